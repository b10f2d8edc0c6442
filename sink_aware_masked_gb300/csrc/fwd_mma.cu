// Forward of sink-aware attention on the warp-level tensor-core path
// (mma.sync m16n8k16, bf16 in, fp32 accumulate), FlashAttention-2 style.
//
// One CTA = 128 query rows of one (sequence, query head); 8 warps, 16 rows
// each.  Key/value tiles of 64 rows stream through a double-buffered,
// XOR-swizzled shared-memory ring filled by cp.async.  Scores live in
// registers, the online softmax runs in the log2 domain, P is re-packed from
// the score accumulators straight into A fragments of the P.V product.
//
// Epilogue (SinkFlex-RL summary page: auxiliary log-sum-exp and the sink
// scaling function; section 5: zero-value sink equivalence):
//   l = ln 2 * (m + log2 sum),  alpha = sigmoid(l - sink[h]),
//   O = alpha * acc / sum,  lse = l.
//
// Only key tiles that intersect the mask are visited: prefix tiles, then the
// causal/window band.  Tiles that are entirely visible skip the predicate.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int D = kHeadDim;
constexpr int BM = 128;
constexpr int BN = 64;
constexpr int NWARP = 8;
constexpr int NTHR = NWARP * 32;
constexpr int SMEM_Q = BM * D * 2;
constexpr int SMEM_KV = BN * D * 2;
constexpr int SMEM_BYTES = SMEM_Q + 4 * SMEM_KV;

struct FwdK {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* sink;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* cu;
  int seqlen;
  long long T;
  int hq, hkv, group;
  MaskParams mask;
  float scale_log2;
  int n_qtiles;
};

__global__ void __launch_bounds__(NTHR, 2) fwd_mma_kernel(const FwdK p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.z);  // longest rows first
  const SeqSpan sp = seq_span(p.cu, p.seqlen, b);
  const int q0 = qt * BM;
  if (q0 >= sp.len) return;
  const int g = h / p.group;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q1 = min(q0 + BM, sp.len) - 1;

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + SMEM_Q;

  const size_t row_q = static_cast<size_t>(p.hq) * D;
  const size_t row_kv = static_cast<size_t>(p.hkv) * D;
  const __nv_bfloat16* qbase = p.q + static_cast<size_t>(sp.start) * row_q + static_cast<size_t>(h) * D;
  const __nv_bfloat16* kbase = p.k + static_cast<size_t>(sp.start) * row_kv + static_cast<size_t>(g) * D;
  const __nv_bfloat16* vbase = p.v + static_cast<size_t>(sp.start) * row_kv + static_cast<size_t>(g) * D;

  for (int i = tid; i < BM * 8; i += NTHR) {
    const int r = i >> 3, c = i & 7, qr = q0 + r;
    const bool ok = qr < sp.len;
    cp_async16(sQ + swz(r, c), qbase + static_cast<size_t>(ok ? qr : 0) * row_q + c * 8, ok);
  }
  cp_async_commit();

  const KeyRange kr = key_range(q0, q1, sp.len, p.mask);
  const int lo_t = kr.lo / BN;
  const int hi_t = kr.hi / BN;
  const int n_pre = min((kr.pre_end + BN - 1) / BN, lo_t);
  const int n_tiles = n_pre + (hi_t - lo_t + 1);

  auto tile_k0 = [&](int i) { return (i < n_pre ? i : lo_t + (i - n_pre)) * BN; };
  auto load_kv = [&](int i, int buf) {
    const int k0 = tile_k0(i);
    const uint32_t dK = sKV + buf * 2 * SMEM_KV, dV = dK + SMEM_KV;
    for (int j = tid; j < BN * 8; j += NTHR) {
      const int r = j >> 3, c = j & 7, kr_ = k0 + r;
      const bool ok = kr_ < sp.len;
      const size_t off = static_cast<size_t>(ok ? kr_ : 0) * row_kv + c * 8;
      cp_async16(dK + swz(r, c), kbase + off, ok);
      cp_async16(dV + swz(r, c), vbase + off, ok);
    }
    cp_async_commit();
  };

  if (n_tiles > 0) load_kv(0, 0);
  cp_async_wait<0>();
  __syncthreads();

  uint32_t qf[4][4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    ldsm_x4(sQ + swz(16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * kk + (lane >> 4)), qf[kk][0], qf[kk][1],
            qf[kk][2], qf[kk][3]);

  float oacc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[j][e] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  const int row_a = q0 + 16 * warp + (lane >> 2);

  for (int i = 0; i < n_tiles; ++i) {
    if (i + 1 < n_tiles) load_kv(i + 1, (i + 1) & 1);
    const int k0 = tile_k0(i);
    const uint32_t tK = sKV + (i & 1) * 2 * SMEM_KV, tV = tK + SMEM_KV;

    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tK + swz(8 * (2 * jp + (lane >> 4)) + (lane & 7), 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma16816(s[2 * jp], qf[kk], b0, b1);
        mma16816(s[2 * jp + 1], qf[kk], b2, b3);
      }
    }

    if (!block_full(q0, BM, k0, BN, sp.len, p.mask)) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = row_a + ((e >> 1) << 3);
          const int kc = k0 + 8 * j + 2 * (lane & 3) + (e & 1);
          if (!visible(r, kc, sp.len, p.mask)) s[j][e] = -INFINITY;
        }
    }

#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float t = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) t = fmaxf(t, fmaxf(s[j][2 * r], s[j][2 * r + 1]));
      t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 1));
      t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 2));
      const float mnew = fmaxf(m_r[r], t * p.scale_log2);
      const float muse = (mnew == -INFINITY) ? 0.f : mnew;
      const float corr = ex2(m_r[r] - muse);
      m_r[r] = mnew;
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        oacc[j][2 * r] *= corr;
        oacc[j][2 * r + 1] *= corr;
        s[j][2 * r] = ex2(fmaf(s[j][2 * r], p.scale_log2, -muse));
        s[j][2 * r + 1] = ex2(fmaf(s[j][2 * r + 1], p.scale_log2, -muse));
        ls += s[j][2 * r] + s[j][2 * r + 1];
      }
      l_r[r] = l_r[r] * corr + ls;
    }

#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tV + swz(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * np + (lane >> 4)), b0, b1, b2, b3);
        mma16816(oacc[2 * np], a, b0, b1);
        mma16816(oacc[2 * np + 1], a, b2, b3);
      }
    }
    cp_async_wait<0>();
    __syncthreads();
  }

  // ---- epilogue: lse, sink scale, normalisation
  const float sinkv = __ldg(p.sink + h);
  float fac[2], lse_r[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_r[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const float lse = (l > 0.f) ? (m_r[r] + __log2f(l)) * kLn2 : -INFINITY;
    const float alpha = 1.f / (1.f + ex2((sinkv - lse) * kLog2e));
    fac[r] = (l > 0.f) ? alpha / l : 0.f;
    lse_r[r] = lse;
  }
  // Stage the bf16 tile in the (now free) Q buffer, then write whole rows.
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = 16 * warp + (lane >> 2) + 8 * r;
      const uint32_t v = pack_bf16(oacc[j][2 * r] * fac[r], oacc[j][2 * r + 1] * fac[r]);
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sQ + swz(row, j) + 4 * (lane & 3)), "r"(v));
    }
  if ((lane & 3) == 0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = row_a + 8 * r;
      if (row < sp.len) p.lse[static_cast<size_t>(h) * p.T + sp.start + row] = lse_r[r];
    }
  }
  __syncthreads();
  __nv_bfloat16* obase = p.o + static_cast<size_t>(sp.start) * row_q + static_cast<size_t>(h) * D;
  for (int i = tid; i < BM * 8; i += NTHR) {
    const int r = i >> 3, c = i & 7;
    if (q0 + r < sp.len) {
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(sQ + swz(r, c)));
      *reinterpret_cast<uint4*>(obase + static_cast<size_t>(q0 + r) * row_q + c * 8) = v;
    }
  }
}

}  // namespace

cudaError_t launch_fwd_mma(const Problem& pr, const FwdArgs& a, cudaStream_t stream) {
  FwdK k;
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.k = static_cast<const __nv_bfloat16*>(a.k);
  k.v = static_cast<const __nv_bfloat16*>(a.v);
  k.sink = a.sink;
  k.o = static_cast<__nv_bfloat16*>(a.o);
  k.lse = a.lse;
  k.cu = pr.cu;
  k.seqlen = pr.seqlen;
  k.T = pr.total_tokens;
  k.hq = pr.hq;
  k.hkv = pr.hkv;
  k.group = pr.hq / pr.hkv;
  k.mask = MaskParams{pr.window, pr.prefix, pr.causal};
  k.scale_log2 = pr.scale * kLog2e;
  k.n_qtiles = ceil_div(pr.seqlen, BM);
  if (k.n_qtiles == 0 || pr.num_seqs == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fwd_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(pr.hq, pr.num_seqs, k.n_qtiles);
  if ((e = prof_begin(g_prof_fwd, stream)) != cudaSuccess) return e;
  fwd_mma_kernel<<<grid, NTHR, SMEM_BYTES, stream>>>(k);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(g_prof_fwd, stream);
}

}  // namespace sa
