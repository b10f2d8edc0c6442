// Backward of sink-aware attention on the warp-level tensor-core path
// (mma.sync m16n8k16, bf16 in, fp32 accumulate).
//
// Math (explicit sink column with zero value; SinkFlex-RL section 5 and the
// summary page's alpha = sigmoid(l - s_h); per-head sink gradient from the
// "GPT-OSS agentic RL training" page):
//   l'  = l + softplus(s_h - l)        log-normaliser including the sink
//   P   = exp(s - l')                  probabilities of the real keys
//   D   = <dO, O>                      O is the final, alpha-scaled output
//   dS  = P (dO.V^T - D)
//   dQ  = scale dS K,  dK = scale dS^T Q,  dV = P^T dO
//   dsink[h] = -sum_rows (1 - alpha) D,   1 - alpha = sigmoid(s_h - l)
//
// Three kernels:
//   bwd_pre   : one pass over O and dO: D, l' (log2 units), per-block partial
//               dsink sums, zeroes the fp32 dQ accumulator.  HBM-bound.
//   bwd_main  : one CTA per (sequence, kv head, 128-key tile).  Loops over the
//               query heads of the GQA group and the 64-row query tiles that
//               intersect the mask; dK and dV stay in registers for the whole
//               loop (no atomics), dQ partials go to the fp32 accumulator with
//               atomic adds.  Probabilities are recomputed from l', nothing of
//               size S x S is ever stored.
//   dq_convert: dQ = scale * accumulator -> bf16; one extra block reduces the
//               dsink partials in a fixed order (deterministic).
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int D = kHeadDim;

// ------------------------------------------------------------------ preprocess
struct PreK {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  const float* sink;
  float* delta;
  float* lse_log2;
  float* dq_accum;
  float* dsink_part;
  long long T;
  int hq;
};

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(x[i]);
    const float2 fy = __bfloat1622float2(y[i]);
    s = fmaf(fx.x, fy.x, s);
    s = fmaf(fx.y, fy.y, s);
  }
  return s;
}

__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreK p) {
  const int sub = threadIdx.x & 7;   // 16-byte chunk of a 128-byte row
  const int hs = threadIdx.x >> 3;   // 0..31
  const long long t0 = static_cast<long long>(blockIdx.x) * kPreTokens;
  const long long t1 = min(t0 + kPreTokens, p.T);
  float acc[kMaxHeadsQ / 32];
#pragma unroll
  for (int i = 0; i < kMaxHeadsQ / 32; ++i) acc[i] = 0.f;
  for (long long t = t0; t < t1; ++t) {
#pragma unroll
    for (int hi = 0; hi < kMaxHeadsQ / 32; ++hi) {
      if (hi * 32 >= p.hq) break;
      const int h = hi * 32 + hs;
      const bool ok = h < p.hq;
      float dot = 0.f;
      if (ok) {
        const size_t base = (static_cast<size_t>(t) * p.hq + h) * D + sub * 8;
        const uint4 ov = __ldg(reinterpret_cast<const uint4*>(p.o + base));
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(p.dout + base));
        dot = dot8_bf16(ov, gv);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4*>(p.dq_accum + base)[0] = z;
        reinterpret_cast<float4*>(p.dq_accum + base)[1] = z;
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      dot += __shfl_xor_sync(0xffffffffu, dot, 4);
      if (ok && sub == 0) {
        const size_t idx = static_cast<size_t>(h) * p.T + t;
        const float l = p.lse[idx];
        const float x = __ldg(p.sink + h) - l;
        const float softplus = fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x)));
        p.lse_log2[idx] = (l + softplus) * kLog2e;
        p.delta[idx] = dot;
        const float one_minus_alpha = 1.f / (1.f + __expf(-x));
        acc[hi] -= one_minus_alpha * dot;
      }
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int hi = 0; hi < kMaxHeadsQ / 32; ++hi) {
      const int h = hi * 32 + hs;
      if (h < p.hq) p.dsink_part[static_cast<size_t>(blockIdx.x) * p.hq + h] = acc[hi];
    }
  }
}

// ------------------------------------------------------------------ main
constexpr int BNK = 128;  // keys per CTA: 8 warps x 16
constexpr int BMQ = 64;   // query rows per step
constexpr int NTHR = 256;
constexpr int TILE_Q = BMQ * D * 2;  // 8 KB
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + BNK * D * 2;  // reused as the dS^T tile after V is in registers
constexpr int OFF_Q = OFF_V + BNK * D * 2;
constexpr int OFF_DO = OFF_Q + 2 * TILE_Q;
constexpr int OFF_L = OFF_DO + 2 * TILE_Q;
constexpr int OFF_DL = OFF_L + 2 * BMQ * 4;
constexpr int SMEM_MAIN = OFF_DL + 2 * BMQ * 4;

struct MainK {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* dout;
  const float* lse_log2;
  const float* delta;
  float* dq_accum;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* cu;
  int seqlen;
  long long T;
  int hq, hkv, group;
  MaskParams mask;
  float scale, scale_log2;
};

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}

__global__ void __launch_bounds__(NTHR, 1) bwd_main_kernel(const MainK p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int g = blockIdx.x, b = blockIdx.y;
  const SeqSpan sp = seq_span(p.cu, p.seqlen, b);
  const int k0 = static_cast<int>(blockIdx.z) * BNK;
  if (k0 >= sp.len) return;
  const int k1 = min(k0 + BNK, sp.len) - 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int qlo, qhi;
  query_range(k0, k1, sp.len, p.mask, qlo, qhi);
  const int qt_lo = qlo / BMQ, nq = qhi / BMQ - qt_lo + 1;
  const int nsteps = p.group * nq;

  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + OFF_K, sV = s0 + OFF_V, sQ = s0 + OFF_Q, sdO = s0 + OFF_DO;
  const uint32_t sL = s0 + OFF_L, sDl = s0 + OFF_DL;
  const float* fL = reinterpret_cast<const float*>(smem + OFF_L);
  const float* fDl = reinterpret_cast<const float*>(smem + OFF_DL);
  const uint32_t sdS = sV;

  const size_t row_q = static_cast<size_t>(p.hq) * D;
  const size_t row_kv = static_cast<size_t>(p.hkv) * D;
  {
    const __nv_bfloat16* kb = p.k + static_cast<size_t>(sp.start) * row_kv + static_cast<size_t>(g) * D;
    const __nv_bfloat16* vb = p.v + static_cast<size_t>(sp.start) * row_kv + static_cast<size_t>(g) * D;
    for (int i = tid; i < BNK * 8; i += NTHR) {
      const int r = i >> 3, c = i & 7, kr = k0 + r;
      const bool ok = kr < sp.len;
      const size_t off = static_cast<size_t>(ok ? kr : 0) * row_kv + c * 8;
      cp_async16(sK + swz(r, c), kb + off, ok);
      cp_async16(sV + swz(r, c), vb + off, ok);
    }
    cp_async_commit();
  }

  auto prefetch = [&](int s, int buf) {
    const int h = g * p.group + s / nq;
    const int q0 = (qt_lo + s % nq) * BMQ;
    const __nv_bfloat16* qb = p.q + static_cast<size_t>(sp.start) * row_q + static_cast<size_t>(h) * D;
    const __nv_bfloat16* ob = p.dout + static_cast<size_t>(sp.start) * row_q + static_cast<size_t>(h) * D;
    for (int i = tid; i < BMQ * 8; i += NTHR) {
      const int r = i >> 3, c = i & 7, qr = q0 + r;
      const bool ok = qr < sp.len;
      const size_t off = static_cast<size_t>(ok ? qr : 0) * row_q + c * 8;
      cp_async16(sQ + buf * TILE_Q + swz(r, c), qb + off, ok);
      cp_async16(sdO + buf * TILE_Q + swz(r, c), ob + off, ok);
    }
    if (tid < 2 * BMQ) {
      const int r = tid & (BMQ - 1), qr = q0 + r;
      const bool ok = qr < sp.len;
      const size_t idx = static_cast<size_t>(h) * p.T + sp.start + (ok ? qr : 0);
      if (tid < BMQ)
        cp_async4(sL + (buf * BMQ + r) * 4, p.lse_log2 + idx, ok);
      else
        cp_async4(sDl + (buf * BMQ + r) * 4, p.delta + idx, ok);
    }
    cp_async_commit();
  };

  prefetch(0, 0);
  cp_async_wait<0>();
  __syncthreads();

  uint32_t kf[4][4], vf[4][4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t off = swz(16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * kk + (lane >> 4));
    ldsm_x4(sK + off, kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3]);
    ldsm_x4(sV + off, vf[kk][0], vf[kk][1], vf[kk][2], vf[kk][3]);
  }
  __syncthreads();  // V tile now lives in registers; its buffer becomes dS^T

  float dva[8][4], dka[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) dva[j][e] = dka[j][e] = 0.f;

  const int key_a = k0 + 16 * warp + (lane >> 2);

  for (int s = 0; s < nsteps; ++s) {
    const int buf = s & 1;
    if (s + 1 < nsteps) prefetch(s + 1, buf ^ 1);
    const int h = g * p.group + s / nq;
    const int q0 = (qt_lo + s % nq) * BMQ;
    const uint32_t tQ = sQ + buf * TILE_Q, tdO = sdO + buf * TILE_Q;

    float st[8][4], dpt[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[j][e] = dpt[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        const uint32_t off = swz(8 * (2 * jp + (lane >> 4)) + (lane & 7), 2 * kk + ((lane >> 3) & 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tQ + off, b0, b1, b2, b3);
        mma16816(st[2 * jp], kf[kk], b0, b1);
        mma16816(st[2 * jp + 1], kf[kk], b2, b3);
        ldsm_x4(tdO + off, b0, b1, b2, b3);
        mma16816(dpt[2 * jp], vf[kk], b0, b1);
        mma16816(dpt[2 * jp + 1], vf[kk], b2, b3);
      }
    }

    const bool full = block_full(q0, BMQ, k0, BNK, sp.len, p.mask);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qc = 8 * j + 2 * (lane & 3) + (e & 1);
        const float lq = fL[buf * BMQ + qc];
        const float dq = fDl[buf * BMQ + qc];
        float pv = ex2(fmaf(st[j][e], p.scale_log2, -lq));
        if (!full) {
          const int key = key_a + ((e >> 1) << 3);
          const int qr = q0 + qc;
          if (!(qr < sp.len && visible(qr, key, sp.len, p.mask))) pv = 0.f;
        }
        st[j][e] = pv;
        dpt[j][e] = pv * (dpt[j][e] - dq);
      }

    // dV += P^T dO, dK += dS^T Q
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ap[4], ad[4];
      ap[0] = pack_bf16(st[2 * kk][0], st[2 * kk][1]);
      ap[1] = pack_bf16(st[2 * kk][2], st[2 * kk][3]);
      ap[2] = pack_bf16(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      ap[3] = pack_bf16(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      ad[0] = pack_bf16(dpt[2 * kk][0], dpt[2 * kk][1]);
      ad[1] = pack_bf16(dpt[2 * kk][2], dpt[2 * kk][3]);
      ad[2] = pack_bf16(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      ad[3] = pack_bf16(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const uint32_t off = swz(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * np + (lane >> 4));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tdO + off, b0, b1, b2, b3);
        mma16816(dva[2 * np], ap, b0, b1);
        mma16816(dva[2 * np + 1], ap, b2, b3);
        ldsm_x4_t(tQ + off, b0, b1, b2, b3);
        mma16816(dka[2 * np], ad, b0, b1);
        mma16816(dka[2 * np + 1], ad, b2, b3);
      }
      // dS^T (bf16) to shared memory for the dQ product
      const int row = 16 * warp + (lane >> 2);
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + swz(row, 2 * kk) + 4 * (lane & 3)), "r"(ad[0]));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + swz(row + 8, 2 * kk) + 4 * (lane & 3)), "r"(ad[1]));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + swz(row, 2 * kk + 1) + 4 * (lane & 3)), "r"(ad[2]));
      asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(sdS + swz(row + 8, 2 * kk + 1) + 4 * (lane & 3)), "r"(ad[3]));
    }
    __syncthreads();

    // dQ(64 x 64) = dS (64 x 128) K (128 x 64); warp owns 16 rows x 32 columns.
    {
      float dqa[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) dqa[n][e] = 0.f;
      const int rq = warp & 3, cq = warp >> 2;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4];
        ldsm_x4_t(sdS + swz(16 * kk + (lane & 7) + 8 * (lane >> 4), 2 * rq + ((lane >> 3) & 1)), a[0], a[1], a[2],
                  a[3]);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sK + swz(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), 4 * cq + 2 * np + (lane >> 4)), b0, b1,
                    b2, b3);
          mma16816(dqa[2 * np], a, b0, b1);
          mma16816(dqa[2 * np + 1], a, b2, b3);
        }
      }
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int qr = q0 + 16 * rq + (lane >> 2) + 8 * e2;
        if (qr < sp.len) {
          float* dst = p.dq_accum + (static_cast<size_t>(sp.start + qr) * p.hq + h) * D + 32 * cq + 2 * (lane & 3);
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            atomicAdd(dst + 8 * n, dqa[n][2 * e2]);
            atomicAdd(dst + 8 * n + 1, dqa[n][2 * e2 + 1]);
          }
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();
  }

  // ---- write dV and dK (scaled) through the Q buffers
  const uint32_t stage = sQ;  // 2 x 8 KB = one 128 x 64 bf16 tile
  __nv_bfloat16* dvb = p.dv + static_cast<size_t>(sp.start) * row_kv + static_cast<size_t>(g) * D;
  __nv_bfloat16* dkb = p.dk + static_cast<size_t>(sp.start) * row_kv + static_cast<size_t>(g) * D;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const float mul = which ? p.scale : 1.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = 16 * warp + (lane >> 2) + 8 * r;
        const float x0 = which ? dka[j][2 * r] : dva[j][2 * r];
        const float x1 = which ? dka[j][2 * r + 1] : dva[j][2 * r + 1];
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(stage + swz(row, j) + 4 * (lane & 3)),
                     "r"(pack_bf16(x0 * mul, x1 * mul)));
      }
    __syncthreads();
    __nv_bfloat16* dst = which ? dkb : dvb;
    for (int i = tid; i < BNK * 8; i += NTHR) {
      const int r = i >> 3, c = i & 7;
      if (k0 + r < sp.len) {
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(stage + swz(r, c)));
        *reinterpret_cast<uint4*>(dst + static_cast<size_t>(k0 + r) * row_kv + c * 8) = v;
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ convert
struct ConvK {
  const float* acc;
  __nv_bfloat16* dq;
  long long n8;  // number of 8-element groups
  float scale;
  const float* part;
  int nparts;
  int hq;
  float* dsink;
};

__global__ void __launch_bounds__(256) dq_convert_kernel(const ConvK p) {
  if (blockIdx.x == gridDim.x - 1) {
    // Fixed-order reduction of the dsink partials: warp w takes heads w, w+8, ...
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < p.hq; h += 8) {
      float s = 0.f;
      for (int i = lane; i < p.nparts; i += 32) s += p.part[static_cast<size_t>(i) * p.hq + h];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) p.dsink[h] = s;
    }
    return;
  }
  const long long stride = static_cast<long long>(gridDim.x - 1) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(p.acc)[2 * i];
    const float4 c = reinterpret_cast<const float4*>(p.acc)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a.x * p.scale, a.y * p.scale);
    o.y = pack_bf16(a.z * p.scale, a.w * p.scale);
    o.z = pack_bf16(c.x * p.scale, c.y * p.scale);
    o.w = pack_bf16(c.z * p.scale, c.w * p.scale);
    reinterpret_cast<uint4*>(p.dq)[i] = o;
  }
}

}  // namespace

cudaError_t launch_bwd(const Problem& pr, const BwdArgs& a, int* status, cudaStream_t stream) {
  const long long T = pr.total_tokens;
  {
    PreK k{static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.sink,
           a.delta, a.lse_log2, a.dq_accum, a.dsink_part, T, pr.hq};
    if (a.preprocess_blocks > 0) bwd_pre_kernel<<<a.preprocess_blocks, 256, 0, stream>>>(k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    cudaError_t e = launch_bwd_tc_main(pr, a, status, stream);
    if (e != cudaSuccess) return e;
  }
  {
    ConvK k{a.dq_accum, static_cast<__nv_bfloat16*>(a.dq), T * pr.hq * D / 8, pr.scale, a.dsink_part,
            a.preprocess_blocks, pr.hq, a.dsink};
    long long blocks = (k.n8 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    dq_convert_kernel<<<static_cast<int>(blocks) + 1, 256, 0, stream>>>(k);
  }
  return cudaGetLastError();
}

}  // namespace sa
