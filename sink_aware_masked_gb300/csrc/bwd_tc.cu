// Backward main kernel of sink-aware attention on the 5th-generation tensor
// cores (tcgen05.mma, Tensor Memory accumulators, TMA operand staging).
//
// Math (sink as a zero-value softmax column; SinkFlex-RL section 5 and the
// summary page's alpha = sigmoid(l - s_h); per-head sink gradient from the
// "GPT-OSS agentic RL training" page).  With l' = l + softplus(s_h - l) and
// D = <dO, O> computed by the preprocess kernel:
//   P^T  = exp(S^T - l')            S^T = scale K Q^T   (keys on TMEM lanes)
//   dS^T = P^T (dP^T - D)           dP^T = V dO^T
//   dV  += P^T dO,  dK += dS^T Q (scale applied at the end),  dQ = dS K
// Nothing of size S x S is stored: P and dS live one 128 x 128 tile at a time.
//
// Work unit (one CTA): 128 keys of one sequence and one kv head; the CTA
// loops over the query heads of the GQA group x the 128-row query tiles that
// can see those keys, so dK and dV accumulate in Tensor Memory without
// atomics.  Warp roles (16 warps, four warpgroups):
//   warp 0      loader: K, V once; per step Q and dO tiles by TMA (2-stage
//               ring) and the 128 l' and D values of the query tile by
//               cp.async, all completing on the stage's full barrier.
//   warp 1      MMA issuer and TMEM owner.  Per step t:
//                 S^T(t+1) = K Q^T, dP^T(t+1) = V dO^T   (SS, K-major)
//                 dV += P^T(t) dO(t)    (A = P^T in TMEM, B = dO MN-major)
//                 dK += dS^T(t) Q(t)    (A = dS^T K-major in smem, B = Q MN-major)
//                 dQ(t) = dS(t) K       (A = the same smem tile read MN-major,
//                                        B = K MN-major)
//               so the tensor core computes the next step's S^T and dP^T while
//               the element-wise warps work on this step.
//   warps 4-11  element-wise, two warpgroups splitting the 128 query columns:
//               thread = key row.  P^T -> TMEM (packed bf16), dS^T -> a
//               double-buffered 128 x 128 bf16 shared tile in the
//               128-byte-swizzled layout both MMAs read; at the end one
//               warpgroup writes dV, the other dK.  Fully visible tiles take
//               a path without the mask predicate.
//   warps 12-15 dQ drain: thread = query row; TMEM -> swizzled fp32 staging
//               tile -> TMA reduce-add into the fp32 dQ accumulator.
// Tensor Memory (512 columns): S^T 128 | dP^T 128 | P^T 64 | dV 64 | dK 64 | dQ 64.
// Every mbarrier wait is bounded; a timeout raises the status word and all
// warps leave through the common exit, which drains copies and MMAs first.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

// Optional timeline instrumentation for performance work: compiled in only
// when SA_BWD_TRACE is defined (never in the library build).
#ifdef SA_BWD_TRACE
__device__ long long* g_bwd_trace;
#define SA_TRACE(role, step, ev)                                                                       \
  do {                                                                                                \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && g_bwd_trace != nullptr && (step) < 1024) \
      g_bwd_trace[((role) * 1024 + (step)) * 8 + (ev)] = clock64();                                   \
  } while (0)
#else
#define SA_TRACE(role, step, ev) \
  do {                           \
  } while (0)
#endif

namespace sa {
namespace {

using namespace tc;

constexpr int D = kHeadDim;
constexpr int BN = 128;  // keys per CTA (TMEM lanes)
constexpr int BM = 128;  // query rows per step
constexpr int NS = 2;    // Q/dO stages
constexpr int NTHR = 512;
// setmaxnreg split of the 512 x 128 launch registers: 128 x 56 (loader/MMA
// warpgroup) + 256 x 168 (two element-wise warpgroups) + 128 x 96 (dQ drain)
// = 62,464 <= 65,536.
constexpr int REGS_LOW = 56, REGS_EW = 168, REGS_DQ = 96;
constexpr int TILE = 128 * D * 2;  // 16 KB
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + TILE;
constexpr int OFF_Q = OFF_V + TILE;
constexpr int OFF_DO = OFF_Q + NS * TILE;
constexpr int OFF_DS = OFF_DO + NS * TILE;     // 2 buffers x 32 KB
constexpr int OFF_STG = OFF_DS + 2 * 2 * TILE;  // 32 KB fp32 dQ staging
constexpr int OFF_L = OFF_STG + 2 * TILE;
constexpr int OFF_DL = OFF_L + NS * BM * 4;
constexpr int SMEM_DYN = OFF_DL + NS * BM * 4 + 1024;

constexpr uint32_t TM_S = 0, TM_DP = 128, TM_P = 256, TM_DV = 320, TM_DK = 384, TM_DQ = 448;

struct BwdTcK {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dq;
  const float* lse_log2;
  const float* delta;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* cu;
  int* status;
  int seqlen;
  long long T;
  int hq, hkv, group;
  MaskParams mask;
  float scale, scale_log2;
};

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[NS], q_empty[NS];
  uint64_t s_full, p_full, pv_done, dq_full, dq_free, kv_done, drain;
};

SA_DEV void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) return;
  }
}

SA_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// One 32-column chunk of the element-wise step for this thread's key row:
// P^T = exp2(S^T * scale * log2(e) - l'), dS^T = P^T (dP^T - D), packed to bf16
// pairs.  FULL skips the mask predicate (every pair of the tile visible).
template <bool FULL>
SA_DEV void ew_chunk(uint32_t tS, uint32_t tDP, uint32_t sL, uint32_t sD, int c, float sl2, int q0, int key, int len,
                     const MaskParams& mask, uint32_t (&pp)[16], uint32_t (&dd)[16]) {
  uint32_t sr[32], dr[32];
  tmem_ld32(tS + 32 * c, sr);
  tmem_ld32(tDP + 32 * c, dr);
  tmem_ld_wait();
  reg_fence32(sr);
  reg_fence32(dr);
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 l4 = ld_shared_f4(sL + (32 * c + e) * 4);
    const float4 d4 = ld_shared_f4(sD + (32 * c + e) * 4);
    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
    float pe[4], de[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      pe[u] = ex2(fmaf(__uint_as_float(sr[e + u]), sl2, -lv[u]));
      de[u] = pe[u] * (__uint_as_float(dr[e + u]) - dv[u]);
      if (!FULL) {
        const int q = q0 + 32 * c + e + u;
        if (!(q < len && visible(q, key, len, mask))) pe[u] = de[u] = 0.f;
      }
    }
    pp[e >> 1] = pack_bf16(pe[0], pe[1]);
    pp[(e >> 1) + 1] = pack_bf16(pe[2], pe[3]);
    dd[e >> 1] = pack_bf16(de[0], de[1]);
    dd[(e >> 1) + 1] = pack_bf16(de[2], de[3]);
  }
}

__global__ void __launch_bounds__(NTHR, 1) bwd_tc_kernel(const __grid_constant__ BwdTcK p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;
  const SeqSpan sp = seq_span(p.cu, p.seqlen, blockIdx.y);
  const int k0 = static_cast<int>(blockIdx.z) * BN;
  if (k0 >= sp.len) return;
  const int k1 = min(k0 + BN, sp.len) - 1;
  int qlo, qhi;
  query_range(k0, k1, sp.len, p.mask, qlo, qhi);
  const int qt_lo = qlo / BM, nq = qhi / BM - qt_lo + 1;
  const int nsteps = p.group * nq;
  auto step_head = [&](int t) { return g * p.group + t / nq; };
  auto step_q0 = [&](int t) { return (qt_lo + t % nq) * BM; };

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t b_kv = smem_u32(&bars.kv_full), b_s = smem_u32(&bars.s_full), b_p = smem_u32(&bars.p_full);
  const uint32_t b_pv = smem_u32(&bars.pv_done), b_dqf = smem_u32(&bars.dq_full), b_dqe = smem_u32(&bars.dq_free);
  const uint32_t b_done = smem_u32(&bars.kv_done), b_dr = smem_u32(&bars.drain);
  auto b_qf = [&](int s) { return smem_u32(&bars.q_full[s]); };
  auto b_qe = [&](int s) { return smem_u32(&bars.q_empty[s]); };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(b_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_qf(s), 33);  // 32 cp.async arrivals + the TMA expect-tx arrival
      mbar_init(b_qe(s), 1);
    }
    mbar_init(b_s, 1);
    mbar_init(b_p, 8);
    mbar_init(b_pv, 1);
    mbar_init(b_dqf, 1);
    mbar_init(b_dqe, 4);
    mbar_init(b_done, 1);
    mbar_init(b_dr, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const Abort ab{&abort_flag, p.status};

  if (warp < 4) {
    regs_dec<REGS_LOW>();
    if (warp == 0) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      tma_prefetch_map(&p.tm_do);
      mbar_expect_tx(b_kv, 2 * TILE);
      tma_load_2d(sb + OFF_K, &p.tm_k, g * D, sp.start + k0, b_kv);
      tma_load_2d(sb + OFF_V, &p.tm_v, g * D, sp.start + k0, b_kv);
    }
    int issued = 0;
    for (int t = 0; t < nsteps; ++t) {
      const int s = t % NS;
      if (t >= NS && !__all_sync(0xffffffffu, mbar_wait(b_qe(s), ((t / NS) - 1) & 1, ab))) break;
      if (lane == 0) SA_TRACE(0, t, 0);
      const int h = step_head(t), q0 = step_q0(t);
      // l' and D of the 128 query rows: asynchronous 4-byte copies that
      // complete on the stage's full barrier (rows past the sequence end read
      // row 0 and are masked by the element-wise warps).
#pragma unroll
      for (int r = lane; r < BM; r += 32) {
        const int qq = q0 + r;
        const size_t idx = static_cast<size_t>(h) * p.T + sp.start + (qq < sp.len ? qq : 0);
        cp_async4(sb + OFF_L + (s * BM + r) * 4, p.lse_log2 + idx);
        cp_async4(sb + OFF_DL + (s * BM + r) * 4, p.delta + idx);
      }
      cp_async_arrive_noinc(b_qf(s));
      if (lane == 0) {
        mbar_expect_tx(b_qf(s), 2 * TILE);
        tma_load_2d(sb + OFF_Q + s * TILE, &p.tm_q, h * D, sp.start + q0, b_qf(s));
        tma_load_2d(sb + OFF_DO + s * TILE, &p.tm_do, h * D, sp.start + q0, b_qf(s));
        SA_TRACE(0, t, 1);
      }
      issued = t + 1;
    }
    if (lane == 0 && abort_flag) {
      wait_drain(b_kv, 0);
      for (int t = max(0, issued - NS); t < issued; ++t) wait_drain(b_qf(t % NS), (t / NS) & 1);
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(BN, BM, false, false);   // S^T, dP^T: 128 keys x 128 queries
      const uint32_t id_kv = idesc_bf16(BN, D, false, true);    // dV, dK: 128 keys x 64
      const uint32_t id_q = idesc_bf16(BM, D, true, true);      // dQ: 128 queries x 64
      const uint32_t sK = sb + OFF_K, sV = sb + OFF_V;
      auto issue_s_dp = [&](int s) {
        const uint32_t sQ = sb + OFF_Q + s * TILE, sO = sb + OFF_DO + s * TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_ss(tmem + TM_S, sdesc_sw128(sK + kk * 32, 16, 1024), sdesc_sw128(sQ + kk * 32, 16, 1024), id_s, kk > 0);
          mma_ss(tmem + TM_DP, sdesc_sw128(sV + kk * 32, 16, 1024), sdesc_sw128(sO + kk * 32, 16, 1024), id_s,
                 kk > 0);
        }
      };
      bool ok = mbar_wait(b_kv, 0, ab) && mbar_wait(b_qf(0), 0, ab);
      if (ok) {
        fence_after_sync();
        issue_s_dp(0);
        mma_commit(b_s);
      }
      for (int t = 0; ok && t < nsteps; ++t) {
        const int s = t % NS, db = t & 1;
        SA_TRACE(1, t, 0);
        if (!(ok = mbar_wait(b_p, t & 1, ab))) break;
        SA_TRACE(1, t, 1);
        fence_after_sync();
        if (t + 1 < nsteps) {
          if (!(ok = mbar_wait(b_qf((t + 1) % NS), ((t + 1) / NS) & 1, ab))) break;
          fence_after_sync();
          SA_TRACE(1, t, 2);
          issue_s_dp((t + 1) % NS);
          mma_commit(b_s);
        }
        SA_TRACE(1, t, 3);
        const uint32_t sQ = sb + OFF_Q + s * TILE, sO = sb + OFF_DO + s * TILE;
        const uint32_t sdS = sb + OFF_DS + db * 2 * TILE;
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk) {
          const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + TM_DV, tmem + TM_P + kk * 8, sdesc_sw128(sO + kk * 2048, 16, 1024), id_kv, acc);
          mma_ss(tmem + TM_DK, sdesc_sw128(sdS + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(sQ + kk * 2048, 16, 1024), id_kv, acc);
        }
        mma_commit(b_pv);
        mma_commit(b_qe(s));  // Q(t), dO(t), l'(t), D(t) have no later reader
        SA_TRACE(1, t, 4);
        if (t > 0) {
          if (!(ok = mbar_wait(b_dqe, (t - 1) & 1, ab))) break;
          fence_after_sync();
        }
        SA_TRACE(1, t, 5);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ss(tmem + TM_DQ, sdesc_sw128(sdS + kk * 2048, TILE, 1024), sdesc_sw128(sK + kk * 2048, 16, 1024), id_q,
                 kk > 0);
        mma_commit(b_dqf);
      }
      if (ok) mma_commit(b_done);
      mma_commit(b_dr);
      wait_drain(b_dr, 0);
    }
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ element-wise
    regs_inc<REGS_EW>();
    const int half = (warp - 4) >> 2;  // query columns [64 * half, 64 * half + 64)
    const int kr = (warp & 3) * 32 + lane;
    const int key = k0 + kr;
    const uint32_t lb = lane_base(warp);
    const uint32_t tS = tmem + TM_S + lb, tDP = tmem + TM_DP + lb, tP = tmem + TM_P + lb;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < nsteps; ++t) {
      const int s = t % NS;
      if (tid == 128) SA_TRACE(2, t, 0);
      ok = __all_sync(0xffffffffu, mbar_wait(b_s, t & 1, ab)) &&
           __all_sync(0xffffffffu, mbar_wait(b_qf(s), (t / NS) & 1, ab));
      if (!ok) break;
      if (tid == 128) SA_TRACE(2, t, 1);
      fence_after_sync();
      const int q0 = step_q0(t);
      const bool full = block_full(q0, BM, k0, BN, sp.len, p.mask);
      const uint32_t rowb = sb + OFF_DS + (t & 1) * 2 * TILE + half * TILE + kr * 128;
      const uint32_t sL = sb + OFF_L + s * BM * 4, sD = sb + OFF_DL + s * BM * 4;
#pragma unroll 1
      for (int cc2 = 0; cc2 < 2; ++cc2) {
        const int c = 2 * half + cc2;
        uint32_t pp[16], dd[16];
        if (full)
          ew_chunk<true>(tS, tDP, sL, sD, c, sl2, q0, key, sp.len, p.mask, pp, dd);
        else
          ew_chunk<false>(tS, tDP, sL, sD, c, sl2, q0, key, sp.len, p.mask, pp, dd);
        if (cc2 == 0 && tid == 128) SA_TRACE(2, t, 2);
        if (cc2 == 0 && t > 0) {
          // P^T of the previous step is read by dV(t-1): wait for it before overwriting.
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_pv, (t - 1) & 1, ab)))) break;
          fence_after_sync();
        }
        if (cc2 == 0 && tid == 128) SA_TRACE(2, t, 3);
        tmem_st16(tP + 16 * c, pp);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int cc = cc2 * 4 + i;
          st_shared_v4(rowb + ((cc ^ (kr & 7)) << 4), dd[4 * i], dd[4 * i + 1], dd[4 * i + 2], dd[4 * i + 3]);
        }
      }
      if (!ok) break;
      tmem_st_wait();
      fence_before_sync();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p);
      if (tid == 128) SA_TRACE(2, t, 4);
    }
    ok = ok && __all_sync(0xffffffffu, mbar_wait(b_done, 0, ab));
    if (ok) {
      // First half writes dV, second half writes dK (scaled).
      fence_after_sync();
      uint32_t a[32], b2[32];
      const uint32_t src = tmem + (half ? TM_DK : TM_DV) + lb;
      tmem_ld32(src, a);
      tmem_ld32(src + 32, b2);
      tmem_ld_wait();
      reg_fence32(a);
      reg_fence32(b2);
      const float mul = half ? p.scale : 1.f;
      if (key < sp.len) {
        __nv_bfloat16* dst = (half ? p.dk : p.dv) + (static_cast<size_t>(sp.start + key) * p.hkv + g) * D;
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          d4[c] = make_uint4(pack_bf16(__uint_as_float(a[8 * c]) * mul, __uint_as_float(a[8 * c + 1]) * mul),
                             pack_bf16(__uint_as_float(a[8 * c + 2]) * mul, __uint_as_float(a[8 * c + 3]) * mul),
                             pack_bf16(__uint_as_float(a[8 * c + 4]) * mul, __uint_as_float(a[8 * c + 5]) * mul),
                             pack_bf16(__uint_as_float(a[8 * c + 6]) * mul, __uint_as_float(a[8 * c + 7]) * mul));
          d4[4 + c] = make_uint4(pack_bf16(__uint_as_float(b2[8 * c]) * mul, __uint_as_float(b2[8 * c + 1]) * mul),
                                 pack_bf16(__uint_as_float(b2[8 * c + 2]) * mul, __uint_as_float(b2[8 * c + 3]) * mul),
                                 pack_bf16(__uint_as_float(b2[8 * c + 4]) * mul, __uint_as_float(b2[8 * c + 5]) * mul),
                                 pack_bf16(__uint_as_float(b2[8 * c + 6]) * mul, __uint_as_float(b2[8 * c + 7]) * mul));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain
    regs_dec<REGS_DQ>();
    const int qr = (warp & 3) * 32 + lane;
    const bool leader = (warp == 12 && lane == 0);
    const uint32_t lb = lane_base(warp);
    const uint32_t tQ = tmem + TM_DQ + lb;
    const uint32_t stg = sb + OFF_STG;
    bool ok = true;
    for (int t = 0; t < nsteps; ++t) {
      if (leader) SA_TRACE(3, t, 0);
      ok = __all_sync(0xffffffffu, mbar_wait(b_dqf, t & 1, ab));
      if (!ok) break;
      if (leader) SA_TRACE(3, t, 1);
      fence_after_sync();
      uint32_t a[32], b2[32];
      tmem_ld32(tQ, a);
      tmem_ld32(tQ + 32, b2);
      tmem_ld_wait();
      reg_fence32(a);
      reg_fence32(b2);
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_dqe);
      const int h = step_head(t), q0 = step_q0(t);
      const bool valid = q0 + qr < sp.len;
      if (leader) bulk_wait_read0();
      if (leader) SA_TRACE(3, t, 2);
      named_sync(1, 128);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t sw = ((i ^ (qr & 7)) << 4) + qr * 128;
        st_shared_v4(stg + sw, valid ? a[4 * i] : 0u, valid ? a[4 * i + 1] : 0u, valid ? a[4 * i + 2] : 0u,
                     valid ? a[4 * i + 3] : 0u);
        st_shared_v4(stg + TILE + sw, valid ? b2[4 * i] : 0u, valid ? b2[4 * i + 1] : 0u,
                     valid ? b2[4 * i + 2] : 0u, valid ? b2[4 * i + 3] : 0u);
      }
      fence_async_smem();
      named_sync(1, 128);
      if (leader) {
        tma_reduce_add_2d(&p.tm_dq, h * D, sp.start + q0, stg);
        tma_reduce_add_2d(&p.tm_dq, h * D + 32, sp.start + q0, stg + TILE);
        bulk_commit();
        SA_TRACE(3, t, 3);
      }
    }
    if (leader) bulk_wait0();
  }
  // ------------------------------------------------------------ common exit
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd_tc_main(const Problem& pr, const BwdArgs& a, int* status, cudaStream_t stream) {
  const int n_kt = ceil_div(pr.seqlen, BN);
  if (n_kt == 0 || pr.num_seqs == 0 || pr.total_tokens == 0) return cudaSuccess;
  BwdTcK k;
  if (!make_rows_map(&k.tm_q, a.q, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_do, a.dout, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_k, a.k, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_v, a.v, pr.total_tokens, pr.hkv, BN) ||
      !make_f32_rows_map(&k.tm_dq, a.dq_accum, pr.total_tokens, pr.hq, BM))
    return cudaErrorInvalidValue;
  k.lse_log2 = a.lse_log2;
  k.delta = a.delta;
  k.dk = static_cast<__nv_bfloat16*>(a.dk);
  k.dv = static_cast<__nv_bfloat16*>(a.dv);
  k.cu = pr.cu;
  k.status = status;
  k.seqlen = pr.seqlen;
  k.T = pr.total_tokens;
  k.hq = pr.hq;
  k.hkv = pr.hkv;
  k.group = pr.hq / pr.hkv;
  k.mask = MaskParams{pr.window, pr.prefix, pr.causal};
  k.scale = pr.scale;
  k.scale_log2 = pr.scale * kLog2e;
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
  if (e != cudaSuccess) return e;
  dim3 grid(pr.hkv, pr.num_seqs, n_kt);
  if ((e = prof_begin(g_prof_bwd, stream)) != cudaSuccess) return e;
  bwd_tc_kernel<<<grid, NTHR, SMEM_DYN, stream>>>(k);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(g_prof_bwd, stream);
}

}  // namespace sa
