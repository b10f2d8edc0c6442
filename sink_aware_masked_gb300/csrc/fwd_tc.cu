// Forward of sink-aware attention on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in Tensor Memory, operands staged by TMA).
//
// Work unit (one CTA): 128 query rows of one sequence for a PAIR of query
// heads of the same GQA group, so both heads share every K/V tile that TMA
// brings in.  Warp roles (12 warps, three warpgroups):
//   warp 0      TMA producer: Q of both heads once, then K and V tiles of
//               128 keys through an NS-stage ring (separate K and V barriers
//               so S = QK^T can start before V lands).
//   warp 1      MMA issuer (one thread) and TMEM owner:
//               S_i = Q_i K_j^T   (M=128, N=128, K=64; A = Q_i in TMEM,
//                                   B = K_j K-major in smem)
//               O_i += P_i V_j    (M=128, N=64,  K=128; A = P_i in TMEM,
//                                   B = V_j MN-major in smem)
//               issued ping-pong between the two heads so the tensor core
//               works on one head while the other head's softmax runs.
//   warps 2-3   idle (they only complete the first warpgroup, which hands
//               its registers to the softmax warpgroups: 64 vs 216 each)
//   warps 4-7   softmax of head 0, warps 8-11 softmax of head 1: the thread
//               in lane l of warp w owns query row 32 * (w % 4) + l (its TMEM
//               lane), so row max and row sum need
//               no shuffles.  Online softmax in log2 units; the O rescale is
//               skipped unless the running max grows by more than 8 (P stays
//               below 2^8, exact in fp32 sums); P is written to TMEM as
//               packed bf16.  One exponential in four runs on the FMA pipe
//               (exp2_fma) to offload the MUFU unit; the row maximum uses independent
//               three-input max chains; scale/subtract and row
//               sums use packed f32x2 arithmetic.  At start each softmax
//               warpgroup copies its head's Q tile into TMEM.
// Tensor Memory (448 of 512 columns): S0 | S1 (128 each; P_i overwrites the
// first 64 columns of S_i) | O0 | O1 (64 each) | Q0 | Q1 (32 each, A operands).
//
// Epilogue (SinkFlex-RL summary page: auxiliary log-sum-exp and the sink
// scaling function; section 5: zero-value sink equivalence):
//   l = ln2 * (m + log2 sum),  alpha = sigmoid(l - sink[h]),  O = alpha * acc / sum.
//
// Key tiles outside the mask are never loaded: the prefix tiles, then the
// causal/window band; fully visible tiles skip the per-element predicate.
// Every mbarrier wait is bounded (see tc.cuh); a timeout raises the library
// status word and every warp leaves through the common exit path, which
// drains outstanding TMA loads and MMAs before Tensor Memory is freed.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

#include <algorithm>

// Optional timeline instrumentation for performance work: compiled in only
// when SA_FWD_TRACE is defined (never in the library build).
#ifdef SA_FWD_TRACE
__device__ long long* g_fwd_trace;
#define SA_TRACE(role, step, ev)                                                                        \
  do {                                                                                                 \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && g_fwd_trace != nullptr && (step) < 256) \
      g_fwd_trace[((role) * 256 + (step)) * 8 + (ev)] = clock64();                                     \
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
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int NS = 3;
constexpr int NTHR = 384;
// Register split after setmaxnreg: 128 x 64 + 256 x 216 = 63,488 <= 384 x 168.
constexpr int REGS_LOW = 64, REGS_HIGH = 216;
constexpr int TILE = BM * D * 2;  // 16 KB: 128 rows x 128 bytes
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + 2 * TILE;
constexpr int OFF_V = OFF_K + NS * TILE;
constexpr int SMEM_DYN = OFF_V + NS * TILE + 1024;  // + alignment slack

// S_i at 128 i (P_i, packed bf16, overwrites its first 64 columns), O_i at
// 256 + 64 i, Q_i (packed bf16, A operand of S_i) at 384 + 32 i.
constexpr uint32_t TM_S = 0, TM_O = 256, TM_Q = 384;

struct FwdTcK {
  CUtensorMap tm_q, tm_k, tm_v;
  const float* sink;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* cu;
  int* status;
  int seqlen;
  long long T;
  int hq, hkv, group, nh;
  MaskParams mask;
  float scale_log2;
  int n_items;
  uint32_t items[4096];  // this launch's slice of the work list: b | (query tile << 16)
};
static_assert(sizeof(FwdTcK) < 32000, "kernel parameter block too large");

struct Bars {
  uint64_t q_full;
  uint64_t k_full[NS], v_full[NS], kv_empty[NS];
  uint64_t s_full[2], p_full[2], q_tmem[2];
  uint64_t o_final, drain;
};

// Waits without the abort short-cut: used on the exit path to let copies and
// MMAs that are still in flight finish before the CTA leaves.
SA_DEV void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) return;
  }
}

__global__ void __launch_bounds__(NTHR, 1) fwd_tc_kernel(const __grid_constant__ FwdTcK p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nh = p.nh;
  const int h0 = static_cast<int>(blockIdx.x) * nh;
  const int g = h0 / p.group;
  const uint32_t item = p.items[blockIdx.y];  // longest first
  const SeqSpan sp = seq_span(p.cu, p.seqlen, static_cast<int>(item & 0xFFFFu));
  const int q0 = static_cast<int>(item >> 16) * BM;
  if (q0 >= sp.len) return;
  const int q1 = min(q0 + BM, sp.len) - 1;
  const KeyRange kr = key_range(q0, q1, sp.len, p.mask);
  const int lo_t = kr.lo / BN, hi_t = kr.hi / BN;
  const int n_pre = min((kr.pre_end + BN - 1) / BN, lo_t);
  const int n_tiles = n_pre + (hi_t - lo_t + 1);
  auto tile_k0 = [&](int j) { return (j < n_pre ? j : lo_t + (j - n_pre)) * BN; };

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t b_q = smem_u32(&bars.q_full), b_of = smem_u32(&bars.o_final), b_dr = smem_u32(&bars.drain);
  auto b_k = [&](int s) { return smem_u32(&bars.k_full[s]); };
  auto b_v = [&](int s) { return smem_u32(&bars.v_full[s]); };
  auto b_e = [&](int s) { return smem_u32(&bars.kv_empty[s]); };
  auto b_s = [&](int i) { return smem_u32(&bars.s_full[i]); };
  auto b_p = [&](int i) { return smem_u32(&bars.p_full[i]); };
  auto b_qt = [&](int i) { return smem_u32(&bars.q_tmem[i]); };

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(b_q, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_k(s), 1);
      mbar_init(b_v(s), 1);
      mbar_init(b_e(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_s(i), 1);
      mbar_init(b_p(i), 4);
      mbar_init(b_qt(i), 4);
    }
    mbar_init(b_of, 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      mbar_expect_tx(b_q, nh * TILE);
      for (int i = 0; i < nh; ++i) tma_load_2d(sb + OFF_Q + i * TILE, &p.tm_q, (h0 + i) * D, sp.start + q0, b_q);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % NS, u = j / NS;
        if (j >= NS && !mbar_wait(b_e(s), (u - 1) & 1, ab)) break;
        const int row = sp.start + tile_k0(j);
        mbar_expect_tx(b_k(s), TILE);
        tma_load_2d(sb + OFF_K + s * TILE, &p.tm_k, g * D, row, b_k(s));
        mbar_expect_tx(b_v(s), TILE);
        tma_load_2d(sb + OFF_V + s * TILE, &p.tm_v, g * D, row, b_v(s));
        issued = j + 1;
      }
      if (abort_flag) {
        wait_drain(b_q, 0);
        for (int j = max(0, issued - NS); j < issued; ++j) {
          wait_drain(b_k(j % NS), (j / NS) & 1);
          wait_drain(b_v(j % NS), (j / NS) & 1);
        }
      }
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Whole warp: descriptors are warp-uniform; one elected lane issues.
    {
      const bool leader = elect_one();
      const uint32_t id_s = idesc_bf16(BM, BN, false, false);
      const uint32_t id_o = idesc_bf16(BM, D, false, true);
      const uint64_t d_k = sdesc_sw128(sb + OFF_K, 16, 1024);  // stage s: + s * TILE
      const uint64_t d_v = sdesc_sw128(sb + OFF_V, 16, 1024);
      auto issue_s = [&](int i, int s) {
        const uint64_t kb = sdesc_add(d_k, s * TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          if (leader) mma_ts(tmem + TM_S + 128 * i, tmem + TM_Q + 32 * i + kk * 8, sdesc_add(kb, kk * 32), id_s, kk > 0);
      };
      auto issue_pv = [&](int i, int s, bool first) {
        const uint64_t vb = sdesc_add(d_v, s * TILE);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          if (leader)
            mma_ts(tmem + TM_O + 64 * i, tmem + TM_S + 128 * i + kk * 8, sdesc_add(vb, kk * 2048), id_o,
                   (!first || kk > 0) ? 1u : 0u);
      };
      bool ok = __all_sync(0xffffffffu, mbar_wait(b_k(0), 0, ab));
      for (int i = 0; i < nh && ok; ++i) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_qt(i), 0, ab)))) break;
        fence_after_sync();
        issue_s(i, 0);
        if (leader) mma_commit(b_s(i));
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % NS;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_v(s), (j / NS) & 1, ab)))) break;
        for (int i = 0; i < nh && ok; ++i) {
          if (lane == 0) SA_TRACE(0, j, 2 * i);
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(b_p(i), j & 1, ab)))) break;
          if (lane == 0) SA_TRACE(0, j, 2 * i + 1);
          fence_after_sync();
          issue_pv(i, s, j == 0);
          if (j + 1 < n_tiles) {
            const int s2 = (j + 1) % NS;
            if (i == 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(b_k(s2), ((j + 1) / NS) & 1, ab)))) break;
            fence_after_sync();
            issue_s(i, s2);
            if (leader) mma_commit(b_s(i));
          }
          if (lane == 0) SA_TRACE(0, j, 4 + i);
        }
        if (ok && leader) mma_commit(b_e(s));
      }
      if (ok && leader) mma_commit(b_of);
      if (leader) mma_commit(b_dr);
      __syncwarp();
      wait_drain(b_dr, 0);
    }
    }
  } else {
    regs_inc<REGS_HIGH>();
    if ((warp - 4) / 4 < nh) {
    // ------------------------------------------------------------ softmax
    const int i = (warp - 4) >> 2;
    const int h = h0 + i;
    const int row = (warp & 3) * 32 + lane;
    const int q = q0 + row;
    const uint32_t lb = lane_base(warp);
    const uint32_t tS = tmem + TM_S + 128 * i + lb, tO = tmem + TM_O + 64 * i + lb;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = __all_sync(0xffffffffu, mbar_wait(b_q, 0, ab));
    if (ok) {
      // Copy this thread's query row into TMEM: the A operand of S_i = Q_i K^T.
      const uint32_t src = sb + OFF_Q + i * TILE + row * 128;
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(src + ((c ^ (row & 7)) << 4)));
        r[4 * c] = v.x, r[4 * c + 1] = v.y, r[4 * c + 2] = v.z, r[4 * c + 3] = v.w;
      }
      tmem_st32(tmem + TM_Q + 32 * i + lb, r);
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qt(i));
    }
    for (int j = 0; ok && j < n_tiles; ++j) {
      if ((warp & 3) == 0 && lane == 0) SA_TRACE(1 + i, j, 0);
      ok = __all_sync(0xffffffffu, mbar_wait(b_s(i), j & 1, ab));
      if (!ok) break;
      if ((warp & 3) == 0 && lane == 0) SA_TRACE(1 + i, j, 1);
      fence_after_sync();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, r[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(r[c]);
#define S_(c) r[(c) >> 5][(c) & 31]
      const int k0 = tile_k0(j);
      if (!block_full(q0, BM, k0, BN, sp.len, p.mask)) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (!visible(q, k0 + c, sp.len, p.mask)) S_(c) = __float_as_uint(-INFINITY);
      }
      // Row maximum as 8 independent three-input chains (no 128-long dependency).
      float pm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pm[k] = fmaxf(__uint_as_float(S_(2 * k)), __uint_as_float(S_(2 * k + 1)));
#pragma unroll
      for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          pm[k] = fmax3(pm[k], __uint_as_float(S_(c + 2 * k)), __uint_as_float(S_(c + 2 * k + 1)));
      const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      const float m_new = fmaxf(m_ref, mx * sl2);
      const bool resc = (m_ref != -INFINITY) && (m_new > m_ref + 8.f);
      float factor = 1.f;
      if (m_ref == -INFINITY) {
        m_ref = m_new;  // nothing accumulated yet: O and the row sum are exactly zero
      } else if (resc) {
        factor = ex2(m_ref - m_new);
        m_ref = m_new;
        l *= factor;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O holds every P.V of earlier tiles: the commit that signalled S for
        // this tile also covered them.
        uint32_t o[2][32];
        tmem_ld32(tO, o[0]);
        tmem_ld32(tO + 32, o[1]);
        tmem_ld_wait();
        reg_fence32(o[0]);
        reg_fence32(o[1]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) o[c][e] = __float_as_uint(__uint_as_float(o[c][e]) * factor);
        tmem_st32(tO, o[0]);
        tmem_st32(tO + 32, o[1]);
      }
      if ((warp & 3) == 0 && lane == 0) SA_TRACE(1 + i, j, 2);
      const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const float2 sl2x2 = make_float2(sl2, sl2), negx2 = make_float2(neg, neg);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = ffma2(make_float2(__uint_as_float(S_(64 * hh + 2 * c)), __uint_as_float(S_(64 * hh + 2 * c + 1))),
                                 sl2x2, negx2);
          float2 e;
          if ((c & 3) == 3) {
            e.x = exp2_fma(x.x);
            e.y = exp2_fma(x.y);
          } else {
            e.x = ex2(x.x);
            e.y = ex2(x.y);
          }
          acc[c & 3] = fadd2(acc[c & 3], e);
          pk[c] = pack_bf16(e.x, e.y);
        }
        // P overwrites the first 64 columns of S_i; the whole S row is
        // already in registers.
        tmem_st32(tS + 32 * hh, pk);
      }
#undef S_
      const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
      const float2 at = fadd2(a01, a23);
      l += at.x + at.y;
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_p(i));
      if ((warp & 3) == 0 && lane == 0) SA_TRACE(1 + i, j, 3);
    }
    ok = ok && __all_sync(0xffffffffu, mbar_wait(b_of, 0, ab));
    if (ok) {
      fence_after_sync();
      uint32_t o[2][32];
      tmem_ld32(tO, o[0]);
      tmem_ld32(tO + 32, o[1]);
      tmem_ld_wait();
      reg_fence32(o[0]);
      reg_fence32(o[1]);
      const float lse = (l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      const float alpha = 1.f / (1.f + ex2((__ldg(p.sink + h) - lse) * kLog2e));
      const float fac = (l > 0.f) ? alpha / l : 0.f;
      if (q < sp.len) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(sp.start + q) * p.hq + h) * D);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
#define O_(e) __uint_as_float(o[c >> 2][(c & 3) * 8 + (e)]) * fac
          uint4 v;
          v.x = pack_bf16(O_(0), O_(1));
          v.y = pack_bf16(O_(2), O_(3));
          v.z = pack_bf16(O_(4), O_(5));
          v.w = pack_bf16(O_(6), O_(7));
#undef O_
          dst[c] = v;
        }
        p.lse[static_cast<size_t>(h) * p.T + sp.start + q] = lse;
      }
    }
    }
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

cudaError_t launch_fwd_tc(const Problem& pr, const FwdArgs& a, int* status, cudaStream_t stream) {
  if (pr.total_tokens == 0 || pr.num_seqs == 0 || pr.seqlen == 0) return cudaSuccess;
  thread_local FwdTcK k;  // 17 KB parameter block; host-side staging, one per host thread
  if (!make_rows_map(&k.tm_q, a.q, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_k, a.k, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_v, a.v, pr.total_tokens, pr.hkv, BN))
    return cudaErrorInvalidValue;
  k.sink = a.sink;
  k.o = static_cast<__nv_bfloat16*>(a.o);
  k.lse = a.lse;
  k.cu = pr.cu;
  k.status = status;
  k.seqlen = pr.seqlen;
  k.T = pr.total_tokens;
  k.hq = pr.hq;
  k.hkv = pr.hkv;
  k.group = pr.hq / pr.hkv;
  k.nh = (k.group % 2 == 0) ? 2 : 1;
  k.mask = MaskParams{pr.window, pr.prefix, pr.causal};
  k.scale_log2 = pr.scale * kLog2e;
  const std::vector<uint32_t> items = fwd_work_list(pr);
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
  if (e != cudaSuccess) return e;
  if ((e = prof_begin(g_prof_fwd, stream)) != cudaSuccess) return e;
  constexpr int kMax = static_cast<int>(sizeof(k.items) / sizeof(k.items[0]));
  for (size_t first = 0; first < items.size(); first += kMax) {
    const int n = static_cast<int>(std::min<size_t>(kMax, items.size() - first));
    std::copy(items.begin() + first, items.begin() + first + n, k.items);
    k.n_items = n;
    dim3 grid(pr.hq / k.nh, n);
    fwd_tc_kernel<<<grid, NTHR, SMEM_DYN, stream>>>(k);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return prof_end(g_prof_fwd, stream);
}

}  // namespace sa
