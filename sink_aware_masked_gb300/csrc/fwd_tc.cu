// Forward of sink-aware attention on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in Tensor Memory, operands staged by TMA).
//
// Persistent kernel: one CTA per SM walks a list of work units.  A unit is
// 128 query rows of one sequence for a PAIR of query heads of the same GQA
// group, so both heads share every K/V tile that TMA brings in.  Units come
// longest-first from the host and are dealt to the CTAs in snake order
// (round r gives unit r*G + c to CTA c on even rounds, r*G + G-1-c on odd
// ones).  Warp roles (12 warps, three warpgroups):
//   warp 0      TMA producer: Q of both heads into one of two Q buffers,
//               then K and V tiles of 128 keys through an NS-stage ring (one
//               barrier per stage).  It runs ahead across unit boundaries.
//   warp 1      S issuer (one elected lane) and TMEM owner:
//               S_i = Q_i K_j^T   (M=128, N=128, K=64; A = Q_i, B = K_j, both
//                                   K-major in smem)
//               for both heads of step t as soon as both softmax warpgroups
//               hold S of step t-1 in registers.
//   warp 2      P.V issuer (one elected lane):
//               O_i += P_i V_j    (M=128, N=64,  K=128; A = P_i in TMEM,
//                                   B = V_j MN-major in smem)
//               by key halves (first half of both heads, then the second) as
//               the softmax hands them over.  The tensor core queues only a
//               few MMAs, so an issuing thread blocks while earlier ones run;
//               with S and P.V in separate warps neither chain of waits
//               stalls the other.  t is the flat sequence of (unit, key tile)
//               steps; barriers both heads pass together (K/V stage, S
//               release, P halves) are shared.
//   warp 3      idle (it only completes the first warpgroup, which hands its
//               registers to the softmax warpgroups: 64 vs 216 each)
//   warps 4-7   softmax of head 0, warps 8-11 softmax of head 1: the thread
//               in lane l of warp w owns query row 32 * (w % 4) + l (its TMEM
//               lane), so row max and row sum need no shuffles.
// Tensor Memory (512 columns): S0 | S1 (128 each) | P0 | P1 (64 each, packed
// bf16) | O0 | O1 (64 each).  P has columns of its own, so a softmax
// warpgroup releases S_i as soon as the tile is in its registers and the
// tensor core computes S_i of the next step while the exponentials of this
// one run.  P is handed over in two 64-key halves with barriers of their own:
// P.V of the first half runs while the second half is exponentiated, and a
// half of P is overwritten one step later, long after its MMAs finished.
//
// Softmax: online softmax in log2 units; the O rescale is skipped unless the
// running max grows by more than 8 (P stays below 2^8, exact in fp32 sums);
// exponentials on the MUFU unit (with two softmax warpgroups per SM sharing
// the pipes, moving a share of them to an FMA polynomial measured slower);
// the row maximum uses independent three-input max chains; scale/subtract
// and row sums use packed f32x2 arithmetic; masked entries of partial tiles
// are cleared from per-32-key visibility bit masks.
//
// Epilogue (SinkFlex-RL summary page: auxiliary log-sum-exp and the sink
// scaling function; section 5: zero-value sink equivalence):
//   l = ln2 * (m + log2 sum),  alpha = sigmoid(l - sink[h]),  O = alpha * acc / sum.
// A tile that lies wholly inside its sequence is written through a staging
// tile per head by one TMA tensor store (row-strided stores from every
// thread took ~2.5 K cycles per unit); the last tile of a sequence, whose
// rows past the end belong to the next packed sequence, is stored row by
// row.
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


namespace sa {
namespace {

using namespace tc;

constexpr int D = kHeadDim;
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int NS = 4;   // K/V ring stages
constexpr int NQB = 2;  // Q buffers (the next unit's Q lands while this one runs)
constexpr int NTHR = 384;
// Register split after setmaxnreg: 128 x 72 + 256 x 216 = 64,512 <= 384 x 168.
constexpr int REGS_LOW = 72, REGS_HIGH = 216;
constexpr int TILE = BM * D * 2;  // 16 KB: 128 rows x 128 bytes
constexpr int OFF_Q = 0;                      // buffer b, head i: + (2 b + i) * TILE
constexpr int OFF_K = OFF_Q + NQB * 2 * TILE;
constexpr int OFF_V = OFF_K + NS * TILE;
constexpr int OFF_OST = OFF_V + NS * TILE;   // head i: + i * TILE, the finished O tile the TMA store reads
constexpr int SMEM_DYN = OFF_OST + 2 * TILE + 1024;  // + alignment slack
static_assert(SMEM_DYN <= 227 * 1024 - 512, "shared memory");

constexpr uint32_t TM_S = 0, TM_P = 256, TM_O = 384;  // + 128 i, + 64 i, + 64 i

struct FwdTcK {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  const float* sink;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* cu;
  int* status;
  int seqlen;
  long long T;
  int hq, hkv, group, nh, npairs;
  MaskParams mask;
  float scale_log2;
  int n_items;
  int n_units;  // n_items * npairs
  uint32_t items[4096];  // this launch's slice of the work list: b | (query tile << 16)
};
static_assert(sizeof(FwdTcK) < 32000, "kernel parameter block too large");

struct Bars {
  uint64_t q_full[NQB], q_empty[NQB];
  uint64_t kv_full[NS], kv_empty[NS];
  uint64_t s_full[2];                 // per head
  uint64_t s_free;                    // both heads' softmax warps
  uint64_t p_full[2], pv_done[2];     // per half of the key tile, both heads
  uint64_t drain;
};

// One work unit as every role sees it.
struct Unit {
  int h0;  // first query head of the pair
  int g;   // key/value head
  SeqSpan sp;
  int q0;
  int lo_t, n_pre, n_tiles;
  SA_DEV int tile_k0(int j) const { return (j < n_pre ? j : lo_t + (j - n_pre)) * BN; }
};

SA_DEV bool get_unit(const FwdTcK& p, int r, Unit& u) {
  // 32-bit: a launch holds at most 4096 items x 128 head pairs.
  const int G = gridDim.x, c = blockIdx.x;
  const int pos = r * G + ((r & 1) ? G - 1 - c : c);
  if (pos >= p.n_units) return false;
  const uint32_t item = p.items[pos / p.npairs];
  u.h0 = (pos % p.npairs) * p.nh;
  u.g = u.h0 / p.group;
  u.sp = seq_span(p.cu, p.seqlen, static_cast<int>(item & 0xFFFFu));
  u.q0 = static_cast<int>(item >> 16) * BM;
  const int q1 = min(u.q0 + BM, u.sp.len) - 1;
  const KeyRange kr = key_range(u.q0, q1, u.sp.len, p.mask);
  u.lo_t = kr.lo / BN;
  u.n_pre = min((kr.pre_end + BN - 1) / BN, u.lo_t);
  u.n_tiles = u.n_pre + (kr.hi / BN - u.lo_t + 1);  // >= 1: the diagonal is always visible
  return true;
}

SA_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

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

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t b_dr = smem_u32(&bars.drain);
  auto b_qf = [&](int b) { return smem_u32(&bars.q_full[b]); };
  auto b_qe = [&](int b) { return smem_u32(&bars.q_empty[b]); };
  auto b_kv = [&](int s) { return smem_u32(&bars.kv_full[s]); };
  auto b_e = [&](int s) { return smem_u32(&bars.kv_empty[s]); };
  auto b_s = [&](int i) { return smem_u32(&bars.s_full[i]); };
  const uint32_t b_sf = smem_u32(&bars.s_free);
  auto b_p = [&](int hf) { return smem_u32(&bars.p_full[hf]); };
  auto b_pv = [&](int hf) { return smem_u32(&bars.pv_done[hf]); };

  if (tid == 0) {
    abort_flag = 0;
    for (int b = 0; b < NQB; ++b) {
      mbar_init(b_qf(b), 1);
      mbar_init(b_qe(b), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_kv(s), 1);
      mbar_init(b_e(s), 2);  // one commit from each MMA issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_s(i), 1);
      mbar_init(b_p(i), 4 * nh);
      mbar_init(b_pv(i), 1);
    }
    mbar_init(b_sf, 4 * nh);
    mbar_init(b_dr, 2);
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
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
        int nq = 0, nt = 0;  // Q loads and K/V tiles issued
        bool ok = true;
        Unit u;
        for (int r = 0; ok && get_unit(p, r, u); ++r) {
          const int qb = r % NQB;
          if (r >= NQB && !(ok = mbar_wait(b_qe(qb), ((r / NQB) - 1) & 1, ab))) break;
          mbar_expect_tx(b_qf(qb), nh * TILE);
          for (int i = 0; i < nh; ++i)
            tma_load_2d(sb + OFF_Q + (2 * qb + i) * TILE, &p.tm_q, (u.h0 + i) * D, u.sp.start + u.q0, b_qf(qb));
          nq = r + 1;
          for (int j = 0; j < u.n_tiles; ++j) {
            const int s = nt % NS;
            if (nt >= NS && !(ok = mbar_wait(b_e(s), ((nt / NS) - 1) & 1, ab))) break;
            const int row = u.sp.start + u.tile_k0(j);
            mbar_expect_tx(b_kv(s), 2 * TILE);
            tma_load_2d(sb + OFF_K + s * TILE, &p.tm_k, u.g * D, row, b_kv(s));
            tma_load_2d(sb + OFF_V + s * TILE, &p.tm_v, u.g * D, row, b_kv(s));
            ++nt;
          }
        }
        if (abort_flag) {
          for (int r = max(0, nq - NQB); r < nq; ++r) wait_drain(b_qf(r % NQB), (r / NQB) & 1);
          for (int t = max(0, nt - NS); t < nt; ++t) wait_drain(b_kv(t % NS), (t / NS) & 1);
        }
      }
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuers
      // Whole warp: descriptors are warp-uniform; one elected lane issues.
      const bool leader = elect_one();
      auto wait_all = [&](uint32_t bar, uint32_t parity) { return mbar_wait_warp(bar, parity, ab); };
      bool ok = true;
      int nt = 0;  // flat step index
      Unit u;
      if (warp == 1) {
        // S_i(t) = Q_i K(t)^T for both heads.
        const uint32_t id_s = idesc_bf16(BM, BN, false, false);
        const uint64_t d_q = sdesc_sw128(sb + OFF_Q, 16, 1024);  // buffer b, head i: + (2 b + i) * TILE
        const uint64_t d_k = sdesc_sw128(sb + OFF_K, 16, 1024);  // stage s: + s * TILE
        for (int r = 0; ok && get_unit(p, r, u); ++r) {
          const int qb = r % NQB;
          if (!(ok = wait_all(b_qf(qb), (r / NQB) & 1))) break;
          for (int j = 0; j < u.n_tiles; ++j, ++nt) {
            const int s = nt % NS;
            // Both tests are issued before either result is needed, so their
            // latencies overlap; a phase still pending falls back to a wait.
            const bool kv_ready = mbar_test_wait(b_kv(s), (nt / NS) & 1);
            const bool s_ready = nt == 0 || mbar_test_wait(b_sf, (nt - 1) & 1);
            if (!__all_sync(0xffffffffu, kv_ready) && !(ok = wait_all(b_kv(s), (nt / NS) & 1))) break;
            if (!__all_sync(0xffffffffu, s_ready) && !(ok = wait_all(b_sf, (nt - 1) & 1))) break;
            fence_after_sync();
            for (int i = 0; i < nh; ++i) {
              const uint64_t qd = sdesc_add(d_q, (2 * qb + i) * TILE), kd = sdesc_add(d_k, s * TILE);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                if (leader) mma_ss(tmem + TM_S + 128 * i, sdesc_add(qd, kk * 32), sdesc_add(kd, kk * 32), id_s, kk > 0);
              if (leader) mma_commit(b_s(i));
            }
            if (leader) {
              if (j == u.n_tiles - 1) mma_commit(b_qe(qb));
              mma_commit(b_e(s));
            }
          }
        }
      } else {
        // O_i += P_i(t) V(t) for both heads, one key half at a time.
        const uint32_t id_o = idesc_bf16(BM, D, false, true);
        const uint64_t d_v = sdesc_sw128(sb + OFF_V, 16, 1024);  // stage s: + s * TILE
        for (int r = 0; ok && get_unit(p, r, u); ++r) {
          for (int j = 0; ok && j < u.n_tiles; ++j, ++nt) {
            const int s = nt % NS;
            const uint64_t vb = sdesc_add(d_v, s * TILE);
            // The V tile landed before S of this step was issued; this
            // acquires the TMA writes for this warp's own MMAs.
            if (!(ok = wait_all(b_kv(s), (nt / NS) & 1))) break;
            for (int hf = 0; hf < 2; ++hf) {
              if (!(ok = wait_all(b_p(hf), nt & 1))) break;
              fence_after_sync();
              for (int i = 0; i < nh; ++i) {
#pragma unroll
                for (int k4 = 0; k4 < BN / 32; ++k4) {
                  const int kk = 4 * hf + k4;
                  if (leader)
                    mma_ts(tmem + TM_O + 64 * i, tmem + TM_P + 64 * i + kk * 8, sdesc_add(vb, kk * 2048), id_o,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
              }
              if (leader) mma_commit(b_pv(hf));
            }
            if (ok && leader) mma_commit(b_e(s));
          }
        }
      }
      if (leader) mma_commit(b_dr);
      __syncwarp();
      wait_drain(b_dr, 0);
    }
  } else {
    regs_inc<REGS_HIGH>();
    if ((warp - 4) / 4 < nh) {
      // ---------------------------------------------------------- softmax
      const int i = (warp - 4) >> 2;
      const int row = (warp & 3) * 32 + lane;
      const uint32_t lb = lane_base(warp);
      const uint32_t tS = tmem + TM_S + 128 * i + lb, tP = tmem + TM_P + 64 * i + lb, tO = tmem + TM_O + 64 * i + lb;
      const float sl2 = p.scale_log2;
      auto wait_all = [&](uint32_t bar, uint32_t parity) { return mbar_wait_warp(bar, parity, ab); };
      bool ok = true;
      int nt = 0;  // flat step index
      Unit u;
      for (int r = 0; ok && get_unit(p, r, u); ++r) {
        const int h = u.h0 + i;
        const int q = u.q0 + row;
        const float sink_h = __ldg(p.sink + h);  // loaded now, used by the epilogue
        float m_ref = -INFINITY, l = 0.f;
        for (int j = 0; j < u.n_tiles; ++j, ++nt) {
          if (!(ok = wait_all(b_s(i), nt & 1))) break;
          fence_after_sync();
          uint32_t r_[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, r_[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c) reg_fence32(r_[c]);
          // S_i is in registers: the tensor core may overwrite it.
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_sf);
          // Early tests of the two halves of the previous step's P.V; the
          // results are used only when P is stored, so their latency hides
          // behind the arithmetic below.
          const bool pv_ready0 = nt == 0 || mbar_test_wait(b_pv(0), (nt - 1) & 1);
          const bool pv_ready1 = nt == 0 || mbar_test_wait(b_pv(1), (nt - 1) & 1);
#define S_(c) r_[(c) >> 5][(c) & 31]
          const int k0 = u.tile_k0(j);
          if (!block_full(u.q0, BM, k0, BN, u.sp.len, p.mask)) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const uint32_t vb = visible_bits(q, k0 + 32 * cc, u.sp.len, p.mask);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                r_[cc][e] = ((vb >> e) & 1u) ? r_[cc][e] : __float_as_uint(-INFINITY);
            }
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
            // O_i must hold every P.V of the previous steps (the second
            // half's commit covers the first half's MMAs).
            if (!(ok = wait_all(b_pv(1), (nt - 1) & 1))) break;
            fence_after_sync();
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
          const float neg = (m_ref == -INFINITY) ? 0.f : -m_ref;
          const float2 sl2x2 = make_float2(sl2, sl2), negx2 = make_float2(neg, neg);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float2 x = ffma2(
                  make_float2(__uint_as_float(S_(64 * hh + 2 * c)), __uint_as_float(S_(64 * hh + 2 * c + 1))), sl2x2,
                  negx2);
              const float2 e = make_float2(ex2(x.x), ex2(x.y));
              acc[c & 3] = fadd2(acc[c & 3], e);
              pk[c] = pack_bf16(e.x, e.y);
            }
            // This half of P_i of the previous step has been consumed.
            if (!__all_sync(0xffffffffu, hh == 0 ? pv_ready0 : pv_ready1) &&
                !(ok = wait_all(b_pv(hh), (nt - 1) & 1)))
              break;
            fence_after_sync();
            tmem_st32(tP + 32 * hh, pk);
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p(hh));
          }
          if (!ok) break;
#undef S_
          const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
          const float2 at = fadd2(a01, a23);
          l += at.x + at.y;
        }
        // The warpgroup's four warps decide together whether to go on: the
        // tile store below meets at named barriers, and a warp whose bounded
        // wait gave up (or saw another role give up) leaves the tile loop
        // early, while a sibling may find its barrier complete.  Every warp
        // of the warpgroup meets the unit's agreement barrier, failed or not.
        if (!ok) {
          named_sync_and(1 + i, 128, false);
          break;
        }
        // ------------------------------------------------------ epilogue
        if (!(ok = named_sync_and(1 + i, 128, wait_all(b_pv(1), (nt - 1) & 1)))) break;
        fence_after_sync();
        uint32_t o[2][32];
        tmem_ld32(tO, o[0]);
        tmem_ld32(tO + 32, o[1]);
        tmem_ld_wait();
        reg_fence32(o[0]);
        reg_fence32(o[1]);
        const float lse = (l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        const float alpha = 1.f / (1.f + ex2((sink_h - lse) * kLog2e));
        const float fac = (l > 0.f) ? alpha / l : 0.f;
#define O_(e) __uint_as_float(o[c >> 2][(c & 3) * 8 + (e)]) * fac
        if (u.q0 + BM <= u.sp.len) {
          // A whole tile of the sequence: the rows go to this head's staging
          // tile (the 128-byte-swizzled layout of the tensor map) and one
          // thread stores it by TMA, so the warps move on to the next unit
          // instead of waiting on 8 row-strided stores each.  The staging
          // tile is free once the previous unit's store has read it.
          const uint32_t ost = sb + OFF_OST + i * TILE;
          const bool issuer = row == 0;
          if (issuer) bulk_wait_read0();
          named_sync(1 + i, 128);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(ost + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4), pack_bf16(O_(0), O_(1)),
                         pack_bf16(O_(2), O_(3)), pack_bf16(O_(4), O_(5)), pack_bf16(O_(6), O_(7)));
          fence_async_smem();
          named_sync(1 + i, 128);
          if (issuer) {
            tma_store_2d(&p.tm_o, h * D, u.sp.start + u.q0, ost);
            bulk_commit();
          }
          p.lse[static_cast<size_t>(h) * p.T + u.sp.start + q] = lse;
        } else if (q < u.sp.len) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<size_t>(u.sp.start + q) * p.hq + h) * D);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 v;
            v.x = pack_bf16(O_(0), O_(1));
            v.y = pack_bf16(O_(2), O_(3));
            v.z = pack_bf16(O_(4), O_(5));
            v.w = pack_bf16(O_(6), O_(7));
            dst[c] = v;
          }
          p.lse[static_cast<size_t>(h) * p.T + u.sp.start + q] = lse;
        }
#undef O_
      }
      if (row == 0) bulk_wait0();  // this thread's tile stores have completed
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

int fwd_tc_launches(const Problem& pr) {
  if (pr.total_tokens == 0 || pr.num_seqs == 0 || pr.seqlen == 0) return 0;
  constexpr size_t kMax = sizeof(FwdTcK::items) / sizeof(FwdTcK::items[0]);
  return static_cast<int>((fwd_work_list(pr).size() + kMax - 1) / kMax);
}

cudaError_t launch_fwd_tc(const Problem& pr, const FwdArgs& a, int* status, cudaStream_t stream) {
  if (pr.total_tokens == 0 || pr.num_seqs == 0 || pr.seqlen == 0) return cudaSuccess;
  thread_local FwdTcK k;  // 17 KB parameter block; host-side staging, one per host thread
  if (!make_rows_map(&k.tm_q, a.q, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_k, a.k, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_v, a.v, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_o, a.o, pr.total_tokens, pr.hq, BM))
    return cudaErrorInvalidValue;
  const int sms = device_sms();
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
  k.npairs = pr.hq / k.nh;
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
    k.n_units = n * k.npairs;
    const int grid = std::min(sms, k.n_units);
    fwd_tc_kernel<<<grid, NTHR, SMEM_DYN, stream>>>(k);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return prof_end(g_prof_fwd, stream);
}

}  // namespace sa
