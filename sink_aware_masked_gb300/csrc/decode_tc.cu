// Decode forward on the 5th-generation tensor cores: row blocks wider than
// 16 (R = group x n in (16, 128]: several new rows per sequence, or large GQA
// groups), and blocks of up to 16 rows on steps that stream at least 128
// key tiles per kv head.  Same split-KV plan, partial format and
// merge as the warp-MMA kernel (decode_common.cuh); only the per-chunk
// partial is computed here.
//
// Few query rows meet 128 keys per tile, so the tile is computed transposed,
// keys on the 128 TMEM lanes and the R query rows (padded to N = 16, 32, 64
// or 128 columns) along the columns:
//   S^T = K Q^T                 M = 128 keys, N, K = 64 dims: A = the K tile
//                               as TMA lands it (K-major), B = Q [N, 64]
//                               (K-major, staged once per CTA)
//   [O^T; l] = [V^T; 1] P^T     M = 128, N, K = 128 keys: A = the V tile read
//                               MN-major (dims 0-63) stacked on a constant
//                               block whose first row is all ones (rows
//                               64-127), B = P stored keys x rows
//                               (MN-major, written by the softmax threads,
//                               eight rows per 16-byte store)
// so TMEM lanes 0-63 accumulate O^T and lane 64 the row sums l_o of exactly
// the bf16 weights the numerator used: the sums over the keys, which lie
// across threads here, come out of the tensor core.  The log-sum-exp takes
// the fp32 sum of the unrounded exponentials instead (one bf16 rounding of a
// dominant key would move lse by up to 2e-3): each thread adds its key's P
// to per-row fp32 partial sums of its own (registers up to 64 rows, TMEM
// columns of its lane above), reduced across the lanes once per CTA.
//
// Softmax without a per-tile row maximum: each row keeps a reference m (log2
// units of the scaled score) and P = 2^{x - m}.  A tile is checked against
// m + 16; only if some score exceeds it (always on the first visible tile of
// a row, rarely afterwards) do the softmax warps compute that tile's row
// maxima (a halving butterfly, N shuffles per warp), move the references and
// rescale the accumulated O^T and l_o columns and the fp32 partial sums.  P
// stays below 2^16, far inside the range of bf16 and of the fp32 sums; the
// result is the same online softmax with a different (exact) reference per
// row, recorded with the partial.
//
// Warp roles: one softmax warpgroup per NC rows (two at 32 columns, else
// one), thread t of warp w owning key 32 (w % 4) + t of the tile (its TMEM
// lane) for the warpgroup's rows; then four role warps: the TMA producers of
// the K and the V tiles (first and third), each through its own ring (a K
// stage is free once S^T of its tile is computed, a V stage once its P.V is,
// so the next K load starts a whole softmax earlier than a shared stage
// would allow), the S^T issuer and TMEM owner (second) and the P.V issuer
// (fourth).  Each issuer blocks on its own barriers, so neither polls nor
// waits behind the other's loads; S^T runs one tile ahead (two S buffers,
// two P buffers).  Every wait is bounded; each softmax warpgroup decides
// together at its named barrier, and every role drains its copies and MMAs
// before TMEM is freed.
#include "decode_common.cuh"

namespace sa {
namespace dec {
namespace {

using namespace tc;

constexpr float kRefSlack = 16.f;  // log2 units a score may exceed its row reference by

template <int N>
struct Cfg {
  // Ring stages.  Two CTAs per SM up to 64 rows; deeper rings measured
  // slower (a third V stage at 32 columns on 8 x 32768 x 4 rows, a third K
  // and V stage at 16 columns on 32 x 8192).
  static constexpr int NK = (N == 128) ? 4 : 2;
  static constexpr int NV = (N == 128) ? 4 : 2;
  static constexpr int CTAS = (N == 128) ? 1 : 2;  // resident CTAs per SM
  // Softmax warpgroups: at 32 columns two, each owning 16 rows (the softmax
  // threads' per-tile work sets the pace; 16 columns a thread measured 0.91
  // of the copy bandwidth against 0.86 for 32), else one owning all N.
  static constexpr int NWG = (N == 32) ? 2 : 1;
  static constexpr int NC = N / NWG;               // rows (TMEM columns) per softmax thread
  static constexpr int NSOFT = 128 * NWG;          // softmax threads; the four role warps follow
  static constexpr int NTHR = NSOFT + 128;
  static constexpr bool SPLIT = N == 64;           // registers moved to the softmax warpgroup
  static constexpr int OFF_K = 0;                  // K stage s at s TILE
  static constexpr int OFF_V = NK * TILE;          // V stage s at OFF_V + s TILE
  static constexpr int OFF_Q = (NK + NV) * TILE;   // [N rows][64] K-major, 8-row groups of 1 KB
  // P buffer, MN-major (keys along the contraction, rows contiguous): key
  // k's row of min(N, 64) bf16 (PRB bytes) in swizzle atoms of 8 keys, N =
  // 128 as two such 64-row columns PATOM apart.
  static constexpr int PRB = (N >= 64 ? 64 : N) * 2;                 // 32, 64 or 128 bytes
  static constexpr int PATOM = BN * PRB;
  static constexpr int PSHIFT = PRB == 128 ? 0 : (PRB == 64 ? 1 : 2);  // 16-byte chunk ^= (key % 8) >> PSHIFT
  static constexpr uint32_t PLAYOUT = PRB == 128 ? 2 : (PRB == 64 ? 4 : 6);  // 128-, 64-, 32-byte swizzle
  static constexpr int PBUF = N * 256;             // one P buffer: 128 keys x N rows of bf16
  static constexpr int OFF_P = OFF_Q + N * 128;    // buffer b at + b PBUF
  static constexpr int OFF_ONES = OFF_P + 2 * PBUF;  // 16 key rows x 128 B, element 0 of each row = 1
  static constexpr int SMEM_DYN = OFF_ONES + 2048 + 1024;  // + alignment slack
  // The fp32 partial row sums live in registers up to 64 rows (at 64 the
  // softmax warpgroup gets 176 registers a thread), in TMEM columns above.
  static constexpr bool L_REGS = N <= 64;
  static constexpr uint32_t TM_S = 0, TM_O = 2 * N, TM_L = 3 * N;  // S buffer b at + b N
  static constexpr uint32_t TM_COLS = ((L_REGS ? 3 : 4) * N <= 128) ? 128 : ((L_REGS ? 3 : 4) * N <= 256 ? 256 : 512);
  static constexpr int UP = (N * 32 + NTHR - 1) / NTHR;    // merge units per thread
  static_assert(!SPLIT || NWG == 1, "the register split assumes one softmax warpgroup");
  static_assert(TM_O + N <= TM_COLS && (L_REGS || TM_L + N <= TM_COLS), "TMEM columns");
  static_assert(CTAS * TM_COLS <= 512, "TMEM of the resident CTAs");
};
// Register split of the 64-row kernel (256 threads), resident twice per SM:
// launched with 128 a thread (65,536 / 512), the softmax warpgroup takes 176
// and the role warps keep 80: 128 x 176 + 128 x 80 = 32,768 = 256 x 128.
constexpr int REGS_LAUNCH = 128, REGS_SOFT = 176, REGS_ROLE = 80;
static_assert(Cfg<64>::NSOFT * REGS_SOFT + (Cfg<64>::NTHR - Cfg<64>::NSOFT) * REGS_ROLE ==
                  Cfg<64>::NTHR * REGS_LAUNCH,
              "register split");

struct Bars {
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t q_full;
  uint64_t s_full[2], p_full[2], p_free[2];
  uint64_t drain_s, drain_o, merge;
};

// Waits without the abort short-cut (exit path: copies and MMAs in flight).
SA_DEV void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) return;
  }
}

SA_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Rows [rlo, rhi) of the block that see `key`: query position L - n + i sees
// the key when key < L, key <= q (causal) and q - key <= w unless key is a
// prefix key; the rows of position i are [i group, (i + 1) group).
SA_DEV void rows_seeing(int key, int L, int n, int group, const MaskParams& m, int& rlo, int& rhi) {
  const int q0 = L - n;
  int ilo = 0, ihi = n - 1;
  if (m.causal) ilo = max(0, key - q0);
  if (m.window >= 0 && key >= m.prefix) ihi = min(ihi, key + m.window - q0);
  if (key >= L || ihi < ilo) {
    rlo = rhi = 0;
    return;
  }
  rlo = ilo * group;
  rhi = (ihi + 1) * group;
}

// In-place halving butterfly over the warp: x holds N values per lane; after
// five exchange steps lane l holds the maxima (SUM: sums) over the 32 lanes
// of entries l N/32 + [0, N/32) in x[0 .. N/32) when N >= 32, and of entry
// l / 2 in x[0] when N = 16 (the last step exchanges the single value whole).
// At each halving step the lanes whose bit is set keep the upper half and
// send the lower one.
template <int N, bool SUM = false>
SA_DEV void lane_butterfly(uint32_t (&x)[N], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int half = N >> (step + 1);
    const bool up = (lane >> (4 - step)) & 1;
    if (half == 0) {
      const float v = __uint_as_float(x[0]);
      const float got = __shfl_xor_sync(0xffffffffu, v, 16 >> step);
      x[0] = __float_as_uint(SUM ? v + got : fmaxf(v, got));
      continue;
    }
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      if (i < half) {
        const float lo = __uint_as_float(x[i]), hi = __uint_as_float(x[i + half]);
        const float got = __shfl_xor_sync(0xffffffffu, up ? lo : hi, 16 >> step);
        const float keep = up ? hi : lo;
        x[i] = __float_as_uint(SUM ? keep + got : fmaxf(keep, got));
      }
    }
  }
}

// Stores the butterfly's results of one warp: dst[e] for the N entries.
template <int N>
SA_DEV void butterfly_store(float* dst, const uint32_t (&x)[N], int lane) {
  if constexpr (N >= 32) {
#pragma unroll
    for (int i = 0; i < N / 32; ++i) dst[lane * (N / 32) + i] = __uint_as_float(x[i]);
  } else {
    if ((lane & 1) == 0) dst[lane >> 1] = __uint_as_float(x[0]);
  }
}

// W (16 or 32) consecutive 32-bit TMEM columns of this thread's lane.
template <int W>
SA_DEV void tmem_ldw(uint32_t taddr, uint32_t* r) {
  if constexpr (W == 32) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(r));
  } else {
    static_assert(W == 16, "chunk width");
    tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
  }
}
template <int W>
SA_DEV void tmem_stw(uint32_t taddr, uint32_t* r) {
  if constexpr (W == 32)
    tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(r));
  else
    tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(r));
}
template <int W>
SA_DEV void reg_fencew(uint32_t* r) {
  if constexpr (W == 32)
    reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(r));
  else
    reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(r));
}

template <int N, int CAP>
__global__ void __launch_bounds__(Cfg<N>::NTHR, Cfg<N>::CTAS) decode_tc_kernel(const __grid_constant__ DecK<CAP> p) {
  using C = Cfg<N>;
  constexpr int NK = C::NK, NV = C::NV, NC = C::NC, NSOFT = C::NSOFT;
  constexpr int CW = NC < 32 ? NC : 32;  // TMEM columns per load or store
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag, is_last;
  __shared__ __align__(16) float m_s[N];    // row reference (log2 units), -inf before a visible key
  __shared__ __align__(16) float thr_s[N];  // (m + kRefSlack) / scale_log2: the bound on the raw score
  __shared__ __align__(16) float neg_s[N];  // -m, 0 while m = -inf
  __shared__ __align__(16) float fac_s[N];  // factor of the last reference move
  __shared__ float red_s[4][N];             // per lane quarter: tile maximum (or sum) of each row
  __shared__ float l_s[N];                  // l_o (TMEM lane 64)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int role = warp - NSOFT / 32;  // 0 K producer, 1 S^T issuer, 2 V producer, 3 P.V issuer; < 0 softmax
  const int item_idx = blockIdx.x, g = blockIdx.y;
  const Chunk ch = chunk_of(p, item_idx);
  const int nt = ch.j1 - ch.j0;  // >= 1: every chunk holds at least one tile

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto b_kf = [&](int s) { return smem_u32(&bars.k_full[s]); };
  auto b_ke = [&](int s) { return smem_u32(&bars.k_empty[s]); };
  auto b_vf = [&](int s) { return smem_u32(&bars.v_full[s]); };
  auto b_ve = [&](int s) { return smem_u32(&bars.v_empty[s]); };
  auto b_sf = [&](int b) { return smem_u32(&bars.s_full[b]); };
  auto b_pf = [&](int b) { return smem_u32(&bars.p_full[b]); };
  auto b_pe = [&](int b) { return smem_u32(&bars.p_free[b]); };
  const uint32_t b_qf = smem_u32(&bars.q_full);

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < NK; ++s) {
      mbar_init(b_kf(s), 1);
      mbar_init(b_ke(s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(b_vf(s), 1);
      mbar_init(b_ve(s), 1);
    }
    mbar_init(b_qf, NSOFT);
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_sf(b), 1);
      mbar_init(b_pf(b), NSOFT / 32);  // one arrival per softmax warp
      mbar_init(b_pe(b), 1);
    }
    mbar_init(smem_u32(&bars.drain_s), 1);
    mbar_init(smem_u32(&bars.drain_o), 1);
    mbar_init(smem_u32(&bars.merge), 1);
    fence_mbar_init();
  }
  if (tid < N) {
    m_s[tid] = -INFINITY;
    thr_s[tid] = -INFINITY;
    neg_s[tid] = 0.f;
  }
  if (role == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::TM_COLS);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const Abort ab{&abort_flag, p.status};

  if (role >= 0) {
    if constexpr (C::SPLIT) regs_dec<REGS_ROLE>();
    if (role == 0 || role == 2) {
      // ---------------------------------------------------------- TMA producers
      // One warp streams the K tiles, another the V tiles, each through its
      // own ring: a K stage is free once S^T of its tile is computed, a V
      // stage once its P.V is, so the next K load starts a whole softmax
      // earlier than a shared K/V stage would allow.
      if (lane == 0) {
        const bool is_k = role == 0;
        const CUtensorMap* map = is_k ? &p.tm_k : &p.tm_v;
        const uint32_t base = sb + (is_k ? C::OFF_K : C::OFF_V);
        const int NS = is_k ? NK : NV;
        tma_prefetch_map(map);
        int issued = 0;
        for (int t = 0; t < nt; ++t) {
          const int s = t % NS;
          if (t >= NS && !mbar_wait(is_k ? b_ke(s) : b_ve(s), ((t / NS) - 1) & 1, ab)) break;
          const uint32_t full = is_k ? b_kf(s) : b_vf(s);
          mbar_expect_tx(full, TILE);
          tma_load_2d(base + s * TILE, map, g * D, ch.sp.start + ch.kt.k0(ch.j0 + t), full);
          issued = t + 1;
        }
        if (abort_flag)
          for (int t = max(0, issued - NS); t < issued; ++t)
            wait_drain(is_k ? b_kf(t % NS) : b_vf(t % NS), (t / NS) & 1);
      }
    } else if (role == 1) {
      // ---------------------------------------------------------- S^T issuer
      // S^T(t) = K(t) Q^T into S buffer t & 1, free again once the softmax
      // warps handed over P(t - 2).
      const bool leader = elect_one();
      const uint32_t id_s = idesc_bf16(128, N, false, false);
      const uint64_t d_q = sdesc_sw128(sb + C::OFF_Q, 16, 1024);
      const uint64_t d_k = sdesc_sw128(sb + C::OFF_K, 16, 1024);
      bool ok = mbar_wait_warp(b_qf, 0, ab);
      for (int t = 0; ok && t < nt; ++t) {
        const int s = t % NK;
        if (!(ok = mbar_wait_warp(b_kf(s), (t / NK) & 1, ab))) break;
        if (t >= 2 && !(ok = mbar_wait_warp(b_pf(t & 1), ((t - 2) >> 1) & 1, ab))) break;
        fence_after_sync();
        const uint64_t dk = sdesc_add(d_k, s * TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          if (leader)
            mma_ss(tmem + C::TM_S + (t & 1) * N, sdesc_add(dk, kk * 32), sdesc_add(d_q, kk * 32), id_s,
                   kk > 0 ? 1u : 0u);
        if (leader) {
          mma_commit(b_sf(t & 1));
          mma_commit(b_ke(s));
        }
        __syncwarp();
      }
      if (leader) mma_commit(smem_u32(&bars.drain_s));
      __syncwarp();
      wait_drain(smem_u32(&bars.drain_s), 0);
    } else {
      // ---------------------------------------------------------- P.V issuer
      // [O^T; l_o] += [V^T; 1] P(t)^T once P(t) is written and V(t) landed.
      const bool leader = elect_one();
      const uint32_t id_o = idesc_bf16(128, N, true, true);
      bool ok = true;
      for (int t = 0; ok && t < nt; ++t) {
        const int s = t % NV;
        if (!(ok = mbar_wait_warp(b_pf(t & 1), (t >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait_warp(b_vf(s), (t / NV) & 1, ab))) break;
        fence_after_sync();
        const uint32_t v_off = C::OFF_V + s * TILE, p_off = C::OFF_P + (t & 1) * C::PBUF;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t a_off = v_off + kk * 2048;  // 16 keys of 128 B rows
          const uint64_t da = sdesc_sw128(sb + a_off, C::OFF_ONES - a_off, 1024);
          const uint64_t db = sdesc_swz(sb + p_off + kk * 16 * C::PRB, C::PATOM, 8 * C::PRB, C::PLAYOUT);
          if (leader) mma_ss(tmem + C::TM_O, da, db, id_o, (t > 0 || kk > 0) ? 1u : 0u);
        }
        if (leader) {
          mma_commit(b_ve(s));
          mma_commit(b_pe(t & 1));
        }
        __syncwarp();
      }
      if (leader) mma_commit(smem_u32(&bars.drain_o));
      __syncwarp();
      wait_drain(smem_u32(&bars.drain_o), 0);
    }
  } else {
    if constexpr (C::SPLIT) regs_inc<REGS_SOFT>();
    // ------------------------------------------------------------ softmax
    // Warpgroup wg owns rows [c0, c0 + NC): their S^T columns, references,
    // sums, P rows and output; thread (warp % 4, lane) owns key 32 (warp % 4)
    // + lane of each tile (its TMEM lane).  Each warpgroup decides at its own
    // named barrier.
    const int wg = warp >> 2, q4 = warp & 3, key = tid & 127, c0 = wg * NC, bar = 1 + wg;
    // Q rows (zero rows up to N) and the constant ones block.
    for (int idx = tid; idx < N * 8; idx += NSOFT) {
      const int r = idx >> 3, c = idx & 7;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < p.R) {
        const int i = r / p.group, jh = r - i * p.group;
        v = __ldg(reinterpret_cast<const uint4*>(
                      p.q + (static_cast<size_t>(ch.b * p.n + i) * p.hq + g * p.group + jh) * D) + c);
      }
      *reinterpret_cast<uint4*>(smem + C::OFF_Q + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
    if (tid < 128) {
      const int r = tid >> 3, c = tid & 7;  // 16 rows x 8 chunks; logical chunk 0 sits at chunk r % 8
      *reinterpret_cast<uint4*>(smem + C::OFF_ONES + tid * 16) = make_uint4(c == (r & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    mbar_arrive(b_qf);

    const uint32_t lb = lane_base(warp);
    // fp32 sums of this key's unrounded P for every owned row (registers or TMEM).
    float lreg[C::L_REGS ? NC : 1];
#pragma unroll
    for (int r = 0; r < (C::L_REGS ? NC : 1); ++r) lreg[r] = 0.f;
    if constexpr (!C::L_REGS) {
      uint32_t z[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) z[e] = 0u;
#pragma unroll
      for (int c = 0; c < NC / 32; ++c) tmem_st32(tmem + lb + C::TM_L + c0 + 32 * c, z);  // NC >= 128 here
      tmem_st_wait();
    }
    const float sl2 = p.scale_log2;
    const int L = ch.sp.len;
    // This thread's key row in a P buffer, and its swizzle.
    const uint32_t p_row = (key >> 3) * (8 * C::PRB) + (key & 7) * C::PRB;
    const int p_swz = (key & 7) >> C::PSHIFT;
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int buf = t & 1;
      ok = mbar_wait_warp(b_sf(buf), (t >> 1) & 1, ab) && ok;
      fence_after_sync();
      const int k0 = ch.kt.k0(ch.j0 + t);
      const bool partial = !block_full(L - p.n, p.n, k0, BN, L, p.mask);
      uint32_t x[NC];  // this key's raw scores for every owned row (-inf where masked); then P
      // S^T stays in TMEM until P(t) is handed over, so the slow path may read it twice.
      auto load_scores = [&]() {
#pragma unroll
        for (int c = 0; c < NC / CW; ++c) tmem_ldw<CW>(tmem + lb + C::TM_S + buf * N + c0 + CW * c, x + CW * c);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < NC / CW; ++c) reg_fencew<CW>(x + CW * c);
        if (partial) {
          int rlo, rhi;
          rows_seeing(k0 + key, L, p.n, p.group, p.mask, rlo, rhi);
#pragma unroll
          for (int r = 0; r < NC; ++r)
            if (c0 + r < rlo || c0 + r >= rhi) x[r] = __float_as_uint(-INFINITY);
        }
      };
      load_scores();
      bool over = false;
#pragma unroll
      for (int r = 0; r < NC; r += 4) {
        const float4 th = *reinterpret_cast<const float4*>(thr_s + c0 + r);
        over |= (__uint_as_float(x[r]) > th.x) | (__uint_as_float(x[r + 1]) > th.y) |
                (__uint_as_float(x[r + 2]) > th.z) | (__uint_as_float(x[r + 3]) > th.w);
      }
      if (named_sync_or(bar, 128, over || !ok)) {
        // A failed wait anywhere in the group: leave together.
        if (!named_sync_and(bar, 128, ok)) break;
        // Row maxima of this tile: a halving butterfly over the lanes (in
        // place), then the four lane quarters in shared memory.
        lane_butterfly<NC>(x, lane);
        butterfly_store<NC>(red_s[q4] + c0, x, lane);
        named_sync(bar, 128);
        bool moved = false;
        if (key < NC) {
          const int r = c0 + key;
          const float M = fmaxf(fmaxf(red_s[0][r], red_s[1][r]), fmaxf(red_s[2][r], red_s[3][r])) * sl2;
          const float m_old = m_s[r];
          float f = 1.f;
          if (M > m_old + kRefSlack) {
            f = (m_old == -INFINITY) ? 0.f : ex2(m_old - M);
            m_s[r] = M;
            thr_s[r] = (M + kRefSlack) / sl2;
            neg_s[r] = -M;
            moved = true;
          }
          fac_s[r] = f;
        }
        if (named_sync_or(bar, 128, moved) && t > 0) {
          auto rescale = [&](uint32_t col) {
#pragma unroll
            for (int c = 0; c < NC / CW; ++c) {
              uint32_t o[CW];
              tmem_ldw<CW>(tmem + lb + col + c0 + CW * c, o);
              tmem_ld_wait();
              reg_fencew<CW>(o);
#pragma unroll
              for (int e = 0; e < CW; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * fac_s[c0 + CW * c + e]);
              tmem_stw<CW>(tmem + lb + col + c0 + CW * c, o);
            }
          };
          if constexpr (C::L_REGS) {
#pragma unroll
            for (int r = 0; r < NC; ++r) lreg[r] *= fac_s[c0 + r];
          } else {
            rescale(C::TM_L);
          }
          // O^T (lanes 0-63) and l_o (lane 64) must hold every P.V so far.
          if (q4 < 3 && (ok = mbar_wait_warp(b_pe((t - 1) & 1), ((t - 1) >> 1) & 1, ab))) {
            fence_after_sync();
            rescale(C::TM_O);
          }
          tmem_st_wait();
        }
        load_scores();
      }
      // P = 2^{x sl2 - m}, stored as bf16 into P buffer buf: this key's row,
      // eight rows per 16-byte chunk.
      if (t >= 2) ok = mbar_wait_warp(b_pe(buf), ((t - 2) >> 1) & 1, ab) && ok;
      if (ok) {
        const uint32_t pb = sb + C::OFF_P + buf * C::PBUF + p_row;
#pragma unroll
        for (int c = 0; c < NC / CW; ++c) {
          uint32_t lt[CW];
          if constexpr (!C::L_REGS) {
            tmem_ldw<CW>(tmem + lb + C::TM_L + c0 + CW * c, lt);
            tmem_ld_wait();
            reg_fencew<CW>(lt);
          }
#pragma unroll
          for (int g8 = 0; g8 < CW / 8; ++g8) {
            const int rl = CW * c + 8 * g8, r0 = c0 + rl;  // first of eight rows: local, global
            const float4 n0 = *reinterpret_cast<const float4*>(neg_s + r0);
            const float4 n1 = *reinterpret_cast<const float4*>(neg_s + r0 + 4);
            const float ngv[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
            float pv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              pv[e] = ex2(fmaf(__uint_as_float(x[rl + e]), sl2, ngv[e]));
              if constexpr (C::L_REGS)
                lreg[rl + e] += pv[e];
              else
                lt[8 * g8 + e] = __float_as_uint(__uint_as_float(lt[8 * g8 + e]) + pv[e]);
            }
            st_shared_v4(pb + (r0 >> 6) * C::PATOM + ((((r0 & 63) >> 3) ^ p_swz) << 4), pack_bf16(pv[0], pv[1]),
                         pack_bf16(pv[2], pv[3]), pack_bf16(pv[4], pv[5]), pack_bf16(pv[6], pv[7]));
          }
          if constexpr (!C::L_REGS) tmem_stw<CW>(tmem + lb + C::TM_L + c0 + CW * c, lt);
        }
        if constexpr (!C::L_REGS) tmem_st_wait();
        fence_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pf(buf));
      }
    }
    // ---------------------------------------------------------- partial out
    ok = named_sync_and(bar, 128, ok);
    if (ok) {
      ok = mbar_wait_warp(b_pe((nt - 1) & 1), ((nt - 1) >> 1) & 1, ab);
      fence_after_sync();
    }
    const size_t part = static_cast<size_t>(item_idx) * p.hkv + g;
    const bool single = ch.nsplit == 1;  // the only chunk: finish the rows here, no workspace round trip
    if (ok && q4 < 3) {
#pragma unroll
      for (int c = 0; c < NC / CW; ++c) {
        uint32_t o[CW];
        tmem_ldw<CW>(tmem + lb + C::TM_O + c0 + CW * c, o);
        tmem_ld_wait();
        reg_fencew<CW>(o);
        if (q4 < 2) {
          if (single) continue;
          float* dst = p.ws_acc + part * p.R * D + key;  // dimension `key` (TMEM lane) of each row
#pragma unroll
          for (int e = 0; e < CW; ++e) {
            const int r = c0 + CW * c + e;
            if (r < p.R) dst[static_cast<size_t>(r) * D] = __uint_as_float(o[e]);
          }
        } else if (lane == 0) {
#pragma unroll
          for (int e = 0; e < CW; ++e) l_s[c0 + CW * c + e] = __uint_as_float(o[e]);
        }
      }
    }
    ok = named_sync_and(bar, 128, ok);  // red_s is reused below
    if (ok) {
      // Row sums of the unrounded exponentials: this lane's partials, summed
      // over the warp, then over the four lane quarters.
#pragma unroll
      for (int c = 0; c < NC / CW; ++c) {
        uint32_t lt[CW];
        if constexpr (C::L_REGS) {
#pragma unroll
          for (int e = 0; e < CW; ++e) lt[e] = __float_as_uint(lreg[CW * c + e]);
        } else {
          tmem_ldw<CW>(tmem + lb + C::TM_L + c0 + CW * c, lt);
          tmem_ld_wait();
          reg_fencew<CW>(lt);
        }
        lane_butterfly<CW, true>(lt, lane);
        butterfly_store<CW>(red_s[q4] + c0 + CW * c, lt, lane);
      }
    }
    ok = named_sync_and(bar, 128, ok);
    if (ok && key < NC && c0 + key < p.R) {
      const int r = c0 + key;
      const float l = red_s[0][r] + red_s[1][r] + red_s[2][r] + red_s[3][r];
      if (single) {
        float lse;
        fac_s[r] = row_scale(p, ch, g, r, m_s[r], l_s[r], l, lse);
        store_lse(p, ch, g, r, lse);
      } else {
        p.ws_ml[part * p.R + r] = make_float4(m_s[r], l_s[r], l, 0.f);
      }
    }
    if (single) {
      ok = named_sync_and(bar, 128, ok);  // fac_s of every owned row
      if (ok && q4 < 2) {
        // Thread `key` holds dimension `key` of every owned row: one bf16
        // per row, 64 contiguous bytes per warp and row.
#pragma unroll
        for (int c = 0; c < NC / CW; ++c) {
          uint32_t o[CW];
          tmem_ldw<CW>(tmem + lb + C::TM_O + c0 + CW * c, o);
          tmem_ld_wait();
          reg_fencew<CW>(o);
#pragma unroll
          for (int e = 0; e < CW; ++e) {
            const int r = c0 + CW * c + e;
            if (r >= p.R) continue;
            const int i = r / p.group, h = g * p.group + (r - i * p.group);
            p.o[(static_cast<size_t>(ch.b * p.n + i) * p.hq + h) * D + key] =
                __float2bfloat16_rn(__uint_as_float(o[e]) * fac_s[r]);
          }
        }
      }
    }
    if constexpr (C::SPLIT) regs_dec<REGS_LAUNCH>();
  }
  // -------------------------------------------------------------- common exit
  fence_before_sync();
  __syncthreads();
  if constexpr (C::SPLIT) {
    if (role >= 0) regs_inc<REGS_LAUNCH>();  // the softmax warpgroup gave its share back before the barrier
  }
  if (role == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, C::TM_COLS);
  }
  if (abort_flag) return;  // written only before the barrier above: every thread reads the same value
  // Recomputed rather than kept live through the role warps' registers.
  const Chunk ch2 = chunk_of(p, blockIdx.x);
  if (ch2.nsplit == 1) return;  // finished by the softmax warps above
  if (!count_partial(p, ch2, blockIdx.y, &is_last)) return;
  merge_partials<C::UP, C::NTHR>(p, ch2, blockIdx.y, blockIdx.x, smem, (NK + NV) * TILE, smem_u32(&bars.merge), ab);
}

template <int N, int CAP>
cudaError_t launch_n(const DecK<CAP>& k, dim3 grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<N, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<N>::SMEM_DYN);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<N, CAP><<<grid, Cfg<N>::NTHR, Cfg<N>::SMEM_DYN, stream>>>(k);
  return cudaGetLastError();
}

}  // namespace

template <int CAP>
cudaError_t launch_decode_tc(const DecK<CAP>& k, dim3 grid, cudaStream_t stream) {
  if (k.R <= 16) return launch_n<16>(k, grid, stream);
  if (k.R <= 32) return launch_n<32>(k, grid, stream);
  if (k.R <= 64) return launch_n<64>(k, grid, stream);
  return launch_n<128>(k, grid, stream);
}

template cudaError_t launch_decode_tc<kSmallItems>(const DecK<kSmallItems>&, dim3, cudaStream_t);
template cudaError_t launch_decode_tc<kDecodeMaxItems>(const DecK<kDecodeMaxItems>&, dim3, cudaStream_t);

}  // namespace dec
}  // namespace sa
