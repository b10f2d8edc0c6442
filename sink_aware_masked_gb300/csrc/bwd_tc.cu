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
// Persistent: one CTA per SM takes work units from a list sorted longest
// first, claiming the next one from a global counter when its loader has
// issued the last loads of the current one (greedy list scheduling: an SM
// that finishes early takes the next unit, whatever the units' costs; the
// claim comes a few steps before the unit is needed, so the loads run on
// across the boundary).  A unit is 128 keys of one sequence and one
// kv head (possibly one query chunk of them); the CTA loops over the query
// heads of the GQA group x the 128-row query tiles that see those keys
// ("steps"), so dK and dV accumulate in Tensor Memory without atomics.  Each
// step's 128 query rows are split into two 64-row halves A and B, each with
// its own S^T / dP^T buffers and element-wise warpgroup, so the tensor core
// works on one half while the other half's element-wise pass runs.  Steps
// are numbered across units, so the Q/dO ring, the per-step barriers and the
// dQ drain run on without a break at unit boundaries.
// Warp roles (16 warps, four warpgroups):
//   warp 0      unit claimer and Q/dO loader: claims the next unit (atomic
//               add on the launch's counter) once it has issued the loads of
//               the current one and publishes the claim in a 4-entry shared
//               ring that every other role reads; per step Q and dO tiles by
//               TMA (NS-stage ring) and the 128 bias rows of the query tile
//               by cp.async, all completing on the stage's full barrier.
//   warp 1      MMA issuer and TMEM owner (whole warp, one elected lane
//               issues).  Per half h of step t, as the element-wise warps
//               hand their results over:
//                 P_h^T ready : dV += P_h^T dO_h, then S_h^T(t+1) = K Q_h^T
//                 dS_h^T ready: dK += dS_h^T Q_h, then dP_h^T(t+1) = V dO_h^T
//               (A = P^T / dS^T / K / V in TMEM, B from shared memory; the
//               next step's S^T and dP^T overwrite the columns the
//               preceding MMA read, which the tensor core runs first), then
//               for the whole step dQ(t) = dS(t) K (A = the dS^T tile in
//               shared memory read MN-major, B = K MN-major).  The first dV
//               product of a unit (which overwrites dV) waits until the
//               element-wise warps have read the previous unit's dK, dV.
//   warp 2      K/V loader: K and V of each unit by TMA into one of KVB
//               buffers, a buffer once every MMA of the unit that used it
//               has completed; the tiles are prefetched into L2 as soon as
//               the unit is claimed.
//   warps 4-7   element-wise for half A, warps 8-11 for half B; thread = key
//               row.  Phase 1: P^T = exp(S^T - l'), packed over the S^T
//               columns just read, then signalled, so dV and the next S^T
//               run while phase 2 computes dS^T = P^T (dP^T - D), packed
//               over the dP^T columns and into a double-buffered 128 x 128
//               bf16 shared tile (128-byte swizzle) for the dQ product.
//               At a unit's start they copy its K and V into TMEM, then read
//               the previous unit's dV (half A) and dK (half B) out of TMEM
//               and write them while the new unit's first products run.
//               Partial tiles clear masked entries with a per-key bit mask
//               of the visible queries (one interval per key).
//   warps 12-15 dQ drain: thread = query row; TMEM -> swizzled fp32 staging
//               tile (32 columns at a time) -> TMA reduce-add into the fp32
//               dQ accumulator.
// Tensor Memory (512 columns): S^T A|B (64 each) | dP^T A|B (64 each) |
// dV 64 | dK 64 | dQ 64 | K 32 | V 32 (bf16 pairs).
// Every mbarrier wait is bounded; a timeout raises the status word and all
// warps leave through the common exit, which drains copies and MMAs first.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

#include <algorithm>

namespace sa {
namespace {

using namespace tc;

constexpr int D = kHeadDim;
constexpr int BN = 128;  // keys per unit (TMEM lanes)
constexpr int BM = 128;  // query rows per step
constexpr int NTHR = 512;
// setmaxnreg split of the 512 x 128 launch registers: 128 x 56 (loader/MMA
// warpgroup) + 256 x 168 (two element-wise warpgroups) + 128 x 96 (dQ drain)
// = 62,464 <= 65,536.
constexpr int REGS_LOW = 56, REGS_EW = 168, REGS_DQ = 96;
constexpr int TILE = 128 * D * 2;  // 16 KB

// Shared memory of a configuration with NS Q/dO stages and KVB K/V buffers.
// Three stages and one K/V buffer fill the 227 KB of a CTA; measured against
// two stages and two K/V buffers (the next unit's K and V loading while the
// current one runs), the third stage is worth more on every workload, the
// short windowed units included.
template <int NS, int KVB>
struct Layout {
  static constexpr int OFF_K = 0;                     // buffer b: + 2 b TILE
  static constexpr int OFF_V = TILE;                  // buffer b: + 2 b TILE
  static constexpr int OFF_Q = 2 * KVB * TILE;
  static constexpr int OFF_DO = OFF_Q + NS * TILE;
  static constexpr int OFF_DS = OFF_DO + NS * TILE;      // 2 buffers x 32 KB
  static constexpr int OFF_STG = OFF_DS + 2 * 2 * TILE;  // 16 KB fp32 dQ staging (32 of the 64 columns at a time)
  // Bias rows of the stage's 128 queries (16 bytes each: -l'/scale and -D as
  // bf16 hi/mid/lo, two zeros), the two 0/1 selector tiles that pick one
  // triple or the other (128 keys x 16 bytes), and a zero block that serves
  // as the upper K half (elements 8-15) of all of them.  All K-major, no
  // swizzle.
  static constexpr int OFF_BIAS = OFF_STG + TILE;          // NS x 2 KB
  static constexpr int OFF_SEL = OFF_BIAS + NS * BM * 16;  // 2 x 2 KB
  static constexpr int OFF_ZERO = OFF_SEL + 2 * BN * 16;   // 2 KB
  static constexpr int SMEM_DYN = OFF_ZERO + BN * 16 + 1024;
  static_assert(SMEM_DYN <= 227 * 1024 - 512, "shared memory");
};

constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 320, TM_DQ = 384, TM_K = 448, TM_V = 480;
constexpr int HALF = BM / 2;
constexpr int kMaxItems = 2048;

struct BwdTcK {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dq;
  // Stores of a warp's 32 finished key rows of dK, dV ([T, Hkv * 64] bf16,
  // boxes of 64 x 32, 128-byte swizzled in shared memory).
  CUtensorMap tm_dk, tm_dv;
  const uint4* bias;  // [Hq, T] rows of 8 bf16
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* cu;
  int* status;
  int seqlen;
  long long T;
  int hq, hkv, group;
  MaskParams mask;
  float scale, scale_log2;
  // Work list slice (longest first); unit u = item u / Hkv, kv head u % Hkv,
  // claimed in increasing u.
  // A key tile whose query range is longer than `qchunk` query tiles is split
  // into chunks, one item each; each chunk writes its partial dK/dV to its
  // own fp32 slot of dkv_acc ([slot][Hkv][2][128 keys][64]: dV, then
  // unscaled dK) and a conversion pass sums the slots of a tile in chunk
  // order.
  int qchunk;
  float* dkv_acc;
  int* unit_counter;  // zero at launch (the preprocess kernel clears it)
  int n_items;
  int n_units;
  BwdItem items[kMaxItems];
};
static_assert(sizeof(BwdTcK) < 32000, "kernel parameter block too large");

// Claimed units in flight: the claimer runs at most NS steps ahead of the
// MMA issuer, and every reader is within a unit of it.
constexpr int kUnitRing = 4;
constexpr int kUnitReaders = 14;  // warps 1, 2 and 4-15 read every claim

template <int NS, int KVB>
struct Bars {
  uint64_t unit_full[kUnitRing], unit_empty[kUnitRing];
  uint64_t kv_full[KVB], kv_empty[KVB];
  uint64_t kv_tmem;                 // K, V of the unit copied into TMEM (8 element-wise warps)
  uint64_t kv_done;                 // every MMA of the unit has completed
  uint64_t dkv_free;                // the unit's dK, dV read out of TMEM (8 element-wise warps)
  uint64_t q_full[NS], q_empty[NS];
  uint64_t s_full[2], dp_full[2];   // per half: S^T / dP^T of the step ready
  uint64_t pt_full[2], ds_full[2];  // per half: packed P^T / dS^T written by the element-wise warps
  uint64_t dq_full, dq_free, drain;
};

// One work unit as every role sees it.
struct Unit {
  BwdItem item;
  int g;  // kv head
  SeqSpan sp;
  int k0;
  int qt_lo, nq, nsteps;
  SA_DEV bool split() const { return item.nchunks > 1; }
};

// Unit number `idx` of the launch; false past the end of the list.
SA_DEV bool decode_unit(const BwdTcK& p, int idx, Unit& u) {
  if (idx < 0 || idx >= p.n_units) return false;
  u.item = p.items[idx / p.hkv];
  u.g = idx % p.hkv;
  u.sp = seq_span(p.cu, p.seqlen, u.item.b);
  u.k0 = static_cast<int>(u.item.kt) * BN;
  if (u.k0 >= u.sp.len) {  // never produced by the host's work list
    u.qt_lo = u.nq = u.nsteps = 0;
    return true;
  }
  const int k1 = min(u.k0 + BN, u.sp.len) - 1;
  int qlo, qhi;
  query_range(u.k0, k1, u.sp.len, p.mask, qlo, qhi);
  u.qt_lo = qlo / BM;
  u.nq = qhi / BM - u.qt_lo + 1;
  if (u.split()) {
    u.qt_lo += u.item.chunk * p.qchunk;
    u.nq = min(p.qchunk, u.nq - u.item.chunk * p.qchunk);
  }
  u.nsteps = u.nq > 0 ? p.group * u.nq : 0;
  return true;
}

SA_DEV int step_head(const BwdTcK& p, const Unit& u, int t) { return u.g * p.group + t / u.nq; }
SA_DEV int step_q0(const Unit& u, int t) { return (u.qt_lo + t % u.nq) * BM; }

SA_DEV void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kTimeoutCycles) return;
  }
}

SA_DEV uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

SA_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// The element-wise pass over one half step (64 queries) for this thread's
// key row, in four 16-column chunks whose Tensor Memory loads are all issued
// before the first wait (the whole phase's arithmetic is then independent
// work for the scheduler).  The MMAs already added -l'/scale to S^T and -D
// to dP^T (a K=16 bias product), so each pair of columns costs one f32x2
// multiply per phase and nothing is read from shared memory.
//
// Phase 1: P^T = exp2((S^T - l'/scale) * scale * log2(e)), masked on partial
// tiles (FULL skips the mask) with the key's visible-query bits; packed P^T
// overwrites the S^T columns already read; fp32 P stays in registers for
// phase 2.
template <bool FULL>
SA_DEV void ew_phase1(uint32_t tS, float sl2, uint32_t vis0, uint32_t vis1, float (&pv)[4][16]) {
  const float2 sl2x2 = make_float2(sl2, sl2);
  uint32_t sr[4][16];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld16(tS + 16 * c, sr[c]);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 4; ++c) reg_fence16(sr[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t (&sc)[16] = sr[c];
    const uint32_t vis = c < 2 ? vis0 : vis1;
    uint32_t pp[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const float2 x = fmul2(make_float2(__uint_as_float(sc[e]), __uint_as_float(sc[e + 1])), sl2x2);
      float2 pe = make_float2(ex2(x.x), ex2(x.y));
      if (!FULL) {
        const int bit = (16 * c + e) & 31;
        if (!(vis & (1u << bit))) pe.x = 0.f;
        if (!(vis & (2u << bit))) pe.y = 0.f;
      }
      pv[c][e] = pe.x;
      pv[c][e + 1] = pe.y;
      pp[e >> 1] = pack_bf16(pe.x, pe.y);
    }
    tmem_st8(tS + 8 * c, pp);
  }
}

// Phase 2: dS^T = P^T (dP^T - D), packed over the dP^T columns already
// read and into this key row of the shared dS^T tile (128-byte swizzle) for
// the dQ product.  Masked entries have P = 0 and so dS = 0.
SA_DEV void ew_phase2(uint32_t tDP, uint32_t rowb, int kr, const float (&pv)[4][16]) {
  uint32_t dr[4][16];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld16(tDP + 16 * c, dr[c]);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 4; ++c) reg_fence16(dr[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t (&dc)[16] = dr[c];
    uint32_t dd[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const float2 de = fmul2(make_float2(pv[c][e], pv[c][e + 1]),
                              make_float2(__uint_as_float(dc[e]), __uint_as_float(dc[e + 1])));
      dd[e >> 1] = pack_bf16(de.x, de.y);
    }
    tmem_st8(tDP + 8 * c, dd);
    st_shared_v4(rowb + (((2 * c) ^ (kr & 7)) << 4), dd[0], dd[1], dd[2], dd[3]);
    st_shared_v4(rowb + (((2 * c + 1) ^ (kr & 7)) << 4), dd[4], dd[5], dd[6], dd[7]);
  }
}

// This thread's key row of a finished unit's dV (half 0) or dK (half 1, with
// the softmax scale), from registers: bf16 into dv / dk, or the fp32 partial
// sums of one chunk of a split tile into the chunk's slot, as row-strided
// 16-byte stores (32 lines per warp instruction).  With STG, a warp whose 32
// bf16 rows are all inside the sequence stages them instead, 128-byte
// swizzled, in its own rows of the first dS^T buffer (no MMA reads it between
// units: every MMA of the finished unit has completed, and the next unit
// writes it in its first phase 2, after waiting for this read), and lane 0
// writes them with one TMA tensor store.  `ds` is the dS^T buffers' base;
// returns true when lane 0 issued a store whose read of shared memory may
// still be in flight.
template <bool STG>
SA_DEV bool write_dkv(const BwdTcK& p, const Unit& u, int half, int kr, uint32_t ds, const uint32_t (&a)[32],
                      const uint32_t (&b2)[32]) {
  const int lane = kr & 31, row0 = kr & ~31;
  const uint32_t srow = ds + half * TILE + kr * 128, sw = kr & 7;
  if (u.split()) {
    // Rows past the sequence end are written too and never read.
    float4* dst = reinterpret_cast<float4*>(
        p.dkv_acc + ((static_cast<size_t>(u.item.slot) * p.hkv + u.g) * 2 + half) * (BN * D) + kr * D);
#pragma unroll
    for (int c = 0; c < 8; ++c)
      dst[c] = make_float4(__uint_as_float(a[4 * c]), __uint_as_float(a[4 * c + 1]), __uint_as_float(a[4 * c + 2]),
                           __uint_as_float(a[4 * c + 3]));
#pragma unroll
    for (int c = 0; c < 8; ++c)
      dst[8 + c] = make_float4(__uint_as_float(b2[4 * c]), __uint_as_float(b2[4 * c + 1]),
                               __uint_as_float(b2[4 * c + 2]), __uint_as_float(b2[4 * c + 3]));
    return false;
  }
  const float mul = half ? p.scale : 1.f;
  if (STG && u.k0 + row0 + 32 <= u.sp.len) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t(&x)[32] = c < 4 ? a : b2;
      const int e = 8 * (c & 3);
      st_shared_v4(srow + ((c ^ sw) << 4), pack_bf16(__uint_as_float(x[e]) * mul, __uint_as_float(x[e + 1]) * mul),
                   pack_bf16(__uint_as_float(x[e + 2]) * mul, __uint_as_float(x[e + 3]) * mul),
                   pack_bf16(__uint_as_float(x[e + 4]) * mul, __uint_as_float(x[e + 5]) * mul),
                   pack_bf16(__uint_as_float(x[e + 6]) * mul, __uint_as_float(x[e + 7]) * mul));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(half ? &p.tm_dk : &p.tm_dv, u.g * D, u.sp.start + u.k0 + row0, ds + half * TILE + row0 * 128);
      bulk_commit();
    }
    return true;
  }
  if (u.k0 + kr < u.sp.len) {
    __nv_bfloat16* dst = (half ? p.dk : p.dv) + (static_cast<size_t>(u.sp.start + u.k0 + kr) * p.hkv + u.g) * D;
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
  return false;
}

// STG: the staged dK / dV stores, for work lists of short units, where each
// unit's drain is a larger share of its time.  Kept out of the other variant:
// its presence alone measured ~1.5 % slower on long causal units.
template <int NS, int KVB, bool STG>
__global__ void __launch_bounds__(NTHR, 1) bwd_tc_kernel(const __grid_constant__ BwdTcK p) {
  using L = Layout<NS, KVB>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars<NS, KVB> bars;
  __shared__ int unit_slot[kUnitRing];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto b_uf = [&](int j) { return smem_u32(&bars.unit_full[j]); };
  auto b_ue = [&](int j) { return smem_u32(&bars.unit_empty[j]); };
  auto b_kvf = [&](int b) { return smem_u32(&bars.kv_full[b]); };
  auto b_kve = [&](int b) { return smem_u32(&bars.kv_empty[b]); };
  const uint32_t b_kvt = smem_u32(&bars.kv_tmem), b_done = smem_u32(&bars.kv_done);
  const uint32_t b_dkv = smem_u32(&bars.dkv_free);
  const uint32_t b_dqf = smem_u32(&bars.dq_full), b_dqe = smem_u32(&bars.dq_free);
  auto b_s = [&](int h) { return smem_u32(&bars.s_full[h]); };
  auto b_dp = [&](int h) { return smem_u32(&bars.dp_full[h]); };
  auto b_pt = [&](int h) { return smem_u32(&bars.pt_full[h]); };
  auto b_ds = [&](int h) { return smem_u32(&bars.ds_full[h]); };
  const uint32_t b_dr = smem_u32(&bars.drain);
  auto b_qf = [&](int s) { return smem_u32(&bars.q_full[s]); };
  auto b_qe = [&](int s) { return smem_u32(&bars.q_empty[s]); };

  if (tid == 0) {
    abort_flag = 0;
    for (int j = 0; j < kUnitRing; ++j) {
      mbar_init(b_uf(j), 1);
      mbar_init(b_ue(j), kUnitReaders);
    }
    for (int b = 0; b < KVB; ++b) {
      mbar_init(b_kvf(b), 1);
      mbar_init(b_kve(b), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_qf(s), 33);  // 32 cp.async arrivals + the TMA expect-tx arrival
      mbar_init(b_qe(s), 1);
    }
    mbar_init(b_kvt, 8);
    mbar_init(b_done, 1);
    mbar_init(b_dkv, 8);
    for (int h = 0; h < 2; ++h) {
      mbar_init(b_s(h), 1);
      mbar_init(b_dp(h), 1);
      mbar_init(b_pt(h), 4);
      mbar_init(b_ds(h), 4);
    }
    mbar_init(b_dqf, 1);
    mbar_init(b_dqe, 4);
    mbar_init(b_dr, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  if (tid < BN) {
    // Selector rows [1,1,1,0,...] (picks -l'/scale) and [0,0,0,1,1,1,0,0]
    // (picks -D) in bf16, and the zero block.
    constexpr uint32_t one = 0x3F80u;
    st_shared_v4(sb + L::OFF_SEL + tid * 16, one | (one << 16), one, 0u, 0u);
    st_shared_v4(sb + L::OFF_SEL + BN * 16 + tid * 16, 0u, one << 16, one | (one << 16), 0u);
    st_shared_v4(sb + L::OFF_ZERO + tid * 16, 0u, 0u, 0u, 0u);
    fence_async_smem();  // generic-proxy writes, read by the tensor core
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const Abort ab{&abort_flag, p.status};
  // This warp's r-th unit from the claim ring (whole warp): 1 = a unit, 0 =
  // the end of the list, -1 = a wait gave up.
  auto take = [&](int r, Unit& u) -> int {
    const int j = r % kUnitRing;
    if (!mbar_wait_warp(b_uf(j), (r / kUnitRing) & 1, ab)) return -1;
    const int idx = *static_cast<volatile int*>(&unit_slot[j]);
    __syncwarp();
    if (lane == 0) mbar_arrive(b_ue(j));
    return decode_unit(p, idx, u) ? 1 : 0;
  };

  if (warp < 4) {
    regs_dec<REGS_LOW>();
    if (warp == 0) {
      // ---------------------------------------------------------- Q/dO loader
      if (lane == 0) {
        tma_prefetch_map(&p.tm_q);
        tma_prefetch_map(&p.tm_do);
      }
      bool ok = true;
      int n = 0;  // steps issued
      Unit u;
      for (int r = 0; ok; ++r) {
        // Claim the CTA's r-th unit and publish it (whole warp, lane 0
        // claims); the slot is free once every reader took claim r - 4.
        const int j = r % kUnitRing;
        if (r >= kUnitRing && !(ok = mbar_wait_warp(b_ue(j), ((r / kUnitRing) - 1) & 1, ab))) break;
        int idx = 0;
        if (lane == 0) {
          idx = atomicAdd(p.unit_counter, 1);
          unit_slot[j] = idx;
          mbar_arrive(b_uf(j));  // release: the readers see the slot with the phase
        }
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (!decode_unit(p, idx, u)) break;
        for (int t = 0; t < u.nsteps; ++t, ++n) {
          const int s = n % NS;
          if (n >= NS && !(ok = mbar_wait_warp(b_qe(s), ((n / NS) - 1) & 1, ab))) break;
          const int h = step_head(p, u, t), q0 = step_q0(u, t);
          // Bias rows of the 128 query rows: asynchronous 16-byte copies that
          // complete on the stage's full barrier (rows past the sequence end
          // read row 0 and are masked by the element-wise warps).
#pragma unroll
          for (int r2 = lane; r2 < BM; r2 += 32) {
            const int qq = q0 + r2;
            const size_t idx = static_cast<size_t>(h) * p.T + u.sp.start + (qq < u.sp.len ? qq : 0);
            cp_async16(sb + L::OFF_BIAS + (s * BM + r2) * 16, p.bias + idx, true);
          }
          cp_async_arrive_noinc(b_qf(s));
          if (lane == 0) {
            mbar_expect_tx(b_qf(s), 2 * TILE);
            tma_load_2d(sb + L::OFF_Q + s * TILE, &p.tm_q, h * D, u.sp.start + q0, b_qf(s));
            tma_load_2d(sb + L::OFF_DO + s * TILE, &p.tm_do, h * D, u.sp.start + q0, b_qf(s));
          }
        }
      }
      if (lane == 0 && abort_flag)
        for (int m = max(0, n - NS); m < n; ++m) wait_drain(b_qf(m % NS), (m / NS) & 1);
    } else if (warp == 2) {
      // ---------------------------------------------------------- K/V loader
      // The whole warp takes the claims; lane 0 issues the loads.
      if (lane == 0) {
        tma_prefetch_map(&p.tm_k);
        tma_prefetch_map(&p.tm_v);
      }
      bool ok = true;
      int ru = 0;  // units loaded
      Unit u;
      for (int r = 0; ok; ++r) {
        const int got = take(r, u);
        if (got <= 0) {
          ok = got == 0;
          break;
        }
        if (u.nsteps == 0) continue;
        const int kb = ru % KVB;
        // The claim comes a few steps before the buffer frees: bring the
        // tiles into L2 now, so that the load at the boundary is short.
        if (lane == 0 && ru >= KVB) {
          tma_prefetch_l2_2d(&p.tm_k, u.g * D, u.sp.start + u.k0);
          tma_prefetch_l2_2d(&p.tm_v, u.g * D, u.sp.start + u.k0);
        }
        if (ru >= KVB && !(ok = mbar_wait_warp(b_kve(kb), ((ru / KVB) - 1) & 1, ab))) break;
        if (lane == 0) {
          mbar_expect_tx(b_kvf(kb), 2 * TILE);
          tma_load_2d(sb + L::OFF_K + 2 * kb * TILE, &p.tm_k, u.g * D, u.sp.start + u.k0, b_kvf(kb));
          tma_load_2d(sb + L::OFF_V + 2 * kb * TILE, &p.tm_v, u.g * D, u.sp.start + u.k0, b_kvf(kb));
        }
        ++ru;
      }
      if (lane == 0 && abort_flag)
        for (int m = max(0, ru - KVB); m < ru; ++m) wait_drain(b_kvf(m % KVB), (m / KVB) & 1);
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this code so every descriptor is warp-uniform; one
      // elected lane issues the MMAs and the commits that track them.
      const bool leader = elect_one();
      const uint32_t id_s = idesc_bf16(BN, HALF, false, false);  // S_h^T, dP_h^T: 128 keys x 64 queries
      const uint32_t id_kv = idesc_bf16(BN, D, false, true);     // dV, dK: 128 keys x 64
      const uint32_t id_q = idesc_bf16(BM, D, true, true);       // dQ: 128 queries x 64
      const uint64_t d_k = sdesc_sw128(sb + L::OFF_K, 16, 1024);   // MN-major B of dQ; buffer b: + 2 b TILE
      const uint64_t d_q = sdesc_sw128(sb + L::OFF_Q, 16, 1024);   // stage s: + s * TILE, half h: + h * 8 KB
      const uint64_t d_o = sdesc_sw128(sb + L::OFF_DO, 16, 1024);
      const uint64_t d_dsm = sdesc_sw128(sb + L::OFF_DS, TILE, 1024);  // MN-major A of dQ (two 64-query blocks)
      // S_h^T = K Q_h^T and dP_h^T = V dO_h^T of the step held in stage s
      // (A = K or V in Tensor Memory, B = the half's 64 query rows, K-major).
      // Bias product first (overwrites): a selector tile times the stage's
      // bias rows of the half adds -l'/scale to S^T and -D to dP^T.
      auto bias_desc = [&](int h, int s) {
        const uint32_t off = L::OFF_BIAS + (s * BM + h * HALF) * 16;
        return sdesc_nosw(sb + off, L::OFF_ZERO - off, 128);
      };
      const uint64_t d_sel_s = sdesc_nosw(sb + L::OFF_SEL, L::OFF_ZERO - L::OFF_SEL, 128);
      const uint64_t d_sel_dp =
          sdesc_nosw(sb + L::OFF_SEL + BN * 16, L::OFF_ZERO - (L::OFF_SEL + BN * 16), 128);
      auto issue_s = [&](int h, int s) {
        const uint64_t q = sdesc_add(d_q, s * TILE + h * HALF * 128);
        if (leader) mma_ss(tmem + TM_S + HALF * h, d_sel_s, bias_desc(h, s), id_s, 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          if (leader) mma_ts(tmem + TM_S + HALF * h, tmem + TM_K + kk * 8, sdesc_add(q, kk * 32), id_s, 1);
      };
      auto issue_dp = [&](int h, int s) {
        const uint64_t o = sdesc_add(d_o, s * TILE + h * HALF * 128);
        if (leader) mma_ss(tmem + TM_DP + HALF * h, d_sel_dp, bias_desc(h, s), id_s, 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          if (leader) mma_ts(tmem + TM_DP + HALF * h, tmem + TM_V + kk * 8, sdesc_add(o, kk * 32), id_s, 1);
      };
      bool ok = true;
      int n = 0, ru = 0;
      Unit u;
      for (int r = 0; ok; ++r) {
        const int got = take(r, u);
        if (got <= 0) {
          ok = got == 0;
          break;
        }
        if (u.nsteps == 0) continue;
        const int kb = ru % KVB;
        // K and V of the unit are in TMEM (the element-wise warps copied them
        // after their TMA landed, which this wait also acquires), and the
        // first stage of the unit has landed.
        if (!(ok = mbar_wait_warp(b_kvt, ru & 1, ab) && mbar_wait_warp(b_kvf(kb), (ru / KVB) & 1, ab) &&
                   mbar_wait_warp(b_qf(n % NS), (n / NS) & 1, ab)))
          break;
        fence_after_sync();
        for (int h = 0; h < 2; ++h) {
          issue_s(h, n % NS);
          if (leader) mma_commit(b_s(h));
        }
        for (int h = 0; h < 2; ++h) {
          issue_dp(h, n % NS);
          if (leader) mma_commit(b_dp(h));
        }
        const uint64_t dk_b = sdesc_add(d_k, 2 * kb * TILE);
        for (int t = 0; ok && t < u.nsteps; ++t, ++n) {
          const int s = n % NS, db = n & 1;
          const bool more = t + 1 < u.nsteps;
          // Phase 1 of each half is done (packed P^T in the S^T columns):
          // dV += P_h^T dO_h, then the next step's S_h^T over those columns
          // (the tensor core runs MMAs in issue order).
          for (int h = 0; h < 2 && ok; ++h) {
            if (!(ok = mbar_wait_warp(b_pt(h), n & 1, ab))) break;
            // The first dV product overwrites dV: the previous unit's dK, dV
            // must have left Tensor Memory.
            if (t == 0 && h == 0 && ru > 0 && !(ok = mbar_wait_warp(b_dkv, (ru - 1) & 1, ab))) break;
            fence_after_sync();
            const uint64_t o = sdesc_add(d_o, s * TILE + h * HALF * 128);
#pragma unroll
            for (int kk = 0; kk < HALF / 16; ++kk)
              if (leader)
                mma_ts(tmem + TM_DV, tmem + TM_S + HALF * h + kk * 8, sdesc_add(o, kk * 2048), id_kv,
                       (t > 0 || h > 0 || kk > 0) ? 1u : 0u);
            if (more) {
              if (h == 0) {
                if (!(ok = mbar_wait_warp(b_qf((n + 1) % NS), ((n + 1) / NS) & 1, ab))) break;
                fence_after_sync();
              }
              issue_s(h, (n + 1) % NS);
              if (leader) mma_commit(b_s(h));
            }
          }
          if (!ok) break;
          // Phase 2 of each half is done (packed dS^T in the dP^T columns):
          // dK += dS_h^T Q_h, then the next step's dP_h^T over those columns.
          for (int h = 0; h < 2 && ok; ++h) {
            if (!(ok = mbar_wait_warp(b_ds(h), n & 1, ab))) break;
            fence_after_sync();
            const uint64_t q = sdesc_add(d_q, s * TILE + h * HALF * 128);
#pragma unroll
            for (int kk = 0; kk < HALF / 16; ++kk)
              if (leader)
                mma_ts(tmem + TM_DK, tmem + TM_DP + HALF * h + kk * 8, sdesc_add(q, kk * 2048), id_kv,
                       (t > 0 || h > 0 || kk > 0) ? 1u : 0u);
            if (more) {
              issue_dp(h, (n + 1) % NS);
              if (leader) mma_commit(b_dp(h));
            }
          }
          if (!ok) break;
          if (leader) mma_commit(b_qe(s));  // Q(n), dO(n), l'(n), D(n) have no later reader
          if (n > 0) {
            if (!(ok = mbar_wait_warp(b_dqe, (n - 1) & 1, ab))) break;
            fence_after_sync();
          }
          const uint64_t dsm = sdesc_add(d_dsm, db * 2 * TILE);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            if (leader) mma_ss(tmem + TM_DQ, sdesc_add(dsm, kk * 2048), sdesc_add(dk_b, kk * 2048), id_q, kk > 0);
          if (leader) mma_commit(b_dqf);
        }
        if (!ok) break;
        // Every MMA of the unit: dK, dV are final and the K/V buffer is free.
        if (leader) {
          mma_commit(b_done);
          mma_commit(b_kve(kb));
        }
        ++ru;
      }
      if (leader) mma_commit(b_dr);
      __syncwarp();
      wait_drain(b_dr, 0);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ element-wise
    regs_inc<REGS_EW>();
    const int half = (warp - 4) >> 2;  // query rows [64 * half, 64 * half + 64) of each step
    const int kr = (warp & 3) * 32 + lane;
    const uint32_t lb = lane_base(warp);
    const uint32_t tS = tmem + TM_S + HALF * half + lb, tDP = tmem + TM_DP + HALF * half + lb;
    const uint32_t tKV = tmem + (half ? TM_V : TM_K) + lb;
    const uint32_t tAcc = tmem + (half ? TM_DK : TM_DV) + lb;
    const float sl2 = p.scale_log2;
    bool ok = true;
    bool stg = false;  // lane 0 has a dK / dV store reading this warp's dS^T rows
    int n = 0, ru = 0;
    Unit u, prev;
    // Reads the finished unit number `idx` (its dV / dK) out of TMEM,
    // releases the columns to the next unit's products, writes it.
    auto drain_unit = [&](const Unit& done, int idx) -> bool {
      if (!mbar_wait_warp(b_done, idx & 1, ab)) return false;
      fence_after_sync();
      uint32_t a[32], b2[32];
      tmem_ld32(tAcc, a);
      tmem_ld32(tAcc + 32, b2);
      tmem_ld_wait();
      reg_fence32(a);
      reg_fence32(b2);
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_dkv);
      stg = write_dkv<STG>(p, done, half, kr, sb + L::OFF_DS, a, b2);
      return true;
    };
    for (int r = 0; ok; ++r) {
      const int got = take(r, u);
      if (got <= 0) {
        ok = got == 0;
        break;
      }
      if (u.nsteps == 0) continue;
      const int kb = ru % KVB;
      if (!(ok = mbar_wait_warp(b_kvf(kb), (ru / KVB) & 1, ab))) break;
      {
        // This thread's row of K (first half) or V (second half) into TMEM,
        // where it is the A operand of S^T = K Q^T / dP^T = V dO^T.  The
        // previous unit's products that read these columns have completed:
        // their results were consumed by this warpgroup's last phase.
        const uint32_t src = sb + (half ? L::OFF_V : L::OFF_K) + 2 * kb * TILE + kr * 128;
        uint32_t rr[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = ld_shared_v4(src + ((c ^ (kr & 7)) << 4));
          rr[4 * c] = v.x, rr[4 * c + 1] = v.y, rr[4 * c + 2] = v.z, rr[4 * c + 3] = v.w;
        }
        tmem_st32(tKV, rr);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_kvt);
      }
      if (ru > 0 && !(ok = drain_unit(prev, ru - 1))) break;
      for (int t = 0; t < u.nsteps; ++t, ++n) {
        if (!(ok = mbar_wait_warp(b_s(half), n & 1, ab))) break;
        fence_after_sync();
        const int qh = step_q0(u, t) + HALF * half;
        const bool full = block_full(qh, HALF, u.k0, BN, u.sp.len, p.mask);
        const uint32_t rowb = sb + L::OFF_DS + (n & 1) * 2 * TILE + half * TILE + kr * 128;
        float pv[4][16];
        if (full) {
          ew_phase1<true>(tS, sl2, 0u, 0u, pv);
        } else {
          const int key = u.k0 + kr;
          ew_phase1<false>(tS, sl2, query_bits(key, qh, u.sp.len, p.mask), query_bits(key, qh + 32, u.sp.len, p.mask),
                           pv);
        }
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pt(half));
        if (!(ok = mbar_wait_warp(b_dp(half), n & 1, ab))) break;
        fence_after_sync();
        if (STG && stg) {
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          stg = false;
        }
        ew_phase2(tDP, rowb, kr, pv);
        tmem_st_wait();
        fence_before_sync();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_ds(half));
      }
      prev = u;
      ++ru;
    }
    if (ok && ru > 0) drain_unit(prev, ru - 1);
    if (STG && lane == 0) bulk_wait0();
  } else {
    // ------------------------------------------------------------ dQ drain
    regs_dec<REGS_DQ>();
    const int qr = (warp & 3) * 32 + lane;
    const bool leader = (warp == 12 && lane == 0);
    const uint32_t lb = lane_base(warp);
    const uint32_t tQ = tmem + TM_DQ + lb;
    const uint32_t stg = sb + L::OFF_STG;
    bool ok = true;
    int n = 0;
    Unit u;
    for (int r = 0; ok; ++r) {
      // The four drain warps decide together: they meet at named barriers,
      // so none may leave the loop while the others go on.
      const int got = take(r, u);
      if (!named_sync_and(1, 128, got >= 0)) {
        ok = false;
        break;
      }
      if (got == 0) break;
      for (int t = 0; t < u.nsteps; ++t, ++n) {
        if (!(ok = named_sync_and(1, 128, mbar_wait_warp(b_dqf, n & 1, ab)))) break;
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
        const int h = step_head(p, u, t), q0 = step_q0(u, t);
        const bool valid = q0 + qr < u.sp.len;
        if (leader) bulk_wait_read0();
        named_sync(1, 128);
        // Columns 0-31, then 32-63, through the one 16 KB staging tile.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t sw = ((i ^ (qr & 7)) << 4) + qr * 128;
          st_shared_v4(stg + sw, valid ? a[4 * i] : 0u, valid ? a[4 * i + 1] : 0u, valid ? a[4 * i + 2] : 0u,
                       valid ? a[4 * i + 3] : 0u);
        }
        fence_async_smem();
        named_sync(1, 128);
        if (leader) {
          tma_reduce_add_2d(&p.tm_dq, h * D, u.sp.start + q0, stg);
          bulk_commit();
          bulk_wait_read0();
        }
        named_sync(1, 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t sw = ((i ^ (qr & 7)) << 4) + qr * 128;
          st_shared_v4(stg + sw, valid ? b2[4 * i] : 0u, valid ? b2[4 * i + 1] : 0u, valid ? b2[4 * i + 2] : 0u,
                       valid ? b2[4 * i + 3] : 0u);
        }
        fence_async_smem();
        named_sync(1, 128);
        if (leader) {
          tma_reduce_add_2d(&p.tm_dq, h * D + 32, u.sp.start + q0, stg);
          bulk_commit();
        }
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

// The conversion pass after the main kernel, one launch with three kinds of
// blocks:
//   dQ     dQ = scale * accumulator -> bf16, two groups of eight values per
//          thread in flight, streaming loads (the accumulator is dead after);
//   dK, dV of split key tiles: the sum of the tile's per-chunk fp32 slots, in
//          chunk order (deterministic), -> bf16 (dK scaled), a flat
//          grid-stride pass over every 8-element group of the split tiles'
//          rows (a few MB spread over a few tiles: one block per tile would
//          leave most SMs idle);
//   dsink  the fixed-order sum of the preprocess partials, one warp per head
//          (deterministic).
struct DkvTile {
  uint32_t code;   // sequence | key tile << 16
  uint32_t slot0;  // slot of chunk 0
  uint32_t nchunks;
};

struct ConvK {
  // dQ
  const float* dq_acc;
  __nv_bfloat16* dq;
  long long n8;  // 8-element groups of dQ
  int q_blocks;
  // split tiles
  const float* dkv_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const int32_t* cu;
  int seqlen, hkv, n_tiles, kv_blocks;
  // dsink
  const float* part;
  int nparts, hq;
  float* dsink;
  float scale;
  DkvTile tiles[2048];
};
static_assert(sizeof(ConvK) < 32000, "kernel parameter block too large");

__global__ void __launch_bounds__(256) convert_kernel(const __grid_constant__ ConvK p) {
  const int bid = static_cast<int>(blockIdx.x);
  if (bid < p.q_blocks) {
    const long long stride = static_cast<long long>(p.q_blocks) * blockDim.x;
    auto emit = [&](long long i, const float4& a, const float4& c) {
      uint4 o;
      o.x = pack_bf16(a.x * p.scale, a.y * p.scale);
      o.y = pack_bf16(a.z * p.scale, a.w * p.scale);
      o.z = pack_bf16(c.x * p.scale, c.y * p.scale);
      o.w = pack_bf16(c.z * p.scale, c.w * p.scale);
      reinterpret_cast<uint4*>(p.dq)[i] = o;
    };
    const float4* acc4 = reinterpret_cast<const float4*>(p.dq_acc);
    long long i = static_cast<long long>(bid) * blockDim.x + threadIdx.x;
    for (; i + stride < p.n8; i += 2 * stride) {
      const float4 a0 = __ldcs(acc4 + 2 * i), c0 = __ldcs(acc4 + 2 * i + 1);
      const float4 a1 = __ldcs(acc4 + 2 * (i + stride)), c1 = __ldcs(acc4 + 2 * (i + stride) + 1);
      emit(i, a0, c0);
      emit(i + stride, a1, c1);
    }
    if (i < p.n8) emit(i, __ldcs(acc4 + 2 * i), __ldcs(acc4 + 2 * i + 1));
    return;
  }
  if (bid < p.q_blocks + p.kv_blocks) {
    const int per_row = p.hkv * 2 * (D / 8);  // 8-element groups per key row
    const long long per_tile = static_cast<long long>(BN) * per_row;
    const long long total = per_tile * p.n_tiles;
    const size_t slot_floats = static_cast<size_t>(p.hkv) * 2 * BN * D;
    for (long long i = (bid - p.q_blocks) * 256LL + threadIdx.x; i < total;
         i += static_cast<long long>(p.kv_blocks) * 256) {
      const int s = static_cast<int>(i / per_tile);
      const int rem0 = static_cast<int>(i - s * per_tile);
      const int r = rem0 / per_row, rem = rem0 - r * per_row;
      const DkvTile tile = p.tiles[s];
      const SeqSpan sp = seq_span(p.cu, p.seqlen, static_cast<int>(tile.code & 0xFFFFu));
      const int k0 = static_cast<int>(tile.code >> 16) * BN;
      if (k0 + r >= sp.len) continue;
      const int g = rem / (2 * (D / 8)), which = (rem / (D / 8)) & 1, c8 = rem % (D / 8);
      const float4* src = reinterpret_cast<const float4*>(
          p.dkv_acc + tile.slot0 * slot_floats + ((static_cast<size_t>(g) * 2 + which) * BN + r) * D + 8 * c8);
      float4 x = __ldcs(src), y = __ldcs(src + 1);
      for (uint32_t c = 1; c < tile.nchunks; ++c) {
        const float4* sc = src + c * (slot_floats / 4);
        const float4 xc = __ldcs(sc), yc = __ldcs(sc + 1);
        x = make_float4(x.x + xc.x, x.y + xc.y, x.z + xc.z, x.w + xc.w);
        y = make_float4(y.x + yc.x, y.y + yc.y, y.z + yc.z, y.w + yc.w);
      }
      const float mul = which ? p.scale : 1.f;
      uint4 o;
      o.x = pack_bf16(x.x * mul, x.y * mul);
      o.y = pack_bf16(x.z * mul, x.w * mul);
      o.z = pack_bf16(y.x * mul, y.y * mul);
      o.w = pack_bf16(y.z * mul, y.w * mul);
      const size_t row = static_cast<size_t>(sp.start + k0 + r);
      *reinterpret_cast<uint4*>((which ? p.dk : p.dv) + (row * p.hkv + g) * D + 8 * c8) = o;
    }
    return;
  }
  // Fixed-order reduction of the dsink partials: one warp per head.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = (bid - p.q_blocks - p.kv_blocks) * 8 + warp;
  if (h >= p.hq) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int i = lane;
  for (; i + 7 * 32 < p.nparts; i += 8 * 32) {
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] += p.part[static_cast<size_t>(i + 32 * u) * p.hq + h];
  }
  for (; i < p.nparts; i += 32) acc[0] += p.part[static_cast<size_t>(i) * p.hq + h];
  float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) p.dsink[h] = sum;
}

// Split tiles of a work list (each tile once, from its chunk 0).
std::vector<DkvTile> split_tiles(const std::vector<BwdItem>& items) {
  std::vector<DkvTile> tiles;
  for (const BwdItem& it : items)
    if (it.nchunks > 1 && it.chunk == 0)
      tiles.push_back({static_cast<uint32_t>(it.b) | (static_cast<uint32_t>(it.kt) << 16), it.slot, it.nchunks});
  return tiles;
}

}  // namespace

size_t bwd_split_acc_bytes(const Problem& pr) {
  if (pr.total_tokens == 0 || pr.num_seqs == 0) return 0;
  const int slots = bwd_split_slots(bwd_work_list(pr, bwd_qchunk(pr)));
  return static_cast<size_t>(slots) * pr.hkv * 2 * BN * D * sizeof(float);
}

int bwd_tc_main_slices(const Problem& pr) {
  if (pr.num_seqs == 0 || pr.total_tokens == 0 || pr.seqlen == 0) return 0;
  return static_cast<int>((bwd_work_list(pr, bwd_qchunk(pr)).size() + kMaxItems - 1) / kMaxItems);
}

int bwd_tc_main_launches(const Problem& pr) {
  if (pr.num_seqs == 0 || pr.total_tokens == 0 || pr.seqlen == 0) return 0;
  const std::vector<BwdItem> items = bwd_work_list(pr, bwd_qchunk(pr));
  constexpr size_t kMaxTiles = sizeof(ConvK::tiles) / sizeof(ConvK::tiles[0]);
  const size_t n_split = split_tiles(items).size();
  // Main kernel slices, then the conversion (its first launch also takes up
  // to kMaxTiles split tiles; more tiles need more launches).
  const size_t extra = n_split > kMaxTiles ? (n_split - 1) / kMaxTiles : 0;
  return static_cast<int>((items.size() + kMaxItems - 1) / kMaxItems + 1 + extra);
}

namespace {

template <int NS, int KVB, bool STG>
cudaError_t launch_main(const BwdTcK& k, int grid, cudaStream_t stream) {
  constexpr int smem = Layout<NS, KVB>::SMEM_DYN;
  cudaError_t e =
      cudaFuncSetAttribute(bwd_tc_kernel<NS, KVB, STG>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_tc_kernel<NS, KVB, STG><<<grid, NTHR, smem, stream>>>(k);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc_main(const Problem& pr, const BwdArgs& a, int* status, cudaStream_t stream) {
  if (pr.num_seqs == 0 || pr.total_tokens == 0 || pr.seqlen == 0) return cudaSuccess;
  thread_local BwdTcK k;  // 25 KB parameter block; host-side staging, one per host thread
  if (!make_rows_map(&k.tm_q, a.q, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_do, a.dout, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_k, a.k, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_v, a.v, pr.total_tokens, pr.hkv, BN) ||
      !make_f32_rows_map(&k.tm_dq, a.dq_accum, pr.total_tokens, pr.hq, BM) ||
      !make_rows_map(&k.tm_dk, a.dk, pr.total_tokens, pr.hkv, 32) ||
      !make_rows_map(&k.tm_dv, a.dv, pr.total_tokens, pr.hkv, 32))
    return cudaErrorInvalidValue;
  k.bias = static_cast<const uint4*>(a.bias);
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
  k.qchunk = bwd_qchunk(pr);
  k.dkv_acc = a.dkv_acc;
  const std::vector<BwdItem> items = bwd_work_list(pr, k.qchunk);
  const std::vector<DkvTile> tiles = split_tiles(items);
  if (!tiles.empty() && a.dkv_acc == nullptr) return cudaErrorInvalidValue;
  // Units of at most 32 steps on average (e.g. a 128-key window with 8 query
  // heads per kv head: 16) take the variant with the staged dK / dV stores.
  const bool short_units =
      !items.empty() && bwd_query_tiles_total(pr) * k.group <= 32LL * static_cast<long long>(items.size());
  const int sms = device_sms();
  cudaError_t e;
  if ((e = prof_begin(g_prof_bwd, stream)) != cudaSuccess) return e;
  for (size_t first = 0; first < items.size(); first += kMaxItems) {
    const int n = static_cast<int>(std::min<size_t>(kMaxItems, items.size() - first));
    std::copy(items.begin() + first, items.begin() + first + n, k.items);
    k.n_items = n;
    k.n_units = n * pr.hkv;
    k.unit_counter = a.unit_counters + first / kMaxItems;
    const int grid = std::min(sms, k.n_units);
    e = short_units ? launch_main<3, 1, true>(k, grid, stream) : launch_main<3, 1, false>(k, grid, stream);
    if (e != cudaSuccess) return e;
  }
  if ((e = prof_end(g_prof_bwd, stream)) != cudaSuccess) return e;
  // Conversion pass: dQ, the split tiles' dK/dV, dsink.
  thread_local ConvK c;
  c.dq_acc = a.dq_accum;
  c.dq = static_cast<__nv_bfloat16*>(a.dq);
  c.n8 = static_cast<long long>(pr.total_tokens) * pr.hq * D / 8;
  c.dkv_acc = a.dkv_acc;
  c.dk = static_cast<__nv_bfloat16*>(a.dk);
  c.dv = static_cast<__nv_bfloat16*>(a.dv);
  c.cu = pr.cu;
  c.seqlen = pr.seqlen;
  c.hkv = pr.hkv;
  c.part = a.dsink_part;
  c.nparts = a.preprocess_blocks;
  c.hq = pr.hq;
  c.dsink = a.dsink;
  c.scale = pr.scale;
  constexpr int kMaxTiles = static_cast<int>(sizeof(c.tiles) / sizeof(c.tiles[0]));
  size_t first = 0;
  do {
    const int n = static_cast<int>(std::min<size_t>(kMaxTiles, tiles.size() - first));
    std::copy(tiles.begin() + first, tiles.begin() + first + n, c.tiles);
    c.n_tiles = n;
    const bool head = first == 0;  // the first launch also converts dQ and reduces dsink
    c.q_blocks = head ? static_cast<int>(std::max<long long>(1, std::min<long long>((c.n8 + 255) / 256, 16LL * sms))) : 0;
    const long long groups = static_cast<long long>(n) * BN * pr.hkv * 2 * (D / 8);
    c.kv_blocks = static_cast<int>(std::min<long long>((groups + 255) / 256, 8LL * sms));
    const int red_blocks = head ? (pr.hq + 7) / 8 : 0;
    convert_kernel<<<c.q_blocks + c.kv_blocks + red_blocks, 256, 0, stream>>>(c);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    first += n;
  } while (first < tiles.size());
  return cudaSuccess;
}

}  // namespace sa
