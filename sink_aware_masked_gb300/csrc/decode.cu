// Decode (rollout-side) forward of sink-aware attention: the last n query
// positions of each sequence against the sequence's whole key/value history.
//
// The pages' policy rollouts sample from the current policy turn by turn
// (SinkFlex-RL, zh page, "Rollout worker"), and the GPT-OSS RL page takes the
// sink-aware forward from an inference-engine FlashAttention fork ("GPT-OSS
// agentic RL training", FlashAttention v3 implementation).  Same mask, sink
// and lse as the full forward: every decode row equals the same row of the
// full-sequence forward.
//
// Few query rows meet a long key history, so the work is a stream over K and
// V bounded by HBM bandwidth (the 8 query heads of a GQA group share every
// key: about 8 FLOP per byte at n = 1).  The key range of each (sequence, kv
// head) is split into chunks of whole 128-key tiles (split-KV); one CTA per
// (chunk, kv head) streams its tiles by TMA through a 2-stage mbarrier ring
// (three such CTAs resident per SM)
// and computes, for the group x n query rows, a partial online softmax
// (running max m in log2 units, row sum l, unnormalised O) with warp-level
// bf16 MMAs.  The last CTA of a (sequence, kv head) to finish (a counter in
// the workspace, incremented after the partial is written and fenced) merges
// the partials of each row,
//     m = max m_i,  l = sum 2^{m_i - m} l_i,  O = sum 2^{m_i - m} O_i / l,
// and only then applies the sink: lse = ln2 (m + log2 l), alpha =
// sigmoid(lse - s_h), O <- alpha O (summary page, sink scaling of the output
// by sigma(l - s_h)); it then clears the counter for the next call.  The
// chunks of a sequence hold equal numbers of tiles (within one).
//
// Rows r of one (sequence, kv head): r = i * group + j is query position
// L - n + i of query head g * group + j.  Warps split the rows into groups of
// at most two 16-row blocks and the keys of each tile among the rest; the
// warps that share rows are merged inside the CTA before the partial is
// written.  Every mbarrier wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

#include <algorithm>
#include <vector>

namespace sa {
namespace {

using namespace tc;

constexpr int D = kHeadDim;
constexpr int BN = 128;           // keys per tile
constexpr int NS = 2;             // K/V stages (three CTAs per SM fit: 65 KB of shared memory each)
constexpr int NTHR = 128;
constexpr int TILE = BN * D * 2;  // 16 KB
constexpr int SMEM_DYN = NS * 2 * TILE + 1024;

// The work list's capacity is a template parameter: a short list keeps the
// kernel parameter block small (a 16 KB block costs ~1.3 us more per launch
// than a small one, a few per cent of a short decode step).
constexpr int kDecodeSmallItems = 256;

template <int CAP>
struct DecK {
  CUtensorMap tm_k, tm_v;
  const __nv_bfloat16* q;  // [B * n, Hq, 64]
  const float* sink;
  __nv_bfloat16* o;        // [B * n, Hq, 64]
  float* lse;              // [Hq, B * n]
  int* counters;           // [B * Hkv] chunks finished; zero between calls
  float* ws_acc;           // [items * Hkv, R, 64] unnormalised O of each partial
  float2* ws_ml;           // [items * Hkv, Rml]: (m in log2 units of the scaled score, l)
  const int32_t* cu;       // key/value offsets or nullptr (uniform length kv_len)
  int* status;
  int kv_len;
  int n, hq, hkv, group, R;
  int Rml;                 // R rounded up to even: (max, sum) blocks are whole 16-byte units
  MaskParams mask;
  float scale_log2;
  int num_seqs;
  int tiles_per_split;  // chunks of a sequence: ceil(tiles / tiles_per_split), equal shares
  int n_items;
  uint32_t items[CAP];  // sequence | (chunk << 16), chunks of a sequence consecutive
};
static_assert(sizeof(DecK<kDecodeMaxItems>) < 32000, "kernel parameter block too large");

// Key tiles that the query rows [L - n, L - 1] see: the prefix tiles below the
// window, then the window/causal band (same arithmetic as the full forward).
struct KeyTiles {
  int lo_t, n_pre, n_tiles;
  SA_DEV int k0(int j) const { return (j < n_pre ? j : lo_t + (j - n_pre)) * BN; }
};

SA_DEV KeyTiles key_tiles(int L, int n, const MaskParams& m) {
  const KeyRange kr = key_range(L - n, L - 1, L, m);
  KeyTiles t;
  t.lo_t = kr.lo / BN;
  t.n_pre = min((kr.pre_end + BN - 1) / BN, t.lo_t);
  t.n_tiles = t.n_pre + (kr.hi / BN - t.lo_t + 1);
  return t;
}

SA_DEV float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
SA_DEV float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// MB: 16-row blocks covering the R rows (1, 2, 4 or 8).
template <int MB, int CAP>
__global__ void __launch_bounds__(NTHR, 3) decode_split_kernel(const __grid_constant__ DecK<CAP> p) {
  constexpr int MBW = MB < 2 ? MB : 2;  // row blocks per warp
  constexpr int WR = MB / MBW;          // warps splitting the rows
  constexpr int WK = 4 / WR;            // warps splitting the keys of a tile
  constexpr int KW = BN / WK;           // keys per warp per tile: 32, 64 or 128
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[NS];
  __shared__ uint64_t merge_bar;
  __shared__ int abort_flag;
  __shared__ float red_m[4][32];  // per warp: running max of its (up to) 32 rows
  __shared__ float red_l[4][32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wr = warp / WK, wk = warp % WK;
  const int item_idx = blockIdx.x, g = blockIdx.y;
  const uint32_t item = p.items[item_idx];
  const int b = static_cast<int>(item & 0xFFFFu), split = static_cast<int>(item >> 16);
  const SeqSpan sp = seq_span(p.cu, p.kv_len, b);
  const int L = sp.len, n = p.n;
  const KeyTiles kt = key_tiles(L, n, p.mask);
  const int nsplit = (kt.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  const int j0 = split * kt.n_tiles / nsplit, j1 = (split + 1) * kt.n_tiles / nsplit;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&full[s]), 1);
    mbar_init(smem_u32(&merge_bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{&abort_flag, p.status};
  auto issue = [&](int j) {
    const int s = (j - j0) % NS;
    const uint32_t bar = smem_u32(&full[s]);
    const int row = sp.start + kt.k0(j);
    mbar_expect_tx(bar, 2 * TILE);
    tma_load_2d(sb + s * 2 * TILE, &p.tm_k, g * D, row, bar);
    tma_load_2d(sb + s * 2 * TILE + TILE, &p.tm_v, g * D, row, bar);
  };
  int issued = j0;  // tiles [j0, issued) have been requested
  if (tid == 0) {
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    for (; issued < min(j0 + NS, j1); ++issued) issue(issued);
  }

  // Q fragments (A operand, row-major 16 x 16) of this warp's row blocks.
  const int row0 = wr * MBW * 16;
  uint32_t qa[MBW][4][4];
#pragma unroll
  for (int mb = 0; mb < MBW; ++mb)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = row0 + mb * 16 + (lane >> 2) + 8 * hr;
      const uint32_t* src = nullptr;
      if (r < p.R) {
        const int i = r / p.group, jh = r - i * p.group;
        src = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(b * n + i) * p.hq + g * p.group + jh) * D);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int c = ks * 8 + (lane & 3);  // 32-bit word index of dims 2c, 2c + 1
        qa[mb][ks][hr] = src ? __ldg(src + c) : 0u;
        qa[mb][ks][2 + hr] = src ? __ldg(src + c + 4) : 0u;
      }
    }

  float o_acc[MBW][8][4];
  float m_run[MBW][2], l_run[MBW][2];
#pragma unroll
  for (int mb = 0; mb < MBW; ++mb) {
#pragma unroll
    for (int dn = 0; dn < 8; ++dn)
#pragma unroll
      for (int e = 0; e < 4; ++e) o_acc[mb][dn][e] = 0.f;
    m_run[mb][0] = m_run[mb][1] = -INFINITY;
    l_run[mb][0] = l_run[mb][1] = 0.f;
  }
  // Query position of each of this thread's rows (rows past R are padding).
  int qpos[MBW][2];
#pragma unroll
  for (int mb = 0; mb < MBW; ++mb)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) qpos[mb][hr] = L - n + (row0 + mb * 16 + (lane >> 2) + 8 * hr) / p.group;
  const float sl2 = p.scale_log2;

  bool failed = false;
  int consumed = j0;
  for (int j = j0; j < j1; ++j) {
    const int s = (j - j0) % NS;
    const bool ok = mbar_wait(smem_u32(&full[s]), ((j - j0) / NS) & 1, ab);
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const int k0 = kt.k0(j);
    const uint32_t kb = sb + s * 2 * TILE, vb = kb + TILE;
    const bool all_visible = block_full(L - n, n, k0, BN, L, p.mask);
#pragma unroll 1
    for (int sub = 0; sub < KW / 32; ++sub) {
      const int kbase = wk * KW + sub * 32;  // first key of this 32-key block within the tile
      float sacc[MBW][4][4];
#pragma unroll
      for (int mb = 0; mb < MBW; ++mb)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mb][nt][e] = 0.f;
      // S = Q K^T: B fragments from the key rows (ldmatrix, 8 keys x 8 dims per matrix).
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int m = lane >> 3;
          const int key = kbase + (2 * np + (m >> 1)) * 8 + (lane & 7);
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kb + swz(key, 2 * ks + (m & 1)), r0, r1, r2, r3);
#pragma unroll
          for (int mb = 0; mb < MBW; ++mb) {
            mma16816(sacc[mb][2 * np], qa[mb][ks], r0, r1);
            mma16816(sacc[mb][2 * np + 1], qa[mb][ks], r2, r3);
          }
        }
      // Online softmax in log2 units; element e of n-tile nt is key
      // kbase + 8 nt + 2 (lane % 4) + (e & 1) of row half e >> 1.
      uint32_t pa[MBW][2][4];
#pragma unroll
      for (int mb = 0; mb < MBW; ++mb) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          float x[8];
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = sacc[mb][nt][2 * hr + e] * sl2;
              if (!all_visible) {
                const int key = k0 + kbase + 8 * nt + 2 * (lane & 3) + e;
                if (!visible(qpos[mb][hr], key, L, p.mask)) v = -INFINITY;
              }
              x[2 * nt + e] = v;
            }
          float mx = x[0];
#pragma unroll
          for (int e = 1; e < 8; ++e) mx = fmaxf(mx, x[e]);
          mx = quad_max(mx);
          const float m_new = fmaxf(m_run[mb][hr], mx);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float factor = ex2(m_run[mb][hr] - m_use);  // 0 while nothing was visible
          m_run[mb][hr] = m_new;
          float sum = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = ex2(x[e] - m_use);
            sum += x[e];
          }
          l_run[mb][hr] = l_run[mb][hr] * factor + sum;
#pragma unroll
          for (int dn = 0; dn < 8; ++dn) {
            o_acc[mb][dn][2 * hr] *= factor;
            o_acc[mb][dn][2 * hr + 1] *= factor;
          }
          // P as the A operand of P V: keys 16 kk + [0, 16) of this block.
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            pa[mb][kk][hr] = pack_bf16(x[4 * kk], x[4 * kk + 1]);
            pa[mb][kk][2 + hr] = pack_bf16(x[4 * kk + 2], x[4 * kk + 3]);
          }
        }
      }
      // O += P V: B fragments from the value rows, transposed (ldmatrix.trans).
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          const int m = lane >> 3;
          const int key = kbase + 16 * kk + (m & 1) * 8 + (lane & 7);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vb + swz(key, 2 * dp + (m >> 1)), r0, r1, r2, r3);
#pragma unroll
          for (int mb = 0; mb < MBW; ++mb) {
            mma16816(o_acc[mb][2 * dp], pa[mb][kk], r0, r1);
            mma16816(o_acc[mb][2 * dp + 1], pa[mb][kk], r2, r3);
          }
        }
    }
    consumed = j + 1;
    __syncthreads();  // every warp is done with stage s
    if (tid == 0 && issued < j1) {
      issue(issued);
      ++issued;
    }
  }
  if (failed) {
    // Let the copies still in flight land before the CTA leaves.
    if (tid == 0)
      for (int j = consumed; j < issued; ++j) {
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&full[(j - j0) % NS]), ((j - j0) / NS) & 1))
          if (clock64() - t0 > kTimeoutCycles) break;
      }
    return;
  }

  // Merge the warps that share rows: common maximum, then sums of l and O.
#pragma unroll
  for (int mb = 0; mb < MBW; ++mb)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l_run[mb][hr] = quad_sum(l_run[mb][hr]);
      if ((lane & 3) == 0) red_m[warp][mb * 16 + (lane >> 2) + 8 * hr] = m_run[mb][hr];
    }
  __syncthreads();
  float* acc_s = reinterpret_cast<float*>(smem);  // [WK][MB * 16][64]; the stages are no longer in use
  constexpr int RP = MB * 16;
#pragma unroll
  for (int mb = 0; mb < MBW; ++mb)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int rl = mb * 16 + (lane >> 2) + 8 * hr;  // row within the warp's block
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < WK; ++w) M = fmaxf(M, red_m[wr * WK + w][rl]);
      const float sc = (m_run[mb][hr] == -INFINITY) ? 0.f : ex2(m_run[mb][hr] - M);
      float* dst = acc_s + (static_cast<size_t>(wk) * RP + row0 + rl) * D + 2 * (lane & 3);
#pragma unroll
      for (int dn = 0; dn < 8; ++dn)
        *reinterpret_cast<float2*>(dst + 8 * dn) =
            make_float2(o_acc[mb][dn][2 * hr] * sc, o_acc[mb][dn][2 * hr + 1] * sc);
      if ((lane & 3) == 0) red_l[warp][rl] = l_run[mb][hr] * sc;
    }
  __syncthreads();
  const size_t part = static_cast<size_t>(item_idx) * p.hkv + g;
  for (int idx = tid; idx < p.R * D; idx += NTHR) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < WK; ++w) a += acc_s[static_cast<size_t>(w) * RP * D + idx];
    p.ws_acc[part * p.R * D + idx] = a;
  }
  for (int r = tid; r < p.R; r += NTHR) {
    const int wr2 = r / (MBW * 16), rl = r - wr2 * MBW * 16;
    float M = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < WK; ++w) {
      M = fmaxf(M, red_m[wr2 * WK + w][rl]);
      l += red_l[wr2 * WK + w][rl];
    }
    p.ws_ml[part * p.Rml + r] = make_float2(M, l);
  }

  // The last chunk of this (sequence, kv head) to finish merges all of them.
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(p.counters + b * p.hkv + g, 1) == nsplit - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // Partials of chunk c: O at ws_acc + (part0 + c Hkv) R 64, (max, sum) at
  // ws_ml + (part0 + c Hkv) Rml.  They are staged in batches through the
  // (now idle) stage buffers by bulk copies, then merged from shared memory
  // with an online rescale per (row, dim pair) unit.
  const size_t part0 = static_cast<size_t>(item_idx - split) * p.hkv + g;
  const uint32_t blk_acc = static_cast<uint32_t>(p.R) * D * 4, blk_ml = static_cast<uint32_t>(p.Rml) * 8;
  const int per_batch = max(1, (NS * 2 * TILE) / static_cast<int>(blk_acc + blk_ml));
  constexpr int UP = MB * 4;  // units per thread: (MB * 16 rows) x 32 dim pairs / 128 threads
  float2 acc[UP];
  float Mu[UP], lu[UP];
#pragma unroll
  for (int k = 0; k < UP; ++k) {
    acc[k] = make_float2(0.f, 0.f);
    Mu[k] = -INFINITY;
    lu[k] = 0.f;
  }
  const float* stg_acc = reinterpret_cast<const float*>(smem);
  const float2* ml_s = reinterpret_cast<const float2*>(smem + per_batch * blk_acc);
  if (tid == 0) fence_proxy_async_global();  // the partials were written through the generic proxy
  for (int c0 = 0, batch = 0; c0 < nsplit; c0 += per_batch, ++batch) {
    const int cnt = min(per_batch, nsplit - c0);
    const uint32_t bar = smem_u32(&merge_bar);
    if (tid == 0) {
      mbar_expect_tx(bar, cnt * (blk_acc + blk_ml));
      for (int c = 0; c < cnt; ++c) {
        const size_t pc = part0 + static_cast<size_t>(c0 + c) * p.hkv;
        bulk_load(sb + c * blk_acc, p.ws_acc + pc * p.R * D, blk_acc, bar);
        bulk_load(sb + per_batch * blk_acc + c * blk_ml, p.ws_ml + pc * p.Rml, blk_ml, bar);
      }
    }
    const bool ok = mbar_wait(bar, batch & 1, ab);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {  // let the copies still in flight land before the CTA leaves
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, batch & 1) && clock64() - t0 < kTimeoutCycles) {
        }
      }
      return;
    }
#pragma unroll
    for (int k = 0; k < UP; ++k) {
      const int u = tid + NTHR * k, r = u >> 5, d2 = u & 31;
      if (r >= p.R) continue;
      for (int c = 0; c < cnt; ++c) {
        const float2 mv = ml_s[c * p.Rml + r];
        if (mv.x == -INFINITY) continue;
        if (mv.x > Mu[k]) {
          const float sc = (Mu[k] == -INFINITY) ? 0.f : ex2(Mu[k] - mv.x);
          acc[k].x *= sc;
          acc[k].y *= sc;
          lu[k] *= sc;
          Mu[k] = mv.x;
        }
        const float w = ex2(mv.x - Mu[k]);
        const float2 a = reinterpret_cast<const float2*>(stg_acc + (static_cast<size_t>(c) * p.R + r) * D)[d2];
        acc[k].x += w * a.x;
        acc[k].y += w * a.y;
        lu[k] += w * mv.y;
      }
    }
    __syncthreads();  // the next batch overwrites the staging buffers
  }
#pragma unroll
  for (int k = 0; k < UP; ++k) {
    const int u = tid + NTHR * k, r = u >> 5, d2 = u & 31;
    if (r >= p.R) continue;
    const float l = lu[k], M = Mu[k];
    const int i = r / p.group, h = g * p.group + (r - i * p.group), bn = b * n + i;
    const float lse = (l > 0.f) ? (M + __log2f(l)) * kLn2 : -INFINITY;
    const float alpha = 1.f / (1.f + ex2((__ldg(p.sink + h) - lse) * kLog2e));
    const float fac = (l > 0.f) ? alpha / l : 0.f;
    reinterpret_cast<uint32_t*>(p.o + (static_cast<size_t>(bn) * p.hq + h) * D)[d2] =
        pack_bf16(acc[k].x * fac, acc[k].y * fac);
    if (d2 == 0) p.lse[static_cast<size_t>(h) * p.num_seqs * n + bn] = lse;
  }
  if (tid == 0) p.counters[b * p.hkv + g] = 0;  // every chunk of this call has counted
}

}  // namespace

DecodePlan decode_plan(const Problem& p, int n) {
  DecodePlan pl;
  const int sms = device_sms();
  std::vector<int> tiles(p.num_seqs);
  long long total = 0;
  for (int b = 0; b < p.num_seqs; ++b) {
    const int len = p.cu_host ? p.cu_host[b + 1] - p.cu_host[b] : p.seqlen;
    // Same arithmetic as key_range() for query rows [len - n, len - 1].
    const int q0 = len - n, hi = len - 1;
    const int lo = (p.window < 0) ? 0 : std::max(0, q0 - p.window);
    const int pre_end = std::max(0, std::min(std::min(p.prefix, lo), hi + 1));
    const int lo_t = lo / BN;
    const int n_pre = std::min((pre_end + BN - 1) / BN, lo_t);
    tiles[b] = n_pre + (hi / BN - lo_t + 1);
    total += tiles[b];
  }
  // Chunks per kv head: `factor` x the SMs / kv heads.  Each CTA pays a
  // pipeline fill and a partial write, and the key stream shares HBM
  // bandwidth, so fewer, longer chunks win until the grid keeps the three
  // resident CTAs per SM busy; the chunks of a sequence are equal, so the CTA
  // count rounds per sequence.  Measured (2 to 6 x the SMs, two-stage ring,
  // three CTAs per SM): a single 16-row block per kv head (one query row per
  // sequence for GQA 8) with at least 1024 key tiles per kv head, e.g.
  // 32 x 8192, wins at 4; fewer tiles (packed trajectories, windows) and
  // wider row blocks (8 x 32768 x 4 rows) win at 2.  At least two tiles per
  // chunk, and no more items than the parameter block holds.
  const int rows = (p.hq / std::max(p.hkv, 1)) * n;
  const int factor = (rows <= 16 && total >= 1024) ? 4 : 2;
  const long long want = std::max<long long>(1, static_cast<long long>(factor) * std::max(sms, 1) / std::max(p.hkv, 1));
  int tps = static_cast<int>(std::max<long long>(2, (total + want - 1) / want));
  for (;;) {
    long long items = 0;
    for (int b = 0; b < p.num_seqs; ++b) items += (tiles[b] + tps - 1) / tps;
    if (items <= kDecodeMaxItems) break;
    tps *= 2;
  }
  pl.tiles_per_split = tps;
  pl.items.clear();
  for (int b = 0; b < p.num_seqs; ++b) {
    const int chunks = (tiles[b] + tps - 1) / tps;
    for (int c = 0; c < chunks; ++c) pl.items.push_back(static_cast<uint32_t>(b) | (static_cast<uint32_t>(c) << 16));
  }
  const int R = (p.hq / p.hkv) * n;
  pl.acc_bytes = pl.items.size() * p.hkv * static_cast<size_t>(R) * D * 4;
  pl.ml_bytes = pl.items.size() * p.hkv * static_cast<size_t>((R + 1) & ~1) * 8;
  pl.counter_bytes = static_cast<size_t>(p.num_seqs) * p.hkv * 4;
  return pl;
}

namespace {

template <int CAP>
cudaError_t launch_decode_cap(const Problem& pr, int n, const DecodeArgs& a, const DecodePlan& pl, int* status,
                              cudaStream_t stream) {
  thread_local DecK<CAP> k;
  if (!make_rows_map(&k.tm_k, a.k, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_v, a.v, pr.total_tokens, pr.hkv, BN))
    return cudaErrorInvalidValue;
  const int group = pr.hq / pr.hkv, R = group * n;
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.sink = a.sink;
  k.o = static_cast<__nv_bfloat16*>(a.o);
  k.lse = a.lse;
  k.counters = a.counters;
  k.num_seqs = pr.num_seqs;
  k.ws_acc = a.ws_acc;
  k.ws_ml = reinterpret_cast<float2*>(a.ws_ml);
  k.cu = pr.cu;
  k.status = status;
  k.kv_len = pr.seqlen;
  k.n = n;
  k.hq = pr.hq;
  k.hkv = pr.hkv;
  k.group = group;
  k.R = R;
  k.Rml = (R + 1) & ~1;
  k.mask = MaskParams{pr.window, pr.prefix, pr.causal};
  k.scale_log2 = pr.scale * kLog2e;
  k.tiles_per_split = pl.tiles_per_split;
  k.n_items = static_cast<int>(pl.items.size());
  std::copy(pl.items.begin(), pl.items.end(), k.items);
  const int mb = R <= 16 ? 1 : R <= 32 ? 2 : R <= 64 ? 4 : 8;
  const dim3 grid(k.n_items, pr.hkv);
  cudaError_t e = prof_begin(g_prof_dec, stream);
  if (e != cudaSuccess) return e;
  switch (mb) {
#define SA_DECODE_CASE(MBV)                                                                                    \
  case MBV:                                                                                                    \
    if ((e = cudaFuncSetAttribute(decode_split_kernel<MBV, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                  SMEM_DYN)) != cudaSuccess)                                                   \
      return e;                                                                                                \
    decode_split_kernel<MBV, CAP><<<grid, NTHR, SMEM_DYN, stream>>>(k);                                        \
    break;
    SA_DECODE_CASE(1)
    SA_DECODE_CASE(2)
    SA_DECODE_CASE(4)
    SA_DECODE_CASE(8)
#undef SA_DECODE_CASE
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(g_prof_dec, stream);
}

}  // namespace

cudaError_t launch_decode(const Problem& pr, int n, const DecodeArgs& a, const DecodePlan& pl, int* status,
                          cudaStream_t stream) {
  if (pr.num_seqs == 0) return cudaSuccess;
  if (pl.items.size() > static_cast<size_t>(kDecodeMaxItems)) return cudaErrorInvalidValue;
  return pl.items.size() <= static_cast<size_t>(kDecodeSmallItems)
             ? launch_decode_cap<kDecodeSmallItems>(pr, n, a, pl, status, stream)
             : launch_decode_cap<kDecodeMaxItems>(pr, n, a, pl, status, stream);
}

}  // namespace sa
