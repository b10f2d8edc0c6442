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
// head) is split into chunks of whole 128-key tiles (split-KV), one CTA per
// (chunk, kv head); the partials are merged by the last CTA of each
// (sequence, kv head) with the sink applied once (decode_common.cuh).
//
// This file holds the plan, the launcher and the kernel for a single 16-row
// block (R = group x n <= 16, e.g. one new row per sequence with GQA 8) on
// steps too small for the tensor-core kernel of decode_tc.cu: the
// CTA streams its tiles by TMA through a 2-stage mbarrier ring (three such
// CTAs resident per SM) and computes a partial online softmax (running max m
// in log2 units, row sum l, unnormalised O) with warp-level bf16 MMAs, the
// four warps splitting the keys of each tile and merging in shared memory
// before the partial is written.  Wider row blocks, and 16-row blocks of
// large steps, run on the tensor-core kernel.  Every mbarrier wait is
// bounded.
#include "decode_common.cuh"

#include <algorithm>
#include <vector>

namespace sa {
namespace {

using namespace tc;
using namespace dec;

constexpr int NS = 2;             // K/V stages (three CTAs per SM fit: 65 KB of shared memory each)
constexpr long long kTcMinTiles = 128;   // key tiles per kv head from which 16 rows go to the tensor cores
constexpr int NTHR = 128;
constexpr int SMEM_DYN = NS * 2 * TILE + 1024;

SA_DEV float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
SA_DEV float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

// MB: 16-row blocks covering the R rows (launched with MB = 1; the body
// also supports 2, 4 and 8).
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
  const Chunk ch = chunk_of(p, item_idx);
  const SeqSpan sp = ch.sp;
  const int b = ch.b, L = sp.len, n = p.n;
  const KeyTiles kt = ch.kt;
  const int j0 = ch.j0, j1 = ch.j1;

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
  auto row_ml = [&](int r, float& M, float& l) {
    const int wr2 = r / (MBW * 16), rl = r - wr2 * MBW * 16;
    M = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int w = 0; w < WK; ++w) {
      M = fmaxf(M, red_m[wr2 * WK + w][rl]);
      l += red_l[wr2 * WK + w][rl];
    }
  };
  if (ch.nsplit == 1) {
    // The only chunk of this (sequence, kv head): finish the rows here,
    // without the round trip through the workspace and the counter.
    for (int u = tid; u < p.R * 32; u += NTHR) {
      const int r = u >> 5, d2 = u & 31;
      float M, l, lse;
      row_ml(r, M, l);
      const float fac = row_scale(p, ch, g, r, M, l, l, lse);
      float2 a = make_float2(0.f, 0.f);
#pragma unroll
      for (int w = 0; w < WK; ++w) {
        const float2 v = reinterpret_cast<const float2*>(acc_s + (static_cast<size_t>(w) * RP + r) * D)[d2];
        a.x += v.x;
        a.y += v.y;
      }
      store_pair(p, ch, g, r, d2, a.x * fac, a.y * fac);
      if (d2 == 0) store_lse(p, ch, g, r, lse);
    }
    return;
  }
  const size_t part = static_cast<size_t>(item_idx) * p.hkv + g;
  for (int idx = tid; idx < p.R * D; idx += NTHR) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < WK; ++w) a += acc_s[static_cast<size_t>(w) * RP * D + idx];
    p.ws_acc[part * p.R * D + idx] = a;
  }
  for (int r = tid; r < p.R; r += NTHR) {
    float M, l;
    row_ml(r, M, l);
    p.ws_ml[part * p.R + r] = make_float4(M, l, l, 0.f);
  }

  // The last chunk of this (sequence, kv head) to finish merges all of them
  // (the stage buffers are idle now).
  __shared__ int is_last;
  if (!count_partial(p, ch, g, &is_last)) return;
  merge_partials<MB * 4, NTHR>(p, ch, g, item_idx, smem, NS * 2 * TILE, smem_u32(&merge_bar), ab);
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
  auto items_at = [&](int t) {
    long long items = 0;
    for (int b = 0; b < p.num_seqs; ++b) items += (tiles[b] + t - 1) / t;
    return items;
  };
  // Kernel: the tensor-core one above 16 rows, and for 16 or fewer from 128
  // key tiles per kv head.  Measured, 16 rows: 2048 tiles (32 x 8192)
  // 6033 against 5429 GB/s, 253 tiles (the packed step) 24.3 against
  // 25.0 us; at 96 tiles (the windowed step, three per CTA) the warp-MMA
  // kernel with its lighter CTAs wins, 14.3 against 16.4 us.
  pl.tensor_core = rows > 16 || total >= kTcMinTiles;
  int tps;
  if (!pl.tensor_core) {
    const int factor = total >= 1024 ? 4 : 2;
    const long long want =
        std::max<long long>(1, static_cast<long long>(factor) * std::max(sms, 1) / std::max(p.hkv, 1));
    tps = static_cast<int>(std::max<long long>(2, (total + want - 1) / want));
    while (items_at(tps) > kDecodeMaxItems) tps *= 2;
  } else {
    // Tensor-core kernel (two CTAs per SM up to 64 rows, one above): each CTA
    // is a latency-bound stream, so the grid must fit in one wave of
    // resident CTAs (a second wave of a few CTAs doubles the step).  The
    // smallest chunk length whose item count fits: items_at() does not grow
    // with the length, so a binary search finds it.
    const int per_sm = rows <= 64 ? 2 : 1;
    const long long fit = std::max<long long>(
        std::max<long long>(1, static_cast<long long>(per_sm) * std::max(sms, 1) / std::max(p.hkv, 1)), p.num_seqs);
    const long long target = std::min<long long>(fit, kDecodeMaxItems);
    int max_tiles = 2;
    for (int b = 0; b < p.num_seqs; ++b) max_tiles = std::max(max_tiles, tiles[b]);
    int lo = static_cast<int>(std::max<long long>(2, (total + target - 1) / target)), hi = std::max(lo, max_tiles);
    while (lo < hi) {
      const int mid = lo + (hi - lo) / 2;
      if (items_at(mid) <= target)
        hi = mid;
      else
        lo = mid + 1;
    }
    tps = lo;
  }
  pl.tiles_per_split = tps;
  pl.items.clear();
  for (int b = 0; b < p.num_seqs; ++b) {
    const int chunks = (tiles[b] + tps - 1) / tps;
    for (int c = 0; c < chunks; ++c) pl.items.push_back(static_cast<uint32_t>(b) | (static_cast<uint32_t>(c) << 16));
  }
  const int R = (p.hq / p.hkv) * n;
  pl.acc_bytes = pl.items.size() * p.hkv * static_cast<size_t>(R) * D * 4;
  pl.ml_bytes = pl.items.size() * p.hkv * static_cast<size_t>(R) * 16;
  pl.counter_bytes = static_cast<size_t>(p.num_seqs) * p.hkv * 4;
  return pl;
}

namespace {

template <int CAP>
cudaError_t launch_decode_cap(const Problem& pr, int n, const DecodeArgs& a, const DecodePlan& pl, int* status,
                              cudaStream_t stream) {
  thread_local DecK<CAP> k;
  if (!fill_params(k, pr, n, a, pl, status)) return cudaErrorInvalidValue;
  const dim3 grid(k.n_items, pr.hkv);
  cudaError_t e = prof_begin(g_prof_dec, stream);
  if (e != cudaSuccess) return e;
  if (!pl.tensor_core) {
    if ((e = cudaFuncSetAttribute(decode_split_kernel<1, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  SMEM_DYN)) != cudaSuccess)
      return e;
    decode_split_kernel<1, CAP><<<grid, NTHR, SMEM_DYN, stream>>>(k);
    e = cudaGetLastError();
  } else {
    e = launch_decode_tc(k, grid, stream);
  }
  if (e != cudaSuccess) return e;
  return prof_end(g_prof_dec, stream);
}

}  // namespace

cudaError_t launch_decode(const Problem& pr, int n, const DecodeArgs& a, const DecodePlan& pl, int* status,
                          cudaStream_t stream) {
  if (pr.num_seqs == 0) return cudaSuccess;
  if (pl.items.size() > static_cast<size_t>(kDecodeMaxItems)) return cudaErrorInvalidValue;
  return pl.items.size() <= static_cast<size_t>(kSmallItems)
             ? launch_decode_cap<kSmallItems>(pr, n, a, pl, status, stream)
             : launch_decode_cap<kDecodeMaxItems>(pr, n, a, pl, status, stream);
}

}  // namespace sa
