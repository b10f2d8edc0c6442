// Pieces shared by the two decode kernels (decode.cu: warp-level MMAs for a
// single 16-row block; decode_tc.cu: tcgen05 for wider row blocks): the
// kernel parameter block, the key tiles a decode row block sees, and the
// merge of the split-KV partials with the sink applied once.
//
// Rows r of one (sequence, kv head): r = i * group + j is query position
// L - n + i of query head g * group + j.  Each CTA handles one chunk of the
// key tiles of one (sequence, kv head) and writes a partial (unnormalised O
// [R, 64], and per row the reference m in log2 units of the scaled score and
// the sum l relative to it); the last CTA of a (sequence, kv head) to finish
// merges the partials of each row,
//     m = max m_i,  l = sum 2^{m_i - m} l_i,  O = sum 2^{m_i - m} O_i / l_o,
// and only then applies the sink: lse = ln2 (m + log2 l), alpha =
// sigmoid(lse - s_h), O <- alpha O (summary page, sink scaling of the output
// by sigma(l - s_h)).  A partial carries two sums: l_o, the one O is
// normalised by (the sum of exactly the weights its numerator used: the
// bf16-rounded P where the tensor core forms it), and l, the fp32 sum of the
// unrounded exponentials that lse is taken from; the warp-MMA kernel writes
// its one fp32 sum into both.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

#include <algorithm>

#include <cuda.h>

namespace sa {
namespace dec {

constexpr int D = kHeadDim;
constexpr int BN = 128;           // keys per tile
constexpr int TILE = BN * D * 2;  // 16 KB

// The work list's capacity is a template parameter: a short list keeps the
// kernel parameter block small (a 16 KB block costs ~1.3 us more per launch
// than a small one, a few per cent of a short decode step).
constexpr int kSmallItems = 256;

template <int CAP>
struct DecK {
  CUtensorMap tm_k, tm_v;
  const __nv_bfloat16* q;  // [B * n, Hq, 64]
  const float* sink;
  __nv_bfloat16* o;        // [B * n, Hq, 64]
  float* lse;              // [Hq, B * n]
  int* counters;           // [B * Hkv] chunks finished; zero between calls
  float* ws_acc;           // [items * Hkv, R, 64] unnormalised O of each partial
  float4* ws_ml;           // [items * Hkv, R]: (m in log2 units of the scaled score, l_o, l, 0)
  const int32_t* cu;       // key/value offsets or nullptr (uniform length kv_len)
  int* status;
  int kv_len;
  int n, hq, hkv, group, R;
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

// The chunk [j0, j1) of key tiles that item `item` of kv head g covers.
struct Chunk {
  int b, split, nsplit, j0, j1;
  SeqSpan sp;
  KeyTiles kt;
};

template <int CAP>
SA_DEV Chunk chunk_of(const DecK<CAP>& p, int item_idx) {
  Chunk c;
  const uint32_t item = p.items[item_idx];
  c.b = static_cast<int>(item & 0xFFFFu);
  c.split = static_cast<int>(item >> 16);
  c.sp = seq_span(p.cu, p.kv_len, c.b);
  c.kt = key_tiles(c.sp.len, p.n, p.mask);
  c.nsplit = (c.kt.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  c.j0 = c.split * c.kt.n_tiles / c.nsplit;
  c.j1 = (c.split + 1) * c.kt.n_tiles / c.nsplit;
  return c;
}

// Counts this CTA's partial (already written by the calling threads) and
// reports whether it was the last of its (sequence, kv head).  Every thread
// of the CTA calls it.
template <int CAP>
SA_DEV bool count_partial(const DecK<CAP>& p, const Chunk& c, int g, int* is_last_sh) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *is_last_sh = atomicAdd(p.counters + c.b * p.hkv + g, 1) == c.nsplit - 1;
  __syncthreads();
  const bool last = *is_last_sh != 0;
  if (last) __threadfence();
  return last;
}

// The sink, applied once to a finished row r of (sequence c.b, kv head g):
// returns the factor O is multiplied by (alpha / l_o) and sets lse from the
// reference M (log2 units) and the fp32 sum l.
template <int CAP>
SA_DEV float row_scale(const DecK<CAP>& p, const Chunk& c, int g, int r, float M, float l_o, float l, float& lse) {
  const int i = r / p.group, h = g * p.group + (r - i * p.group);
  lse = (l > 0.f) ? (M + __log2f(l)) * kLn2 : -INFINITY;
  const float alpha = 1.f / (1.f + ex2((__ldg(p.sink + h) - lse) * kLog2e));
  return (l_o > 0.f) ? alpha / l_o : 0.f;
}

// Output element pair (2 d2, 2 d2 + 1) and lse of row r.
template <int CAP>
SA_DEV void store_pair(const DecK<CAP>& p, const Chunk& c, int g, int r, int d2, float x, float y) {
  const int i = r / p.group, h = g * p.group + (r - i * p.group), bn = c.b * p.n + i;
  reinterpret_cast<uint32_t*>(p.o + (static_cast<size_t>(bn) * p.hq + h) * D)[d2] = pack_bf16(x, y);
}
template <int CAP>
SA_DEV void store_lse(const DecK<CAP>& p, const Chunk& c, int g, int r, float lse) {
  const int i = r / p.group, h = g * p.group + (r - i * p.group), bn = c.b * p.n + i;
  p.lse[static_cast<size_t>(h) * p.num_seqs * p.n + bn] = lse;
}

// Merge of the partials of (sequence c.b, kv head g) by the CTA's NT threads
// (all of them call it).  The partials of chunk s are O at ws_acc +
// (part0 + s Hkv) R 64 and (m, l_o, l) at ws_ml + (part0 + s Hkv) R; they
// are staged in batches through `stage_bytes` of idle shared memory at
// `smem` by bulk copies, then merged from shared memory with an online
// rescale per (row, dim pair) unit.  UP units per thread cover R x 32 dim
// pairs.  Clears the counter for the next call.
template <int UP, int NT, int CAP>
SA_DEV void merge_partials(const DecK<CAP>& p, const Chunk& c, int g, int item_idx, uint8_t* smem, uint32_t stage_bytes,
                           uint32_t merge_bar, const tc::Abort& ab) {
  using namespace tc;
  const int tid = threadIdx.x;
  const uint32_t sb = smem_u32(smem);
  const size_t part0 = static_cast<size_t>(item_idx - c.split) * p.hkv + g;
  const uint32_t blk_acc = static_cast<uint32_t>(p.R) * D * 4, blk_ml = static_cast<uint32_t>(p.R) * 16;
  const int per_batch = max(1, static_cast<int>(stage_bytes / (blk_acc + blk_ml)));
  float2 acc[UP];
  float Mu[UP], lo[UP], lu[UP];
#pragma unroll
  for (int k = 0; k < UP; ++k) {
    acc[k] = make_float2(0.f, 0.f);
    Mu[k] = -INFINITY;
    lo[k] = 0.f;
    lu[k] = 0.f;
  }
  const float* stg_acc = reinterpret_cast<const float*>(smem);
  const float4* ml_s = reinterpret_cast<const float4*>(smem + per_batch * blk_acc);
  if (tid == 0) fence_proxy_async_global();  // the partials were written through the generic proxy
  for (int c0 = 0, batch = 0; c0 < c.nsplit; c0 += per_batch, ++batch) {
    const int cnt = min(per_batch, c.nsplit - c0);
    if (tid == 0) {
      mbar_expect_tx(merge_bar, cnt * (blk_acc + blk_ml));
      for (int s = 0; s < cnt; ++s) {
        const size_t pc = part0 + static_cast<size_t>(c0 + s) * p.hkv;
        bulk_load(sb + s * blk_acc, p.ws_acc + pc * p.R * D, blk_acc, merge_bar);
        bulk_load(sb + per_batch * blk_acc + s * blk_ml, p.ws_ml + pc * p.R, blk_ml, merge_bar);
      }
    }
    const bool ok = mbar_wait(merge_bar, batch & 1, ab);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {  // let the copies still in flight land before the CTA leaves
        const long long t0 = clock64();
        while (!mbar_try_wait(merge_bar, batch & 1) && clock64() - t0 < kTimeoutCycles) {
        }
      }
      return;
    }
#pragma unroll
    for (int k = 0; k < UP; ++k) {
      const int u = tid + NT * k, r = u >> 5, d2 = u & 31;
      if (r >= p.R) continue;
      for (int s = 0; s < cnt; ++s) {
        const float4 mv = ml_s[s * p.R + r];
        if (mv.x == -INFINITY) continue;
        if (mv.x > Mu[k]) {
          const float sc = (Mu[k] == -INFINITY) ? 0.f : ex2(Mu[k] - mv.x);
          acc[k].x *= sc;
          acc[k].y *= sc;
          lo[k] *= sc;
          lu[k] *= sc;
          Mu[k] = mv.x;
        }
        const float w = ex2(mv.x - Mu[k]);
        const float2 a = reinterpret_cast<const float2*>(stg_acc + (static_cast<size_t>(s) * p.R + r) * D)[d2];
        acc[k].x += w * a.x;
        acc[k].y += w * a.y;
        lo[k] += w * mv.y;
        lu[k] += w * mv.z;
      }
    }
    __syncthreads();  // the next batch overwrites the staging buffers
  }
#pragma unroll
  for (int k = 0; k < UP; ++k) {
    const int u = tid + NT * k, r = u >> 5, d2 = u & 31;
    if (r >= p.R) continue;
    float lse;
    const float fac = row_scale(p, c, g, r, Mu[k], lo[k], lu[k], lse);
    store_pair(p, c, g, r, d2, acc[k].x * fac, acc[k].y * fac);
    if (d2 == 0) store_lse(p, c, g, r, lse);
  }
  if (tid == 0) p.counters[c.b * p.hkv + g] = 0;  // every chunk of this call has counted
}

// Host side: the parameter block of one launch.
template <int CAP>
bool fill_params(DecK<CAP>& k, const Problem& pr, int n, const DecodeArgs& a, const DecodePlan& pl, int* status) {
  if (!make_rows_map(&k.tm_k, a.k, pr.total_tokens, pr.hkv, BN) ||
      !make_rows_map(&k.tm_v, a.v, pr.total_tokens, pr.hkv, BN))
    return false;
  const int group = pr.hq / pr.hkv, R = group * n;
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.sink = a.sink;
  k.o = static_cast<__nv_bfloat16*>(a.o);
  k.lse = a.lse;
  k.counters = a.counters;
  k.num_seqs = pr.num_seqs;
  k.ws_acc = a.ws_acc;
  k.ws_ml = reinterpret_cast<float4*>(a.ws_ml);
  k.cu = pr.cu;
  k.status = status;
  k.kv_len = pr.seqlen;
  k.n = n;
  k.hq = pr.hq;
  k.hkv = pr.hkv;
  k.group = group;
  k.R = R;
  k.mask = MaskParams{pr.window, pr.prefix, pr.causal};
  k.scale_log2 = pr.scale * kLog2e;
  k.tiles_per_split = pl.tiles_per_split;
  k.n_items = static_cast<int>(pl.items.size());
  std::copy(pl.items.begin(), pl.items.end(), k.items);
  return true;
}

// The tensor-core kernel for 16 < R <= 128 (decode_tc.cu), one CTA per
// (item, kv head) of `grid`.
template <int CAP>
cudaError_t launch_decode_tc(const DecK<CAP>& k, dim3 grid, cudaStream_t stream);

}  // namespace dec
}  // namespace sa
