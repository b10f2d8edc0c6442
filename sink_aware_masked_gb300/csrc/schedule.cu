// Host-side work lists for the forward and backward kernels.
//
// Work items are sorted longest-first (LPT) and handed to the kernels in
// their parameter blocks, so CTAs are dispatched in order of decreasing
// cost, which bounds the tail when item costs vary (causal masks, packed
// sequences of different lengths, always-visible prefix tiles).  Lists are
// built from the host copy of the sequence offsets: no device-to-host sync.
//
// Forward item  : (sequence, 128-row query tile); cost = key tiles visited.
// Backward item : (sequence, 128-key tile, query chunk); cost = query tiles.
//   A key tile whose query range exceeds `qchunk` query tiles is split into
//   chunks of qchunk; qchunk is chosen so that no item exceeds about half of
//   one SM's average share of the work, and never below 4 (short chunks
//   waste the pipeline fill).  Split tiles accumulate dK/dV in fp32.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <vector>

#include "internal.h"

namespace sa {
namespace {

constexpr int TILE_ROWS = 128;
constexpr int kMaxDevices = 256;
constexpr int kFallbackSms = 152;  // a GB300, when no device answers

struct Span {
  int start, len;
};

std::vector<Span> spans(const Problem& p) {
  std::vector<Span> s(p.num_seqs);
  for (int b = 0; b < p.num_seqs; ++b) {
    if (p.cu_host != nullptr)
      s[b] = {p.cu_host[b], p.cu_host[b + 1] - p.cu_host[b]};
    else
      s[b] = {b * p.seqlen, p.seqlen};
  }
  return s;
}

// Same arithmetic as key_range() / query_range() in common.cuh.
int fwd_tiles_visited(const Problem& p, int q0, int len) {
  const int q1 = std::min(q0 + TILE_ROWS, len) - 1;
  const int hi = p.causal ? std::min(q1, len - 1) : len - 1;
  const int lo = (p.window < 0) ? 0 : std::max(0, q0 - p.window);
  const int pre_end = std::max(0, std::min(std::min(p.prefix, lo), hi + 1));
  const int lo_t = lo / TILE_ROWS, hi_t = hi / TILE_ROWS;
  const int n_pre = std::min((pre_end + TILE_ROWS - 1) / TILE_ROWS, lo_t);
  return n_pre + (hi_t - lo_t + 1);
}

int bwd_query_tiles(const Problem& p, int k0, int len) {
  const int k1 = std::min(k0 + TILE_ROWS, len) - 1;
  const int lo = p.causal ? k0 : 0;
  const int hi = (p.prefix > k0 || p.window < 0) ? len - 1 : std::min(len - 1, k1 + p.window);
  return hi / TILE_ROWS - lo / TILE_ROWS + 1;
}

}  // namespace

int device_sms() {
  static std::atomic<int> cache[kMaxDevices];  // zero until the first query of a device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kFallbackSms;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return kFallbackSms;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

std::vector<uint32_t> fwd_work_list(const Problem& p) {
  struct It {
    int cost;
    uint32_t code;
  };
  std::vector<It> items;
  const auto s = spans(p);
  for (int b = 0; b < p.num_seqs; ++b)
    for (int q0 = 0; q0 < s[b].len; q0 += TILE_ROWS)
      items.push_back({fwd_tiles_visited(p, q0, s[b].len),
                       static_cast<uint32_t>(b) | (static_cast<uint32_t>(q0 / TILE_ROWS) << 16)});
  std::stable_sort(items.begin(), items.end(), [](const It& a, const It& c) { return a.cost > c.cost; });
  std::vector<uint32_t> out(items.size());
  for (size_t i = 0; i < items.size(); ++i) out[i] = items[i].code;
  return out;
}

long long bwd_query_tiles_total(const Problem& p) {
  const auto s = spans(p);
  long long total = 0;
  for (int b = 0; b < p.num_seqs; ++b)
    for (int k0 = 0; k0 < s[b].len; k0 += TILE_ROWS) total += bwd_query_tiles(p, k0, s[b].len);
  return total;
}

int bwd_qchunk(const Problem& p) {
  const auto s = spans(p);
  long long total = 0;
  int longest = 0;
  for (int b = 0; b < p.num_seqs; ++b)
    for (int k0 = 0; k0 < s[b].len; k0 += TILE_ROWS) {
      const int nq = bwd_query_tiles(p, k0, s[b].len);
      total += nq;
      longest = std::max(longest, nq);
    }
  // Per-SM average of query tiles (x kv heads, every CTA covers one kv head).
  const int sms = device_sms();
  const long long per_sm = (total * p.hkv + sms - 1) / sms;
  const int cap = static_cast<int>(std::max<long long>(4, per_sm / 2));
  return std::max(1, std::min(cap, longest));
}

std::vector<BwdItem> bwd_work_list(const Problem& p, int qchunk) {
  struct It {
    int cost;
    BwdItem item;
  };
  std::vector<It> items;
  const auto s = spans(p);
  uint32_t slot = 0;  // chunks of split tiles, in tile then chunk order
  for (int b = 0; b < p.num_seqs; ++b)
    for (int k0 = 0; k0 < s[b].len; k0 += TILE_ROWS) {
      const int nq = bwd_query_tiles(p, k0, s[b].len);
      const int chunks = (nq + qchunk - 1) / qchunk;
      for (int c = 0; c < chunks; ++c) {
        const int cost = std::min(qchunk, nq - c * qchunk);
        items.push_back({cost, BwdItem{static_cast<uint16_t>(b), static_cast<uint16_t>(k0 / TILE_ROWS),
                                       static_cast<uint16_t>(c), static_cast<uint16_t>(chunks),
                                       chunks > 1 ? slot++ : 0u}});
      }
    }
  std::stable_sort(items.begin(), items.end(), [](const It& a, const It& c) { return a.cost > c.cost; });
  std::vector<BwdItem> out(items.size());
  for (size_t i = 0; i < items.size(); ++i) out[i] = items[i].item;
  return out;
}

int bwd_split_slots(const std::vector<BwdItem>& items) {
  int n = 0;
  for (const auto& it : items) n += it.nchunks > 1 ? 1 : 0;
  return n;
}

}  // namespace sa
