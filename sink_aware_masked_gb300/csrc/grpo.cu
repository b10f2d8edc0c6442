// GRPO token loss and its gradient with respect to the policy's token
// log-probabilities, fused into two passes over the tokens.
//
// "Efficient Reinforcement Learning for Long-Horizon Tool-Use Agentic Tasks"
// (SinkFlex-RL), zh page, "Policy update", equations (3)-(7):
//   A_i    = (R_i - mu(R_1..G)) / (sigma(R_1..G) + eps_A)       (3)
//   rho    = exp(logp - logp_old)                                  (4)
//   J      = min(rho A_i, clip(rho, 1 - eps_c, 1 + eps_c) A_i)     (5), (6)
//   L      = -(1 / sum_i T_i) sum J + beta KL                      (7)
// with sigma the population standard deviation of the group's rewards, T_i
// the optimised tokens of rollout i (mask != 0) and the KL term estimated per
// optimised token by k3 = exp(r) - r - 1, r = logp_ref - logp, averaged like
// the policy term.  dL/dlogp = (-dJ + beta (1 - e^r)) / N on optimised
// tokens, dJ = rho A unless the clipped branch is strictly smaller (then 0).
//
// A memory-bound stream (13 bytes read and 4 written per token) over chunks
// of 2048 tokens, each thread taking two 16-byte vectors of a chunk; both
// passes run a persistent grid that strides over the chunks.  Pass 1 counts
// the optimised tokens (one partial per CTA) and computes the advantages
// (one thread per rollout).  Pass 2 needs N = sum_i T_i before it can scale
// the gradient, so every CTA sums the pass-1 counts itself and stages the
// rollout offsets and advantages in shared memory (8 bytes per rollout),
// both while its first chunk's token loads are in flight; it finds each
// vector's rollout by binary search there (the streaming loads would evict
// the offsets from L1), writes dL/dlogp and accumulates partial sums; the
// last CTA to finish reduces the partials in a fixed order (deterministic).
// (Measured and not kept: staging the chunks through a shared-memory ring by
// bulk copies, and per-chunk rollout lists; neither was faster — the pass
// is bound by its per-token instruction latency, not by bytes in flight.)
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace sa {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 2;                          // 16-byte vectors per thread and chunk
constexpr int kTokPerCta = kThreads * kVec * 4;  // 2048 tokens per chunk
constexpr int kRewardStage = 2048;               // rewards of one pass-1 CTA's groups staged up to this
constexpr int kStageRollouts = 6000;             // pass 2 stages offsets and advantages up to this many rollouts
constexpr int kLossCtasPerSm = 4;
constexpr int kCtasPerSm = 4;

struct GrpoK {
  const float* logp;
  const float* logp_old;
  const float* logp_ref;  // nullptr when beta == 0
  const uint8_t* mask;
  const float* rewards;
  const int32_t* cu;
  float* stats;    // [4]: loss, policy term, KL term (unscaled), clipped fraction
  float* dlogp;
  float* adv_out;  // [R] or nullptr
  int* counts;     // workspace [P]: optimised tokens per pass-1 CTA
  float* adv;      // workspace [R]
  float4* part;    // workspace [grid]: sum J, sum k3, clipped count
  unsigned* done;  // workspace: pass-2 CTAs finished
  int R, G, T, chunks, grid, grid2;
  float clip_eps, adv_eps, beta;
};

template <typename T>
SA_DEV T block_sum(T v, T* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  T s = T(0);
  if (threadIdx.x < 32) {
    s = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : T(0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  return s;  // valid in thread 0
}

// Number of nonzero bytes of w.
SA_DEV int nonzero_bytes(uint32_t w) {
  const uint32_t x = ((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w;  // bit 7 of a byte set iff the byte is nonzero
  return __popc(x & 0x80808080u);
}

__global__ void __launch_bounds__(kThreads) grpo_prep_kernel(const GrpoK p) {
  __shared__ int red[kThreads / 32];
  __shared__ float rew_s[kRewardStage];
  const int tid = threadIdx.x;
  // Optimised tokens of the chunks this CTA strides over, 16 per load (the
  // first 128 threads of the CTA cover a 2048-token chunk).
  int n = 0;
  for (int c = blockIdx.x; c < p.chunks && tid < kTokPerCta / 16; c += gridDim.x) {
    const long long t = static_cast<long long>(c) * kTokPerCta + 16LL * tid;
    if (t + 16 <= p.T) {
      const uint4 m = __ldg(reinterpret_cast<const uint4*>(p.mask + t));
      n += nonzero_bytes(m.x) + nonzero_bytes(m.y) + nonzero_bytes(m.z) + nonzero_bytes(m.w);
    } else {
      for (long long u = t; u < p.T && u < t + 16; ++u) n += __ldg(p.mask + u) != 0;
    }
  }
  // Equation (3) for rollouts i = 256 b + tid; the rewards of the block's
  // groups are staged in shared memory by one coalesced load per thread.
  for (int b = blockIdx.x; b * kThreads < p.R; b += gridDim.x) {
    const int r_lo = min(p.R, (b * kThreads / p.G) * p.G);
    const int r_hi = min(p.R, ((min(p.R, b * kThreads + kThreads) + p.G - 1) / p.G) * p.G);
    const bool staged = r_hi - r_lo <= kRewardStage;
    __syncthreads();
    if (staged)
      for (int j = r_lo + tid; j < r_hi; j += kThreads) rew_s[j - r_lo] = __ldg(p.rewards + j);
    __syncthreads();
    const int i = b * kThreads + tid;
    if (i < p.R) {
      // In fp32: FP64 issues at a small fraction of the FP32 rate on this part,
      // and a group's mean and spread need no more than fp32 keeps.
      const int g0 = (i / p.G) * p.G;
      auto rew = [&](int j) { return staged ? rew_s[j - r_lo] : __ldg(p.rewards + j); };
      float mu = 0.f, var = 0.f;
      for (int j = g0; j < g0 + p.G; ++j) mu += rew(j);
      mu /= static_cast<float>(p.G);
      for (int j = g0; j < g0 + p.G; ++j) {
        const float d = rew(j) - mu;
        var += d * d;
      }
      const float a = (rew(i) - mu) / (sqrtf(var / static_cast<float>(p.G)) + p.adv_eps);
      p.adv[i] = a;
      if (p.adv_out) p.adv_out[i] = a;
    }
  }
  n = block_sum(n, red);
  if (tid == 0) {
    p.counts[blockIdx.x] = n;
    if (blockIdx.x == 0) *p.done = 0u;
  }
}

__global__ void __launch_bounds__(kThreads, kLossCtasPerSm) grpo_loss_kernel(const GrpoK p) {
  __shared__ long long red_ll[kThreads / 32];
  __shared__ float3 red_f3[kThreads / 32];
  __shared__ double red_d[kThreads / 32];
  __shared__ float sh_inv_n;
  __shared__ bool is_last;
  extern __shared__ int dyn_s[];  // [R + 1] offsets, then [R] advantages (when staged)
  const int tid = threadIdx.x;
  const bool staged = p.R <= kStageRollouts;
  const int* cu_s = dyn_s;
  const float* adv_s = reinterpret_cast<const float*>(dyn_s + p.R + 1);
  long long n = 0;
  float inv_n = 0.f;
  const float beta = p.beta;
  const float lo = 1.f - p.clip_eps, hi = 1.f + p.clip_eps;
  const int nvec = p.T / 4;
  auto cu_at = [&](int j) { return staged ? cu_s[j] : __ldg(p.cu + j); };
  auto adv_at = [&](int i) { return staged ? adv_s[i] : __ldg(p.adv + i); };
  // Rollout of token t: the last i with cu[i] <= t (skips empty rollouts).
  auto rollout = [&](int t, int a, int b) {  // cu[a] <= t < cu[b]
    while (b - a > 1) {
      const int mid = (a + b) >> 1;
      if (cu_at(mid) <= t) a = mid; else b = mid;
    }
    return a;
  };
  float sj = 0.f, sk = 0.f, sc = 0.f;
  auto token = [&](float x, float xo, float xr, bool m, float A) -> float {
    const float rho = expf(x - xo);
    const float J = fminf(rho * A, fminf(fmaxf(rho, lo), hi) * A);
    const bool clipped = (A > 0.f && rho > hi) || (A < 0.f && rho < lo);
    float g = clipped ? 0.f : -rho * A;
    float k3 = 0.f;
    if (beta != 0.f) {
      const float r = xr - x;
      const float e = expf(r);
      k3 = (e - 1.f) - r;
      g += beta * (1.f - e);
    }
    if (m) {
      sj += J;
      sk += k3;
      sc += clipped ? 1.f : 0.f;
    }
    return m ? g * inv_n : 0.f;
  };
  for (int c = blockIdx.x; c < p.chunks; c += gridDim.x) {
    // The chunk's token loads first.
    float4 lp[kVec], old[kVec], lr[kVec];
    uchar4 mk[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = c * (kTokPerCta / 4) + tid + kThreads * k;
      if (v < nvec) {
        lp[k] = __ldg(reinterpret_cast<const float4*>(p.logp) + v);
        old[k] = __ldg(reinterpret_cast<const float4*>(p.logp_old) + v);
        lr[k] = beta != 0.f ? __ldg(reinterpret_cast<const float4*>(p.logp_ref) + v) : make_float4(0.f, 0.f, 0.f, 0.f);
        mk[k] = __ldg(reinterpret_cast<const uchar4*>(p.mask) + v);
      }
    }
    if (c == static_cast<int>(blockIdx.x)) {
      // N = sum of the pass-1 counts (every CTA sums them itself) and the
      // staged offsets and advantages, while the first chunk's loads are in flight.
      if (staged) {
        for (int j = tid; j <= p.R; j += kThreads) dyn_s[j] = __ldg(p.cu + j);
        for (int j = tid; j < p.R; j += kThreads) reinterpret_cast<float*>(dyn_s + p.R + 1)[j] = __ldg(p.adv + j);
      }
      for (int j = tid; j < p.grid; j += kThreads) n += __ldcg(p.counts + j);
      n = block_sum(n, red_ll);
      if (tid == 0) sh_inv_n = n > 0 ? static_cast<float>(1.0 / static_cast<double>(n)) : 0.f;
      __syncthreads();
      inv_n = sh_inv_n;
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = c * (kTokPerCta / 4) + tid + kThreads * k;
      if (v < nvec) {
        const int t = 4 * v;
        const int i0 = rollout(t, 0, p.R);
        const float a0 = adv_at(i0);
        // The four tokens usually share the rollout; otherwise look each up.
        const bool same = t + 3 < cu_at(i0 + 1);
        float4 d;
        d.x = token(lp[k].x, old[k].x, lr[k].x, mk[k].x != 0, a0);
        d.y = token(lp[k].y, old[k].y, lr[k].y, mk[k].y != 0, same ? a0 : adv_at(rollout(t + 1, i0, p.R)));
        d.z = token(lp[k].z, old[k].z, lr[k].z, mk[k].z != 0, same ? a0 : adv_at(rollout(t + 2, i0, p.R)));
        d.w = token(lp[k].w, old[k].w, lr[k].w, mk[k].w != 0, same ? a0 : adv_at(rollout(t + 3, i0, p.R)));
        reinterpret_cast<float4*>(p.dlogp)[v] = d;
      }
    }
    // The last T % 4 tokens belong to the chunk that would hold vector nvec.
    if (tid == 0 && nvec / (kTokPerCta / 4) == c)
      for (int t = 4 * nvec; t < p.T; ++t)
        p.dlogp[t] = token(__ldg(p.logp + t), __ldg(p.logp_old + t), beta != 0.f ? __ldg(p.logp_ref + t) : 0.f,
                           __ldg(p.mask + t) != 0, adv_at(rollout(t, 0, p.R)));
  }
  // One reduction of the three partial sums.
  float3 s3 = make_float3(sj, sk, sc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s3.x += __shfl_xor_sync(0xffffffffu, s3.x, o);
    s3.y += __shfl_xor_sync(0xffffffffu, s3.y, o);
    s3.z += __shfl_xor_sync(0xffffffffu, s3.z, o);
  }
  __syncthreads();
  if ((tid & 31) == 0) red_f3[tid >> 5] = s3;
  __syncthreads();
  if (tid == 0) {
    float3 t3 = make_float3(0.f, 0.f, 0.f);
    for (int w = 0; w < kThreads / 32; ++w) {
      t3.x += red_f3[w].x;
      t3.y += red_f3[w].y;
      t3.z += red_f3[w].z;
    }
    p.part[blockIdx.x] = make_float4(t3.x, t3.y, t3.z, 0.f);
    __threadfence();
    is_last = atomicAdd(p.done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // Every thread sums a fixed strided subset of the partials, then a fixed
  // shuffle tree: the result does not depend on which CTA finished last.
  double dj = 0.0, dk = 0.0, dc = 0.0;
  for (int j = tid; j < static_cast<int>(gridDim.x); j += kThreads) {
    const float4 v = __ldcg(p.part + j);
    dj += v.x;
    dk += v.y;
    dc += v.z;
  }
  dj = block_sum(dj, red_d);
  dk = block_sum(dk, red_d);
  dc = block_sum(dc, red_d);
  if (tid == 0) {
    const double inv = n > 0 ? 1.0 / static_cast<double>(n) : 0.0;
    const double policy = -dj * inv, kl = dk * inv;
    p.stats[0] = static_cast<float>(policy + static_cast<double>(beta) * kl);
    p.stats[1] = static_cast<float>(policy);
    p.stats[2] = static_cast<float>(kl);
    p.stats[3] = static_cast<float>(dc * inv);
  }
}

int num_chunks(int T) { return std::max(1, (T + kTokPerCta - 1) / kTokPerCta); }

int grid_ctas(int T) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 0;
    if (sms <= 0) sms = 152;
  }
  return std::min(num_chunks(T), kCtasPerSm * sms);
}

int loss_ctas(int T) {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    sms = 152;
  return std::min(num_chunks(T), kLossCtasPerSm * sms);
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t grpo_workspace_bytes(int num_rollouts, int total_tokens) {
  const size_t G = static_cast<size_t>(grid_ctas(total_tokens)), G2 = static_cast<size_t>(loss_ctas(total_tokens));
  return a256(G * 4) + a256(static_cast<size_t>(num_rollouts) * 4) + a256(G2 * 16) + 256;
}

cudaError_t launch_grpo(const GrpoArgs& a, cudaStream_t stream) {
  if (a.num_rollouts == 0) return cudaSuccess;
  const int grid = grid_ctas(a.total_tokens), chunks = num_chunks(a.total_tokens);
  const int grid2 = loss_ctas(a.total_tokens);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  GrpoK k;
  k.logp = a.logp;
  k.logp_old = a.logp_old;
  k.logp_ref = a.kl_beta != 0.f ? a.logp_ref : nullptr;
  k.mask = a.mask;
  k.rewards = a.rewards;
  k.cu = a.cu_tokens;
  k.stats = a.stats;
  k.dlogp = a.dlogp;
  k.adv_out = a.advantages;
  size_t off = 0;
  k.counts = reinterpret_cast<int*>(ws + off);
  off += a256(static_cast<size_t>(grid) * 4);
  k.adv = reinterpret_cast<float*>(ws + off);
  off += a256(static_cast<size_t>(a.num_rollouts) * 4);
  k.part = reinterpret_cast<float4*>(ws + off);
  off += a256(static_cast<size_t>(grid2) * 16);
  k.done = reinterpret_cast<unsigned*>(ws + off);
  k.R = a.num_rollouts;
  k.G = a.group_size;
  k.T = a.total_tokens;
  k.chunks = chunks;
  k.grid = grid;
  k.grid2 = grid2;
  k.clip_eps = a.clip_eps;
  k.adv_eps = a.adv_eps;
  k.beta = a.kl_beta;
  grpo_prep_kernel<<<grid, kThreads, 0, stream>>>(k);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t dyn = a.num_rollouts <= kStageRollouts ? (2 * static_cast<size_t>(a.num_rollouts) + 1) * 4 : 0;
  grpo_loss_kernel<<<grid2, kThreads, dyn, stream>>>(k);
  return cudaGetLastError();
}

}  // namespace sa
