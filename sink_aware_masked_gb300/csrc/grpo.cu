// GRPO token loss and its gradient with respect to the policy's token
// log-probabilities, in one cooperative kernel over the tokens.
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
// A memory-bound stream (13 bytes read and 4 written per token) in a
// persistent grid of co-resident CTAs (a cooperative launch), each CTA
// taking an equal contiguous range of 16-byte vectors (four tokens) in
// batches of two vectors per thread.  Only the final 1/N depends on all
// tokens, so everything else happens before one grid-wide barrier: every
// CTA stages the rollout offsets and computes the advantages in shared
// memory (while its first batch's loads are in flight), bounds the rollouts
// its range touches, finds each vector's rollout by binary lifting within
// them, writes the unscaled gradient (keeping its last batch's in
// registers), counts the optimised tokens and accumulates the partial sums.
// The barrier's arrival word carries the token counts, so the last CTA to
// arrive knows N and publishes it with the release; after the barrier each
// CTA only scales its gradients by 1/N (the earlier batches re-read from
// L2), and the last CTA reduces the partial sums in a fixed order
// (deterministic).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#include <algorithm>

namespace sa {
namespace {

using namespace tc;

constexpr int kThreads = 512;
constexpr int kStageVec = kThreads;              // 16-byte vectors (four tokens) per stage: one per thread
constexpr int kStageBytes = kStageVec * 52;      // logp, logp_old, logp_ref (16 B each) and mask (4 B) per vector
constexpr int kStages = 4;                       // shared-memory ring of stages
constexpr int kStageRollouts = 6000;             // offsets and advantages staged up to this many rollouts
constexpr int kRegStage = 2;                     // offsets and rewards per thread loaded ahead of the tokens
constexpr int kCtasPerSm = 2;
constexpr int kArriveBits = 20;                  // arrival count in the low bits of the barrier word

struct GrpoK {
  const float* logp;
  const float* logp_old;
  const float* logp_ref;  // nullptr when beta == 0
  const uint8_t* mask;
  const float* rewards;
  const int32_t* cu;
  float* stats;     // [4]: loss, policy term, KL term (unscaled), clipped fraction
  float* dlogp;
  float* adv_out;   // [R] or nullptr
  // workspace: [0] arrivals (low kArriveBits bits) plus optimised tokens
  // (high bits), zero between launches; [16] (another 128-byte line, which
  // the waiting CTAs poll) generation (high 32 bits) and the last N (low 32
  // bits).
  unsigned long long* sync;
  float4* part;     // workspace [grid]: sum J, sum k3, clipped count per CTA
  int* status;      // library status word
  int R, G, T, ngroups;
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

SA_DEV unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Acquire-release add at GPU scope (returns the old value).
SA_DEV unsigned long long atom_add_acq_rel_gpu(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], %2;\n" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
SA_DEV void st_release_gpu(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}

// Barrier over the whole (co-resident) grid that also sums one count per
// CTA.  Thread 0 of each CTA adds (count << kArriveBits) + 1 to the arrival
// word (release: its earlier writes, the CTA's partial sums among them, are
// visible to whoever acquires the word later); the CTA that completes it
// (acquire: it then sees every CTA's partial sums) clears the word for the
// next launch and publishes the next generation together with the total,
// which the others poll for.  Only thread 0's own writes are published this
// way, which is all the other CTAs read.  Returns the total in every thread
// (-1 when the wait ran out of time, after raising the status word) and
// whether this CTA arrived last.
SA_DEV long long grid_sync_sum(unsigned long long* sync, long long count, int* status, long long* sh_total,
                               bool* sh_last) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned gen = static_cast<unsigned>(ld_acquire_gpu(sync + 16) >> 32);
    const unsigned long long add = (static_cast<unsigned long long>(count) << kArriveBits) + 1ull;
    const unsigned long long old = atom_add_acq_rel_gpu(sync, add);
    long long total = -1;
    bool last = false;
    if ((old & ((1ull << kArriveBits) - 1ull)) == gridDim.x - 1) {
      total = static_cast<long long>((old + add) >> kArriveBits);
      last = true;
      *reinterpret_cast<volatile unsigned long long*>(sync) = 0ull;  // no CTA touches it again this launch
      st_release_gpu(sync + 16, (static_cast<unsigned long long>(gen + 1u) << 32) | static_cast<unsigned long long>(total));
    } else {
      const long long t0 = clock64();
      for (;;) {
        const unsigned long long w = ld_acquire_gpu(sync + 16);
        if (static_cast<unsigned>(w >> 32) != gen) {
          total = static_cast<long long>(w & 0xFFFFFFFFull);
          break;
        }
        if (clock64() - t0 > kTimeoutCycles) {
          atomicExch(status, kStatusTimeout);
          break;
        }
        __nanosleep(64);
      }
    }
    *sh_total = total;
    *sh_last = last;
  }
  __syncthreads();
  return *sh_total;
}

// Mean and population std + eps of the rewards of one group (shared or
// global memory), by one thread.
SA_DEV float2 group_stats(const float* rew, int g0, int G, float eps) {
  float mu = 0.f, var = 0.f;
  for (int j = g0; j < g0 + G; ++j) mu += rew[j];
  mu /= static_cast<float>(G);
  for (int j = g0; j < g0 + G; ++j) {
    const float d = rew[j] - mu;
    var += d * d;
  }
  return make_float2(mu, sqrtf(var / static_cast<float>(G)) + eps);
}

// Equation (3) for rollout i straight from the rewards (when the advantages
// are not staged).
SA_DEV float advantage_of(const float* rewards, int i, int G, float eps) {
  const float2 st = group_stats(rewards, (i / G) * G, G, eps);
  return (__ldg(rewards + i) - st.x) / st.y;
}

// The same by one warp (lanes stride over the group); valid in every lane.
SA_DEV float2 group_stats_warp(const float* rew, int g0, int G, float eps) {
  const int lane = threadIdx.x & 31;
  float mu = 0.f, var = 0.f;
  for (int j = g0 + lane; j < g0 + G; j += 32) mu += rew[j];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mu += __shfl_xor_sync(0xffffffffu, mu, o);
  mu /= static_cast<float>(G);
  for (int j = g0 + lane; j < g0 + G; j += 32) {
    const float d = rew[j] - mu;
    var += d * d;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) var += __shfl_xor_sync(0xffffffffu, var, o);
  return make_float2(mu, sqrtf(var / static_cast<float>(G)) + eps);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) grpo_kernel(const GrpoK p) {
  __shared__ uint64_t full[kStages];
  __shared__ int range_s[2];  // this CTA's vectors [v_lo, v_hi)
  __shared__ int abort_flag;
  __shared__ int red_i[kThreads / 32];
  __shared__ float3 red_f3[kThreads / 32];
  __shared__ long long sh_total;
  __shared__ bool sh_last;
  // Dynamic shared memory: kStages stages of kStageBytes (logp [512 x 16 B],
  // logp_old, logp_ref, mask [512 x 4 B]), then, when staged, [R + 1]
  // offsets and [R] advantages.
  extern __shared__ __align__(128) uint8_t dyn_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool staged = p.R <= kStageRollouts;
  int* cu_s = reinterpret_cast<int*>(dyn_raw + kStages * kStageBytes);
  float* adv_s = reinterpret_cast<float*>(cu_s + p.R + 1);
  const float beta = p.beta;
  const int nvec = p.T / 4;
  const int G = p.G, ngroups = p.ngroups;
  // This CTA's vectors [v_lo, v_hi): an equal share in units of 32 vectors
  // (128 tokens), in stages of kStageVec vectors.
  // (Thread 0 does the 64-bit divisions; the others read the bounds after
  // the first barrier.)
  int v_lo = 0, v_hi = 0;
  if (tid == 0) {
    const long long n32 = (nvec + 31) / 32;
    v_lo = static_cast<int>(static_cast<long long>(blockIdx.x) * n32 / gridDim.x) * 32;
    v_hi = min(nvec, static_cast<int>(static_cast<long long>(blockIdx.x + 1) * n32 / gridDim.x) * 32);
    range_s[0] = v_lo;
    range_s[1] = v_hi;
  }
  int nstage = (v_hi - v_lo + kStageVec - 1) / kStageVec;
  const uint32_t sbase = smem_u32(dyn_raw);
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
  }
  const Abort ab{&abort_flag, p.status};
  // Stage b: vectors [v0, v1) of the four arrays by bulk copies (16-byte
  // aligned: v0 is a multiple of 32); the mask of the last v1 - v0 mod 4
  // vectors, if any, is read from global memory instead.
  auto issue = [&](int b) {
    const int v0 = v_lo + b * kStageVec, nv = min(kStageVec, v_hi - v0), nvm = nv & ~3;
    const uint32_t bar = smem_u32(&full[b % kStages]);
    const uint32_t dst = sbase + (b % kStages) * kStageBytes;
    mbar_expect_tx(bar, nv * (beta != 0.f ? 48 : 32) + nvm * 4);
    bulk_load(dst, p.logp + 4LL * v0, nv * 16, bar);
    bulk_load(dst + kStageVec * 16, p.logp_old + 4LL * v0, nv * 16, bar);
    if (beta != 0.f) bulk_load(dst + kStageVec * 32, p.logp_ref + 4LL * v0, nv * 16, bar);
    if (nvm > 0) bulk_load(dst + kStageVec * 48, p.mask + 4LL * v0, nvm * 4, bar);
  };

  // Equation (3): every CTA stages all offsets and advantages (CTA 0 also
  // writes the advantages out): the rewards are loaded into the advantage
  // slots, and each group's statistics are computed and its slots
  // overwritten by the thread (G <= 32) or warp that owns the group.  The
  // first offsets and rewards are loaded before the token copies are issued
  // and stored after, so that the statistics are computed while the copies
  // are in flight.  Beyond kStageRollouts rollouts the grid writes the
  // advantages out and each token computes its own.
  int cu_r[kRegStage];
  float rw_r[kRegStage];
  if (staged) {
#pragma unroll
    for (int q = 0; q < kRegStage; ++q) {
      const int j = tid + kThreads * q;
      if (j <= p.R) cu_r[q] = __ldg(p.cu + j);
      if (j < p.R) rw_r[q] = __ldg(p.rewards + j);
    }
  }
  __syncthreads();  // the barriers are initialised, the range is published
  v_lo = range_s[0];
  v_hi = range_s[1];
  nstage = (v_hi - v_lo + kStageVec - 1) / kStageVec;
  if (tid == 0)
    for (int b = 0; b < min(nstage, kStages); ++b) issue(b);
  if (staged) {
    const bool write_adv = p.adv_out != nullptr && blockIdx.x == 0;
#pragma unroll
    for (int q = 0; q < kRegStage; ++q) {
      const int j = tid + kThreads * q;
      if (j <= p.R) cu_s[j] = cu_r[q];
      if (j < p.R) adv_s[j] = rw_r[q];
    }
    for (int j = tid + kThreads * kRegStage; j <= p.R; j += kThreads) {
      cu_s[j] = __ldg(p.cu + j);
      if (j < p.R) adv_s[j] = __ldg(p.rewards + j);
    }
    __syncthreads();
    if (G <= 32) {
      for (int grp = tid; grp < ngroups; grp += kThreads) {
        const int g0 = grp * G;
        const float2 st = group_stats(adv_s, g0, G, p.adv_eps);
        for (int j = g0; j < g0 + G; ++j) {
          const float a = (adv_s[j] - st.x) / st.y;
          adv_s[j] = a;
          if (write_adv) p.adv_out[j] = a;
        }
      }
    } else {
      for (int grp = warp; grp < ngroups; grp += kThreads / 32) {
        const int g0 = grp * G;
        const float2 st = group_stats_warp(adv_s, g0, G, p.adv_eps);  // every lane has read the group
        for (int j = g0 + lane; j < g0 + G; j += 32) {
          const float a = (adv_s[j] - st.x) / st.y;
          adv_s[j] = a;
          if (write_adv) p.adv_out[j] = a;
        }
      }
    }
    __syncthreads();
  } else if (p.adv_out != nullptr) {
    for (int grp = blockIdx.x * kThreads + tid; grp < ngroups; grp += gridDim.x * kThreads) {
      const int g0 = grp * G;
      const float2 st = group_stats(p.rewards, g0, G, p.adv_eps);
      for (int j = g0; j < g0 + G; ++j) p.adv_out[j] = (__ldg(p.rewards + j) - st.x) / st.y;
    }
  }
  auto cu_at = [&](int j) { return staged ? cu_s[j] : __ldg(p.cu + j); };
  auto adv_at = [&](int i) -> float { return staged ? adv_s[i] : advantage_of(p.rewards, i, G, p.adv_eps); };
  // Rollout of token t: the last i with cu[i] <= t (skips empty rollouts),
  // by binary lifting from a over steps top, top / 2, ..., 1 within [a, b]
  // (cu[a] <= t).  The rollouts of this CTA's range bound every search.
  auto lift = [&](int t, int a, int b, int top) {
    for (int step = top; step > 0; step >>= 1)
      if (a + step <= b && cu_at(a + step) <= t) a += step;
    return a;
  };
  auto pow2_floor = [](int x) { return x > 0 ? 1 << (31 - __clz(x)) : 0; };
  const int r_first = v_hi > v_lo ? lift(4 * v_lo, 0, p.R - 1, pow2_floor(p.R - 1)) : 0;
  const int r_last = v_hi > v_lo ? lift(4 * v_hi - 1, r_first, p.R - 1, pow2_floor(p.R - 1 - r_first)) : 0;
  const int top = pow2_floor(r_last - r_first);

  const float lo = 1.f - p.clip_eps, hi = 1.f + p.clip_eps;
  float sj = 0.f, sk = 0.f;
  int nclip = 0, n = 0;
  // One token: returns the unscaled gradient -dJ + beta dk3 (0 when not
  // optimised).  With s = sign(A) and sb = s * (the bound on A's side of the
  // clip), J = |A| min(s rho, sb) and the clip removes the gradient exactly
  // when s rho > sb (sb = +inf for A = 0).
  auto token = [&](float x, float xo, float xr, uint32_t mbyte, float absA, float s, float sb, float A) -> float {
    const float rho = expf(x - xo);
    const float sr = s * rho;
    const float J = absA * fminf(sr, sb);
    const bool clipped = sr > sb;
    float k3 = 0.f, gk = 0.f;  // k3 and beta dk3/dlogp = beta (1 - e^r)
    if (beta != 0.f) {
      const float r = xr - x;
      const float e = expf(r);
      k3 = (e - 1.f) - r;
      gk = fmaf(-beta, e, beta);
    }
    const float g = clipped ? gk : fmaf(-rho, A, gk);
    const bool m = mbyte != 0u;
    if (m) {
      sj += J;
      sk += k3;
      nclip += clipped;
    }
    return m ? g : 0.f;
  };
  auto side = [&](float A, float& absA, float& s, float& sb) {
    absA = fabsf(A);
    s = A > 0.f ? 1.f : -1.f;
    sb = A > 0.f ? hi : (A < 0.f ? -lo : __int_as_float(0x7f800000));
  };
  auto tokens4 = [&](int t, float4 x, float4 xo, float4 xr, uint32_t mw, int i0) -> float4 {
    const float A0 = adv_at(i0);
    float absA, s, sb;
    side(A0, absA, s, sb);
    float4 d;
    if (t + 3 < cu_at(i0 + 1)) {  // the usual case: all four in rollout i0
      d.x = token(x.x, xo.x, xr.x, mw & 0xFFu, absA, s, sb, A0);
      d.y = token(x.y, xo.y, xr.y, mw & 0xFF00u, absA, s, sb, A0);
      d.z = token(x.z, xo.z, xr.z, mw & 0xFF0000u, absA, s, sb, A0);
      d.w = token(x.w, xo.w, xr.w, mw & 0xFF000000u, absA, s, sb, A0);
    } else {  // a rollout ends inside the vector: one token at a time (kept small: rare)
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const float A = adv_at(lift(t + j, i0, r_last, top));
        side(A, absA, s, sb);
        const float xj = j == 0 ? x.x : j == 1 ? x.y : j == 2 ? x.z : x.w;
        const float xoj = j == 0 ? xo.x : j == 1 ? xo.y : j == 2 ? xo.z : xo.w;
        const float xrj = j == 0 ? xr.x : j == 1 ? xr.y : j == 2 ? xr.z : xr.w;
        const float g = token(xj, xoj, xrj, (mw >> (8 * j)) & 0xFFu, absA, s, sb, A);
        if (j == 0) d.x = g; else if (j == 1) d.y = g; else if (j == 2) d.z = g; else d.w = g;
      }
    }
    return d;
  };


  // ---- before the barrier: unscaled gradients, counts and partial sums.
  // Thread tid takes vector tid of each stage; the gradients of the last
  // group of kStages stages stay in registers, earlier ones are written out
  // unscaled (and re-read after the barrier).
  float4 dk[kStages];
  bool failed = false;
  int consumed = 0, issued = min(nstage, kStages);
  for (int b0 = 0; b0 < nstage && !failed; b0 += kStages) {
#pragma unroll
    for (int q = 0; q < kStages; ++q) {
      const int b = b0 + q;
      if (b >= nstage) break;
      const bool ok = mbar_wait(smem_u32(&full[q]), (b / kStages) & 1, ab);
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      const int v0 = v_lo + b * kStageVec, nv = min(kStageVec, v_hi - v0);
      if (tid < nv) {
        const int v = v0 + tid;
        const uint8_t* st = dyn_raw + q * kStageBytes;
        const float4 x = reinterpret_cast<const float4*>(st)[tid];
        const float4 xo = reinterpret_cast<const float4*>(st + kStageVec * 16)[tid];
        const float4 xr =
            beta != 0.f ? reinterpret_cast<const float4*>(st + kStageVec * 32)[tid] : make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t mw = tid < (nv & ~3) ? reinterpret_cast<const uint32_t*>(st + kStageVec * 48)[tid]
                                            : __ldg(reinterpret_cast<const uint32_t*>(p.mask) + v);
        n += nonzero_bytes(mw);
        dk[q] = tokens4(4 * v, x, xo, xr, mw, lift(4 * v, r_first, r_last, top));
      }
      consumed = b + 1;
      if (b + kStages < nstage) {
        __syncthreads();  // every thread is done with this stage's buffer
        if (tid == 0) issue(b + kStages);
        ++issued;
      }
    }
    if (!failed && b0 + kStages < nstage) {
#pragma unroll
      for (int q = 0; q < kStages; ++q) {
        const int v = v_lo + (b0 + q) * kStageVec + tid;
        if (v < v_hi) reinterpret_cast<float4*>(p.dlogp)[v] = dk[q];
      }
    }
  }
  if (failed) {
    // Let the copies still in flight land before the CTA leaves (the grid
    // barrier then runs out of time in the other CTAs too).
    if (tid == 0)
      for (int b = consumed; b < issued; ++b) {
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&full[b % kStages]), (b / kStages) & 1))
          if (clock64() - t0 > kTimeoutCycles) break;
      }
    return;
  }
  // The last T % 4 tokens: thread 0 of the last CTA (its range ends at nvec).
  const bool tail = tid == 0 && blockIdx.x == gridDim.x - 1;
  if (tail)
    for (int t = 4 * nvec; t < p.T; ++t) {
      const uint32_t m = __ldg(p.mask + t);
      n += m != 0u;
      const float A = adv_at(lift(t, 0, p.R - 1, pow2_floor(p.R - 1)));
      float absA, s, sb;
      side(A, absA, s, sb);
      p.dlogp[t] = token(__ldg(p.logp + t), __ldg(p.logp_old + t), beta != 0.f ? __ldg(p.logp_ref + t) : 0.f, m, absA,
                         s, sb, A);
    }
  float3 s3 = make_float3(sj, sk, static_cast<float>(nclip));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s3.x += __shfl_xor_sync(0xffffffffu, s3.x, o);
    s3.y += __shfl_xor_sync(0xffffffffu, s3.y, o);
    s3.z += __shfl_xor_sync(0xffffffffu, s3.z, o);
  }
  if (lane == 0) red_f3[warp] = s3;
  n = block_sum(n, red_i);  // its barriers also publish red_f3
  if (tid == 0) {
    float3 t3 = make_float3(0.f, 0.f, 0.f);
    for (int w = 0; w < kThreads / 32; ++w) {
      t3.x += red_f3[w].x;
      t3.y += red_f3[w].y;
      t3.z += red_f3[w].z;
    }
    p.part[blockIdx.x] = make_float4(t3.x, t3.y, t3.z, 0.f);
  }
  const long long N = grid_sync_sum(p.sync, n, p.status, &sh_total, &sh_last);
  if (N < 0) return;

  // ---- after the barrier: scale by 1/N.
  // fp32 throughout: FP64 issues at a small fraction of the FP32 rate on this part.
  const float inv_n = N > 0 ? __frcp_rn(static_cast<float>(N)) : 0.f;
  auto scale = [&](float4 d) { return make_float4(d.x * inv_n, d.y * inv_n, d.z * inv_n, d.w * inv_n); };
  const int b_keep = nstage > 0 ? ((nstage - 1) / kStages) * kStages : 0;  // first stage held in registers
  for (int b = 0; b < b_keep; ++b) {
    // Written by this same thread before the barrier.
    const int v = v_lo + b * kStageVec + tid;
    if (v < v_hi) {
      float4* d = reinterpret_cast<float4*>(p.dlogp) + v;
      *d = scale(__ldcg(d));
    }
  }
#pragma unroll
  for (int q = 0; q < kStages; ++q) {
    const int v = v_lo + (b_keep + q) * kStageVec + tid;
    if (b_keep + q < nstage && v < v_hi) reinterpret_cast<float4*>(p.dlogp)[v] = scale(dk[q]);
  }
  if (tail)
    for (int t = 4 * nvec; t < p.T; ++t) p.dlogp[t] = __ldcg(p.dlogp + t) * inv_n;

  // ---- the last CTA to arrive: the loss terms from the partial sums.
  if (!sh_last) return;  // thread 0 acquired every CTA's partial sums at the barrier
  // Every thread sums a fixed strided subset of the partials, then a fixed
  // shuffle tree and the eight warp sums in order: the result does not
  // depend on which CTA arrived last.
  float3 t3 = make_float3(0.f, 0.f, 0.f);
  for (int j = tid; j < static_cast<int>(gridDim.x); j += kThreads) {
    const float4 v = __ldcg(p.part + j);
    t3.x += v.x;
    t3.y += v.y;
    t3.z += v.z;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    t3.x += __shfl_xor_sync(0xffffffffu, t3.x, o);
    t3.y += __shfl_xor_sync(0xffffffffu, t3.y, o);
    t3.z += __shfl_xor_sync(0xffffffffu, t3.z, o);
  }
  __syncthreads();
  if (lane == 0) red_f3[warp] = t3;
  __syncthreads();
  if (tid == 0) {
    float dj = 0.f, dk = 0.f, dc = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) {
      dj += red_f3[w].x;
      dk += red_f3[w].y;
      dc += red_f3[w].z;
    }
    const float policy = -dj * inv_n, kl = dk * inv_n;
    p.stats[0] = policy + beta * kl;
    p.stats[1] = policy;
    p.stats[2] = kl;
    p.stats[3] = dc * inv_n;
  }
}

// Grid bound: one CTA per stage of vectors (2048 tokens) at most, and at
// most kCtasPerSm per SM.
int max_ctas(int T) {
  const int sms = device_sms();
  const int by_work = std::max(1, (T / 4 + kStageVec - 1) / kStageVec);
  return std::min(by_work, kCtasPerSm * sms);
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

size_t dyn_bytes(int R) {
  return static_cast<size_t>(kStages) * kStageBytes + (R <= kStageRollouts ? (2 * static_cast<size_t>(R) + 1) * 4 : 0);
}

}  // namespace

size_t grpo_workspace_bytes(int num_rollouts, int total_tokens) {
  (void)num_rollouts;
  return 256 + a256(static_cast<size_t>(max_ctas(total_tokens)) * 16);
}

cudaError_t launch_grpo(const GrpoArgs& a, cudaStream_t stream) {
  if (a.num_rollouts == 0) return cudaSuccess;
  const size_t dyn = dyn_bytes(a.num_rollouts);
  // Every CTA waits at the grid barrier, so the grid must be co-resident.
  cudaError_t e = cudaFuncSetAttribute(grpo_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, grpo_kernel, kThreads, dyn);
  if (e != cudaSuccess) return e;
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  const int sms = device_sms();
  const int grid = std::min(max_ctas(a.total_tokens), per_sm * sms);
  if (grid >= (1 << kArriveBits)) return cudaErrorInvalidConfiguration;
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
  k.sync = reinterpret_cast<unsigned long long*>(ws);
  k.part = reinterpret_cast<float4*>(ws + 256);
  k.status = a.status;
  k.R = a.num_rollouts;
  k.G = a.group_size;
  k.ngroups = a.num_rollouts / a.group_size;
  k.T = a.total_tokens;
  k.clip_eps = a.clip_eps;
  k.adv_eps = a.adv_eps;
  k.beta = a.kl_beta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grpo_kernel, k);
}

}  // namespace sa
