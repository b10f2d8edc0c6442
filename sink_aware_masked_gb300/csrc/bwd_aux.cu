// Backward preprocess of sink-aware attention (the main kernel and the
// conversion pass are in bwd_tc.cu).
//
// Math (explicit sink column with zero value; SinkFlex-RL section 5 and the
// summary page's alpha = sigmoid(l - s_h); per-head sink gradient from the
// "GPT-OSS agentic RL training" page):
//   l'  = l + softplus(s_h - l)        log-normaliser including the sink
//   D   = <dO, O>                      O is the final, alpha-scaled output
//   dsink[h] = -sum_rows (1 - alpha) D,   1 - alpha = sigmoid(s_h - l)
//
//   bwd_pre   : one pass over O and dO: the bias rows (-l'/scale and -D as
//               bf16 hi/mid/lo triples) the main kernel folds into its S^T and
//               dP^T MMAs, per-block partial dsink sums, zeroes the fp32 dQ
//               accumulator (which also brings it into L2 for the main
//               kernel's reduce-adds when it fits) and the main kernel's
//               unit-claim counters.
//               HBM-bound; every thread issues the loads of four tokens
//               before using them.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int D = kHeadDim;

// ------------------------------------------------------------------ preprocess
struct PreK {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  const float* sink;
  uint4* bias;
  float* dq_accum;
  float* dsink_part;
  int* counters;  // the main kernel's unit-claim counters, cleared here
  int n_counters;
  long long T;
  int hq;
  float scale;
};

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fx = __bfloat1622float2(x[i]);
    const float2 fy = __bfloat1622float2(y[i]);
    s = fmaf(fx.x, fy.x, s);
    s = fmaf(fx.y, fy.y, s);
  }
  return s;
}

// Block = kPreTokens tokens x 32 heads (a token group's heads take
// ceil(Hq / 32) consecutive blocks, so that a few thousand tokens still give
// the SMs an even share); thread = (head, 16-byte chunk of a 128-byte row).
// The block walks its tokens in batches of kPreBatch, issuing every load of
// a batch (O, dO, l) before any arithmetic so that enough bytes are in
// flight to reach HBM bandwidth.  The dsink partial sums stay one per
// (token group, head).
constexpr int kPreBatch = 4;

// v as hi + mid + lo, three round-to-nearest bf16 values (the remainder of
// each step is exact in fp32): about 24 significant bits in total.
__device__ __forceinline__ void split3_bf16(float v, uint16_t (&out)[3]) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    out[i] = __bfloat16_as_ushort(b);
    v -= __bfloat162float(b);
  }
}

__global__ void __launch_bounds__(256) bwd_pre_kernel(const PreK p) {
  const int sub = threadIdx.x & 7;  // 16-byte chunk of a 128-byte row
  const int nslots = (p.hq + 31) / 32;
  const int grp = static_cast<int>(blockIdx.x) / nslots;
  const int h = (static_cast<int>(blockIdx.x) - grp * nslots) * 32 + (threadIdx.x >> 3);
  const long long t0 = static_cast<long long>(grp) * kPreTokens;
  const long long t1 = min(t0 + kPreTokens, p.T);
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.n_counters; i += blockDim.x) p.counters[i] = 0;
  {
    const bool ok = h < p.hq;
    const float sk = ok ? __ldg(p.sink + h) : 0.f;
    float part = 0.f;
    for (long long tt = t0; tt < t1; tt += kPreBatch) {
      uint4 ov[kPreBatch], gv[kPreBatch];
      float lv[kPreBatch];
#pragma unroll
      for (int u = 0; u < kPreBatch; ++u) {
        const long long t = tt + u;
        const bool v = ok && t < t1;
        const size_t base = (static_cast<size_t>(v ? t : t0) * p.hq + (ok ? h : 0)) * D + sub * 8;
        ov[u] = v ? __ldg(reinterpret_cast<const uint4*>(p.o + base)) : make_uint4(0, 0, 0, 0);
        gv[u] = v ? __ldg(reinterpret_cast<const uint4*>(p.dout + base)) : make_uint4(0, 0, 0, 0);
        lv[u] = (v && sub == 0) ? __ldg(p.lse + static_cast<size_t>(h) * p.T + t) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kPreBatch; ++u) {
        const long long t = tt + u;
        if (ok && t < t1) {
          const size_t base = (static_cast<size_t>(t) * p.hq + h) * D + sub * 8;
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          reinterpret_cast<float4*>(p.dq_accum + base)[0] = z;
          reinterpret_cast<float4*>(p.dq_accum + base)[1] = z;
        }
      }
#pragma unroll
      for (int u = 0; u < kPreBatch; ++u) {
        const long long t = tt + u;
        float dot = dot8_bf16(ov[u], gv[u]);
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        dot += __shfl_xor_sync(0xffffffffu, dot, 4);
        if (ok && sub == 0 && t < t1) {
          const size_t idx = static_cast<size_t>(h) * p.T + t;
          const float l = lv[u];
          const float x = sk - l;
          const float softplus = fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x)));
          // -l'/scale and -D as three bf16 summands each: the main kernel
          // adds them to S^T and dP^T with one K=16 MMA (a 0/1 selector times
          // these rows), so its element-wise pass reads neither from shared
          // memory; three terms keep about 24 bits of each value.
          // Clamped finite (sink = +inf gives l' = +inf): exp2 of the biased
          // score still underflows to exactly 0, and the selector's zeros
          // times these entries stay 0 instead of NaN.
          uint16_t lb[3], db[3];
          split3_bf16(fminf(fmaxf(-(l + softplus) / p.scale, -1e30f), 1e30f), lb);
          split3_bf16(fminf(fmaxf(-dot, -1e30f), 1e30f), db);
          // Row [l_hi, l_mid, l_lo, d_hi, d_mid, d_lo, 0, 0].
          p.bias[idx] = make_uint4(lb[0] | (static_cast<uint32_t>(lb[1]) << 16),
                                   lb[2] | (static_cast<uint32_t>(db[0]) << 16),
                                   db[1] | (static_cast<uint32_t>(db[2]) << 16), 0u);
          const float one_minus_alpha = 1.f / (1.f + __expf(-x));
          part -= one_minus_alpha * dot;
        }
      }
    }
    if (ok && sub == 0) p.dsink_part[static_cast<size_t>(grp) * p.hq + h] = part;
  }
}

}  // namespace

// Preprocess, then the main kernel and the conversion pass (bwd_tc.cu).
cudaError_t launch_bwd(const Problem& pr, const BwdArgs& a, int* status, cudaStream_t stream) {
  const long long T = pr.total_tokens;
  // No rows: every gradient is empty and dsink is zero.
  if (T == 0 || pr.num_seqs == 0 || pr.seqlen == 0) return cudaMemsetAsync(a.dsink, 0, sizeof(float) * pr.hq, stream);
  PreK k{static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.sink,
         static_cast<uint4*>(a.bias), a.dq_accum, a.dsink_part, a.unit_counters, a.n_unit_counters,
         T, pr.hq, pr.scale};
  if (a.preprocess_blocks > 0) bwd_pre_kernel<<<a.preprocess_blocks * ((pr.hq + 31) / 32), 256, 0, stream>>>(k);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_bwd_tc_main(pr, a, status, stream);
}

}  // namespace sa
