// Packed-sequence front end for multi-turn trajectories of different lengths
// (SinkFlex-RL section 3: long, multi-turn, tool-heavy trajectories).
//
//   varlen_plan : sequence lengths -> offsets cu[0..n] (exclusive prefix sum),
//                 one CTA, warp-shuffle scan with a running carry; no host sync.
//   pack/unpack : [B, Smax, H, D] padded  <->  [T, H, D] packed, 16-byte
//                 vectors; unpack writes zeros into the padding rows.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

__global__ void __launch_bounds__(1024) varlen_plan_kernel(const int32_t* __restrict__ lens, int n,
                                                          int32_t* __restrict__ cu) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    cu[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int i = base + tid;
    int x = (i < n) ? max(lens[i], 0) : 0;
    // inclusive scan inside the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;  // inclusive totals per warp
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (i < n) cu[i + 1] = before + x;
    __syncthreads();
    if (tid == 1023) carry = before + x;
    __syncthreads();
  }
}

struct PackK {
  const uint4* src;
  uint4* dst;
  const int32_t* cu;
  int B, Smax;
  int vec_per_row;  // H * D * 2 / 16
  bool unpack;
};

// One thread per 16-byte vector of the padded tensor.
__global__ void __launch_bounds__(256) pack_kernel(const PackK p) {
  const long long total = static_cast<long long>(p.B) * p.Smax * p.vec_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long row = i / p.vec_per_row;
    const int v = static_cast<int>(i - row * p.vec_per_row);
    const int b = static_cast<int>(row / p.Smax);
    const int r = static_cast<int>(row - static_cast<long long>(b) * p.Smax);
    const int start = p.cu[b];
    const int len = p.cu[b + 1] - start;
    const long long prow = static_cast<long long>(start) + r;
    if (!p.unpack) {
      if (r < len) p.dst[prow * p.vec_per_row + v] = p.src[i];
    } else {
      p.dst[i] = (r < len) ? p.src[prow * p.vec_per_row + v] : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

}  // namespace

cudaError_t launch_varlen_plan(const int32_t* lens, int n, int32_t* cu, cudaStream_t s) {
  varlen_plan_kernel<<<1, 1024, 0, s>>>(lens, n, cu);
  return cudaGetLastError();
}

cudaError_t launch_pack(const void* src, const int32_t* cu, int B, int Smax, int H, int D, void* dst, bool unpack,
                        cudaStream_t s) {
  PackK k{static_cast<const uint4*>(src), static_cast<uint4*>(dst), cu, B, Smax, H * D * 2 / 16, unpack};
  const long long total = static_cast<long long>(B) * Smax * k.vec_per_row;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  const long long cap = 32LL * device_sms();
  if (blocks > cap) blocks = cap;
  pack_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(k);
  return cudaGetLastError();
}

}  // namespace sa
