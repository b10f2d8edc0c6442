// Host-side TMA tensor maps for the [T, H, 64] bf16 token-major tensors.
//
// A tensor is viewed as a 2-D array: inner dimension H * 64 elements (one
// token's row over all heads), outer dimension T tokens.  A box is 64
// elements x `box_rows` tokens, i.e. one head's 128-byte rows of box_rows
// consecutive tokens, written to shared memory with the 128-byte swizzle
// that the tcgen05 shared-memory descriptors expect.  Rows past T are
// zero-filled by the TMA unit.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace sa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Returns false when the driver entry point is missing or the encode fails.
inline bool make_rows_map(CUtensorMap* m, const void* base, long long tokens, int heads, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads) * 64, static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * 64 * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [T, H * 64] accumulator: boxes of 32 floats (128 B) x box_rows tokens,
// 128-byte swizzled in shared memory; used for element-wise reduce-adds.
inline bool make_f32_rows_map(CUtensorMap* m, void* base, long long tokens, int heads, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads) * 64, static_cast<cuuint64_t>(tokens)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * 64 * 4};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sa
