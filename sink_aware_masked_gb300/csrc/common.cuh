// Device-side helpers shared by the sink-aware attention kernels.
//
// Mask: M[q, k] = [k <= q] and ([q - k <= w] or [k < p]) (SinkFlex-RL summary
// page, paragraph on the sink-aware FlexAttention path), with positions
// inside one packed sequence, plus the sequence bound k < len.  The mask is
// pure index arithmetic: no mask tensor exists anywhere.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#define SA_DEV __device__ __forceinline__

namespace sa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Normalised mask parameters: window < 0 means unbounded; the host folds any
// window >= len - 1 into "unbounded" and clamps prefix to the longest
// sequence, which leaves the mask unchanged.
struct MaskParams {
  int window;
  int prefix;
  int causal;
};

SA_DEV bool visible(int q, int k, int len, const MaskParams& m) {
  if (k >= len) return false;
  if (m.causal && k > q) return false;
  return (m.window < 0) || (q - k <= m.window) || (k < m.prefix);
}

struct SeqSpan {
  int start;
  int len;
};

SA_DEV SeqSpan seq_span(const int32_t* cu, int uniform_len, int b) {
  if (cu != nullptr) {
    int s = __ldg(cu + b);
    return {s, __ldg(cu + b + 1) - s};
  }
  return {b * uniform_len, uniform_len};
}

// Key range a block of queries [q0, q1] can see: keys [lo, hi] of the
// window/causal band plus the prefix keys [0, pre_end) below lo.
struct KeyRange {
  int pre_end;  // prefix keys [0, pre_end) that lie below lo
  int lo;
  int hi;       // inclusive; hi < lo means empty
};

SA_DEV KeyRange key_range(int q0, int q1, int len, const MaskParams& m) {
  KeyRange r;
  r.hi = m.causal ? min(q1, len - 1) : len - 1;
  r.lo = (m.window < 0) ? 0 : max(0, q0 - m.window);
  r.pre_end = min(min(m.prefix, r.lo), r.hi + 1);
  if (r.pre_end < 0) r.pre_end = 0;
  return r;
}

// Query range [lo, hi] that can see some key of [k0, k1].
SA_DEV void query_range(int k0, int k1, int len, const MaskParams& m, int& lo, int& hi) {
  lo = m.causal ? k0 : 0;
  if (m.prefix > k0 || m.window < 0)
    hi = len - 1;
  else
    hi = min(len - 1, k1 + m.window);
}

// True when every (q, k) of the block [q0, q0+nq) x [k0, k0+nk) is visible
// and inside the sequence, so the per-element predicate can be skipped.
SA_DEV bool block_full(int q0, int nq, int k0, int nk, int len, const MaskParams& m) {
  const int q1 = q0 + nq - 1, k1 = k0 + nk - 1;
  if (q1 >= len || k1 >= len) return false;
  if (m.causal && k1 > q0) return false;
  return (m.window < 0) || (q1 - k0 <= m.window) || (k1 < m.prefix);
}

// Bit e set for e < n, n clamped to [0, 32].
SA_DEV uint32_t bits_below(int n) { return n <= 0 ? 0u : (n >= 32 ? 0xFFFFFFFFu : (1u << n) - 1u); }

// visible(q, kbase + e, len, m) for e = 0..31 as a bit mask: keys up to the
// causal / sequence bound, and at or above the window's lower edge unless
// they lie in the prefix.
SA_DEV uint32_t visible_bits(int q, int kbase, int len, const MaskParams& m) {
  const int hi = (m.causal ? min(q, len - 1) : len - 1) - kbase;
  uint32_t r = bits_below(hi + 1);
  if (m.window >= 0) r &= ~bits_below(q - m.window - kbase) | bits_below(m.prefix - kbase);
  return r;
}

// visible(qbase + e, key, len, m) and qbase + e < len for e = 0..31 as a bit
// mask: the queries that see one key form a single interval, from the key
// itself (causal) up to the sequence end or, for a key outside the prefix,
// key + w.
SA_DEV uint32_t query_bits(int key, int qbase, int len, const MaskParams& m) {
  if (key >= len) return 0u;
  const int lo = m.causal ? key - qbase : -64;
  int hi = len - 1 - qbase;
  if (m.window >= 0 && key >= m.prefix) hi = min(hi, key + m.window - qbase);
  return bits_below(hi + 1) & ~bits_below(lo);
}

// ---------------------------------------------------------------- PTX helpers
SA_DEV uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// 16-byte async copy global -> shared; zero-fills when !valid.
SA_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
SA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
SA_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

SA_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
SA_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
SA_DEV void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

SA_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Hardware base-2 exponential (MUFU); ex2(-inf) = 0.
SA_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (sm_100 family).
SA_DEV float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed pairs of fp32 (sm_100 family f32x2 instructions).
SA_DEV float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;\n"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
SA_DEV float2 fadd2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;\n"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
SA_DEV float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;\n"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

// Offset in bytes of 16-byte chunk `c` (0..7) of row `r` in a tile whose rows
// are 64 bf16 (128 bytes): chunks are XOR-swizzled by the row's low 3 bits so
// that ldmatrix reads of 8 rows at one chunk column hit 8 different banks.
SA_DEV uint32_t swz(int r, int c) { return static_cast<uint32_t>((r * 8 + (c ^ (r & 7))) * 16); }

}  // namespace sa
