// C ABI of the sink-aware attention library: argument checks, problem
// normalisation, workspace layout and kernel dispatch.  Declarations and the
// contract of every entry point are in include/sinkattn.h.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sinkattn.h"
#include "internal.h"
#include "tc.cuh"

namespace sa {
ProfileEvents g_prof_fwd, g_prof_bwd, g_prof_dec;
}

namespace {

// Device status word raised by kernels that give up a bounded wait.
__device__ int g_device_status = 0;

// Device address of g_device_status for the current device, looked up once
// per device (cudaGetSymbolAddress, under a lock; later calls read the cached
// pointer).  The first lookup on a device is a CUDA runtime call that stream
// capture does not record: make the first call of the library on each device
// outside any capture.
int* status_word() {
  constexpr int kMaxDevices = 256;
  static std::atomic<int*> ptr[kMaxDevices];
  static std::mutex setup;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* p = ptr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  std::lock_guard<std::mutex> lock(setup);
  p = ptr[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess || a == nullptr) return nullptr;
    p = static_cast<int*>(a);
    ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Validates `pr` and fills `out`.  Touches no CUDA API.
sinkattn_status normalise(const sinkattn_problem* pr, sa::Problem& out) {
  if (pr == nullptr) return SINKATTN_ERR_INVALID_ARG;
  if (pr->head_dim != sa::kHeadDim) return SINKATTN_ERR_UNSUPPORTED;
  if (pr->num_heads_kv < 1 || pr->num_heads_q < 1 || pr->num_heads_q % pr->num_heads_kv != 0)
    return SINKATTN_ERR_INVALID_ARG;
  if (pr->num_heads_q > sa::kMaxHeadsQ) return SINKATTN_ERR_UNSUPPORTED;
  if (pr->num_seqs < 0 || pr->seqlen < 0 || pr->total_tokens < 0) return SINKATTN_ERR_INVALID_ARG;
  if (pr->num_seqs > 65535) return SINKATTN_ERR_UNSUPPORTED;
  if (!(pr->scale > 0.f) || !std::isfinite(pr->scale)) return SINKATTN_ERR_INVALID_ARG;
  if (pr->window < -1 || pr->prefix < 0) return SINKATTN_ERR_INVALID_ARG;
  if (pr->causal != 0 && pr->causal != 1) return SINKATTN_ERR_INVALID_ARG;
  if ((pr->cu_seqlens == nullptr) != (pr->cu_seqlens_host == nullptr)) return SINKATTN_ERR_INVALID_ARG;
  if (pr->cu_seqlens == nullptr) {
    const long long t = static_cast<long long>(pr->num_seqs) * pr->seqlen;
    if (t != pr->total_tokens) return SINKATTN_ERR_INVALID_ARG;
  } else {
    const int32_t* cu = pr->cu_seqlens_host;
    if (cu[0] != 0) return SINKATTN_ERR_INVALID_ARG;
    int32_t mx = 0;
    for (int i = 0; i < pr->num_seqs; ++i) {
      const int32_t len = cu[i + 1] - cu[i];
      if (cu[i + 1] < cu[i]) return SINKATTN_ERR_INVALID_ARG;
      if (len > mx) mx = len;
    }
    if (cu[pr->num_seqs] != pr->total_tokens) return SINKATTN_ERR_INVALID_ARG;
    if (mx > pr->seqlen) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned16(pr->cu_seqlens) && pr->num_seqs > 0) return SINKATTN_ERR_ALIGNMENT;
  }
  // 64-bit element counts must stay addressable; the kernels index tokens as int.
  if (static_cast<long long>(pr->total_tokens) * pr->num_heads_q * sa::kHeadDim > (1LL << 40))
    return SINKATTN_ERR_UNSUPPORTED;
  out.num_seqs = pr->num_seqs;
  out.seqlen = pr->seqlen;
  out.cu = pr->cu_seqlens;
  out.cu_host = pr->cu_seqlens_host;
  out.total_tokens = pr->total_tokens;
  out.hq = pr->num_heads_q;
  out.hkv = pr->num_heads_kv;
  // A window reaching the whole sequence is the unbounded window; a prefix
  // covering the whole sequence is the same as the sequence length.
  out.window = (pr->window < 0 || pr->window >= static_cast<int64_t>(pr->seqlen) - 1)
                   ? -1
                   : static_cast<int>(pr->window);
  out.prefix = static_cast<int>(pr->prefix > pr->seqlen ? pr->seqlen : pr->prefix);
  out.causal = pr->causal;
  out.scale = pr->scale;
  return SINKATTN_OK;
}

// One CTA waits on an mbarrier that never completes, with a bounded wait.
__global__ void selftest_wait_kernel(int* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    sa::tc::mbar_init(sa::smem_u32(&bar), 1);
    sa::tc::fence_mbar_init();
  }
  __syncthreads();
  const sa::tc::Abort ab{&abort_flag, status};
  sa::tc::mbar_wait(sa::smem_u32(&bar), 0, ab, limit);
}

struct BwdLayout {
  size_t dq_accum, bias, part, counters, dkv, total;
  int pre_blocks, n_counters;
};

// Backward workspace: fp32 dQ accumulator [T, Hq, 64], bias rows [Hq, T]
// (16 bytes), dsink partial sums [preprocess blocks, Hq], the main kernel's
// unit-claim counters (one int per launch), then the per-chunk dK/dV slots of
// split key tiles.  Every part starts at a 256-byte boundary.  Nothing needs
// to be zero on entry: the preprocess kernel clears the accumulator and the
// counters.
BwdLayout bwd_layout(const sa::Problem& p) {
  BwdLayout l;
  const size_t T = static_cast<size_t>(p.total_tokens), H = static_cast<size_t>(p.hq);
  l.pre_blocks = sa::ceil_div(p.total_tokens, sa::kPreTokens);
  l.n_counters = sa::bwd_tc_main_slices(p);
  l.dq_accum = 0;
  l.bias = l.dq_accum + round_up(T * H * sa::kHeadDim * 4, 256);
  l.part = l.bias + round_up(T * H * 16, 256);
  l.counters = l.part + round_up(static_cast<size_t>(l.pre_blocks) * H * 4, 256);
  l.dkv = l.counters + round_up(static_cast<size_t>(l.n_counters) * 4, 256);
  l.total = l.dkv + round_up(sa::bwd_split_acc_bytes(p), 256) + 256;
  return l;
}

sinkattn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA; }

}  // namespace

extern "C" {

int32_t sinkattn_kernel_launches(const sinkattn_problem* prob, int32_t which) {
  sa::Problem p;
  if (normalise(prob, p) != SINKATTN_OK) return -1;
  if (which == 1) return sa::fwd_tc_launches(p);
  if (which == 2) return (bwd_layout(p).pre_blocks > 0 ? 1 : 0) + sa::bwd_tc_main_launches(p);
  return -1;
}

size_t sinkattn_fwd_workspace_size(const sinkattn_problem* prob) {
  sa::Problem p;
  if (normalise(prob, p) != SINKATTN_OK) return 0;
  return 0;
}

size_t sinkattn_bwd_workspace_size(const sinkattn_problem* prob) {
  sa::Problem p;
  if (normalise(prob, p) != SINKATTN_OK) return 0;
  return bwd_layout(p).total;
}

sinkattn_status sinkattn_fwd(const sinkattn_problem* prob, const void* q, const void* k, const void* v,
                             const float* sink, void* o, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  sa::Problem p;
  sinkattn_status st = normalise(prob, p);
  if (st != SINKATTN_OK) return st;
  (void)workspace;
  (void)workspace_bytes;
  if (p.total_tokens == 0) return SINKATTN_OK;
  if (!q || !k || !v || !sink || !o || !lse) return SINKATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(sink))
    return SINKATTN_ERR_ALIGNMENT;
  sa::FwdArgs a{q, k, v, sink, o, lse};
  int* status = status_word();
  if (status == nullptr) return SINKATTN_ERR_CUDA;
  return from_cuda(sa::launch_fwd_tc(p, a, status, static_cast<cudaStream_t>(stream)));
}

sinkattn_status sinkattn_bwd(const sinkattn_problem* prob, const void* q, const void* k, const void* v,
                             const void* o, const float* lse, const void* dout, const float* sink, void* dq,
                             void* dk, void* dv, float* dsink, void* workspace, size_t workspace_bytes,
                             void* stream) {
  sa::Problem p;
  sinkattn_status st = normalise(prob, p);
  if (st != SINKATTN_OK) return st;
  if (!dsink || !sink) return SINKATTN_ERR_INVALID_ARG;
  if (!aligned16(dsink) || !aligned16(sink)) return SINKATTN_ERR_ALIGNMENT;
  const BwdLayout L = bwd_layout(p);
  if (p.total_tokens > 0) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
      return SINKATTN_ERR_ALIGNMENT;
  }
  if (workspace_bytes < L.total) return SINKATTN_ERR_WORKSPACE;
  if (workspace == nullptr || !aligned16(workspace)) return workspace ? SINKATTN_ERR_ALIGNMENT : SINKATTN_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  sa::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.sink = sink;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dsink = dsink;
  a.dq_accum = reinterpret_cast<float*>(ws + L.dq_accum);
  a.bias = ws + L.bias;
  a.dsink_part = reinterpret_cast<float*>(ws + L.part);
  a.dkv_acc = sa::bwd_split_acc_bytes(p) ? reinterpret_cast<float*>(ws + L.dkv) : nullptr;
  a.unit_counters = reinterpret_cast<int*>(ws + L.counters);
  a.n_unit_counters = L.n_counters;
  a.preprocess_blocks = L.pre_blocks;
  int* status = status_word();
  if (status == nullptr) return SINKATTN_ERR_CUDA;
  return from_cuda(sa::launch_bwd(p, a, status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

struct DecodeLayout {
  sa::DecodePlan plan;
  size_t counters, acc, ml, total;
};

// Validates the decode-specific arguments on top of normalise().
sinkattn_status decode_check(const sa::Problem& p, int32_t q_per_seq) {
  if (q_per_seq < 1) return SINKATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(p.hq / p.hkv) * q_per_seq > 128) return SINKATTN_ERR_UNSUPPORTED;
  if (p.num_seqs > sa::kDecodeMaxItems) return SINKATTN_ERR_UNSUPPORTED;
  for (int b = 0; b < p.num_seqs; ++b) {
    const int len = p.cu_host ? p.cu_host[b + 1] - p.cu_host[b] : p.seqlen;
    if (len < q_per_seq) return SINKATTN_ERR_INVALID_ARG;
  }
  return SINKATTN_OK;
}

DecodeLayout decode_layout(const sa::Problem& p, int32_t q_per_seq) {
  DecodeLayout l;
  l.plan = sa::decode_plan(p, q_per_seq);
  l.counters = 0;
  l.acc = round_up(l.plan.counter_bytes, 256);
  l.ml = l.acc + round_up(l.plan.acc_bytes, 256);
  l.total = l.ml + round_up(l.plan.ml_bytes, 256) + 256;
  return l;
}

}  // namespace

extern "C" {

size_t sinkattn_decode_workspace_size(const sinkattn_problem* kv, int32_t q_per_seq) {
  sa::Problem p;
  if (normalise(kv, p) != SINKATTN_OK || decode_check(p, q_per_seq) != SINKATTN_OK) return 0;
  return decode_layout(p, q_per_seq).total;
}

sinkattn_status sinkattn_decode_fwd(const sinkattn_problem* kv, int32_t q_per_seq, const void* q, const void* k,
                                    const void* v, const float* sink, void* o, float* lse, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  sa::Problem p;
  sinkattn_status st = normalise(kv, p);
  if (st != SINKATTN_OK) return st;
  if ((st = decode_check(p, q_per_seq)) != SINKATTN_OK) return st;
  if (p.num_seqs == 0) return SINKATTN_OK;
  if (!q || !k || !v || !sink || !o || !lse) return SINKATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(sink))
    return SINKATTN_ERR_ALIGNMENT;
  const DecodeLayout L = decode_layout(p, q_per_seq);
  if (workspace_bytes < L.total) return SINKATTN_ERR_WORKSPACE;
  if (workspace == nullptr || !aligned16(workspace)) return workspace ? SINKATTN_ERR_ALIGNMENT : SINKATTN_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  sa::DecodeArgs a{q, k, v, sink, o, lse, reinterpret_cast<float*>(ws + L.acc), ws + L.ml,
                   reinterpret_cast<int*>(ws + L.counters)};
  int* status = status_word();
  if (status == nullptr) return SINKATTN_ERR_CUDA;
  return from_cuda(sa::launch_decode(p, q_per_seq, a, L.plan, status, static_cast<cudaStream_t>(stream)));
}

namespace {

sinkattn_status grpo_check(const sinkattn_grpo_problem* g) {
  if (g == nullptr) return SINKATTN_ERR_INVALID_ARG;
  if (g->num_rollouts < 0 || g->group_size < 1 || g->total_tokens < 0) return SINKATTN_ERR_INVALID_ARG;
  if (g->num_rollouts % g->group_size != 0) return SINKATTN_ERR_INVALID_ARG;
  if (!(g->clip_eps > 0.f) || !std::isfinite(g->clip_eps)) return SINKATTN_ERR_INVALID_ARG;
  if (!(g->adv_eps >= 0.f) || !std::isfinite(g->adv_eps)) return SINKATTN_ERR_INVALID_ARG;
  if (!(g->kl_beta >= 0.f) || !std::isfinite(g->kl_beta)) return SINKATTN_ERR_INVALID_ARG;
  if (g->num_rollouts > 0 && (g->cu_tokens == nullptr || g->cu_tokens_host == nullptr)) return SINKATTN_ERR_INVALID_ARG;
  if (g->num_rollouts > 0) {
    const int32_t* cu = g->cu_tokens_host;
    if (cu[0] != 0 || cu[g->num_rollouts] != g->total_tokens) return SINKATTN_ERR_INVALID_ARG;
    for (int i = 0; i < g->num_rollouts; ++i)
      if (cu[i + 1] < cu[i]) return SINKATTN_ERR_INVALID_ARG;
  }
  return SINKATTN_OK;
}

}  // namespace

size_t sinkattn_grpo_workspace_size(const sinkattn_grpo_problem* g) {
  if (grpo_check(g) != SINKATTN_OK) return 0;
  return sa::grpo_workspace_bytes(g->num_rollouts, g->total_tokens);
}

sinkattn_status sinkattn_grpo_loss(const sinkattn_grpo_problem* g, const float* logp, const float* logp_old,
                                   const float* logp_ref, const uint8_t* mask, const float* rewards, float* stats,
                                   float* dlogp, float* advantages, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  sinkattn_status st = grpo_check(g);
  if (st != SINKATTN_OK) return st;
  if (!stats) return SINKATTN_ERR_INVALID_ARG;
  if (g->num_rollouts == 0) return from_cuda(cudaMemsetAsync(stats, 0, 4 * sizeof(float), static_cast<cudaStream_t>(stream)));
  if (!logp || !logp_old || !mask || !rewards || !dlogp || (g->kl_beta != 0.f && !logp_ref))
    return SINKATTN_ERR_INVALID_ARG;
  if (!aligned16(logp) || !aligned16(logp_old) || !aligned16(mask) || !aligned16(dlogp) ||
      (g->kl_beta != 0.f && !aligned16(logp_ref)))
    return SINKATTN_ERR_ALIGNMENT;
  if (!aligned16(workspace)) return workspace ? SINKATTN_ERR_ALIGNMENT : SINKATTN_ERR_INVALID_ARG;
  if (workspace_bytes < sa::grpo_workspace_bytes(g->num_rollouts, g->total_tokens)) return SINKATTN_ERR_WORKSPACE;
  sa::GrpoArgs a{g->num_rollouts, g->group_size, g->total_tokens, g->cu_tokens, g->clip_eps, g->adv_eps, g->kl_beta,
                 logp, logp_old, logp_ref, mask, rewards, stats, dlogp, advantages, workspace, status_word()};
  if (a.status == nullptr) return SINKATTN_ERR_CUDA;
  return from_cuda(sa::launch_grpo(a, static_cast<cudaStream_t>(stream)));
}

sinkattn_status sinkattn_varlen_plan(const int32_t* seqlens, int32_t num_seqs, int32_t* cu_seqlens_out,
                                     void* stream) {
  if (num_seqs < 0 || cu_seqlens_out == nullptr || (num_seqs > 0 && seqlens == nullptr))
    return SINKATTN_ERR_INVALID_ARG;
  return from_cuda(sa::launch_varlen_plan(seqlens, num_seqs, cu_seqlens_out, static_cast<cudaStream_t>(stream)));
}

static sinkattn_status pack_common(const void* src, const int32_t* cu, int32_t B, int32_t Smax, int32_t H,
                                   int32_t D, void* dst, bool unpack, void* stream) {
  if (B < 0 || Smax < 0 || H < 1 || D < 1) return SINKATTN_ERR_INVALID_ARG;
  if ((static_cast<long long>(H) * D * 2) % 16 != 0) return SINKATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Smax == 0) return SINKATTN_OK;
  if (!src || !cu || !dst) return SINKATTN_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return SINKATTN_ERR_ALIGNMENT;
  return from_cuda(sa::launch_pack(src, cu, B, Smax, H, D, dst, unpack, static_cast<cudaStream_t>(stream)));
}

sinkattn_status sinkattn_pack(const void* padded, const int32_t* cu_seqlens, int32_t B, int32_t Smax, int32_t H,
                              int32_t D, void* packed, void* stream) {
  return pack_common(padded, cu_seqlens, B, Smax, H, D, packed, false, stream);
}

sinkattn_status sinkattn_unpack(const void* packed, const int32_t* cu_seqlens, int32_t B, int32_t Smax, int32_t H,
                                int32_t D, void* padded, void* stream) {
  return pack_common(packed, cu_seqlens, B, Smax, H, D, padded, true, stream);
}

sinkattn_status sinkattn_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SINKATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return SINKATTN_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return SINKATTN_ERR_CUDA;
    return SINKATTN_ERR_TIMEOUT;
  }
  return SINKATTN_OK;
}

sinkattn_status sinkattn_set_profile_events(int32_t kind, void* start, void* stop) {
  if ((start == nullptr) != (stop == nullptr)) return SINKATTN_ERR_INVALID_ARG;
  sa::ProfileEvents ev;
  ev.start = static_cast<cudaEvent_t>(start);
  ev.stop = static_cast<cudaEvent_t>(stop);
  if (kind == 1)
    sa::g_prof_fwd = ev;
  else if (kind == 2)
    sa::g_prof_bwd = ev;
  else if (kind == 3)
    sa::g_prof_dec = ev;
  else
    return SINKATTN_ERR_INVALID_ARG;
  return SINKATTN_OK;
}

sinkattn_status sinkattn_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > 2000000000LL) return SINKATTN_ERR_INVALID_ARG;
  int* status = status_word();
  if (status == nullptr) return SINKATTN_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_cycles);
  return from_cuda(cudaGetLastError());
}

const char* sinkattn_status_string(sinkattn_status s) {
  switch (s) {
    case SINKATTN_OK: return "ok";
    case SINKATTN_ERR_INVALID_ARG: return "invalid argument";
    case SINKATTN_ERR_UNSUPPORTED: return "unsupported problem";
    case SINKATTN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SINKATTN_ERR_WORKSPACE: return "workspace too small";
    case SINKATTN_ERR_CUDA: return "CUDA error";
    case SINKATTN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int32_t sinkattn_version(void) { return 100; }

}  // extern "C"
