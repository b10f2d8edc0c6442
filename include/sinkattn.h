/*
 * sinkattn.h — C ABI of the GB300 (sm_103a) sink-aware attention library.
 *
 * The operation is exact softmax attention under the mask of the SinkFlex-RL
 * paper ("Efficient Reinforcement Learning for Long-Horizon Tool-Use Agentic
 * Tasks", summary page, paragraph on the sink-aware FlexAttention path):
 *
 *     M[q, k] = [k <= q]  and  ( [q - k <= w]  or  [k < p] )
 *
 * with w the local window (inclusive; w + 1 keys including the query) and p
 * the number of always-visible prefix positions, the same mask for every
 * sequence and head.  Scores are s_qk = scale * <Q_q, K_k>.  The attention
 * call returns the output together with the natural-log log-sum-exp
 * l_q = log sum_{k visible} exp(s_qk) (sink excluded), and the output is
 * scaled by alpha_q = sigmoid(l_q - sink[h]), which is the same as appending
 * one more softmax column with logit sink[h] and a zero value vector
 * (section 5, "zero-value sink equivalence").  The backward returns dQ, dK,
 * dV and the per-head sink gradient dL/dS_h ("GPT-OSS agentic RL training"
 * page, FlashAttention v3 implementation), recomputing probabilities from l
 * so that no S x S matrix is ever stored.
 *
 * Layouts (all contiguous, row-major, head_dim innermost):
 *   q, o, dout, dq : bf16 [T, Hq, D]
 *   k, v, dk, dv   : bf16 [T, Hkv, D]
 *   lse            : fp32 [Hq, T]
 *   sink, dsink    : fp32 [Hq]
 * T is the number of tokens of all packed sequences.  Query head h reads
 * key/value head h / (Hq / Hkv) (contiguous GQA groups).  Positions inside
 * the mask are positions inside each packed sequence.
 *
 * Ownership: the caller allocates every buffer, including the workspace,
 * and keeps it alive until the stream has run the work.  The library
 * allocates no device memory and keeps no per-call state.  All device
 * pointers must be 16-byte aligned.  Every call is asynchronous on `stream`
 * (a cudaStream_t passed as void*; NULL = legacy default stream).
 * Outputs are overwritten, never accumulated (dsink included).  No output
 * may alias an input or another output.
 *
 * Errors: argument checks run on the host before anything is launched; a
 * failing check returns its status and launches nothing.  A failed launch
 * returns SINKATTN_ERR_CUDA.  Nothing aborts, exits or traps on the device.
 *
 * First call on a device: the calls that launch kernels (fwd, bwd, decode,
 * GRPO, the wait self-test) look up the device address of the library's
 * status word once per device, with that device current, through
 * cudaGetSymbolAddress (thread-safe).  Make the first such call on each
 * device outside any stream capture; later calls only launch kernels.
 */
#ifndef SINKATTN_H
#define SINKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SINKATTN_OK = 0,
  SINKATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad mask parameter, bad cu_seqlens */
  SINKATTN_ERR_UNSUPPORTED = 2,  /* head_dim other than 64, or sizes beyond the int32 index range */
  SINKATTN_ERR_ALIGNMENT = 3,    /* a device pointer that is not 16-byte aligned */
  SINKATTN_ERR_WORKSPACE = 4,    /* workspace smaller than the matching *_workspace_size() */
  SINKATTN_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
  SINKATTN_ERR_TIMEOUT = 6       /* a kernel gave up a bounded wait (see sinkattn_get_device_status) */
} sinkattn_status;

/* One attention problem.  Uniform batch: cu_seqlens == NULL, num_seqs = B,
 * seqlen = S, total_tokens = B * S.  Packed variable-length sequences:
 * cu_seqlens (device) and cu_seqlens_host (host) hold the same num_seqs + 1
 * offsets, cu[0] = 0, nondecreasing, cu[num_seqs] = total_tokens, and
 * seqlen is the largest cu[i+1] - cu[i]. */
typedef struct {
  int32_t num_seqs;
  int32_t seqlen;
  const int32_t* cu_seqlens;       /* device, [num_seqs + 1], or NULL */
  const int32_t* cu_seqlens_host;  /* host copy of cu_seqlens (NULL iff cu_seqlens is NULL) */
  int32_t total_tokens;
  int32_t num_heads_q;             /* Hq, a multiple of num_heads_kv */
  int32_t num_heads_kv;            /* Hkv >= 1 */
  int32_t head_dim;                /* must be 64 */
  int64_t window;                  /* w >= 0 (inclusive), or -1 for unbounded */
  int64_t prefix;                  /* p >= 0 */
  int32_t causal;                  /* 1: keep [k <= q]; 0: drop that term */
  float scale;                     /* softmax scale, finite and > 0 (1/sqrt(64) usually) */
} sinkattn_problem;

/* Bytes of device workspace that sinkattn_fwd / sinkattn_bwd need for
 * `prob` (0 when the problem is invalid). */
size_t sinkattn_fwd_workspace_size(const sinkattn_problem* prob);
size_t sinkattn_bwd_workspace_size(const sinkattn_problem* prob);

/* Number of kernel launches sinkattn_fwd (which = 1) or sinkattn_bwd /
 * sinkattn_bwd_noalloc (which = 2) make for this problem, from host
 * arithmetic alone (the same work lists the calls build); -1 for an invalid
 * problem or `which`.  Lets a caller count the library's launches without a
 * profiler.  The calls make no other stream operation, except the backward
 * of a problem without tokens, which sets dsink to zero with one memset. */
int32_t sinkattn_kernel_launches(const sinkattn_problem* prob, int32_t which);

/* Forward.  Reads q, k, v (bf16) and sink (fp32 [Hq]); writes
 * o = alpha * softmax_M(s) V (bf16 [T, Hq, 64]) and lse = l (fp32 [Hq, T]).
 * Rows of a sequence are never mixed with rows of another sequence. */
sinkattn_status sinkattn_fwd(const sinkattn_problem* prob,
                             const void* q, const void* k, const void* v, const float* sink,
                             void* o, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Backward.  Reads the forward's inputs, its outputs o and lse, and dout;
 * writes dq, dk, dv (bf16) and dsink (fp32 [Hq]), where
 * dsink[h] = -sum over all rows of (1 - alpha_q) * <dout_q, o_q>.
 * The workspace holds an fp32 dQ accumulator [T, Hq, 64], one 16-byte row
 * per (head, token) with the per-row terms -D and -l'/scale, where
 * l' = l + softplus(sink - l), as three bf16 summands each ([Hq, T]),
 * partial sums of dsink per 8-token group and head, and, when key tiles are split over
 * several work items, per-chunk dK/dV partial sums.
 * Its contents on entry do not matter (the call clears what it accumulates
 * into).  dK, dV and dsink are bitwise reproducible run to run; dQ is summed
 * in arrival order and reproducible to fp32 rounding. */
sinkattn_status sinkattn_bwd(const sinkattn_problem* prob,
                             const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, const float* sink,
                             void* dq, void* dk, void* dv, float* dsink,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Backward without a caller-provided workspace, for callers that cannot
 * allocate device memory (a host program with no device allocator of its
 * own, a runtime whose memory pool is fixed at start-up, a hot loop where an
 * allocation is not acceptable).  The paper has no counterpart: this is a
 * deployment variant of sinkattn_bwd, same arguments minus the workspace,
 * same results.  It uses a 32 MiB workspace compiled into the library as a
 * device array (held by every GPU that loads the library until the process
 * ends) and allocates nothing.  Problems whose sinkattn_bwd_workspace_size()
 * exceeds 32 MiB return SINKATTN_ERR_WORKSPACE and launch nothing.  The
 * first call on each device looks up the array's device address while that
 * device is current; make it before any stream capture.  All calls share
 * the array: calls whose kernels overlap on the GPU race and must be
 * serialised by the caller.  Nothing in the array needs clearing between
 * calls (the kernels clear what they accumulate into). */
sinkattn_status sinkattn_bwd_noalloc(const sinkattn_problem* prob,
                                     const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout, const float* sink,
                                     void* dq, void* dk, void* dv, float* dsink, void* stream);

/* Decode forward: the rollout side of the same attention (SinkFlex-RL,
 * rollout worker: the policy samples turn by turn; GPT-OSS agentic RL page:
 * the sink-aware forward of an inference FlashAttention fork).  `kv`
 * describes the cached sequences exactly as `prob` does for sinkattn_fwd:
 * k, v bf16 [kv->total_tokens, Hkv, 64] hold every position of each
 * sequence.  q bf16 [num_seqs * q_per_seq, Hq, 64] holds, for sequence b,
 * the queries of its last q_per_seq positions L_b - q_per_seq ... L_b - 1
 * in that order (rows b * q_per_seq ...).  Writes o bf16 [num_seqs *
 * q_per_seq, Hq, 64] and lse fp32 [Hq, num_seqs * q_per_seq], each row equal
 * to the same row of sinkattn_fwd over the whole sequence (same mask, sink
 * and lse).  Limits: 1 <= q_per_seq <= every sequence length,
 * (Hq / Hkv) * q_per_seq <= 128 and num_seqs <= 4096, else
 * SINKATTN_ERR_INVALID_ARG / SINKATTN_ERR_UNSUPPORTED.  The workspace
 * (sinkattn_decode_workspace_size bytes, 16-byte aligned) holds the partial
 * results of the key chunks and one counter per (sequence, kv head); its
 * size depends on the device's SM count.  Its first 4 * num_seqs * Hkv bytes
 * (the counters) must be zero before the first call; every completed call
 * leaves them zero, so a workspace zero-filled once can be reused by later
 * calls (not by calls that overlap on the GPU).  After SINKATTN_ERR_TIMEOUT,
 * zero the workspace again. */
size_t sinkattn_decode_workspace_size(const sinkattn_problem* kv, int32_t q_per_seq);
sinkattn_status sinkattn_decode_fwd(const sinkattn_problem* kv, int32_t q_per_seq,
                                    const void* q, const void* k, const void* v, const float* sink,
                                    void* o, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* GRPO token loss and its gradient (SinkFlex-RL, zh page, "Policy update",
 * equations (3)-(7)), the memory-bound step of the same training loop.
 * Rollouts are consecutive groups of group_size (the G rollouts of one
 * prompt); rollout i owns tokens [cu_tokens[i], cu_tokens[i + 1]) of the
 * fp32 arrays logp (current policy), logp_old (sampling policy) and
 * logp_ref (reference policy; may be NULL when kl_beta == 0); mask (uint8,
 * nonzero = optimised token); rewards fp32 [num_rollouts].
 *   A_i = (R_i - mean_group) / (population std of the group + adv_eps)
 *   rho = exp(logp - logp_old),  J = min(rho A_i, clip(rho, 1 -+ clip_eps) A_i)
 *   loss = -(1/N) sum J + kl_beta (1/N) sum (e^r - r - 1),  r = logp_ref - logp
 * with both sums over optimised tokens and N their count.  Writes stats fp32
 * [4] = {loss, -(1/N) sum J, (1/N) sum (e^r - r - 1), fraction of optimised
 * tokens whose gradient the clip removes}, dlogp fp32 [total_tokens] =
 * dloss/dlogp (0 on tokens that are not optimised) and, if non-NULL,
 * advantages fp32 [num_rollouts].  With N = 0 everything is 0.  logp,
 * logp_old, logp_ref, mask and dlogp must be 16-byte aligned.  Workspace:
 * sinkattn_grpo_workspace_size bytes, 16-byte aligned, zero-filled before
 * its first use; every completed call leaves it reusable (its barrier words
 * zero again).  The kernel is one cooperative launch whose CTAs meet at a
 * grid-wide barrier with a bounded wait: if that wait runs out of time the
 * outputs are not written, sinkattn_get_device_status reports TIMEOUT and
 * the workspace must be zero-filled again.
 * Checks: group_size >= 1 dividing num_rollouts, clip_eps > 0, adv_eps >= 0,
 * kl_beta >= 0 (all finite), offsets as for sinkattn_problem. */
typedef struct {
  int32_t num_rollouts;
  int32_t group_size;
  const int32_t* cu_tokens;       /* device [num_rollouts + 1] */
  const int32_t* cu_tokens_host;  /* host copy */
  int32_t total_tokens;
  float clip_eps;
  float adv_eps;
  float kl_beta;
} sinkattn_grpo_problem;
size_t sinkattn_grpo_workspace_size(const sinkattn_grpo_problem* g);
sinkattn_status sinkattn_grpo_loss(const sinkattn_grpo_problem* g, const float* logp, const float* logp_old,
                                   const float* logp_ref, const uint8_t* mask, const float* rewards,
                                   float* stats, float* dlogp, float* advantages,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Packed-sequence front end (multi-turn trajectories of different lengths,
 * SinkFlex-RL section 3).  seqlens: device int32 [num_seqs];
 * cu_seqlens_out: device int32 [num_seqs + 1] receives the exclusive prefix
 * sum (cu[0] = 0).  Fails with INVALID_ARG for num_seqs < 0 or null pointers.
 * A negative length is clamped to 0 on the device. */
sinkattn_status sinkattn_varlen_plan(const int32_t* seqlens, int32_t num_seqs, int32_t* cu_seqlens_out,
                                     void* stream);

/* Padded <-> packed copies of a bf16 [*, H, D] tensor.
 * pack:   padded [B, Smax, H, D] -> packed [cu[B], H, D] (rows past each length are skipped).
 * unpack: packed -> padded; padding rows of `padded` are written with zeros.
 * cu_seqlens is the device copy of the offsets; each length must be <= Smax
 * (rows beyond Smax are not copied).  H * D * 2 bytes must be a multiple of 16. */
sinkattn_status sinkattn_pack(const void* padded, const int32_t* cu_seqlens, int32_t B, int32_t Smax,
                              int32_t H, int32_t D, void* packed, void* stream);
sinkattn_status sinkattn_unpack(const void* packed, const int32_t* cu_seqlens, int32_t B, int32_t Smax,
                                int32_t H, int32_t D, void* padded, void* stream);

/* Synchronises `stream`, then reads and clears the library's device status
 * word: SINKATTN_OK, or SINKATTN_ERR_TIMEOUT when a kernel gave up a bounded
 * wait since the last call (its outputs are then undefined). */
sinkattn_status sinkattn_get_device_status(void* stream);

/* Measurement hook.  kind 1 selects the forward attention kernel, kind 2
 * the backward main kernel, kind 3 the key-chunk kernel of the decode
 * forward (the warp-MMA kernel for at most 16 rows per (sequence, kv head),
 * the tensor-core kernel above).  With non-NULL `start` and `stop` (cudaEvent_t handles passed as
 * void*), every later sinkattn_fwd / sinkattn_bwd / sinkattn_decode_fwd call
 * records `start` on its stream immediately before that kernel's launch and
 * `stop` immediately after it, so the caller can time the kernel alone with
 * cudaEventElapsedTime.  NULL for both clears the hook.  The setting is
 * process-wide and not thread-safe; the events must outlive the calls.
 * Returns INVALID_ARG for an unknown kind or a half-NULL pair. */
sinkattn_status sinkattn_set_profile_events(int32_t kind, void* start, void* stop);

/* Self-test of the bounded waits the kernels use: launches one CTA that
 * waits on an mbarrier nothing ever arrives on, giving up after
 * `limit_cycles` SM cycles (1 .. 2e9) exactly as a kernel's wait does on a
 * timeout.  Afterwards sinkattn_get_device_status() reports
 * SINKATTN_ERR_TIMEOUT once.  Nothing faults or hangs; the context stays
 * usable.  INVALID_ARG for a limit out of range. */
sinkattn_status sinkattn_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/* Static, human-readable name of a status. */
const char* sinkattn_status_string(sinkattn_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t sinkattn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SINKATTN_H */
