// Parameters handed from the C-ABI layer to the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace sa {

constexpr int kHeadDim = 64;
constexpr int kMaxHeadsQ = 256;

// Problem after validation and normalisation (see sinkattn_api.cu).
struct Problem {
  int num_seqs;
  int seqlen;              // uniform length, or the longest packed sequence
  const int32_t* cu;       // device offsets or nullptr (uniform batch)
  const int32_t* cu_host;  // host offsets or nullptr
  int total_tokens;
  int hq, hkv;
  int window;              // -1 = unbounded (any w >= seqlen - 1 is folded into -1)
  int prefix;              // clamped to [0, seqlen]
  int causal;
  float scale;
};

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* sink;
  void* o;
  float* lse;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  const float* sink;
  void* dq;
  void* dk;
  void* dv;
  float* dsink;
  // workspace carve-up
  float* dq_accum;    // [T, Hq, 64] fp32
  // [Hq, T, 8] bf16 per (head, token): -l'/scale and -D (l' = l + softplus(sink - l),
  // D = <dO, O>), each as three bf16 summands (hi, mid, lo), then two zeros;
  // the main kernel adds them to S^T and dP^T through one K=16 MMA.
  void* bias;
  float* dsink_part;  // [preprocess blocks, Hq]
  float* dkv_acc;     // fp32 dK/dV partial sums of split key tiles, one slot per chunk (or nullptr)
  int* unit_counters; // one claim counter per main-kernel launch, cleared by the preprocess kernel
  int n_unit_counters;
  int preprocess_blocks;
};

// Preprocess tokens per block (bounds the number of dsink partial rows).
constexpr int kPreTokens = 8;

// Streaming multiprocessors of the current device, cached per device; 152
// (a GB300) when no device answers, so that host-side plans and the
// workspace sizes they imply are the same with or without a GPU.
int device_sms();

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// One backward work item: key tile `kt` of sequence `b`, query chunk `chunk`
// of `nchunks`.  When nchunks > 1 the item's partial dK/dV go to fp32 slot
// `slot` of the workspace (one slot per chunk; the chunks of one tile hold
// consecutive slots, chunk c at slot - chunk + c), and a conversion pass
// sums a tile's slots in chunk order, so the result does not depend on the
// order in which the chunks ran.
struct BwdItem {
  uint16_t b, kt, chunk, nchunks;
  uint32_t slot;
};

// Work lists (schedule.cu), longest first.
std::vector<uint32_t> fwd_work_list(const Problem& p);  // b | (query tile << 16)
int bwd_qchunk(const Problem& p);
// Query tiles the key tiles of all sequences see (the backward's steps per kv
// head and query head).
long long bwd_query_tiles_total(const Problem& p);
std::vector<BwdItem> bwd_work_list(const Problem& p, int qchunk);
// Partial-sum slots the items of a list use (items with nchunks > 1).
int bwd_split_slots(const std::vector<BwdItem>& items);

// Decode forward (decode.cu): the last n query rows of each sequence against
// its whole key/value history, split over the keys and merged afterwards.
constexpr int kDecodeMaxItems = 4096;  // (sequence, key chunk) items per launch

struct DecodeArgs {
  const void* q;  // [B * n, Hq, 64]
  const void* k;  // [T_kv, Hkv, 64]
  const void* v;
  const float* sink;
  void* o;        // [B * n, Hq, 64]
  float* lse;     // [Hq, B * n]
  float* ws_acc;   // partial unnormalised outputs
  void* ws_ml;     // per partial and row: (max, sum for O, sum for lse, 0) as float4
  int* counters;   // chunks finished per (sequence, kv head); zero between calls
};

struct DecodePlan {
  bool tensor_core = false;      // the tcgen05 kernel (else the warp-MMA one)
  int tiles_per_split = 0;
  std::vector<uint32_t> items;   // sequence | (chunk << 16), sequence-major
  size_t acc_bytes = 0, ml_bytes = 0, counter_bytes = 0;
};

DecodePlan decode_plan(const Problem& p, int n);
cudaError_t launch_decode(const Problem& p, int n, const DecodeArgs& a, const DecodePlan& pl, int* status,
                          cudaStream_t s);

// GRPO token loss (grpo.cu).
struct GrpoArgs {
  int num_rollouts, group_size, total_tokens;
  const int32_t* cu_tokens;  // device [num_rollouts + 1]
  float clip_eps, adv_eps, kl_beta;
  const float* logp;
  const float* logp_old;
  const float* logp_ref;
  const uint8_t* mask;
  const float* rewards;
  float* stats;       // [4]
  float* dlogp;
  float* advantages;  // or nullptr
  void* workspace;   // barrier words zero on entry (left zero on exit)
  int* status;        // library status word (the grid barrier's bounded wait)
};
size_t grpo_workspace_bytes(int num_rollouts, int total_tokens);
cudaError_t launch_grpo(const GrpoArgs& a, cudaStream_t s);

// Optional events recorded around the main kernels (measurement hook).
struct ProfileEvents {
  cudaEvent_t start = nullptr, stop = nullptr;
};
extern ProfileEvents g_prof_fwd, g_prof_bwd, g_prof_dec;

inline cudaError_t prof_begin(const ProfileEvents& e, cudaStream_t s) {
  return e.start ? cudaEventRecord(e.start, s) : cudaSuccess;
}
inline cudaError_t prof_end(const ProfileEvents& e, cudaStream_t s) {
  return e.stop ? cudaEventRecord(e.stop, s) : cudaSuccess;
}

cudaError_t launch_fwd_tc(const Problem& p, const FwdArgs& a, int* status, cudaStream_t s);
// Kernel launches launch_fwd_tc / launch_bwd_tc_main make for a problem (host arithmetic).
int fwd_tc_launches(const Problem& p);
// Launches of launch_bwd_tc_main: the main kernel's work-list slices and the
// conversion pass.
int bwd_tc_main_launches(const Problem& p);
int bwd_tc_main_slices(const Problem& p);  // launches of the main kernel itself (work-list slices)
cudaError_t launch_bwd(const Problem& p, const BwdArgs& a, int* status, cudaStream_t s);
cudaError_t launch_bwd_tc_main(const Problem& p, const BwdArgs& a, int* status, cudaStream_t s);
size_t bwd_split_acc_bytes(const Problem& p);
cudaError_t launch_varlen_plan(const int32_t* seqlens, int n, int32_t* cu, cudaStream_t s);
cudaError_t launch_pack(const void* src, const int32_t* cu, int B, int Smax, int H, int D, void* dst, bool unpack,
                        cudaStream_t s);

}  // namespace sa
