// Internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rlk {

// What the forward saves per row for the backward (the ABI's rlk_row_state,
// 32 bytes).  With c = log2(e) / T:
//   q_i = 2^(z_i c - E) / e^lz for i in S, and S = { i : key(z_i) > key_thr }
//   plus the first `ties` ids (ascending) with key(z_i) == key_thr (all of
//   them when ties == kTiesAll).  key is the order-preserving key of the
//   logits' own type (16-bit for bf16, 32-bit for fp32).
struct RowState {
  float E, lz, H;
  uint32_t key_thr, ties, flags;   // flags: kState* bits | row status << 8
  int32_t kstar;
  float temperature;   // the row's own, when the forward took per-row temperatures; else 0
};
static_assert(sizeof(RowState) == 32, "rlk_row_state is 32 bytes");
constexpr uint32_t kStateValid = 1u;   // the forward finished the row
constexpr uint32_t kStateYIn = 2u;     // the selected token is in S
constexpr uint32_t kTiesAll = 0xFFFFFFFFu;

struct LpeArgs {
  const void* logits;
  int dtype;  // 0 bf16, 1 fp32
  int64_t T, V, ld;
  const int32_t* ids;
  float temperature, top_p;
  float* out_logprob;
  float* out_entropy;
  int32_t* out_k;
  uint32_t* status;
  int only_marked;  // per-row kernel: process only rows whose out_logprob holds a recompute mark
  RowState* state;  // [T] or NULL
  // per-row sampling parameters (NULL: the scalars above for every row)
  const float* temps = nullptr;
  const float* top_ps = nullptr;
};

struct LpeBwdArgs {
  const void* logits;
  int dtype;  // 0 bf16, 1 fp32
  int64_t T, V, ld;
  const int32_t* ids;
  float temperature;
  const RowState* state;
  const float* grad_logprob;   // [T] or NULL
  const float* grad_entropy;   // [T] or NULL
  void* grad_logits;           // [T, ldg]
  int grad_dtype;              // 0 bf16, 1 fp32
  int64_t ldg;
  uint32_t* status;
};

// Quiet-NaN payloads that no arithmetic produces: the streaming kernel leaves
// one in out_logprob for each row that the per-row kernel must recompute --
// the second for a row whose speculative window held too little mass, which
// the per-row kernel then scores in its guaranteed window at once.
constexpr uint32_t kRecomputeMark = 0x7FC0DEADu;
constexpr uint32_t kRecomputeMarkWide = 0x7FC0DEAEu;

struct SupportArgs {
  const void* logits;
  int dtype;  // 0 bf16, 1 fp32
  int64_t T, V, ld;
  const int32_t* ids;
  float temperature;
  const int64_t* offsets;   // [T + 1]
  const int32_t* support;   // [offsets[T]]
  float* out_logprob;
  float* out_entropy;
  uint32_t* status;
  // backward only
  const float* grad_logprob;   // [T] or NULL
  const float* grad_entropy;   // [T] or NULL
  float* grad_support;         // [offsets[T]]
};

struct LossArgs {
  const float *logp_new, *logp_old, *logp_rollout, *logp_ref;
  const uint8_t* mask;
  const float* rewards;
  const int32_t* seq_offsets;
  int32_t n_seq, group_size;
  int64_t n_tok;
  float eps_low, eps_high, tis_cap, kl_coef;
  int agg;
  int loss_type = 0;     // rlk_loss_type
  int is_method = 1;     // rlk_is_method (TIS in rlk_grpo_loss)
  int baseline = 0;      // rlk_baseline
  float ipo_eps = 0.f, band_low = 0.f, band_high = 0.f;
  int nstats = 8;        // slots of out_stats the caller provides
  float* out_loss;
  float* out_grad;
  float* out_stats;
  float* workspace;  // per-sequence partial sums + a few scalars
};

struct LmheadArgs {
  const void* hidden;
  const void* w_vocab;
  int64_t T, H, V;
  const int32_t* ids;
  float temperature;
  float* out_logprob;
  float* out_entropy;
  uint32_t* status;
  void* workspace;
  float* out_lse = nullptr;   // [T] ln sum exp(z / T), for the backward
  float top_p = 1.0f;         // < 1: the chunked path (launch_lmhead_topp)
};

struct LmheadBwdArgs {
  const void* hidden;          // bf16 [T, H]
  const void* w_vocab;         // bf16 [V, H]
  int64_t T, H, V;
  const int32_t* ids;
  float temperature;
  const float* lse;            // [T] from the forward
  const float* entropy;        // [T] from the forward
  const float* grad_logprob;   // [T] or NULL
  const float* grad_entropy;   // [T] or NULL
  float* grad_hidden;          // fp32 [T, H]
  float* grad_w;               // fp32 [V, H]
  int accumulate_w;
  void* workspace;
  size_t workspace_bytes;
};

// Canonical vocabulary partition (vocab_parallel.cu).  Shard s of the
// partition covers global columns [s W, (s + 1) W) clipped to V; a call
// handles n_shards adjacent shards starting at global column first_col, whose
// columns are logits[:, 0 ...] (row stride ld).  partials: 32 bytes per
// (shard, row), [n_shards][T].
struct ShardArgs {
  const void* logits;
  int dtype;
  int64_t T, V, ld, first_col, shard_width;
  int n_shards;
  const int32_t* ids;
  float temperature;
  void* partials;
  // supplied retained set (shard_support_partial_kernel): CSR over global ids
  const int64_t* offsets = nullptr;
  const int32_t* support = nullptr;
};
struct ShardCombineArgs {
  const void* partials;   // [n_shards][T], canonical order, shard 0 first
  int n_shards;
  int64_t T, V, shard_width;
  const int32_t* ids;
  float temperature;
  float* out_logprob;
  float* out_entropy;
  uint32_t* status;
  // top_p < 1: the shards' window counts ([n_shards][T], same order)
  const void* counts = nullptr;
  float top_p = 1.0f;
  int32_t* out_k = nullptr;
};
struct ShardWindowArgs {
  const void* logits;     // bf16: this rank's columns
  int64_t T, V, ld, first_col, shard_width;
  int n_shards;           // this rank's shards
  const int32_t* ids;
  float temperature, top_p;
  const void* all_partials;   // [n_all][T]: every shard's partial, canonical order
  int n_all;
  void* counts;           // [n_shards][T]
};
struct SampleArgs {
  const void* logits;   // bf16
  int64_t T, V, ld;
  float temperature;
  const RowState* state;
  const float* uniforms;
  int32_t* out_ids;
  uint32_t* status;
};
cudaError_t launch_sample(const SampleArgs& a, cudaStream_t stream);
cudaError_t launch_shard_partials(const ShardArgs& a, cudaStream_t stream);
cudaError_t launch_shard_combine(const ShardCombineArgs& a, cudaStream_t stream);
cudaError_t launch_shard_support_partials(const ShardArgs& a, cudaStream_t stream);
cudaError_t launch_shard_window(const ShardWindowArgs& a, cudaStream_t stream);
cudaError_t launch_shard_combine_topp(const ShardCombineArgs& a, cudaStream_t stream);

// Consumes one launch failure injected by rlk_debug_inject_launch_failures.
bool take_injected_failure();

// Number of SMs of the current device (cached per device).
int sm_count();
// Slot 0..63 of the current device for per-device once-only state (kernel
// attributes, occupancy), or -1 (no device / more than 64 devices: the
// callers then redo the work on every call).
int device_slot();

// Launches kernel k as a programmatic dependent of the previous kernel on the
// stream: its launch overlaps that kernel's end, and k calls pdl_wait()
// before it reads anything that kernel wrote.
template <class... KArgs, class... Args>
cudaError_t launch_after(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

cudaError_t launch_logprob_entropy(const LpeArgs& a, cudaStream_t stream);
// Streaming kernel for every bf16 batch of a large vocabulary (lpe_stream.cu).
// wait_limit: clock cycles a device wait may take; withhold: a debug stage
// index the first CTA never issues (-1: none).
bool lpe_stream_eligible(const LpeArgs& a);
cudaError_t launch_lpe_stream(const LpeArgs& a, cudaStream_t stream, long long wait_limit,
                              long long withhold);
// Debug settings of the bounded device waits (rlk_debug.h).
long long debug_wait_limit();       // clock cycles (default about 2^31)
long long debug_take_withheld();    // the stage to withhold in the next launch, or -1
int debug_sampler_mode();           // 1 direct mode (default), 2 direct without its list, 0 radix only

cudaError_t launch_support(const SupportArgs& a, cudaStream_t stream);
cudaError_t launch_logprob_entropy_backward(const LpeBwdArgs& a, cudaStream_t stream);
cudaError_t launch_support_backward(const SupportArgs& a, cudaStream_t stream);

constexpr int kLossPartials = 12;  // floats per sequence in the loss workspace
// Checks rlk_grpo_loss's arguments (all but the workspace) and fills a; returns
// an rlk_status value.  Shared by rlk_grpo_loss and rlk_grpo_loss_noalloc.
int grpo_loss_args(const float* logp_new, const float* logp_old, const float* logp_rollout,
                   const float* logp_ref, const uint8_t* loss_mask, const float* rewards,
                   const int32_t* seq_offsets, int32_t n_seq, int32_t group_size, int64_t n_tok,
                   float eps_low, float eps_high, float tis_cap, float kl_coef, int agg,
                   float* out_loss, float* out_grad, float* out_stats, LossArgs& a);
size_t loss_workspace_bytes(int64_t n_seq);
cudaError_t launch_grpo_loss(const LossArgs& a, cudaStream_t stream);

size_t lmhead_workspace_bytes(int64_t T, int64_t V, int64_t H);
cudaError_t launch_lmhead(const LmheadArgs& a, cudaStream_t stream);
size_t lmhead_bwd_workspace_bytes(int64_t T, int64_t V, int64_t H);
size_t lmhead_topp_workspace_bytes(int64_t T, int64_t V, int64_t H);
cudaError_t launch_lmhead_topp(const LmheadArgs& a, cudaStream_t stream);
cudaError_t launch_lmhead_backward(const LmheadBwdArgs& a, cudaStream_t stream);
// Same, also writing the fp32 logits [T, V] to debug_logits (validation aid).
cudaError_t launch_lmhead_impl(const LmheadArgs& a, float* debug_logits, cudaStream_t stream);

}  // namespace rlk
