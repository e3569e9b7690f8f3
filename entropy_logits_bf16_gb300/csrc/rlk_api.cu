// C ABI of librlk: argument validation, workspace sizes, status strings and
// the launches.  Host-checkable errors return before any CUDA call, so the
// validation paths run without a GPU.

#include <atomic>
#include <cmath>
#include <cstddef>

#include "internal.h"
#include "rlk.h"
#include "rlk_debug.h"

namespace rlk {

int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

int device_slot() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  return dev;
}

}  // namespace rlk

namespace {

bool finite_positive(float x) { return std::isfinite(x) && x > 0.0f; }

}  // namespace

namespace rlk {
// Launch failures injected by rlk_debug_inject_launch_failures: each public
// entry that is about to launch takes one and returns RLK_ERR_CUDA instead.
static std::atomic<int> g_injected_failures{0};
bool take_injected_failure() {
  int n = g_injected_failures.load();
  while (n > 0)
    if (g_injected_failures.compare_exchange_weak(n, n - 1)) return true;
  return false;
}

// Bounded device waits: the limit in clock cycles (about a second at the
// GB300's clocks by default) and a debug stage that the next launch of the
// streaming scorer withholds (rlk_debug_withhold_copy).
constexpr long long kDefaultWaitLimit = 1ll << 31;
static std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
static std::atomic<long long> g_withhold{-1};
long long debug_wait_limit() { return g_wait_limit.load(); }
long long debug_take_withheld() { return g_withhold.exchange(-1); }
// rlk_debug_set_sampler_mode: the ways the sampler may take to a draw
static std::atomic<int> g_sampler_mode{1};
int debug_sampler_mode() { return g_sampler_mode.load(); }

int grpo_loss_args(const float* logp_new, const float* logp_old, const float* logp_rollout,
                   const float* logp_ref, const uint8_t* loss_mask, const float* rewards,
                   const int32_t* seq_offsets, int32_t n_seq, int32_t group_size, int64_t n_tok,
                   float eps_low, float eps_high, float tis_cap, float kl_coef, int agg,
                   float* out_loss, float* out_grad, float* out_stats, LossArgs& a) {
  if (n_seq < 0 || group_size < 1 || n_seq % group_size != 0 || n_tok < 0)
    return RLK_ERR_INVALID_ARG;
  if (!(std::isfinite(eps_low) && eps_low >= 0.0f && std::isfinite(eps_high) && eps_high >= 0.0f))
    return RLK_ERR_INVALID_ARG;
  if (!(std::isfinite(tis_cap) && tis_cap > 0.0f) || !(std::isfinite(kl_coef) && kl_coef >= 0.0f))
    return RLK_ERR_INVALID_ARG;
  if (agg != RLK_AGG_TOKEN_MEAN && agg != RLK_AGG_SEQ_MEAN_TOKEN_MEAN && agg != RLK_AGG_PROMPT_MEAN)
    return RLK_ERR_INVALID_ARG;
  if (!seq_offsets || !out_loss) return RLK_ERR_INVALID_ARG;
  if (n_seq > 0 && (!logp_new || !logp_old || !logp_rollout || !logp_ref || !rewards))
    return RLK_ERR_INVALID_ARG;
  a = LossArgs{};
  a.logp_new = logp_new;
  a.logp_old = logp_old;
  a.logp_rollout = logp_rollout;
  a.logp_ref = logp_ref;
  a.mask = loss_mask;
  a.rewards = rewards;
  a.seq_offsets = seq_offsets;
  a.n_seq = n_seq;
  a.group_size = group_size;
  a.n_tok = n_tok;
  a.eps_low = eps_low;
  a.eps_high = eps_high;
  a.tis_cap = tis_cap;
  a.kl_coef = kl_coef;
  a.agg = agg;
  a.out_loss = out_loss;
  a.out_grad = out_grad;
  a.out_stats = out_stats;
  return RLK_OK;
}
}  // namespace rlk

extern "C" {

int rlk_version(void) { return 100; }

long long rlk_debug_set_wait_limit(long long cycles) {
  return rlk::g_wait_limit.exchange(cycles > 0 ? cycles : rlk::kDefaultWaitLimit);
}

int rlk_debug_withhold_copy(long long stage) {
  rlk::g_withhold.store(stage >= 0 ? stage : -1);
  return 0;
}

int rlk_debug_set_sampler_mode(int mode) {
  return rlk::g_sampler_mode.exchange(mode == 0 || mode == 2 ? mode : 1);
}

const char* rlk_status_string(rlk_status status) {
  switch (status) {
    case RLK_OK: return "ok";
    case RLK_ERR_INVALID_ARG: return "invalid argument";
    case RLK_ERR_UNSUPPORTED: return "unsupported";
    case RLK_ERR_WORKSPACE: return "workspace missing or too small";
    case RLK_ERR_CUDA: return "CUDA error";
    case RLK_ERR_TIMEOUT: return "device wait timed out";
    case RLK_ERR_BAD_INPUT: return "bad input data";
  }
  return "unknown status";
}

size_t rlk_workspace_size(int op, int64_t T, int64_t V, int64_t H) {
  if (T < 0 || V < 0 || H < 0) return 0;
  switch (op) {
    case RLK_OP_LOGPROB_ENTROPY: return 0;
    case RLK_OP_GRPO_LOSS: return rlk::loss_workspace_bytes(V);
    case RLK_OP_LMHEAD: return rlk::lmhead_workspace_bytes(T, V, H);
    case RLK_OP_LMHEAD_BWD: return rlk::lmhead_bwd_workspace_bytes(T, V, H);
    case RLK_OP_LMHEAD_TOPP: return rlk::lmhead_topp_workspace_bytes(T, V, H);
    case RLK_OP_CANONICAL:
      return V < 1 ? 0 : (size_t)V * (size_t)T * sizeof(rlk_shard_partial);
    case RLK_OP_CANONICAL_TOPP:
      return V < 1 ? 0 : (size_t)V * (size_t)T * (sizeof(rlk_shard_partial) + sizeof(rlk_shard_counts));
  }
  return 0;
}

namespace {

rlk_status logprob_entropy_impl(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                int64_t ld, const int32_t* token_ids, float temperature,
                                float top_p, float* out_logprob, float* out_entropy,
                                int32_t* out_nucleus_size, rlk_row_state* out_row_state,
                                bool need_state, uint32_t* out_status_word, rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || ld < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (!(top_p > 0.0f && top_p <= 1.0f)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;   // nothing to read or write; pointers may be NULL
  if (!logits || !token_ids || !out_logprob || !out_entropy) return RLK_ERR_INVALID_ARG;
  if (need_state && !out_row_state) return RLK_ERR_INVALID_ARG;
  const uintptr_t elem = dtype == RLK_BF16 ? 2u : 4u;
  if (reinterpret_cast<uintptr_t>(logits) % elem != 0) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out_row_state) % 16u != 0) return RLK_ERR_INVALID_ARG;
  rlk::LpeArgs a{};
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.ids = token_ids;
  a.temperature = temperature;
  a.top_p = top_p;
  a.out_logprob = out_logprob;
  a.out_entropy = out_entropy;
  a.out_k = out_nucleus_size;
  a.status = out_status_word;
  a.only_marked = 0;
  a.state = reinterpret_cast<rlk::RowState*>(out_row_state);
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_logprob_entropy(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

}  // namespace

rlk_status rlk_logprob_entropy_rows(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                    int64_t ld, const int32_t* token_ids,
                                    const float* temperatures, const float* top_ps,
                                    float* out_logprob, float* out_entropy,
                                    int32_t* out_nucleus_size, rlk_row_state* out_row_state,
                                    uint32_t* out_status_word, rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || ld < V) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!logits || !token_ids || !temperatures || !top_ps || !out_logprob || !out_entropy)
    return RLK_ERR_INVALID_ARG;
  const uintptr_t elem = dtype == RLK_BF16 ? 2u : 4u;
  if (reinterpret_cast<uintptr_t>(logits) % elem != 0 ||
      reinterpret_cast<uintptr_t>(out_row_state) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::LpeArgs a{};
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.ids = token_ids;
  a.temperature = 1.0f;   // placeholders: every row reads its own
  a.top_p = 1.0f;
  a.out_logprob = out_logprob;
  a.out_entropy = out_entropy;
  a.out_k = out_nucleus_size;
  a.status = out_status_word;
  a.only_marked = 0;
  a.state = reinterpret_cast<rlk::RowState*>(out_row_state);
  a.temps = temperatures;
  a.top_ps = top_ps;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_logprob_entropy(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_logprob_entropy(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                               int64_t ld, const int32_t* token_ids, float temperature,
                               float top_p, float* out_logprob, float* out_entropy,
                               int32_t* out_nucleus_size, uint32_t* out_status_word,
                               void* workspace, size_t workspace_bytes, rlk_stream stream) {
  (void)workspace;
  (void)workspace_bytes;
  return logprob_entropy_impl(logits, dtype, T, V, ld, token_ids, temperature, top_p, out_logprob,
                              out_entropy, out_nucleus_size, nullptr, false, out_status_word,
                              stream);
}

rlk_status rlk_logprob_entropy_fwd(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                   int64_t ld, const int32_t* token_ids, float temperature,
                                   float top_p, float* out_logprob, float* out_entropy,
                                   int32_t* out_nucleus_size, rlk_row_state* out_row_state,
                                   uint32_t* out_status_word, rlk_stream stream) {
  return logprob_entropy_impl(logits, dtype, T, V, ld, token_ids, temperature, top_p, out_logprob,
                              out_entropy, out_nucleus_size, out_row_state, true, out_status_word,
                              stream);
}

rlk_status rlk_logprob_entropy_bwd(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                   int64_t ld, const int32_t* token_ids, float temperature,
                                   const rlk_row_state* row_state, const float* grad_logprob,
                                   const float* grad_entropy, void* grad_logits,
                                   rlk_dtype grad_dtype, int64_t ldg, uint32_t* out_status_word,
                                   rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (grad_dtype != RLK_BF16 && grad_dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || ld < V || ldg < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!logits || !token_ids || !row_state || !grad_logits) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % (dtype == RLK_BF16 ? 2u : 4u) != 0 ||
      reinterpret_cast<uintptr_t>(grad_logits) % (grad_dtype == RLK_BF16 ? 2u : 4u) != 0 ||
      reinterpret_cast<uintptr_t>(row_state) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::LpeBwdArgs a;
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.ids = token_ids;
  a.temperature = temperature;
  a.state = reinterpret_cast<const rlk::RowState*>(row_state);
  a.grad_logprob = grad_logprob;
  a.grad_entropy = grad_entropy;
  a.grad_logits = grad_logits;
  a.grad_dtype = grad_dtype == RLK_BF16 ? 0 : 1;
  a.ldg = ldg;
  a.status = out_status_word;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_logprob_entropy_backward(a, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_logprob_entropy_support(const void* logits, rlk_dtype dtype, int64_t T,
                                       int64_t V, int64_t ld, const int32_t* token_ids,
                                       float temperature, const int64_t* support_offsets,
                                       const int32_t* support_ids, float* out_logprob,
                                       float* out_entropy, uint32_t* out_status_word,
                                       rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || ld < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;   // nothing to read or write; pointers may be NULL
  if (!logits || !token_ids || !support_offsets || !out_logprob || !out_entropy)
    return RLK_ERR_INVALID_ARG;
  const uintptr_t elem = dtype == RLK_BF16 ? 2u : 4u;
  if (reinterpret_cast<uintptr_t>(logits) % elem != 0) return RLK_ERR_INVALID_ARG;
  rlk::SupportArgs a{};
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.ids = token_ids;
  a.temperature = temperature;
  a.offsets = support_offsets;
  a.support = support_ids;
  a.out_logprob = out_logprob;
  a.out_entropy = out_entropy;
  a.status = out_status_word;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_support(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_logprob_entropy_support_backward(
    const void* logits, rlk_dtype dtype, int64_t T, int64_t V, int64_t ld,
    const int32_t* token_ids, float temperature, const int64_t* support_offsets,
    const int32_t* support_ids, const float* grad_logprob, const float* grad_entropy,
    float* grad_support, uint32_t* out_status_word, rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || ld < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!logits || !token_ids || !support_offsets || !grad_support) return RLK_ERR_INVALID_ARG;
  const uintptr_t elem = dtype == RLK_BF16 ? 2u : 4u;
  if (reinterpret_cast<uintptr_t>(logits) % elem != 0) return RLK_ERR_INVALID_ARG;
  rlk::SupportArgs a{};
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.ids = token_ids;
  a.temperature = temperature;
  a.offsets = support_offsets;
  a.support = support_ids;
  a.status = out_status_word;
  a.grad_logprob = grad_logprob;
  a.grad_entropy = grad_entropy;
  a.grad_support = grad_support;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_support_backward(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_grpo_loss(const float* logp_new, const float* logp_old,
                         const float* logp_rollout, const float* logp_ref,
                         const uint8_t* loss_mask, const float* rewards,
                         const int32_t* seq_offsets, int32_t n_seq, int32_t group_size,
                         int64_t n_tok, float eps_low, float eps_high, float tis_cap,
                         float kl_coef, rlk_agg agg, float* out_loss,
                         float* out_dloss_dlogp_new, float* out_stats, void* workspace,
                         size_t workspace_bytes, rlk_stream stream) {
  rlk::LossArgs a;
  const int st = rlk::grpo_loss_args(logp_new, logp_old, logp_rollout, logp_ref, loss_mask,
                                     rewards, seq_offsets, n_seq, group_size, n_tok, eps_low,
                                     eps_high, tis_cap, kl_coef, (int)agg, out_loss,
                                     out_dloss_dlogp_new, out_stats, a);
  if (st != RLK_OK) return (rlk_status)st;
  const size_t need = rlk::loss_workspace_bytes(n_seq);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
    return RLK_ERR_WORKSPACE;
  a.workspace = static_cast<float*>(workspace);
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_grpo_loss(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

// The layout the Python binding mirrors (11 four-byte fields).
static_assert(sizeof(rlk_loss_config) == 44, "rlk_loss_config layout");
static_assert(offsetof(rlk_loss_config, is_method) == 24 && offsetof(rlk_loss_config, agg) == 40,
              "rlk_loss_config layout");

rlk_status rlk_policy_loss(const float* logp_new, const float* logp_old,
                           const float* logp_rollout, const float* logp_ref,
                           const uint8_t* loss_mask, const float* rewards,
                           const int32_t* seq_offsets, int32_t n_seq, int32_t group_size,
                           int64_t n_tok, const rlk_loss_config* config, float* out_loss,
                           float* out_dloss_dlogp_new, float* out_stats, void* workspace,
                           size_t workspace_bytes, rlk_stream stream) {
  if (!config) return RLK_ERR_INVALID_ARG;
  const rlk_loss_config c = *config;
  if (c.type != RLK_LOSS_DAPO && c.type != RLK_LOSS_IPO && c.type != RLK_LOSS_ICEPOP)
    return RLK_ERR_INVALID_ARG;
  if (c.is_method != RLK_IS_NONE && c.is_method != RLK_IS_TIS && c.is_method != RLK_IS_MIS)
    return RLK_ERR_INVALID_ARG;
  if (c.baseline != RLK_BASELINE_MEAN && c.baseline != RLK_BASELINE_LENGTH_WEIGHTED)
    return RLK_ERR_INVALID_ARG;
  if (!(std::isfinite(c.ipo_eps) && c.ipo_eps >= 0.0f)) return RLK_ERR_INVALID_ARG;
  if (!(std::isfinite(c.band_low) && std::isfinite(c.band_high) && c.band_low >= 0.0f &&
        c.band_low <= c.band_high))
    return RLK_ERR_INVALID_ARG;
  if (c.is_method == RLK_IS_TIS && !finite_positive(c.is_cap)) return RLK_ERR_INVALID_ARG;
  // The common checks; the cap is checked above only where it is used.
  if (n_seq < 0 || group_size < 1 || n_seq % group_size != 0 || n_tok < 0)
    return RLK_ERR_INVALID_ARG;
  if (!(std::isfinite(c.eps_low) && c.eps_low >= 0.0f && std::isfinite(c.eps_high) &&
        c.eps_high >= 0.0f))
    return RLK_ERR_INVALID_ARG;
  if (!(std::isfinite(c.kl_coef) && c.kl_coef >= 0.0f)) return RLK_ERR_INVALID_ARG;
  if (c.agg != RLK_AGG_TOKEN_MEAN && c.agg != RLK_AGG_SEQ_MEAN_TOKEN_MEAN &&
      c.agg != RLK_AGG_PROMPT_MEAN)
    return RLK_ERR_INVALID_ARG;
  if (!seq_offsets || !out_loss) return RLK_ERR_INVALID_ARG;
  if (n_seq > 0 && (!logp_new || !logp_old || !logp_rollout || !logp_ref || !rewards))
    return RLK_ERR_INVALID_ARG;
  const size_t need = rlk::loss_workspace_bytes(n_seq);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
    return RLK_ERR_WORKSPACE;
  rlk::LossArgs a;
  a.logp_new = logp_new;
  a.logp_old = logp_old;
  a.logp_rollout = logp_rollout;
  a.logp_ref = logp_ref;
  a.mask = loss_mask;
  a.rewards = rewards;
  a.seq_offsets = seq_offsets;
  a.n_seq = n_seq;
  a.group_size = group_size;
  a.n_tok = n_tok;
  a.eps_low = c.eps_low;
  a.eps_high = c.eps_high;
  a.tis_cap = c.is_method == RLK_IS_TIS ? c.is_cap : 1.0f;
  a.kl_coef = c.kl_coef;
  a.agg = c.agg;
  a.loss_type = c.type;
  a.is_method = c.is_method;
  a.baseline = c.baseline;
  a.ipo_eps = c.ipo_eps;
  a.band_low = c.band_low;
  a.band_high = c.band_high;
  a.nstats = RLK_NSTATS_POLICY;
  a.out_loss = out_loss;
  a.out_grad = out_dloss_dlogp_new;
  a.out_stats = out_stats;
  a.workspace = static_cast<float*>(workspace);
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_grpo_loss(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

static_assert(sizeof(rlk_shard_partial) == 32, "rlk_shard_partial is 32 bytes");

rlk_status rlk_shard_partials(const void* logits, rlk_dtype dtype, int64_t T, int64_t V, int64_t ld,
                              int64_t first_col, int64_t shard_width, int32_t n_shards,
                              const int32_t* token_ids, float temperature,
                              rlk_shard_partial* out_partials, rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || shard_width < 1 || n_shards < 1)
    return RLK_ERR_INVALID_ARG;
  if (first_col < 0 || first_col % shard_width != 0) return RLK_ERR_INVALID_ARG;
  const int64_t span = shard_width * (int64_t)n_shards;
  int64_t cols = V - first_col < span ? V - first_col : span;   // shards of padding only: none
  if (cols < 0) cols = 0;
  if (ld < cols) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!logits || !token_ids || !out_partials) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % (dtype == RLK_BF16 ? 2u : 4u) != 0 ||
      reinterpret_cast<uintptr_t>(out_partials) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::ShardArgs a{};
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.first_col = first_col;
  a.shard_width = shard_width;
  a.n_shards = n_shards;
  a.ids = token_ids;
  a.temperature = temperature;
  a.partials = out_partials;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_shard_partials(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_shard_partials_support(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                      int64_t ld, int64_t first_col, int64_t shard_width,
                                      int32_t n_shards, const int32_t* token_ids,
                                      float temperature, const int64_t* support_offsets,
                                      const int32_t* support_ids,
                                      rlk_shard_partial* out_partials, rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || shard_width < 1 || n_shards < 1)
    return RLK_ERR_INVALID_ARG;
  if (first_col < 0 || first_col % shard_width != 0) return RLK_ERR_INVALID_ARG;
  const int64_t span = shard_width * (int64_t)n_shards;
  int64_t cols = V - first_col < span ? V - first_col : span;
  if (cols < 0) cols = 0;
  if (ld < cols) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!logits || !token_ids || !support_offsets || !out_partials) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % (dtype == RLK_BF16 ? 2u : 4u) != 0 ||
      reinterpret_cast<uintptr_t>(out_partials) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::ShardArgs a{};
  a.logits = logits;
  a.dtype = dtype == RLK_BF16 ? 0 : 1;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.first_col = first_col;
  a.shard_width = shard_width;
  a.n_shards = n_shards;
  a.ids = token_ids;
  a.temperature = temperature;
  a.partials = out_partials;
  a.offsets = support_offsets;
  a.support = support_ids;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_shard_support_partials(a, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_shard_combine(const rlk_shard_partial* partials, int32_t n_shards, int64_t T,
                             int64_t V, int64_t shard_width, const int32_t* token_ids,
                             float temperature, float* out_logprob, float* out_entropy,
                             uint32_t* out_status_word, rlk_stream stream) {
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || shard_width < 1 || n_shards < 1)
    return RLK_ERR_INVALID_ARG;
  if (shard_width * (int64_t)n_shards < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!partials || !token_ids || !out_logprob || !out_entropy) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(partials) % 16u != 0) return RLK_ERR_INVALID_ARG;
  rlk::ShardCombineArgs a{};
  a.partials = partials;
  a.n_shards = n_shards;
  a.T = T;
  a.V = V;
  a.shard_width = shard_width;
  a.ids = token_ids;
  a.temperature = temperature;
  a.out_logprob = out_logprob;
  a.out_entropy = out_entropy;
  a.status = out_status_word;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_shard_combine(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_logprob_entropy_canonical(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                         int64_t ld, const int32_t* token_ids, float temperature,
                                         int32_t n_virtual, int64_t padded_vocab,
                                         float* out_logprob, float* out_entropy,
                                         uint32_t* out_status_word, void* workspace,
                                         size_t workspace_bytes, rlk_stream stream) {
  if (n_virtual < 1 || padded_vocab < V || padded_vocab % n_virtual != 0 || ld < V)
    return RLK_ERR_INVALID_ARG;
  if (T > 0 && (!workspace || workspace_bytes < (size_t)n_virtual * (size_t)T * 32u ||
                reinterpret_cast<uintptr_t>(workspace) % 16u != 0))
    return RLK_ERR_WORKSPACE;
  const int64_t W = padded_vocab / n_virtual;
  rlk_shard_partial* part = static_cast<rlk_shard_partial*>(workspace);
  rlk_status st = rlk_shard_partials(logits, dtype, T, V, ld, 0, W, n_virtual, token_ids,
                                     temperature, part, stream);
  if (st != RLK_OK) return st;
  return rlk_shard_combine(part, n_virtual, T, V, W, token_ids, temperature, out_logprob,
                           out_entropy, out_status_word, stream);
}

static_assert(sizeof(rlk_shard_counts) == 8224, "rlk_shard_counts is 8224 bytes");

rlk_status rlk_shard_window_counts(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                   int64_t ld, int64_t first_col, int64_t shard_width,
                                   int32_t n_shards, const int32_t* token_ids, float temperature,
                                   float top_p, const rlk_shard_partial* all_partials,
                                   int32_t n_all, rlk_shard_counts* out_counts, rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || shard_width < 1 || n_shards < 1)
    return RLK_ERR_INVALID_ARG;
  if (first_col < 0 || first_col % shard_width != 0) return RLK_ERR_INVALID_ARG;
  if (n_all < first_col / shard_width + n_shards || shard_width * (int64_t)n_all < V)
    return RLK_ERR_INVALID_ARG;
  const int64_t span = shard_width * (int64_t)n_shards;
  int64_t cols = V - first_col < span ? V - first_col : span;
  if (cols < 0) cols = 0;
  if (ld < cols) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature) || !(top_p > 0.f && top_p < 1.f)) return RLK_ERR_INVALID_ARG;
  if (dtype != RLK_BF16) return RLK_ERR_UNSUPPORTED;
  if (T == 0) return RLK_OK;
  if (!logits || !token_ids || !all_partials || !out_counts) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % 2u != 0 ||
      reinterpret_cast<uintptr_t>(all_partials) % 16u != 0 ||
      reinterpret_cast<uintptr_t>(out_counts) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::ShardWindowArgs a{};
  a.logits = logits;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.first_col = first_col;
  a.shard_width = shard_width;
  a.n_shards = n_shards;
  a.ids = token_ids;
  a.temperature = temperature;
  a.top_p = top_p;
  a.all_partials = all_partials;
  a.n_all = n_all;
  a.counts = out_counts;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_shard_window(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_shard_combine_topp(const rlk_shard_partial* partials, const rlk_shard_counts* counts,
                                  int32_t n_shards, int64_t T, int64_t V, int64_t shard_width,
                                  const int32_t* token_ids, float temperature, float top_p,
                                  float* out_logprob, float* out_entropy, int32_t* out_k,
                                  uint32_t* out_status_word, rlk_stream stream) {
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || shard_width < 1 || n_shards < 1)
    return RLK_ERR_INVALID_ARG;
  if (shard_width * (int64_t)n_shards < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature) || !(top_p > 0.f && top_p < 1.f)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!partials || !counts || !token_ids || !out_logprob || !out_entropy)
    return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(partials) % 16u != 0 ||
      reinterpret_cast<uintptr_t>(counts) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::ShardCombineArgs a{};
  a.partials = partials;
  a.n_shards = n_shards;
  a.T = T;
  a.V = V;
  a.shard_width = shard_width;
  a.ids = token_ids;
  a.temperature = temperature;
  a.out_logprob = out_logprob;
  a.out_entropy = out_entropy;
  a.status = out_status_word;
  a.counts = counts;
  a.top_p = top_p;
  a.out_k = out_k;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_shard_combine_topp(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

rlk_status rlk_logprob_entropy_canonical_topp(const void* logits, rlk_dtype dtype, int64_t T,
                                              int64_t V, int64_t ld, const int32_t* token_ids,
                                              float temperature, float top_p, int32_t n_virtual,
                                              int64_t padded_vocab, float* out_logprob,
                                              float* out_entropy, int32_t* out_k,
                                              uint32_t* out_status_word, void* workspace,
                                              size_t workspace_bytes, rlk_stream stream) {
  if (n_virtual < 1 || padded_vocab < V || padded_vocab % n_virtual != 0 || ld < V)
    return RLK_ERR_INVALID_ARG;
  const size_t part_bytes = (size_t)n_virtual * (size_t)(T > 0 ? T : 0) * sizeof(rlk_shard_partial);
  const size_t need = part_bytes + (size_t)n_virtual * (size_t)(T > 0 ? T : 0) * sizeof(rlk_shard_counts);
  if (T > 0 && (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 16u != 0))
    return RLK_ERR_WORKSPACE;
  const int64_t W = padded_vocab / n_virtual;
  rlk_shard_partial* part = static_cast<rlk_shard_partial*>(workspace);
  rlk_shard_counts* cnt = reinterpret_cast<rlk_shard_counts*>(static_cast<char*>(workspace) + part_bytes);
  rlk_status st = rlk_shard_partials(logits, dtype, T, V, ld, 0, W, n_virtual, token_ids,
                                     temperature, part, stream);
  if (st != RLK_OK) return st;
  st = rlk_shard_window_counts(logits, dtype, T, V, ld, 0, W, n_virtual, token_ids, temperature,
                               top_p, part, n_virtual, cnt, stream);
  if (st != RLK_OK) return st;
  return rlk_shard_combine_topp(part, cnt, n_virtual, T, V, W, token_ids, temperature, top_p,
                                out_logprob, out_entropy, out_k, out_status_word, stream);
}

rlk_status rlk_sample_top_p(const void* logits, rlk_dtype dtype, int64_t T, int64_t V, int64_t ld,
                            float temperature, const rlk_row_state* row_state,
                            const float* uniforms, int32_t* out_ids, uint32_t* out_status_word,
                            rlk_stream stream) {
  if (dtype != RLK_BF16 && dtype != RLK_F32) return RLK_ERR_INVALID_ARG;
  if (T < 0 || V < 1 || V > (int64_t(1) << 24) || ld < V) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (dtype != RLK_BF16) return RLK_ERR_UNSUPPORTED;
  if (T == 0) return RLK_OK;
  if (!logits || !row_state || !uniforms || !out_ids) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % 2u != 0 ||
      reinterpret_cast<uintptr_t>(row_state) % 16u != 0)
    return RLK_ERR_INVALID_ARG;
  rlk::SampleArgs a{};
  a.logits = logits;
  a.T = T;
  a.V = V;
  a.ld = ld;
  a.temperature = temperature;
  a.state = reinterpret_cast<const rlk::RowState*>(row_state);
  a.uniforms = uniforms;
  a.out_ids = out_ids;
  a.status = out_status_word;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  return rlk::launch_sample(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? RLK_OK
             : RLK_ERR_CUDA;
}

static rlk_status lmhead_common(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                int64_t V, const int32_t* token_ids, float temperature,
                                float top_p, float* out_logits, float* out_logprob,
                                float* out_entropy, float* out_lse, uint32_t* out_status_word,
                                void* workspace, size_t workspace_bytes, rlk_stream stream) {
  if (T < 0 || H < 64 || H % 64 != 0 || V < 1 || V > (int64_t(1) << 24)) return RLK_ERR_INVALID_ARG;
  if (T > (int64_t(1) << 30) || H > (int64_t(1) << 20)) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (!(top_p > 0.0f && top_p <= 1.0f)) return RLK_ERR_INVALID_ARG;
  if (!hidden || !w_vocab || !token_ids || !out_logprob || !out_entropy) return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(hidden) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(w_vocab) % 16 != 0)
    return RLK_ERR_INVALID_ARG;
  const bool topp = top_p != 1.0f;
  if (topp && (out_logits || out_lse)) return RLK_ERR_UNSUPPORTED;   // top_p = 1 only
  const size_t need = topp ? rlk::lmhead_topp_workspace_bytes(T, V, H)
                           : rlk::lmhead_workspace_bytes(T, V, H);
  if (need > 0 && (!workspace || workspace_bytes < need ||
                   reinterpret_cast<uintptr_t>(workspace) % 16 != 0))
    return RLK_ERR_WORKSPACE;
  if (T == 0) return RLK_OK;
  rlk::LmheadArgs a;
  a.hidden = hidden;
  a.w_vocab = w_vocab;
  a.T = T;
  a.H = H;
  a.V = V;
  a.ids = token_ids;
  a.temperature = temperature;
  a.out_logprob = out_logprob;
  a.out_entropy = out_entropy;
  a.status = out_status_word;
  a.workspace = workspace;
  a.out_lse = out_lse;
  a.top_p = top_p;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  const cudaError_t e =
      topp ? rlk::launch_lmhead_topp(a, reinterpret_cast<cudaStream_t>(stream))
           : rlk::launch_lmhead_impl(a, out_logits, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return RLK_ERR_UNSUPPORTED;
  return e == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

rlk_status rlk_lmhead_logprob(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                              int64_t V, const int32_t* token_ids, float temperature,
                              float top_p, float* out_logprob, float* out_entropy,
                              uint32_t* out_status_word, void* workspace,
                              size_t workspace_bytes, rlk_stream stream) {
  return lmhead_common(hidden, w_vocab, T, H, V, token_ids, temperature, top_p, nullptr,
                       out_logprob, out_entropy, nullptr, out_status_word, workspace,
                       workspace_bytes, stream);
}

rlk_status rlk_lmhead_logprob_fwd(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                  int64_t V, const int32_t* token_ids, float temperature,
                                  float top_p, float* out_logprob, float* out_entropy,
                                  float* out_lse, uint32_t* out_status_word, void* workspace,
                                  size_t workspace_bytes, rlk_stream stream) {
  if (T > 0 && !out_lse) return RLK_ERR_INVALID_ARG;
  return lmhead_common(hidden, w_vocab, T, H, V, token_ids, temperature, top_p, nullptr,
                       out_logprob, out_entropy, out_lse, out_status_word, workspace,
                       workspace_bytes, stream);
}

rlk_status rlk_lmhead_logprob_bwd(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                  int64_t V, const int32_t* token_ids, float temperature,
                                  const float* lse, const float* entropy,
                                  const float* grad_logprob, const float* grad_entropy,
                                  float* grad_hidden, float* grad_w, int accumulate_grad_w,
                                  void* workspace, size_t workspace_bytes, rlk_stream stream) {
  if (T < 0 || H < 64 || H % 64 != 0 || V < 1 || V > (int64_t(1) << 24)) return RLK_ERR_INVALID_ARG;
  if (T > (int64_t(1) << 30) || H > (int64_t(1) << 20)) return RLK_ERR_INVALID_ARG;
  if (!finite_positive(temperature)) return RLK_ERR_INVALID_ARG;
  if (T == 0) return RLK_OK;
  if (!hidden || !w_vocab || !token_ids || !lse || !entropy || !grad_hidden || !grad_w)
    return RLK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(hidden) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(w_vocab) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(grad_hidden) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(grad_w) % 16 != 0)
    return RLK_ERR_INVALID_ARG;
  const size_t need = rlk::lmhead_bwd_workspace_bytes(T, V, H);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return RLK_ERR_WORKSPACE;
  rlk::LmheadBwdArgs a;
  a.hidden = hidden;
  a.w_vocab = w_vocab;
  a.T = T;
  a.H = H;
  a.V = V;
  a.ids = token_ids;
  a.temperature = temperature;
  a.lse = lse;
  a.entropy = entropy;
  a.grad_logprob = grad_logprob;
  a.grad_entropy = grad_entropy;
  a.grad_hidden = grad_hidden;
  a.grad_w = grad_w;
  a.accumulate_w = accumulate_grad_w != 0;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  if (rlk::take_injected_failure()) return RLK_ERR_CUDA;
  const cudaError_t e =
      rlk::launch_lmhead_backward(a, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return RLK_ERR_UNSUPPORTED;
  return e == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

int rlk_debug_inject_launch_failures(int n) {
  return rlk::g_injected_failures.exchange(n < 0 ? 0 : n);
}

rlk_status rlk_lmhead_logits_debug(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                   int64_t V, const int32_t* token_ids, float temperature,
                                   float* out_logits, float* out_logprob, float* out_entropy,
                                   uint32_t* out_status_word, void* workspace,
                                   size_t workspace_bytes, rlk_stream stream) {
  if (!out_logits) return RLK_ERR_INVALID_ARG;
  return lmhead_common(hidden, w_vocab, T, H, V, token_ids, temperature, 1.0f, out_logits,
                       out_logprob, out_entropy, nullptr, out_status_word, workspace,
                       workspace_bytes, stream);
}

}  // extern "C"
