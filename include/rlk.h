/*
 * rlk.h -- C ABI of librlk: top-p log-probability / entropy of sampled tokens,
 * the GRPO/DAPO loss epilogue, and a fused LM-head variant, for one GB300 GPU.
 *
 * Conventions shared by every entry point
 *  - All pointers are DEVICE pointers unless stated otherwise; scalars are
 *    passed by value.  The caller owns every buffer.  The library never
 *    allocates, frees or synchronises; all work is enqueued on `stream`
 *    (a cudaStream_t; NULL means the legacy default stream).
 *  - Host-checkable argument errors return before any launch and leave every
 *    output untouched.  A failed launch returns RLK_ERR_CUDA.
 *  - Data errors found on the device (a token id outside [0, V), a non-finite
 *    logit) do not abort: the affected row's outputs become NaN and a bit is
 *    OR-ed into *out_status_word (when given); the caller reads it back.
 *  - Results are deterministic: bitwise identical across runs and independent
 *    of how rows are batched (row count, row order, position in the batch).
 *
 * The pages this implements give semantics, not formulas:
 *  - RL-Kernel "Qwen3-8B VIME train-rollout consistency", section "ROCm MI300X
 *    and gfx942": temperature finite and positive; top-p in (0,1]; the
 *    complete retained top-p set with no support cap; top-k and temperature 0
 *    rejected, not ignored; top-p < 1 is scored by the sparse logp /
 *    monitoring-entropy fusion over the retained support, top-p = 1 by the
 *    full-vocabulary strict scorer.
 *  - RL-Kernel "ROCm sparse performance" notes: temperature, softmax, sort and
 *    top-p thresholding keep the sampler's native semantics; train and rollout
 *    log-probabilities must be bitwise equal (fixed reduction order); GRPO
 *    uses standard-deviation normalisation; KL coefficient 0.01.
 *  - LumenRL README, section "Rollout Correction": truncated importance
 *    sampling clips large ratios.
 *  - prime-rl v0.10.0 release notes, section "1. Trainer Performance": the
 *    loss is chunked so full logits need not exist at once.
 */
#ifndef RLK_H_
#define RLK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* same type as cudaStream_t */
typedef struct CUstream_st* rlk_stream;

typedef enum {
  RLK_OK = 0,
  RLK_ERR_INVALID_ARG = 1,   /* a host-checkable argument is invalid          */
  RLK_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. a mode)       */
  RLK_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required    */
  RLK_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed          */
  RLK_ERR_TIMEOUT = 5,       /* reserved: a bounded device wait ran out       */
  RLK_ERR_BAD_INPUT = 6      /* reserved for host-visible data errors         */
} rlk_status;

typedef enum { RLK_BF16 = 0, RLK_F32 = 1 } rlk_dtype;

typedef enum {
  RLK_AGG_TOKEN_MEAN = 0,            /* sum(mask * l) / sum(mask) over the batch (DAPO) */
  RLK_AGG_SEQ_MEAN_TOKEN_MEAN = 1,   /* mean over sequences of each sequence's token mean */
  RLK_AGG_PROMPT_MEAN = 2            /* mean over groups (prompts) of each group's token mean */
} rlk_agg;

/* Policy term of rlk_policy_loss (prime-rl v0.10.0 release notes, section
 * "2. RL Algorithms"). */
typedef enum {
  RLK_LOSS_DAPO = 0,     /* clipped ratio pi_new / pi_old, DAPO clip-higher      */
  RLK_LOSS_IPO = 1,      /* -rho A on tokens with |pi_new - pi_rollout| <= ipo_eps */
  RLK_LOSS_ICEPOP = 2    /* the DAPO term on tokens with rho in the band         */
} rlk_loss_type;

/* Rollout correction weight (LumenRL README, section "Rollout Correction"). */
typedef enum {
  RLK_IS_NONE = 0,       /* w = 1                                                */
  RLK_IS_TIS = 1,        /* w = min(pi_old / pi_rollout, is_cap)                 */
  RLK_IS_MIS = 2         /* w = (pi_old / pi_rollout) / its mean over the batch  */
} rlk_is_method;

/* GRPO advantage baseline. */
typedef enum {
  RLK_BASELINE_MEAN = 0,             /* the group's mean reward                    */
  RLK_BASELINE_LENGTH_WEIGHTED = 1   /* rewards weighted by packed sequence length */
} rlk_baseline;

/* Operation ids for rlk_workspace_size. */
enum { RLK_OP_LOGPROB_ENTROPY = 0, RLK_OP_GRPO_LOSS = 1, RLK_OP_LMHEAD = 2,
       RLK_OP_LMHEAD_BWD = 3, RLK_OP_LMHEAD_TOPP = 4, RLK_OP_CANONICAL = 5,
       RLK_OP_CANONICAL_TOPP = 6 };

/* Bits OR-ed into *out_status_word by the kernels. */
#define RLK_STATUS_BAD_TOKEN_ID 0x1u   /* a token id outside [0, V)          */
#define RLK_STATUS_NONFINITE    0x2u   /* a NaN or +-inf logit in a row      */
#define RLK_STATUS_TIMEOUT      0x4u   /* a bounded device wait ran out; the
                                          rows the kernel had not finished
                                          get NaN outputs (rows finished
                                          before it are valid)              */
#define RLK_STATUS_BAD_SUPPORT  0x8u   /* a supplied retained set that is empty,
                                          lists an id outside [0, V), or whose
                                          offsets decrease                      */
#define RLK_STATUS_NO_STATE     0x10u  /* a row state that no forward wrote
                                          (rlk_logprob_entropy_bwd)           */
#define RLK_STATUS_UNRESOLVED   0x40u  /* rlk_shard_combine_topp: a row whose
                                          window spans more than 4096 values,
                                          whose nucleus boundary falls among the
                                          logits with |z| < 2^-12, or with more
                                          than 65535 equal logits in one shard's
                                          window (NaN outputs)                 */
#define RLK_STATUS_BAD_PARAM    0x20u  /* a per-row temperature that is not
                                          finite and > 0, or a per-row top_p
                                          outside (0, 1]                      */

/* What rlk_logprob_entropy_fwd saves per row for rlk_logprob_entropy_bwd:
 * the row's log-normaliser over its retained set, its entropy and where the
 * set's boundary lies (a value and how many of the ids tied at it are kept).
 * Opaque, 32 bytes, 16-byte aligned in an array of T. */
typedef struct rlk_row_state {
  uint32_t opaque[8];
} rlk_row_state;

/* Slots of the loss statistics vector (float [RLK_NSTATS]); fractions and
 * means are over tokens with mask = 1. */
enum {
  RLK_STAT_LOSS = 0,          /* the loss value                                 */
  RLK_STAT_TOKENS = 1,        /* sum of the mask                                */
  RLK_STAT_CLIP_LOW = 2,      /* fraction with A < 0 and r < 1 - eps_low        */
  RLK_STAT_CLIP_HIGH = 3,     /* fraction with A > 0 and r > 1 + eps_high       */
  RLK_STAT_TIS_MEAN = 4,      /* mean truncated importance weight               */
  RLK_STAT_TIS_CAPPED = 5,    /* fraction whose weight hit the cap              */
  RLK_STAT_K3_MEAN = 6,       /* mean k3 KL estimate                            */
  RLK_STAT_PG_MEAN = 7,       /* mean clipped policy-gradient term              */
  RLK_NSTATS = 8,
  RLK_STAT_MASK_DROPPED = 8,  /* rlk_policy_loss: fraction dropped by the IPO /
                                 IcePop mask                                    */
  RLK_NSTATS_POLICY = 9
};

/* Library version (major * 10000 + minor * 100 + patch). */
int rlk_version(void);

/* Static, NUL-terminated description of a status code; never NULL. */
const char* rlk_status_string(rlk_status status);

/* Bytes of device workspace one call of `op` needs.  Arguments per op:
 *  RLK_OP_LOGPROB_ENTROPY: T rows, V vocabulary, H unused      -> 0
 *  RLK_OP_GRPO_LOSS:       T packed tokens, V = n_seq, H unused
 *  RLK_OP_LMHEAD:          T rows, V vocabulary, H hidden size
 *  RLK_OP_LMHEAD_BWD:      the same (rlk_lmhead_logprob_bwd)
 *  RLK_OP_LMHEAD_TOPP:     the same (rlk_lmhead_logprob with top_p < 1)
 *  RLK_OP_CANONICAL:       T rows, V = the number of virtual shards, H unused
 *  RLK_OP_CANONICAL_TOPP:  the same (rlk_logprob_entropy_canonical_topp)
 * Returns 0 for an unknown op or negative sizes. */
size_t rlk_workspace_size(int op, int64_t T, int64_t V, int64_t H);

/*
 * rlk_logprob_entropy -- per-token top-p log-probability and entropy.
 *
 * For each row t of logits[T, ld] (elements; ld >= V; row-major) with
 * selected token y = token_ids[t]:
 *   x_i = z_i / temperature;  m = max x;  w_i = exp(x_i - m);
 *   rank tokens by (z descending, id ascending), -0 equal to +0;
 *   k* = V if top_p == 1, else the least k whose prefix mass reaches top_p
 *        (sum of w over the first k ranked tokens >= top_p * sum of all w);
 *   S = the first k* ranked tokens (the retained set), Z_S = sum_S w;
 *   out_logprob[t] = (x_y - m) - ln Z_S if y in S, else -INFINITY;
 *   out_entropy[t] = Shannon entropy (nats) of w / Z_S over S;
 *   out_nucleus_size[t] = k*.
 * (The pages fix neither the retained-set rule nor the tie order; this library
 *  keeps a token while the mass ranked strictly ahead of it is < top_p -- the
 *  sampler's cumulative rule -- and keeps equal logits lower id first.)
 *
 * Arguments
 *  logits          device, dtype `dtype`, T x ld elements; base 2-byte (bf16)
 *                  or 4-byte (fp32) aligned.  Read only.
 *  dtype           RLK_BF16 or RLK_F32 (top_p < 1 with fp32 logits takes a
 *                  slower exact path).
 *  T, V, ld        rows, vocabulary size (1 <= V <= 2^24), row stride.
 *  token_ids       device int32[T].
 *  temperature     finite, > 0.   top_p: 0 < top_p <= 1.
 *  out_logprob     device float[T].   out_entropy: device float[T].
 *  out_nucleus_size  device int32[T] or NULL.
 *  out_status_word device uint32[1] or NULL; bits RLK_STATUS_* are OR-ed in.
 *  workspace, workspace_bytes  unused (0 bytes required); may be NULL/0.
 *  stream          CUDA stream.
 * Errors: RLK_ERR_INVALID_ARG for T < 0, V < 1, V > 2^24, ld < V, null
 *  required pointers, a bad dtype, a non-finite or non-positive temperature,
 *  top_p outside (0,1].  T == 0 returns RLK_OK without launching (pointers
 *  may then be NULL).
 */
rlk_status rlk_logprob_entropy(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                               int64_t ld, const int32_t* token_ids, float temperature,
                               float top_p, float* out_logprob, float* out_entropy,
                               int32_t* out_nucleus_size, uint32_t* out_status_word,
                               void* workspace, size_t workspace_bytes, rlk_stream stream);

/*
 * rlk_logprob_entropy_fwd -- rlk_logprob_entropy that also saves, per row,
 * what the backward needs.
 *
 * Outputs and errors as rlk_logprob_entropy, plus
 *  out_row_state   device rlk_row_state[T] (required).  Row t's state is
 *                  written once the row is finished; a row with a status
 *                  gets a state that marks it so.
 */
rlk_status rlk_logprob_entropy_fwd(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                   int64_t ld, const int32_t* token_ids, float temperature,
                                   float top_p, float* out_logprob, float* out_entropy,
                                   int32_t* out_nucleus_size, rlk_row_state* out_row_state,
                                   uint32_t* out_status_word, rlk_stream stream);

/*
 * rlk_logprob_entropy_rows -- rlk_logprob_entropy_fwd with sampling parameters
 * per row.
 *
 * The pages' samplers have no fixed sampling parameter (RL-Kernel "ROCm
 * sparse performance" notes) and test per-row top-p: a batch may mix
 * requests.  Row t uses temperatures[t] and top_ps[t]; c = log2(e) / T and
 * 1 / T are formed per row exactly as the scalar call forms them, so rows
 * with equal parameters give the scalar call's results on the same kernel
 * (at top_p = 1 the entropy numerator is summed in another order: equal
 * within rounding).
 * These rows run on the per-row kernel (the cluster-resident kernel is for
 * one parameter pair per call).
 *
 * Arguments as rlk_logprob_entropy_fwd, with
 *  temperatures, top_ps  device float[T] (required).
 *  out_row_state   device rlk_row_state[T] or NULL; a state records its row's
 *                  temperature, which rlk_logprob_entropy_bwd and
 *                  rlk_sample_top_p then use for that row.
 * A row whose temperature is not finite and > 0 or whose top_p lies outside
 * (0, 1] gets NaN outputs and RLK_STATUS_BAD_PARAM.
 */
rlk_status rlk_logprob_entropy_rows(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                    int64_t ld, const int32_t* token_ids,
                                    const float* temperatures, const float* top_ps,
                                    float* out_logprob, float* out_entropy,
                                    int32_t* out_nucleus_size, rlk_row_state* out_row_state,
                                    uint32_t* out_status_word, rlk_stream stream);

/*
 * rlk_logprob_entropy_bwd -- gradient of the top-p log-probability and
 * entropy with respect to the logits.
 *
 * RL-Kernel "Qwen3-8B VIME train-rollout consistency", section "ROCm MI300X
 * and gfx942": top-p < 1 rows are scored over the complete retained set S,
 * renormalised.  S changes only where a logit crosses its boundary, so
 * almost everywhere it is locally constant and the gradient is that of the
 * softmax restricted to S at temperature T.  For
 *   L = sum_t grad_logprob[t] logprob_t + grad_entropy[t] H_t
 * and q_i = exp(x_i - m) / Z_S over S (as in rlk_logprob_entropy):
 *   grad_logits[t, i] = 0                                         (i not in S)
 *   grad_logits[t, i] = (grad_logprob[t] ([i = y] - q_i) [y in S]
 *                        - grad_entropy[t] q_i (ln q_i + H_t)) / T   (i in S).
 * S is the one the forward selected (ties at the boundary kept lower id
 * first), read from the saved row state.
 *
 * Arguments
 *  logits, dtype, T, V, ld, token_ids, temperature
 *                  the forward's (same values, same contents); a row whose
 *                  state recorded its own temperature (rlk_logprob_entropy_rows)
 *                  uses that one.
 *  row_state       device rlk_row_state[T] from rlk_logprob_entropy_fwd.
 *  grad_logprob    device float[T] or NULL (zero).
 *  grad_entropy    device float[T] or NULL (zero).
 *  grad_logits     device, grad_dtype, T x ldg elements (ldg >= V); every
 *                  element of columns [0, V) is written; NaN for a row whose
 *                  state carries a status (or that no forward wrote).
 *  grad_dtype      RLK_BF16 (rounded to nearest) or RLK_F32.
 *  out_status_word device uint32[1] or NULL: the status bits the forward found
 *                  for rows it could not score, RLK_STATUS_BAD_TOKEN_ID for an
 *                  id outside [0, V), RLK_STATUS_NO_STATE for a state no
 *                  forward wrote.
 *  stream          CUDA stream.
 * Errors: RLK_ERR_INVALID_ARG for T < 0, V < 1, V > 2^24, ld < V, ldg < V,
 *  null required pointers, bad dtypes, a misaligned logits, gradient or state
 *  base, a non-finite or non-positive temperature.  T == 0 returns RLK_OK.
 */
rlk_status rlk_logprob_entropy_bwd(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                   int64_t ld, const int32_t* token_ids, float temperature,
                                   const rlk_row_state* row_state, const float* grad_logprob,
                                   const float* grad_entropy, void* grad_logits,
                                   rlk_dtype grad_dtype, int64_t ldg, uint32_t* out_status_word,
                                   rlk_stream stream);

/*
 * rlk_logprob_entropy_support -- per-token log-probability and entropy over a
 * retained set supplied by the sampler.
 *
 * The sparse path of RL-Kernel "Qwen3-8B VIME train-rollout consistency",
 * section "ROCm MI300X and gfx942", scores the complete retained support the
 * sampler produced rather than recomputing it.  Row t keeps exactly the ids
 * listed in support_ids[support_offsets[t] .. support_offsets[t+1]) (a CSR
 * layout; any order; an id listed twice counts twice):
 *   x_i = z_i / temperature over the listed ids;  m_S = max x;
 *   Z_S = sum exp(x_i - m_S) over the list;
 *   out_logprob[t] = (x_y - m_S) - ln Z_S if y is listed, else -INFINITY;
 *   out_entropy[t] = Shannon entropy (nats) of exp(x - m_S) / Z_S over the list.
 * Only the listed ids' logits are read.  With the list set to the top-p
 * retained set, the outputs equal rlk_logprob_entropy's.
 *
 * Arguments
 *  logits          device, dtype `dtype`, T x ld elements, as for
 *                  rlk_logprob_entropy.  Read only.
 *  T, V, ld        rows, vocabulary size (1 <= V <= 2^24), row stride.
 *  token_ids       device int32[T].
 *  temperature     finite, > 0.
 *  support_offsets device int64[T + 1], nondecreasing (checked per row on the
 *                  device).
 *  support_ids     device int32[support_offsets[T]] (may be NULL when every
 *                  row's list is empty, which is a data error per row).
 *  out_logprob, out_entropy  device float[T].
 *  out_status_word device uint32[1] or NULL.  A row whose selected id is out
 *                  of range (RLK_STATUS_BAD_TOKEN_ID), whose list is empty,
 *                  lists an id out of range or whose offsets decrease
 *                  (RLK_STATUS_BAD_SUPPORT), or whose listed logits include
 *                  a NaN or +-inf (RLK_STATUS_NONFINITE) gets NaN outputs.
 *  stream          CUDA stream.
 * Errors: RLK_ERR_INVALID_ARG for T < 0, V < 1, V > 2^24, ld < V, a bad
 *  dtype, a non-finite or non-positive temperature, or a null required
 *  pointer.  T == 0 returns RLK_OK without launching.
 */
rlk_status rlk_logprob_entropy_support(const void* logits, rlk_dtype dtype, int64_t T,
                                       int64_t V, int64_t ld, const int32_t* token_ids,
                                       float temperature, const int64_t* support_offsets,
                                       const int32_t* support_ids, float* out_logprob,
                                       float* out_entropy, uint32_t* out_status_word,
                                       rlk_stream stream);

/*
 * rlk_logprob_entropy_support_backward -- gradient of the supplied-support
 * scorer with respect to the listed logits.
 *
 * The backward of rlk_logprob_entropy_support with each row's retained set
 * held fixed (the sampler chose it; RL-Kernel "Qwen3-8B VIME train-rollout
 * consistency", section "ROCm MI300X and gfx942", scores that set), for the
 * loss L = sum_t grad_logprob[t] logprob_t + grad_entropy[t] H_t:
 *   q_i = exp(x_i - m_S) / Z_S over the listed ids (as in the forward);
 *   grad_support[j] = dL/dz_i for i = support_ids[j]
 *     = grad_logprob[t] ([i = y] - q_i) / T     (0 when y is not listed)
 *       - grad_entropy[t] q_i (ln q_i + H_t) / T.
 * Unlisted ids have zero gradient and are not written.
 *
 * Arguments: as rlk_logprob_entropy_support, plus
 *  grad_logprob    device float[T] or NULL (all zero).
 *  grad_entropy    device float[T] or NULL (all zero).
 *  grad_support    device float[support_offsets[T]], aligned with
 *                  support_ids; overwritten for every list position of every
 *                  row (NaN for a row with a status).
 * Errors: as rlk_logprob_entropy_support; grad_support may not be NULL.
 */
rlk_status rlk_logprob_entropy_support_backward(
    const void* logits, rlk_dtype dtype, int64_t T, int64_t V, int64_t ld,
    const int32_t* token_ids, float temperature, const int64_t* support_offsets,
    const int32_t* support_ids, const float* grad_logprob, const float* grad_entropy,
    float* grad_support, uint32_t* out_status_word, rlk_stream stream);

/*
 * rlk_grpo_loss -- fused GRPO/DAPO loss with TIS correction and k3 KL.
 *
 * Sequences are packed: sequence s holds tokens [seq_offsets[s], seq_offsets[s+1]),
 * and groups are contiguous runs of group_size sequences (GRPO groups of
 * responses to one prompt; RL-Kernel "ROCm sparse performance" notes: GRPO
 * standard-deviation normalisation).  Per group g with rewards R:
 *   A_s = (R_s - mean_g R) / (std_g R + 1e-6), std with the n-1 divisor (0 when G = 1).
 * Per token t of sequence s (mask m_t, 1 when loss_mask is NULL):
 *   r = exp(logp_new - logp_old);
 *   pg = -min(r A_s, clip(r, 1 - eps_low, 1 + eps_high) A_s)      (DAPO clip-higher);
 *   w = min(exp(logp_old - logp_rollout), tis_cap)                 (TIS; LumenRL
 *        README "Rollout Correction"), a detached weight on pg only;
 *   d = logp_ref - logp_new; k3 = exp(d) - d - 1;
 *   l_t = w pg + kl_coef k3.
 * Aggregation RLK_AGG_TOKEN_MEAN: L = sum m l / sum m (0 if sum m = 0).
 * RLK_AGG_SEQ_MEAN_TOKEN_MEAN: L = mean over sequences with sum m > 0 of
 *   that sequence's token mean.  RLK_AGG_PROMPT_MEAN: the same over groups.
 * Gradient (if out_dloss_dlogp_new): dL/dlogp_new[t] = (weight of t in L) *
 *   (w g_pg + kl_coef (1 - exp(d))), g_pg = -r A when the unclipped term is
 *   the active minimum (ties count as unclipped), else 0.
 *
 * Arguments
 *  logp_new, logp_old, logp_rollout, logp_ref  device float arrays indexed by the
 *                  packed token position t, seq_offsets[0] <= t < seq_offsets[0] + n_tok
 *                  (seq_offsets[0] may be > 0: pass the base of the packed batch).
 *  loss_mask       device uint8[n_tok] (0/1) or NULL for all ones.
 *  rewards         device float[n_seq].
 *  seq_offsets     device int32[n_seq + 1], non-decreasing and within
 *                  [seq_offsets[0], seq_offsets[0] + n_tok] (checked on the device:
 *                  otherwise every sequence's range is clamped to the n_tok tokens, no
 *                  token outside them is read or written, and the loss, the
 *                  statistics and the gradient come out NaN).
 *  n_seq, group_size  n_seq >= 0, group_size >= 1, n_seq % group_size == 0.
 *  eps_low, eps_high  >= 0 and finite; tis_cap > 0; kl_coef >= 0 and finite.
 *  agg             an rlk_agg value.
 *  n_tok           number of packed tokens (seq_offsets[n_seq] - seq_offsets[0]): the
 *                  extent of the per-token arrays and of the gradient.
 *  out_loss        device float[1].
 *  out_dloss_dlogp_new  device float[n_tok] or NULL.
 *  out_stats       device float[RLK_NSTATS] or NULL.
 *  workspace       device scratch of at least rlk_workspace_size(RLK_OP_GRPO_LOSS, n_tok,
 *                  n_seq, 0) bytes, 16-byte aligned; its contents on entry do not matter.
 */
rlk_status rlk_grpo_loss(const float* logp_new, const float* logp_old,
                         const float* logp_rollout, const float* logp_ref,
                         const uint8_t* loss_mask, const float* rewards,
                         const int32_t* seq_offsets, int32_t n_seq, int32_t group_size,
                         int64_t n_tok, float eps_low, float eps_high, float tis_cap,
                         float kl_coef, rlk_agg agg, float* out_loss,
                         float* out_dloss_dlogp_new, float* out_stats, void* workspace,
                         size_t workspace_bytes, rlk_stream stream);

/*
 * rlk_policy_loss -- rlk_grpo_loss with the pages' loss variants.
 *
 * prime-rl v0.10.0 release notes, section "2. RL Algorithms": IPO masks a
 * token whose probability moved too much between the inference engine and the
 * trainer, |pi_train(y) - pi_infer(y)| > eps (eps 0.3, no KL term); IcePop
 * masks a token whose ratio pi_train / pi_infer leaves a fixed band; GRPO gains
 * a length-weighted baseline and prompt-mean aggregation.  LumenRL README,
 * section "Rollout Correction": TIS clips large importance ratios, MIS
 * normalises them.  With pi_train(y) = exp(logp_new), pi_infer(y) =
 * exp(logp_rollout), r = exp(new - old), rho = exp(new - rollout),
 * raw = exp(old - rollout):
 *   A_s = (R_s - b_g) / (std_g R + 1e-6), b_g the group mean or, with
 *     RLK_BASELINE_LENGTH_WEIGHTED, sum_j len_j R_j / sum_j len_j over the
 *     group (len_j = seq_offsets[j+1] - seq_offsets[j]; the plain mean when the
 *     group is empty); std as in rlk_grpo_loss;
 *   RLK_LOSS_DAPO:   pg = -min(r A, clip(r, 1 - eps_low, 1 + eps_high) A);
 *   RLK_LOSS_IPO:    keep = [|exp(new) - exp(rollout)| <= ipo_eps],
 *                    pg = -keep rho A (no clipping; d pg / d new = pg);
 *   RLK_LOSS_ICEPOP: keep = [band_low <= rho <= band_high], pg = keep x the
 *                    DAPO term;
 *   w = 1 (RLK_IS_NONE), min(raw, is_cap) (TIS), raw / mean over mask-1
 *     tokens of raw (MIS), a detached weight on pg;
 *   l_t = w pg + kl_coef k3 (the pages' IPO setting uses kl_coef = 0);
 *   aggregation and gradient as in rlk_grpo_loss, the mask value held fixed.
 * (The pages give only the IPO mask as a formula; the surrogates, MIS and the
 *  length weights above are this library's readings.)
 *
 * Arguments: as rlk_grpo_loss, with the scalars in *config (a host pointer,
 *  read before the call returns) and
 *  out_stats       device float[RLK_NSTATS_POLICY] or NULL (slot
 *                  RLK_STAT_MASK_DROPPED: the fraction of mask-1 tokens the
 *                  IPO / IcePop mask drops; RLK_STAT_TIS_MEAN: mean w).
 *  workspace       as rlk_grpo_loss (rlk_workspace_size(RLK_OP_GRPO_LOSS, ...)).
 * Errors: as rlk_grpo_loss, plus RLK_ERR_INVALID_ARG for a NULL config, an
 *  unknown type / method / baseline / aggregation, ipo_eps not finite and
 *  >= 0, a band that is not finite with 0 <= band_low <= band_high, or (TIS)
 *  is_cap not finite and > 0.
 */
typedef struct rlk_loss_config {
  rlk_loss_type type;
  float eps_low, eps_high;      /* DAPO / IcePop clip bounds                    */
  float ipo_eps;                /* IPO mask threshold                           */
  float band_low, band_high;    /* IcePop band on rho                           */
  rlk_is_method is_method;
  float is_cap;                 /* TIS cap                                      */
  float kl_coef;
  rlk_baseline baseline;
  rlk_agg agg;
} rlk_loss_config;

rlk_status rlk_policy_loss(const float* logp_new, const float* logp_old,
                           const float* logp_rollout, const float* logp_ref,
                           const uint8_t* loss_mask, const float* rewards,
                           const int32_t* seq_offsets, int32_t n_seq, int32_t group_size,
                           int64_t n_tok, const rlk_loss_config* config, float* out_loss,
                           float* out_dloss_dlogp_new, float* out_stats, void* workspace,
                           size_t workspace_bytes, rlk_stream stream);

/* Largest n_seq that rlk_grpo_loss_noalloc accepts. */
#define RLK_NOALLOC_MAX_SEQ 16384

/*
 * rlk_grpo_loss_noalloc -- rlk_grpo_loss for callers that cannot allocate
 * device memory (the pages have no counterpart): a framework that has
 * reserved the whole device for its own pool, code running inside an
 * allocator callback, or a latency-critical loop that bans cudaMalloc because
 * it may synchronise the device.  The caller passes inputs and outputs only.
 *
 * Scratch: a static device array of RLK_NOALLOC_MAX_SEQ * 12 + 4 floats
 * (about 768 KB) inside the library, held by every GPU that loads the library
 * until the process exits.  The first call on each device looks up the
 * array's device address (with that device current) and caches it for the
 * life of the process; make that first call before any stream capture.  A
 * cudaDeviceReset of that device frees the array behind the cached address:
 * do not call this entry point on a device after resetting it.  Every call overwrites what it reads, so nothing
 * needs clearing, and the array keeps the last call's contents.  All calls
 * share the array: calls whose work overlaps on the GPU (different streams or
 * host threads) race and give wrong results -- serialise them.
 *
 * Arguments, semantics and results: as rlk_grpo_loss without the workspace.
 * Errors: as rlk_grpo_loss; n_seq > RLK_NOALLOC_MAX_SEQ returns
 * RLK_ERR_INVALID_ARG; a failed address lookup returns RLK_ERR_CUDA.  Never
 * calls cudaMalloc, cudaFree or any allocating routine.
 */
rlk_status rlk_grpo_loss_noalloc(const float* logp_new, const float* logp_old,
                                 const float* logp_rollout, const float* logp_ref,
                                 const uint8_t* loss_mask, const float* rewards,
                                 const int32_t* seq_offsets, int32_t n_seq, int32_t group_size,
                                 int64_t n_tok, float eps_low, float eps_high, float tis_cap,
                                 float kl_coef, rlk_agg agg, float* out_loss,
                                 float* out_dloss_dlogp_new, float* out_stats, rlk_stream stream);

/*
 * rlk_lmhead_logprob -- the logits path fused with the LM-head GEMM.
 *
 * top_p = 1: logits = hidden[T, H] * w_vocab[V, H]^T are produced tile by
 * tile in tensor-core accumulators and folded into the online max / sum /
 * entropy state; they never reach memory (prime-rl v0.10.0 notes, "1. Trainer
 * Performance": chunked loss; RL-Kernel notes: deterministic GEMM with a
 * fixed reduction order).  Logits are the fp32 accumulations, not rounded
 * to bf16.
 * top_p < 1: the nucleus needs all of a row's logits at once, so the same GEMM
 * emits the logits of at most 4096 rows at a time, rounded to bf16 (the
 * scorer's input type, as an unfused LM head would emit them), into the
 * workspace, and rlk_logprob_entropy scores each chunk there.
 *
 * Arguments
 *  hidden          device bf16 [T, H] row-major, 16-byte aligned.
 *  w_vocab         device bf16 [V, H] row-major, 16-byte aligned.
 *  T, H, V         T >= 0, H a positive multiple of 64, V >= 1.
 *  token_ids       device int32[T].
 *  temperature     finite, > 0.   top_p: 0 < top_p <= 1.
 *  out_logprob, out_entropy  device float[T].
 *  out_status_word device uint32[1] or NULL.
 *  workspace       at least rlk_workspace_size(RLK_OP_LMHEAD, T, V, H) bytes
 *                  (RLK_OP_LMHEAD_TOPP when top_p < 1), 16-byte aligned;
 *                  contents on entry do not matter.
 */
rlk_status rlk_lmhead_logprob(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                              int64_t V, const int32_t* token_ids, float temperature,
                              float top_p, float* out_logprob, float* out_entropy,
                              uint32_t* out_status_word, void* workspace,
                              size_t workspace_bytes, rlk_stream stream);

/*
 * rlk_lmhead_logprob_fwd -- rlk_lmhead_logprob that also writes each row's
 * log-normaliser for the backward.
 *
 * Arguments and errors as rlk_lmhead_logprob, plus
 *  out_lse         device float[T] (required): ln sum_v exp(z_v / T) over the
 *                  row's fp32 logits z (NaN for a row with a status).
 * top_p must be 1 (else RLK_ERR_UNSUPPORTED): the backward is the top_p = 1
 * path's.
 */
rlk_status rlk_lmhead_logprob_fwd(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                  int64_t V, const int32_t* token_ids, float temperature,
                                  float top_p, float* out_logprob, float* out_entropy,
                                  float* out_lse, uint32_t* out_status_word, void* workspace,
                                  size_t workspace_bytes, rlk_stream stream);

/*
 * rlk_lmhead_logprob_bwd -- gradients of the fused LM-head path with respect
 * to hidden and w_vocab.
 *
 * For L = sum_t grad_logprob[t] logprob_t + grad_entropy[t] H_t and
 * z = hidden w_vocab^T (fp32 accumulations of the bf16 inputs), q_v =
 * exp(z_v / T - lse_t):
 *   dz[t, v] = (grad_logprob[t] ([v = y_t] - q_v) - grad_entropy[t] q_v (ln q_v + H_t)) / T,
 *   grad_hidden = dz w_vocab,   grad_w (+)= dz^T hidden.
 * dz is recomputed by the same tensor-core GEMM as the forward, 4096 rows at a
 * time, rounded to bf16 and kept in the workspace (so the gradient logits of at
 * most 4096 rows exist at once: prime-rl v0.10.0 notes, "1. Trainer
 * Performance", the chunked loss); the two weight-side products are tcgen05
 * GEMMs of the library's own (bf16 inputs, fp32 accumulation and outputs, each
 * tile's K in order).  Deterministic for a given T: grad_w sums the chunks in
 * order.
 *
 * Arguments
 *  hidden, w_vocab, T, H, V, token_ids, temperature  the forward's.
 *  lse, entropy    device float[T] from rlk_lmhead_logprob_fwd.
 *  grad_logprob, grad_entropy  device float[T] or NULL (zero).
 *  grad_hidden     device float[T, H] row-major, overwritten.
 *  grad_w          device float[V, H] row-major; overwritten, or added to when
 *                  accumulate_grad_w is non-zero.
 *  workspace       at least rlk_workspace_size(RLK_OP_LMHEAD_BWD, T, V, H)
 *                  bytes (the gradient logits of 4096 rows: 4096 x V bf16),
 *                  16-byte aligned.
 * A row whose lse is NaN (a row the forward could not score) gives NaN in its
 * grad_hidden row and in all of grad_w.
 * Errors: as rlk_lmhead_logprob; RLK_ERR_INVALID_ARG for a NULL lse, entropy,
 *  grad_hidden or grad_w.
 */
rlk_status rlk_lmhead_logprob_bwd(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                  int64_t V, const int32_t* token_ids, float temperature,
                                  const float* lse, const float* entropy,
                                  const float* grad_logprob, const float* grad_entropy,
                                  float* grad_hidden, float* grad_w, int accumulate_grad_w,
                                  void* workspace, size_t workspace_bytes, rlk_stream stream);

/*
 * rlk_sample_top_p -- deterministic top-p sampling.
 *
 * For each row, the id at which the cumulative renormalised probability over
 * the retained set S, taken in ranking order (logit descending, id
 * ascending), first reaches uniforms[t]: the first j in that order with
 * sum_{i <= j} w_i >= u Z_S (RL-Kernel "Qwen3-8B VIME train-rollout
 * consistency", section "ROCm MI300X and gfx942": the sampler's native
 * temperature / softmax / sort / top-p semantics; "ROCm sparse performance"
 * notes: deterministic top-p sampling).  S is the set the forward selected,
 * read from the row state of rlk_logprob_entropy_fwd (whose token_ids do not
 * affect it).  No sort: a radix descent on the 16-bit key of the bf16 logits
 * with exact fixed-point masses (w 2^40, truncated: tokens below 2^-40 of the
 * row maximum count with mass 0), then a scan in id order for the tie.
 *
 * Arguments
 *  logits, T, V, ld, temperature  as the forward's (a row whose state
 *                  recorded its own temperature uses that one); dtype RLK_BF16
 *                  only (RLK_F32: RLK_ERR_UNSUPPORTED).
 *  row_state       device rlk_row_state[T] from rlk_logprob_entropy_fwd.
 *  uniforms        device float[T], each in [0, 1) (clamped).
 *  out_ids         device int32[T]; -1 for a row whose state carries a status.
 *  out_status_word device uint32[1] or NULL (the state's status bits, or
 *                  RLK_STATUS_NO_STATE).
 */
rlk_status rlk_sample_top_p(const void* logits, rlk_dtype dtype, int64_t T, int64_t V, int64_t ld,
                            float temperature, const rlk_row_state* row_state,
                            const float* uniforms, int32_t* out_ids, uint32_t* out_status_word,
                            rlk_stream stream);

/*
 * The canonical vocabulary partition (top_p = 1).
 *
 * RL-Kernel "Qwen3-8B VIME train-rollout consistency", section "Canonical
 * topology strategy": a fixed virtual tensor-parallel degree of 8 and a padded
 * vocabulary of 152576 for every physical topology; a physical rank executes
 * its adjacent virtual shards separately and the shards are combined in the
 * same fixed order (the selected-token log-probability included), so a
 * topology change moves no reduction boundary.  Shard s covers vocabulary
 * columns [s W, (s + 1) W), W = padded_vocab / n_virtual, clipped to V (the
 * padding holds no logits).  The result equals rlk_logprob_entropy's at
 * top_p = 1 within the parity tolerance, and is bitwise the same whatever the
 * number of ranks the shards are spread over.
 */
#define RLK_CANONICAL_TP 8
#define RLK_CANONICAL_VOCAB 152576

/* One row's summary of one shard: its max, sum of exponentials and entropy
 * numerator, and the selected logit when the selected id is in the shard.
 * Opaque, 32 bytes. */
typedef struct rlk_shard_partial {
  float opaque[8];
} rlk_shard_partial;

/*
 * rlk_shard_partials -- the partials of n_shards adjacent shards.
 *
 * Arguments
 *  logits          device bf16 or fp32: the columns of shards first_col / W ..
 *                  first_col / W + n_shards - 1, i.e. global columns
 *                  [first_col, min(first_col + n_shards W, V)), row-major with
 *                  row stride ld (elements).
 *  T, V            rows; the full (unpadded) vocabulary size.
 *  first_col       global index of the first shard's first column, a multiple
 *                  of W (shards wholly in the padding get empty partials).
 *  shard_width     W.
 *  token_ids       device int32[T] (global ids).
 *  out_partials    device rlk_shard_partial[n_shards][T] (shard-major), 16-byte
 *                  aligned.
 * Errors: RLK_ERR_INVALID_ARG for T < 0, V < 1, W < 1, n_shards < 1, a
 *  first_col outside the rules above, ld below the columns given, a bad dtype,
 *  null pointers, a non-finite or non-positive temperature.
 */
rlk_status rlk_shard_partials(const void* logits, rlk_dtype dtype, int64_t T, int64_t V, int64_t ld,
                              int64_t first_col, int64_t shard_width, int32_t n_shards,
                              const int32_t* token_ids, float temperature,
                              rlk_shard_partial* out_partials, rlk_stream stream);

/*
 * rlk_shard_partials_support -- rlk_shard_partials over a retained set
 * supplied by the sampler (CSR, as rlk_logprob_entropy_support): the top_p < 1
 * rows of the pages' sparse path under the canonical partition.  Each shard
 * folds the listed ids that fall in its columns; combined by
 * rlk_shard_combine, the result is rlk_logprob_entropy_support's, and
 * bitwise the same for any number of ranks.  Every shard checks the row's
 * list (empty, decreasing offsets, an id outside [0, V)) and the combine
 * reports RLK_STATUS_BAD_SUPPORT for it; a selected id that is not listed
 * gives a log-probability of -inf.
 *
 * Arguments as rlk_shard_partials, plus support_offsets (device int64[T + 1])
 * and support_ids (device int32[support_offsets[T]], global ids; may be NULL
 * only when every row's list is empty, which is a data error per row).
 */
rlk_status rlk_shard_partials_support(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                      int64_t ld, int64_t first_col, int64_t shard_width,
                                      int32_t n_shards, const int32_t* token_ids,
                                      float temperature, const int64_t* support_offsets,
                                      const int32_t* support_ids,
                                      rlk_shard_partial* out_partials, rlk_stream stream);

/*
 * rlk_shard_combine -- log-probability and entropy from all shards' partials,
 * merged in shard order.
 *
 *  partials        device rlk_shard_partial[n_shards][T], shard 0 first (the
 *                  ranks' outputs gathered in rank order).
 *  n_shards, shard_width  with n_shards W >= V.
 * Data errors as rlk_logprob_entropy (NaN outputs, RLK_STATUS_BAD_TOKEN_ID or
 * RLK_STATUS_NONFINITE), plus the status bits the partials carry
 * (RLK_STATUS_BAD_SUPPORT from rlk_shard_partials_support).
 */
rlk_status rlk_shard_combine(const rlk_shard_partial* partials, int32_t n_shards, int64_t T,
                             int64_t V, int64_t shard_width, const int32_t* token_ids,
                             float temperature, float* out_logprob, float* out_entropy,
                             uint32_t* out_status_word, rlk_stream stream);

/*
 * rlk_logprob_entropy_canonical -- the whole canonical path on one device:
 * rlk_shard_partials over all n_virtual shards (padded_vocab / n_virtual
 * wide) into the workspace, then rlk_shard_combine.
 *
 *  workspace       rlk_workspace_size(RLK_OP_CANONICAL, T, n_virtual, 0) bytes,
 *                  16-byte aligned.
 * Errors: as the two calls; padded_vocab must be >= V and a multiple of
 *  n_virtual.
 */
rlk_status rlk_logprob_entropy_canonical(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                         int64_t ld, const int32_t* token_ids, float temperature,
                                         int32_t n_virtual, int64_t padded_vocab,
                                         float* out_logprob, float* out_entropy,
                                         uint32_t* out_status_word, void* workspace,
                                         size_t workspace_bytes, rlk_stream stream);

/*
 * The canonical partition at top_p < 1, no retained set supplied.
 *
 * The retained set depends on the whole row, so the ranks exchange twice.
 * (1) rlk_shard_partials on every rank, gathered in rank order: every rank
 * now holds all shards' partials, hence the row's max m and Z.  (2)
 * rlk_shard_window_counts: from those every shard derives the same window
 * z >= m - L T, L = ln(V / ((1 - top_p) Z)) + 0.5 (Z relative to the max's
 * weight) -- below it lies less than V e^-L < (1 - top_p) Z of the mass, so
 * the nucleus boundary lies inside -- and counts its logits in the window per
 * bf16 value (all logits of one value carry the same mass; the values with
 * |z| < 2^-12 share one bin whose mass the shard sums in a fixed order),
 * gathered in rank order too.  (3) rlk_shard_combine_topp adds the counts
 * (integers: exact in any order), scans the bins largest value first with a
 * fixed-order double-float prefix to the bin where the retained mass reaches
 * top_p Z (tied logits kept lower id first, as rlk_logprob_entropy) and
 * writes the log-probability of the selected token under the renormalised
 * retained distribution (-inf when it is not retained) and the retained set's
 * entropy.  The result is bitwise the same for any number of ranks, and within
 * the parity tolerance of rlk_logprob_entropy.  bf16 logits only.
 */

/* One row's window counts of one shard.  Opaque, 8224 bytes. */
typedef struct rlk_shard_counts {
  uint32_t opaque[2056];
} rlk_shard_counts;

/*
 * rlk_shard_window_counts -- step (2) above for this rank's n_shards shards.
 *
 *  logits          device bf16, the columns of this rank's shards (as
 *                  rlk_shard_partials).
 *  T, V, ld, first_col, shard_width, n_shards, token_ids, temperature
 *                  as rlk_shard_partials.
 *  top_p           in (0, 1).
 *  all_partials    device rlk_shard_partial[n_all][T]: every shard's partial,
 *                  shard 0 first (rlk_shard_partials of all ranks gathered in
 *                  rank order), 16-byte aligned.
 *  out_counts      device rlk_shard_counts[n_shards][T] (shard-major),
 *                  16-byte aligned.
 * Errors: as rlk_shard_partials, RLK_ERR_UNSUPPORTED for fp32 logits,
 *  RLK_ERR_INVALID_ARG for top_p outside (0, 1) or n_all < first_col / W +
 *  n_shards.  Rows with a bad id or a non-finite logit are left to the
 *  combine, which reports them.
 */
rlk_status rlk_shard_window_counts(const void* logits, rlk_dtype dtype, int64_t T, int64_t V,
                                   int64_t ld, int64_t first_col, int64_t shard_width,
                                   int32_t n_shards, const int32_t* token_ids, float temperature,
                                   float top_p, const rlk_shard_partial* all_partials,
                                   int32_t n_all, rlk_shard_counts* out_counts, rlk_stream stream);

/*
 * rlk_shard_combine_topp -- step (3): log-probability, entropy and nucleus
 * size from all shards' partials and window counts (both [n_shards][T], shard
 * 0 first).
 *
 *  out_k           device int32[T] or NULL: the retained set's size.
 * Data errors: NaN outputs (k = 0) with RLK_STATUS_BAD_TOKEN_ID,
 *  RLK_STATUS_NONFINITE or RLK_STATUS_UNRESOLVED in the status word.
 * Errors: as rlk_shard_combine, RLK_ERR_INVALID_ARG for top_p outside (0, 1).
 */
rlk_status rlk_shard_combine_topp(const rlk_shard_partial* partials, const rlk_shard_counts* counts,
                                  int32_t n_shards, int64_t T, int64_t V, int64_t shard_width,
                                  const int32_t* token_ids, float temperature, float top_p,
                                  float* out_logprob, float* out_entropy, int32_t* out_k,
                                  uint32_t* out_status_word, rlk_stream stream);

/*
 * rlk_logprob_entropy_canonical_topp -- the three steps on one device (all
 * n_virtual shards): partials and counts go to the workspace,
 * rlk_workspace_size(RLK_OP_CANONICAL_TOPP, T, n_virtual, 0) bytes, 16-byte
 * aligned (8256 bytes per row and shard).
 */
rlk_status rlk_logprob_entropy_canonical_topp(const void* logits, rlk_dtype dtype, int64_t T,
                                              int64_t V, int64_t ld, const int32_t* token_ids,
                                              float temperature, float top_p, int32_t n_virtual,
                                              int64_t padded_vocab, float* out_logprob,
                                              float* out_entropy, int32_t* out_k,
                                              uint32_t* out_status_word, void* workspace,
                                              size_t workspace_bytes, rlk_stream stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* RLK_H_ */
