/*
 * rlk_debug.h -- validation aids of librlk (not part of the hot path).
 */
#ifndef RLK_DEBUG_H_
#define RLK_DEBUG_H_

#include "rlk.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * rlk_lmhead_logits_debug -- rlk_lmhead_logprob at top_p = 1 that also writes
 * the fp32 logits it computed, logits[t, v] = sum_k hidden[t, k] w_vocab[v, k],
 * row-major [T, V] into out_logits (device).  The fused path never stores
 * logits; this copy exists only so tests can check the tensor-core GEMM on its
 * own against a library matrix product.  Slow (uncoalesced stores): use small
 * T and V.  Arguments and errors as rlk_lmhead_logprob, plus out_logits
 * (required, device float[T * V]).
 */
rlk_status rlk_lmhead_logits_debug(const void* hidden, const void* w_vocab, int64_t T, int64_t H,
                                   int64_t V, const int32_t* token_ids, float temperature,
                                   float* out_logits, float* out_logprob, float* out_entropy,
                                   uint32_t* out_status_word, void* workspace,
                                   size_t workspace_bytes, rlk_stream stream);

/*
 * rlk_debug_inject_launch_failures -- fault injection on the host.  The next
 * n calls of any entry point that would launch work (after their argument
 * checks pass) return RLK_ERR_CUDA without launching anything and without
 * touching their outputs, as a failed launch would.  n <= 0 clears the count.
 * Returns the count that was pending.  For testing callers' error handling;
 * nothing reaches the GPU.
 */
int rlk_debug_inject_launch_failures(int n);

/*
 * rlk_debug_set_wait_limit -- the number of clock cycles any bounded device
 * wait of the logprob/entropy scorer and the LM-head kernel may take before
 * it gives up (default 2^31, about a second).  A wait that runs out sets
 * RLK_STATUS_TIMEOUT in the call's status word, the rows the kernel has not
 * finished get NaN outputs, copies already issued are allowed to land, and
 * the kernel returns, so the context stays usable.  cycles <= 0 restores the
 * default.  Returns the previous limit.  Not thread-safe with respect to
 * concurrent launches.
 */
long long rlk_debug_set_wait_limit(long long cycles);

/*
 * rlk_debug_withhold_copy -- makes the next rlk_logprob_entropy launch (and
 * the next LM-head forward launch) skip one of the bulk copies of its first
 * CTA: the stage with the given index in that CTA's sequence, for which no
 * copy is issued and no arrival made.  The wait on it then runs out (after
 * the limit set above), which exercises the expiry path; nothing is left in
 * flight.  stage < 0 clears it.  The setting is consumed by one launch.
 * Returns 0.
 */
int rlk_debug_withhold_copy(long long stage);

/*
 * rlk_debug_set_sampler_mode -- the ways rlk_sample_top_p may take to a draw.
 * mode = 1 (the default, also for any value other than 0 and 2): the direct
 * mode where it applies, which bins the retained set by key in one read of
 * the row and ranks the draw's tie group from the list of members it kept;
 * mode = 2: the direct mode without the member list (the tie group is found
 * by a scan of the row in id order, as when the list runs out of room);
 * mode = 0: every row by the radix descent over the 16-bit keys (up to three
 * reads of the row).  All draw the same id (integer arithmetic); this lets
 * tests compare them on the same inputs.  Returns the previous mode.  Not
 * thread-safe with respect to concurrent launches.
 */
int rlk_debug_set_sampler_mode(int mode);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* RLK_DEBUG_H_ */
