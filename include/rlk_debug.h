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

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* RLK_DEBUG_H_ */
