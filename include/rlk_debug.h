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

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* RLK_DEBUG_H_ */
