/*
 * psattn_chunked — prefill chunks in the decode launch, host only.
 *
 * "BatchLLM: Optimizing Large Batched LLM Inference with Global Prefix Sharing
 * and Throughput-oriented Token Batching" (papercache.org summary), sections 2
 * and 6: with chunked prefill, a token batch mixes the queries of prefill
 * chunks with decode tokens, and the attention kernel serves both in one
 * launch.  A chunk of n queries is the last n tokens of its request; query i
 * of the chunk attends to the tokens up to and including its own position.
 *
 * psattn_chunked_expand turns such a batch into an equivalent decode batch
 * for psattn_plan / psattn_decode, so the same fused launch runs it:
 *  - query i of request r becomes a decode row over r's tokens up to its own
 *    position;
 *  - the part of r's suffix before the chunk, rounded down to whole KV
 *    blocks, becomes one more prefix level (child of r's group, or a root),
 *    shared by all n queries: read once for all n * G query rows (the
 *    tensor-core tile when n * G >= 32);
 *  - past that level, the chunk's causal triangle is cut into levels of
 *    level_tokens tokens: level k is shared by every query that sees all of
 *    it, so only the last, partly visible stretch (fewer than level_tokens +
 *    block_size tokens) is each query's own suffix.
 * Every level starts on a KV block boundary, and the levels partition r's
 * suffix in order, so each expanded row's block-table row is a copy of r's
 * row.  A request with n = 1 (a decode request) is copied unchanged.
 *
 * Expanded rows are ordered request by request, query by query: row
 * sum_{r' < r} q_len[r'] + i is query i of request r.  q, out and lse of
 * psattn_decode on the expanded plan use that row order.  New groups are
 * numbered after the given ones, request by request.
 */
#ifndef PSATTN_CHUNKED_H_
#define PSATTN_CHUNKED_H_

#include <stdint.h>

#include "psattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*  shape, block_table, group_of_req, group_parent, prefix_len, suffix_len:
 *                 the batch as psattn_plan takes it (host arrays;
 *                 group_parent may be NULL).
 *  q_len          int32 [num_req]: queries of each request (>= 1); a request
 *                 with q_len >= 2 needs q_len <= suffix_len (its chunk is the
 *                 end of its own suffix).
 *  level_tokens   causal level size, a positive multiple of block_size, or 0
 *                 for none (then each query's own suffix runs from the end of
 *                 the shared level to its position).
 *  out_shape      receives shape with num_req = sum q_len and num_groups =
 *                 given + new groups (also on PSATTN_ERR_NOMEM).
 *  out_block_table  int32 [cap_rows][max_blocks_per_req]
 *  out_group_of_req, out_suffix_len   int32 [cap_rows]
 *  out_group_parent, out_prefix_len   int32 [cap_groups]
 * Host memory only: the caller owns every input and output array (a first
 * call with caps of 0 and NULL outputs returns PSATTN_ERR_NOMEM with the
 * sizes in out_shape), and the call keeps nothing between calls.
 * Errors: PSATTN_ERR_INVALID_ARG (a NULL pointer, a bad length, group id or
 * q_len, level_tokens not a multiple of block_size), PSATTN_ERR_NOMEM (a cap
 * is too small; out_shape says what is needed).  Never aborts. */
int psattn_chunked_expand(const psattn_shape* shape, const int32_t* block_table,
                          const int32_t* group_of_req, const int32_t* group_parent,
                          const int32_t* prefix_len, const int32_t* suffix_len,
                          const int32_t* q_len, int32_t level_tokens, psattn_shape* out_shape,
                          int32_t* out_block_table, int32_t* out_group_of_req,
                          int32_t* out_group_parent, int32_t* out_prefix_len,
                          int32_t* out_suffix_len, int32_t cap_rows, int32_t cap_groups);

/* The same batch with each chunk's suffix as one ragged level, for
 * psattn_plan_ragged (psattn.h): for a request with n >= 2 queries, its whole
 * suffix (the tokens before the chunk and the chunk) becomes one level under
 * its group, shared by all n queries; query i attends to its first
 * out_leaf_len = a + i + 1 tokens of it (a = suffix tokens before the chunk),
 * and has no suffix of its own.  The tensor-core tile then reads the
 * suffix's K/V once for all n * G query rows and masks each row at its
 * position: the chunk's causal attention as one masked contraction.  Requests with n = 1 are copied unchanged
 * (out_leaf_len -1).  Arguments and errors as psattn_chunked_expand, plus
 *  out_leaf_len   int32 [cap_rows] out. */
int psattn_chunked_expand_ragged(const psattn_shape* shape, const int32_t* block_table,
                                 const int32_t* group_of_req, const int32_t* group_parent,
                                 const int32_t* prefix_len, const int32_t* suffix_len,
                                 const int32_t* q_len, psattn_shape* out_shape,
                                 int32_t* out_block_table, int32_t* out_group_of_req,
                                 int32_t* out_group_parent, int32_t* out_prefix_len,
                                 int32_t* out_suffix_len, int32_t* out_leaf_len,
                                 int32_t cap_rows, int32_t cap_groups);

#ifdef __cplusplus
}
#endif

#endif /* PSATTN_CHUNKED_H_ */
