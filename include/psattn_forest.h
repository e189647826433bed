/*
 * psattn_forest — prefix-sharing groups from token ids, host only.
 *
 * These calls produce the grouping metadata the decode kernel consumes
 * (group_of_req, group_parent, prefix_len, suffix_len of psattn.h) from the
 * requests' token ids, and form prefix-homogeneous batches.  They follow:
 *  - "BatchLLM: Optimizing Large Batched LLM Inference with Global Prefix
 *    Sharing and Throughput-oriented Token Batching" (papercache.org summary),
 *    section 4.2: a compact prefix tree over the batch's prompts identifies
 *    the common prefixes explicitly; a dynamic program over that tree
 *    enlarges the first-level prefix to maximise the tokens whose KV is
 *    reused ("saving" of Eq. 2);
 *  - "Requests of a Feather Must Flock Together: Batch Size vs. Prefix
 *    Homogeneity in LLM Inference" (gist.science summary), methodology 1: a
 *    request is a vector of cumulative hashes of fixed-size token chunks; the
 *    active batch keeps the set of its chunk hashes and the waiting requests
 *    sit in a min-heap keyed by their miss count (chunks the batch does not
 *    cover yet), so the best next request is found in O(log W).
 *
 * Conventions
 * -----------
 *  tokens   int32, the requests' token ids back to back; request r owns
 *           tokens[offsets[r] .. offsets[r + 1]) (offsets int64 [R + 1],
 *           offsets[0] = 0, non-decreasing).  Host memory, read only.
 *  chunk    tokens per chunk (>= 1).  Requests are compared in whole chunks
 *           only: two requests share a chunk-prefix of c chunks when their
 *           first c * chunk tokens are equal.  Hashes only index; every
 *           shared chunk is checked token by token, so a hash collision
 *           never merges different prefixes.  With chunk a multiple of the
 *           KV block size every prefix level starts on a block boundary, as
 *           psattn_plan requires.
 *  Outputs are caller-owned host arrays; nothing is kept between calls.
 *  Results are deterministic: group ids are given in depth-first order,
 *  children ordered by the smallest request id that passes through them.
 *  Every call returns a psattn_status (psattn.h) and never aborts.
 */
#ifndef PSATTN_FOREST_H_
#define PSATTN_FOREST_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* flags of psattn_forest_group */
#define PSATTN_FOREST_SINGLE 1u /* one prefix level per request, chosen by the
                                   first-level reuse DP (BatchLLM section 4.2) */

/* Groups the requests by shared chunk-prefixes.
 *
 * Multi-level (flags = 0): the compact prefix tree of the requests' chunk
 * sequences, restricted to chunk-prefixes that two or more requests share.
 * Each node of that tree is one prefix level (group): a maximal run of
 * chunks that the same set of requests passes through; its parent is the
 * level above it (-1 at a root).  A request's group is the deepest level on
 * its path (-1 when it shares no whole chunk with any other request); its
 * suffix is every token past that level (the partial last chunk included).
 * For every two requests, the levels they have in common add up to their
 * longest common prefix rounded down to whole chunks.
 *
 * Single level (PSATTN_FOREST_SINGLE): every group is a root and a request
 * belongs to at most one.  A group is the set of requests that share the
 * first prefix_len tokens (a whole number of chunks along their common
 * path), and the choice maximises the saved tokens
 *     sum over groups of (members - 1) * prefix_len,
 * exactly (a dynamic program over the multi-level tree: at every level,
 * the requests passed up from the levels below and the requests that end
 * there either form the level's group or move up to an ancestor).  Ties
 * are broken deterministically: the fewest requests move up, and a level
 * keeps the smallest ids of the requests that reach it.
 *
 *  group_of_req  int32 [num_req] out
 *  group_parent  int32 [cap] out (all -1 in single-level mode)
 *  prefix_len    int32 [cap] out, tokens each level adds
 *  suffix_len    int32 [num_req] out
 *  cap           capacity of group_parent / prefix_len; num_req - 1 always
 *                suffices.  PSATTN_ERR_NOMEM (and *num_groups = the number
 *                needed) when it is too small.
 *  num_groups    out
 *  saved_tokens  out (may be NULL): sum over levels of (requests through the
 *                level - 1) * tokens of the level.
 * Errors: PSATTN_ERR_INVALID_ARG for a NULL required pointer, num_req < 0,
 * chunk < 1, or offsets that decrease. */
int psattn_forest_group(const int32_t* tokens, const int64_t* offsets, int32_t num_req,
                        int32_t chunk, uint32_t flags, int32_t* group_of_req,
                        int32_t* group_parent, int32_t* prefix_len, int32_t* suffix_len,
                        int32_t cap, int32_t* num_groups, int64_t* saved_tokens);

/* Forms prefix-homogeneous batches with the chunked hash tree (Feather,
 * methodology 1), under a static stopping rule (the paper also learns the
 * rule; that part is not modelled here).
 *
 * Batches are formed one after another.  A batch starts with the waiting
 * request of smallest id; its chunk hashes form the batch's working set.
 * Then, while the batch has fewer than max_batch requests, the waiting
 * request with the fewest misses (whole chunks whose cumulative hash the
 * working set lacks; ties: smallest id) joins if its misses are at most
 * max_new_chunks, and its hashes join the working set; otherwise the batch
 * closes.  Misses only fall while a batch grows: every hash added to the
 * working set lowers the count of each waiting request holding it (an
 * inverted index from hash to requests), and stale heap entries are skipped
 * when popped.
 *
 *  batch_of_req  int32 [num_req] out: batch index of each request
 *  order         int32 [num_req] out: request ids in the order they joined
 *  num_batches   out
 * Errors: PSATTN_ERR_INVALID_ARG for a NULL pointer, num_req < 0, chunk < 1,
 * max_batch < 1, max_new_chunks < 0 or decreasing offsets. */
int psattn_cht_batches(const int32_t* tokens, const int64_t* offsets, int32_t num_req,
                       int32_t chunk, int32_t max_batch, int32_t max_new_chunks,
                       int32_t* batch_of_req, int32_t* order, int32_t* num_batches);

/* The chunked-hash-tree batches of psattn_cht_batches, each turned into the
 * grouping metadata psattn_plan consumes (Feather, methodology 1, forms the
 * prefix-homogeneous batches; within a batch the requests are grouped by
 * their shared chunk-prefixes exactly as psattn_forest_group groups a batch
 * of its own, with the same flags).
 *
 * Batch b's requests, in increasing id order, form its own group forest:
 * its groups are the ids [batch_group_offset[b], batch_group_offset[b + 1]),
 * a group's parent is a group of the same batch (or -1), and a request's
 * group is one of its batch's (or -1).  To plan batch b, take its requests
 * and subtract batch_group_offset[b] from their group ids and from the
 * parents of its groups.
 *
 *  batch_of_req, order, num_batches   as psattn_cht_batches.
 *  batch_group_offset  int32 [num_req + 1] out (num_batches + 1 entries used).
 *  group_of_req, suffix_len  int32 [num_req] out.
 *  group_parent, prefix_len  int32 [cap] out; PSATTN_ERR_NOMEM (with
 *                *num_groups = the number needed) when cap is too small;
 *                num_req - 1 always suffices.
 *  saved_tokens  out (may be NULL): sum of the batches' savings as defined
 *                for psattn_forest_group.
 * Errors: PSATTN_ERR_INVALID_ARG as psattn_cht_batches and psattn_forest_group
 * (NULL pointer, num_req < 0, chunk < 1, max_batch < 1, max_new_chunks < 0,
 * decreasing offsets, unknown flags). */
int psattn_cht_group(const int32_t* tokens, const int64_t* offsets, int32_t num_req,
                     int32_t chunk, int32_t max_batch, int32_t max_new_chunks, uint32_t flags,
                     int32_t* batch_of_req, int32_t* order, int32_t* num_batches,
                     int32_t* batch_group_offset, int32_t* group_of_req, int32_t* group_parent,
                     int32_t* prefix_len, int32_t* suffix_len, int32_t cap, int32_t* num_groups,
                     int64_t* saved_tokens);

#ifdef __cplusplus
}
#endif

#endif /* PSATTN_FOREST_H_ */
