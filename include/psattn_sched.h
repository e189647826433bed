/*
 * psattn_sched — token batches of an offline batch, host only.
 *
 * A simulation of the throughput-oriented token batching of "BatchLLM:
 * Optimizing Large Batched LLM Inference with Global Prefix Sharing and
 * Throughput-oriented Token Batching" (papercache.org summary), section 4.3:
 *  - 4.3.1 requests are scheduled a whole prefix-sharing group at a time,
 *    and every iteration fills its token batch from three queues in this
 *    order: decode tokens, distinct-prompt tokens, common-prefix tokens; a
 *    group's distinct prompts wait until its common prefix is processed;
 *  - 4.3.2 groups are reordered by R_group = 1 / (L_prefix + sum L_distinct)
 *    (Eq. 4: Eq. 3's decode/prefill ratio with the decode length normalised
 *    to one), largest first;
 *  - 4.3.3 memory-centric batching: a prefill chunk joins the batch only if
 *    the KV memory it adds stays within M_threshold, whatever the number of
 *    requests; N_chunk caps the tokens of an iteration.
 * No model runs: an iteration processes its token batch, prefill chunks
 * advance prompt positions, and each decode token advances one request by
 * one output token.  Everything is integer and deterministic.
 *
 * Model (the readings of the section's prose)
 * -----
 *  - Group g has a common prefix of group_prefix[g] tokens; request r
 *    belongs to group group_of_req[r] (-1: a group of its own with no
 *    prefix), has distinct_len[r] prompt tokens and produces decode_len[r]
 *    (>= 1) output tokens, one per iteration, starting the iteration after
 *    its last prompt token was processed.
 *  - Groups are admitted in priority order: input order (the order of each
 *    group's smallest request id), or with PSATTN_SCHED_REORDER by R_group,
 *    largest first (smallest L_prefix + sum L_distinct; ties in input
 *    order).  Groups without requests are skipped.  The common-prefix queue
 *    serves the admitted-but-unfinished prefixes and admits the next group
 *    when the previous prefix is done, within the iteration if budget is
 *    left.  A group's requests enter the distinct queue the iteration after
 *    its prefix is complete (a group without prefix: the iteration after it
 *    is admitted).
 *  - Each iteration, with a budget of n_chunk tokens: (1) every request in
 *    the decode queue (in the order they entered it; ties by request id)
 *    takes one token while budget lasts; (2) requests in the distinct queue
 *    (by group priority, then request id) take min(remaining prompt,
 *    budget) tokens each; (3) the prefix queue likewise.  A prefill chunk
 *    (2, 3) of c tokens is taken only if resident + c <= m_threshold (or
 *    m_threshold < 0); the first one that does not fit ends the prefill
 *    part of the iteration.  So that the run always progresses, a chunk is
 *    also taken when the batch is still empty.  A request whose last prompt
 *    token (prefix or distinct) was processed in iteration t decodes from
 *    iteration t + 1 on; one without any prompt token, from the iteration
 *    after its group was admitted.
 *  - max_requests > 0 adds the request-count limiter the section argues
 *    against: a batch holds at most that many requests (a prefix chunk
 *    counts as one).
 *  - KV memory, in tokens: a group's prefix tokens from the iteration they
 *    are processed until its last request finishes; a request's prompt and
 *    output tokens likewise until it finishes.  A request finishes at the
 *    end of the iteration that produced its last output token.
 *
 * Per iteration i the outputs are iter_tokens[4 i .. 4 i + 3] = decode
 * tokens, distinct-prompt tokens, common-prefix tokens, requests in the
 * batch (a prefix chunk counts as one), and iter_mem[i] = resident KV tokens
 * at the end of the iteration (before that iteration's finished requests are
 * freed).  Returns a psattn_status (psattn.h); never aborts.  Host memory
 * only: the caller owns every input and output array, and the call keeps
 * nothing between calls.
 */
#ifndef PSATTN_SCHED_H_
#define PSATTN_SCHED_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PSATTN_SCHED_REORDER 1u /* admit groups by R_group, largest first */

typedef struct {
  int32_t n_chunk;      /* tokens per iteration (N_chunk), >= 1 */
  int64_t m_threshold;  /* KV-token limit for prefill chunks (M_threshold); < 0: none */
  int32_t max_requests; /* > 0: at most this many requests per batch; 0: no limit */
  uint32_t flags;       /* PSATTN_SCHED_REORDER */
} psattn_sched_params;

/*  group_prefix   int32 [num_groups]   common-prefix tokens per group (>= 0)
 *  group_of_req   int32 [num_req]      -1 or a group id
 *  distinct_len   int32 [num_req]      prompt tokens past the prefix (>= 0)
 *  decode_len     int32 [num_req]      output tokens (>= 1)
 *  group_order    int32 [num_groups + num_req] out: admission order of the
 *                 scheduling groups, numbered 0..num_groups-1 for the given
 *                 groups and num_groups + r for ungrouped request r;
 *                 *num_sched_groups entries are written
 *  iter_tokens    int32 [4 * cap] out
 *  iter_mem       int64 [cap] out
 *  cap            iterations the outputs can hold; PSATTN_ERR_NOMEM (and
 *                 *num_iters = iterations needed) when the run is longer
 *  num_iters      out
 * Errors: PSATTN_ERR_INVALID_ARG for a NULL pointer, negative counts or
 * lengths, decode_len < 1, a group id out of range, n_chunk < 1,
 * max_requests < 0, or a batch of more than 2^29 tokens in all (each used
 * group's prefix once, plus every prompt and output; iterations are counted
 * in int32).  A group with no requests is never admitted.  The run takes one
 * simulated iteration per step, at least the longest output's length. */
int psattn_token_batches(const int32_t* group_prefix, int32_t num_groups,
                         const int32_t* group_of_req, const int32_t* distinct_len,
                         const int32_t* decode_len, int32_t num_req,
                         const psattn_sched_params* params, int32_t* group_order,
                         int32_t* num_sched_groups, int32_t* iter_tokens, int64_t* iter_mem,
                         int32_t cap, int32_t* num_iters);

#ifdef __cplusplus
}
#endif

#endif /* PSATTN_SCHED_H_ */
