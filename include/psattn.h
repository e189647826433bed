/*
 * psattn — batched decode attention over a paged KV cache for requests that
 * share prefixes, on one GB300 (sm_103a).
 *
 * The operation (papercache.org, "BatchLLM: Optimizing Large Batched LLM
 * Inference with Global Prefix Sharing and Throughput-oriented Token
 * Batching", section 2.2, Eq. 1, and section 5 "horizontal fusion"): each
 * decode query's attention is split into a partial over the shared prefix KV
 * of its group, computed once per group, and a partial over its own distinct
 * KV; the partials are reduced exactly by online softmax.  Multi-level
 * prefixes (section 2.2, last paragraph; section 4.2) give one partial per
 * level.  All partials of a batch run in one kernel launch.  The KV cache is
 * paged ("continuous-batching" page, guijiagi.com, PagedAttention section):
 * logically contiguous KV lives in fixed-size physical blocks named by a
 * per-request block table.
 *
 * The result equals, up to rounding, plain attention of every request over
 * its whole token list: softmax(q K^T * scale) V, with LSE = ln sum exp(q K^T
 * * scale).
 *
 * Conventions shared by every call
 * --------------------------------
 *  R = num_req, Hq = num_q_heads, Hkv = num_kv_heads, G = Hq / Hkv (q head h
 *  reads KV head h / G), d = head_dim, B = block_size.
 *
 *  KV pool   [num_pool_blocks][2][Hkv][B][d], index 0 = K, 1 = V, dtype.
 *            One (block, K|V, head) tile of B x d is contiguous.
 *  block table  int32 [R][max_blocks_per_req], row r lists request r's
 *            prefix chain root level first, each level starting at a new
 *            block and occupying ceil(P_level / B) entries, then its
 *            ceil(S_r / B) suffix blocks; unused entries are ignored.
 *  group_of_req int32 [R]: the request's deepest prefix group, -1 = none.
 *  group_parent int32 [num_groups]: parent level of a group, -1 = root; a
 *            NULL pointer means every group is a root (single level).
 *  prefix_len   int32 [num_groups]: tokens a group's level adds (>= 0).
 *  suffix_len   int32 [R]: the request's own tokens, including the decode
 *            token's K/V (>= 0); a request must attend to >= 1 token and to
 *            at most INT32_MAX tokens (its chain and suffix together).
 *  q, out    [R][Hq][d] in dtype; out is rounded to nearest even for bf16.
 *  lse       float32 [R][Hq], natural log of sum(exp(scaled scores)).
 *
 *  Ownership: the caller owns every tensor.  A plan owns its host tables and
 *  one device workspace (work lists, group tables, partial slots, merge
 *  tickets, counters), allocated in psattn_plan and freed by
 *  psattn_plan_destroy.  Every call returns a psattn_status and never aborts.
 *  The library keeps no global state besides the CUDA driver's.
 *
 *  Supported: dtype bf16 with d = 128 (tensor-core paths) or d = 64, fp32
 *  with d = 64 or 128; B = 16; G in {1, 2, 4, 8}.  Anything else returns
 *  PSATTN_ERR_UNSUPPORTED.
 */
#ifndef PSATTN_H_
#define PSATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* psattn_stream_t; /* same type as cudaStream_t */

typedef enum {
    PSATTN_OK = 0,
    PSATTN_ERR_INVALID_ARG = -1,   /* null pointer, bad shape, length < 0, table too narrow */
    PSATTN_ERR_BLOCK_OOB = -2,     /* a block id outside [0, num_pool_blocks) */
    PSATTN_ERR_GROUP_MISMATCH = -3,/* a group member's prefix blocks differ from the group's */
    PSATTN_ERR_EMPTY_REQUEST = -4, /* a request attends to 0 tokens */
    PSATTN_ERR_UNSUPPORTED = -5,   /* dtype / head_dim / block_size / GQA ratio not built */
    PSATTN_ERR_CUDA = -6,          /* a CUDA runtime call failed */
    PSATTN_ERR_DEVICE = -7,        /* the kernel raised its error word (see psattn_plan_status) */
    PSATTN_ERR_NOMEM = -8,         /* host or device allocation failed */
    PSATTN_ERR_GROUP_CYCLE = -9    /* group_parent has a cycle or a bad id */
} psattn_status;

typedef enum { PSATTN_F32 = 0, PSATTN_BF16 = 1 } psattn_dtype;

typedef struct {
    int32_t num_req, num_groups, num_q_heads, num_kv_heads, head_dim, block_size;
    int32_t max_blocks_per_req, num_pool_blocks;
    int32_t dtype; /* psattn_dtype */
    float scale;   /* softmax scale, usually 1/sqrt(head_dim) */
} psattn_shape;

/* Plan flags. */
#define PSATTN_NO_DEDUP 1u   /* ignore groups: every request reads its whole chain itself */
#define PSATTN_FLATTEN 2u    /* collapse each chain into one level per leaf group (BatchLLM
                                section 4.2); needs every non-leaf level to be a whole
                                number of blocks */
#define PSATTN_NO_TENSOR_PREFIX 4u /* run dense prefix groups on the per-warp path */
#define PSATTN_SIMT 8u       /* bf16: use the CUDA-core per-warp path instead of mma.sync */
#define PSATTN_NO_FOLD 16u   /* keep every level its own partial.  By default a parent level
                                (a whole number of blocks) is read by its children's
                                tensor-core items when those, plus the tiles of the level's
                                own requests (none, or at least 8 q rows), need no more
                                128-row tiles than the level itself; info.unique_kv_bytes
                                still counts it once */

typedef struct psattn_plan_s* psattn_plan_t;

typedef struct {
    int64_t warp_items;       /* per-warp work items (suffix and small-group prefix partials) */
    int64_t dense_items;      /* tensor-core prefix tiles */
    int64_t partial_slots;    /* (request, partial) slots in the workspace */
    int64_t workspace_bytes;  /* device bytes owned by the plan */
    int64_t unique_kv_bytes;  /* K+V bytes of every prefix level once per group plus every suffix */
    int64_t planned_kv_bytes; /* K+V bytes the plan's items read (== unique unless NO_DEDUP) */
    int64_t qo_bytes;         /* q + out + lse bytes */
    int32_t suffix_chunk_max; /* largest suffix chunk in tokens */
    int32_t prefix_chunk_max; /* largest prefix chunk in tokens */
    int32_t num_sms;          /* SM count the plan was sized for */
    int32_t grid;             /* CTAs psattn_decode launches */
    int32_t dense_item_warps; /* per-warp item warps per CTA that run beside the tensor-core
                                 items (4; 0 without tensor-core items) */
} psattn_plan_info;

/*
 * Build a plan: validate the inputs, form the prefix-group tables, split every
 * prefix level and suffix into chunks, and lay out the flat work lists
 * (heaviest first, ties broken by kind, group, KV head, chunk).  Reads host
 * arrays only.  Then allocates the plan's device workspace and uploads the
 * tables on `stream` (the upload is complete when this call returns).
 *
 *  shape        host, required.
 *  block_table  host int32 [num_req][max_blocks_per_req].
 *  group_of_req host int32 [num_req].
 *  group_parent host int32 [num_groups], or NULL for single-level groups.
 *  prefix_len   host int32 [num_groups] (may be NULL when num_groups == 0).
 *  suffix_len   host int32 [num_req].
 *  flags        PSATTN_* flags, or 0.
 *  stream       CUDA stream for the allocation and upload (NULL = default stream).
 *  out          receives the plan; set to NULL on error.
 *
 * Errors: INVALID_ARG, UNSUPPORTED, BLOCK_OOB, GROUP_MISMATCH, EMPTY_REQUEST,
 * GROUP_CYCLE (all detected on the host before any device work), NOMEM, CUDA.
 */
int psattn_plan(const psattn_shape* shape, const int32_t* block_table,
                const int32_t* group_of_req, const int32_t* group_parent,
                const int32_t* prefix_len, const int32_t* suffix_len, uint32_t flags,
                psattn_stream_t stream, psattn_plan_t* out);

/*
 * Host-only planning, for a given SM count: the same validation and tables as
 * psattn_plan, with no CUDA call and no device memory.  Such a plan can be
 * inspected (psattn_plan_info, psattn_plan_export) but not run.  num_sms >= 1.
 */
int psattn_plan_host(const psattn_shape* shape, const int32_t* block_table,
                     const int32_t* group_of_req, const int32_t* group_parent,
                     const int32_t* prefix_len, const int32_t* suffix_len, uint32_t flags,
                     int32_t num_sms, psattn_plan_t* out);

/*
 * psattn_plan / psattn_plan_host with ragged leaf levels: leaf_len (host
 * int32 [num_req], or NULL for none) gives, per request, how many tokens of
 * its leaf level (group_of_req[r]) it attends to: the first leaf_len[r]
 * tokens, or all of them for -1.  The level is still read once for all its
 * members; each member row masks the tokens past its own length.  This is
 * how a prefill chunk's causal triangle runs as one shared level
 * (psattn_chunked.h).  Needs the bf16, head_dim 128 path (else
 * PSATTN_ERR_UNSUPPORTED).  INVALID_ARG for a length below -1, above the
 * level, on a request without a group, or with PSATTN_FLATTEN.
 */
int psattn_plan_ragged(const psattn_shape* shape, const int32_t* block_table,
                       const int32_t* group_of_req, const int32_t* group_parent,
                       const int32_t* prefix_len, const int32_t* suffix_len,
                       const int32_t* leaf_len, uint32_t flags, psattn_stream_t stream,
                       psattn_plan_t* out);
int psattn_plan_host_ragged(const psattn_shape* shape, const int32_t* block_table,
                            const int32_t* group_of_req, const int32_t* group_parent,
                            const int32_t* prefix_len, const int32_t* suffix_len,
                            const int32_t* leaf_len, uint32_t flags, int32_t num_sms,
                            psattn_plan_t* out);

/*
 * Run one decode step: the whole fused launch (every prefix partial, every
 * suffix partial and the exact LSE merge) as ONE kernel on `stream`.
 * Asynchronous; the plan's counters and tickets reset themselves at the end of
 * the launch, so steps can follow each other on one stream with no memset.
 * A plan must not run on two streams at once.
 *
 *  q            device [R][Hq][d], dtype, 16-byte aligned.
 *  kv_pool      device [num_pool_blocks][2][Hkv][B][d], dtype, 16-byte aligned.
 *  block_table, group_of_req, prefix_len, suffix_len: device copies with the
 *               contents the plan was built from.  Lengths and block ids are
 *               read here, so a suffix may grow between steps without a new
 *               plan as long as it stays within the block-table columns the
 *               plan saw (the last chunk of each segment runs to its end).
 *  out          device [R][Hq][d], dtype, 16-byte aligned.
 *  lse          device float32 [R][Hq], or NULL.
 *
 * Errors: INVALID_ARG (null or misaligned pointer, host-only plan), CUDA
 * (launch failure).  Inconsistent device tables do not fault: the kernel skips
 * the bad access and raises the plan's error word (psattn_plan_status).
 */
int psattn_decode(psattn_plan_t plan, const void* q, const void* kv_pool,
                  const int32_t* block_table, const int32_t* group_of_req,
                  const int32_t* prefix_len, const int32_t* suffix_len, void* out, float* lse,
                  psattn_stream_t stream);

/*
 * psattn_decode without any device allocation.  The paper has no counterpart:
 * this exists for callers that cannot call cudaMalloc — a process whose device
 * memory is already owned by another allocator (an engine that reserves
 * nearly all of HBM for its KV-cache pool up front), or code on a
 * latency-critical path where cudaMalloc/cudaFree are ruled out because they
 * can synchronise the device.  The workspace psattn_plan would allocate lives
 * instead in one fixed device array of PSATTN_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library keeps until the process
 * exits.
 *
 *  plan   a plan from psattn_plan_host (host tables only, no device memory;
 *         pass the device's SM count) or from psattn_plan.
 *  other arguments: as psattn_decode (device pointers, same layouts).
 *
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  The address
 * is kept per device and looked up again when the device's context has been
 * replaced (after cudaDeviceReset, for instance).  Every call clears the
 * counters and tickets and uploads its plan's tables into the array with
 * asynchronous copies from the plan's host memory, then runs the same fused
 * kernel as psattn_decode, asynchronously on `stream`: keep the plan alive
 * until that work on `stream` has completed.  All calls share the array: calls whose launches overlap on the
 * GPU race and give wrong results.  The kernel's error word is kept in the
 * array and is not reported.  Returns INVALID_ARG (null or misaligned pointer),
 * NOMEM (the plan's workspace exceeds PSATTN_NOALLOC_SCRATCH_BYTES; nothing is
 * launched), CUDA.  Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define PSATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int psattn_decode_noalloc(psattn_plan_t plan, const void* q, const void* kv_pool,
                          const int32_t* block_table, const int32_t* group_of_req,
                          const int32_t* prefix_len, const int32_t* suffix_len, void* out,
                          float* lse, psattn_stream_t stream);

/* Sizes and counts of a plan.  Returns INVALID_ARG on NULL. */
int psattn_plan_info_get(psattn_plan_t plan, psattn_plan_info* info);

/* Plan tables for bit-exact tests.  which: 0 = warp items, 1 = dense items
 * (int32 x 8 each: kind, kv_head, segment, chunk, member_offset, members,
 * partial_index, cost), 2 = per-request table (int32 x 8: slot_base,
 * partials, suffix_column, suffix_chunk_tokens, suffix_chunks, leaf_group, 0,
 * 0), 3 = per-group table (int32 x 8: column_base, chunk_tokens, chunks,
 * representative, member_offset, members, partial_index_0, dense),
 * 4 = member list (int32 request ids), 5 = per-group length offset.
 * Writes at most `cap` int32 values to dst (dst may be NULL) and returns the
 * number of int32 values the table holds, or a negative status. */
int64_t psattn_plan_export(psattn_plan_t plan, int32_t which, int32_t* dst, int64_t cap);

/* Waits for the plan's last psattn_decode launch (an event the library
 * records after each launch; other work on the device is not waited for),
 * then reads and clears the kernel's error word.  When the word is non-zero,
 * the plan's work counters and merge tickets are reset too: a launch that
 * gave up part way may leave tickets short of their count, and the next
 * launch must not merge partials left from it.  Returns
 * PSATTN_OK, PSATTN_ERR_DEVICE (flags in *device_flags when non-NULL: 1 =
 * block id out of range, 2 = group_of_req differs from the plan, 4 = block
 * column beyond the table, 8 = a request with no token, 16 = a bounded wait
 * inside the kernel gave up (the launch's results are incomplete), 32 = the
 * merge bookkeeping found an inconsistency (more arrivals than partials, or a
 * queued unit out of range)), or PSATTN_ERR_CUDA. */
int psattn_plan_status(psattn_plan_t plan, uint32_t* device_flags);

/* Test of the failure path of the kernel's bounded waits, with no fault:
 * launches one wait on an mbarrier that nothing completes, through the same
 * bounded wait the decode kernel uses, with a limit of limit_us microseconds
 * (1 .. 100000).  The wait gives up, the kernel sets error flag 16 and
 * returns; the context stays usable.  Synchronises the device.  Returns
 * PSATTN_ERR_DEVICE with *device_flags = 16 when the wait gave up as it
 * should, PSATTN_OK (flags 0) if it did not, INVALID_ARG or CUDA. */
int psattn_selftest_wait_timeout(uint32_t limit_us, uint32_t* device_flags);

/* Frees the plan and its workspace, after waiting for the plan's last launch.
 * NULL is a no-op. */
void psattn_plan_destroy(psattn_plan_t plan);

/* Static text for a status code. */
const char* psattn_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* PSATTN_H_ */
