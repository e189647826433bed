// Internal tables shared by the host planner (plan.cpp) and the kernels
// (decode.cu).  Everything here is plain data: the planner writes it on the
// host, uploads it once, and the kernels read it.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <vector>

#include <cuda_runtime.h>

#include "psattn.h"

namespace psattn {

constexpr int kBlockSize = 16;       // tokens per KV block (the only size built)
constexpr int kWarpsPerCta = 12;     // warps of the persistent CTA (one CTA per SM)
constexpr int kDenseItemWarps = 4;   // per-warp item warps (8-11) beside the tensor-core items
constexpr int kMmaRows = 8;          // q vectors one mma.sync warp item serves (n = 8)
constexpr int kSimtRows = 4;         // q vectors one CUDA-core warp item serves
constexpr int kDenseRows = 128;      // rows of one tensor-core prefix tile (UMMA M)

// kItemDenseRagged: a dense item on a ragged level whose members all stop
// short of the chunk's end; its span ends `cost` tokens past the chunk start
// (the tiles past every member's limit are skipped).
enum ItemKind : int32_t { kItemSuffix = 0, kItemPrefix = 1, kItemDense = 2, kItemDenseRagged = 3 };

// Kernel variant chosen at plan time from dtype / head_dim / flags.
enum Path : int32_t { kPathMmaBf16D128 = 0, kPathSimtF32D64 = 1, kPathSimtF32D128 = 2,
                      kPathSimtBf16D64 = 3, kPathSimtBf16D128 = 4 };

// One unit of work.  Suffix item: the G q heads of request `seg` against
// chunk `chunk` of its suffix, KV head `kvh`.  Prefix item: members
// [mem_off, mem_off + nmem) of group `seg` (each G q heads) against chunk
// `chunk` of that group's level.  Dense item: the same for up to 128/G
// members on the tensor-core path.
struct Item {
  int32_t kind, kvh, seg, chunk, mem_off, nmem, slot_j, cost;
};
static_assert(sizeof(Item) == 32, "Item layout");

struct ReqInfo {
  int32_t slot_base;       // first partial slot of the request
  int32_t n_partials;      // partials merged into the request's output
  int32_t suffix_col;      // block-table column where the suffix starts
  int32_t suffix_chunk;    // tokens per suffix chunk
  int32_t suffix_nchunks;  // suffix chunks (0 when the suffix is empty)
  int32_t leaf;            // leaf group the plan saw (-1 none)
  int32_t leaf_vis;        // tokens of the leaf level the request attends to (-1: all)
  int32_t pad1;
};
static_assert(sizeof(ReqInfo) == 32, "ReqInfo layout");

struct GroupInfo {
  int32_t col_base;   // block-table column where this level starts
  int32_t chunk_tok;  // tokens per chunk
  int32_t n_chunks;   // chunks of this level (0 when it has no member or no token)
  int32_t rep;        // a member whose block-table row holds the level's blocks
  int32_t mem_off;    // members[mem_off .. mem_off + n_mem)
  int32_t n_mem;
  int32_t slot_j0;    // partial index of chunk 0 within every member's partial list
  int32_t dense;      // 1: tensor-core tiles
};
static_assert(sizeof(GroupInfo) == 32, "GroupInfo layout");

// Device error-word flags.
enum : uint32_t { kErrBlockOob = 1u, kErrGroup = 2u, kErrColumn = 4u, kErrEmpty = 8u,
                  kErrTimeout = 16u, kErrMerge = 32u };

// Counter words at the head of the workspace.
enum : int { kCtrWarp = 0, kCtrDense = 1, kCtrExit = 2, kCtrErr = 3, kCtrWords = 8 };

struct HostPlan {
  psattn_shape shape{};
  uint32_t flags = 0;
  int32_t num_sms = 0;
  int32_t path = 0;
  int32_t grid = 0;
  std::vector<Item> witems, ditems;
  std::vector<ReqInfo> req;
  std::vector<GroupInfo> grp;
  std::vector<int32_t> members;
  std::vector<int32_t> len_add;   // per group: tokens added to prefix_len[g] (FLATTEN)
  int64_t n_slots = 0;
  int64_t unique_kv_bytes = 0, planned_kv_bytes = 0, qo_bytes = 0;
  int32_t suffix_chunk_max = 0, prefix_chunk_max = 0;
  int32_t any_ragged = 0;
};

// Device-side view of a plan's workspace.
struct DevPlan {
  const Item* witems;
  const Item* ditems;
  const ReqInfo* req;
  const GroupInfo* grp;
  const int32_t* members;
  const int32_t* len_add;
  uint32_t* tickets;   // [R][Hkv]
  uint32_t* ctr;       // kCtrWords
  float* opart;        // [slots][Hkv][G][d] unnormalised partial outputs
  float2* mlpart;      // [slots][Hkv][G] (running max in log2 units, sum)
  int32_t n_witems, n_ditems;
  int32_t any_ragged;   // some request sees only part of its leaf level
};

}  // namespace psattn

// Host tables of a plan (plan.cpp), for the library's other translation units.
const psattn::HostPlan* psattn_internal_host_plan(psattn_plan_t plan);

// Implemented in decode.cu.
int psattn_run_wait_selftest(uint32_t* dev_flags, uint64_t limit_ns, void* stream);
int psattn_launch_decode(const psattn::HostPlan& hp, const psattn::DevPlan& dp, const void* q,
                         const void* kv_pool, const int32_t* block_table,
                         const int32_t* group_of_req, const int32_t* prefix_len,
                         const int32_t* suffix_len, void* out, float* lse,
                         psattn_stream_t stream);
