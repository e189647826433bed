// psattn_decode_noalloc: the fused decode for callers that cannot allocate
// device memory.
//
// Who needs it: a serving process whose device memory is owned by another
// allocator (for example an engine that reserves nearly all of HBM for its
// KV-cache pool at start-up, so a later cudaMalloc would fail or fragment that
// pool), and code on a latency-critical path where cudaMalloc / cudaFree are
// not allowed because they can synchronise the whole device.  psattn_plan
// allocates a device workspace per plan; this entry point instead places the
// workspace (work lists, group tables, merge tickets, counters, partial
// results) in one fixed array of PSATTN_NOALLOC_SCRATCH_BYTES that lives in the
// library's own device memory image.  The caller still passes q, the KV pool,
// the tables and the outputs.
//
// Costs and rules:
//  * Every GPU that loads this part of the library holds the array until the
//    process exits.
//  * The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.  Later calls reuse the cached address while
//    the device's context stays the same one (its driver context id); after
//    a cudaDeviceReset the address is looked up again.
//  * The plan's tables reach the array by asynchronous copies from the
//    plan's host memory: the plan must outlive the call's work on its stream.
//  * All calls share the one array and it keeps the last call's contents: each
//    call clears the counters and tickets, then uploads its plan's tables.
//    Calls whose launches overlap on the GPU (different streams, or different
//    host threads without ordering) race on the array and give wrong results.
//  * A plan whose workspace does not fit returns PSATTN_ERR_NOMEM before any
//    device work.  The kernel's error word also lives in the array and is not
//    reported (psattn_plan_status reads only a plan's own workspace).
// No cudaMalloc, cudaFree or other allocating call is made here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "psattn_internal.h"

using namespace psattn;

namespace {

__device__ __align__(256) unsigned char g_scratch[PSATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context id the address belongs to

// Unique id of the calling thread's current driver context (ids are never
// reused within a process); false when there is none or the driver lacks
// the calls, and then the address is looked up on every call.
bool current_context_id(unsigned long long* id) {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static bool tried = false;
  if (!tried) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrentFn>(a);
      get_id = reinterpret_cast<GetIdFn>(b);
    }
    cudaGetLastError();
    tried = true;
  }
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  return get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch on the current device: looked up with the
// device current, and again whenever the device's context has changed.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx = 0;
  bool have_ctx = current_context_id(&ctx);
  if (!g_scratch_addr[dev] || !have_ctx || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return PSATTN_ERR_CUDA;
    }
    // the lookup makes the device's primary context current if none was
    if (!have_ctx) have_ctx = current_context_id(&ctx);
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = have_ctx ? ctx : 0;
  }
  *out = g_scratch_addr[dev];
  return PSATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" int psattn_decode_noalloc(psattn_plan_t plan, const void* q, const void* kv_pool,
                                     const int32_t* block_table, const int32_t* group_of_req,
                                     const int32_t* prefix_len, const int32_t* suffix_len,
                                     void* out, float* lse, psattn_stream_t stream) {
  const HostPlan* hpp = psattn_internal_host_plan(plan);
  if (!hpp) return PSATTN_ERR_INVALID_ARG;
  const HostPlan& hp = *hpp;
  if (hp.shape.num_req == 0) return PSATTN_OK;
  if (!q || !kv_pool || !block_table || !group_of_req || !suffix_len || !out)
    return PSATTN_ERR_INVALID_ARG;
  if (hp.shape.num_groups > 0 && !prefix_len) return PSATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(q) || misaligned(kv_pool) || misaligned(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3))
    return PSATTN_ERR_INVALID_ARG;

  // Workspace layout: the same regions a plan's own workspace holds.
  const int R = hp.shape.num_req, Hkv = hp.shape.num_kv_heads;
  const int G = hp.shape.num_q_heads / Hkv, d = hp.shape.head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + std::max<size_t>(bytes, 1));
    return o;
  };
  const size_t o_ctr = take(sizeof(uint32_t) * kCtrWords);
  const size_t o_tick = take(sizeof(uint32_t) * (size_t)R * Hkv);
  const size_t o_wi = take(sizeof(Item) * hp.witems.size());
  const size_t o_di = take(sizeof(Item) * hp.ditems.size());
  const size_t o_req = take(sizeof(ReqInfo) * hp.req.size());
  const size_t o_grp = take(sizeof(GroupInfo) * hp.grp.size());
  const size_t o_mem = take(sizeof(int32_t) * hp.members.size());
  const size_t o_add = take(sizeof(int32_t) * hp.len_add.size());
  const size_t o_ml = take(sizeof(float2) * (size_t)hp.n_slots * Hkv * G);
  const size_t o_op = take(sizeof(float) * (size_t)hp.n_slots * Hkv * G * d);
  if (off > (size_t)PSATTN_NOALLOC_SCRATCH_BYTES) return PSATTN_ERR_NOMEM;

  void* base_v = nullptr;
  int rc = scratch_address(&base_v);
  if (rc) return rc;
  char* base = static_cast<char*>(base_v);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  // counters and tickets start at zero; the tables are this plan's
  cudaError_t e = cudaMemsetAsync(base + o_ctr, 0, o_wi - o_ctr, st);
  auto put = [&](size_t o, const void* src, size_t bytes) {
    if (e == cudaSuccess && bytes)
      e = cudaMemcpyAsync(base + o, src, bytes, cudaMemcpyHostToDevice, st);
  };
  put(o_wi, hp.witems.data(), sizeof(Item) * hp.witems.size());
  put(o_di, hp.ditems.data(), sizeof(Item) * hp.ditems.size());
  put(o_req, hp.req.data(), sizeof(ReqInfo) * hp.req.size());
  put(o_grp, hp.grp.data(), sizeof(GroupInfo) * hp.grp.size());
  put(o_mem, hp.members.data(), sizeof(int32_t) * hp.members.size());
  put(o_add, hp.len_add.data(), sizeof(int32_t) * hp.len_add.size());
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }

  DevPlan dp;
  dp.ctr = reinterpret_cast<uint32_t*>(base + o_ctr);
  dp.tickets = reinterpret_cast<uint32_t*>(base + o_tick);
  dp.witems = reinterpret_cast<const Item*>(base + o_wi);
  dp.ditems = reinterpret_cast<const Item*>(base + o_di);
  dp.req = reinterpret_cast<const ReqInfo*>(base + o_req);
  dp.grp = reinterpret_cast<const GroupInfo*>(base + o_grp);
  dp.members = reinterpret_cast<const int32_t*>(base + o_mem);
  dp.len_add = reinterpret_cast<const int32_t*>(base + o_add);
  dp.mlpart = reinterpret_cast<float2*>(base + o_ml);
  dp.opart = reinterpret_cast<float*>(base + o_op);
  dp.n_witems = (int32_t)hp.witems.size();
  dp.n_ditems = (int32_t)hp.ditems.size();
  dp.any_ragged = hp.any_ragged;
  return psattn_launch_decode(hp, dp, q, kv_pool, block_table, group_of_req, prefix_len,
                              suffix_len, out, lse, stream);
}
