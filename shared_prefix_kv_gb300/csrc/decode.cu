// The fused decode launch: one persistent kernel runs every partial of the
// batch (prefix chunks and suffix chunks, each against its KV range) and merges
// them exactly by online softmax, with no second kernel.
//
//   papercache.org, "BatchLLM ...", section 2.2 Eq. 1: attention over a
//     request's tokens = online-softmax reduction of partial attentions over a
//     split of those tokens (prefix part, distinct part);
//   same page, section 5: the partials are fused horizontally into one kernel
//     (different thread groups per part, different tile shapes per part);
//   same page, section 6.3.3: a long shared prefix is split along KV ("split-k").
//
// Partial representation (per q vector): m = running max of the scores in
// log2 units (score * scale * log2 e), l = sum of 2^(s - m), o = sum of
// 2^(s - m) * v.  Two partials combine as
//   m' = max(m1, m2), l' = l1 2^(m1-m') + l2 2^(m2-m'), o' = o1 2^(m1-m') + o2 2^(m2-m'),
// and the final output is o / l, LSE = (m + log2 l) * ln 2.
//
// Merge without a reduction kernel: every (request, KV head) has a ticket.
// An item that finishes a partial for it either sees that every other partial
// is already in (ticket == partials - 1) and merges straight from its
// registers, or writes its partial to the plan's slot array, fences, and takes
// a ticket; whoever takes the last ticket merges.  Nothing ever waits on
// another item.  The merger resets the ticket, and the last CTA to leave
// resets the work counters, so consecutive launches need no memset.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <climits>
#include <cstring>

#include "psattn_internal.h"

using namespace psattn;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = kWarpsPerCta * 32;

struct Params {
  CUtensorMap kv_map;  // the pool as [num_blocks * 2 * Hkv * 16 rows][d] bf16, 128B swizzle
  DevPlan dp;
  const void* q;
  const void* pool;
  const int32_t* bt;
  const int32_t* gor;
  const int32_t* plen;
  const int32_t* slen;
  void* out;
  float* lse;
  int R, Hq, Hkv, G, maxb, nblocks;
  float sl2;  // softmax scale * log2(e)
};

// ---------------------------------------------------------------- PTX helpers

// Streaming 128-bit load of KV data: read-only for the whole launch, not kept in L1.
__device__ __forceinline__ uint4 ld_kv(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void raise(const Params& P, uint32_t flag) {
  atomicOr(&P.dp.ctr[kCtrErr], flag);
}

// ------------------------------------------------------------ item resolution

struct Span {
  int rep;       // request whose block-table row names the blocks
  int col0;      // block-table column of the first block of the span
  int t0, t1;    // token range within the segment (t0 is a multiple of 16)
  int nmem;      // members (each contributes G q vectors)
  int mem_off;   // index into the member list (prefix items)
};

__device__ __forceinline__ int member_req(const Params& P, const Item& it, int m) {
  return it.kind == kItemSuffix ? it.seg : __ldg(&P.dp.members[it.mem_off + m]);
}

__device__ __forceinline__ Span resolve(const Params& P, const Item& it) {
  Span s;
  int len, chunk, nchunks, col_base;
  if (it.kind == kItemSuffix) {
    const ReqInfo ri = P.dp.req[it.seg];
    len = __ldg(&P.slen[it.seg]);
    chunk = ri.suffix_chunk;
    nchunks = ri.suffix_nchunks;
    col_base = ri.suffix_col;
    s.rep = it.seg;
    if (__ldg(&P.gor[it.seg]) != ri.leaf && (threadIdx.x & 31) == 0) raise(P, kErrGroup);
  } else {
    const GroupInfo gi = P.dp.grp[it.seg];
    len = __ldg(&P.plen[it.seg]) + __ldg(&P.dp.len_add[it.seg]);
    chunk = gi.chunk_tok;
    nchunks = gi.n_chunks;
    col_base = gi.col_base;
    s.rep = __ldg(&P.dp.members[it.mem_off]);
  }
  s.t0 = it.chunk * chunk;
  s.t1 = (it.chunk == nchunks - 1) ? len : min(len, s.t0 + chunk);
  if (s.t1 < s.t0) s.t1 = s.t0;
  s.col0 = col_base + s.t0 / kBlockSize;
  s.nmem = it.nmem;
  s.mem_off = it.mem_off;
  return s;
}

// Block ids of a span in a sliding 64-entry window: lane i holds the ids of
// local blocks base + i and base + 32 + i.  Out-of-range columns or ids raise
// the error word and read as -1 (the block is skipped, never dereferenced).
struct BlockWin {
  int lo, hi, base;
  __device__ __forceinline__ int fetch(const Params& P, const Span& s, int b, int nb) const {
    if (b >= nb) return -1;
    const int col = s.col0 + b;
    if (col >= P.maxb) {
      raise(P, kErrColumn);
      return -1;
    }
    const int id = __ldg(&P.bt[(size_t)s.rep * P.maxb + col]);
    if (id < 0 || id >= P.nblocks) {
      raise(P, kErrBlockOob);
      return -1;
    }
    return id;
  }
  __device__ __forceinline__ void init(const Params& P, const Span& s, int nb, int lane) {
    base = 0;
    lo = fetch(P, s, lane, nb);
    hi = fetch(P, s, 32 + lane, nb);
  }
  // keep local block bi in [base, base + 32) so that bi + d stays in the window for d < 32
  __device__ __forceinline__ void advance(const Params& P, const Span& s, int bi, int nb, int lane) {
    if (bi >= base + 32) {
      lo = hi;
      base += 32;
      hi = fetch(P, s, base + 32 + lane, nb);
    }
  }
  // warp-uniform b in [base, base + 64)
  __device__ __forceinline__ int get(int b) const {
    const int v = (b - base < 32) ? lo : hi;
    return __shfl_sync(0xffffffffu, v, (b - base) & 31);
  }
};

// Bulk prefetch of one (block, K|V, head) tile into L2 (no register or shared
// memory cost); keeps several tiles per warp in flight ahead of the loads.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

#ifndef PSATTN_PREFETCH_BLOCKS
#define PSATTN_PREFETCH_BLOCKS 2
#endif
constexpr int kPrefetchBlocks = PSATTN_PREFETCH_BLOCKS;  // prefetch distance in blocks (0: off)
static_assert(kPrefetchBlocks >= 0 && kPrefetchBlocks < 32, "prefetch distance");

// ------------------------------------------------------------------- merging

// Unnormalised partial owned by one lane: NR rows (local row index, -1 = none)
// x NS segments of SEG consecutive d values each.
template <int NR, int NS, int SEG>
struct Own {
  int row[NR];
  int d0[NS];
  float v[NR][NS][SEG];
  float m[NR], l[NR];
  bool ml_owner;  // this lane writes m, l and lse of its rows
};

template <typename OutT>
__device__ __forceinline__ void store_out(OutT* dst, const float* v, int n);

template <>
__device__ __forceinline__ void store_out<float>(float* dst, const float* v, int n) {
  for (int i = 0; i < n; i += 4)
    *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}

template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* dst, const float* v, int n) {
  if (n == 8) {
    uint4 w = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                         pack_bf16(v[6], v[7]));
    *reinterpret_cast<uint4*>(dst) = w;
  } else {
    for (int i = 0; i < n; i += 2) *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16(v[i], v[i + 1]);
  }
}

// Finish the partial of one item for every (request, KV head) unit it covers:
// write-and-ticket, or merge, as described at the top of this file.
template <typename OutT, int D, int NR, int NS, int SEG>
__device__ __forceinline__ void finish_item(const Params& P, const Item& it, Own<NR, NS, SEG>& own,
                                            int lane) {
  const int G = P.G, h = it.kvh;
  for (int mu = 0; mu < it.nmem; ++mu) {
    const int r = member_req(P, it, mu);
    const ReqInfo ri = P.dp.req[r];
    uint32_t* ticket = &P.dp.tickets[(size_t)r * P.Hkv + h];
    const uint32_t need = (uint32_t)ri.n_partials - 1u;
    int fast = 0;
    if (lane == 0) fast = ld_acquire(ticket) == need;
    fast = __shfl_sync(0xffffffffu, fast, 0);
    int last = fast;
    if (!fast) {
      const size_t slot = (size_t)ri.slot_base + it.slot_j;
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        const int rho = own.row[k];
        if (rho < mu * G || rho >= (mu + 1) * G) continue;
        const size_t rix = (slot * P.Hkv + h) * G + (rho - mu * G);
        float* dst = P.dp.opart + rix * D;
#pragma unroll
        for (int sg = 0; sg < NS; ++sg)
#pragma unroll
          for (int e = 0; e < SEG; e += 4)
            __stcg(reinterpret_cast<float4*>(dst + own.d0[sg] + e),
                   make_float4(own.v[k][sg][e], own.v[k][sg][e + 1], own.v[k][sg][e + 2],
                               own.v[k][sg][e + 3]));
        if (own.ml_owner) __stcg(&P.dp.mlpart[rix], make_float2(own.m[k], own.l[k]));
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) last = atom_add_acq_rel(ticket, 1u) == need;
      last = __shfl_sync(0xffffffffu, last, 0);
    }
    if (!last) continue;
    __threadfence();
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      const int rho = own.row[k];
      const bool mine = rho >= mu * G && rho < (mu + 1) * G;
      if (!mine) continue;
      const int hl = rho - mu * G;
      float M = own.m[k], L = own.l[k];
      float acc[NS][SEG];
#pragma unroll
      for (int sg = 0; sg < NS; ++sg)
#pragma unroll
        for (int e = 0; e < SEG; ++e) acc[sg][e] = own.v[k][sg][e];
      for (int j = 0; j < ri.n_partials; ++j) {
        if (j == it.slot_j) continue;
        const size_t rix = (((size_t)ri.slot_base + j) * P.Hkv + h) * G + hl;
        // m, l and O of the partial are loaded together (one round trip); an
        // empty partial (m = -inf) is skipped after the loads
        const float2 ml = __ldcg(&P.dp.mlpart[rix]);
        const float* src = P.dp.opart + rix * D;
        float4 w[NS][SEG / 4];
#pragma unroll
        for (int sg = 0; sg < NS; ++sg)
#pragma unroll
          for (int e = 0; e < SEG; e += 4)
            w[sg][e / 4] = __ldcg(reinterpret_cast<const float4*>(src + own.d0[sg] + e));
        if (ml.x == -INFINITY) continue;
        const float Mn = fmaxf(M, ml.x);
        const float a = ex2(M - Mn), b = ex2(ml.x - Mn);
        L = L * a + ml.y * b;
        M = Mn;
#pragma unroll
        for (int sg = 0; sg < NS; ++sg)
#pragma unroll
          for (int e = 0; e < SEG; e += 4) {
            acc[sg][e] = acc[sg][e] * a + w[sg][e / 4].x * b;
            acc[sg][e + 1] = acc[sg][e + 1] * a + w[sg][e / 4].y * b;
            acc[sg][e + 2] = acc[sg][e + 2] * a + w[sg][e / 4].z * b;
            acc[sg][e + 3] = acc[sg][e + 3] * a + w[sg][e / 4].w * b;
          }
      }
      const int hq = h * G + hl;
      const bool empty = !(L > 0.f);
      const float inv = empty ? 0.f : 1.f / L;
      OutT* dst = reinterpret_cast<OutT*>(P.out) + ((size_t)r * P.Hq + hq) * D;
#pragma unroll
      for (int sg = 0; sg < NS; ++sg) {
        float o[SEG];
#pragma unroll
        for (int e = 0; e < SEG; ++e) o[e] = acc[sg][e] * inv;
        store_out<OutT>(dst + own.d0[sg], o, SEG);
      }
      if (own.ml_owner) {
        if (empty) raise(P, kErrEmpty);
        if (P.lse) P.lse[(size_t)r * P.Hq + hq] = empty ? -INFINITY : (M + __log2f(L)) * kLn2;
      }
    }
    __syncwarp();
    if (lane == 0) st_relaxed(ticket, 0u);
  }
}

// ------------------------------------------ bf16, d = 128: mma.sync warp item
//
// A warp serves up to 8 q vectors ("rows") that share a KV head and a token
// range, one 16-token block at a time, reading each K and V tile of the block
// once with coalesced 128-bit loads that feed the tensor-core fragments
// directly (no shared-memory staging):
//   S[rows x 16 tok] = Q[rows x 128] . K^T     (m16n8k16, rows padded to 16,
//                                                tokens as two n-tiles of 8)
//   O^T[128 x rows] += V^T[128 x 16 tok] . P^T (m16n8k16, d as 8 m-tiles,
//                                                rows as the n = 8 dimension)
// The d index is permuted consistently between Q and K (the reduction order
// does not matter), so lane (g, tig) loads 16-byte chunks tig, tig+4, tig+8,
// tig+12 of K rows g and g+8 and uses them unchanged as B fragments.  For V,
// lane (g, tig) loads chunks g and g+8 of tokens 2tig, 2tig+1, 2tig+8, 2tig+9
// and forms the A fragments with byte permutes; m-tile i, m-row g then holds
// d = 8g + i and m-row g+8 holds d = 64 + 8g + i.  The S accumulator of row g
// sits exactly where the P^T B fragment needs it, so softmax needs shuffles
// only for the row max / sum.

__device__ __forceinline__ void mma_item(const Params& P, const Item& it, int lane) {
  constexpr int D = 128;
  const int g = lane >> 2, tig = lane & 3;
  const int G = P.G, h = it.kvh;
  const Span s = resolve(P, it);
  const int nrows = s.nmem * G;

  // Q fragments: row g, slice k: chunk (tig + 4*(k>>1)), words 2(k&1) and 2(k&1)+1.
  // lim: tokens of the span row g attends to (less than the span only on a
  // ragged leaf level, whose members see its first leaf_vis tokens)
  uint32_t qa0[8], qa2[8];
  int lim = INT_MAX;
  if (g < nrows) {
    const int r = member_req(P, it, g / G);
    if (P.dp.any_ragged && it.kind != kItemSuffix) {
      const ReqInfo ri = P.dp.req[r];
      if (ri.leaf_vis >= 0 && ri.leaf == it.seg) lim = ri.leaf_vis - s.t0;
    }
    const __nv_bfloat16* qp =
        reinterpret_cast<const __nv_bfloat16*>(P.q) + ((size_t)r * P.Hq + h * G + g % G) * D;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(qp + 8 * (tig + 4 * u)));
      qa0[2 * u] = w.x; qa2[2 * u] = w.y; qa0[2 * u + 1] = w.z; qa2[2 * u + 1] = w.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) qa0[k] = qa2[k] = 0u;
  }

  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // row g; l_run is this lane's share

  const int nb = (s.t1 > s.t0) ? (s.t1 - s.t0 + kBlockSize - 1) / kBlockSize : 0;
  const size_t head_stride = (size_t)kBlockSize * D;  // elements of one (block, K|V, head) tile
  const __nv_bfloat16* pool = reinterpret_cast<const __nv_bfloat16*>(P.pool);
  const uint32_t tile_bytes = (uint32_t)(head_stride * sizeof(__nv_bfloat16));
  BlockWin win;
  win.init(P, s, nb, lane);
  auto prefetch_block = [&](int id) {
    prefetch_l2(pool + ((size_t)id * 2 * P.Hkv + h) * head_stride, tile_bytes);
    prefetch_l2(pool + (((size_t)id * 2 + 1) * P.Hkv + h) * head_stride, tile_bytes);
  };
  // lane i already holds the id of local block i: no shuffle (a full-mask
  // shuffle here would be reached by only some lanes)
  if (lane < kPrefetchBlocks && win.lo >= 0) prefetch_block(win.lo);
  uint4 kr[2][4];
  int id_next = nb > 0 ? win.get(0) : -1;
  auto load_k = [&](int id) {
    const __nv_bfloat16* kb = pool + ((size_t)id * 2 * P.Hkv + h) * head_stride;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) kr[j][u] = ld_kv(kb + (8 * j + g) * D + 8 * (tig + 4 * u));
  };
  if (id_next >= 0) load_k(id_next);

  for (int bi = 0; bi < nb; ++bi) {
    win.advance(P, s, bi, nb, lane);
    if (kPrefetchBlocks > 0 && bi + kPrefetchBlocks < nb) {
      const int pid = win.get(bi + kPrefetchBlocks);
      if (lane == 0 && pid >= 0) prefetch_block(pid);
    }
    const int id = id_next;
    const int nvalid = min(kBlockSize, s.t1 - (s.t0 + bi * kBlockSize));
    uint4 vr[4][2];
    const int tv[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
    if (id >= 0) {
      const __nv_bfloat16* vb = pool + (((size_t)id * 2 + 1) * P.Hkv + h) * head_stride;
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int c = 0; c < 2; ++c) vr[t][c] = ld_kv(vb + tv[t] * D + 8 * (g + 8 * c));
    }
    float acc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 kv = kr[j][k >> 1];
        mma16816(acc[j], qa0[k], 0u, qa2[k], 0u, (k & 1) ? kv.z : kv.x, (k & 1) ? kv.w : kv.y);
      }
    }
    if (bi + 1 < nb) {
      id_next = win.get(bi + 1);
      if (id_next >= 0) load_k(id_next);
    }
    if (id < 0) continue;

    // scores of row g for tokens 2tig, 2tig+1, 2tig+8, 2tig+9
    float x[4] = {acc[0][0], acc[0][1], acc[1][0], acc[1][1]};
    float mx = -INFINITY;
    const int tok0 = bi * kBlockSize;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i] = (tv[i] < nvalid && tok0 + tv[i] < lim) ? x[i] * P.sl2 : -INFINITY;
      mx = fmaxf(mx, x[i]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // -inf only for a row that has seen no token yet (padding rows, or a
    // ragged row past its limit): then O and l are 0 and stay 0
    const float m_new = fmaxf(m_run, mx);
    const float mref = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = ex2(m_run - mref);
    float p[4], psum = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      p[i] = ex2(x[i] - mref);
      psum += p[i];
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    // rescale O^T columns (rows 2tig, 2tig+1) by their rows' alpha
    const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * tig);
    const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * tig + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= a0; o[i][1] *= a1; o[i][2] *= a0; o[i][3] *= a1;
    }
    // tokens past the segment end may hold anything (even NaN): zero their V
    if (nvalid < kBlockSize) {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (tv[t] >= nvalid) vr[t][0] = vr[t][1] = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint32_t pb0 = pack_bf16(p[0], p[1]), pb1 = pack_bf16(p[2], p[3]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t sel = (i & 1) ? 0x7632u : 0x5410u;
      const int w = i >> 1;
      const uint32_t* x0 = reinterpret_cast<const uint32_t*>(&vr[0][0]);
      const uint32_t* x1 = reinterpret_cast<const uint32_t*>(&vr[1][0]);
      const uint32_t* y0 = reinterpret_cast<const uint32_t*>(&vr[0][1]);
      const uint32_t* y1 = reinterpret_cast<const uint32_t*>(&vr[1][1]);
      const uint32_t* z0 = reinterpret_cast<const uint32_t*>(&vr[2][0]);
      const uint32_t* z1 = reinterpret_cast<const uint32_t*>(&vr[3][0]);
      const uint32_t* u0 = reinterpret_cast<const uint32_t*>(&vr[2][1]);
      const uint32_t* u1 = reinterpret_cast<const uint32_t*>(&vr[3][1]);
      mma16816(o[i], __byte_perm(x0[w], x1[w], sel), __byte_perm(y0[w], y1[w], sel),
               __byte_perm(z0[w], z1[w], sel), __byte_perm(u0[w], u1[w], sel), pb0, pb1);
    }
  }

  // full row sum of row g
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

  Own<2, 2, 8> own;
  own.row[0] = (2 * tig < nrows) ? 2 * tig : -1;
  own.row[1] = (2 * tig + 1 < nrows) ? 2 * tig + 1 : -1;
  own.d0[0] = 8 * g;
  own.d0[1] = 64 + 8 * g;
  own.m[0] = __shfl_sync(0xffffffffu, m_run, 8 * tig);
  own.l[0] = __shfl_sync(0xffffffffu, l_run, 8 * tig);
  own.m[1] = __shfl_sync(0xffffffffu, m_run, 8 * tig + 4);
  own.l[1] = __shfl_sync(0xffffffffu, l_run, 8 * tig + 4);
  own.ml_owner = (g == 0);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    own.v[0][0][i] = o[i][0];
    own.v[1][0][i] = o[i][1];
    own.v[0][1][i] = o[i][2];
    own.v[1][1][i] = o[i][3];
  }
  finish_item<__nv_bfloat16, D>(P, it, own, lane);
}

// ---------------------------------------------- CUDA-core (SIMT) warp item
//
// Up to 4 rows; lanes split one token row into 16-byte slices (LPR lanes per
// row, TPW tokens per warp load).  Each lane group keeps its own online-softmax
// state over its tokens; the groups are merged with shuffles at the end.

template <typename T>
__device__ __forceinline__ void widen16(const uint4 w, float* f);

template <>
__device__ __forceinline__ void widen16<float>(const uint4 w, float* f) {
  f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
  f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
}

template <>
__device__ __forceinline__ void widen16<__nv_bfloat16>(const uint4 w, float* f) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

template <typename T, int D>
__device__ __forceinline__ void simt_item(const Params& P, const Item& it, int lane) {
  constexpr int EPL = 16 / (int)sizeof(T);          // elements per lane load
  constexpr int LPR = D / EPL;                      // lanes per token row
  constexpr int TPW = 32 / LPR;                     // tokens per warp load
  constexpr int NR = kSimtRows;
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row split");
  const int tau = lane / LPR, sl = lane % LPR;
  const int G = P.G, h = it.kvh;
  const Span s = resolve(P, it);
  const int nrows = s.nmem * G;

  float qf[NR][EPL];
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    if (k < nrows) {
      const int r = member_req(P, it, k / G);
      const T* qp = reinterpret_cast<const T*>(P.q) + ((size_t)r * P.Hq + h * G + k % G) * D;
      widen16<T>(__ldg(reinterpret_cast<const uint4*>(qp + sl * EPL)), qf[k]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) qf[k][e] = 0.f;
    }
  }
  float m[NR], l[NR], o[NR][EPL];
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    m[k] = -INFINITY; l[k] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[k][e] = 0.f;
  }
  const int nb = (s.t1 > s.t0) ? (s.t1 - s.t0 + kBlockSize - 1) / kBlockSize : 0;
  const size_t head_stride = (size_t)kBlockSize * D;
  const T* pool = reinterpret_cast<const T*>(P.pool);
  const uint32_t tile_bytes = (uint32_t)(head_stride * sizeof(T));
  BlockWin win;
  win.init(P, s, nb, lane);
  if (lane < kPrefetchBlocks && win.lo >= 0) {
    prefetch_l2(pool + ((size_t)win.lo * 2 * P.Hkv + h) * head_stride, tile_bytes);
    prefetch_l2(pool + (((size_t)win.lo * 2 + 1) * P.Hkv + h) * head_stride, tile_bytes);
  }
  for (int bi = 0; bi < nb; ++bi) {
    win.advance(P, s, bi, nb, lane);
    if (kPrefetchBlocks > 0 && bi + kPrefetchBlocks < nb) {
      const int pid = win.get(bi + kPrefetchBlocks);
      if (lane == 0 && pid >= 0) {
        prefetch_l2(pool + ((size_t)pid * 2 * P.Hkv + h) * head_stride, tile_bytes);
        prefetch_l2(pool + (((size_t)pid * 2 + 1) * P.Hkv + h) * head_stride, tile_bytes);
      }
    }
    const int id = win.get(bi);
    if (id < 0) continue;
    const int nvalid = min(kBlockSize, s.t1 - (s.t0 + bi * kBlockSize));
    const T* kb = pool + ((size_t)id * 2 * P.Hkv + h) * head_stride;
    const T* vb = kb + (size_t)P.Hkv * head_stride;
#pragma unroll
    for (int tk = 0; tk < kBlockSize / TPW; ++tk) {
      const int t = tk * TPW + tau;
      float kf[EPL], vf[EPL];
      widen16<T>(ld_kv(kb + t * D + sl * EPL), kf);
      widen16<T>(ld_kv(vb + t * D + sl * EPL), vf);
      const bool valid = t < nvalid;
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qf[k][e], kf[e], dot);
#pragma unroll
        for (int off = 1; off < LPR; off <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        if (valid) {
          const float x = dot * P.sl2;
          const float mn = fmaxf(m[k], x);
          const float a = ex2(m[k] - mn), pw = ex2(x - mn);
          l[k] = l[k] * a + pw;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[k][e] = o[k][e] * a + pw * vf[e];
          m[k] = mn;
        }
      }
    }
  }
  // merge the TPW token groups (lanes tau*LPR + sl, same sl)
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[k], off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[k], off);
      const float mn = fmaxf(m[k], m2);
      const float a = (m[k] == -INFINITY) ? 0.f : ex2(m[k] - mn);
      const float b = (m2 == -INFINITY) ? 0.f : ex2(m2 - mn);
      l[k] = l[k] * a + l2 * b;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float o2 = __shfl_xor_sync(0xffffffffu, o[k][e], off);
        o[k][e] = o[k][e] * a + o2 * b;
      }
      m[k] = mn;
    }
  }
  Own<NR, 1, EPL> own;
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    own.row[k] = (tau == 0 && k < nrows) ? k : -1;
    own.m[k] = m[k];
    own.l[k] = l[k];
#pragma unroll
    for (int e = 0; e < EPL; ++e) own.v[k][0][e] = o[k][e];
  }
  own.d0[0] = sl * EPL;
  own.ml_owner = (lane == 0);
  finish_item<T, D>(P, it, own, lane);
}

// ------------------------------------ tensor-core prefix tile (tcgen05 + TMA)
//
// A dense item is (group, KV head, chunk of the group's level, up to 128/G
// members): 128 rows of q (member x q head of the KV head; padding rows are
// zero) against the chunk's K/V, read once for all rows (the prefix partial as
// a matrix product, BatchLLM section 2.2).  Eight warps of the CTA run it:
//
//   warps 0-3   softmax and epilogue, thread t owning row t (= TMEM lane t);
//   warp 4      lane 0 issues the S = Q K^T MMAs and their commits;
//   warps 5, 6  TMA producers of the K and the V tiles;
//   warp 7      lane 0 issues the PV MMAs and their commits.
// Warps 8-11 run per-warp items meanwhile (one per SM sub-partition).
//
// For each 128-token tile g (counted across items, so the rings continue):
//   TMA       K(g), V(g): 8 paged blocks x 2 halves of d, 128B-swizzled boxes
//             of 16 rows x 64 columns from the pool (tensor map over the pool
//             as [rows = block*2*Hkv*16][d]), into K and V rings of three
//             stages; a stage is refilled as soon as the MMA that read it is
//             done;
//   S(g)      = Q K(g)^T, tcgen05.mma kind::f16 M 128 N 128 K 128, fp32 into
//             TMEM buffer g & 1 (columns 0-127 or 128-255);
//   softmax   reads S(g) from TMEM, keeps a running max m in log2 units that
//             moves only when the tile max exceeds it by more than 8 (then O
//             is rescaled in TMEM), writes P = 2^(s - m) as bf16 pairs back
//             into TMEM (columns 384-447 or 448-511, one row per lane);
//   PV(g)     O += P V(g), P as the A operand straight from TMEM, V as the
//             MN-major B operand from shared memory, fp32 in TMEM columns
//             256-383.
// S(g + 1) is issued while the softmax works on S(g), so the tensor core and
// the softmax overlap.  Every wait is bounded: on a timeout the CTA
// raises the error word, sets an abort flag that makes every later wait
// return at once, and leaves its dense work.

constexpr int kTileTok = 128;
constexpr uint32_t kTileBytes = 128 * 128 * 2;          // one 128 x 128 bf16 operand tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;         // one 64-column half (K atom)
constexpr int kStages = 3;                              // K and V ring depth
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTileBytes;                  // kStages K stages
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;  // kStages V stages
// between items the K stages hold the epilogue's O staging, [128][kERow]
// fp32 (a row of 128 values and a 16-byte pad)
constexpr uint32_t kOffE = kOffK;
constexpr int kERow = 132;
static_assert(128 * kERow * 4 <= kStages * kTileBytes, "O staging overruns the K stages");
static_assert((kERow * 4) % 16 == 0, "bulk copies need 16-byte aligned staging rows");
constexpr int kMaxDenseBlocks = 512;                    // chunk <= 8192 tokens
constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;  // 21 mbarriers
constexpr uint32_t kOffMisc = kOffBar + 168;
constexpr uint32_t kDenseSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
static_assert(kDenseSmemBytes <= 232448, "dense tile shared memory exceeds 227 KB");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;                        // O accumulator columns
constexpr uint32_t kTmemP = 384;                        // two P buffers of 64 columns
// A row's running max m moves only when the row's sum of P = 2^(s - m) over
// a tile exceeds 2^PSATTN_RESCALE_LOG2_SUM (then some P exceeds 2^8: m is at
// least 8 below the row's values).  P, O and l stay far inside the bf16 and
// fp32 ranges below that, so only this bound on their size matters.
#ifndef PSATTN_RESCALE_LOG2_SUM
#define PSATTN_RESCALE_LOG2_SUM 15
#endif
constexpr float kRescaleSumLimit = (float)(1u << PSATTN_RESCALE_LOG2_SUM);
constexpr uint64_t kWaitLimitNs = 2000000000ull;        // 2 s per wait
constexpr int kDenseThreads = 256;                      // warps 0-7


__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier; false on timeout or when
// another thread of the dense group has already given up (*abort != 0).
// Parity waits are sound only when the waiter knows the previous phase has
// completed and the next one cannot complete before it looks: every wait in
// this file is placed so that both hold (a stage, buffer or product two phases
// ahead always depends on something the waiter itself has not yet released).
__device__ __forceinline__ bool mbar_wait_ns(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  return mbar_wait_ns(bar, parity, abort, kWaitLimitNs);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}


__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One bulk copy of `bytes` (a multiple of 16) from shared to global memory
// by the TMA engine; both addresses 16-byte aligned.  The shared source must
// have been made visible to the async proxy (fence_proxy_async) first.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}

// Commits this thread's bulk copies and waits until they are complete (the
// global writes done, the shared sources read); the writes are then ordered
// before this thread's later generic-proxy operations.
__device__ __forceinline__ void bulk_commit_and_wait() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// named barrier 1 over the 256 threads of warps 0-7 (the dense group)
// (non-aligned form: lanes of the MMA and producer warps may arrive apart)
__device__ __forceinline__ void dense_sync() { asm volatile("barrier.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with the A operand read from TMEM (rows in lanes 0-127, K along
// columns, two bf16 per 32-bit column).
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane; the caller waits
// (tmem_wait_st) before the values are published
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane, without the wait
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (start, leading and stride
// byte offsets in 16-byte units; bits 46-48 fixed 0b001; layout 2 = SW128).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = 128, N = 128;
// b_mn_major selects an MN-major B operand.
__host__ __device__ constexpr uint32_t idesc_bf16_m128_n128(bool b_mn_major) {
  return (1u << 4)            // D format fp32
         | (1u << 7)          // A format bf16
         | (1u << 10)         // B format bf16
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((128u >> 3) << 17)  // N / 8
         | ((128u >> 4) << 24); // M / 16
}


struct DenseState {
  uint8_t* smem;       // 1024-aligned
  uint32_t sbase;      // its shared-space address
  uint32_t tmem;       // TMEM base address
  uint32_t g;          // tiles this CTA has run so far (drives every ring phase)
  uint32_t xph;        // completions of the softmax threads' exchange barrier so far
  volatile int* abort;
  // softmax threads: the item's member tickets (lane mu: member mu's unit
  // r * Hkv + h and partial count)
  uint32_t pend_unit;
  int pend_np;
  int pend_valid;      // this lane has a member
  int pend_any;        // the warp has tickets pending (same in every lane)
};

// mbarrier slots.  Tile g uses K/V stage g % kStages (completion number
// g / kStages on that stage's barriers) and TMEM S and P buffers g % 2
// (completion number g / 2).
//   k[st], v[st]      K / V of the stage landed (TMA byte count)
//   kfree[st]         S of the stage's tile done (its K may be overwritten)
//   vfree[st]         PV of the stage's tile done (its V may be overwritten)
//   s[b]              S(g) in TMEM buffer b
//   sfree[b]          the four softmax warps have read S buffer b
//   p[b]              the four softmax warps have written P buffer b (one
//                     barrier per buffer: a warp a tile ahead arrives on the
//                     other one and cannot complete a phase for a tile the
//                     slower warps have not finished)
//   pfree[b]          PV of P buffer b done (P may be rewritten; O updated)
//   x                 all 128 softmax threads reached the same point of an
//                     item's epilogue (the exchange between row copies)
__device__ __forceinline__ uint32_t bar_k(const DenseState& d, uint32_t st) { return d.sbase + kOffBar + 8u * st; }
__device__ __forceinline__ uint32_t bar_v(const DenseState& d, uint32_t st) { return d.sbase + kOffBar + 24u + 8u * st; }
__device__ __forceinline__ uint32_t bar_s(const DenseState& d, uint32_t b) { return d.sbase + kOffBar + 48u + 8u * b; }
__device__ __forceinline__ uint32_t bar_sfree(const DenseState& d, uint32_t b) { return d.sbase + kOffBar + 64u + 8u * b; }
__device__ __forceinline__ uint32_t bar_p(const DenseState& d, uint32_t b) { return d.sbase + kOffBar + 80u + 8u * b; }
__device__ __forceinline__ uint32_t bar_pfree(const DenseState& d, uint32_t b) { return d.sbase + kOffBar + 96u + 8u * b; }
__device__ __forceinline__ uint32_t bar_kfree(const DenseState& d, uint32_t st) { return d.sbase + kOffBar + 112u + 8u * st; }
__device__ __forceinline__ uint32_t bar_vfree(const DenseState& d, uint32_t st) { return d.sbase + kOffBar + 136u + 8u * st; }
__device__ __forceinline__ uint32_t bar_x(const DenseState& d) { return d.sbase + kOffBar + 160u; }

// Row copies of a small dense item.  An item of at most 32 (64) q rows runs
// each row as 4 (2) copies in the four (two) TMEM lane quadrants: copy c of
// row rho sits at lane c * width + rho and takes only the tile columns
// [c * width, (c + 1) * width) of every tile, with its own running max, sum
// and O.  Each softmax thread then passes over 32 (64) columns of a tile
// instead of 128, and the copies are merged by their maxima in the epilogue
// (the online-softmax combination of partials over disjoint token sets).
__device__ __forceinline__ int copy_width(int nrows) {
  return nrows <= 32 ? 32 : (nrows <= 64 ? 64 : kTileTok);
}

// Block-table lookup for the K or V tile of local tile j, by the 32 lanes of a
// producer warp: lanes 0-15 each take one of the tile's 8 blocks (lane / 2)
// and one 64-column half of it (lane % 2); returns the pool row of that block
// half's 16 tokens, -1 for lanes without one (bad ids raise the error word
// and are skipped).
__device__ __forceinline__ int kv_row(const Params& P, const Span& s, int h, int kv, int j, int nb,
                                      int lane) {
  const int b = j * (kTileTok / kBlockSize) + (lane >> 1);
  int row = -1;
  if (lane < 16 && b < nb) {
    const int col = s.col0 + b;
    if (col >= P.maxb) {
      raise(P, kErrColumn);
    } else {
      const int id = __ldg(&P.bt[(size_t)s.rep * P.maxb + col]);
      if (id < 0 || id >= P.nblocks) raise(P, kErrBlockOob);
      else row = ((id * 2 + kv) * P.Hkv + h) * kBlockSize;
    }
  }
  return row;
}

// TMA of one K or V tile into stage st from the rows kv_row looked up; lane 0
// first posts the byte count.
__device__ __forceinline__ void issue_kv(const Params& P, const DenseState& d, int kv, uint32_t st,
                                         int row, int lane) {
  const uint32_t valid = __ballot_sync(0xffffffffu, row >= 0);
  const uint32_t bar = kv ? bar_v(d, st) : bar_k(d, st);
  if (lane == 0) mbar_expect_tx(bar, (uint32_t)__popc(valid) * (kBlockSize * 64u * 2u));
  __syncwarp();
  if (row >= 0) {
    const uint32_t dst = d.sbase + (kv ? kOffV : kOffK) + st * kTileBytes + (lane & 1) * kHalfBytes +
                         (uint32_t)(lane >> 1) * (kBlockSize * 128u);
    tma_load_2d(dst, &P.kv_map, (lane & 1) * 64, row, bar);
  }
}

// The tensor-core issue of one item, split over two threads so that neither
// waits behind the other: issuing a tcgen05.mma blocks while the tensor core
// is busy, and S(g + 1) should not queue behind PV(g - 1), which waits for
// the slowest softmax warp.  (Commits track the committing thread's own
// MMAs.)
//   lane 0 of warp 4: S(g) once K(g) has landed and the softmax is done with
//     S(g - 2); commits to s[g % 2] and kfree[stage].
//   lane 0 of warp 7: PV(g) once P(g) is written and V(g) has landed;
//     commits to pfree[g % 2] and vfree[stage].
// Parity soundness (see mbar_wait): each thread saw the previous completion
// of every barrier it waits on (its own earlier wait, or the previous item),
// and the next completion needs an MMA it has not issued yet: K(g + 3) needs
// kfree for S(g), sfree for S(g) needs S(g), V(g + 3) needs vfree for PV(g),
// and P(g + 2) needs the softmax's wait for PV(g) (P buffer reuse).
__device__ void mma_s_item(const Params& P, DenseState& d, int ntiles) {
  if ((threadIdx.x & 31) != 0) return;
  const uint32_t g0 = d.g;
  const uint32_t idesc_s = idesc_bf16_m128_n128(false);
  const uint64_t qdesc = sw128_desc(d.sbase + kOffQ, 16, 1024);
  for (int j = 0; j < ntiles; ++j) {
    const uint32_t g = g0 + j, b = g & 1, st = g % kStages;
    if (!mbar_wait(bar_k(d, st), (g / kStages) & 1, d.abort)) return;
    if (g >= 2 && !mbar_wait(bar_sfree(d, b), ((g >> 1) - 1) & 1, d.abort)) return;
    tc_fence_after();
    const uint64_t kdesc = sw128_desc(d.sbase + kOffK + st * kTileBytes, 16, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t koff = ((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4;
      tc_mma(d.tmem + b * 128, qdesc + koff, kdesc + koff, idesc_s, k > 0);
    }
    tc_commit(bar_s(d, b));
    tc_commit(bar_kfree(d, st));
  }
}

__device__ void mma_pv_item(const Params& P, DenseState& d, int ntiles) {
  if ((threadIdx.x & 31) != 0) return;
  const uint32_t g0 = d.g;
  const uint32_t idesc_o = idesc_bf16_m128_n128(true);
  for (int j = 0; j < ntiles; ++j) {
    const uint32_t g = g0 + j, st = g % kStages;
    if (!mbar_wait(bar_p(d, g & 1), (g >> 1) & 1, d.abort)) return;
    if (!mbar_wait(bar_v(d, st), (g / kStages) & 1, d.abort)) return;
    tc_fence_after();
    const uint64_t vdesc = sw128_desc(d.sbase + kOffV + st * kTileBytes, kHalfBytes, 1024);
#pragma unroll
    for (int k = 0; k < 8; ++k)  // 16 tokens of P = 8 TMEM columns per step
      tc_mma_ta(d.tmem + kTmemO, d.tmem + kTmemP + (g & 1) * 64 + k * 8,
                vdesc + ((k * 16 * 128) >> 4), idesc_o, (j > 0 || k > 0));
    tc_commit(bar_pfree(d, g & 1));
    tc_commit(bar_vfree(d, st));
  }
}

// The producer warps' part of one item: warp 5 issues the K copies, warp 6
// the V copies.  The first kStages tiles go straight into their stages (the
// previous item is done with every stage); tile g >= kStages waits for the
// stage's previous tile g - kStages to be consumed (kfree / vfree).  The block
// ids of a tile are looked up before that wait, so the lookup's latency
// overlaps it.
__device__ void producer_item(const Params& P, DenseState& d, const Span& s, int h, int kv, int nb,
                              int ntiles) {
  const int lane = threadIdx.x & 31;
  const uint32_t g0 = d.g;
  auto wait0 = [&](uint32_t bar, uint32_t parity) -> bool {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, d.abort);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  for (int j = 0; j < ntiles; ++j) {
    const uint32_t g = g0 + j, st = g % kStages;
    const int row = kv_row(P, s, h, kv, j, nb, lane);
    if (j >= kStages &&
        !wait0(kv ? bar_vfree(d, st) : bar_kfree(d, st), ((g / kStages) - 1) & 1))
      return;
    issue_kv(P, d, kv, st, row, lane);
  }
}

// The Q tile of one item (threads 0-127); returns the request of the
// thread's row (-1 past the item's rows).  Tile row t holds q row t % width
// (copy_width): small items repeat their rows in every lane quadrant.
__device__ int prepare_item(const Params& P, DenseState& d, const Item& it, int nrows) {
  const int tid = threadIdx.x, G = P.G, h = it.kvh;
  const int rho = tid % copy_width(nrows);
  // Q tile, K-major, 128B swizzle: 16-byte chunk c of row t at
  // atom (c / 8), row t, position (c % 8) ^ (t % 8)
  uint8_t* qs = d.smem + kOffQ;
  const __nv_bfloat16* qp = nullptr;
  int r = -1;
  if (rho < nrows) {
    r = member_req(P, it, rho / G);
    qp = reinterpret_cast<const __nv_bfloat16*>(P.q) + ((size_t)r * P.Hq + h * G + rho % G) * 128;
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint4 w = qp ? __ldg(reinterpret_cast<const uint4*>(qp + 8 * c)) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalfBytes + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)) = w;
  }
  fence_proxy_async();
  return r;
}

// Row max of S(g) (scaled to log2 units) over the valid columns of the NQ
// groups of 32 columns at sa.
template <int NQ>
__device__ __forceinline__ float tile_max(uint32_t sa, float sl2, int tile_valid) {
  float mxa[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mxa[i] = -INFINITY;
#pragma unroll
  for (int q4 = 0; q4 < NQ; ++q4) {
    float v[32];
    tmem_ld32(sa + q4 * 32, v);
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (q4 * 32 + e < tile_valid) mxa[e & 7] = fmaxf(mxa[e & 7], v[e]);
  }
  return fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
               fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7]))) * sl2;
}

// One pass over NQ x 32 columns of S(g) of this thread's row: P = 2^(s * sl2
// - m) as bf16 pairs into the row's TMEM lane at pa (token 2c and 2c + 1 in
// column c, the lower token in the low half), columns past tile_valid as 0
// (kFull: every column is valid, no masks).  Returns the row sum of P (fp32).
// The next 32 columns of S are loaded while this 32 are computed.
template <int NQ, bool kFull>
__device__ __forceinline__ float softmax_pass(uint32_t sa, float sl2, float m, int tile_valid,
                                              uint32_t pa) {
  const float2 sl2_2 = make_float2(sl2, sl2), negm_2 = make_float2(-m, -m);
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  uint32_t r[2][32];
  tmem_ld32_async(sa, r[0]);
  tmem_wait_ld();
#pragma unroll
  for (int q4 = 0; q4 < NQ; ++q4) {
    if (q4 + 1 < NQ) tmem_ld32_async(sa + (q4 + 1) * 32, r[(q4 + 1) & 1]);
    const uint32_t* v = r[q4 & 1];
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                  sl2_2, negm_2);
      float p0 = ex2(x.x), p1 = ex2(x.y);
      if (!kFull) {
        const int c = q4 * 32 + e;
        p0 = c < tile_valid ? p0 : 0.f;
        p1 = c + 1 < tile_valid ? p1 : 0.f;
      }
      acc[(e >> 1) & 1] = __fadd2_rn(acc[(e >> 1) & 1], make_float2(p0, p1));
      const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
      pk[e >> 1] = *reinterpret_cast<const uint32_t*>(&pp);
    }
    tmem_st16(pa + q4 * 16, pk);
    if (q4 + 1 < NQ) tmem_wait_ld();
  }
  tmem_wait_st();
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}

// The passes are separate functions: scheduled on their own, away from the
// rest of the kernel, the full pass runs about twice as fast.
template <int NQ>
__device__ __noinline__ float softmax_pass_full(uint32_t sa, float sl2, float m, uint32_t pa) {
  return softmax_pass<NQ, true>(sa, sl2, m, NQ * 32, pa);
}
template <int NQ>
__device__ __noinline__ float softmax_pass_masked(uint32_t sa, float sl2, float m, int tile_valid,
                                                  uint32_t pa) {
  return softmax_pass<NQ, false>(sa, sl2, m, tile_valid, pa);
}

// nq (4, 2 or 1 groups of 32 columns) is the same in every thread of the
// item.  tile_valid may differ between the warp's rows (a ragged leaf
// level); full or masked is chosen for the whole warp (tcgen05.ld is
// warp-collective).
__device__ __forceinline__ float softmax_pass_any(int nq, uint32_t sa, float sl2, float m,
                                                  int tile_valid, uint32_t pa) {
  const bool full = __all_sync(0xffffffffu, tile_valid == nq * 32);
  if (nq == 4) return full ? softmax_pass_full<4>(sa, sl2, m, pa)
                           : softmax_pass_masked<4>(sa, sl2, m, tile_valid, pa);
  if (nq == 2) return full ? softmax_pass_full<2>(sa, sl2, m, pa)
                           : softmax_pass_masked<2>(sa, sl2, m, tile_valid, pa);
  return full ? softmax_pass_full<1>(sa, sl2, m, pa)
              : softmax_pass_masked<1>(sa, sl2, m, tile_valid, pa);
}

__device__ __forceinline__ float tile_max_any(int nq, uint32_t sa, float sl2, int tile_valid) {
  if (nq == 4) return tile_max<4>(sa, sl2, tile_valid);
  if (nq == 2) return tile_max<2>(sa, sl2, tile_valid);
  return tile_max<1>(sa, sl2, tile_valid);
}

// Cold path of the softmax: some row's tile sum of P outgrew the limit (its
// running max is stale).  Recompute P for the warp (rows that did not grow keep their
// max), then rescale O and l of the grown rows once PV(g - 1) is complete.
__device__ __noinline__ bool softmax_regrow(const Params& P, DenseState& d, int nq, uint32_t sa,
                                            uint32_t trow, int tile_valid, uint32_t pa,
                                            uint32_t g, bool grow, float* m_run, float* l_run,
                                            float* psum) {
  // tcgen05.ld is warp-collective: every lane reads the tile max, then selects
  const float tmax = tile_max_any(nq, sa, P.sl2, tile_valid);
  const float m_new = grow ? tmax : *m_run;
  // equal maxima (also a row that has seen no token: both -inf) need no rescale
  const float alpha = (m_new == *m_run) ? 1.f : ex2(*m_run - m_new);
  *psum = softmax_pass_any(nq, sa, P.sl2, m_new, tile_valid, pa);
  // PV(g - 1) done: pfree of its buffer, completion (g - 1) / 2
  if (!mbar_wait(bar_pfree(d, (g - 1) & 1), ((g - 1) >> 1) & 1, d.abort)) return false;
  tc_fence_after();
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    float o[32];
    tmem_ld32(trow + kTmemO + q4 * 32, o);
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] *= alpha;
    tmem_st32(trow + kTmemO + q4 * 32, o);
  }
  *l_run *= alpha;
  *m_run = m_new;
  return true;
}

// ---- merge queue.  A dense item that turns out to be the last partial of a
// (request, KV head) unit does not merge it: it puts the unit into its CTA's
// ring in shared memory (r * Hkv + h + 1 per entry, 0 = empty) and moves on;
// the CTA's other warps merge queued units between their own items, and every
// warp drains the ring before the CTA ends.  `count` is claimed before an
// entry is written or read, so head and tail never run more than a ring
// apart; a writer still waits for its slot to be cleared (its previous reader
// may not be done with it), and a reader for the entry to appear.  Both waits
// are bounded.  A full ring makes the pushing warp merge the unit itself.
constexpr int kMqCap = 256;
struct MergeRing {
  uint32_t e[kMqCap];
  int count, head, tail;
};

__device__ __forceinline__ bool ring_wait(volatile uint32_t* e, bool want_empty) {
  const uint64_t t0 = global_ns();
  while ((*e == 0u) != want_empty)
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// By lane 0 of a warp whose lanes acquired the unit's partials (its ticket).
__device__ bool mq_push(const Params& P, MergeRing& q, uint32_t unit) {
  if (atomicAdd(&q.count, 1) >= kMqCap) {
    atomicSub(&q.count, 1);
    return false;
  }
  const int pos = atomicAdd(&q.tail, 1) & (kMqCap - 1);
  volatile uint32_t* e = &q.e[pos];
  if (!ring_wait(e, true)) {
    raise(P, kErrTimeout);
    return true;  // (the unit is lost; the error word says so)
  }
  // Release at CTA scope: the reader is a warp of this CTA, and the partials
  // this warp acquired (gpu scope, through the ticket) come with the entry.
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32((const void*)e)),
               "r"(unit + 1u)
               : "memory");
  return true;
}

// One unit from the ring, or -1 when it is empty (lane 0 claims, the warp gets
// the answer).
__device__ int mq_pop(const Params& P, MergeRing& q, int lane) {
  int v = -1;
  if (lane == 0) {
    volatile int* cnt = &q.count;
    int c = *cnt;
    for (int tries = 0; c > 0; ++tries) {
      if (tries > (1 << 20)) {  // never expected: the count keeps changing under it
        raise(P, kErrMerge);
        break;
      }
      if (atomicCAS(&q.count, c, c - 1) == c) {
        const int pos = atomicAdd(&q.head, 1) & (kMqCap - 1);
        volatile uint32_t* e = &q.e[pos];
        if (ring_wait(e, false)) {
          uint32_t x;  // acquire at CTA scope: the pusher's partials are visible
          asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(x) : "r"(smem_u32((const void*)e)) : "memory");
          v = (int)x - 1;
          *e = 0u;
        } else {
          raise(P, kErrTimeout);
        }
        break;
      }
      c = *cnt;
    }
  }
  v = __shfl_sync(0xffffffffu, v, 0);
  __syncwarp();  // the whole warp is ordered after lane 0's acquire
  return v;
}

// Merge of one queued unit (request r, KV head h), every partial read from the
// partial store: four rows per round, lane = (row of the round, 16 values of
// d), one online-softmax step per partial; output bf16 (queued units come
// only from tensor-core items).  (Loading several partials per step before
// combining them made the whole launch about twice as slow.)
__device__ __noinline__ void merge_unit(const Params& P, int unit, int lane) {
  const int G = P.G, r = unit / P.Hkv, h = unit % P.Hkv;
  if (r < 0 || r >= P.R) {
    if (lane == 0) raise(P, kErrMerge);
    return;
  }
  const ReqInfo ri = P.dp.req[r];
  const size_t jstride = (size_t)P.Hkv * G;
  const int sub = lane >> 3, d0 = (lane & 7) * 16;
  for (int r0 = 0; r0 < G; r0 += 4) {
    const int hl = r0 + sub;
    if (hl >= G) continue;
    const size_t base = ((size_t)ri.slot_base * P.Hkv + h) * G + hl;
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    float M = -INFINITY, L = 0.f;
#pragma unroll 4
    for (int j = 0; j < ri.n_partials; ++j) {
      const size_t rix = base + j * jstride;
      const float2 ml = __ldcg(&P.dp.mlpart[rix]);
      const float4* src = reinterpret_cast<const float4*>(P.dp.opart + rix * 128 + d0);
      float4 o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = __ldcg(src + k);
      if (ml.x == -INFINITY) continue;
      const float Mn = fmaxf(M, ml.x);
      const float a = ex2(M - Mn), b = ex2(ml.x - Mn);
      L = L * a + ml.y * b;
      M = Mn;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[4 * k] = acc[4 * k] * a + o[k].x * b;
        acc[4 * k + 1] = acc[4 * k + 1] * a + o[k].y * b;
        acc[4 * k + 2] = acc[4 * k + 2] * a + o[k].z * b;
        acc[4 * k + 3] = acc[4 * k + 3] * a + o[k].w * b;
      }
    }
    const bool empty = !(L > 0.f);
    const float inv = empty ? 0.f : 1.f / L;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] *= inv;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(P.out) + ((size_t)r * P.Hq + h * G + hl) * 128 + d0;
    store_out<__nv_bfloat16>(out, acc, 8);
    store_out<__nv_bfloat16>(out + 8, acc + 8, 8);
    if ((lane & 7) == 0) {
      if (empty) raise(P, kErrEmpty);
      if (P.lse) P.lse[(size_t)r * P.Hq + h * G + hl] = empty ? -INFINITY : (M + __log2f(L)) * kLn2;
    }
  }
}

// The member tickets of the softmax warp's item, once its partial rows are
// written (lane mu: member mu).  The last arriver of a unit queues its merge;
// a full ring makes the warp merge it here.  (Taking the tickets a tile into
// the next item instead, to hide the fence, was tried: a launch then
// occasionally never finished, and no bounded wait fired; see the design
// notes.)
__device__ void settle_tickets(const Params& P, DenseState& d, MergeRing& ring) {
  const int lane = threadIdx.x & 31;
  __threadfence();
  __syncwarp();
  bool last = false;
  if (d.pend_valid) {
    uint32_t* ticket = &P.dp.tickets[d.pend_unit];
    const uint32_t old = atom_add_acq_rel(ticket, 1u);
    if (old >= (uint32_t)d.pend_np) raise(P, kErrMerge);  // more arrivals than partials
    last = old == (uint32_t)d.pend_np - 1u;
    if (last) st_relaxed(ticket, 0u);  // every partial is in: ready for the next launch
  }
  d.pend_valid = 0;
  d.pend_any = 0;
  const uint32_t lastmask = __ballot_sync(0xffffffffu, last);
  __syncwarp();  // the acquiring lanes' view, for lane 0's push and the whole warp
  for (uint32_t m = lastmask; m; m &= m - 1) {
    const int mu = __ffs(m) - 1;
    const uint32_t unit = __shfl_sync(0xffffffffu, d.pend_unit, mu);
    int ok = 1;
    if (lane == 0) ok = mq_push(P, ring, unit);
    if (!__shfl_sync(0xffffffffu, ok, 0)) merge_unit(P, (int)unit, lane);  // ring full
  }
}

// The softmax warps' part of one item, then the epilogue.  r_row is the
// request of this thread's row (-1 past the item's rows).  Returns early
// (abort set) on a timeout.
// All 128 softmax threads at the same point (bounded; false on abort).
__device__ __forceinline__ bool softmax_threads_sync(DenseState& d) {
  mbar_arrive(bar_x(d));
  const bool ok = mbar_wait(bar_x(d), d.xph & 1, d.abort);
  ++d.xph;
  return ok;
}

__device__ void softmax_item(const Params& P, DenseState& d, MergeRing& ring, const Item& it,
                             int t0, int ntok, int ntiles, int nrows, int r_row) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t g0 = d.g;
  const uint32_t trow = d.tmem + ((uint32_t)(warp * 32) << 16);
  // this thread's row copy: tile columns [col0, col0 + cw) of every tile
  const int cw = copy_width(nrows), nq = cw / 32, ncopy = kTileTok / cw;
  const int col0 = (tid / cw) * cw;
  if (ncopy > 1) {
    // P columns outside a copy's slice stay 0 for the whole item, so each
    // copy's PV sums only its own tokens.  Both P buffers are idle here: the
    // previous item waited for its last PV.
    uint32_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
    for (int c = 0; c < 128; c += 16) tmem_st16(trow + kTmemP + c, z);
    tmem_wait_st();
  }
  // the row's partial slots, needed only at the end (the load hides behind the tiles)
  // row_end: tokens of the item's span the row attends to (fewer than the
  // span only on a ragged leaf level, whose members see its first leaf_vis
  // tokens; 0 when the row sees none of this chunk)
  int sb_row = 0, np_row = 0, row_end = ntok;
  if (r_row >= 0) {
    const ReqInfo ri = P.dp.req[r_row];
    sb_row = ri.slot_base;
    np_row = ri.n_partials;
    if (ri.leaf_vis >= 0 && ri.leaf == it.seg) row_end = max(0, min(ntok, ri.leaf_vis - t0));
  }
  float m_run = -INFINITY, l_run = 0.f;
  for (int j = 0; j < ntiles; ++j) {
    const uint32_t g = g0 + j, b = g & 1;
    const int tile_valid = min(kTileTok, ntok - j * kTileTok);  // the item's tokens (V rows)
    // this row copy's valid columns of its slice
    const int row_valid = max(0, min(cw, min(tile_valid, row_end - j * kTileTok) - col0));
    const uint32_t pa = trow + kTmemP + b * 64 + col0 / 2;
    if (!mbar_wait(bar_s(d, b), (g >> 1) & 1, d.abort)) return;
    // P buffer b was last read by PV(g - 2)
    if (j >= 2 && !mbar_wait(bar_pfree(d, b), ((g >> 1) - 1) & 1, d.abort)) return;
    tc_fence_after();
    const uint32_t sa = trow + b * 128 + col0;
    // P against the running max (the tile's own max on the first tile of the
    // item, when O is still empty); rows whose tile sum outgrew the limit are
    // redone with their new max (rare)
    if (j == 0) m_run = tile_max_any(nq, sa, P.sl2, row_valid);
    float psum = softmax_pass_any(nq, sa, P.sl2, m_run, row_valid, pa);
    const bool grow = psum > kRescaleSumLimit;
    if (j > 0 && __any_sync(0xffffffffu, grow)) {
      if (!softmax_regrow(P, d, nq, sa, trow, row_valid, pa, g, grow, &m_run, &l_run, &psum))
        return;
    }
    l_run = (j == 0) ? psum : l_run + psum;
    // S(g) has been read: the MMA warp may reuse this TMEM buffer
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_sfree(d, b));
    if (tile_valid < kTileTok) {
      // rows past the chunk end may hold anything (even NaN): zero them in V
      // before PV reads them (0 * NaN would poison O)
      const uint32_t st = g % kStages;
      if (!mbar_wait(bar_v(d, st), (g / kStages) & 1, d.abort)) return;
      if (tid >= tile_valid) {
        uint8_t* vs = d.smem + kOffV + st * kTileBytes;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(vs + (c >> 3) * kHalfBytes + tid * 128 + (c & 7) * 16) =
              make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_p(d, b));
  }
  // O is final once PV(last) is done; its commit on pfree of the last P
  // buffer covers every earlier MMA too.  The wait is sound: that barrier's
  // previous completion (PV(last - 2)) has happened and its next one needs
  // this warp's P of the next item.  (A barrier that every PV completes would
  // not do: PV(last) may complete before the warp first looks, and a wait for
  // PV(last - 1) by parity then names a completion that never comes.)
  if (ntiles > 0) {
    const uint32_t gl = g0 + ntiles - 1;
    if (!mbar_wait(bar_pfree(d, gl & 1), (gl >> 1) & 1, d.abort)) return;
    tc_fence_after();
  }

  // ---- epilogue.  Each row leaves as one bulk copy (cp.async.bulk, run by
  // the TMA engine) of a staging row in shared memory: 512 B of fp32 partial
  // output, or 256 B of bf16 output for a (request, KV head) unit whose only
  // partial this is.  E is [128][kERow] fp32 over the idle K stages, a row
  // per thread; the 16-byte pad makes the row-per-thread accesses free of
  // bank conflicts.
  const int G = P.G, h = it.kvh;
  float* E = reinterpret_cast<float*>(d.smem + kOffE);
  float4* Erow = reinterpret_cast<float4*>(E + tid * kERow);
  fence_proxy_async();  // E overlays K stages the TMA and the tensor cores used
  // Row copies: the row's maximum over its copies, each copy's O and l
  // scaled to it; copy 0's threads then add the copies' rows into theirs
  // (the V stages are idle and hold the exchange).
  float fac = 1.f, m_out = m_run, l_out = l_run;
  float* X = reinterpret_cast<float*>(d.smem + kOffV);  // [2][128]: m, then scaled l
  const int rho = tid % cw;
  if (ncopy > 1) {
    X[tid] = m_run;
    if (!softmax_threads_sync(d)) return;
    float mx = -INFINITY;
    for (int c = 0; c < ncopy; ++c) mx = fmaxf(mx, X[rho + c * cw]);
    // a copy that saw no token (m = -inf, O = 0, l = 0) adds nothing
    fac = (m_run == -INFINITY) ? 0.f : ex2(m_run - mx);
    X[128 + tid] = l_run * fac;
    m_out = mx;
  }
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    float o[32];
    if (ntiles > 0) {
      tmem_ld32(trow + kTmemO + q4 * 32, o);  // warp-collective: every lane
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      Erow[q4 * 8 + (e >> 2)] = make_float4(o[e] * fac, o[e + 1] * fac, o[e + 2] * fac, o[e + 3] * fac);
  }
  if (ncopy > 1) {
    if (!softmax_threads_sync(d)) return;  // every copy's rows and l written
    l_out = 0.f;
    for (int c = 0; c < ncopy; ++c) l_out += X[128 + rho + c * cw];
    if (tid < cw) {
      for (int j = 0; j < 32; ++j) {
        float4 v = Erow[j];
        for (int c = 1; c < ncopy; ++c) {
          const float4 w = reinterpret_cast<const float4*>(E + (tid + c * cw) * kERow)[j];
          v.x += w.x;
          v.y += w.y;
          v.z += w.z;
          v.w += w.w;
        }
        Erow[j] = v;
      }
    }
  }
  // copy 0's threads write their rows.  A row whose unit has this one partial
  // gets its output and LSE here: no partial slot, no ticket, no merge.
  // (Merging here with partials already in would put their loads on the
  // tensor-core path: the merges stay with the per-warp item warps.)
  const bool writer = tid < cw;
  if (writer && tid < nrows && r_row >= 0) {
    if (np_row > 1) {
      const size_t prow = (((size_t)sb_row + it.slot_j) * P.Hkv + h) * G + tid % G;
      __stcg(&P.dp.mlpart[prow], make_float2(m_out, l_out));
      fence_proxy_async();
      bulk_store(P.dp.opart + prow * 128, Erow, 128 * 4);
    } else {
      const bool empty = !(l_out > 0.f);
      const float inv = empty ? 0.f : 1.f / l_out;
      // bf16 in place: quad j (8 B) lands below float4 j, which is read first
      uint2* Eb = reinterpret_cast<uint2*>(Erow);
      for (int j = 0; j < 32; ++j) {
        const float4 v = Erow[j];
        Eb[j] = make_uint2(pack_bf16(v.x * inv, v.y * inv), pack_bf16(v.z * inv, v.w * inv));
      }
      const size_t orow = (size_t)r_row * P.Hq + h * G + tid % G;
      if (empty) raise(P, kErrEmpty);
      if (P.lse) P.lse[orow] = empty ? -INFINITY : (m_out + __log2f(l_out)) * kLn2;
      fence_proxy_async();
      bulk_store(reinterpret_cast<__nv_bfloat16*>(P.out) + orow * 128, Erow, 128 * 2);
    }
    // the row is in global memory (and its staging read) before the tickets
    // below publish it and before the next item's K tiles land over E
    bulk_commit_and_wait();
  }
  tc_fence_before();
  __syncwarp();
  // this warp's members: lane mu speaks for member mu (rows warp * 32 + mu * G ..)
  const int mpw = 32 / G, src = (lane < mpw ? lane : 0) * G;
  const int r_m = __shfl_sync(0xffffffffu, r_row, src);
  const int np_m = __shfl_sync(0xffffffffu, np_row, src);
  // lane mu takes member mu's ticket (units with more than one partial); the
  // last arriver of a unit queues its merge
  d.pend_valid = writer && lane < mpw && warp * 32 + lane * G < nrows && r_m >= 0 && np_m > 1;
  d.pend_unit = (uint32_t)(d.pend_valid ? r_m : 0) * P.Hkv + h;
  d.pend_np = np_m;
  d.pend_any = 1;
  settle_tickets(P, d, ring);
}

// Dense items of this CTA, run by warps 0-7 (256 threads).
__device__ void dense_loop(const Params& P, uint8_t* smem_raw, MergeRing& ring) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool control = (tid == 128);
  DenseState d;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  d.smem = smem_raw + pad;
  d.sbase = raw + pad;
  d.g = 0;
  d.xph = 0;
  d.pend_unit = 0;
  d.pend_np = 0;
  d.pend_valid = 0;
  d.pend_any = 0;
  volatile int* s_idx = reinterpret_cast<volatile int*>(d.smem + kOffMisc);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(d.smem + kOffMisc + 8);
  d.abort = reinterpret_cast<volatile int*>(d.smem + kOffMisc + 16);
  if (control) {
    *d.abort = 0;
    for (uint32_t st = 0; st < (uint32_t)kStages; ++st) {
      mbar_init(bar_k(d, st), 1);
      mbar_init(bar_v(d, st), 1);
      mbar_init(bar_kfree(d, st), 1);
      mbar_init(bar_vfree(d, st), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      mbar_init(bar_s(d, b), 1);
      mbar_init(bar_sfree(d, b), 4);
      mbar_init(bar_p(d, b), 4);
      mbar_init(bar_pfree(d, b), 1);
    }
    mbar_init(bar_x(d), 128);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  dense_sync();
  tc_fence_after();
  d.tmem = *reinterpret_cast<volatile uint32_t*>(s_tmem);
  for (;;) {
    if (control) *s_idx = (int)atomicAdd(&P.dp.ctr[kCtrDense], 1u);
    dense_sync();
    const int idx = *s_idx;
    const bool stop = idx >= P.dp.n_ditems || *d.abort;
    dense_sync();
    if (stop) break;
    const int4* ip = reinterpret_cast<const int4*>(P.dp.ditems + idx);
    const int4 a = __ldg(ip), b = __ldg(ip + 1);
    const Item it{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const Span s = resolve(P, it);
    const int nrows = s.nmem * P.G;
    int ntok = s.t1 - s.t0;
    if (it.kind == kItemDenseRagged) ntok = min(ntok, it.cost);  // no row sees further
    if (ntok > kMaxDenseBlocks * kBlockSize) {  // device lengths beyond what was planned
      if (control) raise(P, kErrColumn);
      ntok = kMaxDenseBlocks * kBlockSize;
    }
    const int nb = (ntok + kBlockSize - 1) / kBlockSize;
    const int ntiles = (ntok + kTileTok - 1) / kTileTok;
    int r_row = -1;
    if (tid < 128) r_row = prepare_item(P, d, it, nrows);
    dense_sync();
    if (tid < 128) softmax_item(P, d, ring, it, s.t0, ntok, ntiles, nrows, r_row);
    else if (warp == 4) mma_s_item(P, d, ntiles);
    else if (warp == 7) mma_pv_item(P, d, ntiles);
    else if (warp == 5 || warp == 6) producer_item(P, d, s, it.kvh, warp - 5, nb, ntiles);
    tc_fence_before();
    dense_sync();
    d.g += ntiles;
  }
  if (*d.abort && control) {
    raise(P, kErrTimeout);
    // give tensor-core work already issued time to drain before the TMEM is released
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  tc_fence_before();
  dense_sync();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(d.tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------ the launch

// PSATTN_SUFFIX_SIMT=1 (build define, for measurement): on the bf16 d = 128
// path, suffix items run on the CUDA-core item (shuffle-reduced dot
// products) instead of mma.sync, everything else unchanged.
#ifndef PSATTN_SUFFIX_SIMT
#define PSATTN_SUFFIX_SIMT 0
#endif

template <int PATH>
__device__ __forceinline__ void run_item(const Params& P, const Item& it, int lane) {
  if constexpr (PATH == kPathMmaBf16D128 && PSATTN_SUFFIX_SIMT) {
    if (it.kind == kItemSuffix && P.G <= kSimtRows) simt_item<__nv_bfloat16, 128>(P, it, lane);
    else mma_item(P, it, lane);
  } else if constexpr (PATH == kPathMmaBf16D128) mma_item(P, it, lane);
  else if constexpr (PATH == kPathSimtF32D64) simt_item<float, 64>(P, it, lane);
  else if constexpr (PATH == kPathSimtF32D128) simt_item<float, 128>(P, it, lane);
  else if constexpr (PATH == kPathSimtBf16D64) simt_item<__nv_bfloat16, 64>(P, it, lane);
  else simt_item<__nv_bfloat16, 128>(P, it, lane);
}

template <int PATH>
__global__ void __launch_bounds__(kThreads, 1) psattn_fused_decode(const __grid_constant__ Params P) {
  const int lane = threadIdx.x & 31;
  // tensor-core items run (and may queue merges) while s_dense_active is set
  __shared__ volatile int s_dense_active;
  __shared__ MergeRing ring;
  constexpr bool kMma = PATH == kPathMmaBf16D128;
  const bool queue = kMma && P.dp.n_ditems > 0;
  if constexpr (kMma) {
    extern __shared__ uint8_t dyn_smem[];
    if (queue) {
      for (int i = threadIdx.x; i < kMqCap; i += blockDim.x) ring.e[i] = 0u;
      if (threadIdx.x == 0) {
        ring.count = ring.head = ring.tail = 0;
        s_dense_active = 1;
      }
      __syncthreads();
      if (threadIdx.x < kDenseThreads) {
        dense_loop(P, dyn_smem, ring);
        if (threadIdx.x == 0) s_dense_active = 0;
      }
    }
  }
  for (;;) {
    int idx = 0;
    if (lane == 0) idx = (int)atomicAdd(&P.dp.ctr[kCtrWarp], 1u);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    if (idx >= P.dp.n_witems) break;
    const int4* ip = reinterpret_cast<const int4*>(P.dp.witems + idx);
    const int4 a = __ldg(ip), b = __ldg(ip + 1);
    const Item it{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    run_item<PATH>(P, it, lane);
    if (queue) {  // the queued merges, between items
      for (int u = mq_pop(P, ring, lane); u >= 0; u = mq_pop(P, ring, lane)) merge_unit(P, u, lane);
    }
  }
  if (queue) {
    // Drain the ring.  While this CTA's tensor-core items run, more merges may
    // come (sleep between looks); once they are done, empty means done.
    uint64_t t0 = global_ns();
    for (;;) {
      const int u = mq_pop(P, ring, lane);
      if (u >= 0) {
        merge_unit(P, u, lane);
        t0 = global_ns();
        continue;
      }
      if (!s_dense_active) break;
      if (global_ns() - t0 > kWaitLimitNs) {  // the CTA's tensor-core items never finished
        if (lane == 0) raise(P, kErrTimeout);
        break;
      }
      __nanosleep(1000);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&P.dp.ctr[kCtrExit], 1u) == gridDim.x - 1) {
      atomicExch(&P.dp.ctr[kCtrWarp], 0u);
      atomicExch(&P.dp.ctr[kCtrDense], 0u);
      atomicExch(&P.dp.ctr[kCtrExit], 0u);
    }
  }
}

template <int PATH>
cudaError_t launch(const Params& P, int grid, cudaStream_t st) {
  const uint32_t smem = (PATH == kPathMmaBf16D128 && P.dp.n_ditems > 0) ? kDenseSmemBytes : 0;
  if (smem) {
    // the attribute is set once per device the process launches on (it holds
    // for the function on the current device); concurrent first launches on
    // one device only set it twice
    constexpr int kMaxDevices = 64;
    static std::atomic<bool> attr_set[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(psattn_fused_decode<PATH>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_release);
    }
  }
  psattn_fused_decode<PATH><<<grid, kThreads, smem, st>>>(P);
  return cudaGetLastError();
}

// Tensor map of the pool for the dense tiles: a 2-D bf16 tensor of
// [num_blocks * 2 * Hkv * 16 rows][d = 128 columns], boxes of 16 rows x 64
// columns with the 128-byte swizzle the tcgen05 descriptors expect.
int encode_kv_map(CUtensorMap* map, const void* pool, int nblocks, int hkv) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
      cudaGetLastError();
      return PSATTN_ERR_CUDA;
    }
    fn = reinterpret_cast<EncodeFn>(p);
  }
  const cuuint64_t dims[2] = {128, (cuuint64_t)nblocks * 2 * hkv * kBlockSize};
  const cuuint64_t strides[1] = {128 * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PSATTN_OK : PSATTN_ERR_CUDA;
}

// One wait that nothing completes (an mbarrier no thread arrives on), run
// through the same bounded wait as the decode kernel with a short limit: the
// wait gives up, sets the abort flag and the error word, and the kernel
// returns.  For testing the bounded-wait path without a fault.
__global__ void psattn_selftest_wait(uint32_t* flags, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait_ns(smem_u32(&bar), 0, &abort, limit_ns);
    if (!ok && abort) atomicOr(flags, (uint32_t)kErrTimeout);
  }
}

}  // namespace

int psattn_run_wait_selftest(uint32_t* dev_flags, uint64_t limit_ns, void* stream) {
  psattn_selftest_wait<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev_flags, limit_ns);
  return cudaGetLastError() == cudaSuccess ? PSATTN_OK : PSATTN_ERR_CUDA;
}

int psattn_launch_decode(const HostPlan& hp, const DevPlan& dp, const void* q, const void* kv_pool,
                         const int32_t* block_table, const int32_t* group_of_req,
                         const int32_t* prefix_len, const int32_t* suffix_len, void* out,
                         float* lse, psattn_stream_t stream) {
  Params P;
  P.dp = dp;
  P.q = q;
  P.pool = kv_pool;
  P.bt = block_table;
  P.gor = group_of_req;
  P.plen = prefix_len;
  P.slen = suffix_len;
  P.out = out;
  P.lse = lse;
  P.R = hp.shape.num_req;
  P.Hq = hp.shape.num_q_heads;
  P.Hkv = hp.shape.num_kv_heads;
  P.G = P.Hq / P.Hkv;
  P.maxb = hp.shape.max_blocks_per_req;
  P.nblocks = hp.shape.num_pool_blocks;
  P.sl2 = hp.shape.scale * kLog2e;
  std::memset(&P.kv_map, 0, sizeof(P.kv_map));
  if (hp.path == kPathMmaBf16D128 && dp.n_ditems > 0) {
    const int rc = encode_kv_map(&P.kv_map, kv_pool, P.nblocks, P.Hkv);
    if (rc) return rc;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (hp.path) {
    case kPathMmaBf16D128: e = launch<kPathMmaBf16D128>(P, hp.grid, st); break;
    case kPathSimtF32D64: e = launch<kPathSimtF32D64>(P, hp.grid, st); break;
    case kPathSimtF32D128: e = launch<kPathSimtF32D128>(P, hp.grid, st); break;
    case kPathSimtBf16D64: e = launch<kPathSimtBf16D64>(P, hp.grid, st); break;
    default: e = launch<kPathSimtBf16D128>(P, hp.grid, st); break;
  }
  if (e != cudaSuccess) return PSATTN_ERR_CUDA;
  return PSATTN_OK;
}
