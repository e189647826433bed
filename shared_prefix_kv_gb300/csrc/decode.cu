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
#define PSATTN_PREFETCH_BLOCKS 3
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
        const float2 ml = __ldcg(&P.dp.mlpart[rix]);
        if (ml.x == -INFINITY) continue;
        const float Mn = fmaxf(M, ml.x);
        const float a = ex2(M - Mn), b = ex2(ml.x - Mn);
        L = L * a + ml.y * b;
        M = Mn;
        const float* src = P.dp.opart + rix * D;
#pragma unroll
        for (int sg = 0; sg < NS; ++sg)
#pragma unroll
          for (int e = 0; e < SEG; e += 4) {
            const float4 w = __ldcg(reinterpret_cast<const float4*>(src + own.d0[sg] + e));
            acc[sg][e] = acc[sg][e] * a + w.x * b;
            acc[sg][e + 1] = acc[sg][e + 1] * a + w.y * b;
            acc[sg][e + 2] = acc[sg][e + 2] * a + w.z * b;
            acc[sg][e + 3] = acc[sg][e + 3] * a + w.w * b;
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
  uint32_t qa0[8], qa2[8];
  if (g < nrows) {
    const int r = member_req(P, it, g / G);
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
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i] = (tv[i] < nvalid) ? x[i] * P.sl2 : -INFINITY;
      mx = fmaxf(mx, x[i]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);  // finite: the block has a valid token
    const float alpha = ex2(m_run - m_new);
    float p[4], psum = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      p[i] = ex2(x[i] - m_new);
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
// a matrix product, BatchLLM section 2.2).  Warps 0-3 of the CTA run it: thread
// 0 issues the TMA copies and the tcgen05 MMAs, and all 128 threads do the
// softmax and the epilogue, thread t owning row t (= TMEM lane t).
//
// Per 128-token tile j (stage j & 1 of a double-buffered K/V ring):
//   TMA: 8 paged blocks x {K, V} x 2 halves of d, 128B-swizzled boxes of
//        16 rows x 64 columns straight from the pool (tensor map over the pool
//        as [rows = block*2*Hkv*16][d]);
//   S = Q K^T   tcgen05.mma kind::f16, M 128, N 128, K 128 (8 steps), fp32 in
//               TMEM columns [0, 128); Q and K are K-major;
//   softmax     tcgen05.ld of S, running max m in log2 units, raised only when
//               the tile max exceeds it by more than 8 (then O is rescaled in
//               TMEM), P = 2^(s - m) as bf16 into a 128B-swizzled K-major tile;
//   O += P V    tcgen05.mma, N 128 (d), K 128 tokens, V as the MN-major B
//               operand, fp32 in TMEM columns [128, 256).
// Every wait is bounded; a timeout raises the error word and ends the dense
// work of the CTA without touching the rest.

constexpr int kTileTok = 128;
constexpr uint32_t kTileBytes = 128 * 128 * 2;          // one 128 x 128 bf16 operand tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;         // one 64-column half (K atom)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTileBytes;                  // 2 stages
constexpr uint32_t kOffV = 3 * kTileBytes;              // 2 stages
constexpr uint32_t kOffP = 5 * kTileBytes;
constexpr uint32_t kOffIds = 6 * kTileBytes;            // block ids of the chunk
constexpr int kMaxDenseBlocks = 512;                    // chunk <= 8192 tokens
constexpr uint32_t kOffBar = kOffIds + kMaxDenseBlocks * 4;
constexpr uint32_t kOffMisc = kOffBar + 64;
constexpr uint32_t kDenseSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleThreshold = 8.0f;               // log2 units
constexpr uint64_t kWaitLimitNs = 2000000000ull;        // 2 s per wait

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

// Bounded wait for phase `parity` of an mbarrier; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// named barrier 1 over the 128 threads of warps 0-3
__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// barrier that also ORs a flag over the 128 threads (uniform abort decisions)
__device__ __forceinline__ bool group_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 1, 128, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

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
  uint8_t* smem;      // 1024-aligned
  uint32_t sbase;     // its shared-space address
  uint32_t tmem;      // TMEM base (lane 0, column of S)
  uint32_t ph_kv0, ph_kv1, ph_s, ph_o;
};

__device__ __forceinline__ uint32_t bar_kv(const DenseState& d, int st) {
  return d.sbase + kOffBar + 8u * st;
}
__device__ __forceinline__ uint32_t bar_s(const DenseState& d) { return d.sbase + kOffBar + 16; }
__device__ __forceinline__ uint32_t bar_o(const DenseState& d) { return d.sbase + kOffBar + 24; }

// TMA of tile j of the chunk into stage j & 1 (thread 0 only).
__device__ __forceinline__ void issue_tile(const Params& P, const DenseState& d, int j, int nb,
                                           int h) {
  const int st = j & 1;
  const int* ids = reinterpret_cast<const int*>(d.smem + kOffIds);
  const int b0 = j * (kTileTok / kBlockSize), b1 = min(nb, b0 + kTileTok / kBlockSize);
  uint32_t bytes = 0;
  for (int b = b0; b < b1; ++b)
    if (ids[b] >= 0) bytes += 4u * kBlockSize * 64u * 2u;  // K and V x two 16 x 64 halves
  const uint32_t bar = bar_kv(d, st);
  mbar_expect_tx(bar, bytes);
  const uint32_t ks = d.sbase + kOffK + st * kTileBytes, vs = d.sbase + kOffV + st * kTileBytes;
  for (int b = b0; b < b1; ++b) {
    const int id = ids[b];
    if (id < 0) continue;
    const int rk = ((id * 2 + 0) * P.Hkv + h) * kBlockSize;
    const int rv = ((id * 2 + 1) * P.Hkv + h) * kBlockSize;
    const uint32_t off = (uint32_t)(b - b0) * (kBlockSize * 128u);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      tma_load_2d(ks + half * kHalfBytes + off, &P.kv_map, half * 64, rk, bar);
      tma_load_2d(vs + half * kHalfBytes + off, &P.kv_map, half * 64, rv, bar);
    }
  }
}

// One dense item.  Returns false when a wait timed out (uniform over the group).
__device__ bool dense_item(const Params& P, DenseState& d, const Item& it) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G, h = it.kvh;
  const Span s = resolve(P, it);
  const int nrows = s.nmem * G;
  int ntok = s.t1 - s.t0;
  if (ntok > kMaxDenseBlocks * kBlockSize) {  // device lengths beyond what was planned
    if (tid == 0) raise(P, kErrColumn);
    ntok = kMaxDenseBlocks * kBlockSize;
  }
  const int nb = (ntok + kBlockSize - 1) / kBlockSize;
  const int ntiles = (ntok + kTileTok - 1) / kTileTok;

  // block ids of the chunk -> shared memory (bad ids raise the error word, read -1)
  int* ids = reinterpret_cast<int*>(d.smem + kOffIds);
  for (int b = tid; b < nb; b += 128) {
    int id = -1;
    const int col = s.col0 + b;
    if (col >= P.maxb) {
      raise(P, kErrColumn);
    } else {
      id = __ldg(&P.bt[(size_t)s.rep * P.maxb + col]);
      if (id < 0 || id >= P.nblocks) {
        raise(P, kErrBlockOob);
        id = -1;
      }
    }
    ids[b] = id;
  }
  // Q tile, K-major, 128B swizzle: 16-byte chunk c of row t at
  // atom (c / 8), row t, position (c % 8) ^ (t % 8)
  {
    uint8_t* qs = d.smem + kOffQ;
    const __nv_bfloat16* qp = nullptr;
    if (tid < nrows) {
      const int r = member_req(P, it, tid / G);
      qp = reinterpret_cast<const __nv_bfloat16*>(P.q) + ((size_t)r * P.Hq + h * G + tid % G) * 128;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 w = qp ? __ldg(reinterpret_cast<const uint4*>(qp + 8 * c)) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(qs + (c >> 3) * kHalfBytes + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)) = w;
    }
  }
  fence_proxy_async();
  group_sync();
  if (tid == 0 && ntiles > 0) issue_tile(P, d, 0, nb, h);

  const uint32_t trow = d.tmem + ((uint32_t)(warp * 32) << 16);
  const uint32_t idesc_s = idesc_bf16_m128_n128(false), idesc_o = idesc_bf16_m128_n128(true);
  float m_run = -INFINITY, l_run = 0.f;
  for (int j = 0; j < ntiles; ++j) {
    const int st = j & 1;
    const int tile_valid = min(kTileTok, ntok - j * kTileTok);
    bool to = !mbar_wait(bar_kv(d, st), st ? d.ph_kv1 : d.ph_kv0);
    if (st) d.ph_kv1 ^= 1; else d.ph_kv0 ^= 1;
    if (tile_valid < kTileTok && tid >= tile_valid) {
      // rows past the chunk end: stale or poisoned V would give 0 * NaN
      uint8_t* vs = d.smem + kOffV + st * kTileBytes;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(vs + (c >> 3) * kHalfBytes + tid * 128 + (c & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      fence_proxy_async();
    }
    if (group_sync_or(to)) return false;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t qa = d.sbase + kOffQ, ka = d.sbase + kOffK + st * kTileBytes;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t koff = (k >> 2) * kHalfBytes + (k & 3) * 32;
        tc_mma(d.tmem, sw128_desc(qa + koff, 16, 1024), sw128_desc(ka + koff, 16, 1024), idesc_s,
               k > 0);
      }
      tc_commit(bar_s(d));
    }
    to = !mbar_wait(bar_s(d), d.ph_s);
    d.ph_s ^= 1;
    if (j > 0) {
      to |= !mbar_wait(bar_o(d), d.ph_o);
      d.ph_o ^= 1;
    }
    if (group_sync_or(to)) return false;
    tc_fence_after();
    // the other stage is free now (its S and PV products are complete)
    if (tid == 0 && j + 1 < ntiles) issue_tile(P, d, j + 1, nb, h);

    // row max of the tile
    float mx = -INFINITY;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[32];
      tmem_ld32(trow + q4 * 32, v);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (q4 * 32 + e < tile_valid) mx = fmaxf(mx, v[e] * P.sl2);
    }
    const float m_new = (mx > m_run + kRescaleThreshold) ? mx : m_run;
    const float alpha = ex2(m_run - m_new);
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float o[32];
        tmem_ld32(trow + 128 + q4 * 32, o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] *= alpha;
        tmem_st32(trow + 128 + q4 * 32, o);
      }
    }
    m_run = m_new;
    // P = 2^(s - m) as bf16, K-major 128B-swizzled like Q
    float psum = 0.f;
    uint8_t* ps = d.smem + kOffP;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float v[32];
      tmem_ld32(trow + q4 * 32, v);
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float p0 = (q4 * 32 + e < tile_valid) ? ex2(v[e] * P.sl2 - m_run) : 0.f;
        const float p1 = (q4 * 32 + e + 1 < tile_valid) ? ex2(v[e + 1] * P.sl2 - m_run) : 0.f;
        psum += p0 + p1;
        pk[e >> 1] = pack_bf16(p0, p1);
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int jj = (q4 & 1) * 4 + cc;
        *reinterpret_cast<uint4*>(ps + (q4 >> 1) * kHalfBytes + tid * 128 + ((jj ^ (tid & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      }
    }
    l_run = l_run * alpha + psum;
    fence_proxy_async();
    tc_fence_before();
    group_sync();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t pa = d.sbase + kOffP, va = d.sbase + kOffV + st * kTileBytes;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t poff = (k >> 2) * kHalfBytes + (k & 3) * 32;
        tc_mma(d.tmem + 128, sw128_desc(pa + poff, 16, 1024),
               sw128_desc(va + k * (16 * 128), kHalfBytes, 1024), idesc_o, (j > 0 || k > 0));
      }
      tc_commit(bar_o(d));
    }
  }
  bool to = false;
  if (ntiles > 0) {
    to = !mbar_wait(bar_o(d), d.ph_o);
    d.ph_o ^= 1;
  }
  if (group_sync_or(to)) return false;
  tc_fence_after();

  // epilogue: row tid -> partial slot, then tickets and merges per member
  const bool valid_row = tid < nrows;
  int r = -1, hl = 0;
  ReqInfo ri{};
  size_t rix = 0;
  if (valid_row) {
    r = member_req(P, it, tid / G);
    hl = tid % G;
    ri = P.dp.req[r];
    rix = (((size_t)ri.slot_base + it.slot_j) * P.Hkv + h) * G + hl;
  }
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    float o[32];
    if (ntiles > 0) {
      tmem_ld32(trow + 128 + q4 * 32, o);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
    }
    if (valid_row) {
      float* dst = P.dp.opart + rix * 128 + q4 * 32;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        __stcg(reinterpret_cast<float4*>(dst + e), make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]));
    }
  }
  if (valid_row) __stcg(&P.dp.mlpart[rix], make_float2(m_run, l_run));
  __threadfence();
  __syncwarp();
  // one ticket per member: its G rows are lanes [lead, lead + G) of this warp
  const int lead = lane - (lane % G);
  int last = 0;
  if (valid_row && hl == 0) {
    uint32_t* ticket = &P.dp.tickets[(size_t)r * P.Hkv + h];
    last = atom_add_acq_rel(ticket, 1u) == (uint32_t)ri.n_partials - 1u;
    if (last) st_relaxed(ticket, 0u);
  }
  last = __shfl_sync(0xffffffffu, last, lead);
  if (valid_row && last) {
    __threadfence();
    float M = -INFINITY, L = 0.f;
    for (int j = 0; j < ri.n_partials; ++j) {
      const size_t jx = (((size_t)ri.slot_base + j) * P.Hkv + h) * G + hl;
      const float2 ml = __ldcg(&P.dp.mlpart[jx]);
      if (ml.x == -INFINITY) continue;
      const float Mn = fmaxf(M, ml.x);
      L = L * ex2(M - Mn) + ml.y * ex2(ml.x - Mn);
      M = Mn;
    }
    const bool empty = !(L > 0.f);
    const float inv = empty ? 0.f : 1.f / L;
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(P.out) + ((size_t)r * P.Hq + h * G + hl) * 128;
    for (int c8 = 0; c8 < 128; c8 += 32) {
      float acc[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] = 0.f;
      for (int j = 0; j < ri.n_partials; ++j) {
        const size_t jx = (((size_t)ri.slot_base + j) * P.Hkv + h) * G + hl;
        const float2 ml = __ldcg(&P.dp.mlpart[jx]);
        if (ml.x == -INFINITY) continue;
        const float w = ex2(ml.x - M) * inv;
        const float* src = P.dp.opart + jx * 128 + c8;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(src + e));
          acc[e] += w * x.x; acc[e + 1] += w * x.y; acc[e + 2] += w * x.z; acc[e + 3] += w * x.w;
        }
      }
#pragma unroll
      for (int e = 0; e < 32; e += 8) store_out<__nv_bfloat16>(dst + c8 + e, acc + e, 8);
    }
    if (empty) raise(P, kErrEmpty);
    if (P.lse) P.lse[(size_t)r * P.Hq + h * G + hl] = empty ? -INFINITY : (M + __log2f(L)) * kLn2;
  }
  // the next item overwrites Q, P and TMEM only after every thread is past here
  tc_fence_before();
  group_sync();
  return true;
}

// Dense items of this CTA, run by warps 0-3.
__device__ void dense_loop(const Params& P, uint8_t* smem_raw) {
  const int tid = threadIdx.x, warp = tid >> 5;
  DenseState d;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  d.smem = smem_raw + pad;
  d.sbase = raw + pad;
  d.ph_kv0 = d.ph_kv1 = d.ph_s = d.ph_o = 0;
  volatile int* s_idx = reinterpret_cast<volatile int*>(d.smem + kOffMisc);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(d.smem + kOffMisc + 8);
  if (tid == 0) {
    mbar_init(bar_kv(d, 0), 1);
    mbar_init(bar_kv(d, 1), 1);
    mbar_init(bar_s(d), 1);
    mbar_init(bar_o(d), 1);
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
  group_sync();
  tc_fence_after();
  d.tmem = *reinterpret_cast<volatile uint32_t*>(s_tmem);
  for (;;) {
    if (tid == 0) *s_idx = (int)atomicAdd(&P.dp.ctr[kCtrDense], 1u);
    group_sync();
    const int idx = *s_idx;
    group_sync();
    if (idx >= P.dp.n_ditems) break;
    const int4* ip = reinterpret_cast<const int4*>(P.dp.ditems + idx);
    const int4 a = __ldg(ip), b = __ldg(ip + 1);
    const Item it{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (!dense_item(P, d, it)) {
      // a wait gave up: wait (bounded) for this CTA's tensor-core work to drain
      // before the TMEM is released
      if (tid == 0) {
        raise(P, kErrTimeout);
        tc_commit(bar_s(d));
        mbar_wait(bar_s(d), d.ph_s);
      }
      break;
    }
  }
  tc_fence_before();
  group_sync();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(d.tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------ the launch

template <int PATH>
__device__ __forceinline__ void run_item(const Params& P, const Item& it, int lane) {
  if constexpr (PATH == kPathMmaBf16D128) mma_item(P, it, lane);
  else if constexpr (PATH == kPathSimtF32D64) simt_item<float, 64>(P, it, lane);
  else if constexpr (PATH == kPathSimtF32D128) simt_item<float, 128>(P, it, lane);
  else if constexpr (PATH == kPathSimtBf16D64) simt_item<__nv_bfloat16, 64>(P, it, lane);
  else simt_item<__nv_bfloat16, 128>(P, it, lane);
}

template <int PATH>
__global__ void __launch_bounds__(kThreads, 1) psattn_fused_decode(const __grid_constant__ Params P) {
  const int lane = threadIdx.x & 31;
  if constexpr (PATH == kPathMmaBf16D128) {
    extern __shared__ uint8_t dyn_smem[];
    if (P.dp.n_ditems > 0 && threadIdx.x < 128) dense_loop(P, dyn_smem);
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
    static bool attr_set = false;  // once per process; the attribute is per function
    if (!attr_set) {
      cudaError_t e = cudaFuncSetAttribute(psattn_fused_decode<PATH>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      attr_set = true;
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

}  // namespace

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
