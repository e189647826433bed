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
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "psattn_internal.h"

using namespace psattn;

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = kWarpsPerCta * 32;

struct Params {
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

// Block ids of a span, 32 at a time in a register of every lane; returns the
// physical id of local block bi (warp-uniform), or -1 when it is out of range.
struct BlockIds {
  int cache, base;
  __device__ __forceinline__ BlockIds() : cache(-1), base(-64) {}
  __device__ __forceinline__ int get(const Params& P, const Span& s, int bi, int nb, int lane) {
    if (bi - base >= 32 || bi < base) {
      base = bi;
      int id = -1;
      const int b = bi + lane;
      if (b < nb) {
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
      }
      cache = id;
    }
    return __shfl_sync(0xffffffffu, cache, bi - base);
  }
};

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
  BlockIds ids;
  uint4 kr[2][4];
  int id_next = nb > 0 ? ids.get(P, s, 0, nb, lane) : -1;
  auto load_k = [&](int id) {
    const __nv_bfloat16* kb = pool + ((size_t)id * 2 * P.Hkv + h) * head_stride;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u) kr[j][u] = ld_kv(kb + (8 * j + g) * D + 8 * (tig + 4 * u));
  };
  if (id_next >= 0) load_k(id_next);

  for (int bi = 0; bi < nb; ++bi) {
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
      id_next = ids.get(P, s, bi + 1, nb, lane);
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
  BlockIds ids;
  for (int bi = 0; bi < nb; ++bi) {
    const int id = ids.get(P, s, bi, nb, lane);
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
__global__ void __launch_bounds__(kThreads, 1) psattn_fused_decode(const Params P) {
  const int lane = threadIdx.x & 31;
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
  psattn_fused_decode<PATH><<<grid, kThreads, 0, st>>>(P);
  return cudaGetLastError();
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
