// Host planner and the C ABI around it (psattn_plan, psattn_plan_host,
// psattn_decode's host side, info/export/status/destroy).
//
// Planning follows BatchLLM's description of the fused prefix-sharing kernel
// (papercache.org, "BatchLLM ...", section 5 "horizontal fusion"): the prefix
// partials and the distinct (suffix) partials of a whole batch become one flat
// list of work items, run by one persistent launch, with different tile shapes
// for the two kinds.  A long shared prefix is split along its KV range ("split-k",
// section 6.3.3) so that a few large groups still fill every SM; the pieces are
// merged like any other partial (Eq. 1, online softmax).  Multi-level prefixes
// (section 2.2 last paragraph, section 4.2) give one partial list per level, or
// one level per leaf under PSATTN_FLATTEN (the paper's first-level enlargement,
// applied here to an existing tree rather than re-derived by its DP).
//
// Everything here is integer work and deterministic: the same inputs and SM
// count give byte-identical tables.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <new>

#include "psattn_internal.h"

using namespace psattn;

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Groups with at least this many q rows (members x G) run as tensor-core tiles.
// Measured on the skewed workload (many small groups over long prefixes):
// 8 rows 0.347 ms, 16 rows 0.353, 32 rows 0.377, 64 rows 0.410; the
// tensor-core tile reads a group's prefix once even when it is mostly empty,
// where per-warp items of 8 rows would read it once per item.
constexpr int kDenseMinRows = 8;
constexpr int kDenseTileTok = 128;    // tokens per tensor-core K/V tile
constexpr int kDenseMaxChunk = 8192;  // tokens per dense item

struct Inputs {
  const psattn_shape* s;
  const int32_t *bt, *gor, *gpar, *plen, *slen;
  uint32_t flags;
  const int32_t* leaf_len = nullptr;  // ragged leaf levels (NULL: none)
};

int check_shape(const psattn_shape* s, uint32_t flags, int32_t* path) {
  if (!s) return PSATTN_ERR_INVALID_ARG;
  if (s->num_req < 0 || s->num_groups < 0 || s->num_q_heads <= 0 || s->num_kv_heads <= 0 ||
      s->head_dim <= 0 || s->block_size <= 0 || s->num_pool_blocks <= 0 ||
      (s->num_req > 0 && s->max_blocks_per_req <= 0) || !std::isfinite(s->scale))
    return PSATTN_ERR_INVALID_ARG;
  if (s->num_q_heads % s->num_kv_heads) return PSATTN_ERR_INVALID_ARG;
  const int G = s->num_q_heads / s->num_kv_heads;
  if (s->block_size != kBlockSize) return PSATTN_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PSATTN_ERR_UNSUPPORTED;
  if (s->dtype == PSATTN_BF16) {
    if (s->head_dim == 128 && !(flags & PSATTN_SIMT)) *path = kPathMmaBf16D128;
    else if (s->head_dim == 128) *path = kPathSimtBf16D128;
    else if (s->head_dim == 64) *path = kPathSimtBf16D64;
    else return PSATTN_ERR_UNSUPPORTED;
  } else if (s->dtype == PSATTN_F32) {
    if (s->head_dim == 64) *path = kPathSimtF32D64;
    else if (s->head_dim == 128) *path = kPathSimtF32D128;
    else return PSATTN_ERR_UNSUPPORTED;
  } else {
    return PSATTN_ERR_UNSUPPORTED;
  }
  const int rows = (*path == kPathMmaBf16D128) ? kMmaRows : kSimtRows;
  if (G > rows) return PSATTN_ERR_UNSUPPORTED;
  return PSATTN_OK;
}

// Chain of group g, root first.  Returns false on a bad id or a cycle.
bool chain_of(const Inputs& in, int32_t g, std::vector<int32_t>& out) {
  out.clear();
  const int ng = in.s->num_groups;
  while (g >= 0) {
    if (g >= ng || (int)out.size() > ng) return false;
    out.push_back(g);
    g = in.gpar ? in.gpar[g] : -1;
    if (g < -1) return false;
  }
  std::reverse(out.begin(), out.end());
  return true;
}

int build(const Inputs& in, int32_t num_sms, HostPlan& hp) {
  const psattn_shape& s = *in.s;
  int32_t path = 0;
  int rc = check_shape(in.s, in.flags, &path);
  if (rc) return rc;
  if (s.num_req > 0 && (!in.bt || !in.gor || !in.slen)) return PSATTN_ERR_INVALID_ARG;
  if (s.num_groups > 0 && !in.plen) return PSATTN_ERR_INVALID_ARG;
  if (num_sms < 1) return PSATTN_ERR_INVALID_ARG;

  const int R = s.num_req, NG = s.num_groups, Hkv = s.num_kv_heads;
  const int G = s.num_q_heads / Hkv, B = s.block_size, maxb = s.max_blocks_per_req;
  const bool no_dedup = in.flags & PSATTN_NO_DEDUP;
  const bool flatten = in.flags & PSATTN_FLATTEN;

  hp.shape = s;
  hp.flags = in.flags;
  hp.num_sms = num_sms;
  hp.path = path;
  hp.grid = num_sms;

  // ---- groups: ids, lengths, cycles
  for (int g = 0; g < NG; ++g) {
    if (in.plen[g] < 0) return PSATTN_ERR_INVALID_ARG;
    if (in.gpar && (in.gpar[g] < -1 || in.gpar[g] >= NG)) return PSATTN_ERR_GROUP_CYCLE;
  }
  std::vector<int32_t> ch;
  for (int g = 0; g < NG; ++g)
    if (!chain_of(in, g, ch)) return PSATTN_ERR_GROUP_CYCLE;

  // ---- requests: chains, token counts, block-table columns and ids
  // Internal chain of a request: the original chain, or its leaf alone under FLATTEN.
  std::vector<std::vector<int32_t>> rchain(R);
  hp.len_add.assign(NG, 0);
  for (int r = 0; r < R; ++r) {
    const int32_t leaf = in.gor[r];
    if (leaf < -1 || leaf >= NG) return PSATTN_ERR_INVALID_ARG;
    if (in.slen[r] < 0) return PSATTN_ERR_INVALID_ARG;
    if (!chain_of(in, leaf, ch)) return PSATTN_ERR_GROUP_CYCLE;
    int64_t tokens = in.slen[r], cols = ceil_div(in.slen[r], B);
    for (size_t i = 0; i < ch.size(); ++i) {
      tokens += in.plen[ch[i]];
      cols += ceil_div(in.plen[ch[i]], B);
      if (flatten && i + 1 < ch.size() && in.plen[ch[i]] % B) return PSATTN_ERR_UNSUPPORTED;
    }
    // the kernel and the flattened chains count a request's tokens (its whole
    // chain and suffix, seen or not) in int32
    if (tokens > INT32_MAX) return PSATTN_ERR_INVALID_ARG;
    if (in.leaf_len && in.leaf_len[r] != -1) {
      // a ragged leaf: the request sees the first leaf_len tokens of its leaf
      // level (the tensor-core and mma.sync paths mask per row)
      if (leaf < 0 || flatten || in.leaf_len[r] < 0 || in.leaf_len[r] > in.plen[leaf])
        return PSATTN_ERR_INVALID_ARG;
      if (path != kPathMmaBf16D128) return PSATTN_ERR_UNSUPPORTED;
      tokens -= in.plen[leaf] - in.leaf_len[r];
    }
    if (tokens < 1) return PSATTN_ERR_EMPTY_REQUEST;
    if (cols > maxb) return PSATTN_ERR_INVALID_ARG;
    const int32_t* row = in.bt + (int64_t)r * maxb;
    for (int64_t c = 0; c < cols; ++c)
      if (row[c] < 0 || row[c] >= s.num_pool_blocks) return PSATTN_ERR_BLOCK_OOB;
    if (flatten && !ch.empty()) {
      int32_t add = 0;
      for (size_t i = 0; i + 1 < ch.size(); ++i) add += in.plen[ch[i]];
      hp.len_add[leaf] = add;
      rchain[r].assign(1, leaf);
    } else {
      rchain[r] = ch;
    }
  }

  // ---- members per (internal) group and column bases
  auto level_len = [&](int g) -> int64_t { return (int64_t)in.plen[g] + hp.len_add[g]; };
  std::vector<std::vector<int32_t>> mem(NG);
  std::vector<int32_t> col_base(NG, -1);
  auto gather_members = [&]() {
    for (auto& m : mem) m.clear();
    col_base.assign(NG, -1);
    for (int r = 0; r < R; ++r) {
      int64_t col = 0;
      for (int32_t g : rchain[r]) {
        mem[g].push_back(r);
        col_base[g] = (int32_t)col;  // identical for every member: same chain prefix
        col += ceil_div(level_len(g), B);
      }
    }
  };
  gather_members();
  // levels the roofline counts once each (before any folding below)
  std::vector<char> level_used(NG, 0);
  for (int g = 0; g < NG; ++g) level_used[g] = !mem[g].empty();

  // ---- dedup check: every member reads the same physical blocks as the first
  if (!no_dedup) {
    for (int g = 0; g < NG; ++g) {
      if (mem[g].size() < 2) continue;
      const int64_t nb = ceil_div(level_len(g), B);
      const int32_t* a = in.bt + (int64_t)mem[g][0] * maxb + col_base[g];
      for (size_t k = 1; k < mem[g].size(); ++k) {
        const int32_t* b = in.bt + (int64_t)mem[g][k] * maxb + col_base[g];
        if (std::memcmp(a, b, sizeof(int32_t) * nb)) return PSATTN_ERR_GROUP_MISMATCH;
      }
    }
  }

  const int rows_w = (path == kPathMmaBf16D128) ? kMmaRows : kSimtRows;
  const int mpi = no_dedup ? 1 : std::max(1, rows_w / G);  // members per warp prefix item
  const int mpt = kDenseRows / G;                          // members per dense tile
  // the TMA row coordinate of a block is an int32: (block * 2 + kv) * Hkv * 16
  const bool tma_ok = (int64_t)s.num_pool_blocks * 2 * Hkv * B <= INT32_MAX;
  const bool tensor = !no_dedup && !(in.flags & PSATTN_NO_TENSOR_PREFIX) &&
                      path == kPathMmaBf16D128 && tma_ok;

  // ---- folding parent levels into their children's tensor-core items.
  // Every 128-row tile of a level reads the whole level.  When the members of
  // a level that sit in child groups run on tensor-core tiles there, and those
  // children's tiles plus the tiles of the level's own requests are no more
  // than the level needs anyway, each child's tiles can read the level first
  // and then their own tokens: the same K/V reads and tile rows, and per
  // member below the level one partial, one item epilogue and one merge step
  // fewer (the first-level enlargement of BatchLLM section 4.2, applied where
  // it costs no extra reads).  The level keeps items for its own requests
  // only.  Its blocks lead each child's span, so it must be a whole number of
  // blocks.
  if (tensor && !flatten && !(in.flags & PSATTN_NO_FOLD) && in.gpar) {
    std::vector<int64_t> direct(NG, 0), child_tiles(NG, 0);
    std::vector<char> small_child(NG, 0), fold(NG, 0);
    for (int r = 0; r < R; ++r)
      if (in.gor[r] >= 0) ++direct[in.gor[r]];
    for (int g = 0; g < NG; ++g) {
      const int32_t par = in.gpar[g];
      if (par < 0 || mem[g].empty()) continue;
      child_tiles[par] += ceil_div((int64_t)mem[g].size(), mpt);
      if ((int64_t)mem[g].size() * G < kDenseMinRows) small_child[par] = 1;
    }
    bool any = false;
    for (int g = 0; g < NG; ++g) {
      // the level's own requests keep tiles of their own, so they too must
      // fill one (no per-warp item re-reading the level)
      const bool own_ok = direct[g] == 0 || direct[g] * G >= kDenseMinRows;
      fold[g] = !mem[g].empty() && in.plen[g] > 0 && in.plen[g] % B == 0 && own_ok &&
                !small_child[g] && child_tiles[g] > 0 &&
                child_tiles[g] + ceil_div(direct[g], mpt) <=
                    ceil_div((int64_t)mem[g].size(), mpt);
      any = any || fold[g];
    }
    if (any) {
      std::vector<int32_t> kept;
      for (int r = 0; r < R; ++r) {
        kept.clear();
        int32_t pending = 0;  // tokens of folded levels above the next kept one
        const size_t n = rchain[r].size();
        for (size_t i = 0; i < n; ++i) {
          const int32_t g = rchain[r][i];
          if (fold[g] && i + 1 < n) {  // a request's own level stays its own
            pending += in.plen[g];
            continue;
          }
          hp.len_add[g] = pending;  // the same for every member: same chain above g
          pending = 0;
          kept.push_back(g);
        }
        rchain[r] = kept;
      }
      gather_members();
    }
  }

  // ---- dense classification and work estimates (token x KV-head units)
  std::vector<int32_t> dense(NG, 0);
  int64_t w_warp = 0, w_dense = 0;
  for (int g = 0; g < NG; ++g) {
    if (mem[g].empty() || level_len(g) == 0) continue;
    const int64_t rows = (int64_t)mem[g].size() * G;
    dense[g] = tensor && rows >= kDenseMinRows;
    if (dense[g]) w_dense += ceil_div(mem[g].size(), mpt) * level_len(g);
    else w_warp += ceil_div(mem[g].size(), mpi) * level_len(g);
  }
  for (int r = 0; r < R; ++r) w_warp += in.slen[r];

  // Chunk targets: a warp item at most a warp's average share of the warp
  // work; dense items about one per SM (capped at kDenseMaxChunk tokens).
  // Measured: more, smaller items cost more in per-item epilogues, tickets
  // and merges than they gain in balance; the per-warp items fill the gaps.
  const int64_t warps = (int64_t)num_sms * kWarpsPerCta;
  const int64_t c_warp = std::max<int64_t>(64, round_up(ceil_div(w_warp * Hkv, warps), B));
  const int64_t c_dense = std::min<int64_t>(
      kDenseMaxChunk,
      std::max<int64_t>(256, round_up(ceil_div(w_dense * Hkv, (int64_t)num_sms), kDenseTileTok)));
  auto chunking = [&](int64_t len, int64_t target, int32_t* chunk, int32_t* n, int64_t unit) {
    if (len <= 0) { *chunk = (int32_t)B; *n = 0; return; }
    int64_t k = ceil_div(len, target);
    int64_t c = std::min(round_up(ceil_div(len, k), unit), round_up(target, unit));
    *chunk = (int32_t)c;
    *n = (int32_t)ceil_div(len, c);
  };

  hp.grp.assign(NG, GroupInfo{});
  hp.members.clear();
  for (int g = 0; g < NG; ++g) {
    GroupInfo& gi = hp.grp[g];
    gi.col_base = col_base[g] < 0 ? 0 : col_base[g];
    gi.mem_off = (int32_t)hp.members.size();
    gi.n_mem = (int32_t)mem[g].size();
    gi.rep = mem[g].empty() ? -1 : mem[g][0];
    gi.dense = dense[g];
    gi.slot_j0 = -1;
    if (mem[g].empty()) { gi.chunk_tok = B; gi.n_chunks = 0; continue; }
    chunking(level_len(g), dense[g] ? c_dense : c_warp, &gi.chunk_tok, &gi.n_chunks,
             dense[g] ? kDenseTileTok : B);
    hp.members.insert(hp.members.end(), mem[g].begin(), mem[g].end());
    hp.prefix_chunk_max = std::max(hp.prefix_chunk_max, gi.n_chunks ? gi.chunk_tok : 0);
  }

  // ---- partial slots
  hp.req.assign(R, ReqInfo{});
  int64_t slot = 0;
  for (int r = 0; r < R; ++r) {
    ReqInfo& ri = hp.req[r];
    int32_t j = 0;
    int64_t col = 0;
    for (int32_t g : rchain[r]) {
      GroupInfo& gi = hp.grp[g];
      if (gi.slot_j0 < 0) gi.slot_j0 = j;  // same j for all members (same chain prefix)
      j += gi.n_chunks;
      col += ceil_div(level_len(g), B);
    }
    ri.suffix_col = (int32_t)col;
    chunking(in.slen[r], c_warp, &ri.suffix_chunk, &ri.suffix_nchunks, B);
    hp.suffix_chunk_max = std::max(hp.suffix_chunk_max, ri.suffix_nchunks ? ri.suffix_chunk : 0);
    j += ri.suffix_nchunks;
    ri.slot_base = (int32_t)slot;
    ri.n_partials = j;
    ri.leaf = in.gor[r];
    // a ragged leaf's visible tokens, counted from the start of its level's
    // span (which folded levels above it lead)
    ri.leaf_vis = in.leaf_len ? in.leaf_len[r] : -1;
    if (ri.leaf_vis >= 0) ri.leaf_vis += hp.len_add[ri.leaf];
    if (ri.leaf_vis >= 0) hp.any_ragged = 1;
    slot += j;
    if (slot > INT32_MAX / 2) return PSATTN_ERR_NOMEM;
  }
  for (auto& gi : hp.grp)
    if (gi.slot_j0 < 0) gi.slot_j0 = 0;
  hp.n_slots = slot;

  // ---- items
  auto seg_tokens = [](int64_t len, int32_t chunk, int32_t n, int32_t c) -> int32_t {
    int64_t lo = (int64_t)c * chunk, hi = (c == n - 1) ? len : std::min<int64_t>(len, lo + chunk);
    return (int32_t)std::max<int64_t>(0, hi - lo);
  };
  hp.witems.clear();
  hp.ditems.clear();
  const int64_t tb = 2LL * Hkv * s.head_dim * (s.dtype == PSATTN_F32 ? 4 : 2);
  int64_t planned_tok = 0;
  for (int g = 0; g < NG; ++g) {
    const GroupInfo& gi = hp.grp[g];
    if (gi.n_chunks == 0) continue;
    const int per = gi.dense ? mpt : mpi;
    for (int32_t m0 = 0; m0 < gi.n_mem; m0 += per) {
      const int32_t nm = std::min<int32_t>(per, gi.n_mem - m0);
      // on a ragged level, the farthest token any member of the item sees
      int64_t reach = 0;
      bool short_all = gi.dense != 0;
      for (int32_t m = m0; m < m0 + nm; ++m) {
        const ReqInfo& ri = hp.req[hp.members[gi.mem_off + m]];
        const bool ragged = ri.leaf_vis >= 0 && ri.leaf == g;
        const int64_t lim = ragged ? ri.leaf_vis : level_len(g);
        if (!ragged) short_all = false;
        reach = std::max(reach, lim);
      }
      for (int32_t c = 0; c < gi.n_chunks; ++c) {
        int32_t t = seg_tokens(level_len(g), gi.chunk_tok, gi.n_chunks, c);
        int32_t kind = gi.dense ? kItemDense : kItemPrefix;
        if (short_all) {  // tensor-core item on a ragged level: skip the tiles no row sees
          const int64_t lo = (int64_t)c * gi.chunk_tok;
          t = (int32_t)std::max<int64_t>(0, std::min<int64_t>(t, reach - lo));
          kind = kItemDenseRagged;
        }
        planned_tok += t;
        for (int h = 0; h < Hkv; ++h) {
          Item it{kind, h, g, c, gi.mem_off + m0, nm, gi.slot_j0 + c, t};
          (gi.dense ? hp.ditems : hp.witems).push_back(it);
        }
      }
    }
  }
  for (int r = 0; r < R; ++r) {
    const ReqInfo& ri = hp.req[r];
    const int32_t j0 = ri.n_partials - ri.suffix_nchunks;
    for (int32_t c = 0; c < ri.suffix_nchunks; ++c) {
      const int32_t t = seg_tokens(in.slen[r], ri.suffix_chunk, ri.suffix_nchunks, c);
      planned_tok += t;
      for (int h = 0; h < Hkv; ++h) hp.witems.push_back(Item{kItemSuffix, h, r, c, 0, 1, j0 + c, t});
    }
  }
  // Heaviest first; ties: prefix before suffix, then segment, chunk, KV head, members.
  auto order = [](const Item& a, const Item& b) {
    if (a.cost != b.cost) return a.cost > b.cost;
    if (a.kind != b.kind) return a.kind > b.kind;
    if (a.seg != b.seg) return a.seg < b.seg;
    if (a.chunk != b.chunk) return a.chunk < b.chunk;
    if (a.kvh != b.kvh) return a.kvh < b.kvh;
    return a.mem_off < b.mem_off;
  };
  std::stable_sort(hp.witems.begin(), hp.witems.end(), order);
  std::stable_sort(hp.ditems.begin(), hp.ditems.end(), order);

  // ---- byte accounting (K+V of all KV heads per token = tb)
  // (a folded level once, however many children read it; under FLATTEN each
  // leaf's whole chain, the bytes that mode must read)
  int64_t uniq_tok = 0;
  for (int g = 0; g < NG; ++g)
    if (level_used[g]) uniq_tok += flatten ? level_len(g) : in.plen[g];
  for (int r = 0; r < R; ++r) uniq_tok += in.slen[r];
  hp.unique_kv_bytes = uniq_tok * tb;
  hp.planned_kv_bytes = planned_tok * tb;
  hp.qo_bytes = (int64_t)R * s.num_q_heads *
                (2LL * s.head_dim * (s.dtype == PSATTN_F32 ? 4 : 2) + 4);
  return PSATTN_OK;
}

}  // namespace

struct psattn_plan_s {
  HostPlan hp;
  bool on_device = false;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  size_t reset_bytes = 0;        // counters + tickets at the head of ws
  cudaEvent_t done = nullptr;    // recorded after every launch on this plan
  cudaStream_t aux = nullptr;    // the plan's own stream for status reads and resets
  DevPlan dp{};
};

namespace {

int plan_common(const psattn_shape* shape, const int32_t* bt, const int32_t* gor,
                const int32_t* gpar, const int32_t* plen, const int32_t* slen, uint32_t flags,
                int32_t num_sms, psattn_plan_t* out, std::unique_ptr<psattn_plan_s>& p,
                const int32_t* leaf_len = nullptr) {
  if (!out) return PSATTN_ERR_INVALID_ARG;
  *out = nullptr;
  p.reset(new (std::nothrow) psattn_plan_s());
  if (!p) return PSATTN_ERR_NOMEM;
  Inputs in{shape, bt, gor, gpar, plen, slen, flags, leaf_len};
  try {
    return build(in, num_sms, p->hp);
  } catch (const std::bad_alloc&) {
    return PSATTN_ERR_NOMEM;
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int upload(psattn_plan_s* p, cudaStream_t stream) {
  HostPlan& hp = p->hp;
  const int R = hp.shape.num_req, Hkv = hp.shape.num_kv_heads;
  const int G = hp.shape.num_q_heads / Hkv, d = hp.shape.head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + std::max<size_t>(bytes, 1)); return o; };
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
  p->ws_bytes = off;
  p->reset_bytes = o_wi - o_ctr;
  if (cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p->aux, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  if (cudaMalloc(&p->ws, off) != cudaSuccess) {
    cudaGetLastError();
    p->ws = nullptr;
    return PSATTN_ERR_NOMEM;
  }
  char* base = static_cast<char*>(p->ws);
  DevPlan& dp = p->dp;
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
  cudaError_t e = cudaMemsetAsync(base + o_ctr, 0, o_wi - o_ctr, stream);  // counters + tickets
  auto put = [&](size_t o, const void* src, size_t bytes) {
    if (e == cudaSuccess && bytes) e = cudaMemcpyAsync(base + o, src, bytes, cudaMemcpyHostToDevice, stream);
  };
  put(o_wi, hp.witems.data(), sizeof(Item) * hp.witems.size());
  put(o_di, hp.ditems.data(), sizeof(Item) * hp.ditems.size());
  put(o_req, hp.req.data(), sizeof(ReqInfo) * hp.req.size());
  put(o_grp, hp.grp.data(), sizeof(GroupInfo) * hp.grp.size());
  put(o_mem, hp.members.data(), sizeof(int32_t) * hp.members.size());
  put(o_add, hp.len_add.data(), sizeof(int32_t) * hp.len_add.size());
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  p->on_device = true;
  return PSATTN_OK;
}

// Releases what upload() created (any part of it may be missing).
void release_device(psattn_plan_s* p) {
  if (p->done) cudaEventSynchronize(p->done);
  if (p->ws) cudaFree(p->ws);
  if (p->done) cudaEventDestroy(p->done);
  if (p->aux) cudaStreamDestroy(p->aux);
  cudaGetLastError();
  p->ws = nullptr;
  p->done = nullptr;
  p->aux = nullptr;
}

}  // namespace

const psattn::HostPlan* psattn_internal_host_plan(psattn_plan_t plan) {
  return plan ? &plan->hp : nullptr;
}

extern "C" {

int psattn_plan_host(const psattn_shape* shape, const int32_t* block_table,
                     const int32_t* group_of_req, const int32_t* group_parent,
                     const int32_t* prefix_len, const int32_t* suffix_len, uint32_t flags,
                     int32_t num_sms, psattn_plan_t* out) {
  std::unique_ptr<psattn_plan_s> p;
  int rc = plan_common(shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
                       flags, num_sms, out, p);
  if (rc) return rc;
  *out = p.release();
  return PSATTN_OK;
}

int psattn_plan_host_ragged(const psattn_shape* shape, const int32_t* block_table,
                            const int32_t* group_of_req, const int32_t* group_parent,
                            const int32_t* prefix_len, const int32_t* suffix_len,
                            const int32_t* leaf_len, uint32_t flags, int32_t num_sms,
                            psattn_plan_t* out) {
  std::unique_ptr<psattn_plan_s> p;
  int rc = plan_common(shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
                       flags, num_sms, out, p, leaf_len);
  if (rc) return rc;
  *out = p.release();
  return PSATTN_OK;
}

int psattn_plan_ragged(const psattn_shape* shape, const int32_t* block_table,
                       const int32_t* group_of_req, const int32_t* group_parent,
                       const int32_t* prefix_len, const int32_t* suffix_len,
                       const int32_t* leaf_len, uint32_t flags, psattn_stream_t stream,
                       psattn_plan_t* out) {
  if (!out) return PSATTN_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  std::unique_ptr<psattn_plan_s> p;
  int rc = plan_common(shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
                       flags, sms, out, p, leaf_len);
  if (rc) return rc;
  rc = upload(p.get(), reinterpret_cast<cudaStream_t>(stream));
  if (rc) {
    release_device(p.get());
    return rc;
  }
  *out = p.release();
  return PSATTN_OK;
}

int psattn_plan(const psattn_shape* shape, const int32_t* block_table,
                const int32_t* group_of_req, const int32_t* group_parent,
                const int32_t* prefix_len, const int32_t* suffix_len, uint32_t flags,
                psattn_stream_t stream, psattn_plan_t* out) {
  if (!out) return PSATTN_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  std::unique_ptr<psattn_plan_s> p;
  int rc = plan_common(shape, block_table, group_of_req, group_parent, prefix_len, suffix_len,
                       flags, sms, out, p);
  if (rc) return rc;
  rc = upload(p.get(), reinterpret_cast<cudaStream_t>(stream));
  if (rc) {
    release_device(p.get());
    return rc;
  }
  *out = p.release();
  return PSATTN_OK;
}

int psattn_decode(psattn_plan_t plan, const void* q, const void* kv_pool,
                  const int32_t* block_table, const int32_t* group_of_req,
                  const int32_t* prefix_len, const int32_t* suffix_len, void* out, float* lse,
                  psattn_stream_t stream) {
  if (!plan || !plan->on_device) return PSATTN_ERR_INVALID_ARG;
  const HostPlan& hp = plan->hp;
  if (hp.shape.num_req == 0) return PSATTN_OK;
  if (!q || !kv_pool || !block_table || !group_of_req || !suffix_len || !out)
    return PSATTN_ERR_INVALID_ARG;
  if (hp.shape.num_groups > 0 && !prefix_len) return PSATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(q) || misaligned(kv_pool) || misaligned(out) ||
      (reinterpret_cast<uintptr_t>(lse) & 3))
    return PSATTN_ERR_INVALID_ARG;
  const int rc = psattn_launch_decode(hp, plan->dp, q, kv_pool, block_table, group_of_req,
                                     prefix_len, suffix_len, out, lse, stream);
  if (rc) return rc;
  // marks the end of this launch for psattn_plan_status and psattn_plan_destroy
  if (cudaEventRecord(plan->done, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  return PSATTN_OK;
}

int psattn_plan_info_get(psattn_plan_t plan, psattn_plan_info* info) {
  if (!plan || !info) return PSATTN_ERR_INVALID_ARG;
  const HostPlan& hp = plan->hp;
  info->warp_items = (int64_t)hp.witems.size();
  info->dense_items = (int64_t)hp.ditems.size();
  info->partial_slots = hp.n_slots;
  info->workspace_bytes = (int64_t)plan->ws_bytes;
  info->unique_kv_bytes = hp.unique_kv_bytes;
  info->planned_kv_bytes = hp.planned_kv_bytes;
  info->qo_bytes = hp.qo_bytes;
  info->suffix_chunk_max = hp.suffix_chunk_max;
  info->prefix_chunk_max = hp.prefix_chunk_max;
  info->num_sms = hp.num_sms;
  info->grid = hp.grid;
  info->dense_item_warps = hp.ditems.empty() ? 0 : kDenseItemWarps;
  return PSATTN_OK;
}

int64_t psattn_plan_export(psattn_plan_t plan, int32_t which, int32_t* dst, int64_t cap) {
  if (!plan) return PSATTN_ERR_INVALID_ARG;
  const HostPlan& hp = plan->hp;
  const int32_t* src = nullptr;
  int64_t n = 0;
  switch (which) {
    case 0: src = reinterpret_cast<const int32_t*>(hp.witems.data()); n = 8 * (int64_t)hp.witems.size(); break;
    case 1: src = reinterpret_cast<const int32_t*>(hp.ditems.data()); n = 8 * (int64_t)hp.ditems.size(); break;
    case 2: src = reinterpret_cast<const int32_t*>(hp.req.data()); n = 8 * (int64_t)hp.req.size(); break;
    case 3: src = reinterpret_cast<const int32_t*>(hp.grp.data()); n = 8 * (int64_t)hp.grp.size(); break;
    case 4: src = hp.members.data(); n = (int64_t)hp.members.size(); break;
    case 5: src = hp.len_add.data(); n = (int64_t)hp.len_add.size(); break;
    default: return PSATTN_ERR_INVALID_ARG;
  }
  if (dst && n) std::memcpy(dst, src, sizeof(int32_t) * (size_t)std::min(n, std::max<int64_t>(cap, 0)));
  return n;
}

int psattn_plan_status(psattn_plan_t plan, uint32_t* device_flags) {
  if (device_flags) *device_flags = 0;
  if (!plan) return PSATTN_ERR_INVALID_ARG;
  if (!plan->on_device) return PSATTN_OK;
  // Waits for the plan's last launch only (its event), then reads the error
  // word on the plan's own stream, so other work on the device runs on.
  uint32_t w = 0;
  cudaError_t e = cudaEventSynchronize(plan->done);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&w, plan->dp.ctr + kCtrErr, sizeof w, cudaMemcpyDeviceToHost, plan->aux);
  if (e == cudaSuccess) e = cudaStreamSynchronize(plan->aux);
  // A launch that raised the word may have ended with merge tickets that
  // never reached their count (a bounded wait gave up, or the merge
  // bookkeeping disagreed): the counters, tickets and the word itself all
  // start again from zero, so the next launch cannot merge stale partials.
  if (e == cudaSuccess && w) e = cudaMemsetAsync(plan->ws, 0, plan->reset_bytes, plan->aux);
  if (e == cudaSuccess && w) e = cudaStreamSynchronize(plan->aux);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  if (device_flags) *device_flags = w;
  return w ? PSATTN_ERR_DEVICE : PSATTN_OK;
}

int psattn_selftest_wait_timeout(uint32_t limit_us, uint32_t* device_flags) {
  if (device_flags) *device_flags = 0;
  if (limit_us < 1 || limit_us > 100000) return PSATTN_ERR_INVALID_ARG;
  uint32_t* d = nullptr;
  uint32_t w = 0;
  bool ok = cudaMalloc(&d, sizeof w) == cudaSuccess;
  ok = ok && cudaMemset(d, 0, sizeof w) == cudaSuccess;
  ok = ok && psattn_run_wait_selftest(d, 1000ull * limit_us, nullptr) == PSATTN_OK;
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  ok = ok && cudaMemcpy(&w, d, sizeof w, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (d) cudaFree(d);
  if (!ok) {
    cudaGetLastError();
    return PSATTN_ERR_CUDA;
  }
  if (device_flags) *device_flags = w;
  return w ? PSATTN_ERR_DEVICE : PSATTN_OK;
}

void psattn_plan_destroy(psattn_plan_t plan) {
  if (!plan) return;
  release_device(plan);  // waits for the plan's last launch first
  delete plan;
}

const char* psattn_status_string(int status) {
  switch (status) {
    case PSATTN_OK: return "ok";
    case PSATTN_ERR_INVALID_ARG: return "invalid argument";
    case PSATTN_ERR_BLOCK_OOB: return "block id out of range";
    case PSATTN_ERR_GROUP_MISMATCH: return "group member's prefix blocks differ from the group's";
    case PSATTN_ERR_EMPTY_REQUEST: return "request attends to no token";
    case PSATTN_ERR_UNSUPPORTED: return "unsupported dtype, head_dim, block_size or GQA ratio";
    case PSATTN_ERR_CUDA: return "CUDA runtime error";
    case PSATTN_ERR_DEVICE: return "kernel raised its error word";
    case PSATTN_ERR_NOMEM: return "out of memory";
    case PSATTN_ERR_GROUP_CYCLE: return "group_parent has a cycle or a bad id";
    default: return "unknown status";
  }
}

}  // extern "C"
