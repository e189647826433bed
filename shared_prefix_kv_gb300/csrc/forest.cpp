// Prefix-sharing groups and prefix-homogeneous batches from token ids, on
// the host.  The contract is in psattn_forest.h:
//  - psattn_forest_group: the compact prefix tree of BatchLLM section 4.2
//    ("BatchLLM: Optimizing Large Batched LLM Inference with Global Prefix
//    Sharing and Throughput-oriented Token Batching"), either as multi-level
//    groups or enlarged to one level per request by a dynamic program that
//    maximises the reused tokens;
//  - psattn_cht_batches: the chunked hash tree of Feather ("Requests of a
//    Feather Must Flock Together", methodology 1) forming batches by
//    smallest miss count.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <queue>
#include <unordered_map>
#include <unordered_set>
#include <utility>
#include <vector>

#include "psattn.h"
#include "psattn_forest.h"

namespace {

// splitmix64's output function (S. Vigna): mixes one 64-bit word.
inline uint64_t mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

struct Requests {
  const int32_t* tokens;
  const int64_t* offsets;
  int32_t R;
  int32_t chunk;
  int64_t len(int32_t r) const { return offsets[r + 1] - offsets[r]; }
  int64_t full_chunks(int32_t r) const { return len(r) / chunk; }
  const int32_t* chunk_at(int32_t r, int64_t i) const { return tokens + offsets[r] + i * chunk; }
  bool same_chunk(int32_t a, int32_t b, int64_t i) const {
    return std::memcmp(chunk_at(a, i), chunk_at(b, i), sizeof(int32_t) * (size_t)chunk) == 0;
  }
};

bool valid(const int32_t* tokens, const int64_t* offsets, int32_t R, int32_t chunk) {
  if (R < 0 || chunk < 1 || !offsets) return false;
  if (R > 0 && offsets[0] != 0) return false;
  for (int32_t r = 0; r < R; ++r)
    if (offsets[r + 1] < offsets[r]) return false;
  if (R > 0 && offsets[R] > 0 && !tokens) return false;
  return true;
}

// Cumulative chunk hashes: h[r][i] identifies chunks 0..i of request r (the
// hash of chunk i chained onto the hash of chunks 0..i-1).
std::vector<std::vector<uint64_t>> cumulative_hashes(const Requests& q) {
  std::vector<std::vector<uint64_t>> h((size_t)q.R);
  for (int32_t r = 0; r < q.R; ++r) {
    const int64_t n = q.full_chunks(r);
    h[r].resize((size_t)n);
    uint64_t acc = 0x2545F4914F6CDD1Dull;
    for (int64_t i = 0; i < n; ++i) {
      const int32_t* c = q.chunk_at(r, i);
      uint64_t x = mix64(acc ^ (uint64_t)(i + 1));
      for (int32_t t = 0; t < q.chunk; ++t) x = mix64(x ^ (uint32_t)c[t]);
      acc = x;
      h[r][(size_t)i] = acc;
    }
  }
  return h;
}

// The chunk trie: one node per distinct chunk-prefix of the requests (node 0
// is the empty prefix).  A node is looked up by its cumulative hash and then
// confirmed by its parent and the tokens of its own chunk, so requests share
// a node exactly when their chunk-prefixes are equal.
struct Trie {
  struct Node {
    int32_t parent = -1;
    int32_t depth = 0;  // chunks from the root to the end of this node
    int32_t rep = -1;   // smallest request id through the node
    int32_t count = 0;  // requests through the node
    std::vector<int32_t> children;
  };
  std::vector<Node> nodes;
  std::vector<std::vector<int32_t>> path;  // per request: node of each of its chunks
};

Trie build_trie(const Requests& q, const std::vector<std::vector<uint64_t>>& h) {
  Trie t;
  t.nodes.emplace_back();  // root
  t.path.resize((size_t)q.R);
  std::unordered_map<uint64_t, std::vector<int32_t>> index;
  for (int32_t r = 0; r < q.R; ++r) {
    int32_t cur = 0;
    const int64_t n = q.full_chunks(r);
    t.path[r].reserve((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
      std::vector<int32_t>& cand = index[h[r][(size_t)i]];
      int32_t next = -1;
      for (int32_t c : cand)
        if (t.nodes[c].parent == cur && q.same_chunk(t.nodes[c].rep, r, i)) {
          next = c;
          break;
        }
      if (next < 0) {
        next = (int32_t)t.nodes.size();
        Trie::Node nd;
        nd.parent = cur;
        nd.depth = t.nodes[cur].depth + 1;
        nd.rep = r;
        t.nodes.push_back(nd);
        t.nodes[cur].children.push_back(next);
        cand.push_back(next);
      }
      t.nodes[next].count += 1;
      t.path[r].push_back(next);
      cur = next;
    }
  }
  return t;
}

// Prefix levels: maximal runs of trie nodes that the same two or more
// requests pass through (a run continues from a node into a child exactly
// when every request through the node goes on into that child).
struct Levels {
  struct Level {
    int32_t parent = -1;     // level above, -1 at a root
    int32_t chunks = 0;      // chunks of this level
    int32_t end_depth = 0;   // chunks from the root to the end of this level
    int32_t count = 0;       // requests through the level
    int32_t rep = -1;        // smallest request id through the level
    int32_t ending = 0;      // requests whose deepest level this is
    std::vector<int32_t> children;  // ordered by rep
  };
  std::vector<Level> lv;            // in depth-first order (the group ids)
  std::vector<int32_t> deepest;     // per request: its deepest level, -1 = none
};

Levels build_levels(const Requests& q, const Trie& t) {
  const int32_t N = (int32_t)t.nodes.size();
  // start[n]: n opens a level (shared, and its parent is the root or a node
  // some request through it does not continue into n)
  std::vector<char> shared((size_t)N, 0), start((size_t)N, 0);
  for (int32_t n = 1; n < N; ++n) shared[n] = t.nodes[n].count >= 2;
  for (int32_t n = 1; n < N; ++n) {
    if (!shared[n]) continue;
    const int32_t p = t.nodes[n].parent;
    start[n] = (p == 0) || (t.nodes[p].count != t.nodes[n].count);
  }
  // level of every shared node: follow each start down its single-child run
  std::vector<int32_t> level_of((size_t)N, -1);
  Levels L;
  // depth-first over start nodes, children ordered by rep (node ids grow with
  // the first request that created them, so ordering by rep is ordering by id
  // of the smallest request through them)
  std::function<void(int32_t, int32_t)> visit = [&](int32_t s, int32_t parent_level) {
    const int32_t id = (int32_t)L.lv.size();
    L.lv.emplace_back();
    L.lv[id].parent = parent_level;
    L.lv[id].count = t.nodes[s].count;
    L.lv[id].rep = t.nodes[s].rep;
    if (parent_level >= 0) L.lv[parent_level].children.push_back(id);
    int32_t n = s, len = 0;
    for (;;) {
      level_of[n] = id;
      ++len;
      int32_t cont = -1;
      for (int32_t c : t.nodes[n].children)
        if (shared[c] && !start[c]) cont = c;  // (at most one: same count as n)
      if (cont < 0) break;
      n = cont;
    }
    L.lv[id].chunks = len;
    L.lv[id].end_depth = t.nodes[n].depth;
    // child levels start at shared children of the run's last node
    std::vector<int32_t> kids;
    for (int32_t c : t.nodes[n].children)
      if (shared[c] && start[c]) kids.push_back(c);
    std::sort(kids.begin(), kids.end(),
              [&](int32_t a, int32_t b) { return t.nodes[a].rep < t.nodes[b].rep; });
    for (int32_t c : kids) visit(c, id);
  };
  std::vector<int32_t> roots;
  for (int32_t c : t.nodes[0].children)
    if (shared[c]) roots.push_back(c);
  std::sort(roots.begin(), roots.end(),
            [&](int32_t a, int32_t b) { return t.nodes[a].rep < t.nodes[b].rep; });
  for (int32_t c : roots) visit(c, -1);
  L.deepest.assign((size_t)q.R, -1);
  for (int32_t r = 0; r < q.R; ++r) {
    for (int32_t n : t.path[r])
      if (level_of[n] >= 0) L.deepest[r] = level_of[n];
    if (L.deepest[r] >= 0) L.lv[L.deepest[r]].ending += 1;
  }
  return L;
}

// ---- single level: the first-level reuse DP (BatchLLM section 4.2)
//
// Over the level tree (d_v = tokens from the root to the end of level v,
// e_v = requests whose deepest level is v): F_v(u) is the largest saving
// inside v's subtree when exactly u of its requests are left for an
// ancestor to group.  The requests reaching v are the ones its children pass
// up plus the e_v ending at v; all of them share v's prefix, so the x of
// them kept at v form v's group and save (x - 1) * d_v (nothing for x < 2).
//   H_v(K) = max { sum_c F_c(k_c) : sum_c k_c = K }          (children merged)
//   F_v(u) = max_K { H_v(K) + save_v(K + e_v - u) : K + e_v >= u }
// The answer is max_K H_root(K) over the root levels (requests left at the
// root share nothing).  Counts are chosen top down from the stored argmax
// choices; then, bottom up, every level keeps the smallest request ids of
// those reaching it and passes the largest ones up.
struct Dp {
  std::vector<std::vector<int64_t>> F;             // per level, index u
  std::vector<std::vector<int32_t>> bestK;         // per level, index u
  std::vector<std::vector<std::vector<int32_t>>> split;  // per level, per child: k_c by merged K
  std::vector<std::vector<int64_t>> Hfinal;        // per level: H_v
};

constexpr int64_t kNeg = INT64_MIN / 4;

// merges children tables; returns H and fills the per-child choice tables
std::vector<int64_t> merge_children(const std::vector<int32_t>& kids,
                                    const std::vector<std::vector<int64_t>>& F,
                                    std::vector<std::vector<int32_t>>* choices) {
  std::vector<int64_t> H(1, 0);
  choices->clear();
  for (int32_t c : kids) {
    const std::vector<int64_t>& Fc = F[c];
    std::vector<int64_t> Hn(H.size() + Fc.size() - 1, kNeg);
    std::vector<int32_t> ch(Hn.size(), 0);
    for (size_t K = 0; K < H.size(); ++K) {
      if (H[K] == kNeg) continue;
      for (size_t k = 0; k < Fc.size(); ++k) {
        if (Fc[k] == kNeg) continue;
        const int64_t v = H[K] + Fc[k];
        if (v > Hn[K + k]) {  // strict: among equal totals the smallest k for this child
          Hn[K + k] = v;
          ch[K + k] = (int32_t)k;
        }
      }
    }
    H.swap(Hn);
    choices->push_back(std::move(ch));
  }
  return H;
}

int64_t single_level(const Levels& L, std::vector<int32_t>* keep_level /* per request */,
                     const std::vector<int32_t>& deepest) {
  const int32_t NL = (int32_t)L.lv.size();
  Dp dp;
  dp.F.resize((size_t)NL);
  dp.bestK.resize((size_t)NL);
  dp.split.resize((size_t)NL);
  // children before parents: levels are numbered depth first, so in reverse
  for (int32_t v = NL - 1; v >= 0; --v) {
    const Levels::Level& lv = L.lv[v];
    const std::vector<int64_t> H = merge_children(lv.children, dp.F, &dp.split[v]);
    const int64_t d = lv.end_depth;  // in chunks; scaled to tokens by the caller
    const int32_t n = lv.count;      // = (H.size() - 1) + ending
    dp.F[v].assign((size_t)n + 1, kNeg);
    dp.bestK[v].assign((size_t)n + 1, 0);
    for (int32_t u = 0; u <= n; ++u) {
      for (size_t K = 0; K < H.size(); ++K) {
        if (H[K] == kNeg) continue;
        const int64_t x = (int64_t)K + lv.ending - u;
        if (x < 0) continue;
        const int64_t val = H[K] + (x >= 2 ? (x - 1) * d : 0);
        if (val > dp.F[v][u]) {  // strict: the smallest K among equals
          dp.F[v][u] = val;
          dp.bestK[v][u] = (int32_t)K;
        }
      }
    }
  }
  // the root: every root level passes some requests up to "no group"
  std::vector<int32_t> roots;
  for (int32_t v = 0; v < NL; ++v)
    if (L.lv[v].parent < 0) roots.push_back(v);
  std::vector<std::vector<int32_t>> root_split;
  const std::vector<int64_t> Hroot = merge_children(roots, dp.F, &root_split);
  int64_t best = kNeg;
  size_t bestK = 0;
  for (size_t K = 0; K < Hroot.size(); ++K)
    if (Hroot[K] > best) {  // smallest K among equals: keep requests grouped
      best = Hroot[K];
      bestK = K;
    }
  // counts, top down: u[v] = requests level v passes up
  std::vector<int32_t> u((size_t)NL, 0);
  auto distribute = [&](const std::vector<int32_t>& kids,
                        const std::vector<std::vector<int32_t>>& choice, size_t K) {
    for (int32_t i = (int32_t)kids.size() - 1; i >= 0; --i) {
      const int32_t k = choice[(size_t)i][K];
      u[kids[(size_t)i]] = k;
      K -= (size_t)k;
    }
  };
  distribute(roots, root_split, bestK);
  for (int32_t v = 0; v < NL; ++v)  // parents before children (depth-first numbering)
    distribute(L.lv[v].children, dp.split[v], (size_t)dp.bestK[v][u[v]]);
  // requests, bottom up: a level keeps the smallest ids reaching it
  std::vector<std::vector<int32_t>> up((size_t)NL);
  std::vector<std::vector<int32_t>> ending((size_t)NL);
  for (int32_t r = 0; r < (int32_t)deepest.size(); ++r)
    if (deepest[r] >= 0) ending[deepest[r]].push_back(r);
  keep_level->assign(deepest.size(), -1);
  for (int32_t v = NL - 1; v >= 0; --v) {
    std::vector<int32_t> reach = ending[v];
    for (int32_t c : L.lv[v].children) reach.insert(reach.end(), up[c].begin(), up[c].end());
    std::sort(reach.begin(), reach.end());
    const size_t keep = reach.size() - (size_t)u[v];
    if (keep >= 2)
      for (size_t i = 0; i < keep; ++i) (*keep_level)[reach[i]] = v;
    up[v].assign(reach.begin() + (ptrdiff_t)keep, reach.end());
  }
  return best;
}

// ---- chunked hash tree batches (Feather, methodology 1)

void cht_batches(const Requests& q, const std::vector<std::vector<uint64_t>>& h,
                 int32_t max_batch, int32_t max_new, int32_t* batch_of_req, int32_t* order,
                 int32_t* num_batches) {
  const int32_t R = q.R;
  // inverted index: cumulative chunk hash -> requests holding it (each
  // request holds a given cumulative hash at most once: it fixes the position)
  std::unordered_map<uint64_t, std::vector<int32_t>> holders;
  for (int32_t r = 0; r < R; ++r)
    for (uint64_t x : h[r]) holders[x].push_back(r);
  std::vector<char> waiting((size_t)R, 1);
  std::vector<int32_t> miss((size_t)R, 0);
  int32_t placed = 0, nb = 0, next_seed = 0;
  using Entry = std::pair<int32_t, int32_t>;  // (misses, request id): min-heap
  while (placed < R) {
    while (!waiting[next_seed]) ++next_seed;
    const int32_t seed = next_seed;
    std::unordered_set<uint64_t> work(h[seed].begin(), h[seed].end());
    waiting[seed] = 0;
    batch_of_req[seed] = nb;
    order[placed++] = seed;
    int32_t size = 1;
    std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
    for (int32_t r = 0; r < R; ++r) {
      if (!waiting[r]) continue;
      int32_t m = 0;
      for (uint64_t x : h[r]) m += work.count(x) ? 0 : 1;
      miss[r] = m;
      heap.emplace(m, r);
    }
    while (size < max_batch && !heap.empty()) {
      const Entry top = heap.top();
      heap.pop();
      const int32_t r = top.second;
      if (!waiting[r] || top.first != miss[r]) continue;  // stale entry
      if (top.first > max_new) break;                     // nothing else may join
      waiting[r] = 0;
      batch_of_req[r] = nb;
      order[placed++] = r;
      ++size;
      for (uint64_t x : h[r]) {
        if (!work.insert(x).second) continue;
        for (int32_t w : holders[x])
          if (waiting[w]) heap.emplace(--miss[w], w);
      }
    }
    ++nb;
  }
  *num_batches = nb;
}

// Groups one set of requests (the body of psattn_forest_group): fills
// group_of_req / suffix_len per request and group_parent / prefix_len per
// group, and the saved tokens.
struct Grouping {
  std::vector<int32_t> gor, slen, gpar, plen;
  int64_t saved = 0;
};

void group_requests(const Requests& q, uint32_t flags, Grouping* out) {
  const auto h = cumulative_hashes(q);
  const Trie t = build_trie(q, h);
  const Levels L = build_levels(q, t);
  out->gor.assign((size_t)q.R, -1);
  out->slen.assign((size_t)q.R, 0);
  out->gpar.clear();
  out->plen.clear();
  const int32_t chunk = q.chunk;
  if (flags & PSATTN_FOREST_SINGLE) {
    std::vector<int32_t> keep;
    out->saved = single_level(L, &keep, L.deepest) * chunk;
    // groups: the levels that keep two or more requests, in level order
    std::vector<int32_t> gid(L.lv.size(), -1);
    for (int32_t r = 0; r < q.R; ++r)
      if (keep[r] >= 0) gid[keep[r]] = 0;
    for (size_t v = 0; v < L.lv.size(); ++v)
      if (gid[v] == 0) {
        gid[v] = (int32_t)out->plen.size();
        out->gpar.push_back(-1);
        out->plen.push_back(L.lv[v].end_depth * chunk);
      }
    for (int32_t r = 0; r < q.R; ++r) {
      const int32_t v = keep[r];
      out->gor[r] = v >= 0 ? gid[v] : -1;
      out->slen[r] = (int32_t)(q.len(r) - (v >= 0 ? (int64_t)L.lv[v].end_depth * chunk : 0));
    }
    return;
  }
  out->saved = 0;
  for (const auto& lv : L.lv) {
    out->saved += (int64_t)(lv.count - 1) * lv.chunks * chunk;
    out->gpar.push_back(lv.parent);
    out->plen.push_back(lv.chunks * chunk);
  }
  for (int32_t r = 0; r < q.R; ++r) {
    const int32_t v = L.deepest[r];
    out->gor[r] = v;
    out->slen[r] = (int32_t)(q.len(r) - (v >= 0 ? (int64_t)L.lv[v].end_depth * chunk : 0));
  }
}

}  // namespace

extern "C" {

int psattn_forest_group(const int32_t* tokens, const int64_t* offsets, int32_t num_req,
                        int32_t chunk, uint32_t flags, int32_t* group_of_req,
                        int32_t* group_parent, int32_t* prefix_len, int32_t* suffix_len,
                        int32_t cap, int32_t* num_groups, int64_t* saved_tokens) {
  if (!valid(tokens, offsets, num_req, chunk) || !num_groups ||
      (num_req > 0 && (!group_of_req || !suffix_len)) || cap < 0 ||
      (cap > 0 && (!group_parent || !prefix_len)) || (flags & ~PSATTN_FOREST_SINGLE))
    return PSATTN_ERR_INVALID_ARG;
  const Requests q{tokens, offsets, num_req, chunk};
  try {
    Grouping gr;
    group_requests(q, flags, &gr);
    const int32_t ng = (int32_t)gr.plen.size();
    *num_groups = ng;
    if (saved_tokens) *saved_tokens = gr.saved;
    if (ng > cap) return PSATTN_ERR_NOMEM;
    for (int32_t v = 0; v < ng; ++v) {
      group_parent[v] = gr.gpar[v];
      prefix_len[v] = gr.plen[v];
    }
    for (int32_t r = 0; r < num_req; ++r) {
      group_of_req[r] = gr.gor[r];
      suffix_len[r] = gr.slen[r];
    }
    return PSATTN_OK;
  } catch (...) {
    return PSATTN_ERR_NOMEM;
  }
}

int psattn_cht_group(const int32_t* tokens, const int64_t* offsets, int32_t num_req,
                     int32_t chunk, int32_t max_batch, int32_t max_new_chunks, uint32_t flags,
                     int32_t* batch_of_req, int32_t* order, int32_t* num_batches,
                     int32_t* batch_group_offset, int32_t* group_of_req, int32_t* group_parent,
                     int32_t* prefix_len, int32_t* suffix_len, int32_t cap, int32_t* num_groups,
                     int64_t* saved_tokens) {
  if (!valid(tokens, offsets, num_req, chunk) || !num_batches || !num_groups ||
      max_batch < 1 || max_new_chunks < 0 || cap < 0 || !batch_group_offset ||
      (num_req > 0 && (!batch_of_req || !order || !group_of_req || !suffix_len)) ||
      (cap > 0 && (!group_parent || !prefix_len)) || (flags & ~PSATTN_FOREST_SINGLE))
    return PSATTN_ERR_INVALID_ARG;
  const Requests q{tokens, offsets, num_req, chunk};
  try {
    const auto h = cumulative_hashes(q);
    int32_t nb = 0;
    cht_batches(q, h, max_batch, max_new_chunks, batch_of_req, order, &nb);
    *num_batches = nb;
    // each batch's requests in increasing id order
    std::vector<std::vector<int32_t>> members((size_t)nb);
    for (int32_t r = 0; r < num_req; ++r) members[batch_of_req[r]].push_back(r);
    std::vector<int32_t> gpar_all, plen_all;
    int64_t saved = 0;
    batch_group_offset[0] = 0;
    std::vector<int32_t> btok;
    std::vector<int64_t> boff;
    for (int32_t b = 0; b < nb; ++b) {
      // the batch's token ids back to back
      const std::vector<int32_t>& m = members[b];
      btok.clear();
      boff.assign(1, 0);
      for (int32_t r : m) {
        btok.insert(btok.end(), tokens + offsets[r], tokens + offsets[r + 1]);
        boff.push_back((int64_t)btok.size());
      }
      if (btok.empty()) btok.push_back(0);
      const Requests sub{btok.data(), boff.data(), (int32_t)m.size(), chunk};
      Grouping gr;
      group_requests(sub, flags, &gr);
      const int32_t base = (int32_t)plen_all.size();
      for (size_t v = 0; v < gr.plen.size(); ++v) {
        gpar_all.push_back(gr.gpar[v] >= 0 ? base + gr.gpar[v] : -1);
        plen_all.push_back(gr.plen[v]);
      }
      for (size_t i = 0; i < m.size(); ++i) {
        group_of_req[m[i]] = gr.gor[i] >= 0 ? base + gr.gor[i] : -1;
        suffix_len[m[i]] = gr.slen[i];
      }
      saved += gr.saved;
      batch_group_offset[b + 1] = (int32_t)plen_all.size();
    }
    const int32_t ng = (int32_t)plen_all.size();
    *num_groups = ng;
    if (saved_tokens) *saved_tokens = saved;
    if (ng > cap) return PSATTN_ERR_NOMEM;
    for (int32_t v = 0; v < ng; ++v) {
      group_parent[v] = gpar_all[v];
      prefix_len[v] = plen_all[v];
    }
    return PSATTN_OK;
  } catch (...) {
    return PSATTN_ERR_NOMEM;
  }
}

int psattn_cht_batches(const int32_t* tokens, const int64_t* offsets, int32_t num_req,
                       int32_t chunk, int32_t max_batch, int32_t max_new_chunks,
                       int32_t* batch_of_req, int32_t* order, int32_t* num_batches) {
  if (!valid(tokens, offsets, num_req, chunk) || !num_batches || max_batch < 1 ||
      max_new_chunks < 0 || (num_req > 0 && (!batch_of_req || !order)))
    return PSATTN_ERR_INVALID_ARG;
  const Requests q{tokens, offsets, num_req, chunk};
  try {
    const auto h = cumulative_hashes(q);
    cht_batches(q, h, max_batch, max_new_chunks, batch_of_req, order, num_batches);
    return PSATTN_OK;
  } catch (...) {
    return PSATTN_ERR_NOMEM;
  }
}

}  // extern "C"
