// Token batches of an offline batch: group scheduling over three queues,
// R_group reordering and memory-centric batching, after BatchLLM section 4.3
// (include/psattn_sched.h states the model).  Host only.
#include "psattn.h"
#include "psattn_sched.h"

#include <algorithm>
#include <cstdint>
#include <vector>

namespace {

struct SchedGroup {
  int64_t prefix = 0;          // common-prefix tokens
  int64_t key = 0;             // L_prefix + sum L_distinct (R_group = 1 / key)
  int32_t first = 0;           // smallest member id: the input order
  int32_t id = 0;              // g, or num_groups + r for an ungrouped request
  std::vector<int32_t> members;  // ascending ids
};

struct Req {
  int64_t prompt_left = 0;  // distinct tokens not yet processed
  int64_t out_left = 0;     // output tokens not yet produced
  int64_t own = 0;          // resident tokens of the request (prompt + output)
  int32_t sg = -1;          // scheduling group (index into the priority order)
  int32_t eligible_at = -1; // first iteration its distinct chunks may run
  int32_t decode_at = -1;   // first iteration it may decode (-1: not yet known)
  bool done = false;
};

constexpr int64_t kMaxTotalTokens = int64_t(1) << 29;

}  // namespace

extern "C" int psattn_token_batches(const int32_t* group_prefix, int32_t num_groups,
                                    const int32_t* group_of_req, const int32_t* distinct_len,
                                    const int32_t* decode_len, int32_t num_req,
                                    const psattn_sched_params* prm, int32_t* group_order,
                                    int32_t* num_sched_groups, int32_t* iter_tokens,
                                    int64_t* iter_mem, int32_t cap, int32_t* num_iters) {
  if (num_groups < 0 || num_req < 0 || cap < 0 || !prm || !group_order || !num_sched_groups ||
      !num_iters || (cap > 0 && (!iter_tokens || !iter_mem)) ||
      (num_groups > 0 && !group_prefix) ||
      (num_req > 0 && (!group_of_req || !distinct_len || !decode_len)))
    return PSATTN_ERR_INVALID_ARG;
  if (prm->n_chunk < 1 || prm->max_requests < 0) return PSATTN_ERR_INVALID_ARG;
  for (int32_t g = 0; g < num_groups; ++g)
    if (group_prefix[g] < 0) return PSATTN_ERR_INVALID_ARG;
  for (int32_t r = 0; r < num_req; ++r)
    if (group_of_req[r] < -1 || group_of_req[r] >= num_groups || distinct_len[r] < 0 ||
        decode_len[r] < 1)
      return PSATTN_ERR_INVALID_ARG;

  // ---- scheduling groups and their priority order
  std::vector<SchedGroup> sg;
  std::vector<int32_t> sg_of_group((size_t)num_groups, -1);
  for (int32_t r = 0; r < num_req; ++r) {
    const int32_t g = group_of_req[r];
    int32_t s;
    if (g < 0) {
      s = (int32_t)sg.size();
      sg.emplace_back();
      sg[s].id = num_groups + r;
      sg[s].first = r;
    } else {
      s = sg_of_group[g];
      if (s < 0) {
        s = sg_of_group[g] = (int32_t)sg.size();
        sg.emplace_back();
        sg[s].id = g;
        sg[s].first = r;
        sg[s].prefix = group_prefix[g];
        sg[s].key = group_prefix[g];
      }
    }
    sg[s].members.push_back(r);
    sg[s].key += distinct_len[r];
  }
  // sg is already in input order (first member ascending)
  std::vector<int32_t> order(sg.size());
  for (size_t i = 0; i < sg.size(); ++i) order[i] = (int32_t)i;
  if (prm->flags & PSATTN_SCHED_REORDER)
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return sg[a].key < sg[b].key; });
  for (size_t i = 0; i < order.size(); ++i) group_order[i] = sg[order[i]].id;
  *num_sched_groups = (int32_t)order.size();

  std::vector<Req> rq((size_t)num_req);
  std::vector<int32_t> rank_of_sg(sg.size());
  for (size_t i = 0; i < order.size(); ++i) rank_of_sg[order[i]] = (int32_t)i;
  std::vector<int32_t> left_in_sg(sg.size());
  for (size_t s = 0; s < sg.size(); ++s) {
    left_in_sg[s] = (int32_t)sg[s].members.size();
    for (int32_t r : sg[s].members) {
      rq[r].prompt_left = distinct_len[r];
      rq[r].out_left = decode_len[r];
      rq[r].sg = rank_of_sg[s];
    }
  }
  // by priority rank: prefix tokens processed so far, members in rank order
  const int32_t NS = (int32_t)order.size();
  std::vector<int64_t> pre_done((size_t)NS, 0);
  std::vector<int32_t> dq;  // distinct queue: requests by (rank, id)
  for (int32_t k = 0; k < NS; ++k)
    for (int32_t r : sg[order[k]].members) dq.push_back(r);
  // decode queue entries: (first iteration, request id), kept sorted
  std::vector<std::pair<int32_t, int32_t>> decq;

  int64_t total = 0;
  for (int32_t k = 0; k < NS; ++k) {
    total += sg[order[k]].prefix;
    for (int32_t r : sg[order[k]].members) total += (int64_t)distinct_len[r] + decode_len[r];
  }
  // iterations are counted in int32 (the tables and the decode queue's start
  // iterations): a batch must keep its total tokens below kMaxTotalTokens
  if (total > kMaxTotalTokens) return PSATTN_ERR_INVALID_ARG;
  const int64_t guard = 2 * total + 2 * (int64_t)NS + 4;

  int64_t resident = 0;
  int32_t cur = 0;         // rank of the group whose prefix is being served
  size_t dq_head = 0;      // first distinct-queue entry that may still have work
  int32_t finished = 0;
  int64_t it = 0;
  std::vector<int32_t> fin;
  while (finished < num_req) {
    // every iteration but (rarely) one in two processes a token: never reached
    if (it >= guard) return PSATTN_ERR_INVALID_ARG;
    const int32_t t = (int32_t)it;
    int64_t budget = prm->n_chunk;
    int32_t nreq = 0, ndec = 0;
    int64_t ndis = 0, npre = 0;
    const bool capped = prm->max_requests > 0;
    auto room = [&]() { return !capped || nreq < prm->max_requests; };
    fin.clear();
    // (1) decode tokens, in queue order
    std::sort(decq.begin(), decq.end());
    for (const auto& e : decq) {
      if (budget == 0 || !room()) break;
      if (e.first > t) break;  // sorted: later entries start later too
      Req& q = rq[e.second];
      --budget;
      ++nreq;
      ++ndec;
      ++resident;
      ++q.own;
      if (--q.out_left == 0) fin.push_back(e.second);
    }
    if (!fin.empty()) {
      std::vector<char> gone((size_t)num_req, 0);
      for (int32_t r : fin) gone[r] = 1;
      decq.erase(std::remove_if(decq.begin(), decq.end(),
                                [&](const std::pair<int32_t, int32_t>& e) { return gone[e.second] != 0; }),
                 decq.end());
    }
    // (2) distinct-prompt chunks, (3) common-prefix chunks; memory gate
    bool prefill_open = true;
    auto fits = [&](int64_t c) {
      const bool empty = (nreq == 0);
      return empty || prm->m_threshold < 0 || resident + c <= prm->m_threshold;
    };
    while (dq_head < dq.size() && rq[dq[dq_head]].eligible_at >= 0 && rq[dq[dq_head]].prompt_left == 0 &&
           rq[dq[dq_head]].decode_at >= 0)
      ++dq_head;
    for (size_t i = dq_head; i < dq.size() && prefill_open; ++i) {
      if (budget == 0 || !room()) break;
      const int32_t r = dq[i];
      Req& q = rq[r];
      if (q.eligible_at < 0 || q.eligible_at > t) break;  // rank order: later groups are later
      if (q.prompt_left == 0) continue;
      const int64_t c = std::min<int64_t>(q.prompt_left, budget);
      if (!fits(c)) {
        prefill_open = false;
        break;
      }
      budget -= c;
      ++nreq;
      ndis += c;
      resident += c;
      q.own += c;
      q.prompt_left -= c;
      if (q.prompt_left == 0) {
        q.decode_at = t + 1;
        decq.emplace_back(t + 1, r);
      }
    }
    while (prefill_open && cur < NS) {
      const SchedGroup& G = sg[order[cur]];
      const int64_t rem = G.prefix - pre_done[cur];
      if (rem > 0) {
        if (budget == 0 || !room()) break;
        const int64_t c = std::min<int64_t>(rem, budget);
        if (!fits(c)) {
          prefill_open = false;
          break;
        }
        budget -= c;
        ++nreq;
        npre += c;
        resident += c;
        pre_done[cur] += c;
        if (pre_done[cur] < G.prefix) break;  // budget spent inside this prefix
      }
      // prefix complete (or none): members may start next iteration
      for (int32_t r : G.members) {
        rq[r].eligible_at = t + 1;
        if (rq[r].prompt_left == 0) {  // no distinct prompt: decodes next
          rq[r].decode_at = t + 1;
          decq.emplace_back(t + 1, r);
        }
      }
      ++cur;
    }
    if (it < cap) {
      iter_tokens[4 * it] = ndec;
      iter_tokens[4 * it + 1] = (int32_t)ndis;
      iter_tokens[4 * it + 2] = (int32_t)npre;
      iter_tokens[4 * it + 3] = nreq;
      iter_mem[it] = resident;
    }
    // free what finished in this iteration
    for (int32_t r : fin) {
      Req& q = rq[r];
      q.done = true;
      resident -= q.own;
      q.own = 0;
      ++finished;
      const int32_t s = order[q.sg];
      if (--left_in_sg[s] == 0) resident -= sg[s].prefix;
    }
    ++it;
  }
  *num_iters = (int32_t)std::min<int64_t>(it, INT32_MAX);
  return it > cap ? PSATTN_ERR_NOMEM : PSATTN_OK;
}
