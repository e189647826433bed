// Prefill chunks as decode rows with shared causal levels
// (include/psattn_chunked.h states the expansion).  Host only.
#include "psattn.h"
#include "psattn_chunked.h"

#include <cstdint>
#include <cstring>
#include <vector>

namespace {

struct Layout {
  int64_t A = 0;      // tokens of the shared level of the earlier suffix (whole blocks)
  int64_t a = 0;      // suffix tokens before the chunk
  int32_t levels = 0; // causal levels
};

Layout layout_of(int32_t S, int32_t n, int32_t B, int32_t W) {
  Layout L;
  if (n < 2) return L;
  L.a = (int64_t)S - n;
  L.A = (L.a / B) * B;
  if (W > 0) {
    const int64_t e_last = L.a - L.A + n - 1;  // last query's position past A (inclusive)
    L.levels = (int32_t)((e_last + 1) / W);
  }
  return L;
}

// ragged: the request's whole suffix is one level whose member i sees its
// first a + i + 1 tokens (out_leaf_len; a = suffix tokens before the chunk),
// instead of a level for the earlier suffix, level_tokens-sized causal levels
// and own suffixes.
int expand(const psattn_shape* shape, const int32_t* block_table, const int32_t* group_of_req,
           const int32_t* group_parent, const int32_t* prefix_len, const int32_t* suffix_len,
           const int32_t* q_len, int32_t level_tokens, bool ragged, psattn_shape* out_shape,
           int32_t* out_block_table, int32_t* out_group_of_req, int32_t* out_group_parent,
           int32_t* out_prefix_len, int32_t* out_suffix_len, int32_t* out_leaf_len,
           int32_t cap_rows, int32_t cap_groups) {
  if (!shape || !out_shape || cap_rows < 0 || cap_groups < 0) return PSATTN_ERR_INVALID_ARG;
  const int32_t R = shape->num_req, NG = shape->num_groups, B = shape->block_size;
  const int32_t maxb = shape->max_blocks_per_req;
  if (R < 0 || NG < 0 || B < 1 || (R > 0 && maxb < 1)) return PSATTN_ERR_INVALID_ARG;
  if ((R > 0 && (!block_table || !group_of_req || !suffix_len || !q_len)) ||
      (NG > 0 && !prefix_len))
    return PSATTN_ERR_INVALID_ARG;
  if (level_tokens < 0 || (level_tokens > 0 && level_tokens % B)) return PSATTN_ERR_INVALID_ARG;
  for (int32_t g = 0; g < NG; ++g)
    if (prefix_len[g] < 0 || (group_parent && (group_parent[g] < -1 || group_parent[g] >= NG)))
      return PSATTN_ERR_INVALID_ARG;
  int64_t rows = 0, groups = NG;
  for (int32_t r = 0; r < R; ++r) {
    const int32_t n = q_len[r], S = suffix_len[r];
    if (n < 1 || S < 0 || group_of_req[r] < -1 || group_of_req[r] >= NG ||
        (n >= 2 && n > S))
      return PSATTN_ERR_INVALID_ARG;
    const Layout L = layout_of(S, n, B, ragged ? 0 : level_tokens);
    rows += n;
    groups += ragged ? (n >= 2 ? 1 : 0) : (L.A > 0 ? 1 : 0) + L.levels;
  }
  if (rows > INT32_MAX || groups > INT32_MAX) return PSATTN_ERR_INVALID_ARG;
  *out_shape = *shape;
  out_shape->num_req = (int32_t)rows;
  out_shape->num_groups = (int32_t)groups;
  if (rows > cap_rows || groups > cap_groups) return PSATTN_ERR_NOMEM;
  if ((rows > 0 && (!out_block_table || !out_group_of_req || !out_suffix_len ||
                    (ragged && !out_leaf_len))) ||
      (groups > 0 && (!out_group_parent || !out_prefix_len)))
    return PSATTN_ERR_INVALID_ARG;

  for (int32_t g = 0; g < NG; ++g) {
    out_prefix_len[g] = prefix_len[g];
    out_group_parent[g] = group_parent ? group_parent[g] : -1;
  }
  int32_t ng = NG;
  int64_t k = 0;
  for (int32_t r = 0; r < R; ++r) {
    const int32_t n = q_len[r], S = suffix_len[r], W = ragged ? 0 : level_tokens;
    const int32_t* src = block_table + (size_t)r * maxb;
    const Layout L = layout_of(S, n, B, W);
    int32_t top = group_of_req[r];  // deepest level every query of r shares
    if (!ragged && L.A > 0) {
      out_prefix_len[ng] = (int32_t)L.A;
      out_group_parent[ng] = top;
      top = ng++;
    }
    int32_t causal = -1;  // the ragged level (ragged mode)
    if (ragged && n >= 2) {
      out_prefix_len[ng] = S;
      out_group_parent[ng] = top;
      causal = ng++;
    }
    const int32_t first_level = ng;
    for (int32_t j = 0; j < L.levels; ++j) {
      out_prefix_len[ng] = W;
      out_group_parent[ng] = j == 0 ? top : ng - 1;
      ++ng;
    }
    for (int32_t i = 0; i < n; ++i, ++k) {
      std::memcpy(out_block_table + (size_t)k * maxb, src, sizeof(int32_t) * (size_t)maxb);
      if (ragged) out_leaf_len[k] = -1;
      if (n < 2) {
        out_group_of_req[k] = group_of_req[r];
        out_suffix_len[k] = S;
        continue;
      }
      if (ragged) {
        out_group_of_req[k] = causal;
        out_suffix_len[k] = 0;
        out_leaf_len[k] = (int32_t)(L.a + i + 1);
        continue;
      }
      const int64_t e = L.a - L.A + i;  // position past A, inclusive
      const int32_t m = W > 0 ? (int32_t)((e + 1) / W) : 0;
      out_group_of_req[k] = m > 0 ? first_level + m - 1 : top;
      out_suffix_len[k] = (int32_t)(e + 1 - (int64_t)m * (W > 0 ? W : 0));
    }
  }
  return PSATTN_OK;
}

}  // namespace

extern "C" int psattn_chunked_expand(const psattn_shape* shape, const int32_t* block_table,
                                     const int32_t* group_of_req, const int32_t* group_parent,
                                     const int32_t* prefix_len, const int32_t* suffix_len,
                                     const int32_t* q_len, int32_t level_tokens,
                                     psattn_shape* out_shape, int32_t* out_block_table,
                                     int32_t* out_group_of_req, int32_t* out_group_parent,
                                     int32_t* out_prefix_len, int32_t* out_suffix_len,
                                     int32_t cap_rows, int32_t cap_groups) {
  return expand(shape, block_table, group_of_req, group_parent, prefix_len, suffix_len, q_len,
                level_tokens, false, out_shape, out_block_table, out_group_of_req,
                out_group_parent, out_prefix_len, out_suffix_len, nullptr, cap_rows, cap_groups);
}

extern "C" int psattn_chunked_expand_ragged(
    const psattn_shape* shape, const int32_t* block_table, const int32_t* group_of_req,
    const int32_t* group_parent, const int32_t* prefix_len, const int32_t* suffix_len,
    const int32_t* q_len, psattn_shape* out_shape, int32_t* out_block_table,
    int32_t* out_group_of_req, int32_t* out_group_parent, int32_t* out_prefix_len,
    int32_t* out_suffix_len, int32_t* out_leaf_len, int32_t cap_rows, int32_t cap_groups) {
  return expand(shape, block_table, group_of_req, group_parent, prefix_len, suffix_len, q_len, 0,
                true, out_shape, out_block_table, out_group_of_req, out_group_parent,
                out_prefix_len, out_suffix_len, out_leaf_len, cap_rows, cap_groups);
}
