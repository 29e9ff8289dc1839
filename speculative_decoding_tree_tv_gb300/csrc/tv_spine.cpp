// tv_build_spine_tree: GOOSE's anisotropic spine tree, built on the host from
// the drafter's candidate lists (GOOSE §2A: a deep chain of context-matched
// tokens, branches of transition tokens forking off every spine node, wide
// near the root and narrower deeper down; §2B Proposition 2: the branch
// allocation falls linearly with depth; §2C: the spine ratio follows an
// exponential moving average of the observed acceptance of the spine).
//
// The tree goes to tv_tree_build / tv_attn_verify / tv_accept_* as it is:
// parent[] in breadth-first order with the spine child first at every depth,
// which is also the order in which the greedy walk prefers the spine.
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "treeverify.h"
#include "tv_nvtx.h"

namespace {

// Usable branch candidates of one spine position: best first up to the first
// -1, without the spine's own token there and without repeats.
int usable_candidates(const int32_t* row, int K, int skip, int32_t* out) {
  int n = 0;
  for (int k = 0; k < K && row[k] >= 0; ++k) {
    const int32_t t = row[k];
    if (t == skip) continue;
    bool seen = false;
    for (int i = 0; i < n && !seen; ++i) seen = (out[i] == t);
    if (!seen) out[n++] = t;
  }
  return n;
}

}  // namespace

extern "C" tv_status tv_build_spine_tree(const int32_t* spine_tokens, int S,
                                         const int32_t* branch_tokens, int Sb, int K,
                                         int root_token, int budget, float spine_ratio,
                                         int32_t* parent, int32_t* tokens, int32_t* n_nodes) {
  TV_NVTX_RANGE("tv_build_spine_tree");
  if (S < 0 || Sb < 0 || K < 0 || budget < 1 || !parent || !tokens || !n_nodes)
    return TV_ERR_INVALID_ARG;
  if (!(spine_ratio >= 0.0f && spine_ratio <= 1.0f)) return TV_ERR_INVALID_ARG;
  if ((S > 0 && !spine_tokens) || (Sb > 0 && K > 0 && !branch_tokens)) return TV_ERR_INVALID_ARG;
  // spine length, then branch points: spine nodes 0 .. m-1
  const int spine_len = std::min(S, (int)std::llround((double)spine_ratio * (budget - 1)));
  const int rest = budget - 1 - spine_len;
  const int points = std::min(spine_len + 1, Sb);
  std::vector<int32_t> cand((size_t)std::max(points, 0) * std::max(K, 1));
  std::vector<int> avail(std::max(points, 0)), width(std::max(points, 0), 0);
  for (int j = 0; j < points; ++j) {
    const int skip = (j < spine_len) ? spine_tokens[j] : -1;
    avail[j] = usable_candidates(branch_tokens + (size_t)j * K, K, skip, cand.data() + (size_t)j * K);
  }
  // widths proportional to (points - j): the integer parts, then the leftover
  // one by one from the root; a position short of candidates passes the
  // rest on to the next one
  if (points > 0 && rest > 0) {
    const long long tri = (long long)points * (points + 1) / 2;
    long long assigned = 0;
    for (int j = 0; j < points; ++j) {
      width[j] = (int)(rest * (long long)(points - j) / tri);
      assigned += width[j];
    }
    for (int j = 0; assigned < rest; j = (j + 1) % points, ++assigned) ++width[j];
    int spill = 0;
    for (int j = 0; j < points; ++j) {
      const int want = width[j] + spill;
      width[j] = std::min(want, avail[j]);
      spill = want - width[j];
    }
  }
  // breadth-first: level t holds spine node t (t <= spine_len), then the
  // branches of spine node t - 1
  int n = 0;
  parent[n] = -1;
  tokens[n++] = root_token;
  int above = 0;  // spine node t - 1
  const int levels = std::max(spine_len, points);
  for (int t = 1; t <= levels; ++t) {
    const int from = above;
    if (t <= spine_len) {
      parent[n] = from;
      tokens[n] = spine_tokens[t - 1];
      above = n++;
    }
    if (t <= points)
      for (int k = 0; k < width[t - 1]; ++k) {
        parent[n] = from;
        tokens[n++] = cand[(size_t)(t - 1) * K + k];
      }
  }
  *n_nodes = n;
  return TV_OK;
}

extern "C" float tv_spine_ratio_update(float ratio, float observed_accept_rate, float beta) {
  const float r = (1.0f - beta) * ratio + beta * observed_accept_rate;
  return std::min(1.0f, std::max(0.0f, r));
}
