// Plain CPU oracle for tree-based speculative verification.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
// statement of what the GPU library computes.  Only the test suite, the
// smoke check and the bench's CPU-baseline leg may build, load or call it;
// the GPU path never does, and the two share no code.
//
// Everything is written as the plain definition: explicit ancestor sets
// obtained by walking parent links, fp64 arithmetic, full sorts, brute force.
// No blocking, fusion or reordering beyond what the definition states.  Loops
// over independent rows (attention rows, argmax rows) may run on several
// threads (OpenMP); each row is still computed start to finish by one thread
// in the order written, so the results do not depend on the thread count.
//
// Sources (page title, section):
//   [OPT]   "OPT-Tree: Speculative Decoding with Adaptive Draft Tree Structure",
//           §2 Preliminaries (tree attention mask; longest matching branch
//           under greedy sampling) and §3 (node scores, monotone path scores).
//   [SPEC]  "Speculative Decoding" concept page, "The protocol" steps 1-4
//           (accept with min(1, p/q), residual (p-q)+ resampling, lossless).
//   [TALON] "TALON: confidence-aware speculative decoding with adaptive token
//           trees", §5.1 (token budget B), §5.2.1 (confidence-gated
//           expansion: candidate pool, path score s(c) = prod p_d, anchor,
//           alpha gate, budget truncation), §5.2.2 (root Top-K).
//   [GOOSE] "GOOSE: Anisotropic Speculation Trees", §2C (one forward pass
//           verifies the whole tree; greedy walk).
//   The commit of the accepted branch into the cache follows [SPEC] step 4
//   and [OPT] §2 (see or_commit_path); the expected acceptance length of a
//   tree follows [OPT] §3 (see or_expected_accept), and so do OPT-Tree's
//   greedy expansion and subtree selection (or_expand_topn, or_select_topn).
//   [PHILOX] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
//           1, 2, 3" (SC'11): the Philox4x64-10 counter-based generator.
//
// Readings where the pages are silent (each also listed in the design notes):
//   * node 0 is the token right after the cached prefix and is always
//     accepted; logits row v is the target distribution over v's children;
//     accept_len counts accepted draft tokens (node 0 excluded).
//   * argmax ties go to the lowest token index; "longest branch" ties go to
//     the lowest node index.
//   * tree K/V of node j lives at cache slot kv_len[b] + j; GQA kv head of
//     query head h is h / (Hq / Hkv); scale 0 means 1/sqrt(D).
//   * stochastic acceptance on a tree tests children in ascending index;
//     after a rejection the target becomes norm((r - q)+) with the same q.
//
// Decisions taken on floating point (accept tests, sampling, gating) also
// report a margin: the distance of the decision quantity from its threshold,
// so tests can tell a genuine disagreement from a rounding-order tie.

#include <stdint.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

const int ST_OK = 0;
const int ST_INVALID_ARG = 1;
const int ST_INVALID_TREE = 2;
const int ST_INVALID_TOKEN = 6;

double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

// A tree is valid when node 0 is the only root and every other node's parent
// comes earlier (a topological numbering).
bool tree_is_valid(const int32_t* parent, int N) {
  if (N < 1 || parent[0] != -1) return false;
  for (int i = 1; i < N; ++i)
    if (parent[i] < 0 || parent[i] >= i) return false;
  return true;
}

// Explicit ancestor-or-self set of node i, from i up to the root.
std::vector<int> ancestors_of(const int32_t* parent, int i) {
  std::vector<int> a;
  for (int x = i; x >= 0; x = parent[x]) a.push_back(x);
  return a;
}

int depth_of(const int32_t* parent, int i) {
  int d = 0;
  for (int x = i; parent[x] >= 0; x = parent[x]) ++d;
  return d;
}

// ---------------------------------------------------------------------------
// Philox4x64-10 [PHILOX]: ten rounds of two 64x64->128 multiplies with the
// published multipliers, key bumped by the published Weyl constants.
// ---------------------------------------------------------------------------
void philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
  const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
  uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { k0 += W0; k1 += W1; }
    unsigned __int128 p0 = (unsigned __int128)M0 * x0;
    unsigned __int128 p1 = (unsigned __int128)M1 * x2;
    uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    x0 = hi1 ^ x1 ^ k0;
    x1 = lo1;
    x2 = hi0 ^ x3 ^ k1;
    x3 = lo0;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// The single random word used by a decision: counter (offset, sequence,
// node, purpose<<32 | ordinal), key (seed, 0); first output word.
const uint64_t PURPOSE_ACCEPT = 0;  // accept test of the ordinal-th child
const uint64_t PURPOSE_SAMPLE = 1;  // the final draw (residual or bonus)

uint64_t draw_word(uint64_t seed, uint64_t offset, int b, int node, uint64_t purpose,
                   uint32_t ordinal) {
  uint64_t ctr[4] = {offset, (uint64_t)b, (uint64_t)node, (purpose << 32) | ordinal};
  uint64_t key[2] = {seed, 0};
  uint64_t out[4];
  philox4x64_10(ctr, key, out);
  return out[0];
}

// 53-bit uniform in [0,1): the top 53 bits of the word, scaled by 2^-53.
double uniform53(uint64_t w) { return (double)(w >> 11) * (1.0 / 9007199254740992.0); }

// Natural-log partition of a logits row at temperature T: log sum exp(l/T).
double row_logsumexp(const float* row, int V, double T) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) m = std::max(m, (double)row[v] / T);
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp((double)row[v] / T - m);
  return m + log(s);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Tree encoding [OPT §2, §3]: the tree attention mask lets node i see exactly
// its ancestors and itself.  depth[i] = number of edges from the root;
// anc_mask[i] has bit j set iff j is on the path root..i.
// ---------------------------------------------------------------------------
int or_tree_build(const int32_t* parent, int B, int N, int32_t* depth, uint64_t* anc_mask,
                  int32_t* status) {
  if (B < 0 || N < 1) return ST_INVALID_ARG;
  const int W = (N + 63) / 64;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (size_t)b * N;
    int32_t* dep = depth + (size_t)b * N;
    uint64_t* anc = anc_mask + (size_t)b * N * W;
    memset(anc, 0, sizeof(uint64_t) * N * W);
    if (!tree_is_valid(par, N)) {
      status[b] = ST_INVALID_TREE;
      for (int i = 0; i < N; ++i) dep[i] = -1;
      continue;
    }
    status[b] = ST_OK;
    for (int i = 0; i < N; ++i) {
      dep[i] = depth_of(par, i);
      for (int a : ancestors_of(par, i)) anc[(size_t)i * W + a / 64] |= 1ULL << (a % 64);
    }
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// Tree-verify attention [OPT §2; GOOSE §2C; SPEC "Why it is a win"]: for the
// query of node i and head h, attend over the cached prefix 0..L_b-1 and the
// tree slots L_b + j of the ancestors-or-self j of i.  The kv head of query
// head h is h / (Hq/Hkv).  Computed for the requested rows only:
// rows[3r..3r+2] = (b, i, h).  out[r*D + d] gets the output, lse[r] the
// natural-log normaliser log sum_j exp(scale * q.k_j).
// ---------------------------------------------------------------------------
// Threads used by the loops over independent rows (OpenMP); n <= 0 keeps
// the runtime's default (one per core).
void or_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int or_attn_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                 const int32_t* kv_len, const int32_t* parent, int B, int N, int Hq,
                 int Hkv, int D, int Lcap, double scale, const int32_t* rows, int n_rows,
                 double* out, double* lse) {
  if (Hkv < 1 || Hq % Hkv != 0 || N < 1 || D < 1) return ST_INVALID_ARG;
  if (scale == 0.0) scale = 1.0 / sqrt((double)D);
  const int G = Hq / Hkv;
  for (int r = 0; r < n_rows; ++r) {
    const int b = rows[3 * r], i = rows[3 * r + 1], h = rows[3 * r + 2];
    if (b < 0 || b >= B || i < 0 || i >= N || h < 0 || h >= Hq) return ST_INVALID_ARG;
    if (!tree_is_valid(parent + (size_t)b * N, N)) return ST_INVALID_TREE;
    if (kv_len[b] < 0 || kv_len[b] + N > Lcap) return ST_INVALID_ARG;
  }
  // Rows are independent: each is computed by one thread, start to finish.
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < n_rows; ++r) {
    const int b = rows[3 * r], i = rows[3 * r + 1], h = rows[3 * r + 2];
    const int32_t* par = parent + (size_t)b * N;
    const int L = kv_len[b];
    const int kvh = h / G;

    std::vector<int> keys;  // cache positions visible to (b, i)
    for (int j = 0; j < L; ++j) keys.push_back(j);
    std::vector<int> anc = ancestors_of(par, i);
    std::sort(anc.begin(), anc.end());
    for (int a : anc) keys.push_back(L + a);

    const uint16_t* qrow = q + (((size_t)b * N + i) * Hq + h) * D;
    const uint16_t* kbase = k + ((size_t)b * Hkv + kvh) * (size_t)Lcap * D;
    const uint16_t* vbase = v + ((size_t)b * Hkv + kvh) * (size_t)Lcap * D;

    std::vector<double> s(keys.size());
    double m = -INFINITY;
    for (size_t t = 0; t < keys.size(); ++t) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += bf16_to_double(qrow[d]) * bf16_to_double(kbase[(size_t)keys[t] * D + d]);
      s[t] = dot * scale;
      m = std::max(m, s[t]);
    }
    // softmax weights w_t = exp(s_t - max), the normaliser their sum
    std::vector<double> w(keys.size());
    double denom = 0.0;
    for (size_t t = 0; t < keys.size(); ++t) {
      w[t] = exp(s[t] - m);
      denom += w[t];
    }
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
      for (size_t t = 0; t < keys.size(); ++t)
        acc += w[t] * bf16_to_double(vbase[(size_t)keys[t] * D + d]);
      out[(size_t)r * D + d] = acc / denom;
    }
    lse[r] = m + log(denom);
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// Greedy acceptance [OPT §2 "longest branch matching the target's
// highest-probability sequence"; GOOSE §2C greedy walk].
//   argmax[i]  = first index of the largest logit in row i;
//   a node is valid iff every edge p->c on its root path has
//              tokens[c] == argmax[p]   (checked by brute force per node);
//   end        = deepest valid node, ties to the lowest index;
//   accept_len = depth[end]; path = root..end padded with -1;
//   bonus      = argmax[end] (the target's own next token).
// ---------------------------------------------------------------------------
int or_accept_greedy(const float* logits, const int32_t* tokens, const int32_t* parent, int B,
                     int N, int V, int32_t* argmax, int32_t* accept_len, int32_t* end_node,
                     int32_t* path, int32_t* bonus, int32_t* status) {
  if (B < 0 || N < 1 || V < 1) return ST_INVALID_ARG;
  // argmax of every node row (rows are independent: one thread each)
#pragma omp parallel for schedule(static)
  for (long long row_i = 0; row_i < (long long)B * N; ++row_i) {
    const float* row = logits + (size_t)row_i * V;
    int best = 0;
    for (int t = 1; t < V; ++t)
      if (row[t] > row[best]) best = t;
    argmax[row_i] = best;
  }
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (size_t)b * N;
    const int32_t* tok = tokens + (size_t)b * N;
    const int32_t* am = argmax + (size_t)b * N;
    for (int i = 0; i < N; ++i) path[(size_t)b * N + i] = -1;
    accept_len[b] = end_node[b] = bonus[b] = -1;
    if (!tree_is_valid(par, N)) { status[b] = ST_INVALID_TREE; continue; }
    bool tok_ok = true;
    for (int i = 1; i < N; ++i)
      if (tok[i] < 0 || tok[i] >= V) tok_ok = false;
    if (!tok_ok) { status[b] = ST_INVALID_TOKEN; continue; }
    status[b] = ST_OK;

    int end = 0, end_depth = 0;
    for (int e = 0; e < N; ++e) {
      bool valid = true;
      for (int c = e; par[c] >= 0; c = par[c])
        if (tok[c] != am[par[c]]) valid = false;
      const int de = depth_of(par, e);
      if (valid && de > end_depth) { end = e; end_depth = de; }
    }
    std::vector<int> anc = ancestors_of(par, end);  // end .. root
    for (size_t t = 0; t < anc.size(); ++t) path[(size_t)b * N + (anc.size() - 1 - t)] = anc[t];
    accept_len[b] = end_depth;
    end_node[b] = end;
    bonus[b] = am[end];
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// Stochastic acceptance [SPEC "The protocol", step 3 and the lossless
// remark], extended to a tree: start at node 0 with target r = p_0.  At node
// v, test its children c (ascending index, draft token x = tokens[c]):
// accept with probability min(1, r(x)/q_v(x)) -- draw u, accept iff
// u < r(x)/q_v(x), and always when q_v(x) = 0.  On acceptance descend to c
// (r := p_c).  On rejection r := norm((r - q_v)+) (unchanged if that mass is
// not positive).  If every child is rejected, draw the output token from r;
// if v has no children, draw the bonus token from p_v.  p_v, q_v are
// softmax(logits/T) of row v.
//
// Random words: Philox4x64-10 keyed by (seed, 0), counter (offset, b, v,
// purpose<<32 | ordinal), each turned into a 53-bit uniform u.  Accept
// tests compare u with the fp64 ratio.  The final draw walks the fp64
// probabilities in ascending token order: the token is the smallest k whose
// cumulative mass exceeds u * (total mass); if rounding leaves none, the last
// token with positive mass.
//
// margin_accept[b] = smallest |u - ratio| / ratio over tree b's accept tests;
// margin_path[b, d] = the same over the accept tests made at the walk's node
// of depth d (INFINITY where none was made), so a comparison can locate the
// first decision that sits near its threshold;
// margin_draw[b] = distance of u * total from the nearest cumulative boundary
// of its final draw, divided by total; draw_alt[b] = the token a draw would
// give on the other side of that boundary (the previous or next token with
// positive mass; -1 if there is none).
// ---------------------------------------------------------------------------
int or_accept_sample(const float* p_logits, const float* q_logits, const int32_t* tokens,
                     const int32_t* parent, int B, int N, int V, float temperature,
                     uint64_t seed, uint64_t offset, int32_t* accept_len, int32_t* end_node,
                     int32_t* path, int32_t* out_token, int32_t* status, double* margin_accept,
                     double* margin_path, double* margin_draw, int32_t* draw_alt) {
  if (B < 0 || N < 1 || V < 1 || !(temperature > 0.0f)) return ST_INVALID_ARG;
  const double T = (double)temperature;
  std::vector<double> r(V), q(V);
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (size_t)b * N;
    const int32_t* tok = tokens + (size_t)b * N;
    for (int i = 0; i < N; ++i) {
      path[(size_t)b * N + i] = -1;
      margin_path[(size_t)b * N + i] = INFINITY;
    }
    accept_len[b] = end_node[b] = out_token[b] = draw_alt[b] = -1;
    margin_accept[b] = margin_draw[b] = INFINITY;
    if (!tree_is_valid(par, N)) { status[b] = ST_INVALID_TREE; continue; }
    bool tok_ok = true;
    for (int i = 1; i < N; ++i)
      if (tok[i] < 0 || tok[i] >= V) tok_ok = false;
    if (!tok_ok) { status[b] = ST_INVALID_TOKEN; continue; }
    status[b] = ST_OK;

    int node = 0, node_depth = 0;
    int out = -1;
    for (;;) {
      const float* prow = p_logits + ((size_t)b * N + node) * V;
      const float* qrow = q_logits + ((size_t)b * N + node) * V;
      const double lp = row_logsumexp(prow, V, T);
      const double lq = row_logsumexp(qrow, V, T);
      for (int t = 0; t < V; ++t) {
        r[t] = exp((double)prow[t] / T - lp);
        q[t] = exp((double)qrow[t] / T - lq);
      }
      std::vector<int> kids;
      for (int c = node + 1; c < N; ++c)
        if (par[c] == node) kids.push_back(c);

      int accepted = -1;
      for (size_t o = 0; o < kids.size(); ++o) {
        const int x = tok[kids[o]];
        const double u = uniform53(draw_word(seed, offset, b, node, PURPOSE_ACCEPT, (uint32_t)o));
        bool acc;
        if (q[x] == 0.0) {
          acc = true;
        } else {
          const double ratio = r[x] / q[x];
          acc = u < ratio;
          if (ratio > 0.0) {
            const double mg = fabs(u - ratio) / ratio;
            margin_accept[b] = std::min(margin_accept[b], mg);
            double& md = margin_path[(size_t)b * N + node_depth];
            md = std::min(md, mg);
          }
        }
        if (acc) { accepted = kids[o]; break; }
        double z = 0.0;
        for (int t = 0; t < V; ++t) z += std::max(r[t] - q[t], 0.0);
        if (z > 0.0)
          for (int t = 0; t < V; ++t) r[t] = std::max(r[t] - q[t], 0.0) / z;
      }
      if (accepted >= 0) {
        node = accepted;
        ++node_depth;
        continue;
      }

      // Final draw from r (the residual, or p_node at a leaf).
      const double u = uniform53(draw_word(seed, offset, b, node, PURPOSE_SAMPLE, 0));
      double total = 0.0;
      for (int t = 0; t < V; ++t) total += r[t];
      const double target = u * total;
      double cum = 0.0;
      int last_pos = -1;
      bool lower_closer = false;  // the nearest boundary lies below the drawn token
      for (int t = 0; t < V; ++t) {
        const double rt = r[t];
        if (rt > 0.0) last_pos = t;
        const double before = cum;
        cum += rt;
        if (out < 0 && cum > target) {
          out = t;
          margin_draw[b] = std::min(cum - target, target - before) / total;
          lower_closer = (target - before) <= (cum - target);
        }
      }
      if (out < 0) out = last_pos;
      if (lower_closer) {
        for (int t = out - 1; t >= 0 && draw_alt[b] < 0; --t)
          if (r[t] > 0.0) draw_alt[b] = t;
      } else {
        for (int t = out + 1; t < V && draw_alt[b] < 0; ++t)
          if (r[t] > 0.0) draw_alt[b] = t;
      }
      break;
    }
    std::vector<int> anc = ancestors_of(par, node);
    for (size_t t = 0; t < anc.size(); ++t) path[(size_t)b * N + (anc.size() - 1 - t)] = anc[t];
    accept_len[b] = depth_of(par, node);
    end_node[b] = node;
    out_token[b] = out;
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// TALON layer expansion [TALON §5.1, §5.2.1, §5.2.2].
//   Row v of draft_logits is the draft distribution p_d(. | path to
//   frontier_node[v]); frontier_logscore[v] = log s(frontier_node[v]).
//   Candidate (v, c) has log s = frontier_logscore[v] + log softmax(row v)[c].
//   layer == 1: keep the Top-K tokens of the single (root) row -- no gate.
//   layer >= 2: anchor = max log s over all candidates; keep those with
//              log s >= log(alpha) + anchor.
//   Either way at most R = budget - n_nodes are kept, the best scores first
//   (ties: parent node ascending, token ascending).  Kept nodes are appended
//   at ids n_nodes.. in (parent asc, score desc, token asc) order.
// margin = smallest |log s - threshold| over candidates, and the gap between
// the last kept and the first dropped score when they have different
// parents (absolute, log domain).  Candidates of one row differ only by their
// fp32 logits, so their order is exact and carries no margin.
// ---------------------------------------------------------------------------
struct Cand {
  double ls;
  int parent;
  int token;
};

int or_expand_gated(const float* draft_logits, const int32_t* frontier_node,
                    const float* frontier_logscore, int F, int V, int layer, int topk,
                    float alpha, int budget, int32_t* tree_parent, int32_t* tree_token,
                    float* tree_logscore, int32_t* n_nodes, double* margin) {
  *margin = INFINITY;
  if (F < 0 || V < 1 || layer < 1 || budget < 1) return ST_INVALID_ARG;
  if (layer == 1 && (F != 1 || topk < 1)) return ST_INVALID_ARG;
  if (layer >= 2 && !(alpha > 0.0f && alpha <= 1.0f)) return ST_INVALID_ARG;
  const int n0 = *n_nodes;
  const int R = budget - n0;
  if (R <= 0 || F == 0) return ST_OK;

  std::vector<Cand> all;
  all.reserve((size_t)F * V);
  for (int v = 0; v < F; ++v) {
    const float* row = draft_logits + (size_t)v * V;
    const double lse = row_logsumexp(row, V, 1.0);
    for (int c = 0; c < V; ++c)
      all.push_back({(double)frontier_logscore[v] + ((double)row[c] - lse), frontier_node[v], c});
  }
  auto better = [](const Cand& a, const Cand& b) {
    if (a.ls != b.ls) return a.ls > b.ls;
    if (a.parent != b.parent) return a.parent < b.parent;
    return a.token < b.token;
  };
  std::vector<Cand> pass;
  int limit = R;
  if (layer == 1) {
    pass = all;
    limit = std::min(topk, R);
  } else {
    double anchor = -INFINITY;
    for (const Cand& c : all) anchor = std::max(anchor, c.ls);
    const double thr = log((double)alpha) + anchor;
    for (const Cand& c : all) {
      if (c.ls >= thr) pass.push_back(c);
      if (c.ls != thr) *margin = std::min(*margin, fabs(c.ls - thr));
    }
  }
  std::sort(pass.begin(), pass.end(), better);
  if ((int)pass.size() > limit) {
    if (pass[limit - 1].parent != pass[limit].parent)
      *margin = std::min(*margin, pass[limit - 1].ls - pass[limit].ls);
    pass.resize(limit);
  }
  std::sort(pass.begin(), pass.end(), [](const Cand& a, const Cand& b) {
    if (a.parent != b.parent) return a.parent < b.parent;
    if (a.ls != b.ls) return a.ls > b.ls;
    return a.token < b.token;
  });
  for (size_t t = 0; t < pass.size(); ++t) {
    tree_parent[n0 + t] = pass[t].parent;
    tree_token[n0 + t] = pass[t].token;
    tree_logscore[n0 + t] = (float)pass[t].ls;
  }
  *n_nodes = n0 + (int)pass.size();
  return ST_OK;
}

// ---------------------------------------------------------------------------
// OPT-Tree greedy expansion, one layer [OPT] §3: a node's score is the
// product of the draft probabilities along its path (kept as its log); the
// frontier nodes are expanded, every child of every frontier node is a
// candidate (log score = the parent's + the child's log draft probability),
// and the layer keeps the `width` best candidates, which become the next
// frontier.  Ties go to the lower (parent, token).  The kept candidates are
// appended at n_nodes.. in (parent asc, score desc, token asc) order; a layer
// keeps at most capacity - n_nodes.  margin: the score gap at the cut between
// candidates of different parents (rounding can only reorder those).
// ---------------------------------------------------------------------------
int or_expand_topn(const float* draft_logits, const int32_t* frontier_node,
                   const float* frontier_logscore, int F, int V, int width, int capacity,
                   int32_t* tree_parent, int32_t* tree_token, float* tree_logscore,
                   int32_t* n_nodes, double* margin) {
  *margin = INFINITY;
  if (F < 0 || V < 1 || width < 1 || capacity < 1) return ST_INVALID_ARG;
  const int n0 = *n_nodes;
  const int limit = std::min(width, capacity - n0);
  if (limit <= 0 || F == 0) return ST_OK;
  std::vector<Cand> all;
  all.reserve((size_t)F * V);
  for (int v = 0; v < F; ++v) {
    const float* row = draft_logits + (size_t)v * V;
    const double lse = row_logsumexp(row, V, 1.0);
    for (int c = 0; c < V; ++c)
      all.push_back({(double)frontier_logscore[v] + ((double)row[c] - lse), frontier_node[v], c});
  }
  auto better = [](const Cand& a, const Cand& b) {
    if (a.ls != b.ls) return a.ls > b.ls;
    if (a.parent != b.parent) return a.parent < b.parent;
    return a.token < b.token;
  };
  // the best limit + 1 in order (a library partial sort), then the cut
  const size_t head = std::min(all.size(), (size_t)limit + 1);
  std::partial_sort(all.begin(), all.begin() + head, all.end(), better);
  if (all.size() > (size_t)limit) {
    if (all[limit - 1].parent != all[limit].parent)
      *margin = all[limit - 1].ls - all[limit].ls;
    all.resize(limit);
  }
  std::sort(all.begin(), all.end(), [](const Cand& a, const Cand& b) {
    if (a.parent != b.parent) return a.parent < b.parent;
    if (a.ls != b.ls) return a.ls > b.ls;
    return a.token < b.token;
  });
  for (size_t t = 0; t < all.size(); ++t) {
    tree_parent[n0 + t] = all[t].parent;
    tree_token[n0 + t] = all[t].token;
    tree_logscore[n0 + t] = (float)all[t].ls;
  }
  *n_nodes = n0 + (int)all.size();
  return ST_OK;
}

// ---------------------------------------------------------------------------
// OPT-Tree subtree selection [OPT] §3: of a candidate tree whose scores never
// rise from a node to its child, keep the n best-scoring nodes (ties to the
// lower node id, so a parent always ranks before its child); by that
// monotonicity they contain the root and every kept node's parent, i.e. they
// form a subtree, the one of n nodes with the largest sum of scores.
//   parent, token, logscore [B, M]; n_nodes [B] nodes in use (1..M).
//   out_* [B, n]: the kept nodes renumbered in their original order (so still
//   topological); out_src = the node's id in the input; rows k..n-1 (k =
//   min(n, n_nodes)) are -1 / 0.  expected[b] = sum of exp(logscore) over the
//   kept nodes other than the root (the expected acceptance length).
//   status: ST_INVALID_TREE for a malformed parent array or a kept node whose
//   parent is not kept (scores not monotone), ST_INVALID_ARG for a NaN score
//   or n_nodes outside 1..M; outputs of such a tree are -1 / 0.
// ---------------------------------------------------------------------------
int or_select_topn(const int32_t* parent, const int32_t* token, const float* logscore,
                   const int32_t* n_nodes, int B, int M, int n, int32_t* out_parent,
                   int32_t* out_token, float* out_logscore, int32_t* out_src, float* expected,
                   int32_t* status) {
  if (B < 0 || M < 1 || n < 1) return ST_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (size_t)b * M;
    const float* ls = logscore + (size_t)b * M;
    int32_t* op = out_parent + (size_t)b * n;
    int32_t* ot = out_token + (size_t)b * n;
    float* ol = out_logscore + (size_t)b * n;
    int32_t* os = out_src + (size_t)b * n;
    for (int j = 0; j < n; ++j) {
      op[j] = -1;
      ot[j] = -1;
      ol[j] = 0.0f;
      os[j] = -1;
    }
    expected[b] = 0.0f;
    const int m = n_nodes[b];
    int st = ST_OK;
    if (m < 1 || m > M) st = ST_INVALID_ARG;
    for (int i = 0; st == ST_OK && i < m; ++i) {
      if (i == 0 ? par[0] != -1 : (par[i] < 0 || par[i] >= i)) st = ST_INVALID_TREE;
      else if (std::isnan(ls[i])) st = ST_INVALID_ARG;
    }
    if (st == ST_OK) {
      std::vector<int> order(m);
      for (int i = 0; i < m; ++i) order[i] = i;
      std::sort(order.begin(), order.end(), [&](int a, int c) {
        if (ls[a] != ls[c]) return ls[a] > ls[c];
        return a < c;
      });
      const int k = std::min(n, m);
      std::vector<char> kept(m, 0);
      for (int r = 0; r < k; ++r) kept[order[r]] = 1;
      std::vector<int> newid(m, -1);
      int next = 0;
      for (int i = 0; i < m; ++i)
        if (kept[i]) newid[i] = next++;
      for (int i = 1; i < m; ++i)
        if (kept[i] && !kept[par[i]]) st = ST_INVALID_TREE;
      if (st == ST_OK) {
        double e = 0.0;
        for (int i = 0; i < m; ++i) {
          if (!kept[i]) continue;
          const int j = newid[i];
          op[j] = i == 0 ? -1 : newid[par[i]];
          ot[j] = token[(size_t)b * M + i];
          ol[j] = ls[i];
          os[j] = i;
          if (i != 0) e += exp((double)ls[i]);
        }
        expected[b] = (float)e;
      }
    }
    status[b] = st;
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// Commit of the accepted branch: [SPEC] "The protocol" step 4 (the accepted
// tokens and the correction extend the prefix) with [OPT] §2 (the accepted
// tokens are one root-to-node branch of the tree).  With the branch
// path[0..a] (path[0] = 0), the K and V rows of its nodes move from their
// tree slots kv_len + path[d] to the consecutive positions kv_len + d, one
// row after another in increasing d; the new prefix holds a + 1 more tokens
// (node 0 and the a accepted draft tokens).  A path that does not start at 0,
// is not strictly increasing, leaves the tree or the cache is rejected and
// its sequence left as it was.
int or_commit_path(uint16_t* k, uint16_t* v, const int32_t* kv_len, const int32_t* path,
                   const int32_t* accept_len, int B, int N, int Hkv, int D, int Lcap,
                   int32_t* new_kv_len, int32_t* status) {
  if (B < 0 || N < 1 || Hkv < 1 || D < 1 || Lcap < 1) return ST_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int L = kv_len[b], a = accept_len[b];
    const int32_t* pth = path + (size_t)b * N;
    bool ok = L >= 0 && a >= 0 && a < N && pth[0] == 0;
    for (int d = 1; ok && d <= a; ++d) ok = pth[d] > pth[d - 1] && pth[d] < N;
    if (ok) ok = (long long)L + pth[a] < (long long)Lcap;
    status[b] = ok ? ST_OK : ST_INVALID_ARG;
    new_kv_len[b] = ok ? L + a + 1 : L;
    if (!ok) continue;
    for (int h = 0; h < Hkv; ++h) {
      const size_t base = ((size_t)b * Hkv + h) * (size_t)Lcap;
      for (int d = 1; d <= a; ++d) {
        const size_t dst = (base + (size_t)(L + d)) * D;
        const size_t src = (base + (size_t)(L + pth[d])) * D;
        for (int e = 0; e < D; ++e) {
          k[dst + e] = k[src + e];
          v[dst + e] = v[src + e];
        }
      }
    }
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// Expected acceptance length of a draft tree, [OPT] §3: a node's score is
// the product of the draft probabilities along its path from the root, and
// the expected acceptance length is approximated by the sum of the scores of
// the tree's draft nodes (node 0, the last accepted token, scores 1 and
// counts no draft token).  prob[b, i] is node i's draft probability given its
// parent; prob[b, 0] is not read.  A tree that is not in topological order or
// a probability outside [0, 1] sets the sequence's status and leaves its
// outputs at 0.
int or_expected_accept(const int32_t* parent, const float* prob, int B, int N, double* score,
                       double* expected, int32_t* status) {
  if (B < 0 || N < 1) return ST_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parent + (size_t)b * N;
    const float* pr = prob + (size_t)b * N;
    expected[b] = 0.0;
    for (int i = 0; i < N; ++i) score[(size_t)b * N + i] = 0.0;
    if (!tree_is_valid(par, N)) { status[b] = ST_INVALID_TREE; continue; }
    bool ok = true;
    for (int i = 1; i < N; ++i)
      if (!(pr[i] >= 0.0f && pr[i] <= 1.0f)) ok = false;
    if (!ok) { status[b] = ST_INVALID_ARG; continue; }
    status[b] = ST_OK;
    double e = 0.0;
    for (int v = 0; v < N; ++v) {
      double s = 1.0;
      for (int u = v; u > 0; u = par[u]) s *= (double)pr[u];
      score[(size_t)b * N + v] = s;
      if (v > 0) e += s;
    }
    expected[b] = e;
  }
  return ST_OK;
}

// ---------------------------------------------------------------------------
// GOOSE anisotropic spine tree, [GOOSE] §2A (the spine: a chain of
// context-matched tokens; branches of transition tokens fork off every spine
// node; more of the budget to the spine where its acceptance is high, the
// rest as branches wide near the root and narrower deeper down) and §2B
// Proposition 2 (the optimal branch allocation decreases linearly with
// depth).  Readings where the pages give no formula:
//   * the spine takes d = min(S, round(ratio * (budget - 1))) nodes;
//   * branch point j (spine node j, j = 0 .. m-1, m = min(d + 1, Sb)) gets
//     w_j = floor(R (m - j) / (m (m + 1) / 2)) of the R = budget - 1 - d
//     branch nodes, the remainder one each from j = 0 on;
//   * a branch point with fewer usable candidates (row j of branch_tokens,
//     best first, -1 ends the row, the spine's own token at that depth
//     skipped, repeats skipped) passes the rest on to j + 1, j + 2, ...;
//   * nodes are numbered breadth-first, the spine child first at each depth.
int or_build_spine_tree(const int32_t* spine_tokens, int S, const int32_t* branch_tokens, int Sb,
                        int K, int root_token, int budget, float spine_ratio, int32_t* parent,
                        int32_t* tokens, int32_t* n_nodes) {
  if (S < 0 || Sb < 0 || K < 0 || budget < 1 || !(spine_ratio >= 0.0f && spine_ratio <= 1.0f))
    return ST_INVALID_ARG;
  int d = (int)llround((double)spine_ratio * (double)(budget - 1));
  d = std::min(d, S);
  const int R = budget - 1 - d;
  const int m = std::min(d + 1, Sb);
  // usable candidates of each branch point
  std::vector<std::vector<int>> cand(m);
  for (int j = 0; j < m; ++j) {
    const int spine_tok = (j < S) ? spine_tokens[j] : -1;  // the spine child's token at depth j+1
    for (int k = 0; k < K; ++k) {
      const int t = branch_tokens[(size_t)j * K + k];
      if (t < 0) break;
      if (j < d && t == spine_tok) continue;
      if (std::find(cand[j].begin(), cand[j].end(), t) != cand[j].end()) continue;
      cand[j].push_back(t);
    }
  }
  std::vector<int> w(m, 0);
  if (m > 0 && R > 0) {
    const long long T = (long long)m * (m + 1) / 2;
    int given = 0;
    for (int j = 0; j < m; ++j) {
      w[j] = (int)((long long)R * (m - j) / T);
      given += w[j];
    }
    for (int j = 0; given < R; ++j, ++given) w[j % m] += 1;
    int carry = 0;
    for (int j = 0; j < m; ++j) {
      w[j] += carry;
      carry = 0;
      if (w[j] > (int)cand[j].size()) {
        carry = w[j] - (int)cand[j].size();
        w[j] = (int)cand[j].size();
      }
    }
  }
  // breadth-first numbering: depth t holds spine node t (if t <= d), then the
  // branches of spine node t - 1
  int n = 0;
  parent[n] = -1;
  tokens[n] = root_token;
  ++n;
  int spine_id = 0;  // id of spine node t - 1 while depth t is numbered
  const int depth_max = std::max(d, m);
  for (int t = 1; t <= depth_max; ++t) {
    const int up = spine_id;
    if (t <= d) {
      parent[n] = up;
      tokens[n] = spine_tokens[t - 1];
      spine_id = n;
      ++n;
    }
    if (t - 1 < m)
      for (int k = 0; k < w[t - 1]; ++k) {
        parent[n] = up;
        tokens[n] = cand[t - 1][k];
        ++n;
      }
  }
  *n_nodes = n;
  return ST_OK;
}

// Philox4x64-10 block (exposed for the generator's own pins).
void or_philox4x64_10(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  philox4x64_10(ctr, key, out);
}

// The random word a decision uses (see or_accept_sample).
uint64_t or_draw_word(uint64_t seed, uint64_t offset, int b, int node, int purpose,
                      uint32_t ordinal) {
  return draw_word(seed, offset, b, node, (uint64_t)purpose, ordinal);
}

}  // extern "C"
