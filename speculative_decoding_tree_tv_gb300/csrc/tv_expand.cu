// tv_expand_gated: one layer of TALON's budget-driven tree expansion
// (TALON §5.1 token budget; §5.2.2 root Top-K; §5.2.1 confidence-gated
// expansion: candidate pool = all children of the frontier, path score
// s(c) = prod p_d, anchor = max s, keep s >= alpha * s_anchor, and keep the
// best-scoring ones when more survive than the remaining budget).
// tv_expand_topn: one layer of OPT-Tree's greedy expansion (OPT-Tree §3:
// every child of every frontier node is a candidate, scored by its path's
// draft probability, and the layer keeps the `width` best); the same
// launches without the gate, plus the floor kernel.
//
// Three launches (four for OPT-Tree layers), all on the caller's stream:
//   1. stats:   per (frontier row, 2048-logit chunk) max and sum exp, one warp
//               per chunk and eight chunks per CTA; each lane also lists the
//               largest of the 64 logits it read (value and token) and the
//               chunk records a bound u over everything else (the largest
//               lane's second largest); warp 0 of the last CTA of
//               a row to finish forms the row's log-normaliser lse_v and
//               offset off_v = logscore_v - lse_v (log s of token c in row v
//               is off_v + logit) and raises the layer's anchor (the best
//               score) with one atomic max;
//   1b. floor:  (OPT-Tree layers only) one CTA sets the layer's floor to
//               (just under) the limit-th best score among the chunks'
//               maxima: they are distinct candidates, so the layer's
//               limit-th best scores at least that much, and it is close to
//               the cut;
//   2. filter:  one CTA per row turns the fp64 gate (if
//               any) and the layer's floor into an fp32 logit threshold for
//               the row, and appends the (row, token) candidates that pass,
//               with their order-preserving fp64 score keys (at most the
//               layer's limit per chunk, its best ones).  It reads the logits
//               again only for a chunk whose bound u is at or above the
//               threshold; otherwise the chunk's maximum (no candidate) or its
//               lane-maximum list (every candidate; one warp per such chunk
//               appends them directly), so the rows stream from memory once
//               per layer when few candidates share a chunk, the usual case
//               above an OPT-Tree floor.  A re-read chunk holding
//               more than `limit` candidates raises the floor to its limit-th
//               best key: the layer's limit-th best is at least that, so
//               chunks that run later skip everything below it;
//   3. select:  one CTA keeps the best `limit` candidates, ties to the lower
//               (parent, token): up to 1024 candidates by their ranks (each
//               counted by up to 32 threads), beyond that by a radix select on
//               the score keys starting at the first byte in which the keys
//               differ; it orders them
//               (parent asc, score desc, token asc: each kept candidate's
//               position is the number of kept candidates before it, counted
//               by up to 32 threads; a bitonic sort beyond 1024 kept),
//               appends them to the tree and returns the control words
//               (candidate count, anchor, floor) to zero for the next call.
// Scores are fp64 in the log domain; logits stay fp32.
#define TV_UNIT 4
#include <algorithm>
#include <climits>

#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kExpThreads = 256;
constexpr int kStatsWarps = 8;   // chunks per stats CTA, one warp each
constexpr int kFiltGroup = 256;  // chunks per filter CTA at most (one thread each for the flags)
constexpr int kExpChunk = 2048;
constexpr int kSelThreads = 1024;
constexpr int kMaxBudget = 2048;
constexpr int kTieCap = 1024;
constexpr int kSelBatch = 8;  // key loads in flight per thread in the select passes
constexpr int kSelStageKeys = 16384;  // candidates whose keys the select stages in shared memory
constexpr int kFoldBins = 2048;  // the statistics pass's floor histogram: 1/64-nat bins, 32 nats

struct ExpPartial {
  double s;  // sum of exp(x - m) over the chunk
  float m;   // the chunk's largest logit
  float u;   // every logit of the chunk outside its lane-maximum list is <= u
};
// One entry of a chunk's lane-maximum list: the largest logit of the 64 a
// lane of the stats warp read, and its token (-1: the lane read nothing).
struct ExpCand {
  float v;
  int t;
};
struct ExpRow {
  double off;  // logscore_v - lse_v
  float m;     // the row's maximum logit
  float pad;
};
struct ExpCtl {
  int count;                 // candidates appended by the filter (returned to 0)
  int limit;                 // how many may be kept
  int n0;                    // nodes in the tree before this layer
  unsigned int rows_done;    // rows whose statistics are complete (returned to 0)
  unsigned long long anchor;  // order-preserving key of the best score (returned to 0)
  unsigned long long floor;   // key no kept candidate lies below (returned to 0)
};

struct ExpWs {
  ExpCtl* ctl;
  unsigned int* arrivals;  // [kMaxBudget] chunks of each row done by the stats pass (returned to 0)
  unsigned int* hist;      // [kFoldBins] chunk maxima per distance bin (returned to 0)
  ExpRow* rows;
  ExpPartial* part;
  ExpCand* cand;             // [row][chunk][32] lane maxima of each chunk
  unsigned long long* list;  // (row << 32) | token
  unsigned long long* keys;  // order-preserving fp64 score key of list[i]
};

// The control words (ExpCtl, then one arrival counter per possible row) sit at
// fixed offsets, so that what one call returns to zero is where the next call
// looks, whatever its number of frontier rows; the per-row and per-chunk
// regions after them move with F and are written before they are read.
__host__ __device__ inline size_t exp_arrivals_offset() { return align_up(sizeof(ExpCtl), 256); }
__host__ __device__ inline size_t exp_hist_offset() {
  return exp_arrivals_offset() + align_up((size_t)kMaxBudget * sizeof(unsigned int), 256);
}
__host__ __device__ inline size_t exp_offsets(int F, int V, size_t* rows_off, size_t* part_off,
                                              size_t* cand_off, size_t* list_off,
                                              size_t* keys_off) {
  const int chunks = (V + kExpChunk - 1) / kExpChunk;
  size_t o = exp_hist_offset() + align_up((size_t)kFoldBins * sizeof(unsigned int), 256);
  *rows_off = o;
  o += align_up((size_t)F * sizeof(ExpRow), 256);
  *part_off = o;
  o += align_up((size_t)F * chunks * sizeof(ExpPartial), 256);
  *cand_off = o;
  o += align_up((size_t)F * chunks * 32 * sizeof(ExpCand), 256);
  *list_off = o;
  o += align_up((size_t)F * V * sizeof(unsigned long long), 256);
  *keys_off = o;
  o += align_up((size_t)F * V * sizeof(unsigned long long), 256);
  return o;
}

__device__ __forceinline__ unsigned int arrive_acq_rel(unsigned int* p, unsigned int n) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(n)
               : "memory");
  return old;
}

constexpr float kLog2e = 1.4426950408889634f;
// 2^x on the special-function unit (ex2.approx.ftz): relative error about
// 2^-22, below the fp32 rounding of the logits it is applied to.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One warp per 2048-logit chunk (64 logits a lane, all loads in flight at
// once), kStatsWarps chunks of one row per CTA.  Each warp writes its chunk's
// partial (max, sum of exp(x - max)); the CTA then arrives on the row's counter
// with its number of chunks, and warp 0 of the row's last CTA combines the
// row's partials.
//
// fold (OPT-Tree layers with at least `cap` chunks): the floor under the
// layer's limit-th best score is found here instead of by exp_floor_kernel.
// Its reference is A0, the best frontier score, which no child's score
// exceeds (a row's normaliser is at least its largest term), so every
// distance below it is >= 0; the layer's best score lies within log V of it
// (a row's best child has probability >= 1 / V).  The row's last CTA counts
// each chunk maximum's distance below A0 in 1/64-nat bins (32 nats), and the
// layer's last row (acquiring every row's counts; its whole CTA, 8 bins a
// thread) finds the first bin from the top at which the count reaches
// `limit`: the floor is that bin's lower edge less a 1e-3
// nat margin for the fp32 distances, a little under the limit-th best chunk
// maximum and so under the limit-th best score (chunk maxima are distinct
// candidates).  Fewer than `limit` counted: no floor, as in exp_floor_kernel.
// The histogram and the row counter are returned to zero.
__global__ void __launch_bounds__(kStatsWarps * 32)
exp_stats_kernel(const float* __restrict__ logits, int V, int chunks,
                 const float* __restrict__ frontier_logscore, int fold, int cap, int budget,
                 const int32_t* __restrict__ n_nodes, ExpWs ws) {
  __shared__ int s_last;
  __shared__ unsigned int s_done;
  __shared__ float s_a0;
  __shared__ unsigned int s_wsum[kStatsWarps];
  pdl_trigger();
  pdl_wait();
  ExpPartial* __restrict__ part = ws.part;
  const int row = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * kStatsWarps + warp;
  const float* x = logits + (size_t)row * V;
  if (c < chunks) {
    const int start = c * kExpChunk;
    const int stop = min(V, start + kExpChunk);
    constexpr int kPer = kExpChunk / 32;
    float a[kPer];
    if ((V & 3) == 0) {  // rows 16-byte aligned; a chunk holds whole float4s
      const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
      for (int u = 0; u < kPer / 4; ++u) {
        const int e = start + 4 * (lane + 32 * u);
        const float4 f = (e < stop) ? ld_stream_f4(x4 + (e >> 2))
                                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        a[4 * u + 0] = f.x;
        a[4 * u + 1] = f.y;
        a[4 * u + 2] = f.z;
        a[4 * u + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = start + lane + 32 * u;
        a[u] = (e < stop) ? __ldg(x + e) : -INFINITY;
      }
    }
    // the lane's largest logit (first of its ties) and second largest (a tie
    // with the largest counts): everything the lane read but did not list is
    // <= its second largest
    float v1 = -INFINITY, v2 = -INFINITY;
    int u1 = -1;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      if (a[u] > v1) {
        v2 = v1;
        v1 = a[u];
        u1 = u;
      } else {
        v2 = fmaxf(v2, a[u]);
      }
    }
    const int t1 = (u1 < 0) ? -1
                   : ((V & 3) == 0) ? start + 4 * (lane + 32 * (u1 >> 2)) + (u1 & 3)
                                    : start + lane + 32 * u1;
    ws.cand[((size_t)row * chunks + c) * 32 + lane] = ExpCand{v1, t1};
    const float ub = warp_max(v2);
    const float m = warp_max(v1);
    const float ml = m * kLog2e;
    float sl = 0.0f;
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      sl += (a[u] == -INFINITY) ? 0.0f : ex2_approx(fmaf(a[u], kLog2e, -ml));
    const double sd = warp_sum_d((double)sl);
    if (lane == 0) {
      part[(size_t)row * chunks + c] = ExpPartial{sd, m, ub};
      __threadfence();  // the partial is visible before the CTA arrives
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int mine = (unsigned int)min(kStatsWarps, chunks - (int)blockIdx.x * kStatsWarps);
    // the last arrival (acquire) sees every partial of the row
    s_last = TV_IN(row, kMaxBudget) &&
             (arrive_acq_rel(&ws.arrivals[row], mine) + mine == (unsigned int)chunks);
  }
  __syncthreads();
  if (!s_last) return;  // uniform over the CTA
  const int F = (int)gridDim.y;
  if (warp == 0) {
    // warp 0 of the row's last CTA: normaliser, offset and best score of the
    // row.  Exponentials on the SFU (fp32; fp64 runs at a small fraction of
    // the fp32 rate here), the sum itself in fp64, the logarithm in one lane.
    const ExpPartial* p = part + (size_t)row * chunks;
    float mr = -INFINITY;
    for (int k = lane; k < chunks; k += 32) mr = fmaxf(mr, __ldcg(&p[k].m));
    mr = warp_max(mr);
    double sr = 0.0;
    for (int k = lane; k < chunks; k += 32)
      sr += __ldcg(&p[k].s) * (double)ex2_approx((__ldcg(&p[k].m) - mr) * kLog2e);
    sr = warp_sum_d(sr);
    double off = 0.0;
    if (lane == 0) {
      off = (double)frontier_logscore[row] - ((double)mr + log(sr));
      ws.arrivals[row] = 0u;
      ws.rows[row].off = off;
      ws.rows[row].m = mr;
      atomicMax(&ws.ctl->anchor, double_key(off + (double)mr));
    }
    if (fold) {
      off = __shfl_sync(0xffffffffu, off, 0);
      float a0 = -INFINITY;
      for (int r = lane; r < F; r += 32) a0 = fmaxf(a0, __ldg(frontier_logscore + r));
      a0 = warp_max(a0);
      const float av = (float)((double)a0 - off);  // A0 - off, once per row in fp64
      for (int k = lane; k < chunks; k += 32) {
        const float d = (av - __ldcg(&p[k].m)) * 64.0f;  // >= 0 up to rounding
        if (d < (float)kFoldBins) atomicAdd(&ws.hist[max(0, (int)d)], 1u);
      }
      __threadfence();  // this lane's counts are performed before the row arrives
      __syncwarp();
      if (lane == 0) {
        s_done = arrive_acq_rel(&ws.ctl->rows_done, 1u) + 1u;
        s_a0 = a0;
      }
    }
  }
  if (!fold) return;
  __syncthreads();
  if (s_done != (unsigned int)F) return;
  // the layer's last row: every row's counts are in (acquired by thread 0;
  // the barrier orders the reads below after it).  Thread t holds bins
  // [8t, 8t + 8), nearest to A0 first.
  static_assert(kFoldBins == 8 * kStatsWarps * 32, "8 bins a thread");
  const int t = threadIdx.x;
  const uint4 h0 = __ldcg(reinterpret_cast<const uint4*>(ws.hist) + 2 * t);
  const uint4 h1 = __ldcg(reinterpret_cast<const uint4*>(ws.hist) + 2 * t + 1);
  const unsigned int hb[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
  unsigned int tsum = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) tsum += hb[i];
  unsigned int incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  for (int w = 0; w < warp; ++w) incl += s_wsum[w];
  const unsigned int above = incl - tsum;  // maxima in bins nearer to A0
  const int remaining = budget - __ldcg(n_nodes);
  const int limit = min(remaining > 0 ? remaining : 0, cap);
  const unsigned int need = (unsigned int)limit;
  if (limit > 0 && above < need && incl >= need) {
    // the first of this thread's bins (nearest A0 first) at which the count
    // reaches `need`
    int bin = 8 * t + 7;
    unsigned int run = above;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      run += hb[i];
      if (run >= need) {
        bin = 8 * t + i;
        break;
      }
    }
    // every maximum counted up to this bin lies above A0 - (bin + 1) / 64, up
    // to the fp32 rounding of its distance, which the margin covers
    ws.ctl->floor = double_key((double)s_a0 - (double)(bin + 1) / 64.0 - 1e-3);
  }
  reinterpret_cast<uint4*>(ws.hist)[2 * t] = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<uint4*>(ws.hist)[2 * t + 1] = make_uint4(0u, 0u, 0u, 0u);
  if (t == 0) ws.ctl->rows_done = 0u;
}

// Smallest fp32 value >= x (x finite).
__device__ __forceinline__ float float_ceil_of(double x) {
  float f = (float)x;
  if ((double)f < x) f = nextafterf(f, INFINITY);
  return f;
}

// Inverse of double_key.
__device__ __forceinline__ double key_double(unsigned long long k) {
  const unsigned long long u = (k & 0x8000000000000000ull) ? (k & 0x7fffffffffffffffull) : ~k;
  return __longlong_as_double((long long)u);
}

constexpr int kFloorThreads = 1024;
constexpr int kFloorBins = 2048;      // bins below the anchor ...
constexpr double kFloorBinsPerNat = 64.0;  // ... each 1/64 nat wide (32 nats in all)
constexpr int kFloorBatch = 16;       // chunk maxima a thread loads at once

// One CTA: a floor under the layer's limit-th best score from the chunks'
// maxima (distinct candidates, so at least `limit` candidates score as much
// as the limit-th best of them).  Each maximum's distance below the anchor
// (the layer's best score) is counted in 1/64-nat bins; the first bin from
// the top at which the count reaches `limit` gives the floor, its lower edge
// less a margin (a little under the exact value, which is all a floor needs).
// The distances are fp32 (the row's offset from the anchor once per row in
// fp64); the 1e-3-nat margin covers their rounding.  Maxima more than 32 nats
// down are not counted; if fewer than `limit` are left there is no floor (it
// stays 0).  With fewer chunks than `limit` (a few rows: the root layer) the
// lanes' maxima of the statistics pass (32 per chunk, also distinct
// candidates) are counted instead, and with fewer of those every logit.
__global__ void __launch_bounds__(kFloorThreads)
exp_floor_kernel(const float* __restrict__ logits, int V, int F, int chunks, int cap, int budget,
                 const int32_t* __restrict__ n_nodes, ExpWs ws) {
  __shared__ unsigned int s_hist[kFloorBins];
  __shared__ float s_av[kMaxBudget];  // anchor - off_v, per frontier row
  __shared__ unsigned int s_wsum[kFloorThreads / 32];
  __shared__ int s_bin;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int remaining = budget - *n_nodes;
  const int limit = min(remaining > 0 ? remaining : 0, cap);
  // the values counted: the chunks' maxima; with fewer chunks than `limit`,
  // the lanes' maxima of the statistics pass (32 per chunk); with fewer
  // still, every logit.  Each is a distinct candidate.
  const int mode = (F * chunks >= limit) ? 0 : ((long long)F * chunks * 32 >= limit) ? 1 : 2;
  const int per_row = mode == 0 ? chunks : mode == 1 ? chunks * 32 : V;
  const int total = F * per_row;
  if (limit == 0 || total < limit || !TV_CHECK(F <= kMaxBudget)) return;
  const double anchor = key_double(ws.ctl->anchor);
  for (int i = tid; i < kFloorBins; i += kFloorThreads) s_hist[i] = 0u;
  for (int r = tid; r < F; r += kFloorThreads) s_av[r] = (float)(anchor - ws.rows[r].off);
  if (tid == 0) s_bin = -1;
  __syncthreads();
  const float inv_per_row = 1.0f / (float)per_row;
  for (int i0 = 0; i0 < total; i0 += kFloorBatch * kFloorThreads) {
    float mx[kFloorBatch];  // a batch of values, their loads in flight together
#pragma unroll
    for (int u = 0; u < kFloorBatch; ++u) {
      const int i = i0 + tid + u * kFloorThreads;
      mx[u] = (i >= total) ? -INFINITY
              : mode == 0  ? __ldcg(&ws.part[i].m)
              : mode == 1  ? __ldcg(&ws.cand[i].v)
                           : __ldg(logits + i);
    }
#pragma unroll
    for (int u = 0; u < kFloorBatch; ++u) {
      const int i = i0 + tid + u * kFloorThreads;
      int r = (int)((float)i * inv_per_row);  // the row of value i, corrected to be exact
      r -= (r * per_row > i);
      r += ((r + 1) * per_row <= i);
      const float d = (s_av[min(r, F - 1)] - mx[u]) * (float)kFloorBinsPerNat;  // >= 0
      if (i < total && d < (float)kFloorBins) atomicAdd(&s_hist[max(0, (int)d)], 1u);
    }
  }
  __syncthreads();
  // cumulative counts from the top bin: each thread holds two adjacent bins
  const int b0 = 2 * tid;
  const unsigned int c0 = s_hist[b0], c1 = s_hist[b0 + 1];
  unsigned int incl = c0 + c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  unsigned int before = 0u;
  for (int w = 0; w < warp; ++w) before += s_wsum[w];
  const unsigned int above = before + incl - (c0 + c1);  // maxima in higher bins
  const unsigned int need = (unsigned int)limit;
  if (above < need && above + c0 + c1 >= need) s_bin = (above + c0 >= need) ? b0 : b0 + 1;
  __syncthreads();
  if (tid == 0 && s_bin >= 0) {
    // every maximum counted up to bin b lies above anchor - (b + 1) / 64, up
    // to the fp32 rounding of its distance, which the margin covers
    const double fl = anchor - (double)(s_bin + 1) / kFloorBinsPerNat - 1e-3;
    ws.ctl->floor = double_key(fl);
  }
}

// kExpChunk / kExpThreads logits of one chunk per thread
constexpr int kFiltPer = kExpChunk / kExpThreads;

// Element j of a thread's share of a chunk: with 16-byte rows two float4s
// (4 (tid + 256 u) + k, j = 4u + k), otherwise tid + 256 j.
__device__ __forceinline__ int filt_elem(bool vec, int tid, int j) {
  return vec ? 4 * (tid + kExpThreads * (j >> 2)) + (j & 3) : tid + kExpThreads * j;
}

// One CTA per (frontier row, group of chunks): the whole row (up to
// kFiltGroup chunks) once there are 32 rows or more, else four chunks, so
// that the root layer's re-read chunks spread over CTAs.  Thread 0 turns
// the fp64 gate (if any) and the layer's floor into an fp32 logit threshold
// for the row.  Per chunk, the candidates (logit >= the threshold) are
// gathered in shared memory with their score keys, from one of three places:
// none if the chunk's maximum is below the threshold (most chunks); the
// chunk's lane-maximum list if the threshold lies above the chunk's bound u
// (every logit outside the list is <= u, so the list holds every candidate);
// else the chunk itself, read again.  When there are more candidates than
// the layer may keep (`limit`), only the chunk's best `limit` under the
// output's total order (score desc, then token asc within a row) are
// appended: the layer's best `limit` overall are among them, and the select
// kernel then sees at most chunks x limit candidates per row.  gated: TALON's
// alpha gate against the anchor (limit = the remaining budget); otherwise
// every child is a candidate and limit = min(cap, remaining).
__global__ void __launch_bounds__(kExpThreads)
exp_filter_kernel(const float* __restrict__ logits, int V, int cpc, int gated, int cap, int budget,
                  double log_alpha, const int32_t* __restrict__ n_nodes, ExpWs ws) {
  __shared__ unsigned long long s_key[kExpChunk];
  __shared__ int s_tok[kExpChunk];
  __shared__ unsigned int s_hist[256];
  __shared__ unsigned int s_tiebits[kExpChunk / 32];
  __shared__ int s_cnt, s_base, s_digit, s_need, s_out;
  __shared__ unsigned long long s_kmin, s_kmax;
  __shared__ float s_thr;
  __shared__ int s_limit;
  __shared__ int s_chunks[kFiltGroup];  // (chunk offset << 2) | 1 list or 2 re-read
  __shared__ int s_wcount[kExpThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int row = gridDim.y - 1 - blockIdx.y;
  const int group = gridDim.x - 1 - blockIdx.x;
  const int chunks = ceil_div(V, kExpChunk);
  const int c0 = group * cpc;
  const int nc = min(min(cpc, kFiltGroup), chunks - c0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* x = logits + (size_t)row * V;
  const bool vec = (V & 3) == 0;
  const double off = ws.rows[row].off;
  if (tid == 0) {
    const int n0 = *n_nodes;
    const int remaining = budget - n0;
    const int limit = min(remaining > 0 ? remaining : 0, cap);
    float thr;
    if (!gated || limit == 0) {
      thr = limit == 0 ? INFINITY : -INFINITY;
    } else {
      // s = off_v + logit >= log(alpha) + anchor  <=>  logit >= m_v + (d_v + log(alpha)),
      // d_v = anchor - best_v >= 0 (best_v = off_v + m_v), exactly 0 in the anchor's row
      const double anchor = key_double(ws.ctl->anchor);
      const double m = (double)ws.rows[row].m;
      const double d = anchor - (off + m);
      thr = float_ceil_of(m + (d + log_alpha));
    }
    const unsigned long long fk = *(volatile unsigned long long*)&ws.ctl->floor;
    if (limit > 0 && fk != 0ull) {
      // the smallest logit whose score off + logit can round to the floor or
      // above, taken a little low (a superset passes; the selects are exact)
      const double fs = key_double(fk);
      const double xs = (fs - off) - 4e-16 * (fabs(fs) + fabs(off));
      thr = fmaxf(thr, nextafterf((float)xs, -INFINITY));
    }
    if (c0 == 0 && row == 0) {
      ws.ctl->limit = limit;
      ws.ctl->n0 = n0;
    }
    s_thr = thr;
    s_limit = limit;
  }
  __syncthreads();
  const float thr = s_thr;
  if (!(thr < INFINITY)) return;
  const int limit = s_limit;
  const unsigned long long row_hi = (unsigned long long)row << 32;
  // a whole warp offers one value per lane; the passing ones go to the
  // chunk's candidate list in shared memory
  auto push = [&](bool pass, float lg, int e) {
    const unsigned int bal = __ballot_sync(0xffffffffu, pass);
    if (bal == 0u) return;
    int slot0 = 0;
    if (lane == 0) slot0 = atomicAdd(&s_cnt, __popc(bal));
    slot0 = __shfl_sync(0xffffffffu, slot0, 0);
    if (pass) {
      const int slot = slot0 + __popc(bal & ((1u << lane) - 1u));
      if (TV_IN(slot, kExpChunk)) {
        s_key[slot] = double_key(off + (double)lg);
        s_tok[slot] = e;
      }
    }
  };
  // the chunks holding a candidate, in order, one thread per chunk: by the
  // list when the threshold lies above the chunk's bound, else by a re-read
  int flag = 0;
  if (tid < nc) {
    const ExpPartial pc = ws.part[(size_t)row * chunks + c0 + tid];
    flag = (pc.m >= thr) ? ((thr > pc.u) ? 1 : 2) : 0;
  }
  const unsigned int fb = __ballot_sync(0xffffffffu, flag != 0);
  if (lane == 0) s_wcount[warp] = __popc(fb);
  __syncthreads();
  int before = 0, nflag = 0;
#pragma unroll
  for (int w = 0; w < kExpThreads / 32; ++w) {
    before += (w < warp) ? s_wcount[w] : 0;
    nflag += s_wcount[w];
  }
  if (flag) s_chunks[before + __popc(fb & ((1u << lane) - 1u))] = (tid << 2) | flag;
  __syncthreads();
  // chunks decided by their list: one warp each, appended straight to the
  // layer's candidates (at most 32 from a chunk)
  for (int q = warp; q < nflag; q += kExpThreads / 32) {
    if ((s_chunks[q] & 3) != 1) continue;  // warp-uniform
    const int c = c0 + (s_chunks[q] >> 2);
    const int start = c * kExpChunk;
    const int stop = min(V, start + kExpChunk);
    const ExpCand e = ws.cand[((size_t)row * chunks + c) * 32 + lane];
    const bool pass = e.t >= 0 && e.v >= thr && TV_IN(e.t - start, stop - start);
    const unsigned int bal = __ballot_sync(0xffffffffu, pass);
    if (bal == 0u) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(&ws.ctl->count, __popc(bal));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (pass) {
      const int slot = base + __popc(bal & ((1u << lane) - 1u));
      if (TV_IN((long long)slot, (long long)gridDim.y * V)) {
        ws.list[slot] = row_hi | (unsigned int)e.t;
        ws.keys[slot] = double_key(off + (double)e.v);
      }
    }
  }
  // chunks read again, by the whole CTA one after another
  for (int q = 0; q < nflag; ++q) {
    const int c = c0 + (s_chunks[q] >> 2);
    if ((s_chunks[q] & 3) == 1) continue;  // uniform: done above
    const int start = c * kExpChunk;
    const int stop = min(V, start + kExpChunk);
    if (tid == 0) {
      s_cnt = 0;
      s_out = 0;
      s_kmin = ~0ull;
      s_kmax = 0ull;
    }
    __syncthreads();
    {
      // the chunk again, all of a thread's loads in flight at once
      float a[kFiltPer];
      if (vec) {
        const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
        for (int u = 0; u < kFiltPer / 4; ++u) {
          const int e = start + 4 * (tid + kExpThreads * u);
          const float4 f = (e < stop) ? __ldg(x4 + (e >> 2))
                                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          a[4 * u + 0] = f.x;
          a[4 * u + 1] = f.y;
          a[4 * u + 2] = f.z;
          a[4 * u + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < kFiltPer; ++j) {
          const int e = start + tid + kExpThreads * j;
          a[j] = (e < stop) ? __ldg(x + e) : -INFINITY;
        }
      }
#pragma unroll
      for (int j = 0; j < kFiltPer; ++j) {
        const int e = start + filt_elem(vec, tid, j);
        push((e < stop) && (a[j] >= thr), a[j], e);
      }
    }
    __syncthreads();
    const int n = s_cnt;
    if (n == 0) continue;
    if (n <= limit) {  // everything passes on
      if (tid == 0) s_base = atomicAdd(&ws.ctl->count, n);
      __syncthreads();
      for (int i = tid; i < n; i += kExpThreads) {
        if (!TV_IN((long long)s_base + i, (long long)gridDim.y * V)) continue;
        ws.list[s_base + i] = row_hi | (unsigned int)s_tok[i];
        ws.keys[s_base + i] = s_key[i];
      }
      __syncthreads();
      continue;
    }
    // radix select of the limit-th largest key T among the n (the bytes above
    // the highest one in which the smallest and largest key differ are common)
    for (int i = tid; i < kExpChunk / 32; i += kExpThreads) s_tiebits[i] = 0u;
    unsigned long long kmin = ~0ull, kmax = 0ull;
    for (int i = tid; i < n; i += kExpThreads) {
      kmin = min(kmin, s_key[i]);
      kmax = max(kmax, s_key[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (lane == 0) {
      atomicMin(&s_kmin, kmin);
      atomicMax(&s_kmax, kmax);
    }
    __syncthreads();
    const unsigned long long diff = s_kmin ^ s_kmax;
    const int top = diff ? ((63 - __clzll((long long)diff)) & ~7) : 0;
    unsigned long long mask = (top >= 56) ? 0ull : (~0ull << (top + 8));
    unsigned long long prefix = s_kmax & mask;
    int need = limit;
    for (int shift = top; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kExpThreads) s_hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n; i += kExpThreads) {
        const unsigned long long k = s_key[i];
        if ((k & mask) == prefix) atomicAdd(&s_hist[(k >> shift) & 255ull], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // digits from the top: lane l holds digits 255 - 8l .. 248 - 8l
        int cnt[8], lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          cnt[i] = (int)s_hist[255 - 8 * lane - i];
          lsum += cnt[i];
        }
        int incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int above = incl - lsum;
        if (above < need && incl >= need) {
          int cum = above;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (cum + cnt[i] >= need) {
              s_digit = 255 - 8 * lane - i;
              s_need = need - cum;
              break;
            }
            cum += cnt[i];
          }
        }
      }
      __syncthreads();
      prefix |= (unsigned long long)s_digit << shift;
      mask |= 0xffull << shift;
      need = s_need;
      __syncthreads();
    }
    const unsigned long long T = prefix;
    // at least `limit` candidates of this chunk score T or more
    if (tid == 0) atomicMax(&ws.ctl->floor, T);
    // ties at T: the `need` lowest tokens, found through a bitmap of the chunk
    for (int i = tid; i < n; i += kExpThreads)
      if (s_key[i] == T && TV_IN(s_tok[i] - start, kExpChunk))
        atomicOr(&s_tiebits[(s_tok[i] - start) >> 5], 1u << ((s_tok[i] - start) & 31));
    if (tid == 0) s_base = atomicAdd(&ws.ctl->count, limit);
    __syncthreads();
    // the cutoff token: the need-th set bit of the bitmap, by one warp
    if (warp == 0) {
      int before = 0;
      for (int w0 = 0; w0 < kExpChunk / 32; w0 += 32) {
        const unsigned int bits = s_tiebits[w0 + lane];
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int tot = __shfl_sync(0xffffffffu, incl, 31);
        if (before + tot >= need) {
          const int ex = before + incl - c;  // set bits before this lane's word
          if (ex < need && ex + c >= need) {
            unsigned int b = bits;
            for (int r = need - ex; r > 1; --r) b &= b - 1u;  // drop the lower set bits
            s_digit = start + ((w0 + lane) << 5) + (__ffs(b) - 1);  // the need-th tie token
          }
          break;
        }
        before += tot;
      }
    }
    __syncthreads();
    const int last_tie = s_digit;
    for (int i = tid; i < n; i += kExpThreads) {
      const unsigned long long k = s_key[i];
      if (k > T || (k == T && s_tok[i] <= last_tie)) {
        const int slot = s_base + atomicAdd(&s_out, 1);
        if (!TV_IN((long long)slot, (long long)gridDim.y * V)) continue;
        ws.list[slot] = row_hi | (unsigned int)s_tok[i];
        ws.keys[slot] = k;
      }
    }
    __syncthreads();
  }
}

struct Kept {
  unsigned long long key;  // order-preserving score key
  int row;
  int token;
};

// order of the output: row (parent) asc, score desc, token asc
__device__ __forceinline__ bool out_before(const Kept& a, const Kept& b) {
  if (a.row != b.row) return a.row < b.row;
  if (a.key != b.key) return a.key > b.key;
  return a.token < b.token;
}

// order of the selection: score desc, then the lower (row, token)
__device__ __forceinline__ bool sel_before(const Kept& a, const Kept& b) {
  if (a.key != b.key) return a.key > b.key;
  if (a.row != b.row) return a.row < b.row;
  return a.token < b.token;
}

// Ascending bitonic sort of n_pow2 entries under out_before (kOut) or
// sel_before, by the whole CTA.
template <bool kOut>
__device__ void bitonic_sort_kept(Kept* s, int n_pow2) {
  for (int k = 2; k <= n_pow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const Kept a = s[i], b = s[ixj];
          const bool b_first = kOut ? out_before(b, a) : sel_before(b, a);
          const bool a_first = kOut ? out_before(a, b) : sel_before(a, b);
          if (up ? b_first : a_first) {
            s[i] = b;
            s[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__device__ void bitonic_sort_u64(unsigned long long* s, int n_pow2) {
  for (int k = 2; k <= n_pow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const bool swap = up ? (s[ixj] < s[i]) : (s[i] < s[ixj]);
          if (swap) {
            const unsigned long long t = s[i];
            s[i] = s[ixj];
            s[ixj] = t;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Threads per candidate when ranking k candidates with kSelThreads threads:
// the largest power of two <= kSelThreads / k, at most a warp.
__device__ __forceinline__ int rank_split(int k) {
  int t = 1;
  while (t < 32 && 2 * t * k <= kSelThreads) t <<= 1;
  return t;
}

__global__ void __launch_bounds__(kSelThreads)
exp_select_kernel(const float* __restrict__ logits, int V, int F, int budget,
                  const int32_t* __restrict__ frontier_node,
                  int32_t* __restrict__ tree_parent, int32_t* __restrict__ tree_token,
                  float* __restrict__ tree_logscore, int32_t* __restrict__ n_nodes, ExpWs ws) {
  // the per-warp histograms of the radix passes and the kept list are never
  // live at the same time: they share one buffer
  static_assert((kSelThreads / 32) * 256 * sizeof(unsigned int) <= kMaxBudget * sizeof(Kept), "");
  __shared__ __align__(16) unsigned char s_buf[kMaxBudget * sizeof(Kept)];
  Kept* s_kept = reinterpret_cast<Kept*>(s_buf);
  auto s_hist = reinterpret_cast<unsigned int (*)[256]>(s_buf);  // [warp][digit]
  __shared__ unsigned long long s_ties[kTieCap];
  __shared__ int s_n, s_nt, s_digit, s_need;
  __shared__ unsigned long long s_min, s_kmin, s_kmax;
  // the candidates' keys, staged once so that the radix passes read shared
  // memory; once the kept set is known, the same space holds it in output order
  extern __shared__ unsigned long long s_stage[];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const ExpCtl ctl = *ws.ctl;
  const int count = ctl.count, limit = ctl.limit;
  const int lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_n = 0;
    s_nt = 0;
    s_kmin = ~0ull;
    s_kmax = 0ull;
  }
  __syncthreads();
  int k;  // candidates kept, in s_kept[0, k) in no particular order
  if (count <= limit) {
    // every candidate is kept
    k = TV_CHECK(count <= kMaxBudget) ? count : 0;
    for (int j = tid; j < k; j += kSelThreads) {
      const unsigned long long c = ws.list[j];
      s_kept[j] = Kept{ws.keys[j], (int)(c >> 32), (int)(c & 0xffffffffu)};
    }
    __syncthreads();
  } else if (count <= kSelThreads) {
    // a few more than are kept: each candidate's rank under the selection
    // order (score desc, then the lower (row, token)) is the number of
    // candidates before it, counted by rank_split(count) threads; the first
    // `limit` ranks land in order at the start of s_stage and are copied back
    for (int j = tid; j < count; j += kSelThreads) {
      const unsigned long long c = ws.list[j];
      s_kept[j] = Kept{ws.keys[j], (int)(c >> 32), (int)(c & 0xffffffffu)};
    }
    __syncthreads();
    Kept* s_sel = reinterpret_cast<Kept*>(s_stage);
    const int tpc = rank_split(count);
    const int i = tid / tpc, part = tid % tpc;
    int r = 0;
    Kept me{};
    if (i < count) {
      me = s_kept[i];
      for (int j = part; j < count; j += tpc) r += sel_before(s_kept[j], me);
    }
    for (int o = tpc >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (i < count && part == 0 && r < limit) s_sel[r] = me;
    __syncthreads();
    k = limit;
    for (int j = tid; j < k; j += kSelThreads) s_kept[j] = s_sel[j];
    __syncthreads();
  } else {
    // radix select of T = the limit-th largest key, need = how many keys == T
    // to take.  The bytes above the highest one in which the smallest and the
    // largest key differ are common to all keys and skipped.
    const bool staged = count <= kSelStageKeys;
    if (staged) {
      for (int j = tid; j < count; j += kSelThreads) s_stage[j] = ws.keys[j];
      __syncthreads();
    }
    const unsigned long long* K = staged ? s_stage : ws.keys;
    unsigned long long kmin = ~0ull, kmax = 0ull;
    for (int j0 = tid; j0 < count; j0 += kSelBatch * kSelThreads) {
      unsigned long long kb[kSelBatch];
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        const int j = j0 + u * kSelThreads;
        kb[u] = (j < count) ? K[j] : K[0];
      }
#pragma unroll
      for (int u = 0; u < kSelBatch; ++u) {
        kmin = min(kmin, kb[u]);
        kmax = max(kmax, kb[u]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (lane == 0) {
      atomicMin(&s_kmin, kmin);
      atomicMax(&s_kmax, kmax);
    }
    __syncthreads();
    const unsigned long long diff = s_kmin ^ s_kmax;
    const int top = diff ? ((63 - __clzll((long long)diff)) & ~7) : 0;
    unsigned long long mask = (top >= 56) ? 0ull : (~0ull << (top + 8));
    unsigned long long prefix = s_kmax & mask;
    int need = limit;
    // Once the digit holding the limit-th key has at most kSelThreads keys
    // (the bucket [b_lo, b_hi]), the keys above it are kept, and the `need`
    // best of the bucket are found by their ranks: the remaining passes and
    // the ties are skipped.
    bool bucketed = false;
    unsigned long long b_lo = 0ull, b_hi = 0ull;
    for (int shift = top; shift >= 0; shift -= 8) {
      for (int i = tid; i < (kSelThreads / 32) * 256; i += kSelThreads) (&s_hist[0][0])[i] = 0u;
      __syncthreads();
      for (int j0 = tid; j0 < count; j0 += kSelBatch * kSelThreads) {
        unsigned long long kb[kSelBatch];
#pragma unroll
        for (int u = 0; u < kSelBatch; ++u) {
          const int j = j0 + u * kSelThreads;
          kb[u] = (j < count) ? K[j] : ~prefix;  // ~prefix never matches the prefix
        }
#pragma unroll
        for (int u = 0; u < kSelBatch; ++u)
          if ((kb[u] & mask) == prefix && (j0 + u * kSelThreads) < count)
            atomicAdd(&s_hist[warp][(kb[u] >> shift) & 255ull], 1u);
      }
      __syncthreads();
      if (tid < 256) {
        unsigned int t = 0u;
#pragma unroll 8
        for (int w = 0; w < kSelThreads / 32; ++w) t += s_hist[w][tid];
        s_hist[0][tid] = t;
      }
      __syncthreads();
      if (warp == 0) {
        // digits from the top: lane l sums digits 255 - 8l .. 248 - 8l, an
        // exclusive scan over lanes gives the count above each lane's digits
        int cnt[8], lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          cnt[i] = (int)s_hist[0][255 - 8 * lane - i];
          lsum += cnt[i];
        }
        int incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int above = incl - lsum;
        if (above < need && incl >= need) {
          int cum = above;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (cum + cnt[i] >= need) {
              s_digit = 255 - 8 * lane - i;
              s_need = need - cum;
              break;
            }
            cum += cnt[i];
          }
        }
      }
      __syncthreads();
      const int bucket = (int)s_hist[0][s_digit];
      prefix |= (unsigned long long)s_digit << shift;
      mask |= 0xffull << shift;
      need = s_need;
      __syncthreads();
      if (bucket <= kSelThreads && limit - need + bucket <= kMaxBudget) {  // uniform
        bucketed = true;
        b_lo = prefix;
        b_hi = prefix | ((1ull << shift) - 1ull);
        break;
      }
    }
    if (bucketed) {
      // the keys above the bucket go to s_kept[0, limit - need), the bucket
      // after them; then the bucket's `need` best, by their ranks, are placed
      // in s_stage (its keys are no longer needed) and copied back
      const int n_gt = limit - need;
      for (int j = tid; j < count; j += kSelThreads) {
        const unsigned long long kj = K[j];
        if (kj < b_lo) continue;
        const unsigned long long c = ws.list[j];
        const int slot = (kj > b_hi) ? atomicAdd(&s_n, 1) : n_gt + atomicAdd(&s_nt, 1);
        if (TV_IN(slot, kMaxBudget)) s_kept[slot] = Kept{kj, (int)(c >> 32), (int)(c & 0xffffffffu)};
      }
      __syncthreads();
      const int nb = s_nt;
      Kept* s_win = reinterpret_cast<Kept*>(s_stage);
      const Kept* s_bk = s_kept + n_gt;
      const int tpc = rank_split(nb);
      const int i = tid / tpc, part = tid % tpc;
      int r = 0;
      Kept me{};
      if (i < nb) {
        me = s_bk[i];
        for (int j = part; j < nb; j += tpc) r += sel_before(s_bk[j], me);
      }
      for (int o = tpc >> 1; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
      if (i < nb && part == 0 && r < need) s_win[r] = me;
      __syncthreads();
      for (int j = tid; j < need; j += kSelThreads)
        if (TV_IN(n_gt + j, kMaxBudget)) s_kept[n_gt + j] = s_win[j];
      k = limit;
      __syncthreads();
    } else {
      const unsigned long long T = prefix;
      for (int j = tid; j < count; j += kSelThreads) {
        const unsigned long long kj = K[j];
        if (kj > T) {
          const unsigned long long c = ws.list[j];
          const int slot = atomicAdd(&s_n, 1);
          if (TV_IN(slot, kMaxBudget)) s_kept[slot] = Kept{kj, (int)(c >> 32), (int)(c & 0xffffffffu)};
        } else if (kj == T) {
          const int slot = atomicAdd(&s_nt, 1);
          if (slot < kTieCap) s_ties[slot] = ws.list[j];
        }
      }
      __syncthreads();
      const int n_gt = s_n, n_ties = s_nt;
      if (n_ties <= kTieCap) {
        // take the `need` lowest (row, token) among the ties
        int p2 = 1;
        while (p2 < n_ties) p2 <<= 1;
        for (int i = n_ties + tid; i < p2; i += kSelThreads) s_ties[i] = ~0ull;
        __syncthreads();
        bitonic_sort_u64(s_ties, p2);
        for (int i = tid; i < need; i += kSelThreads)
          if (TV_IN(n_gt + i, kMaxBudget) && TV_IN(i, kTieCap))
            s_kept[n_gt + i] = Kept{T, (int)(s_ties[i] >> 32), (int)(s_ties[i] & 0xffffffffu)};
      } else {
        // very many exact ties: pick them one by one in (row, token) order
        unsigned long long last = 0ull;
        bool first = true;
        for (int r = 0; r < need; ++r) {
          if (tid == 0) s_min = ~0ull;
          __syncthreads();
          unsigned long long mine = ~0ull;
          for (int j = tid; j < count; j += kSelThreads) {
            const unsigned long long c = ws.list[j];
            if ((first || c > last) && c < mine && K[j] == T) mine = c;
          }
          atomicMin(&s_min, mine);
          __syncthreads();
          last = s_min;
          first = false;
          if (tid == 0 && TV_IN(n_gt + r, kMaxBudget))
            s_kept[n_gt + r] = Kept{T, (int)(last >> 32), (int)(last & 0xffffffffu)};
          __syncthreads();
        }
      }
      k = limit;
      __syncthreads();
    }
  }
  // the output order (parent asc, score desc, token asc).  Up to 1024 kept:
  // each candidate's position is the number of kept candidates before it,
  // counted by rank_split(k) threads over interleaved shares; the positions
  // are distinct (the order is total) and the candidates land in s_stage,
  // whose keys are no longer needed.  More: a bitonic sort in place.
  const Kept* ordered = s_kept;
  if (k <= kSelThreads) {
    Kept* s_ord = reinterpret_cast<Kept*>(s_stage);
    const int tpc = rank_split(k);
    const int i = tid / tpc, part = tid % tpc;
    int pos = 0;
    Kept me{};
    if (i < k) {
      me = s_kept[i];
      for (int j = part; j < k; j += tpc) pos += out_before(s_kept[j], me);
    }
    for (int o = tpc >> 1; o > 0; o >>= 1) pos += __shfl_xor_sync(0xffffffffu, pos, o);
    if (i < k && part == 0 && TV_IN(pos, k)) s_ord[pos] = me;
    __syncthreads();
    ordered = s_ord;
  } else {
    int p2 = 1;
    while (p2 < k) p2 <<= 1;
    for (int i = k + tid; i < p2; i += kSelThreads) s_kept[i] = Kept{0ull, INT_MAX, INT_MAX};
    __syncthreads();
    bitonic_sort_kept<true>(s_kept, p2);
  }
  const int n0 = ctl.n0;
  for (int i = tid; i < k; i += kSelThreads) {
    const Kept c = ordered[i];
    if (!(TV_IN(c.row, F) && TV_IN(c.token, V) && TV_IN(n0 + i, budget))) continue;
    tree_parent[n0 + i] = frontier_node[c.row];
    tree_token[n0 + i] = c.token;
    // the key is the order-preserving image of the fp64 score off + logit the
    // filter formed: the score itself, without reading the logit again
    tree_logscore[n0 + i] = (float)key_double(c.key);
  }
  if (tid == 0) {
    *n_nodes = n0 + k;
    ws.ctl->count = 0;   // the next call starts from zero
    ws.ctl->anchor = 0ull;
    ws.ctl->floor = 0ull;
  }
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_expand_workspace_size(int F, int V) {
  if (F <= 0 || V <= 0) return 256;
  size_t a, b, c, d, e;
  return tv::exp_offsets(F, V, &a, &b, &c, &d, &e);
}

namespace tv {
namespace {

// The three launches of one layer; the caller has checked the arguments.
tv_status launch_layer(const float* draft_logits, const int32_t* frontier_node,
                       const float* frontier_logscore, int F, int V, int gated, int cap,
                       double log_alpha, int budget, int32_t* tree_parent, int32_t* tree_token,
                       float* tree_logscore, int32_t* n_nodes, void* workspace,
                       cudaStream_t stream) {
  size_t rows_off, part_off, cand_off, list_off, keys_off;
  exp_offsets(F, V, &rows_off, &part_off, &cand_off, &list_off, &keys_off);
  char* base = static_cast<char*>(workspace);
  ExpWs ws;
  ws.ctl = reinterpret_cast<ExpCtl*>(base);
  ws.arrivals = reinterpret_cast<unsigned int*>(base + exp_arrivals_offset());
  ws.hist = reinterpret_cast<unsigned int*>(base + exp_hist_offset());
  ws.rows = reinterpret_cast<ExpRow*>(base + rows_off);
  ws.part = reinterpret_cast<ExpPartial*>(base + part_off);
  ws.cand = reinterpret_cast<ExpCand*>(base + cand_off);
  ws.list = reinterpret_cast<unsigned long long*>(base + list_off);
  ws.keys = reinterpret_cast<unsigned long long*>(base + keys_off);
  const int chunks = ceil_div(V, kExpChunk);
  // chunks per filter CTA: a whole row once there are enough rows to fill the
  // GPU; a few rows (the root layer) spread over more CTAs, since the chunks a
  // list cannot decide are read again one after another within a CTA
  const int cpc = F >= 32 ? kFiltGroup : 4;
  // the select stages up to kSelStageKeys keys
  if (!set_dyn_smem(exp_select_kernel, (int)(kSelStageKeys * sizeof(unsigned long long))))
    return TV_ERR_CUDA;
  // OPT-Tree layers with at least `cap` chunks (every one but the root's) find
  // their floor in the statistics pass; the others launch the floor kernel
  const int fold = (!gated && (long long)F * chunks >= cap) ? 1 : 0;
  if (launch_pdl(exp_stats_kernel, dim3(ceil_div(chunks, kStatsWarps), F), dim3(kStatsWarps * 32),
                 0, stream, draft_logits, V, chunks, frontier_logscore, fold, cap, budget,
                 (const int32_t*)n_nodes, ws) != cudaSuccess ||
      (!gated && !fold && launch_pdl(exp_floor_kernel, dim3(1), dim3(kFloorThreads), 0, stream,
                            draft_logits, V, F, chunks, cap, budget, (const int32_t*)n_nodes,
                            ws) != cudaSuccess) ||
      launch_pdl(exp_filter_kernel, dim3(ceil_div(chunks, cpc), F), dim3(kExpThreads), 0,
                 stream, draft_logits, V, cpc, gated,
                 cap, budget, log_alpha, (const int32_t*)n_nodes, ws) != cudaSuccess ||
      launch_pdl(exp_select_kernel, dim3(1), dim3(kSelThreads),
                 (size_t)kSelStageKeys * sizeof(unsigned long long), stream, draft_logits, V, F,
                 budget, frontier_node, tree_parent, tree_token, tree_logscore, n_nodes,
                 ws) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}

// Checks shared by both entry points (F == 0 has already returned).
tv_status check_layer(const float* draft_logits, const int32_t* frontier_node,
                      const float* frontier_logscore, int F, int V, int32_t* tree_parent,
                      int32_t* tree_token, float* tree_logscore, int32_t* n_nodes,
                      void* workspace, size_t ws_bytes) {
  if (!draft_logits || !frontier_node || !frontier_logscore || !tree_parent || !tree_token ||
      !tree_logscore || !n_nodes)
    return TV_ERR_INVALID_ARG;
  if ((size_t)F * V >= (1ull << 31)) return TV_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < tv_expand_workspace_size(F, V)) return TV_ERR_WORKSPACE;
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(draft_logits) & 15)) return TV_ERR_INVALID_ARG;
  return TV_OK;
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_expand_gated(const float* draft_logits, const int32_t* frontier_node,
                                     const float* frontier_logscore, int F, int V, int layer,
                                     int topk, float alpha, int budget, int32_t* tree_parent,
                                     int32_t* tree_token, float* tree_logscore, int32_t* n_nodes,
                                     void* workspace, size_t ws_bytes, cudaStream_t stream) {
  TV_NVTX_RANGE("tv_expand_gated");
  if (F < 0 || V < 1 || layer < 1 || budget < 1) return TV_ERR_INVALID_ARG;
  if (budget > tv::kMaxBudget || F > tv::kMaxBudget) return TV_ERR_UNSUPPORTED;
  if (layer == 1 && (F != 1 || topk < 1)) return TV_ERR_INVALID_ARG;
  if (layer >= 2 && !(alpha > 0.0f && alpha <= 1.0f)) return TV_ERR_INVALID_ARG;
  if (F == 0) return TV_OK;
  const tv_status st = tv::check_layer(draft_logits, frontier_node, frontier_logscore, F, V,
                                       tree_parent, tree_token, tree_logscore, n_nodes, workspace,
                                       ws_bytes);
  if (st != TV_OK) return st;
  // the root layer keeps its Top-K ungated; deeper layers gate, up to the budget
  const int gated = layer >= 2;
  const int cap = gated ? INT_MAX : topk;
  return tv::launch_layer(draft_logits, frontier_node, frontier_logscore, F, V, gated, cap,
                          gated ? log((double)alpha) : 0.0, budget, tree_parent, tree_token,
                          tree_logscore, n_nodes, workspace, stream);
}

extern "C" tv_status tv_expand_topn(const float* draft_logits, const int32_t* frontier_node,
                                    const float* frontier_logscore, int F, int V, int width,
                                    int capacity, int32_t* tree_parent, int32_t* tree_token,
                                    float* tree_logscore, int32_t* n_nodes, void* workspace,
                                    size_t ws_bytes, cudaStream_t stream) {
  TV_NVTX_RANGE("tv_expand_topn");
  if (F < 0 || V < 1 || width < 1 || capacity < 1) return TV_ERR_INVALID_ARG;
  if (width > tv::kMaxBudget || F > tv::kMaxBudget) return TV_ERR_UNSUPPORTED;
  if (F == 0) return TV_OK;
  const tv_status st = tv::check_layer(draft_logits, frontier_node, frontier_logscore, F, V,
                                       tree_parent, tree_token, tree_logscore, n_nodes, workspace,
                                       ws_bytes);
  if (st != TV_OK) return st;
  return tv::launch_layer(draft_logits, frontier_node, frontier_logscore, F, V, 0, width, 0.0,
                          capacity, tree_parent, tree_token, tree_logscore, n_nodes, workspace,
                          stream);
}
