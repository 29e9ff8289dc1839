// tv_accept_sample: stochastic, lossless acceptance over a verified tree
// (Speculative Decoding concept page, "The protocol" step 3: accept with
// probability min(1, p/q), resample from the normalised (p - q)+ on
// rejection; the accepted sequence follows the target exactly).
//
// One launch: a thread-block cluster of 8 CTAs (16 for vocabularies above
// 204,800) per sequence walks that sequence's tree (when there are more trees
// than clusters resident at once, the clusters take them deepest first).  CTA `rank` owns a slice
// of the vocabulary and keeps, for the node being visited, its slice of the p
// and q rows in shared memory, token-major; thread t owns the float4 groups
// t, t + 512, t + 1024, ... of the slice, so global and shared accesses are
// both contiguous across a warp.  A visit
//   * brings the node's two row slices in by bulk copies (rows 16-byte
//     aligned; plain coalesced loads otherwise) and asks the L2 for the first
//     child's slices, the likeliest next visit (the root's slices are asked
//     for before the dependent-launch wait);
//   * forms the softmax normalisers with one cluster exchange: every CTA
//     publishes its slice's (max, sum of exp(x - max)) and each combines the
//     pairs, one lane per rank, in the same butterfly order;
//   * computes, one thread per child, p(x) and q(x) of every child's token
//     for the accept tests;
//   * tests the children in index order; a rejection is one pass that sums
//     (r - q)+ over the slice (the update of r itself is applied lazily by
//     the next pass) and one cluster exchange of the sums.
// The final draw gives each thread a contiguous run of the slice, scans the
// runs' masses across the CTA, exchanges the slices' masses, and only the run
// holding the target replays its tokens.  The cached slice holds exp(x - its
// maximum); the factors that make it r and q are applied where it is read, so
// a visit whose first child is accepted never rescales it.
//
// All CTAs of a cluster take the same decisions from the same inputs (accept
// tests by each CTA's thread 0 from the exchanged normalisers; the draw's
// owner from the exchanged masses), so they follow the same walk.  Element
// values are fp32; sums across threads and CTAs are compensated fp32 pairs
// (TwoSum), combined in a fixed order.  fp64 runs at a small fraction of the
// fp32 rate on this part, so it is used only where the 53-bit uniform meets a
// probability: the accept comparison and the draw's target.
#define TV_UNIT 3
#include <climits>
#include <map>
#include <mutex>
#include <tuple>
#include <cstdlib>

#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kMaxRejects = kMaxNodes;
constexpr int kMaxRounds = 16;                // float4 groups per thread and row slice
constexpr size_t kWalkCacheMax = 200 * 1024;  // shared memory for the two row slices

// Tokens in the slice of each CTA (a multiple of 4): CTA `rank` owns
// [rank * S, min(V, (rank + 1) * S)).
__host__ __device__ inline int slice_len(int V, int cluster) {
  return ((ceil_div(V, cluster) + 3) / 4) * 4;
}
__host__ __device__ inline size_t cache_bytes(int V, int cluster) {
  return (size_t)2 * slice_len(V, cluster) * sizeof(float);
}
inline bool walk_cluster_fits(int V, int cl) {
  return cache_bytes(V, cl) <= kWalkCacheMax &&
         ceil_div(slice_len(V, cl) / 4, kWalkThreads) <= kMaxRounds;
}
// Trees a walk launch orders by depth (more than the clusters resident at once).
constexpr int kMaxOrderTrees = 64;

// 8 CTAs per tree when the slices fit, else 16, else 0 (unsupported).  The
// environment variable TV_WALK_CLUSTER=16 (or 8) replaces the choice where
// the slices fit, for tests and tuning; it is read on every call.
inline int walk_cluster(int V) {
  const char* e = getenv("TV_WALK_CLUSTER");
  if (e) {
    const int want = atoi(e);
    if ((want == 8 || want == 16) && walk_cluster_fits(V, want)) return want;
  }
  for (int cl = 8; cl <= kMaxCluster; cl *= 2)
    if (walk_cluster_fits(V, cl)) return cl;
  return 0;
}

// Sums across threads as unevaluated pairs hi + lo of fp32 values, each
// addition exact up to the last bits of lo (Knuth's TwoSum), so about twice
// the fp32 precision at fp32 speed; fp64 runs at a small fraction of the
// fp32 rate on this part.
struct DF {
  float hi, lo;
};
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const float s = a.hi + b.hi;
  const float v = s - a.hi;
  float e = (a.hi - (s - v)) + (b.hi - v);
  e += a.lo + b.lo;
  const float hi = s + e;
  return DF{hi, e - (hi - s)};
}
__device__ __forceinline__ double df_val(DF a) { return (double)a.hi + (double)a.lo; }
__device__ __forceinline__ DF df_of_double(double d) {
  const float hi = (float)d;
  return DF{hi, (float)(d - (double)hi)};
}
// Order of normalised pairs (|lo| at most half an ulp of hi, as df_add leaves them).
__device__ __forceinline__ bool df_le(DF a, DF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo <= b.lo);
}
__device__ __forceinline__ bool df_lt(DF a, DF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}
// DF times a float (TwoProd by fma), normalised.
__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const float p = a.hi * b;
  const float e = fmaf(a.hi, b, -p) + a.lo * b;
  const float hi = p + e;
  return DF{hi, e - (hi - p)};
}
constexpr float kLog2e = 1.4426950408889634f;
// 2^x on the special-function unit (ex2.approx.ftz): relative error about
// 2^-22, below the fp32 rounding of the probabilities it makes.
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ DF df_shfl_xor(DF a, int o) {
  return DF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ DF df_shfl_up(DF a, int o) {
  return DF{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  return v;
}
// Inclusive prefix over the lanes of a warp.
__device__ __forceinline__ DF warp_scan_df(DF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y = df_shfl_up(v, o);
    if (lane >= o) v = df_add(v, y);
  }
  return v;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void dsmem_st_s32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Ask the L2 for `bytes` (a multiple of 16, 16-byte aligned) of global memory.

__global__ void __launch_bounds__(kWalkThreads)
walk_kernel(const float* __restrict__ p_logits, const float* __restrict__ q_logits,
            const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
            const int32_t* __restrict__ depth, int N, int V, float inv_t, uint64_t seed,
            uint64_t offset, int32_t* __restrict__ accept_len, int32_t* __restrict__ end_node,
            int32_t* __restrict__ path, int32_t* __restrict__ out_token,
            int32_t* __restrict__ status, int order_trees) {
  // this CTA's slices of the visited node's rows, token-major: p side (logit,
  // then probability, then residual), then q side
  extern __shared__ __align__(16) float s_cache[];
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int32_t s_par[kMaxNodes], s_dep[kMaxNodes], s_tok[kMaxNodes], s_kids[kMaxNodes];
  __shared__ float s_kpx[kMaxNodes], s_kqx[kMaxNodes];  // p(x), q(x) of each child's token
  __shared__ float s_invz[kMaxRejects];
  __shared__ int s_wcount[kWalkWarps];
  __shared__ float s_wmax[2][kWalkWarps];
  __shared__ DF s_wsum[2][kWalkWarps];
  __shared__ DF s_wtot[kWalkWarps];  // draw: each warp's mass, then the mass before it
  __shared__ float s_norm[4];  // 1/S_p, 1/S_q, M_p, M_q
  __shared__ float s_scale[2];  // this slice's factors exp(m - M) / S
  __shared__ DF s_lt;           // draw: the slice's mass, then the target minus the mass
                                // before this slice (owner only)
  __shared__ int s_found, s_zpos, s_last, s_result;
  __shared__ int s_err;
  // what this CTA shows the cluster: two phases, so that writing the next
  // value never races with another CTA still reading the previous one
  __shared__ __align__(16) float s_pub_f[2][8];
  __shared__ int s_pub_i[2];
  __shared__ __align__(16) float s_all_f[kMaxCluster][8];
  __shared__ int s_all_i[kMaxCluster];
  pdl_trigger();
  const int cl = (int)cluster_nctarank();
  const int rank = (int)sm100::cluster_ctarank();
  int b = blockIdx.x / cl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool bulk = (V & 3) == 0;
  const int S = slice_len(V, cl);
  const int s_lo = min(V, rank * S), s_hi = min(V, s_lo + S);
  const uint32_t slice_bytes = (uint32_t)(s_hi - s_lo) * 4u;
  // Every walk starts at the root: its two slices, and the tree arrays, into
  // the L2 while the previous kernel finishes.  A prefetch changes no result
  // (the loads proper come after the wait and read the L2, where the
  // previous kernel's writes land).
  if (bulk && tid == 0 && slice_bytes > 0) {
    sm100::bulk_prefetch_l2(p_logits + (size_t)b * N * V + s_lo, slice_bytes);
    sm100::bulk_prefetch_l2(q_logits + (size_t)b * N * V + s_lo, slice_bytes);
  }
  if (tid * 32 < N) {
    sm100::line_prefetch_l2(parent + (size_t)b * N + tid * 32);
    sm100::line_prefetch_l2(tokens + (size_t)b * N + tid * 32);
    sm100::line_prefetch_l2(depth + (size_t)b * N + tid * 32);
  }
  pdl_wait();
  if (order_trees) {
    // More trees than clusters fit on the GPU at once: the clusters that
    // start first take the deepest trees (a walk visits at most depth + 1
    // nodes), ties to the lower index, so that the ones left for the
    // clusters that start late are the shortest.  Every CTA of a cluster
    // computes the same permutation from the same depth arrays.
    __shared__ int s_maxdep[kMaxOrderTrees];
    __shared__ int s_b;
    const int nb = (int)gridDim.x / cl;
    for (int i = tid; i < nb; i += kWalkThreads) s_maxdep[i] = 0;
    if (tid == 0) s_b = b;
    __syncthreads();
    for (int i = tid; i < nb * N; i += kWalkThreads)
      if (TV_IN(i / N, kMaxOrderTrees)) atomicMax(&s_maxdep[i / N], __ldg(depth + i));
    __syncthreads();
    for (int t = tid; t < nb; t += kWalkThreads) {
      int r = 0;
      for (int u = 0; u < nb; ++u)
        r += (s_maxdep[u] > s_maxdep[t]) || (s_maxdep[u] == s_maxdep[t] && u < t);
      if (r == b) s_b = t;  // b is still this cluster's position
    }
    __syncthreads();
    b = s_b;
  }
  int phase = 0;
  // publish eight floats and an int, wait for the cluster, read everyone's in
  // rank order
  auto exchange = [&](float4 a, float4 c, int i) {
    if (tid == 0) {
      *reinterpret_cast<float4*>(&s_pub_f[phase][0]) = a;
      *reinterpret_cast<float4*>(&s_pub_f[phase][4]) = c;
      s_pub_i[phase] = i;
    }
    sm100::cluster_sync();
    if (tid < 2 * cl) {
      const int r = tid >> 1, k = tid & 1;
      *reinterpret_cast<float4*>(&s_all_f[r][4 * k]) =
          sm100::dsmem_ld_f32x4(sm100::dsmem_map(sm100::smem_u32(&s_pub_f[phase][4 * k]), r));
      if (k == 0) s_all_i[r] = sm100::dsmem_ld_s32(sm100::dsmem_map(sm100::smem_u32(&s_pub_i[phase]), r));
    }
    __syncthreads();
    phase ^= 1;
  };

  const int32_t* par = parent + (size_t)b * N;
  const int32_t* tok = tokens + (size_t)b * N;
  if (tid == 0) {
    sm100::mbar_init(&s_bar, 1);
    sm100::mbar_fence_init();
    s_err = 0;
  }
  int bad_tree = 0, bad_tok = 0;
  for (int i = tid; i < N; i += kWalkThreads) {
    const int p = par[i];
    s_par[i] = p;
    s_dep[i] = depth[(size_t)b * N + i];
    bad_tree |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    const int x = tok[i];
    s_tok[i] = x;
    if (i > 0) bad_tok |= (x < 0 || x >= V);
  }
  bad_tree = __syncthreads_or(bad_tree);
  if (!bad_tree)
    for (int i = tid; i < N; i += kWalkThreads)
      bad_tree |= (i == 0) ? (s_dep[0] != 0) : (s_dep[i] != s_dep[s_par[i]] + 1);
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  int32_t* pth = path + (size_t)b * N;
  if (bad_tree || bad_tok) {  // the same in every CTA of the cluster: all leave here
    if (rank == 0) {
      for (int i = tid; i < N; i += kWalkThreads) pth[i] = -1;
      if (tid == 0) {
        accept_len[b] = end_node[b] = out_token[b] = -1;
        status[b] = bad_tree ? TV_ERR_INVALID_TREE : TV_ERR_INVALID_TOKEN;
      }
    }
    return;
  }

  const int n4 = (s_hi - s_lo + 3) / 4;  // float4 groups; a ragged last one is padded
  const int rounds = ceil_div(n4, kWalkThreads);
  float4* const c_p = reinterpret_cast<float4*>(s_cache);
  float4* const c_q = reinterpret_cast<float4*>(s_cache + S);
  uint32_t bar_parity = 0;

  int node = 0;
  int result = -1;
  (void)TV_CHECK(s_hi - s_lo <= S && cl <= kMaxCluster && N <= kMaxNodes);
  for (;;) {
    if (!TV_IN(node, N)) node = 0;
    const float* prow = p_logits + ((size_t)b * N + node) * V;
    const float* qrow = q_logits + ((size_t)b * N + node) * V;
    // ---- the node's two row slices into shared memory (every thread's
    // reads of the previous visit's slices are ordered before the copy)
    sm100::fence_async_smem();
    __syncthreads();
    if (bulk) {
      if (tid == 0 && slice_bytes > 0) {
        sm100::mbar_expect_tx(&s_bar, 2u * slice_bytes);
        sm100::bulk_load_global(c_p, prow + s_lo, slice_bytes, &s_bar);
        sm100::bulk_load_global(c_q, qrow + s_lo, slice_bytes, &s_bar);
      }
    } else {
      float* cp = s_cache;
      float* cq = s_cache + S;
      for (int k = tid; k < 4 * n4; k += kWalkThreads) {
        const int t = s_lo + k;
        cp[k] = (t < s_hi) ? __ldg(prow + t) : -INFINITY;
        cq[k] = (t < s_hi) ? __ldg(qrow + t) : -INFINITY;
      }
    }
    // ---- the children, in index order (one per thread: N <= kWalkThreads)
    const bool is_kid = tid > node && tid < N && s_par[tid] == node;
    const unsigned kb = __ballot_sync(0xffffffffu, is_kid);
    if (lane == 0) s_wcount[warp] = __popc(kb);
    __syncthreads();
    int before = 0, nkids = 0;
#pragma unroll
    for (int w = 0; w < kWalkWarps; ++w) {
      before += (w < warp) ? s_wcount[w] : 0;
      nkids += s_wcount[w];
    }
    if (is_kid && TV_IN(before + __popc(kb & ((1u << lane) - 1u)), N))
      s_kids[before + __popc(kb & ((1u << lane) - 1u))] = tid;
    __syncthreads();
    float kp = 0.0f, kq = 0.0f;
    if (tid < nkids) {  // the children's tokens' logits, for the accept tests
      const int x = s_tok[s_kids[tid]];
      if (TV_IN(x, V)) {
        kp = __ldg(prow + x) * inv_t;
        kq = __ldg(qrow + x) * inv_t;
      }
    }
    if (bulk && tid == 0 && nkids > 0 && slice_bytes > 0) {  // the likeliest next visit
      const size_t row1 = (size_t)b * N + s_kids[0];
      sm100::bulk_prefetch_l2(p_logits + row1 * V + s_lo, slice_bytes);
      sm100::bulk_prefetch_l2(q_logits + row1 * V + s_lo, slice_bytes);
    }
    if (bulk && slice_bytes > 0) {
      bool ok = sm100::mbar_wait(&s_bar, bar_parity);
      if (!ok) ok = sm100::mbar_wait(&s_bar, bar_parity);  // a copy must not outlive the CTA
      if (!ok) s_err = 1;
      bar_parity ^= 1u;
    } else {
      __syncthreads();
    }
    // ---- slice maxima of logit / T (inv_t > 0 keeps the order, so the
    // maximum of the scaled values is the scaled maximum)
    float mp = -INFINITY, mq = -INFINITY;
#pragma unroll 4
    for (int j = 0; j < rounds; ++j) {
      const int f = tid + j * kWalkThreads;
      if (f < n4) {
        const float4 a = c_p[f], c = c_q[f];
        mp = fmaxf(mp, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
        mq = fmaxf(mq, fmaxf(fmaxf(c.x, c.y), fmaxf(c.z, c.w)));
      }
    }
    mp = warp_max(mp) * inv_t;
    mq = warp_max(mq) * inv_t;
    if (lane == 0) {
      s_wmax[0][warp] = mp;
      s_wmax[1][warp] = mq;
    }
    __syncthreads();
    mp = -INFINITY;
    mq = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWalkWarps; ++w) {
      mp = fmaxf(mp, s_wmax[0][w]);
      mq = fmaxf(mq, s_wmax[1][w]);
    }
    // ---- exp(x - slice max), kept in place; sums per thread, then per CTA
    float sp = 0.0f, sq = 0.0f;
#pragma unroll 4
    for (int j = 0; j < rounds; ++j) {
      const int f = tid + j * kWalkThreads;
      if (f < n4) {
        float4 a = c_p[f], c = c_q[f];
        a = make_float4(ex2f(fmaf(a.x, inv_t, -mp) * kLog2e), ex2f(fmaf(a.y, inv_t, -mp) * kLog2e),
                        ex2f(fmaf(a.z, inv_t, -mp) * kLog2e), ex2f(fmaf(a.w, inv_t, -mp) * kLog2e));
        c = make_float4(ex2f(fmaf(c.x, inv_t, -mq) * kLog2e), ex2f(fmaf(c.y, inv_t, -mq) * kLog2e),
                        ex2f(fmaf(c.z, inv_t, -mq) * kLog2e), ex2f(fmaf(c.w, inv_t, -mq) * kLog2e));
        c_p[f] = a;
        c_q[f] = c;
        sp += (a.x + a.y) + (a.z + a.w);
        sq += (c.x + c.y) + (c.z + c.w);
      }
    }
    {
      const DF wp = warp_sum_df(DF{sp, 0.0f}), wq = warp_sum_df(DF{sq, 0.0f});
      if (lane == 0) {
        s_wsum[0][warp] = wp;
        s_wsum[1][warp] = wq;
      }
    }
    __syncthreads();
    DF tp{0.0f, 0.0f}, tq{0.0f, 0.0f};
    if (tid == 0)
      for (int w = 0; w < kWalkWarps; ++w) {
        tp = df_add(tp, s_wsum[0][w]);
        tq = df_add(tq, s_wsum[1][w]);
      }
    // ---- one exchange: every slice's (max, sum); normalisers in rank order
    exchange(make_float4(mp, tp.hi, tp.lo, 0.0f), make_float4(mq, tq.hi, tq.lo, 0.0f), 0);
    if (warp < 2) {  // warp 0: p, warp 1: q; lane r takes rank r's (max, sum)
      const int k = 4 * warp;
      const float m_r = (lane < cl) ? s_all_f[lane][k] : -INFINITY;
      const float M = warp_max(m_r);
      DF t{0.0f, 0.0f};
      if (lane < cl && s_all_f[lane][k + 1] > 0.0f)
        t = df_mul_f(DF{s_all_f[lane][k + 1], s_all_f[lane][k + 2]}, ex2f((m_r - M) * kLog2e));
      t = warp_sum_df(t);  // the same butterfly in every CTA: identical normalisers
      if (lane == 0) {
        const float inv = 1.0f / (t.hi + t.lo);
        const float mine = (warp == 0) ? mp : mq;
        s_norm[warp] = inv;
        s_norm[2 + warp] = M;
        s_scale[warp] = (mine == -INFINITY) ? 0.0f : ex2f((mine - M) * kLog2e) * inv;
      }
    }
    __syncthreads();
    // the children's p(x), q(x) for the accept tests; the slice itself stays
    // as exp(x - slice max) and is scaled (by s_scale) where it is read
    if (tid < nkids) {
      s_kpx[tid] = ex2f((kp - s_norm[2]) * kLog2e) * s_norm[0];
      s_kqx[tid] = ex2f((kq - s_norm[3]) * kLog2e) * s_norm[1];
    }
    __syncthreads();

    int n_rej = 0;    // residual normalisations so far
    int applied = 0;  // of them applied to the p side of the cache
    float rs = s_scale[0];        // the p side holds r / rs until a pass stores r itself
    const float qs = s_scale[1];  // the q side always holds q / qs
    // the residual r of group f (and q) with every pending normalisation
    // applied (r <- (r - q)+ / Z_j); r is stored back when `store` or when an
    // update was pending, and the pass then sets rs = 1
    auto residual = [&](int f, float4& q, bool store) {
      const float4 c = c_q[f];
      q = make_float4(c.x * qs, c.y * qs, c.z * qs, c.w * qs);
      const float4 a = c_p[f];
      float4 r = make_float4(a.x * rs, a.y * rs, a.z * rs, a.w * rs);
      if (applied < n_rej) {
        for (int j = applied; j < n_rej; ++j) {
          const float z = s_invz[j];
          r = make_float4(fmaxf(r.x - q.x, 0.0f) * z, fmaxf(r.y - q.y, 0.0f) * z,
                          fmaxf(r.z - q.z, 0.0f) * z, fmaxf(r.w - q.w, 0.0f) * z);
        }
        store = true;
      }
      if (store) c_p[f] = r;
      return r;
    };
    int accepted = -1;
    for (int kid = 0; kid < nkids; ++kid) {
      // accept test in fp64 on the child's token x
      if (tid == 0) {
        float r = s_kpx[kid];
        const float qx = s_kqx[kid];
        for (int j = 0; j < n_rej; ++j) r = fmaxf(r - qx, 0.0f) * s_invz[j];
        const double u = decision_uniform(seed, offset, b, node, 0u, (uint32_t)kid);
        s_found = (qx == 0.0f) || (u < (double)(r / qx));
      }
      __syncthreads();
      if (s_found) {
        accepted = s_kids[kid];
        break;
      }
      // rejection: Z = sum_t (r(t) - q(t))+ over the row, from every CTA's slice
      float zs = 0.0f;
#pragma unroll 4
      for (int j = 0; j < rounds; ++j) {
        const int f = tid + j * kWalkThreads;
        if (f < n4) {
          float4 q;
          const float4 r = residual(f, q, false);
          zs += (fmaxf(r.x - q.x, 0.0f) + fmaxf(r.y - q.y, 0.0f)) +
                (fmaxf(r.z - q.z, 0.0f) + fmaxf(r.w - q.w, 0.0f));
        }
      }
      if (applied < n_rej) rs = 1.0f;  // uniform: every group was stored
      applied = n_rej;
      {
        const DF wz = warp_sum_df(DF{zs, 0.0f});
        if (lane == 0) s_wsum[0][warp] = wz;
      }
      __syncthreads();
      DF tz{0.0f, 0.0f};
      if (tid == 0)
        for (int w = 0; w < kWalkWarps; ++w) tz = df_add(tz, s_wsum[0][w]);
      exchange(make_float4(tz.hi, tz.lo, 0.0f, 0.0f), make_float4(0.0f, 0.0f, 0.0f, 0.0f), 0);
      if (tid == 0) {
        DF z{0.0f, 0.0f};
        for (int r = 0; r < cl; ++r) z = df_add(z, DF{s_all_f[r][0], s_all_f[r][1]});
        const float zf = z.hi + z.lo;
        s_zpos = (zf > 0.0f) ? 1 : 0;
        if (zf > 0.0f && n_rej < kMaxRejects) s_invz[n_rej] = 1.0f / zf;
      }
      __syncthreads();
      if (s_zpos && n_rej < kMaxRejects) ++n_rej;  // z <= 0 leaves r as it is
    }
    if (accepted >= 0) {
      node = accepted;
      continue;
    }
    // ---- final draw from the current residual (p_node itself when nothing
    // was rejected).  For the draw, thread t takes a contiguous run of the
    // slice, float4 groups [t P4, (t + 1) P4), so token order is (rank,
    // thread, group, element).  It reads its groups in an order rotated by t
    // (conflict-free), stores r itself, and sums its run as a float pair; a
    // block-wide scan of the runs gives every thread [lo, hi), and the runs
    // tile the slice exactly.
    const int P4 = ceil_div(n4, kWalkThreads);
    DF run{0.0f, 0.0f};
    int last_pos = -1;
    for (int k = 0; k < P4; ++k) {
      const int g = tid * P4 + (k + tid) % P4;
      if (g < n4) {
        float4 q;
        const float4 r = residual(g, q, true);
        run = df_add(run, DF{(r.x + r.y) + (r.z + r.w), 0.0f});
        const int t = s_lo + 4 * g;
        const int lp = (r.w > 0.0f) ? t + 3 : (r.z > 0.0f) ? t + 2 : (r.y > 0.0f) ? t + 1
                                                                      : (r.x > 0.0f) ? t : -1;
        last_pos = max(last_pos, lp);
      }
    }
    applied = n_rej;
    rs = 1.0f;
    const DF incl = warp_scan_df(run);
    const DF excl = DF{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
    if (lane == 31) s_wtot[warp] = incl;
    if (tid == 0) {
      s_last = -1;
      s_result = -1;
    }
    __syncthreads();
    last_pos = __reduce_max_sync(0xffffffffu, last_pos);
    if (lane == 0) atomicMax(&s_last, last_pos);
    if (warp == 0) {  // mass before each warp's runs, and the slice's mass
      DF base{0.0f, 0.0f};
      for (int w = 0; w < kWalkWarps; ++w) {
        const DF tw = s_wtot[w];
        __syncwarp();
        if (lane == 0) s_wtot[w] = base;
        base = df_add(base, tw);
      }
      if (lane == 0) s_lt = base;  // the slice's mass, until the exchange
    }
    __syncthreads();
    const DF wbase = s_wtot[warp];
    const DF lo = (lane == 0) ? wbase : df_add(wbase, excl);
    const DF hi = df_add(wbase, incl);
    // the slices' masses and last positive tokens, in rank order
    exchange(make_float4(s_lt.hi, s_lt.lo, 0.0f, 0.0f), make_float4(0.0f, 0.0f, 0.0f, 0.0f), s_last);
    if (tid == 0) {
      DF before_cta{0.0f, 0.0f}, total{0.0f, 0.0f};
      int last_all = -1;
      for (int r = 0; r < cl; ++r) {
        const DF m_r{s_all_f[r][0], s_all_f[r][1]};
        if (r < rank) before_cta = df_add(before_cta, m_r);
        total = df_add(total, m_r);
        last_all = max(last_all, s_all_i[r]);
      }
      // the target u * total, formed once in fp64 and held as a float pair
      const DF target = df_of_double(decision_uniform(seed, offset, b, node, 1u, 0u) * df_val(total));
      const DF mine{s_all_f[rank][0], s_all_f[rank][1]};
      s_found = (mine.hi > 0.0f && df_le(before_cta, target) && df_lt(target, df_add(before_cta, mine)))
                    ? 1 : 0;
      s_lt = df_add(target, DF{-before_cta.hi, -before_cta.lo});
      s_last = last_all;
    }
    __syncthreads();
    if (s_found) {  // this slice holds the target: the run holding it replays its tokens
      const DF lt = s_lt;
      if (df_lt(lo, hi) && df_le(lo, lt) && df_lt(lt, hi)) {
        DF cum = lo;
        int pick = -1, last_mine = -1;
        for (int g = tid * P4; g < min(n4, (tid + 1) * P4); ++g) {
          const float4 r = c_p[g];
          const float e[4] = {r.x, r.y, r.z, r.w};
          for (int k = 0; k < 4; ++k) {
            if (!(e[k] > 0.0f)) continue;
            last_mine = s_lo + 4 * g + k;
            cum = df_add(cum, DF{e[k], 0.0f});
            if (pick < 0 && df_lt(lt, cum)) pick = last_mine;
          }
        }
        if (pick < 0) pick = last_mine;  // rounding at the run's end: its last token with mass
        dsmem_st_s32(sm100::dsmem_map(sm100::smem_u32(&s_result), 0), pick);
      }
    }
    result = -2;  // rank 0 reads s_result after the final cluster barrier
    break;
  }
  // no CTA may leave while another still reads its shared memory; the draw's
  // pick reaches rank 0 before this barrier.  A CTA whose copy timed out
  // reports it after rank 0 has written the status.
  if (rank == 0 && tid == 0) status[b] = s_err ? TV_ERR_TIMEOUT : TV_OK;
  sm100::cluster_sync();
  if (rank != 0) {
    if (tid == 0 && s_err) atomicMax(status + b, (int)TV_ERR_TIMEOUT);
    return;
  }
  if (result == -2) result = (s_result >= 0) ? s_result : s_last;
  if (!TV_IN(result, V)) result = -1;
  const int end_depth = s_dep[node];
  for (int i = tid; i < N; i += kWalkThreads)
    if (i > end_depth) pth[i] = -1;
  if (tid == 0) {
    for (int x = node, d = end_depth; x >= 0 && TV_IN(d, N) && TV_IN(x, N); x = s_par[x], --d)
      pth[d] = x;
    accept_len[b] = end_depth;
    end_node[b] = node;
    out_token[b] = result;
  }
}

// The walk kernel as clusters of `cl` CTAs, with programmatic dependent launch.
// Clusters of `cl` walk CTAs (with `smem` bytes each) the device holds at
// once, per device and shape (0 if the query fails).
int resident_walk_clusters(int cl, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> cache;
  const auto key = std::make_tuple(current_device(), cl, smem);
  std::lock_guard<std::mutex> lock(mu);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cl * kMaxOrderTrees), 1, 1);
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)cl;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, walk_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[key] = n;
  return n;
}

template <typename... Args>
cudaError_t launch_walk(int B, int cl, size_t smem, cudaStream_t stream, Args... args) {
  if (!set_dyn_smem(walk_kernel, (int)kWalkCacheMax) ||
      !set_func_attr(reinterpret_cast<const void*>(walk_kernel),
                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1))
    return cudaErrorInvalidValue;
  // deepest trees first when some clusters must wait for others to finish
  const int resident = resident_walk_clusters(cl, smem);
  const int order_trees = (resident > 0 && B > resident && B <= kMaxOrderTrees) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * cl), 1, 1);
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, walk_kernel, args..., order_trees);
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_accept_sample_workspace_size(int B, int N, int V) {
  (void)B;
  (void)N;
  (void)V;
  return 0;
}

extern "C" tv_status tv_accept_sample(const float* p_logits, const float* q_logits,
                                      const int32_t* tokens, const int32_t* parent,
                                      const int32_t* depth, int B, int N, int V,
                                      float temperature, uint64_t seed, uint64_t offset,
                                      int32_t* accept_len, int32_t* end_node, int32_t* path,
                                      int32_t* out_token, int32_t* status, void* workspace,
                                      size_t ws_bytes, cudaStream_t stream) {
  TV_NVTX_RANGE("tv_accept_sample");
  (void)workspace;
  (void)ws_bytes;
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1) return TV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!p_logits || !q_logits || !tokens || !parent || !depth || !accept_len || !end_node ||
      !path || !out_token || !status)
    return TV_ERR_INVALID_ARG;
  const int cl = tv::walk_cluster(V);
  if (cl == 0 || (long long)B * cl > 0x7fffffffll) return TV_ERR_UNSUPPORTED;
  if ((V & 3) == 0 && ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits)) & 15))
    return TV_ERR_INVALID_ARG;
  const float inv_t = 1.0f / temperature;
  if (tv::launch_walk(B, cl, tv::cache_bytes(V, cl), stream, p_logits, q_logits, tokens, parent,
                      depth, N, V, inv_t, seed, offset, accept_len, end_node, path, out_token,
                      status) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
