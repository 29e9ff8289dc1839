// tv_accept_sample: stochastic, lossless acceptance over a verified tree
// (Speculative Decoding concept page, "The protocol" step 3: accept with
// probability min(1, p/q), resample from the normalised (p - q)+ on
// rejection; the accepted sequence follows the target exactly).
//
// One launch: a thread-block cluster of 8 CTAs (16 for vocabularies above
// 204,800) per sequence walks that sequence's tree.  CTA `rank` owns a slice
// of the vocabulary and keeps, for the node being visited, the slice of p and
// q in shared memory.  Visiting a node loads its two rows once (16-byte
// loads, all in flight), forms the softmax normalisers from cluster-wide
// maxima and sums, and turns the cached slice into probabilities; every
// rejection is then one in-place update of the cached residual, and the
// final draw an inverse-CDF search across the cluster.  Only the rows of the
// nodes the walk visits are ever read.
//
// All CTAs of a cluster take the same decisions from the same inputs (the
// accept tests in fp64 by each CTA's thread 0, the normalisers from sums
// combined in rank order), so they follow the same walk; sums over a row are
// exchanged through distributed shared memory, one cluster barrier each.
// Element values are fp32 (expf); every sum is carried in fp64 across
// threads and CTAs and every decision (accept test, draw) is taken in fp64.
#include <climits>

#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

constexpr int kWalkThreads = 512;
constexpr int kMaxCluster = 16;
constexpr int kMaxRejects = kMaxNodes;
constexpr size_t kWalkCacheMax = 200 * 1024;  // shared memory for the cached slice

// Vocabulary slice of a CTA and its per-thread runs, so that (rank, thread)
// order is token order: slice [rank * S, (rank + 1) * S), thread t the P
// tokens [t * P, (t + 1) * P) of it; S and P multiples of 4.
struct Slicing {
  int S, P;
};
__host__ __device__ inline Slicing slicing(int V, int cluster) {
  Slicing s;
  s.S = ((ceil_div(V, cluster) + 3) / 4) * 4;
  s.P = ((ceil_div(s.S, kWalkThreads) + 3) / 4) * 4;
  return s;
}
__host__ __device__ inline size_t cache_bytes(int V, int cluster) {
  return (size_t)2 * slicing(V, cluster).P * kWalkThreads * sizeof(float);
}
// 8 CTAs per tree when the cache fits, else 16, else 0 (unsupported).
inline int walk_cluster(int V) {
  if (cache_bytes(V, 8) <= kWalkCacheMax) return 8;
  if (cache_bytes(V, 16) <= kWalkCacheMax) return 16;
  return 0;
}

struct RowNorm {
  float m;       // row max of logit / T
  float inv_s;   // 1 / sum exp(a - m), rounded to fp32
  double s;      // sum exp(a - m)
};

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
__device__ __forceinline__ DF df_of(const KahanF& k) {  // k.s - k.c
  return df_add(DF{k.s, 0.0f}, DF{-k.c, 0.0f});
}
__device__ __forceinline__ DF df_shfl_xor(DF a, int o) {
  return DF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ DF df_shfl_up(DF a, int o) {
  return DF{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}

// Block-wide sum over kWalkThreads threads (fixed order); every thread gets
// the result as a double.
__device__ double block_sum_df(DF v, DF* scratch, double* out) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  const int tid = threadIdx.x;
  __syncthreads();
  if ((tid & 31) == 0) scratch[tid >> 5] = v;
  __syncthreads();
  if (tid < 32) {
    DF w = (tid < kWalkThreads / 32) ? scratch[tid] : DF{0.0f, 0.0f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = df_add(w, df_shfl_xor(w, o));
    if (tid == 0) *out = (double)w.hi + (double)w.lo;
  }
  __syncthreads();
  return *out;
}
__device__ float block_max_f(float v, float* scratch) {
  v = warp_max(v);
  const int tid = threadIdx.x;
  __syncthreads();
  if ((tid & 31) == 0) scratch[tid >> 5] = v;
  __syncthreads();
  if (tid < 32) {
    float w = (tid < kWalkThreads / 32) ? scratch[tid] : -INFINITY;
    w = warp_max(w);
    if (tid == 0) scratch[32] = w;
  }
  __syncthreads();
  return scratch[32];
}

// Loads this thread's tokens [t0, t1) of a row pair and calls
// fn(k, p_logit, q_logit) with k = index of the token in the run, up to 32
// tokens per round with every load of the round in flight (16-byte loads when
// the rows are 16-byte aligned; t0 is then a multiple of 4).
template <class Fn>
__device__ __forceinline__ void load_run(const float* prow, const float* qrow, int t0, int t1,
                                         bool vec, Fn&& fn) {
  constexpr int kTile = 32;
  for (int base = t0; base < t1; base += kTile) {
    float pa[kTile], qa[kTile];
    if (vec) {
#pragma unroll
      for (int u = 0; u < kTile / 4; ++u) {
        const int e = base + 4 * u;
        const float4 x = (e < t1) ? ld_stream_f4(reinterpret_cast<const float4*>(prow + e))
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const float4 y = (e < t1) ? ld_stream_f4(reinterpret_cast<const float4*>(qrow + e))
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        pa[4 * u] = x.x; pa[4 * u + 1] = x.y; pa[4 * u + 2] = x.z; pa[4 * u + 3] = x.w;
        qa[4 * u] = y.x; qa[4 * u + 1] = y.y; qa[4 * u + 2] = y.z; qa[4 * u + 3] = y.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kTile; ++u) {
        const int e = base + u;
        pa[u] = (e < t1) ? __ldg(prow + e) : 0.0f;
        qa[u] = (e < t1) ? __ldg(qrow + e) : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < kTile; ++u)
      if (base + u < t1) fn(base + u - t0, pa[u], qa[u]);
  }
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__global__ void __launch_bounds__(kWalkThreads)
walk_kernel(const float* __restrict__ p_logits, const float* __restrict__ q_logits,
            const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
            const int32_t* __restrict__ depth, int N, int V, float inv_t, uint64_t seed,
            uint64_t offset, int32_t* __restrict__ accept_len, int32_t* __restrict__ end_node,
            int32_t* __restrict__ path, int32_t* __restrict__ out_token,
            int32_t* __restrict__ status) {
  // this CTA's slice of the visited node's rows, [2][P][kWalkThreads]:
  // p-side (logit / T, then the residual r) and q-side (logit / T, then q),
  // element-major so that the threads of a warp hit distinct banks
  extern __shared__ float s_cache[];
  __shared__ int32_t s_par[kMaxNodes], s_dep[kMaxNodes];
  __shared__ int32_t s_first[kMaxNodes], s_next[kMaxNodes];  // children lists, index order
  __shared__ int32_t s_kids[kMaxNodes];                      // children of the visited node
  __shared__ float s_kp[kMaxNodes], s_kq[kMaxNodes];         // their tokens' logits
  __shared__ int s_nkids;
  __shared__ RowNorm s_pn, s_qn;
  __shared__ float s_invz[kMaxRejects];
  __shared__ double s_red[33];
  __shared__ DF s_redd[kWalkThreads / 32];
  __shared__ DF s_scan[kWalkThreads / 32];
  __shared__ float s_redf[33];
  __shared__ int s_found, s_last_pos;
  // what this CTA shows the cluster: two phases, so that writing the next
  // value never races with another CTA still reading the previous one
  __shared__ double s_pub_d[2][2];
  __shared__ int s_pub_i[2];
  __shared__ double s_all_d[kMaxCluster][2];
  __shared__ int s_all_i[kMaxCluster];
  pdl_trigger();
  pdl_wait();
  const int cl = (int)cluster_nctarank();
  const int rank = (int)sm100::cluster_ctarank();
  const int b = blockIdx.x / cl;
  const int tid = threadIdx.x;
  int phase = 0;
  // publish (d0, d1, i), wait for the cluster, read everyone's in rank order
  auto exchange = [&](double d0, double d1, int i) {
    if (tid == 0) {
      s_pub_d[phase][0] = d0;
      s_pub_d[phase][1] = d1;
      s_pub_i[phase] = i;
    }
    sm100::cluster_sync();
    if (tid < cl) {
      const uint32_t a = sm100::dsmem_map(sm100::smem_u32(&s_pub_d[phase][0]), tid);
      s_all_d[tid][0] = sm100::dsmem_ld_f64(a);
      s_all_d[tid][1] = sm100::dsmem_ld_f64(a + 8);
      s_all_i[tid] = sm100::dsmem_ld_s32(sm100::dsmem_map(sm100::smem_u32(&s_pub_i[phase]), tid));
    }
    __syncthreads();
    phase ^= 1;
  };

  const int32_t* par = parent + (size_t)b * N;
  const int32_t* tok = tokens + (size_t)b * N;
  int bad_tree = 0, bad_tok = 0;
  for (int i = tid; i < N; i += kWalkThreads) {
    const int p = par[i];
    s_par[i] = p;
    s_dep[i] = depth[(size_t)b * N + i];
    bad_tree |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    if (i > 0) bad_tok |= (tok[i] < 0 || tok[i] >= V);
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

  if (tid == 0) {
    for (int i = 0; i < N; ++i) s_first[i] = -1;
    for (int c = N - 1; c >= 1; --c) {
      s_next[c] = s_first[s_par[c]];
      s_first[s_par[c]] = c;
    }
  }
  __syncthreads();

  const bool vec = (V & 3) == 0;
  const Slicing sl = slicing(V, cl);
  const int s_lo = min(V, rank * sl.S), s_hi = min(V, s_lo + sl.S);
  const int t0 = min(s_hi, s_lo + tid * sl.P), t1 = min(s_hi, t0 + sl.P);
  const int nmine = t1 - t0;
  float* s_r = s_cache;
  float* s_q = s_cache + (size_t)sl.P * kWalkThreads;
  auto at = [&](int k) { return (size_t)k * kWalkThreads + tid; };

  int node = 0;
  int result = -1;
  for (;;) {
    const float* prow = p_logits + ((size_t)b * N + node) * V;
    const float* qrow = q_logits + ((size_t)b * N + node) * V;
    // ---- visit: the children's logits for the accept tests, fetched while the
    // slice loads; softmax normalisers from cluster-wide maxima and sums
    if (tid == 0) {
      int n = 0;
      for (int c = s_first[node]; c >= 0; c = s_next[c]) s_kids[n++] = c;
      s_nkids = n;
    }
    __syncthreads();
    const int nkids = s_nkids;
    for (int j = tid; j < nkids; j += kWalkThreads) {
      const int x = tok[s_kids[j]];
      s_kp[j] = __ldg(prow + x);
      s_kq[j] = __ldg(qrow + x);
    }
    float mp = -INFINITY, mq = -INFINITY;
    load_run(prow, qrow, t0, t1, vec, [&](int k, float a, float bq) {
      const float x = a * inv_t, y = bq * inv_t;
      s_r[at(k)] = x;
      s_q[at(k)] = y;
      mp = fmaxf(mp, x);
      mq = fmaxf(mq, y);
    });
    mp = block_max_f(mp, s_redf);
    mq = block_max_f(mq, s_redf);
    exchange((double)mp, (double)mq, 0);
    float Mp = -INFINITY, Mq = -INFINITY;
    for (int r = 0; r < cl; ++r) {
      Mp = fmaxf(Mp, (float)s_all_d[r][0]);
      Mq = fmaxf(Mq, (float)s_all_d[r][1]);
    }
    // exponentials once, kept in the cache; their sums
    KahanF sp, sq;
    for (int k = 0; k < nmine; ++k) {
      const float ep = expf(s_r[at(k)] - Mp), eq = expf(s_q[at(k)] - Mq);
      s_r[at(k)] = ep;
      s_q[at(k)] = eq;
      sp.add(ep);
      sq.add(eq);
    }
    const double sp_cta = block_sum_df(df_of(sp), s_redd, &s_red[32]);
    const double sq_cta = block_sum_df(df_of(sq), s_redd, &s_red[32]);
    exchange(sp_cta, sq_cta, 0);
    if (tid == 0) {  // fp64 runs at a small fraction of the fp32 rate: once per CTA
      double Sp = 0.0, Sq = 0.0;
      for (int r = 0; r < cl; ++r) {
        Sp += s_all_d[r][0];
        Sq += s_all_d[r][1];
      }
      s_pn = RowNorm{Mp, (float)(1.0 / Sp), Sp};
      s_qn = RowNorm{Mq, (float)(1.0 / Sq), Sq};
    }
    __syncthreads();
    const RowNorm pn = s_pn, qn = s_qn;
    // the slice as probabilities: r = p, q
    for (int k = 0; k < nmine; ++k) {
      s_r[at(k)] *= pn.inv_s;
      s_q[at(k)] *= qn.inv_s;
    }
    int n_rej = 0;    // residual normalisations so far
    int applied = 0;  // of them applied to s_r
    // calls fn(token, r, q) for this thread's tokens in token order, r brought
    // up to date (n_rej updates r <- (r - q)+ / Z_j)
    auto visit = [&](auto&& fn) {
      for (int k = 0; k < nmine; ++k) {
        float r = s_r[at(k)];
        const float q = s_q[at(k)];
        if (applied < n_rej) {
          for (int j = applied; j < n_rej; ++j) r = fmaxf(r - q, 0.0f) * s_invz[j];
          s_r[at(k)] = r;
        }
        fn(t0 + k, r, q);
      }
      applied = n_rej;
    };
    int accepted = -1;
    int ordinal = 0;
    for (int kid = 0; kid < nkids; ++kid) {
      const int c = s_kids[kid];
      // accept test in fp64 on the single token x
      if (tid == 0) {
        const double ax = (double)(s_kp[kid] * inv_t);
        const double bx = (double)(s_kq[kid] * inv_t);
        double r = exp(ax - (double)pn.m) / pn.s;
        const double qx = exp(bx - (double)qn.m) / qn.s;
        for (int j = 0; j < n_rej; ++j) r = fmax(r - qx, 0.0) * (double)s_invz[j];
        const double u = decision_uniform(seed, offset, b, node, 0u, (uint32_t)ordinal);
        s_found = (qx == 0.0) || (u < r / qx);
      }
      __syncthreads();
      if (s_found) {
        accepted = c;
        break;
      }
      // rejection: Z = sum_t (r(t) - q(t))+ over the row, from every CTA's slice
      KahanF acc;
      visit([&](int, float r, float q) { acc.add(fmaxf(r - q, 0.0f)); });
      const double zc = block_sum_df(df_of(acc), s_redd, &s_red[32]);
      exchange(zc, 0.0, 0);
      double z = 0.0;
      for (int r = 0; r < cl; ++r) z += s_all_d[r][0];
      if (z > 0.0 && n_rej < kMaxRejects) {
        if (tid == 0) s_invz[n_rej] = (float)(1.0 / z);
        ++n_rej;
      }
      __syncthreads();
      ++ordinal;
    }
    if (accepted >= 0) {
      node = accepted;
      continue;
    }
    // final draw from the current residual (p_node itself when nothing was rejected)
    KahanF acc;
    int last_pos = -1;
    visit([&](int t, float r, float) {
      acc.add(r);
      if (r > 0.0f) last_pos = t;
    });
    // exclusive scan of per-thread masses inside the CTA (compensated pairs)
    // the scan adds the same per-thread values the boundary test and the
    // replay use (the compensated sums' leading parts), so that the runs'
    // intervals tile [0, total) without gaps or overlaps
    const DF dmass = DF{acc.s, 0.0f};
    const double mass = (double)acc.s;
    DF incl = dmass;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const DF y = df_shfl_up(incl, o);
      if (lane >= o) incl = df_add(incl, y);
    }
    if (lane == 31) s_scan[warp] = incl;
    if (tid == 0) {
      s_found = -1;
      s_last_pos = -1;
    }
    __syncthreads();
    if (warp == 0) {
      const DF w = (lane < kWalkThreads / 32) ? s_scan[lane] : DF{0.0f, 0.0f};
      DF wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const DF y = df_shfl_up(wi, o);
        if (lane >= o) wi = df_add(wi, y);
      }
      // exclusive prefix of warp totals; this CTA's mass
      if (lane < kWalkThreads / 32) s_scan[lane] = df_add(wi, DF{-w.hi, -w.lo});
      if (lane == kWalkThreads / 32 - 1) s_red[32] = (double)wi.hi + (double)wi.lo;
    }
    atomicMax(&s_last_pos, last_pos);
    __syncthreads();
    // the cluster's masses and last positive tokens, in rank order
    exchange(s_red[32], 0.0, s_last_pos);
    double before_cta = 0.0, total = 0.0;
    int last_all = -1;
    for (int r = 0; r < cl; ++r) {
      if (r < rank) before_cta += s_all_d[r][0];
      total += s_all_d[r][0];
      last_all = max(last_all, s_all_i[r]);
    }
    const double u = decision_uniform(seed, offset, b, node, 1u, 0u);
    const double target = u * total;
    const DF excl = df_add(incl, DF{-dmass.hi, -dmass.lo});  // this thread's exclusive prefix
    const double before = before_cta + ((double)s_scan[warp].hi + (double)s_scan[warp].lo) +
                          ((double)excl.hi + (double)excl.lo);
    if (mass > 0.0 && before + mass > target && before <= target) {
      // This run holds the boundary (the lowest such run wins if rounding
      // makes several).  Replaying the run's compensated sum in the same
      // order ends exactly at `mass`, so the search always finds a token.
      KahanF run;
      int pick = -1;
      visit([&](int t, float r, float) {
        if (pick >= 0) return;
        run.add(r);
        if (before + (double)run.s > target) pick = t;
      });
      if (pick >= 0) atomicMin(reinterpret_cast<unsigned int*>(&s_found), (unsigned int)pick);
    }
    __syncthreads();
    // the lowest pick of the cluster, else the last token with positive mass
    exchange(0.0, 0.0, s_found);
    int pick = -1;
    for (int r = 0; r < cl; ++r)
      if (s_all_i[r] >= 0 && (pick < 0 || s_all_i[r] < pick)) pick = s_all_i[r];
    result = (pick >= 0) ? pick : last_all;
    break;
  }
  // no CTA may leave while another still reads its shared memory
  sm100::cluster_sync();
  if (rank != 0) return;
  const int end_depth = s_dep[node];
  for (int i = tid; i < N; i += kWalkThreads)
    if (i > end_depth) pth[i] = -1;
  if (tid == 0) {
    for (int x = node, d = end_depth; x >= 0; x = s_par[x], --d) pth[d] = x;
    accept_len[b] = end_depth;
    end_node[b] = node;
    out_token[b] = result;
    status[b] = TV_OK;
  }
}

// The walk kernel as clusters of `cl` CTAs, with programmatic dependent launch.
template <typename... Args>
cudaError_t launch_walk(int B, int cl, size_t smem, cudaStream_t stream, Args... args) {
  static bool attrs_set = false;
  if (!attrs_set) {
    cudaError_t e = cudaFuncSetAttribute(walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kWalkCacheMax);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(walk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attrs_set = true;
  }
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
  return cudaLaunchKernelEx(&cfg, walk_kernel, args...);
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
