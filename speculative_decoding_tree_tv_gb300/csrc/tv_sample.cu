// tv_accept_sample: stochastic, lossless acceptance over a verified tree
// (Speculative Decoding concept page, "The protocol" step 3: accept with
// probability min(1, p/q), resample from the normalised (p - q)+ on
// rejection; the accepted sequence follows the target exactly).
//
// Two launches on the caller's stream:
//   1. row_stats_kernel streams every p and q row once (8192 logits per CTA)
//      and leaves per-chunk (max, sum exp) partials in the workspace;
//   2. walk_kernel, one cluster of 8 CTAs per sequence, combines the partials
//      of the rows it visits into fp64 normalisers and walks the tree.  A
//      rejection triggers one pass over the node's row (each CTA an eighth
//      of it) to normalise the next residual; the final draw is an
//      inverse-CDF search over the residual across the cluster.
// Element values are fp32 (expf); every sum is carried in fp64 and every
// decision (accept test, draw) is taken in fp64.
#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

constexpr int kStatThreads = 256;
constexpr int kStatChunk = 8192;
constexpr int kWalkThreads = 512;
constexpr int kWalkCluster = 8;  // CTAs per tree in the walk
constexpr int kWalkTile = 32;    // tokens a walk thread holds per round
constexpr int kMaxRejects = kMaxNodes;

struct RowPartial {
  double s;  // sum of exp(a - m) over the chunk, a = logit / T
  float m;   // chunk max of a
  float pad;
};

__global__ void __launch_bounds__(kStatThreads)
row_stats_kernel(const float* __restrict__ p_logits, const float* __restrict__ q_logits, int rows,
                 int V, int chunks, float inv_t, RowPartial* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x / chunks;
  const int chunk = blockIdx.x % chunks;
  const int which = blockIdx.y;  // 0: p, 1: q
  const float* x = (which ? q_logits : p_logits) + (size_t)row * V;
  const int start = chunk * kStatChunk;
  const int stop = min(V, start + kStatChunk);
  const int tid = threadIdx.x;
  constexpr int kPer = kStatChunk / kStatThreads;  // 32 values per thread
  float a[kPer];
  if ((V & 3) == 0) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll
    for (int u = 0; u < kPer / 4; ++u) {
      const int e = start + 4 * (tid + u * kStatThreads);
      float4 f = (e < stop) ? ld_stream_f4(x4 + (e >> 2))
                            : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      a[4 * u + 0] = f.x * inv_t;
      a[4 * u + 1] = f.y * inv_t;
      a[4 * u + 2] = f.z * inv_t;
      a[4 * u + 3] = f.w * inv_t;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = start + tid + u * kStatThreads;
      a[u] = (e < stop) ? __ldg(x + e) * inv_t : -INFINITY;
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < kPer; ++u) m = fmaxf(m, a[u]);
  __shared__ float s_m[kStatThreads / 32];
  __shared__ double s_s[kStatThreads / 32];
  m = warp_max(m);
  if ((tid & 31) == 0) s_m[tid >> 5] = m;
  __syncthreads();
  m = s_m[0];
#pragma unroll
  for (int w = 1; w < kStatThreads / 32; ++w) m = fmaxf(m, s_m[w]);
  float s = 0.0f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) s += (a[u] == -INFINITY) ? 0.0f : expf(a[u] - m);
  double sd = warp_sum_d((double)s);
  if ((tid & 31) == 0) s_s[tid >> 5] = sd;
  __syncthreads();
  if (tid == 0) {
    double tot = 0.0;
#pragma unroll
    for (int w = 0; w < kStatThreads / 32; ++w) tot += s_s[w];
    RowPartial r;
    r.s = tot;
    r.m = m;
    r.pad = 0.0f;
    part[((size_t)which * rows + row) * chunks + chunk] = r;
  }
}

// Block-wide fp64 sum over kWalkThreads threads (fixed order); every thread
// gets the result.
__device__ double block_sum_d(double v, double* scratch) {
  v = warp_sum_d(v);
  const int tid = threadIdx.x;
  __syncthreads();
  if ((tid & 31) == 0) scratch[tid >> 5] = v;
  __syncthreads();
  if (tid < 32) {
    double w = (tid < kWalkThreads / 32) ? scratch[tid] : 0.0;
    w = warp_sum_d(w);
    if (tid == 0) scratch[32] = w;
  }
  __syncthreads();
  return scratch[32];
}

struct RowNorm {
  float m;       // row max of logit / T
  float inv_s;   // 1 / sum exp(a - m), rounded to fp32
  double s;      // sum exp(a - m)
};

// Chunk partials -> row normaliser.  The chunk scale factors are fp32
// exponentials (a few ulp; fp64 runs at a small fraction of the fp32 rate),
// the sum is fp64.
__device__ RowNorm combine_partials(const RowPartial* p, int chunks) {
  RowNorm r;
  float m = -INFINITY;
  for (int c = 0; c < chunks; ++c) m = fmaxf(m, p[c].m);
  double s = 0.0;
  for (int c = 0; c < chunks; ++c) s += p[c].s * (double)expf(p[c].m - m);
  r.m = m;
  r.s = s;
  r.inv_s = (float)(1.0 / s);
  return r;
}

// The residual chain of one token: r = p, then r <- (r - q)+ / Z_j for each
// rejection so far (Z_j its normaliser).
__device__ __forceinline__ float residual(float a, float bq, float inv_t, const RowNorm& pn,
                                          const RowNorm& qn, int n_rej, const float* invz,
                                          float* q_out) {
  float r = expf(a * inv_t - pn.m) * pn.inv_s;
  const float q = expf(bq * inv_t - qn.m) * qn.inv_s;
  for (int j = 0; j < n_rej; ++j) r = fmaxf(r - q, 0.0f) * invz[j];
  *q_out = q;
  return r;
}

// Calls fn(token, p_logit, q_logit) for the tokens [t0, t1) in order, loading
// up to kWalkTile of them at a time (all loads of a round in flight; 16-byte
// loads when the rows are 16-byte aligned and t0 is a multiple of 4).
template <class Fn>
__device__ __forceinline__ void for_tokens(const float* prow, const float* qrow, int t0, int t1,
                                           bool vec, Fn&& fn) {
  for (int base = t0; base < t1; base += kWalkTile) {
    float pa[kWalkTile], qa[kWalkTile];
    if (vec) {
#pragma unroll
      for (int u = 0; u < kWalkTile / 4; ++u) {
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
      for (int u = 0; u < kWalkTile; ++u) {
        const int e = base + u;
        pa[u] = (e < t1) ? __ldg(prow + e) : 0.0f;
        qa[u] = (e < t1) ? __ldg(qrow + e) : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < kWalkTile; ++u)
      if (base + u < t1) fn(base + u, pa[u], qa[u]);
  }
}

// One tree per thread-block cluster of kWalkCluster CTAs.  CTA `rank` owns
// the vocabulary slice [rank * S, (rank + 1) * S) and, inside it, thread t a
// contiguous run of P tokens, so (rank, thread) order is token order.  Every
// CTA takes the same decisions from the same inputs (the accept tests in
// fp64 by its thread 0, the normalisers from cluster-wide sums added in rank
// order), so all of them follow the same walk; sums over the row are
// exchanged through distributed shared memory, one cluster barrier each.
__global__ void __launch_bounds__(kWalkThreads)
walk_kernel(const float* __restrict__ p_logits, const float* __restrict__ q_logits,
            const int32_t* __restrict__ tokens, const int32_t* __restrict__ parent,
            const int32_t* __restrict__ depth, int N, int V, int chunks, float inv_t,
            uint64_t seed, uint64_t offset, const RowPartial* __restrict__ part,
            int32_t* __restrict__ accept_len, int32_t* __restrict__ end_node,
            int32_t* __restrict__ path, int32_t* __restrict__ out_token,
            int32_t* __restrict__ status) {
  pdl_trigger();
  pdl_wait();
  const int rank = (int)sm100::cluster_ctarank();
  const int b = blockIdx.x / kWalkCluster;
  const int tid = threadIdx.x;
  const int rows = (gridDim.x / kWalkCluster) * N;
  __shared__ int32_t s_par[kMaxNodes], s_dep[kMaxNodes];
  __shared__ float s_invz[kMaxRejects];
  __shared__ double s_red[33];
  __shared__ RowNorm s_pn, s_qn;
  __shared__ int s_found, s_last_pos;
  __shared__ double s_scan[kWalkThreads / 32];
  // what this CTA shows the cluster: two phases, so that writing the next
  // value never races with another CTA still reading the previous one
  __shared__ double s_pub_d[2];
  __shared__ int s_pub_i[2];
  __shared__ double s_all_d[kWalkCluster];
  __shared__ int s_all_i[kWalkCluster];
  int phase = 0;
  // publish (d, i), wait for the cluster, read everyone's in rank order
  auto exchange = [&](double d, int i) {
    if (tid == 0) {
      s_pub_d[phase] = d;
      s_pub_i[phase] = i;
    }
    sm100::cluster_sync();
    if (tid < kWalkCluster) {
      s_all_d[tid] = sm100::dsmem_ld_f64(sm100::dsmem_map(sm100::smem_u32(&s_pub_d[phase]), tid));
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

  const bool vec = (V & 3) == 0;
  const int S = ((ceil_div(V, kWalkCluster) + 3) / 4) * 4;
  const int P = ((ceil_div(S, kWalkThreads) + 3) / 4) * 4;
  const int s_lo = min(V, rank * S), s_hi = min(V, s_lo + S);
  const int t0 = min(s_hi, s_lo + tid * P), t1 = min(s_hi, t0 + P);

  int node = 0;
  int result = -1;
  for (;;) {
    const float* prow = p_logits + ((size_t)b * N + node) * V;
    const float* qrow = q_logits + ((size_t)b * N + node) * V;
    if (tid == 0) {
      s_pn = combine_partials(part + ((size_t)0 * rows + (size_t)b * N + node) * chunks, chunks);
      s_qn = combine_partials(part + ((size_t)1 * rows + (size_t)b * N + node) * chunks, chunks);
    }
    __syncthreads();
    const RowNorm pn = s_pn, qn = s_qn;
    int n_rej = 0;  // residual normalisations applied so far
    int accepted = -1;
    int ordinal = 0;
    for (int c = node + 1; c < N; ++c) {
      if (s_par[c] != node) continue;
      // accept test in fp64 on the single token x
      if (tid == 0) {
        const int x = tok[c];
        const double ax = (double)(__ldg(prow + x) * inv_t);
        const double bx = (double)(__ldg(qrow + x) * inv_t);
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
      for_tokens(prow, qrow, t0, t1, vec, [&](int, float a, float bq) {
        float q;
        const float r = residual(a, bq, inv_t, pn, qn, n_rej, s_invz, &q);
        acc.add(fmaxf(r - q, 0.0f));
      });
      const double zc = block_sum_d((double)acc.s, s_red);
      exchange(zc, 0);
      double z = 0.0;
      for (int r = 0; r < kWalkCluster; ++r) z += s_all_d[r];
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
    for_tokens(prow, qrow, t0, t1, vec, [&](int t, float a, float bq) {
      float q;
      const float r = residual(a, bq, inv_t, pn, qn, n_rej, s_invz, &q);
      acc.add(r);
      if (r > 0.0f) last_pos = t;
    });
    // exclusive scan of per-thread masses (fp64) inside the CTA
    const double mass = (double)acc.s;
    double incl = mass;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_scan[warp] = incl;
    if (tid == 0) {
      s_found = -1;
      s_last_pos = -1;
    }
    __syncthreads();
    if (warp == 0) {
      double w = (lane < kWalkThreads / 32) ? s_scan[lane] : 0.0;
      double wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < kWalkThreads / 32) s_scan[lane] = wi - w;  // exclusive prefix of warp totals
      if (lane == kWalkThreads / 32 - 1) s_red[32] = wi;    // this CTA's mass
    }
    atomicMax(&s_last_pos, last_pos);
    __syncthreads();
    // the cluster's masses and last positive tokens, in rank order
    exchange(s_red[32], s_last_pos);
    double before_cta = 0.0, total = 0.0;
    int last_all = -1;
    for (int r = 0; r < kWalkCluster; ++r) {
      if (r < rank) before_cta += s_all_d[r];
      total += s_all_d[r];
      last_all = max(last_all, s_all_i[r]);
    }
    const double u = decision_uniform(seed, offset, b, node, 1u, 0u);
    const double target = u * total;
    const double before = before_cta + s_scan[warp] + (incl - mass);
    if (mass > 0.0 && before + mass > target && before <= target) {
      // This slice holds the boundary (the lowest such slice wins if rounding
      // makes several).  Replaying the slice's compensated sum in the same
      // order ends exactly at `mass`, so the search always finds a token.
      KahanF run;
      int pick = -1;
      for_tokens(prow, qrow, t0, t1, vec, [&](int t, float a, float bq) {
        if (pick >= 0) return;
        float q;
        const float r = residual(a, bq, inv_t, pn, qn, n_rej, s_invz, &q);
        run.add(r);
        if (before + (double)run.s > target) pick = t;
      });
      if (pick >= 0) atomicMin(reinterpret_cast<unsigned int*>(&s_found), (unsigned int)pick);
    }
    __syncthreads();
    // the lowest pick of the cluster, else the last token with positive mass
    exchange(0.0, s_found);
    int pick = -1;
    for (int r = 0; r < kWalkCluster; ++r)
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

// The walk kernel as clusters of kWalkCluster CTAs, with programmatic
// dependent launch.
template <typename... Args>
cudaError_t launch_walk(dim3 grid, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kWalkCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, walk_kernel, args...);
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_accept_sample_workspace_size(int B, int N, int V) {
  if (B <= 0 || N <= 0 || V <= 0) return 256;
  const int chunks = tv::ceil_div(V, tv::kStatChunk);
  return tv::align_up((size_t)2 * B * N * chunks * sizeof(tv::RowPartial), 256);
}

extern "C" tv_status tv_accept_sample(const float* p_logits, const float* q_logits,
                                      const int32_t* tokens, const int32_t* parent,
                                      const int32_t* depth, int B, int N, int V,
                                      float temperature, uint64_t seed, uint64_t offset,
                                      int32_t* accept_len, int32_t* end_node, int32_t* path,
                                      int32_t* out_token, int32_t* status, void* workspace,
                                      size_t ws_bytes, cudaStream_t stream) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1) return TV_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!p_logits || !q_logits || !tokens || !parent || !depth || !accept_len || !end_node ||
      !path || !out_token || !status)
    return TV_ERR_INVALID_ARG;
  if ((size_t)B * N * tv::ceil_div(V, tv::kStatChunk) > 0x7fffffffu) return TV_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < tv_accept_sample_workspace_size(B, N, V)) return TV_ERR_WORKSPACE;
  if ((V & 3) == 0 && ((reinterpret_cast<uintptr_t>(p_logits) | reinterpret_cast<uintptr_t>(q_logits)) & 15))
    return TV_ERR_INVALID_ARG;
  const int chunks = tv::ceil_div(V, tv::kStatChunk);
  const float inv_t = 1.0f / temperature;
  auto* part = static_cast<tv::RowPartial*>(workspace);
  dim3 g1(chunks * B * N, 2);
  if (tv::launch_pdl(tv::row_stats_kernel, g1, dim3(tv::kStatThreads), 0, stream, p_logits,
                     q_logits, B * N, V, chunks, inv_t, part) != cudaSuccess ||
      tv::launch_walk(dim3(B * tv::kWalkCluster), stream, p_logits, q_logits, tokens, parent,
                      depth, N, V, chunks, inv_t, seed, offset, (const tv::RowPartial*)part,
                      accept_len, end_node, path, out_token, status) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
