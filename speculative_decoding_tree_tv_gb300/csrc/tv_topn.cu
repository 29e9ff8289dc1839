// tv_select_topn: OPT-Tree's subtree selection (OPT-Tree §3: of the
// candidate tree grown layer by layer, keep the n nodes with the highest
// scores; because a node's score, the product of the draft probabilities
// along its path, never exceeds its parent's, those n nodes contain the root
// and each other's parents and so form the subtree of n nodes with the
// largest expected acceptance length).
//
// One CTA per tree, every step in shared memory:
//   1. the fp32 log scores become order-preserving 32-bit keys (-0 as +0),
//      while the parent array is checked (topological, single root);
//   2. a radix select over the keys, one byte per pass from the top, finds
//      T = the key of the k-th best node (k = min(n, nodes)) and how many of
//      the nodes scoring exactly T are taken (the lowest ids: a parent ties
//      ahead of its child);
//   3. each thread owns a contiguous run of ids; a block scan ranks the ties,
//      a second one numbers the kept nodes in id order (so the subtree stays
//      topological) and the new numbers overwrite the keys;
//   4. every kept node writes its renumbered parent, token, score and source
//      id; a kept node whose parent was cut (scores that rise along a path)
//      marks the tree invalid.  The sum of exp(score) over the kept draft
//      nodes (the expected acceptance length) is reduced in fp64.
#define TV_UNIT 8
#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kTopnThreads = 1024;
constexpr int kTopnWarps = kTopnThreads / 32;
constexpr int kTopnMaxNodes = 16384;
constexpr int kTopnRun = kTopnMaxNodes / kTopnThreads;  // ids per thread at most
static_assert(kTopnRun <= 32, "a thread's kept flags fit one 32-bit word");
constexpr unsigned int kCut = 0xffffffffu;              // "not kept" in the renumbering

__device__ __forceinline__ unsigned int score_key(float f) {
  unsigned int u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v over the block (1024 threads); *total = the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = s_warp[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi - w;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + incl - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kTopnThreads)
select_topn_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                   const float* __restrict__ logscore, const int32_t* __restrict__ n_nodes, int M,
                   int n, int32_t* __restrict__ out_parent, int32_t* __restrict__ out_token,
                   float* __restrict__ out_logscore, int32_t* __restrict__ out_src,
                   float* __restrict__ expected, int32_t* __restrict__ status) {
  extern __shared__ unsigned int s_key[];  // [M]: score keys, then the new ids
  __shared__ unsigned int s_hist[256];
  __shared__ int s_warp[33];
  __shared__ double s_e[kTopnWarps];
  __shared__ int s_digit, s_need;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* par = parent + (size_t)b * M;
  const float* ls = logscore + (size_t)b * M;
  int32_t* op = out_parent + (size_t)b * n;
  int32_t* ot = out_token + (size_t)b * n;
  float* ol = out_logscore + (size_t)b * n;
  int32_t* os = out_src + (size_t)b * n;
  const int m_in = __ldg(n_nodes + b);
  int st = (m_in < 1 || m_in > M) ? TV_ERR_INVALID_ARG : TV_OK;
  const int m = (st == TV_OK) ? m_in : 0;  // no shared memory is touched for a bad count
  // 1. keys and checks
  int bad_tree = 0, bad_arg = 0;
  if (st == TV_OK) {
    for (int i = tid; i < m; i += kTopnThreads) {
      const int p = __ldg(par + i);
      const float f = __ldg(ls + i);
      bad_tree |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
      bad_arg |= (f != f);
      s_key[i] = score_key(f);
    }
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_arg = __syncthreads_or(bad_arg);
  if (st == TV_OK && bad_tree) st = TV_ERR_INVALID_TREE;
  if (st == TV_OK && bad_arg) st = TV_ERR_INVALID_ARG;
  const int k = (st == TV_OK) ? min(n, m) : 0;
  // 2. T = the k-th largest key; need = how many keys equal to T are kept
  unsigned int T = 0u;
  int need = 0;
  if (k > 0 && k < m) {
    unsigned int prefix = 0u, mask = 0u;
    need = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kTopnThreads) s_hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < m; i += kTopnThreads) {
        const unsigned int key = s_key[i];
        if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds digits 255 - 8l .. 248 - 8l; a scan over lanes gives
        // the count of keys above each lane's digits
        int cnt[8], lsum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = (int)s_hist[255 - 8 * lane - j];
          lsum += cnt[j];
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
          for (int j = 0; j < 8; ++j) {
            if (cum + cnt[j] >= need) {
              s_digit = 255 - 8 * lane - j;
              s_need = need - cum;
              break;
            }
            cum += cnt[j];
          }
        }
      }
      __syncthreads();
      prefix |= (unsigned int)s_digit << shift;
      mask |= 0xffu << shift;
      need = s_need;
      __syncthreads();
    }
    T = prefix;
  }
  // 3. ranks of the ties, then the new numbers, over contiguous runs of ids
  const int run = (m + kTopnThreads - 1) / kTopnThreads;
  const int lo = min(m, tid * run), hi = TV_CHECK(run <= 32) ? min(m, lo + run) : lo;
  unsigned int keep = 0u;  // bit j: id lo + j is kept
  if (k > 0) {
    if (k == m) {
      keep = (hi > lo) ? (0xffffffffu >> (32 - (hi - lo))) : 0u;
    } else {
      int ties = 0;
      for (int i = lo; i < hi; ++i) ties += (s_key[i] == T);
      int total;
      int rank = block_exclusive_scan(ties, s_warp, &total);
      for (int i = lo; i < hi; ++i) {
        const unsigned int key = s_key[i];
        bool kept = key > T;
        if (key == T) kept = rank++ < need;
        keep |= (unsigned int)kept << (i - lo);
      }
    }
  }
  __syncthreads();  // every run has been read before any is overwritten
  {
    int total;
    int id = block_exclusive_scan(__popc(keep), s_warp, &total);
    for (int i = lo; i < hi; ++i) s_key[i] = ((keep >> (i - lo)) & 1u) ? (unsigned int)id++ : kCut;
  }
  __syncthreads();
  // 4. the renumbered subtree
  int broken = 0;
  double e = 0.0;
  if (k > 0) {
    for (int i = tid; i < m; i += kTopnThreads) {
      const unsigned int j = s_key[i];
      if (j == kCut) continue;
      if (j >= (unsigned int)k) {  // cannot happen: k nodes are numbered 0..k-1
        broken = 1;
        continue;
      }
      int np = -1;
      if (i > 0) {
        const int pi = __ldg(par + i);
        const unsigned int pj = TV_IN(pi, m) ? s_key[pi] : kCut;
        broken |= (pj == kCut);
        np = (int)pj;
      }
      const float f = __ldg(ls + i);
      op[j] = np;
      ot[j] = __ldg(token + (size_t)b * M + i);
      ol[j] = f;
      os[j] = i;
      if (i > 0) e += (double)expf(f);
    }
  }
  broken = __syncthreads_or(broken);
  if (st == TV_OK && broken) st = TV_ERR_INVALID_TREE;
  const int first_blank = (st == TV_OK) ? k : 0;
  for (int j = first_blank + tid; j < n; j += kTopnThreads) {
    op[j] = -1;
    ot[j] = -1;
    ol[j] = 0.0f;
    os[j] = -1;
  }
  e = warp_sum_d(e);
  if (lane == 0) s_e[warp] = e;
  __syncthreads();
  if (tid == 0) {
    double tot = 0.0;
    for (int w = 0; w < kTopnWarps; ++w) tot += s_e[w];
    expected[b] = (st == TV_OK) ? (float)tot : 0.0f;
    status[b] = st;
  }
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_select_topn(const int32_t* parent, const int32_t* token,
                                    const float* logscore, const int32_t* n_nodes, int B, int M,
                                    int n, int32_t* out_parent, int32_t* out_token,
                                    float* out_logscore, int32_t* out_src, float* expected,
                                    int32_t* status, cudaStream_t stream) {
  TV_NVTX_RANGE("tv_select_topn");
  if (B < 0 || M < 1 || n < 1) return TV_ERR_INVALID_ARG;
  if (M > tv::kTopnMaxNodes) return TV_ERR_UNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!parent || !token || !logscore || !n_nodes || !out_parent || !out_token || !out_logscore ||
      !out_src || !expected || !status)
    return TV_ERR_INVALID_ARG;
  // up to 64 KB of keys
  if (!tv::set_dyn_smem(tv::select_topn_kernel, (int)(tv::kTopnMaxNodes * sizeof(unsigned int))))
    return TV_ERR_CUDA;
  if (tv::launch_pdl(tv::select_topn_kernel, dim3((unsigned)B), dim3(tv::kTopnThreads),
                     (size_t)M * sizeof(unsigned int), stream, parent, token, logscore, n_nodes, M,
                     n, out_parent, out_token, out_logscore, out_src, expected,
                     status) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
