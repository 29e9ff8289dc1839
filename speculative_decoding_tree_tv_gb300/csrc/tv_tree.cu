// tv_tree_build: parent[] -> depth[] and ancestor-or-self bitmasks, the tree
// attention mask of OPT-Tree §2 (a node attends to its ancestors and itself).
#define TV_UNIT 1
#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

constexpr int kTreeThreads = 256;

// One CTA per sequence.  Each thread walks its nodes up to the root; the
// walk length is the node depth (<= N - 1), and N <= 512, so the whole tree
// costs at most N * depth shared-memory steps spread over 256 threads.
__global__ void __launch_bounds__(kTreeThreads)
tree_build_kernel(const int32_t* __restrict__ parent, int N, int W, int32_t* __restrict__ depth,
                  uint64_t* __restrict__ anc_mask, int32_t* __restrict__ status) {
  __shared__ int32_t s_par[kMaxNodes];
  __shared__ uint64_t s_anc[kMaxNodes * kMaxWords];
  pdl_trigger();
  const int b = blockIdx.x;
  const int32_t* par = parent + (size_t)b * N;
  // the parent row into the L2 while the previous kernel finishes (a hint:
  // the reads below come after the wait)
  if (threadIdx.x * 32 < N) sm100::line_prefetch_l2(par + threadIdx.x * 32);
  pdl_wait();
  int32_t* dep = depth + (size_t)b * N;
  uint64_t* anc = anc_mask + (size_t)b * N * W;

  int bad = 0;
  if (!TV_CHECK(N <= kMaxNodes && N * W <= kMaxNodes * kMaxWords)) return;
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int p = par[i];
    s_par[i] = p;
    bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
  }
  if (W > 1)
    for (int w = threadIdx.x; w < N * W; w += blockDim.x) s_anc[w] = 0ull;
  bad = __syncthreads_or(bad);
  if (bad) {
    for (int i = threadIdx.x; i < N; i += blockDim.x) dep[i] = -1;
    for (int w = threadIdx.x; w < N * W; w += blockDim.x) anc[w] = 0ull;
    if (threadIdx.x == 0) status[b] = TV_ERR_INVALID_TREE;
    return;
  }
  if (W == 1) {
    // up to 64 nodes: the mask of a node is one word, built in a register and
    // stored straight to global memory
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
      int d = -1;
      uint64_t m = 0ull;
      for (int x = i; x >= 0 && TV_IN(x, N); x = s_par[x]) {
        m |= 1ull << x;
        ++d;
      }
      dep[i] = d;
      anc[i] = m;
    }
  } else {
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
      int d = -1;
      uint64_t* row = s_anc + i * W;
      for (int x = i; x >= 0 && TV_IN(x, N); x = s_par[x]) {
        row[x >> 6] |= 1ull << (x & 63);
        ++d;
      }
      dep[i] = d;
    }
    __syncthreads();
    for (int w = threadIdx.x; w < N * W; w += blockDim.x) anc[w] = s_anc[w];
  }
  if (threadIdx.x == 0) status[b] = TV_OK;
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_tree_build(const int32_t* parent, int B, int N, int32_t* depth,
                                   uint64_t* anc_mask, int32_t* status, cudaStream_t stream) {
  TV_NVTX_RANGE("tv_tree_build");
  if (B < 0 || N < 1 || N > TV_MAX_NODES) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!parent || !depth || !anc_mask || !status) return TV_ERR_INVALID_ARG;
  const int W = tv::ceil_div(N, 64);
  if (tv::launch_pdl(tv::tree_build_kernel, dim3(B), dim3(tv::kTreeThreads), 0, stream, parent, N,
                     W, depth, anc_mask, status) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
