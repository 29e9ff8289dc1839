// tv_expected_accept: the expected acceptance length of a draft tree
// (OPT-Tree §3: a node's score is the product of the draft probabilities
// along its path from the root; the expected acceptance length is
// approximated by the sum of the scores of the tree's draft nodes).
//
// One CTA per tree.  The path products come from pointer jumping in shared
// memory: after round r a node holds the product over itself and its
// 2^r - 1 nearest ancestors (node 0 contributes 1) and points to its 2^r-th
// ancestor, so ceil(log2 N) rounds give every node its whole path.  The sum
// over draft nodes is reduced per warp in fp32 and across warps in fp64.
#define TV_UNIT 7
#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kExpectThreads = 512;  // one node per thread (N <= 512)

__global__ void __launch_bounds__(kExpectThreads)
expected_kernel(const int32_t* __restrict__ parent, const float* __restrict__ prob, int N,
                float* __restrict__ score, float* __restrict__ expected,
                int32_t* __restrict__ status) {
  __shared__ int32_t s_jump[2][kMaxNodes];
  __shared__ float s_prod[2][kMaxNodes];
  __shared__ float s_warp[kExpectThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  const bool in = i < N && TV_CHECK(N <= kMaxNodes);
  int bad_tree = 0, bad_prob = 0;
  if (in) {
    const int p = __ldg(parent + (size_t)b * N + i);
    const float q = (i == 0) ? 1.0f : __ldg(prob + (size_t)b * N + i);
    bad_tree = (i == 0) ? (p != -1) : (p < 0 || p >= i);
    bad_prob = !(q >= 0.0f && q <= 1.0f);
    s_jump[0][i] = (i == 0) ? -1 : p;
    s_prod[0][i] = q;
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_prob = __syncthreads_or(bad_prob);
  if (bad_tree || bad_prob) {
    if (in && score) score[(size_t)b * N + i] = 0.0f;
    if (i == 0) {
      expected[b] = 0.0f;
      status[b] = bad_tree ? TV_ERR_INVALID_TREE : TV_ERR_INVALID_ARG;
    }
    return;
  }
  int cur = 0;
  for (int span = 1; span < N; span <<= 1) {
    if (in) {
      int j = s_jump[cur][i];
      if (!TV_CHECK(j < i)) j = -1;
      s_prod[cur ^ 1][i] = (j < 0) ? s_prod[cur][i] : s_prod[cur][i] * s_prod[cur][j];
      s_jump[cur ^ 1][i] = (j < 0) ? -1 : s_jump[cur][j];
    }
    __syncthreads();
    cur ^= 1;
  }
  const float sc = in ? s_prod[cur][i] : 0.0f;
  if (in && score) score[(size_t)b * N + i] = sc;
  const float w = warp_sum((in && i > 0) ? sc : 0.0f);
  if ((i & 31) == 0) s_warp[i >> 5] = w;
  __syncthreads();
  if (i == 0) {
    double e = 0.0;
    for (int k = 0; k < kExpectThreads / 32; ++k) e += (double)s_warp[k];
    expected[b] = (float)e;
    status[b] = TV_OK;
  }
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_expected_accept(const int32_t* parent, const float* prob, int B, int N,
                                        float* score, float* expected, int32_t* status,
                                        cudaStream_t stream) {
  TV_NVTX_RANGE("tv_expected_accept");
  if (B < 0 || N < 1 || N > TV_MAX_NODES) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!parent || !prob || !expected || !status) return TV_ERR_INVALID_ARG;
  if (tv::launch_pdl(tv::expected_kernel, dim3((unsigned)B), dim3(tv::kExpectThreads), 0, stream,
                     parent, prob, N, score, expected, status) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
