// tv_commit_path: move the accepted branch's K/V rows from their tree slots to
// consecutive cache positions (Speculative Decoding concept page, "The
// protocol" step 4: the accepted tokens and the correction extend the prefix;
// OPT-Tree §2: the accepted tokens are one root-to-node branch of the tree).
//
// One CTA per (sequence, kv head).  Row d of the branch (1 <= d <= a) moves
// from slot kv_len + path[d] to slot kv_len + d.  The path is strictly
// increasing from 0, so path[d] >= d: a destination never lies past the
// sources still to be read.  Rows move in batches; a batch reads all of its
// sources (16-byte chunks, coalesced along the row) before any thread writes
// a destination, and every later batch reads only slots past this batch's
// destinations, so the copy is exact in place.
#define TV_UNIT 6
#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kCommitThreads = 256;
constexpr int kCommitChunks = 4;  // 16-byte chunks a thread carries per batch

__global__ void __launch_bounds__(kCommitThreads)
commit_kernel(uint4* __restrict__ k, uint4* __restrict__ v, const int32_t* __restrict__ kv_len,
              const int32_t* __restrict__ path, const int32_t* __restrict__ accept_len, int N,
              int Hkv, int C /* 16-byte chunks per row */, int Lcap,
              int32_t* __restrict__ new_kv_len, int32_t* __restrict__ status) {
  __shared__ int32_t s_path[kMaxNodes];
  pdl_trigger();
  pdl_wait();  // the path and the tree rows come from earlier kernels
  const int b = blockIdx.x / Hkv, h = blockIdx.x % Hkv;
  const int tid = threadIdx.x;
  const int L = __ldg(kv_len + b), a = __ldg(accept_len + b);
  int bad = !(L >= 0 && a >= 0 && a < N && TV_CHECK(N <= kMaxNodes));
  if (!bad)
    for (int d = tid; d <= a; d += kCommitThreads) {
      const int p = __ldg(path + (size_t)b * N + d);
      s_path[d] = p;
      bad |= (d == 0) ? (p != 0) : (p >= N);
    }
  bad = __syncthreads_or(bad);
  if (!bad)
    for (int d = 1 + tid; d <= a; d += kCommitThreads) bad |= (s_path[d] <= s_path[d - 1]);
  bad = __syncthreads_or(bad);
  if (!bad) bad = (long long)L + s_path[a] >= (long long)Lcap;
  if (h == 0 && tid == 0) {
    status[b] = bad ? TV_ERR_INVALID_ARG : TV_OK;
    new_kv_len[b] = bad ? L : L + a + 1;
  }
  if (bad) return;
  const size_t base = ((size_t)b * Hkv + h) * (size_t)Lcap + (size_t)L;  // slot kv_len of this head
  const int per_row = 2 * C;                                            // K and V chunks of a row
  const int rows_per_batch = max(1, kCommitThreads * kCommitChunks / per_row);
  for (int d0 = 1; d0 <= a; d0 += rows_per_batch) {
    const int items = (min(a + 1, d0 + rows_per_batch) - d0) * per_row;
    uint4 buf[kCommitChunks];
#pragma unroll
    for (int u = 0; u < kCommitChunks; ++u) {
      const int w = tid + u * kCommitThreads;
      if (w < items) {
        const int d = d0 + w / per_row, t = (w / C) & 1, c = w % C;
        if (s_path[d] != d && TV_CHECK(s_path[d] > 0 && L + s_path[d] < Lcap))
          buf[u] = (t ? v : k)[(base + s_path[d]) * C + c];
      }
    }
    __syncthreads();  // every source of the batch is read before any destination is written
#pragma unroll
    for (int u = 0; u < kCommitChunks; ++u) {
      const int w = tid + u * kCommitThreads;
      if (w < items) {
        const int d = d0 + w / per_row, t = (w / C) & 1, c = w % C;
        if (s_path[d] != d && TV_CHECK(L + d < Lcap)) (t ? v : k)[(base + d) * C + c] = buf[u];
      }
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_commit_path(tv_bf16* k, tv_bf16* v, const int32_t* kv_len,
                                    const int32_t* path, const int32_t* accept_len, int B, int N,
                                    int Hkv, int D, int Lcap, int32_t* new_kv_len,
                                    int32_t* status, cudaStream_t stream) {
  TV_NVTX_RANGE("tv_commit_path");
  if (B < 0 || N < 1 || N > TV_MAX_NODES || Hkv < 1 || Lcap < 1) return TV_ERR_INVALID_ARG;
  if (D < 8 || D % 8 != 0 || D > 1024) return TV_ERR_UNSUPPORTED;
  if (B == 0) return TV_OK;
  if (!k || !v || !kv_len || !path || !accept_len || !new_kv_len || !status)
    return TV_ERR_INVALID_ARG;
  if (new_kv_len == kv_len) return TV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return TV_ERR_INVALID_ARG;
  if ((long long)B * Hkv > 0x7fffffffll) return TV_ERR_UNSUPPORTED;
  if (tv::launch_pdl(tv::commit_kernel, dim3((unsigned)(B * Hkv)), dim3(tv::kCommitThreads), 0,
                     stream, reinterpret_cast<uint4*>(k), reinterpret_cast<uint4*>(v), kv_len, path,
                     accept_len, N, Hkv, D / 8, Lcap, new_kv_len, status) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
