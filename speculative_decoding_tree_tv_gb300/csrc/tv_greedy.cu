// tv_accept_greedy: vocabulary-streaming argmax over every tree node's
// target logits, then the longest matching branch (OPT-Tree §2: under greedy
// sampling the longest branch matching the target's highest-probability
// sequence is accepted; GOOSE §2C greedy walk).
//
// One launch.  CTA (chunk, row) streams 8192 logits of one row with 16-byte
// non-allocating loads, reduces them to (max, lowest index) and folds that
// into the row's 64-bit key (order-preserving float bits, inverted index)
// with atomicMax.  The CTA that finishes a sequence last (per-sequence
// arrival counter) runs the tree scan for it:
//   match[i] = tokens[i] == argmax[parent[i]],
//   valid[i] = AND of match over the root path (pointer jumping),
//   end      = deepest valid node, ties to the lowest index,
// and returns the workspace to zero (keys swapped out with atomicExch, the
// counter reset).
#include <climits>

#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kGreedyThreads = 256;
constexpr int kGreedyChunk = 8192;  // logits per CTA: 8 float4 per thread
constexpr int kScanNodesPerThread = (kMaxNodes + kGreedyThreads - 1) / kGreedyThreads;

struct GreedyWs {
  unsigned long long* keys;  // [B*N]
  unsigned int* arrivals;    // [B]
};

__host__ __device__ inline size_t greedy_keys_bytes(int B, int N) {
  return align_up((size_t)B * N * sizeof(unsigned long long), 256);
}

__device__ __forceinline__ unsigned long long pack_key(ArgMax a) {
  return ((unsigned long long)float_key(a.v) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)a.i);
}

__global__ void __launch_bounds__(kGreedyThreads)
greedy_kernel(const float* __restrict__ logits, const int32_t* __restrict__ tokens,
              const int32_t* __restrict__ parent, const int32_t* __restrict__ depth, int N, int V,
              int chunks, int32_t* __restrict__ argmax_out, int32_t* __restrict__ accept_len,
              int32_t* __restrict__ end_node, int32_t* __restrict__ path,
              int32_t* __restrict__ bonus, int32_t* __restrict__ status, GreedyWs ws) {
  const int row = blockIdx.x / chunks;
  const int b = row / N;
  const int tid = threadIdx.x;
  const int start = (blockIdx.x % chunks) * kGreedyChunk;
  const int stop = min(V, start + kGreedyChunk);
  const float* x = logits + (size_t)row * V;

  ArgMax best{-INFINITY, INT_MAX};
  if ((V & 3) == 0) {
    // rows start 16-byte aligned: vector body, all loads issued first
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float4 buf[kGreedyChunk / (4 * kGreedyThreads)];
#pragma unroll
    for (int u = 0; u < kGreedyChunk / (4 * kGreedyThreads); ++u) {
      const int e = start + 4 * (tid + u * kGreedyThreads);
      buf[u] = (e < stop) ? ld_stream_f4(x4 + (e >> 2)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < kGreedyChunk / (4 * kGreedyThreads); ++u) {
      const int e = start + 4 * (tid + u * kGreedyThreads);
      if (e < stop) {
        if (buf[u].x > best.v) best = {buf[u].x, e};
        if (buf[u].y > best.v) best = {buf[u].y, e + 1};
        if (buf[u].z > best.v) best = {buf[u].z, e + 2};
        if (buf[u].w > best.v) best = {buf[u].w, e + 3};
      }
    }
  } else {
    for (int e = start + tid; e < stop; e += kGreedyThreads) {
      const float v = __ldg(x + e);
      if (v > best.v) best = {v, e};
    }
  }
  if (best.i == INT_MAX) best.i = start;  // all -inf: any index of the chunk, lowest first

  __shared__ ArgMax s_red[kGreedyThreads / 32];
  __shared__ int s_last;
  best = warp_argmax(best);
  if ((tid & 31) == 0) s_red[tid >> 5] = best;
  __syncthreads();
  if (tid < 32) {
    ArgMax a = (tid < kGreedyThreads / 32) ? s_red[tid] : ArgMax{-INFINITY, INT_MAX};
    a = warp_argmax(a);
    if (tid == 0) {
      atomicMax(ws.keys + row, pack_key(a));
      __threadfence();
      const unsigned int prev = atomicAdd(ws.arrivals + b, 1u);
      s_last = (prev == (unsigned int)(N * chunks - 1));
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---------------- tree scan for sequence b (last CTA only) ----------------
  __shared__ int32_t s_par[kMaxNodes], s_dep[kMaxNodes], s_am[kMaxNodes];
  __shared__ int32_t s_valid[kMaxNodes], s_jump[kMaxNodes];
  __shared__ unsigned int s_best;
  const int32_t* par = parent + (size_t)b * N;
  const int32_t* tok = tokens + (size_t)b * N;
  const int32_t* dep = depth + (size_t)b * N;
  int bad_tree = 0, bad_tok = 0;
  for (int i = tid; i < N; i += kGreedyThreads) {
    const unsigned long long key = atomicExch(ws.keys + (size_t)b * N + i, 0ull);
    const int am = (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu));
    s_am[i] = am;
    argmax_out[(size_t)b * N + i] = am;
    const int p = par[i];
    s_par[i] = p;
    s_dep[i] = dep[i];
    bad_tree |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    if (i > 0) {
      const int t = tok[i];
      bad_tok |= (t < 0 || t >= V);
    }
  }
  if (tid == 0) {
    ws.arrivals[b] = 0u;
    s_best = 0u;
  }
  bad_tree = __syncthreads_or(bad_tree);
  if (!bad_tree) {
    for (int i = tid; i < N; i += kGreedyThreads)
      bad_tree |= (i == 0) ? (s_dep[0] != 0) : (s_dep[i] != s_dep[s_par[i]] + 1);
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  int32_t* pth = path + (size_t)b * N;
  if (bad_tree || bad_tok) {
    for (int i = tid; i < N; i += kGreedyThreads) pth[i] = -1;
    if (tid == 0) {
      accept_len[b] = end_node[b] = bonus[b] = -1;
      status[b] = bad_tree ? TV_ERR_INVALID_TREE : TV_ERR_INVALID_TOKEN;
    }
    return;
  }
  for (int i = tid; i < N; i += kGreedyThreads) {
    s_valid[i] = (i == 0) ? 1 : (tok[i] == s_am[s_par[i]]);
    s_jump[i] = s_par[i];
  }
  __syncthreads();
  // pointer jumping: after r rounds s_valid[i] covers 2^r edges above i
  for (int span = 1; span < N; span <<= 1) {
    int nv[kScanNodesPerThread], nj[kScanNodesPerThread];
#pragma unroll
    for (int k = 0; k < kScanNodesPerThread; ++k) {
      const int i = tid + k * kGreedyThreads;
      if (i < N) {
        const int j = s_jump[i];
        nv[k] = s_valid[i] & (j < 0 ? 1 : s_valid[j]);
        nj[k] = j < 0 ? -1 : s_jump[j];
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kScanNodesPerThread; ++k) {
      const int i = tid + k * kGreedyThreads;
      if (i < N) {
        s_valid[i] = nv[k];
        s_jump[i] = nj[k];
      }
    }
    __syncthreads();
  }
  // deepest valid node, lowest index on ties
  unsigned int mine = 0u;
  for (int i = tid; i < N; i += kGreedyThreads)
    if (s_valid[i]) mine = max(mine, ((unsigned int)s_dep[i] << 16) | (0xffffu - (unsigned int)i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, o));
  if ((tid & 31) == 0) atomicMax(&s_best, mine);
  __syncthreads();
  const int end = (int)(0xffffu - (s_best & 0xffffu));
  const int end_depth = s_dep[end];
  for (int i = tid; i < N; i += kGreedyThreads)
    if (i > end_depth) pth[i] = -1;
  if (tid == 0) {
    for (int x2 = end, d = end_depth; x2 >= 0; x2 = s_par[x2], --d) pth[d] = x2;
    accept_len[b] = end_depth;
    end_node[b] = end;
    bonus[b] = s_am[end];
    status[b] = TV_OK;
  }
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_accept_greedy_workspace_size(int B, int N, int V) {
  (void)V;
  if (B <= 0 || N <= 0) return 256;
  return tv::greedy_keys_bytes(B, N) + tv::align_up((size_t)B * sizeof(unsigned int), 256);
}

extern "C" tv_status tv_accept_greedy(const float* logits, const int32_t* tokens,
                                      const int32_t* parent, const int32_t* depth, int B, int N,
                                      int V, int32_t* argmax, int32_t* accept_len,
                                      int32_t* end_node, int32_t* path, int32_t* bonus,
                                      int32_t* status, void* workspace, size_t ws_bytes,
                                      cudaStream_t stream) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!logits || !tokens || !parent || !depth || !argmax || !accept_len || !end_node || !path ||
      !bonus || !status)
    return TV_ERR_INVALID_ARG;
  if ((size_t)B * N * tv::ceil_div(V, tv::kGreedyChunk) > 0x7fffffffu) return TV_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < tv_accept_greedy_workspace_size(B, N, V)) return TV_ERR_WORKSPACE;
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) != 0) return TV_ERR_INVALID_ARG;
  tv::GreedyWs ws;
  ws.keys = static_cast<unsigned long long*>(workspace);
  ws.arrivals = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) +
                                                tv::greedy_keys_bytes(B, N));
  const int chunks = tv::ceil_div(V, tv::kGreedyChunk);
  dim3 grid(chunks * B * N);
  tv::greedy_kernel<<<grid, tv::kGreedyThreads, 0, stream>>>(
      logits, tokens, parent, depth, N, V, chunks, argmax, accept_len, end_node, path, bonus,
      status, ws);
  TV_CHECK_LAUNCH();
  return TV_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of tv_accept_greedy.
//
// Some callers cannot allocate device memory where they need acceptance: a
// serving loop whose device memory was planned and reserved once at start-up,
// a plug-in running inside another framework's execution that is handed no
// allocator, or a real-time path where an allocation (and the synchronisation
// it may imply) is not allowed.  This entry point takes no workspace.  Its
// scratch -- one 64-bit key per node row and one arrival counter per sequence
// -- lives in a fixed-size file-scope __device__ array, which every GPU that
// loads this library holds until the process exits.
#include <mutex>

namespace tv {
namespace {

constexpr long long kStaticMaxRows = 65536;  // B * N
constexpr int kStaticMaxSeqs = 4096;         // B
constexpr size_t kStaticKeyBytes = (size_t)kStaticMaxRows * sizeof(unsigned long long);
constexpr size_t kStaticScratchBytes = kStaticKeyBytes + (size_t)kStaticMaxSeqs * sizeof(unsigned int);

__device__ __align__(256) unsigned char g_greedy_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_greedy_scratch_addr[kMaxDevices];  // device address of the array, per device
std::mutex g_greedy_scratch_mu;

}  // namespace
}  // namespace tv

extern "C" tv_status tv_accept_greedy_noalloc(const float* logits, const int32_t* tokens,
                                              const int32_t* parent, const int32_t* depth, int B,
                                              int N, int V, int32_t* argmax, int32_t* accept_len,
                                              int32_t* end_node, int32_t* path, int32_t* bonus,
                                              int32_t* status, cudaStream_t stream) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!logits || !tokens || !parent || !depth || !argmax || !accept_len || !end_node || !path ||
      !bonus || !status)
    return TV_ERR_INVALID_ARG;
  if ((long long)B * N > tv::kStaticMaxRows || B > tv::kStaticMaxSeqs) return TV_ERR_UNSUPPORTED;
  if ((size_t)B * N * tv::ceil_div(V, tv::kGreedyChunk) > 0x7fffffffu) return TV_ERR_UNSUPPORTED;
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) != 0) return TV_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  if (dev < 0 || dev >= tv::kMaxDevices) return TV_ERR_UNSUPPORTED;
  void* base = nullptr;
  {
    // first call on this device: look up where the array lives on it
    std::lock_guard<std::mutex> lock(tv::g_greedy_scratch_mu);
    if (!tv::g_greedy_scratch_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, tv::g_greedy_scratch) != cudaSuccess || !addr) {
        (void)cudaGetLastError();
        return TV_ERR_CUDA;
      }
      tv::g_greedy_scratch_addr[dev] = addr;
    }
    base = tv::g_greedy_scratch_addr[dev];
  }
  // The array keeps whatever the previous call left; the keys and counters
  // this call uses must start at zero.
  char* b8 = static_cast<char*>(base);
  if (cudaMemsetAsync(b8, 0, (size_t)B * N * sizeof(unsigned long long), stream) != cudaSuccess ||
      cudaMemsetAsync(b8 + tv::kStaticKeyBytes, 0, (size_t)B * sizeof(unsigned int), stream) !=
          cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  tv::GreedyWs ws;
  ws.keys = reinterpret_cast<unsigned long long*>(b8);
  ws.arrivals = reinterpret_cast<unsigned int*>(b8 + tv::kStaticKeyBytes);
  const int chunks = tv::ceil_div(V, tv::kGreedyChunk);
  tv::greedy_kernel<<<dim3(chunks * B * N), tv::kGreedyThreads, 0, stream>>>(
      logits, tokens, parent, depth, N, V, chunks, argmax, accept_len, end_node, path, bonus,
      status, ws);
  TV_CHECK_LAUNCH();
  return TV_OK;
}
