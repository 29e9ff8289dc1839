// tv_accept_greedy: vocabulary-streaming argmax over every tree node's
// target logits, then the longest matching branch (OPT-Tree §2: under greedy
// sampling the longest branch matching the target's highest-probability
// sequence is accepted; GOOSE §2C greedy walk).
//
// One launch.  CTA c handles work item c = (row, chunk): a contiguous chunk
// of one row's logits.  Items are numbered row-major, so the CTAs resident at
// any moment sweep one contiguous stretch of memory (which keeps every DRAM
// channel busy), and the chunk length is chosen so that all items fit in one
// wave of resident CTAs.  Each thread keeps 8 16-byte non-allocating loads in
// flight; the CTA reduces its chunk to (max, lowest index) and folds it into
// the row's 64-bit key (order-preserving float bits, inverted index) with
// atomicMax.  The CTA that completes a sequence's N * chunks arrivals runs
// that tree's scan:
//   match[i] = tokens[i] == argmax[parent[i]],
//   valid[i] = AND of match over the root path (pointer jumping),
//   end      = deepest valid node, ties to the lowest index,
// and returns the workspace to zero (keys swapped out with atomicExch,
// counter reset).  No CTA waits for another.
#include <climits>
#include <mutex>

#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kGreedyThreads = 256;
constexpr int kGreedyCtasPerSm = 4;  // resident CTAs per SM assumed when sizing chunks
constexpr int kLoadsInFlight = 8;  // vector loads per thread per batch
constexpr int kScanNodesPerThread = (kMaxNodes + kGreedyThreads - 1) / kGreedyThreads;

struct GreedyWs {
  unsigned long long* keys;  // [B*N]
  unsigned int* arrivals;    // [B]
};

struct GreedyArgs {
  const float* logits;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* depth;
  int B, N, V;
  int chunks;          // work items per row
  int chunk_units;     // vectors (or scalars) per work item
  int32_t* argmax;
  int32_t* accept_len;
  int32_t* end_node;
  int32_t* path;
  int32_t* bonus;
  int32_t* status;
  GreedyWs ws;
};

__host__ __device__ inline size_t greedy_keys_bytes(int B, int N) {
  return align_up((size_t)B * N * sizeof(unsigned long long), 256);
}

__device__ __forceinline__ unsigned long long pack_key(ArgMax a) {
  return ((unsigned long long)float_key(a.v) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)a.i);
}

// Block-wide argmax; every thread gets the result.
__device__ ArgMax block_argmax(ArgMax a, ArgMax* s_red) {
  a = warp_argmax(a);
  const int tid = threadIdx.x;
  __syncthreads();
  if ((tid & 31) == 0) s_red[tid >> 5] = a;
  __syncthreads();
  ArgMax r = s_red[0];
#pragma unroll
  for (int w = 1; w < kGreedyThreads / 32; ++w) r = argmax_combine(r, s_red[w]);
  return r;
}

// Longest matching branch of tree b (run by one CTA after every row key of b is final).
__device__ void tree_scan(const GreedyArgs& g, int b) {
  __shared__ int32_t s_par[kMaxNodes], s_dep[kMaxNodes], s_am[kMaxNodes];
  __shared__ int32_t s_valid[kMaxNodes], s_jump[kMaxNodes];
  __shared__ unsigned int s_best;
  const int tid = threadIdx.x;
  const int N = g.N;
  const int32_t* par = g.parent + (size_t)b * N;
  const int32_t* tok = g.tokens + (size_t)b * N;
  const int32_t* dep = g.depth + (size_t)b * N;
  int bad_tree = 0, bad_tok = 0;
  __syncthreads();
  for (int i = tid; i < N; i += kGreedyThreads) {
    const unsigned long long key = atomicExch(g.ws.keys + (size_t)b * N + i, 0ull);
    const int am = (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu));
    s_am[i] = am;
    g.argmax[(size_t)b * N + i] = am;
    const int p = par[i];
    s_par[i] = p;
    s_dep[i] = dep[i];
    bad_tree |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    if (i > 0) {
      const int t = tok[i];
      bad_tok |= (t < 0 || t >= g.V);
    }
  }
  if (tid == 0) {
    g.ws.arrivals[b] = 0u;
    s_best = 0u;
  }
  bad_tree = __syncthreads_or(bad_tree);
  if (!bad_tree) {
    for (int i = tid; i < N; i += kGreedyThreads)
      bad_tree |= (i == 0) ? (s_dep[0] != 0) : (s_dep[i] != s_dep[s_par[i]] + 1);
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  int32_t* pth = g.path + (size_t)b * N;
  if (bad_tree || bad_tok) {
    for (int i = tid; i < N; i += kGreedyThreads) pth[i] = -1;
    if (tid == 0) {
      g.accept_len[b] = g.end_node[b] = g.bonus[b] = -1;
      g.status[b] = bad_tree ? TV_ERR_INVALID_TREE : TV_ERR_INVALID_TOKEN;
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
    for (int x = end, d = end_depth; x >= 0; x = s_par[x], --d) pth[d] = x;
    g.accept_len[b] = end_depth;
    g.end_node[b] = end;
    g.bonus[b] = s_am[end];
    g.status[b] = TV_OK;
  }
}

// VEC = 4: rows are 16-byte aligned and read as float4; VEC = 1: scalars.
template <int VEC>
__global__ void __launch_bounds__(kGreedyThreads)
greedy_kernel(const GreedyArgs g) {
  __shared__ ArgMax s_red[kGreedyThreads / 32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the logits may come from the previous kernel
  const int U = g.V / VEC;  // units per row
  const long long row = blockIdx.x / g.chunks;
  const int base = (int)(blockIdx.x % g.chunks) * g.chunk_units;
  const int n = min(g.chunk_units, U - base);
  const int b = (int)(row / g.N);
  ArgMax best{-INFINITY, INT_MAX};
  if (VEC == 4) {
    const float4* x4 = reinterpret_cast<const float4*>(g.logits + row * (long long)g.V) + base;
    for (int k0 = 0; k0 < n; k0 += kLoadsInFlight * kGreedyThreads) {
      float4 buf[kLoadsInFlight];
#pragma unroll
      for (int j = 0; j < kLoadsInFlight; ++j) {
        const int k = k0 + j * kGreedyThreads + tid;
        buf[j] = (k < n) ? ld_stream_f4(x4 + k)
                         : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int j = 0; j < kLoadsInFlight; ++j) {
        const int k = k0 + j * kGreedyThreads + tid;
        const int e = 4 * (base + k);
        if (k < n) {
          if (buf[j].x > best.v) best = {buf[j].x, e};
          if (buf[j].y > best.v) best = {buf[j].y, e + 1};
          if (buf[j].z > best.v) best = {buf[j].z, e + 2};
          if (buf[j].w > best.v) best = {buf[j].w, e + 3};
        }
      }
    }
  } else {
    const float* x = g.logits + row * (long long)g.V + base;
    for (int k = tid; k < n; k += kGreedyThreads) {
      const float v = __ldg(x + k);
      if (v > best.v) best = {v, base + k};
    }
  }
  if (best.i == INT_MAX) best.i = VEC * base;  // only -inf seen: lowest index of the chunk
  best = block_argmax(best, s_red);
  if (tid == 0) {
    atomicMax(g.ws.keys + row, pack_key(best));
    __threadfence();
    const unsigned int prev = atomicAdd(g.ws.arrivals + b, 1u);
    s_last = (prev == (unsigned int)(g.N * g.chunks - 1));
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    tree_scan(g, b);
  }
}

tv_status launch_greedy(const GreedyArgs& in, cudaStream_t stream) {
  GreedyArgs g = in;
  const int VEC = ((g.V & 3) == 0) ? 4 : 1;
  const int U = g.V / VEC;
  const long long rows = (long long)g.B * g.N;
  // chunks per row: as many as fit one wave of resident CTAs, at least one
  const long long slots = (long long)device_sm_count() * kGreedyCtasPerSm;
  int chunks = (int)(slots / rows);
  chunks = max(1, min(chunks, ceil_div(U, kGreedyThreads)));
  g.chunk_units = ceil_div(U, chunks);
  g.chunks = ceil_div(U, g.chunk_units);
  const long long ctas = rows * g.chunks;
  const cudaError_t err =
      VEC == 4 ? launch_pdl(greedy_kernel<4>, dim3((unsigned)ctas), dim3(kGreedyThreads), 0, stream, g)
               : launch_pdl(greedy_kernel<1>, dim3((unsigned)ctas), dim3(kGreedyThreads), 0, stream, g);
  if (err != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}

tv_status check_greedy_args(const float* logits, const int32_t* tokens, const int32_t* parent,
                            const int32_t* depth, int B, int N, int V, int32_t* argmax,
                            int32_t* accept_len, int32_t* end_node, int32_t* path, int32_t* bonus,
                            int32_t* status) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || V < 1) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!logits || !tokens || !parent || !depth || !argmax || !accept_len || !end_node || !path ||
      !bonus || !status)
    return TV_ERR_INVALID_ARG;
  if ((long long)B * N * (long long)V >= (1ll << 40) || (long long)B * N * ((V + 255) / 256) > 0x7fffffffll)
    return TV_ERR_UNSUPPORTED;
  if ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) != 0) return TV_ERR_INVALID_ARG;
  return TV_OK;
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
  const tv_status st = tv::check_greedy_args(logits, tokens, parent, depth, B, N, V, argmax,
                                             accept_len, end_node, path, bonus, status);
  if (st != TV_OK || B == 0) return st;
  if (!workspace || ws_bytes < tv_accept_greedy_workspace_size(B, N, V)) return TV_ERR_WORKSPACE;
  tv::GreedyArgs g = {};
  g.logits = logits;
  g.tokens = tokens;
  g.parent = parent;
  g.depth = depth;
  g.B = B;
  g.N = N;
  g.V = V;
  g.argmax = argmax;
  g.accept_len = accept_len;
  g.end_node = end_node;
  g.path = path;
  g.bonus = bonus;
  g.status = status;
  g.ws.keys = static_cast<unsigned long long*>(workspace);
  g.ws.arrivals = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) +
                                                  tv::greedy_keys_bytes(B, N));
  return tv::launch_greedy(g, stream);
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
  const tv_status st = tv::check_greedy_args(logits, tokens, parent, depth, B, N, V, argmax,
                                             accept_len, end_node, path, bonus, status);
  if (st != TV_OK || B == 0) return st;
  if ((long long)B * N > tv::kStaticMaxRows || B > tv::kStaticMaxSeqs) return TV_ERR_UNSUPPORTED;
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
  tv::GreedyArgs g = {};
  g.logits = logits;
  g.tokens = tokens;
  g.parent = parent;
  g.depth = depth;
  g.B = B;
  g.N = N;
  g.V = V;
  g.argmax = argmax;
  g.accept_len = accept_len;
  g.end_node = end_node;
  g.path = path;
  g.bonus = bonus;
  g.status = status;
  g.ws.keys = reinterpret_cast<unsigned long long*>(b8);
  g.ws.arrivals = reinterpret_cast<unsigned int*>(b8 + tv::kStaticKeyBytes);
  return tv::launch_greedy(g, stream);
}
