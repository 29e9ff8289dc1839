// tv_accept_greedy: vocabulary-streaming argmax over every tree node's
// target logits, then the longest matching branch (OPT-Tree §2: under greedy
// sampling the longest branch matching the target's highest-probability
// sequence is accepted; GOOSE §2C greedy walk).
//
// One launch.  CTA c handles work item c = (row, chunk): a contiguous chunk
// of one row's logits.  Items are numbered row-major, so the CTAs resident at
// any moment sweep one contiguous stretch of memory (which keeps every DRAM
// channel busy), and the chunk length is chosen so that all items fit in one
// wave of resident CTAs.  With 16-byte-aligned rows the chunk (about 51 KB for
// a 128K vocabulary) is brought into shared memory by bulk copies, so every
// byte of the logits is requested at once without holding registers.  The
// CTA reduces its chunk to (max, lowest index) and folds it into the row's
// 64-bit key (order-preserving float bits, inverted index) with atomicMax.
// The CTA that completes a sequence's N * chunks arrivals runs that tree's
// scan:
//   match[i] = tokens[i] == argmax[parent[i]],
//   valid[i] = AND of match over the root path (pointer jumping),
//   end      = deepest valid node, ties to the lowest index,
// and returns the workspace to zero (keys swapped out with atomicExch,
// counter reset).  No CTA waits for another.
#define TV_UNIT 2
#include <climits>
#include <mutex>

#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

constexpr int kGreedyThreads = 256;

// Reporting limit (SM cycles) of the waits for a CTA's chunk copies: the
// regular bound unless a test has shortened it (tv_debug_set_wait_limit).
// The second wait that keeps copies from outliving the CTA always takes the
// regular bound.
__constant__ long long c_copy_wait_limit = sm100::kWaitLimitCycles;
constexpr int kGreedyCtasPerSm = 4;  // resident CTAs per SM assumed when sizing chunks
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

// Shared-memory arrays of one tree scan.
struct ScanSmem {
  int32_t par[kMaxNodes], tok[kMaxNodes], dep[kMaxNodes];
  int32_t am[kMaxNodes], valid[kMaxNodes], jump[kMaxNodes];
  unsigned int best;
};

// Pull sequence b's parent, token and depth arrays into L2 while the logits
// stream, so that the scan's reads of them are L2 hits.
__device__ __forceinline__ void prefetch_tree(const GreedyArgs& g, int b) {
  const int lines = ceil_div(g.N * (int)sizeof(int32_t), 128);
  const int t = threadIdx.x;
  if (t < 3 * lines) {
    const int32_t* arr = (t < lines) ? g.parent : (t < 2 * lines) ? g.tokens : g.depth;
    const char* addr = reinterpret_cast<const char*>(arr + (size_t)b * g.N) + (t % lines) * 128;
    sm100::line_prefetch_l2(addr);
  }
}

// Longest matching branch of tree b (run by one CTA after every row key of b
// is final).  `err` is a status to report instead of success (a timed-out
// copy in some CTA of the sequence), or TV_OK.
__device__ void tree_scan(const GreedyArgs& g, int b, ScanSmem& sm, int err) {
  const int tid = threadIdx.x;
  const int N = g.N;
  const size_t o = (size_t)b * N;
  int32_t* pth = g.path + o;
  if (err != TV_OK) {
    // a copy of some CTA timed out: report it without reading the row keys,
    // and without touching shared memory, where a copy may still be landing
    for (int i = tid; i < N; i += kGreedyThreads) {
      (void)atomicExch(g.ws.keys + o + i, 0ull);
      g.argmax[o + i] = -1;
      pth[i] = -1;
    }
    if (tid == 0) {
      g.ws.arrivals[b] = 0u;
      g.accept_len[b] = g.end_node[b] = g.bonus[b] = -1;
      g.status[b] = err;
    }
    return;
  }
  int bad_tree = !TV_CHECK(N <= kMaxNodes), bad_tok = 0;
  __syncthreads();
  for (int i = tid; i < N && !bad_tree; i += kGreedyThreads) {
    const unsigned long long key = atomicExch(g.ws.keys + o + i, 0ull);
    int am = (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu));
    if (!TV_IN(am, g.V)) am = 0;
    sm.am[i] = am;
    g.argmax[o + i] = am;
    const int p = __ldcg(g.parent + o + i);
    sm.par[i] = p;
    sm.dep[i] = __ldcg(g.depth + o + i);
    const int tk = __ldcg(g.tokens + o + i);
    sm.tok[i] = tk;
    bad_tree |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    if (i > 0) bad_tok |= (tk < 0 || tk >= g.V);
  }
  if (tid == 0) {
    g.ws.arrivals[b] = 0u;
    sm.best = 0u;
  }
  bad_tree = __syncthreads_or(bad_tree);
  if (!bad_tree) {
    for (int i = tid; i < N; i += kGreedyThreads)
      bad_tree |= (i == 0) ? (sm.dep[0] != 0) : (sm.dep[i] != sm.dep[sm.par[i]] + 1);
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  if (bad_tree || bad_tok) {
    for (int i = tid; i < N; i += kGreedyThreads) pth[i] = -1;
    if (tid == 0) {
      g.accept_len[b] = g.end_node[b] = g.bonus[b] = -1;
      g.status[b] = bad_tree ? TV_ERR_INVALID_TREE : TV_ERR_INVALID_TOKEN;
    }
    return;
  }
  for (int i = tid; i < N; i += kGreedyThreads) {
    sm.valid[i] = (i == 0) ? 1 : TV_IN(sm.par[i], i) && (sm.tok[i] == sm.am[sm.par[i]]);
    sm.jump[i] = sm.par[i];
  }
  __syncthreads();
  // pointer jumping: after r rounds valid[i] covers 2^r edges above i
  for (int span = 1; span < N; span <<= 1) {
    int nv[kScanNodesPerThread], nj[kScanNodesPerThread];
#pragma unroll
    for (int k = 0; k < kScanNodesPerThread; ++k) {
      const int i = tid + k * kGreedyThreads;
      if (i < N) {
        int j = sm.jump[i];
        if (!TV_CHECK(j < i)) j = -1;
        nv[k] = sm.valid[i] & (j < 0 ? 1 : sm.valid[j]);
        nj[k] = j < 0 ? -1 : sm.jump[j];
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kScanNodesPerThread; ++k) {
      const int i = tid + k * kGreedyThreads;
      if (i < N) {
        sm.valid[i] = nv[k];
        sm.jump[i] = nj[k];
      }
    }
    __syncthreads();
  }
  // deepest valid node, lowest index on ties
  unsigned int mine = 0u;
  for (int i = tid; i < N; i += kGreedyThreads)
    if (sm.valid[i]) mine = max(mine, ((unsigned int)sm.dep[i] << 16) | (0xffffu - (unsigned int)i));
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, w));
  if ((tid & 31) == 0) atomicMax(&sm.best, mine);
  __syncthreads();
  int end = (int)(0xffffu - (sm.best & 0xffffu));
  if (!TV_IN(end, N)) end = 0;
  const int end_depth = sm.dep[end];
  for (int i = tid; i < N; i += kGreedyThreads)
    if (i > end_depth) pth[i] = -1;
  if (tid == 0) {
    for (int x = end, d = end_depth; x >= 0 && TV_IN(d, N) && TV_IN(x, N); x = sm.par[x], --d)
      pth[d] = x;
    g.accept_len[b] = end_depth;
    g.end_node[b] = end;
    g.bonus[b] = sm.am[end];
    g.status[b] = TV_OK;
  }
}

__device__ __forceinline__ void red_max_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// The same scan for trees of at most 64 nodes, by one warp in registers:
// node i lives in lane i % 32, slot i / 32, and an array is read at another
// node with two shuffles.  Pointer jumping keeps each round's jump table
// (ancestor at distance 2^r), from which every lane lifts the end node to the
// depth of the path entries it writes.
constexpr int kWarpScanMax = 64;

__device__ __forceinline__ int gather2(const int (&v)[2], int j) {
  const int lo = __shfl_sync(0xffffffffu, v[0], j & 31);
  const int hi = __shfl_sync(0xffffffffu, v[1], j & 31);
  return (j < 32) ? lo : hi;
}

// A tree of at most 64 nodes as one warp holds it: node i in lane i % 32,
// slot i / 32.  Every CTA's first warp loads its sequence's tree while the
// logits stream, so that the CTA which completes the sequence only has the
// row keys left to fetch.
struct TreeRegs {
  int par[2], dep[2], tok[2];
};

__device__ __forceinline__ TreeRegs load_tree_regs(const GreedyArgs& g, int b) {
  const int lane = threadIdx.x & 31;
  const size_t o = (size_t)b * g.N;
  TreeRegs t;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    const bool in = i < g.N;
    t.par[s] = in ? __ldcg(g.parent + o + i) : -1;
    t.dep[s] = in ? __ldcg(g.depth + o + i) : 0;
    t.tok[s] = in ? __ldcg(g.tokens + o + i) : 0;
  }
  return t;
}

__device__ void warp_scan(const GreedyArgs& g, int b, int err, const TreeRegs& tr) {
  const int lane = threadIdx.x & 31;
  const int N = g.N;
  const size_t o = (size_t)b * N;
  int am[2];
  const int(&par)[2] = tr.par;
  const int(&dep)[2] = tr.dep;
  const int(&tok)[2] = tr.tok;
  bool in[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    in[s] = i < N;
    const unsigned long long key = in[s] ? atomicExch(g.ws.keys + o + i, 0ull) : 0ull;
    am[s] = (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu));
    if (in[s] && !TV_IN(am[s], g.V)) am[s] = 0;
    if (in[s]) g.argmax[o + i] = am[s];
  }
  if (lane == 0) g.ws.arrivals[b] = 0u;
  int bad_tree = 0, bad_tok = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    if (in[s]) {
      bad_tree |= (i == 0) ? (par[s] != -1) : (par[s] < 0 || par[s] >= i);
      if (i > 0) bad_tok |= (tok[s] < 0 || tok[s] >= g.V);
    }
  }
  bad_tree = __any_sync(0xffffffffu, bad_tree);
  if (!bad_tree) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int i = lane + 32 * s;
      const int dp = gather2(dep, max(par[s], 0));
      if (in[s]) bad_tree |= (i == 0) ? (dep[s] != 0) : (dep[s] != dp + 1);
    }
    bad_tree = __any_sync(0xffffffffu, bad_tree);
  }
  bad_tok = __any_sync(0xffffffffu, bad_tok);
  int32_t* pth = g.path + o;
  if (bad_tree || bad_tok || err != TV_OK) {
#pragma unroll
    for (int s = 0; s < 2; ++s)
      if (in[s]) pth[lane + 32 * s] = -1;
    if (lane == 0) {
      g.accept_len[b] = g.end_node[b] = g.bonus[b] = -1;
      g.status[b] = err != TV_OK ? err : bad_tree ? TV_ERR_INVALID_TREE : TV_ERR_INVALID_TOKEN;
    }
    return;
  }
  int val[2], jmp[2], lift[6][2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    const int amp = gather2(am, max(par[s], 0));
    val[s] = in[s] ? ((i == 0) ? 1 : (tok[s] == amp)) : 0;
    jmp[s] = par[s];
  }
  // after round r, val[i] covers 2^(r+1) edges above i; lift[r] = ancestor at distance 2^r
#pragma unroll
  for (int r = 0; r < 6; ++r) {
    lift[r][0] = jmp[0];
    lift[r][1] = jmp[1];
    if ((1 << r) >= N) continue;  // uniform
    int nv[2], nj[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int j = jmp[s];
      const int vj = gather2(val, max(j, 0));
      const int jj = gather2(jmp, max(j, 0));
      nv[s] = val[s] & (j < 0 ? 1 : vj);
      nj[s] = j < 0 ? -1 : jj;
    }
    val[0] = nv[0];
    val[1] = nv[1];
    jmp[0] = nj[0];
    jmp[1] = nj[1];
  }
  // deepest valid node, lowest index on ties
  unsigned int mine = 0u;
#pragma unroll
  for (int s = 0; s < 2; ++s)
    if (in[s] && val[s])
      mine = max(mine, ((unsigned int)dep[s] << 16) | (0xffffu - (unsigned int)(lane + 32 * s)));
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, w));
  const int end = (int)(0xffffu - (mine & 0xffffu));
  const int end_depth = (int)(mine >> 16);
  // path[d] = ancestor of end at distance end_depth - d, for d <= end_depth
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int d = lane + 32 * s;
    const int k = max(end_depth - d, 0);
    int x = end;
#pragma unroll
    for (int r = 0; r < 6; ++r) {
      int lr[2] = {lift[r][0], lift[r][1]};
      const int up = gather2(lr, max(x, 0));
      if ((k >> r) & 1) x = up;
    }
    if (d < N) pth[d] = (d <= end_depth) ? x : -1;
  }
  const int bonus = gather2(am, end);
  if (lane == 0) {
    g.accept_len[b] = end_depth;
    g.end_node[b] = end;
    g.bonus[b] = bonus;
    g.status[b] = TV_OK;
  }
}

// Fold the CTA's (max, lowest index) into the row key, count the arrival, and
// run the tree scan if this CTA completes the sequence.  A timed-out copy
// sets bit 31 of the arrival counter, which the scan reports.
__device__ __forceinline__ void finish_item(const GreedyArgs& g, long long row, int b, ArgMax best,
                                            ArgMax* s_red, int* s_last, bool timed_out,
                                            ScanSmem& sm, const TreeRegs& tr) {
  best = block_argmax(best, s_red);
  if (threadIdx.x == 0) {
    // the key update needs no answer; the arrival is a release (ordering the
    // update before it) and an acquire (the last arrival sees every update)
    if (TV_IN(row, (long long)g.B * g.N) && TV_IN(best.i, g.V))
      red_max_u64(g.ws.keys + row, pack_key(best));
    const unsigned int prev = atom_add_acq_rel(g.ws.arrivals + b, timed_out ? 0x80000001u : 1u);
    const bool last = ((prev & 0x7fffffffu) == (unsigned int)(g.N * g.chunks - 1));
    *s_last = last ? (((prev >> 31) | (timed_out ? 1u : 0u)) ? 2 : 1) : 0;
  }
  __syncthreads();
  if (*s_last) {
    const int err = *s_last == 2 ? TV_ERR_TIMEOUT : TV_OK;
    if (g.N <= kWarpScanMax) {
      if (threadIdx.x < 32) warp_scan(g, b, err, tr);
    } else {
      tree_scan(g, b, sm, err);
    }
  }
}

// Rows 16-byte aligned (V % 4 == 0): the CTA's chunk of one row is brought
// into shared memory by bulk copies (two pieces, each on its own mbarrier),
// so the whole chunk is in flight at once without holding registers; the
// reduction then reads shared memory.  The chunk buffer is reused by the scan.
constexpr int kGreedyPieces = 2;

__global__ void __launch_bounds__(kGreedyThreads)
greedy_bulk_kernel(const GreedyArgs g) {
  extern __shared__ __align__(128) uint8_t g_smem[];
  __shared__ __align__(8) uint64_t s_bar[kGreedyPieces];
  __shared__ ArgMax s_red[kGreedyThreads / 32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int U = g.V / 4;
  const long long row = blockIdx.x / g.chunks;
  const int base = (int)(blockIdx.x % g.chunks) * g.chunk_units;
  const int n = min(g.chunk_units, U - base);
  const int b = (int)(row / g.N);
  const int per = TV_CHECK(n >= 1 && n <= g.chunk_units) ? ceil_div(n, kGreedyPieces) : 0;
  if (tid == 0) {
    for (int q = 0; q < kGreedyPieces; ++q) sm100::mbar_init(&s_bar[q], 1);
    sm100::mbar_fence_init();
  }
  __syncthreads();
  pdl_trigger();
  // The chunk (and the tree) into the L2 while the previous kernel finishes.
  // A prefetch changes no result: if the previous kernel writes the logits,
  // its writes land in the same L2 and the copies below, issued after the
  // wait, read them.
  const float4* src = reinterpret_cast<const float4*>(g.logits + row * (long long)g.V) + base;
  if (tid == 0) sm100::bulk_prefetch_l2(src, (uint32_t)n * 16u);
  prefetch_tree(g, b);
  pdl_wait();  // the logits may come from the previous kernel
  if (tid == 0) {
    for (int q = 0; q < kGreedyPieces; ++q) {
      const int q0 = q * per, qn = min(per, n - q0);
      if (qn <= 0) break;
      sm100::mbar_expect_tx(&s_bar[q], (uint32_t)qn * 16u);
      sm100::bulk_load_global(g_smem + (size_t)q0 * 16, src + q0, (uint32_t)qn * 16u, &s_bar[q]);
    }
  }
  TreeRegs tr{};
  if (g.N <= kWarpScanMax && tid < 32) tr = load_tree_regs(g, b);
  // four independent compare chains, one per float4 lane: each sees its
  // indices in increasing order, so a strict compare keeps the lowest index
  // of its maximum, and the combine below breaks ties to the lower index
  ArgMax c4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) c4[j] = {-INFINITY, INT_MAX};
  bool ok = true;
  const float4* x4 = reinterpret_cast<const float4*>(g_smem);
  for (int q = 0; q < kGreedyPieces; ++q) {
    const int q0 = q * per, qn = min(per, n - q0);
    if (qn <= 0) break;
    if (!sm100::mbar_wait_for(&s_bar[q], 0, c_copy_wait_limit)) {
      ok = false;  // every copy of this CTA is waited for again (bounded) below
      continue;
    }
#pragma unroll 4
    for (int k = q0 + tid; k < q0 + qn; k += kGreedyThreads) {
      const float4 v = x4[k];
      const int e = 4 * (base + k);
      if (v.x > c4[0].v) c4[0] = {v.x, e};
      if (v.y > c4[1].v) c4[1] = {v.y, e + 1};
      if (v.z > c4[2].v) c4[2] = {v.z, e + 2};
      if (v.w > c4[3].v) c4[3] = {v.w, e + 3};
    }
  }
  ArgMax best = argmax_combine(argmax_combine(c4[0], c4[1]), argmax_combine(c4[2], c4[3]));
  if (best.i == INT_MAX) best.i = 4 * base;  // only -inf seen: lowest index of the chunk
  const bool timed_out = __syncthreads_or(!ok) != 0;
  if (timed_out && tid == 0) {
    // no copy may still be landing when the CTA leaves or the last CTA reuses
    // the chunk buffer for the tree scan: a second bounded wait on every piece
    // (the scan skips shared memory altogether when a timeout is reported)
    for (int q = 0; q < kGreedyPieces; ++q)
      if (q * per < n) (void)sm100::mbar_wait(&s_bar[q], 0);
  }
  // the chunk buffer is dead once every thread has reduced it (the block
  // reduction below starts with a barrier)
  finish_item(g, row, b, best, s_red, &s_last, timed_out, *reinterpret_cast<ScanSmem*>(g_smem),
              tr);
}

// Rows not 16-byte aligned (V % 4 != 0): scalar loads.
__global__ void __launch_bounds__(kGreedyThreads)
greedy_scalar_kernel(const GreedyArgs g) {
  __shared__ ArgMax s_red[kGreedyThreads / 32];
  __shared__ int s_last;
  __shared__ ScanSmem s_scan;
  const int tid = threadIdx.x;
  pdl_trigger();
  const long long row = blockIdx.x / g.chunks;
  const int base = (int)(blockIdx.x % g.chunks) * g.chunk_units;
  const int n = min(g.chunk_units, g.V - base);
  const int b = (int)(row / g.N);
  const float* x = g.logits + row * (long long)g.V + base;
  // the chunk's lines (and the tree) into the L2 before the wait (a hint)
  for (int k = tid * 32; k < n; k += kGreedyThreads * 32) sm100::line_prefetch_l2(x + k);
  prefetch_tree(g, b);
  pdl_wait();  // the logits may come from the previous kernel
  TreeRegs tr{};
  if (g.N <= kWarpScanMax && tid < 32) tr = load_tree_regs(g, b);
  ArgMax best{-INFINITY, INT_MAX};
  for (int k = tid; k < n; k += kGreedyThreads) {
    const float v = __ldg(x + k);
    if (v > best.v) best = {v, base + k};
  }
  if (best.i == INT_MAX) best.i = base;  // only -inf seen: lowest index of the chunk
  finish_item(g, row, b, best, s_red, &s_last, false, s_scan, tr);
}

// Largest chunk a CTA stages (4 CTAs of this size, plus their static shared
// memory, fit the 228 KB of an SM); bigger rows take more chunks per row.
constexpr int kGreedyChunkMaxBytes = 55296;

tv_status launch_greedy(const GreedyArgs& in, cudaStream_t stream) {
  GreedyArgs g = in;
  const bool bulk = (g.V & 3) == 0;
  const int U = bulk ? g.V / 4 : g.V;
  const long long rows = (long long)g.B * g.N;
  // chunks per row: as many as fit one wave of resident CTAs, at least one
  const long long slots = (long long)device_sm_count() * kGreedyCtasPerSm;
  int chunks = (int)(slots / rows);
  chunks = max(1, min(chunks, ceil_div(U, kGreedyThreads)));
  if (bulk)  // a staged chunk must fit its shared-memory budget
    while ((long long)ceil_div(U, chunks) * 16 > kGreedyChunkMaxBytes) ++chunks;
  g.chunk_units = ceil_div(U, chunks);
  g.chunks = ceil_div(U, g.chunk_units);
  const long long ctas = rows * g.chunks;
  cudaError_t err;
  if (bulk) {
    const size_t smem = max((size_t)g.chunk_units * 16, sizeof(ScanSmem));
    if (!set_dyn_smem(greedy_bulk_kernel, kGreedyChunkMaxBytes)) return TV_ERR_CUDA;
    err = launch_pdl(greedy_bulk_kernel, dim3((unsigned)ctas), dim3(kGreedyThreads), smem, stream, g);
  } else {
    err = launch_pdl(greedy_scalar_kernel, dim3((unsigned)ctas), dim3(kGreedyThreads), 0, stream, g);
  }
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
  TV_NVTX_RANGE("tv_accept_greedy");
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
  TV_NVTX_RANGE("tv_accept_greedy_noalloc");
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

// ---------------------------------------------------------------------------
// Test hook: the reporting limit of tv_accept_greedy's chunk-copy waits on the
// current device (see the header).
extern "C" tv_status tv_debug_set_wait_limit(long long cycles) {
  if (cycles < 0 && cycles != TV_WAIT_LIMIT_DEFAULT) return TV_ERR_INVALID_ARG;
  const long long v = (cycles == TV_WAIT_LIMIT_DEFAULT) ? tv::sm100::kWaitLimitCycles : cycles;
  if (cudaMemcpyToSymbol(tv::c_copy_wait_limit, &v, sizeof(v)) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}
