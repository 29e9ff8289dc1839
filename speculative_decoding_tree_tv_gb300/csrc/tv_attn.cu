// tv_attn_verify: tree-verify attention on the 5th-generation tensor cores
// (OPT-Tree §2: all tree tokens are verified in one target pass under the
// tree attention mask; a node sees the cached prefix, its ancestors and
// itself).
//
// One CTA owns up to 256 query rows of one (sequence, kv head): two row
// blocks of 128 TMEM lanes.  Rows are the GQA group's (node, head) pairs,
// node-major; a row block holds nb = floor(128 / G) whole nodes, so both
// blocks share every K/V tile and the cache is streamed once per kv head.
// The CTA covers a range of 128-key tiles of the key range [0, kv_len + N).
// Warp roles (320 threads):
//   warps 0-3, 4-7  softmax of row block 0, 1: one thread per query row (TMEM
//                   lane), online softmax over the tile's 128 keys in the
//                   log2 domain with lazy rescaling; the tree mask is applied
//                   as 32-bit visibility words;
//   warp 8          producer: TMA loads (128-byte swizzle) of Q once and of
//                   the K tiles (lane 0) and V tiles (lane 1);
//   warp 9          MMA issuer: S_r = Q_r K^T and O_r += P_r V with
//                   tcgen05.mma (bf16 operands in shared memory, fp32
//                   accumulators in TMEM), each issued as soon as its inputs
//                   are ready, so the next tile's S overlaps this tile's
//                   softmax; zeroes V rows past the end of the key range so
//                   that stale cache slots never reach a result.
// Unsplit, each softmax thread normalises its row and writes it.  When the
// key range is split across CTAs, each split stores its normalised bf16
// partial rows to the workspace (chunk-major: each warp store writes 512
// contiguous bytes), with (max, sum) pairs
// beside them, and a merge kernel chained by programmatic dependent launch
// combines the partials of every row.  Every wait is bounded.
#define TV_UNIT 5
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cstdio>
#include <cstdlib>
#include <cuda_bf16.h>

#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

using namespace sm100;

constexpr int kRB = 128;              // rows per row block = TMEM lanes
constexpr int kBN = 128;              // keys per tile
constexpr float kRescaleLog2 = 8.0f;  // keep a stale max while within 2^8
constexpr int kAtomBytes = 16384;     // 128 rows x 128 bytes
constexpr int kMaxSplit = 64;         // splits of one CTA's key range
constexpr int kPrefetchTiles = 4;     // tiles of a split's range prefetched into the L2
constexpr int kMaxOrderSeqs = 64;     // sequences a launch orders longest first

// Shape of a CTA: RBS row blocks of 128 query rows (one or two), 128 softmax
// threads per row block, then the K producer, MMA and V producer warps (the
// two loads wait on different barriers, so each has a warp of its own) and,
// with two row blocks, a second MMA warp: each row block's products are issued
// by a warp of their own.  Two row
// blocks share every K/V tile (the cache is streamed once per kv head); one
// row block gives twice the CTAs.  In both the softmax writes P(t) over the
// first 64 columns of the S buffer it read (bf16 pairs), from where PV(t)
// reads it (tcgen05.mma with A in TMEM), and a later S into that buffer is
// issued after PV(t) (the tensor core runs one thread's instructions in issue
// order).  Both fill 224 KB of shared memory (D = 128):
//   one row block:  Q 32 KB, three K stages, three V stages.  S is
//     double-buffered in TMEM: S(t + 1) is computed while the softmax of tile
//     t runs, and S(t + 2) follows PV(t).
//   two row blocks: Q 64 KB, two K stages, three V stages.  One S buffer per
//     row block (S and O of two row blocks fill the 512 columns), so S_r(t + 1)
//     follows PV_r(t).  The two row blocks run in step: both softmaxes, then
//     the four products back to back (a product run beside a softmax shares
//     TMEM traffic with it and runs slower).
// TMEM: S of (row block r, buffer u) at column 128 (r kSBufs + u), O_r at
// 128 RBS kSBufs + 128 r; 512 columns either way.
template <int RBS>
struct Shape {
  static constexpr int kRows = RBS * kRB;
  static constexpr int kThreads = RBS * kRB + 32 * (RBS == 2 ? 4 : 3);
  static constexpr int kProducerWarp = RBS * 4;  // K loads
  static constexpr int kMmaWarp = RBS * 4 + 1;   // products of row block 0
  static constexpr int kVProducerWarp = RBS * 4 + 2;
  static constexpr int kMmaWarp1 = RBS * 4 + 3;  // products of row block 1 (two row blocks)
  static constexpr int kKStages = (RBS == 1) ? 3 : 2;
  static constexpr int kVStages = 3;
  static constexpr int kPBufs = (RBS == 1) ? 2 : 1;
  static constexpr int kSBufs = (RBS == 1) ? 2 : 1;
  static constexpr uint32_t kTmemCols = 512u;
};

struct AttnParams {
  // tree encoding in the same launch (trees of up to 64 nodes): the parent
  // array in; depth, ancestor masks and tree status out (written by the first
  // CTA of each sequence); each CTA keeps the masks it needs in shared memory
  const int32_t* parent;
  int32_t* depth_out;
  uint64_t* anc_out;
  int32_t* tree_status;
  int fuse_tree;
  const uint16_t* k;  // caches, for the L2 prefetch of a split's first tiles
  const uint16_t* v;
  uint16_t* out;
  float* lse;
  int32_t* status;
  const int32_t* kv_len;
  const uint64_t* anc;
  uint16_t* part;   // split partials [unit][nsplit][D / 8][CTA rows] 16-byte chunks of 8 bf16
  float2* part_ml;  // their (running max in the log2 domain, running sum) [unit][nsplit][CTA rows]
  int N, Hq, Hkv, G, Lcap, W;
  int nb;           // nodes per row block: floor(128 / G)
  int mtiles;       // CTAs along the node axis: ceil(N / (row blocks x nb))
  int nsplit;       // splits of the key range
  int units;        // (sequence, kv head, node tile) units: B x Hkv x mtiles
  int order_seqs;   // launch the sequences longest first (more CTAs than one wave)
  float scale_log2;
};

template <int D, int RBS>
struct Layout {
  static constexpr int A = D / 64;                   // 128-byte atoms per row of Q, K, V
  static constexpr int kTile = A * kAtomBytes;       // one K or V tile (128 keys)
  static constexpr int kQ = 0;                       // Q [row block][atom]
  static constexpr int kK = kQ + RBS * A * kAtomBytes;  // K ring [stage][atom]
  static constexpr int kV = kK + Shape<RBS>::kKStages * kTile;  // V ring [stage][atom]
  static constexpr int kBytes = kV + Shape<RBS>::kVStages * kTile;
  static constexpr int kDyn = kBytes + 1024;         // slack for 1024-byte alignment
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Two bf16 halves of a 32-bit word back to fp32 (exact).
__device__ __forceinline__ float2 unpack_bf16(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Two fp32 lanes at once (Blackwell f32x2 instructions), round to nearest.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<const float2*>(&d);
}

// 2^x on the special-function unit (ex2.approx, flush-to-zero); 2^-inf = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Every lane of the warp waits; the warp goes on only if all of them saw the
// phase complete, so a timeout never splits a warp at a .sync.aligned op.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// 32 bits of the ancestor bit-string starting at bit `pos` (0 <= pos < 64*W).
__device__ __forceinline__ uint32_t anc_bits32(const uint64_t* anc, int W, int pos) {
  const int wi = TV_IN(pos >> 6, W) ? pos >> 6 : 0, sh = pos & 63;
  const uint64_t lo = anc[wi];  // global (from tv_tree_build) or shared (built in this launch)
  const uint64_t hi = (sh != 0 && wi + 1 < W) ? anc[wi + 1] : 0ull;
  return (uint32_t)((lo >> sh) | (sh ? (hi << (64 - sh)) : 0ull));
}

// Visibility of the 32 keys j0 + 32c .. j0 + 32c + 31 for one query row:
// prefix keys (< L) always, tree slot L + a iff a is an ancestor-or-self of
// the row's node, nothing at or beyond L + N.
__device__ __forceinline__ uint32_t visibility32(int c, int j0, int L, int keys, int N,
                                                 const uint64_t* anc, int W) {
  const int lo = 32 * c;
  const int pre = L - j0;   // columns [0, pre) are prefix keys
  const int end = keys - j0;
  const uint32_t pm = (pre >= lo + 32) ? 0xffffffffu : (pre <= lo ? 0u : ((1u << (pre - lo)) - 1u));
  const uint32_t em = (end >= lo + 32) ? 0xffffffffu : (end <= lo ? 0u : ((1u << (end - lo)) - 1u));
  uint32_t tm = 0u;
  const int x = lo - pre;   // tree index of column lo
  if (x + 32 > 0 && x < N) tm = (x >= 0) ? anc_bits32(anc, W, x) : (anc_bits32(anc, W, 0) << (-x));
  return (pm | tm) & em;
}

constexpr int kFusedTreeMax = 64;  // nodes a fused tree encoding handles (one mask word)

// Node j's value from a tree held by a warp (node i in lane i % 32, slot i / 32).
__device__ __forceinline__ int gather_i(const int (&v)[2], int j) {
  const int lo = __shfl_sync(0xffffffffu, v[0], j & 31);
  const int hi = __shfl_sync(0xffffffffu, v[1], j & 31);
  return j < 32 ? lo : hi;
}
__device__ __forceinline__ uint64_t gather_u64(const uint64_t (&v)[2], int j) {
  const uint64_t lo = __shfl_sync(0xffffffffu, v[0], j & 31);
  const uint64_t hi = __shfl_sync(0xffffffffu, v[1], j & 31);
  return j < 32 ? lo : hi;
}

// Tree encoding of sequence b by one warp (N <= 64; OPT-Tree §2: a node
// attends to its ancestors and itself): depth and ancestor-or-self masks by
// pointer jumping -- after round r a node's mask holds itself and its 2^(r+1)
// - 1 nearest ancestors, and its depth counts the edges jumped.  An invalid
// parent array (parent[0] != -1, or parent[i] outside [0, i)) gives depth -1
// and empty masks, as tv_tree_build does.  The masks go to shared memory; the
// first CTA of the sequence also writes the outputs of tv_tree_build.
__device__ void tree_in_warp(const AttnParams& p, int b, uint64_t* s_anc, bool write_out) {
  const int lane = threadIdx.x & 31, N = p.N;
  const int32_t* par_g = p.parent + (size_t)b * N;
  int par[2], jmp[2], dep[2];
  uint64_t anc[2];
  int bad = 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    par[s] = i < N ? par_g[i] : -1;
    if (i < N) bad |= (i == 0) ? (par[s] != -1) : (par[s] < 0 || par[s] >= i);
    anc[s] = i < N ? (1ull << i) : 0ull;
    jmp[s] = par[s];
    dep[s] = (i < N && par[s] >= 0) ? 1 : 0;
  }
  bad = __any_sync(0xffffffffu, bad);
  if (!bad) {
#pragma unroll
    for (int r = 0; r < 6; ++r) {
      int nj[2], nd[2];
      uint64_t na[2];
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int j = jmp[s], jj = max(j, 0);
        const int dj = gather_i(dep, jj), jjmp = gather_i(jmp, jj);
        const uint64_t aj = gather_u64(anc, jj);
        nd[s] = j >= 0 ? dep[s] + dj : dep[s];
        na[s] = j >= 0 ? (anc[s] | aj) : anc[s];
        nj[s] = j >= 0 ? jjmp : -1;
      }
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        dep[s] = nd[s];
        anc[s] = na[s];
        jmp[s] = nj[s];
      }
    }
  }
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int i = lane + 32 * s;
    if (i >= N) continue;
    const uint64_t a = bad ? 0ull : anc[s];
    s_anc[i] = a;
    if (write_out) {
      p.depth_out[(size_t)b * N + i] = bad ? -1 : dep[s];
      p.anc_out[(size_t)b * N + i] = a;
    }
  }
  if (write_out && lane == 0) p.tree_status[b] = bad ? TV_ERR_INVALID_TREE : TV_OK;
}

template <int D, int RBS>
__global__ void __launch_bounds__(Shape<RBS>::kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Lay = Layout<D, RBS>;
  using Sh = Shape<RBS>;
  constexpr int A = Lay::A;
  constexpr int kKStages = Sh::kKStages, kVStages = Sh::kVStages, kPBufs = Sh::kPBufs;
  constexpr int kSBufs = Sh::kSBufs;
  constexpr uint32_t kOCol = 128u * RBS * kSBufs;  // first O column
  constexpr int kProducerWarp = Sh::kProducerWarp, kMmaWarp = Sh::kMmaWarp;
  constexpr int kVProducerWarp = Sh::kVProducerWarp;
  constexpr uint32_t kTmemCols = Sh::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Lay::kQ;
  uint8_t* sK = smem + Lay::kK;
  uint8_t* sV = smem + Lay::kV;

  __shared__ __align__(8) uint64_t bar_q;
  __shared__ __align__(8) uint64_t bar_k_full[kKStages], bar_k_empty[kKStages];
  __shared__ __align__(8) uint64_t bar_v_full[kVStages], bar_v_empty[kVStages];
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ __align__(8) uint64_t bar_vzero;  // the last tile's V rows past the range are cleared
  __shared__ __align__(8) uint64_t bar_s_full[2][kSBufs];
  // one P barrier per P buffer: with two buffers the softmax may finish P(t + 1)
  // before the MMA warp has seen P(t), and a shared barrier would then be two
  // phases ahead of the parity it is tested for
  __shared__ __align__(8) uint64_t bar_p_full[2][kPBufs];
  __shared__ __align__(8) uint64_t bar_o_done[2][kPBufs];  // PV(t) of a row block, per P buffer
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ uint64_t s_anc[kFusedTreeMax];     // masks built in this launch
  __shared__ __align__(8) uint64_t bar_tree;    // they are ready

  // Barriers, TMEM and descriptor prefetches need nothing from the previous
  // kernel, so they are set up before waiting for it.
  pdl_trigger();
  const int split = blockIdx.x, mt = blockIdx.y;
  // With order_seqs the CTAs' sequences are set after the wait (longest
  // first); kv heads and node tiles keep their launch order.
  int b = (int)blockIdx.z / p.Hkv;
  const int kvh = (int)blockIdx.z % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N, G = p.G, nb = p.nb;
  const int node0 = mt * RBS * nb;               // first node of this CTA
  const int nrb = (RBS == 2 && node0 + nb < N) ? 2 : 1;  // row blocks holding a node
  const bool is_softmax = warp < 4 * RBS;
  const int rb = (warp >> 2) & 1;                // softmax warps: row block
  const int row = tid & (kRB - 1);               // softmax warps: row = TMEM lane
  const int nodel = row / G;
  const int node = node0 + rb * nb + nodel;
  const bool act = is_softmax && rb < nrb;       // warp-uniform
  const int h = kvh * G + row % G;
  const bool valid_row = act && nodel < nb && node < N && TV_CHECK(h < p.Hq && (int)blockIdx.z < p.units);

  // Split ranges come from the cache capacity, so the first tile's loads can
  // be issued before kv_len arrives; tiles past the key range are dropped.
  const int tiles_cap = ceil_div(p.Lcap, kBN);
  const int t_begin = (int)(((long long)split * tiles_cap) / p.nsplit);
  const int t_end = (int)(((long long)(split + 1) * tiles_cap) / p.nsplit);
  // tiles issued during setup, one per stage
  const int preK = min(kKStages, t_end - t_begin), preV = min(kVStages, t_end - t_begin);
  const bool first_issued = preK > 0;
  __shared__ int s_kvl[kMaxOrderSeqs];
  __shared__ int s_b;
  if (tid == 0) {
    mbar_init(&bar_q, 1);
    // a K or V stage is free, and the tensor core idle at the end, once the
    // products of every row block holding a node are done (one commit each)
    for (int st = 0; st < kKStages; ++st) {
      mbar_init(&bar_k_full[st], 1);
      mbar_init(&bar_k_empty[st], nrb);
    }
    for (int st = 0; st < kVStages; ++st) {
      mbar_init(&bar_v_full[st], 1);
      mbar_init(&bar_v_empty[st], nrb);
    }
    mbar_init(&bar_drain, nrb);
    mbar_init(&bar_vzero, 1);
    mbar_init(&bar_tree, 32);
    for (int r = 0; r < 2; ++r) {
      for (int u = 0; u < kSBufs; ++u) mbar_init(&bar_s_full[r][u], 1);
      for (int u = 0; u < kPBufs; ++u) mbar_init(&bar_p_full[r][u], kRB);
      for (int u = 0; u < kPBufs; ++u) mbar_init(&bar_o_done[r][u], 1);
    }
    mbar_fence_init();
    s_abort = 0;
    if (first_issued) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    if (first_issued && !p.order_seqs) {
      const int y0 = (int)blockIdx.z * p.Lcap + t_begin * kBN;
      // This CTA's Q rows and the first tiles of its key range into the L2
      // while the previous kernel finishes.  Prefetches are hints (the L2 is
      // where every SM reads and writes), so they change no result even if
      // the previous kernel writes these inputs; the loads come after the wait.
      for (int r = 0; r < nrb; ++r)
#pragma unroll
        for (int a = 0; a < A; ++a) tma_prefetch_l2_3d(&tmQ, a * 64, kvh * G, b * N + node0 + r * nb);
      if (p.fuse_tree)  // the parent row, 256 bytes at most: every line it touches
        for (int i = 0; i < N; i += 32) line_prefetch_l2(p.parent + (size_t)b * N + i);
      const int rows = min(min(t_end - t_begin, kPrefetchTiles) * kBN, p.Lcap - t_begin * kBN);
      if (rows > 0) {
        bulk_prefetch_l2(p.k + (size_t)y0 * D, (uint32_t)rows * D * 2u);
        bulk_prefetch_l2(p.v + (size_t)y0 * D, (uint32_t)rows * D * 2u);
      }
    }
  }
  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
  pdl_wait();  // everything below may read what the previous kernel wrote
  if (p.order_seqs) {
    // the sequence at this CTA's launch position among the sequences sorted
    // by key range, longest first (ties to the lower index): the CTAs that
    // start late, after the first wave, get the short ones
    const int nbs = (int)gridDim.z / p.Hkv;
    if (tid < nbs && TV_IN(tid, kMaxOrderSeqs)) s_kvl[tid] = __ldg(p.kv_len + tid);
    if (tid == 0) s_b = b;
    __syncthreads();
    if (tid < nbs && TV_IN(tid, kMaxOrderSeqs)) {
      int r = 0;
      for (int u = 0; u < nbs; ++u) r += (s_kvl[u] > s_kvl[tid]) || (s_kvl[u] == s_kvl[tid] && u < tid);
      if (r == b) s_b = tid;  // b is still the launch position
    }
    __syncthreads();
    b = s_b;
  }
  const int bh = b * p.Hkv + kvh;
  const int y0 = bh * p.Lcap + t_begin * kBN;
  const int L = __ldg(p.kv_len + b);
  if (tid == 0) {
    if (first_issued) {
      // Q: box {64 dims, G heads, nb nodes} per (row block, atom); rows come
      // out node-major, matching the row numbering
      mbar_expect_tx(&bar_q, (uint32_t)(nrb * A * 64 * G * nb * 2));
      for (int r = 0; r < nrb; ++r)
#pragma unroll
        for (int a = 0; a < A; ++a)
          tma_load_3d(sQ + (r * A + a) * kAtomBytes, &tmQ, &bar_q, a * 64, kvh * G,
                      b * N + node0 + r * nb);
      for (int t = 0; t < max(preK, preV); ++t) {
        if (t < preK) {
          mbar_expect_tx(&bar_k_full[t], Lay::kTile);
#pragma unroll
          for (int a = 0; a < A; ++a)
            tma_load_2d(sK + t * Lay::kTile + a * kAtomBytes, &tmK, &bar_k_full[t], a * 64,
                        y0 + t * kBN);
        }
        if (t < preV) {
          mbar_expect_tx(&bar_v_full[t], Lay::kTile);
#pragma unroll
          for (int a = 0; a < A; ++a)
            tma_load_2d(sV + t * Lay::kTile + a * kAtomBytes, &tmV, &bar_v_full[t], a * 64,
                        y0 + t * kBN);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // fused tree encoding: the V producer warp builds the masks before its own
  // work (the first V tiles were issued during setup), in the CTAs whose key
  // range reaches the tree's own slots and in the first CTA of the sequence,
  // which writes the encoding out; softmax warps wait for the masks before the
  // first tile that needs them
  const bool writes_tree = split == 0 && mt == 0 && kvh == 0;
  if (p.fuse_tree && warp == kVProducerWarp && (writes_tree || t_end * kBN > L)) {
    tree_in_warp(p, b, s_anc, writes_tree);
    mbar_arrive(&bar_tree);  // every lane: its shared-memory writes are released
  }

  if (L < 0 || L + N > p.Lcap) {  // uniform over the CTA; the merge kernel skips it too
    if (split == 0 && valid_row) {
      uint4* o = reinterpret_cast<uint4*>(p.out + (((size_t)b * N + node) * p.Hq + h) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
      if (p.lse) p.lse[((size_t)b * N + node) * p.Hq + h] = 0.0f;
    }
    if (split == 0 && mt == 0 && kvh == 0 && tid == 0 && p.status) p.status[b] = TV_ERR_INVALID_ARG;
    if (tid == 0 && first_issued) {  // no copy may be in flight when the CTA leaves
      mbar_wait(&bar_q, 0);
      for (int t = 0; t < preK; ++t) mbar_wait(&bar_k_full[t], 0);
      for (int t = 0; t < preV; ++t) mbar_wait(&bar_v_full[t], 0);
    }
    __syncwarp();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  if (split == 0 && mt == 0 && kvh == 0 && tid == 0 && p.status) p.status[b] = TV_OK;
  const int keys = L + N;
  // tiles of this split inside the key range; an empty split only writes its statistics
  const int T = max(0, min(t_end, ceil_div(keys, kBN)) - t_begin);

  float m_run = -INFINITY, l_run = 0.0f;  // softmax threads: running max (log2) and sum

  if (first_issued && (warp == kProducerWarp || warp == kVProducerWarp)) {
    // ----------------------------------------------------------- producers
    // the first tiles of each ring (and Q) were issued during setup; lane 0
    // of one warp loads K, lane 0 of another V, each into a ring of its own depth
    if (lane == 0) {
      const bool isV = warp == kVProducerWarp;
      uint64_t* full = isV ? bar_v_full : bar_k_full;
      uint64_t* empty = isV ? bar_v_empty : bar_k_empty;
      const CUtensorMap* map = isV ? &tmV : &tmK;
      uint8_t* dst = isV ? sV : sK;
      const int stages = isV ? kVStages : kKStages;
      int issued = isV ? preV : preK;
      for (int t = issued; t < T; ++t) {
        const int st = t % stages;
        const bool freed = mbar_wait(&empty[st], ((t / stages) & 1) ^ 1);
        if (!freed || s_abort) {
          // checked build: which ring gave up
          if (!freed && isV) (void)TV_CHECK(false);
          if (!freed && !isV) (void)TV_CHECK(false);
          s_abort = 1;
          break;
        }
        mbar_expect_tx(&full[st], Lay::kTile);
#pragma unroll
        for (int a = 0; a < A; ++a)
          tma_load_2d(dst + st * Lay::kTile + a * kAtomBytes, map, &full[st], a * 64,
                      y0 + t * kBN);
        issued = t + 1;
      }
      // the CTA must not move on while its copies are in flight: the last
      // tile issued into each stage has landed
      if (!isV) mbar_wait(&bar_q, 0);
      for (int t = max(0, issued - stages); t < issued; ++t)
        mbar_wait(&full[t % stages], (t / stages) & 1);
    }
  } else if (T > 0 && (warp == kMmaWarp || (RBS == 2 && warp == Sh::kMmaWarp1 && nrb == 2))) {
    // ----------------------------------------------------------------- MMA
    // One warp per row block r issues its products in the fixed order
    // S_r(0), [S_r(1),] then PV_r(t) followed by the next S into the buffer
    // that held P_r(t) (the tensor core runs one thread's instructions in issue
    // order).  S_r(t) needs K(t); PV_r(t) needs V(t) and P_r(t).  With two row
    // blocks the two warps issue independently, so that neither warp's own
    // issue overhead leaves the tensor core idle between products.
    const int r = (warp == kMmaWarp) ? 0 : 1;
    constexpr uint32_t idS = idesc_bf16_f32(kRB, kBN, 0, 0);
    constexpr uint32_t idO = idesc_bf16_f32(kRB, D, 0, 1);
    bool ok = warp_wait(&bar_q, 0);
    if (!ok) (void)TV_CHECK(false);
    // S_r(t) = Q_r K(t)^T into row block r's S buffer (lane 0)
    auto issue_s = [&](int t) {
      const uint32_t k0 = smem_u32(sK) + (t % kKStages) * Lay::kTile;
      const uint32_t q0 = smem_u32(sQ) + r * A * kAtomBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
        mma_bf16(tmem + 128 * (r * kSBufs + t % kSBufs), sw128_desc(q0 + off, 16, 1024),
                 sw128_desc(k0 + off, 16, 1024), idS, kk > 0);
      }
      mma_commit(&bar_s_full[r][t % kSBufs]);
      mma_commit(&bar_k_empty[t % kKStages]);  // K(t) is free once every S(t) is done
    };
    // O_r += P_r(t) V(t) over the 16-key steps that hold a key of the range.
    // The V rows of the last step past the range (at most 15; only the tile
    // that ends the key range has them) are cleared first, as the cache may
    // hold anything there: by row block 0's warp, which row block 1's waits for.
    auto issue_pv = [&](int t) -> bool {
      const int valid = min(kBN, keys - (t_begin + t) * kBN);
      const int nk = (valid + 15) >> 4;
      const int z1 = min(kBN, nk * 16);
      if (valid < z1) {
        if (r == 0) {
#pragma unroll
          for (int a = 0; a < A; ++a)
            for (int zr = valid + (lane >> 3); zr < z1; zr += 4)
              *reinterpret_cast<uint4*>(sV + (t % kVStages) * Lay::kTile + a * kAtomBytes +
                                        zr * 128 + ((lane & 7) << 4)) = make_uint4(0, 0, 0, 0);
          fence_async_smem();
          __syncwarp();
          if (nrb == 2 && lane == 0) mbar_arrive(&bar_vzero);
        } else if (!warp_wait(&bar_vzero, 0)) {
          return false;
        }
      }
      __syncwarp();
      if (lane == 0) {
        tc_fence_after();
        const uint32_t v0 = smem_u32(sV) + (t % kVStages) * Lay::kTile;
        const uint32_t tP = tmem + 128 * (r * kSBufs + t % kSBufs);  // P over S: 8 columns per 16 keys
        for (int kk = 0; kk < nk; ++kk)
          mma_bf16_ts(tmem + kOCol + 128 * r, tP + 8 * kk,
                      sw128_desc(v0 + kk * 16 * 128, kAtomBytes, 1024), idO, (t > 0) || (kk > 0));
        mma_commit(&bar_o_done[r][t % kPBufs]);
        mma_commit(&bar_v_empty[t % kVStages]);  // V(t) is free once every PV(t) is done
      }
      __syncwarp();
      return true;
    };
    // Each input is awaited with a blocking wait, which leaves the issue slots
    // of this scheduler to the softmax warps that share it.
    auto s_in_order = [&](int t) -> bool {
      if (!warp_wait(&bar_k_full[t % kKStages], (t / kKStages) & 1)) return false;
      tc_fence_after();
      if (lane == 0) issue_s(t);
      __syncwarp();
      return true;
    };
    auto pv_in_order = [&](int t) -> bool {
      if (!(warp_wait(&bar_v_full[t % kVStages], (t / kVStages) & 1) &&
            warp_wait(&bar_p_full[r][t % kPBufs], (t / kPBufs) & 1)))
        return false;
      tc_fence_after();
      return issue_pv(t);
    };
    for (int t = 0; ok && t < min(T, kSBufs); ++t) ok = s_in_order(t);
    for (int t = 0; ok && t < T; ++t) {
      ok = pv_in_order(t);
      if (ok && t + kSBufs < T) ok = s_in_order(t + kSBufs);
    }
    if (!ok) (void)TV_CHECK(false);
    if (!ok) s_abort = 1;
    if (lane == 0) {  // all issued tensor-core work retires before TMEM is read or released
      mma_commit(&bar_drain);
      // (a warp that gave up may leave the other's commit missing: bounded)
      if (!mbar_wait(&bar_drain, 0)) s_abort = 1;
    }
    __syncwarp();
  } else if (T > 0 && act) {
    // ------------------------------------------------------------- softmax
    const uint64_t* anc = p.fuse_tree ? s_anc + (valid_row ? node : 0)
                                      : p.anc + ((size_t)b * N + (valid_row ? node : 0)) * p.W;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS0 = tmem + 128 * (rb * kSBufs), tO = tmem + kOCol + 128 * rb;
    const float sc = p.scale_log2;
    bool ok = true;
    bool tree_ready = !p.fuse_tree;  // masks built in this launch: awaited when first needed
    for (int t = 0; ok && t < T; ++t) {
      // the mask words (their ancestor loads) are ready before S is
      const int j0 = (t_begin + t) * kBN;
      if (!tree_ready && j0 + kBN > L) {  // this tile reaches the tree's own key slots
        ok = warp_wait(&bar_tree, 0);
        if (!ok) (void)TV_CHECK(false);
        if (!ok) break;
        tree_ready = true;
      }
      uint32_t vis[4] = {0u, 0u, 0u, 0u};
      if (valid_row) {
        if (j0 + kBN <= L) {  // all prefix keys
#pragma unroll
          for (int c = 0; c < 4; ++c) vis[c] = 0xffffffffu;
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) vis[c] = visibility32(c, j0, L, keys, N, anc, p.W);
        }
      }
      ok = warp_wait(&bar_s_full[rb][t % kSBufs], (t / kSBufs) & 1);
      if (!ok) (void)TV_CHECK(false);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
      const uint32_t tS = tS0 + 128 * (t % kSBufs);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_base + 32 * c, sr[c]);
      tmem_wait_ld();
      tc_fence_before();

      // hidden keys become -inf; most tiles are all visible (prefix keys)
      if ((vis[0] & vis[1] & vis[2] & vis[3]) != 0xffffffffu) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!((vis[c] >> e) & 1u)) sr[c][e] = __float_as_uint(-INFINITY);
      }
      // row maximum over eight independent chains
      float mx8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx8[j] = __uint_as_float(sr[0][j]);
#pragma unroll
      for (int k = 8; k < kBN; k += 8)
#pragma unroll
        for (int j = 0; j < 8; ++j) mx8[j] = fmaxf(mx8[j], __uint_as_float(sr[k >> 5][(k & 31) + j]));
      const float tmax = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * sc;
      float corr = 1.0f;
      bool need = false;
      const float m_new = fmaxf(m_run, tmax);
      if (m_run == -INFINITY) {
        m_run = m_new;
      } else if (m_new > m_run + kRescaleLog2) {
        corr = ex2(m_run - m_new);
        m_run = m_new;
        need = true;
      }
      // 2^(s sc - m) pairwise (f32x2 FMA, then the special-function unit); a
      // hidden key gives 2^-inf = 0.  Four pairwise partial sums.
      float2 ps2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
      {
        // 32 keys at a time -> 16 columns of P (bf16 pairs, lower key in the
        // lower half) over the S columns this thread has already read
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_run, -m_run);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pw[16];
          if (m_run == -INFINITY) {  // nothing visible yet: P = 0
#pragma unroll
            for (int i = 0; i < 16; ++i) pw[i] = 0u;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 y = ffma2(make_float2(__uint_as_float(sr[c][2 * i]),
                                                 __uint_as_float(sr[c][2 * i + 1])),
                                     sc2, nm2);
              const float2 x = make_float2(ex2(y.x), ex2(y.y));
              ps2[i & 3] = fadd2(ps2[i & 3], x);
              pw[i] = pack_bf16(x.x, x.y);
            }
          }
          tmem_st16(tS + lane_base + 16 * c, pw);
        }
        tmem_wait_st();
      }
      const float2 ps_a = fadd2(ps2[0], ps2[1]), ps_b = fadd2(ps2[2], ps2[3]);
      const float2 ps_ab = fadd2(ps_a, ps_b);
      l_run = l_run * corr + (ps_ab.x + ps_ab.y);
      // rescale O after the exponentials, when S no longer holds registers
      if (__any_sync(0xffffffffu, need)) {
        // O holds every tile up to t - 1 once PV(t - 1) retired: with one S
        // buffer, S(t) was issued after it and has completed
        if (kSBufs > 1) {
          ok = warp_wait(&bar_o_done[rb][(t - 1) % kPBufs], ((t - 1) / kPBufs) & 1);
          if (!ok) (void)TV_CHECK(false);
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + lane_base + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
          tmem_st32(tO + lane_base + c, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(&bar_p_full[rb][t % kPBufs]);
    }
    if (ok) {
      ok = warp_wait(&bar_o_done[rb][(T - 1) % kPBufs], ((T - 1) / kPBufs) & 1);
      if (!ok) (void)TV_CHECK(false);
    }
    if (!ok) s_abort = 1;
    tc_fence_after();
  }

  // ------------------------------------------------------------ epilogue
  // Each softmax warpgroup finishes its row block as soon as its last PV
  // retired, while the other one may still be working.
  const bool split_kv = p.nsplit > 1;
  const size_t unit = (size_t)bh * p.mtiles + mt;  // (sequence, kv head, node tile)
  if (act) {
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + kOCol + 128 * rb;
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    const int crow = rb * kRB + row;  // row of the CTA
    const size_t slot = unit * p.nsplit + split;
    const bool slot_ok = !split_kv || TV_CHECK(unit < (size_t)p.units && split < p.nsplit);
    if (split_kv && slot_ok) p.part_ml[slot * Sh::kRows + crow] = make_float2(m_run, l_run);
    if (T > 0 && slot_ok) {
      uint32_t o[D / 32][32];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + lane_base + 32 * c, o[c]);  // warp-wide
      tmem_wait_ld();
      if (split_kv) {
        // normalised bf16 partial row (bf16 keeps the fp32 exponent range), chunk-major: the lanes of a warp hold
        // consecutive rows, so every store instruction writes 512 contiguous bytes
        uint4* dst = reinterpret_cast<uint4*>(p.part) + slot * (D / 8) * Sh::kRows + crow;
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[(size_t)(4 * c + q) * Sh::kRows] = make_uint4(
                pack_bf16(__uint_as_float(o[c][8 * q + 0]) * inv, __uint_as_float(o[c][8 * q + 1]) * inv),
                pack_bf16(__uint_as_float(o[c][8 * q + 2]) * inv, __uint_as_float(o[c][8 * q + 3]) * inv),
                pack_bf16(__uint_as_float(o[c][8 * q + 4]) * inv, __uint_as_float(o[c][8 * q + 5]) * inv),
                pack_bf16(__uint_as_float(o[c][8 * q + 6]) * inv, __uint_as_float(o[c][8 * q + 7]) * inv));
      } else if (valid_row) {
        // the whole key range was here: write the output row
        uint4* orow = reinterpret_cast<uint4*>(p.out + (((size_t)b * N + node) * p.Hq + h) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            orow[4 * c + q] = make_uint4(
                pack_bf16(__uint_as_float(o[c][8 * q + 0]) * inv, __uint_as_float(o[c][8 * q + 1]) * inv),
                pack_bf16(__uint_as_float(o[c][8 * q + 2]) * inv, __uint_as_float(o[c][8 * q + 3]) * inv),
                pack_bf16(__uint_as_float(o[c][8 * q + 4]) * inv, __uint_as_float(o[c][8 * q + 5]) * inv),
                pack_bf16(__uint_as_float(o[c][8 * q + 6]) * inv, __uint_as_float(o[c][8 * q + 7]) * inv));
        if (p.lse)
          p.lse[((size_t)b * N + node) * p.Hq + h] =
              l_run > 0.0f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();  // every role is done; TMA and MMA work has retired
  if (s_abort && tid == 0 && p.status) atomicMax(p.status + b, (int)TV_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Merge of the split-KV partials: for every query row, weights
// 2^(m_s - M) * l_s over the nsplit partials, normalised, applied to the
// normalised bf16 partial rows.  A CTA takes 32 rows x 2 chunks of one unit;
// its 8 warps are (chunk, slot group): warp (c, g) takes slots g, g + 4, ...
// of chunk c for 32 consecutive rows, so every load is one contiguous 512-byte
// (chunk) or 256-byte (statistics) segment and all of a thread's loads are in
// flight together (in batches of 6).  The four slot groups are folded in
// shared memory.  Four CTAs fit an SM, so a unit's 64 CTAs of the merge of a
// one-wave attention grid run in one wave too.
constexpr int kMergeRows = 32, kMergeChunks = 2, kMergeGroups = 4, kMergeBatch = 6;

template <int D, int RBS>
__global__ void __launch_bounds__(256, 4)
attn_merge_kernel(const AttnParams p) {
  constexpr int kC16 = D / 8;
  constexpr int kRows = Shape<RBS>::kRows;
  constexpr int kCtaPerUnit = (kRows / kMergeRows) * (kC16 / kMergeChunks);
  constexpr int kSPT = kMaxSplit / kMergeGroups;  // slots per thread at most
  __shared__ float s_m[kMergeGroups][kMergeChunks][kMergeRows];
  __shared__ float s_l[kMergeGroups][kMergeChunks][kMergeRows];
  __shared__ float4 s_acc[kMergeGroups][kMergeChunks][2][kMergeRows];
  pdl_trigger();
  pdl_wait();  // the partials come from the attention kernel
  const int unit = blockIdx.x / kCtaPerUnit;
  const int sub = blockIdx.x % kCtaPerUnit;
  if (!TV_IN(unit, p.units)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cl = warp % kMergeChunks, g = warp / kMergeChunks;
  const int crow = (sub % (kRows / kMergeRows)) * kMergeRows + lane;
  const int ch = (sub / (kRows / kMergeRows)) * kMergeChunks + cl;
  const int bh = unit / p.mtiles, mt = unit % p.mtiles;
  const int b = bh / p.Hkv, kvh = bh % p.Hkv;
  const int L = __ldg(p.kv_len + b);  // checked once the loads below are in flight
  const int ns = p.nsplit;
  const float2* ml = p.part_ml + (size_t)unit * ns * kRows + crow;
  const uint4* src = reinterpret_cast<const uint4*>(p.part) + (size_t)unit * ns * kC16 * kRows +
                     (size_t)ch * kRows + crow;
  float M = -INFINITY, Ls = 0.0f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  for (int k0 = 0; k0 < kSPT; k0 += kMergeBatch) {
    if (g + kMergeGroups * k0 >= ns) break;
    float2 st[kMergeBatch];
    uint4 x[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const int sl = g + kMergeGroups * (k0 + k);
      const bool in = sl < ns;
      st[k] = in ? __ldg(ml + (size_t)sl * kRows) : make_float2(-INFINITY, 0.0f);
      x[k] = in ? __ldg(src + (size_t)sl * kC16 * kRows) : make_uint4(0, 0, 0, 0);
    }
    float mb = M;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) mb = fmaxf(mb, st[k].x);
    if (mb == -INFINITY) continue;  // nothing visible so far
    const float rs = (M == -INFINITY) ? 0.0f : ex2(M - mb);
    Ls *= rs;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= rs;
    M = mb;
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      // an empty split (max -inf) never wrote its rows: select, do not multiply
      if (st[k].x == -INFINITY) continue;
      const float w = ex2(st[k].x - M) * st[k].y;
      Ls += w;
      const uint32_t xw[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16(xw[e]);
        acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
      }
    }
  }
  s_m[g][cl][lane] = M;
  s_l[g][cl][lane] = Ls;
  s_acc[g][cl][0][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  s_acc[g][cl][1][lane] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (g != 0) return;
  if (L < 0 || L + p.N > p.Lcap) return;  // the attention kernel zeroed these outputs
  const int rbk = crow / kRB, rl = crow % kRB;
  const int nodel = rl / p.G;
  const int node = mt * RBS * p.nb + rbk * p.nb + nodel;
  if (nodel >= p.nb || node >= p.N) return;
  const int h = kvh * p.G + rl % p.G;
  if (!TV_IN(h, p.Hq)) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int q = 0; q < kMergeGroups; ++q) Mt = fmaxf(Mt, s_m[q][cl][lane]);
  float Lt = 0.0f;
  float o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.0f;
#pragma unroll
  for (int q = 0; q < kMergeGroups; ++q) {
    const float mq = s_m[q][cl][lane];
    if (mq == -INFINITY) continue;
    const float sc = ex2(mq - Mt);
    Lt = fmaf(sc, s_l[q][cl][lane], Lt);
    const float4 a0 = s_acc[q][cl][0][lane], a1 = s_acc[q][cl][1][lane];
    o[0] = fmaf(sc, a0.x, o[0]);
    o[1] = fmaf(sc, a0.y, o[1]);
    o[2] = fmaf(sc, a0.z, o[2]);
    o[3] = fmaf(sc, a0.w, o[3]);
    o[4] = fmaf(sc, a1.x, o[4]);
    o[5] = fmaf(sc, a1.y, o[5]);
    o[6] = fmaf(sc, a1.z, o[6]);
    o[7] = fmaf(sc, a1.w, o[7]);
  }
  const float inv = Lt > 0.0f ? 1.0f / Lt : 0.0f;
  const size_t orow = ((size_t)b * p.N + node) * p.Hq + h;
  *reinterpret_cast<uint4*>(p.out + orow * D + 8 * ch) =
      make_uint4(pack_bf16(o[0] * inv, o[1] * inv), pack_bf16(o[2] * inv, o[3] * inv),
                 pack_bf16(o[4] * inv, o[5] * inv), pack_bf16(o[6] * inv, o[7] * inv));
  if (ch == 0 && p.lse)
    p.lse[orow] = Lt > 0.0f ? (Mt + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
}

// --------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      (void)cudaGetLastError();
  }
  return fn;
}

struct SplitPlan {
  int rbs;          // row blocks of 128 rows per CTA (1 or 2)
  int nb, mtiles, nsplit;
  long long units;  // (sequence, kv head, node tile) triples
};

// Rough costs in tenths of a microsecond, fitted to the measured times of
// forced plans on GB300 over the tiny, Llama-3-8B spine, TALON, ragged-batch
// and long-context shapes:
//   * a CTA's fixed part (launch into the SM, setup, the first tile's loads
//     and compute, epilogue), for 128-row and 256-row CTAs;
//   * each further 128-key tile.  A 256-row CTA's tile is four 128 x 128 x 128
//     products (S and PV of each row block), about 0.5 us each on the tensor
//     core at this instruction shape.  A 128-row CTA pipelines two tiles, but
//     the L2 serves each kv head's tile once per node tile, and its period
//     grows with the number of node tiles streaming the same cache;
//   * the merge kernel: mostly its launch boundary, plus the partial bytes.
constexpr long long kCostFixed[3] = {0, 43, 54};
constexpr long long kCostMergeBase = 45;
constexpr long long kCostMergePer10MB = 5;  // tenths of a microsecond per 10 MB of partials

long long tile_cost(int rbs, int mtiles) {
  return rbs == 2 ? 26 : 9 + (long long)min(mtiles - 1, 6);
}

// Choose the CTA height and split count that minimise
// (waves of CTAs) x (CTA cost) + merge cost, preferring the taller CTA and
// fewer splits on ties.  One CTA fits an SM (its shared memory decides).
// The environment variable TV_ATTN_PLAN="rows,splits" (rows 128 or 256,
// splits 1 .. min(64, key tiles)) replaces the choice, for tests and tuning;
// anything else in it is ignored.  It is read on every call.
bool plan_override(int N, int nb, int tiles_max, SplitPlan& sp) {
  const char* e = getenv("TV_ATTN_PLAN");
  int rows = 0, ns = 0;
  if (!e || sscanf(e, "%d,%d", &rows, &ns) != 2) return false;
  if ((rows != kRB && rows != 2 * kRB) || ns < 1 || ns > kMaxSplit || ns > tiles_max) return false;
  sp.rbs = rows / kRB;
  sp.nb = nb;
  sp.mtiles = ceil_div(N, sp.rbs * nb);
  sp.nsplit = ns;
  return true;
}

SplitPlan plan_splits(int B, int N, int Hq, int Hkv, int Lcap, int D) {
  SplitPlan best_sp{};
  const int G = Hq / Hkv;
  const int nb = kRB / G;
  const int tiles_max = ceil_div(Lcap, kBN);
  if (plan_override(N, nb, tiles_max, best_sp)) {
    best_sp.units = (long long)B * Hkv * best_sp.mtiles;
    return best_sp;
  }
  const long long slots = device_sm_count();
  long long best = -1;
  for (int rbs = 2; rbs >= 1; --rbs) {
    SplitPlan sp;
    sp.rbs = rbs;
    sp.nb = nb;
    sp.mtiles = ceil_div(N, rbs * nb);
    sp.units = (long long)B * Hkv * sp.mtiles;
    const long long tile = tile_cost(rbs, sp.mtiles);
    for (int ns = 1; ns <= kMaxSplit && ns <= tiles_max; ++ns) {
      const long long waves = (sp.units * ns + slots - 1) / slots;
      const long long tiles_per_cta = (tiles_max + ns - 1) / ns;
      const long long cta = kCostFixed[rbs] + (tiles_per_cta - 1) * tile;
      const long long part_bytes = sp.units * ns * kRB * rbs * (long long)D * 2;
      const long long merge =
          ns > 1 ? kCostMergeBase + kCostMergePer10MB * part_bytes / 10000000ll : 0;
      const long long cost = waves * cta + merge;
      if (best < 0 || cost < best) {
        best = cost;
        sp.nsplit = ns;
        best_sp = sp;
      }
    }
  }
  return best_sp;
}

// Workspace bytes of a plan: bf16 partial rows, then their (max, sum) pairs.
size_t plan_workspace(const SplitPlan& sp, int D) {
  if (sp.nsplit <= 1) return 0;
  const size_t rows = (size_t)sp.units * sp.nsplit * kRB * sp.rbs;
  return align_up(rows * D * 2, 256) + align_up(rows * 8, 256);
}

template <int D, int RBS>
bool set_smem_once() {
  return set_dyn_smem(attn_tc_kernel<D, RBS>, Layout<D, RBS>::kDyn);
}

template <int D, int RBS>
cudaError_t launch_grids(const SplitPlan& sp, int BH, cudaStream_t stream, const CUtensorMap& tmQ,
                         const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& p) {
  cudaError_t e = launch_pdl(attn_tc_kernel<D, RBS>, dim3(sp.nsplit, sp.mtiles, BH),
                             dim3(Shape<RBS>::kThreads, 1, 1), (size_t)Layout<D, RBS>::kDyn,
                             stream, tmQ, tmK, tmV, p);
  if (e != cudaSuccess || sp.nsplit <= 1) return e;
  const long long ctas =
      sp.units * (Shape<RBS>::kRows / kMergeRows) * ((D / 8) / kMergeChunks);
  return launch_pdl(attn_merge_kernel<D, RBS>, dim3((unsigned)ctas, 1, 1), dim3(256, 1, 1), 0,
                    stream, p);
}

// Tree encoding done in the attention launch (nullptr parent: masks given).
struct FusedTree {
  const int32_t* parent = nullptr;
  int32_t* depth = nullptr;
  uint64_t* anc_mask = nullptr;
  int32_t* status = nullptr;
};

template <int D>
tv_status launch_attn(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v, const int32_t* kv_len,
                      const uint64_t* anc_mask, int B, int N, int Hq, int Hkv, int Lcap,
                      float scale_log2, tv_bf16* out, float* lse, int32_t* status,
                      void* workspace, size_t ws_bytes, cudaStream_t stream,
                      const FusedTree& ft = FusedTree()) {
  const SplitPlan sp = plan_splits(B, N, Hq, Hkv, Lcap, D);
  const size_t need = plan_workspace(sp, D);
  if (need > 0 && (workspace == nullptr || ws_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return TV_ERR_WORKSPACE;
  auto encode = tensor_map_encoder();
  if (!encode) return TV_ERR_CUDA;
  if (!(sp.rbs == 2 ? set_smem_once<D, 2>() : set_smem_once<D, 1>())) return TV_ERR_CUDA;
  const int G = Hq / Hkv;
  const cuuint32_t estr[3] = {1, 1, 1};
  // Q as [B * N tokens][Hq heads][D]; a box is {64 dims, G heads, nb nodes}
  CUtensorMap tmQ, tmK, tmV;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)B * N};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)sp.nb};
    if (encode(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<tv_bf16*>(q), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TV_ERR_INVALID_ARG;
  }
  // K and V as [B * Hkv * Lcap slots][D]; a box is {64 dims, 128 keys}
  {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)B * Hkv * Lcap};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, kBN};
    if (encode(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<tv_bf16*>(k), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TV_ERR_INVALID_ARG;
    if (encode(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<tv_bf16*>(v), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return TV_ERR_INVALID_ARG;
  }
  AttnParams p;
  p.parent = ft.parent;
  p.depth_out = ft.depth;
  p.anc_out = ft.anc_mask;
  p.tree_status = ft.status;
  p.fuse_tree = ft.parent != nullptr;
  p.k = reinterpret_cast<const uint16_t*>(k);
  p.v = reinterpret_cast<const uint16_t*>(v);
  p.out = out;
  p.lse = lse;
  p.status = status;
  p.kv_len = kv_len;
  p.anc = anc_mask;
  p.part = nullptr;
  p.part_ml = nullptr;
  if (need > 0) {
    const size_t rows = (size_t)sp.units * sp.nsplit * kRB * sp.rbs;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.part = reinterpret_cast<uint16_t*>(ws);
    p.part_ml = reinterpret_cast<float2*>(ws + align_up(rows * D * 2, 256));
  }
  p.N = N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.Lcap = Lcap;
  p.W = ceil_div(N, 64);
  p.nb = sp.nb;
  p.mtiles = sp.mtiles;
  p.nsplit = sp.nsplit;
  p.units = B * Hkv * sp.mtiles;
  // more CTAs than one wave (one CTA per SM) and several sequences: the
  // longest start first, so that the CTAs left for later waves are short
  p.order_seqs = (B > 1 && B <= kMaxOrderSeqs &&
                  (long long)sp.nsplit * sp.units > (long long)device_sm_count()) ? 1 : 0;
  p.scale_log2 = scale_log2;
  const cudaError_t e = sp.rbs == 2 ? launch_grids<D, 2>(sp, B * Hkv, stream, tmQ, tmK, tmV, p)
                                     : launch_grids<D, 1>(sp, B * Hkv, stream, tmQ, tmK, tmV, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}

bool attn_shape_ok(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  return B >= 0 && N >= 1 && N <= TV_MAX_NODES && Hq >= 1 && Hkv >= 1 && Lcap >= N &&
         Hq % Hkv == 0 && Hq / Hkv <= kRB && (D == 64 || D == 128);
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  if (!tv::attn_shape_ok(B, N, Hq, Hkv, D, Lcap) || B == 0) return 0;
  return tv::plan_workspace(tv::plan_splits(B, N, Hq, Hkv, Lcap, D), D);
}

extern "C" tv_status tv_attn_plan(int B, int N, int Hq, int Hkv, int D, int Lcap, int32_t* info) {
  if (!info || !tv::attn_shape_ok(B, N, Hq, Hkv, D, Lcap) || B == 0) return TV_ERR_INVALID_ARG;
  const tv::SplitPlan sp = tv::plan_splits(B, N, Hq, Hkv, Lcap, D);
  info[0] = tv::kRB * sp.rbs;
  info[1] = sp.mtiles;
  info[2] = sp.nsplit;
  info[3] = (int32_t)(sp.units * sp.nsplit);
  return TV_OK;
}

namespace tv {
namespace {

// Host-side checks shared by both attention entry points.
tv_status check_attn_args(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v,
                          const int32_t* kv_len, const void* mask_or_parent, int B, int N, int Hq,
                          int Hkv, int D, int Lcap, float scale, const tv_bf16* out) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || Hq < 1 || Hkv < 1 || Lcap < N) return TV_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return TV_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TV_ERR_UNSUPPORTED;
  if (Hq / Hkv > kRB) return TV_ERR_UNSUPPORTED;
  if (!(scale >= 0.0f) || !isfinite(scale)) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!q || !k || !v || !kv_len || !mask_or_parent || !out) return TV_ERR_INVALID_ARG;
  if ((long long)B * Hkv > 65535 || (long long)B * Hkv * Lcap > 0x7fffffffll ||
      (long long)B * N > 0x7fffffffll)
    return TV_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15)
    return TV_ERR_INVALID_ARG;
  return TV_OK;
}

tv_status attn_dispatch(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v,
                        const int32_t* kv_len, const uint64_t* anc_mask, int B, int N, int Hq,
                        int Hkv, int D, int Lcap, float scale, tv_bf16* out, float* lse,
                        int32_t* status, void* workspace, size_t ws_bytes, cudaStream_t stream,
                        const FusedTree& ft) {
  const float sc = (scale == 0.0f) ? 1.0f / sqrtf((float)D) : scale;
  const float scale_log2 = sc * 1.4426950408889634f;
  if (D == 128)
    return launch_attn<128>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out,
                            lse, status, workspace, ws_bytes, stream, ft);
  return launch_attn<64>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out, lse,
                         status, workspace, ws_bytes, stream, ft);
}

}  // namespace
}  // namespace tv

extern "C" tv_status tv_attn_verify(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v,
                                    const int32_t* kv_len, const uint64_t* anc_mask, int B, int N,
                                    int Hq, int Hkv, int D, int Lcap, float scale, tv_bf16* out,
                                    float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                                    cudaStream_t stream) {
  TV_NVTX_RANGE("tv_attn_verify");
  const tv_status st =
      tv::check_attn_args(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, D, Lcap, scale, out);
  if (st != TV_OK || B == 0) return st;
  return tv::attn_dispatch(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, D, Lcap, scale, out, lse,
                           status, workspace, ws_bytes, stream, tv::FusedTree());
}

extern "C" tv_status tv_attn_verify_tree(const int32_t* parent, const tv_bf16* q,
                                         const tv_bf16* k, const tv_bf16* v,
                                         const int32_t* kv_len, int B, int N, int Hq, int Hkv,
                                         int D, int Lcap, float scale, tv_bf16* out, float* lse,
                                         int32_t* status, int32_t* depth, uint64_t* anc_mask,
                                         int32_t* tree_status, void* workspace, size_t ws_bytes,
                                         cudaStream_t stream) {
  TV_NVTX_RANGE("tv_attn_verify_tree");
  const tv_status st =
      tv::check_attn_args(q, k, v, kv_len, parent, B, N, Hq, Hkv, D, Lcap, scale, out);
  if (st != TV_OK || B == 0) return st;
  if (!depth || !anc_mask || !tree_status) return TV_ERR_INVALID_ARG;
  if (N > tv::kFusedTreeMax) {
    // masks of more than one word: the tree encoding runs as its own launch
    const tv_status ts = tv_tree_build(parent, B, N, depth, anc_mask, tree_status, stream);
    if (ts != TV_OK) return ts;
    return tv::attn_dispatch(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, D, Lcap, scale, out, lse,
                             status, workspace, ws_bytes, stream, tv::FusedTree());
  }
  tv::FusedTree ft;
  ft.parent = parent;
  ft.depth = depth;
  ft.anc_mask = anc_mask;
  ft.status = tree_status;
  return tv::attn_dispatch(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, D, Lcap, scale, out, lse,
                           status, workspace, ws_bytes, stream, ft);
}
