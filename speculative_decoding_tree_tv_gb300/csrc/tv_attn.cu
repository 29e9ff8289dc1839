// tv_attn_verify: tree-verify attention on the 5th-generation tensor cores
// (OPT-Tree §2: all tree tokens are verified in one target pass under the
// tree attention mask; a node sees the cached prefix, its ancestors and
// itself).
//
// One CTA owns 128 query rows of one (sequence, kv head) -- the GQA group's
// rows (node, head) flattened as node * G + g -- and a range of 128-key tiles
// of that kv head's key range [0, kv_len + N).  Warp roles (320 threads):
//   warps 0-7  softmax, two groups of four warps.  Group h owns keys
//              64h .. 64h+63 of every tile and runs its own online softmax
//              (log2 domain, lazy rescaling) with its own accumulator O_h in
//              TMEM; thread (group h, lane) = one query row = one TMEM lane.
//              The tree mask is applied as 32-bit visibility words;
//   warp 8     producer: TMA loads of K and V tiles (128-byte swizzle) into a
//              two-stage ring;
//   warp 9     MMA: S = Q K^T, then O_h += P_h V_h for each key half, with
//              tcgen05.mma (bf16 operands in shared memory, fp32 accumulators
//              in TMEM); zeroes V rows past the end of the key range so that
//              stale cache slots never reach a result.
// When one CTA covers the whole key range, the two halves are merged in shared
// memory and the CTA writes the output rows.  When the key range is split
// across CTAs, each split stages its two normalised fp16 partials and stores
// them to the workspace with one bulk copy, its (max, sum) statistics beside
// them; a merge kernel, chained by programmatic dependent launch, combines
// the 2 x nsplit partials of every row.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

using namespace sm100;

constexpr int kBM = 128;              // query rows per CTA = TMEM lanes
constexpr int kBN = 128;              // keys per tile (two halves of 64)
constexpr int kStages = 2;            // K/V ring depth
constexpr int kSoftmaxThreads = 256;  // two groups of four warps
constexpr int kThreads = kSoftmaxThreads + 64;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale max while within 2^8
constexpr int kAtomBytes = 16384;     // 128 rows x 128 bytes
constexpr int kMaxSplit = 32;         // splits of one row tile's key range

struct AttnParams {
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  int32_t* status;
  const int32_t* kv_len;
  const uint64_t* anc;
  __half* part;    // split partials [unit][2 * nsplit][128][D] fp16, chunks swizzled
  float2* part_ml; // their (running max in the log2 domain, running sum) [unit][2 * nsplit][128]
  int N, Hq, Hkv, G, Lcap, W;
  int nsplit;      // splits per row tile
  float scale_log2;
};

template <int D>
struct Layout {
  static constexpr int A = D / 64;                 // 128-byte atoms per row of Q, K, V
  static constexpr int kQ = 0;
  static constexpr int kP = kQ + A * kAtomBytes;
  static constexpr int kKV = kP + 2 * kAtomBytes;  // P: 128 rows x 128 keys bf16
  static constexpr int kStage = 2 * A * kAtomBytes;
  static constexpr int kBytes = kKV + kStages * kStage;
  static constexpr int kDyn = kBytes + 1024;       // slack for 1024-byte alignment
  // TMEM: S at [0, 128), O_0 at [128, 128 + D), O_1 at [128 + D, 128 + 2D)
  static constexpr uint32_t kTmemCols = (128 + 2 * D <= 256) ? 256u : 512u;
  // epilogue staging at kQ (Q and P are dead by then): 2 groups x 128 fp16 rows
  static_assert(2 * kBM * D * 2 <= kKV, "staging must fit Q + P");
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Every lane of the warp waits; the warp goes on only if all of them saw the
// phase complete, so a timeout never splits a warp at a .sync.aligned op.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// 32 bits of the ancestor bit-string starting at bit `pos` (0 <= pos < 64*W).
__device__ __forceinline__ uint32_t anc_bits32(const uint64_t* anc, int W, int pos) {
  const int wi = pos >> 6, sh = pos & 63;
  const uint64_t lo = __ldg(anc + wi);
  const uint64_t hi = (sh != 0 && wi + 1 < W) ? __ldg(anc + wi + 1) : 0ull;
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

// fp32 row buffers are stored with the 16-byte chunks of a row XOR-swizzled by
// the row index, so that threads writing different rows hit different banks.
__device__ __forceinline__ int swz_chunk(int row, int chunk) { return chunk ^ (row & 7); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const AttnParams p) {
  using Lay = Layout<D>;
  constexpr int A = Lay::A;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + Lay::kQ;
  uint8_t* sP = smem + Lay::kP;
  uint8_t* sKV = smem + Lay::kKV;

  __shared__ __align__(8) uint64_t bar_kv_full[kStages], bar_kv_empty[kStages];
  __shared__ __align__(8) uint64_t bar_q, bar_s_full, bar_s_free, bar_drain;
  __shared__ __align__(8) uint64_t bar_p_full[2], bar_o_done[2];
  __shared__ float s_gm[2][kBM], s_gl[2][kBM];  // per group: running max and sum of each row
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  pdl_wait();  // everything below may read what the previous kernel wrote
  pdl_trigger();
  const int split = blockIdx.x, mt = blockIdx.y, bh = blockIdx.z;
  const int b = bh / p.Hkv, kvh = bh % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = (tid < kSoftmaxThreads) ? (tid >> 7) : 0;  // softmax group: key half
  const int row = tid & (kBM - 1);                            // softmax threads: query row
  const int N = p.N;
  const int L = p.kv_len[b];
  const int rows_total = N * p.G;
  const int r = mt * kBM + row;
  const bool is_softmax = tid < kSoftmaxThreads;
  const bool valid_row = is_softmax && (r < rows_total);
  const int node = valid_row ? r / p.G : 0;
  const int h = kvh * p.G + (valid_row ? r % p.G : 0);
  const int nranks = p.nsplit;

  if (L < 0 || L + N > p.Lcap) {  // the merge kernel skips this sequence too
    if (split == 0 && valid_row && grp == 0) {
      uint4* o = reinterpret_cast<uint4*>(p.out + (((size_t)b * N + node) * p.Hq + h) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
      if (p.lse) p.lse[((size_t)b * N + node) * p.Hq + h] = 0.0f;
    }
    if (split == 0 && mt == 0 && kvh == 0 && tid == 0 && p.status) p.status[b] = TV_ERR_INVALID_ARG;
    return;
  }
  if (split == 0 && mt == 0 && kvh == 0 && tid == 0 && p.status) p.status[b] = TV_OK;
  const int keys = L + N;
  const int tiles = ceil_div(keys, kBN);
  // balanced split of this sequence's tiles; an empty split still merges
  const int t_begin = (int)(((long long)split * tiles) / nranks);
  const int T = (int)(((long long)(split + 1) * tiles) / nranks) - t_begin;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_q, kSoftmaxThreads);
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_s_free, kSoftmaxThreads);
    mbar_init(&bar_p_full[0], kBM);
    mbar_init(&bar_p_full[1], kBM);
    mbar_init(&bar_o_done[0], 1);
    mbar_init(&bar_o_done[1], 1);
    mbar_init(&bar_drain, 1);
    mbar_fence_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&s_tmem, Lay::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem;
  const uint32_t tO0 = tmem + 128, tO1 = tmem + 128 + D;

  float m_run = -INFINITY, l_run = 0.0f;  // softmax threads: running max (log2) and sum

  if (T > 0 && warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int row0 = bh * p.Lcap;
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        const uint32_t ph = (t / kStages) & 1;
        if (!mbar_wait(&bar_kv_empty[s], ph ^ 1u) || s_abort) {
          s_abort = 1;
          break;
        }
        uint8_t* sK = sKV + s * Lay::kStage;
        uint8_t* sV = sK + A * kAtomBytes;
        mbar_expect_tx(&bar_kv_full[s], 2 * A * kAtomBytes);
        const int y = row0 + (t_begin + t) * kBN;
#pragma unroll
        for (int a = 0; a < A; ++a) {
          tma_load_2d(sK + a * kAtomBytes, &tmK, &bar_kv_full[s], a * 64, y);
          tma_load_2d(sV + a * kAtomBytes, &tmV, &bar_kv_full[s], a * 64, y);
        }
        issued = t + 1;
      }
      // the CTA must not move on while its copies are in flight
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(&bar_kv_full[t % kStages], (t / kStages) & 1);
    }
  } else if (T > 0 && warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, 0, 0);
    constexpr uint32_t idO = idesc_bf16_f32(kBM, D, 0, 1);
    bool ok = warp_wait(&bar_q, 0);
    for (int t = 0; ok && t < T; ++t) {
      const int s = t % kStages;
      uint8_t* sK = sKV + s * Lay::kStage;
      uint8_t* sV = sK + A * kAtomBytes;
      ok = warp_wait(&bar_kv_full[s], (t / kStages) & 1);
      if (!ok) break;
      const int j0 = (t_begin + t) * kBN;
      const int valid = min(kBN, keys - j0);
      if (valid < kBN) {
        // V rows past the key range: whatever the cache holds there, make it 0
        const int rows = kBN - valid;
        for (int idx = lane; idx < rows * 8 * A; idx += 32) {
          const int a = idx / (rows * 8);
          const int rem = idx - a * rows * 8;
          *reinterpret_cast<uint4*>(sV + a * kAtomBytes + (valid + (rem >> 3)) * 128 +
                                    ((rem & 7) << 4)) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
      }
      __syncwarp();
      if (t > 0) {
        ok = warp_wait(&bar_s_free, (t - 1) & 1);
        if (!ok) break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          mma_bf16(tS, sw128_desc(q0 + off, 16, 1024), sw128_desc(k0 + off, 16, 1024), idS,
                   kk > 0);
        }
        mma_commit(&bar_s_full);
      }
      __syncwarp();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        ok = warp_wait(&bar_p_full[hf], t & 1);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          // O_hf += P[:, 64hf .. 64hf+63] * V[64hf .. 64hf+63, :]
          const uint32_t p0 = smem_u32(sP) + hf * kAtomBytes;
          const uint32_t v0 = smem_u32(sV) + hf * 64 * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(hf ? tO1 : tO0, sw128_desc(p0 + kk * 32, 16, 1024),
                     sw128_desc(v0 + kk * 16 * 128, kAtomBytes, 1024), idO, (t > 0) || (kk > 0));
          mma_commit(&bar_o_done[hf]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&bar_kv_empty[s]);
      __syncwarp();
    }
    if (!ok) s_abort = 1;
    if (lane == 0) {  // all issued tensor-core work retires before TMEM is read or released
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0);
    }
  } else if (T > 0 && is_softmax) {
    // ------------------------------------------------------------- softmax
    {
      const uint4* qrow =
          reinterpret_cast<const uint4*>(p.q + (((size_t)b * N + node) * p.Hq + h) * D);
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) {  // this group's half of the row's chunks
        const int c = grp * (D / 16) + cc;
        const uint4 v = valid_row ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * kAtomBytes + row * 128 +
                                  (((c & 7) ^ (row & 7)) << 4)) = v;
      }
      fence_async_smem();
      mbar_arrive(&bar_q);
    }
    const uint64_t* anc = p.anc + ((size_t)b * N + node) * p.W;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = grp ? tO1 : tO0;
    const float sc = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      ok = warp_wait(&bar_s_full, t & 1);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(tS + lane_base + grp * 64, sr[0]);
      tmem_ld32(tS + lane_base + grp * 64 + 32, sr[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_s_free);

      const int j0 = (t_begin + t) * kBN;
      float mx[2] = {-INFINITY, -INFINITY};
      if (valid_row && j0 + kBN <= L) {  // all prefix keys: nothing to mask
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx[c] = fmaxf(mx[c], __uint_as_float(sr[c][e]));
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint32_t vis = valid_row ? visibility32(2 * grp + c, j0, L, keys, N, anc, p.W) : 0u;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float x = ((vis >> e) & 1u) ? __uint_as_float(sr[c][e]) : -INFINITY;
            sr[c][e] = __float_as_uint(x);
            mx[c] = fmaxf(mx[c], x);
          }
        }
      }
      const float tmax = fmaxf(mx[0], mx[1]) * sc;
      float corr = 1.0f;
      bool need = false;
      const float m_new = fmaxf(m_run, tmax);
      if (m_run == -INFINITY) {
        m_run = m_new;
      } else if (m_new > m_run + kRescaleLog2) {
        corr = exp2f(m_run - m_new);
        m_run = m_new;
        need = true;
      }
      uint32_t pk[32];
      float ps[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (m_run == -INFINITY) {  // nothing visible yet: P = 0
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = 0u;
      } else {
        const float neg_m = -m_run;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float x0 = exp2f(fmaf(__uint_as_float(sr[c][e]), sc, neg_m));
            const float x1 = exp2f(fmaf(__uint_as_float(sr[c][e + 1]), sc, neg_m));
            ps[2 * c + ((e >> 4) & 1)] += x0 + x1;
            pk[(c * 32 + e) >> 1] = pack_bf16(x0, x1);
          }
        }
      }
      l_run = l_run * corr + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      // this group's P half and O_h are free once its previous PV retired
      if (t > 0) {
        ok = warp_wait(&bar_o_done[grp], (t - 1) & 1);
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, need)) {
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
      uint8_t* prow = sP + grp * kAtomBytes + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_full[grp]);
    }
    if (ok) ok = warp_wait(&bar_o_done[grp], (T - 1) & 1);
    if (!ok) s_abort = 1;
    tc_fence_after();
  }

  // ------------------------------------------------------------ epilogue
  tc_fence_before();
  __syncthreads();  // every role is done; TMA and MMA work has retired
  tc_fence_after();
  if (s_abort && tid == 0 && p.status) atomicMax(p.status + b, (int)TV_ERR_TIMEOUT);
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  // Each softmax thread stages its group's normalised O row in fp16 at kQ
  // (Q and P are dead now) as [group][row][D], 16-byte chunks swizzled by the
  // row, with the group's running (max, sum) beside it.
  uint8_t* sStage = smem + Lay::kQ;
  const bool split_kv = p.nsplit > 1;
  const size_t unit = (size_t)bh * gridDim.y + mt;  // (sequence, kv head, row tile)
  if (is_softmax) {
    s_gm[grp][row] = m_run;
    s_gl[grp][row] = l_run;
    if (split_kv) {
      const size_t si = (unit * (2 * p.nsplit) + 2 * split + grp) * kBM + row;
      p.part_ml[si] = make_float2(m_run, l_run);
    }
    uint32_t o[D / 32][32];
    if (T > 0) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32((grp ? tO1 : tO0) + lane_base + 32 * c, o[c]);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) o[c][e] = 0u;
    }
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    uint8_t* srow = sStage + (size_t)(grp * kBM + row) * D * 2;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // four 16-byte chunks of 8 halves
        uint32_t hw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 hv = __floats2half2_rn(__uint_as_float(o[c][8 * e + 2 * j]) * inv,
                                               __uint_as_float(o[c][8 * e + 2 * j + 1]) * inv);
          hw[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        *reinterpret_cast<uint4*>(srow + swz_chunk(row, 4 * c + e) * 16) =
            make_uint4(hw[0], hw[1], hw[2], hw[3]);
      }
    }
    if (split_kv) fence_async_smem();  // the bulk store reads the staging area
  }
  __syncthreads();
  if (split_kv) {
    // the partial rows go to the workspace; tv_attn_merge finishes them
    if (tid == 0 && T > 0) {
      __half* dst = p.part + (unit * (2 * p.nsplit) + 2 * split) * kBM * D;
      bulk_store_global(dst, smem_u32(sStage), (uint32_t)(2 * kBM * D * 2));
      bulk_commit();
      bulk_wait_all();
    }
  } else {
    // merge the two key halves of each row here.  A warp takes 32 / (D / 8)
    // rows; the lanes of a row cover its 16-byte fp16 chunks.
    constexpr int kC16 = D / 8;
    constexpr int kRowsPerWarp = 32 / kC16;
    const int sub = lane / kC16, ch = lane % kC16;
    for (int rb = warp * kRowsPerWarp; rb < kBM; rb += (kThreads / 32) * kRowsPerWarp) {
      const int lr = rb + sub;
      const int gr = mt * kBM + lr;
      if (gr >= rows_total) continue;
      const float m0 = s_gm[0][lr], m1 = s_gm[1][lr];
      const float M = fmaxf(m0, m1);
      const float w0 = (m0 == -INFINITY) ? 0.0f : exp2f(m0 - M) * s_gl[0][lr];
      const float w1 = (m1 == -INFINITY) ? 0.0f : exp2f(m1 - M) * s_gl[1][lr];
      const float L = w0 + w1;
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      const uint4 x0 = *reinterpret_cast<const uint4*>(sStage + (size_t)lr * D * 2 + swz_chunk(lr, ch) * 16);
      const uint4 x1 = *reinterpret_cast<const uint4*>(sStage + (size_t)(kBM + lr) * D * 2 + swz_chunk(lr, ch) * 16);
      const uint32_t a[4] = {x0.x, x0.y, x0.z, x0.w}, c1[4] = {x1.x, x1.y, x1.z, x1.w};
      uint32_t u[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&a[j]));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&c1[j]));
        u[j] = pack_bf16((w0 * f0.x + w1 * f1.x) * inv, (w0 * f0.y + w1 * f1.y) * inv);
      }
      const size_t orow = ((size_t)b * N + gr / p.G) * p.Hq + kvh * p.G + gr % p.G;
      *reinterpret_cast<uint4*>(p.out + orow * D + 8 * ch) = make_uint4(u[0], u[1], u[2], u[3]);
      if (ch == 0 && p.lse)
        p.lse[orow] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Lay::kTmemCols);
}

// Merge of the split-KV partials: for every query row, weights
// exp2(m_s - M) * l_s over the 2 * nsplit partials (two key halves per
// split), normalised, applied to the normalised fp16 partial rows.  A CTA
// takes kRows = 256 / (D / 8) rows of one row tile; kC16 = D / 8 threads per
// row.  Every load of a phase is issued before the first one is used, so the
// kernel pays about one L2 round trip per phase.
template <int D>
__global__ void __launch_bounds__(256)
attn_merge_kernel(const AttnParams p, int mtiles) {
  constexpr int kC16 = D / 8;
  constexpr int kRows = 256 / kC16;
  constexpr int kMaxSlots = 2 * kMaxSplit;
  constexpr int kSPT = kMaxSlots / kC16;  // statistics phase: slots per thread
  constexpr int kBatch = 16;              // accumulation phase: loads in flight per thread
  __shared__ float s_w[kMaxSlots][kRows];
  __shared__ float s_inv[kRows], s_lse[kRows];
  pdl_wait();  // the partials come from the attention kernel
  pdl_trigger();
  const int cpu = kBM / kRows;  // CTAs per row tile
  const int unit = blockIdx.x / cpu;
  const int rbase = (blockIdx.x % cpu) * kRows;
  const int bh = unit / mtiles, mt = unit % mtiles;
  const int b = bh / p.Hkv, kvh = bh % p.Hkv;
  const int L = p.kv_len[b];
  if (L < 0 || L + p.N > p.Lcap) return;  // the attention kernel zeroed these outputs
  const int nslots = 2 * p.nsplit;
  const int tid = threadIdx.x;
  const int r = tid / kC16, j = tid % kC16;  // row of this CTA; lane within the row's group
  const int row = rbase + r;
  const size_t sbase = (size_t)unit * nslots * kBM;
  {
    // statistics: the kC16 threads of a row take slots j, j + kC16, ...
    float2 ml[kSPT];
#pragma unroll
    for (int k = 0; k < kSPT; ++k) {
      const int sl = j + kC16 * k;
      ml[k] = sl < nslots ? __ldg(p.part_ml + sbase + (size_t)sl * kBM + row)
                          : make_float2(-INFINITY, 0.0f);
    }
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kSPT; ++k) M = fmaxf(M, ml[k].x);
#pragma unroll
    for (int o = kC16 / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Ls = 0.0f;
#pragma unroll
    for (int k = 0; k < kSPT; ++k) {
      const int sl = j + kC16 * k;
      const float w = (ml[k].x == -INFINITY) ? 0.0f : exp2f(ml[k].x - M) * ml[k].y;
      if (sl < nslots) s_w[sl][r] = w;
      Ls += w;
    }
#pragma unroll
    for (int o = kC16 / 2; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (j == 0) {
      s_inv[r] = Ls > 0.0f ? 1.0f / Ls : 0.0f;
      s_lse[r] = Ls > 0.0f ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
    }
  }
  __syncthreads();
  const int gr = mt * kBM + row;
  if (gr >= p.N * p.G) return;
  const int ch = j;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(p.part) +
                       ((size_t)unit * nslots * kBM + row) * D * 2 + swz_chunk(row, ch) * 16;
  for (int s0 = 0; s0 < nslots; s0 += kBatch) {
    uint4 x[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      x[k] = (s0 + k < nslots) ? __ldg(reinterpret_cast<const uint4*>(src + (size_t)(s0 + k) * kBM * D * 2))
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (s0 + k >= nslots) break;
      const float w = s_w[s0 + k][r];
      if (w == 0.0f) continue;  // an empty split: its rows were never written
      const uint32_t xw[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xw[e]));
        acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
      }
    }
  }
  const float inv = s_inv[r];
  const size_t orow = ((size_t)b * p.N + gr / p.G) * p.Hq + kvh * p.G + gr % p.G;
  uint4 u;
  u.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  u.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  u.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  u.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(p.out + orow * D + 8 * ch) = u;
  if (ch == 0 && p.lse) p.lse[orow] = s_lse[r];
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
  int mtiles, nsplit;
  long long units;  // (sequence, kv head, row tile) triples
};

// Choose the split count that minimises
// (waves of CTAs) x (tiles per CTA + fixed cost) + merge cost, preferring
// fewer splits.  One CTA fits an SM (its shared memory decides that).
SplitPlan plan_splits(int B, int N, int Hq, int Hkv, int Lcap) {
  SplitPlan sp;
  const int G = Hq / Hkv;
  sp.mtiles = ceil_div(N * G, kBM);
  sp.units = (long long)B * Hkv * sp.mtiles;
  const int tiles_max = ceil_div(Lcap, kBN);
  const long long slots = device_sm_count();
  long long best = -1;
  sp.nsplit = 1;
  for (int ns = 1; ns <= kMaxSplit && ns <= tiles_max; ++ns) {
    const long long waves = (sp.units * ns + slots - 1) / slots;
    const long long tiles_per_cta = (tiles_max + ns - 1) / ns;
    const long long cost = waves * (tiles_per_cta * 4 + 10) + (ns > 1 ? 6 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      sp.nsplit = ns;
    }
  }
  return sp;
}

// Workspace bytes of a plan: fp16 partial rows, then their (max, sum) pairs.
size_t plan_workspace(const SplitPlan& sp, int D) {
  if (sp.nsplit <= 1) return 0;
  const size_t rows = (size_t)sp.units * 2 * sp.nsplit * kBM;
  return align_up(rows * D * 2, 256) + align_up(rows * 8, 256);
}

template <int D>
tv_status launch_attn(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v, const int32_t* kv_len,
                      const uint64_t* anc_mask, int B, int N, int Hq, int Hkv, int Lcap,
                      float scale_log2, tv_bf16* out, float* lse, int32_t* status,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  using Lay = Layout<D>;
  const SplitPlan sp = plan_splits(B, N, Hq, Hkv, Lcap);
  const size_t need = plan_workspace(sp, D);
  if (need > 0 && (workspace == nullptr || ws_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return TV_ERR_WORKSPACE;
  auto encode = tensor_map_encoder();
  if (!encode) return TV_ERR_CUDA;
  static bool smem_set = false;
  if (!smem_set) {
    if (cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay::kDyn) != cudaSuccess) {
      (void)cudaGetLastError();
      return TV_ERR_CUDA;
    }
    smem_set = true;
  }
  CUtensorMap tmK, tmV;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)B * Hkv * Lcap};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64, kBN};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<tv_bf16*>(k), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TV_ERR_INVALID_ARG;
  if (encode(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<tv_bf16*>(v), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TV_ERR_INVALID_ARG;
  AttnParams p;
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.status = status;
  p.kv_len = kv_len;
  p.anc = anc_mask;
  p.part = nullptr;
  p.part_ml = nullptr;
  if (need > 0) {
    const size_t rows = (size_t)sp.units * 2 * sp.nsplit * kBM;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.part = reinterpret_cast<__half*>(ws);
    p.part_ml = reinterpret_cast<float2*>(ws + align_up(rows * D * 2, 256));
  }
  p.N = N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Lcap = Lcap;
  p.W = ceil_div(N, 64);
  p.nsplit = sp.nsplit;
  p.scale_log2 = scale_log2;
  if (launch_pdl(attn_tc_kernel<D>, dim3(sp.nsplit, sp.mtiles, B * Hkv), dim3(kThreads, 1, 1),
                 (size_t)Lay::kDyn, stream, tmK, tmV, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  if (sp.nsplit > 1) {
    constexpr int kRows = 256 / (D / 8);
    const long long ctas = sp.units * (kBM / kRows);
    if (launch_pdl(attn_merge_kernel<D>, dim3((unsigned)ctas, 1, 1), dim3(256, 1, 1), 0, stream, p,
                   sp.mtiles) != cudaSuccess) {
      (void)cudaGetLastError();
      return TV_ERR_CUDA;
    }
  }
  return TV_OK;
}

bool attn_shape_ok(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  return B >= 0 && N >= 1 && N <= TV_MAX_NODES && Hq >= 1 && Hkv >= 1 && Lcap >= N &&
         Hq % Hkv == 0 && (D == 64 || D == 128);
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  if (!tv::attn_shape_ok(B, N, Hq, Hkv, D, Lcap) || B == 0) return 0;
  return tv::plan_workspace(tv::plan_splits(B, N, Hq, Hkv, Lcap), D);
}

extern "C" tv_status tv_attn_verify(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v,
                                    const int32_t* kv_len, const uint64_t* anc_mask, int B, int N,
                                    int Hq, int Hkv, int D, int Lcap, float scale, tv_bf16* out,
                                    float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                                    cudaStream_t stream) {
  if (B < 0 || N < 1 || N > TV_MAX_NODES || Hq < 1 || Hkv < 1 || Lcap < N) return TV_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return TV_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return TV_ERR_UNSUPPORTED;
  if (!(scale >= 0.0f) || !isfinite(scale)) return TV_ERR_INVALID_ARG;
  if (B == 0) return TV_OK;
  if (!q || !k || !v || !kv_len || !anc_mask || !out) return TV_ERR_INVALID_ARG;
  if ((long long)B * Hkv > 65535 || (long long)B * Hkv * Lcap > 0x7fffffffll) return TV_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15)
    return TV_ERR_INVALID_ARG;
  const float sc = (scale == 0.0f) ? 1.0f / sqrtf((float)D) : scale;
  const float scale_log2 = sc * 1.4426950408889634f;
  if (D == 128)
    return tv::launch_attn<128>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out,
                                lse, status, workspace, ws_bytes, stream);
  return tv::launch_attn<64>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out, lse,
                             status, workspace, ws_bytes, stream);
}
