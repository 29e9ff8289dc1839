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
// The two halves are merged in shared memory.  When the key range is split
// across CTAs, the splits of one row tile form a thread-block cluster: each
// pushes its (max, sum, O) partial into the owner CTA's shared memory with
// remote stores, and after one cluster barrier each owner reduces its rows.
// No global scratch, no second launch; every mbarrier wait is bounded.
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
constexpr int kMaxCluster = 16;

struct AttnParams {
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  int32_t* status;
  const int32_t* kv_len;
  const uint64_t* anc;
  int N, Hq, Hkv, G, Lcap, W;
  int nsplit;  // splits per row tile (= cluster size when > 1)
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
  // merge statistics at kQ (Q and P are dead by then): three [slot][row]
  // float arrays of 2 * 16 slots x 64 rows (or 2 slots x 128 rows)
  static_assert(3 * 2 * kMaxCluster * (kBM / 2) * 4 <= kKV, "merge statistics must fit Q + P");
  // receive buffer at kKV: fp16 rows, two slots per rank, ceil(128 / nsplit) rows each
  static_assert(2 * (kBM + kMaxCluster) * D * 2 <= kStages * kStage, "receive buffer");
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
  float* sStat = reinterpret_cast<float*>(smem + Lay::kQ);  // merge statistics, at the end
  __half* sRecv = reinterpret_cast<__half*>(sKV);           // partial O rows, at the end

  __shared__ __align__(8) uint64_t bar_kv_full[kStages], bar_kv_empty[kStages];
  __shared__ __align__(8) uint64_t bar_q, bar_s_full, bar_s_free, bar_drain;
  __shared__ __align__(8) uint64_t bar_p_full[2], bar_o_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_M[kBM], s_L[kBM];  // merged max and sum of the rows this CTA owns

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
  const bool clustered = nranks > 1;

  if (L < 0 || L + N > p.Lcap) {  // uniform over the whole cluster: all of it leaves
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

  // 1. Every CTA of the cluster must be past its main loop before anyone
  //    writes into its Q/P and K/V space, which now hold the merge buffers.
  if (clustered) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  // 2. Every softmax thread hands its group's partial for its row -- running
  //    max, sum and the normalised O row in fp16 -- to the rank owning the row
  //    (itself without a cluster), slot 2 * split + group.
  const int per = ceil_div(kBM, nranks);  // rows per owner rank
  const int slots = 2 * nranks;
  float* s_mx = sStat;                    // [slot][per] partial max (log2)
  float* s_sm = sStat + 2 * kMaxCluster * kBM / 2;          // [slot][per] partial sum
  float* s_cf = sStat + 2 * (2 * kMaxCluster * kBM / 2);    // [slot][per] merge weight
  if (is_softmax) {
    const int owner = row / per, lr = row - owner * per;
    const int sl = 2 * split + grp;
    const int si = sl * per + lr;
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    const uint32_t rrow = smem_u32(sRecv) + (uint32_t)(si * D * 2);
    if (clustered) {
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dsmem_map(smem_u32(s_mx + si), owner)),
                   "f"(m_run)
                   : "memory");
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dsmem_map(smem_u32(s_sm + si), owner)),
                   "f"(l_run)
                   : "memory");
    } else {
      s_mx[si] = m_run;
      s_sm[si] = l_run;
    }
    const uint32_t rbase = clustered ? dsmem_map(rrow, owner) : rrow;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      if (T > 0) {
        tmem_ld32((grp ? tO1 : tO0) + lane_base + c, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {  // four 16-byte chunks of 8 halves
        uint32_t hw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __half2 hv = __floats2half2_rn(__uint_as_float(o[8 * e + 2 * j]) * inv,
                                               __uint_as_float(o[8 * e + 2 * j + 1]) * inv);
          hw[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const uint32_t addr = rbase + (uint32_t)(swz_chunk(lr, c / 8 + e) * 16);
        if (clustered)
          asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(hw[0]),
                       "r"(hw[1]), "r"(hw[2]), "r"(hw[3])
                       : "memory");
        else
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(hw[0]),
                       "r"(hw[1]), "r"(hw[2]), "r"(hw[3])
                       : "memory");
      }
    }
  }
  if (clustered) {
    cluster_sync();  // every partial has landed in its owner's shared memory
  } else {
    __syncthreads();
  }
  // 3. owners merge their rows: weights exp2(m_s - M) * l_s / sum, then a
  //    weighted sum of the normalised partial rows
  const int row0 = split * per, nrows = max(0, min(kBM, row0 + per) - row0);
  for (int lr = tid; lr < nrows; lr += kThreads) {
    float M = -INFINITY;
    for (int sl = 0; sl < slots; ++sl) M = fmaxf(M, s_mx[sl * per + lr]);
    float lsum = 0.0f;
    for (int sl = 0; sl < slots; ++sl) {
      const float ms = s_mx[sl * per + lr];
      const float w = (ms == -INFINITY) ? 0.0f : exp2f(ms - M) * s_sm[sl * per + lr];
      s_cf[sl * per + lr] = w;
      lsum += w;
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    for (int sl = 0; sl < slots; ++sl) s_cf[sl * per + lr] *= inv;
    s_M[lr] = M;
    s_L[lr] = lsum;
  }
  __syncthreads();
  constexpr int kC16 = D / 8;  // 16-byte chunks of an fp16 row
  for (int idx = tid; idx < nrows * kC16; idx += kThreads) {
    const int lr = idx / kC16, ch = idx % kC16;
    const int gr = mt * kBM + row0 + lr;
    if (gr >= rows_total) continue;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int sl = 0; sl < slots; ++sl) {
      const float cw = s_cf[sl * per + lr];
      if (cw == 0.0f) continue;
      const uint4 x = *reinterpret_cast<const uint4*>(
          reinterpret_cast<const uint8_t*>(sRecv) + (size_t)(sl * per + lr) * D * 2 +
          swz_chunk(lr, ch) * 16);
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xw[j]));
        acc[2 * j] += cw * f.x;
        acc[2 * j + 1] += cw * f.y;
      }
    }
    const size_t orow = ((size_t)b * N + gr / p.G) * p.Hq + kvh * p.G + gr % p.G;
    uint4 u;
    u.x = pack_bf16(acc[0], acc[1]);
    u.y = pack_bf16(acc[2], acc[3]);
    u.z = pack_bf16(acc[4], acc[5]);
    u.w = pack_bf16(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(p.out + orow * D + 8 * ch) = u;
    if (ch == 0 && p.lse)
      p.lse[orow] = s_L[lr] > 0.0f ? (s_M[lr] + log2f(s_L[lr])) * 0.69314718055994531f : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Lay::kTmemCols);
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

// How many clusters of each size (1..16) of this kernel the device can hold
// at once; entry 1 is the number of CTAs that fit (one per SM).
template <int D>
const int* cluster_capacity() {
  static int cap[kMaxCluster + 1] = {0};
  static bool done = false;
  if (!done) {
    using Lay = Layout<D>;
    cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kDyn);
    cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    (void)cudaGetLastError();
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 0;
    (void)cudaGetLastError();
    cap[1] = sms;
    for (int cs = 2; cs <= kMaxCluster; ++cs) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = Lay::kDyn;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = cs;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<D>, &cfg) != cudaSuccess) n = 0;
      (void)cudaGetLastError();
      cap[cs] = n;
    }
    done = true;
  }
  return cap;
}

struct SplitPlan {
  int mtiles, nsplit;
};

// Choose the split count (= cluster size) that minimises
// (waves of clusters) x (tiles per CTA + fixed cost), preferring fewer splits.
// Without a device (capacities unknown) the plan assumes 152 SMs and clusters
// of up to 8.
SplitPlan plan_splits(int B, int N, int Hq, int Hkv, int Lcap, const int* cap) {
  SplitPlan sp;
  const int G = Hq / Hkv;
  sp.mtiles = ceil_div(N * G, kBM);
  const long long units = (long long)B * Hkv * sp.mtiles;
  const int tiles_max = ceil_div(Lcap, kBN);
  long long best = -1;
  sp.nsplit = 1;
  for (int ns = 1; ns <= kMaxCluster && ns <= tiles_max; ++ns) {
    long long slots;
    if (cap[1] > 0)
      slots = (ns == 1) ? cap[1] : cap[ns];
    else
      slots = (ns <= 8) ? 152 / ns : 0;
    if (slots <= 0) continue;
    const long long waves = (units + slots - 1) / slots;
    const long long tiles_per_cta = (tiles_max + ns - 1) / ns;
    const long long cost = waves * (tiles_per_cta * 4 + 10) + (ns > 1 ? 4 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      sp.nsplit = ns;
    }
  }
  return sp;
}

template <int D>
tv_status launch_attn(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v, const int32_t* kv_len,
                      const uint64_t* anc_mask, int B, int N, int Hq, int Hkv, int Lcap,
                      float scale_log2, tv_bf16* out, float* lse, int32_t* status,
                      cudaStream_t stream) {
  using Lay = Layout<D>;
  auto encode = tensor_map_encoder();
  if (!encode) return TV_ERR_CUDA;
  const int* cap = cluster_capacity<D>();
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
  const SplitPlan sp = plan_splits(B, N, Hq, Hkv, Lcap, cap);
  AttnParams p;
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.status = status;
  p.kv_len = kv_len;
  p.anc = anc_mask;
  p.N = N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Lcap = Lcap;
  p.W = ceil_div(N, 64);
  p.nsplit = sp.nsplit;
  p.scale_log2 = scale_log2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sp.nsplit, sp.mtiles, B * Hkv);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Lay::kDyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = sp.nsplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = sp.nsplit > 1 ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, attn_tc_kernel<D>, tmK, tmV, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  (void)B; (void)N; (void)Hq; (void)Hkv; (void)D; (void)Lcap;
  return 0;
}

extern "C" tv_status tv_attn_verify(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v,
                                    const int32_t* kv_len, const uint64_t* anc_mask, int B, int N,
                                    int Hq, int Hkv, int D, int Lcap, float scale, tv_bf16* out,
                                    float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                                    cudaStream_t stream) {
  (void)workspace;
  (void)ws_bytes;
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
                                lse, status, stream);
  return tv::launch_attn<64>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out, lse,
                             status, stream);
}
