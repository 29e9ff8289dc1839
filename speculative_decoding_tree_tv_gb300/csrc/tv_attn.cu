// tv_attn_verify: tree-verify attention on the 5th-generation tensor cores
// (OPT-Tree §2: all tree tokens are verified in one target pass under the
// tree attention mask; a node sees the cached prefix, its ancestors and
// itself).
//
// One CTA owns 128 query rows of one (sequence, kv head) -- the GQA group's
// rows (node, head) flattened as node * G + g -- and a range of 128-key tiles
// of that kv head's key range [0, kv_len + N) (split-KV).  Warp roles:
//   warps 0-3  softmax: one TMEM lane (= query row) per thread; load Q into
//              shared memory, read S tiles from TMEM, apply the tree mask and
//              the online softmax (log2 domain, lazy rescaling), write P (bf16)
//              to shared memory, rescale O in TMEM when the running max grows;
//   warp 4     producer: TMA loads of K and V tiles (128-byte swizzle) into a
//              two-stage ring;
//   warp 5     MMA: S = Q K^T and O += P V with tcgen05.mma (bf16 operands
//              from shared memory, fp32 accumulators in TMEM); zeroes V rows
//              past the end of the key range so that stale cache slots never
//              reach a result.
// Splits write unnormalised (O, max, sum) partials to the workspace; the last
// split to finish a (sequence, kv head, row tile) merges them (arrival
// counter, no waiting).  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "tv_common.cuh"
#include "tv_sm100.cuh"

namespace tv {
namespace {

using namespace sm100;

constexpr int kBM = 128;             // query rows per CTA = TMEM lanes
constexpr int kBN = 128;             // keys per tile
constexpr int kStages = 2;           // K/V ring depth
constexpr int kThreads = 192;        // 4 softmax warps + producer + MMA
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256;  // S at [0, 128), O at [128, 128 + D)
constexpr float kRescaleLog2 = 8.0f;  // keep a stale max while within 2^8
constexpr int kAtomBytes = 16384;    // 128 rows x 128 bytes

struct AttnParams {
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  int32_t* status;
  const int32_t* kv_len;
  const uint64_t* anc;
  float* part;               // split partials
  unsigned int* arrivals;    // per (sequence, kv head, row tile)
  int N, Hq, Hkv, G, Lcap, W;
  int mtiles, tps, nsplit;
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
  static constexpr int kPartFloats = kBM * (D + 2);
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void set_status(int32_t* status, int b, int code) {
  if (status) atomicMax(status + b, code);
}

// Every lane of the warp waits; the warp goes on only if all of them saw the
// phase complete, so a timeout never splits a warp at a .sync.aligned op.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

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
  __shared__ __align__(8) uint64_t bar_q, bar_s_full, bar_s_free, bar_p_full, bar_o_done, bar_drain;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_last;

  const int split = blockIdx.x, mt = blockIdx.y, bh = blockIdx.z;
  const int b = bh / p.Hkv, kvh = bh % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  const int L = p.kv_len[b];
  const int rows_total = N * p.G;
  const int r = mt * kBM + tid;  // query row of softmax threads
  const bool valid_row = (tid < kBM) && (r < rows_total);
  const int node = valid_row ? r / p.G : 0;
  const int h = kvh * p.G + (valid_row ? r % p.G : 0);

  if (L < 0 || L + N > p.Lcap) {
    if (split == 0 && valid_row) {
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
  const int nsplit_b = ceil_div(tiles, p.tps);
  if (split >= nsplit_b) return;
  const int t_begin = split * p.tps;
  const int T = min(tiles, t_begin + p.tps) - t_begin;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_q, kBM);
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_s_free, kBM);
    mbar_init(&bar_p_full, kBM);
    mbar_init(&bar_o_done, 1);
    mbar_init(&bar_drain, 1);
    mbar_fence_init();
    s_abort = 0;
    s_last = 0;
  }
  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tS = tmem, tO = tmem + 128;

  float m_run = -INFINITY, l_run = 0.0f;  // softmax threads: running max (log2) and sum

  if (warp == kProducerWarp) {
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
      // the CTA must not retire while its copies are in flight
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(&bar_kv_full[t % kStages], (t / kStages) & 1);
    }
  } else if (warp == kMmaWarp) {
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
      ok = warp_wait(&bar_p_full, t & 1);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t p0 = smem_u32(sP), v0 = smem_u32(sV);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t offp = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          mma_bf16(tO, sw128_desc(p0 + offp, 16, 1024),
                   sw128_desc(v0 + kk * 16 * 128, kAtomBytes, 1024), idO, (t > 0) || (kk > 0));
        }
        mma_commit(&bar_o_done);
        mma_commit(&bar_kv_empty[s]);
      }
      __syncwarp();
    }
    if (!ok) s_abort = 1;
    if (lane == 0) {  // all issued tensor-core work retires before TMEM is released
      mma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------- softmax
    {
      const uint16_t* qrow = p.q + (((size_t)b * N + node) * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = valid_row ? __ldg(reinterpret_cast<const uint4*>(qrow) + c)
                                  : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * kAtomBytes + tid * 128 +
                                  (((c & 7) ^ (tid & 7)) << 4)) = v;
      }
      fence_async_smem();
      mbar_arrive(&bar_q);
    }
    const uint64_t* anc = p.anc + ((size_t)b * N + node) * p.W;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      ok = warp_wait(&bar_s_full, t & 1);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_base + c * 32, sr[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bar_s_free);

      const int j0 = (t_begin + t) * kBN;
      const bool prefix_only = valid_row && (j0 + kBN <= L);
      // ancestor words covering tree slots a = j0 + k - L of this tile
      const int a0 = j0 - L;
      const int wb = a0 > 0 ? (a0 >> 6) : 0;
      uint64_t w0 = 0, w1 = 0, w2 = 0;
      if (valid_row && !prefix_only && j0 + kBN > L) {
        w0 = (wb < p.W) ? __ldg(anc + wb) : 0;
        w1 = (wb + 1 < p.W) ? __ldg(anc + wb + 1) : 0;
        w2 = (wb + 2 < p.W) ? __ldg(anc + wb + 2) : 0;
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int k = c * 32 + e;
          bool vis = prefix_only;
          if (!prefix_only && valid_row) {
            const int j = j0 + k;
            if (j < L) {
              vis = true;
            } else if (j < keys) {
              const int a = j - L;
              const int w = (a >> 6) - wb;
              const uint64_t word = (w == 0) ? w0 : ((w == 1) ? w1 : w2);
              vis = (word >> (a & 63)) & 1ull;
            }
          }
          const float sv = vis ? __uint_as_float(sr[c][e]) * p.scale_log2 : -INFINITY;
          sr[c][e] = __float_as_uint(sv);
          tmax = fmaxf(tmax, sv);
        }
      }
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
      float psum = 0.0f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float x0 = (m_run == -INFINITY) ? 0.0f : exp2f(__uint_as_float(sr[c][e]) - m_run);
          const float x1 =
              (m_run == -INFINITY) ? 0.0f : exp2f(__uint_as_float(sr[c][e + 1]) - m_run);
          psum += x0 + x1;
          pk[(c * 32 + e) >> 1] = pack_bf16(x0, x1);
        }
      }
      l_run = l_run * corr + psum;
      // P and O are free once the previous tile's PV has retired
      if (t > 0) {
        ok = warp_wait(&bar_o_done, (t - 1) & 1);
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
#pragma unroll
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(sP + (c >> 3) * kAtomBytes + tid * 128 +
                                  (((c & 7) ^ (tid & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_full);
    }
    if (ok) ok = warp_wait(&bar_o_done, (T - 1) & 1);
    if (!ok) s_abort = 1;
    tc_fence_after();
    // ------------------------------------------------------------ epilogue
    const size_t orow = ((size_t)b * N + node) * p.Hq + h;
    if (nsplit_b == 1) {
      const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + lane_base + c, o);
        tmem_wait_ld();
        if (valid_row) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D + c);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[8 * e + 0]) * inv_l, __uint_as_float(o[8 * e + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(o[8 * e + 2]) * inv_l, __uint_as_float(o[8 * e + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(o[8 * e + 4]) * inv_l, __uint_as_float(o[8 * e + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(o[8 * e + 6]) * inv_l, __uint_as_float(o[8 * e + 7]) * inv_l);
            dst[e] = v;
          }
        }
      }
      if (valid_row && p.lse)
        p.lse[orow] = l_run > 0.0f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    } else {
      float* part = p.part + (((size_t)bh * p.mtiles + mt) * p.nsplit + split) * Lay::kPartFloats;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + lane_base + c, o);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(part + (size_t)tid * D + c);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                               __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
      }
      part[kBM * D + tid] = m_run;
      part[kBM * D + kBM + tid] = l_run;
      __threadfence();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0) set_status(p.status, b, TV_ERR_TIMEOUT);
  if (nsplit_b > 1) {
    if (tid == 0) {
      __threadfence();
      const unsigned int prev = atomicAdd(p.arrivals + (size_t)bh * p.mtiles + mt, 1u);
      s_last = (prev == (unsigned int)(nsplit_b - 1));
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (tid == 0) p.arrivals[(size_t)bh * p.mtiles + mt] = 0u;
      if (valid_row) {
        const float* base = p.part + ((size_t)bh * p.mtiles + mt) * p.nsplit * Lay::kPartFloats;
        float M = -INFINITY;
        for (int s = 0; s < nsplit_b; ++s)
          M = fmaxf(M, __ldcg(base + (size_t)s * Lay::kPartFloats + kBM * D + tid));
        float acc[D];
#pragma unroll
        for (int d = 0; d < D; ++d) acc[d] = 0.0f;
        float lsum = 0.0f;
        for (int s = 0; s < nsplit_b; ++s) {
          const float* ps = base + (size_t)s * Lay::kPartFloats;
          const float ms = __ldcg(ps + kBM * D + tid);
          const float ls = __ldcg(ps + kBM * D + kBM + tid);
          const float w = (ms == -INFINITY) ? 0.0f : exp2f(ms - M);
          lsum += w * ls;
          const float4* os = reinterpret_cast<const float4*>(ps + (size_t)tid * D);
#pragma unroll
          for (int d4 = 0; d4 < D / 4; ++d4) {
            const float4 v = __ldcg(os + d4);
            acc[4 * d4 + 0] += w * v.x;
            acc[4 * d4 + 1] += w * v.y;
            acc[4 * d4 + 2] += w * v.z;
            acc[4 * d4 + 3] += w * v.w;
          }
        }
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
        const size_t orow = ((size_t)b * N + node) * p.Hq + h;
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) {
          uint4 v;
          v.x = pack_bf16(acc[8 * e + 0] * inv, acc[8 * e + 1] * inv);
          v.y = pack_bf16(acc[8 * e + 2] * inv, acc[8 * e + 3] * inv);
          v.z = pack_bf16(acc[8 * e + 4] * inv, acc[8 * e + 5] * inv);
          v.w = pack_bf16(acc[8 * e + 6] * inv, acc[8 * e + 7] * inv);
          dst[e] = v;
        }
        if (p.lse) p.lse[orow] = lsum > 0.0f ? (M + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else {
      (void)cudaGetLastError();
      n = 152;
    }
  }
  return n;
}

struct SplitPlan {
  int mtiles, tps, nsplit;
};

// Split the key range so that the grid fills the SMs: minimise
// (waves of CTAs) x (tiles per split), preferring fewer splits on ties.
SplitPlan plan_splits(int B, int N, int Hq, int Hkv, int Lcap) {
  SplitPlan sp;
  const int G = Hq / Hkv;
  sp.mtiles = ceil_div(N * G, kBM);
  const long long units = (long long)B * Hkv * sp.mtiles;
  const int tiles_max = ceil_div(Lcap, kBN);
  const int sms = sm_count();
  long long best = -1;
  sp.tps = tiles_max;
  sp.nsplit = 1;
  for (int ns = 1; ns <= tiles_max && ns <= 64; ++ns) {
    const int tps = ceil_div(tiles_max, ns);
    const int nsplit = ceil_div(tiles_max, tps);
    if (nsplit != ns) continue;
    const long long waves = (units * nsplit + sms - 1) / sms;
    const long long cost = waves * (tps + 1) * 4 + (nsplit > 1 ? 2 : 0);
    if (best < 0 || cost < best) {
      best = cost;
      sp.tps = tps;
      sp.nsplit = nsplit;
    }
  }
  return sp;
}

size_t counters_bytes(int B, int Hkv, int mtiles) {
  return align_up((size_t)B * Hkv * mtiles * sizeof(unsigned int), 256);
}

template <int D>
tv_status launch_attn(const tv_bf16* q, const tv_bf16* k, const tv_bf16* v, const int32_t* kv_len,
                      const uint64_t* anc_mask, int B, int N, int Hq, int Hkv, int Lcap,
                      float scale_log2, tv_bf16* out, float* lse, int32_t* status,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  using Lay = Layout<D>;
  auto encode = tensor_map_encoder();
  if (!encode) return TV_ERR_CUDA;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay::kDyn) != cudaSuccess) {
      (void)cudaGetLastError();
      return TV_ERR_CUDA;
    }
    attr_set = true;
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
  const SplitPlan sp = plan_splits(B, N, Hq, Hkv, Lcap);
  AttnParams p;
  p.q = q;
  p.out = out;
  p.lse = lse;
  p.status = status;
  p.kv_len = kv_len;
  p.anc = anc_mask;
  p.arrivals = static_cast<unsigned int*>(workspace);
  p.part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                    counters_bytes(B, Hkv, sp.mtiles));
  p.N = N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Lcap = Lcap;
  p.W = ceil_div(N, 64);
  p.mtiles = sp.mtiles;
  p.tps = sp.tps;
  p.nsplit = sp.nsplit;
  p.scale_log2 = scale_log2;
  if (sp.nsplit > 1) {
    // the arrival counters start at zero whatever the workspace held before
    if (cudaMemsetAsync(workspace, 0, counters_bytes(B, Hkv, sp.mtiles), stream) != cudaSuccess) {
      (void)cudaGetLastError();
      return TV_ERR_CUDA;
    }
  }
  dim3 grid(sp.nsplit, sp.mtiles, B * Hkv);
  attn_tc_kernel<D><<<grid, kThreads, Lay::kDyn, stream>>>(tmK, tmV, p);
  TV_CHECK_LAUNCH();
  return TV_OK;
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Lcap < N || (D != 64 && D != 128))
    return 256;
  const tv::SplitPlan sp = tv::plan_splits(B, N, Hq, Hkv, Lcap);
  size_t bytes = tv::counters_bytes(B, Hkv, sp.mtiles);
  if (sp.nsplit > 1)
    bytes += (size_t)B * Hkv * sp.mtiles * sp.nsplit * tv::kBM * (D + 2) * sizeof(float);
  return bytes;
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
  if (!workspace || ws_bytes < tv_attn_workspace_size(B, N, Hq, Hkv, D, Lcap))
    return TV_ERR_WORKSPACE;
  const float sc = (scale == 0.0f) ? 1.0f / sqrtf((float)D) : scale;
  const float scale_log2 = sc * 1.4426950408889634f;
  if (D == 128)
    return tv::launch_attn<128>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out,
                                lse, status, workspace, ws_bytes, stream);
  return tv::launch_attn<64>(q, k, v, kv_len, anc_mask, B, N, Hq, Hkv, Lcap, scale_log2, out, lse,
                             status, workspace, ws_bytes, stream);
}
