// tv_attn_verify: tree-verify attention (OPT-Tree §2: every tree token is
// scored in one target pass under the tree attention mask; a node sees the
// cached prefix, its ancestors and itself).
//
// Warp-per-query-row kernel: CTA (row block, kv head, sequence) holds 8 warps,
// each owning one (node, query head) row of the GQA group of that kv head, so
// the CTA's rows share every K/V line through L1.  Scores use an online
// softmax in the log2 domain with fp32 accumulation.
#include "tv_common.cuh"

namespace tv {
namespace {

constexpr int kAttnWarps = 8;
constexpr int kKeyBlock = 8;  // keys scored together for shuffle-chain ILP

template <int D>
struct Lane {
  static constexpr int E = D / 32;  // elements per lane
};

template <int D>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float (&x)[D / 32]) {
  constexpr int E = D / 32;
  if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(u.x << 16);
    x[1] = __uint_as_float(u.x & 0xffff0000u);
    x[2] = __uint_as_float(u.y << 16);
    x[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    x[0] = __uint_as_float(u << 16);
    x[1] = __uint_as_float(u & 0xffff0000u);
  }
}

__device__ __forceinline__ uint16_t to_bf16(float f) {
  // round to nearest even (finite inputs)
  uint32_t u = __float_as_uint(f);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

template <int D>
__global__ void __launch_bounds__(kAttnWarps * 32)
attn_warp_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                 const uint16_t* __restrict__ v, const int32_t* __restrict__ kv_len,
                 const uint64_t* __restrict__ anc_mask, int N, int Hq, int Hkv, int Lcap,
                 float scale_log2, uint16_t* __restrict__ out, float* __restrict__ lse,
                 int32_t* __restrict__ status) {
  constexpr int E = D / 32;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kAttnWarps + warp;
  const int L = kv_len[b];
  const bool bad = (L < 0) || (L + N > Lcap);
  if (blockIdx.x == 0 && kvh == 0 && threadIdx.x == 0 && status)
    status[b] = bad ? TV_ERR_INVALID_ARG : TV_OK;
  if (r >= N * G) return;
  const int i = r / G, h = kvh * G + r % G;
  uint16_t* orow = out + (((size_t)b * N + i) * Hq + h) * D;
  if (bad) {
    for (int e = lane; e < D; e += 32) orow[e] = 0;
    if (lse && lane == 0) lse[((size_t)b * N + i) * Hq + h] = 0.0f;
    return;
  }
  float qv[E];
  load_bf16<D>(q + (((size_t)b * N + i) * Hq + h) * D + lane * E, qv);
  const uint16_t* kb = k + ((size_t)b * Hkv + kvh) * (size_t)Lcap * D + lane * E;
  const uint16_t* vb = v + ((size_t)b * Hkv + kvh) * (size_t)Lcap * D + lane * E;
  const int W = (N + 63) >> 6;
  const uint64_t* anc = anc_mask + ((size_t)b * N + i) * W;

  float m = -INFINITY, l = 0.0f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.0f;

  auto consume = [&](float s, const float (&vv)[E]) {
    const float m_new = fmaxf(m, s);
    const float c = exp2f(m - m_new);
    const float p = exp2f(s - m_new);
    l = l * c + p;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = o[e] * c + p * vv[e];
    m = m_new;
  };

  // prefix keys, kKeyBlock at a time
  int j = 0;
  for (; j + kKeyBlock <= L; j += kKeyBlock) {
    float s[kKeyBlock];
#pragma unroll
    for (int t = 0; t < kKeyBlock; ++t) {
      float kv[E];
      load_bf16<D>(kb + (size_t)(j + t) * D, kv);
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc += qv[e] * kv[e];
      s[t] = acc;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1)
#pragma unroll
      for (int t = 0; t < kKeyBlock; ++t) s[t] += __shfl_xor_sync(0xffffffffu, s[t], o2);
#pragma unroll
    for (int t = 0; t < kKeyBlock; ++t) {
      float vv[E];
      load_bf16<D>(vb + (size_t)(j + t) * D, vv);
      consume(s[t] * scale_log2, vv);
    }
  }
  for (; j < L; ++j) {
    float kv[E], vv[E];
    load_bf16<D>(kb + (size_t)j * D, kv);
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc += qv[e] * kv[e];
    acc = warp_sum(acc);
    load_bf16<D>(vb + (size_t)j * D, vv);
    consume(acc * scale_log2, vv);
  }
  // tree keys: ancestors-or-self of node i
  for (int w = 0; w < W; ++w) {
    uint64_t bits = anc[w];
    while (bits) {
      const int a = w * 64 + __ffsll((long long)bits) - 1;
      bits &= bits - 1;
      if (a >= N) break;
      float kv[E], vv[E];
      load_bf16<D>(kb + (size_t)(L + a) * D, kv);
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc += qv[e] * kv[e];
      acc = warp_sum(acc);
      load_bf16<D>(vb + (size_t)(L + a) * D, vv);
      consume(acc * scale_log2, vv);
    }
  }
  const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
  if constexpr (E == 4) {
    uint2 u;
    u.x = (uint32_t)to_bf16(o[0] * inv_l) | ((uint32_t)to_bf16(o[1] * inv_l) << 16);
    u.y = (uint32_t)to_bf16(o[2] * inv_l) | ((uint32_t)to_bf16(o[3] * inv_l) << 16);
    *reinterpret_cast<uint2*>(orow + lane * E) = u;
  } else {
    const uint32_t u = (uint32_t)to_bf16(o[0] * inv_l) | ((uint32_t)to_bf16(o[1] * inv_l) << 16);
    *reinterpret_cast<uint32_t*>(orow + lane * E) = u;
  }
  if (lse && lane == 0)
    lse[((size_t)b * N + i) * Hq + h] = (l > 0.0f) ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace
}  // namespace tv

extern "C" size_t tv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int Lcap) {
  (void)B; (void)N; (void)Hq; (void)Hkv; (void)D; (void)Lcap;
  return 256;
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
  if (B > 65535 || Hkv > 65535) return TV_ERR_UNSUPPORTED;
  (void)workspace;
  (void)ws_bytes;
  const float sc = (scale == 0.0f) ? 1.0f / sqrtf((float)D) : scale;
  const float scale_log2 = sc * 1.4426950408889634f;
  const int G = Hq / Hkv;
  dim3 grid(tv::ceil_div(N * G, tv::kAttnWarps), Hkv, B);
  if (D == 128)
    tv::attn_warp_kernel<128><<<grid, tv::kAttnWarps * 32, 0, stream>>>(
        q, k, v, kv_len, anc_mask, N, Hq, Hkv, Lcap, scale_log2, out, lse, status);
  else
    tv::attn_warp_kernel<64><<<grid, tv::kAttnWarps * 32, 0, stream>>>(
        q, k, v, kv_len, anc_mask, N, Hq, Hkv, Lcap, scale_log2, out, lse, status);
  TV_CHECK_LAUNCH();
  return TV_OK;
}
