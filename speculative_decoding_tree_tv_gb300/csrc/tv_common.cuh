// Shared device helpers for libtreeverify (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "treeverify.h"
#include "tv_nvtx.h"

#define TV_CHECK_LAUNCH()                                   \
  do {                                                      \
    if (cudaPeekAtLastError() != cudaSuccess) {             \
      (void)cudaGetLastError();                             \
      return TV_ERR_CUDA;                                   \
    }                                                       \
  } while (0)

// Bounds-checked builds.  Compiled with -DTV_CHECKED, every index a kernel
// computes from its inputs or its launch geometry is checked before the
// access it guards: a failed check skips that access and records the first
// failing site of the translation unit, (TV_UNIT << 16) | line, in a device
// word that tv_debug_check_take() reads and clears.  No check traps.  In the
// regular build TV_CHECK(cond) is the constant true and the guarded access is
// unconditional.  Each source file defines TV_UNIT (its number in
// treeverify.h) before including this header.
#ifndef TV_UNIT
#define TV_UNIT 0
#endif

namespace tv {

// the host-side reader of one translation unit's check word (checked builds):
// returns the recorded site (0: none) and clears it, or -1 on a CUDA error
using CheckReader = int (*)();
void register_check_reader(CheckReader reader);

#ifdef TV_CHECKED
namespace {
__device__ int g_check_site;
int take_check_site() {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_check_site, sizeof v) != cudaSuccess ||
      cudaMemcpyToSymbol(g_check_site, &zero, sizeof zero) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return v;
}
struct CheckRegistrar {
  CheckRegistrar() { register_check_reader(&take_check_site); }
};
const CheckRegistrar g_check_registrar;
}  // namespace
__device__ __forceinline__ bool check_site(bool ok, int line) {
  if (!ok) atomicCAS(&g_check_site, 0, (TV_UNIT << 16) | line);
  return ok;
}
#define TV_CHECK(cond) (::tv::check_site(static_cast<bool>(cond), __LINE__))
#else
#define TV_CHECK(cond) true
#endif
// 0 <= i < n
#define TV_IN(i, n) TV_CHECK((i) >= 0 && (i) < (n))

constexpr int kMaxNodes = TV_MAX_NODES;
constexpr int kMaxWords = (kMaxNodes + 63) / 64;

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Order-preserving map of a finite float to uint32 (larger float -> larger
// key).  -0 is folded onto +0 so that the two compare equal.
__device__ __forceinline__ uint32_t float_key(float x) {
  uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// Order-preserving map of a double to uint64.
__device__ __forceinline__ uint64_t double_key(double x) {
  uint64_t u = (uint64_t)__double_as_longlong(x == 0.0 ? 0.0 : x);
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// (value, index) argmax combine: larger value wins, ties -> lower index.
struct ArgMax {
  float v;
  int i;
};
__device__ __forceinline__ ArgMax argmax_combine(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}
__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = argmax_combine(a, b);
  }
  return a;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the previous kernel on the stream is still
// running; it must call pdl_wait() before touching anything that kernel
// writes (the wait returns once that kernel has completed and its memory
// operations are visible).  pdl_trigger() lets the next kernel start early;
// since that kernel waits in turn, every kernel here triggers first thing.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Compensated (Kahan) fp32 accumulation.
struct KahanF {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float x) {
    float y = x - c;
    float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

// ---------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): ten rounds of two 64x64 -> 128-bit multiplies
// with the published multipliers; the key is bumped by the published Weyl
// increments between rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void philox4x64_10(const uint64_t ctr[4], uint64_t k0, uint64_t k1,
                                              uint64_t out[4]) {
  const uint64_t kMul0 = 0xD2E7470EE14C6C93ull, kMul1 = 0xCA5A826395121157ull;
  const uint64_t kWeyl0 = 0x9E3779B97F4A7C15ull, kWeyl1 = 0xBB67AE8584CAA73Bull;
  uint64_t a = ctr[0], b = ctr[1], c = ctr[2], d = ctr[3];
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round) {
      k0 += kWeyl0;
      k1 += kWeyl1;
    }
    const uint64_t lo_a = kMul0 * a, hi_a = __umul64hi(kMul0, a);
    const uint64_t lo_c = kMul1 * c, hi_c = __umul64hi(kMul1, c);
    a = hi_c ^ b ^ k0;
    b = lo_c;
    c = hi_a ^ d ^ k1;
    d = lo_a;
  }
  out[0] = a;
  out[1] = b;
  out[2] = c;
  out[3] = d;
}

// Uniform in [0, 1) for one decision of the stochastic acceptance walk.
__device__ __forceinline__ double decision_uniform(uint64_t seed, uint64_t offset, int b, int node,
                                                   uint32_t purpose, uint32_t ordinal) {
  const uint64_t ctr[4] = {offset, (uint64_t)b, (uint64_t)node,
                           ((uint64_t)purpose << 32) | ordinal};
  uint64_t out[4];
  philox4x64_10(ctr, seed, 0ull, out);
  return (double)(out[0] >> 11) * (1.0 / 9007199254740992.0);
}

// ------------------------------------------------------------------- host
constexpr int kMaxDevicesCached = 64;

// Ordinal of the current device, or -1 if none can be queried.
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return dev;
}

// SMs of the current device (152 on GB300 when no device can be queried),
// looked up once per device.
inline int device_sm_count() {
  static std::atomic<int> cache[kMaxDevicesCached];
  const int dev = current_device();
  if (dev >= 0 && dev < kMaxDevicesCached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int v = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      v <= 0) {
    (void)cudaGetLastError();
    return 152;
  }
  if (dev < kMaxDevicesCached) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Set a kernel attribute on the current device.  Attributes are per device,
// so each (kernel, attribute) pair is set once per device: a registry of
// device bit-words under a lock.
inline bool set_func_attr(const void* kernel, cudaFuncAttribute attr, int value) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, uint64_t> done;
  const int dev = current_device();
  if (dev < 0) return false;
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  uint64_t& word = done[{kernel, (int)attr}];
  if (bit && (word & bit)) return true;
  if (cudaFuncSetAttribute(kernel, attr, value) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  word |= bit;
  return true;
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device.
template <typename Kernel>
inline bool set_dyn_smem(Kernel kernel, int bytes) {
  return set_func_attr(reinterpret_cast<const void*>(kernel),
                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Launch with programmatic stream serialisation (see pdl_wait/pdl_trigger).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace tv
