// Library-wide entry points: status strings, version, workspace clearing, the
// checked build's status word.
#define TV_UNIT 9
#include "tv_common.cuh"

#include <vector>

namespace tv {
namespace {
std::mutex& readers_mutex() {
  static std::mutex m;
  return m;
}
std::vector<CheckReader>& readers() {
  static std::vector<CheckReader> r;
  return r;
}
}  // namespace
void register_check_reader(CheckReader reader) {
  std::lock_guard<std::mutex> lock(readers_mutex());
  readers().push_back(reader);
}
}  // namespace tv

extern "C" int tv_checked_build(void) {
#ifdef TV_CHECKED
  return 1;
#else
  return 0;
#endif
}

extern "C" tv_status tv_debug_check_take(int32_t* site) {
  if (!site) return TV_ERR_INVALID_ARG;
  *site = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(tv::readers_mutex());
  for (tv::CheckReader r : tv::readers()) {
    const int v = r();
    if (v < 0) return TV_ERR_CUDA;
    if (v != 0 && *site == 0) *site = v;
  }
  return TV_OK;
}

extern "C" const char* tv_status_string(tv_status s) {
  switch (s) {
    case TV_OK: return "TV_OK";
    case TV_ERR_INVALID_ARG: return "TV_ERR_INVALID_ARG";
    case TV_ERR_INVALID_TREE: return "TV_ERR_INVALID_TREE";
    case TV_ERR_UNSUPPORTED: return "TV_ERR_UNSUPPORTED";
    case TV_ERR_CUDA: return "TV_ERR_CUDA";
    case TV_ERR_TIMEOUT: return "TV_ERR_TIMEOUT";
    case TV_ERR_INVALID_TOKEN: return "TV_ERR_INVALID_TOKEN";
    case TV_ERR_WORKSPACE: return "TV_ERR_WORKSPACE";
  }
  return "TV_ERR_UNKNOWN";
}

extern "C" int tv_version(void) { return 100; }

extern "C" tv_status tv_workspace_clear(void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (ws_bytes == 0) return TV_OK;
  if (!workspace) return TV_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, ws_bytes, stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return TV_ERR_CUDA;
  }
  return TV_OK;
}

namespace tv {
namespace {
// buf[i] = i for i < n, each store guarded by the check 0 <= i < logical_n
__global__ void check_selftest_kernel(int32_t* buf, int n, int logical_n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && TV_IN(i, logical_n)) buf[i] = i;
}
}  // namespace
}  // namespace tv

extern "C" tv_status tv_debug_check_selftest(int32_t* buf, int n, int logical_n,
                                             cudaStream_t stream) {
  if (!buf || n < 0 || logical_n < 0) return TV_ERR_INVALID_ARG;
  if (n == 0) return TV_OK;
  tv::check_selftest_kernel<<<tv::ceil_div(n, 256), 256, 0, stream>>>(buf, n, logical_n);
  TV_CHECK_LAUNCH();
  return TV_OK;
}
