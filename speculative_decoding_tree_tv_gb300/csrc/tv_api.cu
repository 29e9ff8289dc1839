// Library-wide entry points: status strings, version, workspace clearing.
#include "tv_common.cuh"

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
