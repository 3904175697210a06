// kda_static_ws.cu -- kda_fwd for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs where
// cudaMalloc is off limits (a host framework that owns every allocation
// through its own pool and forbids others, an embedded runtime that must
// not grow its memory footprint after start-up, or a plugin with no handle
// to the application's allocator).  For them this file provides one extra
// entry point that behaves like kda_fwd but takes its workspace from a
// fixed array compiled into the library instead of from the caller.
//
// The array lives in device global memory of every GPU that loads this
// library, for as long as the process runs: kStaticWorkspaceBytes (64 MiB)
// per device.  Problems whose workspace would be larger are rejected.
#include <mutex>

#include "../../include/kda.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;   // 64 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device.  In host code
// the array's name only stands in for the symbol; its device address must be
// looked up once per device, with that device current.
kda_status static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_device_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
    g_device_ptr[dev] = p;
  }
  *out = g_device_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_fwd_static_workspace(const kda_shape* shape, const void* q, const void* k,
                                               const void* v, const void* g, const void* beta, float scale,
                                               void* out, const float* A_log, const float* dt_bias,
                                               float lower_bound, const void* initial_state,
                                               kda_state_dtype init_dtype, void* final_state,
                                               kda_state_dtype final_dtype, const int64_t* cu_seqlens,
                                               kda_stream_t stream) {
  size_t need = 0;
  kda_status st = kda_workspace_size(shape, &need);
  if (st != KDA_OK) return st;
  if (need > kStaticWorkspaceBytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  st = static_workspace_address(&ws);
  if (st != KDA_OK) return st;
  // Nothing in the workspace has to start at zero: every call rebuilds its
  // work lists, counters and error word before any kernel reads them.
  return kda_fwd(shape, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, init_dtype,
                 final_state, final_dtype, cu_seqlens, ws, kStaticWorkspaceBytes, stream);
}
