// attn_bwd_static_ws: the backward pass for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain a workspace: code running inside a
// CUDA-graph replay or another library's callback where allocation is
// forbidden, runtimes whose allocator is owned by someone else and not
// reachable from the call site, or embedded / real-time settings that ban
// cudaMalloc after start-up.  For them this entry point runs the same
// schedule -> preprocess -> main -> reduce sequence as attn_bwd, with the
// workspace taken from a fixed-size device array that is part of this
// library's module instead of from the caller.
//
// The array is a file-scope __device__ variable of ATTN_BWD_STATIC_WS_BYTES
// bytes.  Every GPU that loads the library holds those bytes until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it is only a stand-in symbol), so the device address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call made while it is the current device.  The
// address is cached per device ordinal and belongs to the primary context of
// that device: a cudaDeviceReset (which unloads the module) or a non-primary
// context would need a new lookup, and the header declares both unsupported.
#include <mutex>

#include "common.cuh"

namespace {

// 256-byte aligned like every workspace attn_bwd accepts.
static __device__ __align__(256) unsigned char g_static_workspace[ATTN_BWD_STATIC_WS_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_lookup_mutex;
void* g_device_address[kMaxDevices];   // per device ordinal, filled on first use

int static_workspace_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_lookup_mutex);
  if (g_device_address[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_device_address[dev] = p;
  }
  *out = g_device_address[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_static_ws(const attn_bwd_params* p, cudaStream_t stream) {
  size_t need = 0;
  int st = attn_bwd_workspace_size(p, &need);
  if (st != ATTN_OK) return st;
  if (need > (size_t)ATTN_BWD_STATIC_WS_BYTES) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  st = static_workspace_address(&ws);
  if (st != ATTN_OK) return st;
  // attn_bwd initialises every part of the workspace it reads (header words,
  // LSE/D rows, work list, the zeroed atomic dq_acc slice; deterministic
  // slices are written before they are read), so the previous call's
  // contents left in the shared array never leak into this one.
  return attn_bwd(p, ws, (size_t)ATTN_BWD_STATIC_WS_BYTES, stream);
}
