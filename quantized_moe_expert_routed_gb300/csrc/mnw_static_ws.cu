// mnw_static_ws.cu -- the whole MoE layer without any device allocation.
//
// Some callers cannot hand the library a workspace and cannot allocate one:
// for example a plugin running inside a serving process whose device memory
// is owned up front by another allocator that gives plugins no allocation
// hook, or a latency-critical path that must not pay the implicit device
// synchronisation of cudaMalloc/cudaFree.  For them, mnw_moe_forward_static()
// runs the same kernels as mnw_moe_forward() with its intermediates in a
// fixed-size array compiled into this library.  The caller still passes (and
// owns) the inputs and the output.
//
// The array lives in device memory on every GPU that loads the library, for
// as long as the library stays loaded (until process exit in practice), so
// it is kept modest: MNW_STATIC_WS_BYTES.  Requests needing more return
// MNW_E_WORKSPACE_TOO_SMALL before anything is enqueued.
//
// All calls share the one array: calls that overlap on the GPU (different
// streams, or different host threads, on the same device) race on it and
// corrupt each other's intermediates; serialise them on one stream.  The array
// keeps the previous call's contents; the only value that must start at zero,
// the device error word, is cleared by every call.
#include <cstring>
#include <mutex>

#include "mnw_internal.h"

namespace mnw {
namespace {

// 32 MiB: enough for the 256-token decode batch of the W4A16 workload
// (H = 2048, I = 512, top-8 needs about 19 MB).
constexpr size_t kStaticWsBytes = size_t(32) << 20;
static_assert(kStaticWsBytes == MNW_STATIC_WS_BYTES, "header and library disagree on the static workspace size");

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// Device address of g_static_ws, looked up once per device.  In host code the
// symbol is only a host-side stand-in, never a device address.  The cached
// address belongs to the device's primary context: after cudaDeviceReset the
// library must not be used again in this process.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

int static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MNW_E_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return MNW_E_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MNW_OK;
}

}  // namespace
}  // namespace mnw

extern "C" int mnw_moe_forward_static(const mnw_moe_layer* layer, int act, const void* x, const int32_t* ids,
                                      const float* w, int T, int k, void* out, uint32_t* err, mnw_stream stream) {
  if (!layer || T < 0 || k < 1) return MNW_E_INVALID_ARG;
  if (T == 0) {
    // nothing to run; the caller's error word still reports this call (no error)
    if (err && cudaMemsetAsync(err, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return MNW_E_CUDA;
    return MNW_OK;
  }
  const size_t need = mnw_moe_workspace_size(layer, act, T, k);
  if (need == 0) return MNW_E_INVALID_ARG;
  if (need > mnw::kStaticWsBytes) return MNW_E_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  int rc = mnw::static_ws_address(&ws);
  if (rc != MNW_OK) return rc;
  rc = mnw_moe_forward(layer, act, x, ids, w, T, k, out, ws, mnw::kStaticWsBytes, stream);
  if (rc != MNW_OK) return rc;
  if (err && cudaMemcpyAsync(err, mnw_moe_workspace_error_word(ws), sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MNW_E_CUDA;
  return MNW_OK;
}
