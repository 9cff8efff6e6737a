// rar_static_ws.cu -- rar_allreduce_static: the ring AllReduce for callers that
// must not allocate device memory. The pages have no counterpart to this entry
// point; it exists for the callers described in include/rar.h.
//
// The workspace of the call lives in a file-scope device array of
// RAR_STATIC_WORKSPACE_BYTES, created when the library is loaded onto a device
// and held until the process exits. In host code `g_static_ws` names a host-side
// stand-in, not device memory, so the host never passes it to a kernel: at
// set-up, once per device and with that device current, cudaGetSymbolAddress
// gives the array's device address, which is cached and passed on as the
// workspace pointer.
#include <cuda_runtime.h>

#include <mutex>

#include "rar.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[RAR_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_static_ws_addr[kMaxDevices] = {nullptr};

// Device address of this device's array (looked up on first use per device).
rar_status static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return RAR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return RAR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_static_ws_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return RAR_ERR_CUDA;
    }
    g_static_ws_addr[dev] = p;
  }
  *out = g_static_ws_addr[dev];
  return RAR_OK;
}

}  // namespace

extern "C" RAR_API rar_status rar_allreduce_static(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                                   size_t count, rar_dtype dtype, rar_redop op,
                                                   const int* ring_order, uint64_t channelMask, rar_proto proto,
                                                   size_t buffSize, int chunkSteps, void* stream) {
  const size_t need = rar_workspace_bytes(nranks, channelMask, proto, buffSize);
  if (need == 0) return RAR_ERR_ARG;
  if (need > (size_t)RAR_STATIC_WORKSPACE_BYTES) return RAR_ERR_WORKSPACE;
  void* ws = nullptr;
  rar_status st = static_ws_address(&ws);
  if (st != RAR_OK) return st;
  if (count > 0) {
    // Every call starts from a cleared workspace: step counters, status,
    // abort flag and FIFO lines of the bytes this call uses are zeroed.
    st = rar_workspace_init(ws, need, nranks, channelMask, proto, buffSize, stream);
    if (st != RAR_OK) return st;
  }
  return rar_allreduce(sendbufs, recvbufs, nranks, count, dtype, op, ring_order, channelMask, proto, buffSize,
                       chunkSteps, ws, (size_t)RAR_STATIC_WORKSPACE_BYTES, stream);
}
