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
#include "rar_launch.h"

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
  // Every argument check first (rar_allreduce's codes, in its order), so
  // that a refused call makes no CUDA call and enqueues nothing.
  rar::RingArgs a;
  int grid = 0;
  rar_status st = rar::check_ring_call(rar::kAllReduce, sendbufs, recvbufs, nranks, count, dtype, op, ring_order, 1,
                                       channelMask, proto, buffSize, chunkSteps, 0u, &a, &grid);
  if (st != RAR_OK) return st;
  const int64_t need = rar::workspace_bytes_for(nranks, a.geo.nchan, a.geo.buff_size);
  if (need > (int64_t)RAR_STATIC_WORKSPACE_BYTES) return RAR_ERR_WORKSPACE;
  if (grid == 0) return RAR_OK;  // an empty call: nothing to clear or run
  void* ws = nullptr;
  st = static_ws_address(&ws);
  if (st != RAR_OK) return st;
  // Every call starts from a cleared workspace: header, status, abort flag
  // and step counters. Simple writes every FIFO byte before it reads it, so
  // its slots need no clearing; LL and LL128 accept lines by their flags, so
  // their FIFO lines are zeroed too (a line left by an earlier call could
  // otherwise carry a flag this call expects).
  const int64_t clear = a.geo.proto == rar::kSimple ? rar::kHeaderBytes + rar::conn_region_bytes(nranks, a.geo.nchan)
                                                    : need;
  st = rar::clear_workspace(ws, clear, nranks, channelMask, (int)proto, a.geo.buff_size, stream);
  if (st != RAR_OK) return st;
  a.ws = (char*)ws;
  return rar::launch_ring(a, grid, stream);
}
