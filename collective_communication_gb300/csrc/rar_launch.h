// rar_launch.h -- host-side launchers of the kernels of librar.so.
#pragma once

#include <cuda_runtime.h>

#include "rar_device.cuh"

namespace rar {

// Cooperative launch of one block per (rank, channel); grid = nranks * C.
cudaError_t launch_ring_simple(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out);
cudaError_t launch_ring_line(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out);

struct OneShotArgs {
  const void* send[kMaxRanks];
  void* recv[kMaxRanks];
  int nranks;
  int dtype;
  int64_t count;
};
cudaError_t launch_oneshot(const OneShotArgs& a, cudaStream_t stream);

}  // namespace rar
