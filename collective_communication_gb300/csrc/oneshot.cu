// oneshot.cu -- one-shot AllReduce over N virtual ranks: every rank reads all
// peers' inputs and reduces them itself.
//
// Pages cited (by title, then section):
//   [OS89] "perf(osar): all-reduce 5커널 → 3커널 (가드·웨이트 프롤로그 융합) - #89"
//          (the one-shot kernel: each rank copies in, then reduces all peers)
//   [NOTES] "NCCL" notes (cishoon.github.io), section "5 Symmetric Memory" (a
//          rank reads a peer's buffer by pointer; one kernel, one hop)
//
// On one GPU the ranks' buffers are already addressable by pointer, so the
// copy-in / signal / wait stages of the page's kernel have nothing to move or
// wait for: the N inputs are read directly, and since every rank's result is
// the same sum, each pack is reduced once and written to all N outputs.
//
// Sum: binary32, in user-rank order 0..N-1, starting from x_0 (no added
// zero), rounded once to bf16 for bf16 data.
#include "rar_launch.h"

namespace rar {

constexpr int kOneShotThreads = 256;

template <typename T>
struct OsPack;
template <>
struct OsPack<float> {
  static constexpr int kElems = 4;
  __device__ static __forceinline__ void widen(uint4 u, float (&v)[8]) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  }
  __device__ static __forceinline__ uint4 narrow(const float (&v)[8]) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
};
template <>
struct OsPack<uint16_t> {
  static constexpr int kElems = 8;
  __device__ static __forceinline__ void widen(uint4 u, float (&v)[8]) {
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
    v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
  }
  __device__ static __forceinline__ uint4 narrow(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
  }
};

template <typename T>
__device__ __forceinline__ float os_scalar(const T* p);
template <>
__device__ __forceinline__ float os_scalar<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float os_scalar<uint16_t>(const uint16_t* p) { return __uint_as_float((uint32_t)*p << 16); }
template <typename T>
__device__ __forceinline__ void os_store_scalar(T* p, float v);
template <>
__device__ __forceinline__ void os_store_scalar<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void os_store_scalar<uint16_t>(uint16_t* p, float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  *p = *reinterpret_cast<uint16_t*>(&b);
}

// Every rank's result is the same value, so each 16-byte pack is reduced
// once and stored to all N outputs (the N ranks' blocks of the page's kernel
// would each read all N inputs: N times the reads for the same sums). Peers
// are read in batches of kBatch ranks: every load of a batch is issued before
// any is added, so a thread keeps kBatch 16-byte loads in flight; the
// additions then run strictly in rank order.
constexpr int kBatch = 8;

template <typename T>
__global__ void __launch_bounds__(kOneShotThreads) oneshot_kernel(const __grid_constant__ OneShotArgs a) {
  constexpr int P = OsPack<T>::kElems;
  const int N = a.nranks;
  const int64_t npack = a.count / P;
  const int64_t stride = (int64_t)gridDim.x * kOneShotThreads;
  for (int64_t p = (int64_t)blockIdx.x * kOneShotThreads + threadIdx.x; p < npack; p += stride) {
    float acc[8];
    for (int q0 = 0; q0 < N; q0 += kBatch) {
      uint4 w[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; b++)
        if (q0 + b < N) w[b] = ld_stream_v4(reinterpret_cast<const T*>(a.send[q0 + b]) + p * P);
#pragma unroll
      for (int b = 0; b < kBatch; b++) {
        if (q0 + b < N) {
          float v[8];
          OsPack<T>::widen(w[b], v);
          if (q0 + b == 0) {
#pragma unroll
            for (int j = 0; j < P; j++) acc[j] = v[j];  // the sum starts at x_0
          } else {
#pragma unroll
            for (int j = 0; j < P; j++) acc[j] = __fadd_rn(acc[j], v[j]);
          }
        }
      }
    }
    const uint4 r = OsPack<T>::narrow(acc);
    for (int q = 0; q < N; q++) st_v4(reinterpret_cast<T*>(a.recv[q]) + p * P, r);
  }
  // ragged end (fewer than one 16-byte pack): block 0
  if (blockIdx.x == 0) {
    for (int64_t e = npack * P + threadIdx.x; e < a.count; e += kOneShotThreads) {
      float acc = os_scalar<T>(reinterpret_cast<const T*>(a.send[0]) + e);
      for (int q = 1; q < N; q++) acc = __fadd_rn(acc, os_scalar<T>(reinterpret_cast<const T*>(a.send[q]) + e));
      for (int q = 0; q < N; q++) os_store_scalar<T>(reinterpret_cast<T*>(a.recv[q]) + e, acc);
    }
  }
}

cudaError_t launch_oneshot(const OneShotArgs& a, cudaStream_t stream) {
  const int P = a.dtype == kF32 ? 4 : 8;
  const int64_t npack = a.count / P;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  static int sm_count[64] = {0};
  int sms = device < 64 ? sm_count[device] : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    if (device < 64) sm_count[device] = sms;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  // enough blocks to fill every SM several times over, never more than needed
  int64_t blocks = div_up(npack, kOneShotThreads);
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kOneShotThreads);
  if (a.dtype == kF32) return cudaLaunchKernelEx(&cfg, oneshot_kernel<float>, a);
  return cudaLaunchKernelEx(&cfg, oneshot_kernel<uint16_t>, a);
}

}  // namespace rar
