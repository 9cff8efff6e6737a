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
// wait for: each rank's blocks read the N inputs directly. Block b serves
// rank b % N and tile b / N; the N blocks of a tile are adjacent in launch
// order, so they run together and the N-fold reads of one input tile are
// served mostly from L2.
//
// Sum: binary32, in user-rank order 0..N-1, starting from x_0 (no added
// zero), rounded once to bf16 for bf16 data.
#include <cstdio>

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

// Input loads of the one-shot: streamed past L1. The API refuses a receive
// buffer that overlaps any send buffer, so no store of the kernel can meet
// these loads and they carry no memory clobber: the compiler may issue all of
// a pack's peer loads back to back.
__device__ __forceinline__ uint4 os_load_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The ragged end (fewer elements than one 16-byte pack), done by tile 0 of
// each rank with the same rank-order sum, before the packs (so that nothing
// of it stays live across the pack loop).
template <typename T>
__device__ __forceinline__ void oneshot_ragged_end(const OneShotArgs& a, int rank, int64_t npack) {
  constexpr int P = OsPack<T>::kElems;
  T* out = reinterpret_cast<T*>(a.recv[rank]);
  for (int64_t e = npack * P + threadIdx.x; e < a.count; e += kOneShotThreads) {
    float acc = os_scalar<T>(reinterpret_cast<const T*>(a.send[0]) + e);
    for (int q = 1; q < a.nranks; q++) acc = __fadd_rn(acc, os_scalar<T>(reinterpret_cast<const T*>(a.send[q]) + e));
    os_store_scalar<T>(out + e, acc);
  }
}

// 1 to 8 ranks: the rank count is a template argument, so a pack's NR peer
// loads are issued together with no per-rank guard, and the kernel fits in
// 32 registers: 8 blocks of 256 threads (every warp slot of the SM) stay
// resident to cover the L2 latency of the N-fold reads. (With the rank count
// a runtime value the kernel needed about 60 registers, half the warps.)
template <typename T, int NR>
__global__ void __launch_bounds__(kOneShotThreads, 8) oneshot_kernel(const __grid_constant__ OneShotArgs a) {
  constexpr int P = OsPack<T>::kElems;
  const int rank = blockIdx.x % NR;
  const int64_t tile = blockIdx.x / NR;
  const int64_t ntiles = gridDim.x / NR;
  const int64_t npack = a.count / P;
  if (tile == 0) oneshot_ragged_end<T>(a, rank, npack);
  for (int64_t p = tile * kOneShotThreads + threadIdx.x; p < npack; p += ntiles * kOneShotThreads) {
    uint4 w[NR];
#pragma unroll
    for (int q = 0; q < NR; q++) w[q] = os_load_v4(reinterpret_cast<const T*>(a.send[q]) + p * P);
    float acc[8];
#pragma unroll
    for (int q = 0; q < NR; q++) {
      float v[8];
      OsPack<T>::widen(w[q], v);
#pragma unroll
      for (int j = 0; j < P; j++) acc[j] = q == 0 ? v[j] : __fadd_rn(acc[j], v[j]);  // the sum starts at x_0
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.recv[rank]) + p * P) = OsPack<T>::narrow(acc);
  }
}

// More than 8 ranks: peers are read in batches of kBatch, every load of a
// batch issued before any is added; the additions run strictly in rank order.
constexpr int kBatch = 8;

template <typename T>
__global__ void __launch_bounds__(kOneShotThreads) oneshot_wide_kernel(const __grid_constant__ OneShotArgs a) {
  constexpr int P = OsPack<T>::kElems;
  const int N = a.nranks;
  const int rank = blockIdx.x % N;
  const int64_t tile = blockIdx.x / N;
  const int64_t ntiles = gridDim.x / N;
  const int64_t npack = a.count / P;
  if (tile == 0) oneshot_ragged_end<T>(a, rank, npack);
  T* out = reinterpret_cast<T*>(a.recv[rank]);
  for (int64_t p = tile * kOneShotThreads + threadIdx.x; p < npack; p += ntiles * kOneShotThreads) {
    float acc[8];
    for (int q0 = 0; q0 < N; q0 += kBatch) {
      uint4 w[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; b++)
        if (q0 + b < N) w[b] = os_load_v4(reinterpret_cast<const T*>(a.send[q0 + b]) + p * P);
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
    st_v4(out + p * P, OsPack<T>::narrow(acc));
  }
}

template <typename T>
static const void* oneshot_kernel_for(int nranks) {
  switch (nranks) {
    case 1: return (const void*)oneshot_kernel<T, 1>;
    case 2: return (const void*)oneshot_kernel<T, 2>;
    case 3: return (const void*)oneshot_kernel<T, 3>;
    case 4: return (const void*)oneshot_kernel<T, 4>;
    case 5: return (const void*)oneshot_kernel<T, 5>;
    case 6: return (const void*)oneshot_kernel<T, 6>;
    case 7: return (const void*)oneshot_kernel<T, 7>;
    case 8: return (const void*)oneshot_kernel<T, 8>;
    default: return (const void*)oneshot_wide_kernel<T>;
  }
}

cudaError_t launch_oneshot(const OneShotArgs& a, cudaStream_t stream) {
  const int P = a.dtype == kF32 ? 4 : 8;
  const int64_t npack = a.count / P;
  int device = 0, sms = 0;
  const cudaError_t e = current_device_sms(&device, &sms);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  // enough tiles to fill every SM 8 blocks deep, never more than needed
  int64_t tiles = div_up(npack, (int64_t)kOneShotThreads);
  const int64_t cap = div_up((int64_t)sms * 8, a.nranks);
  if (tiles > cap) tiles = cap;
  if (tiles < 1) tiles = 1;
  cfg.gridDim = dim3((unsigned)(tiles * a.nranks));
  cfg.blockDim = dim3(kOneShotThreads);
  const void* fn = a.dtype == kF32 ? oneshot_kernel_for<float>(a.nranks) : oneshot_kernel_for<uint16_t>(a.nranks);
  if (trace_on())
    std::fprintf(stderr, "rar trace: oneshot nranks=%d count=%lld dtype=%s grid=%u (block b: rank b %% %d, tile b / %d) "
                 "threads=%d kernel=%s\n", a.nranks, (long long)a.count, a.dtype == kF32 ? "f32" : "bf16",
                 cfg.gridDim.x, a.nranks, a.nranks, kOneShotThreads,
                 a.nranks <= 8 ? "oneshot_kernel" : "oneshot_wide_kernel");
  void* params[] = {const_cast<OneShotArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, params);
}

}  // namespace rar
