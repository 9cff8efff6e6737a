// oneshot_staged.cu -- one-shot AllReduce in the staged form: every rank
// copies its input into a staging slot, publishes a sequence number once all
// of its blocks have copied, waits for every peer's number, then reduces the
// N staged copies. One launch per call, no reset between calls, so a CUDA
// graph of calls can be replayed any number of times.
//
// Pages cited (by title, then section):
//   [OS89] "perf(osar): all-reduce 5커널 → 3커널 (가드·웨이트 프롤로그 융합) - #89"
//          the five-kernel collective (guard, copy-in, signal, wait, reduce),
//          why guard and wait fold into the copy and reduce kernels (every
//          block can poll the same monotonic globals by itself), and the
//          follow-up single-kernel form: a monotonic done counter that every
//          launch advances by exactly its fixed grid, so the block whose
//          atomicAdd returns (grid - 1) modulo the grid is this launch's last
//          block to finish copying and publishes the sequence number; no reset
//          is needed, so CUDA graph replay works.
//
// Per call, for user rank r (blocks b with b % N == r, G blocks per rank):
//   guard    s = tx_seq[r] (read before this block copies); the staging slot
//            s % RING was last read in call s - RING: wait until every rank's
//            ack_seq has reached s - RING + 1.
//   copy     slot (r, s % RING) <- input of rank r (grid-stride over G blocks).
//   signal   fence, atomicAdd(done[r], 1); the block that gets (G-1) mod G
//            publishes tx_seq[r] = s + 1 (release).
//   wait     every block waits until tx_seq[q] >= s + 1 for all q (acquire).
//   reduce   out_r = T(sum over q = 0..N-1 of slot (q, s % RING)), binary32, in
//            user-rank order, rounded once for bf16; rank r's blocks take
//            chunks of packs from a counter grab[r][s % RING].
//   ack      fence, atomicAdd(read[r], 1); the last block resets grab[r][s %
//            RING] and publishes ack_seq[r] = s + 1: rank r has finished
//            reading call s's slots.
// A block reads tx_seq before its own atomicAdd, and the block that publishes
// s + 1 exists only after every block of the launch has added, so no block of
// this launch can read s + 1 at entry. All N*G blocks wait on each other, so
// the launch is cooperative (all blocks resident, or the launch is refused).
// Every wait is bounded; a wait that runs out raises the workspace's abort
// flag and every other wait then ends too.
#include <cstdio>

#include "rar_launch.h"

namespace rar {

constexpr int kStagedThreads = 256;
constexpr int64_t kGrabPacks = 2 * kStagedThreads;  // packs of one reduce chunk

__device__ __forceinline__ OsHeader* os_header(const StagedArgs& a) { return (OsHeader*)a.ws; }
__device__ __forceinline__ OsControl* os_control(const StagedArgs& a, int rank) {
  return (OsControl*)(a.ws + kHeaderBytes) + rank;
}
// Slot (rank, s mod kStagingSlots); slot_bytes is the workspace's, from its header.
__device__ __forceinline__ char* os_slot(const StagedArgs& a, int64_t slot_bytes, int rank, uint64_t s) {
  return a.ws + a.stage_offset + ((int64_t)rank * kStagingSlots + (int64_t)(s % kStagingSlots)) * slot_bytes;
}

template <typename T>
struct StPack;
template <>
struct StPack<float> {
  static constexpr int kElems = 4;
  __device__ static __forceinline__ void widen(uint4 u, float (&v)[8]) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  }
  __device__ static __forceinline__ uint4 narrow(const float (&v)[8]) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
  __device__ static __forceinline__ float scalar(const char* p) { return __uint_as_float(ld_cg_u32(p)); }
  __device__ static __forceinline__ void store_scalar(float* p, float v) { *p = v; }
};
template <>
struct StPack<uint16_t> {
  static constexpr int kElems = 8;
  __device__ static __forceinline__ void widen(uint4 u, float (&v)[8]) {
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
    v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
  }
  __device__ static __forceinline__ uint4 narrow(const float (&v)[8]) {
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
  }
  __device__ static __forceinline__ float scalar(const char* p) {
    uint16_t h;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p) : "memory");
    return __uint_as_float((uint32_t)h << 16);
  }
  __device__ static __forceinline__ void store_scalar(uint16_t* p, float v) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    *p = *reinterpret_cast<uint16_t*>(&b);
  }
};

// One thread's bounded wait until *p >= want. Returns false when it gave up.
__device__ __forceinline__ bool os_wait_at_least(const StagedArgs& a, const uint64_t* p, uint64_t want,
                                                 uint64_t info) {
  Spin sp;
  while (ld_acquire_u64(p) < want) {
    if (sp.poll_h(os_header(a), a.timeout_ns, info, want)) return false;
  }
  return true;
}

// NR > 0: the rank count as a template argument (up to 8 ranks), so that a
// pack's NR slot loads are issued together with no per-rank guard; NR == 0:
// any rank count, the slots read in batches of 8 ranks.
template <typename T, int NR>
__global__ void __launch_bounds__(kStagedThreads, kStagedBlocksPerSm) oneshot_staged_kernel(const __grid_constant__ StagedArgs a) {
  constexpr int P = StPack<T>::kElems;
  constexpr int kBatchRanks = 8;
  __shared__ uint64_t sh_s;
  __shared__ int64_t sh_slot_bytes;
  __shared__ int sh_stop;
  __shared__ int64_t sh_chunk[2];
  const int N = a.nranks, G = a.blocks_per_rank;
  const int rank = blockIdx.x % N;
  const int j = blockIdx.x / N;
  const uint64_t info = (uint64_t)blockIdx.x << 32;
  OsHeader* h = os_header(a);
  OsControl* me = os_control(a, rank);

  // ---- entry check and guard ----
  if (threadIdx.x == 0) {
    sh_stop = 0;
    sh_slot_bytes = h->slot_bytes;
    if (h->magic != kStagedMagic || h->nranks != N || h->dtype != a.dtype || h->blocks_per_rank != G ||
        a.count > h->max_count || a.count * (int64_t)sizeof(T) > h->slot_bytes) {
      report_failure(h, kErrWorkspace, info, 0);
      sh_stop = 1;
    } else if (ld_relaxed_u32(&h->abort) != 0u) {
      atomicCAS(&h->status, 0u, kErrAbort);
      sh_stop = 1;
    } else {
      sh_s = ld_acquire_u64(&me->tx_seq);
    }
  }
  __syncthreads();
  if (sh_stop) return;
  const uint64_t s = sh_s;
  const int64_t sb = sh_slot_bytes;
  // guard: thread q < N waits for rank q's acknowledgement (the N waits run
  // side by side; the block barrier then orders the copy after all of them)
  if (threadIdx.x < N && s + 1 > kStagingSlots &&
      !os_wait_at_least(a, &os_control(a, threadIdx.x)->ack_seq, s + 1 - kStagingSlots,
                        info | (1u << 24) | threadIdx.x))
    sh_stop = 1;
  __syncthreads();
  if (sh_stop) return;

  // ---- copy the rank's input into its slot ----
  const int64_t npack = a.count / P;
  {
    const T* src = reinterpret_cast<const T*>(a.send[rank]);
    char* dst = os_slot(a, sb, rank, s);
    // kCopyUnroll loads in flight per thread before their stores (one at a
    // time, the copy was bound by the loads' latency)
    constexpr int kCopyUnroll = 4;
    const int64_t stride = (int64_t)G * kStagedThreads;
    int64_t p = (int64_t)j * kStagedThreads + threadIdx.x;
    for (; p + (kCopyUnroll - 1) * stride < npack; p += kCopyUnroll * stride) {
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; u++) v[u] = ld_stream_v4(src + (p + u * stride) * P);
#pragma unroll
      for (int u = 0; u < kCopyUnroll; u++) st_v4(dst + (p + u * stride) * 16, v[u]);
    }
    for (; p < npack; p += stride) st_v4(dst + p * 16, ld_stream_v4(src + p * P));
    if (j == 0)
      for (int64_t e = npack * P + threadIdx.x; e < a.count; e += kStagedThreads)
        reinterpret_cast<T*>(dst)[e] = src[e];
  }
  __syncthreads();

  // ---- signal, then wait for every peer ----
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();  // the block's copies are visible before its count
    const uint64_t old = atom_add_acq_rel_u64(&me->done, 1);
    if (old % (uint64_t)G == (uint64_t)G - 1) st_release_u64(&me->tx_seq, s + 1);
    sh_chunk[0] = (int64_t)atomicAdd(reinterpret_cast<unsigned long long*>(&me->grab[s % kStagingSlots]), 1ull);
  }
  // thread q < N waits for rank q's sequence number, side by side
  if (threadIdx.x < N && !os_wait_at_least(a, &os_control(a, threadIdx.x)->tx_seq, s + 1, info | (2u << 24) | threadIdx.x))
    sh_stop = 1;
  __syncthreads();
  if (sh_stop) return;

  // ---- reduce the N staged copies, in user-rank order ----
  // The rank's packs go out in chunks of kGrabPacks from a counter of the
  // slot, so that blocks on SMs with more L2 bandwidth take more chunks (the
  // first chunk was taken before the wait). The call's last reader resets the
  // counter before it acknowledges; the slot's next call passes the guard
  // only after that.
  T* out = reinterpret_cast<T*>(a.recv[rank]);
  const int64_t nchunks = (npack + kGrabPacks - 1) / kGrabPacks;
  unsigned long long* grab = reinterpret_cast<unsigned long long*>(&me->grab[s % kStagingSlots]);
  for (int cur = 0;; cur ^= 1) {
    const int64_t chunk = sh_chunk[cur];
    if (chunk >= nchunks) break;
    if (threadIdx.x == 0) sh_chunk[cur ^ 1] = (int64_t)atomicAdd(grab, 1ull);  // the next chunk, ahead
    const int64_t p_end = (chunk + 1) * kGrabPacks < npack ? (chunk + 1) * kGrabPacks : npack;
    for (int64_t p = chunk * kGrabPacks + threadIdx.x; p < p_end; p += kStagedThreads) {
      float acc[8];
      if constexpr (NR > 0) {
        const char* slot0 = os_slot(a, sb, 0, s) + p * 16;
        const int64_t rank_stride = (int64_t)kStagingSlots * sb;  // slot (q, s) to slot (q + 1, s)
        uint4 w[NR];
#pragma unroll
        for (int q = 0; q < NR; q++) w[q] = ld_cg_v4(slot0 + q * rank_stride);
#pragma unroll
        for (int q = 0; q < NR; q++) {
          float v[8];
          StPack<T>::widen(w[q], v);
#pragma unroll
          for (int k = 0; k < P; k++) acc[k] = q == 0 ? v[k] : __fadd_rn(acc[k], v[k]);  // the sum starts at x_0
        }
      } else {
        for (int q0 = 0; q0 < N; q0 += kBatchRanks) {
          uint4 w[kBatchRanks];
#pragma unroll
          for (int b = 0; b < kBatchRanks; b++)
            if (q0 + b < N) w[b] = ld_cg_v4(os_slot(a, sb, q0 + b, s) + p * 16);
#pragma unroll
          for (int b = 0; b < kBatchRanks; b++) {
            if (q0 + b < N) {
              float v[8];
              StPack<T>::widen(w[b], v);
              if (q0 + b == 0) {
#pragma unroll
                for (int k = 0; k < P; k++) acc[k] = v[k];  // the sum starts at x_0
              } else {
#pragma unroll
                for (int k = 0; k < P; k++) acc[k] = __fadd_rn(acc[k], v[k]);
              }
            }
          }
        }
      }
      st_v4(out + p * P, StPack<T>::narrow(acc));
    }
    __syncthreads();  // every thread has read sh_chunk[cur]; thread 0's next chunk is visible
  }
  if (j == 0) {
    for (int64_t e = npack * P + threadIdx.x; e < a.count; e += kStagedThreads) {
      float acc = StPack<T>::scalar(os_slot(a, sb, 0, s) + e * (int64_t)sizeof(T));
      for (int q = 1; q < N; q++) acc = __fadd_rn(acc, StPack<T>::scalar(os_slot(a, sb, q, s) + e * (int64_t)sizeof(T)));
      StPack<T>::store_scalar(out + e, acc);
    }
  }
  __syncthreads();

  // ---- acknowledge: this rank has read call s's slots ----
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();
    const uint64_t old = atom_add_acq_rel_u64(&me->read, 1);
    if (old % (uint64_t)G == (uint64_t)G - 1) {
      st_relaxed_u64(&me->grab[s % kStagingSlots], 0);  // every block of this call has taken its last chunk
      if (a.fault != kFaultDropAck) st_release_u64(&me->ack_seq, s + 1);
    }
  }
}

template <typename T>
static const void* staged_kernel_for(int nranks) {
  switch (nranks) {
    case 1: return (const void*)oneshot_staged_kernel<T, 1>;
    case 2: return (const void*)oneshot_staged_kernel<T, 2>;
    case 3: return (const void*)oneshot_staged_kernel<T, 3>;
    case 4: return (const void*)oneshot_staged_kernel<T, 4>;
    case 5: return (const void*)oneshot_staged_kernel<T, 5>;
    case 6: return (const void*)oneshot_staged_kernel<T, 6>;
    case 7: return (const void*)oneshot_staged_kernel<T, 7>;
    case 8: return (const void*)oneshot_staged_kernel<T, 8>;
    default: return (const void*)oneshot_staged_kernel<T, 0>;
  }
}

int staged_blocks_per_rank(int nranks, int sms) {
  const int g = sms * kStagedBlocksPerSm / nranks;
  return g < 1 ? 1 : g;
}

cudaError_t launch_oneshot_staged(const StagedArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3((unsigned)(a.nranks * a.blocks_per_rank));
  cfg.blockDim = dim3(kStagedThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (trace_on())
    std::fprintf(stderr, "rar trace: oneshot_staged nranks=%d count=%lld dtype=%s grid=%u blocks_per_rank=%d "
                 "threads=%d kernel=oneshot_staged_kernel (cooperative)\n", a.nranks, (long long)a.count,
                 a.dtype == kF32 ? "f32" : "bf16", cfg.gridDim.x, a.blocks_per_rank, kStagedThreads);
  const void* fn = a.dtype == kF32 ? staged_kernel_for<float>(a.nranks) : staged_kernel_for<uint16_t>(a.nranks);
  void* params[] = {const_cast<StagedArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, fn, params);
}

}  // namespace rar
