// ring_simple.cu -- ring AllReduce, Simple protocol, all N virtual ranks in
// one launch (one block per (rank, channel)).
//
// Pages cited (by title, then section):
//   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
//         sections "Simple 的线程角色", "Simple 的 Credit 与 Step", "发布顺序与 Fence",
//         "Slice Size", "Primitive API 是模板组合"
//   [C12] "NCCL 专家课程 12：Ring AllReduce 逐步推导、真实 Ring 与 Channel 并行"
//         sections "源码步骤一" .. "源码步骤五"
//
// Block organisation (the page's wait / worker / post roles, on Blackwell
// mbarriers instead of paired named barriers, so the roles run decoupled):
//   warp 0, lane 0  waiter: for slice i, waits until the receive FIFO holds it
//                   (tail >= step + StepPerSlice) and the send FIFO has room
//                   (head + NCCL_STEPS >= step + StepPerSlice), then arrives on
//                   full[i % D];
//   warps 2..       workers: wait full[i % D], move the slice with 16-byte
//                   vector loads/stores (reduce in binary32), arrive done[i % D];
//   warp 1, lane 0  poster: waits done[i % D], then fence.acq_rel.gpu and
//                   publish tail (payload first, then the tail), publish head,
//                   arrive empty[i % D] so the waiter may reuse the slot.
// The waiter may run up to D slices ahead of the poster. Empty slices still
// wait and post, so both ends of every connection count the same steps.
#include "rar_device.cuh"

namespace rar {

constexpr int kDepth = 4;  // mbarrier ring depth

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<float> {
  static constexpr int kPack = 4;  // elements per 16-byte pack
  static constexpr int kUnroll = 4;
};
template <>
struct ElemTraits<uint16_t> {
  static constexpr int kPack = 8;
  static constexpr int kUnroll = 2;
};

// --- 16-byte pack helpers --------------------------------------------------
// x: user input pack (T) widened to binary32.
template <typename T>
__device__ __forceinline__ void load_input_pack(const T* p, float (&v)[ElemTraits<T>::kPack]);
template <>
__device__ __forceinline__ void load_input_pack<float>(const float* p, float (&v)[4]) {
  uint4 u = ld_stream_v4(p);
  v[0] = __uint_as_float(u.x);
  v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z);
  v[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void load_input_pack<uint16_t>(const uint16_t* p, float (&v)[8]) {
  uint4 u = ld_stream_v4(p);
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x);
  v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z);
  v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}

// Partial sums in the FIFO are binary32: kPack * 4 bytes per pack.
template <int P>
__device__ __forceinline__ void load_partial_pack(const char* p, float (&v)[P]) {
#pragma unroll
  for (int q = 0; q < P / 4; q++) {
    uint4 u = ld_cg_v4(p + 16 * q);
    v[4 * q + 0] = __uint_as_float(u.x);
    v[4 * q + 1] = __uint_as_float(u.y);
    v[4 * q + 2] = __uint_as_float(u.z);
    v[4 * q + 3] = __uint_as_float(u.w);
  }
}
template <int P>
__device__ __forceinline__ void store_partial_pack(char* p, const float (&v)[P]) {
#pragma unroll
  for (int q = 0; q < P / 4; q++)
    st_v4(p + 16 * q, make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                                 __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])));
}
// Final values (T): one 16-byte pack. For bf16 the binary32 sum is rounded
// once here (round to nearest even).
template <typename T>
__device__ __forceinline__ uint4 to_final_pack(const float (&v)[ElemTraits<T>::kPack]);
template <>
__device__ __forceinline__ uint4 to_final_pack<float>(const float (&v)[4]) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
template <>
__device__ __forceinline__ uint4 to_final_pack<uint16_t>(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// --- scalar helpers for the ragged end of a slice --------------------------
template <typename T>
__device__ __forceinline__ float load_input_scalar(const T* p);
template <>
__device__ __forceinline__ float load_input_scalar<float>(const float* p) {
  return __uint_as_float(ld_cg_u32(p));
}
template <>
__device__ __forceinline__ float load_input_scalar<uint16_t>(const uint16_t* p) {
  uint16_t h;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p) : "memory");
  return __uint_as_float((uint32_t)h << 16);
}
template <typename T>
__device__ __forceinline__ T final_scalar(float v);
template <>
__device__ __forceinline__ float final_scalar<float>(float v) { return v; }
template <>
__device__ __forceinline__ uint16_t final_scalar<uint16_t>(float v) {
  __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&b);
}
template <typename T>
__device__ __forceinline__ T load_final_scalar(const char* p);
template <>
__device__ __forceinline__ float load_final_scalar<float>(const char* p) { return __uint_as_float(ld_cg_u32(p)); }
template <>
__device__ __forceinline__ uint16_t load_final_scalar<uint16_t>(const char* p) {
  uint16_t h;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p) : "memory");
  return h;
}

// --- the five primitives on one slice --------------------------------------
// in/out: user buffers at the slice's first element; rslot/sslot: FIFO bytes
// of the slice on the receive / send connection.
template <typename T, int PRIM>
__device__ __forceinline__ void move_slice(const T* __restrict__ in, T* __restrict__ out, const char* rslot,
                                           char* sslot, int64_t nelem, int wt, int nwt) {
  constexpr int P = ElemTraits<T>::kPack;
  constexpr int U = ElemTraits<T>::kUnroll;
  constexpr bool kIn = PRIM == kSend || PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend;
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend;
  constexpr bool kRecvFinal = PRIM == kRecvCopySend || PRIM == kRecv;
  constexpr bool kSendPartial = PRIM == kSend || PRIM == kRecvReduceSend;
  constexpr bool kSendFinal = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv;

  const int64_t npack = nelem / P;
  for (int64_t p0 = wt; p0 < npack; p0 += (int64_t)nwt * U) {
    float x[U][P];
    float part[U][P];
    uint4 fin[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      int64_t p = p0 + (int64_t)u * nwt;
      if (p < npack) {
        if (kIn) load_input_pack<T>(in + p * P, x[u]);
        if (kRecvPartial) load_partial_pack<P>(rslot + p * P * 4, part[u]);
        if (kRecvFinal) fin[u] = ld_cg_v4(rslot + p * 16);
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      int64_t p = p0 + (int64_t)u * nwt;
      if (p < npack) {
        if (PRIM == kSend) {
          store_partial_pack<P>(sslot + p * P * 4, x[u]);
        } else if (PRIM == kRecvReduceSend) {
#pragma unroll
          for (int j = 0; j < P; j++) part[u][j] = __fadd_rn(part[u][j], x[u][j]);
          store_partial_pack<P>(sslot + p * P * 4, part[u]);
        } else if (PRIM == kRecvReduceCopySend) {
#pragma unroll
          for (int j = 0; j < P; j++) part[u][j] = __fadd_rn(part[u][j], x[u][j]);
          fin[u] = to_final_pack<T>(part[u]);
        }
        if (kOut) st_v4(out + p * P, fin[u]);
        if (kSendFinal) st_v4(sslot + p * 16, fin[u]);
        (void)kSendPartial;
      }
    }
  }
  // ragged end: fewer than P elements, one per thread
  for (int64_t e = npack * P + wt; e < nelem; e += nwt) {
    float xv = 0.f, pv = 0.f;
    T fv{};
    if (kIn) xv = load_input_scalar<T>(in + e);
    if (kRecvPartial) pv = __uint_as_float(ld_cg_u32(rslot + e * 4));
    if (kRecvFinal) fv = load_final_scalar<T>(rslot + e * sizeof(T));
    if (PRIM == kSend) {
      *reinterpret_cast<float*>(sslot + e * 4) = xv;
    } else if (PRIM == kRecvReduceSend) {
      *reinterpret_cast<float*>(sslot + e * 4) = __fadd_rn(pv, xv);
    } else if (PRIM == kRecvReduceCopySend) {
      fv = final_scalar<T>(__fadd_rn(pv, xv));
    }
    if (kOut) out[e] = fv;
    if (kSendFinal) *reinterpret_cast<T*>(sslot + e * sizeof(T)) = fv;
  }
}

template <typename T>
__device__ __forceinline__ void move_slice_any(int prim, const T* in, T* out, const char* rslot, char* sslot,
                                               int64_t nelem, int wt, int nwt) {
  switch (prim) {
    case kSend: move_slice<T, kSend>(in, out, rslot, sslot, nelem, wt, nwt); break;
    case kRecvReduceSend: move_slice<T, kRecvReduceSend>(in, out, rslot, sslot, nelem, wt, nwt); break;
    case kRecvReduceCopySend: move_slice<T, kRecvReduceCopySend>(in, out, rslot, sslot, nelem, wt, nwt); break;
    case kRecvCopySend: move_slice<T, kRecvCopySend>(in, out, rslot, sslot, nelem, wt, nwt); break;
    default: move_slice<T, kRecv>(in, out, rslot, sslot, nelem, wt, nwt); break;
  }
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT, 1) ring_simple_kernel(const __grid_constant__ RingArgs a) {
  constexpr int kWorkers = NT - 64;  // warps 2.. are workers
  __shared__ uint64_t bar_full[kDepth], bar_done[kDepth], bar_empty[kDepth];
  __shared__ volatile int sh_abort;
  __shared__ int sh_chan;
  __shared__ uint64_t sh_base_send, sh_base_recv;

  const Geometry& g = a.geo;
  if (threadIdx.x == 0) sh_chan = -1;
  __syncthreads();
  int rank, dense;
  map_block(a, &rank, &dense, &sh_chan);
  __syncthreads();
  const int N = g.nranks;
  const int ring_idx = a.ring_index[rank];
  const int e_send = ring_idx, e_recv = (ring_idx + N - 1) % N;
  ConnCounters* cs = conn_at(a, dense, e_send);
  ConnCounters* cr = conn_at(a, dense, e_recv);
  char* fifo_send = fifo_at(a, dense, e_send);
  const char* fifo_recv = fifo_at(a, dense, e_recv);

  if (threadIdx.x == 0) {
    sh_abort = entry_check(a) ? 0 : 1;
    for (int d = 0; d < kDepth; d++) {
      mbar_init(&bar_full[d], 1);
      mbar_init(&bar_done[d], kWorkers);
      mbar_init(&bar_empty[d], 1);
    }
    // This block alone writes the tail of its send edge and the head of its
    // receive edge; both equal the previous call's final step. Slices start
    // on a multiple of NCCL_STEPS so that no slice wraps around the ring.
    sh_base_send = round_up_steps(ld_relaxed_u64(&cs->tail));
    sh_base_recv = round_up_steps(ld_relaxed_u64(&cr->head));
    reinterpret_cast<uint8_t*>(a.ws + kTraceOffset)[blockIdx.x] = (uint8_t)sh_chan;
  }
  __syncthreads();
  if (sh_abort) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t sps = (uint64_t)g.sps;
  const uint64_t base_send = sh_base_send, base_recv = sh_base_recv;
  const uint64_t info = ((uint64_t)blockIdx.x << 32);
  SliceCursor c;
  cursor_begin(g, dense, ring_idx, c);

  if (warp == 0) {
    if (lane != 0) return;
    // ---- waiter ----
    uint64_t rstep = base_recv, sstep = base_send, tail_seen = 0, head_seen = 0;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      if (use > 0 && !mbar_wait(a, &bar_empty[d], (use - 1) & 1u, info | (1u << 24) | i)) sh_abort = 1;
      if (!sh_abort && row_recvs(c.prim)) {
        Spin sp;
        while (tail_seen < rstep + sps) {
          tail_seen = ld_acquire_u64(&cr->tail);
          if (tail_seen >= rstep + sps) break;
          if (sp.poll(a, info | (2u << 24) | i, rstep + sps)) { sh_abort = 1; break; }
        }
      }
      if (!sh_abort && row_sends(c.prim)) {
        Spin sp;
        // Until the receiver's first release in this call, its head may still
        // hold the previous call's final step (< base_send): all slots free.
        while ((head_seen > base_send ? head_seen : base_send) + kSteps < sstep + sps) {
          head_seen = ld_acquire_u64(&cs->head);
          if ((head_seen > base_send ? head_seen : base_send) + kSteps >= sstep + sps) break;
          if (sp.poll(a, info | (3u << 24) | i, sstep + sps)) { sh_abort = 1; break; }
        }
      }
      mbar_arrive(&bar_full[d]);
      if (sh_abort) break;
      if (row_recvs(c.prim)) rstep += sps;
      if (row_sends(c.prim)) sstep += sps;
    }
  } else if (warp == 1) {
    if (lane != 0) return;
    // ---- poster ----
    uint64_t rstep = base_recv, sstep = base_send;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      if (!mbar_wait(a, &bar_done[d], use & 1u, info | (4u << 24) | i)) { sh_abort = 1; break; }
      if (sh_abort) break;
      if (row_sends(c.prim)) {
        sstep += sps;
        fence_acq_rel_gpu();  // the workers' payload is visible before the tail
        st_relaxed_u64(&cs->tail, sstep);
      }
      if (row_recvs(c.prim)) {
        rstep += sps;
        if (a.fault != kFaultDropHead) st_relaxed_u64(&cr->head, rstep);  // release the slots read
      }
      mbar_arrive(&bar_empty[d]);
    }
  } else {
    // ---- workers ----
    const int wt = threadIdx.x - 64;
    const T* in = reinterpret_cast<const T*>(a.send[rank]);
    T* out = reinterpret_cast<T*>(a.recv[rank]);
    const int64_t step_bytes = g.step_bytes;
    uint64_t rstep = base_recv, sstep = base_send;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      bool ok = mbar_wait(a, &bar_full[d], use & 1u, info | (5u << 24) | i);
      if (!ok || sh_abort) {
        mbar_arrive(&bar_done[d]);
        break;
      }
      const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
      char* sslot = fifo_send + (int64_t)(sstep % kSteps) * step_bytes;
      move_slice_any<T>(c.prim, in + c.offset, out + c.offset, rslot, sslot, c.nelem, wt, kWorkers);
      mbar_arrive(&bar_done[d]);
      if (row_recvs(c.prim)) rstep += sps;
      if (row_sends(c.prim)) sstep += sps;
    }
  }
}

// Host-side launch of the Simple kernel (declared in rar_launch.h).
cudaError_t launch_ring_simple(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out) {
  constexpr int kThreads = 544;  // 2 control warps + 15 worker warps (the page's Simple blockX)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (threads_out) *threads_out = kThreads;
  if (a.geo.dtype == kF32) return cudaLaunchKernelEx(&cfg, ring_simple_kernel<float, kThreads>, a);
  return cudaLaunchKernelEx(&cfg, ring_simple_kernel<uint16_t, kThreads>, a);
}

}  // namespace rar
