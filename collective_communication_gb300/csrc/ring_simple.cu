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
// Block organisation: the page's wait / worker / post roles, decoupled by
// shared-memory mbarriers, with the workers' loads moved onto the TMA engine:
//   warp 0, lane 0  waiter: for slice i, waits until the receive FIFO holds it
//                   (tail >= step + StepPerSlice) and the send FIFO has room
//                   (head + NCCL_STEPS >= step + StepPerSlice), both polled in
//                   one loop; arrives ready[i % D].
//   warp 1, lane 0  loader: streams the slice in tiles of kTileElems elements:
//                   bulk copies (cp.async.bulk) of the user input (the first
//                   tile's as soon as a stage is free, before ready[i % D]) and,
//                   after ready[i % D], of the received FIFO bytes into a ring
//                   of smem stages, completion counted in bytes on full[stage].
//   warps 3..10     workers: per tile, wait full[stage], reduce from shared
//                   memory in binary32, store the FIFO output and the user output
//                   with 16-byte stores, release the stage (empty[stage]); after
//                   the slice's last tile arrive done[i % D].
//   warp 2, lane 0  poster: after ready[i % D] and done[i % D], publish the head
//                   (the slots read), then fence.acq_rel.gpu and publish the
//                   tail (payload first, then the tail); arrive free[i % D] so
//                   the waiter may reuse the slot.
// Up to D slices are in flight between waiter and poster, and up to
// `nstages` tiles between loader and workers (about 190 KB of loads in flight
// per SM). Empty slices still wait and post, so both ends of every connection
// count the same steps.
#include <cstdio>

#include "rar_launch.h"

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

// --- one tile of a slice ---------------------------------------------------
// s_in / s_rcv: the tile's user input and received FIFO bytes in shared
// memory (the pack-aligned prefix of `covered` elements); g_in / g_out: user
// buffers at the slice's first element; rslot / sslot: the slice's FIFO bytes
// on the receive / send connection; e0: the tile's first element in the slice.
// DIRECT (all-gather hops of the direct mode): final values go straight to
// the next rank's output (g_next) instead of the send FIFO, and a received
// final is already in this rank's own output (staged from there, not from the
// FIFO), so it is neither stored again nor, on the last row, moved at all.
// covered == 0 (a slice whose user pointers are not 16-byte aligned, which
// only a ragged block of the halves gives): every element takes the scalar path.
template <typename T, int PRIM, bool DIRECT>
__device__ __forceinline__ void tile_compute(const char* s_in, const char* s_rcv, const T* __restrict__ g_in,
                                             T* __restrict__ g_out, T* __restrict__ g_next, const char* rslot,
                                             char* sslot, int64_t e0, int ne, int covered, int ct, int nct,
                                             uint64_t out_policy) {
  constexpr int P = ElemTraits<T>::kPack;
  constexpr bool kReduce = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kFinalOfSum = PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kIn = PRIM == kSend || kReduce || PRIM == kCopySend;
  constexpr bool kRecvPartial = kReduce;
  constexpr bool kRecvFinal = (PRIM == kRecvCopySend || PRIM == kRecv) && !(DIRECT && PRIM == kRecv);
  constexpr bool kSendPartial = PRIM == kSend || PRIM == kRecvReduceSend;
  constexpr bool kForward = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kCopySend;
  constexpr bool kSendFinal = kForward && !DIRECT;
  constexpr bool kSendNext = kForward && DIRECT;
  constexpr bool kOut = kFinalOfSum || PRIM == kCopySend || ((PRIM == kRecvCopySend || PRIM == kRecv) && !DIRECT);
  if constexpr (DIRECT && PRIM == kRecv) return;  // the data is already in place
  constexpr int U = 4;
  const int npacks = covered / P;
  for (int j0 = ct; j0 < npacks; j0 += nct * U) {
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int j = j0 + u * nct;
      if (j < npacks) {
        const int64_t e = e0 + (int64_t)j * P;
        float x[P], v[P];
        uint4 fin, w = make_uint4(0u, 0u, 0u, 0u);
        if (kIn) w = *reinterpret_cast<const uint4*>(s_in + j * 16);
        if (kIn && PRIM != kCopySend) {
          if constexpr (P == 4) {
            x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
            x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
          } else {
            x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
            x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
          }
        }
        if (kRecvPartial) {
#pragma unroll
          for (int q = 0; q < P / 4; q++) {
            const float4 w = *reinterpret_cast<const float4*>(s_rcv + j * P * 4 + 16 * q);
            v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
          }
#pragma unroll
          for (int k = 0; k < P; k++) v[k] = __fadd_rn(v[k], x[k]);
        } else if (PRIM == kSend) {
#pragma unroll
          for (int k = 0; k < P; k++) v[k] = x[k];
        }
        if (kRecvFinal) fin = *reinterpret_cast<const uint4*>(s_rcv + j * 16);
        if (kFinalOfSum) fin = to_final_pack<T>(v);
        if (PRIM == kCopySend) fin = w;  // the input is already a final value
        if (kSendPartial) store_partial_pack<P>(sslot + e * 4, v);
        if (kSendFinal) st_v4(sslot + e * (int64_t)sizeof(T), fin);
        if (kSendNext) st_v4(g_next + e, fin);  // read back by the next rank: default L2 policy
        if (kOut) st_v4_policy(g_out + e, fin, out_policy);  // streamed out: evict-first in L2
      }
    }
  }
  // the last < P elements of a slice: plain loads straight from global memory
  for (int k = covered + ct; k < ne; k += nct) {
    const int64_t e = e0 + k;
    float xv = 0.f, pv = 0.f;
    T fv{};
    if (kIn && PRIM != kCopySend) xv = load_input_scalar<T>(g_in + e);
    if (PRIM == kCopySend) fv = load_final_scalar<T>(reinterpret_cast<const char*>(g_in + e));
    if (kRecvPartial) pv = __uint_as_float(ld_cg_u32(rslot + e * 4));
    if (kRecvFinal)
      fv = DIRECT ? load_final_scalar<T>(reinterpret_cast<const char*>(g_out + e))
                  : load_final_scalar<T>(rslot + e * (int64_t)sizeof(T));
    if (PRIM == kSend) {
      *reinterpret_cast<float*>(sslot + e * 4) = xv;
    } else if (PRIM == kRecvReduceSend) {
      *reinterpret_cast<float*>(sslot + e * 4) = __fadd_rn(pv, xv);
    } else if (kFinalOfSum) {
      fv = final_scalar<T>(__fadd_rn(pv, xv));
    }
    if (kOut) g_out[e] = fv;
    if (kSendFinal) *reinterpret_cast<T*>(sslot + e * (int64_t)sizeof(T)) = fv;
    if (kSendNext) g_next[e] = fv;
  }
}

template <typename T, bool DIRECT>
__device__ __forceinline__ void tile_compute_prim(int prim, const char* s_in, const char* s_rcv, const T* g_in,
                                                  T* g_out, T* g_next, const char* rslot, char* sslot, int64_t e0,
                                                  int ne, int covered, int ct, int nct, uint64_t pol) {
  switch (prim) {
    case kSend:
      tile_compute<T, kSend, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct, nct, pol);
      break;
    case kRecvReduceSend:
      tile_compute<T, kRecvReduceSend, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct,
                                               nct, pol);
      break;
    case kRecvReduceCopySend:
      tile_compute<T, kRecvReduceCopySend, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered,
                                                   ct, nct, pol);
      break;
    case kRecvCopySend:
      tile_compute<T, kRecvCopySend, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct,
                                             nct, pol);
      break;
    case kRecvReduceCopy:
      tile_compute<T, kRecvReduceCopy, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct,
                                               nct, pol);
      break;
    case kCopySend:
      tile_compute<T, kCopySend, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct, nct,
                                         pol);
      break;
    default:
      tile_compute<T, kRecv, DIRECT>(s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct, nct, pol);
      break;
  }
}

template <typename T>
__device__ __forceinline__ void tile_compute_any(bool direct, int prim, const char* s_in, const char* s_rcv,
                                                 const T* g_in, T* g_out, T* g_next, const char* rslot, char* sslot,
                                                 int64_t e0, int ne, int covered, int ct, int nct, uint64_t pol) {
  if (direct)
    tile_compute_prim<T, true>(prim, s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct, nct, pol);
  else
    tile_compute_prim<T, false>(prim, s_in, s_rcv, g_in, g_out, g_next, rslot, sslot, e0, ne, covered, ct, nct, pol);
}

// Rows of the direct mode: all-gather sends go to the next rank's output,
// all-gather receives find their data in this rank's own output.
__device__ __forceinline__ bool direct_send_row(bool direct, int prim) {
  return direct && (prim == kRecvReduceCopySend || prim == kRecvCopySend || prim == kCopySend);
}
__device__ __forceinline__ bool direct_recv_row(bool direct, int prim) {
  return direct && (prim == kRecvCopySend || prim == kRecv);
}

constexpr int kTileElems = 8192;    // elements per bulk-copied tile
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;  // dynamic shared memory for the stage ring
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = 32 * kComputeWarps;
constexpr int kSimpleThreads = 32 * 3 + kComputeThreads;  // waiter, loader, poster + workers

template <typename T>
__host__ __device__ constexpr int stage_bytes() { return kTileElems * ((int)sizeof(T) + 4); }
template <typename T>
__host__ __device__ constexpr int max_stages() {
  return kSmemBudget / stage_bytes<T>() < kMaxStages ? kSmemBudget / stage_bytes<T>() : kMaxStages;
}

__device__ __forceinline__ bool recv_is_partial(int prim) { return row_recvs_partial(prim); }

// A slice's user pointers all 16-byte aligned: its packs may be bulk-copied
// and stored 16 bytes at a time.
template <typename T>
__device__ __forceinline__ bool user_vec_ok(const T* in, const T* out, const T* next) {
  return (((uintptr_t)in | (uintptr_t)out | (uintptr_t)next) & 15u) == 0;
}

// Split point of the Simple kernel's two-block form: 16 elements keep every
// part's user and FIFO bytes 16-byte aligned for both element types.
constexpr int kSimpleSplitAlign = 16;

template <typename T, int SPLIT>
__global__ void __launch_bounds__(kSimpleThreads, 1) ring_simple_kernel(const __grid_constant__ RingArgs a,
                                                                        int nstages) {
  extern __shared__ __align__(128) char smem[];
  __shared__ uint64_t bar_ready[kDepth], bar_done[kDepth], bar_free[kDepth];
  __shared__ uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
  __shared__ volatile int sh_abort;
  __shared__ int sh_chan;
  __shared__ uint64_t sh_base_send, sh_base_recv;
  constexpr int P = ElemTraits<T>::kPack;
  constexpr int SB = stage_bytes<T>();

  const Geometry& g = a.geo;
  if (threadIdx.x == 0) sh_chan = -1;
  __syncthreads();
  // blocks [0, N * C) move the first part of every slice (all of it unless
  // the launch splits), blocks [N * C, 2 * N * C) the rest
  const int nblk = g.nranks * g.nchan;
  const int half = SPLIT == 1 ? 0 : (int)blockIdx.x / nblk;
  int rank, dense;
  map_block_index(a, SPLIT == 1 ? (int)blockIdx.x : (int)blockIdx.x % nblk, &rank, &dense, &sh_chan);
  __syncthreads();
  const int N = g.nranks;
  const int ring_idx = ring_index_of(a, dense, rank);
  const int e_send = ring_idx, e_recv = (ring_idx + N - 1) % N;
  ConnCounters* cs = conn_at(a, dense, e_send);
  ConnCounters* cr = conn_at(a, dense, e_recv);
  uint64_t* s_tail = conn_tail(cs, half);  // this part's published steps
  const uint64_t* r_tail = conn_tail(cr, half);
  uint64_t* r_head = conn_head(cr, half);
  char* fifo_send = fifo_at(a, dense, e_send);
  const char* fifo_recv = fifo_at(a, dense, e_recv);

  if (threadIdx.x == 0) {
    const uint64_t tail0 = ld_relaxed_u64(s_tail), head0 = ld_relaxed_u64(r_head);  // with the header
    sh_abort = entry_check(a) ? 0 : 1;
    for (int d = 0; d < kDepth; d++) {
      mbar_init(&bar_ready[d], 1);
      mbar_init(&bar_done[d], kComputeThreads);
      mbar_init(&bar_free[d], 1);
    }
    for (int st = 0; st < kMaxStages; st++) {
      mbar_init(&bar_full[st], 1);
      mbar_init(&bar_empty[st], kComputeWarps);
    }
    // This block alone writes the tail of its send edge and the head of its
    // receive edge; both equal the previous call's final step. Slices start
    // on a multiple of NCCL_STEPS so that no slice wraps around the ring.
    sh_base_send = round_up_steps(tail0);
    sh_base_recv = round_up_steps(head0);
    reinterpret_cast<uint8_t*>(a.ws + kTraceOffset)[blockIdx.x] = (uint8_t)sh_chan;
  }
  __syncthreads();
  if (sh_abort) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t sps = (uint64_t)g.sps;
  const uint64_t base_send = sh_base_send, base_recv = sh_base_recv;
  const uint64_t info = ((uint64_t)blockIdx.x << 32);
  const int64_t step_bytes = g.step_bytes;
  const T* in = reinterpret_cast<const T*>(a.send[rank]);
  T* out = reinterpret_cast<T*>(a.recv[rank]);
  const bool direct = a.direct != 0;
  T* next_out = reinterpret_cast<T*>(a.recv[next_rank_of(a, dense, ring_idx)]);
  SliceCursor c;
  cursor_begin(g, dense, ring_idx, c);

  if (warp == 0) {
    if (lane != 0) return;
    // ---- waiter ----
    uint64_t rstep = base_recv, sstep = base_send, tail_seen = 0, head_seen = 0, head_seen1 = 0;
    // the send credit: the receiver's head (both parts' heads when the launch
    // splits: each slice's split point follows its size, so a later slice in
    // the same slot can give one part bytes that the other part's receiver
    // read before)
    auto credit = [&]() -> uint64_t {
      const uint64_t h0 = head_seen > base_send ? head_seen : base_send;
      if (SPLIT == 1) return h0;
      const uint64_t h1 = head_seen1 > base_send ? head_seen1 : base_send;
      return h0 < h1 ? h0 : h1;
    };
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      if (use > 0 && !mbar_wait(a, &bar_free[d], (use - 1) & 1u, info | (1u << 24) | i)) sh_abort = 1;
      if (!sh_abort && !slice_in_bounds(a, dense, c, rstep, sstep, info | i)) sh_abort = 1;
      // The slice's data (tail) and the room for what it sends (head) are
      // polled in one loop, both loads in flight at once, so a credit that
      // needs a poll adds no round trip after the tail. Until the receiver's
      // first release in this call, its head may still hold the previous
      // call's final step (< base_send): all slots free. The head is read
      // relaxed: the receiver publishes it only after its reads of the slot
      // have returned, and the slot is written only after the value is seen.
      bool need_t = !sh_abort && row_recvs(c.prim) && tail_seen < rstep + sps;
      bool need_h = !sh_abort && row_sends(c.prim) && !direct_send_row(direct, c.prim) &&  // direct sends fill no slot
                    credit() + kSteps < sstep + sps;
      Spin sp;
      while (need_t || need_h) {
        uint64_t h = 0, h1 = 0;
        if (need_h) {
          h = ld_relaxed_u64(&cs->head);
          if (SPLIT == 2) h1 = ld_relaxed_u64(&cs->head_h1);
        }
        if (need_t) {
          tail_seen = ld_acquire_u64(r_tail);
          need_t = tail_seen < rstep + sps;
        }
        if (need_h) {
          head_seen = h > head_seen ? h : head_seen;
          head_seen1 = h1 > head_seen1 ? h1 : head_seen1;
          need_h = credit() + kSteps < sstep + sps;
        }
        if (!(need_t || need_h)) break;
        if (sp.poll(a, info | ((need_t ? 2u : 3u) << 24) | i, need_t ? rstep + sps : sstep + sps)) {
          sh_abort = 1;
          break;
        }
      }
      mbar_arrive(&bar_ready[d]);
      if (sh_abort) break;
      if (row_recvs(c.prim)) rstep += sps;
      if (row_sends(c.prim)) sstep += sps;
    }
  } else if (warp == 1) {
    if (lane != 0) return;
    // ---- loader ----
    const uint64_t pol = l2_policy_evict_first();
    uint64_t rstep = base_recv;
    uint32_t gt = 0;  // tiles issued so far
    uint64_t sstep_l = base_send;  // for the debug bounds check only
    for (uint32_t i = 0; c.valid && !sh_abort; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      const int prim = c.prim;
      if (!slice_in_bounds(a, dense, c, rstep, sstep_l, info | i)) {
        sh_abort = 1;
        break;
      }
      if (row_sends(prim)) sstep_l += sps;
      int64_t in_off, out_off;
      slice_offsets(a, dense, c, &in_off, &out_off);
      const bool vec = user_vec_ok(in + in_off, out + out_off, direct ? next_out + out_off : nullptr);
      const bool has_in = row_reads_input(prim);
      const bool has_rcv = row_recvs(prim);
      // direct mode: a forwarded final is staged from this rank's own output,
      // the last row moves nothing
      const bool rcv_own_out = direct_recv_row(direct, prim);
      const bool rcv_bytes = has_rcv && !(rcv_own_out && prim == kRecv);
      const int rcv_eb = recv_is_partial(prim) ? 4 : (int)sizeof(T);
      const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
      int64_t lo, hi;
      split_range(c.nelem, half, SPLIT, kSimpleSplitAlign, &lo, &hi);
      const int ntiles = (int)div_up(hi - lo, kTileElems);
      // The slice's first tile copies its input as soon as a stage is free,
      // before the wait for the slice's tail and credit (the input does not
      // depend on the peers; copying it early takes its HBM latency off the
      // chain of handoffs).
      bool ready = false;
      for (int k = 0; k < ntiles || !ready; k++) {
        if (k >= ntiles) {  // an empty slice: only the wait
          if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (6u << 24) | i) || sh_abort) sh_abort = 1;
          ready = true;
          break;
        }
        const uint32_t st = gt % nstages, su = gt / nstages;
        if (su > 0 && !mbar_wait(a, &bar_empty[st], (su - 1) & 1u, info | (7u << 24) | i)) {
          sh_abort = 1;
          break;
        }
        const int64_t e0 = lo + (int64_t)k * kTileElems;
        const int ne = (int)imin(kTileElems, hi - e0);
        const int covered = vec ? ne / P * P : 0;
        const uint32_t b_in = has_in ? (uint32_t)covered * (uint32_t)sizeof(T) : 0u;
        const uint32_t b_rcv = rcv_bytes ? (uint32_t)covered * (uint32_t)rcv_eb : 0u;
        char* s_in = smem + (int64_t)st * SB;
        char* s_rcv = s_in + kTileElems * (int)sizeof(T);
        if (b_in) {
          mbar_expect_tx(&bar_full[st], b_in);
          tma_load_1d(s_in, in + in_off + e0, b_in, &bar_full[st], pol);
        }
        if (!ready) {
          ready = true;
          if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (6u << 24) | i) || sh_abort) {
            mbar_arrive_expect_tx(&bar_full[st], 0u);  // the phase completes once the input landed
            gt++;
            sh_abort = 1;
            break;
          }
          if (has_rcv) fence_proxy_async_global();  // the tail acquired by the waiter, before bulk reads of the FIFO
        }
        mbar_arrive_expect_tx(&bar_full[st], b_rcv);
        if (b_rcv)
          tma_load_1d(s_rcv, rcv_own_out ? reinterpret_cast<const char*>(out + out_off + e0) : rslot + e0 * rcv_eb,
                      b_rcv, &bar_full[st], pol);
        gt++;
      }
      if (has_rcv) rstep += sps;
    }
    // Never leave with bulk copies in flight: wait (time-bounded, whatever
    // the abort flag says) until the last tile issued to every stage landed.
    for (uint32_t st = 0; st < (uint32_t)nstages && st < gt; st++) {
      const uint32_t last = (gt - 1 - st) / nstages * nstages + st;  // last tile issued to stage st
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bar_full[st], (last / nstages) & 1u)) {
        if (global_timer_ns() - t0 > a.timeout_ns) {
          report_failure(header_of(a), kErrTimeout, info | (8u << 24), last);
          break;
        }
      }
    }
  } else if (warp == 2) {
    if (lane != 0) return;
    // ---- poster ----
    uint64_t rstep = base_recv, sstep = base_send;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (4u << 24) | i) ||
          !mbar_wait(a, &bar_done[d], use & 1u, info | (4u << 24) | i)) {
        sh_abort = 1;
        break;
      }
      if (sh_abort) break;
      // the head first: the slots read need no fence (their bytes have been
      // read), and the sender waits on it
      if (row_recvs(c.prim)) {
        rstep += sps;
        if (a.fault != kFaultDropHead) st_relaxed_u64(r_head, rstep);  // release the slots read
      }
      if (row_sends(c.prim)) {
        sstep += sps;
        fence_acq_rel_gpu();  // the workers' payload is visible before the tail
        st_relaxed_u64(s_tail, sstep);
      }
      mbar_arrive(&bar_free[d]);
    }
    // without a split, the second part's counters follow this call's final
    // steps (a later split call starts both parts from them)
    if (SPLIT == 1 && !sh_abort) {
      st_relaxed_u64(&cs->tail_h1, sstep);
      st_relaxed_u64(&cr->head_h1, rstep);
    }
  } else {
    // ---- workers ----
    const int ct = threadIdx.x - 96;
    const uint64_t out_pol = l2_policy_evict_first();
    uint64_t rstep = base_recv, sstep = base_send;
    uint32_t gt = 0;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kDepth, use = i / kDepth;
      // Gate every slice on the waiter (which the poster paces), so the
      // workers never run more than D slices ahead, even across empty slices.
      if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (5u << 24) | i) || sh_abort) {
        mbar_arrive(&bar_done[d]);
        sh_abort = 1;
        break;
      }
      const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
      char* sslot = fifo_send + (int64_t)(sstep % kSteps) * step_bytes;
      int64_t in_off, out_off;
      slice_offsets(a, dense, c, &in_off, &out_off);
      const bool vec = user_vec_ok(in + in_off, out + out_off, direct ? next_out + out_off : nullptr);
      int64_t lo, hi;
      split_range(c.nelem, half, SPLIT, kSimpleSplitAlign, &lo, &hi);
      const int ntiles = (int)div_up(hi - lo, kTileElems);
      bool stop = false;
      for (int k = 0; k < ntiles; k++, gt++) {
        const uint32_t st = gt % nstages, su = gt / nstages;
        if (!mbar_wait(a, &bar_full[st], su & 1u, info | (5u << 24) | i) || sh_abort) {
          stop = true;
          break;
        }
        const int64_t e0 = lo + (int64_t)k * kTileElems;
        const int ne = (int)imin(kTileElems, hi - e0);
        const char* s_in = smem + (int64_t)st * SB;
        const char* s_rcv = s_in + kTileElems * (int)sizeof(T);
        tile_compute_any<T>(direct, c.prim, s_in, s_rcv, in + in_off, out + out_off, next_out + out_off, rslot,
                            sslot, e0, ne, vec ? ne / P * P : 0, ct, kComputeThreads, out_pol);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_empty[st]);
      }
      mbar_arrive(&bar_done[d]);
      if (stop) {
        sh_abort = 1;
        break;
      }
      if (row_recvs(c.prim)) rstep += sps;
      if (row_sends(c.prim)) sstep += sps;
    }
  }
}

// Host-side launch of the Simple kernel (declared in rar_launch.h).
template <typename T, int SPLIT>
cudaError_t launch_simple_form(const RingArgs& a, cudaLaunchConfig_t cfg, int device, int nstages, int smem,
                               int key) {
  if (!setup_done(device, key)) {
    const cudaError_t e = cudaFuncSetAttribute(ring_simple_kernel<T, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               max_stages<T>() * stage_bytes<T>());
    if (e != cudaSuccess) return e;
    mark_setup_done(device, key);
  }
  cfg.gridDim = dim3(cfg.gridDim.x * (unsigned)SPLIT);
  if (trace_on())
    std::fprintf(stderr, "rar trace:   kernel ring_simple_kernel<%s> grid %u threads %d stages %d smem %d split %d\n",
                 sizeof(T) == 4 ? "float" : "bf16", cfg.gridDim.x, kSimpleThreads, nstages, smem, SPLIT);
  return cudaLaunchKernelEx(&cfg, ring_simple_kernel<T, SPLIT>, a, nstages);
}

// First-loop chunks of at least this many elements split a grid that fits the
// SMs twice over two blocks per (rank, channel); smaller messages keep one
// block per pair (their time is the hand-off chain, not the SMs' stores).
constexpr int64_t kSimpleSplitMinChunk = 65536;

cudaError_t launch_ring_simple(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out) {
  int device = 0, sms = 0;
  cudaError_t e = current_device_sms(&device, &sms);
  if (e != cudaSuccess) return e;
  // One block per SM gets the deep stage ring; grids larger than the SM
  // count use two stages so that several blocks fit on an SM.
  const bool f32 = a.geo.dtype == kF32;
  const int deep = f32 ? max_stages<float>() : max_stages<uint16_t>();
  const int nstages = grid <= sms ? deep : 2;
  const int smem = nstages * (f32 ? stage_bytes<float>() : stage_bytes<uint16_t>());
  // The workers' stores are bound by their SM's store rate: when twice the
  // grid fits one block per SM, two blocks per (rank, channel) each move a
  // part of every slice on twice the SMs.
  const int64_t first_chunk = loop_chunk_count(a.geo, imin(a.geo.per_channel, a.geo.count));
  const bool split = 2 * grid <= sms && first_chunk >= kSimpleSplitMinChunk;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSimpleThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (threads_out) *threads_out = kSimpleThreads;
  if (f32)
    return split ? launch_simple_form<float, 2>(a, cfg, device, nstages, smem, kSetupSimpleF32Split)
                 : launch_simple_form<float, 1>(a, cfg, device, nstages, smem, kSetupSimpleF32);
  return split ? launch_simple_form<uint16_t, 2>(a, cfg, device, nstages, smem, kSetupSimpleBf16Split)
               : launch_simple_form<uint16_t, 1>(a, cfg, device, nstages, smem, kSetupSimpleBf16);
}

}  // namespace rar
