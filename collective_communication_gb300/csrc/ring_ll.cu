// ring_ll.cu -- ring AllReduce, LL and LL128 protocols, all N virtual ranks in
// one launch (one block per (rank, channel)).
//
// Pages cited (by title, then section):
//   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
//         sections "LL：Data 与 Flag 同 Line", "LL128：15/16 Payload",
//         "Simple 的 Credit 与 Step" (the head credit both protocols share)
//   [C12] "NCCL 专家课程 12：Ring AllReduce 逐步推导、真实 Ring 与 Channel 并行"
//         sections "源码步骤一" .. "源码步骤五"
//
// One chunk = one slice = one FIFO step. A step's data is ready when the
// flags inside its lines equal step + 1 (a generation that grows with the
// connection's step count, so a slot reused NCCL_STEPS steps later never
// matches a stale line). Every thread polls the lines it consumes. The head
// credit (head + NCCL_STEPS >= step + 1) is checked by thread 0 for the next
// step while the block still works on the current one; one block barrier per
// step then releases the data threads and lets thread 0 publish the head.
//
// LL line (16 B): {data_lo, flag, data_hi, flag}, 8 payload bytes; payload
// bytes [8j, 8j+8) of the step go to line j.
// LL128 line (128 B): 16 x 64-bit words, words 0..14 payload, word 15 the flag.
// A warp moves 4 lines (512 B) per 16-byte-per-lane access; lane l holds bytes
// [16l, 16l+16) of the group, i.e. line l/8, words 2(l%8), 2(l%8)+1; the lane
// with l%8 == 7 holds word 14 (payload) and word 15 (flag). The 480 payload
// bytes of group g map to the lanes so that every user access stays aligned:
// lanes with l%8 < 7 carry group bytes 16*(7*(l/8) + l%8) .. +16, the four
// flag lanes carry bytes 448 + 8*(l/8) .. +8.
#include "rar_device.cuh"

namespace rar {

constexpr uint32_t kFullMask = 0xffffffffu;

template <typename T>
struct LLUnit;
template <>
struct LLUnit<float> {
  static constexpr int kElems = 2;       // elements per 8 payload bytes of T
  static constexpr int kPartLines = 1;   // lines per unit of binary32 partial sums
};
template <>
struct LLUnit<uint16_t> {
  static constexpr int kElems = 4;
  static constexpr int kPartLines = 2;
};

// Load n (<= kmax) consecutive input elements, widened to binary32; zeros past n.
template <typename T, int KMAX>
__device__ __forceinline__ void load_input_n(const T* p, int n, float (&v)[KMAX]);
template <int KMAX>
__device__ __forceinline__ void load_input_n_f32(const float* p, int n, float (&v)[KMAX]) {
  if (n == KMAX && KMAX == 4) {
    uint4 u = ld_stream_v4(p);
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  } else if (n == KMAX && KMAX == 2) {
    uint2 u = ld_stream_v2(p);
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
  } else {
#pragma unroll
    for (int j = 0; j < KMAX; j++) v[j] = j < n ? __uint_as_float(ld_cg_u32(p + j)) : 0.f;
  }
}
template <int KMAX>
__device__ __forceinline__ void load_input_n_bf16(const uint16_t* p, int n, float (&v)[KMAX]) {
  if (n == KMAX && KMAX == 4) {
    uint2 u = ld_stream_v2(p);
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  } else if (n == KMAX && KMAX == 2) {
    uint32_t u = ld_cg_u32(p);
    v[0] = bf16lo(u); v[1] = bf16hi(u);
  } else {
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
      uint16_t h = 0;
      if (j < n) asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p + j) : "memory");
      v[j] = __uint_as_float((uint32_t)h << 16);
    }
  }
}
template <>
__device__ __forceinline__ void load_input_n<float, 4>(const float* p, int n, float (&v)[4]) { load_input_n_f32<4>(p, n, v); }
template <>
__device__ __forceinline__ void load_input_n<float, 2>(const float* p, int n, float (&v)[2]) { load_input_n_f32<2>(p, n, v); }
template <>
__device__ __forceinline__ void load_input_n<uint16_t, 4>(const uint16_t* p, int n, float (&v)[4]) { load_input_n_bf16<4>(p, n, v); }
template <>
__device__ __forceinline__ void load_input_n<uint16_t, 2>(const uint16_t* p, int n, float (&v)[2]) { load_input_n_bf16<2>(p, n, v); }

// Store the first n elements of T held as raw bits in w (little-endian).
template <typename T>
__device__ __forceinline__ void store_out_n(T* p, int n, int kmax, uint4 w) {
  const int bytes = kmax * (int)sizeof(T);
  if (n == kmax) {
    if (bytes == 16) { st_v4(p, w); return; }
    if (bytes == 8) { st_v2(p, make_uint2(w.x, w.y)); return; }
    if (bytes == 4) { *reinterpret_cast<uint32_t*>(p) = w.x; return; }
  }
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
  for (int j = 0; j < n; j++) {
    if (sizeof(T) == 4) {
      reinterpret_cast<uint32_t*>(p)[j] = wd[j];
    } else {
      reinterpret_cast<uint16_t*>(p)[j] = (uint16_t)(wd[j >> 1] >> ((j & 1) * 16));
    }
  }
}

__device__ __forceinline__ uint32_t round_bf16_pair(float lo, float hi) { return pack_bf16x2(lo, hi); }

// ---------------------------------------------------------------------------
// LL
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool ll_ready(const uint4& v, uint32_t flag) { return v.y == flag && v.w == flag; }

// Poll one line until both flags equal `flag` (bounded). Returns false when
// the wait gave up; v holds the last value read.
__device__ __forceinline__ bool ll_poll(const RingArgs& a, const char* p, uint32_t flag, uint4& v,
                                        volatile int* sh_abort, uint64_t info) {
  Spin sp;
  while (!ll_ready(v, flag)) {
    if (*sh_abort) return false;
    if (sp.poll(a, info, flag)) { *sh_abort = 1; return false; }
    v = ld_volatile_v4(p);
  }
  return true;
}

template <typename T, int PRIM, int NT>
__device__ __forceinline__ void ll_slice(const RingArgs& a, const T* in, T* out, const char* rslot, char* sslot,
                                         int64_t nelem, uint32_t rflag, uint32_t sflag, volatile int* sh_abort,
                                         uint64_t info) {
  constexpr int K = LLUnit<T>::kElems;
  constexpr int PL = LLUnit<T>::kPartLines;
  constexpr int UL = 4;
  constexpr bool kIn = PRIM == kSend || PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend;
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend;
  constexpr bool kRecvFinal = PRIM == kRecvCopySend || PRIM == kRecv;
  constexpr bool kSendPartial = PRIM == kSend || PRIM == kRecvReduceSend;
  constexpr bool kSendFinal = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv;
  constexpr int RL = kRecvPartial ? PL : 1;

  const int64_t nunits = div_up(nelem, K);
  for (int64_t u0 = threadIdx.x; u0 < nunits; u0 += (int64_t)NT * UL) {
    uint4 rl[UL][RL];
    float x[UL][K];
#pragma unroll
    for (int u = 0; u < UL; u++) {
      const int64_t unit = u0 + (int64_t)u * NT;
      if (unit < nunits) {
        if (kRecvPartial || kRecvFinal) {
#pragma unroll
          for (int l = 0; l < RL; l++) rl[u][l] = ld_volatile_v4(rslot + (unit * RL + l) * 16);
        }
        if (kIn) load_input_n<T, K>(in + unit * K, (int)imin(K, nelem - unit * K), x[u]);
      }
    }
    if (kRecvPartial || kRecvFinal) {
#pragma unroll
      for (int u = 0; u < UL; u++) {
        const int64_t unit = u0 + (int64_t)u * NT;
        if (unit < nunits) {
#pragma unroll
          for (int l = 0; l < RL; l++)
            if (!ll_ready(rl[u][l], rflag) &&
                !ll_poll(a, rslot + (unit * RL + l) * 16, rflag, rl[u][l], sh_abort, info))
              return;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UL; u++) {
      const int64_t unit = u0 + (int64_t)u * NT;
      if (unit >= nunits) continue;
      const int kv = (int)imin(K, nelem - unit * K);
      float v[K];
      if (kRecvPartial) {
#pragma unroll
        for (int l = 0; l < PL; l++) {
          v[2 * l] = __uint_as_float(rl[u][l].x);
          v[2 * l + 1] = __uint_as_float(rl[u][l].z);
        }
#pragma unroll
        for (int j = 0; j < K; j++) v[j] = __fadd_rn(v[j], x[u][j]);
      } else if (PRIM == kSend) {
#pragma unroll
        for (int j = 0; j < K; j++) v[j] = x[u][j];
      }
      if (kSendPartial) {
#pragma unroll
        for (int l = 0; l < PL; l++)
          st_volatile_v4(sslot + (unit * PL + l) * 16,
                         make_uint4(__float_as_uint(v[2 * l]), sflag, __float_as_uint(v[2 * l + 1]), sflag));
      } else {
        // final values: 8 bytes of T
        uint2 f;
        if (kRecvFinal) {
          f = make_uint2(rl[u][0].x, rl[u][0].z);
        } else if (sizeof(T) == 4) {
          f = make_uint2(__float_as_uint(v[0]), __float_as_uint(v[1]));
        } else {
          f = make_uint2(round_bf16_pair(v[0], v[1]), round_bf16_pair(v[2], v[3]));  // rounded once
        }
        if (kOut) store_out_n<T>(out + unit * K, kv, K, make_uint4(f.x, f.y, 0u, 0u));
        if (kSendFinal) st_volatile_v4(sslot + unit * 16, make_uint4(f.x, sflag, f.y, sflag));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// LL128
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t ll128_flag_of(const uint4& v) { return ((uint64_t)v.w << 32) | v.z; }

// Warp-uniform wait until every flag lane of the group sees `flag`.
__device__ __forceinline__ bool ll128_poll(const RingArgs& a, const char* p, uint64_t flag, bool flag_lane, uint4& v,
                                        volatile int* sh_abort, uint64_t info) {
  Spin sp;
  const int lane = threadIdx.x & 31;
  while (true) {
    const bool need = flag_lane && ll128_flag_of(v) != flag;
    if (!__any_sync(kFullMask, need)) return true;
    int stop = *sh_abort;
    if (lane == 0 && !stop && sp.poll(a, info, flag)) { *sh_abort = 1; stop = 1; }
    stop = __shfl_sync(kFullMask, stop, 0);
    if (stop) return false;
    v = ld_volatile_v4(p);
  }
}

// Lane geometry inside a 4-line group.
struct LL128Lane {
  int lane;
  bool flag_lane;
  int piece_off;   // payload byte offset of the lane's piece inside the group
  int piece_bytes; // 16, or 8 for flag lanes
  __device__ __forceinline__ LL128Lane() {
    lane = threadIdx.x & 31;
    const int q = lane >> 3, t8 = lane & 7;
    flag_lane = (t8 == 7);
    piece_off = flag_lane ? 448 + 8 * q : 16 * (7 * q + t8);
    piece_bytes = flag_lane ? 8 : 16;
  }
};

// Same payload element size on both sides (all rows except bf16's owner row).
template <typename T, int PRIM, int NT>
__device__ __forceinline__ void ll128_slice(const RingArgs& a, const T* in, T* out, const char* rslot, char* sslot,
                                            int64_t nelem, uint64_t rflag, uint64_t sflag, volatile int* sh_abort,
                                            uint64_t info) {
  constexpr int NW = NT / 32;
  constexpr int UG = 2;
  constexpr bool kIn = PRIM == kSend || PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend;
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend;
  constexpr bool kHasRecv = PRIM != kSend;
  constexpr bool kHasSend = PRIM != kRecv;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv;
  // payload element bytes of this row (both sides)
  constexpr int EB = (PRIM == kSend || PRIM == kRecvReduceSend) ? 4
                   : (PRIM == kRecvReduceCopySend) ? 4  // f32 only here
                   : (int)sizeof(T);
  constexpr int KMAX = 16 / EB;
  const LL128Lane L;
  const int warp = threadIdx.x >> 5;
  const int kmax = L.piece_bytes / EB;
  const int64_t ngroups = div_up(nelem * EB, 480);
  for (int64_t g0 = warp; g0 < ngroups; g0 += (int64_t)NW * UG) {
    uint4 rv[UG];
    float x[UG][4];
#pragma unroll
    for (int u = 0; u < UG; u++) {
      const int64_t g = g0 + (int64_t)u * NW;
      if (g < ngroups) {
        if (kHasRecv) rv[u] = ld_volatile_v4(rslot + g * 512 + 16 * L.lane);
        if (kIn) {
          const int64_t e0 = (g * 480 + L.piece_off) / EB;
          const int kv = (int)imax(0, imin(kmax, nelem - e0));
          if (L.flag_lane) {
            float t[2];
            load_input_n<T, 2>(in + e0, kv, t);
            x[u][0] = t[0]; x[u][1] = t[1]; x[u][2] = 0.f; x[u][3] = 0.f;
          } else {
            load_input_n<T, 4>(in + e0, kv, x[u]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UG; u++) {
      const int64_t g = g0 + (int64_t)u * NW;
      if (g >= ngroups) continue;  // uniform across the warp
      if (kHasRecv && !ll128_poll(a, rslot + g * 512 + 16 * L.lane, rflag, L.flag_lane, rv[u], sh_abort, info)) return;
      const int64_t e0 = (g * 480 + L.piece_off) / EB;
      const int kv = (int)imax(0, imin(kmax, nelem - e0));
      uint4 pay;
      if (kRecvPartial || PRIM == kSend) {
        float v[4];
        if (kRecvPartial) {
          v[0] = __uint_as_float(rv[u].x); v[1] = __uint_as_float(rv[u].y);
          v[2] = __uint_as_float(rv[u].z); v[3] = __uint_as_float(rv[u].w);
#pragma unroll
          for (int j = 0; j < 4; j++) v[j] = __fadd_rn(v[j], x[u][j]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; j++) v[j] = x[u][j];
        }
#pragma unroll
        for (int j = 0; j < 4; j++)
          if (j >= kv) v[j] = 0.f;
        pay = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
      } else {
        pay = rv[u];  // final values pass through unchanged
      }
      if (kOut && kv > 0) store_out_n<T>(out + e0, kv, kmax, pay);
      if (kHasSend) {
        if (L.flag_lane) {
          pay.z = (uint32_t)sflag;
          pay.w = (uint32_t)(sflag >> 32);
        }
        st_volatile_v4(sslot + g * 512 + 16 * L.lane, pay);
      }
      (void)KMAX;
    }
  }
}

// bf16 owner row: binary32 partial sums arrive (120 elements per group) and
// bf16 finals leave (240 elements per group). A warp reduces the two receive
// groups 2g and 2g+1, rounds once to bf16, writes the output, stages the 240
// bf16 values in shared memory and rewrites them in the send layout.
template <int NT>
__device__ __forceinline__ void ll128_owner_bf16(const RingArgs& a, const uint16_t* in, uint16_t* out,
                                                 const char* rslot, char* sslot, int64_t nelem, uint64_t rflag,
                                                 uint64_t sflag, volatile int* sh_abort, uint64_t info,
                                                 uint16_t* stage) {
  constexpr int NW = NT / 32;
  const LL128Lane L;
  const int warp = threadIdx.x >> 5;
  uint16_t* st = stage + warp * 240;
  const int64_t nrecv = div_up(nelem * 4, 480), nsend = div_up(nelem * 2, 480);
  for (int64_t gs = warp; gs < nsend; gs += NW) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int64_t gr = 2 * gs + h;
      if (gr >= nrecv) break;  // uniform
      const char* rp = rslot + gr * 512 + 16 * L.lane;
      uint4 rv = ld_volatile_v4(rp);
      const int kmax = L.piece_bytes / 4;
      const int64_t e0 = (gr * 480 + L.piece_off) / 4;
      const int kv = (int)imax(0, imin(kmax, nelem - e0));
      float x[4];
      if (L.flag_lane) {
        float t[2];
        load_input_n<uint16_t, 2>(in + e0, kv, t);
        x[0] = t[0]; x[1] = t[1]; x[2] = 0.f; x[3] = 0.f;
      } else {
        load_input_n<uint16_t, 4>(in + e0, kv, x);
      }
      if (!ll128_poll(a, rp, rflag, L.flag_lane, rv, sh_abort, info)) return;
      float v[4] = {__fadd_rn(__uint_as_float(rv.x), x[0]), __fadd_rn(__uint_as_float(rv.y), x[1]),
                    __fadd_rn(__uint_as_float(rv.z), x[2]), __fadd_rn(__uint_as_float(rv.w), x[3])};
      const uint4 w = make_uint4(round_bf16_pair(v[0], v[1]), round_bf16_pair(v[2], v[3]), 0u, 0u);
      if (kv > 0) store_out_n<uint16_t>(out + e0, kv, kmax, w);
      const int64_t loc = e0 - gs * 240;  // in [0, 240)
      for (int j = 0; j < kv; j++) st[loc + j] = (uint16_t)((j < 2 ? w.x : w.y) >> ((j & 1) * 16));
    }
    __syncwarp();
    {
      const int kmax = L.piece_bytes / 2;
      const int64_t e0 = (gs * 480 + L.piece_off) / 2;
      const int kv = (int)imax(0, imin(kmax, nelem - e0));
      const int loc = (int)(e0 - gs * 240);
      uint32_t wd[4] = {0u, 0u, 0u, 0u};
      for (int j = 0; j < kv; j++) wd[j >> 1] |= (uint32_t)st[loc + j] << ((j & 1) * 16);
      uint4 pay = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      if (L.flag_lane) {
        pay.z = (uint32_t)sflag;
        pay.w = (uint32_t)(sflag >> 32);
      }
      st_volatile_v4(sslot + gs * 512 + 16 * L.lane, pay);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
__device__ __noinline__ bool wait_credit(const RingArgs& a, ConnCounters* cs, uint64_t base_send, uint64_t step,
                                         uint64_t* head_seen, uint64_t info) {
  Spin sp;
  while (true) {
    const uint64_t h = *head_seen > base_send ? *head_seen : base_send;
    if (h + kSteps >= step + 1) return true;
    *head_seen = ld_acquire_u64(&cs->head);
    const uint64_t h2 = *head_seen > base_send ? *head_seen : base_send;
    if (h2 + kSteps >= step + 1) return true;
    if (sp.poll(a, info, step + 1)) return false;
  }
}

template <typename T, int PROTO, int NT>
__device__ __forceinline__ void line_slice(int prim, const RingArgs& a, const T* in, T* out, const char* rslot,
                                           char* sslot, int64_t nelem, uint64_t rstep, uint64_t sstep,
                                           volatile int* sh_abort, uint64_t info, uint16_t* stage) {
  if (PROTO == kLL) {
    const uint32_t rf = (uint32_t)(rstep + 1), sf = (uint32_t)(sstep + 1);
    switch (prim) {
      case kSend: ll_slice<T, kSend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      case kRecvReduceSend: ll_slice<T, kRecvReduceSend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      case kRecvReduceCopySend: ll_slice<T, kRecvReduceCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      case kRecvCopySend: ll_slice<T, kRecvCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      default: ll_slice<T, kRecv, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
    }
  } else {
    const uint64_t rf = rstep + 1, sf = sstep + 1;
    switch (prim) {
      case kSend: ll128_slice<T, kSend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      case kRecvReduceSend: ll128_slice<T, kRecvReduceSend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      case kRecvReduceCopySend:
        if constexpr (sizeof(T) == 4)
          ll128_slice<T, kRecvReduceCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info);
        else
          ll128_owner_bf16<NT>(a, reinterpret_cast<const uint16_t*>(in), reinterpret_cast<uint16_t*>(out), rslot,
                               sslot, nelem, rf, sf, sh_abort, info, stage);
        break;
      case kRecvCopySend: ll128_slice<T, kRecvCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      default: ll128_slice<T, kRecv, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
    }
  }
}

template <typename T, int PROTO, int NT>
__global__ void __launch_bounds__(NT, 1) ring_line_kernel(const __grid_constant__ RingArgs a) {
  __shared__ volatile int sh_abort;
  __shared__ int sh_chan;
  __shared__ uint64_t sh_base_send, sh_base_recv;
  __shared__ __align__(16) uint16_t stage[(PROTO == kLL128 && sizeof(T) == 2) ? (NT / 32) * 240 : 8];

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
    // Both counters belong to this block and equal the previous call's final step.
    sh_base_send = ld_relaxed_u64(&cs->tail);
    sh_base_recv = ld_relaxed_u64(&cr->head);
    reinterpret_cast<uint8_t*>(a.ws + kTraceOffset)[blockIdx.x] = (uint8_t)sh_chan;
  }
  __syncthreads();
  if (sh_abort) return;

  const T* in = reinterpret_cast<const T*>(a.send[rank]);
  T* out = reinterpret_cast<T*>(a.recv[rank]);
  const int64_t step_bytes = g.step_bytes;
  const uint64_t base_send = sh_base_send;
  const uint64_t info = ((uint64_t)blockIdx.x << 32);
  uint64_t rstep = sh_base_recv, sstep = base_send, head_seen = 0;
  SliceCursor c;
  cursor_begin(g, dense, ring_idx, c);
  if (threadIdx.x == 0 && c.valid && row_sends(c.prim) &&
      !wait_credit(a, cs, base_send, sstep, &head_seen, info | (3u << 24)))
    sh_abort = 1;
  __syncthreads();
  uint32_t i = 0;
  while (c.valid && !sh_abort) {
    const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
    char* sslot = fifo_send + (int64_t)(sstep % kSteps) * step_bytes;
    line_slice<T, PROTO, NT>(c.prim, a, in + c.offset, out + c.offset, rslot, sslot, c.nelem, rstep, sstep,
                             &sh_abort, info | (2u << 24) | i, stage);
    SliceCursor nx = c;
    cursor_next(g, nx);
    const uint64_t nsstep = sstep + (row_sends(c.prim) ? 1 : 0);
    // credit for the next step, taken while the block finishes this one
    if (threadIdx.x == 0 && nx.valid && row_sends(nx.prim) && !sh_abort &&
        !wait_credit(a, cs, base_send, nsstep, &head_seen, info | (3u << 24) | (i + 1)))
      sh_abort = 1;
    __syncthreads();
    if (threadIdx.x == 0 && row_recvs(c.prim) && !sh_abort && a.fault != kFaultDropHead)
      st_relaxed_u64(&cr->head, rstep + 1);  // every thread has read this step's lines
    if (row_recvs(c.prim)) rstep++;
    sstep = nsstep;
    c = nx;
    i++;
  }
  // the sender's step count carries over to the next call
  if (threadIdx.x == 0 && !sh_abort) st_relaxed_u64(&cs->tail, sstep);
}

cudaError_t launch_ring_line(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out) {
  constexpr int kThreadsLL = 512;     // the page's LL blockX
  constexpr int kThreadsLL128 = 640;  // the page's LL128 blockX (20 warps)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool f32 = a.geo.dtype == kF32;
  if (a.geo.proto == kLL) {
    cfg.blockDim = dim3(kThreadsLL);
    if (threads_out) *threads_out = kThreadsLL;
    return f32 ? cudaLaunchKernelEx(&cfg, ring_line_kernel<float, kLL, kThreadsLL>, a)
               : cudaLaunchKernelEx(&cfg, ring_line_kernel<uint16_t, kLL, kThreadsLL>, a);
  }
  cfg.blockDim = dim3(kThreadsLL128);
  if (threads_out) *threads_out = kThreadsLL128;
  return f32 ? cudaLaunchKernelEx(&cfg, ring_line_kernel<float, kLL128, kThreadsLL128>, a)
             : cudaLaunchKernelEx(&cfg, ring_line_kernel<uint16_t, kLL128, kThreadsLL128>, a);
}

}  // namespace rar
