// ring_ll.cu -- ring AllReduce (and its ReduceScatter and AllGather halves),
// LL and LL128 protocols, all N virtual ranks in one launch (one block per
// (rank, channel)).
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
#include <cstdio>

#include "rar_launch.h"

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

// The first n (<= kmax) elements of T at p as raw bits, little-endian, zeros
// past n; kmax * sizeof(T) is 16 or 8 bytes.
template <typename T>
__device__ __forceinline__ uint4 load_raw_n(const T* p, int n, int kmax) {
  const int bytes = kmax * (int)sizeof(T);
  if (n == kmax && bytes == 16) return ld_stream_v4(p);
  if (n == kmax && bytes == 8) {
    const uint2 u = ld_stream_v2(p);
    return make_uint4(u.x, u.y, 0u, 0u);
  }
  uint32_t wd[4] = {0u, 0u, 0u, 0u};
  for (int j = 0; j < n; j++) {
    if constexpr (sizeof(T) == 4) {
      wd[j] = ld_cg_u32(p + j);
    } else {
      uint16_t h;
      asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(p + j) : "memory");
      wd[j >> 1] |= (uint32_t)h << ((j & 1) * 16);
    }
  }
  return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

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
    v = ld_line_v4(p);
  }
  return true;
}

template <typename T, int PRIM, int NT>
__device__ __forceinline__ void ll_slice(const RingArgs& a, const T* in, T* out, const char* rslot, char* sslot,
                                         int64_t nelem, uint32_t rflag, uint32_t sflag, bool clean,
                                         volatile int* sh_abort, uint64_t info) {
  constexpr int K = LLUnit<T>::kElems;
  constexpr int PL = LLUnit<T>::kPartLines;
  constexpr int UL = 1;
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kIn = PRIM == kSend || kRecvPartial || PRIM == kCopySend;
  constexpr bool kRecvFinal = PRIM == kRecvCopySend || PRIM == kRecv;
  constexpr bool kSendPartial = PRIM == kSend || PRIM == kRecvReduceSend;
  constexpr bool kSendFinal = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kCopySend;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv ||
                        PRIM == kRecvReduceCopy || PRIM == kCopySend;
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
          for (int l = 0; l < RL; l++) rl[u][l] = ld_line_v4(rslot + (unit * RL + l) * 16);
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
      } else if (PRIM == kSend || PRIM == kCopySend) {
        // copySend: a bf16 input widened and rounded back is the same value
#pragma unroll
        for (int j = 0; j < K; j++) v[j] = x[u][j];
      }
      if (kSendPartial) {
#pragma unroll
        for (int l = 0; l < PL; l++)
          st_line_v4(sslot + (unit * PL + l) * 16,
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
        if (kSendFinal) st_line_v4(sslot + unit * 16, make_uint4(f.x, sflag, f.y, sflag));
      }
    }
  }
  // flag-wrap mode: the rest of the slot gets the current flag (no payload)
  if ((kSendPartial || kSendFinal) && clean) {
    const int64_t sent = nunits * (kSendPartial ? PL : 1);
    const int64_t slot_lines = a.geo.step_bytes / 16;
    for (int64_t l = sent + threadIdx.x; l < slot_lines; l += NT)
      st_line_v4(sslot + l * 16, make_uint4(0u, sflag, 0u, sflag));
  }
}

// ---------------------------------------------------------------------------
// LL128
// ---------------------------------------------------------------------------

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
    v = ld_line_v4(p);
  }
}

// Same payload element size on both sides (all rows except bf16's owner row).
template <typename T, int PRIM, int NT>
__device__ __forceinline__ void ll128_slice(const RingArgs& a, const T* in, T* out, const char* rslot, char* sslot,
                                            int64_t nelem, uint64_t rflag, uint64_t sflag, volatile int* sh_abort,
                                            uint64_t info) {
  constexpr int NW = NT / 32;
  constexpr int UG = 1;
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kIn = PRIM == kSend || kRecvPartial;  // copySend loads its input raw
  constexpr bool kHasRecv = PRIM != kSend && PRIM != kCopySend;
  constexpr bool kHasSend = PRIM != kRecv && PRIM != kRecvReduceCopy;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv ||
                        PRIM == kRecvReduceCopy || PRIM == kCopySend;
  // payload element bytes of this row (the received side for recvReduceCopy)
  constexpr int EB = (PRIM == kSend || PRIM == kRecvReduceSend) ? 4
                   : (PRIM == kRecvReduceCopySend) ? 4  // f32 only here
                   : (PRIM == kRecvReduceCopy) ? 4
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
        if (kHasRecv) rv[u] = ld_line_v4(rslot + g * 512 + 16 * L.lane);
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
        if (PRIM == kRecvReduceCopy && sizeof(T) == 2)  // bf16 output, rounded once
          pay = make_uint4(round_bf16_pair(v[0], v[1]), round_bf16_pair(v[2], v[3]), 0u, 0u);
        else
          pay = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
      } else if (PRIM == kCopySend) {
        pay = kv > 0 ? load_raw_n<T>(in + e0, kv, kmax) : make_uint4(0u, 0u, 0u, 0u);  // already final
      } else {
        pay = rv[u];  // final values pass through unchanged
      }
      if (kOut && kv > 0) store_out_n<T>(out + e0, kv, kmax, pay);
      if (kHasSend) {
        if (L.flag_lane) {
          pay.z = (uint32_t)sflag;
          pay.w = (uint32_t)(sflag >> 32);
        }
        st_line_v4(sslot + g * 512 + 16 * L.lane, pay);
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
      uint4 rv = ld_line_v4(rp);
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
      st_line_v4(sslot + gs * 512 + 16 * L.lane, pay);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
__device__ __noinline__ bool wait_credit(const RingArgs& a, const uint64_t* head, uint64_t base_send, uint64_t step,
                                         uint64_t* head_seen, uint64_t info) {
  Spin sp;
  while (true) {
    const uint64_t h = *head_seen > base_send ? *head_seen : base_send;
    if (h + kSteps >= step + 1) return true;
    *head_seen = ld_acquire_u64(head);
    const uint64_t h2 = *head_seen > base_send ? *head_seen : base_send;
    if (h2 + kSteps >= step + 1) return true;
    if (sp.poll(a, info, step + 1)) return false;
  }
}

// Send credit of a split connection: both halves of the receiver must have
// released the slot. (Each step's split point follows the step's size, so a
// later step in the same slot can give one half lines that the other half's
// receiver read in the earlier step.)
__device__ __noinline__ bool wait_credit_both(const RingArgs& a, ConnCounters* cs, uint64_t base_send, uint64_t step,
                                              uint64_t (&seen)[2], uint64_t info) {
  Spin sp;
  auto ok = [&]() {
    const uint64_t h0 = seen[0] > base_send ? seen[0] : base_send;
    const uint64_t h1 = seen[1] > base_send ? seen[1] : base_send;
    return (h0 < h1 ? h0 : h1) + kSteps >= step + 1;
  };
  while (true) {
    if (ok()) return true;
    const uint64_t h0 = ld_acquire_u64(&cs->head), h1 = ld_acquire_u64(&cs->head_h1);
    seen[0] = h0 > seen[0] ? h0 : seen[0];
    seen[1] = h1 > seen[1] ? h1 : seen[1];
    if (ok()) return true;
    if (sp.poll(a, info, step + 1)) return false;
  }
}

// Pacing (thread 0, before a large step): wait until the LAST line of the
// step carries the step's flag. All ranks run at the same speed on one GPU, so
// without this a receiver chases its sender line by line and most of its
// early loads see stale flags, each costing another L2 round trip. The wait
// is only a hint about progress: every line is still accepted by its own flag
// alone. Steps that fit in one pass of the block (<= one unit per thread for
// LL, <= one group per warp for LL128) keep pure line-by-line streaming.
template <typename T, int PROTO, int NT>
__device__ __noinline__ bool pace_wait(const RingArgs& a, const char* rslot, int prim, int64_t nelem, uint64_t rstep,
                                       uint64_t info) {
  if (nelem <= 0 || !row_recvs(prim)) return true;
  const bool partial = row_recvs_partial(prim);
  Spin sp;
  if (PROTO == kLL) {
    constexpr int K = LLUnit<T>::kElems;
    const int64_t nunits = div_up(nelem, K);
    if (nunits <= NT) return true;
    const int64_t lines = nunits * (partial ? LLUnit<T>::kPartLines : 1);
    const char* p = rslot + (lines - 1) * 16;
    const uint32_t flag = ll_flag(a, rstep);
    uint4 v = ld_line_v4(p);
    while (!ll_ready(v, flag)) {
      if (sp.poll(a, info, flag)) return false;
      v = ld_line_v4(p);
    }
    return true;
  } else {
    const int64_t ngroups = div_up(nelem * (partial ? 4 : (int64_t)sizeof(T)), 480);
    if (ngroups <= NT / 32) return true;
    const uint64_t* p = reinterpret_cast<const uint64_t*>(rslot + (4 * (ngroups - 1) + 3) * 128 + 120);
    const uint64_t flag = rstep + 1;
    while (true) {
      uint64_t f;
      f = ld_relaxed_u64(p);
      if (f == flag) return true;
      if (sp.poll(a, info, flag)) return false;
    }
  }
}

template <typename T, int PROTO, int NT>
__device__ __forceinline__ void line_slice(int prim, const RingArgs& a, const T* in, T* out, const char* rslot,
                                           char* sslot, int64_t nelem, uint64_t rstep, uint64_t sstep,
                                           volatile int* sh_abort, uint64_t info, uint16_t* stage) {
  if (PROTO == kLL) {
    const uint32_t rf = ll_flag(a, rstep), sf = ll_flag(a, sstep);
    const bool clean = ll_cleanup_step(a, sstep);
    switch (prim) {
      case kSend: ll_slice<T, kSend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info); break;
      case kRecvReduceSend:
        ll_slice<T, kRecvReduceSend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info);
        break;
      case kRecvReduceCopySend:
        ll_slice<T, kRecvReduceCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info);
        break;
      case kRecvCopySend:
        ll_slice<T, kRecvCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info);
        break;
      case kRecvReduceCopy:
        ll_slice<T, kRecvReduceCopy, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info);
        break;
      case kCopySend: ll_slice<T, kCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info); break;
      default: ll_slice<T, kRecv, NT>(a, in, out, rslot, sslot, nelem, rf, sf, clean, sh_abort, info); break;
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
      case kRecvReduceCopy:
        ll128_slice<T, kRecvReduceCopy, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info);
        break;
      case kCopySend: ll128_slice<T, kCopySend, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
      default: ll128_slice<T, kRecv, NT>(a, in, out, rslot, sslot, nelem, rf, sf, sh_abort, info); break;
    }
  }
}

// Checks (thread 0) before a group of steps: the debug bounds of each of the
// next `steps` slices from cursor c, and the send credit of the last send
// among them; with one step per group also the pacing wait. False if a
// check failed or a wait gave up.
template <typename T, int PROTO, int NT>
__device__ __forceinline__ bool line_group_checks(const RingArgs& a, const Geometry& g, int dense, SliceCursor c,
                                                  int steps, uint64_t rstep, uint64_t sstep, ConnCounters* cs,
                                                  uint64_t base_send, uint64_t* head_seen, const char* fifo_recv,
                                                  uint64_t info) {
  const SliceCursor first = c;
  const uint64_t rstep0 = rstep;
  uint64_t last_send = 0;
  bool sends = false;
  for (int k = 0; k < steps && c.valid; k++) {
    if (!slice_in_bounds(a, dense, c, rstep, sstep, info | k)) return false;
    if (row_sends(c.prim)) {
      last_send = sstep++;
      sends = true;
    }
    if (row_recvs(c.prim)) rstep++;
    cursor_next(g, c);
  }
  if (sends && !wait_credit(a, &cs->head, base_send, last_send, head_seen, info | (3u << 24))) return false;
  if (steps == 1)
    return pace_wait<T, PROTO, NT>(a, fifo_recv + (int64_t)(rstep0 % kSteps) * g.step_bytes, first.prim, first.nelem,
                                   rstep0, info | (9u << 24));
  return true;
}

// Polling form. `epoch` steps per group: 1 = the block meets at a barrier
// after every step (head published, next step's credit and pacing checked);
// kSteps / 2 = steps whose lines the block covers in one pass (small
// messages): each thread then moves from step to step on its own lines, the
// block meets only every `epoch` steps (and at the end), where it publishes
// the head of every step read and takes the credit for the next group's
// sends. Lines are accepted by their flags either way; the group is at most
// half the FIFO, so no slot is written again before its reader's head covers
// it. (With a barrier per step, the block waits at every step for its slowest
// thread's poll.)
template <typename T, int PROTO, int NT>
__global__ void __launch_bounds__(NT, 1) ring_line_kernel(const __grid_constant__ RingArgs a, int epoch) {
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
  const int ring_idx = ring_index_of(a, dense, rank);
  const int e_send = ring_idx, e_recv = (ring_idx + N - 1) % N;
  ConnCounters* cs = conn_at(a, dense, e_send);
  ConnCounters* cr = conn_at(a, dense, e_recv);
  char* fifo_send = fifo_at(a, dense, e_send);
  const char* fifo_recv = fifo_at(a, dense, e_recv);
  if (threadIdx.x == 0) {
    // Both counters belong to this block and equal the previous call's final
    // step; they are read together with the header (one round trip, not two).
    const uint64_t tail0 = ld_relaxed_u64(&cs->tail), head0 = ld_relaxed_u64(&cr->head);
    sh_abort = entry_check(a) ? 0 : 1;
    sh_base_send = tail0;
    sh_base_recv = head0;
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
  if (threadIdx.x == 0 && c.valid &&
      !line_group_checks<T, PROTO, NT>(a, g, dense, c, epoch, rstep, sstep, cs, base_send, &head_seen, fifo_recv,
                                       info))
    sh_abort = 1;
  __syncthreads();
  uint32_t i = 0;
  int in_group = 0;
  uint64_t head_published = rstep;
  bool go = c.valid && !sh_abort;
  while (go) {
    const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
    char* sslot = fifo_send + (int64_t)(sstep % kSteps) * step_bytes;
    int64_t in_off, out_off;
    slice_offsets(a, dense, c, &in_off, &out_off);
    line_slice<T, PROTO, NT>(c.prim, a, in + in_off, out + out_off, rslot, sslot, c.nelem, rstep, sstep, &sh_abort,
                             info | (2u << 24) | i, stage);
    SliceCursor nx = c;
    cursor_next(g, nx);
    const uint64_t nsstep = sstep + (row_sends(c.prim) ? 1 : 0);
    const uint64_t nrstep = rstep + (row_recvs(c.prim) ? 1 : 0);
    if (++in_group >= epoch || !nx.valid) {
      int aborted;
      if (epoch == 1) {
        // checks and credit for the next step, taken while the block finishes this one
        if (threadIdx.x == 0 && nx.valid && !sh_abort &&
            !line_group_checks<T, PROTO, NT>(a, g, dense, nx, 1, nrstep, nsstep, cs, base_send, &head_seen,
                                             fifo_recv, info | (i + 1)))
          sh_abort = 1;
        aborted = __syncthreads_or(sh_abort);  // the same value for every thread
        if (threadIdx.x == 0 && !aborted && nrstep > head_published && a.fault != kFaultDropHead) {
          st_relaxed_u64(&cr->head, nrstep);  // every thread has read this step's lines
          head_published = nrstep;
        }
      } else {
        // the head of every step read first, then the credit of the next
        // group: a block that waits for its receiver's head has published
        // its own, so the waits around the ring cannot close a cycle
        aborted = __syncthreads_or(sh_abort);
        if (threadIdx.x == 0 && !aborted) {
          if (nrstep > head_published && a.fault != kFaultDropHead) {
            st_relaxed_u64(&cr->head, nrstep);  // every thread has read these steps' lines
            head_published = nrstep;
          }
          if (nx.valid && !line_group_checks<T, PROTO, NT>(a, g, dense, nx, epoch, nrstep, nsstep, cs, base_send,
                                                           &head_seen, fifo_recv, info | (i + 1)))
            sh_abort = 1;
        }
        if (nx.valid && !aborted) aborted = __syncthreads_or(sh_abort);
      }
      in_group = 0;
      go = nx.valid && !aborted;
    }
    rstep = nrstep;
    sstep = nsstep;
    c = nx;
    i++;
  }
  // the sender's step count carries over to the next call; the counters of
  // the second half of a split connection follow (no block of this launch
  // moves that half)
  if (threadIdx.x == 0 && !sh_abort) {
    st_relaxed_u64(&cs->tail, sstep);
    st_relaxed_u64(&cs->tail_h1, sstep);
    st_relaxed_u64(&cr->head_h1, rstep);
  }
}

// ---------------------------------------------------------------------------
// LL128, bulk form: the same lines, flags and head credits, with the loads of
// large steps moved onto the TMA engine (used from first-loop chunks of
// kL8BulkMinChunk elements; a tile may be partial). Roles as in the Simple
// kernel:
//   warp 0, lane 0  waiter: send credit (head + NCCL_STEPS >= step + 1);
//                   arrives ready[i % D].
//   warp 1, lane 0  loader: per tile of 64 line groups (kL8TileElems
//                   elements; rows that move bf16 finals and read no input
//                   fill them with 2 * kL8TileElems elements; LL:
//                   kLLTileElems), a bulk copy of the tile's user input into a
//                   smem stage as soon as the stage is free, a pacing wait for
//                   the flag of the tile's last received line (the flags of up
//                   to kPaceBatch tiles read together; LL: the step's last line,
//                   once per step), then a bulk copy of the tile's received lines.
//   warps 3..18     workers: per 4-line group, check every line's flag in
//                   shared memory (a line that is not yet there is re-polled
//                   from global memory until its flag matches), reduce, store
//                   the output and write the outgoing lines, one warp access
//                   per 4 lines, flag word included.
//   warp 2, lane 0  poster: publishes the head once the step's lines are read.
// A line is accepted only by its own flag, exactly as in the polling form.
// LL128's split instance (SPLIT = 2) runs two blocks per (rank, channel):
// each moves a fixed part of every step's elements with the roles above, keeps
// its own head counter, and takes a slot's credit from both receiver parts.
// ---------------------------------------------------------------------------
constexpr int kL8TileElems = 7680;   // 64 groups of binary32 payload, 32 groups of bf16 payload
constexpr int kL8TileGroups = kL8TileElems * 4 / 480;
constexpr int kL8BulkMinChunk = 960;  // chunks at least this long take the bulk form (measured: 480-7680)
constexpr int kL8Warps = 16;
constexpr int kL8WorkThreads = 32 * kL8Warps;
constexpr int kL8Threads = 32 * 3 + kL8WorkThreads;
constexpr int kL8Depth = 4;
constexpr int kL8MaxStages = 8;
constexpr int kL8SmemBudget = 200 * 1024;

template <typename T>
__host__ __device__ constexpr int l8_stage_bytes() { return kL8TileGroups * 512 + kL8TileElems * (int)sizeof(T); }
template <typename T>
__host__ __device__ constexpr int l8_max_stages() {
  return kL8SmemBudget / l8_stage_bytes<T>() < kL8MaxStages ? kL8SmemBudget / l8_stage_bytes<T>() : kL8MaxStages;
}

// Input element j of the tile (binary32): from the staged prefix, or from
// global memory past it (the last < 16 bytes of a slice).
template <typename T>
__device__ __forceinline__ float l8_input(const char* s_in, const T* g_tile, int j, int covered) {
  if (j < covered) {
    if constexpr (sizeof(T) == 4) return reinterpret_cast<const float*>(s_in)[j];
    else return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(s_in)[j] << 16);
  }
  if constexpr (sizeof(T) == 4) return __uint_as_float(ld_cg_u32(g_tile + j));
  uint16_t h;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(g_tile + j) : "memory");
  return __uint_as_float((uint32_t)h << 16);
}

// The lane's kmax (4, or 2 for flag lanes) input elements at tile element el,
// widened to binary32, zeros past kv: one shared-memory vector load when the
// whole piece is staged, element by element otherwise.
template <typename T>
__device__ __forceinline__ void l8_input_piece(const char* s_in, const T* g_tile, int el, int kv, int kmax,
                                               int covered, float (&x)[4]) {
  if (kv == kmax && el + kv <= covered) {
    if constexpr (sizeof(T) == 4) {
      if (kmax == 4) {
        const float4 w = *reinterpret_cast<const float4*>(s_in + el * 4);
        x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
      } else {
        const float2 w = *reinterpret_cast<const float2*>(s_in + el * 4);
        x[0] = w.x; x[1] = w.y; x[2] = 0.f; x[3] = 0.f;
      }
    } else {
      if (kmax == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(s_in + el * 2);
        x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(s_in + el * 2);
        x[0] = bf16lo(w); x[1] = bf16hi(w); x[2] = 0.f; x[3] = 0.f;
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; j++) x[j] = j < kv ? l8_input<T>(s_in, g_tile, el + j, covered) : 0.f;
}

// The lane's kmax elements of T at tile element el as raw bits (kmax *
// sizeof(T) = 16 or 8 bytes), zeros past kv: from shared memory when the whole
// piece is staged, element by element otherwise.
template <typename T>
__device__ __forceinline__ uint4 l8_raw_piece(const char* s_in, const T* g_tile, int el, int kv, int kmax,
                                              int covered) {
  const int bytes = kmax * (int)sizeof(T);
  if (kv == kmax && el + kv <= covered) {
    if (bytes == 16) return *reinterpret_cast<const uint4*>(s_in + el * (int)sizeof(T));
    const uint2 w = *reinterpret_cast<const uint2*>(s_in + el * (int)sizeof(T));
    return make_uint4(w.x, w.y, 0u, 0u);
  }
  uint32_t wd[4] = {0u, 0u, 0u, 0u};
  for (int j = 0; j < kv; j++) {
    const int e = el + j;
    uint32_t bits;
    if (e < covered) {
      bits = sizeof(T) == 4 ? reinterpret_cast<const uint32_t*>(s_in)[e]
                            : (uint32_t)reinterpret_cast<const uint16_t*>(s_in)[e];
    } else if constexpr (sizeof(T) == 4) {
      bits = ld_cg_u32(g_tile + e);
    } else {
      uint16_t h;
      asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(h) : "l"(g_tile + e) : "memory");
      bits = h;
    }
    if (sizeof(T) == 4) wd[j] = bits;
    else wd[j >> 1] |= bits << ((j & 1) * 16);
  }
  return make_uint4(wd[0], wd[1], wd[2], wd[3]);
}

// Check a group's flags as staged; re-poll stale lines from global memory.
__device__ __forceinline__ bool l8_accept(const RingArgs& a, uint4& v, const char* gline, uint64_t flag, bool flag_lane,
                                          volatile int* sh_abort, uint64_t info) {
  const bool need = flag_lane && ll128_flag_of(v) != flag;
  if (!__any_sync(kFullMask, need)) return true;
  v = ld_line_v4(gline);
  return ll128_poll(a, gline, flag, flag_lane, v, sh_abort, info);
}

template <typename T, int PRIM>
__device__ __forceinline__ void l8_tile_same_layout(const RingArgs& a, const char* s_lines, const char* s_in,
                                                    const T* g_in_tile, T* g_out_tile, const char* g_rlines,
                                                    char* g_slines, int ne, int covered, uint64_t rflag, uint64_t sflag,
                                                    volatile int* sh_abort, uint64_t info, int w) {
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kHasRecv = PRIM != kSend && PRIM != kCopySend;
  constexpr bool kHasSend = PRIM != kRecv && PRIM != kRecvReduceCopy;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv ||
                        PRIM == kRecvReduceCopy || PRIM == kCopySend;
  constexpr int EB = (PRIM == kSend || kRecvPartial) ? 4 : (int)sizeof(T);
  const LL128Lane L;
  const int kmax = L.piece_bytes / EB;
  const int ng = (int)div_up((int64_t)ne * EB, 480);
  for (int gl = w; gl < ng; gl += kL8Warps) {
    uint4 rv = make_uint4(0u, 0u, 0u, 0u);
    bool ok = true;
    if (kHasRecv) {
      rv = *reinterpret_cast<const uint4*>(s_lines + gl * 512 + 16 * L.lane);
      ok = l8_accept(a, rv, g_rlines + gl * 512 + 16 * L.lane, rflag, L.flag_lane, sh_abort, info);
    }
    if (!ok) return;  // uniform across the warp
    const int el = (gl * 480 + L.piece_off) / EB;
    const int kv = (int)imax(0, imin(kmax, ne - el));
    uint4 pay;
    if (kRecvPartial || PRIM == kSend) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (kRecvPartial) {
        v[0] = __uint_as_float(rv.x); v[1] = __uint_as_float(rv.y);
        v[2] = __uint_as_float(rv.z); v[3] = __uint_as_float(rv.w);
      }
      float x[4];
      l8_input_piece<T>(s_in, g_in_tile, el, kv, kmax, covered, x);
#pragma unroll
      for (int j = 0; j < 4; j++) v[j] = j < kv ? (kRecvPartial ? __fadd_rn(v[j], x[j]) : x[j]) : 0.f;
      if (PRIM == kRecvReduceCopy && sizeof(T) == 2)  // bf16 output, rounded once
        pay = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), 0u, 0u);
      else
        pay = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
    } else if (PRIM == kCopySend) {
      pay = l8_raw_piece<T>(s_in, g_in_tile, el, kv, kmax, covered);  // already final
    } else {
      pay = rv;  // final values pass through unchanged
    }
    if (kOut && kv > 0) store_out_n<T>(g_out_tile + el, kv, kmax, pay);
    if (kHasSend) {
      if (L.flag_lane) {
        pay.z = (uint32_t)sflag;
        pay.w = (uint32_t)(sflag >> 32);
      }
      st_line_v4(g_slines + gl * 512 + 16 * L.lane, pay);
    }
  }
}

// A lane's piece of a full group (every element present and staged): the
// input word that holds it, read as one aligned shared-memory vector. A flag
// lane's piece is half as long and may sit in the upper half of that word.
template <typename T, int EB>
__device__ __forceinline__ void l8_full_input(const char* s_in, int el, float (&x)[4]) {
  if constexpr (sizeof(T) == 4) {
    const int bo = el * 4;
    const float4 w4 = *reinterpret_cast<const float4*>(s_in + (bo & ~15));
    const bool hi = (bo & 8) != 0;
    x[0] = hi ? w4.z : w4.x;
    x[1] = hi ? w4.w : w4.y;
    x[2] = w4.z;
    x[3] = w4.w;
  } else {
    const int bo = el * 2;
    const uint2 w2 = *reinterpret_cast<const uint2*>(s_in + (bo & ~7));
    const uint32_t lo = (bo & 4) ? w2.y : w2.x;
    x[0] = bf16lo(lo);
    x[1] = bf16hi(lo);
    x[2] = bf16lo(w2.y);
    x[3] = bf16hi(w2.y);
  }
}
template <typename T>
__device__ __forceinline__ uint4 l8_full_raw(const char* s_in, int el) {
  const int bo = el * (int)sizeof(T);  // payload bytes of the piece = group layout bytes
  const uint4 w = *reinterpret_cast<const uint4*>(s_in + (bo & ~15));
  return (bo & 8) ? make_uint4(w.z, w.w, 0u, 0u) : w;
}
// Store a lane's output piece: kmax elements of T (16 / EB of them, half as
// many on flag lanes) from the raw bits in w.
template <typename T, int EB>
__device__ __forceinline__ void l8_full_store(T* p, bool flag_lane, uint4 w) {
  constexpr int kBytes = 16 / EB * (int)sizeof(T);  // 16, or 8 for bf16 from binary32 partial sums
  if constexpr (kBytes == 16) {
    if (flag_lane) st_v2(p, make_uint2(w.x, w.y));
    else st_v4(p, w);
  } else {
    if (flag_lane) *reinterpret_cast<uint32_t*>(p) = w.x;
    else st_v2(p, make_uint2(w.x, w.y));
  }
}

// Same values and lines as l8_tile_same_layout for a full tile (TE elements,
// all input staged): every group is whole, so the lanes need no element
// bounds and each warp's groups are known at compile time.
template <typename T, int PRIM, int TE>
__device__ __forceinline__ void l8_tile_full(const RingArgs& a, const char* s_lines, const char* s_in,
                                             T* g_out_tile, const char* g_rlines, char* g_slines, uint64_t rflag,
                                             uint64_t sflag, volatile int* sh_abort, uint64_t info, int w) {
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kHasRecv = PRIM != kSend && PRIM != kCopySend;
  constexpr bool kHasSend = PRIM != kRecv && PRIM != kRecvReduceCopy;
  constexpr bool kOut = PRIM == kRecvReduceCopySend || PRIM == kRecvCopySend || PRIM == kRecv ||
                        PRIM == kRecvReduceCopy || PRIM == kCopySend;
  constexpr int EB = (PRIM == kSend || kRecvPartial) ? 4 : (int)sizeof(T);
  constexpr int NG = TE * EB / 480;
  static_assert(TE * EB % 480 == 0 && NG <= kL8TileGroups, "a tile is whole groups of one stage");
  constexpr int GPW = (NG + kL8Warps - 1) / kL8Warps;  // groups of a warp: w, w + 16, ...
  const int gw = NG % kL8Warps == 0 || w < NG % kL8Warps ? GPW : GPW - 1;
  const LL128Lane L;
  uint4 rv[GPW];
  if (kHasRecv) {
#pragma unroll
    for (int q = 0; q < GPW; q++)
      if (q < gw) rv[q] = *reinterpret_cast<const uint4*>(s_lines + (w + q * kL8Warps) * 512 + 16 * L.lane);
#pragma unroll
    for (int q = 0; q < GPW; q++)
      if (q < gw &&
          !l8_accept(a, rv[q], g_rlines + (w + q * kL8Warps) * 512 + 16 * L.lane, rflag, L.flag_lane, sh_abort, info))
        return;  // uniform across the warp
  }
#pragma unroll
  for (int q = 0; q < GPW; q++) {
    if (q >= gw) break;
    const int gl = w + q * kL8Warps;
    const int el = (gl * 480 + L.piece_off) / EB;
    uint4 pay;
    if constexpr (kRecvPartial || PRIM == kSend) {
      float x[4];
      l8_full_input<T, EB>(s_in, el, x);
      float v[4];
      if constexpr (kRecvPartial) {
        v[0] = __fadd_rn(__uint_as_float(rv[q].x), x[0]);
        v[1] = __fadd_rn(__uint_as_float(rv[q].y), x[1]);
        v[2] = __fadd_rn(__uint_as_float(rv[q].z), x[2]);
        v[3] = __fadd_rn(__uint_as_float(rv[q].w), x[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = x[j];
      }
      if constexpr (PRIM == kRecvReduceCopy && sizeof(T) == 2)  // bf16 output, rounded once
        pay = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), 0u, 0u);
      else
        pay = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
    } else if constexpr (PRIM == kCopySend) {
      pay = l8_full_raw<T>(s_in, el);  // already final
    } else {
      pay = rv[q];  // final values pass through unchanged
    }
    if constexpr (kOut) l8_full_store<T, (PRIM == kRecvReduceCopy ? 4 : (int)sizeof(T))>(g_out_tile + el, L.flag_lane, pay);
    if constexpr (kHasSend) {
      if (L.flag_lane) {
        pay.z = (uint32_t)sflag;
        pay.w = (uint32_t)(sflag >> 32);
      }
      st_line_v4(g_slines + gl * 512 + 16 * L.lane, pay);
    }
  }
}

// bf16 owner row: binary32 partial sums in (120 elements per group), bf16
// finals out (240 elements per group). The finals are written over the staged
// bf16 input (each element by the lane that read it), then re-read in the
// send layout after a barrier of the worker warps.
__device__ __forceinline__ void l8_tile_owner_bf16(const RingArgs& a, const char* s_lines, char* s_in,
                                                   const uint16_t* g_in_tile, uint16_t* g_out_tile,
                                                   const char* g_rlines, char* g_slines, int ne, int covered,
                                                   uint64_t rflag, uint64_t sflag, volatile int* sh_abort,
                                                   uint64_t info, int w, uint64_t* bar_fin, uint32_t* fin_uses) {
  const LL128Lane L;
  uint16_t* fin = reinterpret_cast<uint16_t*>(s_in);
  const int ngr = (int)div_up((int64_t)ne * 4, 480), ngs = (int)div_up((int64_t)ne * 2, 480);
  bool ok = true;
  for (int gl = w; gl < ngr && ok; gl += kL8Warps) {
    uint4 rv = *reinterpret_cast<const uint4*>(s_lines + gl * 512 + 16 * L.lane);
    ok = l8_accept(a, rv, g_rlines + gl * 512 + 16 * L.lane, rflag, L.flag_lane, sh_abort, info);
    if (!ok) break;
    const int kmax = L.piece_bytes / 4;
    const int el = (gl * 480 + L.piece_off) / 4;
    const int kv = (int)imax(0, imin(kmax, ne - el));
    const float p[4] = {__uint_as_float(rv.x), __uint_as_float(rv.y), __uint_as_float(rv.z), __uint_as_float(rv.w)};
    float x[4], v[4];
    l8_input_piece<uint16_t>(s_in, g_in_tile, el, kv, kmax, covered, x);
#pragma unroll
    for (int j = 0; j < 4; j++) v[j] = j < kv ? __fadd_rn(p[j], x[j]) : 0.f;
    const uint4 wv = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), 0u, 0u);  // rounded once
    if (kv > 0) store_out_n<uint16_t>(g_out_tile + el, kv, kmax, wv);
    // a whole piece in one shared-memory store: el is a multiple of 4 (of 2 on
    // a flag lane), so the 8 (4) bytes are aligned
    if (kv == kmax && kmax == 4) *reinterpret_cast<uint2*>(fin + el) = make_uint2(wv.x, wv.y);
    else if (kv == kmax) *reinterpret_cast<uint32_t*>(fin + el) = wv.x;
    else
      for (int j = 0; j < kv; j++) fin[el + j] = (uint16_t)((j < 2 ? wv.x : wv.y) >> ((j & 1) * 16));
  }
  // every worker warp passes this barrier once per owner tile, on every path;
  // the wait is bounded like every other wait of the kernel
  __syncwarp();
  if (L.lane == 0) mbar_arrive(bar_fin);
  const bool passed = mbar_wait(a, bar_fin, (*fin_uses) & 1u, info);
  (*fin_uses)++;
  if (!passed || *sh_abort) {
    *sh_abort = 1;
    return;
  }
  for (int gl = w; gl < ngs; gl += kL8Warps) {
    const int kmax = L.piece_bytes / 2;
    const int el = (gl * 480 + L.piece_off) / 2;
    const int kv = (int)imax(0, imin(kmax, ne - el));
    uint32_t wd[4] = {0u, 0u, 0u, 0u};
    if (kv == kmax && kmax == 8) {  // 16-byte aligned: el * 2 = 480 * gl + piece_off
      const uint4 q = *reinterpret_cast<const uint4*>(fin + el);
      wd[0] = q.x; wd[1] = q.y; wd[2] = q.z; wd[3] = q.w;
    } else if (kv == kmax) {  // a flag lane's 8 bytes, 8-byte aligned
      const uint2 q = *reinterpret_cast<const uint2*>(fin + el);
      wd[0] = q.x; wd[1] = q.y;
    } else {
#pragma unroll
      for (int j = 0; j < 8; j++)
        if (j < kv) wd[j >> 1] |= (uint32_t)fin[el + j] << ((j & 1) * 16);
    }
    uint4 pay = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    if (L.flag_lane) {
      pay.z = (uint32_t)sflag;
      pay.w = (uint32_t)(sflag >> 32);
    }
    st_line_v4(g_slines + gl * 512 + 16 * L.lane, pay);
  }
}

// bf16 owner row, full tile (kL8TileElems elements, all input staged): warp
// w takes the outgoing groups w and w + kL8Warps and, for each, the two
// received groups 2g and 2g + 1 that hold its 240 elements; a lane rounds its
// sums once to bf16, stores its output piece and writes the finals over its
// own piece of the staged input (pieces are disjoint, so only this warp
// touches these elements), and after a warp barrier the warp re-reads them
// in the send layout. No barrier across warps.
__device__ __forceinline__ void l8_tile_owner_bf16_full(const RingArgs& a, const char* s_lines, char* s_in,
                                                        uint16_t* g_out_tile, const char* g_rlines, char* g_slines,
                                                        uint64_t rflag, uint64_t sflag, volatile int* sh_abort,
                                                        uint64_t info, int w) {
  constexpr int NS = kL8TileElems * 2 / 480;  // outgoing groups of a tile
  static_assert(NS % kL8Warps == 0, "whole outgoing groups per warp");
  const LL128Lane L;
  uint16_t* fin = reinterpret_cast<uint16_t*>(s_in);
#pragma unroll
  for (int q = 0; q < NS / kL8Warps; q++) {
    const int gs = w + q * kL8Warps;
    uint4 rv[2];
#pragma unroll
    for (int h = 0; h < 2; h++) rv[h] = *reinterpret_cast<const uint4*>(s_lines + (2 * gs + h) * 512 + 16 * L.lane);
#pragma unroll
    for (int h = 0; h < 2; h++)
      if (!l8_accept(a, rv[h], g_rlines + (2 * gs + h) * 512 + 16 * L.lane, rflag, L.flag_lane, sh_abort, info))
        return;  // uniform across the warp
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int el = ((2 * gs + h) * 480 + L.piece_off) / 4;
      float x[4];
      l8_full_input<uint16_t, 4>(s_in, el, x);
      const float v0 = __fadd_rn(__uint_as_float(rv[h].x), x[0]), v1 = __fadd_rn(__uint_as_float(rv[h].y), x[1]);
      const float v2 = __fadd_rn(__uint_as_float(rv[h].z), x[2]), v3 = __fadd_rn(__uint_as_float(rv[h].w), x[3]);
      const uint4 wv = make_uint4(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3), 0u, 0u);  // rounded once
      l8_full_store<uint16_t, 4>(g_out_tile + el, L.flag_lane, wv);
      if (L.flag_lane) *reinterpret_cast<uint32_t*>(fin + el) = wv.x;  // 2 elements, 4-byte aligned
      else *reinterpret_cast<uint2*>(fin + el) = make_uint2(wv.x, wv.y);  // 4 elements, 8-byte aligned
    }
    __syncwarp();
    const int es = (gs * 480 + L.piece_off) / 2;
    uint4 pay;
    if (L.flag_lane) {
      const uint2 f = *reinterpret_cast<const uint2*>(fin + es);  // 4 elements, 8-byte aligned
      pay = make_uint4(f.x, f.y, (uint32_t)sflag, (uint32_t)(sflag >> 32));
    } else {
      pay = *reinterpret_cast<const uint4*>(fin + es);  // 8 elements, 16-byte aligned
    }
    st_line_v4(g_slines + gs * 512 + 16 * L.lane, pay);
  }
}

template <typename T>
__device__ __forceinline__ void l8_tile_any(int prim, const RingArgs& a, const char* s_lines, char* s_in,
                                            const T* g_in_tile, T* g_out_tile, const char* g_rlines, char* g_slines,
                                            int ne, int te, int covered, uint64_t rflag, uint64_t sflag,
                                            volatile int* sh_abort, uint64_t info, int w, uint64_t* bar_fin,
                                            uint32_t* fin_uses) {
  if (ne == te && covered == ne) {
#define RAR_L8_FULL(P) l8_tile_full<T, P, kL8TileElems>(a, s_lines, s_in, g_out_tile, g_rlines, g_slines, rflag, sflag, sh_abort, info, w)
#define RAR_L8_FULL2(P) l8_tile_full<T, P, 2 * kL8TileElems>(a, s_lines, s_in, g_out_tile, g_rlines, g_slines, rflag, sflag, sh_abort, info, w)
    switch (prim) {
      case kSend: RAR_L8_FULL(kSend); return;
      case kRecvReduceSend: RAR_L8_FULL(kRecvReduceSend); return;
      case kRecvReduceCopySend:
        if constexpr (sizeof(T) == 4) {
          RAR_L8_FULL(kRecvReduceCopySend);
        } else {
          l8_tile_owner_bf16_full(a, s_lines, s_in, reinterpret_cast<uint16_t*>(g_out_tile), g_rlines, g_slines,
                                  rflag, sflag, sh_abort, info, w);
        }
        return;
      case kRecvCopySend:
        if constexpr (sizeof(T) == 2) {
          if (te == 2 * kL8TileElems) {
            RAR_L8_FULL2(kRecvCopySend);
            return;
          }
        }
        RAR_L8_FULL(kRecvCopySend);
        return;
      case kRecvReduceCopy: RAR_L8_FULL(kRecvReduceCopy); return;
      case kCopySend: RAR_L8_FULL(kCopySend); return;
      default:
        if constexpr (sizeof(T) == 2) {
          if (te == 2 * kL8TileElems) {
            RAR_L8_FULL2(kRecv);
            return;
          }
        }
        RAR_L8_FULL(kRecv);
        return;
    }
#undef RAR_L8_FULL2
#undef RAR_L8_FULL
  }
  switch (prim) {
    case kSend:
      l8_tile_same_layout<T, kSend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered, rflag,
                                    sflag, sh_abort, info, w);
      break;
    case kRecvReduceSend:
      l8_tile_same_layout<T, kRecvReduceSend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne,
                                              covered, rflag, sflag, sh_abort, info, w);
      break;
    case kRecvReduceCopySend:
      if constexpr (sizeof(T) == 4)
        l8_tile_same_layout<T, kRecvReduceCopySend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne,
                                                    covered, rflag, sflag, sh_abort, info, w);
      else
        l8_tile_owner_bf16(a, s_lines, s_in, reinterpret_cast<const uint16_t*>(g_in_tile),
                           reinterpret_cast<uint16_t*>(g_out_tile), g_rlines, g_slines, ne, covered, rflag, sflag,
                           sh_abort, info, w, bar_fin, fin_uses);
      break;
    case kRecvCopySend:
      l8_tile_same_layout<T, kRecvCopySend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered,
                                            rflag, sflag, sh_abort, info, w);
      break;
    case kRecvReduceCopy:
      l8_tile_same_layout<T, kRecvReduceCopy>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne,
                                              covered, rflag, sflag, sh_abort, info, w);
      break;
    case kCopySend:
      l8_tile_same_layout<T, kCopySend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered,
                                        rflag, sflag, sh_abort, info, w);
      break;
    default:
      l8_tile_same_layout<T, kRecv>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered, rflag,
                                    sflag, sh_abort, info, w);
      break;
  }
}

// ---------------------------------------------------------------------------
// LL, bulk form: the same roles as LL128's, for LL lines. A tile of
// kLLTileElems elements starts on a line boundary of both FIFOs; its received
// lines are bulk-copied into shared memory, every worker thread takes whole
// units (the elements of one outgoing line, or of one received line on rows
// that send nothing), accepts each line only by its two flags (a line not yet
// there is re-polled from global memory), reduces, stores the output and
// writes the outgoing line with one 16-byte store.
// ---------------------------------------------------------------------------
// 8192 elements: one tile per default step (32 KiB of binary32 payload), 2 stages;
// 1920-, 3840- and 4096-element tiles were measured slower at every size
constexpr int kLLTileElems = 8192;
constexpr int kLLTileLineBytes = kLLTileElems * 4 / 8 * 16;  // binary32 payload: 8 bytes per 16-byte line
constexpr int kLLBulkMinChunk = 1024;  // chunks at least this long take the bulk form (measured: 1-8192)

template <int PROTO>
__host__ __device__ constexpr int bulk_tile_elems() { return PROTO == kLL ? kLLTileElems : kL8TileElems; }
// Elements of a row's tile. LL128 sizes a tile by its 64 line groups: rows
// that move bf16 finals and read no input (recvCopySend, recv) put twice the
// elements of a binary32 row in them, so that their tiles carry as many
// lines as the reduce-scatter rows' and the per-tile costs (pacing, stage
// hand-off) are spread over as many bytes. Every other row: kL8TileElems.
template <typename T, int PROTO>
__device__ __forceinline__ int bulk_row_tile(int prim) {
  if (PROTO == kLL128 && sizeof(T) == 2 && (prim == kRecvCopySend || prim == kRecv)) return 2 * kL8TileElems;
  return bulk_tile_elems<PROTO>();
}
template <int PROTO>
__host__ __device__ constexpr int bulk_line_bytes() { return PROTO == kLL ? kLLTileLineBytes : kL8TileGroups * 512; }
template <typename T, int PROTO>
__host__ __device__ constexpr int bulk_stage_bytes() {
  return bulk_line_bytes<PROTO>() + bulk_tile_elems<PROTO>() * (int)sizeof(T);
}
template <typename T, int PROTO>
__host__ __device__ constexpr int bulk_max_stages() {
  return kL8SmemBudget / bulk_stage_bytes<T, PROTO>() < kL8MaxStages ? kL8SmemBudget / bulk_stage_bytes<T, PROTO>()
                                                                     : kL8MaxStages;
}

// KU input elements of the tile from element e, widened to binary32, zeros
// past kv: one shared-memory load when all of them are staged.
template <typename T, int KU>
__device__ __forceinline__ void ll_input_unit(const char* s_in, const T* g_tile, int e, int kv, int covered,
                                              float (&x)[4]) {
  if (kv == KU && e + KU <= covered) {
    if constexpr (sizeof(T) == 4) {
      const float2 w = *reinterpret_cast<const float2*>(s_in + e * 4);
      x[0] = w.x; x[1] = w.y; x[2] = 0.f; x[3] = 0.f;
    } else if constexpr (KU == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(s_in + e * 2);
      x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(s_in + e * 2);
      x[0] = bf16lo(w); x[1] = bf16hi(w); x[2] = 0.f; x[3] = 0.f;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; j++) x[j] = j < kv && j < KU ? l8_input<T>(s_in, g_tile, e + j, covered) : 0.f;
}

template <typename T, int PRIM>
__device__ __forceinline__ void ll_bulk_tile(const RingArgs& a, const char* s_lines, const char* s_in,
                                             const T* g_in_tile, T* g_out_tile, const char* g_rlines, char* g_slines,
                                             int ne, int covered, uint32_t rflag, uint32_t sflag,
                                             volatile int* sh_abort, uint64_t info, int ct, int nct) {
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kHasRecv = PRIM != kSend && PRIM != kCopySend;
  constexpr bool kHasSend = PRIM != kRecv && PRIM != kRecvReduceCopy;
  constexpr bool kIn = PRIM == kSend || kRecvPartial || PRIM == kCopySend;
  constexpr bool kFinalOfSum = PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kOut = kFinalOfSum || PRIM == kRecvCopySend || PRIM == kRecv || PRIM == kCopySend;
  constexpr int EBR = kRecvPartial ? 4 : (int)sizeof(T);                                 // received element bytes
  constexpr int EBS = (PRIM == kSend || PRIM == kRecvReduceSend) ? 4 : (int)sizeof(T);  // sent element bytes
  constexpr int KU = 8 / (kHasSend ? EBS : EBR);  // elements of a unit
  constexpr int LPU = kHasRecv ? KU * EBR / 8 : 0;  // received lines of a unit (2 for bf16's owner row)
  const int nunits = (ne + KU - 1) / KU;
  for (int u = ct; u < nunits; u += nct) {
    const int e = u * KU;
    const int kv = ne - e < KU ? ne - e : KU;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t fin0 = 0u, fin1 = 0u;  // the unit's final values as raw bits (8 bytes)
    if (kHasRecv) {
#pragma unroll
      for (int l = 0; l < (LPU > 0 ? LPU : 1); l++) {
        // a unit's second line (bf16's owner row) exists only if it holds elements
        if (l > 0 && e + l * (8 / EBR) >= ne) break;
        const int li = u * LPU + l;
        uint4 rl = *reinterpret_cast<const uint4*>(s_lines + li * 16);
        if (!ll_ready(rl, rflag)) {
          rl = ld_line_v4(g_rlines + li * 16);
          if (!ll_ready(rl, rflag) && !ll_poll(a, g_rlines + li * 16, rflag, rl, sh_abort, info)) return;
        }
        if (kRecvPartial) {
          v[2 * l] = __uint_as_float(rl.x);
          v[2 * l + 1] = __uint_as_float(rl.z);
        } else {
          fin0 = rl.x;
          fin1 = rl.z;
        }
      }
    }
    float x[4];
    if (kIn) ll_input_unit<T, KU>(s_in, g_in_tile, e, kv, covered, x);
    if (PRIM == kSend) {
#pragma unroll
      for (int j = 0; j < 4; j++) v[j] = x[j];
    } else if (kRecvPartial) {
#pragma unroll
      for (int j = 0; j < 4; j++) v[j] = j < kv ? __fadd_rn(v[j], x[j]) : 0.f;
    }
    if (kFinalOfSum || PRIM == kCopySend) {
      const float* f = PRIM == kCopySend ? x : v;  // a bf16 input widened and rounded back is itself
      if constexpr (sizeof(T) == 4) {
        fin0 = __float_as_uint(f[0]);
        fin1 = __float_as_uint(f[1]);
      } else {
        fin0 = round_bf16_pair(f[0], f[1]);
        fin1 = round_bf16_pair(f[2], f[3]);
      }
    }
    if (kOut && kv > 0) store_out_n<T>(g_out_tile + e, kv, KU, make_uint4(fin0, fin1, 0u, 0u));
    if (kHasSend) {
      uint4 line;
      if (EBS == 4 && (PRIM == kSend || PRIM == kRecvReduceSend))
        line = make_uint4(__float_as_uint(v[0]), sflag, __float_as_uint(v[1]), sflag);
      else
        line = make_uint4(fin0, sflag, fin1, sflag);
      st_line_v4(g_slines + u * 16, line);
    }
  }
}

// Same values and lines as ll_bulk_tile for a whole tile (kLLTileElems
// elements, all input staged): every unit is full, so the threads need no
// element bounds and each thread's units are known at compile time.
template <typename T, int PRIM>
__device__ __forceinline__ void ll_bulk_tile_full(const RingArgs& a, const char* s_lines, const char* s_in,
                                                  T* g_out_tile, const char* g_rlines, char* g_slines, uint32_t rflag,
                                                  uint32_t sflag, volatile int* sh_abort, uint64_t info, int ct) {
  constexpr bool kRecvPartial = PRIM == kRecvReduceSend || PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kHasRecv = PRIM != kSend && PRIM != kCopySend;
  constexpr bool kHasSend = PRIM != kRecv && PRIM != kRecvReduceCopy;
  constexpr bool kIn = PRIM == kSend || kRecvPartial || PRIM == kCopySend;
  constexpr bool kFinalOfSum = PRIM == kRecvReduceCopySend || PRIM == kRecvReduceCopy;
  constexpr bool kOut = kFinalOfSum || PRIM == kRecvCopySend || PRIM == kRecv || PRIM == kCopySend;
  constexpr int EBR = kRecvPartial ? 4 : (int)sizeof(T);
  constexpr int EBS = (PRIM == kSend || PRIM == kRecvReduceSend) ? 4 : (int)sizeof(T);
  constexpr int KU = 8 / (kHasSend ? EBS : EBR);
  constexpr int LPU = kHasRecv ? KU * EBR / 8 : 0;
  constexpr int NU = kLLTileElems / KU;  // units of a whole tile
  constexpr int RPT = (NU + kL8WorkThreads - 1) / kL8WorkThreads;
  static_assert(kLLTileElems % KU == 0, "whole units");
#pragma unroll
  for (int r = 0; r < RPT; r++) {
    const int u = ct + r * kL8WorkThreads;
    if (NU % kL8WorkThreads != 0 && u >= NU) break;
    const int e = u * KU;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t fin0 = 0u, fin1 = 0u;
    if constexpr (kHasRecv) {
#pragma unroll
      for (int l = 0; l < LPU; l++) {
        const int li = u * LPU + l;
        uint4 rl = *reinterpret_cast<const uint4*>(s_lines + li * 16);
        if (!ll_ready(rl, rflag)) {
          rl = ld_line_v4(g_rlines + li * 16);
          if (!ll_ready(rl, rflag) && !ll_poll(a, g_rlines + li * 16, rflag, rl, sh_abort, info)) return;
        }
        if constexpr (kRecvPartial) {
          v[2 * l] = __uint_as_float(rl.x);
          v[2 * l + 1] = __uint_as_float(rl.z);
        } else {
          fin0 = rl.x;
          fin1 = rl.z;
        }
      }
    }
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (kIn) {
      if constexpr (sizeof(T) == 4) {
        const float2 w = *reinterpret_cast<const float2*>(s_in + e * 4);
        x[0] = w.x;
        x[1] = w.y;
      } else if constexpr (KU == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(s_in + e * 2);
        x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(s_in + e * 2);
        x[0] = bf16lo(w);
        x[1] = bf16hi(w);
      }
    }
    if constexpr (PRIM == kSend) {
#pragma unroll
      for (int j = 0; j < 4; j++) v[j] = x[j];
    } else if constexpr (kRecvPartial) {
#pragma unroll
      for (int j = 0; j < KU; j++) v[j] = __fadd_rn(v[j], x[j]);
    }
    if constexpr (kFinalOfSum || PRIM == kCopySend) {
      const float* f = PRIM == kCopySend ? x : v;
      if constexpr (sizeof(T) == 4) {
        fin0 = __float_as_uint(f[0]);
        fin1 = __float_as_uint(f[1]);
      } else {
        fin0 = round_bf16_pair(f[0], f[1]);
        fin1 = round_bf16_pair(f[2], f[3]);
      }
    }
    if constexpr (kOut) {
      if constexpr (KU * sizeof(T) == 8) st_v2(g_out_tile + e, make_uint2(fin0, fin1));
      else *reinterpret_cast<uint32_t*>(g_out_tile + e) = fin0;
    }
    if constexpr (kHasSend) {
      uint4 line;
      if constexpr (EBS == 4 && (PRIM == kSend || PRIM == kRecvReduceSend))
        line = make_uint4(__float_as_uint(v[0]), sflag, __float_as_uint(v[1]), sflag);
      else
        line = make_uint4(fin0, sflag, fin1, sflag);
      st_line_v4(g_slines + u * 16, line);
    }
  }
}

template <typename T>
__device__ __forceinline__ void ll_bulk_tile_any(int prim, const RingArgs& a, const char* s_lines, const char* s_in,
                                                 const T* g_in_tile, T* g_out_tile, const char* g_rlines,
                                                 char* g_slines, int ne, int covered, uint32_t rflag,
                                                 uint32_t sflag, volatile int* sh_abort, uint64_t info, int ct,
                                                 int nct) {
  if (ne == kLLTileElems && covered == ne && nct == kL8WorkThreads) {
#define RAR_LL_FULL(P) ll_bulk_tile_full<T, P>(a, s_lines, s_in, g_out_tile, g_rlines, g_slines, rflag, sflag, sh_abort, info, ct)
    switch (prim) {
      case kSend: RAR_LL_FULL(kSend); return;
      case kRecvReduceSend: RAR_LL_FULL(kRecvReduceSend); return;
      case kRecvReduceCopySend: RAR_LL_FULL(kRecvReduceCopySend); return;
      case kRecvCopySend: RAR_LL_FULL(kRecvCopySend); return;
      case kRecvReduceCopy: RAR_LL_FULL(kRecvReduceCopy); return;
      case kCopySend: RAR_LL_FULL(kCopySend); return;
      default: RAR_LL_FULL(kRecv); return;
    }
#undef RAR_LL_FULL
  }
  switch (prim) {
    case kSend:
      ll_bulk_tile<T, kSend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered, rflag, sflag,
                             sh_abort, info, ct, nct);
      break;
    case kRecvReduceSend:
      ll_bulk_tile<T, kRecvReduceSend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered,
                                       rflag, sflag, sh_abort, info, ct, nct);
      break;
    case kRecvReduceCopySend:
      ll_bulk_tile<T, kRecvReduceCopySend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered,
                                           rflag, sflag, sh_abort, info, ct, nct);
      break;
    case kRecvCopySend:
      ll_bulk_tile<T, kRecvCopySend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered,
                                     rflag, sflag, sh_abort, info, ct, nct);
      break;
    case kRecvReduceCopy:
      ll_bulk_tile<T, kRecvReduceCopy>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered,
                                       rflag, sflag, sh_abort, info, ct, nct);
      break;
    case kCopySend:
      ll_bulk_tile<T, kCopySend>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered, rflag,
                                 sflag, sh_abort, info, ct, nct);
      break;
    default:
      ll_bulk_tile<T, kRecv>(a, s_lines, s_in, g_in_tile, g_out_tile, g_rlines, g_slines, ne, covered, rflag, sflag,
                             sh_abort, info, ct, nct);
      break;
  }
}

// Pacing of the bulk form: wait (bounded) until the last of the received
// lines, `bytes` of them starting at `lines`, carries the flag of step
// `rstep`. Only a heuristic for when to copy: every line is still
// accepted by its own flag. False if the wait gave up.
template <int PROTO>
__device__ __forceinline__ bool tile_last_line_wait(const RingArgs& a, const char* lines, uint32_t bytes,
                                                    uint64_t rstep, uint64_t info) {
  Spin sp;
  if constexpr (PROTO == kLL128) {
    const uint64_t* p = reinterpret_cast<const uint64_t*>(lines + bytes - 8);  // flag word of the group's line 3
    while (ld_relaxed_u64(p) != rstep + 1) {
      if (sp.poll(a, info, rstep + 1)) return false;
    }
  } else {
    const char* p = lines + bytes - 16;
    const uint32_t flag = ll_flag(a, rstep);
    while (!ll_ready(ld_line_v4(p), flag)) {
      if (sp.poll(a, info, flag)) return false;
    }
  }
  return true;
}

constexpr int kPaceBatch = 8;
// LL128 pacing over several tiles at once, in two parts: the flags of the
// last lines of tiles k .. k + kPaceBatch - 1 of a step are loaded first
// (issued before the loader's wait for a free stage, so that their round trip
// overlaps that wait: f32 on 12 channels +2.5 %), then l8_tiles_ready_f
// returns the last tile of the prefix that carries the flag, after waiting
// (bounded) for tile k itself when none does yet, or -1 if the wait gave up.
__device__ __forceinline__ void l8_flags_issue(const char* rslot, int k, int ntiles, int64_t nelem, int te, int eb,
                                               uint64_t (&f)[kPaceBatch]) {
#pragma unroll
  for (int j = 0; j < kPaceBatch; j++) {
    f[j] = 0;
    if (k + j < ntiles) {
      const int64_t g_end = div_up(imin((int64_t)(k + j + 1) * te, nelem) * eb, 480);
      f[j] = ld_relaxed_u64(reinterpret_cast<const uint64_t*>(rslot + g_end * 512 - 8));
    }
  }
}
__device__ __forceinline__ int l8_tiles_ready_f(const RingArgs& a, const char* rslot, int k, int ntiles, int64_t nelem,
                                                int te, int eb, uint64_t rstep, uint64_t info,
                                                const uint64_t (&f)[kPaceBatch]) {
  int n = 0;
#pragma unroll
  for (int j = 0; j < kPaceBatch; j++)
    if (n == j && k + j < ntiles && f[j] == rstep + 1) n = j + 1;
  if (n > 0) return k + n - 1;
  const int64_t g_end = div_up(imin((int64_t)(k + 1) * te, nelem) * eb, 480);
  return tile_last_line_wait<kLL128>(a, rslot, (uint32_t)(g_end * 512), rstep, info) ? k : -1;
}

// The split point of LL128's bulk form: whole 4-line groups of bf16 payload
// (240 elements, two groups of binary32), so that both parts start on a group
// boundary whichever type a row's lines carry, and a row's received and sent
// lines of one part cover the same elements.
constexpr int kSplitAlign = 240;
constexpr int64_t kL8SplitMinChunk = kL8TileElems;  // first-loop chunks that split (one whole tile)

template <typename T, int PROTO, int SPLIT>
__global__ void __launch_bounds__(kL8Threads, 1) ring_line_bulk_kernel(const __grid_constant__ RingArgs a,
                                                                        int nstages) {
  extern __shared__ __align__(128) char smem[];
  __shared__ uint64_t bar_ready[kL8Depth], bar_done[kL8Depth], bar_free[kL8Depth];
  __shared__ uint64_t bar_full[kL8MaxStages], bar_empty[kL8MaxStages], bar_fin;
  __shared__ volatile int sh_abort;
  __shared__ int sh_chan;
  __shared__ uint64_t sh_base_send, sh_base_recv;
  constexpr int P = 16 / (int)sizeof(T);
  constexpr int LB = bulk_line_bytes<PROTO>();
  constexpr int SB = bulk_stage_bytes<T, PROTO>();

  const Geometry& g = a.geo;
  if (threadIdx.x == 0) sh_chan = -1;
  __syncthreads();
  // blocks [0, N * C) move the first half of every step (all of it unless
  // the launch splits), blocks [N * C, 2 * N * C) the second half
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
  uint64_t* r_head = conn_head(cr, half);  // this block's releases
  uint64_t* s_tail = conn_tail(cs, half);
  char* fifo_send = fifo_at(a, dense, e_send);
  const char* fifo_recv = fifo_at(a, dense, e_recv);
  if (threadIdx.x == 0) {
    const uint64_t tail0 = ld_relaxed_u64(s_tail), head0 = ld_relaxed_u64(r_head);  // with the header
    sh_abort = entry_check(a) ? 0 : 1;
    for (int d = 0; d < kL8Depth; d++) {
      mbar_init(&bar_ready[d], 1);
      mbar_init(&bar_done[d], kL8WorkThreads);
      mbar_init(&bar_free[d], 1);
    }
    for (int st = 0; st < kL8MaxStages; st++) {
      mbar_init(&bar_full[st], 1);
      mbar_init(&bar_empty[st], kL8Warps);
    }
    mbar_init(&bar_fin, kL8Warps);
    // Both counters belong to this block (this half) and equal the previous
    // call's final step.
    sh_base_send = tail0;
    sh_base_recv = head0;
    reinterpret_cast<uint8_t*>(a.ws + kTraceOffset)[blockIdx.x] = (uint8_t)sh_chan;
  }
  __syncthreads();
  if (sh_abort) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t base_send = sh_base_send, base_recv = sh_base_recv;
  const uint64_t info = ((uint64_t)blockIdx.x << 32);
  const int64_t step_bytes = g.step_bytes;
  const T* in = reinterpret_cast<const T*>(a.send[rank]);
  T* out = reinterpret_cast<T*>(a.recv[rank]);
  SliceCursor c;
  cursor_begin(g, dense, ring_idx, c);

  if (warp == 0) {
    if (lane != 0) return;
    // ---- waiter ----
    uint64_t rstep = base_recv, sstep = base_send, head_seen = 0;
    uint64_t seen2[2] = {0, 0};  // split launches: both halves' heads
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kL8Depth, use = i / kL8Depth;
      if (use > 0 && !mbar_wait(a, &bar_free[d], (use - 1) & 1u, info | (1u << 24) | i)) sh_abort = 1;
      if (!sh_abort && !slice_in_bounds(a, dense, c, rstep, sstep, info | i)) sh_abort = 1;
      if (!sh_abort && row_sends(c.prim)) {
        bool ok;
        if constexpr (SPLIT == 1)
          ok = wait_credit(a, &cs->head, base_send, sstep, &head_seen, info | (3u << 24) | i);
        else
          ok = wait_credit_both(a, cs, base_send, sstep, seen2, info | (3u << 24) | i);
        if (!ok) sh_abort = 1;
      }
      mbar_arrive(&bar_ready[d]);
      if (sh_abort) break;
      if (row_recvs(c.prim)) rstep++;
      if (row_sends(c.prim)) sstep++;
    }
  } else if (warp == 1) {
    if (lane != 0) return;
    // ---- loader ----
    const uint64_t pol = l2_policy_evict_first();
    uint64_t rstep = base_recv;
    uint32_t gt = 0;
    uint64_t sstep_l = base_send;  // for the debug bounds check only
    for (uint32_t i = 0; c.valid && !sh_abort; i++, cursor_next(g, c)) {
      const uint32_t d = i % kL8Depth, use = i / kL8Depth;
      if (!slice_in_bounds(a, dense, c, rstep, sstep_l, info | i)) {
        sh_abort = 1;
        break;
      }
      if (row_sends(c.prim)) sstep_l++;
      if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (6u << 24) | i) || sh_abort) {
        sh_abort = 1;
        break;
      }
      const int prim = c.prim;
      int64_t in_off, out_off;
      slice_offsets(a, dense, c, &in_off, &out_off);
      const bool has_in = row_reads_input(prim);
      const bool has_rcv = row_recvs(prim);
      const int eb = row_recvs_partial(prim) ? 4 : (int)sizeof(T);
      const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
      const int te = bulk_row_tile<T, PROTO>(prim);
      int64_t lo, hi;
      split_range(c.nelem, half, SPLIT, kSplitAlign, &lo, &hi);
      const int64_t nh = hi - lo;
      const char* rslot_h = rslot + (PROTO == kLL128 ? lo * eb / 480 * 512 : lo * eb / 8 * 16);  // the half's lines
      const int ntiles = (int)div_up(nh, te);
      int ready_upto = -1;  // LL128: the last tile of this step known to carry its flags
      for (int k = 0; k < ntiles; k++) {
        const uint32_t st = gt % nstages, su = gt / nstages;
        uint64_t pf[kPaceBatch];
        if constexpr (PROTO == kLL128) {
          if (has_rcv && k > ready_upto) l8_flags_issue(rslot_h, k, ntiles, nh, te, eb, pf);
        }
        if (su > 0 && !mbar_wait(a, &bar_empty[st], (su - 1) & 1u, info | (7u << 24) | i)) {
          sh_abort = 1;
          break;
        }
        const int64_t e0 = lo + (int64_t)k * te;
        const int ne = (int)imin(te, hi - e0);
        const int covered = ne / P * P;
        const uint32_t b_in = has_in ? (uint32_t)covered * (uint32_t)sizeof(T) : 0u;
        // the tile's received lines: whole 4-line groups (LL128) or 16-byte lines (LL)
        const uint32_t b_rcv = !has_rcv ? 0u
                               : PROTO == kLL128 ? (uint32_t)div_up((int64_t)ne * eb, 480) * 512u
                                                 : (uint32_t)div_up((int64_t)ne * eb, 8) * 16u;
        const int64_t r_off = PROTO == kLL128 ? e0 * eb / 480 * 512 : e0 * eb / 8 * 16;
        char* s_lines = smem + (int64_t)st * SB;
        char* s_in = s_lines + LB;
        // the input (which does not depend on the sender) is copied ahead of
        // the pacing wait and the lines
        const bool pace = b_rcv && (PROTO == kLL128 ? k > ready_upto : k == 0);
        if (b_in) {
          mbar_expect_tx(&bar_full[st], b_in);
          tma_load_1d(s_in, in + in_off + e0, b_in, &bar_full[st], pol);
        }
        // pacing: LL128 copies a tile's lines once the tile's last line
        // carries the flag, so that they move while the sender still writes
        // the step's later tiles (the flags of several tiles are read
        // together); LL waits once for the step's last line (measured:
        // per-tile waits made LL slower)
        bool paced = true;
        if constexpr (PROTO == kLL128) {
          if (pace) {
            ready_upto = l8_tiles_ready_f(a, rslot_h, k, ntiles, nh, te, eb, rstep, info | (9u << 24) | i, pf);
            paced = ready_upto >= 0;
            if (paced) fence_proxy_async_global();
          }
        } else if (pace) {
          paced = tile_last_line_wait<PROTO>(a, rslot_h, (uint32_t)div_up(nh * eb, 8) * 16u, rstep,
                                             info | (9u << 24) | i);
          if (paced) fence_proxy_async_global();
        }
        if (!paced) {
          mbar_arrive_expect_tx(&bar_full[st], 0u);  // the phase completes once the input landed
          gt++;
          sh_abort = 1;
          break;
        }
        mbar_arrive_expect_tx(&bar_full[st], b_rcv);
        if (b_rcv) tma_load_1d(s_lines, rslot + r_off, b_rcv, &bar_full[st], pol);
        gt++;
      }
      if (has_rcv) rstep++;
    }
    for (uint32_t st = 0; st < (uint32_t)nstages && st < gt; st++) {
      const uint32_t last = (gt - 1 - st) / nstages * nstages + st;
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
    bool aborted = false;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kL8Depth, use = i / kL8Depth;
      if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (4u << 24) | i) ||
          !mbar_wait(a, &bar_done[d], use & 1u, info | (4u << 24) | i) || sh_abort) {
        sh_abort = 1;
        aborted = true;
        break;
      }
      if (row_recvs(c.prim)) {
        rstep++;
        if (a.fault != kFaultDropHead) st_relaxed_u64(r_head, rstep);  // every line of this half was read
      }
      if (row_sends(c.prim)) sstep++;
      mbar_arrive(&bar_free[d]);
    }
    if (!aborted) {
      // the sender's step count carries over to the next call; without a
      // split, the second half's counters follow
      st_relaxed_u64(s_tail, sstep);
      if (SPLIT == 1) {
        st_relaxed_u64(&cs->tail_h1, sstep);
        st_relaxed_u64(&cr->head_h1, rstep);
      }
    }
  } else {
    // ---- workers ----
    const int w = warp - 3;
    uint64_t rstep = base_recv, sstep = base_send;
    uint32_t gt = 0, fin_uses = 0;
    for (uint32_t i = 0; c.valid; i++, cursor_next(g, c)) {
      const uint32_t d = i % kL8Depth, use = i / kL8Depth;
      if (!mbar_wait(a, &bar_ready[d], use & 1u, info | (5u << 24) | i) || sh_abort) {
        mbar_arrive(&bar_done[d]);
        sh_abort = 1;
        break;
      }
      const int eb_r = row_recvs_partial(c.prim) ? 4 : (int)sizeof(T);
      const int eb_s = row_sends_partial(c.prim) ? 4 : (int)sizeof(T);
      const char* rslot = fifo_recv + (int64_t)(rstep % kSteps) * step_bytes;
      char* sslot = fifo_send + (int64_t)(sstep % kSteps) * step_bytes;
      int64_t in_off, out_off;
      slice_offsets(a, dense, c, &in_off, &out_off);
      const int te = bulk_row_tile<T, PROTO>(c.prim);
      int64_t lo, hi;
      split_range(c.nelem, half, SPLIT, kSplitAlign, &lo, &hi);
      const int ntiles = (int)div_up(hi - lo, te);
      bool stop = false;
      for (int k = 0; k < ntiles; k++, gt++) {
        const uint32_t st = gt % nstages, su = gt / nstages;
        if (!mbar_wait(a, &bar_full[st], su & 1u, info | (5u << 24) | i)) sh_abort = 1;
        const int64_t e0 = lo + (int64_t)k * te;
        const int ne = (int)imin(te, hi - e0);
        char* s_lines = smem + (int64_t)st * SB;
        char* s_in = s_lines + LB;
        if constexpr (PROTO == kLL128) {
          // the tile runs on every path so that the workers' barrier counts match
          l8_tile_any<T>(c.prim, a, s_lines, s_in, in + in_off + e0, out + out_off + e0,
                         rslot + e0 * eb_r / 480 * 512, sslot + e0 * eb_s / 480 * 512, sh_abort ? 0 : ne, te,
                         ne / P * P, rstep + 1, sstep + 1, &sh_abort, info | (10u << 24) | i, w, &bar_fin,
                         &fin_uses);
        } else {
          ll_bulk_tile_any<T>(c.prim, a, s_lines, s_in, in + in_off + e0, out + out_off + e0,
                              rslot + e0 * eb_r / 8 * 16, sslot + e0 * eb_s / 8 * 16, sh_abort ? 0 : ne, ne / P * P,
                              ll_flag(a, rstep), ll_flag(a, sstep), &sh_abort, info | (10u << 24) | i,
                              threadIdx.x - 96, kL8WorkThreads);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_empty[st]);
        if (sh_abort) {
          stop = true;
          break;
        }
      }
      mbar_arrive(&bar_done[d]);
      if (stop) break;
      if (row_recvs(c.prim)) rstep++;
      if (row_sends(c.prim)) sstep++;
    }
  }
}

template <int PROTO, int SPLIT>
cudaError_t launch_bulk(const RingArgs& a, cudaLaunchConfig_t cfg, bool f32, int device, int* threads_out) {
  const int nstages = f32 ? bulk_max_stages<float, PROTO>() : bulk_max_stages<uint16_t, PROTO>();
  const int smem = nstages * (f32 ? bulk_stage_bytes<float, PROTO>() : bulk_stage_bytes<uint16_t, PROTO>());
  static_assert(PROTO == kLL128 || SPLIT == 1, "only LL128's bulk form splits");
  const int key = PROTO == kLL ? (f32 ? kSetupBulkLLF32 : kSetupBulkLLBf16)
                  : SPLIT == 1 ? (f32 ? kSetupBulkLL128F32 : kSetupBulkLL128Bf16)
                               : (f32 ? kSetupBulkLL128F32Split : kSetupBulkLL128Bf16Split);  // per device
  if (!setup_done(device, key)) {
    const cudaError_t e = f32 ? cudaFuncSetAttribute(ring_line_bulk_kernel<float, PROTO, SPLIT>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                              : cudaFuncSetAttribute(ring_line_bulk_kernel<uint16_t, PROTO, SPLIT>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mark_setup_done(device, key);
  }
  cfg.gridDim = dim3(cfg.gridDim.x * (unsigned)SPLIT);
  cfg.blockDim = dim3(kL8Threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  if (threads_out) *threads_out = kL8Threads;
  if (trace_on())
    std::fprintf(stderr,
                 "rar trace:   kernel ring_line_bulk_kernel<%s, %s> grid %u threads %d stages %d smem %d split %d\n",
                 f32 ? "float" : "bf16", PROTO == kLL ? "LL" : "LL128", cfg.gridDim.x, kL8Threads, nstages, smem,
                 SPLIT);
  return f32 ? cudaLaunchKernelEx(&cfg, ring_line_bulk_kernel<float, PROTO, SPLIT>, a, nstages)
             : cudaLaunchKernelEx(&cfg, ring_line_bulk_kernel<uint16_t, PROTO, SPLIT>, a, nstages);
}

void trace_polling(const char* proto, bool f32, int grid, int threads) {
  if (trace_on())
    std::fprintf(stderr, "rar trace:   kernel ring_line_kernel<%s, %s, %d> grid %d threads %d\n", f32 ? "float" : "bf16",
                 proto, threads, grid, threads);
}

cudaError_t launch_ring_line(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out) {
  // Polling forms: 256 threads when a step is a few passes of the block at
  // most (fewer threads per barrier: lower latency), 1024 threads for large
  // LL steps (more warps in flight).
  constexpr int kThreadsSmall = 256;
  constexpr int kThreadsLarge = 1024;
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
  const int64_t first_chunk = loop_chunk_count(a.geo, imin(a.geo.per_channel, a.geo.count));
  int device = 0, sms = 0;
  const cudaError_t e = current_device_sms(&device, &sms);
  if (e != cudaSuccess) return e;
  // Steps per barrier group of the polling form: a group of kSteps / 2 steps
  // when every step's lines fit one pass of the block (no pacing wait is
  // needed) and flags do not wrap; else one step.
  auto epoch_for = [&](int threads) -> int {
    if (a.ll_flag_max != 0) return 1;
    const bool one_pass = a.geo.proto == kLL
                              ? div_up(first_chunk, f32 ? LLUnit<float>::kElems : LLUnit<uint16_t>::kElems) <= threads
                              : div_up(first_chunk * 4, 480) <= threads / 32;
    return one_pass ? kSteps / 2 : 1;
  };
  // LL: the bulk form from 1024-element chunks (not in the flag-wrap test
  // mode, whose slot cleanup lives in the polling form); below that the
  // polling form has the lower latency
  // (one block per (rank, channel): LL's steps are one tile each, paced
  // once per step, and a split over two blocks measured no faster)
  if (a.geo.proto == kLL && first_chunk >= kLLBulkMinChunk && grid <= sms && a.ll_flag_max == 0)
    return launch_bulk<kLL, 1>(a, cfg, f32, device, threads_out);
  if (a.geo.proto == kLL) {
    // 256 threads when a step is one pass of them; larger steps take 1024
    // threads, so that a step is still one pass (barrier groups: at 256 KiB
    // per rank on 12 channels, 27.5 against 34.4 us with 256 threads in two
    // passes and a barrier per step). The flag-wrap test mode, which keeps a
    // barrier per step, stays at 256 threads up to 8 passes.
    const bool small = div_up(first_chunk, f32 ? LLUnit<float>::kElems : LLUnit<uint16_t>::kElems) <=
                       (a.ll_flag_max ? 8 : 1) * kThreadsSmall;
    if (small) {
      cfg.blockDim = dim3(kThreadsSmall);
      if (threads_out) *threads_out = kThreadsSmall;
      trace_polling("LL", f32, grid, kThreadsSmall);
      const int ep = epoch_for(kThreadsSmall);
      return f32 ? cudaLaunchKernelEx(&cfg, ring_line_kernel<float, kLL, kThreadsSmall>, a, ep)
                 : cudaLaunchKernelEx(&cfg, ring_line_kernel<uint16_t, kLL, kThreadsSmall>, a, ep);
    }
    cfg.blockDim = dim3(kThreadsLarge);
    if (threads_out) *threads_out = kThreadsLarge;
    trace_polling("LL", f32, grid, kThreadsLarge);
    const int ep = epoch_for(kThreadsLarge);
    return f32 ? cudaLaunchKernelEx(&cfg, ring_line_kernel<float, kLL, kThreadsLarge>, a, ep)
               : cudaLaunchKernelEx(&cfg, ring_line_kernel<uint16_t, kLL, kThreadsLarge>, a, ep);
  }
  // LL128: the bulk form from 960-element chunks, the polling form (lowest
  // latency) for smaller messages.
  // Two blocks per (rank, channel), each a fixed half of every step, when
  // twice the grid still fits one block per SM and a step holds at least one
  // whole tile: the bulk form is bound by its blocks' instruction issue, and
  // a mask of few channels leaves SMs idle; smaller steps are bound by their
  // hand-off chain, which a split only lengthens (measured: 512 KiB per rank
  // on 4 ranks and 12 channels, 2732-element chunks, 19.0 against 17.5 us).
  // Not in the flag-wrap test mode, whose slot cleanup lives in the polling
  // form anyway.
  if (first_chunk >= kL8BulkMinChunk && grid <= sms) {
    if (2 * grid <= sms && first_chunk >= kL8SplitMinChunk && a.ll_flag_max == 0)
      return launch_bulk<kLL128, 2>(a, cfg, f32, device, threads_out);
    return launch_bulk<kLL128, 1>(a, cfg, f32, device, threads_out);
  }
  cfg.blockDim = dim3(kThreadsSmall);
  if (threads_out) *threads_out = kThreadsSmall;
  trace_polling("LL128", f32, grid, kThreadsSmall);
  const int ep = epoch_for(kThreadsSmall);
  return f32 ? cudaLaunchKernelEx(&cfg, ring_line_kernel<float, kLL128, kThreadsSmall>, a, ep)
             : cudaLaunchKernelEx(&cfg, ring_line_kernel<uint16_t, kLL128, kThreadsSmall>, a, ep);
}

}  // namespace rar
