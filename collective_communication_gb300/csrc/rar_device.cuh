// rar_device.cuh -- workspace layout, kernel arguments and device helpers
// (inline PTX for loads/stores with explicit scope and caching, fences,
// mbarriers, bounded waits) of librar.so. sm_103a only.
//
// Pages cited (by title, then section):
//   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
//   [NOTES] "NCCL" notes (cishoon.github.io), section "Memory Model（acquire / release
//           真正在做什么）"
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "rar_geometry.h"

namespace rar {

// ---------------------------------------------------------------------------
// Workspace layout (device memory owned by the caller).
//   [0, 4096)            WsHeader, then a per-block channel-id trace at 2048
//   [4096, 4096 + R)     one ConnCounters record (256 B) per connection
//   [4096 + R, ...)      one FIFO of buff_size bytes per connection
// R = align_up(C * N * 256, 4096). Connection (dense channel n, ring edge e)
// is number n * N + e; edge e runs from ring index e to ring index e + 1.
// ---------------------------------------------------------------------------
constexpr uint32_t kMagic = 0x31524152u;  // "RAR1"
constexpr int64_t kHeaderBytes = 4096;
constexpr int64_t kTraceOffset = 2048;
constexpr int64_t kConnBytes = 256;

struct WsHeader {
  uint32_t magic;
  uint32_t status;     // first device failure (rar_status), 0 if none
  uint32_t abort;      // raised by the first block that gives up
  int32_t nranks;
  uint64_t mask;
  int32_t proto;
  int32_t pad0;
  int64_t buff_size;   // resolved (never 0)
  uint64_t err_info;   // where the first failure happened: block << 32 | role << 24 | slice
  uint64_t err_step;   // the step it waited for
};

// head: steps the receiver has released; tail: steps the sender has published
// (Simple), or the sender's step count at the end of a call (LL, LL128). Each
// on its own 128-byte line so that the two sides' polls do not share a line.
// head_h1 / tail_h1: the same counters of the second half of a connection
// whose steps a split LL128 launch moves with two blocks per (rank, channel)
// (each half a fixed element range of every step). Every call ends with both
// halves' counters at the call's final step, so that any form may follow.
struct ConnCounters {
  uint64_t head;
  uint64_t pad0[7];
  uint64_t head_h1;
  uint64_t pad0b[7];
  uint64_t tail;
  uint64_t pad1[7];
  uint64_t tail_h1;
  uint64_t pad1b[7];
};
static_assert(sizeof(ConnCounters) == 256, "one connection's counters fill kConnBytes");

inline int64_t conn_region_bytes(int nranks, int nchan) {
  return align_up((int64_t)nranks * nchan * kConnBytes, 4096);
}
inline int64_t workspace_bytes_for(int nranks, int nchan, int64_t buff_size) {
  return kHeaderBytes + conn_region_bytes(nranks, nchan) + (int64_t)nranks * nchan * buff_size;
}

// Status codes written by kernels (mirror rar_status).
constexpr uint32_t kErrWorkspace = 4;
constexpr uint32_t kErrTimeout = 7;
constexpr uint32_t kErrAbort = 8;
constexpr uint32_t kErrBounds = 9;  // debug builds: a slice outside its buffers

// Fault injection for tests (a wait that nothing satisfies; the wait runs out
// of time and the launch ends with RAR_ERR_TIMEOUT).
constexpr int kFaultNone = 0;
constexpr int kFaultDropHead = 1;   // receivers never publish their head
constexpr int kFaultDropAck = 2;    // staged one-shot: ranks never acknowledge their reads
constexpr int kFaultBoundsView = 3;  // debug builds: the bounds check sees each slice one buffer further on

struct RingArgs {
  const void* send[kMaxRanks];
  void* recv[kMaxRanks];
  uint8_t ring_index[kMaxChannels * kMaxRanks];  // [dense channel * kMaxRanks + user rank] -> ring index
  uint8_t ring_rank[kMaxChannels * kMaxRanks];   // [dense channel * kMaxRanks + ring index] -> user rank
  int direct;                  // Simple: all-gather hops write the next rank's output directly
  Geometry geo;
  uint64_t mask;
  char* ws;                    // workspace base
  int64_t conn_offset;         // byte offset of the ConnCounters array
  int64_t fifo_offset;         // byte offset of the FIFO array
  uint64_t timeout_ns;
  int fault;
  uint32_t ll_flag_max;        // LL: 0 = flag step + 1 (32 bits); else flags wrap at this power of two
};

// ---------------------------------------------------------------------------
// PTX wrappers. Scope .gpu: every party (the N ranks' blocks) is an SM of the
// same GPU, so the system scope the pages need for peers across NVLink, the
// CPU proxy or a NIC is not required here ([NOTES] Memory Model).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Returns the old value.
__device__ __forceinline__ uint64_t atom_add_acq_rel_u64(uint64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// FIFO payload reads: cached in L2 only, so a slot reused NCCL_STEPS steps
// later is never served from a stale L1 line.
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_cg_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_cg_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// User input reads: streamed, not kept in L1. (Not the non-coherent path:
// an in-place call writes the same buffer later in the kernel.)
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
// Line polls and line stores of LL / LL128: one 16-byte access each, so a
// line's data and its flag(s) travel together ([C23] "LL：Data 与 Flag 同 Line").
// Strong relaxed accesses at GPU scope: every reader and writer is an SM of
// this GPU, so they meet in L2. (The system-scope volatile form the page
// uses, for peers across NVLink, serialises a thread's polls.)
__device__ __forceinline__ uint4 ld_line_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_line_v4(void* p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// mbarrier in shared memory (one phase bit per completed round).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Arrive once and add `bytes` to the transaction count the current phase
// waits for (the bytes of the bulk copies that complete on this barrier).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Add `bytes` to the current phase's transaction count without arriving:
// the phase cannot complete before the pending arrival, so copies issued
// under this count may land before the rest of the phase is set up.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// TMA bulk copy global -> shared (no tensor map; 16-byte aligned addresses,
// size a multiple of 16). Completion is counted on `bar` in bytes. The L2
// policy marks the source lines evict-first: each is read exactly once.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_1d(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
// Store with an L2 eviction policy (user output: evict-first, so that the
// streaming output does not push FIFO lines out of L2).
__device__ __forceinline__ void st_v4_policy(void* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}
// Orders this thread's earlier generic-proxy accesses (here: the acquire of a
// FIFO tail) before its later async-proxy (bulk copy) accesses of global memory.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Failure reporting and bounded waits ([C23] checkAbort in the wait loops).
// ---------------------------------------------------------------------------
__device__ __forceinline__ WsHeader* header_of(const RingArgs& a) { return (WsHeader*)a.ws; }

// First failure wins the status word; every failure raises the abort flag.
// H: any workspace header with status, abort, err_info and err_step.
template <typename H>
__device__ __forceinline__ void report_failure(H* h, uint32_t code, uint64_t info, uint64_t step) {
  if (atomicCAS(&h->status, 0u, code) == 0u) {
    h->err_info = info;
    h->err_step = step;
  }
  atomicExch(&h->abort, 1u);
}

// Iteration backstop, in case the timer misbehaves: far above what any
// legitimate wait needs, still a finite wait.
constexpr uint32_t kMaxSpinChecks = 1u << 24;

// State of one bounded wait. poll() returns true when the wait must give up
// (time limit passed, or another block raised the abort flag).
struct Spin {
  uint64_t t0;
  uint32_t iters;
  uint32_t checks;
  __device__ __forceinline__ Spin() : t0(0), iters(0), checks(0) {}
  template <typename H>
  __device__ __forceinline__ bool poll_h(H* h, uint64_t timeout_ns, uint64_t info, uint64_t step) {
    if ((++iters & 63u) != 0u) return false;
    if (ld_relaxed_u32(&h->abort) != 0u) return true;
    uint64_t now = global_timer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > timeout_ns || ++checks > kMaxSpinChecks) {
      report_failure(h, kErrTimeout, info, step);
      return true;
    }
    return false;
  }
  __device__ __forceinline__ bool poll(const RingArgs& a, uint64_t info, uint64_t step) {
    return poll_h(header_of(a), a.timeout_ns, info, step);
  }
};

// Bounded wait on an mbarrier phase. Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(const RingArgs& a, uint64_t* bar, uint32_t parity, uint64_t info) {
  Spin sp;
  while (!mbar_try_wait(bar, parity)) {
    if (sp.poll(a, info, parity)) return false;
  }
  return true;
}

__device__ __forceinline__ ConnCounters* conn_at(const RingArgs& a, int dense_channel, int edge) {
  return (ConnCounters*)(a.ws + a.conn_offset) + ((int64_t)dense_channel * a.geo.nranks + edge);
}
// Elements [lo, hi) of a slice of ne elements that part `half` of a launch
// split over two blocks per (rank, channel) moves: the first part rounded up
// to a multiple of `align` elements (the protocol's layout unit), the rest to
// the second. Both ends of a connection compute the same split from the same
// slice.
__device__ __forceinline__ void split_range(int64_t ne, int half, int nsplit, int64_t align, int64_t* lo,
                                            int64_t* hi) {
  if (nsplit == 1) {
    *lo = 0;
    *hi = ne;
    return;
  }
  const int64_t m = imin(ne, div_up(ne, 2 * align) * align);
  *lo = half ? m : 0;
  *hi = half ? ne : m;
}

// The head / tail of half `half` of a connection (0 unless a launch splits it).
__device__ __forceinline__ uint64_t* conn_head(ConnCounters* c, int half) { return half ? &c->head_h1 : &c->head; }
__device__ __forceinline__ uint64_t* conn_tail(ConnCounters* c, int half) { return half ? &c->tail_h1 : &c->tail; }
__device__ __forceinline__ char* fifo_at(const RingArgs& a, int dense_channel, int edge) {
  return a.ws + a.fifo_offset + ((int64_t)dense_channel * a.geo.nranks + edge) * a.geo.buff_size;
}

// Block -> (rank, dense channel, channel id). Block b serves rank b / C and
// the (b % C)-th set bit of the mask; each thread below 64 tests one bit the
// way the page's kernel entry does: n = popcount(mask & ((1 << id) - 1))
// ([C23] "Kernel 如何把 Block 映射到 Channel").
__device__ __forceinline__ void map_block_index(const RingArgs& a, int b, int* rank, int* dense, int* sh_chan_id) {
  int C = a.geo.nchan;
  *rank = b / C;
  *dense = b % C;
  int tid = threadIdx.x;
  if (tid < kMaxChannels && ((a.mask >> tid) & 1ull)) {
    uint64_t below = tid == 0 ? 0ull : (a.mask & ((1ull << tid) - 1ull));
    if (__popcll(below) == *dense) *sh_chan_id = tid;
  }
}
__device__ __forceinline__ void map_block(const RingArgs& a, int* rank, int* dense, int* sh_chan_id) {
  map_block_index(a, (int)blockIdx.x, rank, dense, sh_chan_id);
}

// Ring index of user rank `rank` on dense channel `dense`, and the user rank
// that follows it on that channel's ring.
__device__ __forceinline__ int ring_index_of(const RingArgs& a, int dense, int rank) {
  return a.ring_index[dense * kMaxRanks + rank];
}
// LL flag of a step ([C23] "LL：Data 与 Flag 同 Line"): step + 1, or, in the
// wrap test mode, step + 1 modulo the power of two ll_flag_max.
__device__ __forceinline__ uint32_t ll_flag(const RingArgs& a, uint64_t step) {
  return a.ll_flag_max ? (uint32_t)((step + 1) & (uint64_t)(a.ll_flag_max - 1)) : (uint32_t)(step + 1);
}
// Wrap mode: on the last NCCL_STEPS steps of every half flag period (once per
// slot every ll_flag_max / 2 steps) the sender rewrites every line of its slot
// past its slice with the current flag, so that no line is ever older than
// half a period when it is read and none can carry a later step's flag.
__device__ __forceinline__ bool ll_cleanup_step(const RingArgs& a, uint64_t step) {
  if (a.ll_flag_max == 0) return false;
  const uint64_t half = a.ll_flag_max / 2;
  return step % half >= half - kSteps;
}

__device__ __forceinline__ int rank_at_index(const RingArgs& a, int dense, int ring_idx) {
  return a.ring_rank[dense * kMaxRanks + ring_idx];
}
__device__ __forceinline__ int next_rank_of(const RingArgs& a, int dense, int ring_idx) {
  return rank_at_index(a, dense, (ring_idx + 1) % a.geo.nranks);
}

// Element offsets of the current slice in the rank's input and output.
// AllReduce: the same offset in both. The halves: a ReduceScatter input and
// an AllGather output hold nranks blocks of geo.count elements, block b
// belonging to user rank b; a slice of the chunk with ring index c lies in
// the block of the user rank at ring index c. The other buffer holds one block.
__device__ __forceinline__ void slice_offsets(const RingArgs& a, int dense, const SliceCursor& c, int64_t* in_off,
                                              int64_t* out_off) {
  const Geometry& g = a.geo;
  if (g.kind == kAllReduce) {
    *in_off = *out_off = c.offset;
    return;
  }
  const int64_t blk = (int64_t)rank_at_index(a, dense, c.chunk) * g.count;
  *in_off = c.offset + (g.kind == kReduceScatter ? blk : 0);
  *out_off = c.offset + (g.kind == kAllGather ? blk : 0);
}

// Debug builds (-DRAR_DEBUG): before a slice is used, check that its user
// ranges lie inside the rank's buffers and that its bytes on the wire (a
// binary32 bound for both types) fit its FIFO slot(s); a violation records
// RAR_ERR_BOUNDS with the block, slice and offset in the workspace header and
// the caller aborts instead of touching memory. Release builds: always true.
__device__ __forceinline__ bool slice_in_bounds(const RingArgs& a, int dense, const SliceCursor& c, uint64_t rstep,
                                                uint64_t sstep, uint64_t info) {
#ifdef RAR_DEBUG
  const Geometry& g = a.geo;
  int64_t in_off, out_off;
  slice_offsets(a, dense, c, &in_off, &out_off);
  const int64_t N = g.nranks;
  const int64_t in_len = g.kind == kReduceScatter ? N * g.count : g.count;
  const int64_t out_len = g.kind == kAllGather ? N * g.count : g.count;
  if (a.fault == kFaultBoundsView) {  // the check's own view only; the slice's accesses keep their offsets
    in_off += in_len;
    out_off += out_len;
  }
  // an empty slice touches no user memory (its offset may lie past the end)
  bool ok = c.nelem >= 0 && (c.nelem == 0 || (in_off >= 0 && out_off >= 0 && in_off + c.nelem <= in_len &&
                                              out_off + c.nelem <= out_len));
  const int64_t b4 = c.nelem * 4;
  if (g.proto == kSimple) {
    ok = ok && b4 <= (int64_t)g.sps * g.step_bytes;
    if (row_recvs(c.prim)) ok = ok && (int64_t)(rstep % kSteps) + g.sps <= kSteps;
    if (row_sends(c.prim)) ok = ok && (int64_t)(sstep % kSteps) + g.sps <= kSteps;
  } else if (g.proto == kLL) {
    ok = ok && div_up(b4, 8) * 16 <= g.step_bytes;
  } else {
    ok = ok && div_up(b4, 480) * 512 <= g.step_bytes;
  }
  if (!ok) report_failure(header_of(a), kErrBounds, info | (11u << 24), (uint64_t)c.offset);
  return ok;
#else
  (void)a; (void)dense; (void)c; (void)rstep; (void)sstep; (void)info;
  return true;
#endif
}

// Entry check shared by the ring kernels (thread 0): the workspace must be
// initialised for this configuration and not aborted. Returns true to run.
__device__ __forceinline__ bool entry_check(const RingArgs& a) {
  WsHeader* h = header_of(a);
  if (h->magic != kMagic || h->nranks != a.geo.nranks || h->mask != a.mask || h->proto != a.geo.proto ||
      h->buff_size != a.geo.buff_size) {
    report_failure(h, kErrWorkspace, (uint64_t)blockIdx.x << 32, 0);
    return false;
  }
  if (ld_relaxed_u32(&h->abort) != 0u) {
    atomicCAS(&h->status, 0u, kErrAbort);
    return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t round_up_steps(uint64_t v) {
  return (v + kSteps - 1) / kSteps * kSteps;
}

// LL128: lane geometry inside a group of 4 lines (512 bytes) moved by one
// warp access of 16 bytes per lane. Lane l holds bytes [16l, 16l+16) of the
// group: line l/8, 64-bit words 2(l%8) and 2(l%8)+1. Word 15 of each line is
// its flag, held by the lane with l%8 == 7 next to payload word 14. The 480
// payload bytes of a group are spread over the lanes so that every user
// access stays aligned: lanes with l%8 < 7 carry group payload bytes
// 16*(7*(l/8) + l%8) .. +16, the four flag lanes carry bytes 448 + 8*(l/8) .. +8.
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


__device__ __forceinline__ uint64_t ll128_flag_of(const uint4& v) { return ((uint64_t)v.w << 32) | v.z; }

// bf16 helpers: widening is exact (a bf16 is the upper half of a binary32);
// narrowing is round-to-nearest-even by the hardware conversion.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace rar
