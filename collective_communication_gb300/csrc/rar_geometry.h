// rar_geometry.h -- chunk geometry of the ring AllReduce, shared by the host
// launcher (argument checks, workspace sizing, rar_describe_geometry) and the
// device kernels of librar.so.
//
// Pages cited (by title, then section):
//   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
//   [C12] "NCCL 专家课程 12：Ring AllReduce 逐步推导、真实 Ring 与 Channel 并行"
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define RAR_HD __host__ __device__ __forceinline__
#else
#define RAR_HD inline
#endif

namespace rar {

constexpr int kSteps = 8;  // NCCL_STEPS: slots per connector FIFO ([C23] "Simple 的 Credit 与 Step")
constexpr int kMaxRanks = 32;
constexpr int kMaxChannels = 64;

enum Proto : int { kLL = 0, kLL128 = 1, kSimple = 2 };
enum Dtype : int { kF32 = 0, kBF16 = 1 };

// Collectives built on the ring: AllReduce, and its two halves on their own
// ([C12] "Ring AllReduce 不只是“绕一圈”": AllReduce = ReduceScatter + AllGather).
enum Kind : int { kAllReduce = 0, kReduceScatter = 1, kAllGather = 2 };

// Rows of the per-rank schedule ([C12] "源码步骤一" .. "源码步骤五").
enum Prim : int {
  kSend = 0,                // raw local input -> next
  kRecvReduceSend = 1,      // prev + local -> next
  kRecvReduceCopySend = 2,  // prev + local -> output and next (owner row)
  kRecvCopySend = 3,        // prev -> output and next
  kRecv = 4,                // prev -> output
  kRecvReduceCopy = 5,      // prev + local -> output (ReduceScatter's owner row)
  kCopySend = 6             // local -> output and next (AllGather's first row)
};

RAR_HD int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }
RAR_HD int64_t align_up(int64_t a, int64_t b) { return div_up(a, b) * b; }
RAR_HD int64_t imin(int64_t a, int64_t b) { return a < b ? a : b; }
RAR_HD int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }

RAR_HD int rows_per_loop(int kind, int n) { return kind == kAllReduce ? 2 * n - 1 : n; }

RAR_HD int prim_of_row(int kind, int n, int s) {
  if (kind == kReduceScatter) return s == 0 ? kSend : s < n - 1 ? kRecvReduceSend : kRecvReduceCopy;
  if (kind == kAllGather) return s == 0 ? kCopySend : s < n - 1 ? kRecvCopySend : kRecv;
  return s == 0 ? kSend
       : s < n - 1 ? kRecvReduceSend
       : s == n - 1 ? kRecvReduceCopySend
       : s < 2 * n - 2 ? kRecvCopySend
       : kRecv;
}
// Chunk (ring index of its owner) of row s for ring index i: every formula of
// the page, (i + n - j) with its own loop counter j, is (i - s - 1) mod n for
// the row number s. The AllGather half starts at the rank's own chunk, so its
// row s carries chunk (i - s) mod n.
RAR_HD int chunk_of_row(int kind, int n, int i, int s) {
  const int d = kind == kAllGather ? s : s + 1;
  return ((i - d) % n + 2 * n) % n;
}
RAR_HD bool row_recvs(int prim) { return prim != kSend && prim != kCopySend; }
RAR_HD bool row_sends(int prim) { return prim != kRecv && prim != kRecvReduceCopy; }
RAR_HD bool row_reads_input(int prim) {
  return prim == kSend || prim == kRecvReduceSend || prim == kRecvReduceCopySend || prim == kRecvReduceCopy ||
         prim == kCopySend;
}
// Partial sums (binary32) cross the reduce-scatter hops; final values (T)
// cross the all-gather hops.
RAR_HD bool row_sends_partial(int prim) { return prim == kSend || prim == kRecvReduceSend; }
RAR_HD bool row_recvs_partial(int prim) {
  return prim == kRecvReduceSend || prim == kRecvReduceCopySend || prim == kRecvReduceCopy;
}

RAR_HD int64_t default_buff_size(int proto) {
  return proto == kSimple ? (int64_t)4 << 20   // "default" row of [C23] "Simple Buffer Sweep"
       : proto == kLL ? (int64_t)512 << 10     // one LL step = buffer/8, half of it payload
       : (int64_t)4915200;                     // 8 steps x 4800 lines x 128 B: 576000 B chunks
}

// Resolved per-call geometry.
struct Geometry {
  int kind;             // kAllReduce, kReduceScatter or kAllGather
  int proto, dtype, nranks, nchan;
  int64_t count;        // elements per rank (AllReduce) or per rank block (ReduceScatter, AllGather)
  int elem_bytes;       // sizeof(T)
  int align_elems;      // 16 / sizeof(T)
  int64_t buff_size;    // FIFO bytes per connection
  int64_t step_bytes;   // buff_size / kSteps
  int64_t chunk_elems;  // elements of a full chunk
  int64_t step_elems;   // binary32 elements per Simple step
  int sps;              // steps per slice
  int spc;              // slices per chunk
  int64_t per_channel;  // elements per channel (the last ones may get fewer)
};

// Returns 0 on success, 1 for a bad argument.
RAR_HD int make_geometry(Geometry* g, int proto, int dtype, int nranks, uint64_t mask, int64_t count,
                         int64_t buff_size, int chunk_steps, int kind = kAllReduce) {
  if (kind != kAllReduce && kind != kReduceScatter && kind != kAllGather) return 1;
  g->kind = kind;
  if (nranks < 2 || nranks > kMaxRanks) return 1;
  if (dtype != kF32 && dtype != kBF16) return 1;
  if (proto != kLL && proto != kLL128 && proto != kSimple) return 1;
  if (mask == 0 || count < 0) return 1;
  if (chunk_steps != 1 && chunk_steps != 2 && chunk_steps != 4) return 1;
  int c = 0;
  for (int b = 0; b < kMaxChannels; b++) c += (int)((mask >> b) & 1u);
  g->proto = proto;
  g->dtype = dtype;
  g->nranks = nranks;
  g->nchan = c;
  g->count = count;
  g->elem_bytes = dtype == kF32 ? 4 : 2;
  g->align_elems = 16 / g->elem_bytes;
  if (buff_size == 0) buff_size = default_buff_size(proto);
  g->buff_size = buff_size;
  g->step_bytes = buff_size / kSteps;
  g->step_elems = g->step_bytes / 4;
  // A chunk is sized in 4-byte elements for both types, so that the binary32
  // partial sums of bf16 fit the same FIFO slots; for f32 this is exactly
  // buffer / NCCL_STEPS * chunkSteps / sizeof(T) ([C23] "Buffer 到 Chunk 的实测公式").
  if (proto == kSimple) {
    if (buff_size % 4096 != 0 || buff_size < 4096) return 1;
    g->sps = chunk_steps >= 2 ? chunk_steps / 2 : 1;  // StepPerSlice
    g->spc = chunk_steps / g->sps;                    // SlicePerChunk
    g->chunk_elems = g->step_bytes * chunk_steps / 4;
  } else if (proto == kLL) {
    if (buff_size % 4096 != 0 || buff_size < 4096) return 1;
    g->sps = 1;
    g->spc = 1;
    g->chunk_elems = g->step_bytes / 2 / 4;  // 8 payload bytes per 16-byte line
  } else {
    // whole groups of 4 lines (one warp access) per step
    if (buff_size % 4096 != 0 || buff_size < 4096) return 1;
    g->sps = 1;
    g->spc = 1;
    g->chunk_elems = (g->step_bytes / 128) * 120 / 4 / 32 * 32;  // 120 payload bytes per line
  }
  if (g->chunk_elems < 32) return 1;
  g->per_channel = align_up(div_up(count, c), g->align_elems);
  return 0;
}

RAR_HD void channel_range(const Geometry& g, int n, int64_t* grid_offset, int64_t* channel_count) {
  int64_t off = g.per_channel * n;
  *grid_offset = off;
  *channel_count = off >= g.count ? 0 : imin(g.per_channel, g.count - off);
}

// Elements of the channel range one loop covers: AllReduce splits a loop into
// nranks chunks of the rank's buffer; the two halves move one chunk of every
// rank block per loop (the block is the chunk).
RAR_HD int64_t loop_count(const Geometry& g) {
  return g.kind == kAllReduce ? (int64_t)g.nranks * g.chunk_elems : g.chunk_elems;
}

// Chunk size of a loop whose remainder is rem: full chunks, except in the
// short last loop, split over the ranks and aligned up to 16/sizeof(T)
// ([C12] "runRing 的数据切分"); for the halves, the remainder itself.
RAR_HD int64_t loop_chunk_count(const Geometry& g, int64_t rem) {
  if (g.kind != kAllReduce) return imin(rem, g.chunk_elems);
  return rem < loop_count(g) ? align_up(div_up(rem, g.nranks), g.align_elems) : g.chunk_elems;
}

RAR_HD int64_t chunk_nelem(int64_t chunk_count, int64_t rem, int c) {
  int64_t off = chunk_count * c;
  return rem > off ? imin(chunk_count, rem - off) : 0;
}

// [C23] "Slice Size": the larger of an even split in units of 16 elements and
// 1/32 of a slice's FIFO capacity, aligned to 16 elements (so every slice
// starts on a 16-byte boundary for both element types). LL and LL128: one
// slice per chunk.
RAR_HD int64_t slice_size(const Geometry& g, int64_t nelem) {
  if (g.proto != kSimple) return nelem;
  return align_up(imax(div_up(nelem, 16 * (int64_t)g.spc) * 16, g.step_elems * g.sps / 32), 16);
}

// Walks one block's slices in order: loops x rows x slices per chunk. Every
// role of a block walks the same sequence.
struct SliceCursor {
  int64_t grid_offset, channel_count;
  int64_t elem_offset, rem, chunk_count;
  int s, k;
  int ring_index;
  bool valid;
  // current slice
  int prim;
  int chunk;       // ring index of the chunk's owner
  int64_t offset;  // AllReduce: user element offset; halves: offset inside the rank block
  int64_t nelem;
};

RAR_HD void cursor_fill(const Geometry& g, SliceCursor& c) {
  int n = g.nranks;
  int ch = chunk_of_row(g.kind, n, c.ring_index, c.s);
  int64_t ne, base;
  if (g.kind == kAllReduce) {
    ne = chunk_nelem(c.chunk_count, c.rem, ch);
    base = c.grid_offset + c.elem_offset + c.chunk_count * ch;
  } else {
    ne = c.chunk_count;  // the same range of every rank block
    base = c.grid_offset + c.elem_offset;
  }
  int64_t ss = slice_size(g, ne);
  int64_t so = ss * c.k;
  c.prim = prim_of_row(g.kind, n, c.s);
  c.chunk = ch;
  c.offset = base + so;
  c.nelem = ne > so ? imin(ss, ne - so) : 0;  // empty slices still wait and post
}

RAR_HD void cursor_begin(const Geometry& g, int dense_channel, int ring_index, SliceCursor& c) {
  channel_range(g, dense_channel, &c.grid_offset, &c.channel_count);
  c.ring_index = ring_index;
  c.elem_offset = 0;
  c.s = 0;
  c.k = 0;
  c.valid = c.channel_count > 0;
  if (c.valid) {
    c.rem = c.channel_count;
    c.chunk_count = loop_chunk_count(g, c.rem);
    cursor_fill(g, c);
  }
}

RAR_HD void cursor_next(const Geometry& g, SliceCursor& c) {
  if (++c.k < g.spc) { cursor_fill(g, c); return; }
  c.k = 0;
  if (++c.s < rows_per_loop(g.kind, g.nranks)) { cursor_fill(g, c); return; }
  c.s = 0;
  c.elem_offset += loop_count(g);
  if (c.elem_offset >= c.channel_count) { c.valid = false; return; }
  c.rem = c.channel_count - c.elem_offset;
  c.chunk_count = loop_chunk_count(g, c.rem);
  cursor_fill(g, c);
}

}  // namespace rar
