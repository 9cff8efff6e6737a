/*
 * oracle.c -- plain, slow CPU oracle for the ring AllReduce over N virtual
 * ranks and for the one-shot AllReduce variant.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The product (the CUDA
 * library and its Python binding) never loads, links or calls it, and the two
 * share no source, header, table or constant generator.
 *
 * Pages cited (by title, then section):
 *   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
 *         (blog.cptz.space)
 *   [C12] "NCCL 专家课程 12：Ring AllReduce 逐步推导、真实 Ring 与 Channel 并行"
 *         (blog.cptz.space)
 *   [OS89] "perf(osar): all-reduce 5커널 → 3커널 (가드·웨이트 프롤로그 융합) - #89"
 *         (github.com/choiceoh/stkernel pull request 89)
 *
 * Where the pages leave a step open, the reading taken is named in a comment
 * ("Reading: ...") at the place it is used.
 *
 * Arithmetic: every floating-point addition is one IEEE-754 binary32 add in
 * round-to-nearest-even. Build with -ffp-contract=off and without fast-math so
 * that the C compiler keeps exactly these operations.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Constants and codes (exported values are mirrored in oracle.py).    */
/* ------------------------------------------------------------------ */

/* NCCL_STEPS: slots in every connector FIFO ring ([C23] "Simple 的 Credit 与 Step"). */
#define NSTEPS 8
#define MAXCH 64
#define MAXR 64

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_LL = 0, ORC_LL128 = 1, ORC_SIMPLE = 2 };
enum {
  ORC_OK = 0,
  ORC_EARG = 1,      /* bad argument */
  ORC_ERING = 2,     /* ring_order is not a ring over all ranks */
  ORC_EDEADLOCK = 3, /* simulation stopped with ranks still waiting */
  ORC_ECHECK = 4,    /* an internal invariant of the simulation failed */
  ORC_ENOMEM = 5
};
/* Primitive of each row of the per-rank ring schedule ([C12] "源码步骤一..五"). */
enum {
  ORC_SEND = 0,
  ORC_RECV_REDUCE_SEND = 1,
  ORC_RECV_REDUCE_COPY_SEND = 2,
  ORC_RECV_COPY_SEND = 3,
  ORC_RECV = 4,
  /* the halves as collectives of their own ([C12] "源码步骤三": the owner row is
   * the last recv+reduce of ReduceScatter fused with the first send of AllGather) */
  ORC_RECV_REDUCE_COPY = 5, /* ReduceScatter's last row: recv + reduce, write the output */
  ORC_COPY_SEND = 6         /* AllGather's first row: copy the input to the output and send it */
};
/* Collective run on the ring ([C12] "Ring AllReduce 不只是“绕一圈”"). */
enum { ORC_ALLREDUCE = 0, ORC_REDUCE_SCATTER = 1, ORC_ALL_GATHER = 2 };

static size_t div_up(size_t a, size_t b) { return (a + b - 1) / b; }
static size_t align_up(size_t a, size_t b) { return div_up(a, b) * b; }
static size_t min_sz(size_t a, size_t b) { return a < b ? a : b; }
static size_t max_sz(size_t a, size_t b) { return a > b ? a : b; }

/* ------------------------------------------------------------------ */
/* bf16 <-> f32                                                        */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of a binary32; widening is exact. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round binary32 to bf16, round-to-nearest-even. Method: add 0x7FFF plus the
 * lowest kept bit to the 32-bit pattern and truncate (the usual integer form
 * of RNE; a carry out of the mantissa bumps the exponent, which is also what
 * RNE does at a binade edge and at overflow to infinity). NaN stays NaN and is
 * made quiet. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void orc_bf16_round(const float* x, uint16_t* y, size_t n) {
  for (size_t i = 0; i < n; i++) y[i] = f32_to_bf16_rne(x[i]);
}

/* Value of element e of rank buffer `buf`, widened to binary32. */
static float load_as_f32(const void* buf, int dtype, size_t e) {
  if (dtype == ORC_F32) return ((const float*)buf)[e];
  return bf16_to_f32(((const uint16_t*)buf)[e]);
}

/* Store a binary32 value as element e of `buf`; bf16 is rounded once here. */
static void store_from_f32(void* buf, int dtype, size_t e, float v) {
  if (dtype == ORC_F32)
    ((float*)buf)[e] = v;
  else
    ((uint16_t*)buf)[e] = f32_to_bf16_rne(v);
}

/* ------------------------------------------------------------------ */
/* Ring setup ([C12] "ring index 如何计算", "Graph 如何变成完整 ring") */
/* ------------------------------------------------------------------ */

/*
 * ring_order[i] is the user rank at place i of the ring; the ring's `next`
 * direction runs from place i to place i+1 (mod n).
 *
 * First the ring is checked the way the page's ring builder does: start at
 * rank 0, follow `next` n times recording each rank; every rank must be seen
 * once and the walk must come back to rank 0 ("ring does not loop back").
 *
 * Then, for every user rank r (the setupChannel computation):
 *   ixZero = place of rank 0, ixRank = place of rank r,
 *   index[r] = (ixRank - ixZero + n) % n          (ring index / position)
 *   user_ranks[r*n + i] = ring_order[(i + ixRank) % n]   (ring seen from r)
 *   prev[r] = rank before r, next[r] = rank after r.
 * Any output pointer may be NULL.
 */
int orc_ring_setup(int n, const int* ring_order, int* index, int* prev, int* next,
                   int* user_ranks) {
  if (n < 1 || n > MAXR || ring_order == NULL) return ORC_EARG;
  int nxt[MAXR], seen[MAXR], place[MAXR];
  for (int r = 0; r < n; r++) { nxt[r] = -1; seen[r] = 0; place[r] = -1; }
  for (int i = 0; i < n; i++) {
    int r = ring_order[i];
    if (r < 0 || r >= n) return ORC_ERING;
    if (place[r] != -1) return ORC_ERING; /* rank listed twice */
    place[r] = i;
    nxt[r] = ring_order[(i + 1) % n];
  }
  int cur = 0;
  for (int i = 0; i < n; i++) {
    if (cur < 0 || seen[cur]) return ORC_ERING;
    seen[cur] = 1;
    cur = nxt[cur];
  }
  if (cur != 0) return ORC_ERING; /* ring does not loop back */
  int ixZero = place[0];
  for (int r = 0; r < n; r++) {
    int ixRank = place[r];
    if (index) index[r] = (ixRank - ixZero + n) % n;
    if (prev) prev[r] = ring_order[(ixRank - 1 + n) % n];
    if (next) next[r] = ring_order[(ixRank + 1) % n];
    if (user_ranks)
      for (int i = 0; i < n; i++) user_ranks[r * n + i] = ring_order[(i + ixRank) % n];
  }
  return ORC_OK;
}

/* rank_at[j] = user rank whose ring index is j. */
static int rank_at_index(int n, const int* ring_order, int* rank_at) {
  int index[MAXR];
  int st = orc_ring_setup(n, ring_order, index, NULL, NULL, NULL);
  if (st != ORC_OK) return st;
  for (int r = 0; r < n; r++) rank_at[index[r]] = r;
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Ring schedule ([C12] "源码步骤一..五", "rank0 的完整操作序列")       */
/* ------------------------------------------------------------------ */

/*
 * For the rank with ring index i, its 2n-1 schedule rows s = 0..2n-2:
 *   s = 0          send                        chunk (i-1) mod n
 *   s = 1..n-2     recvReduceSend              chunk (i-s-1) mod n
 *   s = n-1        recvReduceCopySend (owner)  chunk i
 *   s = n..2n-3    recvCopySend                chunk (i-s-1) mod n
 *   s = 2n-2       recv                        chunk (i+1) mod n
 * Each formula on the page is of the form (i + n - j) with its own loop
 * counter j; every one of them equals (i - s - 1) mod n for the row number s.
 */
static int prim_of_row(int n, int s) {
  if (s == 0) return ORC_SEND;
  if (s < n - 1) return ORC_RECV_REDUCE_SEND;
  if (s == n - 1) return ORC_RECV_REDUCE_COPY_SEND;
  if (s < 2 * n - 2) return ORC_RECV_COPY_SEND;
  return ORC_RECV;
}

static int chunk_of_row(int n, int i, int s) { return ((i - s - 1) % n + 2 * n) % n; }

/*
 * The halves on their own, n rows each (reading: the AllReduce rows split at
 * the owner row, whose recv+reduce ends ReduceScatter and whose send starts
 * AllGather, [C12] "源码步骤三"):
 *   ReduceScatter  s = 0 send, s = 1..n-2 recvReduceSend, s = n-1 recvReduceCopy;
 *                  chunk (i-s-1) mod n, as in the AllReduce rows 0..n-1.
 *   AllGather      s = 0 copySend, s = 1..n-2 recvCopySend, s = n-1 recv;
 *                  chunk (i-s) mod n, as in the AllReduce rows n-1..2n-2.
 */
static int rows_of_kind(int kind, int n) { return kind == ORC_ALLREDUCE ? 2 * n - 1 : n; }

static int prim_of_kind_row(int kind, int n, int s) {
  if (kind == ORC_REDUCE_SCATTER)
    return s == 0 ? ORC_SEND : s < n - 1 ? ORC_RECV_REDUCE_SEND : ORC_RECV_REDUCE_COPY;
  if (kind == ORC_ALL_GATHER) return s == 0 ? ORC_COPY_SEND : s < n - 1 ? ORC_RECV_COPY_SEND : ORC_RECV;
  return prim_of_row(n, s);
}

static int chunk_of_kind_row(int kind, int n, int i, int s) {
  if (kind == ORC_ALL_GATHER) return ((i - s) % n + 2 * n) % n;
  return chunk_of_row(n, i, s);
}

int orc_schedule(int n, int ring_index, int* prim, int* chunk) {
  if (n < 1 || ring_index < 0 || ring_index >= n) return ORC_EARG;
  if (n == 1) return ORC_EARG;
  for (int s = 0; s < 2 * n - 1; s++) {
    prim[s] = prim_of_row(n, s);
    chunk[s] = chunk_of_row(n, ring_index, s);
  }
  return ORC_OK;
}

/* Rows of one collective kind; returns the row count, or -1. */
int orc_schedule_kind(int kind, int n, int ring_index, int* prim, int* chunk) {
  if (kind < ORC_ALLREDUCE || kind > ORC_ALL_GATHER) return -1;
  if (n < 2 || ring_index < 0 || ring_index >= n) return -1;
  int rows = rows_of_kind(kind, n);
  for (int s = 0; s < rows; s++) {
    prim[s] = prim_of_kind_row(kind, n, s);
    chunk[s] = chunk_of_kind_row(kind, n, ring_index, s);
  }
  return rows;
}

/* ------------------------------------------------------------------ */
/* Geometry ([C23] "Kernel 如何把 Block 映射到 Channel",                */
/*           "Buffer 到 Chunk 的实测公式", "Slice Size", "LL", "LL128"; */
/*           [C12] "runRing 的数据切分", "多 channel 如何并行")          */
/* ------------------------------------------------------------------ */

typedef struct {
  int kind;             /* ORC_ALLREDUCE, ORC_REDUCE_SCATTER or ORC_ALL_GATHER */
  int proto, dtype, nranks, nchan;
  int chan_id[MAXCH];   /* dense channel n -> channel id */
  size_t count;         /* elements per rank (AllReduce) or per rank block (the halves) */
  size_t elem_bytes;    /* sizeof(T) */
  size_t align_elems;   /* 16 / sizeof(T) */
  size_t step_bytes;    /* FIFO bytes per step (line bytes for LL and LL128) */
  size_t chunk_elems;   /* elements of a full chunk */
  size_t step_elems;    /* binary32 payload elements per Simple step */
  int sps;              /* steps per slice */
  int spc;              /* slices per chunk */
  size_t per_channel;   /* elements given to each channel (last may get fewer) */
} geom_t;

size_t orc_default_buffsize(int proto) {
  switch (proto) {
    case ORC_SIMPLE: return (size_t)4 << 20; /* 4 MiB: the "default" row of the buffer sweep */
    case ORC_LL: return (size_t)512 << 10;   /* 8 lines x 512 threads x 8 steps x 16 B */
    case ORC_LL128: return (size_t)4915200;  /* 8 steps x 4800 lines x 128 B: a 576000 B chunk */
    default: return 0;
  }
}

/*
 * Reading (block -> channel): block n of a launch serves the n-th set bit of
 * channelMask; that bit's id is the channel id. The page computes, for every
 * set bit id, n = popcount(mask & ((1<<id)-1)).
 */
int orc_mask_channels(uint64_t mask, int* chan_id) {
  int c = 0;
  for (int id = 0; id < MAXCH; id++) {
    if (!((mask >> id) & 1u)) continue;
    uint64_t below = (id == 0) ? 0 : (mask & ((((uint64_t)1) << id) - 1));
    int n = __builtin_popcountll(below);
    chan_id[n] = id;
    c++;
  }
  return c;
}

static int geom_init(geom_t* g, int proto, int dtype, int nranks, uint64_t mask,
                     size_t count, size_t buffSize, int chunkSteps) {
  memset(g, 0, sizeof *g);
  if (nranks < 2 || nranks > MAXR) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  if (mask == 0) return ORC_EARG;
  g->proto = proto;
  g->dtype = dtype;
  g->nranks = nranks;
  g->count = count;
  g->elem_bytes = dtype == ORC_F32 ? 4 : 2;
  g->align_elems = 16 / g->elem_bytes;
  g->nchan = orc_mask_channels(mask, g->chan_id);
  if (buffSize == 0) buffSize = orc_default_buffsize(proto);
  /* Reading (bf16 on the ring): partial sums cross the reduce-scatter hops
   * as binary32, so a chunk is sized in 4-byte elements for both types;
   * for f32 this is exactly buffer/NCCL_STEPS*chunkSteps/sizeof(T). */
  if (proto == ORC_SIMPLE) {
    if (buffSize % 4096 != 0) return ORC_EARG;
    if (chunkSteps != 1 && chunkSteps != 2 && chunkSteps != 4 && chunkSteps != 8)
      return ORC_EARG;
    g->step_bytes = buffSize / NSTEPS;
    /* Reading (slices): StepPerSlice = chunkSteps/2, SlicePerChunk = 2
     * (1 and 1 when chunkSteps is 1). */
    g->sps = chunkSteps >= 2 ? chunkSteps / 2 : 1;
    g->spc = chunkSteps / g->sps;
    g->step_elems = g->step_bytes / 4;
    g->chunk_elems = g->step_bytes * (size_t)chunkSteps / 4;
  } else if (proto == ORC_LL) {
    if (buffSize % 4096 != 0) return ORC_EARG;
    g->step_bytes = buffSize / NSTEPS;
    g->sps = 1;
    g->spc = 1;
    /* one step per chunk; each 16-byte line carries 8 payload bytes */
    g->chunk_elems = g->step_bytes / 2 / 4;
  } else if (proto == ORC_LL128) {
    /* Reading: whole groups of 4 lines per step (a multiple of 4096 bytes). */
    if (buffSize % 4096 != 0) return ORC_EARG;
    g->step_bytes = buffSize / NSTEPS;
    g->sps = 1;
    g->spc = 1;
    /* one step per chunk; each 128-byte line carries 120 payload bytes;
     * reading: rounded down to a multiple of 32 elements */
    g->chunk_elems = (g->step_bytes / 128) * 120 / 4 / 32 * 32;
  } else {
    return ORC_EARG;
  }
  if (g->chunk_elems < 32) return ORC_EARG;
  /* Reading (channel partition): each channel gets a contiguous range of
   * alignUp(divUp(count, C), 16/sizeof(T)) elements, in dense order; the last
   * channels may get fewer or none. */
  g->per_channel = align_up(div_up(count, (size_t)g->nchan), g->align_elems);
  return ORC_OK;
}

static void channel_range(const geom_t* g, int n, size_t* gridOffset, size_t* channelCount) {
  size_t off = g->per_channel * (size_t)n;
  *gridOffset = off;
  *channelCount = off >= g->count ? 0 : min_sz(g->per_channel, g->count - off);
}

/* Elements of a channel's range one loop covers. AllReduce: n chunks of the
 * rank's buffer. Reading (the halves): the channel range is a range of every
 * rank block, and one loop moves one chunk of it from every block. */
static size_t loop_count_of(const geom_t* g) {
  return g->kind == ORC_ALLREDUCE ? (size_t)g->nranks * g->chunk_elems : g->chunk_elems;
}

/* Per-loop chunk size: full chunks, except in the last, short loop where the
 * remainder is split over the n ranks and aligned up to 16/sizeof(T)
 * ([C12] "runRing 的数据切分"). The halves: the remainder, at most a chunk. */
static size_t loop_chunk_count(const geom_t* g, size_t remCount) {
  if (g->kind != ORC_ALLREDUCE) return min_sz(remCount, g->chunk_elems);
  size_t loopCount = loop_count_of(g);
  if (remCount < loopCount) return align_up(div_up(remCount, (size_t)g->nranks), g->align_elems);
  return g->chunk_elems;
}

/* Elements of chunk c in a loop whose remainder is remCount. */
static size_t chunk_nelem(size_t chunkCount, size_t remCount, int c) {
  size_t chunkOffset = chunkCount * (size_t)c;
  return remCount > chunkOffset ? min_sz(chunkCount, remCount - chunkOffset) : 0;
}

/* Slice size of a chunk of nelem elements ([C23] "Slice Size"): the larger of
 * an even split over SlicePerChunk slices in units of 16 elements and 1/32 of
 * the FIFO capacity of one slice, aligned to 16 elements (the page's text;
 * the 1/32 floor is not always a multiple of 16 for the buffer sizes allowed
 * here). LL and LL128 use one slice per chunk. */
static size_t slice_size(const geom_t* g, size_t nelem) {
  if (g->proto != ORC_SIMPLE) return nelem;
  return align_up(max_sz(div_up(nelem, 16 * (size_t)g->spc) * 16, g->step_elems * (size_t)g->sps / 32), 16);
}

/*
 * Geometry summary for tests:
 *   out[0] step_bytes, out[1] chunk_elems, out[2] steps per slice,
 *   out[3] slices per chunk, out[4] C (active channels), out[5] per-channel
 *   element count, out[6..6+C) channel ids (dense order),
 *   out[6+C + 2n], out[6+C + 2n+1] = gridOffset, channelCount of channel n.
 */
int orc_geometry(int proto, int dtype, int nranks, uint64_t mask, size_t count,
                 size_t buffSize, int chunkSteps, int64_t* out) {
  geom_t g;
  int st = geom_init(&g, proto, dtype, nranks, mask, count, buffSize, chunkSteps);
  if (st != ORC_OK) return st;
  out[0] = (int64_t)g.step_bytes;
  out[1] = (int64_t)g.chunk_elems;
  out[2] = g.sps;
  out[3] = g.spc;
  out[4] = g.nchan;
  out[5] = (int64_t)g.per_channel;
  for (int n = 0; n < g.nchan; n++) out[6 + n] = g.chan_id[n];
  for (int n = 0; n < g.nchan; n++) {
    size_t go, cc;
    channel_range(&g, n, &go, &cc);
    out[6 + g.nchan + 2 * n] = (int64_t)go;
    out[6 + g.nchan + 2 * n + 1] = (int64_t)cc;
  }
  return ORC_OK;
}

/*
 * Loop table of one channel for tests: for loop l, rows[3l..3l+2] =
 * elemOffset, remCount, chunkCount. Returns the number of loops (or -1 when
 * max_loops is too small).
 */
int64_t orc_channel_loops(int proto, int dtype, int nranks, uint64_t mask, size_t count,
                          size_t buffSize, int chunkSteps, int n, int64_t* rows,
                          int64_t max_loops) {
  geom_t g;
  if (geom_init(&g, proto, dtype, nranks, mask, count, buffSize, chunkSteps) != ORC_OK) return -1;
  if (n < 0 || n >= g.nchan) return -1;
  size_t go, cc;
  channel_range(&g, n, &go, &cc);
  size_t loopCount = (size_t)nranks * g.chunk_elems;
  int64_t l = 0;
  for (size_t elemOffset = 0; elemOffset < cc; elemOffset += loopCount, l++) {
    if (l >= max_loops) return -1;
    size_t rem = cc - elemOffset;
    rows[3 * l] = (int64_t)elemOffset;
    rows[3 * l + 1] = (int64_t)rem;
    rows[3 * l + 2] = (int64_t)loop_chunk_count(&g, rem);
  }
  return l;
}

/* ------------------------------------------------------------------ */
/* LL and LL128 line formats ([C23] "LL：Data 与 Flag 同 Line",         */
/*                           "LL128：15/16 Payload")                   */
/* ------------------------------------------------------------------ */

/*
 * LL line: 16 bytes = four 32-bit words {data1, flag1, data2, flag2}; data1 is
 * the low half and data2 the high half of 8 payload bytes. Payload bytes
 * [8j, 8j+8) go to line j; the last line is zero-padded.
 */
void orc_ll_encode(const uint8_t* payload, size_t nbytes, uint32_t flag, uint32_t* lines) {
  size_t nlines = div_up(nbytes, 8);
  for (size_t j = 0; j < nlines; j++) {
    uint8_t b[8] = {0};
    memcpy(b, payload + 8 * j, min_sz(8, nbytes - 8 * j));
    uint32_t lo, hi;
    memcpy(&lo, b, 4);
    memcpy(&hi, b + 4, 4);
    lines[4 * j + 0] = lo;
    lines[4 * j + 1] = flag;
    lines[4 * j + 2] = hi;
    lines[4 * j + 3] = flag;
  }
}

/* A line is accepted only when both flags equal the expected one. Returns 0
 * and fills payload when every line is accepted, else 1 + the first line not
 * accepted (payload then untouched from that line on). */
size_t orc_ll_decode(const uint32_t* lines, size_t nbytes, uint32_t flag, uint8_t* payload) {
  size_t nlines = div_up(nbytes, 8);
  for (size_t j = 0; j < nlines; j++) {
    if (lines[4 * j + 1] != flag || lines[4 * j + 3] != flag) return j + 1;
    uint8_t b[8];
    memcpy(b, &lines[4 * j + 0], 4);
    memcpy(b + 4, &lines[4 * j + 2], 4);
    memcpy(payload + 8 * j, b, min_sz(8, nbytes - 8 * j));
  }
  return 0;
}

/*
 * LL128 line: 128 bytes = sixteen 64-bit words; words 0..14 carry 120 payload
 * bytes, word 15 carries the flag. Reading: payload bytes [120l, 120l+120) go
 * to line l in order; the last line is zero-padded.
 */
void orc_ll128_encode(const uint8_t* payload, size_t nbytes, uint64_t flag, uint64_t* lines) {
  size_t nlines = div_up(nbytes, 120);
  for (size_t l = 0; l < nlines; l++) {
    uint8_t b[120] = {0};
    memcpy(b, payload + 120 * l, min_sz(120, nbytes - 120 * l));
    memcpy(&lines[16 * l], b, 120);
    lines[16 * l + 15] = flag;
  }
}

size_t orc_ll128_decode(const uint64_t* lines, size_t nbytes, uint64_t flag, uint8_t* payload) {
  size_t nlines = div_up(nbytes, 120);
  for (size_t l = 0; l < nlines; l++) {
    if (lines[16 * l + 15] != flag) return l + 1;
    memcpy(payload + 120 * l, &lines[16 * l], min_sz(120, nbytes - 120 * l));
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Step-by-step ring simulation                                        */
/* ------------------------------------------------------------------ */

/*
 * Connection e of a channel is the ring edge from ring index e to ring index
 * e+1. It has a FIFO of NSTEPS slots of step_bytes each, a head (steps the
 * receiver has released) and a tail (steps the sender has published; Simple
 * only -- LL and LL128 publish through the flags inside the lines).
 */
typedef struct {
  uint8_t* fifo;
  uint64_t head, tail;
  /* LL sessions only (orc_ll_session_sim): per line of the FIFO, the step its
   * content was written for (NEVER if never written); the receiver's lines of
   * the pending slice accepted so far, and their payload */
  uint64_t* wstep;
  uint8_t* acc;
  uint8_t* pbuf;
} conn_t;

#define NEVER UINT64_MAX

typedef struct {
  const geom_t* g;
  const void* const* send;  /* per user rank */
  void* const* recv;        /* per user rank */
  const int* rank_at;       /* ring index -> user rank */
  conn_t* conn;             /* per ring edge */
  uint64_t sstep[MAXR], rstep[MAXR]; /* per ring index: send / recv step */
  int64_t* sends;           /* per user rank, counted per slice */
  int64_t* recvs;
  uint8_t* pay_in;          /* scratch payload */
  uint8_t* pay_out;
  float* vals;              /* scratch binary32 values */
  int direct;               /* Simple only: all-gather hops write the next rank's output */
  /* LL sessions: line-by-line acceptance, the flag period and its cleanup */
  int session;
  uint32_t flag_max;        /* 0: flag = step + 1 (32 bits); else (step + 1) mod flag_max */
  int cleanup;
  int64_t stale_accepts;    /* lines accepted whose content was written for another step */
  int64_t max_stale_age;    /* largest step distance of a stale line a receiver polled */
} sim_t;

/* LL flag of a step ([C23] "LL：Data 与 Flag 同 Line": production flag = step + 1;
 * the test mode wraps it at 0x100). */
static uint32_t ll_flag_of(const sim_t* S, uint64_t step) {
  return S->flag_max ? (uint32_t)((step + 1) % S->flag_max) : (uint32_t)(step + 1);
}

/* Reading of the page's cleanup: the sender rewrites the rest of its slot
 * (every line past its slice) with the current flag on the last NCCL_STEPS
 * steps of every half flag period, i.e. once per slot every flag_max/2 steps.
 * A line of a slot is then never older than flag_max/2 steps when it is read,
 * so no stale line can carry the flag of the step being read. */
static int ll_cleanup_step(const sim_t* S, uint64_t step) {
  if (!S->cleanup || S->flag_max == 0) return 0;
  uint64_t half = S->flag_max / 2;
  return step % half >= half - NSTEPS;
}

/* One slice of one rank's program. */
typedef struct {
  int prim;
  size_t in_el;  /* element of the rank's input where the slice starts */
  size_t out_el; /* element of the rank's output where the slice starts */
  size_t nelem;
} slice_t;

/*
 * Payload of a hop: rows that send a partial sum (send, recvReduceSend) carry
 * binary32; rows that send the final value (recvReduceCopySend,
 * recvCopySend) carry T. For f32 both are binary32.
 */
static int sends_partial(int prim) { return prim == ORC_SEND || prim == ORC_RECV_REDUCE_SEND; }
static int recvs_partial(int prim) {
  return prim == ORC_RECV_REDUCE_SEND || prim == ORC_RECV_REDUCE_COPY_SEND || prim == ORC_RECV_REDUCE_COPY;
}
static int has_recv(int prim) { return prim != ORC_SEND && prim != ORC_COPY_SEND; }
static int has_send(int prim) { return prim != ORC_RECV && prim != ORC_RECV_REDUCE_COPY; }

static size_t payload_bytes(const geom_t* g, int partial, size_t nelem) {
  return nelem * (partial ? 4 : g->elem_bytes);
}

/* Encode nelem values (binary32 in vals) into payload bytes of the given kind. */
static void pack_values(const geom_t* g, int partial, const float* vals, size_t nelem, uint8_t* out) {
  if (partial || g->dtype == ORC_F32) {
    memcpy(out, vals, nelem * 4);
  } else {
    for (size_t j = 0; j < nelem; j++) {
      uint16_t h = f32_to_bf16_rne(vals[j]);
      memcpy(out + 2 * j, &h, 2);
    }
  }
}

static void unpack_values(const geom_t* g, int partial, const uint8_t* in, size_t nelem, float* vals) {
  if (partial || g->dtype == ORC_F32) {
    memcpy(vals, in, nelem * 4);
  } else {
    for (size_t j = 0; j < nelem; j++) {
      uint16_t h;
      memcpy(&h, in + 2 * j, 2);
      vals[j] = bf16_to_f32(h);
    }
  }
}

/* Try to receive a slice: returns 1 and fills pay_in when the data is there. */
static int fifo_try_recv(sim_t* S, int e, uint64_t step, size_t nbytes) {
  const geom_t* g = S->g;
  conn_t* c = &S->conn[e];
  uint8_t* slot = c->fifo + (step % NSTEPS) * g->step_bytes;
  if (S->session) {
    /* every line on its own, as the GPU's threads poll theirs: a line whose
     * two flags equal the step's flag is taken, whenever it was written */
    uint32_t flag = ll_flag_of(S, step);
    size_t nlines = div_up(nbytes, 8), line0 = (step % NSTEPS) * (g->step_bytes / 16);
    const uint32_t* L = (const uint32_t*)slot;
    int all = 1;
    for (size_t j = 0; j < nlines; j++) {
      if (c->acc[j]) continue;
      uint64_t ws = c->wstep[line0 + j];
      if (ws != step && ws != NEVER && (int64_t)(step - ws) > S->max_stale_age) S->max_stale_age = (int64_t)(step - ws);
      if (L[4 * j + 1] == flag && L[4 * j + 3] == flag) {
        memcpy(c->pbuf + 8 * j, &L[4 * j], 4);
        memcpy(c->pbuf + 8 * j + 4, &L[4 * j + 2], 4);
        c->acc[j] = 1;
        if (ws != step) S->stale_accepts++;
      } else {
        all = 0;
      }
    }
    if (!all) return 0;
    memcpy(S->pay_in, c->pbuf, nbytes);
    memset(c->acc, 0, nlines);
    return 1;
  }
  if (g->proto == ORC_SIMPLE) {
    if (c->tail < step + (uint64_t)g->sps) return 0;
    memcpy(S->pay_in, slot, nbytes);
    return 1;
  }
  if (g->proto == ORC_LL)
    return orc_ll_decode((const uint32_t*)slot, nbytes, (uint32_t)(step + 1), S->pay_in) == 0;
  return orc_ll128_decode((const uint64_t*)slot, nbytes, step + 1, S->pay_in) == 0;
}

/* Credit check for the sender: the slots it is about to fill must have been
 * released, head + NCCL_STEPS >= step + StepPerSlice. */
static int fifo_can_send(sim_t* S, int e, uint64_t step) {
  return S->conn[e].head + NSTEPS >= step + (uint64_t)S->g->sps;
}

static int fifo_send(sim_t* S, int e, uint64_t step, size_t nbytes) {
  const geom_t* g = S->g;
  conn_t* c = &S->conn[e];
  uint8_t* slot = c->fifo + (step % NSTEPS) * g->step_bytes;
  if (g->proto == ORC_SIMPLE) {
    if ((step % NSTEPS) + (uint64_t)g->sps > NSTEPS) return ORC_ECHECK; /* slice would wrap */
    if (nbytes > (size_t)g->sps * g->step_bytes) return ORC_ECHECK;
    memcpy(slot, S->pay_out, nbytes);
    c->tail = step + (uint64_t)g->sps; /* payload first, then the tail */
  } else if (g->proto == ORC_LL && S->session) {
    size_t nlines = div_up(nbytes, 8), slines = g->step_bytes / 16, line0 = (step % NSTEPS) * slines;
    if (nlines > slines) return ORC_ECHECK;
    uint32_t flag = ll_flag_of(S, step);
    orc_ll_encode(S->pay_out, nbytes, flag, (uint32_t*)slot);
    for (size_t j = 0; j < nlines; j++) c->wstep[line0 + j] = step;
    if (ll_cleanup_step(S, step)) {
      uint32_t* L = (uint32_t*)slot;
      for (size_t j = nlines; j < slines; j++) {
        L[4 * j] = 0;
        L[4 * j + 1] = flag;
        L[4 * j + 2] = 0;
        L[4 * j + 3] = flag;
        c->wstep[line0 + j] = step;
      }
    }
  } else if (g->proto == ORC_LL) {
    if (div_up(nbytes, 8) * 16 > g->step_bytes) return ORC_ECHECK;
    orc_ll_encode(S->pay_out, nbytes, (uint32_t)(step + 1), (uint32_t*)slot);
  } else {
    if (div_up(nbytes, 120) * 128 > g->step_bytes) return ORC_ECHECK;
    orc_ll128_encode(S->pay_out, nbytes, step + 1, (uint64_t*)slot);
  }
  return ORC_OK;
}

/*
 * Execute slice `sl` for the rank at ring index i if its waits are met.
 * Returns 1 when executed, 0 when it must wait, or -(error).
 */
static int sim_try_slice(sim_t* S, int i, const slice_t* sl) {
  const geom_t* g = S->g;
  int n = g->nranks;
  int r = S->rank_at[i];
  int e_send = i, e_recv = (i - 1 + n) % n;
  int prim = sl->prim;
  size_t nelem = sl->nelem;
  /* Direct all-gather ([C23] "发布顺序与 Fence", direct read/write; [C12]
   * "源码步骤三" .. "源码步骤五"): a hop that carries a final value writes it
   * straight into the next rank's output at the same offset instead of a FIFO
   * slot, then publishes the tail as usual; its receiver waits for the tail and
   * finds the value already in its own output. No slot is filled, so the
   * sender skips the credit wait; the step counters advance as before. */
  /* AllGather's first row sends a final value too, so it writes directly as well. */
  int direct_send = S->direct && (prim == ORC_RECV_REDUCE_COPY_SEND || prim == ORC_RECV_COPY_SEND ||
                                  prim == ORC_COPY_SEND);
  int direct_recv = S->direct && (prim == ORC_RECV_COPY_SEND || prim == ORC_RECV);
  int r_next = S->rank_at[(i + 1) % n];
  if (has_send(prim) && !direct_send && !fifo_can_send(S, e_send, S->sstep[i])) return 0;
  if (direct_recv) {
    if (S->conn[e_recv].tail < S->rstep[i] + (uint64_t)g->sps) return 0;
    for (size_t j = 0; j < nelem; j++) S->vals[j] = load_as_f32(S->recv[r], g->dtype, sl->out_el + j);
  } else if (has_recv(prim)) {
    size_t nb = payload_bytes(g, recvs_partial(prim), nelem);
    if (!fifo_try_recv(S, e_recv, S->rstep[i], nb)) return 0;
    unpack_values(g, recvs_partial(prim), S->pay_in, nelem, S->vals);
  }
  /* The arithmetic of the primitives ([C12] "源码步骤一..五"). */
  for (size_t j = 0; j < nelem; j++) {
    size_t ie = sl->in_el + j, oe = sl->out_el + j;
    switch (prim) {
      case ORC_SEND:
        S->vals[j] = load_as_f32(S->send[r], g->dtype, ie); /* the raw local input, no reduction */
        break;
      case ORC_RECV_REDUCE_SEND:
        S->vals[j] = S->vals[j] + load_as_f32(S->send[r], g->dtype, ie);
        break;
      case ORC_RECV_REDUCE_COPY_SEND:
      case ORC_RECV_REDUCE_COPY: {
        float v = S->vals[j] + load_as_f32(S->send[r], g->dtype, ie); /* the last reduction */
        store_from_f32(S->recv[r], g->dtype, oe, v); /* rounded once for bf16 */
        S->vals[j] = load_as_f32(S->recv[r], g->dtype, oe); /* forward the stored value */
        break;
      }
      case ORC_COPY_SEND:
        S->vals[j] = load_as_f32(S->send[r], g->dtype, ie);
        store_from_f32(S->recv[r], g->dtype, oe, S->vals[j]); /* exact: the value is already T */
        break;
      case ORC_RECV_COPY_SEND:
      case ORC_RECV:
        if (!direct_recv) store_from_f32(S->recv[r], g->dtype, oe, S->vals[j]);
        break;
    }
  }
  if (has_send(prim)) {
    if (direct_send) {
      /* the same block offset in the next rank's output */
      for (size_t j = 0; j < nelem; j++) store_from_f32(S->recv[r_next], g->dtype, sl->out_el + j, S->vals[j]);
      S->conn[e_send].tail = S->sstep[i] + (uint64_t)g->sps; /* data first, then the tail */
    } else {
      size_t nb = payload_bytes(g, sends_partial(prim), nelem);
      pack_values(g, sends_partial(prim), S->vals, nelem, S->pay_out);
      int st = fifo_send(S, e_send, S->sstep[i], nb);
      if (st != ORC_OK) return -st;
    }
    S->sstep[i] += (uint64_t)g->sps;
    S->sends[r]++;
  }
  if (has_recv(prim)) {
    S->rstep[i] += (uint64_t)g->sps;
    S->conn[e_recv].head = S->rstep[i]; /* release the slots just read */
    S->recvs[r]++;
  }
  /* credit bound: never more than NCCL_STEPS steps outstanding on an edge
   * (direct all-gather steps occupy no slot, so the bound holds for FIFO use only) */
  if (!S->direct)
    for (int e = 0; e < n; e++)
      if (S->conn[e].tail > S->conn[e].head + NSTEPS) return -ORC_ECHECK;
  return 1;
}

/*
 * The program of the rank at ring index i on one channel: loops x rows x
 * slices. AllReduce: chunk c of a loop is a piece of every rank's buffer, at
 * the same offset in input and output. The halves (reading, the collectives'
 * usual shapes): a ReduceScatter input and an AllGather output hold n blocks
 * of `count` elements, block b belonging to user rank b; a chunk with ring
 * index c is the loop's range of the block of user rank rank_at[c], and the
 * other side (ReduceScatter output, AllGather input) holds one block.
 */
static size_t build_program(const geom_t* g, const int* rank_at, int i, size_t gridOffset,
                            size_t channelCount, slice_t* prog) {
  int n = g->nranks;
  size_t loopCount = loop_count_of(g);
  size_t k = 0;
  for (size_t elemOffset = 0; elemOffset < channelCount; elemOffset += loopCount) {
    size_t rem = channelCount - elemOffset;
    size_t chunkCount = loop_chunk_count(g, rem);
    for (int s = 0; s < rows_of_kind(g->kind, n); s++) {
      int c = chunk_of_kind_row(g->kind, n, i, s);
      size_t nelem, base;
      if (g->kind == ORC_ALLREDUCE) {
        nelem = chunk_nelem(chunkCount, rem, c);
        base = gridOffset + elemOffset + chunkCount * (size_t)c;
      } else {
        nelem = chunkCount;
        base = gridOffset + elemOffset;
      }
      size_t blk = (size_t)rank_at[c] * g->count;
      size_t ss = slice_size(g, nelem);
      for (int q = 0; q < g->spc; q++) {
        size_t so = ss * (size_t)q;
        slice_t sl;
        sl.prim = prim_of_kind_row(g->kind, n, s);
        sl.in_el = base + so + (g->kind == ORC_REDUCE_SCATTER ? blk : 0);
        sl.out_el = base + so + (g->kind == ORC_ALL_GATHER ? blk : 0);
        sl.nelem = nelem > so ? min_sz(ss, nelem - so) : 0; /* empty slices still run */
        if (prog) prog[k] = sl;
        k++;
      }
    }
  }
  return k;
}

/*
 * Step-by-step simulation of one ring collective call over all channels.
 * kind: ORC_ALLREDUCE (send[r], recv[r]: `count` elements), ORC_REDUCE_SCATTER
 * (send[r]: nranks*count, recv[r]: count) or ORC_ALL_GATHER (send[r]: count,
 * recv[r]: nranks*count); elements are binary32 or bf16 bit patterns.
 * sends/recvs (optional, per user rank) count the slices each rank sent and
 * received; loops_out (optional, per dense channel) the chunk loops of each
 * channel.
 * Ranks are run round-robin; each runs its next slices until a wait is not
 * met. When a full round makes no progress while work remains, the result is
 * ORC_EDEADLOCK.
 */
int orc_ring_collective_sim(int kind, const void* const* send, void* const* recv, int nranks, size_t count,
                            int dtype, const int* ring_order, int nrings, uint64_t mask, int proto,
                            size_t buffSize, int chunkSteps, int direct, int64_t* sends, int64_t* recvs,
                            int64_t* loops_out) {
  geom_t g;
  if (kind < ORC_ALLREDUCE || kind > ORC_ALL_GATHER) return ORC_EARG;
  int st = geom_init(&g, proto, dtype, nranks, mask, count, buffSize, chunkSteps);
  if (st != ORC_OK) return st;
  g.kind = kind;
  if (nrings != 1 && nrings != g.nchan) return ORC_EARG;
  if (direct && proto != ORC_SIMPLE) return ORC_EARG;
  /* ReduceScatter has no hop that carries a final value: nothing to write directly */
  if (direct && kind == ORC_REDUCE_SCATTER) return ORC_EARG;
  int rank_at[MAXR];
  for (int ch = 0; ch < nrings; ch++) {
    st = rank_at_index(nranks, ring_order + (size_t)ch * nranks, rank_at);
    if (st != ORC_OK) return st;
  }
  int64_t dummy_s[MAXR] = {0}, dummy_r[MAXR] = {0};
  if (!sends) sends = dummy_s;
  if (!recvs) recvs = dummy_r;
  for (int r = 0; r < nranks; r++) { sends[r] = 0; recvs[r] = 0; }

  size_t max_payload = (size_t)g.sps * g.step_bytes + 256;
  conn_t* conn = calloc((size_t)nranks, sizeof(conn_t));
  uint8_t* fifo = calloc((size_t)nranks * NSTEPS, g.step_bytes);
  uint8_t* pin = malloc(max_payload);
  uint8_t* pout = malloc(max_payload);
  float* vals = malloc(sizeof(float) * (g.chunk_elems + 64));
  slice_t* prog[MAXR] = {0};
  size_t cursor[MAXR];
  int rc = ORC_OK;
  if (!conn || !fifo || !pin || !pout || !vals) { rc = ORC_ENOMEM; goto done; }

  sim_t S;
  memset(&S, 0, sizeof S);
  S.g = &g;
  S.send = send;
  S.recv = recv;
  S.rank_at = rank_at;
  S.conn = conn;
  S.sends = sends;
  S.recvs = recvs;
  S.pay_in = pin;
  S.pay_out = pout;
  S.vals = vals;
  S.direct = direct;

  for (int ch = 0; ch < g.nchan; ch++) {
    /* this channel's ring ([C12] "GRAPH 重建：N=4": channels may use different ring orders) */
    rank_at_index(nranks, ring_order + (nrings == 1 ? 0 : (size_t)ch * nranks), rank_at);
    size_t gridOffset, channelCount;
    channel_range(&g, ch, &gridOffset, &channelCount);
    /* a fresh connector set per channel: FIFOs zeroed, steps from 0 */
    memset(fifo, 0, (size_t)nranks * NSTEPS * g.step_bytes);
    for (int e = 0; e < nranks; e++) {
      conn[e].fifo = fifo + (size_t)e * NSTEPS * g.step_bytes;
      conn[e].head = conn[e].tail = 0;
    }
    size_t nslices = 0;
    for (int i = 0; i < nranks; i++) {
      S.sstep[i] = S.rstep[i] = 0;
      nslices = build_program(&g, rank_at, i, gridOffset, channelCount, NULL);
      free(prog[i]);
      prog[i] = malloc(sizeof(slice_t) * (nslices ? nslices : 1));
      if (!prog[i]) { rc = ORC_ENOMEM; goto done; }
      build_program(&g, rank_at, i, gridOffset, channelCount, prog[i]);
      cursor[i] = 0;
    }
    if (loops_out) loops_out[ch] = (int64_t)div_up(channelCount, loop_count_of(&g));
    int finished = 0;
    while (finished < nranks) {
      int progressed = 0;
      for (int i = 0; i < nranks; i++) {
        while (cursor[i] < nslices) {
          int r = sim_try_slice(&S, i, &prog[i][cursor[i]]);
          if (r < 0) { rc = -r; goto done; }
          if (r == 0) break;
          cursor[i]++;
          progressed = 1;
          if (cursor[i] == nslices) finished++;
        }
      }
      if (nslices == 0) break;
      if (!progressed) { rc = ORC_EDEADLOCK; goto done; }
    }
    /* after a call every edge has released everything it published */
    for (int e = 0; e < nranks; e++)
      if (g.proto == ORC_SIMPLE && conn[e].head != conn[e].tail) { rc = ORC_ECHECK; goto done; }
  }
done:
  for (int i = 0; i < nranks; i++) free(prog[i]);
  free(conn);
  free(fifo);
  free(pin);
  free(pout);
  free(vals);
  return rc;
}

int orc_ring_allreduce_sim(const void* const* send, void* const* recv, int nranks, size_t count,
                           int dtype, const int* ring_order, int nrings, uint64_t mask, int proto,
                           size_t buffSize, int chunkSteps, int direct, int64_t* sends, int64_t* recvs,
                           int64_t* loops_out) {
  return orc_ring_collective_sim(ORC_ALLREDUCE, send, recv, nranks, count, dtype, ring_order, nrings, mask,
                                 proto, buffSize, chunkSteps, direct, sends, recvs, loops_out);
}

/*
 * A sequence of ring AllReduce calls on one LL workspace, as the library runs
 * them: the connector FIFOs and every rank's step counters persist from call
 * to call (nothing is cleared between calls, [C23] "LL：Data 与 Flag 同 Line":
 * the monotonic generation makes old lines mismatch). Receivers take each
 * 16-byte line on its own as soon as both its flags equal the step's flag,
 * the way the GPU's threads poll their lines, so a stale line that happens to
 * carry the right flag is taken: the simulation counts such lines.
 *
 * Call k uses counts[k] elements per rank, send[k*nranks + r] and
 * recv[k*nranks + r]. flag_max 0: production flags (step + 1, 32 bits);
 * otherwise a power of two >= 64, flags (step + 1) mod flag_max (the page's
 * test mode wraps at 0x100), with the slot cleanup when `cleanup` is set
 * (tests turn it off to show what it prevents). Outputs: stale_accepts (lines
 * taken whose content was written for another step) and max_stale_age (the
 * largest step distance between a polled stale line's write and the poll).
 */
int orc_ll_session_sim(int ncalls, const size_t* counts, const void* const* send, void* const* recv,
                       int nranks, int dtype, const int* ring_order, int nrings, uint64_t mask,
                       size_t buffSize, uint32_t flag_max, int cleanup, int64_t* stale_accepts,
                       int64_t* max_stale_age) {
  if (ncalls < 0) return ORC_EARG;
  if (flag_max != 0 && (flag_max < 64 || (flag_max & (flag_max - 1)) != 0)) return ORC_EARG;
  geom_t g;
  int st = geom_init(&g, ORC_LL, dtype, nranks, mask, 0, buffSize, 4);
  if (st != ORC_OK) return st;
  if (nrings != 1 && nrings != g.nchan) return ORC_EARG;
  int rank_at[MAXR];
  for (int ch = 0; ch < nrings; ch++) {
    st = rank_at_index(nranks, ring_order + (size_t)ch * nranks, rank_at);
    if (st != ORC_OK) return st;
  }
  size_t nconn = (size_t)g.nchan * nranks, slines = g.step_bytes / 16;
  conn_t* conn = calloc(nconn, sizeof(conn_t));
  uint8_t* fifo = calloc(nconn * NSTEPS, g.step_bytes);
  uint64_t* wstep = malloc(sizeof(uint64_t) * nconn * NSTEPS * slines);
  uint8_t* acc = calloc(nconn, slines);
  uint8_t* pbuf = calloc(nconn, slines * 8);
  uint64_t* steps = calloc((size_t)2 * nconn, sizeof(uint64_t)); /* per channel and ring index: send, recv */
  uint8_t* pin = malloc(g.step_bytes);
  uint8_t* pout = malloc(g.step_bytes);
  float* vals = malloc(sizeof(float) * (g.chunk_elems + 64));
  slice_t* prog[MAXR] = {0};
  size_t cursor[MAXR];
  int64_t sends[MAXR], recvs[MAXR];
  int rc = ORC_OK;
  sim_t S;
  memset(&S, 0, sizeof S);
  if (!conn || !fifo || !wstep || !acc || !pbuf || !steps || !pin || !pout || !vals) { rc = ORC_ENOMEM; goto done; }
  for (size_t k = 0; k < nconn * NSTEPS * slines; k++) wstep[k] = NEVER;
  for (size_t e = 0; e < nconn; e++) {
    conn[e].fifo = fifo + e * NSTEPS * g.step_bytes;
    conn[e].wstep = wstep + e * NSTEPS * slines;
    conn[e].acc = acc + e * slines;
    conn[e].pbuf = pbuf + e * slines * 8;
  }
  S.g = &g;
  S.rank_at = rank_at;
  S.sends = sends;
  S.recvs = recvs;
  S.pay_in = pin;
  S.pay_out = pout;
  S.vals = vals;
  S.session = 1;
  S.flag_max = flag_max;
  S.cleanup = cleanup;
  for (int k = 0; k < ncalls; k++) {
    g.count = counts[k];
    g.per_channel = align_up(div_up(g.count, (size_t)g.nchan), g.align_elems);
    S.send = send + (size_t)k * nranks;
    S.recv = recv + (size_t)k * nranks;
    if (g.count == 0) continue; /* an empty call advances nothing */
    for (int ch = 0; ch < g.nchan; ch++) {
      rank_at_index(nranks, ring_order + (nrings == 1 ? 0 : (size_t)ch * nranks), rank_at);
      size_t gridOffset, channelCount;
      channel_range(&g, ch, &gridOffset, &channelCount);
      S.conn = conn + (size_t)ch * nranks;
      size_t nslices = 0;
      for (int i = 0; i < nranks; i++) {
        S.sstep[i] = steps[2 * ((size_t)ch * nranks + i)];
        S.rstep[i] = steps[2 * ((size_t)ch * nranks + i) + 1];
        nslices = build_program(&g, rank_at, i, gridOffset, channelCount, NULL);
        free(prog[i]);
        prog[i] = malloc(sizeof(slice_t) * (nslices ? nslices : 1));
        if (!prog[i]) { rc = ORC_ENOMEM; goto done; }
        build_program(&g, rank_at, i, gridOffset, channelCount, prog[i]);
        cursor[i] = 0;
      }
      int finished = 0;
      while (finished < nranks && nslices > 0) {
        int progressed = 0;
        for (int i = 0; i < nranks; i++) {
          while (cursor[i] < nslices) {
            int r = sim_try_slice(&S, i, &prog[i][cursor[i]]);
            if (r < 0) { rc = -r; goto done; }
            if (r == 0) break;
            cursor[i]++;
            progressed = 1;
            if (cursor[i] == nslices) finished++;
          }
        }
        if (!progressed) { rc = ORC_EDEADLOCK; goto done; }
      }
      for (int i = 0; i < nranks; i++) {
        steps[2 * ((size_t)ch * nranks + i)] = S.sstep[i];
        steps[2 * ((size_t)ch * nranks + i) + 1] = S.rstep[i];
      }
    }
  }
done:
  if (stale_accepts) *stale_accepts = S.stale_accepts;
  if (max_stale_age) *max_stale_age = S.max_stale_age;
  for (int i = 0; i < nranks; i++) free(prog[i]);
  free(conn);
  free(fifo);
  free(wstep);
  free(acc);
  free(pbuf);
  free(steps);
  free(pin);
  free(pout);
  free(vals);
  return rc;
}

/* ------------------------------------------------------------------ */
/* Closed form of the ring result                                      */
/* ------------------------------------------------------------------ */

/*
 * The value the ring leaves in every rank's output, written out directly:
 * element e lies in chunk c of some loop of some channel. Its partial sum
 * starts at ring index c+1 with that rank's raw input and travels forward,
 * each rank adding its own input, until the owner (ring index c) adds its
 * input last ([C12] "源码步骤一..三"):
 *   acc = x[c+1]; acc = acc + x[c+2]; ...; acc = acc + x[c]   (indices mod n)
 * where x[j] is the input of the rank with ring index j. bf16 inputs are
 * widened exactly, the sum is binary32, and the result is rounded to bf16
 * once. Every rank gets the same value.
 */
static float ring_fold(const geom_t* g, const void* const* send, const int* rank_at, int c,
                       size_t el) {
  int n = g->nranks;
  float acc = load_as_f32(send[rank_at[(c + 1) % n]], g->dtype, el);
  for (int k = 2; k <= n; k++) acc = acc + load_as_f32(send[rank_at[(c + k) % n]], g->dtype, el);
  return acc;
}

int orc_ring_allreduce_closed(const void* const* send, void* const* recv, int nranks, size_t count,
                              int dtype, const int* ring_order, int nrings, uint64_t mask, int proto,
                              size_t buffSize, int chunkSteps) {
  geom_t g;
  int st = geom_init(&g, proto, dtype, nranks, mask, count, buffSize, chunkSteps);
  if (st != ORC_OK) return st;
  if (nrings != 1 && nrings != g.nchan) return ORC_EARG;
  int rank_at[MAXR];
  size_t loopCount = (size_t)nranks * g.chunk_elems;
  for (int ch = 0; ch < g.nchan; ch++) {
    st = rank_at_index(nranks, ring_order + (nrings == 1 ? 0 : (size_t)ch * nranks), rank_at);
    if (st != ORC_OK) return st;
    size_t gridOffset, channelCount;
    channel_range(&g, ch, &gridOffset, &channelCount);
    for (size_t elemOffset = 0; elemOffset < channelCount; elemOffset += loopCount) {
      size_t rem = channelCount - elemOffset;
      size_t chunkCount = loop_chunk_count(&g, rem);
      for (int c = 0; c < nranks; c++) {
        size_t nelem = chunk_nelem(chunkCount, rem, c);
        size_t base = gridOffset + elemOffset + chunkCount * (size_t)c;
        for (size_t j = 0; j < nelem; j++) {
          float v = ring_fold(&g, send, rank_at, c, base + j);
          for (int r = 0; r < nranks; r++) store_from_f32(recv[r], dtype, base + j, v);
        }
      }
    }
  }
  return ORC_OK;
}

/*
 * Closed form of the halves ([C12] "Ring AllReduce 不只是“绕一圈”": AllReduce is
 * ReduceScatter followed by AllGather).
 * ReduceScatter: element j of rank r's output is block r, element j, folded
 *   along the ring of j's channel exactly as an AllReduce chunk whose owner is
 *   r: it starts at the rank after r on the ring and ends with r's own input,
 *     out_r[j] = T(x[c+1][r*count+j] + x[c+2][r*count+j] + ... + x[c][r*count+j])
 *   with c the ring index of r and x[i] the input of the rank at ring index i.
 * AllGather: out_r[q*count + j] = in_q[j] for every pair of ranks (a copy).
 * The channel of element j is the one whose range of the block holds j.
 */
int orc_ring_halves_closed(int kind, const void* const* send, void* const* recv, int nranks, size_t count,
                           int dtype, const int* ring_order, int nrings, uint64_t mask, int proto,
                           size_t buffSize, int chunkSteps) {
  geom_t g;
  if (kind != ORC_REDUCE_SCATTER && kind != ORC_ALL_GATHER) return ORC_EARG;
  int st = geom_init(&g, proto, dtype, nranks, mask, count, buffSize, chunkSteps);
  if (st != ORC_OK) return st;
  g.kind = kind;
  if (nrings != 1 && nrings != g.nchan) return ORC_EARG;
  int rank_at[MAXR], index[MAXR];
  for (int ch = 0; ch < g.nchan; ch++) {
    st = rank_at_index(nranks, ring_order + (nrings == 1 ? 0 : (size_t)ch * nranks), rank_at);
    if (st != ORC_OK) return st;
    for (int c = 0; c < nranks; c++) index[rank_at[c]] = c;
    size_t gridOffset, channelCount;
    channel_range(&g, ch, &gridOffset, &channelCount);
    for (size_t j = gridOffset; j < gridOffset + channelCount; j++) {
      for (int r = 0; r < nranks; r++) {
        if (kind == ORC_REDUCE_SCATTER) {
          float v = ring_fold(&g, send, rank_at, index[r], (size_t)r * count + j);
          store_from_f32(recv[r], dtype, j, v);
        } else {
          for (int q = 0; q < nranks; q++)
            store_from_f32(recv[r], dtype, (size_t)q * count + j, load_as_f32(send[q], dtype, j));
        }
      }
    }
  }
  return ORC_OK;
}

/*
 * The same value at m chosen element indices only, for sizes where a full
 * evaluation is too slow. sampled[r][k] is the input of user rank r at element
 * idx[k] (the caller gathers them); count is the full per-rank element count,
 * which fixes the geometry. Writes out[k] as T (binary32 or bf16 bits), and
 * chunk_out[k] (optional) = the chunk index c that element idx[k] lies in.
 */
int orc_ring_closed_at(const void* const* sampled, int nranks, size_t count, int dtype,
                       const int* ring_order, int nrings, uint64_t mask, int proto, size_t buffSize,
                       int chunkSteps, const int64_t* idx, size_t m, void* out,
                       int32_t* chunk_out) {
  geom_t g;
  int st = geom_init(&g, proto, dtype, nranks, mask, count, buffSize, chunkSteps);
  if (st != ORC_OK) return st;
  if (nrings != 1 && nrings != g.nchan) return ORC_EARG;
  int rank_at[MAXR];
  size_t loopCount = (size_t)nranks * g.chunk_elems;
  for (size_t k = 0; k < m; k++) {
    if (idx[k] < 0 || (size_t)idx[k] >= count) return ORC_EARG;
    size_t el = (size_t)idx[k];
    int ch = (int)(el / g.per_channel);
    st = rank_at_index(nranks, ring_order + (nrings == 1 ? 0 : (size_t)ch * nranks), rank_at);
    if (st != ORC_OK) return st;
    size_t gridOffset, channelCount;
    channel_range(&g, ch, &gridOffset, &channelCount);
    size_t off = el - gridOffset;
    size_t elemOffset = off / loopCount * loopCount;
    size_t rem = channelCount - elemOffset;
    size_t chunkCount = loop_chunk_count(&g, rem);
    int c = (int)((off - elemOffset) / chunkCount);
    if (c >= nranks || (off - elemOffset) - chunkCount * (size_t)c >= chunk_nelem(chunkCount, rem, c))
      return ORC_ECHECK;
    /* sample k plays the role of element el */
    store_from_f32(out, dtype, k, ring_fold(&g, sampled, rank_at, c, k));
    if (chunk_out) chunk_out[k] = c;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* One-shot AllReduce ([OS89] one-shot kernel description)             */
/* ------------------------------------------------------------------ */

/*
 * Every rank reads all peers' inputs and reduces them itself; the sum is
 * binary32, taken in user-rank order 0..n-1, and (for bf16) rounded once:
 *   out_r[e] = T(((x_0[e] + x_1[e]) + x_2[e]) + ... + x_{n-1}[e]).
 * Each rank's output is computed from the inputs, rank by rank.
 */
int orc_oneshot(const void* const* send, void* const* recv, int nranks, size_t count, int dtype) {
  if (nranks < 1 || nranks > MAXR) return ORC_EARG;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_EARG;
  for (int r = 0; r < nranks; r++) {
    for (size_t e = 0; e < count; e++) {
      float acc = load_as_f32(send[0], dtype, e);
      for (int q = 1; q < nranks; q++) acc = acc + load_as_f32(send[q], dtype, e);
      store_from_f32(recv[r], dtype, e, acc);
    }
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Credit / flag state model ([C23] "状态机故障注入")                    */
/* ------------------------------------------------------------------ */

/*
 * A deterministic discrete model of one connector: a producer and a consumer
 * share a FIFO of `slots` slots and move `total` steps. Step t carries the
 * value t. Each side's step is split into micro-operations; the model checker
 * explores every interleaving of the two sides (the state is the pair of
 * program counters, which fixes the FIFO contents) and reports:
 *   outcome 0 COMPLETE   every interleaving finishes all steps correctly;
 *   outcome 1 STALL      some interleaving reaches a state with no enabled
 *                        micro-operation before the end (deadlock / blocked);
 *   outcome 2 CORRUPT    some interleaving lets the consumer accept a value
 *                        that is not the one produced for that step;
 * corruption is reported in preference to a stall.
 * res[0] outcome, res[1] kinds of corruption seen (bit 0: an older
 * generation accepted; bit 1: a slot accepted before its data was ever
 * written), res[2]/res[3] producer/consumer steps
 * done at the first stall found (by smallest producer progress), res[4]
 * number of states explored.
 *
 * Protocols and faults (the nine rows of the page's table):
 *   Simple: 0 normal head/tail, 1 receiver drops its head update,
 *           2 tail published before the payload;
 *   LL:     0 both flags = step+1, 1 second flag never written,
 *           2 constant flag (the same value every generation);
 *   LL128:  0 line with flag word, 1 flag word never written,
 *           2 flag word written before the data words.
 */
enum { M_COMPLETE = 0, M_STALL = 1, M_CORRUPT = 2 };

typedef struct {
  int proto, fault, slots, total;
  /* FIFO slot contents, derived from the producer position */
  int64_t data[NSTEPS], flag1[NSTEPS], flag2[NSTEPS];
  int64_t head, tail;
} mstate_t;

/* micro-operations per step */
static int prod_ops(int proto, int fault) {
  if (proto == ORC_SIMPLE) return 2;           /* payload, tail (or reversed) */
  if (proto == ORC_LL128 && fault == 2) return 2; /* flag word, then data */
  return 1;                                    /* whole line in one store */
}
static int cons_ops(void) { return 2; }        /* read (after wait), release head */

/* Rebuild slot contents and head/tail from the two program counters. */
static void model_rebuild(mstate_t* m, int pt, int pp, int ct, int cp) {
  for (int s = 0; s < m->slots; s++) { m->data[s] = -1; m->flag1[s] = 0; m->flag2[s] = 0; }
  m->head = 0;
  m->tail = 0;
  for (int t = 0; t <= pt && t < m->total; t++) {
    int ops_done = (t < pt) ? prod_ops(m->proto, m->fault) : pp;
    int s = t % m->slots;
    int64_t flag = (m->proto == ORC_LL && m->fault == 2) ? 1 : t + 1;
    if (m->proto == ORC_SIMPLE) {
      int payload_op = (m->fault == 2) ? 1 : 0;
      int tail_op = (m->fault == 2) ? 0 : 1;
      if (ops_done > payload_op) m->data[s] = t;
      if (ops_done > tail_op) m->tail = t + 1;
    } else if (m->proto == ORC_LL) {
      if (ops_done >= 1) {
        m->data[s] = t;
        m->flag1[s] = flag;
        if (m->fault != 1) m->flag2[s] = flag; /* fault 1: second flag never written */
      }
    } else { /* LL128 */
      if (m->fault == 2) {
        if (ops_done >= 1) m->flag1[s] = flag;
        if (ops_done >= 2) m->data[s] = t;
      } else if (ops_done >= 1) {
        m->data[s] = t;
        if (m->fault != 1) m->flag1[s] = flag;
      }
    }
  }
  for (int t = 0; t <= ct && t < m->total; t++) {
    int ops_done = (t < ct) ? cons_ops() : cp;
    if (ops_done >= 2 && !(m->proto == ORC_SIMPLE && m->fault == 1)) m->head = t + 1;
  }
}

/* Is the consumer's wait for step u met, given the current contents? */
static int cons_ready(const mstate_t* m, int u) {
  int s = u % m->slots;
  int64_t flag = (m->proto == ORC_LL && m->fault == 2) ? 1 : u + 1;
  if (m->proto == ORC_SIMPLE) return m->tail >= u + 1;
  if (m->proto == ORC_LL) return m->flag1[s] == flag && m->flag2[s] == flag;
  return m->flag1[s] == flag;
}

int orc_state_model(int proto, int fault, int slots, int total, int64_t* res) {
  if (slots < 1 || slots > NSTEPS || total < 1 || total > 4096) return ORC_EARG;
  if (proto != ORC_SIMPLE && proto != ORC_LL && proto != ORC_LL128) return ORC_EARG;
  if (fault < 0 || fault > 2) return ORC_EARG;
  int P = prod_ops(proto, fault), Q = cons_ops();
  /* state = (producer step, producer op, consumer step, consumer op) */
  size_t dim_p = (size_t)(total + 1) * (size_t)P, dim_c = (size_t)(total + 1) * (size_t)Q;
  uint8_t* seen = calloc(dim_p * dim_c, 1);
  int32_t* stack = malloc(sizeof(int32_t) * 4 * dim_p * dim_c + 16);
  if (!seen || !stack) { free(seen); free(stack); return ORC_ENOMEM; }
  mstate_t m;
  memset(&m, 0, sizeof m);
  m.proto = proto;
  m.fault = fault;
  m.slots = slots;
  m.total = total;
  int outcome = M_COMPLETE, kind = 0;
  int64_t stall_p = -1, stall_c = -1, explored = 0;
  size_t sp = 0;
#define KEY(a, b, c, d) (((size_t)(a) * P + (b)) * dim_c + (size_t)(c) * Q + (d))
  stack[sp++] = 0; stack[sp++] = 0; stack[sp++] = 0; stack[sp++] = 0;
  seen[KEY(0, 0, 0, 0)] = 1;
  while (sp > 0) {
    int cp = stack[--sp], ct = stack[--sp], pp = stack[--sp], pt = stack[--sp];
    explored++;
    if (pt == total && ct == total) continue; /* finished */
    model_rebuild(&m, pt, pp, ct, cp);
    int moves = 0;
    /* producer micro-op */
    if (pt < total) {
      int enabled = 1;
      if (pp == 0) enabled = (m.head + slots >= pt + 1); /* credit before the first write */
      if (enabled) {
        int npt = pt, npp = pp + 1;
        if (npp == P) { npt++; npp = 0; }
        moves++;
        if (!seen[KEY(npt, npp, ct, cp)]) {
          seen[KEY(npt, npp, ct, cp)] = 1;
          stack[sp++] = npt; stack[sp++] = npp; stack[sp++] = ct; stack[sp++] = cp;
        }
      }
    }
    /* consumer micro-op */
    if (ct < total) {
      int enabled = 1;
      if (cp == 0) {
        enabled = cons_ready(&m, ct);
        if (enabled) {
          int64_t got = m.data[ct % slots];
          if (got != ct) {
            outcome = M_CORRUPT;
            kind |= (got >= 0 && got < ct) ? 1 : 2;
            enabled = 0; /* this path is already wrong; do not continue it */
            moves++;
          }
        }
      }
      if (enabled) {
        int nct = ct, ncp = cp + 1;
        if (ncp == Q) { nct++; ncp = 0; }
        moves++;
        if (!seen[KEY(pt, pp, nct, ncp)]) {
          seen[KEY(pt, pp, nct, ncp)] = 1;
          stack[sp++] = pt; stack[sp++] = pp; stack[sp++] = nct; stack[sp++] = ncp;
        }
      }
    }
    if (moves == 0) {
      if (outcome == M_COMPLETE) outcome = M_STALL;
      if (stall_p < 0 || pt < stall_p) { stall_p = pt; stall_c = ct; }
    }
  }
#undef KEY
  free(seen);
  free(stack);
  res[0] = outcome;
  res[1] = kind;
  res[2] = stall_p;
  res[3] = stall_c;
  res[4] = explored;
  return ORC_OK;
}
