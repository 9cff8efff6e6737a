// rar_api.cu -- the C ABI of librar.so (declared in include/rar.h): argument
// checks, ring setup, workspace sizing and initialisation, launches, status.
//
// Pages cited (by title, then section):
//   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
//   [C12] "NCCL 专家课程 12：Ring AllReduce 逐步推导、真实 Ring 与 Channel 并行"
//         sections "ring index 如何计算", "Graph 如何变成完整 ring"
//   [OS89] "perf(osar): all-reduce 5커널 → 3커널 (가드·웨이트 프롤로그 융합) - #89"
//          (review finding: an empty input must not advance any state)
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "rar.h"
#include "rar_launch.h"

namespace rar {
namespace {

std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<int> g_fault{0};
std::atomic<uint32_t> g_ll_flag_max{0};

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

}  // namespace

bool trace_on() {
  static const bool on = [] {
    const char* env = std::getenv("RAR_TRACE");
    return env != nullptr && env[0] != '\0' && std::strcmp(env, "0") != 0;
  }();
  return on;
}

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<uint32_t> g_setup[kMaxDevices];
}  // namespace

cudaError_t current_device_sms(int* device, int* sms) {
  cudaError_t e = cudaGetDevice(device);
  if (e != cudaSuccess) return e;
  const bool cached = *device >= 0 && *device < kMaxDevices;
  if (cached) {
    const int v = g_sm_count[*device].load(std::memory_order_relaxed);
    if (v != 0) {
      *sms = v;
      return cudaSuccess;
    }
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *device);
  if (e == cudaSuccess && cached) g_sm_count[*device].store(*sms, std::memory_order_relaxed);
  return e;
}

bool setup_done(int device, int key) {
  return device >= 0 && device < kMaxDevices && ((g_setup[device].load(std::memory_order_acquire) >> key) & 1u);
}

void mark_setup_done(int device, int key) {
  if (device >= 0 && device < kMaxDevices) g_setup[device].fetch_or(1u << key, std::memory_order_release);
}

namespace {

uint64_t spin_timeout_ns() {
  uint64_t t = g_timeout_ns.load(std::memory_order_relaxed);
  if (t != 0) return t;
  const char* env = std::getenv("RAR_SPIN_TIMEOUT_NS");
  if (env != nullptr) {
    unsigned long long v = std::strtoull(env, nullptr, 10);
    if (v > 0) return (uint64_t)v;
  }
  return kDefaultTimeoutNs;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

const char* kind_name(int kind) {
  return kind == kReduceScatter ? "reduce_scatter" : kind == kAllGather ? "all_gather" : "allreduce";
}
const char* proto_name(int proto) { return proto == kLL ? "LL" : proto == kLL128 ? "LL128" : "Simple"; }

// One call's resolved geometry ([C23] "Kernel 如何把 Block 映射到 Channel";
// [C12] "runRing 的数据切分"): grid, block -> channel, per-channel range and
// loops, chunk and slice sizes.
void trace_geometry(int kind, const Geometry& g, uint64_t mask, int nrings, bool direct) {
  std::fprintf(stderr,
               "rar trace: %s nranks=%d count=%lld dtype=%s proto=%s mask=0x%llx grid=%d buff=%lld "
               "step_bytes=%lld chunk_elems=%lld steps_per_slice=%d slices_per_chunk=%d per_channel=%lld "
               "rings=%d direct=%d\n",
               kind_name(kind), g.nranks, (long long)g.count, g.dtype == kF32 ? "f32" : "bf16", proto_name(g.proto),
               (unsigned long long)mask, g.nranks * g.nchan, (long long)g.buff_size, (long long)g.step_bytes,
               (long long)g.chunk_elems, g.sps, g.spc, (long long)g.per_channel, nrings, direct ? 1 : 0);
  int n = 0;
  for (int b = 0; b < kMaxChannels; b++) {
    if (((mask >> b) & 1ull) == 0) continue;
    int64_t go, cc;
    channel_range(g, n, &go, &cc);
    std::fprintf(stderr,
                 "rar trace:   channel %d id %d blocks %d+%d*rank offset %lld count %lld loops %lld first_chunk %lld\n",
                 n, b, n, g.nchan, (long long)go, (long long)cc, (long long)div_up(cc, loop_count(g)),
                 (long long)(cc > 0 ? loop_chunk_count(g, cc) : 0));
    n++;
  }
}

// Ring setup ([C12] "ring index 如何计算"): check that following `next` from
// rank 0 visits every rank once and comes back ("ring does not loop back"),
// then ring_index[r] = (place(r) - place(0) + n) % n.
rar_status setup_ring(int n, const int* ring_order, int* ring_index) {
  if (ring_order == nullptr) return RAR_ERR_ARG;
  int place[kMaxRanks], nxt[kMaxRanks];
  bool seen[kMaxRanks];
  for (int r = 0; r < n; r++) { place[r] = -1; nxt[r] = -1; seen[r] = false; }
  for (int i = 0; i < n; i++) {
    const int r = ring_order[i];
    if (r < 0 || r >= n || place[r] != -1) return RAR_ERR_RING;
    place[r] = i;
    nxt[r] = ring_order[(i + 1) % n];
  }
  int cur = 0;
  for (int i = 0; i < n; i++) {
    if (cur < 0 || seen[cur]) return RAR_ERR_RING;
    seen[cur] = true;
    cur = nxt[cur];
  }
  if (cur != 0) return RAR_ERR_RING;
  for (int r = 0; r < n; r++) ring_index[r] = (place[r] - place[0] + n) % n;
  return RAR_OK;
}

bool overlaps(const void* a, const void* b, int64_t bytes) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + (uintptr_t)bytes && y < x + (uintptr_t)bytes;
}
bool overlaps2(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return abytes > 0 && bbytes > 0 && x < y + (uintptr_t)bbytes && y < x + (uintptr_t)abytes;
}

// Buffers: non-null, 16-byte aligned; a receive buffer may coincide exactly
// with its own rank's send buffer (in place) and must not overlap anything
// else. With allow_in_place false it may not touch any send buffer.
rar_status check_buffers(const void* const* send, void* const* recv, int n, int64_t bytes, bool allow_in_place) {
  if (send == nullptr || recv == nullptr) return RAR_ERR_ARG;
  for (int r = 0; r < n; r++) {
    if (send[r] == nullptr || recv[r] == nullptr) return RAR_ERR_ARG;
    if (!aligned16(send[r]) || !aligned16(recv[r])) return RAR_ERR_ALIGN;
  }
  for (int r = 0; r < n; r++) {
    for (int q = 0; q < n; q++) {
      if (q != r && overlaps(recv[r], recv[q], bytes)) return RAR_ERR_ARG;
      if (overlaps(recv[r], send[q], bytes)) {
        const bool in_place = allow_in_place && q == r && recv[r] == send[r];
        if (!in_place) return RAR_ERR_ARG;
      }
    }
  }
  return RAR_OK;
}

rar_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return RAR_OK;
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();  // the launch was refused; do not leave it sticky
    return RAR_ERR_CORESIDENCY;
  }
  (void)cudaGetLastError();
  return RAR_ERR_CUDA;
}

__global__ void init_staged_header_kernel(char* ws, int nranks, int dtype, int blocks_per_rank, int64_t max_count,
                                          int64_t slot_bytes) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    OsHeader* h = reinterpret_cast<OsHeader*>(ws);
    h->status = 0;
    h->abort = 0;
    h->nranks = nranks;
    h->dtype = dtype;
    h->blocks_per_rank = blocks_per_rank;
    h->max_count = max_count;
    h->slot_bytes = slot_bytes;
    h->err_info = 0;
    h->err_step = 0;
    h->magic = kStagedMagic;
  }
}

cudaError_t device_sms(int* sms) {
  int device = 0;
  return current_device_sms(&device, sms);
}

__global__ void init_header_kernel(char* ws, int nranks, uint64_t mask, int proto, int64_t buff_size) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    WsHeader* h = reinterpret_cast<WsHeader*>(ws);
    h->status = 0;
    h->abort = 0;
    h->nranks = nranks;
    h->mask = mask;
    h->proto = proto;
    h->buff_size = buff_size;
    h->err_info = 0;
    h->err_step = 0;
    h->magic = kMagic;
  }
}

// Buffers of the halves. ReduceScatter: send nranks blocks, recv one;
// AllGather: send one block, recv nranks. All non-null and 16-byte aligned;
// no receive buffer overlaps another one or another rank's send buffer. A
// rank's own pair may overlap only in the in-place shape, where the one-block
// buffer is the rank's own block of the other (ReduceScatter: recv == send +
// rank*block; AllGather: send == recv + rank*block).
rar_status check_half_buffers(int kind, const void* const* send, void* const* recv, int n, int64_t block) {
  if (send == nullptr || recv == nullptr) return RAR_ERR_ARG;
  const int64_t sbytes = kind == kReduceScatter ? n * block : block;
  const int64_t rbytes = kind == kReduceScatter ? block : n * block;
  for (int r = 0; r < n; r++) {
    if (send[r] == nullptr || recv[r] == nullptr) return RAR_ERR_ARG;
    if (!aligned16(send[r]) || !aligned16(recv[r])) return RAR_ERR_ALIGN;
  }
  for (int r = 0; r < n; r++) {
    for (int q = 0; q < n; q++) {
      if (q != r && overlaps2(recv[r], rbytes, recv[q], rbytes)) return RAR_ERR_ARG;
      if (!overlaps2(recv[r], rbytes, send[q], sbytes)) continue;
      const char* own = kind == kReduceScatter ? (const char*)send[r] + r * block : (const char*)recv[r] + r * block;
      const void* one = kind == kReduceScatter ? (const void*)recv[r] : send[r];
      if (q != r || own != one) return RAR_ERR_ARG;
    }
  }
  return RAR_OK;
}

}  // namespace

// Every check of one ring call that does not involve the workspace, in the
// order rar_allreduce reports them (operation, sizes, enums, flags, rings,
// buffers), and the kernel arguments except the workspace fields. Enqueues
// nothing; *grid is 0 for an empty call.
rar_status check_ring_call(int kind, const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                           rar_dtype dtype, rar_redop op, const int* ring_orders, int nrings, uint64_t channelMask,
                           rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags, RingArgs* a,
                           int* grid) {
  if (op != RAR_SUM) return RAR_ERR_ARG;
  if (nranks < 2 || nranks > kMaxRanks) return RAR_ERR_ARG;
  if (count > (size_t)INT64_MAX / 4 / (size_t)nranks) return RAR_ERR_ARG;
  if ((flags & ~(unsigned)RAR_FLAG_DIRECT) != 0) return RAR_ERR_ARG;
  const bool direct = (flags & RAR_FLAG_DIRECT) != 0;
  if (direct && proto != RAR_SIMPLE) return RAR_ERR_ARG;
  // ReduceScatter carries no final value from rank to rank: nothing to write directly
  if (direct && kind == kReduceScatter) return RAR_ERR_ARG;
  Geometry g;
  if (make_geometry(&g, (int)proto, (int)dtype, nranks, channelMask, (int64_t)count, (int64_t)buffSize,
                    chunkSteps, kind) != 0)
    return RAR_ERR_ARG;
  if (nrings != 1 && nrings != g.nchan) return RAR_ERR_ARG;
  if (ring_orders == nullptr) return RAR_ERR_ARG;
  std::memset(a, 0, sizeof *a);
  // one ring for every channel, or one per dense channel ([C12] "GRAPH 重建：N=4")
  for (int ch = 0; ch < g.nchan; ch++) {
    int idx[kMaxRanks];
    const rar_status st = setup_ring(nranks, ring_orders + (nrings == 1 ? 0 : (size_t)ch * nranks), idx);
    if (st != RAR_OK) return st;
    for (int r = 0; r < nranks; r++) {
      a->ring_index[ch * kMaxRanks + r] = (uint8_t)idx[r];
      a->ring_rank[ch * kMaxRanks + idx[r]] = (uint8_t)r;
    }
  }
  const int64_t block = (int64_t)count * g.elem_bytes;
  // LL and LL128 move user data in 8- and 16-byte pieces: the halves' blocks
  // must start on 16-byte boundaries (Simple moves a ragged block elementwise)
  if (kind != kAllReduce && proto != RAR_SIMPLE && block % 16 != 0) return RAR_ERR_ALIGN;
  rar_status st = kind == kAllReduce ? check_buffers(sendbufs, recvbufs, nranks, block, true)
                                     : check_half_buffers(kind, sendbufs, recvbufs, nranks, block);
  if (st != RAR_OK) return st;
  if (trace_on()) trace_geometry(kind, g, channelMask, nrings, direct);
  for (int r = 0; r < nranks; r++) {
    a->send[r] = sendbufs[r];
    a->recv[r] = recvbufs[r];
  }
  a->geo = g;
  a->mask = channelMask;
  a->conn_offset = kHeaderBytes;
  a->fifo_offset = kHeaderBytes + conn_region_bytes(nranks, g.nchan);
  a->timeout_ns = spin_timeout_ns();
  a->fault = g_fault.load(std::memory_order_relaxed);
  a->ll_flag_max = g.proto == kLL ? g_ll_flag_max.load(std::memory_order_relaxed) : 0u;
  a->direct = direct ? 1 : 0;
  *grid = count == 0 ? 0 : nranks * g.nchan;
  return RAR_OK;
}

rar_status launch_ring(const RingArgs& a, int grid, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = (a.geo.proto == kSimple) ? launch_ring_simple(a, grid, s, nullptr)
                                           : launch_ring_line(a, grid, s, nullptr);
  return from_cuda(e);
}

rar_status clear_workspace(void* workspace, int64_t clear_bytes, int nranks, uint64_t channelMask, int proto,
                           int64_t buff_size, void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(workspace, 0, (size_t)clear_bytes, s);
  if (e != cudaSuccess) return from_cuda(e);
  init_header_kernel<<<1, 32, 0, s>>>((char*)workspace, nranks, channelMask, proto, buff_size);
  return from_cuda(cudaGetLastError());
}

namespace {

// One ring collective of any kind: argument checks, ring tables, launch.
rar_status run_ring(int kind, const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                    rar_dtype dtype, rar_redop op, const int* ring_orders, int nrings, uint64_t channelMask,
                    rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags, void* workspace,
                    size_t workspaceBytes, void* stream) {
  RingArgs a;
  int grid = 0;
  rar_status st = check_ring_call(kind, sendbufs, recvbufs, nranks, count, dtype, op, ring_orders, nrings,
                                  channelMask, proto, buffSize, chunkSteps, flags, &a, &grid);
  if (st != RAR_OK) return st;
  if (workspace == nullptr) return RAR_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return RAR_ERR_ALIGN;
  if ((int64_t)workspaceBytes < workspace_bytes_for(nranks, a.geo.nchan, a.geo.buff_size)) return RAR_ERR_WORKSPACE;
  // An empty call enqueues nothing and advances no step counter ([OS89],
  // review of the empty-input case).
  if (grid == 0) return RAR_OK;
  a.ws = (char*)workspace;
  return launch_ring(a, grid, stream);
}

}  // namespace
}  // namespace rar

using namespace rar;

extern "C" {

size_t rar_workspace_bytes(int nranks, uint64_t channelMask, rar_proto proto, size_t buffSize) {
  Geometry g;
  if (make_geometry(&g, (int)proto, kF32, nranks, channelMask, 0, (int64_t)buffSize, 4) != 0) return 0;
  return (size_t)workspace_bytes_for(nranks, g.nchan, g.buff_size);
}

rar_status rar_workspace_init(void* workspace, size_t workspaceBytes, int nranks, uint64_t channelMask,
                              rar_proto proto, size_t buffSize, void* stream) {
  Geometry g;
  if (make_geometry(&g, (int)proto, kF32, nranks, channelMask, 0, (int64_t)buffSize, 4) != 0) return RAR_ERR_ARG;
  if (workspace == nullptr) return RAR_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return RAR_ERR_ALIGN;
  const int64_t need = workspace_bytes_for(nranks, g.nchan, g.buff_size);
  if ((int64_t)workspaceBytes < need) return RAR_ERR_WORKSPACE;
  return clear_workspace(workspace, need, nranks, channelMask, (int)proto, g.buff_size, stream);
}

rar_status rar_allreduce_ex(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                            rar_dtype dtype, rar_redop op, const int* ring_orders, int nrings, uint64_t channelMask,
                            rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags, void* workspace,
                            size_t workspaceBytes, void* stream) {
  return run_ring(kAllReduce, sendbufs, recvbufs, nranks, count, dtype, op, ring_orders, nrings, channelMask, proto,
                  buffSize, chunkSteps, flags, workspace, workspaceBytes, stream);
}

rar_status rar_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t recvcount,
                              rar_dtype dtype, rar_redop op, const int* ring_orders, int nrings,
                              uint64_t channelMask, rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags,
                              void* workspace, size_t workspaceBytes, void* stream) {
  return run_ring(kReduceScatter, sendbufs, recvbufs, nranks, recvcount, dtype, op, ring_orders, nrings, channelMask,
                  proto, buffSize, chunkSteps, flags, workspace, workspaceBytes, stream);
}

rar_status rar_all_gather(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t sendcount,
                          rar_dtype dtype, const int* ring_orders, int nrings, uint64_t channelMask, rar_proto proto,
                          size_t buffSize, int chunkSteps, unsigned flags, void* workspace, size_t workspaceBytes,
                          void* stream) {
  return run_ring(kAllGather, sendbufs, recvbufs, nranks, sendcount, dtype, RAR_SUM, ring_orders, nrings,
                  channelMask, proto, buffSize, chunkSteps, flags, workspace, workspaceBytes, stream);
}

rar_status rar_allreduce(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                         rar_dtype dtype, rar_redop op, const int* ring_order, uint64_t channelMask,
                         rar_proto proto, size_t buffSize, int chunkSteps, void* workspace, size_t workspaceBytes,
                         void* stream) {
  return rar_allreduce_ex(sendbufs, recvbufs, nranks, count, dtype, op, ring_order, 1, channelMask, proto, buffSize,
                          chunkSteps, 0u, workspace, workspaceBytes, stream);
}

rar_status rar_oneshot(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                       rar_dtype dtype, rar_redop op, void* stream) {
  if (op != RAR_SUM) return RAR_ERR_ARG;
  if (nranks < 1 || nranks > kMaxRanks) return RAR_ERR_ARG;
  if (dtype != RAR_F32 && dtype != RAR_BF16) return RAR_ERR_ARG;
  if (count > (size_t)INT64_MAX / 4) return RAR_ERR_ARG;
  const int64_t esz = dtype == RAR_F32 ? 4 : 2;
  rar_status st = check_buffers(sendbufs, recvbufs, nranks, (int64_t)count * esz, false);
  if (st != RAR_OK) return st;
  if (count == 0) return RAR_OK;
  OneShotArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < nranks; r++) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }
  a.nranks = nranks;
  a.dtype = (int)dtype;
  a.count = (int64_t)count;
  return from_cuda(launch_oneshot(a, (cudaStream_t)stream));
}

size_t rar_oneshot_workspace_bytes(int nranks, size_t max_count, rar_dtype dtype) {
  if (nranks < 1 || nranks > kMaxRanks) return 0;
  if (dtype != RAR_F32 && dtype != RAR_BF16) return 0;
  if (max_count == 0 || max_count > (size_t)INT64_MAX / 64 / (size_t)nranks) return 0;
  return (size_t)staged_workspace_bytes(nranks, (int64_t)max_count, dtype == RAR_F32 ? 4 : 2);
}

rar_status rar_oneshot_workspace_init(void* workspace, size_t workspaceBytes, int nranks, size_t max_count,
                                      rar_dtype dtype, void* stream) {
  const size_t need = rar_oneshot_workspace_bytes(nranks, max_count, dtype);
  if (need == 0) return RAR_ERR_ARG;
  if (workspace == nullptr) return RAR_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return RAR_ERR_ALIGN;
  if (workspaceBytes < need) return RAR_ERR_WORKSPACE;
  int sms = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return from_cuda(e);
  cudaStream_t s = (cudaStream_t)stream;
  // header and counters only: a slot's bytes are always written before they are read
  e = cudaMemsetAsync(workspace, 0, (size_t)staged_stage_offset(nranks), s);
  if (e != cudaSuccess) return from_cuda(e);
  const int eb = dtype == RAR_F32 ? 4 : 2;
  init_staged_header_kernel<<<1, 32, 0, s>>>((char*)workspace, nranks, (int)dtype,
                                             staged_blocks_per_rank(nranks, sms), (int64_t)max_count,
                                             staged_slot_bytes((int64_t)max_count, eb));
  return from_cuda(cudaGetLastError());
}

rar_status rar_oneshot_staged(const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                              rar_dtype dtype, rar_redop op, void* workspace, size_t workspaceBytes, void* stream) {
  if (op != RAR_SUM) return RAR_ERR_ARG;
  if (nranks < 1 || nranks > kMaxRanks) return RAR_ERR_ARG;
  if (dtype != RAR_F32 && dtype != RAR_BF16) return RAR_ERR_ARG;
  if (count > (size_t)INT64_MAX / 64 / (size_t)nranks) return RAR_ERR_ARG;
  const int eb = dtype == RAR_F32 ? 4 : 2;
  rar_status st = check_buffers(sendbufs, recvbufs, nranks, (int64_t)count * eb, true);
  if (st != RAR_OK) return st;
  if (workspace == nullptr) return RAR_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return RAR_ERR_ALIGN;
  // An empty call enqueues nothing and advances no sequence number ([OS89],
  // review of the empty-input case).
  if (count == 0) return RAR_OK;
  if ((int64_t)workspaceBytes < staged_workspace_bytes(nranks, (int64_t)count, eb)) return RAR_ERR_WORKSPACE;
  int sms = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return from_cuda(e);
  StagedArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < nranks; r++) {
    a.send[r] = sendbufs[r];
    a.recv[r] = recvbufs[r];
  }
  a.nranks = nranks;
  a.dtype = (int)dtype;
  a.blocks_per_rank = staged_blocks_per_rank(nranks, sms);
  a.fault = g_fault.load(std::memory_order_relaxed);
  a.count = (int64_t)count;
  a.ws = (char*)workspace;
  a.stage_offset = staged_stage_offset(nranks);  // the slot size comes from the workspace header
  a.timeout_ns = spin_timeout_ns();
  return from_cuda(launch_oneshot_staged(a, (cudaStream_t)stream));
}

rar_status rar_get_status(void* workspace, void* stream) {
  if (workspace == nullptr) return RAR_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return from_cuda(e);
  uint32_t status = 0;
  e = cudaMemcpy(&status, (char*)workspace + offsetof(WsHeader, status), sizeof status, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return from_cuda(e);
  if (status != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy((char*)workspace + offsetof(WsHeader, status), &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return (rar_status)status;
}

const char* rar_strerror(rar_status status) {
  switch (status) {
    case RAR_OK: return "success";
    case RAR_ERR_ARG: return "invalid argument";
    case RAR_ERR_RING: return "ring_order is not one ring over all ranks (ring does not loop back)";
    case RAR_ERR_ALIGN: return "buffer or workspace not aligned (16 bytes; workspace 256 bytes)";
    case RAR_ERR_WORKSPACE: return "workspace too small or not initialised for this configuration";
    case RAR_ERR_CORESIDENCY: return "the (rank, channel) blocks cannot all be resident on the GPU at once";
    case RAR_ERR_CUDA: return "a CUDA runtime call failed";
    case RAR_ERR_TIMEOUT: return "a device wait ran past its time limit; the workspace is aborted";
    case RAR_ERR_ABORT: return "the workspace was aborted by an earlier failure; re-initialise it";
    case RAR_ERR_BOUNDS: return "a slice fell outside its buffers (debug library); the workspace is aborted";
  }
  return "unknown status";
}

void rar_set_spin_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns, std::memory_order_relaxed); }

void rar_debug_set_fault(int fault) { g_fault.store(fault, std::memory_order_relaxed); }

rar_status rar_debug_set_ll_flag_wrap(uint32_t flag_max) {
  if (flag_max != 0 && (flag_max < 64 || flag_max > (1u << 31) || (flag_max & (flag_max - 1)) != 0))
    return RAR_ERR_ARG;
  g_ll_flag_max.store(flag_max, std::memory_order_relaxed);
  return RAR_OK;
}

rar_status rar_describe_geometry(int nranks, size_t count, rar_dtype dtype, uint64_t channelMask, rar_proto proto,
                                 size_t buffSize, int chunkSteps, int64_t* out) {
  if (out == nullptr) return RAR_ERR_ARG;
  Geometry g;
  if (make_geometry(&g, (int)proto, (int)dtype, nranks, channelMask, (int64_t)count, (int64_t)buffSize,
                    chunkSteps) != 0)
    return RAR_ERR_ARG;
  const int C = g.nchan;
  out[0] = g.step_bytes;
  out[1] = g.chunk_elems;
  out[2] = g.sps;
  out[3] = g.spc;
  out[4] = C;
  out[5] = g.per_channel;
  int n = 0;
  for (int b = 0; b < kMaxChannels; b++)
    if ((channelMask >> b) & 1ull) out[6 + n++] = b;
  for (int c = 0; c < C; c++) {
    int64_t go, cc;
    channel_range(g, c, &go, &cc);
    out[6 + C + 2 * c] = go;
    out[6 + C + 2 * c + 1] = cc;
    out[6 + 3 * C + c] = div_up(cc, loop_count(g));
  }
  return RAR_OK;
}

}  // extern "C"
