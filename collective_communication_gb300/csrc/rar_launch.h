// rar_launch.h -- host-side launchers of the kernels of librar.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "rar.h"
#include "rar_device.cuh"

namespace rar {

// ---- ring calls (rar_api.cu) ----
// Every check of a ring call that does not involve the workspace (the codes
// and their order are rar_allreduce's) and the kernel arguments except the
// workspace fields; enqueues nothing. *grid is 0 for an empty call.
rar_status check_ring_call(int kind, const void* const* sendbufs, void* const* recvbufs, int nranks, size_t count,
                           rar_dtype dtype, rar_redop op, const int* ring_orders, int nrings, uint64_t channelMask,
                           rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags, RingArgs* a,
                           int* grid);
// The kernel of a checked call (a.ws set) on `stream`.
rar_status launch_ring(const RingArgs& a, int grid, void* stream);
// Zero the first clear_bytes of a ring workspace and write its header for
// this configuration, on `stream`.
rar_status clear_workspace(void* workspace, int64_t clear_bytes, int nranks, uint64_t channelMask, int proto,
                           int64_t buff_size, void* stream);

// Cooperative launch of one block per (rank, channel); grid = nranks * C.
cudaError_t launch_ring_simple(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out);
cudaError_t launch_ring_line(const RingArgs& a, int grid, cudaStream_t stream, int* threads_out);

struct OneShotArgs {
  const void* send[kMaxRanks];
  void* recv[kMaxRanks];
  int nranks;
  int dtype;
  int64_t count;
};
cudaError_t launch_oneshot(const OneShotArgs& a, cudaStream_t stream);

// ---- staged one-shot (oneshot_staged.cu) ----
// Workspace: a 4 KiB header, one OsControl per rank (rounded up to 4 KiB),
// then kStagingSlots slots of slot_bytes per rank.
constexpr uint32_t kStagedMagic = 0x32534152u;  // "RAS2"
constexpr int kStagingSlots = 4;                // slots per rank, reused round-robin
constexpr int kStagedBlocksPerSm = 4;           // grid = nranks * (SMs * 4 / nranks) blocks

struct OsHeader {
  uint32_t magic;
  uint32_t status;  // first device failure (rar_status), 0 if none: same offset as the ring header's
  uint32_t abort;
  int32_t nranks;
  int32_t dtype;
  int32_t blocks_per_rank;
  int64_t max_count;   // elements a slot holds
  int64_t slot_bytes;
  uint64_t err_info;
  uint64_t err_step;
};
static_assert(offsetof(OsHeader, status) == offsetof(WsHeader, status), "status word at one offset");

// Per-rank sequence numbers and counters, each on its own 128-byte line; all
// monotonic across calls.
struct OsControl {
  uint64_t tx_seq;  // calls whose slot this rank has completely written
  uint64_t pad0[15];
  uint64_t ack_seq;  // calls whose slots this rank has completely read
  uint64_t pad1[15];
  uint64_t done;  // blocks that finished copying, over all calls
  uint64_t pad2[15];
  uint64_t read;  // blocks that finished reducing, over all calls
  uint64_t pad3[15];
  uint64_t grab[kStagingSlots];  // reduce chunks handed out in the call using each slot (reset after it)
  uint64_t pad4[16 - kStagingSlots];
};

struct StagedArgs {
  const void* send[kMaxRanks];
  void* recv[kMaxRanks];
  int nranks;
  int dtype;
  int blocks_per_rank;
  int fault;
  int64_t count;
  char* ws;
  int64_t stage_offset;
  uint64_t timeout_ns;
};

inline int64_t staged_slot_bytes(int64_t max_count, int elem_bytes) { return align_up(max_count * elem_bytes, 256); }
inline int64_t staged_stage_offset(int nranks) {
  return kHeaderBytes + align_up((int64_t)nranks * (int64_t)sizeof(OsControl), 4096);
}
inline int64_t staged_workspace_bytes(int nranks, int64_t max_count, int elem_bytes) {
  return staged_stage_offset(nranks) + (int64_t)nranks * kStagingSlots * staged_slot_bytes(max_count, elem_bytes);
}
int staged_blocks_per_rank(int nranks, int sms);

// Host-side tracing: RAR_TRACE set to anything but "0" in the environment
// makes every call print its resolved geometry and kernel to stderr.
bool trace_on();

// The current device and its SM count (cached per device; safe from several
// host threads).
cudaError_t current_device_sms(int* device, int* sms);
// One-time host setup per device (kernel attributes): true once `key` has
// been marked done on `device`; mark_setup_done records it. Setting an
// attribute twice from racing threads is harmless, so no lock is taken.
bool setup_done(int device, int key);
void mark_setup_done(int device, int key);
enum SetupKey : int {
  kSetupSimpleF32 = 0, kSetupSimpleBf16, kSetupBulkLLF32, kSetupBulkLLBf16, kSetupBulkLL128F32, kSetupBulkLL128Bf16,
  kSetupBulkLL128F32Split, kSetupBulkLL128Bf16Split, kSetupSimpleF32Split, kSetupSimpleBf16Split
};
cudaError_t launch_oneshot_staged(const StagedArgs& a, cudaStream_t stream);

}  // namespace rar
