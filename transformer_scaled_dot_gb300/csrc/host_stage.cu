// host_stage.cu -- copy streams and per-workspace events of the host-buffer
// entry points (the ordering rules are in host_stage.h).
//
// State: per device one non-blocking copy stream; a table of workspaces
// (device, base address) with two events each -- `staged` (recorded on the
// copy stream after a call's input copies) and `computed` (recorded on the
// caller's stream after the computation that read them). A workspace seen
// for the first time, or again after its entry was evicted, first gets
// `computed` recorded on the caller's stream, so its first copy waits for
// everything the stream had before it. Streams and events live as long as
// the process: they are never destroyed, so nothing depends on the order of
// static destruction against the CUDA runtime's own teardown.
#include "host_stage.h"

#include <cstdint>

namespace tsd {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kWorkspaceSlots = 64;

struct WorkspaceSlot {
  int device = -1;
  const void* base = nullptr;
  cudaEvent_t staged = nullptr;
  cudaEvent_t computed = nullptr;
  uint64_t last_use = 0;
};

std::mutex g_mutex;
cudaStream_t g_copy_stream[kMaxDevices] = {};
WorkspaceSlot g_slots[kWorkspaceSlots];
uint64_t g_use_clock = 0;

}  // namespace

HostStage::HostStage(const void* workspace, cudaStream_t stream)
    : lock_(g_mutex), stream_(stream) {
  int dev = 0;
  err_ = cudaGetDevice(&dev);
  if (err_ != cudaSuccess) return;
  if (dev < 0 || dev >= kMaxDevices) {
    err_ = cudaErrorInvalidDevice;
    return;
  }
  if (g_copy_stream[dev] == nullptr) {
    err_ = cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking);
    if (err_ != cudaSuccess) {
      g_copy_stream[dev] = nullptr;
      return;
    }
  }
  copy_ = g_copy_stream[dev];
  // the workspace's slot: a hit, else an empty slot, else the least recently used
  WorkspaceSlot* slot = nullptr;
  WorkspaceSlot* victim = &g_slots[0];
  for (WorkspaceSlot& s : g_slots) {
    if (s.device == dev && s.base == workspace) {
      slot = &s;
      break;
    }
    if (s.last_use < victim->last_use) victim = &s;
  }
  bool fresh = false;
  if (slot == nullptr) {
    slot = victim;
    if (slot->staged == nullptr || slot->device != dev) {
      // events belong to the device current at their creation
      cudaEvent_t a = nullptr, b = nullptr;
      err_ = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
      if (err_ == cudaSuccess) err_ = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
      if (err_ != cudaSuccess) return;
      // an evicted slot's events may still be pending in a stream; their
      // destruction is deferred by the runtime until they complete
      if (slot->staged != nullptr) cudaEventDestroy(slot->staged);
      if (slot->computed != nullptr) cudaEventDestroy(slot->computed);
      slot->staged = a;
      slot->computed = b;
    }
    slot->device = dev;
    slot->base = workspace;
    fresh = true;
  }
  slot->last_use = ++g_use_clock;
  staged_ = slot->staged;
  computed_ = slot->computed;
  if (fresh) {
    err_ = cudaEventRecord(computed_, stream_);
    if (err_ != cudaSuccess) return;
  }
  // refill the staging region only after the last computation that read it
  err_ = cudaStreamWaitEvent(copy_, computed_, 0);
}

cudaError_t HostStage::copy_in(void* dst_dev, const void* src_host, size_t bytes) {
  if (err_ != cudaSuccess || bytes == 0) return err_;
  err_ = cudaMemcpyAsync(dst_dev, src_host, bytes, cudaMemcpyHostToDevice, copy_);
  return err_;
}

cudaError_t HostStage::inputs_ready() {
  if (err_ != cudaSuccess) return err_;
  err_ = cudaEventRecord(staged_, copy_);
  if (err_ == cudaSuccess) err_ = cudaStreamWaitEvent(stream_, staged_, 0);
  return err_;
}

cudaError_t HostStage::computed() {
  if (err_ != cudaSuccess) return err_;
  err_ = cudaEventRecord(computed_, stream_);
  return err_;
}

cudaError_t HostStage::copy_out(void* dst_host, const void* src_dev, size_t bytes) {
  if (err_ != cudaSuccess || bytes == 0) return err_;
  err_ = cudaMemcpyAsync(dst_host, src_dev, bytes, cudaMemcpyDeviceToHost, stream_);
  return err_;
}

}  // namespace tsd
