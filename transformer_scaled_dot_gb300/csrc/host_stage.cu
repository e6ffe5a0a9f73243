// host_stage.cu -- copy streams and per-workspace events of the host-buffer
// entry points (the ordering rules are in host_stage.h).
//
// State: per device one non-blocking copy stream and one result stream; a
// table of workspaces (device, base address) with three events each --
// `staged` (recorded on the copy stream after a call's input copies),
// `computed` (recorded on the caller's stream after the computation that
// read them) and `out_free` (recorded on the result stream after an
// asynchronous result copy read the workspace's result staging). A workspace
// seen for the first time, or again after its entry was evicted, first gets
// `computed` and `out_free` recorded on the caller's stream, after that
// stream has been made to wait for every result copy issued so far on the
// result stream (one of them may still read this workspace from a use before
// its entry was evicted), so its first copy waits for everything the stream
// had before it and its first computation for every earlier result copy.
// Streams and events live as long as
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
  cudaEvent_t out_free = nullptr;  // the last asynchronous result copy has read the staging
  uint64_t last_use = 0;
};

std::mutex g_mutex;
cudaStream_t g_copy_stream[kMaxDevices] = {};
cudaStream_t g_result_stream[kMaxDevices] = {};
cudaEvent_t g_join_event[kMaxDevices] = {};

cudaError_t make_stream(cudaStream_t* s) {
  if (*s != nullptr) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  if (e != cudaSuccess) *s = nullptr;
  return e;
}
WorkspaceSlot g_slots[kWorkspaceSlots];
uint64_t g_use_clock = 0;

// `stream` waits for everything issued so far on the device's result stream.
// Caller holds g_mutex.
cudaError_t join_result_locked(int dev, cudaStream_t stream) {
  if (g_result_stream[dev] == nullptr) return cudaSuccess;  // nothing was ever issued there
  if (g_join_event[dev] == nullptr) {
    cudaError_t e = cudaEventCreateWithFlags(&g_join_event[dev], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      g_join_event[dev] = nullptr;
      return e;
    }
  }
  cudaError_t e = cudaEventRecord(g_join_event[dev], g_result_stream[dev]);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, g_join_event[dev], 0);
  return e;
}

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
  err_ = make_stream(&g_copy_stream[dev]);
  if (err_ == cudaSuccess) err_ = make_stream(&g_result_stream[dev]);
  if (err_ != cudaSuccess) return;
  copy_ = g_copy_stream[dev];
  result_ = g_result_stream[dev];
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
      cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
      for (cudaEvent_t& x : ev)
        if (err_ == cudaSuccess) err_ = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
      if (err_ != cudaSuccess) {
        for (cudaEvent_t x : ev)
          if (x != nullptr) cudaEventDestroy(x);
        return;
      }
      // an evicted slot's events may still be pending in a stream; their
      // destruction is deferred by the runtime until they complete
      if (slot->staged != nullptr) cudaEventDestroy(slot->staged);
      if (slot->computed != nullptr) cudaEventDestroy(slot->computed);
      if (slot->out_free != nullptr) cudaEventDestroy(slot->out_free);
      slot->staged = ev[0];
      slot->computed = ev[1];
      slot->out_free = ev[2];
    }
    slot->device = dev;
    slot->base = workspace;
    fresh = true;
  }
  slot->last_use = ++g_use_clock;
  staged_ = slot->staged;
  computed_ = slot->computed;
  out_free_ = slot->out_free;
  if (fresh) {
    // a result copy from this workspace's earlier use (before its entry was
    // evicted, or under another slot's events) may still be reading its
    // result staging: the caller's stream waits for all of them first
    err_ = join_result_locked(dev, stream_);
    if (err_ == cudaSuccess) err_ = cudaEventRecord(computed_, stream_);
    if (err_ == cudaSuccess) err_ = cudaEventRecord(out_free_, stream_);
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
  // the computation rewrites the result staging: after the last
  // asynchronous copy that read it
  if (err_ == cudaSuccess) err_ = cudaStreamWaitEvent(stream_, out_free_, 0);
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

cudaError_t HostStage::copy_out_async(void* dst_host, const void* src_dev, size_t bytes) {
  if (err_ != cudaSuccess) return err_;
  err_ = cudaStreamWaitEvent(result_, computed_, 0);
  if (err_ == cudaSuccess && bytes != 0)
    err_ = cudaMemcpyAsync(dst_host, src_dev, bytes, cudaMemcpyDeviceToHost, result_);
  if (err_ == cudaSuccess) err_ = cudaEventRecord(out_free_, result_);
  return err_;
}

cudaError_t host_join(cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  return join_result_locked(dev, stream);
}

}  // namespace tsd
