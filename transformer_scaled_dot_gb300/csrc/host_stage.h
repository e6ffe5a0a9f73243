// host_stage.h -- the runtime behind the host-buffer entry points (internal).
//
// A host-staged call copies its inputs from host memory into a staging region
// of the caller's device workspace, runs the device entry point on the staged
// copies, and copies the result back to host memory. The host-to-device copies
// run on a library-owned copy stream (one per device, created on first use),
// ordered only after the last computation that read the same workspace's
// staging region; the computation and the copy back run on the caller's
// stream. So a caller that alternates two workspaces over consecutive calls
// gets call i+1's input copy overlapped with call i's computation and result
// copy, while every call stays ordered on its stream: once the stream has
// passed a call, its result is in host memory. The asynchronous variant
// copies the result on a library-owned result stream instead, so that it
// also overlaps the next call's computation; the result is in host memory
// once the stream has passed a later host_join. A workspace's next
// computation waits for the result copy that last read its staging region.
#pragma once

#include <cstddef>
#include <mutex>

#include <cuda_runtime.h>

namespace tsd {

class HostStage {
 public:
  // Takes the library-wide lock for the call's enqueue (a few microseconds):
  // the per-workspace events are shared state.
  HostStage(const void* workspace, cudaStream_t stream);
  HostStage(const HostStage&) = delete;
  HostStage& operator=(const HostStage&) = delete;

  cudaError_t status() const { return err_; }
  // host -> device on the copy stream (nothing for 0 bytes)
  cudaError_t copy_in(void* dst_dev, const void* src_host, size_t bytes);
  // the caller's stream waits for every copy_in so far
  cudaError_t inputs_ready();
  // marks the point on the caller's stream after which the workspace's
  // staged inputs are no longer read (the next call may refill them)
  cudaError_t computed();
  // device -> host on the caller's stream
  cudaError_t copy_out(void* dst_host, const void* src_dev, size_t bytes);
  // device -> host on the library's result stream (after the computation):
  // it overlaps the next call's computation; host_join orders it
  cudaError_t copy_out_async(void* dst_host, const void* src_dev, size_t bytes);

 private:
  std::unique_lock<std::mutex> lock_;
  cudaStream_t stream_ = nullptr;
  cudaStream_t copy_ = nullptr;
  cudaStream_t result_ = nullptr;
  cudaEvent_t staged_ = nullptr;
  cudaEvent_t computed_ = nullptr;
  cudaEvent_t out_free_ = nullptr;
  cudaError_t err_ = cudaSuccess;
};

// `stream` waits for every result copy issued so far (copy_out_async) on
// the current device.
cudaError_t host_join(cudaStream_t stream);

}  // namespace tsd
