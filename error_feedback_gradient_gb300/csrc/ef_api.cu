// Host-side common entry points of libefgrad: status strings, last CUDA
// error, device checks, the per-thread profiling hook and the workspace
// status read-back.
#include <cuda_runtime.h>

#include <mutex>

#include "ef_common.cuh"

namespace ef {

namespace {

thread_local int32_t t_last_cuda_error = 0;
thread_local int64_t t_launches = 0;

struct ProfSlot {
  cudaEvent_t start = nullptr;
  cudaEvent_t stop = nullptr;
};
constexpr int kProfSlots = 5;
thread_local ProfSlot t_prof[kProfSlots];

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_known[kMaxDevices] = {false};

}  // namespace

ef_status cuda_fail(cudaError_t err) {
  t_last_cuda_error = (int32_t)err;
  return EF_ERR_CUDA;
}

ef_status check_launch() {
  ++t_launches;
  cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? EF_OK : cuda_fail(err);
}

ef_status current_device(DeviceInfo* out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= kMaxDevices) return EF_ERR_ARCH;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_known[dev]) {
      cudaDeviceProp p;
      err = cudaGetDeviceProperties(&p, dev);
      if (err != cudaSuccess) return cuda_fail(err);
      DeviceInfo d;
      d.sms = p.multiProcessorCount;
      d.major = p.major;
      d.minor = p.minor;
      d.max_smem_optin = p.sharedMemPerBlockOptin;
      g_dev[dev] = d;
      g_dev_known[dev] = true;
    }
    *out = g_dev[dev];
  }
  if (out->major != 10 || out->minor != 3) return EF_ERR_ARCH;
  return EF_OK;
}

void prof_begin(int kernel_id, cudaStream_t s) {
  if (kernel_id > 0 && kernel_id < kProfSlots && t_prof[kernel_id].start)
    cudaEventRecord(t_prof[kernel_id].start, s);
}

void prof_end(int kernel_id, cudaStream_t s) {
  if (kernel_id > 0 && kernel_id < kProfSlots && t_prof[kernel_id].stop)
    cudaEventRecord(t_prof[kernel_id].stop, s);
}

namespace {

// Tile 1 of a fresh state array waits on tile 0, which is never published.
__global__ void selftest_wait_kernel(uint64_t* states, int32_t* status, uint64_t limit_ns) {
  lookback_warp(states, 1, 0, 1, status, limit_ns);
}

}  // namespace
}  // namespace ef

extern "C" {

ef_status ef_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                   void* stream) {
  if (!workspace) return EF_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < 512)
    return EF_ERR_WORKSPACE;
  if (limit_ns < 1000000 || limit_ns > 10000000000ll) return EF_ERR_ARG;
  ef::DeviceInfo dev;
  ef_status st = ef::current_device(&dev);
  if (st != EF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  cudaError_t err = cudaMemsetAsync(ws, 0, 512, s);
  if (err != cudaSuccess) return ef::cuda_fail(err);
  ef::selftest_wait_kernel<<<1, 32, 0, s>>>(reinterpret_cast<uint64_t*>(ws + 256),
                                            reinterpret_cast<int32_t*>(ws),
                                            (uint64_t)limit_ns);
  return ef::check_launch();
}

int32_t ef_abi_version(void) { return EF_ABI_VERSION; }

int32_t ef_last_cuda_error(void) { return ef::t_last_cuda_error; }

int64_t ef_kernel_launches(void) { return ef::t_launches; }

const char* ef_status_string(ef_status s) {
  switch (s) {
    case EF_OK: return "ok";
    case EF_ERR_NULL: return "a required pointer is NULL";
    case EF_ERR_SIZE: return "size out of range";
    case EF_ERR_K: return "k out of range for its segment";
    case EF_ERR_SEGMENTS: return "segment offsets do not rise from 0 to n";
    case EF_ERR_ALIAS: return "an output overlaps another buffer";
    case EF_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case EF_ERR_WORKERS: return "worker count out of range";
    case EF_ERR_ARG: return "invalid argument value";
    case EF_ERR_ALIGN: return "pointer not 4-byte aligned";
    case EF_ERR_ARCH: return "current device is not compute capability 10.3";
    case EF_ERR_CUDA: return "a CUDA call failed";
    case EF_ERR_DEVICE_TIMEOUT: return "device-side bounded wait ran out";
    case EF_ERR_PACKET: return "malformed packet (unsorted, out of range or wrong count)";
    case EF_ERR_INTERNAL: return "device-side consistency check failed";
    case EF_ERR_CAPACITY: return "more elements kept than the packet holds";
    default: return "unknown status";
  }
}

ef_status ef_workspace_status(const void* workspace, void* stream, int32_t* device_status) {
  if (!workspace || !device_status) return EF_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return ef::cuda_fail(err);
  int32_t v = 0;
  err = cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return ef::cuda_fail(err);
  *device_status = v;
  return EF_OK;
}

ef_status ef_profile_events(int32_t kernel_id, void* start_event, void* stop_event) {
  if (kernel_id <= 0 || kernel_id >= ef::kProfSlots) return EF_ERR_ARG;
  if ((start_event == nullptr) != (stop_event == nullptr)) return EF_ERR_NULL;
  ef::t_prof[kernel_id].start = static_cast<cudaEvent_t>(start_event);
  ef::t_prof[kernel_id].stop = static_cast<cudaEvent_t>(stop_event);
  return EF_OK;
}

}  // extern "C"
