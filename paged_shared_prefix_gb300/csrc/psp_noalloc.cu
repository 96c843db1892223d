// psp_noalloc.cu -- a variant of psp_run that allocates nothing.
//
// Some callers cannot allocate device memory at the point where they run a
// decode step: a serving engine that has already reserved nearly all of HBM for
// its KV-cache pool and its weights, a framework plugin or custom-op callback
// whose host framework forbids raw device allocation on that path, or a
// latency-critical loop that cannot afford the device-wide synchronisation an
// allocation may cause.  psp_run_noalloc lets them run the step without a
// caller-allocated workspace: the plan arrays, the partial results and the
// status word live in one file-scope device array of fixed size, and the call
// itself makes no cudaMalloc, cudaFree or other allocating call.
#include <cuda_runtime.h>

#include <mutex>

#include "psp.h"
#include "psp_internal.h"

namespace {

// Size of the static scratch.  Every GPU on which this library's device code is
// loaded holds it for the life of the process.
constexpr size_t kScratchBytes = size_t{64} << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" PSP_API psp_status psp_run_noalloc(psp_handle* h, const psp_tensors* t, void* stream) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return psp::set_error(h, PSP_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices) return psp::set_error(h, PSP_ERR_UNSUPPORTED, "device ordinal above 63");
  unsigned char* scratch = nullptr;
  {
    // once per device, with that device current: the device address of the array
    // (its name in host code is only a host-side stand-in)
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || !p)
        return psp::set_error(h, PSP_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    scratch = g_scratch_ptr[dev];
  }
  return psp::bind_image_and_run(h, scratch, kScratchBytes, t, static_cast<cudaStream_t>(stream));
}
