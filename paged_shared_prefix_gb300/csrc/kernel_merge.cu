// kernel_merge.cu -- the device-side token-flat lowering of the block tables,
// the dense-branch dispatch and the bounded-wait self test.  (The log-sum-exp
// merge itself runs inside the prefix and suffix kernels, psp_merge.cuh.)
//
// Expansion: kv_indices[kv_indptr[b] + t] = page[b][t >> s] << s | (t & mask)
// for every context token t, reconstructing request b's block table from its
// group's shared pages and its suffix pages ("The 25% Page-Size Slowdown That
// Wasn't", "Four meanings of page size": B x context_length indices).
#include <cuda_runtime.h>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_sm100.cuh"

namespace psp {
namespace {

using namespace dev;

__global__ void __launch_bounds__(256) expand_kernel(const StepParams p, int32_t* out) {
  const int b = blockIdx.x;
  const int start = p.suffix_start[b];
  const int len = start + p.suffix_len[b];
  const int g = p.req_group[b];
  const int32_t* shared = (start > 0 && g >= 0) ? p.group_page_indices + p.group_page_indptr[g] : nullptr;
  const int32_t* own = p.suffix_page_indices + p.suffix_page_indptr[b];
  const int s = p.page_shift;
  const int mask = (1 << s) - 1;
  int32_t* dst = out + p.kv_indptr[b];
  for (int t = threadIdx.x; t < len; t += blockDim.x) {
    int32_t page;
    if (t < start) {
      page = shared[t >> s];
    } else {
      page = own[(t - start) >> s];
    }
    dst[t] = (page << s) | (t & mask);
  }
}

// Failure-detection self test: waits on an mbarrier that nothing completes,
// with the given poll budget, and must come back with the timeout recorded in
// the status word (site 99) instead of hanging.
__global__ void wait_selftest_kernel(int32_t* status, uint32_t polls) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    sm100::mbar_init(b, 1);
    sm100::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) sm100::mbar_wait_polls(b, 0, status, 99, polls);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* status, uint32_t polls, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, polls);
  return cudaGetLastError();
}

cudaError_t launch_expand_kv_indices(const StepParams& p, int32_t* out, cudaStream_t s) {
  if (p.batch == 0) return cudaSuccess;
  expand_kernel<<<p.batch, 256, 0, s>>>(p, out);
  return cudaGetLastError();
}

cudaError_t launch_prefix_dense(const StepParams& p, int num_items, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  if (p.kv_dtype == PSP_KV_F32) return launch_prefix_simt(p, num_items, true, s);
  if (dense_tc_supported(p)) return launch_prefix_dense_tc(p, num_items, s);
  return launch_prefix_dense_mma(p, num_items, s);
}

}  // namespace psp
