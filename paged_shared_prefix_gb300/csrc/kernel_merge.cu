// kernel_merge.cu -- log-sum-exp merge of the partial results of one decode
// step, and the device-side token-flat lowering of the block tables.
//
// Merge: for each (request b, query head hq) the partial states of the shared
// prefix (one per prefix chunk of b's group, row member*G + j) and of b's
// suffix splits are combined in a fixed order (prefix chunks, then splits):
//   M = max_i lse_i,  w_i = 2^(lse_i - M),  O = sum_i w_i O_i / sum_i w_i,
//   LSE = (M + log2 sum_i w_i) * ln 2
// where every O_i is already normalised and lse_i is its log2 normaliser.
// An empty part has lse = -inf and weight 0.  This is the cascade merge that
// joins the prefix result with each request's suffix attention ("GraniKV",
// section 3); the fixed order makes the result independent of the page size.
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

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const StepParams p) {
  constexpr int kPer = D / 32;  // floats per lane
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.batch * p.hq) return;
  const int b = row / p.hq;
  const int hq = row - b * p.hq;
  const int G = p.group;
  const int h = hq / G;
  const int j = hq - h * G;
  const int g = p.req_group[b];
  int c0 = 0, c1 = 0, m_eff = 0, prow = 0;
  if (g >= 0) {
    c0 = p.group_chunk_indptr[g];
    c1 = p.group_chunk_indptr[g + 1];
    m_eff = p.group_m_eff[g];
    prow = p.req_member[b] * G + j;
  }
  const int s0 = p.split_indptr[b], s1 = p.split_indptr[b + 1];

  float mmax = neg_inf();
  for (int c = c0; c < c1; ++c)
    mmax = fmaxf(mmax, p.lse_pre[p.chunk_row_offset[c] + static_cast<int64_t>(h) * m_eff + prow]);
  for (int s = s0; s < s1; ++s) mmax = fmaxf(mmax, p.lse_suf[(static_cast<int64_t>(s) * p.hkv + h) * G + j]);

  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float sum = 0.f;
  auto add = [&](int64_t r, const float* obuf, const float* lbuf) {
    const float w = exp2f(lbuf[r] - mmax);
    sum += w;
    const float* src = obuf + r * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
    }
  };
  for (int c = c0; c < c1; ++c) add(p.chunk_row_offset[c] + static_cast<int64_t>(h) * m_eff + prow, p.o_pre, p.lse_pre);
  for (int s = s0; s < s1; ++s) add((static_cast<int64_t>(s) * p.hkv + h) * G + j, p.o_suf, p.lse_suf);

  const float inv = 1.f / sum;
  const int64_t obase = static_cast<int64_t>(row) * D + lane * kPer;
  if (p.o_dtype == PSP_KV_BF16) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) + obase;
    if constexpr (kPer == 4) {
      uint2 v;
      v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(o) = v;
    } else {
      *reinterpret_cast<uint32_t*>(o) = pack_bf16(acc[0] * inv, acc[1] * inv);
    }
  } else {
    float* o = static_cast<float*>(p.o) + obase;
#pragma unroll
    for (int k = 0; k < kPer; ++k) o[k] = acc[k] * inv;
  }
  if (p.lse && lane == 0) p.lse[row] = (mmax + log2f(sum)) * 0.6931471805599453f;
}

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

cudaError_t launch_merge(const StepParams& p, cudaStream_t s) {
  const int rows = p.batch * p.hq;
  if (rows == 0) return cudaSuccess;
  dim3 grid((rows + 7) / 8);
  if (p.head_dim == 128) merge_kernel<128><<<grid, 256, 0, s>>>(p);
  else merge_kernel<64><<<grid, 256, 0, s>>>(p);
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
