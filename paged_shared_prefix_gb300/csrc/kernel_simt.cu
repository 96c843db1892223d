// kernel_simt.cu -- fp32 K/V path of the step (CUDA-core FMA, fp32 throughout).
//
// Used for fp32 caches only, where tensor-core inputs would round the keys and
// values.  One kernel serves both work kinds: a suffix item is (split, KV head)
// over the G query heads of one request; a prefix item is (chunk, row block,
// KV head) over stacked group rows.  The CTA stages 32-token K/V tiles in
// shared memory through the page list; each warp owns one query row at a
// time (lane = token for the scores, lane = head-dim slice for the values) and
// keeps an online-softmax state.  Output: the same normalised fp32 partial
// (O, log2-LSE) rows as the tensor-core kernels.
#include <cuda_runtime.h>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"

namespace psp {
namespace {

using namespace dev;

constexpr int kWarps = 8;
constexpr int kTok = 32;

template <int D>
__global__ void __launch_bounds__(kWarps * 32) simt_kernel(const StepParams p, int mode, const int32_t* item_chunk,
                                                           const int32_t* item_rb, int rows_per_block) {
  __shared__ float ks[kTok][D + 1];
  __shared__ float vs[kTok][D];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (mode == 1) pdl_launch_dependents();  // prefix items: the suffix kernel may start early
  const int h = blockIdx.x % p.hkv;  // KV head fastest (neighbouring heads' rows are adjacent)
  const int item = blockIdx.x / p.hkv;
  const int G = p.group;
  const float* kpool = static_cast<const float*>(p.k_pool);
  const float* vpool = static_cast<const float*>(p.v_pool);
  const float* q = static_cast<const float*>(p.q);

  // ---- work item: token list, token range, rows
  const int32_t* list;
  int shift, t0, t1, n_rows, m_eff = 0, b_suffix = 0;
  int64_t out_base;
  const int32_t* members = nullptr;
  int row0 = 0;
  if (mode == 0) {  // suffix split
    const int split = item;
    b_suffix = p.split_req[split];
    t0 = p.split_begin[split];
    t1 = p.split_end[split];
    if (p.token_flat) {
      list = p.kv_indices + p.kv_indptr[b_suffix] + p.suffix_start[b_suffix];
      shift = 0;
    } else {
      list = p.suffix_page_indices + p.suffix_page_indptr[b_suffix];
      shift = p.page_shift;
    }
    n_rows = G;
    out_base = (static_cast<int64_t>(split) * p.hkv + h) * G;
  } else {  // prefix chunk x row block
    const int ci = item_chunk[item];
    const int g = p.chunk_group[ci];
    t0 = p.chunk_begin[ci];
    t1 = p.chunk_end[ci];
    m_eff = p.group_m_eff[g];
    members = p.group_members + p.group_member_indptr[g];
    if (p.token_flat) {
      list = p.kv_indices + p.kv_indptr[members[0]];
      shift = 0;
    } else {
      list = p.group_page_indices + p.group_page_indptr[g];
      shift = p.page_shift;
    }
    row0 = item_rb[item] * rows_per_block;
    n_rows = min(rows_per_block, m_eff - row0);
    out_base = p.chunk_row_offset[ci] + static_cast<int64_t>(h) * m_eff + row0;
  }
  const int64_t row_stride = static_cast<int64_t>(p.hkv) * D;
  constexpr int kPer = D / 32;
  // a request with a single partial (no shared prefix, one split) writes its output directly;
  // a single-split request of a prefix group merges after its write (the prefix kernel ran earlier)
  const bool one_split = mode == 0 && p.split_indptr[b_suffix + 1] - p.split_indptr[b_suffix] == 1;
  const bool direct = one_split && p.req_group[b_suffix] < 0;
  const bool solo = one_split && !p.concurrent;

  for (int rbase = 0; rbase < n_rows; rbase += kWarps) {
    const int r = rbase + warp;
    const bool live = r < n_rows;
    // query row of this warp (staged in shared memory for the score loop)
    const float* qrow = q;
    if (live) {
      if (mode == 0) {
        qrow = q + (static_cast<int64_t>(b_suffix) * p.hq + h * G + r) * D;
      } else {
        const int R = row0 + r, mem = R / G, j = R - mem * G;
        qrow = q + (static_cast<int64_t>(members[mem]) * p.hq + h * G + j) * D;
      }
    }
    __shared__ float qs[kWarps][D];
#pragma unroll
    for (int k = 0; k < kPer; ++k) qs[warp][lane + 32 * k] = live ? qrow[lane + 32 * k] : 0.f;
    float m = neg_inf(), l = 0.f;
    float acc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = 0.f;

    for (int tb = t0; tb < t1; tb += kTok) {
      __syncthreads();  // previous tile fully consumed
      for (int e = threadIdx.x; e < kTok * D; e += kWarps * 32) {
        const int tt = e / D, dd = e - tt * D;
        const int t = tb + tt;
        float kx = 0.f, vx = 0.f;
        if (t < t1) {
          const int64_t off = slot_of(list, t, shift) * row_stride + static_cast<int64_t>(h) * D + dd;
          kx = kpool[off];
          vx = vpool[off];
        }
        ks[tt][dd] = kx;
        vs[tt][dd] = vx;
      }
      __syncthreads();
      if (!live) continue;
      // lane = token: score
      const int t = tb + lane;
      float sc = 0.f;
#pragma unroll 8
      for (int dd = 0; dd < D; ++dd) sc = fmaf(qs[warp][dd], ks[lane][dd], sc);
      sc = (t < t1) ? sc * p.scale_log2 : neg_inf();
      float mx = sc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(m, mx);
      const float alpha = exp2f(m - mn);
      const float pr = exp2f(sc - mn);
      float ps = pr;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l = l * alpha + ps;
      m = mn;
#pragma unroll
      for (int k = 0; k < kPer; ++k) acc[k] *= alpha;
      for (int tt = 0; tt < kTok; ++tt) {
        const float pt = __shfl_sync(0xffffffffu, pr, tt);
#pragma unroll
        for (int k = 0; k < kPer; ++k) acc[k] = fmaf(pt, vs[tt][lane + 32 * k], acc[k]);
      }
    }
    if (live && direct) {
      const int64_t orow = static_cast<int64_t>(b_suffix) * p.hq + h * G + r;
#pragma unroll
      for (int k = 0; k < kPer; ++k) store_final(p, orow, lane + 32 * k, acc[k] / l);
      if (lane == 0 && p.lse) p.lse[orow] = (m + log2f(l)) * 0.6931471805599453f;
    } else if (live) {
      float* orow = (mode == 0 ? p.o_suf : p.o_pre) + (out_base + r) * D;
#pragma unroll
      for (int k = 0; k < kPer; ++k) orow[lane + 32 * k] = acc[k] / l;
      if (lane == 0) (mode == 0 ? p.lse_suf : p.lse_pre)[out_base + r] = m + log2f(l);
    }
  }
  if (direct) return;
  // arrive once per (request, KV head) this CTA contributed to; the completing arrival merges
  __threadfence();
  __syncthreads();
  __shared__ int flags[kDenseRows];  // one per member of a row block (G >= 1)
  if (mode == 0) {
    if (threadIdx.x == 0) flags[0] = (solo || arrive_is_last(p, b_suffix, h)) ? 1 : 0;
    __syncthreads();
    if (flags[0])
      for (int j0 = warp; j0 < G; j0 += kWarps) merge_rows<D, 32>(p, b_suffix, h, j0, lane);
  } else {
    prefix_arrive_and_merge<D>(p, members, h, row0, n_rows, flags);
    prefix_rows_done(p, n_rows);
  }
}

cudaError_t launch_simt(const StepParams& p, int mode, int n, const int32_t* chunks, const int32_t* rbs, int rows,
                        cudaStream_t s) {
  const int grid = n * p.hkv;
  if (p.head_dim == 128) {
    simt_kernel<128><<<grid, kWarps * 32, 0, s>>>(p, mode, chunks, rbs, rows);
  } else {
    simt_kernel<64><<<grid, kWarps * 32, 0, s>>>(p, mode, chunks, rbs, rows);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_suffix_simt(const StepParams& p, int num_splits, cudaStream_t s) {
  if (num_splits <= 0) return cudaSuccess;
  return launch_simt(p, 0, num_splits, nullptr, nullptr, 0, s);
}

cudaError_t launch_prefix_simt(const StepParams& p, int num_items, bool dense, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  return dense ? launch_simt(p, 1, num_items, p.item_chunk_dense, p.item_rb_dense, kDenseRows, s)
               : launch_simt(p, 1, num_items, p.item_chunk_cascade, p.item_rb_cascade, kCascadeRows, s);
}

}  // namespace psp
