// psp_merge.cuh -- log-sum-exp merge of the partial results of one
// (request, query head) row, performed by whichever CTA delivers the last
// partial of its (request, KV head).
//
// Every (b, h) expects one partial per prefix chunk of each read-once group b
// belongs to (one group, or a path of nested groups) plus one per suffix split
// of b.  A CTA that has written its partials fences them and adds one arrival
// on the (b, h) counter; the CTA that brings the count to the
// expected total merges the G rows of (b, h) and resets the counter to zero
// for the next step.  No CTA ever waits for another.  A request with exactly
// one suffix split skips the counter when the prefix kernels run before the
// suffix kernel on one stream: its suffix CTA merges the (complete) prefix
// partials directly.  With concurrent prefix and suffix kernels every row with
// more than one part goes through its counter.
//
// Merge of a row: with every O_i normalised and lse_i its log2 normaliser,
//   M = max_i lse_i,  w_i = 2^(lse_i - M),  O = sum_i w_i O_i / sum_i w_i,
//   LSE = (M + log2 sum_i w_i) * ln 2,
// in a fixed order (prefix chunks level by level from the outermost, then splits),
// so the result does not depend on which CTA merges ("GraniKV", section 3: the
// prefix result is merged with each request's suffix attention).
#pragma once

#include "psp_device.cuh"
#include "psp_internal.h"

namespace psp {
namespace dev {

// Number of partial results (b, h) receives this step.
__device__ __forceinline__ int expected_parts(const StepParams& p, int b) {
  return p.req_part_indptr[b + 1] - p.req_part_indptr[b] + p.split_indptr[b + 1] - p.split_indptr[b];
}

// One arrival on (b, h) after this CTA's partials for it are written and fenced.
// Returns true for the arrival that completes (b, h).
__device__ __forceinline__ bool arrive_is_last(const StepParams& p, int b, int h) {
  int32_t* cnt = p.counters + static_cast<int64_t>(b) * p.hkv + h;
  const int expected = expected_parts(p, b);
  const int old = atomicAdd(cnt, 1);
  if (old + 1 == expected) {
    __threadfence();   // see every other CTA's partials before reading them
    *cnt = 0;          // ready for the next step (later kernels are stream-ordered)
    return true;
  }
  return false;
}

// Accumulation of one part of a merged row: weight 2^(lse - mmax) times the part's
// D/LANES elements of this lane (row r of obuf / lbuf).
template <int D, int LANES>
struct MergeAcc {
  static constexpr int kPer = D / LANES;           // elements per lane
  static constexpr int kW = kPer % 4 == 0 ? 4 : 2;  // elements per vector access
  static_assert(kPer % kW == 0, "whole vectors per lane");
  float acc[kPer];
  float sum;
  __device__ __forceinline__ MergeAcc() : sum(0.f) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  }
  __device__ __forceinline__ void add(int64_t r, const float* obuf, const float* lbuf, float mmax, int sub) {
    const float w = exp2f(__ldcg(lbuf + r) - mmax);
    sum += w;
    const float* src = obuf + r * D + sub * kPer;
#pragma unroll
    for (int v = 0; v < kPer; v += kW) {
      if constexpr (kW == 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(src + v));
        acc[v] = fmaf(w, x.x, acc[v]);
        acc[v + 1] = fmaf(w, x.y, acc[v + 1]);
        acc[v + 2] = fmaf(w, x.z, acc[v + 2]);
        acc[v + 3] = fmaf(w, x.w, acc[v + 3]);
      } else {
        const float2 x = __ldcg(reinterpret_cast<const float2*>(src + v));
        acc[v] = fmaf(w, x.x, acc[v]);
        acc[v + 1] = fmaf(w, x.y, acc[v + 1]);
      }
    }
  }
  // o and lse of row (b, h * G + j)
  __device__ __forceinline__ void store(const StepParams& p, int b, int h, int j, int sub, float mmax) const {
    const float inv = 1.f / sum;
    const int64_t row = static_cast<int64_t>(b) * p.hq + h * p.group + j;
    const int64_t obase = row * D + sub * kPer;
    if (p.o_dtype == PSP_KV_BF16) {
      uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.o) + obase);
#pragma unroll
      for (int v = 0; v < kPer; v += 2) o[v / 2] = pack_bf16(acc[v] * inv, acc[v + 1] * inv);
    } else {
      float* o = static_cast<float*>(p.o) + obase;
#pragma unroll
      for (int v = 0; v < kPer; ++v) o[v] = acc[v] * inv;
    }
    if (p.lse && sub == 0) p.lse[row] = (mmax + log2f(sum)) * 0.6931471805599453f;
  }
};

// Warp-cooperative merge of rows j0 .. j0 + 32/LANES - 1 (those below G) of (b, h): LANES
// lanes per row, each owning D/LANES consecutive elements, every row at once, and no
// store before the last load, so that the loads of every part of every row can be in
// flight together (a merge costs a few dependent global round trips, not a few per row:
// the request's part list, then its partial rows).  LANES = 4 merges a whole (request,
// KV head) in one warp; more lanes per row use fewer registers per lane.  The prefix
// parts come in plan order (chunks of each read-once group, the outermost group first),
// then the suffix splits.
template <int D, int LANES>
__device__ __forceinline__ void merge_rows(const StepParams& p, int b, int h, int j0, int lane) {
  const int G = p.group;
  const int j = j0 + lane / LANES;
  const int sub = lane % LANES;
  if (j >= G) return;
  const int q0 = p.req_part_indptr[b], q1 = p.req_part_indptr[b + 1];
  const int s0 = p.split_indptr[b], s1 = p.split_indptr[b + 1];
  auto pre_row = [&](int q) {
    const int2 part = __ldg(p.req_part + q);
    return static_cast<int64_t>(part.x) + static_cast<int64_t>(h) * part.y + j;
  };
  float mmax = neg_inf();
  for (int q = q0; q < q1; ++q) mmax = fmaxf(mmax, __ldcg(p.lse_pre + pre_row(q)));
  for (int s = s0; s < s1; ++s) mmax = fmaxf(mmax, __ldcg(p.lse_suf + (static_cast<int64_t>(s) * p.hkv + h) * G + j));
  MergeAcc<D, LANES> a;
  for (int q = q0; q < q1; ++q) a.add(pre_row(q), p.o_pre, p.lse_pre, mmax, sub);
  for (int s = s0; s < s1; ++s) a.add((static_cast<int64_t>(s) * p.hkv + h) * G + j, p.o_suf, p.lse_suf, mmax, sub);
  a.store(p, b, h, j, sub, mmax);
}

// Writes one row's final result directly (the row has exactly one partial).
__device__ __forceinline__ void store_final(const StepParams& p, int64_t row, int d, float value) {
  if (p.o_dtype == PSP_KV_BF16) {
    static_cast<__nv_bfloat16*>(p.o)[row * p.head_dim + d] = __float2bfloat16_rn(value);
  } else {
    static_cast<float*>(p.o)[row * p.head_dim + d] = value;
  }
}

// Writes four consecutive elements (d a multiple of 4) of one row's final result.
__device__ __forceinline__ void store_final4(const StepParams& p, int64_t row, int d, float4 v) {
  const int64_t off = row * p.head_dim + d;
  if (p.o_dtype == PSP_KV_BF16) {
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + off) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(p.o) + off) = v;
  }
}

// Prefix kernels launched ahead of a dependent suffix kernel that does not wait for them
// (the concurrent form): after this CTA's partials and arrivals are complete, count its
// rows as done, so that suffix CTAs can see that the whole prefix is finished.  Called by
// every thread of the CTA.
__device__ __forceinline__ void prefix_rows_done(const StepParams& p, int n_rows) {
  if (!p.pdl || !p.concurrent) return;  // only the concurrent form reads the count
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.prefix_done, n_rows);
  }
}

// Whether member b of a prefix row block must arrive on its (b, h) counter: every
// request does, unless it has exactly one suffix split and the prefix kernels run
// before the suffix kernel (that split then merges the prefix partials itself).
__device__ __forceinline__ bool prefix_member_arrives(const StepParams& p, int b) {
  return p.concurrent || p.split_indptr[b + 1] - p.split_indptr[b] != 1;
}

// Prefix kernels: after this CTA's partial rows [row0, row0 + n) of head h are
// written by the calling warp group, arrive once per member whose G rows all lie
// in the range and merge the members that this arrival completes.  Members with
// exactly one suffix split are skipped: their suffix CTA (a later launch) merges
// the prefix partials itself.  Called by every thread of the CTA after a
// __syncthreads() that follows the writes.  `flags` is shared scratch of at
// least n / G ints.
template <int D>
__device__ __forceinline__ void prefix_arrive_and_merge(const StepParams& p, const int32_t* members, int h, int row0,
                                                        int n, int* flags) {
  const int G = p.group;
  const int n_members = n / G;  // row blocks hold whole members (G divides the block)
  for (int m = threadIdx.x; m < n_members; m += blockDim.x) {
    const int b = members[(row0 / G) + m];
    flags[m] = (prefix_member_arrives(p, b) && arrive_is_last(p, b, h)) ? 1 : 0;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int m = warp; m < n_members; m += nwarps)
    if (flags[m]) merge_rows<D, 32 / kMaxGroupSize>(p, members[(row0 / G) + m], h, 0, lane);
}

// As prefix_arrive_and_merge, with flags[m] (m < n / G) already holding
// prefix_member_arrives() for each member of the block, computed early so that
// the loads are off the kernel's tail.  Called by every thread after a
// __syncthreads() that follows the partial writes (each writer fenced its own).
template <int D>
__device__ __forceinline__ void prefix_arrive_and_merge_flagged(const StepParams& p, const int32_t* members, int h,
                                                                int row0, int n, int* flags) {
  const int G = p.group;
  const int n_members = n / G;
  for (int m = threadIdx.x; m < n_members; m += blockDim.x)
    if (flags[m]) flags[m] = arrive_is_last(p, members[(row0 / G) + m], h) ? 1 : 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int m = warp; m < n_members; m += nwarps)
    if (flags[m]) merge_rows<D, 32 / kMaxGroupSize>(p, members[(row0 / G) + m], h, 0, lane);
}

}  // namespace dev
}  // namespace psp
