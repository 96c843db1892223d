// psp_suffix_epi.cuh -- the end of one suffix (split, KV head) CTA, shared by the
// suffix kernels: the prefetch of a single-split request's shared-prefix
// partial rows, and the combination of the CTA's partial softmax states into
// either the request's final output (merged with those prefix rows) or a
// normalised partial (O, log2-LSE) that goes through the (request, KV head)
// counter ("GraniKV", section 3: the prefix result is merged with each
// request's suffix attention; the merge itself is in psp_merge.cuh).
#pragma once

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"

namespace psp {
namespace dev {

constexpr int kPreRows = 16;  // prefix partial rows (chunks x query heads) prefetched per single-split request

// The split's descriptor (its first 32 bytes): two 16-byte loads, issued together.
__device__ __forceinline__ SplitDesc load_split_desc(const StepParams& p, int split) {
  const int4* src = reinterpret_cast<const int4*>(p.split_desc + split);
  const int4 a = __ldg(src), b = __ldg(src + 1);
  SplitDesc d;
  d.b = a.x;
  d.t0 = a.y;
  d.t1 = a.z;
  d.list_paged = a.w;
  d.list_flat = b.x;
  d.part0 = b.y;
  d.n_parts = b.z;
  d.one_split = b.w;
  return d;
}

// The same record read again late in a CTA (volatile, so the compiler keeps the first
// read's registers free in between instead of reusing them).
__device__ __forceinline__ SplitDesc reload_split_desc(const StepParams& p, int split) {
  const int4* src = reinterpret_cast<const int4*>(p.split_desc + split);
  int4 a, b;
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];\n" : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w) : "l"(src));
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];\n" : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w) : "l"(src + 1));
  SplitDesc d;
  d.b = a.x;
  d.t0 = a.y;
  d.t1 = a.z;
  d.list_paged = a.w;
  d.list_flat = b.x;
  d.part0 = b.y;
  d.n_parts = b.z;
  d.one_split = b.w;
  return d;
}

// What the end of a suffix CTA needs to know about its request.
struct SuffixCta {
  int split, h, b;
  int part0, n_parts;  // b's prefix parts [part0, part0 + n_parts) (one per chunk of each read-once group)
  bool one_split;      // b has exactly one suffix split
  bool solo;         // one suffix split and the prefix kernels complete before its rows are read
  bool pre_smem;     // solo, and the prefix rows fit the shared-memory prefetch area
  bool wait_prefix;  // dependent launch, sequential form: prefix rows only after the prefix grid
  bool late;         // dependent launch, concurrent form, and the prefix was complete at the start
};

// pre_rows: capacity of the caller's prefix-row prefetch area (at most kPreRows).
__device__ __forceinline__ SuffixCta suffix_cta(const StepParams& p, const SplitDesc& d, int split, int h,
                                                int pre_rows = kPreRows) {
  SuffixCta c;
  c.split = split;
  c.h = h;
  c.b = d.b;
  c.part0 = d.part0;
  c.n_parts = d.n_parts;
  c.one_split = d.one_split != 0;
  c.solo = !p.concurrent && c.one_split;
  c.late = false;
  c.pre_smem = c.solo && c.n_parts > 0 && c.n_parts * p.group <= pre_rows;
  c.wait_prefix = p.pdl && !p.concurrent;
  return c;
}

// The state of a CTA that found its prefix rows complete (suffix_cta_late).
__device__ __forceinline__ void suffix_cta_mark_late(const StepParams& p, SuffixCta& c, int pre_rows) {
  c.late = true;
  c.solo = true;
  c.pre_smem = c.n_parts * p.group <= pre_rows;
}

// Concurrent form: a one-split request whose CTA finds every prefix row done (the prefix
// CTAs count their rows after their partials and arrivals) merges like a solo request of
// the sequential form, from prefetched rows, without its counter.  Called by every thread
// once the CTA's first copies are in flight (the check is a round trip); returns true when
// the caller should prefetch the prefix rows now.
__device__ __forceinline__ bool suffix_cta_late(const StepParams& p, SuffixCta& c, int pre_rows = kPreRows) {
  if (!(p.pdl && p.concurrent && c.one_split && c.n_parts > 0)) return false;
  __shared__ int prefix_complete;
  if (threadIdx.x == 0)
    prefix_complete = *reinterpret_cast<volatile int32_t*>(p.prefix_done) == p.prefix_rows_total;
  __syncthreads();
  if (!prefix_complete) return false;
  __threadfence();  // the prefix partials were fenced before their rows were counted
  suffix_cta_mark_late(p, c, pre_rows);
  return c.pre_smem;
}

// cp.async of b's prefix partial rows of head h into pre_o [part * G + j][D] and
// pre_l [part * G + j], by NT threads numbered tid = 0 .. NT - 1 (the caller commits
// and waits).
template <int D, int NT>
__device__ __forceinline__ void prefetch_prefix_rows(const StepParams& p, const SuffixCta& c, float* pre_o,
                                                     float* pre_l, int tid = threadIdx.x) {
  const int G = p.group;
  constexpr int kRowChunks = D * 4 / 16;
  for (int e = tid; e < c.n_parts * G * (kRowChunks + 1); e += NT) {
    const int ch = e / (G * (kRowChunks + 1));
    const int rem = e - ch * G * (kRowChunks + 1);
    const int j = rem / (kRowChunks + 1);
    const int q = rem - j * (kRowChunks + 1);
    const int2 part = __ldg(p.req_part + c.part0 + ch);
    const int64_t row = static_cast<int64_t>(part.x) + static_cast<int64_t>(c.h) * part.y + j;
    if (q < kRowChunks) {
      cp_async_16(smem_u32(pre_o + (ch * G + j) * D + q * 4), p.o_pre + row * D + q * 4, true);
    } else {
      cp_async_4(smem_u32(pre_l + ch * G + j), p.lse_pre + row);
    }
  }
}

// Combines NSTATE partial softmax states of the CTA's G query heads (red [state][8][D]
// unnormalised outputs, ms [state][8] log2-domain maxima, ls [state][8] sums, all in
// shared memory and complete) and delivers the result.  A single-split request writes
// its final output, merged with its prefix rows when they are in pre_o / pre_l; any
// other writes its normalised partial and arrives on the (b, h) counter, and the
// arrival that completes (b, h) merges it.  Called by all NT threads of the CTA, after
// a __syncthreads() that follows the writes of red / ms / ls (and, for pre_smem, of
// the prefetched rows).
template <int D, int NSTATE, int NT>
__device__ __forceinline__ void suffix_finish(const StepParams& p, const SuffixCta& c, const float* red,
                                              const float* ms, const float* ls, const float* pre_o,
                                              const float* pre_l, float out_scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int b = c.b, h = c.h;
  const bool one_split = c.one_split;
  const bool only_part = one_split && c.n_parts == 0;
  const bool direct = only_part || (c.solo && c.pre_smem);
  // Launched as a dependent of a still running prefix kernel: a one-split request whose
  // prefix partials are all complete (every prefix row counted done) merges them here like
  // a solo request; otherwise its part goes through the (request, KV head) counter.
  bool ready = c.late;
  if (!c.late && p.pdl && p.concurrent && one_split && c.n_parts > 0) {
    __shared__ int prefix_ready;
    if (threadIdx.x == 0) prefix_ready = *reinterpret_cast<volatile int32_t*>(p.prefix_done) == p.prefix_rows_total;
    __syncthreads();
    ready = prefix_ready != 0;
    if (ready) __threadfence();  // the prefix partials were fenced before their rows were counted
  }
  const bool solo_global = (c.solo && !direct) || ready;  // read the prefix partials from global memory
  // the G rows of (b, h) over the CTA's warps, one row per warp at a time
  auto merge_cta_rows = [&](int bb) {
    for (int j0 = warp; j0 < G; j0 += NT / 32) merge_rows<D, 32>(p, bb, h, j0, lane);
  };
  const int64_t row0 = (static_cast<int64_t>(c.split) * p.hkv + h) * G;
  const int64_t orow0 = static_cast<int64_t>(b) * p.hq + h * G;
  // Per row (one thread per query head): the weight of each warp's state in the CTA's own
  // part O_s = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w (times the value scale, log2-LSE
  // M + log2(sum)), and for a direct merge the weights of the prefix chunks and of O_s.
  // The direct merge repeats merge_rows' arithmetic in its order (the own part as it would
  // be written, then the parts weighted by 2^(lse - max), summed by fmaf in the fixed order,
  // times 1 / sum), so a row's result does not depend on which CTA merges it.
  __shared__ float s_coef[NSTATE * 8];  // [warp state][row]
  __shared__ float s_cpre[kPreRows];    // [part * G + row]: 2^(lse_part - max)
  __shared__ float s_own[8], s_inv[8], s_lse[8];
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float mmax = neg_inf();
#pragma unroll
    for (int w = 0; w < NSTATE; ++w) mmax = fmaxf(mmax, ms[w * 8 + g]);
    float sc[NSTATE];
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < NSTATE; ++w) {
      sc[w] = exp2f(ms[w * 8 + g] - mmax);
      sum += ls[w * 8 + g] * sc[w];
    }
    const float f = out_scale / sum;
#pragma unroll
    for (int w = 0; w < NSTATE; ++w) s_coef[w * 8 + g] = sc[w] * f;
    const float lse_own = mmax + log2f(sum);
    if (direct) {
      float big = neg_inf();
      for (int ch = 0; ch < c.n_parts; ++ch) big = fmaxf(big, pre_l[ch * G + g]);
      big = fmaxf(big, lse_own);
      float wsum = 0.f;
      for (int ch = 0; ch < c.n_parts; ++ch) {
        const float w = exp2f(pre_l[ch * G + g] - big);
        s_cpre[ch * G + g] = w;
        wsum += w;
      }
      const float w_own = exp2f(lse_own - big);
      wsum += w_own;
      s_own[g] = w_own;
      s_inv[g] = 1.f / wsum;
      s_lse[g] = big + log2f(wsum);
    } else {
      s_lse[g] = lse_own;
    }
  }
  __syncthreads();
  // every element: a few FMAs over four consecutive d, one vector store
  constexpr int kQuads = D / 4;
  for (int e = threadIdx.x; e < G * kQuads; e += NT) {
    const int g = e / kQuads;
    const int d = (e - g * kQuads) * 4;
    float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float4& acc, float cf, float4 v) {
      acc.x = fmaf(cf, v.x, acc.x);
      acc.y = fmaf(cf, v.y, acc.y);
      acc.z = fmaf(cf, v.z, acc.z);
      acc.w = fmaf(cf, v.w, acc.w);
    };
#pragma unroll
    for (int w = 0; w < NSTATE; ++w)
      add(os, s_coef[w * 8 + g], *reinterpret_cast<const float4*>(red + (w * 8 + g) * D + d));
    if (direct) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int ch = 0; ch < c.n_parts; ++ch)
        add(acc, s_cpre[ch * G + g], *reinterpret_cast<const float4*>(pre_o + (ch * G + g) * D + d));
      add(acc, s_own[g], os);
      const float inv = s_inv[g];
      store_final4(p, orow0 + g, d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
      if (d == 0 && p.lse) p.lse[orow0 + g] = s_lse[g] * 0.6931471805599453f;
      // every prefix arrival on (b, h) was made and nothing else arrives: clear it for the next step
      if (c.late && e == 0) p.counters[static_cast<int64_t>(b) * p.hkv + h] = 0;
    } else {
      *reinterpret_cast<float4*>(p.o_suf + (row0 + g) * D + d) = os;
      if (d == 0) p.lse_suf[row0 + g] = s_lse[g];
    }
  }
  if (!direct) {
    __threadfence();
    __syncthreads();
    if (solo_global) {  // every other part of (b, h) is already complete
      merge_cta_rows(b);
      // every prefix arrival on (b, h) was made and nothing else arrives: clear it for the next step
      if (ready && threadIdx.x == 0) p.counters[static_cast<int64_t>(b) * p.hkv + h] = 0;
    } else {
      __shared__ int last;
      if (threadIdx.x == 0) last = arrive_is_last(p, b, h) ? 1 : 0;
      __syncthreads();
      if (last) merge_cta_rows(b);
    }
  }
}

// End of every suffix CTA.  Launched as a dependent of the prefix kernel and never
// waiting for it (the concurrent form), the grid's last CTA waits for the prefix grid,
// so this grid (and the stream after it) completes only after the prefix kernel; in the
// sequential form every CTA has waited already.  suffix_grid_arrive counts the CTA (thread
// 0, right after its main loop, so that the atomic's round trip overlaps the epilogue) and
// returns whether it was the last; suffix_grid_tail, at the very end, does the last CTA's
// waiting.  A reset of the prefix-row count while other CTAs finish only sends their
// one-split merges through the counter, which is always correct.
__device__ __forceinline__ bool suffix_grid_arrive(const StepParams& p) {
  return p.pdl && p.concurrent && threadIdx.x == 0 && atomicAdd(p.done_ctas, 1) == static_cast<int>(gridDim.x) - 1;
}
__device__ __forceinline__ void suffix_grid_tail(const StepParams& p, bool last) {
  if (!last) return;
  *p.done_ctas = 0;  // ready for the next step (stream-ordered)
  pdl_wait_primary();
  *p.prefix_done = 0;  // every prefix CTA has counted its rows
}

}  // namespace dev
}  // namespace psp
