// kernel_prefix_cascade.cu -- shared-prefix attention for the stacked queries
// of a prefix group, small-M tiled loop ("GraniKV", section 3: below the
// dispatcher threshold the prefix runs as a tiled cascade loop and is merged
// with the suffix).
//
// The M_eff = members x G queries of one KV head are stacked as rows
// R = member * G + j (query head h*G + j of the member-th request).  One CTA
// takes NW*16 consecutive rows and one chunk of the shared prefix; every
// 64-token K/V tile of the chunk is staged once in shared memory (16-byte
// cp.async gathers through the group's page list, multi-stage) and used by all
// NW warps, so the prefix is read once per row block instead of once per
// request.  Each warp runs the FlashAttention-2 register pipeline on its 16
// rows: S = Q K^T (m16n8k16, fp32 accumulate), online softmax with quad
// shuffles, O += P V with P taken straight from the score fragments.  fp8-e4m3
// tiles are converted to f16 in registers; their scales fold into the score
// and output scalars.  Output: one normalised fp32 partial (O, log2-LSE) per
// (chunk, head, row).
#include <cuda_runtime.h>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"

namespace psp {
namespace {

using namespace dev;

constexpr int kTile = 64;  // tokens per staged tile

template <int KV, int D>
struct PreCfg {
  static constexpr int kElem = (KV == PSP_KV_BF16) ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kTileBytes = kTile * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOTiles = D / 8;  // n8 tiles of the value product
};

template <int KV, int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) prefix_cascade_kernel(const StepParams p, const int32_t* item_chunk,
                                                                 const int32_t* item_rb, int ctas_per_item) {
  using C = PreCfg<KV, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // an item's row block may span several CTAs of NW * 16 rows each
  pdl_launch_dependents();  // the step's suffix kernel may start filling free SMs
  const int h = blockIdx.x % p.hkv;  // KV head fastest (neighbouring heads' rows are adjacent)
  const int cta = blockIdx.x / p.hkv;
  const int item = cta / ctas_per_item;
  const int ci = item_chunk[item];
  const int rb = item_rb[item] * ctas_per_item + (cta - item * ctas_per_item);
  const int g = p.chunk_group[ci];
  const int t0 = p.chunk_begin[ci];
  const int t1 = p.chunk_end[ci];
  const int G = p.group;
  const int m_eff = p.group_m_eff[g];
  const int32_t* members = p.group_members + p.group_member_indptr[g];

  const int32_t* list;
  int shift;
  if (p.token_flat) {
    list = p.kv_indices + p.kv_indptr[members[0]];
    shift = 0;
  } else {
    list = p.group_page_indices + p.group_page_indptr[g];
    shift = p.page_shift;
  }
  const int64_t row_stride = static_cast<int64_t>(p.hkv) * C::kRowBytes;
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k_pool) + static_cast<int64_t>(h) * C::kRowBytes;
  const unsigned char* vbase = static_cast<const unsigned char*>(p.v_pool) + static_cast<int64_t>(h) * C::kRowBytes;

  // -------- query fragments (A operand, rows r and r+8 of this warp's 16)
  const int rr = lane >> 2;
  const int qc = lane & 3;
  const int row_lo = rb * NW * 16 + warp * 16 + rr;
  const int row_hi = row_lo + 8;
  uint32_t qa[D / 16][4];
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    auto qrow = [&](int R) -> const __nv_bfloat16* {
      const int mem = R / G, j = R - mem * G;
      return q + (static_cast<int64_t>(members[mem]) * p.hq + h * G + j) * D;
    };
    const bool lo_ok = row_lo < m_eff, hi_ok = row_hi < m_eff;
    const __nv_bfloat16* qlo = lo_ok ? qrow(row_lo) : q;
    const __nv_bfloat16* qhi = hi_ok ? qrow(row_hi) : q;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if constexpr (KV == PSP_KV_BF16) {
        const uint32_t* l32 = reinterpret_cast<const uint32_t*>(qlo + ks * 16);
        const uint32_t* h32 = reinterpret_cast<const uint32_t*>(qhi + ks * 16);
        qa[ks][0] = lo_ok ? __ldg(l32 + qc) : 0u;
        qa[ks][1] = hi_ok ? __ldg(h32 + qc) : 0u;
        qa[ks][2] = lo_ok ? __ldg(l32 + 4 + qc) : 0u;
        qa[ks][3] = hi_ok ? __ldg(h32 + 4 + qc) : 0u;
      } else {
        // k-slot permutation matching the fp8 key fragments: (2c,2c+1) <- d 4c,4c+1; (2c+8,2c+9) <- 4c+2,4c+3
        const uint2 vl = lo_ok ? __ldg(reinterpret_cast<const uint2*>(qlo + ks * 16 + 4 * qc)) : make_uint2(0u, 0u);
        const uint2 vh = hi_ok ? __ldg(reinterpret_cast<const uint2*>(qhi + ks * 16 + 4 * qc)) : make_uint2(0u, 0u);
        qa[ks][0] = pack_f16(bf16_bits_to_float(vl.x & 0xffff), bf16_bits_to_float(vl.x >> 16));
        qa[ks][1] = pack_f16(bf16_bits_to_float(vh.x & 0xffff), bf16_bits_to_float(vh.x >> 16));
        qa[ks][2] = pack_f16(bf16_bits_to_float(vl.y & 0xffff), bf16_bits_to_float(vl.y >> 16));
        qa[ks][3] = pack_f16(bf16_bits_to_float(vh.y & 0xffff), bf16_bits_to_float(vh.y >> 16));
      }
    }
  }
  float score_scale = p.scale_log2;
  float out_scale = 1.f;
  if constexpr (KV == PSP_KV_FP8) {
    score_scale *= __ldg(p.k_scale + h);
    out_scale = __ldg(p.v_scale + h);
  }

  const int n_tiles = (t1 - t0 + kTile - 1) / kTile;
  auto issue = [&](int i) {
    const int tb = t0 + i * kTile;
    unsigned char* kdst = smem + (i % NST) * C::kStageBytes;
    constexpr int kChunksTotal = kTile * C::kChunks;
    constexpr int kIters = (kChunksTotal + NW * 32 - 1) / (NW * 32);
    // all block-table lookups first (independent loads in flight together), then the
    // copies: a lookup issued between copies (asm with a memory clobber) would wait alone
    int64_t off[kIters];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int e = threadIdx.x + it * NW * 32;
      const int r = e / C::kChunks;
      const int t = tb + r;
      off[it] = (e < kChunksTotal && t < t1) ? slot_of(list, t, shift) * row_stride + (e - r * C::kChunks) * 16 : -1;
    }
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const int e = threadIdx.x + it * NW * 32;
      if (e >= kChunksTotal) break;
      const int r = e / C::kChunks;
      const int c = e - r * C::kChunks;
      const bool valid = off[it] >= 0;
      const uint32_t d = smem_u32(kdst + r * C::kRowBytes + swz<C::kChunks>(r, c) * 16);
      cp_async_16(d, kbase + (valid ? off[it] : 0), valid);
      cp_async_16(d + C::kTileBytes, vbase + (valid ? off[it] : 0), valid);
    }
  };

  float o[C::kOTiles][4];
#pragma unroll
  for (int t = 0; t < C::kOTiles; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m_lo = neg_inf(), m_hi = neg_inf(), l_lo = 0.f, l_hi = 0.f;

#pragma unroll
  for (int i = 0; i < NST - 1; ++i) {
    if (i < n_tiles) issue(i);
    cp_async_commit();
  }
  for (int i = 0; i < n_tiles; ++i) {
    cp_async_wait<NST - 2>();
    __syncthreads();
    const unsigned char* kt = smem + (i % NST) * C::kStageBytes;
    const unsigned char* vt = kt + C::kTileBytes;

    // ---- S = Q K^T : 16 rows x 64 tokens (8 n-tiles)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    {
      const int j = lane >> 3;
      if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
          for (int np = 0; np < 4; ++np) {  // pairs of n-tiles
            const int row = 16 * np + (j >> 1) * 8 + (lane & 7);
            const int ch = 2 * ks + (j & 1);
            uint32_t b[4];
            ldsm_x4(b, smem_u32(kt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            mma_bf16(s[2 * np], qa[ks], b[0], b[1]);
            mma_bf16(s[2 * np + 1], qa[ks], b[2], b[3]);
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
          for (int nq = 0; nq < 2; ++nq) {  // quads of n-tiles
            const int row = 32 * nq + j * 8 + (lane & 7);
            uint32_t b[4];
            ldsm_x4(b, smem_u32(kt + row * C::kRowBytes + swz<C::kChunks>(row, ks) * 16));
#pragma unroll
            for (int u = 0; u < 4; ++u)
              mma_f16(s[4 * nq + u], qa[ks], e4m3x2_to_f16x2(b[u]), e4m3x2_to_f16x2(b[u] >> 16));
          }
        }
      }
    }

    // ---- online softmax (rows lane>>2 and +8; columns 2c, 2c+1 of each n-tile)
    const int tb = t0 + i * kTile;
    float mx_lo = neg_inf(), mx_hi = neg_inf();
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int t = tb + 8 * nt + 2 * qc;
      const bool v0 = t < t1, v1 = t + 1 < t1;
      s[nt][0] = v0 ? s[nt][0] * score_scale : neg_inf();
      s[nt][1] = v1 ? s[nt][1] * score_scale : neg_inf();
      s[nt][2] = v0 ? s[nt][2] * score_scale : neg_inf();
      s[nt][3] = v1 ? s[nt][3] * score_scale : neg_inf();
      mx_lo = fmaxf(mx_lo, fmaxf(s[nt][0], s[nt][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(s[nt][2], s[nt][3]));
    }
    mx_lo = xor_max<1, 2>(mx_lo);
    mx_hi = xor_max<1, 2>(mx_hi);
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float a_lo = exp2f(m_lo - mn_lo), a_hi = exp2f(m_hi - mn_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    l_lo *= a_lo;
    l_hi *= a_hi;
#pragma unroll
    for (int t = 0; t < C::kOTiles; ++t) {
      o[t][0] *= a_lo;
      o[t][1] *= a_lo;
      o[t][2] *= a_hi;
      o[t][3] *= a_hi;
    }
    uint32_t pa[4][4];  // P as A fragments, one per 16-token k-step
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = exp2f(s[nt][0] - mn_lo), p1 = exp2f(s[nt][1] - mn_lo);
      const float p2 = exp2f(s[nt][2] - mn_hi), p3 = exp2f(s[nt][3] - mn_hi);
      l_lo += p0 + p1;
      l_hi += p2 + p3;
      const int kk = nt >> 1, hi = nt & 1;
      if constexpr (KV == PSP_KV_BF16) {
        pa[kk][2 * hi] = pack_bf16(p0, p1);
        pa[kk][2 * hi + 1] = pack_bf16(p2, p3);
      } else {
        pa[kk][2 * hi] = pack_f16(p0, p1);
        pa[kk][2 * hi + 1] = pack_f16(p2, p3);
      }
    }

    // ---- O += P V
    {
      const int j = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int row = 16 * kk + (j & 1) * 8 + (lane & 7);
        if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
          for (int np = 0; np < C::kOTiles / 2; ++np) {
            const int ch = 2 * np + (j >> 1);
            uint32_t b[4];
            ldsm_x4_t(b, smem_u32(vt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            mma_bf16(o[2 * np], pa[kk], b[0], b[1]);
            mma_bf16(o[2 * np + 1], pa[kk], b[2], b[3]);
          }
        } else {
#pragma unroll
          for (int qp = 0; qp < C::kChunks / 2; ++qp) {
            const int ch = 2 * qp + (j >> 1);
            uint32_t b[4];
            ldsm_x4_t(b, smem_u32(vt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            // b[0]: tokens 0-7 chunk 2qp, b[1]: tokens 8-15 chunk 2qp, b[2]/b[3]: chunk 2qp+1
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t x_lo = e4m3x2_to_f16x2(__byte_perm(b[2 * u], 0, 0x20));
              const uint32_t x_hi = e4m3x2_to_f16x2(__byte_perm(b[2 * u + 1], 0, 0x20));
              const uint32_t y_lo = e4m3x2_to_f16x2(__byte_perm(b[2 * u], 0, 0x31));
              const uint32_t y_hi = e4m3x2_to_f16x2(__byte_perm(b[2 * u + 1], 0, 0x31));
              mma_f16(o[2 * (2 * qp + u)], pa[kk], x_lo, x_hi);
              mma_f16(o[2 * (2 * qp + u) + 1], pa[kk], y_lo, y_hi);
            }
          }
        }
      }
    }
    __syncthreads();
    const int nx = i + NST - 1;
    if (nx < n_tiles) issue(nx);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // -------- normalise and write this warp's rows
  l_lo = xor_sum<1, 2>(l_lo);
  l_hi = xor_sum<1, 2>(l_hi);
  const int64_t base = p.chunk_row_offset[ci] + static_cast<int64_t>(h) * m_eff;
  const float inv_lo = out_scale / l_lo, inv_hi = out_scale / l_hi;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int R = half ? row_hi : row_lo;
    if (R >= m_eff) continue;
    const float inv = half ? inv_hi : inv_lo;
    float* orow = p.o_pre + (base + R) * D;
    if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
      for (int t = 0; t < C::kOTiles; ++t)
        *reinterpret_cast<float2*>(orow + 8 * t + 2 * qc) = make_float2(o[t][2 * half] * inv, o[t][2 * half + 1] * inv);
    } else {
#pragma unroll
      for (int q = 0; q < C::kChunks; ++q)  // tiles X (even d) and Y (odd d) of 16-code chunk q
        *reinterpret_cast<float4*>(orow + 16 * q + 4 * qc) =
            make_float4(o[2 * q][2 * half] * inv, o[2 * q + 1][2 * half] * inv, o[2 * q][2 * half + 1] * inv,
                        o[2 * q + 1][2 * half + 1] * inv);
    }
    if (qc == 0) p.lse_pre[base + R] = (half ? m_hi : m_lo) + log2f(half ? l_hi : l_lo);
  }
  // arrive for every member of this row block; the arrival that completes a member merges it
  __threadfence();
  __syncthreads();
  const int row0 = rb * NW * 16;
  prefix_arrive_and_merge<D>(p, members, h, row0, min(NW * 16, m_eff - row0), reinterpret_cast<int*>(smem));
  prefix_rows_done(p, min(NW * 16, m_eff - row0));
}

template <int KV, int D, int NW, int NST>
cudaError_t launch_t(const StepParams& p, const int32_t* chunks, const int32_t* rbs, int n, int per_item,
                     cudaStream_t s) {
  using C = PreCfg<KV, D>;
  const int bytes = NST * C::kStageBytes;
  auto kern = prefix_cascade_kernel<KV, D, NW, NST>;
  cudaError_t e = ensure_smem_limit<prefix_cascade_kernel<KV, D, NW, NST>>(bytes);
  if (e != cudaSuccess) return e;
  const int grid = n * per_item * p.hkv;
  kern<<<grid, NW * 32, bytes, s>>>(p, chunks, rbs, per_item);
  return cudaGetLastError();
}

template <int NW>
cudaError_t launch_rows(const StepParams& p, const int32_t* chunks, const int32_t* rbs, int n, int per_item,
                        cudaStream_t s) {
  if (p.kv_dtype == PSP_KV_BF16)
    return p.head_dim == 128 ? launch_t<PSP_KV_BF16, 128, NW, 3>(p, chunks, rbs, n, per_item, s)
                             : launch_t<PSP_KV_BF16, 64, NW, 4>(p, chunks, rbs, n, per_item, s);
  return p.head_dim == 128 ? launch_t<PSP_KV_FP8, 128, NW, 4>(p, chunks, rbs, n, per_item, s)
                           : launch_t<PSP_KV_FP8, 64, NW, 4>(p, chunks, rbs, n, per_item, s);
}

}  // namespace

cudaError_t launch_prefix_cascade(const StepParams& p, int num_items, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  if (p.kv_dtype == PSP_KV_F32) return launch_prefix_simt(p, num_items, false, s);
  return launch_rows<kCascadeRows / 16>(p, p.item_chunk_cascade, p.item_rb_cascade, num_items, 1, s);
}

// Dense branch with the same register pipeline (head_dim 64): each 256-row item as
// two CTAs of 128 rows (8 warps).
cudaError_t launch_prefix_dense_mma(const StepParams& p, int num_items, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  return launch_rows<8>(p, p.item_chunk_dense, p.item_rb_dense, num_items, kDenseRows / 128, s);
}

}  // namespace psp
