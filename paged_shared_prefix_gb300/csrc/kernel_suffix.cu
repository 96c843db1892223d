// kernel_suffix.cu -- split-KV paged decode over each request's private suffix.
//
// Persistent warps.  Every (split, KV head) of the plan is one work item; a
// warp takes items in the plan's order (longest split first) from a work
// counter and processes each item alone: all G query heads of the KV head over
// the split's tokens, so every suffix K/V byte is read from HBM exactly once
// per step.  Keys and values are gathered token by token through the block
// table (page granularity 1 << page_shift; at page size 1, or in token-flat
// mode, the list is the per-token kv_indices) with 16-byte cp.async copies into
// the warp's multi-stage shared-memory ring ("The 25% Page-Size Slowdown That
// Wasn't", "When source beats intuition": each token's K/V row is a contiguous
// burst, so only the address generation depends on the page size).  The ring
// runs continuously across items: the next item's query rows and first
// sub-tiles are already in flight while the current item finishes, so item
// boundaries cost no pipeline refill.
//
// Per 16-token sub-tile: scores S^T = K Q^T on mma.sync m16n8k16 (tokens on M,
// the <= 8 query heads on N), online softmax on the accumulator fragments
// (three shuffles per max), P^T turned into the B operand of the value product
// by an in-register 8x8 transpose (movmatrix), O^T += V^T P^T.  fp8-e4m3 codes
// are converted to f16 in registers (exact); the per-head scales fold into the
// score and output scalars.
//
// Item epilogue: the normalised result goes through the just-consumed ring
// stage to coalesced row writes.  A request with one split and no shared
// prefix writes its output; otherwise the warp writes a partial (O, log2-LSE)
// and either merges at once (one split, prefix partials complete because the
// prefix kernel ran earlier on the stream) or adds an arrival on the (request,
// KV head) counter and merges if it completed it (psp_merge.cuh).
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"

namespace psp {
namespace {

using namespace dev;

template <int KV, int D>
struct SufCfg {
  static constexpr int kElem = (KV == PSP_KV_BF16) ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kTileBytes = 16 * kRowBytes;   // one 16-token sub-tile of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
  static constexpr int kMTiles = D / 16;              // m16 tiles of the value product
  static constexpr int kQBytes = 8 * D * 2;           // up to 8 bf16 query rows of one item
  static_assert(kStageBytes >= 8 * D * 4, "a ring stage holds an item's fp32 result rows");
};

struct Item {
  int b, h, t0, t1, nsub;
  const int32_t* list;
  int shift;
};

__device__ __forceinline__ Item describe(const StepParams& p, int id) {
  Item it;
  if (id < 0) {
    it.b = it.h = it.t0 = it.t1 = it.nsub = it.shift = 0;
    it.list = nullptr;
    return it;
  }
  const int code = p.suffix_items[id];
  const int split = code / p.hkv;
  it.h = code - split * p.hkv;
  it.b = p.split_req[split];
  it.t0 = p.split_begin[split];
  it.t1 = p.split_end[split];
  it.nsub = (it.t1 - it.t0 + 15) >> 4;
  if (p.token_flat) {
    it.list = p.kv_indices + p.kv_indptr[it.b] + p.suffix_start[it.b];
    it.shift = 0;
  } else {
    it.list = p.suffix_page_indices + p.suffix_page_indptr[it.b];
    it.shift = p.page_shift;
  }
  return it;
}

template <int KV, int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) suffix_kernel(const StepParams p, int n_items) {
  using C = SufCfg<KV, D>;
  constexpr int kWarpBytes = NST * C::kStageBytes + 2 * C::kQBytes + 64;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  unsigned char* ring = smem + warp * kWarpBytes;
  unsigned char* qbuf = ring + NST * C::kStageBytes;            // [2][8][D] bf16
  float* lse_buf = reinterpret_cast<float*>(qbuf + 2 * C::kQBytes);  // [8]
  const int64_t row_stride = static_cast<int64_t>(p.hkv) * C::kRowBytes;

  // ---- work queue: cur (being consumed), nxt (issued after cur), one fetch in flight
  auto fetch_raw = [&]() -> int { return lane == 0 ? atomicAdd(p.work, 1) : 0; };
  auto settle = [&](int raw) -> int {
    const int v = __shfl_sync(0xffffffffu, raw, 0);
    return v < n_items ? v : -1;
  };
  int cur_id = settle(fetch_raw());
  int nxt_id = settle(fetch_raw());
  int pending = fetch_raw();
  Item cur = describe(p, cur_id);
  Item nxt = describe(p, nxt_id);
  int cur_seq = 0;            // item sequence number of cur (selects its query buffer)
  bool iss_on_next = false;   // issue cursor on nxt instead of cur
  int n_consumed = 0;         // sub-tiles consumed by this warp
  int iss_sub = 0;            // next sub-tile of the item the issue cursor is on
  int n_issued = 0;           // sub-tiles issued by this warp: one cp.async group each

  // The next sub-tile in item order as one cp.async group (with the item's query rows
  // before its first sub-tile); nothing, and no group, when nothing is left to issue.
  // Sub-tile k always lands in ring stage k % NST and is the k-th group of the warp.
  auto issue_one = [&]() {
    if (n_issued - n_consumed >= NST) return;
    if (!iss_on_next && iss_sub >= cur.nsub && nxt_id >= 0) {
      iss_on_next = true;
      iss_sub = 0;
    }
    Item it;
    it.b = iss_on_next ? nxt.b : cur.b;
    it.h = iss_on_next ? nxt.h : cur.h;
    it.t0 = iss_on_next ? nxt.t0 : cur.t0;
    it.t1 = iss_on_next ? nxt.t1 : cur.t1;
    it.nsub = iss_on_next ? nxt.nsub : cur.nsub;
    it.list = iss_on_next ? nxt.list : cur.list;
    it.shift = iss_on_next ? nxt.shift : cur.shift;
    const int seq = iss_on_next ? cur_seq + 1 : cur_seq;
    if ((iss_on_next || cur_id >= 0) && iss_sub < it.nsub) {
      if (iss_sub == 0) {
        // the item's query rows (bf16), zero rows beyond G
        unsigned char* qdst = qbuf + (seq & 1) * C::kQBytes;
        const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(p.q) +
                                    (static_cast<int64_t>(it.b) * p.hq + it.h * G) * D;
        constexpr int kQChunks = 8 * D * 2 / 16;
        for (int e = lane; e < kQChunks; e += 32) {
          const int g = e / (D * 2 / 16);
          cp_async_16(smem_u32(qdst + e * 16), g < G ? qsrc + e * 8 : qsrc, g < G);
        }
      }
      const int tb = it.t0 + iss_sub * 16;
      unsigned char* kdst = ring + (n_issued % NST) * C::kStageBytes;
      const unsigned char* kbase = static_cast<const unsigned char*>(p.k_pool) + static_cast<int64_t>(it.h) * C::kRowBytes;
      const unsigned char* vbase = static_cast<const unsigned char*>(p.v_pool) + static_cast<int64_t>(it.h) * C::kRowBytes;
      constexpr int kRowsPerPass = 32 / C::kChunks;
      const int c = lane % C::kChunks;
#pragma unroll
      for (int k = 0; k < 16 / kRowsPerPass; ++k) {
        const int r = lane / C::kChunks + k * kRowsPerPass;
        const int t = tb + r;
        const bool valid = t < it.t1;
        const int64_t off = valid ? slot_of(it.list, t, it.shift) * row_stride + c * 16 : 0;
        const uint32_t d = smem_u32(kdst + r * C::kRowBytes + swz<C::kChunks>(r, c) * 16);
        cp_async_16(d, kbase + off, valid);
        cp_async_16(d + C::kTileBytes, vbase + off, valid);
      }
      ++iss_sub;
      ++n_issued;
      cp_async_commit();
    }
  };

#pragma unroll 1
  for (int i = 0; i < NST - 1; ++i) issue_one();

  while (cur_id >= 0) {
    // ---- per item: scales, query fragments (after its first sub-tile has landed)
    float score_scale = p.scale_log2;
    float out_scale = 1.f;
    if constexpr (KV == PSP_KV_FP8) {
      score_scale *= __ldg(p.k_scale + cur.h);
      out_scale = __ldg(p.v_scale + cur.h);
    }
    uint32_t qf[D / 16][2];
    float o[C::kMTiles][4];
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = neg_inf(), m1 = neg_inf();  // running max of query heads 2c, 2c+1 (log2 domain)
    float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums

#pragma unroll 1
    for (int cs = 0; cs < cur.nsub; ++cs) {
      cp_async_wait_upto<NST>(n_issued - 1 - n_consumed);  // sub-tile n_consumed has landed
      __syncwarp();
      if (cs == 0) {
        const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(qbuf + (cur_seq & 1) * C::kQBytes) +
                                    (lane >> 2) * D;
        const int qc = lane & 3;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          if constexpr (KV == PSP_KV_BF16) {
            const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow + ks * 16);
            qf[ks][0] = q32[qc];
            qf[ks][1] = q32[4 + qc];
          } else {
            // k-slots (2c, 2c+1) <- d = 4c, 4c+1 and (2c+8, 2c+9) <- d = 4c+2, 4c+3 (matches the
            // byte order the fp8 key fragments arrive in)
            const uint2 v = *reinterpret_cast<const uint2*>(qrow + ks * 16 + 4 * qc);
            qf[ks][0] = pack_f16(bf16_bits_to_float(v.x & 0xffff), bf16_bits_to_float(v.x >> 16));
            qf[ks][1] = pack_f16(bf16_bits_to_float(v.y & 0xffff), bf16_bits_to_float(v.y >> 16));
          }
        }
      }
      const unsigned char* kt = ring + (n_consumed % NST) * C::kStageBytes;
      const unsigned char* vt = kt + C::kTileBytes;
      // ---- S^T (16 tokens x 8 query heads)
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int j = lane >> 3;
        const int row = (lane & 7) + (j & 1) * 8;
        if constexpr (KV == PSP_KV_BF16) {
  #pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t a[4];
            const int ch = 2 * ks + (j >> 1);
            ldsm_x4(a, smem_u32(kt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            mma_bf16(s, a, qf[ks][0], qf[ks][1]);
          }
        } else {
  #pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            uint32_t r[4];
            const int ch = 2 * kk + (j >> 1);
            ldsm_x4(r, smem_u32(kt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            const uint32_t a0[4] = {e4m3x2_to_f16x2(r[0]), e4m3x2_to_f16x2(r[1]), e4m3x2_to_f16x2(r[0] >> 16),
                                    e4m3x2_to_f16x2(r[1] >> 16)};
            const uint32_t a1[4] = {e4m3x2_to_f16x2(r[2]), e4m3x2_to_f16x2(r[3]), e4m3x2_to_f16x2(r[2] >> 16),
                                    e4m3x2_to_f16x2(r[3] >> 16)};
            mma_f16(s, a0, qf[2 * kk][0], qf[2 * kk][1]);
            mma_f16(s, a1, qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
          }
        }
      }

      // ---- online softmax on the fragments: rows = tokens (lane>>2, +8), cols = heads (2c, 2c+1)
      const int tb = cur.t0 + cs * 16;
      const bool v_lo = tb + (lane >> 2) < cur.t1;
      const bool v_hi = tb + (lane >> 2) + 8 < cur.t1;
      const float s0 = v_lo ? s[0] * score_scale : neg_inf();
      const float s1 = v_lo ? s[1] * score_scale : neg_inf();
      const float s2 = v_hi ? s[2] * score_scale : neg_inf();
      const float s3 = v_hi ? s[3] * score_scale : neg_inf();
      const float mx0 = xor_max<4, 16>(fmaxf(s0, s2));
      const float mx1 = xor_max<4, 16>(fmaxf(s1, s3));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
      const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
      const float p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
      l0 = l0 * a0 + p0 + p2;
      l1 = l1 * a1 + p1 + p3;
      m0 = mn0;
      m1 = mn1;
  #pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      uint32_t pb0, pb1;  // P^T as the B operand (k = token, n = query head)
      if constexpr (KV == PSP_KV_BF16) {
        pb0 = movmatrix_t(pack_bf16(p0, p1));
        pb1 = movmatrix_t(pack_bf16(p2, p3));
      } else {
        pb0 = movmatrix_t(pack_f16(p0, p1));
        pb1 = movmatrix_t(pack_f16(p2, p3));
      }

      // ---- O^T += V^T P^T
      {
        const int j = lane >> 3;
        const int row = (lane & 7) + (j >> 1) * 8;
        if constexpr (KV == PSP_KV_BF16) {
  #pragma unroll
          for (int mt = 0; mt < C::kMTiles; ++mt) {
            uint32_t a[4];
            const int ch = 2 * mt + (j & 1);
            ldsm_x4_t(a, smem_u32(vt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            mma_bf16(o[mt], a, pb0, pb1);
          }
        } else {
  #pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[4];
            const int ch = 2 * cc + (j & 1);
            ldsm_x4_t(r, smem_u32(vt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
            // each register: (token 2c: d 2p, 2p+1), (token 2c+1: d 2p, 2p+1); split even / odd d
            const uint32_t ax[4] = {e4m3x2_to_f16x2(__byte_perm(r[0], 0, 0x20)),
                                    e4m3x2_to_f16x2(__byte_perm(r[1], 0, 0x20)),
                                    e4m3x2_to_f16x2(__byte_perm(r[2], 0, 0x20)),
                                    e4m3x2_to_f16x2(__byte_perm(r[3], 0, 0x20))};
            const uint32_t ay[4] = {e4m3x2_to_f16x2(__byte_perm(r[0], 0, 0x31)),
                                    e4m3x2_to_f16x2(__byte_perm(r[1], 0, 0x31)),
                                    e4m3x2_to_f16x2(__byte_perm(r[2], 0, 0x31)),
                                    e4m3x2_to_f16x2(__byte_perm(r[3], 0, 0x31))};
            mma_f16(o[2 * cc], ax, pb0, pb1);
            mma_f16(o[2 * cc + 1], ay, pb0, pb1);
          }
        }
      }

      __syncwarp();
      issue_one();
      ++n_consumed;
    }

    // ---- item epilogue: normalise through the just-consumed stage, write or merge
    {
      float* stage = reinterpret_cast<float*>(ring + ((n_consumed - 1) % NST) * C::kStageBytes);  // [8][D]
      l0 = xor_sum<4, 16>(l0);
      l1 = xor_sum<4, 16>(l1);
      const float inv0 = out_scale / l0, inv1 = out_scale / l1;
      const int c2 = 2 * (lane & 3);
      const int rr = lane >> 2;
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          int d;
          if constexpr (KV == PSP_KV_BF16) {
            d = 16 * mt + 8 * half + rr;
          } else {
            d = 32 * (mt >> 1) + 16 * half + 2 * rr + (mt & 1);
          }
          stage[c2 * D + d] = o[mt][2 * half] * inv0;
          stage[(c2 + 1) * D + d] = o[mt][2 * half + 1] * inv1;
        }
      }
      if (lane < 4) {
        lse_buf[c2] = m0 + log2f(l0);
        lse_buf[c2 + 1] = m1 + log2f(l1);
      }
      __syncwarp();
      const int b = cur.b, h = cur.h;
      const int n_split = p.split_indptr[b + 1] - p.split_indptr[b];
      const bool has_prefix = p.req_group[b] >= 0;
      constexpr int kPer = D / 32;
      if (n_split == 1 && !has_prefix) {
        // the only part of these rows: final output
        const int64_t orow0 = static_cast<int64_t>(b) * p.hq + h * G;
        for (int g = 0; g < G; ++g) {
          const float* src = stage + g * D + lane * kPer;
          if (p.o_dtype == PSP_KV_BF16) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + (orow0 + g) * D + lane * kPer;
            if constexpr (kPer == 4) {
              *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(src[0], src[1]), pack_bf16(src[2], src[3]));
            } else {
              *reinterpret_cast<uint32_t*>(dst) = pack_bf16(src[0], src[1]);
            }
          } else {
            float* dst = static_cast<float*>(p.o) + (orow0 + g) * D + lane * kPer;
#pragma unroll
            for (int k = 0; k < kPer; ++k) dst[k] = src[k];
          }
          if (lane == 0 && p.lse) p.lse[orow0 + g] = lse_buf[g] * 0.6931471805599453f;
        }
      } else {
        // a partial: write it, then merge now (single split with complete prefix partials)
        // or through the (request, KV head) arrival counter
        const int split = p.suffix_items[cur_id] / p.hkv;
        const int64_t row0 = (static_cast<int64_t>(split) * p.hkv + h) * G;
        for (int g = 0; g < G; ++g) {
          const float* src = stage + g * D + lane * kPer;
          float* dst = p.o_suf + (row0 + g) * D + lane * kPer;
          if constexpr (kPer == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(src[0], src[1], src[2], src[3]);
          } else {
            *reinterpret_cast<float2*>(dst) = make_float2(src[0], src[1]);
          }
          if (lane == 0) p.lse_suf[row0 + g] = lse_buf[g];
        }
        __threadfence();
        __syncwarp();
        int merge = 0;
        if (n_split == 1 && !p.concurrent) {
          merge = 1;
        } else {
          merge = lane == 0 ? (arrive_is_last(p, b, h) ? 1 : 0) : 0;
          merge = __shfl_sync(0xffffffffu, merge, 0);
        }
        if (merge)
          for (int g = 0; g < G; ++g) merge_row<D>(p, b, h * G + g, lane);
      }
      __syncwarp();
    }

    // ---- next item (the issue cursor is already on it, or past it)
    cur = nxt;
    cur_id = nxt_id;
    ++cur_seq;
    iss_on_next = false;
    nxt_id = settle(pending);
    nxt = describe(p, nxt_id);
    pending = nxt_id >= 0 ? fetch_raw() : 0;
  }
  cp_async_wait<0>();

  // the last warp to finish resets the work counter for the next step
  __threadfence();
  if (lane == 0) {
    const int total = gridDim.x * NW;
    if (atomicAdd(p.work + 1, 1) == total - 1) {
      p.work[0] = 0;
      p.work[1] = 0;
    }
  }
}

constexpr int kPreRows = 16;  // prefix partial rows (chunks x query heads) prefetched per single-split request

// Per-CTA variant: one CTA per (split, KV head), 4 warps interleaving 16-token sub-tiles.
template <int KV, int D>
struct SufCfgCta {
  static constexpr int kElem = (KV == PSP_KV_BF16) ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kTileBytes = 16 * kRowBytes;   // one 16-token sub-tile of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
  static constexpr int kMTiles = D / 16;              // m16 tiles of the value product
};

template <int KV, int D, int NW, int NST>
__global__ void __launch_bounds__(NW * 32) suffix_cta_kernel(const StepParams p) {
  using C = SufCfgCta<KV, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int b = p.split_req[split];
  const int t0 = p.split_begin[split];
  const int t1 = p.split_end[split];
  const int G = p.group;

  const int32_t* list;
  int shift;
  if (p.token_flat) {
    list = p.kv_indices + p.kv_indptr[b] + p.suffix_start[b];
    shift = 0;
  } else {
    list = p.suffix_page_indices + p.suffix_page_indptr[b];
    shift = p.page_shift;
  }
  const int64_t row_stride = static_cast<int64_t>(p.hkv) * C::kRowBytes;
  const unsigned char* kbase = static_cast<const unsigned char*>(p.k_pool) + static_cast<int64_t>(h) * C::kRowBytes;
  const unsigned char* vbase = static_cast<const unsigned char*>(p.v_pool) + static_cast<int64_t>(h) * C::kRowBytes;
  unsigned char* ring = smem + warp * (NST * C::kStageBytes);

  const int n_sub = (t1 - t0 + 15) >> 4;
  const int my_n = n_sub > warp ? (n_sub - warp + NW - 1) / NW : 0;

  // A request with one suffix split merges its shared-prefix partials here: the prefix
  // kernel ran earlier on the stream, so its rows are complete.  They are prefetched into
  // a shared-memory area of their own, in the first cp.async group of every thread.
  const int g_req = p.req_group[b];
  const bool solo = !p.concurrent && p.split_indptr[b + 1] - p.split_indptr[b] == 1;
  const int c0 = g_req >= 0 ? p.group_chunk_indptr[g_req] : 0;
  const int n_chunks = g_req >= 0 ? p.group_chunk_indptr[g_req + 1] - c0 : 0;
  const bool pre_smem = solo && n_chunks > 0 && n_chunks * G <= kPreRows;
  float* pre_o = reinterpret_cast<float*>(smem + NW * NST * C::kStageBytes);   // [chunk * G + j][D]
  float* pre_l = pre_o + kPreRows * D;                                           // [chunk * G + j]
  if (pre_smem) {
    const int m_eff = p.group_m_eff[g_req];
    const int prow = p.req_member[b] * G;
    constexpr int kRowChunks = D * 4 / 16;
    for (int e = threadIdx.x; e < n_chunks * G * (kRowChunks + 1); e += NW * 32) {
      const int c = e / (G * (kRowChunks + 1));
      const int rem = e - c * G * (kRowChunks + 1);
      const int j = rem / (kRowChunks + 1);
      const int q = rem - j * (kRowChunks + 1);
      const int64_t row = p.chunk_row_offset[c0 + c] + static_cast<int64_t>(h) * m_eff + prow + j;
      if (q < kRowChunks) {
        cp_async_16(smem_u32(pre_o + (c * G + j) * D + q * 4), p.o_pre + row * D + q * 4, true);
      } else {
        cp_async_4(smem_u32(pre_l + c * G + j), p.lse_pre + row);
      }
    }
  }

  // -------- query fragments: B operand of S^T = K Q^T (k = head dim, n = query head)
  const int qg = lane >> 2;  // query head within the group (B fragment column)
  const int qc = lane & 3;
  uint32_t qf[D / 16][2];
  {
    const bool live = qg < G;
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<int64_t>(b) * p.hq + h * G + (live ? qg : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      if constexpr (KV == PSP_KV_BF16) {
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow + ks * 16);
        qf[ks][0] = live ? __ldg(q32 + qc) : 0u;
        qf[ks][1] = live ? __ldg(q32 + 4 + qc) : 0u;
      } else {
        // k-slots (2c, 2c+1) <- d = 4c, 4c+1 and (2c+8, 2c+9) <- d = 4c+2, 4c+3 (matches the
        // byte order the fp8 key fragments arrive in)
        const uint2 v = live ? __ldg(reinterpret_cast<const uint2*>(qrow + ks * 16 + 4 * qc)) : make_uint2(0u, 0u);
        qf[ks][0] = pack_f16(bf16_bits_to_float(v.x & 0xffff), bf16_bits_to_float(v.x >> 16));
        qf[ks][1] = pack_f16(bf16_bits_to_float(v.y & 0xffff), bf16_bits_to_float(v.y >> 16));
      }
    }
  }
  float score_scale = p.scale_log2;
  float out_scale = 1.f;
  if constexpr (KV == PSP_KV_FP8) {
    score_scale *= __ldg(p.k_scale + h);
    out_scale = __ldg(p.v_scale + h);
  }

  // -------- asynchronous gather of one 16-token sub-tile (K and V) into ring stage i % NST
  auto issue = [&](int i) {
    const int tb = t0 + (warp + i * NW) * 16;
    unsigned char* kdst = ring + (i % NST) * C::kStageBytes;
    constexpr int kRowsPerPass = 32 / C::kChunks;
    const int c = lane % C::kChunks;
#pragma unroll
    for (int k = 0; k < 16 / kRowsPerPass; ++k) {
      const int r = lane / C::kChunks + k * kRowsPerPass;
      const int t = tb + r;
      const bool valid = t < t1;
      const int64_t off = valid ? slot_of(list, t, shift) * row_stride + c * 16 : 0;
      const uint32_t d = smem_u32(kdst + r * C::kRowBytes + swz<C::kChunks>(r, c) * 16);
      cp_async_16(d, kbase + off, valid);
      cp_async_16(d + C::kTileBytes, vbase + off, valid);
    }
  };

  float o[C::kMTiles][4];
#pragma unroll
  for (int mt = 0; mt < C::kMTiles; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = neg_inf(), m1 = neg_inf();  // running max of query heads 2c, 2c+1 (log2 domain)
  float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums

#pragma unroll
  for (int i = 0; i < NST - 1; ++i) {
    if (i < my_n) issue(i);
    cp_async_commit();
  }

  for (int i = 0; i < my_n; ++i) {
    cp_async_wait<NST - 2>();
    __syncwarp();
    const unsigned char* kt = ring + (i % NST) * C::kStageBytes;
    const unsigned char* vt = kt + C::kTileBytes;

    // ---- S^T (16 tokens x 8 query heads)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int j = lane >> 3;
      const int row = (lane & 7) + (j & 1) * 8;
      if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          const int ch = 2 * ks + (j >> 1);
          ldsm_x4(a, smem_u32(kt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
          mma_bf16(s, a, qf[ks][0], qf[ks][1]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
          uint32_t r[4];
          const int ch = 2 * kk + (j >> 1);
          ldsm_x4(r, smem_u32(kt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
          const uint32_t a0[4] = {e4m3x2_to_f16x2(r[0]), e4m3x2_to_f16x2(r[1]), e4m3x2_to_f16x2(r[0] >> 16),
                                  e4m3x2_to_f16x2(r[1] >> 16)};
          const uint32_t a1[4] = {e4m3x2_to_f16x2(r[2]), e4m3x2_to_f16x2(r[3]), e4m3x2_to_f16x2(r[2] >> 16),
                                  e4m3x2_to_f16x2(r[3] >> 16)};
          mma_f16(s, a0, qf[2 * kk][0], qf[2 * kk][1]);
          mma_f16(s, a1, qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
        }
      }
    }

    // ---- online softmax on the fragments: rows = tokens (lane>>2, +8), cols = heads (2c, 2c+1)
    const int tb = t0 + (warp + i * NW) * 16;
    const bool v_lo = tb + (lane >> 2) < t1;
    const bool v_hi = tb + (lane >> 2) + 8 < t1;
    const float s0 = v_lo ? s[0] * score_scale : neg_inf();
    const float s1 = v_lo ? s[1] * score_scale : neg_inf();
    const float s2 = v_hi ? s[2] * score_scale : neg_inf();
    const float s3 = v_hi ? s[3] * score_scale : neg_inf();
    const float mx0 = xor_max<4, 16>(fmaxf(s0, s2));
    const float mx1 = xor_max<4, 16>(fmaxf(s1, s3));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
    const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
    const float p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
    l0 = l0 * a0 + p0 + p2;
    l1 = l1 * a1 + p1 + p3;
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
      o[mt][0] *= a0;
      o[mt][1] *= a1;
      o[mt][2] *= a0;
      o[mt][3] *= a1;
    }
    uint32_t pb0, pb1;  // P^T as the B operand (k = token, n = query head)
    if constexpr (KV == PSP_KV_BF16) {
      pb0 = movmatrix_t(pack_bf16(p0, p1));
      pb1 = movmatrix_t(pack_bf16(p2, p3));
    } else {
      pb0 = movmatrix_t(pack_f16(p0, p1));
      pb1 = movmatrix_t(pack_f16(p2, p3));
    }

    // ---- O^T += V^T P^T
    {
      const int j = lane >> 3;
      const int row = (lane & 7) + (j >> 1) * 8;
      if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt) {
          uint32_t a[4];
          const int ch = 2 * mt + (j & 1);
          ldsm_x4_t(a, smem_u32(vt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
          mma_bf16(o[mt], a, pb0, pb1);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[4];
          const int ch = 2 * cc + (j & 1);
          ldsm_x4_t(r, smem_u32(vt + row * C::kRowBytes + swz<C::kChunks>(row, ch) * 16));
          // each register: (token 2c: d 2p, 2p+1), (token 2c+1: d 2p, 2p+1); split even / odd d
          const uint32_t ax[4] = {e4m3x2_to_f16x2(__byte_perm(r[0], 0, 0x20)),
                                  e4m3x2_to_f16x2(__byte_perm(r[1], 0, 0x20)),
                                  e4m3x2_to_f16x2(__byte_perm(r[2], 0, 0x20)),
                                  e4m3x2_to_f16x2(__byte_perm(r[3], 0, 0x20))};
          const uint32_t ay[4] = {e4m3x2_to_f16x2(__byte_perm(r[0], 0, 0x31)),
                                  e4m3x2_to_f16x2(__byte_perm(r[1], 0, 0x31)),
                                  e4m3x2_to_f16x2(__byte_perm(r[2], 0, 0x31)),
                                  e4m3x2_to_f16x2(__byte_perm(r[3], 0, 0x31))};
          mma_f16(o[2 * cc], ax, pb0, pb1);
          mma_f16(o[2 * cc + 1], ay, pb0, pb1);
        }
      }
    }
    __syncwarp();
    const int nx = i + NST - 1;
    if (nx < my_n) issue(nx);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // -------- combine the warps' partial states through shared memory
  l0 = xor_sum<4, 16>(l0);
  l1 = xor_sum<4, 16>(l1);
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [NW][8][D]
  float* ms = red + NW * 8 * D;                 // [NW][8]
  float* ls = ms + NW * 8;                      // [NW][8]
  const int c2 = 2 * (lane & 3);
  if (lane < 4) {
    ms[warp * 8 + c2] = m0;
    ms[warp * 8 + c2 + 1] = m1;
    ls[warp * 8 + c2] = l0;
    ls[warp * 8 + c2 + 1] = l1;
  }
  {
    const int rr = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        int d;
        if constexpr (KV == PSP_KV_BF16) {
          d = 16 * mt + 8 * half + rr;
        } else {
          d = 32 * (mt >> 1) + 16 * half + 2 * rr + (mt & 1);
        }
        red[(warp * 8 + c2) * D + d] = o[mt][2 * half];
        red[(warp * 8 + c2 + 1) * D + d] = o[mt][2 * half + 1];
      }
    }
  }
  __syncthreads();
  // A single-split request writes its final output here: its own result merged with the
  // prefetched prefix partials (none without a shared prefix).  Otherwise write the partial
  // and let the last arrival of (b, h) merge.
  const bool only_part = p.split_indptr[b + 1] - p.split_indptr[b] == 1 && n_chunks == 0;
  const bool direct = only_part || (solo && pre_smem);
  const bool solo_global = solo && !direct;   // too many prefix chunks to prefetch: read them here
  const int64_t row0 = (static_cast<int64_t>(split) * p.hkv + h) * G;
  const int64_t orow0 = static_cast<int64_t>(b) * p.hq + h * G;
  for (int e = threadIdx.x; e < G * D; e += NW * 32) {
    const int g = e / D;
    const int d = e - g * D;
    float mmax = neg_inf();
#pragma unroll
    for (int w = 0; w < NW; ++w) mmax = fmaxf(mmax, ms[w * 8 + g]);
    float acc = 0.f, sum = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sc = exp2f(ms[w * 8 + g] - mmax);
      sum += ls[w * 8 + g] * sc;
      acc += red[(w * 8 + g) * D + d] * sc;
    }
    if (direct) {
      // own part: O_s = acc / sum * out_scale with log2-LSE mmax + log2(sum); prefix chunks first
      float lse_own = mmax + log2f(sum);
      float big = lse_own;
      for (int c = 0; c < n_chunks; ++c) big = fmaxf(big, pre_l[c * G + g]);
      float wsum = 0.f, out = 0.f;
      for (int c = 0; c < n_chunks; ++c) {
        const float w = exp2f(pre_l[c * G + g] - big);
        wsum += w;
        out = fmaf(w, pre_o[(c * G + g) * D + d], out);
      }
      const float w_own = exp2f(lse_own - big);
      wsum += w_own;
      out = fmaf(w_own, acc / sum * out_scale, out);
      store_final(p, orow0 + g, d, out / wsum);
      if (d == 0 && p.lse) p.lse[orow0 + g] = (big + log2f(wsum)) * 0.6931471805599453f;
    } else {
      p.o_suf[(row0 + g) * D + d] = acc / sum * out_scale;
      if (d == 0) p.lse_suf[row0 + g] = mmax + log2f(sum);
    }
  }
  if (direct) return;
  __threadfence();
  __syncthreads();
  if (solo_global) {  // every other part of (b, h) is already complete
    for (int rr = warp; rr < G; rr += NW) merge_row<D>(p, b, h * G + rr, lane);
    return;
  }
  __shared__ int last;
  if (threadIdx.x == 0) last = arrive_is_last(p, b, h) ? 1 : 0;
  __syncthreads();
  if (last)
    for (int rr = warp; rr < G; rr += NW) merge_row<D>(p, b, h * G + rr, lane);
}

template <int KV, int D, int NW, int NST>
cudaError_t launch_cta(const StepParams& p, int num_splits, cudaStream_t s) {
  using C = SufCfgCta<KV, D>;
  const int ring = NW * NST * C::kStageBytes;
  const int epi = (NW * 8 * D + 2 * NW * 8) * 4;
  const int bytes = (ring > epi ? ring : epi) + kPreRows * (D + 1) * 4;
  auto kern = suffix_cta_kernel<KV, D, NW, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(num_splits, p.hkv);
  kern<<<grid, NW * 32, bytes, s>>>(p);
  return cudaGetLastError();
}

int num_sms_of_current_device() {
  static int cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev);
  return cached[dev];
}

template <int KV, int D, int NW, int NST>
cudaError_t launch_t(const StepParams& p, int num_splits, cudaStream_t s) {
  using C = SufCfg<KV, D>;
  const int bytes = NW * (NST * C::kStageBytes + 2 * C::kQBytes + 64);
  auto kern = suffix_kernel<KV, D, NW, NST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NW * 32, bytes);
  if (e != cudaSuccess) return e;
  const int n_items = num_splits * p.hkv;
  const int sms = num_sms_of_current_device();
  int grid = (per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
  const int needed = (n_items + NW - 1) / NW;
  if (grid > needed) grid = needed;
  kern<<<grid, NW * 32, bytes, s>>>(p, n_items);
  return cudaGetLastError();
}

// Ring depth per warp for d = 128 (PSP_SUFFIX_STAGES overrides it for tuning sweeps):
// fewer stages leave room for more resident warps per SM.
int suffix_stages(int fallback) {
  static const int env = [] {
    const char* v = std::getenv("PSP_SUFFIX_STAGES");
    return v ? std::atoi(v) : 0;
  }();
  return env > 0 ? env : fallback;
}

}  // namespace

cudaError_t launch_suffix(const StepParams& p, int num_splits, cudaStream_t s) {
  if (num_splits <= 0) return cudaSuccess;
  static const int impl = [] {
    const char* v = std::getenv("PSP_SUFFIX_IMPL");
    return v ? std::atoi(v) : 1;
  }();
  if (p.kv_dtype == PSP_KV_BF16) {
    if (p.head_dim != 128) return launch_t<PSP_KV_BF16, 64, 4, 4>(p, num_splits, s);
    if (impl == 1) return launch_cta<PSP_KV_BF16, 128, 4, 3>(p, num_splits, s);
    switch (suffix_stages(3)) {
      case 2: return launch_t<PSP_KV_BF16, 128, 4, 2>(p, num_splits, s);
      case 4: return launch_t<PSP_KV_BF16, 128, 4, 4>(p, num_splits, s);
      default: return launch_t<PSP_KV_BF16, 128, 4, 3>(p, num_splits, s);
    }
  }
  if (p.kv_dtype == PSP_KV_FP8) {
    if (p.head_dim != 128) return launch_t<PSP_KV_FP8, 64, 4, 6>(p, num_splits, s);
    if (impl == 1) return launch_cta<PSP_KV_FP8, 128, 4, 3>(p, num_splits, s);
    switch (suffix_stages(3)) {
      case 2: return launch_t<PSP_KV_FP8, 128, 4, 2>(p, num_splits, s);
      case 4: return launch_t<PSP_KV_FP8, 128, 4, 4>(p, num_splits, s);
      case 5: return launch_t<PSP_KV_FP8, 128, 4, 5>(p, num_splits, s);
      default: return launch_t<PSP_KV_FP8, 128, 4, 3>(p, num_splits, s);
    }
  }
  return launch_suffix_simt(p, num_splits, s);
}

}  // namespace psp
