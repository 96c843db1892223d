// kernel_suffix.cu -- split-KV paged decode over each request's private suffix.
//
// One CTA per (split, KV head).  The CTA serves all G query heads of its KV
// head, so every suffix K/V byte is read from HBM exactly once per step.
// Keys and values are gathered token by token through the block table (page
// granularity 1 << page_shift; at page size 1, or in token-flat mode, the
// list is the per-token kv_indices) with 16-byte cp.async copies into a
// per-warp multi-stage shared-memory ring ("The 25% Page-Size Slowdown That
// Wasn't", "When source beats intuition": each token's K/V row is a contiguous
// burst, so only the address generation depends on the page size).
//
// Each warp owns 16-token sub-tiles w, w+NW, ... of the split.  Scores are the
// tensor-core product S^T = K Q^T (m16n8k16, tokens on M, the <= 8 query
// heads on N), the online softmax runs on the accumulator fragments with a
// three-step shuffle max per tile, P^T is turned into the B operand of the
// second product by an in-register 8x8 transpose (movmatrix), and the value
// product is O^T = V^T P^T.  fp8-e4m3 keys/values enter both products as
// e4m3 mma.sync operands (m16n8k32, two sub-tiles per iteration, the query
// rows and P quantised to e4m3); the per-head scales fold into the score and
// output scalars.  The warps' partial states are combined through shared memory and
// written as one normalised fp32 partial (O, log2-LSE) per (split, head, q).
#include <cuda_runtime.h>

#include <cstdlib>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"
#include "psp_suffix_epi.cuh"

namespace psp {
namespace {

using namespace dev;

constexpr int kTablePrefetch = 8;  // sub-tiles (per warp) between a table prefetch and its use

template <int KV, int D>
struct SufCfg {
  static constexpr int kElem = (KV == PSP_KV_BF16) ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunks = kRowBytes / 16;
  static constexpr int kTileBytes = 16 * kRowBytes;   // one 16-token sub-tile of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
  static constexpr int kMTiles = D / 16;              // m16 tiles of the value product
  // prefix-row prefetch area: kPreRows rows, or one prefix chunk of <= 8 heads where the
  // 16-row area would keep a 3-stage e4m3 ring (48 KB) from four resident CTAs per SM
  template <int NST>
  __host__ __device__ static constexpr int pre_rows() { return (KV == PSP_KV_FP8 && D == 128 && NST == 3) ? 8 : kPreRows; }
  // resident CTAs per SM the register allocation must allow: four for that e4m3 ring (128
  // registers a thread), three for the 2-stage bf16 ring (170; shared memory allows three),
  // otherwise whatever the compiler chooses
  template <int NST>
  __host__ __device__ static constexpr int min_ctas() { return (KV == PSP_KV_FP8 && D == 128 && NST == 3) ? 4 : (KV == PSP_KV_BF16 && D == 128 && NST == 2) ? 3 : 1; }
};

// PT (page tiles): the block table is paged with pages of >= 16 tokens, so each 16-token
// sub-tile lies in one page; a sub-tile then costs one table entry and one address
// computation, its rows following at a fixed stride.  Otherwise (page size < 16, or the
// token-flat kv_indices) every row is looked up on its own.
template <int KV, int D, int NW, int NST, bool PT>
__global__ void __launch_bounds__(NW * 32, SufCfg<KV, D>::template min_ctas<NST>()) suffix_kernel(const StepParams p) {
  using C = SufCfg<KV, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // one-dimensional grid, KV head fastest: the Hkv CTAs of a split run side by side, so
  // the heads' rows of each token (adjacent in the pool) are read at about the same time
  const int h = blockIdx.x % p.hkv;
  const int split = blockIdx.x / p.hkv;
  const SplitDesc sd = load_split_desc(p, split);
  // page size >= 16: a 16-token sub-tile lies in one page, and the pages of the split's first
  // sub-tiles sit in its descriptor, loaded beside it, so the ring's first copies wait for no
  // block-table load
  const bool desc_pages = !p.token_flat && p.page_shift >= 4;
  int32_t first_pg[NST];
#pragma unroll
  for (int i = 0; i < NST; ++i) {
    const int st = warp + i * NW;
    first_pg[i] = (desc_pages && st < kDescPages) ? __ldg(p.split_desc[split].first_page + st) : -1;
  }
  const int b = sd.b;
  const int t0 = sd.t0;
  const int t1 = sd.t1;
  const int G = p.group;

  const int32_t* list;
  int shift;
  if (p.token_flat) {
    list = p.kv_indices + sd.list_flat;
    shift = 0;
  } else {
    list = p.suffix_page_indices + sd.list_paged;
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
  // a shared-memory area of their own, in the first cp.async group of every thread (a
  // dependent launch that keeps the sequential protocol reads them only after the prefix
  // grid has completed, below, after this CTA's own stream; one in the concurrent form
  // prefetches them once its first copies are in flight if the prefix is complete by then).
  constexpr int kPre = C::template pre_rows<NST>();
  SuffixCta cta = suffix_cta(p, sd, split, h, kPre);
  float* pre_o = reinterpret_cast<float*>(smem + NW * NST * C::kStageBytes);   // [chunk * G + j][D]
  float* pre_l = pre_o + kPre * D;                                               // [chunk * G + j]
  if (cta.pre_smem && !cta.wait_prefix) prefetch_prefix_rows<D, NW * 32>(p, cta, pre_o, pre_l);

  // -------- query fragments: B operand of S^T = K Q^T (k = head dim, n = query head)
  const int qg = lane >> 2;  // query head within the group (B fragment column)
  const int qc = lane & 3;
  // bf16: m16n8k16 fragments (two bf16 per register).  fp8: m16n8k32 e4m3 fragments (four
  // codes per register: d = 32kk + 4c .. 4c+3 and 32kk + 16 + 4c .. +3), the query row
  // quantised to e4m3 with its own scale amax/448, folded into the score scale below.
  constexpr int kQFrag = (KV == PSP_KV_BF16) ? D / 16 : D / 32;
  uint32_t qf[kQFrag][2];
  float q_scale = 1.f;  // fp8: this lane's query head's scale
  {
    const bool live = qg < G;
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<int64_t>(b) * p.hq + h * G + (live ? qg : 0)) * D;
    if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow + ks * 16);
        qf[ks][0] = live ? __ldg(q32 + qc) : 0u;
        qf[ks][1] = live ? __ldg(q32 + 4 + qc) : 0u;
      }
    } else {
      uint2 v[kQFrag][2];
#pragma unroll
      for (int kk = 0; kk < kQFrag; ++kk)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          v[kk][hf] = live ? __ldg(reinterpret_cast<const uint2*>(qrow + kk * 32 + hf * 16 + 4 * qc)) : make_uint2(0u, 0u);
      float amax = 0.f;
#pragma unroll
      for (int kk = 0; kk < kQFrag; ++kk)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t w[2] = {v[kk][hf].x, v[kk][hf].y};
#pragma unroll
          for (int e = 0; e < 2; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[e] & 0xffff)), fabsf(bf16_bits_to_float(w[e] >> 16))));
        }
      amax = xor_max<1, 2>(amax);  // the four lanes of this query head
      q_scale = amax > 0.f ? amax / 448.f : 1.f;
      const float inv = 1.f / q_scale;
#pragma unroll
      for (int kk = 0; kk < kQFrag; ++kk)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const uint2 w = v[kk][hf];
          qf[kk][hf] = e4m3x4_from_floats(bf16_bits_to_float(w.x & 0xffff) * inv, bf16_bits_to_float(w.x >> 16) * inv,
                                          bf16_bits_to_float(w.y & 0xffff) * inv, bf16_bits_to_float(w.y >> 16) * inv);
        }
    }
  }
  float score_scale = p.scale_log2;  // per accumulator column below (sc0: head 2c, sc1: head 2c+1)
  float out_scale = 1.f;
  if constexpr (KV == PSP_KV_FP8) {
    score_scale *= __ldg(p.k_scale + h);
    out_scale = __ldg(p.v_scale + h);
  }
  float sc0 = score_scale, sc1 = score_scale;
  if constexpr (KV == PSP_KV_FP8) {
    sc0 *= __shfl_sync(0xffffffffu, q_scale, 8 * qc);      // lanes 4n.. hold query head n
    sc1 *= __shfl_sync(0xffffffffu, q_scale, 8 * qc + 4);
  }

  // -------- asynchronous gather of one 16-token sub-tile (K and V) into ring stage i % NST
  // (the callers keep the stage index, so no division by a ring depth of 3 runs per copy).
  // The block-table entries of a sub-tile's rows are loaded one iteration ahead of its
  // copies (load_pages), so no copy waits on a dependent table load: the copies are
  // asm statements with a memory clobber, which keeps the compiler from hoisting the
  // next row's table load above the previous row's copy.
  constexpr int kRowsPerPass = 32 / C::kChunks;
  constexpr int kRowIters = 16 / kRowsPerPass;
  constexpr int kPgSlots = PT ? 1 : kRowIters;  // table entries a lane holds per sub-tile
  const int mask = (1 << shift) - 1;
  // page tiles: this lane's first source bytes (its row within a pass, its 16-byte chunk)
  const unsigned char* klane = nullptr;
  const unsigned char* vlane = nullptr;
  if constexpr (PT) {
    const int64_t lane_off = static_cast<int64_t>(lane / C::kChunks) * row_stride + (lane % C::kChunks) * 16;
    klane = kbase + lane_off;
    vlane = vbase + lane_off;
  }
  auto load_pages = [&](int i, int32_t (&pg)[kPgSlots]) {
    const int tb = t0 + (warp + i * NW) * 16;
    if constexpr (PT) {
      pg[0] = __ldg(list + (tb >> shift));  // callers pass only sub-tiles of the split (tb < t1)
    } else {
#pragma unroll
      for (int k = 0; k < kRowIters; ++k) {
        const int t = tb + lane / C::kChunks + k * kRowsPerPass;
        pg[k] = t < t1 ? __ldg(list + (t >> shift)) : -1;
      }
    }
  };
  // the same for the ring's first NST sub-tiles, from the descriptor where it holds them
  auto load_first_pages = [&](int i, int32_t (&pg)[kPgSlots]) {
    if (desc_pages && warp + i * NW < kDescPages) {
      if constexpr (PT) {
        pg[0] = first_pg[i];
      } else {
        const int tb = t0 + (warp + i * NW) * 16;
#pragma unroll
        for (int k = 0; k < kRowIters; ++k) pg[k] = tb + lane / C::kChunks + k * kRowsPerPass < t1 ? first_pg[i] : -1;
      }
    } else {
      load_pages(i, pg);
    }
  };
  auto issue = [&](int i, int stage, const int32_t (&pg)[kPgSlots]) {
    const int tb = t0 + (warp + i * NW) * 16;
    unsigned char* kdst = ring + stage * C::kStageBytes;
    const int c = lane % C::kChunks;
    if constexpr (PT) {
      // one page holds the whole sub-tile: its first row, then kRowsPerPass rows per pass
      const int64_t base = ((static_cast<int64_t>(pg[0]) << shift) | (tb & mask)) * row_stride;
      const unsigned char* ks = klane + base;
      const unsigned char* vs = vlane + base;
      const int64_t pass = static_cast<int64_t>(kRowsPerPass) * row_stride;
#pragma unroll
      for (int k = 0; k < kRowIters; ++k) {
        const int r = lane / C::kChunks + k * kRowsPerPass;
        const bool valid = tb + r < t1;
        const uint32_t d = smem_u32(kdst + r * C::kRowBytes + swz<C::kChunks>(r, c) * 16);
        cp_async_16(d, valid ? ks + k * pass : ks, valid);
        cp_async_16(d + C::kTileBytes, valid ? vs + k * pass : vs, valid);
      }
    } else {
#pragma unroll
      for (int k = 0; k < kRowIters; ++k) {
        const int r = lane / C::kChunks + k * kRowsPerPass;
        const bool valid = pg[k] >= 0;
        const int64_t slot = (static_cast<int64_t>(pg[k]) << shift) | ((tb + r) & mask);
        const int64_t off = valid ? slot * row_stride + c * 16 : 0;
        const uint32_t d = smem_u32(kdst + r * C::kRowBytes + swz<C::kChunks>(r, c) * 16);
        cp_async_16(d, kbase + off, valid);
        cp_async_16(d + C::kTileBytes, vbase + off, valid);
      }
    }
  };

  float o[C::kMTiles][4];
#pragma unroll
  for (int mt = 0; mt < C::kMTiles; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = neg_inf(), m1 = neg_inf();  // running max of query heads 2c, 2c+1 (log2 domain)
  float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums

  // Sub-tiles per iteration: bf16 takes one; fp8 takes two, so that the value product runs
  // as e4m3 mma.sync with k = 32 tokens (m16n8k32) and the code needs no conversion of its own
  // (on sm_103a the instruction itself unpacks the codes to f16 for the tensor cores).
  constexpr int U = (KV == PSP_KV_FP8) ? 2 : 1;
  static_assert(NST >= U + 1, "the ring holds the sub-tiles of one iteration and at least one in flight");
  // fp8: the running max is kept 8 below the true max, so P <= 2^8 (inside e4m3's range and
  // clear of its subnormals); l carries the same factor, so O / l and m + log2(l) are exact.
  constexpr float kPShift = (KV == PSP_KV_FP8) ? 8.f : 0.f;

  // Ring schedule: sub-tiles 0 .. NST-1 are issued before the loop (one cp.async group each).
  // Each iteration waits for its own U sub-tiles and refills their stages, with the sub-tiles
  // NST further on, as soon as their fragments are in registers (after the score products),
  // so every sub-tile is issued an iteration or more before it is needed (a refill at the top
  // of the next iteration would leave the second of an e4m3 iteration's sub-tiles only a
  // moment to arrive).  The block-table entries of a sub-tile are loaded one iteration
  // before its copies, so no copy waits on a dependent table load.
  int32_t pages[U][kPgSlots];
#pragma unroll
  for (int i = 0; i < NST; ++i) {
    if (i < my_n) {
      load_first_pages(i, pages[0]);
      issue(i, i, pages[0]);
    }
    cp_async_commit();
  }
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (NST + u < my_n) load_pages(NST + u, pages[u]);
  // Concurrent form: the check of the prefix rows (a round trip and a CTA barrier) comes
  // after every first copy is in flight; a late CTA's prefix rows join the next cp.async
  // group, which the loop waits for one iteration later than its first sub-tiles.
  if (suffix_cta_late(p, cta, kPre)) prefetch_prefix_rows<D, NW * 32>(p, cta, pre_o, pre_l);
  // e4m3: only the late flag is carried through the loop, the rest of the CTA's request
  // state is read again after it (registers are that kernel's limit; bf16 keeps it)
  const bool late = cta.late;

  // ring stage of sub-tile i0 (i0 % NST, kept as a running index)
  auto wrap = [](int x) { return x >= NST ? x - NST : x; };  // x < 2 * NST
  int st0 = 0;
  for (int i0 = 0; i0 < my_n; i0 += U, st0 = wrap(st0 + U)) {
    // refill the stages of sub-tiles i0 + u with the sub-tiles NST further on
    auto refill = [&]() {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int nx = i0 + NST + u;
        if (nx < my_n) issue(nx, wrap(st0 + u), pages[u]);
        cp_async_commit();
        if (nx + U < my_n) load_pages(nx + U, pages[u]);  // in flight while this iteration computes
        // the block-table entries of a sub-tile kTablePrefetch iterations later, pulled into L2
        // now: at small page sizes every sub-tile reads its own 64 bytes of the table, and a
        // DRAM round trip taken only one iteration ahead of the copies would stall them
        const int pf = nx + U + kTablePrefetch;
        if (lane == 0 && pf < my_n) prefetch_l2(list + ((t0 + (warp + pf * NW) * 16) >> shift));
      }
    };
    cp_async_wait<NST - U>();
    __syncwarp();

    // ---- fragment loads of K (A operand of S^T) and V (A operand of O^T).  bf16 loads
    // both for the whole iteration first, so their shared-memory latencies overlap each
    // other and the softmax; fp8 loads V once the score products have consumed K, so the
    // two sets of fragments never hold registers at the same time (the loads are volatile
    // asm: the compiler keeps them in source order)
    constexpr int kKFrag = (KV == PSP_KV_BF16) ? D / 16 : D / 32;
    constexpr int kVFrag = (KV == PSP_KV_BF16) ? C::kMTiles : D / 32;
    uint32_t kf[U][kKFrag][4], vf[U][kVFrag][4];
    const bool second = (U == 1) || (i0 + 1 < my_n);  // fp8: the iteration's second sub-tile exists
    const int lj = lane >> 3;
    const int krow = (lane & 7) + (lj & 1) * 8;
    const int vrow = (lane & 7) + (lj >> 1) * 8;
    auto load_v = [&]() {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const unsigned char* vt = ring + wrap(st0 + u) * C::kStageBytes + C::kTileBytes;
#pragma unroll
        for (int f = 0; f < kVFrag; ++f)
          ldsm_x4_t(vf[u][f], smem_u32(vt + vrow * C::kRowBytes + swz<C::kChunks>(vrow, 2 * f + (lj & 1)) * 16));
      }
      if (!second) {
        // no second sub-tile: its stage holds stale codes (possibly NaN), so its value
        // fragments are zero and its scores are masked below
#pragma unroll
        for (int f = 0; f < kVFrag; ++f) vf[U - 1][f][0] = vf[U - 1][f][1] = vf[U - 1][f][2] = vf[U - 1][f][3] = 0u;
      }
    };
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const unsigned char* kt = ring + wrap(st0 + u) * C::kStageBytes;
#pragma unroll
      for (int f = 0; f < kKFrag; ++f)
        ldsm_x4(kf[u][f], smem_u32(kt + krow * C::kRowBytes + swz<C::kChunks>(krow, 2 * f + (lj >> 1)) * 16));
    }
    if constexpr (KV == PSP_KV_BF16) load_v();

    // ---- S^T (16 tokens x 8 query heads) per sub-tile; two accumulators halve the mma chain
    float x[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (KV == PSP_KV_BF16) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) mma_bf16((ks & 1) ? sb : sa, kf[u][ks], qf[ks][0], qf[ks][1]);
      } else {
        // the ldmatrix fragments of 16 rows x 32 codes are the e4m3 A operand as they stand
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) mma_e4m3((kk & 1) ? sb : sa, kf[u][kk], qf[kk][0], qf[kk][1]);
      }
      // rows = tokens (lane>>2, +8), cols = heads (2c, 2c+1)
      const int tb = t0 + (warp + (i0 + u) * NW) * 16;
      const bool live = (u == 0) || second;
      const bool v_lo = live && tb + (lane >> 2) < t1;
      const bool v_hi = live && tb + (lane >> 2) + 8 < t1;
      x[u][0] = v_lo ? (sa[0] + sb[0]) * sc0 : neg_inf();
      x[u][1] = v_lo ? (sa[1] + sb[1]) * sc1 : neg_inf();
      x[u][2] = v_hi ? (sa[2] + sb[2]) * sc0 : neg_inf();
      x[u][3] = v_hi ? (sa[3] + sb[3]) * sc1 : neg_inf();
    }

    if constexpr (KV != PSP_KV_BF16) load_v();
    __syncwarp();  // every lane's fragment loads of these stages come first
    refill();

    // ---- online softmax over the iteration's tokens
    float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
    for (int u = 1; u < U; ++u) {
      mx0 = fmaxf(mx0, fmaxf(x[u][0], x[u][2]));
      mx1 = fmaxf(mx1, fmaxf(x[u][1], x[u][3]));
    }
    mx0 = xor_max<4, 16>(mx0) - kPShift;
    mx1 = xor_max<4, 16>(mx1) - kPShift;
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    float pr[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      pr[u][0] = ex2_ftz(x[u][0] - mn0);
      pr[u][1] = ex2_ftz(x[u][1] - mn1);
      pr[u][2] = ex2_ftz(x[u][2] - mn0);
      pr[u][3] = ex2_ftz(x[u][3] - mn1);
    }
    // fp8 (bound by its instruction count): rescale only when some running max moved,
    // which stops once the maxima settle; bf16 (bound by memory) rescales every sub-tile
    if (KV != PSP_KV_FP8 || __any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
      const float a0 = ex2_ftz(m0 - mn0), a1 = ex2_ftz(m1 - mn1);
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      m0 = mn0;
      m1 = mn1;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      l0 += pr[u][0] + pr[u][2];
      l1 += pr[u][1] + pr[u][3];
    }

    // ---- O^T += V^T P^T
    if constexpr (KV == PSP_KV_BF16) {
      // P^T as the B operand (k = token, n = query head) by an in-register 8x8 transpose
      const uint32_t pb0 = movmatrix_t(pack_bf16(pr[0][0], pr[0][1]));
      const uint32_t pb1 = movmatrix_t(pack_bf16(pr[0][2], pr[0][3]));
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) mma_bf16(o[mt], vf[0][mt], pb0, pb1);
    } else {
      // k = 32 tokens per product, ordered (2c, 2c+1, 2c+8, 2c+9) of sub-tile 0 at k = 4c..4c+3
      // and the same tokens of sub-tile 1 at k = 16+4c..: the transposed f16 probabilities of
      // head g become four e4m3 codes per register, and the value fragments are regrouped
      // to the same token order by byte permutes (even and odd d separately)
      uint32_t pb[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t lo = movmatrix_t(pack_f16(pr[u][0], pr[u][1]));  // tokens 2c, 2c+1 of head g
        const uint32_t hi = movmatrix_t(pack_f16(pr[u][2], pr[u][3]));  // tokens 2c+8, 2c+9
        pb[u] = e4m3x2_from_f16x2(lo) | (e4m3x2_from_f16x2(hi) << 16);
      }
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        // vf[u][cc][0]: (token 2c: d 32cc+2g, +1), (token 2c+1: same d); [2]: tokens 2c+8, 2c+9;
        // [1], [3]: the same for d 32cc+16+2g, +1
        const uint32_t ae[4] = {__byte_perm(vf[0][cc][0], vf[0][cc][2], 0x6420), __byte_perm(vf[0][cc][1], vf[0][cc][3], 0x6420),
                                __byte_perm(vf[U - 1][cc][0], vf[U - 1][cc][2], 0x6420),
                                __byte_perm(vf[U - 1][cc][1], vf[U - 1][cc][3], 0x6420)};
        const uint32_t ao[4] = {__byte_perm(vf[0][cc][0], vf[0][cc][2], 0x7531), __byte_perm(vf[0][cc][1], vf[0][cc][3], 0x7531),
                                __byte_perm(vf[U - 1][cc][0], vf[U - 1][cc][2], 0x7531),
                                __byte_perm(vf[U - 1][cc][1], vf[U - 1][cc][3], 0x7531)};
        mma_e4m3(o[2 * cc], ae, pb[0], pb[U - 1]);
        mma_e4m3(o[2 * cc + 1], ao, pb[0], pb[U - 1]);
      }
    }
  }
  if constexpr (KV == PSP_KV_FP8) {
    cta = suffix_cta(p, reload_split_desc(p, split), split, h, kPre);
    if (late) suffix_cta_mark_late(p, cta, kPre);
  }
  const bool grid_last = suffix_grid_arrive(p);
  cp_async_commit();  // copies issued after the loop's last commit (a warp without refills)
  cp_async_wait<0>();
  if (cta.wait_prefix) {
    pdl_wait_primary();  // every prefix partial and prefix arrival of this step is complete
    if (cta.pre_smem) {
      prefetch_prefix_rows<D, NW * 32>(p, cta, pre_o, pre_l);
      cp_async_commit();
      cp_async_wait<0>();
    }
  }

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
  suffix_finish<D, NW, NW * 32>(p, cta, red, ms, ls, pre_o, pre_l, out_scale);
  suffix_grid_tail(p, grid_last);
}

template <int KV, int D, int NW, int NST, bool PT>
cudaError_t launch_pt(const StepParams& p, int num_splits, cudaStream_t s) {
  using C = SufCfg<KV, D>;
  const int ring = NW * NST * C::kStageBytes;
  const int epi = (NW * 8 * D + 2 * NW * 8) * 4;
  const int bytes = (ring > epi ? ring : epi) + C::template pre_rows<NST>() * (D + 1) * 4;
  auto kern = suffix_kernel<KV, D, NW, NST, PT>;
  cudaError_t e = ensure_smem_limit<suffix_kernel<KV, D, NW, NST, PT>>(bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_splits * p.hkv);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KV, int D, int NW, int NST>
cudaError_t launch_t(const StepParams& p, int num_splits, cudaStream_t s) {
  if (!p.token_flat && p.page_shift >= 4) return launch_pt<KV, D, NW, NST, true>(p, num_splits, s);
  return launch_pt<KV, D, NW, NST, false>(p, num_splits, s);
}

}  // namespace

// Ring depth per warp for d = 128 (PSP_SUFFIX_STAGES overrides it for tuning sweeps):
// fewer stages leave room for more resident CTAs per SM.
int suffix_stages(int fallback) {
  static const int env = [] {
    const char* v = std::getenv("PSP_SUFFIX_STAGES");
    return v ? std::atoi(v) : 0;
  }();
  return env > 0 ? env : fallback;
}

cudaError_t launch_suffix(const StepParams& p, int num_splits, cudaStream_t s) {
  if (num_splits <= 0) return cudaSuccess;
  if (p.kv_dtype == PSP_KV_BF16) {
    if (p.head_dim != 128) return launch_t<PSP_KV_BF16, 64, 4, 4>(p, num_splits, s);
    switch (suffix_stages(2)) {  // 2 stages: three CTAs per SM (measured best with 5 split CTAs per SM)
      case 3: return launch_t<PSP_KV_BF16, 128, 4, 3>(p, num_splits, s);
      case 4: return launch_t<PSP_KV_BF16, 128, 4, 4>(p, num_splits, s);
      default: return launch_t<PSP_KV_BF16, 128, 4, 2>(p, num_splits, s);
    }
  }
  if (p.kv_dtype == PSP_KV_FP8) {
    if (p.head_dim != 128) return launch_t<PSP_KV_FP8, 64, 4, 6>(p, num_splits, s);
    switch (suffix_stages(3)) {  // 3 stages, 128 registers: four CTAs per SM (measured best)
      case 4: return launch_t<PSP_KV_FP8, 128, 4, 4>(p, num_splits, s);
      case 5: return launch_t<PSP_KV_FP8, 128, 4, 5>(p, num_splits, s);
      default: return launch_t<PSP_KV_FP8, 128, 4, 3>(p, num_splits, s);
    }
  }
  return launch_suffix_simt(p, num_splits, s);
}

}  // namespace psp
