// kernel_prefix_dense.cu -- dense shared-prefix attention on the 5th-generation
// tensor cores (tcgen05), the branch the dispatcher takes at large M_eff
// ("GraniKV", section 3: above the threshold the shared prefix runs as a dense
// matmul over all stacked queries; section 2: the prefix is read once per step
// instead of once per request).
//
// One CTA = 256 stacked query rows of one KV head (rows R = member * G + j, in
// two 128-row tiles A and B) x one chunk of the shared prefix, in 128-token
// K/V tiles that both query tiles share:
//   warps 8 and 9 (producers, keys and values) TMA-load each K and V tile page
//                      by page from the paged pool (3-D tensor map [slot][kv
//                      head][d], boxes of up to 64 tokens x 128 bytes, 128-byte
//                      swizzle) into rings of 2 (bf16) or 4 (e4m3) stages;
//   warp 10 (MMA)      one thread issues, per K/V tile j,
//                        S_A = Q_A K_j^T, S_B = Q_B K_j^T       (M=128, N=128)
//                        O_A += P_A V_j, S_A(j+1), O_B += P_B V_j, S_B(j+1)
//                      with fp32 accumulators in tensor memory (S_A, S_B, O_A,
//                      O_B: all 512 columns) and P read from tensor memory; in
//                      this order the tensor core runs one tile's products while
//                      the other tile's softmax warps work;
//   warps 0-3 / 4-7    (softmax, tiles A / B) one thread per row: read the S
//                      row, online softmax with lazy rescaling (the running max
//                      only moves when it grows by more than 2^8, and O is then
//                      rescaled in tensor memory), write P back over S, and at
//                      the end normalise O and write the fp32 partial row and
//                      its log2-LSE.
// fp8-e4m3 caches use kind::f8f6f4: the e4m3 K/V tiles are loaded as stored,
// each query row is quantised to e4m3 with its own scale amax/448 (folded, with
// the per-head key scale, into the softmax scale), and P is written to tensor
// memory as e4m3 (P <= 2^8 under the lazy bound, inside the e4m3 range); the
// value scale is applied to the normalised output.
// Every mbarrier wait is bounded; on timeout the kernel records the site in the
// device status word and unwinds (draining its own TMA copies, freeing its
// tensor memory) instead of hanging.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"
#include "psp_sm100.cuh"

namespace psp {
namespace {

using namespace dev;
using namespace sm100;

constexpr int kRows = 128;                 // UMMA M (stacked query rows per tile)
constexpr int kTok = 128;                  // tokens per K/V tile (N of S, K of PV)
constexpr int kD = 128;                    // head dim (K of S, N of PV)
constexpr int kThreads = 352;              // warps 0-7 softmax, 8 K producer, 9 V producer, 10 MMA
constexpr uint32_t kTmemCols = 512;        // S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512)
constexpr float kRescaleLog2 = 8.f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <bool FP8>
struct DenseCfg {
  static constexpr uint32_t kElem = FP8 ? 1 : 2;
  static constexpr int kStages = FP8 ? 4 : 2;                // K and V ring depth
  static constexpr uint32_t kTileBytes = kTok * kD * kElem;  // one K or V tile
  static constexpr uint32_t kQBytes = kRows * kD * kElem;    // one query tile
  static constexpr uint32_t kHalves = FP8 ? 1 : 2;           // 128-byte column blocks of a row
  static constexpr uint32_t kHalf = kTileBytes / kHalves;
  static constexpr uint32_t kQHalf = kQBytes / kHalves;
  static constexpr int kBoxElems = 128 / kElem;              // d elements per TMA box row
  static constexpr int kKStep = 32 / kElem;                  // K elements per MMA instruction
  static constexpr uint32_t kOffQ = 0;                       // Q_A, Q_B
  static constexpr uint32_t kOffK = kOffQ + 2 * kQBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
  // barriers: q_ready, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], pv_done[2], o_full, final
  static constexpr int kBarQ = 0, kBarKFull = 1, kBarKEmpty = 1 + kStages, kBarVFull = 1 + 2 * kStages,
                       kBarVEmpty = 1 + 3 * kStages, kBarSFull = 1 + 4 * kStages, kBarPFull = 3 + 4 * kStages,
                       kBarPvDone = 5 + 4 * kStages, kBarOFull = 7 + 4 * kStages, kBarFinal = 8 + 4 * kStages,
                       kNumBars = 9 + 4 * kStages;
  static constexpr uint32_t kOffTmem = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffFlag = kOffTmem + 8;
  static constexpr uint32_t kSmemBytes = kOffFlag + 8 + 1024;  // + alignment slack
  static constexpr uint32_t kIdescS = FP8 ? idesc_e4m3(kRows, kTok, false) : idesc_f16(kRows, kTok, 1, false);
  static constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3(kRows, kD, true) : idesc_f16(kRows, kD, 1, true);
};

template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_dense_kernel(const StepParams p, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, int num_slots) {
  using C = DenseCfg<FP8>;
  constexpr int NS = C::kStages;
  constexpr uint32_t kTileBytes = C::kTileBytes;
  constexpr uint32_t kHalf = C::kHalf;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  auto bar = [&](int i) { return base + C::kOffBar + 8u * i; };
  volatile int* failed = reinterpret_cast<volatile int*>(gbase + C::kOffFlag);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ci = p.item_chunk_dense[blockIdx.x];
  const int rb = p.item_rb_dense[blockIdx.x];  // 256-row block
  const int h = blockIdx.y;
  const int g = p.chunk_group[ci];
  const int t0 = p.chunk_begin[ci];
  const int t1 = p.chunk_end[ci];
  const int n_tiles = (t1 - t0 + kTok - 1) / kTok;
  const int G = p.group;
  const int m_eff = p.group_m_eff[g];
  const int row_base = rb * 2 * kRows;
  const bool tile_b = row_base + kRows < m_eff;  // tile B holds live rows
  const int32_t* members = p.group_members + p.group_member_indptr[g];
  int32_t* status = p.status;

  if (threadIdx.x == 0) {
    *failed = 0;
    mbar_init(bar(C::kBarQ), tile_b ? 256 : 128);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
      mbar_init(bar(C::kBarVFull + s), 1);
      mbar_init(bar(C::kBarVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), 128);
      mbar_init(bar(C::kBarPvDone + t), 1);
    }
    mbar_init(bar(C::kBarOFull), 1);
    mbar_init(bar(C::kBarFinal), 1);
    fence_mbar_init();
  }
  if (warp == 10) {
    tmem_alloc(base + C::kOffTmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);

  if (warp == 8 || warp == 9) {
    // ------------------------------------------------- producers: warp 8 keys, warp 9 values
    if (lane == 0) {
      const bool is_v = warp == 9;
      const CUtensorMap* map = is_v ? &vmap : &kmap;
      prefetch_tmap(map);
      const int full0 = is_v ? C::kBarVFull : C::kBarKFull;
      const int empty0 = is_v ? C::kBarVEmpty : C::kBarKEmpty;
      const uint32_t ring = base + (is_v ? C::kOffV : C::kOffK);
      const int32_t* list;
      int shift;
      if (p.token_flat) {
        list = p.kv_indices + p.kv_indptr[members[0]];
        shift = 0;
      } else {
        list = p.group_page_indices + p.group_page_indptr[g];
        shift = p.page_shift;
      }
      const int mask = (1 << shift) - 1;
      const int br = min(1 << shift, 64);  // rows per TMA box; boxes never straddle a page
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(bar(empty0 + s), ((j / NS) - 1) & 1, status, is_v ? 2 : 1)) break;
        mbar_arrive_tx(bar(full0 + s), kTileBytes);
        const uint32_t dst = ring + s * kTileBytes;
        for (int r = 0; r < kTok; r += br) {
          const int tok = t0 + j * kTok + r;
          const int slot = tok < t1 ? ((__ldg(list + (tok >> shift)) << shift) | (tok & mask)) : num_slots;
#pragma unroll
          for (uint32_t hf = 0; hf < C::kHalves; ++hf)
            tma_load_3d(dst + hf * kHalf + r * 128, map, hf * C::kBoxElems, h, slot, bar(full0 + s));
        }
        issued = j + 1;
      }
      // drain: the last load issued on each stage must have landed before the CTA may exit
      for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(bar(full0 + j % NS), (j / NS) & 1, status, 3);
    }
  } else if (warp == 10) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      bool ok = mbar_wait(bar(C::kBarQ), 0, status, 4);
      tc_fence_after();
      // S_t = Q_t K_j^T into the S columns of tile t
      auto issue_s = [&](int t, int j) {
        const uint32_t kbase = base + C::kOffK + (j % NS) * kTileBytes;
        const uint32_t qbase = base + C::kOffQ + t * C::kQBytes;
#pragma unroll
        for (int ks = 0; ks < kD / C::kKStep; ++ks) {
          // K-major operands: 32 bytes of K per instruction inside a 128-byte swizzled row
          const uint32_t off = (ks & 3) * 32;
          const uint64_t adesc = sw128_desc(qbase + (ks >> 2) * C::kQHalf + off, 16, 1024);
          const uint64_t bdesc = sw128_desc(kbase + (ks >> 2) * kHalf + off, 16, 1024);
          if constexpr (FP8) {
            mma_ss_f8(tmem + t * kTok, adesc, bdesc, C::kIdescS, ks > 0 ? 1u : 0u);
          } else {
            mma_ss(tmem + t * kTok, adesc, bdesc, C::kIdescS, ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(C::kBarSFull + t));
      };
      // O_t += P_t V_j (P from the S columns of tile t)
      auto issue_pv = [&](int t, int j) {
        const uint32_t vbase = base + C::kOffV + (j % NS) * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kTok / C::kKStep; ++ks) {
          // V is the MN-major B operand: K (tokens) advances by whole 128-byte rows
          const uint64_t bdesc = sw128_desc(vbase + ks * C::kKStep * 128, kHalf, 1024);
          const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
          if constexpr (FP8) {
            mma_ts_f8(tmem + 256 + t * kD, tmem + t * kTok + ks * 8, bdesc, C::kIdescPV, acc);
          } else {
            mma_ts(tmem + 256 + t * kD, tmem + t * kTok + ks * 8, bdesc, C::kIdescPV, acc);
          }
        }
        mma_commit(bar(C::kBarPvDone + t));
      };
      if (ok && n_tiles > 0) {
        ok = mbar_wait(bar(C::kBarKFull), 0, status, 7);
        tc_fence_after();
        if (ok) {
          issue_s(0, 0);
          if (tile_b) issue_s(1, 0);
          mma_commit(bar(C::kBarKEmpty));
        }
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const bool more = j + 1 < n_tiles;
        ok = mbar_wait(bar(C::kBarPFull + 0), j & 1, status, 5) &&
             mbar_wait(bar(C::kBarVFull + j % NS), (j / NS) & 1, status, 6);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, j);
        if (more) {
          ok = mbar_wait(bar(C::kBarKFull + (j + 1) % NS), ((j + 1) / NS) & 1, status, 7);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, j + 1);  // S_A's columns are reused only after PV_A(j) (issued above) has read P_A(j)
        }
        if (tile_b) {
          ok = mbar_wait(bar(C::kBarPFull + 1), j & 1, status, 5);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, j);
          if (more) issue_s(1, j + 1);
        }
        mma_commit(bar(C::kBarVEmpty + j % NS));
        if (more) mma_commit(bar(C::kBarKEmpty + (j + 1) % NS));
      }
      mma_commit(bar(C::kBarOFull));
      mma_commit(bar(C::kBarFinal));
      mbar_wait(bar(C::kBarFinal), 0, status, 8);  // every MMA of this CTA has completed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- softmax warps
    const int t = warp >> 2;                   // query tile (0 = A, 1 = B)
    const int r = threadIdx.x & 127;           // row of the tile = TMEM lane
    const int R = row_base + t * kRows + r;
    const bool live = R < m_eff;
    const bool active = t == 0 || tile_b;
    float q_scale = 1.f;  // fp8: this row's quantisation scale
    if (active) {
      const uint4* qrow = nullptr;
      if (live) {
        const int mem = R / G, jq = R - mem * G;
        qrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                              (static_cast<int64_t>(members[mem]) * p.hq + h * G + jq) * kD);
      }
      const uint32_t qoff = C::kOffQ + t * C::kQBytes;
      // all 16 loads of the row in flight before the first shared store (the compiler
      // cannot move global loads across generic stores that might alias them)
      uint4 v[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = live ? __ldg(qrow + c) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (FP8) {
        // the row's amax, then e4m3 codes of q / (amax / 448)
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
          for (int k = 0; k < 4; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[k] & 0xffff)), fabsf(bf16_bits_to_float(w[k] >> 16))));
        }
        q_scale = amax > 0.f ? amax / 448.f : 1.f;
        const float inv = 1.f / q_scale;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16 e4m3 codes per 16-byte chunk
          const uint32_t w[8] = {v[2 * c].x,     v[2 * c].y,     v[2 * c].z,     v[2 * c].w,
                                 v[2 * c + 1].x, v[2 * c + 1].y, v[2 * c + 1].z, v[2 * c + 1].w};
          uint32_t out[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            out[k] = e4m3x4_from_floats(
                bf16_bits_to_float(w[2 * k] & 0xffff) * inv, bf16_bits_to_float(w[2 * k] >> 16) * inv,
                bf16_bits_to_float(w[2 * k + 1] & 0xffff) * inv, bf16_bits_to_float(w[2 * k + 1] >> 16) * inv);
          *reinterpret_cast<uint4*>(gbase + qoff + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
              make_uint4(out[0], out[1], out[2], out[3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(gbase + qoff + (c >> 3) * C::kQHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v[c];
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::kBarQ));
    }
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = t * kTok, o_col = 256 + t * kD;
    float scale = p.scale_log2;  // > 0, so max(x) * scale = max(x * scale)
    float out_scale = 1.f;
    if constexpr (FP8) {
      scale *= __ldg(p.k_scale + h) * q_scale;
      out_scale = __ldg(p.v_scale + h);
    }
    float m_used = neg_inf(), l = 0.f;
    bool ok = active;
    for (int j = 0; j < n_tiles && ok; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarSFull + t), j & 1, status, 9));
      if (!ok) break;
      tc_fence_after();
      float x[kTok];
      {
        uint32_t u[kTok / 32][32];
#pragma unroll
        for (int c = 0; c < kTok / 32; ++c) tmem_ld32(lane_addr + s_col + c * 32, u[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kTok / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(u[c][i]);
      }
      const int valid = t1 - (t0 + j * kTok);
      if (valid < kTok) {
#pragma unroll
        for (int i = 0; i < kTok; ++i) x[i] = i < valid ? x[i] : neg_inf();
      }
      // tile max with eight independent accumulators (short dependency chains)
      float mx[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx[a] = x[a];
#pragma unroll
      for (int i = 8; i < kTok; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * scale;
      const bool need = mt > m_used + kRescaleLog2;
      float alpha = 1.f;
      if (need) {
        alpha = ex2(m_used - mt);
        m_used = mt;
        l *= alpha;
      }
      const float neg_m = -m_used;
      float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if constexpr (FP8) {
        uint32_t u[kTok / 4];  // four e4m3 probabilities per column
#pragma unroll
        for (int i = 0; i < kTok / 4; ++i) {
          const float a = ex2(fmaf(x[4 * i], scale, neg_m)), b = ex2(fmaf(x[4 * i + 1], scale, neg_m));
          const float c2 = ex2(fmaf(x[4 * i + 2], scale, neg_m)), d2 = ex2(fmaf(x[4 * i + 3], scale, neg_m));
          sm[i & 7] += (a + b) + (c2 + d2);
          u[i] = e4m3x4_from_floats(a, b, c2, d2);
        }
        tmem_st32(lane_addr + s_col, u);
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t u[32];  // two bf16 probabilities per column
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float a = ex2(fmaf(x[c * 64 + 2 * i], scale, neg_m));
            const float b = ex2(fmaf(x[c * 64 + 2 * i + 1], scale, neg_m));
            sm[i & 7] += a + b;
            u[i] = pack_bf16(a, b);
          }
          tmem_st32(lane_addr + s_col + c * 32, u);
        }
      }
      l += ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O_t holds the products of tiles < j; wait for the last of them, then rescale this row
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarPvDone + t), (j - 1) & 1, status, 10));
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(lane_addr + o_col + c * 32, u);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
            tmem_st32(lane_addr + o_col + c * 32, u);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBarPFull + t));
    }
    // epilogue: O / l -> fp32 partial row, log2-LSE
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(C::kBarOFull), 0, status, 11));
    if (ok) {
      tc_fence_after();
      const int64_t row = p.chunk_row_offset[ci] + static_cast<int64_t>(h) * m_eff + R;
      float4* dst = live ? reinterpret_cast<float4*>(p.o_pre + row * kD) : nullptr;
      const float inv = out_scale / l;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(lane_addr + o_col + c * 32, u);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[c * 8 + i] = make_float4(__uint_as_float(u[4 * i]) * inv, __uint_as_float(u[4 * i + 1]) * inv,
                                         __uint_as_float(u[4 * i + 2]) * inv, __uint_as_float(u[4 * i + 3]) * inv);
        }
      }
      if (live) p.lse_pre[row] = m_used + __log2f(l);
      __threadfence();
    }
    if (active && !ok) *failed = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 10) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // arrive for every member of this row block (shared memory is free now: every MMA and
  // TMA copy of this CTA has completed); the arrival that completes a member merges it
  if (!*failed) {
    const int n_rows = min(2 * kRows, m_eff - row_base);
    __syncthreads();
    prefix_arrive_and_merge<kD>(p, members, h, row_base, n_rows, reinterpret_cast<int*>(gbase));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Pool [slots][Hkv][d] as a 3-D tensor; box = 128 bytes of d x 1 head x rows tokens, 128-byte swizzle.
cudaError_t make_pool_map(CUtensorMap* map, const void* pool, int64_t slots, int hkv, int rows, bool fp8) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t elem = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(slots)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * elem, static_cast<cuuint64_t>(hkv) * kD * elem};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem), 1, static_cast<cuuint32_t>(rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool FP8>
cudaError_t launch_t(const StepParams& p, int num_items, cudaStream_t s) {
  const int64_t slots = static_cast<int64_t>(p.num_pages) * p.page_size;
  if (slots >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  const int rows = p.token_flat ? 1 : (p.page_size < 64 ? p.page_size : 64);
  CUtensorMap kmap, vmap;
  cudaError_t e = make_pool_map(&kmap, p.k_pool, slots, p.hkv, rows, FP8);
  if (e != cudaSuccess) return e;
  e = make_pool_map(&vmap, p.v_pool, slots, p.hkv, rows, FP8);
  if (e != cudaSuccess) return e;
  constexpr uint32_t bytes = DenseCfg<FP8>::kSmemBytes;
  static_assert(bytes <= 232448, "dense prefix CTA exceeds the shared memory of one SM");
  e = cudaFuncSetAttribute(prefix_dense_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(num_items, p.hkv);
  prefix_dense_kernel<FP8><<<grid, kThreads, bytes, s>>>(p, kmap, vmap, static_cast<int>(slots));
  return cudaGetLastError();
}

}  // namespace

// True when the tcgen05 dense kernel serves this configuration (bf16 or e4m3 K/V, d = 128).
bool dense_tc_supported(const StepParams& p) {
  return (p.kv_dtype == PSP_KV_BF16 || p.kv_dtype == PSP_KV_FP8) && p.head_dim == kD;
}

cudaError_t launch_prefix_dense_tc(const StepParams& p, int num_items, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  return p.kv_dtype == PSP_KV_FP8 ? launch_t<true>(p, num_items, s) : launch_t<false>(p, num_items, s);
}

}  // namespace psp
