// kernel_prefix_dense.cu -- dense shared-prefix attention on the 5th-generation
// tensor cores (tcgen05), the branch the dispatcher takes at large M_eff
// ("GraniKV", section 3: above the threshold the shared prefix runs as a dense
// matmul over all stacked queries; section 2: the prefix is read once per step
// instead of once per request).
//
// One CTA = 256 stacked query rows of one KV head (rows R = member * G + j, in
// two 128-row tiles A and B) x one chunk of the shared prefix, in 128-token
// K/V tiles that both query tiles share:
//   warp 8          (producer) TMA-loads K and V tiles page by page from the
//                   paged pool (3-D tensor maps [slot][kv head][d], boxes of up to
//                   64 tokens x 128 bytes, 128-byte swizzle): K_0 into a slot of
//                   its own, then ring stage j holds V_j and K_{j+1}, the operands
//                   that one issue step consumes, behind a single barrier;
//   warp 9          (MMA) one thread issues, per K/V tile j and query tile t,
//                     O_t += P_t V_j, then S_t = Q_t K_{j+1}^T  (M=128, N=128)
//                   with fp32 accumulators in tensor memory (S_A, S_B, O_A, O_B:
//                   all 512 columns) and P read from tensor memory where the
//                   softmax wrote it over S; tile A's products run while tile B's
//                   softmax works and the other way round;
//   warps 0-3 / 4-7 (softmax, tiles A / B) one thread per row: read the S row,
//                   online softmax, write P back over S, and at the end normalise O
//                   and write the fp32 partial row and its log2-LSE.  With bf16 the
//                   two groups take turns at the exponentials of a tile (A(j), B(j),
//                   A(j+1), ..., handed over on two barriers): groups left to
//                   themselves fall into step, computing at the same time and then
//                   waiting together for the tensor pipe (measured on GB300: 4% on the
//                   bf16 agent batch; e4m3 tiles, whose softmax is bound by the latency
//                   of one warp rather than by the shared units, run 18% slower in turns).
// The MMA warp runs its waits as a whole warp with one lane issuing (measured on
// GB300: a completed mbarrier costs 100-200 cycles to poll, more from one lane
// than from a whole warp, and one lane issuing while the rest of its warp polls
// another barrier is slowed several-fold), and one barrier covers V_j and
// K_{j+1}, so each issue step has a single wait for its operands.
// The online softmax rescales lazily: the running max only moves when it grows
// by more than 2^8, and O is then rescaled in tensor memory.
// fp8-e4m3 caches use kind::f8f6f4: the e4m3 K/V tiles are loaded as stored,
// each query row is quantised to e4m3 with its own scale amax/448 (folded, with
// the per-head key scale, into the softmax scale), and P is written to tensor
// memory as e4m3 (P <= 2^8 under the lazy bound, inside the e4m3 range); the
// value scale is applied to the normalised output.
// Every mbarrier wait is bounded and also watches a CTA-wide abort flag: on a
// timeout the kernel records the site in the device status word, raises the flag
// so that every other role stops waiting, and unwinds (draining its own TMA
// copies and tensor-core products, freeing its tensor memory) instead of hanging.
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

constexpr int kRows = 128;                   // UMMA M (stacked query rows per tile)
constexpr int kTok = 128;                    // tokens per K/V tile (N of S, K of PV)
constexpr int kD = 128;                      // head dim (K of S, N of PV)
constexpr int kGroup = 128;                  // threads of one softmax group (one per tile row)
constexpr int kWarpP = 8, kWarpM = 9;        // producer and MMA warps
constexpr int kThreads = 2 * kGroup + 64;
constexpr uint32_t kTmemCols = 512;          // S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512)
constexpr float kRescaleLog2 = 8.f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <bool FP8>
struct DenseCfg {
  static constexpr uint32_t kElem = FP8 ? 1 : 2;
  static constexpr int kStages = FP8 ? 5 : 2;                // ring depth, stages of (V_j, K_{j+1})
  static constexpr uint32_t kTileBytes = kTok * kD * kElem;  // one K or V tile
  static constexpr uint32_t kQBytes = kRows * kD * kElem;    // one query tile
  static constexpr uint32_t kHalves = FP8 ? 1 : 2;           // 128-byte column blocks of a row
  static constexpr uint32_t kHalf = kTileBytes / kHalves;
  static constexpr uint32_t kQHalf = kQBytes / kHalves;
  static constexpr int kBoxElems = 128 / kElem;              // d elements per TMA box row
  static constexpr int kKStep = 32 / kElem;                  // K elements per MMA instruction
  static constexpr uint32_t kOffQ = 0;                       // Q_A, Q_B (each reused as its tile's epilogue staging)
  static constexpr uint32_t kOffK0 = kOffQ + 2 * kQBytes;   // K_0
  static constexpr uint32_t kOffRing = kOffK0 + kTileBytes;  // stage s: V at +0, K at +kTileBytes
  static constexpr uint32_t kStageBytes = 2 * kTileBytes;
  static constexpr uint32_t kOffBar = kOffRing + kStages * kStageBytes;
  // barriers: k0_full, full[S], empty[S], q_full[2], s_full[2], p_full[2], o_full[2], drain, turn[2]
  static constexpr int kBarK0 = 0, kBarFull = 1, kBarEmpty = 1 + kStages, kBarQFull = 1 + 2 * kStages,
                       kBarSFull = kBarQFull + 2, kBarPFull = kBarSFull + 2, kBarOFull = kBarPFull + 2,
                       kBarDrain = kBarOFull + 2, kBarTurn = kBarDrain + 1, kNumBars = kBarTurn + 2;
  static constexpr uint32_t kOffTmem = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffAbort = kOffTmem + 8;       // int: a role gave up (CTA-wide)
  static constexpr uint32_t kOffAny = kOffAbort + 8;        // int: some member must arrive
  static constexpr uint32_t kOffFlags = kOffAny + 8;        // int flags[2 * kRows]: member must arrive
  static constexpr uint32_t kSmemBytes = kOffFlags + 2 * kRows * 4 + 1024;  // + alignment slack
  static constexpr uint32_t kIdescS = FP8 ? idesc_e4m3(kRows, kTok, false) : idesc_f16(kRows, kTok, 1, false);
  static constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3(kRows, kD, true) : idesc_f16(kRows, kD, 1, true);
  static_assert(4 * 32 * 32 * 4 <= kQBytes, "epilogue staging (4 warps x 32 x 32 fp32) must fit in one Q tile");
};

// Pages of fewer than 16 tokens: one TMA box per page would leave the copy engine issuing a
// box (or two) for every token, so the producer warp gathers a tile's rows itself with 16-byte
// cp.async copies, into the layout the boxes give: chunk c of row r at r * 128 + ((c ^ (r & 7))
// << 4) of each 128-byte column block (the 128-byte swizzle of a 1024-byte-aligned tile).
// Lane l holds the pool slots of rows l, l + 32, l + 64 and l + 96 of tile j (-1 at or past
// t1, whose rows are zero-filled).
__device__ __forceinline__ void tile_slots(int (&slot)[4], const int32_t* list, int shift, int t0, int t1, int j,
                                           int lane) {
  const int mask = (1 << shift) - 1;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int tok = t0 + j * kTok + q * 32 + lane;
    slot[q] = tok < t1 ? ((__ldg(list + (tok >> shift)) << shift) | (tok & mask)) : -1;
  }
}
// Lane l copies chunk l % 8 of rows l / 8 + 4 i, taking each row's slot from the lane that
// holds it.  The caller commits the copies.
template <bool FP8>
__device__ __forceinline__ void gather_tile(const unsigned char* pool, int hkv, int h, uint32_t dst,
                                            const int (&slot)[4], int lane) {
  using C = DenseCfg<FP8>;
  constexpr int64_t kRowBytes = static_cast<int64_t>(kD) * C::kElem;  // one head's row of a token
  const int c = lane & 7;
#pragma unroll
  for (int i = 0; i < kTok / 4; ++i) {
    const int r = (lane >> 3) + 4 * i;
    const int s = __shfl_sync(0xffffffffu, slot[i >> 3], (lane >> 3) + 4 * (i & 7));  // row r's slot
    const bool valid = s >= 0;
    const unsigned char* src = pool + (valid ? (static_cast<int64_t>(s) * hkv + h) * kRowBytes : 0) + c * 16;
    const uint32_t d = dst + r * 128 + ((c ^ (r & 7)) << 4);
#pragma unroll
    for (uint32_t hf = 0; hf < C::kHalves; ++hf) cp_async_16(d + hf * C::kHalf, src + hf * 128, valid);
  }
}

// GATHER: the producer gathers tiles with cp.async (pages of 1 or 2 tokens, token-flat
// lists); otherwise with TMA boxes of one page each.
template <bool FP8, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_dense_kernel(const StepParams p, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, int num_slots) {
  using C = DenseCfg<FP8>;
  constexpr int NS = C::kStages;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  auto bar = [&](int i) { return base + C::kOffBar + 8u * i; };
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + C::kOffAbort);
  volatile int* any_arrive = reinterpret_cast<volatile int*>(gbase + C::kOffAny);
  int* flags = reinterpret_cast<int*>(gbase + C::kOffFlags);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  dev::pdl_launch_dependents();  // the step's suffix kernel may start filling free SMs
  const int h = blockIdx.x % p.hkv;  // KV head fastest (neighbouring heads' rows are adjacent)
  const int item = blockIdx.x / p.hkv;
  // the work item's record: two 16-byte loads, issued together
  const int4 da = __ldg(reinterpret_cast<const int4*>(p.item_desc_dense + item));
  const int4 db = __ldg(reinterpret_cast<const int4*>(p.item_desc_dense + item) + 1);
  const int rb = da.y;  // 256-row block
  const int t0 = da.z;
  const int t1 = da.w;
  const int n_tiles = (t1 - t0 + kTok - 1) / kTok;
  const int G = p.group;
  const int m_eff = db.x;
  const int row_base = rb * 2 * kRows;
  const int n_rows = min(2 * kRows, m_eff - row_base);
  const bool tile_b = n_rows > kRows;  // tile B holds live rows
  const int32_t* members = p.group_members + db.y;
  const int list_base = db.z;    // the group's block list, or its first member's kv_indices
  const int row_offset = db.w;   // the chunk's first prefix-partial row
  int32_t* status = p.status;

  if (threadIdx.x == 0) {
    *abort = n_tiles > 0 ? 0 : 1;
    *any_arrive = 0;
    if (n_tiles <= 0) atomicCAS(status, 0, kDevTimeout | (12 << 8));  // never planned: empty chunk
    mbar_init(bar(C::kBarK0), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarQFull + t), kGroup / 32);  // one arrival per warp
      mbar_init(bar(C::kBarSFull + t), 1);
      mbar_init(bar(C::kBarPFull + t), kGroup / 32);
      mbar_init(bar(C::kBarOFull + t), 1);
      mbar_init(bar(C::kBarTurn + t), kGroup / 32);  // one arrival per warp of the other group
    }
    mbar_init(bar(C::kBarDrain), 1);
    fence_mbar_init();
  }
  if (warp == kWarpP) {
    tmem_alloc(base + C::kOffTmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);
  const bool run = !*abort;

  if (warp == kWarpP) {
    // ---------------------------------------------------------------- producer
    // the whole warp: lane 0 waits and sets the expected bytes, every lane issues boxes
    if (run) {
      const int32_t* list;
      int shift;
      if (p.token_flat) {
        list = p.kv_indices + list_base;
        shift = 0;
      } else {
        list = p.group_page_indices + list_base;
        shift = p.page_shift;
      }
      if constexpr (GATHER) {
        // small pages: the warp gathers every tile with cp.async (gather_tile).  Stage s (K_0
        // is stage -1) is arrived on once its copies have landed and been made visible to the
        // tensor cores' proxy, which the warp checks for at the top of iteration s + L, so the
        // copies of L stages stay in flight (L = NS - 1 keeps the producer from waiting on a
        // stage the consumer has yet to receive).
        constexpr int L = NS - 1;
        const unsigned char* kpool = static_cast<const unsigned char*>(p.k_pool);
        const unsigned char* vpool = static_cast<const unsigned char*>(p.v_pool);
        auto stage_bar = [&](int st) { return st < 0 ? bar(C::kBarK0) : bar(C::kBarFull + st % NS); };
        int cur[4], nxt[4];
        tile_slots(cur, list, shift, t0, t1, 0, lane);
        gather_tile<FP8>(kpool, p.hkv, h, base + C::kOffK0, cur, lane);
        cp_async_commit();
        int arrived = -2;  // the last stage arrived on
        int j = 0;
        for (; j < n_tiles; ++j) {
          if (j - L >= -1) {
            cp_async_wait<L - 1>();  // stage j - L and every earlier one have landed
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(stage_bar(j - L));
            arrived = j - L;
          }
          const int st = j % NS;
          if (j >= NS) {
            int ok = 0;
            if (lane == 0) ok = wait_or_abort(bar(C::kBarEmpty + st), ((j / NS) - 1) & 1, abort, status, 1) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
          }
          const uint32_t dst = base + C::kOffRing + st * C::kStageBytes;
          gather_tile<FP8>(vpool, p.hkv, h, dst, cur, lane);  // V_j: the rows of K_j
          if (j + 1 < n_tiles) {
            tile_slots(nxt, list, shift, t0, t1, j + 1, lane);
            gather_tile<FP8>(kpool, p.hkv, h, dst + C::kTileBytes, nxt, lane);
#pragma unroll
            for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
          }
          cp_async_commit();
        }
        // drain: every copy lands before the CTA may exit; the stages issued but not yet
        // arrived on (after an abort, stages nobody waits for)
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          for (int st = arrived + 1; st < j; ++st) mbar_arrive(stage_bar(st));
        __syncwarp();
      } else {
      if (lane == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
        mbar_arrive_tx(bar(C::kBarK0), C::kTileBytes);
      }
      __syncwarp();
      load_tile<kTok, C::kHalf, C::kHalves, C::kBoxElems>(&kmap, base + C::kOffK0, bar(C::kBarK0), list, shift, h, t0, t1,
                                                    0, num_slots, lane);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NS;
        if (j >= NS) {
          int ok = 0;
          if (lane == 0) ok = wait_or_abort(bar(C::kBarEmpty + st), ((j / NS) - 1) & 1, abort, status, 1) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        const bool more = j + 1 < n_tiles;
        const uint32_t full = bar(C::kBarFull + st), dst = base + C::kOffRing + st * C::kStageBytes;
        if (lane == 0) mbar_arrive_tx(full, more ? 2 * C::kTileBytes : C::kTileBytes);
        __syncwarp();
        load_tile<kTok, C::kHalf, C::kHalves, C::kBoxElems>(&vmap, dst, full, list, shift, h, t0, t1, j, num_slots, lane);
        if (more)
          load_tile<kTok, C::kHalf, C::kHalves, C::kBoxElems>(&kmap, dst + C::kTileBytes, full, list, shift, h, t0, t1,
                                                        j + 1, num_slots, lane);
        issued = j + 1;
      }
      // drain: every load issued must have landed before the CTA may exit (plain bounded waits)
      if (lane == 0) {
        mbar_wait(bar(C::kBarK0), 0, status, 3);
        for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(bar(C::kBarFull + j % NS), (j / NS) & 1, status, 3);
      }
      __syncwarp();
      }
    }
  } else if (warp == kWarpM) {
    // -------------------------------------------------------------------- MMA
    // The whole warp runs the loop and its waits; lane 0 issues.
    if (run) {
      // S_t = Q_t K^T (K tile at kbase) into the S columns of tile t
      auto issue_s = [&](int t, uint32_t kbase) {
        const uint32_t qbase = base + C::kOffQ + t * C::kQBytes;
#pragma unroll
        for (int ks = 0; ks < kD / C::kKStep; ++ks) {
          // K-major operands: 32 bytes of K per instruction inside a 128-byte swizzled row
          const uint32_t off = (ks & 3) * 32;
          const uint64_t adesc = sw128_desc(qbase + (ks >> 2) * C::kQHalf + off, 16, 1024);
          const uint64_t bdesc = sw128_desc(kbase + (ks >> 2) * C::kHalf + off, 16, 1024);
          if constexpr (FP8) {
            mma_ss_f8(tmem + t * kTok, adesc, bdesc, C::kIdescS, ks > 0 ? 1u : 0u);
          } else {
            mma_ss(tmem + t * kTok, adesc, bdesc, C::kIdescS, ks > 0 ? 1u : 0u);
          }
        }
      };
      // O_t += P_t V (V tile at vbase; P from the S columns of tile t)
      auto issue_pv = [&](int t, uint32_t vbase, bool accumulate) {
#pragma unroll
        for (int ks = 0; ks < kTok / C::kKStep; ++ks) {
          // V is the MN-major B operand: K (tokens) advances by whole 128-byte rows
          const uint64_t bdesc = sw128_desc(vbase + ks * C::kKStep * 128, C::kHalf, 1024);
          const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
          if constexpr (FP8) {
            mma_ts_f8(tmem + 256 + t * kD, tmem + t * kTok + ks * 8, bdesc, C::kIdescPV, acc);
          } else {
            mma_ts(tmem + 256 + t * kD, tmem + t * kTok + ks * 8, bdesc, C::kIdescPV, acc);
          }
        }
      };
      auto all = [](bool v) { return __all_sync(0xffffffffu, v); };
      bool ok = all(wait_or_abort(bar(C::kBarQFull), 0, abort, status, 4)) &&
                (!tile_b || all(wait_or_abort(bar(C::kBarQFull + 1), 0, abort, status, 4))) &&
                all(wait_or_abort(bar(C::kBarK0), 0, abort, status, 7));
      if (ok && lane == 0) {
        tc_fence_after();
        issue_s(0, base + C::kOffK0);
        mma_commit(bar(C::kBarSFull));
        if (tile_b) {
          issue_s(1, base + C::kOffK0);
          mma_commit(bar(C::kBarSFull + 1));
        }
      }
      __syncwarp();
      for (int j = 0; j < n_tiles && ok; ++j) {
        const bool more = j + 1 < n_tiles;
        const int st = j % NS;
        const uint32_t sb = base + C::kOffRing + st * C::kStageBytes;
        for (int t = 0; t < (tile_b ? 2 : 1) && ok; ++t) {
          ok = all(wait_or_abort(bar(C::kBarPFull + t), j & 1, abort, status, 5)) &&
               (t > 0 || all(wait_or_abort(bar(C::kBarFull + st), (j / NS) & 1, abort, status, 6)));
          if (ok && lane == 0) {
            tc_fence_after();
            issue_pv(t, sb, j > 0);
            // S_t's columns are overwritten only after PV_t(j) (issued first) has read P_t(j)
            if (more) issue_s(t, sb + C::kTileBytes);
            mma_commit(bar((more ? C::kBarSFull : C::kBarOFull) + t));
          }
          __syncwarp();
        }
        if (ok && lane == 0) mma_commit(bar(C::kBarEmpty + st));
        __syncwarp();
      }
    }
    if (lane == 0) {
      // every product of the CTA has completed before the tensor memory is freed
      mma_commit(bar(C::kBarDrain));
      mbar_wait(bar(C::kBarDrain), 0, status, 8);
    }
    __syncwarp();
  } else if (run && (warp < 4 || tile_b)) {
    // ------------------------------------------------------- softmax warps (A: 0-3, B: 4-7)
    const int t = warp >> 2;                   // query tile (0 = A, 1 = B)
    const int r = threadIdx.x & 127;           // row of the tile = TMEM lane
    const int R = row_base + t * kRows + r;
    const bool live = R < m_eff;

    // members of the block that must arrive on their (b, h) counter after the partials
    // are written; looked up now, so the loads are off the kernel's tail
    if (t == 0) {
      for (int m = r; m < n_rows / G; m += kGroup) {
        const int f = prefix_member_arrives(p, members[row_base / G + m]) ? 1 : 0;
        flags[m] = f;
        if (f) *any_arrive = 1;
      }
    }

    // ---- Q tile t into shared memory (K-major, 128-byte swizzle), e4m3 per-row scaled for fp8
    float q_scale = 1.f;
    {
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
    }

      // one arrival per warp: 32 arrivals on one barrier word serialise (measured ~500 cycles
      // for a 128-thread group), one per warp after a warp sync does not
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBarQFull + t));

    const uint32_t s_full = bar(C::kBarSFull + t), o_full = bar(C::kBarOFull + t);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = t * kTok, o_col = 256 + t * kD;
    float scale = p.scale_log2;  // > 0, so max(x) * scale = max(x * scale)
    float out_scale = 1.f;
    if constexpr (FP8) {
      scale *= __ldg(p.k_scale + h) * q_scale;
      out_scale = __ldg(p.v_scale + h);
    }
    float m_used = neg_inf(), l = 0.f;
    bool ok = true;
    constexpr bool kTurns = !FP8;
    // hands the exponentials over to the other group (one arrival per warp)
    auto pass_turn = [&]() {
      if (kTurns && tile_b) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarTurn + 1 - t));
      }
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      // S_t(j) complete, and with it every earlier product (one issuing thread), so O_t
      // holds exactly the tiles < j.  __all_sync: the warp leaves the poll loop together
      // before its aligned tcgen05 loads.
      ok = __all_sync(0xffffffffu, wait_or_abort(s_full, j & 1, abort, status, 9));
      if (!ok) break;
      tc_fence_after();
      const int valid = t1 - (t0 + j * kTok);
      // the whole S row in registers (bf16 tiles; e4m3 tiles only when they need the max)
      float x[kTok];
      auto load_row = [&]() {
        uint32_t u[kTok / 32][32];
#pragma unroll
        for (int c = 0; c < kTok / 32; ++c) tmem_ld32(lane_addr + s_col + c * 32, u[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kTok / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(u[c][i]);
        if (valid < kTok) {
#pragma unroll
          for (int i = 0; i < kTok; ++i) x[i] = i < valid ? x[i] : neg_inf();
        }
      };
      if constexpr (!FP8) load_row();
      // this group's turn at the exponentials (the other group finished its previous tile)
      if (kTurns && tile_b && (t == 1 || j > 0)) {
        ok = __all_sync(0xffffffffu, wait_or_abort(bar(C::kBarTurn + t), (t == 1 ? j : j - 1) & 1, abort, status, 13));
        if (!ok) break;
      }
      // tile max with eight independent accumulators (short dependency chains)
      auto tile_max = [&]() {
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = x[a];
#pragma unroll
        for (int i = 8; i < kTok; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
        return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
               scale;
      };
      bool need = false;
      float alpha = 1.f;
      if constexpr (FP8) {
        // The probabilities of a tile must stay <= 2^8 (inside e4m3).  After the first tile
        // the max pass is skipped: they are computed against the current reference, and since
        // all are >= 0 their sum bounds each of them, so a tile sum <= 2^8 proves the bound.
        // Only a larger sum (rare: the scores rose) takes the max and, if it moved by more
        // than 2^8, rebases; that tile, the first and a ragged last tile are computed again
        // from the whole row.
        uint32_t u[kTok / 4];  // four e4m3 probabilities per column
        const float2 scale2 = make_float2(scale, scale);
        auto make_p = [&](float m) {
          const float2 neg_m2 = make_float2(-m, -m);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int i = 0; i < kTok / 4; ++i) {
            const float2 y0 = __ffma2_rn(make_float2(x[4 * i], x[4 * i + 1]), scale2, neg_m2);
            const float2 y1 = __ffma2_rn(make_float2(x[4 * i + 2], x[4 * i + 3]), scale2, neg_m2);
            const float2 p0 = make_float2(ex2(y0.x), ex2(y0.y)), p1 = make_float2(ex2(y1.x), ex2(y1.y));
            acc[i & 3] = __fadd2_rn(acc[i & 3], __fadd2_rn(p0, p1));
            u[i] = e4m3x4_from_floats(p0.x, p0.y, p1.x, p1.y);
          }
          const float2 s = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
          return s.x + s.y;
        };
        // The S row streamed from tensor memory in 32-column pieces, the next piece loading
        // while this one computes: a full tile needs neither its max nor a register copy of
        // the whole row (the row fills most of a thread's registers).
        auto stream_p = [&](float m) {
          const float2 neg_m2 = make_float2(-m, -m);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          uint32_t ra[32], rb[32];
          tmem_ld32(lane_addr + s_col, ra);
          tmem_wait_ld_regs(ra);
#pragma unroll
          for (int c = 0; c < kTok / 32; ++c) {
            uint32_t(&cur)[32] = (c & 1) ? rb : ra;
            uint32_t(&nxt)[32] = (c & 1) ? ra : rb;
            if (c + 1 < kTok / 32) tmem_ld32(lane_addr + s_col + (c + 1) * 32, nxt);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(cur[4 * k]), __uint_as_float(cur[4 * k + 1])),
                                           scale2, neg_m2);
              const float2 y1 = __ffma2_rn(
                  make_float2(__uint_as_float(cur[4 * k + 2]), __uint_as_float(cur[4 * k + 3])), scale2, neg_m2);
              const float2 p0 = make_float2(ex2(y0.x), ex2(y0.y)), p1 = make_float2(ex2(y1.x), ex2(y1.y));
              acc[k & 3] = __fadd2_rn(acc[k & 3], __fadd2_rn(p0, p1));
              u[c * 8 + k] = e4m3x4_from_floats(p0.x, p0.y, p1.x, p1.y);
            }
            if (c + 1 < kTok / 32) tmem_wait_ld_regs(nxt);
          }
          const float2 s = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
          return s.x + s.y;
        };
        float tile_sum = 0.f;
        bool whole = j == 0 || valid < kTok;  // first tile (no reference max yet) or ragged
        if (!whole) {
          tile_sum = stream_p(m_used);
          // warp-uniform (the row reload below is a warp-collective tensor-memory load); a
          // row whose own sum passed recomputes the same probabilities against the same max
          whole = __any_sync(0xffffffffu, !(tile_sum <= 256.f));  // also catches an infinite sum
        }
        if (whole) {
          load_row();
          const float mt = tile_max();
          if (j == 0) {
            need = true;
            m_used = mt;
          } else if (mt > m_used + kRescaleLog2) {
            need = true;
            alpha = ex2(m_used - mt);
            m_used = mt;
            l *= alpha;
          }
          tile_sum = make_p(m_used);
        }
        l += tile_sum;
        pass_turn();
        tmem_st32(lane_addr + s_col, u);
      } else {
        const float mt = tile_max();
        need = mt > m_used + kRescaleLog2;
        if (need) {
          alpha = ex2(m_used - mt);
          m_used = mt;
          l *= alpha;
        }
        const float neg_m = -m_used;
        float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
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
        l += ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
        pass_turn();
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // rescale this warp's rows of O_t
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
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBarPFull + t));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(o_full, 0, abort, status, 11));
    if (ok) {
      // ---- epilogue: O / l -> fp32 partial rows, log2-LSE.  Each warp transposes its 32 rows
      // through 4 KB of its tile's Q area (free: every product of the group has completed) so
      // that the global stores are whole 128-byte row segments.
      tc_fence_after();
      const int wq = warp & 3;
      float* stage = reinterpret_cast<float*>(gbase + C::kOffQ + t * C::kQBytes + wq * 4096);  // [32][32]
      const int row0 = row_base + t * kRows + wq * 32;  // block row of lane 0
      const int live_rows = min(32, m_eff - row0);
      const int64_t grow0 = row_offset + static_cast<int64_t>(h) * m_eff + row0;
      const float inv = out_scale / l;
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(lane_addr + o_col + c * 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 8; ++q)  // 16-byte chunk q of this lane's row, XOR-swizzled by row
          *reinterpret_cast<float4*>(stage + lane * 32 + ((q ^ (lane & 7)) << 2)) =
              make_float4(__uint_as_float(u[4 * q]) * inv, __uint_as_float(u[4 * q + 1]) * inv,
                          __uint_as_float(u[4 * q + 2]) * inv, __uint_as_float(u[4 * q + 3]) * inv);
        __syncwarp();
#pragma unroll
        for (int k0 = 0; k0 < 32; k0 += 4) {  // four rows per instruction, eight lanes per row
          const int row = k0 + (lane >> 3);
          if (row < live_rows) {
            const float4 val = *reinterpret_cast<const float4*>(stage + row * 32 + (((lane & 7) ^ (row & 7)) << 2));
            *reinterpret_cast<float4*>(p.o_pre + (grow0 + row) * kD + c * 32 + (lane & 7) * 4) = val;
          }
        }
        __syncwarp();
      }
      if (live) p.lse_pre[grow0 + lane] = m_used + __log2f(l);
      __threadfence();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpP) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // arrivals of the block's members whose (b, h) counters need them; the arrival that
  // completes a member merges it (shared memory is free: every product and copy is done)
  if (!*abort && *any_arrive) prefix_arrive_and_merge_flagged<kD>(p, members, h, row_base, n_rows, flags);
  if (!*abort) prefix_rows_done(p, n_rows);
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
  const int grid = num_items * p.hkv;
  // one TMA box per page costs the copy engine more than the producer warp's own 16-byte
  // copies once pages hold few tokens: up to 2 for e4m3 (dense kernel on the e4m3 batch:
  // 1,148 against 375 us at page size 1, 346 against ~375 us at 4), up to 4 for bf16 (agent
  // batch: 49.2 against 43.5 us at page size 4, 34.9 against 43.2 us at 8)
  if (p.token_flat || p.page_shift <= (FP8 ? 1 : 2)) {
    e = ensure_smem_limit<prefix_dense_kernel<FP8, true>>(bytes);
    if (e != cudaSuccess) return e;
    prefix_dense_kernel<FP8, true><<<grid, kThreads, bytes, s>>>(p, kmap, vmap, static_cast<int>(slots));
  } else {
    e = ensure_smem_limit<prefix_dense_kernel<FP8, false>>(bytes);
    if (e != cudaSuccess) return e;
    prefix_dense_kernel<FP8, false><<<grid, kThreads, bytes, s>>>(p, kmap, vmap, static_cast<int>(slots));
  }
  return cudaGetLastError();
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// True when the tcgen05 dense kernel serves this configuration (bf16 or e4m3 K/V, d = 128).
bool dense_tc_supported(const StepParams& p) {
  return (p.kv_dtype == PSP_KV_BF16 || p.kv_dtype == PSP_KV_FP8) && p.head_dim == kD;
}

cudaError_t launch_prefix_dense_tc(const StepParams& p, int num_items, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  return p.kv_dtype == PSP_KV_FP8 ? launch_t<true>(p, num_items, s) : launch_t<false>(p, num_items, s);
}

}  // namespace psp
