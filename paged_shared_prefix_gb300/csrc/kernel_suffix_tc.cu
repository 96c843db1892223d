// kernel_suffix_tc.cu -- split-KV paged decode over each request's private
// suffix for fp8-e4m3 K/V at d = 128, on the 5th-generation tensor cores, as
// one persistent CTA per SM.  Selected with PSP_SUFFIX_TC=1: it is exact, but on
// GB300 it measured slower than the mma.sync kernel in kernel_suffix.cu, which
// stays the default (its per-item epilogue throttles the stream; see the design
// notes for the measurements).
//
// Same work as the suffix kernel in kernel_suffix.cu (one item = one (split, KV
// head); all G <= 8 query heads of the KV head are served from one read of each
// K/V byte), but both products run natively on e4m3 codes with kind::f8f6f4
// tcgen05.mma, so no key or value code is converted on the CUDA cores, and the
// CTA streams item after item through one pipeline that never drains:
//   warp 11 (schedule)   takes items from a grid-wide counter and resolves them (split,
//                        KV head, request, token range) up to 16 items ahead, copying
//                        each item's block-table entries into shared memory (a lookup
//                        from global memory is one DRAM round trip per tile);
//   warp 8 (producer)    TMA-loads the items' K and V rows through the block table in
//                        128-token tiles (3-D pool maps [slot][kv head][d], boxes of
//                        min(page size, 64) tokens, 128-byte swizzle), K and V of a tile
//                        in one ring stage whose metadata names the item and the tile,
//                        with the block-table entries of the next tile already loaded;
//   warp 10 (queries)    quantises the next item's query rows to e4m3 (per-row scale
//                        amax/448) into one of two query buffers;
//   warp 9 (MMA)         one lane issues, whichever is ready first, S^T = K Q^T
//                        (M = 128 tokens, N = 16: the query heads padded, K = 128)
//                        into one of two TMEM score buffers, and O^T += V^T P^T
//                        (M = 128 = d, N = 16, K = 128 tokens) into one of two TMEM
//                        output buffers, with V read MN-major straight from its tile
//                        and P^T from shared memory;
//   warps 0-3 (softmax)  one thread per token row of a tile (= TMEM lane): scores of
//                        its 8 heads, exp2 against a reference max per head, the P^T
//                        row as 8 e4m3 codes;
//   warps 4-7 (epilogue) one thread per d (= TMEM lane of O^T): at an item's end,
//                        normalise its output and deliver it (merged with the
//                        request's shared-prefix rows, or as a partial through the
//                        (request, KV head) counter) while the next item streams.
// The reference max moves lazily: a tile whose scores would give a probability above
// 2^8 (near e4m3's largest finite value) starts an exchange of the tile's maxima among
// the softmax warps, after which that tile's max maps to 2^4 (small probabilities stay
// clear of e4m3's subnormals) and O^T is rescaled in tensor memory; otherwise a tile
// costs the softmax warps one barrier.  The per-KV-head key scale folds into the score
// scale and the value scale into the output ("GraniKV", section 2: each request's
// private suffix is read through its block table).
// Every mbarrier wait is bounded and watches a CTA-wide abort flag; each warp group
// takes its decisions to leave through barrier reductions, so no warp waits at a
// barrier for one that has left.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>

#include "psp_device.cuh"
#include "psp_internal.h"
#include "psp_merge.cuh"
#include "psp_sm100.cuh"
#include "psp_suffix_epi.cuh"

namespace psp {
namespace {

using namespace dev;
using namespace sm100;

constexpr int kTok = 128;             // tokens per K/V tile (M of the score product, K of the value product)
constexpr int kD = 128;               // head dim (K of the score product, M of the value product)
constexpr int kN = 16;                // query heads padded to the MMA's smallest N at M = 128
constexpr int kWarpE = 4, kWarpP = 8, kWarpM = 9, kWarpQ = 10, kWarpS = 11;
constexpr int kThreads = 384;
constexpr int kMaxBoxes = 4;          // TMA boxes of a tile per producer lane (page size 1: 128 / 32)
constexpr int kTabEntries = 160;      // block-table entries staged per item (2048 tokens at page size 16)
constexpr int kSlots = 16;            // items in flight inside one CTA, at most
constexpr uint32_t kTmemCols = 64;    // S^T buffers [0, 16) [16, 32), O^T buffers [32, 48) [48, 64)
constexpr uint32_t kOCol = 32;
constexpr float kPMaxLog2 = 8.f;      // a probability above 2^8 moves the reference max
constexpr float kPTopLog2 = 4.f;      // after a move the tile's max maps to 2^4
constexpr uint32_t kTileBytes = kTok * kD;   // one e4m3 K or V tile
constexpr uint32_t kQBytes = kN * kD;        // one e4m3 query buffer
constexpr uint32_t kPBytes = kTok * kN;      // one e4m3 P^T buffer
constexpr uint32_t kIdescS = idesc_e4m3(kTok, kN, false);
constexpr uint32_t kIdescPV = idesc_e4m3(kD, kN, true, true);

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

template <int NS>
struct TcCfg {
  static constexpr uint32_t kStageBytes = 2 * kTileBytes;           // K at +0, V at +kTileBytes
  static constexpr uint32_t kOffQ = NS * kStageBytes;                // 2 query buffers [16][128], 128-byte swizzle
  static constexpr uint32_t kOffP = kOffQ + 2 * kQBytes;             // 2 P^T buffers [128][16] (MN-major)
  static constexpr uint32_t kOffPre = kOffP + 2 * kPBytes;           // prefix rows [16][D] f32 + [16] f32
  static constexpr uint32_t kOffF = kOffPre + (kPreRows * kD + kPreRows) * 4;
  // floats: qsc [2][8] score scales, mrec [2][8] maxima, lrec [2][4][8] sums, wmax [4][8],
  // hw [8][kPreRows + 2] per-head delivery weights (up to kPreRows prefix chunks at G = 1)
  static constexpr uint32_t kOffMeta = kOffF + (128 + 8 * (kPreRows + 2)) * 4;  // int4 per ring stage
  static constexpr uint32_t kOffItem = kOffMeta + NS * 16;           // 8 ints per item slot
  static constexpr uint32_t kOffTab = kOffItem + kSlots * 64;        // int [kSlots][kTabEntries]
  static constexpr uint32_t kOffBar = kOffTab + kSlots * kTabEntries * 4;
  static constexpr int kFull = 0, kEmpty = NS, kSFull = 2 * NS, kPFull = kSFull + 2, kODone = kPFull + 2,
                       kQFull = kODone + 1, kQFree = kQFull + 2, kOReady = kQFree + 2, kOFree = kOReady + 2,
                       kItemDone = kOFree + 2, kRecFree = kItemDone + 2, kIqFull = kRecFree + 2,
                       kIqFree = kIqFull + kSlots, kDrain = kIqFree + kSlots, kNumBars = kDrain + 1;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem base, abort, ready, last
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
};

template <int NS>
__global__ void __launch_bounds__(kThreads, 1)
    suffix_tc_kernel(const StepParams p, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, int num_slots, int total_items) {
  using C = TcCfg<NS>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  auto bar = [&](int i) { return base + C::kOffBar + 8u * i; };
  volatile int* abort = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 4);
  volatile int* flag_ready = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 8);
  volatile int* flag_last = reinterpret_cast<volatile int*>(gbase + C::kOffMisc + 12);
  float* fl = reinterpret_cast<float*>(gbase + C::kOffF);
  float* qsc = fl;         // [buffer][8] score scales of the queued items
  float* mrec = fl + 16;   // [buffer][8] reference maxima of a finished item
  float* lrec = fl + 32;   // [buffer][warp][8] sums of a finished item
  float* wmax = fl + 96;   // [warp][8] tile maxima
  constexpr int kHw = kPreRows + 2;
  float* hw = fl + 128;    // [head][kHw]: own factor, prefix-chunk weights, log-sum-exp
  volatile int* meta = reinterpret_cast<volatile int*>(gbase + C::kOffMeta);  // per stage {item, tile, tiles, valid rows}
  auto meta_get = [&](int st) { return make_int4(meta[4 * st], meta[4 * st + 1], meta[4 * st + 2], meta[4 * st + 3]); };
  // item record (16 ints): split, h, b, t0, t1, tiles, list, staged, value scale (bits), one split,
  // first prefix chunk, prefix chunks, solo, prefix rows in shared memory
  volatile int* items = reinterpret_cast<volatile int*>(gbase + C::kOffItem);
  const int* tab = reinterpret_cast<const int*>(gbase + C::kOffTab);
  float* pre_o = reinterpret_cast<float*>(gbase + C::kOffPre);
  float* pre_l = pre_o + kPreRows * kD;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int32_t* status = p.status;

  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(C::kFull + s), 1);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::kSFull + i), 1);
      mbar_init(bar(C::kPFull + i), 4);     // one arrival per softmax warp
      mbar_init(bar(C::kQFull + i), 1);
      mbar_init(bar(C::kQFree + i), 5);     // the last score product's commit + the 4 softmax warps
      mbar_init(bar(C::kOReady + i), 1);
      mbar_init(bar(C::kOFree + i), 1);
      mbar_init(bar(C::kItemDone + i), 4);  // one arrival per softmax warp
      mbar_init(bar(C::kRecFree + i), 1);
    }
    mbar_init(bar(C::kODone), 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(C::kIqFull + s), 1);
      mbar_init(bar(C::kIqFree + s), 3);    // the producer, the query warp and the epilogue
    }
    mbar_init(bar(C::kDrain), 1);
    fence_mbar_init();
  }
  if (warp == kWarpP) {
    tmem_alloc(base + C::kOffMisc, kTmemCols);
    tmem_relinquish();
  } else if (warp == kWarpQ) {
    // rows 8..15 of both query buffers: the heads that pad N to 16 stay zero
    for (int i = lane; i < 2 * 64; i += 32) {
      const uint32_t off = C::kOffQ + (i >> 6) * kQBytes + 8 * 128 + (i & 63) * 16;
      *reinterpret_cast<uint4*>(gbase + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffMisc);

  if (warp == kWarpS) {
    // ---------------------------------------------------------------- schedule
    // lane 0 takes tickets (item = split * Hkv + KV head, KV head fastest); the warp
    // publishes each resolved item in the next slot of the item ring (the end of the work
    // as split -1), with the block-table entries of its tokens staged beside it when they
    // fit (entry e of the slot = table entry (t0 >> shift) + e)
    const int shift = p.token_flat ? 0 : p.page_shift;
    const int32_t* table = p.token_flat ? p.kv_indices : p.suffix_page_indices;
    int ticket = 0, next = 0;
    if (lane == 0) ticket = atomicAdd(p.work_next, 1);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    for (int k = 0;; ++k) {
      const int slot = k % kSlots;
      const bool end = ticket >= total_items;
      int split = -1, h = 0, b = 0, t0 = 0, t1 = 0, n = 0, list = 0;
      if (!end) {
        if (lane == 0) next = atomicAdd(p.work_next, 1);  // in flight while this item resolves
        split = ticket / p.hkv;
        h = ticket - split * p.hkv;
        b = p.split_req[split];
        t0 = p.split_begin[split];
        t1 = p.split_end[split];
        n = (t1 - t0 + kTok - 1) / kTok;
        list = p.token_flat ? p.kv_indptr[b] + p.suffix_start[b] : p.suffix_page_indptr[b];
      }
      // everything the epilogue needs about the item, resolved here (well ahead of its use)
      SuffixCta cta{};
      float vs = 0.f;
      int one_split = 0;
      if (!end) {
        cta = suffix_cta(p, split, h);
        vs = __ldg(p.v_scale + h);
        one_split = p.split_indptr[b + 1] - p.split_indptr[b] == 1;
      }
      int ok = 1;
      if (k >= kSlots && lane == 0) ok = wait_or_abort_sleep(bar(C::kIqFree + slot), ((k / kSlots) - 1) & 1, abort, status, 32);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int first = t0 >> shift;
      const int cnt = end ? 0 : ((t1 - 1) >> shift) - first + 1;
      const bool staged = cnt <= kTabEntries;
      if (!end && staged) {
        int* t = const_cast<int*>(tab) + slot * kTabEntries;
        for (int e = lane; e < cnt; e += 32) t[e] = __ldg(table + list + first + e);
      }
      __syncwarp();
      if (lane == 0) {
        volatile int* it = items + slot * 16;
        it[0] = split;
        it[1] = h;
        it[2] = b;
        it[3] = t0;
        it[4] = t1;
        it[5] = n;
        it[6] = list;
        it[7] = staged ? 1 : 0;
        it[8] = __float_as_int(vs);
        it[9] = one_split;
        it[10] = cta.c0;
        it[11] = cta.n_chunks;
        it[12] = cta.solo ? 1 : 0;
        it[13] = cta.pre_smem ? 1 : 0;
        mbar_arrive(bar(C::kIqFull + slot));
      }
      __syncwarp();
      if (end) break;
      ticket = __shfl_sync(0xffffffffu, next, 0);
    }
  } else if (warp == kWarpP) {
    // ---------------------------------------------------------------- producer
    auto lane0_wait = [&](uint32_t b, uint32_t parity, int site) {
      int ok = 0;
      if (lane == 0) ok = wait_or_abort_sleep(b, parity, abort, status, site) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
    }
    const int32_t* table = p.token_flat ? p.kv_indices : p.suffix_page_indices;
    const int shift = p.token_flat ? 0 : p.page_shift;
    const int mask = (1 << shift) - 1;
    const int br = min(1 << shift, 64);  // rows per TMA box
    // pool slots of this lane's boxes (box i: rows (lane + 32 i) br ..) of tile j of an
    // item; rows at or past t1 read slot num_slots, out of the map (zero fill)
    struct Item {
      int split, h, t0, t1, n, first;
      const int32_t* list;  // the item's block-table row in global memory
      const int* staged;    // its entries from `first` on in shared memory, or null
    };
    auto lookup = [&](const Item& it, int j, int (&sl)[kMaxBoxes]) {
#pragma unroll
      for (int i = 0; i < kMaxBoxes; ++i) {
        const int r = (lane + 32 * i) * br;
        const int tok = it.t0 + j * kTok + r;
        int slot = num_slots;
        if (r < kTok && tok < it.t1) {
          const int e = tok >> shift;
          slot = ((it.staged ? it.staged[e - it.first] : __ldg(it.list + e)) << shift) | (tok & mask);
        }
        sl[i] = slot;
      }
    };
    auto read_item = [&](int k, Item& it) {
      const int slot = k % kSlots;
      if (!lane0_wait(bar(C::kIqFull + slot), (k / kSlots) & 1, 33)) return false;
      volatile int* v = items + slot * 16;
      it.split = v[0];
      it.h = v[1];
      it.t0 = v[3];
      it.t1 = v[4];
      it.n = v[5];
      it.list = table + v[6];
      it.first = it.t0 >> shift;
      it.staged = v[7] ? tab + slot * kTabEntries : nullptr;
      return true;
    };
    Item cur;
    int sl[kMaxBoxes];
    bool ok = read_item(0, cur), marker = false;
    if (ok && cur.split >= 0) lookup(cur, 0, sl);
    int k = 0, gl = 0;
    while (ok && cur.split >= 0) {
      Item nxt = cur;
      for (int j = 0; j < cur.n; ++j, ++gl) {
        // the next tile's block-table entries are in flight while this tile waits for its stage
        int sn[kMaxBoxes];
        if (j + 1 < cur.n) {
          lookup(cur, j + 1, sn);
        } else {
          if (!(ok = read_item(k + 1, nxt))) break;
          if (nxt.split >= 0) lookup(nxt, 0, sn);
        }
        const int st = gl % NS;
        if (gl >= NS && !(ok = lane0_wait(bar(C::kEmpty + st), ((gl / NS) - 1) & 1, 34))) break;
        const uint32_t full = bar(C::kFull + st), dst = base + st * C::kStageBytes;
        if (lane == 0) {
          meta[4 * st] = k;
          meta[4 * st + 1] = j;
          meta[4 * st + 2] = cur.n;
          meta[4 * st + 3] = cur.t1 - (cur.t0 + j * kTok);
          mbar_arrive_tx(full, 2 * kTileBytes);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kMaxBoxes; ++i) {
          const int r = (lane + 32 * i) * br;
          if (r < kTok) {
            tma_load_3d(dst + r * 128, &kmap, 0, cur.h, sl[i], full);
            tma_load_3d(dst + kTileBytes + r * 128, &vmap, 0, cur.h, sl[i], full);
          }
        }
#pragma unroll
        for (int i = 0; i < kMaxBoxes; ++i) sl[i] = sn[i];
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(bar(C::kIqFree + k % kSlots));
      ++k;
      cur = nxt;
    }
    if (ok) {
      // end marker: a stage without copies whose metadata stops the MMA and softmax warps
      const int st = gl % NS;
      if (gl < NS || lane0_wait(bar(C::kEmpty + st), ((gl / NS) - 1) & 1, 34)) {
        if (lane == 0) {
          meta[4 * st] = -1;
          mbar_arrive(bar(C::kFull + st));
        }
        marker = true;
      }
    }
    // drain: every issued copy has landed before the CTA may exit (the marker's stage
    // reused tile gl - NS's barrier after that tile was consumed)
    if (lane == 0)
      for (int t = max(0, gl - NS + (marker ? 1 : 0)); t < gl; ++t)
        mbar_wait(bar(C::kFull + t % NS), (t / NS) & 1, status, 35);
    __syncwarp();
  } else if (warp == kWarpM) {
    // -------------------------------------------------------------------- MMA
    auto all = [](bool v) { return __all_sync(0xffffffffu, v); };
    // S^T = K Q^T for tile g into score buffer g & 1 (both operands K-major, 32 bytes of d per step)
    auto issue_s = [&](int g, int qb) {
      const uint32_t kb = base + (g % NS) * C::kStageBytes, qbase = base + C::kOffQ + qb * kQBytes;
#pragma unroll
      for (int ks = 0; ks < kD / 32; ++ks)
        mma_ss_f8(tmem + (g & 1) * kN, sw128_desc(kb + ks * 32, 16, 1024), sw128_desc(qbase + ks * 32, 16, 1024),
                  kIdescS, ks > 0 ? 1u : 0u);
    };
    // O^T += V^T P^T for tile g into output buffer ob: V is the MN-major A operand as loaded
    // (K = tokens advance by whole 128-byte rows), P^T the MN-major B operand [token][16 heads]
    auto issue_pv = [&](int g, int ob, bool accumulate) {
      const uint32_t vb = base + (g % NS) * C::kStageBytes + kTileBytes, pb = base + C::kOffP + (g & 1) * kPBytes;
#pragma unroll
      for (int ks = 0; ks < kTok / 32; ++ks)
        mma_ss_f8(tmem + kOCol + ob * kN, sw128_desc(vb + ks * 32 * 128, kTileBytes, 1024),
                  plain_desc(pb + ks * 32 * kN, 128), kIdescPV, (accumulate || ks > 0) ? 1u : 0u);
    };
    auto meta_of = [&](int g) { return meta_get(g % NS); };
    // the score product of tile g (item m.x, tile m.y of m.z), or the end marker's signal
    auto start_tile = [&](int g, int4 m) {
      if (m.x < 0) {
        if (lane == 0) mma_commit(bar(C::kSFull + (g & 1)));  // nothing to wait for: the softmax reads the marker
        __syncwarp();
        return true;
      }
      const int qb = m.x & 1;
      if (m.y == 0 && !all(wait_or_abort_sleep(bar(C::kQFull + qb), (m.x >> 1) & 1, abort, status, 36))) return false;
      if (lane == 0) {
        tc_fence_after();
        issue_s(g, qb);
        mma_commit(bar(C::kSFull + (g & 1)));
        if (m.y == m.z - 1) mma_commit(bar(C::kQFree + qb));  // the item's last read of its query buffer
      }
      __syncwarp();
      return true;
    };
    // Issue whichever product is ready: the score product of tile gs once its copy has
    // landed and its score buffer is free (the softmax of tile gs - 2 is done, gp >= gs - 1),
    // the value product of tile gp once its probabilities are written.  Neither waits for
    // the other, so a stage is released as soon as its tile's value product completes.
    int gs = 0, gp = 0, end_at = -1;
    int4 mt0 = make_int4(-1, 0, 0, 0), mt1 = mt0;  // metadata of the tiles in flight (by tile parity)
    bool ok = true;
    uint32_t idle = 0;
    while (ok) {
      bool progress = false;
      if (end_at < 0 && gs <= gp + 1 && all(mbar_test_wait(bar(C::kFull + gs % NS), (gs / NS) & 1))) {
        const int4 m = meta_of(gs);
        if (!(ok = start_tile(gs, m))) break;
        if (m.x < 0) end_at = gs;
        if (gs & 1) mt1 = m; else mt0 = m;
        ++gs;
        progress = true;
      }
      if (gp < gs && gp != end_at && all(mbar_test_wait(bar(C::kPFull + (gp & 1)), (gp >> 1) & 1))) {
        const int4 m = (gp & 1) ? mt1 : mt0;
        const int ob = m.x & 1;
        // the item's first product overwrites its output buffer: the epilogue of item m.x - 2 has read it
        if (m.y == 0 && m.x >= 2 &&
            !(ok = all(wait_or_abort_sleep(bar(C::kOFree + ob), ((m.x >> 1) - 1) & 1, abort, status, 40))))
          break;
        if (lane == 0) {
          tc_fence_after();
          issue_pv(gp, ob, m.y > 0);
          mma_commit(bar(C::kODone));
          mma_commit(bar(C::kEmpty + gp % NS));
          if (m.y == m.z - 1) mma_commit(bar(C::kOReady + ob));
        }
        __syncwarp();
        ++gp;
        progress = true;
      }
      if (end_at >= 0 && gp == end_at) break;
      if (progress) {
        idle = 0;
      } else if ((++idle & 255) != 0) {
        __nanosleep(32);  // leaves the sub-partition's issue slots to working warps
      } else if (*abort || idle >= (1u << 24)) {
        if (!*abort) {
          atomicCAS(status, 0, kDevTimeout | (38 << 8));
          *abort = 1;
        }
        ok = false;
      }
    }
    if (lane == 0) {
      // every product of the CTA has completed before the tensor memory is freed
      mma_commit(bar(C::kDrain));
      mbar_wait(bar(C::kDrain), 0, status, 41);
    }
    __syncwarp();
  } else if (warp == kWarpQ) {
    // -------------------------------------------------------------- query rows
    for (int k = 0;; ++k) {
      const int slot = k % kSlots;
      if (!__all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kIqFull + slot), (k / kSlots) & 1, abort, status, 42))) break;
      const int split = items[slot * 16], h = items[slot * 16 + 1], b = items[slot * 16 + 2];
      if (split < 0) break;
      const int qb = k & 1;
      // the buffer's previous item (k - 2) has had its last score product and its scales read
      if (k >= 2 && !__all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kQFree + qb), ((k >> 1) - 1) & 1, abort, status, 43)))
        break;
      const int G = p.group;
      const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) + (static_cast<int64_t>(b) * p.hq + h * G) * kD;
      uint2 v[8];  // lane: d = 4 lane .. 4 lane + 3 of each query row
#pragma unroll
      for (int g = 0; g < 8; ++g)
        v[g] = g < G ? __ldg(reinterpret_cast<const uint2*>(qrow + g * kD) + lane) : make_uint2(0u, 0u);
      const float kscale = p.scale_log2 * __ldg(p.k_scale + h);
      unsigned char* qbuf = gbase + C::kOffQ + qb * kQBytes;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const float f0 = bf16_bits_to_float(v[g].x & 0xffff), f1 = bf16_bits_to_float(v[g].x >> 16);
        const float f2 = bf16_bits_to_float(v[g].y & 0xffff), f3 = bf16_bits_to_float(v[g].y >> 16);
        const float amax = xor_max<1, 16>(fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3))));
        const float qs = amax > 0.f ? amax / 448.f : 1.f;
        const float inv = 1.f / qs;
        // bytes 4 lane .. 4 lane + 3 of row g: 16-byte chunk lane / 4, XOR-swizzled by the row
        *reinterpret_cast<uint32_t*>(qbuf + g * 128 + (((lane >> 2) ^ g) << 4) + (lane & 3) * 4) =
            e4m3x4_from_floats(f0 * inv, f1 * inv, f2 * inv, f3 * inv);
        if (lane == 0) qsc[qb * 8 + g] = qs * kscale;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(C::kQFull + qb));
        mbar_arrive(bar(C::kIqFree + slot));
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------- softmax warps 0-3
    const int r = threadIdx.x;  // token row of a tile = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float sc[8], M[8], L[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      sc[g] = 0.f;
      M[g] = neg_inf();
      L[g] = 0.f;
    }
    bool bad = false;
    for (int g = 0;; ++g) {
      const int buf = g & 1;
      const bool got =
          !bad && __all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kSFull + buf), (g >> 1) & 1, abort, status, 44));
      int4 m = make_int4(-1, 0, 0, 0);
      float x[8];
      bool need = false;
      if (got) m = meta_get(g % NS);
      if (m.x >= 0) {
        if (m.y == 0) {
          // a new item: its score scales were written before its first score product
#pragma unroll
          for (int h8 = 0; h8 < 8; ++h8) {
            sc[h8] = qsc[(m.x & 1) * 8 + h8];
            M[h8] = neg_inf();
            L[h8] = 0.f;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::kQFree + (m.x & 1)));
        }
        tc_fence_after();
        uint32_t u[8];
        tmem_ld8(lane_addr + buf * kN, u);
        tmem_wait_ld();
        const bool valid = r < m.w;
#pragma unroll
        for (int h8 = 0; h8 < 8; ++h8) {
          x[h8] = valid ? __uint_as_float(u[h8]) * sc[h8] : neg_inf();
          need |= x[h8] > M[h8] + kPMaxLog2;
        }
      }
      // one barrier per tile; a second only when some warp stops or a reference max moves
      if (group_bar_or(1, 128, !got || m.x < 0 || need)) {
        if (group_bar_or(1, 128, !got || m.x < 0)) break;  // a failed wait, or the end of the work
        // the tile's maxima over its 128 tokens, the same in every thread
#pragma unroll
        for (int h8 = 0; h8 < 8; ++h8) {
          const float wm = xor_max<1, 16>(x[h8]);
          if (lane == 0) wmax[warp * 8 + h8] = wm;
        }
        named_bar_sync(1, 128);
        float alpha[8];
        bool moved = false;
#pragma unroll
        for (int h8 = 0; h8 < 8; ++h8) {
          const float tm = fmaxf(fmaxf(wmax[h8], wmax[8 + h8]), fmaxf(wmax[16 + h8], wmax[24 + h8]));
          alpha[h8] = 1.f;
          if (tm > M[h8] + kPMaxLog2) {
            const float mn = tm - kPTopLog2;
            alpha[h8] = ex2(M[h8] - mn);
            M[h8] = mn;
            moved = true;
          }
        }
        if (moved) {  // the same in every thread
#pragma unroll
          for (int h8 = 0; h8 < 8; ++h8) L[h8] *= alpha[h8];
          if (m.y > 0) {
            // O^T holds exactly the item's tiles before g once the product of tile g - 1 has
            // completed (the product of tile g waits for this warp); rescale this warp's rows
            if (__all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kODone), (g - 1) & 1, abort, status, 45))) {
              tc_fence_after();
              const uint32_t oc = lane_addr + kOCol + (m.x & 1) * kN;
              uint32_t o[8];
              tmem_ld8(oc, o);
              tmem_wait_ld();
#pragma unroll
              for (int h8 = 0; h8 < 8; ++h8) o[h8] = __float_as_uint(__uint_as_float(o[h8]) * alpha[h8]);
              tmem_st8(oc, o);
              tmem_wait_st();
            } else {
              bad = true;  // the abort flag is up: the next tile's barrier takes every warp out
            }
          }
        }
        // wmax is written again only after a later tile's first barrier, which every thread
        // reaches after its reads above
      }
      // row r of P^T: the 8 heads' e4m3 probabilities, the 8 padding heads zero
      float pr[8];
#pragma unroll
      for (int h8 = 0; h8 < 8; ++h8) {
        pr[h8] = ex2(x[h8] - M[h8]);
        L[h8] += pr[h8];
      }
      *reinterpret_cast<uint4*>(gbase + C::kOffP + buf * kPBytes + r * kN) =
          make_uint4(e4m3x4_from_floats(pr[0], pr[1], pr[2], pr[3]), e4m3x4_from_floats(pr[4], pr[5], pr[6], pr[7]),
                     0u, 0u);
      if (r >= m.w) {
        // a row past the item's end: the rest of a partly used page may hold any bytes, and
        // 0 * NaN would reach every output of the value product, so the row is zeroed (the
        // wait re-observes the tile's completed copy before the generic-proxy writes)
        if (wait_or_abort_sleep(bar(C::kFull + g % NS), (g / NS) & 1, abort, status, 46)) {
          uint4* vrow = reinterpret_cast<uint4*>(gbase + (g % NS) * C::kStageBytes + kTileBytes + r * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kPFull + buf));
      if (m.y == m.z - 1) {
        // the item's last tile: this warp's sums and the reference maxima for the epilogue,
        // once the epilogue of item m.x - 2 has read the records of this buffer
        const int rb = m.x & 1;
        if (m.x >= 2 &&
            !__all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kRecFree + rb), ((m.x >> 1) - 1) & 1, abort, status, 47)))
          bad = true;
        if (!bad) {
#pragma unroll
          for (int h8 = 0; h8 < 8; ++h8) {
            const float s = xor_sum<1, 16>(L[h8]);
            if (lane == 0) lrec[rb * 32 + warp * 8 + h8] = s;
            if (warp == 0 && lane == h8) mrec[rb * 8 + h8] = M[h8];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::kItemDone + rb));
        }
      }
    }
  } else if (warp < kWarpE + 4) {
    // ------------------------------------------------------ epilogue warps 4-7
    const int d = threadIdx.x - kWarpE * 32;  // row of O^T = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int G = p.group;
    bool waited_primary = false;
    for (int k = 0;; ++k) {
      const int slot = k % kSlots;
      const bool got =
          __all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kIqFull + slot), (k / kSlots) & 1, abort, status, 48));
      const int split = got ? items[slot * 16] : -1;
      if (group_bar_or(2, 128, !got || split < 0)) break;
      const int h = items[slot * 16 + 1];
      SuffixCta cta;
      {
        volatile int* it = items + slot * 16;
        cta.split = split;
        cta.h = h;
        cta.b = it[2];
        cta.c0 = it[10];
        cta.n_chunks = it[11];
        cta.solo = it[12] != 0;
        cta.pre_smem = it[13] != 0;
        cta.wait_prefix = p.pdl && !p.concurrent;
      }
      if (cta.wait_prefix && !waited_primary) {
        pdl_wait_primary();  // prefix partials are read only after the prefix grid has completed
        waited_primary = true;
      }
      if (cta.pre_smem) prefetch_prefix_rows<kD, 128>(p, cta, pre_o, pre_l, d);
      cp_async_commit();
      const float vs = __int_as_float(items[slot * 16 + 8]);
      const int b = cta.b;
      const bool one_split = items[slot * 16 + 9] != 0;
      // the item's softmax records and its last value product
      const int ob = k & 1;
      const bool ok =
          __all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kItemDone + ob), (k >> 1) & 1, abort, status, 49)) &&
          __all_sync(0xffffffffu, wait_or_abort_sleep(bar(C::kOReady + ob), (k >> 1) & 1, abort, status, 50));
      if (group_bar_or(2, 128, !ok)) break;
      tc_fence_after();
      uint32_t u[8];
      tmem_ld8(lane_addr + kOCol + ob * kN, u);
      tmem_wait_ld();
      float Mx[8], Ls[8];
#pragma unroll
      for (int h8 = 0; h8 < 8; ++h8) {
        Mx[h8] = mrec[ob * 8 + h8];
        Ls[h8] = (lrec[ob * 32 + h8] + lrec[ob * 32 + 8 + h8]) + (lrec[ob * 32 + 16 + h8] + lrec[ob * 32 + 24 + h8]);
      }
      tc_fence_before();
      named_bar_sync(2, 128);  // every epilogue thread holds its O^T row and the records
      if (d == 0) {
        mbar_arrive(bar(C::kOFree + ob));
        mbar_arrive(bar(C::kRecFree + ob));
        mbar_arrive(bar(C::kIqFree + slot));
      }
      cp_async_wait<0>();
      // Launched as a dependent of a still running prefix kernel: a one-split request whose
      // prefix partials are all complete merges them here like a solo request.
      bool ready = false;
      if (p.pdl && p.concurrent && one_split && cta.n_chunks > 0) {
        if (d == 0) *flag_ready = *reinterpret_cast<volatile int32_t*>(p.prefix_done) == p.prefix_rows_total;
        named_bar_sync(2, 128);
        ready = *flag_ready != 0;
        if (ready) __threadfence();  // the prefix partials were fenced before their rows were counted
      }
      named_bar_sync(2, 128);  // the prefetched prefix rows are visible to every thread
      const bool only_part = one_split && cta.n_chunks == 0;
      const bool direct = only_part || (cta.solo && cta.pre_smem);
      const bool solo_global = (cta.solo && !direct) || ready;
      const int64_t row0 = (static_cast<int64_t>(split) * p.hkv + h) * G;
      const int64_t orow0 = static_cast<int64_t>(b) * p.hq + h * G;
      // per head, once: the own part's factor (value scale / sum) and log2-LSE, and for a
      // direct delivery the weights of the prefix chunks' rows and of the own part, all
      // divided by their sum (prefix chunks first, then the own part)
      if (d < G) {
        // SFU approximations and one reciprocal: this runs as one dependent chain per head
        // on a few lanes of one warp, between the item's end and its delivery
        const int hd = d;
        float lse_own = 0.f, l_own = 1.f;
#pragma unroll
        for (int h8 = 0; h8 < 8; ++h8)
          if (h8 == hd) {
            lse_own = Mx[h8] + __log2f(Ls[h8]);
            l_own = Ls[h8];
          }
        float* w = hw + hd * kHw;
        if (direct) {
          float big = lse_own;
          for (int ch = 0; ch < cta.n_chunks; ++ch) big = fmaxf(big, pre_l[ch * G + hd]);
          const float w_own = ex2(lse_own - big);
          float wsum = w_own;
          for (int ch = 0; ch < cta.n_chunks; ++ch) {
            const float wc = ex2(pre_l[ch * G + hd] - big);
            w[1 + ch] = wc;
            wsum += wc;
          }
          const float inv = __frcp_rn(wsum);
          for (int ch = 0; ch < cta.n_chunks; ++ch) w[1 + ch] *= inv;
          w[0] = w_own * inv * vs * __frcp_rn(l_own);
          w[kHw - 1] = big + __log2f(wsum);
          if (p.lse) p.lse[orow0 + hd] = w[kHw - 1] * 0.6931471805599453f;
        } else {
          w[0] = vs * __frcp_rn(l_own);
          w[kHw - 1] = lse_own;
        }
      }
      named_bar_sync(2, 128);
#pragma unroll
      for (int h8 = 0; h8 < 8; ++h8) {
        if (h8 < G) {
          const float* w = hw + h8 * kHw;
          float out = __uint_as_float(u[h8]) * w[0];
          if (direct) {
            for (int ch = 0; ch < cta.n_chunks; ++ch) out = fmaf(w[1 + ch], pre_o[(ch * G + h8) * kD + d], out);
            store_final(p, orow0 + h8, d, out);
          } else {
            p.o_suf[(row0 + h8) * kD + d] = out;
            if (d == 0) p.lse_suf[row0 + h8] = w[kHw - 1];
          }
        }
      }
      if (!direct) {
        __threadfence();
        named_bar_sync(2, 128);
        bool merge = solo_global;
        if (!solo_global) {
          if (d == 0) *flag_last = arrive_is_last(p, b, h) ? 1 : 0;
          named_bar_sync(2, 128);
          merge = *flag_last != 0;
        }
        if (merge)
          for (int rr = warp - kWarpE; rr < G; rr += 4) merge_row<kD>(p, b, h * G + rr, lane);
        // every prefix arrival on (b, h) was made and nothing else arrives: clear it for the next step
        if (ready && d == 0) p.counters[static_cast<int64_t>(b) * p.hkv + h] = 0;
      }
      named_bar_sync(2, 128);  // the prefix-row area and the flags are free for the next item
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpP) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // the grid's last CTA returns the work counter to zero for the next step (every CTA
    // has taken its last item before it counts itself here)
    __threadfence();
    if (atomicAdd(p.work_done, 1) == static_cast<int>(gridDim.x) - 1) {
      *p.work_next = 0;
      *p.work_done = 0;
    }
  }
  // sequential dependent launch: every CTA has waited for the prefix grid before it ends
  if (p.pdl && !p.concurrent) pdl_wait_primary();
  suffix_grid_tail(p);
}

template <int NS>
cudaError_t launch_t(const StepParams& p, int num_splits, cudaStream_t s) {
  const int64_t slots = static_cast<int64_t>(p.num_pages) * p.page_size;
  if (slots >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  const int rows = p.token_flat ? 1 : (p.page_size < 64 ? p.page_size : 64);
  CUtensorMap kmap, vmap;
  cudaError_t e = make_pool_map(&kmap, p.k_pool, slots, p.hkv, rows, true);
  if (e != cudaSuccess) return e;
  e = make_pool_map(&vmap, p.v_pool, slots, p.hkv, rows, true);
  if (e != cudaSuccess) return e;
  constexpr uint32_t bytes = TcCfg<NS>::kSmemBytes;
  static_assert(bytes <= 232448, "suffix CTA exceeds the shared memory of one SM");
  auto kern = suffix_tc_kernel<NS>;
  e = ensure_smem_limit<suffix_tc_kernel<NS>>(bytes);
  if (e != cudaSuccess) return e;
  const int total = num_splits * p.hkv;
  const int grid = total < p.num_sms ? total : (p.num_sms > 0 ? p.num_sms : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, p, kmap, vmap, static_cast<int>(slots), total);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Ring depth of the tensor-core suffix kernel (PSP_SUFFIX_TC_STAGES overrides it for
// tuning sweeps): 6 stages of 32 KB (K and V of 128 tokens) per SM.
cudaError_t launch_suffix_tc(const StepParams& p, int num_splits, cudaStream_t s) {
  static const int env = [] {
    const char* v = std::getenv("PSP_SUFFIX_TC_STAGES");
    return v ? std::atoi(v) : 0;
  }();
  switch (env) {
    case 4: return launch_t<4>(p, num_splits, s);
    case 5: return launch_t<5>(p, num_splits, s);
    default: return launch_t<6>(p, num_splits, s);
  }
}

}  // namespace psp
