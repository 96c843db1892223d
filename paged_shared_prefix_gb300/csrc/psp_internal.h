// psp_internal.h -- structures shared by the host side (plan, C ABI) and the
// kernels of the paged shared-prefix decode step.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

// Element type codes (same values as the public PSP_DTYPE_*).
#define PSP_KV_F32 0
#define PSP_KV_BF16 1
#define PSP_KV_FP8 2

namespace psp {

constexpr int kMaxGroupSize = 8;        // query heads per KV head handled per CTA row set
constexpr int kTileTokens = 64;         // partition granule (tokens)
constexpr int kCascadeRows = 64;        // stacked query rows per cascade prefix CTA
constexpr int kDenseRows = 256;         // stacked query rows per dense prefix CTA (two 128-row tiles)
constexpr int kWorkspaceAlign = 256;

// Device status codes written instead of faulting.
constexpr int32_t kDevOk = 0;
constexpr int32_t kDevTimeout = 1;
constexpr int32_t kDevBadIndex = 2;

// Everything a kernel of the step reads: configuration, caller tensors, the
// uploaded plan and the partial-result buffers in the workspace.
// Everything a suffix CTA needs to know about its split, in one 128-byte record, so that
// the CTA's first load is not followed by loads that depend on it (each is a DRAM round
// trip before the first K/V copy can be issued).
struct SplitDesc {
  int32_t b;           // request
  int32_t t0, t1;      // suffix tokens [t0, t1) of b
  int32_t list_paged;  // b's first entry in suffix_page_indices
  int32_t list_flat;   // b's first suffix entry in kv_indices (kv_indptr[b] + suffix_start[b])
  int32_t part0;       // b's prefix parts [part0, part0 + n_parts) of req_part (none: 0, 0)
  int32_t n_parts;
  int32_t one_split;   // 1: b has exactly one suffix split
  int32_t pad[8];
  // page size >= 16: the page of 16-token sub-tile s (tokens t0 + 16s ..) for s < kDescPages,
  // -1 past t1, so that a CTA's first copies need no block-table load; unused below 16
  int32_t first_page[16];
};
constexpr int kDescPages = 16;
static_assert(sizeof(SplitDesc) == 128, "one 128-byte record per split");
constexpr int kSplitDescInts = static_cast<int>(sizeof(SplitDesc) / sizeof(int32_t));

// Everything a dense prefix CTA needs about its work item in one 32-byte record (two 16-byte
// loads), so that its member list and block list are one dependent load away, not four.
struct DenseItemDesc {
  int32_t chunk;       // prefix chunk
  int32_t rb;          // 256-row block of the chunk's group
  int32_t t0, t1;      // the chunk's context tokens [t0, t1)
  int32_t m_eff;       // stacked rows of the group
  int32_t member_base; // the group's first entry in group_members
  int32_t list_base;   // the group's first entry in group_page_indices, or (token-flat) its first
                       // member's first entry in kv_indices
  int32_t row_offset;  // chunk_row_offset of the chunk
};
static_assert(sizeof(DenseItemDesc) == 32, "one 32-byte record per dense item");

struct StepParams {
  // configuration
  int32_t batch;
  int32_t hq, hkv, group, head_dim;
  int32_t page_size, page_shift;     // page_size == 1 << page_shift
  int32_t kv_dtype, q_dtype, o_dtype;
  int32_t num_pages;
  int32_t token_flat;                // read K/V through kv_indices (page size 1 view)
  int32_t concurrent;                // prefix and suffix kernels may run at the same time
  int32_t pdl;                       // the suffix kernel is a programmatic dependent of the prefix kernel
  float scale_log2;                  // log2(e) / sqrt(head_dim)

  // caller tensors (device)
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const float* k_scale;
  const float* v_scale;
  void* o;
  float* lse;

  // plan (device int32 arrays, see plan layout)
  const int32_t* suffix_page_indptr;   // [B+1]
  const int32_t* suffix_page_indices;
  const int32_t* suffix_start;         // [B]
  const int32_t* suffix_len;           // [B]
  const int32_t* split_indptr;         // [B+1]
  const int32_t* split_req;            // [S]
  const int32_t* split_begin;          // [S]
  const int32_t* split_end;            // [S]
  const SplitDesc* split_desc;         // [S]
  const int32_t* req_group;            // [B] deepest read-once group of b, else -1
  const int32_t* req_part_indptr;      // [B+1] b's prefix parts: one per chunk of each read-once
  const int2* req_part;                //   group of b, outermost first; .x = the chunk's first partial
                                       //   row + b's member index x G, .y = the group's M_eff, so that
                                       //   query head j of KV head h is row .x + h * .y + j
  const int32_t* group_page_indptr;    // [NG+1]
  const int32_t* group_page_indices;
  const int32_t* group_m_eff;          // [NG]
  const int32_t* group_shared_len;     // [NG]
  const int32_t* group_member_indptr;  // [NG+1]
  const int32_t* group_members;        // members (with descendants'), increasing request id
  const int32_t* group_chunk_indptr;   // [NG+1]
  const int32_t* chunk_group;          // [NC]
  const int32_t* chunk_begin;          // [NC] context tokens (the group's own segment)
  const int32_t* chunk_end;            // [NC]
  const int32_t* chunk_row_offset;     // [NC] first prefix-partial row of the chunk
  const DenseItemDesc* item_desc_dense;  // dense prefix work items, one record each
  const int32_t* item_chunk_dense;     // dense prefix work items: (chunk, row block)
  const int32_t* item_rb_dense;
  const int32_t* item_chunk_cascade;   // cascade prefix work items
  const int32_t* item_rb_cascade;
  const int32_t* kv_indptr;            // [B+1] token-flat offsets
  int32_t* kv_indices;                 // [sum kv_len] (token-flat mode)

  // partial results: O normalised (fp32) and log2-domain LSE
  float* o_suf;                        // [(S * Hkv + h) * G + j][D]
  float* lse_suf;
  float* o_pre;                        // [chunk_row_offset[c] + h * M_eff + r][D]
  float* lse_pre;
  int32_t* status;                     // device status word
  int32_t* counters;                   // [B * Hkv] arrivals of partial results (zero between steps)
  int32_t* done_ctas;                  // suffix CTAs finished this step (zero between steps)
  int32_t* prefix_done;                // prefix rows (x heads) whose partials and arrivals are done
  int32_t prefix_rows_total;           // its value once the whole prefix kernel has finished
};

// Byte offsets of every array inside the workspace (256-byte aligned each).
struct PlanLayout {
  size_t suffix_page_indptr, suffix_page_indices, suffix_start, suffix_len;
  size_t split_indptr, split_req, split_begin, split_end, split_desc;
  size_t req_group, req_part_indptr, req_part;
  size_t group_page_indptr, group_page_indices, group_m_eff, group_shared_len;
  size_t group_member_indptr, group_members, group_chunk_indptr;
  size_t chunk_group, chunk_begin, chunk_end, chunk_row_offset;
  size_t item_desc_dense, item_chunk_dense, item_rb_dense, item_chunk_cascade, item_rb_cascade;
  size_t kv_indptr;
  size_t plan_bytes;       // end of the uploaded integer region
  size_t status;
  size_t counters;         // right after status; both cleared at every upload
  size_t zero_end;
  size_t o_suf, lse_suf, o_pre, lse_pre;
  size_t kv_indices;
  size_t total;
};

// Launchers (each returns the launch's cudaError_t; nothing is launched for 0 items).
cudaError_t launch_suffix(const StepParams& p, int num_splits, cudaStream_t s);
cudaError_t launch_prefix_cascade(const StepParams& p, int num_items, cudaStream_t s);
cudaError_t launch_prefix_dense(const StepParams& p, int num_items, cudaStream_t s);
cudaError_t launch_expand_kv_indices(const StepParams& p, int32_t* out, cudaStream_t s);
cudaError_t launch_suffix_simt(const StepParams& p, int num_splits, cudaStream_t s);
cudaError_t launch_prefix_simt(const StepParams& p, int num_items, bool dense, cudaStream_t s);
cudaError_t launch_prefix_dense_mma(const StepParams& p, int num_items, cudaStream_t s);
cudaError_t launch_prefix_dense_tc(const StepParams& p, int num_items, cudaStream_t s);
bool dense_tc_supported(const StepParams& p);
cudaError_t launch_wait_selftest(int32_t* status, uint32_t polls, cudaStream_t s);

// Workspace-free entry point support (defined in psp_api.cpp).
}  // namespace psp

struct psp_handle;
typedef int32_t psp_status;
struct psp_tensors;

namespace psp {
psp_status set_error(psp_handle* h, psp_status code, const char* msg);
psp_status bind_image_and_run(psp_handle* h, unsigned char* ws, size_t cap, const psp_tensors* t, cudaStream_t s);
}  // namespace psp
