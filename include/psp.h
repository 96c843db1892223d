/*
 * psp.h -- paged shared-prefix decode attention on GB300 (sm_103a): C ABI.
 *
 * One decode step of attention: every request b contributes one query token
 * per query head and attends to its kv_len[b] context tokens, whose keys and
 * values sit in a pool of fixed-size physical pages reached through the
 * request's block table ("Track C Document 10 -- Shrinking the footprint",
 * PagedAttention answer: blocks handed out on demand, anywhere in memory).
 * Requests that share a prefix (a prefix group) reference the same physical
 * pages for it; the step reads those pages from HBM once, computes the
 * prefix scores and values for all M_eff = members x GQA-group stacked
 * queries at once, and merges that partial result with each request's
 * private-suffix attention by a log-sum-exp merge ("GraniKV: asymmetric KV
 * cache paging for shared-prefix agents", section 2 "Reuse saves prefill,
 * not decode reads" and section 3 "Per-step dispatcher").
 *
 * The result is exactly standard attention, O = softmax(q K^T / sqrt(d)) V
 * and LSE = ln(sum exp(q k / sqrt(d))) per (request, query head); paging
 * and sharing only change which bytes are read, not the math (runbook page,
 * "Does PagedAttention change the maths of attention?").
 *
 * Calls, in step order:
 *   psp_create            validate a configuration, make a handle (no CUDA calls)
 *   psp_plan              host-only: validate one batch's block tables and build
 *                         the step's integer plan (prefix/suffix split, M_eff,
 *                         dense/cascade branch, split-KV partition)
 *   psp_workspace_size    device bytes the plan needs (caller allocates)
 *   psp_upload            copy the plan into the caller's workspace (async H2D)
 *   psp_run               launch the step's kernels on the caller's stream
 * plus psp_step_host (the whole step from host buffers), psp_expand_kv_indices
 * (the token-flat lowering), read-back and diagnostics.
 *
 * Conventions for every call:
 *   - Return PSP_OK (0) or a negative psp_status; never throw, never abort.
 *     Invalid input is reported before anything is launched or copied.
 *     psp_last_error() holds a one-line description of the last failure.
 *   - Device pointers are plain CUDA device addresses on the current device;
 *     host pointers are ordinary (optionally pinned) host memory.  The caller
 *     owns every buffer and stream; the library owns only the handle and the
 *     pinned host staging it allocates for plan uploads.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Launches and copies are asynchronous on it.
 *   - A handle serves one stream at a time and is not thread-safe.
 *
 * Environment overrides, for measurements and tuning sweeps (read when a
 * handle is created, or once per process where marked; the defaults are the
 * values measured best on GB300):
 *   PSP_DENSE_THRESHOLD     dispatcher threshold T when psp_config.dense_threshold
 *                           is 0 (default 16)
 *   PSP_SPLIT_MIN_TILES     smallest split in 64-token granules (default 4)
 *   PSP_SPLIT_CTAS_PER_SM   split-KV target, (split, KV head) items per SM (default 5)
 *   PSP_PREFIX_MIN_TILES,   prefix-chunk partition: smallest chunk in 64-token granules
 *   PSP_PREFIX_CTAS_PER_SM  (default 4) and prefix CTAs per SM (default 1)
 *   PSP_PDL_FORM            prefix -> suffix dependent launch: 0 chosen by the prefix
 *                           grid's size and chunk length (default), 1 sequential,
 *                           2 concurrent
 *   PSP_SUFFIX_STAGES       suffix ring depth per warp at d = 128 (default 2 for bf16,
 *                           3 for e4m3; once per process)
 *   PSP_NUM_SMS             SM count the partition is sized for when psp_config.num_sms
 *                           is 0 (reproducible partitions across GPUs); unset or 0 = the
 *                           current device's count
 *   PSP_NVTX                1: psp_plan, psp_upload, psp_run and each kernel launch are named
 *                           NVTX ranges (for a profiler's timeline); default 0
 *   PSP_PLAN_THREADS        host threads (the calling one included, at most 16) that
 *                           compare group members' shared pages in psp_plan when the batch
 *                           lists at least 131072 page ids (default 8, never more than the
 *                           host's hardware threads; 1 = the calling thread);
 *                           the workers are made on first use and joined by psp_destroy
 *   PSP_LOG                 1: psp_plan writes one line per planned step to stderr,
 *                           "psp_step " and a JSON object: shapes and dtypes, page size,
 *                           block-table and kv_indices lengths, suffix and shared tokens,
 *                           splits, chunks and CTAs, per group its members, M_eff,
 *                           shared tokens, branch and chunks, and "coerced": false
 *                           (nothing is ever coerced); default 0
 * The plan outputs depend on the partition constants; psp_plan_info_get reports
 * the values a plan was built with.
 */
#ifndef PSP_H_
#define PSP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PSP_ABI_VERSION 3

#if defined(__GNUC__)
#define PSP_API __attribute__((visibility("default")))
#else
#define PSP_API
#endif

typedef int32_t psp_status;
#define PSP_OK 0
#define PSP_ERR_INVALID_ARGUMENT (-1) /* null pointer, bad size, inconsistent arrays, a group
                                         tree whose parent is not a lower group or whose
                                         child prefix is shorter than its parent's */
#define PSP_ERR_UNSUPPORTED (-2)      /* configuration not built (see psp_create); never coerced */
#define PSP_ERR_PAGE_OUT_OF_RANGE (-3)/* a page id < 0 or >= num_pages */
#define PSP_ERR_LENGTH (-4)           /* kv_len < 1, or page count != ceil(kv_len / page_size) */
#define PSP_ERR_PREFIX_MISMATCH (-5)  /* group members (descendants' requests included)
                                         disagree on their shared pages, or a member's context
                                         is shorter than its group's prefix */
#define PSP_ERR_NO_PLAN (-6)          /* run/upload/query before a successful plan/upload */
#define PSP_ERR_WORKSPACE (-7)        /* workspace NULL, too small or not 256-byte aligned */
#define PSP_ERR_CUDA (-8)             /* a CUDA runtime call failed (text in psp_last_error) */
#define PSP_ERR_DEVICE_TIMEOUT (-9)   /* a kernel's bounded wait ran out (psp_device_status) */
#define PSP_ERR_HOST_ALLOC (-10)      /* host memory for the plan could not be allocated */
#define PSP_ERR_CAPACITY (-11)        /* a caller buffer is too small (size in *needed) */

/* Element types. */
#define PSP_DTYPE_F32 0
#define PSP_DTYPE_BF16 1
#define PSP_DTYPE_FP8_E4M3 2 /* OCP e4m3 ("fn"): value = code * per-KV-head fp32 scale */

/* Prefix branch chosen per group by the dispatcher. */
#define PSP_BRANCH_NONE 0    /* no member, or the group's own segment is shorter than one page */
#define PSP_BRANCH_CASCADE 1 /* small-M tiled loop over the stacked queries */
#define PSP_BRANCH_DENSE 2   /* 128-row tensor-core tiles over the stacked queries */
#define PSP_BRANCH_PAGED 3   /* reading the group's segment once does not pay at this size, or
                                the group lies below a paged group: every member reads it
                                through its own block table, as unshared tokens (a root group's
                                plan then equals the plan without the group) */

/* Flags for psp_config.flags. */
#define PSP_FLAG_TOKEN_FLAT 1 /* lower block tables to per-token kv_indices on the device
                                 (psp_expand_kv_indices) inside psp_run and read K/V
                                 through them; results are bit-identical to page mode */
#define PSP_FLAG_CONCURRENT 2 /* run the prefix kernels on an internal stream forked from
                                 and joined back into the caller's stream, concurrently
                                 with the suffix kernel (tensor-core work overlapping the
                                 HBM stream); every multi-part row then merges through
                                 its arrival counter.  Ignored by psp_run_noalloc. */

/*
 * Step configuration.  Supported (anything else -> PSP_ERR_UNSUPPORTED):
 *   head_dim 64 or 128; num_q_heads = G * num_kv_heads with G in {1, 2, 4, 8};
 *   kv_dtype F32 with q_dtype F32; kv_dtype BF16 or FP8_E4M3 with q_dtype BF16;
 *   o_dtype F32 or BF16; page_size a power of two in [1, 1024].
 */
typedef struct psp_config {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t q_dtype;
  int32_t kv_dtype;
  int32_t o_dtype;
  int32_t page_size;       /* tokens per physical page */
  int32_t num_pages;       /* pages in the K pool (and the V pool) */
  int32_t num_sms;         /* SMs the partition is sized for; 0 = PSP_NUM_SMS if set, else the
                              current device's count */
  int32_t dense_threshold; /* M_eff at or above which a group takes the dense branch;
                              0 = the built-in value measured on GB300 */
  int32_t flags;           /* PSP_FLAG_* */
  int32_t read_once_min_tokens; /* a group's prefix is read once only if its shared tokens
                                   reach this; 0 = the built-in GB300 value, < 0 = no minimum */
  int32_t read_once_min_mib;    /* ... and only if reading once saves at least this many MiB,
                                   (members - 1) x shared tokens x 2 x Hkv x d x element size;
                                   0 = the built-in GB300 value, < 0 = no minimum */
} psp_config;

/*
 * One step's block tables, in host memory (read during psp_plan only).
 *   kv_len[B]            context tokens of request b, including the token being decoded
 *   page_indptr[B+1]     CSR offsets: request b's pages are page_indices[page_indptr[b] ..
 *                        page_indptr[b+1]), in logical order; there must be exactly
 *                        ceil(kv_len[b] / page_size) of them (the last may be partial)
 *   page_indices[...]    physical page ids in [0, num_pages); at page_size 1 these are the
 *                        token-flat kv_indices
 *   prefix_group[B]      group id in [0, num_groups) or -1; NULL = no sharing at all
 *   group_prefix_len[g]  tokens of group g's shared prefix (counted from the context's first
 *                        token); only its floor(P / page_size) full pages are shared
 *                        (block-aligned matching), the remaining tokens stay in each
 *                        member's private suffix
 *   group_parent[g]      nested prefixes (a radix tree of shared beginnings, "Track C
 *                        Document 10", the vLLM-or-SGLang answer; per-user sharing on top of
 *                        a global prefix in its cache table): -1 for a root, else a group of
 *                        lower index whose prefix is no longer than g's; NULL = every group
 *                        is a root.  A request of group g is a member of g and of every
 *                        ancestor of g; group g's own segment is its shared pages from
 *                        floor(P_parent / page_size) on, read once for all of its members.
 * Every member of a group must list the group's floor(P / page_size) shared page ids.
 */
typedef struct psp_batch {
  int32_t batch_size;
  const int32_t* kv_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  const int32_t* prefix_group;
  int32_t num_groups;
  const int32_t* group_prefix_len;
  const int32_t* group_parent;
} psp_batch;

/*
 * Device tensors of one step (row-major, densely packed, caller-owned).
 *   q       [B, Hq, d]                        q_dtype
 *   k_pool  [num_pages, page_size, Hkv, d]    kv_dtype (token-major within a page)
 *   v_pool  [num_pages, page_size, Hkv, d]    kv_dtype
 *   k_scale, v_scale [Hkv] fp32               FP8_E4M3 only (NULL otherwise)
 *   o       [B, Hq, d]                        o_dtype (written)
 *   lse     [B, Hq] fp32, natural log         written if not NULL
 * All pointers 16-byte aligned.
 */
typedef struct psp_tensors {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const float* k_scale;
  const float* v_scale;
  void* o;
  float* lse;
} psp_tensors;

/* Counts and constants of the current plan (psp_plan_info). */
typedef struct psp_plan_info {
  int32_t batch_size;
  int32_t num_groups;
  int32_t num_splits;          /* suffix splits over all requests */
  int32_t num_chunks;          /* prefix chunks over all groups */
  int64_t suffix_pages;        /* entries of the suffix page lists */
  int64_t group_pages;         /* entries of the group prefix page lists (whole prefixes) */
  int64_t kv_indices_len;      /* sum of kv_len (token-flat lowering length) */
  int64_t suffix_tokens;       /* sum of suffix lengths */
  int64_t shared_tokens;       /* sum of the groups' own segments read once per step */
  int64_t workspace_bytes;     /* device workspace the plan needs */
  int32_t suffix_ctas;         /* (split, kv head) work items */
  int32_t prefix_dense_ctas;   /* (chunk, row block, kv head) items of dense groups */
  int32_t prefix_cascade_ctas; /* same for cascade groups */
  int32_t merge_rows;          /* (request, query head) rows merged */
  /* partition constants (see psp_plan) */
  int32_t num_sms;
  int32_t dense_threshold;
  int32_t tile_tokens;
  int32_t split_min_tiles;
  int32_t split_ctas_per_sm;
  int32_t prefix_rows_dense;
  int32_t prefix_rows_cascade;
  int32_t prefix_min_tiles;
  int32_t prefix_ctas_per_sm;
  int32_t read_once_min_tokens; /* as resolved (-1: no minimum) */
  int32_t read_once_min_mib;    /* as resolved (-1: no minimum) */
  int32_t token_bytes;          /* K + V bytes of one token over all KV heads */
} psp_plan_info;

/* Plan arrays readable with psp_plan_query (all int32). */
#define PSP_FIELD_SUFFIX_START 0        /* [B] first private token = shared pages * page_size */
#define PSP_FIELD_SUFFIX_LEN 1          /* [B] private tokens, kv_len - suffix_start */
#define PSP_FIELD_SUFFIX_PAGE_INDPTR 2  /* [B+1] */
#define PSP_FIELD_SUFFIX_PAGE_INDICES 3 /* suffix page lists, logical order */
#define PSP_FIELD_SPLIT_INDPTR 4        /* [B+1] splits of request b */
#define PSP_FIELD_SPLIT_BEGIN 5         /* [num_splits] token offset within the suffix */
#define PSP_FIELD_SPLIT_END 6           /* [num_splits] exclusive */
#define PSP_FIELD_GROUP_SHARED_LEN 7    /* [num_groups] tokens of the own segment read once */
#define PSP_FIELD_GROUP_PAGE_INDPTR 8   /* [num_groups+1] */
#define PSP_FIELD_GROUP_PAGE_INDICES 9  /* per read-once group its whole shared page list,
                                           ancestors' pages first */
#define PSP_FIELD_GROUP_M_EFF 10        /* [num_groups] members (descendants' requests
                                           included) x (Hq / Hkv) */
#define PSP_FIELD_GROUP_BRANCH 11       /* [num_groups] PSP_BRANCH_* */
#define PSP_FIELD_GROUP_ROW_BLOCKS 12   /* [num_groups] stacked-query row blocks */
#define PSP_FIELD_GROUP_CHUNK_INDPTR 13 /* [num_groups+1] */
#define PSP_FIELD_CHUNK_BEGIN 14        /* [num_chunks] context token (inside the group's own
                                           segment, which starts at its parent's shared end) */
#define PSP_FIELD_CHUNK_END 15          /* [num_chunks] exclusive */
#define PSP_FIELD_KV_INDPTR 16          /* [B+1] offsets of the token-flat lowering */
#define PSP_FIELD_REQ_LEVEL_INDPTR 17   /* [B+1] CSR offsets of each request's read-once groups */
#define PSP_FIELD_REQ_LEVEL_GROUP 18    /* those groups, outermost first (merge order) */

typedef struct psp_handle psp_handle;

/* Library version string, e.g. "psp 0.1 sm_103a" (static storage). */
PSP_API const char* psp_version(void);

/* Text of a status code (static storage). */
PSP_API const char* psp_status_string(psp_status status);

/* Validates cfg (see psp_config) and allocates a handle.  Makes no CUDA call.
 * Errors: INVALID_ARGUMENT (NULL, non-positive sizes, Hq not a multiple of Hkv),
 * UNSUPPORTED (a combination that is not built; nothing is coerced). */
PSP_API psp_status psp_create(const psp_config* cfg, psp_handle** out);

/* Frees the handle, its pinned staging and its planning threads (joined).  Waits for no
 * device work: the caller must not destroy a handle whose upload is still in flight.
 * NULL is ignored. */
PSP_API void psp_destroy(psp_handle* h);

/* Description of the handle's last failure ("" if none; static to the handle). */
PSP_API const char* psp_last_error(const psp_handle* h);

/*
 * Host-only planning of one step (no CUDA call unless cfg.num_sms == 0, which
 * queries the current device's SM count once).  Validates the batch (see
 * psp_batch) and builds, in token units independent of the page size:
 *  - per group (its members: its own requests and its descendants'): M_eff =
 *    members x (Hq / Hkv), its own segment (shared tokens from its parent's
 *    floor(P_parent / page_size) pages to its floor(P_g / page_size) pages)
 *    and the branch ("GraniKV", section 3 Per-step dispatcher): NONE without
 *    members or without a full page in the segment; PAGED below a PAGED group,
 *    or when reading the segment once does not pay (its tokens below
 *    read_once_min_tokens, or (members - 1) x its tokens x token_bytes below
 *    read_once_min_mib MiB; the built-in values 1024 tokens and 64 MiB are the
 *    GB300 refit); else DENSE if M_eff >= dense_threshold, else CASCADE.  A
 *    DENSE or CASCADE group's segment is read once; a PAGED group shares
 *    nothing (shared length 0, no chunks);
 *  - per request: its read-once groups, outermost first (each contributes
 *    its prefix partials to the merge), shared pages n_sh = floor(P / page_size)
 *    of the deepest of them (0 without one), suffix_start = n_sh * page_size,
 *    suffix_len = kv_len - suffix_start, the suffix page list = pages[n_sh:]
 *    ("Track C Document 10", block-aligned prefix matching);
 *  - the split-KV partition: with granule tile_tokens, T_b = ceil(S_b / tile)
 *    granules per suffix, W = Hkv * sum T_b, C = max(split_min_tiles,
 *    ceil(W / (split_ctas_per_sm * num_sms))) granules per split, and split s
 *    of request b covering suffix tokens [tile*s*C, min(tile*(s+1)*C, S_b));
 *  - the prefix partition of each read-once segment: R = ceil(M_eff / rows) row
 *    blocks (rows = 256 dense, 64 cascade), TP = ceil(shared / tile) granules, n = max(1,
 *    min(floor(prefix_ctas_per_sm * num_sms / (Hkv * R)), floor(TP /
 *    prefix_min_tiles))), CP = ceil(TP / n), chunk c covering the segment's
 *    tokens [tile*c*CP, min(tile*(c+1)*CP, shared)), offset by the segment's
 *    first context token.
 * A successful plan replaces the previous one (its upload becomes invalid).
 * Errors: INVALID_ARGUMENT, PAGE_OUT_OF_RANGE, LENGTH, PREFIX_MISMATCH,
 * HOST_ALLOC, CUDA (only when querying the SM count). */
PSP_API psp_status psp_plan(psp_handle* h, const psp_batch* batch);

/* Counts and constants of the current plan.  Errors: NO_PLAN. */
PSP_API psp_status psp_plan_info_get(const psp_handle* h, psp_plan_info* out);

/* Device workspace bytes the current plan needs (plan arrays, fp32 partial
 * results, the token-flat indices in TOKEN_FLAT mode, a device status word and
 * per-(request, KV head) merge counters).
 * Errors: NO_PLAN. */
PSP_API psp_status psp_workspace_size(const psp_handle* h, size_t* bytes);

/* Copies one plan array to host memory dst (capacity cap_bytes).  *needed (if
 * not NULL) receives the array's size in bytes.  Errors: NO_PLAN,
 * INVALID_ARGUMENT (unknown field), CAPACITY (dst too small; nothing copied). */
PSP_API psp_status psp_plan_query(const psp_handle* h, int32_t field, void* dst, size_t cap_bytes,
                          size_t* needed);

/* Binds a caller-allocated device workspace (>= psp_workspace_size bytes,
 * 256-byte aligned) to the current plan and enqueues the plan's host-to-device
 * copy on `stream` (from pinned staging the library owns).  Clears the device
 * status word and the merge counters.  The staging is reused by the next upload of this handle after
 * the previous copy has completed (the call synchronises on its own event).
 * Errors: NO_PLAN, WORKSPACE, CUDA, HOST_ALLOC. */
PSP_API psp_status psp_upload(psp_handle* h, void* workspace, size_t workspace_bytes, void* stream);

/* Launches one decode step on `stream`: the prefix kernel of every group
 * (dense or cascade branch), then the split-KV suffix kernel (in TOKEN_FLAT
 * mode, first the device kv_indices expansion).  The log-sum-exp merge that
 * writes o and lse runs inside those kernels: the CTA that delivers the last
 * partial result of a (request, KV head) merges its rows.  Reads the uploaded plan; t must match the planned
 * batch and configuration.  Errors: NO_PLAN, INVALID_ARGUMENT, CUDA. */
PSP_API psp_status psp_run(psp_handle* h, const psp_tensors* t, void* stream);

/* Host-buffer variant of one whole step, synchronous: enqueue the copy of q_host
 * (pinned, [B, Hq, d] q_dtype) to dev->q, psp_plan(batch) on the host while that
 * copy runs, upload into `workspace`, psp_run, copy dev->o and dev->lse back to
 * o_host and lse_host (lse_host may be NULL), then wait for the stream.
 * dev->q/o/lse are device staging buffers, dev's pools and scales are the
 * resident cache.  Errors: as the calls it makes (a planning error returns with
 * the query copy already enqueued on the stream). */
PSP_API psp_status psp_step_host(psp_handle* h, const psp_batch* batch, const void* q_host,
                         void* o_host, float* lse_host, const psp_tensors* dev,
                         void* workspace, size_t workspace_bytes, void* stream);

/* The token-flat lowering on the device ("The 25% Page-Size Slowdown That
 * Wasn't", "Four meanings of page size": B x context_length indices at every
 * page size): kv_indices[kv_indptr[b] + t] = page[b][t / ps] * ps + t % ps for
 * t < kv_len[b], written to the device array kv_indices (capacity cap entries,
 * >= psp_plan_info.kv_indices_len).  Needs an uploaded plan.
 * Errors: NO_PLAN, CAPACITY, CUDA. */
PSP_API psp_status psp_expand_kv_indices(psp_handle* h, int32_t* kv_indices, int64_t cap, void* stream);

/* Per-kernel device timing.  When enabled, psp_run records CUDA events around
 * each launch it makes; psp_kernel_times (after the stream has completed)
 * writes up to cap elapsed times in milliseconds, in launch order, and their
 * names (static strings) if names is not NULL; *count receives how many.
 * Errors: INVALID_ARGUMENT, CUDA. */
PSP_API psp_status psp_set_kernel_timing(psp_handle* h, int32_t enable);
PSP_API psp_status psp_kernel_times(psp_handle* h, float* ms, const char** names, int32_t cap,
                            int32_t* count);

/* Reads (synchronously) the device status word in the bound workspace into
 * *code: 0, or the code a kernel recorded instead of faulting -- low byte 1 =
 * a bounded mbarrier wait ran out (upper bits: the wait site), 2 = an index
 * found out of range.  Returns PSP_ERR_DEVICE_TIMEOUT when a wait ran out.
 * Errors: NO_PLAN, CUDA, DEVICE_TIMEOUT. */
PSP_API psp_status psp_device_status(psp_handle* h, int32_t* code);

/* Workspace-free variant of psp_run, for callers that cannot allocate device
 * memory where they run the step: an engine that has reserved nearly all HBM
 * for its KV pool and weights, a framework plugin or custom-op callback that
 * must not allocate on that path, or a latency-critical loop that cannot take
 * the synchronisation an allocation may cause.  (It has no counterpart on the
 * pages; the step it runs is exactly psp_run's.)
 * Needs a successful psp_plan; instead of psp_upload's caller workspace it
 * uses one file-scope static device array of 64 MiB, held for the life of the
 * process on every GPU where the library's device code is loaded.  It copies
 * the plan into that array from the handle's host image (pageable copy, no
 * staging), clears the status word and the merge counters, binds the array
 * as the handle's workspace
 * (psp_device_status reads it afterwards) and launches the step on `stream`.
 * It calls no cudaMalloc, cudaFree or other allocating routine and records no
 * kernel timing events.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  Every call, from any handle, shares the one
 * array, which keeps the last call's contents: calls whose work overlaps on
 * the GPU race with each other, so serialise them (one stream, or events).
 * A plan whose workspace (psp_workspace_size) exceeds 64 MiB is rejected with
 * PSP_ERR_WORKSPACE before anything is copied or launched; so is any call that
 * psp_run's own argument checks would reject (the call then leaves the array and
 * the handle's workspace binding untouched, and a call that fails after the copy
 * restores the binding).  After a successful call the handle stays bound to the
 * shared array: psp_device_status reads its status word, and psp_run or
 * psp_expand_kv_indices on the handle use it as their workspace, until the next
 * psp_upload binds one of the caller's; calls from other handles may overwrite
 * the array in between.
 * Errors: INVALID_ARGUMENT, NO_PLAN, WORKSPACE, UNSUPPORTED (device ordinal >
 * 63), CUDA. */
PSP_API psp_status psp_run_noalloc(psp_handle* h, const psp_tensors* t, void* stream);

/* Failure-detection self test: launches one kernel that waits, with a budget
 * of `polls` polls, on an mbarrier nothing completes, so that the wait runs out
 * and records its timeout (site 99) in the status word instead of hanging.
 * Read the result with psp_device_status after the stream completes.  Needs
 * an uploaded plan (for the workspace).  Errors: INVALID_ARGUMENT, NO_PLAN, CUDA. */
PSP_API psp_status psp_wait_selftest(psp_handle* h, int32_t polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PSP_H_ */
