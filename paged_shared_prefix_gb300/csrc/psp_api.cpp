// psp_api.cpp -- the C ABI of the paged shared-prefix decode step: handle and
// configuration checks, the host-side plan (block-aligned prefix split,
// dispatcher, split-KV partition), workspace layout, plan upload and the
// ordered kernel launches of one step.
#include "psp.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "psp_internal.h"

namespace {

using psp::PlanLayout;
using psp::StepParams;

// Dense/cascade threshold used when the configuration passes 0.  The pages fit
// 1024 on A100 and ask for a refit per GPU ("GraniKV", section 3).  This value
// is the GB300 refit: over a 4096-token prefix, 8 KV heads, GQA groups 1-8 and
// M_eff from 16 to 4096, the tcgen05 dense kernel was never slower than the
// cascade kernel (17.0 vs 18.4 us at M_eff 16, 86 vs 301 us at 4096), so the
// smallest swept M_eff is the threshold.
constexpr int32_t kDefaultDenseThreshold = 16;

// Minimums for reading a group's prefix once (else the group takes the paged branch): at
// least this many shared tokens, and at least this much HBM traffic saved, (members - 1) x
// shared tokens x bytes per token.  GB300 refit: a sweep over prefix lengths 128-4096,
// 8-256 members and bf16 / e4m3 caches, read-once step against the same batch planned
// without groups; these minimums gave the least total loss against the faster choice per
// point (0.20 in summed log time ratios, against 5.06 for always reading once).
constexpr int32_t kReadOnceMinTokens = 1024;
constexpr int32_t kReadOnceMinMiB = 64;

constexpr int32_t kSplitMinTiles = 4;
constexpr int32_t kConcurrentChunkTokens = 4096;  // prefix chunk length from which the concurrent form runs
constexpr int32_t kSplitCtasPerSm = 5;  // measured on GB300 with 2-stage bf16 rings: 5 (split, head) CTAs per SM
constexpr int32_t kPrefixMinTiles = 4;
constexpr int32_t kPrefixCtasPerSm = 1;  // a dense prefix CTA fills an SM (all of tensor memory)

thread_local std::string g_create_error;

int env_int(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (!v || !*v) return fallback;
  char* end = nullptr;
  long x = std::strtol(v, &end, 10);
  return (end && *end == 0 && x > 0 && x < (1L << 30)) ? static_cast<int>(x) : fallback;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align_up(size_t x) { return (x + psp::kWorkspaceAlign - 1) / psp::kWorkspaceAlign * psp::kWorkspaceAlign; }

int dtype_bytes(int32_t t) {
  switch (t) {
    case PSP_DTYPE_F32: return 4;
    case PSP_DTYPE_BF16: return 2;
    case PSP_DTYPE_FP8_E4M3: return 1;
  }
  return 0;
}

// A few host threads for the plan's comparisons of members' shared pages in large batches
// (made on first use, joined when the handle is destroyed).  run(n, f) calls f(i) once for
// every item i in [0, n): the calling thread starts on the items at once and the workers
// take items from the same counter as they wake, so a worker that wakes late costs the call
// nothing (it finds the items taken, or the job gone).  Returns when every call has.
class HostPool {
 public:
  explicit HostPool(int workers) {
    for (int i = 0; i < workers; ++i) threads_.emplace_back([this] { loop(); });
  }
  ~HostPool() {
    {
      std::lock_guard<std::mutex> g(m_);
      stop_ = true;
    }
    cv_.notify_all();
    for (std::thread& t : threads_) t.join();
  }
  int size() const { return static_cast<int>(threads_.size()) + 1; }
  void run(int n, const std::function<void(int)>& f) {
    {
      std::lock_guard<std::mutex> g(m_);
      job_ = &f;
      n_ = n;
      next_.store(0, std::memory_order_relaxed);
      ++gen_;
    }
    cv_.notify_all();
    drain(f);
    // every item is taken: withdraw the job from workers still waking, then wait for the
    // ones inside it to finish their items
    std::unique_lock<std::mutex> l(m_);
    job_ = nullptr;
    done_.wait(l, [&] { return active_ == 0; });
  }

 private:
  void drain(const std::function<void(int)>& f) {
    for (int i = next_.fetch_add(1, std::memory_order_relaxed); i < n_; i = next_.fetch_add(1, std::memory_order_relaxed))
      f(i);
  }
  void loop() {
    uint64_t seen = 0;
    for (;;) {
      const std::function<void(int)>* job = nullptr;
      {
        std::unique_lock<std::mutex> l(m_);
        cv_.wait(l, [&] { return stop_ || gen_ != seen; });
        if (stop_) return;
        seen = gen_;
        if (!job_) continue;  // the run has already ended
        job = job_;
        ++active_;
      }
      drain(*job);
      std::lock_guard<std::mutex> g(m_);
      if (--active_ == 0) done_.notify_one();
    }
  }
  std::vector<std::thread> threads_;
  std::mutex m_;
  std::condition_variable cv_, done_;
  const std::function<void(int)>* job_ = nullptr;
  int n_ = 0, active_ = 0;
  std::atomic<int> next_{0};
  uint64_t gen_ = 0;
  bool stop_ = false;
};

struct HostPlan {
  int32_t B = 0, NG = 0, NS = 0, NC = 0;
  std::vector<int32_t> suffix_page_indptr, suffix_page_indices, suffix_start, suffix_len;
  std::vector<int32_t> split_indptr, split_req, split_begin, split_end;
  std::vector<int32_t> split_desc;  // kSplitDescInts per split (psp::SplitDesc)
  std::vector<int32_t> req_group, req_member, req_level_indptr, req_level_group;
  std::vector<int32_t> req_part_indptr, req_part;  // req_part: (first row + member x G, M_eff) pairs
  std::vector<int32_t> group_page_indptr, group_page_indices, group_m_eff, group_shared_len;
  std::vector<int32_t> group_branch, group_row_blocks;
  std::vector<int32_t> group_member_indptr, group_members, group_chunk_indptr;
  std::vector<int32_t> chunk_group, chunk_begin, chunk_end, chunk_row_offset;
  std::vector<int32_t> item_chunk_dense, item_rb_dense, item_chunk_cascade, item_rb_cascade;
  std::vector<int32_t> item_desc_dense;  // 8 ints per dense item (psp::DenseItemDesc)
  std::vector<int32_t> kv_indptr;
  int64_t kv_indices_len = 0, suffix_tokens = 0, shared_tokens = 0, pre_rows = 0;
  PlanLayout layout{};
  psp_plan_info info{};
  std::vector<unsigned char> image;  // the uploaded integer region, laid out as in the workspace

  // Empties the plan for the next step, keeping every array's allocation (a decode loop
  // plans every step with arrays of about the same sizes).
  void clear() {
    B = NG = NS = NC = 0;
    for (std::vector<int32_t>* v :
         {&suffix_page_indptr, &suffix_page_indices, &suffix_start, &suffix_len, &split_indptr, &split_req,
          &split_begin, &split_end, &split_desc, &req_group, &req_member, &req_level_indptr, &req_level_group,
          &req_part_indptr, &req_part, &group_page_indptr, &group_page_indices,
          &group_m_eff, &group_shared_len, &group_branch, &group_row_blocks, &group_member_indptr, &group_members,
          &group_chunk_indptr, &chunk_group, &chunk_begin, &chunk_end, &chunk_row_offset, &item_chunk_dense,
          &item_rb_dense, &item_chunk_cascade, &item_rb_cascade, &kv_indptr, &item_desc_dense})
      v->clear();
    kv_indices_len = suffix_tokens = shared_tokens = pre_rows = 0;
    layout = PlanLayout{};
    info = psp_plan_info{};
    image.clear();
  }
};

}  // namespace

// A named NVTX range over a scope when enabled (one push and one pop; nothing otherwise).
struct NvtxRange {
  bool on;
  NvtxRange(bool enable, const char* name) : on(enable) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
};

struct psp_handle {
  psp_config cfg{};
  int32_t group = 1;
  int32_t page_shift = 0;
  int32_t split_min_tiles = kSplitMinTiles;
  int32_t split_ctas_per_sm = kSplitCtasPerSm;
  int32_t prefix_min_tiles = kPrefixMinTiles;
  int32_t prefix_ctas_per_sm = kPrefixCtasPerSm;
  int32_t num_sms_resolved = 0;

  bool planned = false;
  HostPlan plan;

  // upload state
  unsigned char* staging = nullptr;
  size_t staging_bytes = 0;
  cudaEvent_t staging_done = nullptr;
  unsigned char* workspace = nullptr;
  size_t workspace_bytes = 0;
  bool uploaded = false;

  // concurrent prefix: side stream and fork/join events (created on first use)
  cudaStream_t side = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  bool allow_concurrent = true;   // false on the workspace-free path (no object creation)
  int32_t pdl_form = 0;           // dependent-launch form: 0 by grid size, 1 sequential, 2 concurrent
  bool log = false;               // PSP_LOG: one structured line per plan on stderr
  int32_t plan_threads = 1;       // PSP_PLAN_THREADS: threads comparing shared pages in large plans
  int32_t env_num_sms = 0;        // PSP_NUM_SMS: SM count used when cfg.num_sms is 0 (0 = query the device)
  bool nvtx = false;              // PSP_NVTX: name psp_plan, psp_upload, psp_run and each launch as NVTX ranges
  std::unique_ptr<HostPool> pool; // its workers (made on first use)

  // per-kernel timing
  bool timing = false;
  std::vector<cudaEvent_t> events;       // 2 per launch
  std::vector<const char*> event_names;
  int recorded = 0;

  std::string last_error;
};

namespace {

psp_status fail(psp_handle* h, psp_status code, const std::string& msg) {
  if (h) h->last_error = msg;
  else g_create_error = msg;
  return code;
}

psp_status cuda_fail(psp_handle* h, cudaError_t e, const char* what) {
  std::string msg = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return fail(h, PSP_ERR_CUDA, msg);
}

// ----------------------------------------------------------------- planning

psp_status validate_batch(psp_handle* h, const psp_batch* bt) {
  const psp_config& c = h->cfg;
  if (!bt) return fail(h, PSP_ERR_INVALID_ARGUMENT, "batch is NULL");
  if (bt->batch_size < 0) return fail(h, PSP_ERR_INVALID_ARGUMENT, "negative batch size");
  if (bt->num_groups < 0) return fail(h, PSP_ERR_INVALID_ARGUMENT, "negative group count");
  const int B = bt->batch_size;
  if (B > 0 && (!bt->kv_len || !bt->page_indptr || !bt->page_indices))
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "kv_len/page_indptr/page_indices NULL");
  if (bt->num_groups > 0 && !bt->group_prefix_len)
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "group_prefix_len NULL");
  if (B > 0 && bt->page_indptr[0] != 0) return fail(h, PSP_ERR_INVALID_ARGUMENT, "page_indptr[0] != 0");
  const int64_t ps = c.page_size;
  int64_t total = 0;
  // The shared pages of a group member after the first are compared with the first
  // member's (build_plan), whose pages are range-checked in full here, so they are not
  // range-checked a second time.
  std::vector<int32_t> first_member(std::max(bt->num_groups, 0), -1);
  for (int b = 0; b < B; ++b) {
    const int64_t L = bt->kv_len[b];
    if (L < 1) return fail(h, PSP_ERR_LENGTH, "kv_len[" + std::to_string(b) + "] < 1");
    const int64_t n = static_cast<int64_t>(bt->page_indptr[b + 1]) - bt->page_indptr[b];
    if (n != cdiv(L, ps))
      return fail(h, PSP_ERR_LENGTH, "request " + std::to_string(b) + " has " + std::to_string(n) +
                                         " pages for kv_len " + std::to_string(L));
    // range check as a branch-free min / max pass (it vectorises); the offending id is
    // searched for only to word the error
    int64_t skip = 0;
    const int g = bt->prefix_group ? bt->prefix_group[b] : -1;
    if (g >= 0 && g < bt->num_groups && bt->group_prefix_len[g] >= 0) {
      if (first_member[g] < 0) {
        first_member[g] = b;
      } else {
        skip = std::min<int64_t>(n, bt->group_prefix_len[g] / ps);
      }
    }
    const int32_t* pg = bt->page_indices + bt->page_indptr[b];
    int32_t lo = INT32_MAX, hi = INT32_MIN;
    for (int64_t i = skip; i < n; ++i) {
      lo = std::min(lo, pg[i]);
      hi = std::max(hi, pg[i]);
    }
    if (n > skip && (lo < 0 || hi >= c.num_pages)) {
      const int32_t bad = lo < 0 ? lo : hi;
      return fail(h, PSP_ERR_PAGE_OUT_OF_RANGE,
                  "page id " + std::to_string(bad) + " of request " + std::to_string(b) + " outside [0, num_pages)");
    }
    total += L;
    if (total > INT32_MAX) return fail(h, PSP_ERR_INVALID_ARGUMENT, "sum of kv_len exceeds int32");
  }
  for (int g = 0; g < bt->num_groups; ++g)
    if (bt->group_prefix_len[g] < 0) return fail(h, PSP_ERR_INVALID_ARGUMENT, "negative group prefix length");
  // nested groups: a parent has a lower index and a prefix no longer than its child's
  if (bt->group_parent)
    for (int g = 0; g < bt->num_groups; ++g) {
      const int par = bt->group_parent[g];
      if (par < -1 || par >= g)
        return fail(h, PSP_ERR_INVALID_ARGUMENT, "group_parent[" + std::to_string(g) + "] is not -1 or a lower group");
      if (par >= 0 && bt->group_prefix_len[par] > bt->group_prefix_len[g])
        return fail(h, PSP_ERR_INVALID_ARGUMENT, "group " + std::to_string(g) + " has a shorter prefix than its parent");
    }
  return PSP_OK;
}

// Range check of every page id in request order (the slow path behind a failed group
// comparison: an out-of-range id takes precedence over a prefix mismatch).
psp_status full_range_check(psp_handle* h, const psp_batch* bt) {
  for (int b = 0; b < bt->batch_size; ++b)
    for (int64_t i = bt->page_indptr[b]; i < bt->page_indptr[b + 1]; ++i) {
      const int32_t pg = bt->page_indices[i];
      if (pg < 0 || pg >= h->cfg.num_pages)
        return fail(h, PSP_ERR_PAGE_OUT_OF_RANGE,
                    "page id " + std::to_string(pg) + " of request " + std::to_string(b) + " outside [0, num_pages)");
    }
  return PSP_OK;
}

psp_status build_plan(psp_handle* h, const psp_batch* bt, HostPlan& P) {
  const psp_config& c = h->cfg;
  const int B = bt->batch_size, NG = bt->num_groups, Hkv = c.num_kv_heads, G = h->group;
  const int64_t ps = c.page_size;
  const int64_t tile = psp::kTileTokens;
  const int32_t threshold = c.dense_threshold > 0 ? c.dense_threshold : kDefaultDenseThreshold;
  const int32_t min_tokens = c.read_once_min_tokens > 0 ? c.read_once_min_tokens
                             : c.read_once_min_tokens == 0 ? kReadOnceMinTokens : -1;
  const int32_t min_mib = c.read_once_min_mib > 0 ? c.read_once_min_mib : c.read_once_min_mib == 0 ? kReadOnceMinMiB : -1;
  const int64_t token_bytes = 2LL * Hkv * c.head_dim * dtype_bytes(c.kv_dtype);
  const int64_t sms = h->num_sms_resolved;
  P.clear();
  P.B = B;
  P.NG = NG;

  // --- groups: the tree (checked in validate_batch; NULL parents: every group a root), the
  //     members of each group (its own requests and its descendants'), increasing request id
  const int32_t* parent = bt->group_parent;
  auto parent_of = [&](int g) { return parent ? parent[g] : -1; };
  auto pages_of = [&](int g) -> int64_t { return g >= 0 ? bt->group_prefix_len[g] / ps : 0; };
  std::vector<int32_t> lead(NG, -1), count(NG, 0);
  P.req_group.assign(B, -1);
  P.req_member.assign(B, -1);
  int64_t chain_len = 0;
  for (int b = 0; b < B; ++b) {
    const int g = bt->prefix_group ? bt->prefix_group[b] : -1;
    if (g == -1) continue;
    if (g < -1 || g >= NG) return fail(h, PSP_ERR_INVALID_ARGUMENT, "prefix_group out of range");
    if (bt->group_prefix_len[g] > bt->kv_len[b])
      return fail(h, PSP_ERR_PREFIX_MISMATCH, "group prefix longer than the context of request " + std::to_string(b));
    if (lead[g] < 0) lead[g] = b;
    for (int a = g; a >= 0; a = parent_of(a)) {
      ++count[a];
      ++chain_len;
    }
  }
  P.group_member_indptr.assign(NG + 1, 0);
  for (int g = 0; g < NG; ++g) P.group_member_indptr[g + 1] = P.group_member_indptr[g] + count[g];
  P.group_members.assign(std::max<int64_t>(P.group_member_indptr[NG], 0), 0);
  // per request, its groups from its own up to the root with its index among each one's members
  std::vector<int32_t> chain_indptr(B + 1, 0), chain_group(chain_len), chain_member(chain_len);
  {
    std::vector<int32_t> cursor(P.group_member_indptr.begin(), P.group_member_indptr.end() - 1);
    int64_t k = 0;
    for (int b = 0; b < B; ++b) {
      const int g = bt->prefix_group ? bt->prefix_group[b] : -1;
      for (int a = g; a >= 0; a = parent_of(a), ++k) {
        chain_group[k] = a;
        chain_member[k] = cursor[a] - P.group_member_indptr[a];
        P.group_members[cursor[a]++] = b;
      }
      chain_indptr[b + 1] = static_cast<int32_t>(k);
    }
  }
  // every member lists its group's shared pages: against the first request of its own group
  // over the whole prefix (that request's pages were range-checked in full), and against the
  // first member of every group on its path over that group's own segment (needed only where
  // the first member is not the first request of the group itself).  Large batches split the
  // requests over a few host threads; the first mismatching request in request order is the
  // one reported either way.
  auto first_mismatch = [&](int b0, int b1) {
    for (int b = b0; b < b1; ++b) {
      const int g = bt->prefix_group ? bt->prefix_group[b] : -1;
      if (g < 0) continue;
      const int32_t* mine = bt->page_indices + bt->page_indptr[b];
      bool same = true;
      const int64_t n_sh = pages_of(g);
      if (b != lead[g] && n_sh > 0)
        same = std::memcmp(mine, bt->page_indices + bt->page_indptr[lead[g]], static_cast<size_t>(n_sh) * sizeof(int32_t)) == 0;
      for (int a = g; same && a >= 0; a = parent_of(a)) {
        const int rep = P.group_members[P.group_member_indptr[a]];
        if (rep == b || (a == g && rep == lead[g])) continue;
        const int64_t lo = pages_of(parent_of(a)), hi = pages_of(a);
        if (hi > lo)
          same = std::memcmp(mine + lo, bt->page_indices + bt->page_indptr[rep] + lo,
                             static_cast<size_t>(hi - lo) * sizeof(int32_t)) == 0;
      }
      if (!same) return b;
    }
    return -1;
  };
  int bad = -1;
  const int64_t compared = chain_len > 0 ? static_cast<int64_t>(bt->page_indptr[B]) : 0;  // bounds the pages compared
  const int parts = compared >= (int64_t{1} << 17) ? std::min<int>(h->plan_threads, B) : 1;
  if (parts > 1 && !h->pool) {
    try {
      h->pool.reset(new HostPool(parts - 1));
    } catch (...) {  // no threads to be had: compare on the calling thread
      h->plan_threads = 1;
    }
  }
  if (parts > 1 && h->pool) {
    // items of about 16k compared page ids, in request order
    const int64_t per_item = std::max<int64_t>(1, (int64_t{1} << 14) * B / compared);
    const int n = static_cast<int>(cdiv(B, per_item));
    std::vector<int> found(n, -1);
    const std::function<void(int)> part = [&](int i) {
      found[i] = first_mismatch(static_cast<int>(per_item * i), static_cast<int>(std::min<int64_t>(B, per_item * (i + 1))));
    };
    h->pool->run(n, part);
    for (int i = 0; i < n && bad < 0; ++i) bad = found[i];
  } else {
    bad = first_mismatch(0, B);
  }
  if (bad >= 0) {
    const psp_status range = full_range_check(h, bt);
    if (range) return range;
    return fail(h, PSP_ERR_PREFIX_MISMATCH, "request " + std::to_string(bad) + " does not share the prefix pages of its group");
  }

  // --- per group: M_eff, the branch of its own segment, shared pages, row blocks, chunks
  //     (a group below a paged group is paged: a request's unshared tokens stay one range)
  P.group_shared_len.assign(NG, 0);
  P.group_m_eff.assign(NG, 0);
  P.group_branch.assign(NG, PSP_BRANCH_NONE);
  P.group_row_blocks.assign(NG, 0);
  P.group_page_indptr.assign(NG + 1, 0);
  P.group_chunk_indptr.assign(NG + 1, 0);
  std::vector<char> below_paged(NG, 0);
  for (int g = 0; g < NG; ++g) {
    const int par = parent_of(g);
    if (par >= 0) below_paged[g] = below_paged[par] || P.group_branch[par] == PSP_BRANCH_PAGED;
    const int64_t n_sh = pages_of(g);
    const int64_t seg0 = pages_of(par) * ps;  // first token of the group's own segment
    const int64_t seg = count[g] > 0 ? n_sh * ps - seg0 : 0;
    const int64_t m_eff = static_cast<int64_t>(count[g]) * G;
    int branch = PSP_BRANCH_NONE;
    if (m_eff > 0 && seg > 0) {
      const int64_t saved = static_cast<int64_t>(count[g] - 1) * seg * token_bytes;
      if (below_paged[g] || (min_tokens > 0 && seg < min_tokens) ||
          (min_mib > 0 && saved < (static_cast<int64_t>(min_mib) << 20)))
        branch = PSP_BRANCH_PAGED;
      else
        branch = m_eff >= threshold ? PSP_BRANCH_DENSE : PSP_BRANCH_CASCADE;
    }
    const bool once = branch == PSP_BRANCH_DENSE || branch == PSP_BRANCH_CASCADE;
    const int64_t shared = once ? seg : 0;
    P.group_shared_len[g] = static_cast<int32_t>(shared);
    P.group_m_eff[g] = static_cast<int32_t>(m_eff);
    if (once) {  // the whole prefix, the ancestors' pages first
      const int32_t* src = bt->page_indices + bt->page_indptr[P.group_members[P.group_member_indptr[g]]];
      P.group_page_indices.insert(P.group_page_indices.end(), src, src + n_sh);
    }
    P.group_page_indptr[g + 1] = static_cast<int32_t>(P.group_page_indices.size());
    P.group_branch[g] = branch;
    if (once) {
      const int64_t rows = branch == PSP_BRANCH_DENSE ? psp::kDenseRows : psp::kCascadeRows;
      const int64_t rb = cdiv(m_eff, rows);
      const int64_t tiles = cdiv(shared, tile);
      const int64_t fit = (static_cast<int64_t>(h->prefix_ctas_per_sm) * sms) / (Hkv * rb);
      const int64_t most = tiles / h->prefix_min_tiles;
      int64_t n = std::max<int64_t>(1, std::min(fit, most));
      const int64_t per = cdiv(tiles, n);
      n = cdiv(tiles, per);
      P.group_row_blocks[g] = static_cast<int32_t>(rb);
      for (int64_t ci = 0; ci < n; ++ci) {
        const int32_t chunk_id = static_cast<int32_t>(P.chunk_begin.size());
        P.chunk_group.push_back(g);
        P.chunk_begin.push_back(static_cast<int32_t>(seg0 + ci * per * tile));
        P.chunk_end.push_back(static_cast<int32_t>(seg0 + std::min((ci + 1) * per * tile, shared)));
        P.chunk_row_offset.push_back(static_cast<int32_t>(P.pre_rows));
        P.pre_rows += static_cast<int64_t>(Hkv) * m_eff;
        for (int64_t r = 0; r < rb; ++r) {
          if (branch == PSP_BRANCH_DENSE) {
            P.item_chunk_dense.push_back(chunk_id);
            P.item_rb_dense.push_back(static_cast<int32_t>(r));
          } else {
            P.item_chunk_cascade.push_back(chunk_id);
            P.item_rb_cascade.push_back(static_cast<int32_t>(r));
          }
        }
      }
      P.shared_tokens += shared;
    }
    P.group_chunk_indptr[g + 1] = static_cast<int32_t>(P.chunk_begin.size());
  }
  if (P.pre_rows > INT32_MAX) return fail(h, PSP_ERR_INVALID_ARGUMENT, "prefix partial rows exceed int32");
  P.NC = static_cast<int32_t>(P.chunk_begin.size());

  // --- per request: the read-once groups on its path, outermost first (their prefix partials
  //     are merged in this order), and the suffix after the deepest of them
  P.req_level_indptr.assign(B + 1, 0);
  P.req_part_indptr.assign(B + 1, 0);
  P.suffix_page_indptr.assign(B + 1, 0);
  P.suffix_start.assign(B, 0);
  P.suffix_len.assign(B, 0);
  P.kv_indptr.assign(B + 1, 0);
  for (int b = 0; b < B; ++b) {
    int64_t n_sh = 0;
    for (int32_t k = chain_indptr[b + 1] - 1; k >= chain_indptr[b]; --k) {
      const int a = chain_group[k];
      if (P.group_branch[a] != PSP_BRANCH_DENSE && P.group_branch[a] != PSP_BRANCH_CASCADE) continue;
      P.req_level_group.push_back(a);
      for (int32_t c = P.group_chunk_indptr[a]; c < P.group_chunk_indptr[a + 1]; ++c) {
        P.req_part.push_back(P.chunk_row_offset[c] + chain_member[k] * G);
        P.req_part.push_back(P.group_m_eff[a]);
      }
      P.req_group[b] = a;
      P.req_member[b] = chain_member[k];
      n_sh = pages_of(a);
    }
    P.req_level_indptr[b + 1] = static_cast<int32_t>(P.req_level_group.size());
    P.req_part_indptr[b + 1] = static_cast<int32_t>(P.req_part.size() / 2);
    P.suffix_start[b] = static_cast<int32_t>(n_sh * ps);
    P.suffix_len[b] = static_cast<int32_t>(bt->kv_len[b] - n_sh * ps);
    const int32_t* pages = bt->page_indices + bt->page_indptr[b];
    const int64_t npg = bt->page_indptr[b + 1] - bt->page_indptr[b];
    P.suffix_page_indices.insert(P.suffix_page_indices.end(), pages + n_sh, pages + npg);
    P.suffix_page_indptr[b + 1] = static_cast<int32_t>(P.suffix_page_indices.size());
    P.kv_indptr[b + 1] = P.kv_indptr[b] + bt->kv_len[b];
    P.suffix_tokens += P.suffix_len[b];
  }
  P.kv_indices_len = P.kv_indptr[B];

  // --- one record per dense work item (its chunk, group, token range and list bases)
  P.item_desc_dense.assign(P.item_chunk_dense.size() * 8, 0);
  for (size_t it = 0; it < P.item_chunk_dense.size(); ++it) {
    const int32_t ci = P.item_chunk_dense[it], g = P.chunk_group[ci];
    const int32_t mb = P.group_member_indptr[g];
    psp::DenseItemDesc d{};
    d.chunk = ci;
    d.rb = P.item_rb_dense[it];
    d.t0 = P.chunk_begin[ci];
    d.t1 = P.chunk_end[ci];
    d.m_eff = P.group_m_eff[g];
    d.member_base = mb;
    d.list_base = (c.flags & PSP_FLAG_TOKEN_FLAT) ? P.kv_indptr[P.group_members[mb]] : P.group_page_indptr[g];
    d.row_offset = P.chunk_row_offset[ci];
    std::memcpy(P.item_desc_dense.data() + it * 8, &d, sizeof(d));
  }

  // --- split-KV partition of the suffixes (token units, page-size independent)
  int64_t granules = 0;
  for (int b = 0; b < B; ++b) granules += cdiv(P.suffix_len[b], tile);
  const int64_t target = static_cast<int64_t>(h->split_ctas_per_sm) * sms;
  const int64_t per_split = std::max<int64_t>(h->split_min_tiles, cdiv(static_cast<int64_t>(Hkv) * granules, target));
  P.split_indptr.assign(B + 1, 0);
  for (int b = 0; b < B; ++b) {
    const int64_t S = P.suffix_len[b];
    for (int64_t lo = 0; lo < S; lo += per_split * tile) {
      P.split_req.push_back(b);
      P.split_begin.push_back(static_cast<int32_t>(lo));
      P.split_end.push_back(static_cast<int32_t>(std::min(lo + per_split * tile, S)));
    }
    P.split_indptr[b + 1] = static_cast<int32_t>(P.split_req.size());
  }
  P.NS = static_cast<int32_t>(P.split_req.size());
  P.split_desc.assign(static_cast<size_t>(P.NS) * psp::kSplitDescInts, 0);
  for (int32_t si = 0; si < P.NS; ++si) {
    psp::SplitDesc d{};
    const int32_t b = P.split_req[si];
    d.b = b;
    d.t0 = P.split_begin[si];
    d.t1 = P.split_end[si];
    d.list_paged = P.suffix_page_indptr[b];
    d.list_flat = P.kv_indptr[b] + P.suffix_start[b];
    d.part0 = P.req_part_indptr[b];
    d.n_parts = P.req_part_indptr[b + 1] - d.part0;
    d.one_split = P.split_indptr[b + 1] - P.split_indptr[b] == 1 ? 1 : 0;
    const int32_t* spages = P.suffix_page_indices.data() + d.list_paged;
    const int shift = h->page_shift;  // page_size == 1 << shift: no division per entry
    for (int k = 0; k < psp::kDescPages; ++k) {
      const int32_t t = d.t0 + 16 * k;
      d.first_page[k] = (ps >= 16 && t < d.t1) ? spages[t >> shift] : -1;
    }
    std::memcpy(P.split_desc.data() + static_cast<size_t>(si) * psp::kSplitDescInts, &d, sizeof(d));
  }
  if (static_cast<int64_t>(P.NS) * Hkv > INT32_MAX / psp::kMaxGroupSize)
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "too many splits");

  // --- workspace layout
  PlanLayout& L = P.layout;
  size_t off = 0;
  auto place = [&](size_t& field, size_t bytes) { field = off; off = align_up(off + std::max<size_t>(bytes, 4)); };
  auto n32 = [](const std::vector<int32_t>& v) { return v.size() * sizeof(int32_t); };
  place(L.suffix_page_indptr, n32(P.suffix_page_indptr));
  place(L.suffix_page_indices, n32(P.suffix_page_indices));
  place(L.suffix_start, n32(P.suffix_start));
  place(L.suffix_len, n32(P.suffix_len));
  place(L.split_indptr, n32(P.split_indptr));
  place(L.split_req, n32(P.split_req));
  place(L.split_begin, n32(P.split_begin));
  place(L.split_end, n32(P.split_end));
  place(L.split_desc, n32(P.split_desc));
  place(L.req_group, n32(P.req_group));
  place(L.req_part_indptr, n32(P.req_part_indptr));
  place(L.req_part, n32(P.req_part));
  place(L.group_page_indptr, n32(P.group_page_indptr));
  place(L.group_page_indices, n32(P.group_page_indices));
  place(L.group_m_eff, n32(P.group_m_eff));
  place(L.group_shared_len, n32(P.group_shared_len));
  place(L.group_member_indptr, n32(P.group_member_indptr));
  place(L.group_members, n32(P.group_members));
  place(L.group_chunk_indptr, n32(P.group_chunk_indptr));
  place(L.chunk_group, n32(P.chunk_group));
  place(L.chunk_begin, n32(P.chunk_begin));
  place(L.chunk_end, n32(P.chunk_end));
  place(L.chunk_row_offset, n32(P.chunk_row_offset));
  place(L.item_desc_dense, n32(P.item_desc_dense));
  place(L.item_chunk_dense, n32(P.item_chunk_dense));
  place(L.item_rb_dense, n32(P.item_rb_dense));
  place(L.item_chunk_cascade, n32(P.item_chunk_cascade));
  place(L.item_rb_cascade, n32(P.item_rb_cascade));
  place(L.kv_indptr, n32(P.kv_indptr));
  L.plan_bytes = off;
  L.status = off;
  L.counters = off + 64;
  L.zero_end = L.counters + static_cast<size_t>(B) * Hkv * sizeof(int32_t);
  off = align_up(L.zero_end);
  const size_t D = c.head_dim;
  const size_t suf_rows = static_cast<size_t>(P.NS) * Hkv * G;
  place(L.o_suf, suf_rows * D * sizeof(float));
  place(L.lse_suf, suf_rows * sizeof(float));
  place(L.o_pre, static_cast<size_t>(P.pre_rows) * D * sizeof(float));
  place(L.lse_pre, static_cast<size_t>(P.pre_rows) * sizeof(float));
  place(L.kv_indices, (c.flags & PSP_FLAG_TOKEN_FLAT) ? static_cast<size_t>(P.kv_indices_len) * 4 : 0);
  L.total = off;

  // host image of the integer region
  // (through zero_end: the status word and the merge counters upload as zeros with the plan)
  P.image.assign(L.zero_end, 0);
  auto put = [&](size_t off, const std::vector<int32_t>& v) {
    if (!v.empty()) std::memcpy(P.image.data() + off, v.data(), v.size() * sizeof(int32_t));
  };
  put(L.suffix_page_indptr, P.suffix_page_indptr);
  put(L.suffix_page_indices, P.suffix_page_indices);
  put(L.suffix_start, P.suffix_start);
  put(L.suffix_len, P.suffix_len);
  put(L.split_indptr, P.split_indptr);
  put(L.split_req, P.split_req);
  put(L.split_begin, P.split_begin);
  put(L.split_end, P.split_end);
  put(L.split_desc, P.split_desc);
  put(L.req_group, P.req_group);
  put(L.req_part_indptr, P.req_part_indptr);
  put(L.req_part, P.req_part);
  put(L.group_page_indptr, P.group_page_indptr);
  put(L.group_page_indices, P.group_page_indices);
  put(L.group_m_eff, P.group_m_eff);
  put(L.group_shared_len, P.group_shared_len);
  put(L.group_member_indptr, P.group_member_indptr);
  put(L.group_members, P.group_members);
  put(L.group_chunk_indptr, P.group_chunk_indptr);
  put(L.chunk_group, P.chunk_group);
  put(L.chunk_begin, P.chunk_begin);
  put(L.chunk_end, P.chunk_end);
  put(L.chunk_row_offset, P.chunk_row_offset);
  put(L.item_desc_dense, P.item_desc_dense);
  put(L.item_chunk_dense, P.item_chunk_dense);
  put(L.item_rb_dense, P.item_rb_dense);
  put(L.item_chunk_cascade, P.item_chunk_cascade);
  put(L.item_rb_cascade, P.item_rb_cascade);
  put(L.kv_indptr, P.kv_indptr);

  psp_plan_info& I = P.info;
  I.batch_size = B;
  I.num_groups = NG;
  I.num_splits = P.NS;
  I.num_chunks = P.NC;
  I.suffix_pages = static_cast<int64_t>(P.suffix_page_indices.size());
  I.group_pages = static_cast<int64_t>(P.group_page_indices.size());
  I.kv_indices_len = P.kv_indices_len;
  I.suffix_tokens = P.suffix_tokens;
  I.shared_tokens = P.shared_tokens;
  I.workspace_bytes = static_cast<int64_t>(L.total);
  I.suffix_ctas = P.NS * Hkv;
  I.prefix_dense_ctas = static_cast<int32_t>(P.item_chunk_dense.size()) * Hkv;
  I.prefix_cascade_ctas = static_cast<int32_t>(P.item_chunk_cascade.size()) * Hkv;
  I.merge_rows = B * c.num_q_heads;
  I.num_sms = static_cast<int32_t>(sms);
  I.dense_threshold = threshold;
  I.tile_tokens = psp::kTileTokens;
  I.split_min_tiles = h->split_min_tiles;
  I.split_ctas_per_sm = h->split_ctas_per_sm;
  I.prefix_rows_dense = psp::kDenseRows;
  I.prefix_rows_cascade = psp::kCascadeRows;
  I.prefix_min_tiles = h->prefix_min_tiles;
  I.prefix_ctas_per_sm = h->prefix_ctas_per_sm;
  I.read_once_min_tokens = min_tokens;
  I.read_once_min_mib = min_mib;
  I.token_bytes = static_cast<int32_t>(token_bytes);
  return PSP_OK;
}

const std::vector<int32_t>* field_vector(const HostPlan& P, int32_t field) {
  switch (field) {
    case PSP_FIELD_SUFFIX_START: return &P.suffix_start;
    case PSP_FIELD_SUFFIX_LEN: return &P.suffix_len;
    case PSP_FIELD_SUFFIX_PAGE_INDPTR: return &P.suffix_page_indptr;
    case PSP_FIELD_SUFFIX_PAGE_INDICES: return &P.suffix_page_indices;
    case PSP_FIELD_SPLIT_INDPTR: return &P.split_indptr;
    case PSP_FIELD_SPLIT_BEGIN: return &P.split_begin;
    case PSP_FIELD_SPLIT_END: return &P.split_end;
    case PSP_FIELD_GROUP_SHARED_LEN: return &P.group_shared_len;
    case PSP_FIELD_GROUP_PAGE_INDPTR: return &P.group_page_indptr;
    case PSP_FIELD_GROUP_PAGE_INDICES: return &P.group_page_indices;
    case PSP_FIELD_GROUP_M_EFF: return &P.group_m_eff;
    case PSP_FIELD_GROUP_BRANCH: return &P.group_branch;
    case PSP_FIELD_GROUP_ROW_BLOCKS: return &P.group_row_blocks;
    case PSP_FIELD_GROUP_CHUNK_INDPTR: return &P.group_chunk_indptr;
    case PSP_FIELD_CHUNK_BEGIN: return &P.chunk_begin;
    case PSP_FIELD_CHUNK_END: return &P.chunk_end;
    case PSP_FIELD_KV_INDPTR: return &P.kv_indptr;
    case PSP_FIELD_REQ_LEVEL_INDPTR: return &P.req_level_indptr;
    case PSP_FIELD_REQ_LEVEL_GROUP: return &P.req_level_group;
  }
  return nullptr;
}

StepParams make_params(const psp_handle* h, const psp_tensors* t) {
  const psp_config& c = h->cfg;
  const HostPlan& P = h->plan;
  const PlanLayout& L = P.layout;
  unsigned char* ws = h->workspace;
  StepParams p{};
  p.batch = P.B;
  p.hq = c.num_q_heads;
  p.hkv = c.num_kv_heads;
  p.group = h->group;
  p.head_dim = c.head_dim;
  p.page_size = c.page_size;
  p.page_shift = h->page_shift;
  p.kv_dtype = c.kv_dtype;
  p.q_dtype = c.q_dtype;
  p.o_dtype = c.o_dtype;
  p.num_pages = c.num_pages;
  p.token_flat = (c.flags & PSP_FLAG_TOKEN_FLAT) ? 1 : 0;
  p.concurrent = ((c.flags & PSP_FLAG_CONCURRENT) && h->allow_concurrent) ? 1 : 0;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c.head_dim)));
  if (t) {
    p.q = t->q;
    p.k_pool = t->k_pool;
    p.v_pool = t->v_pool;
    p.k_scale = t->k_scale;
    p.v_scale = t->v_scale;
    p.o = t->o;
    p.lse = t->lse;
  }
  auto I = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  p.suffix_page_indptr = I(L.suffix_page_indptr);
  p.suffix_page_indices = I(L.suffix_page_indices);
  p.suffix_start = I(L.suffix_start);
  p.suffix_len = I(L.suffix_len);
  p.split_indptr = I(L.split_indptr);
  p.split_req = I(L.split_req);
  p.split_begin = I(L.split_begin);
  p.split_end = I(L.split_end);
  p.split_desc = reinterpret_cast<const psp::SplitDesc*>(I(L.split_desc));
  p.req_group = I(L.req_group);
  p.req_part_indptr = I(L.req_part_indptr);
  p.req_part = reinterpret_cast<const int2*>(I(L.req_part));
  p.group_page_indptr = I(L.group_page_indptr);
  p.group_page_indices = I(L.group_page_indices);
  p.group_m_eff = I(L.group_m_eff);
  p.group_shared_len = I(L.group_shared_len);
  p.group_member_indptr = I(L.group_member_indptr);
  p.group_members = I(L.group_members);
  p.group_chunk_indptr = I(L.group_chunk_indptr);
  p.chunk_group = I(L.chunk_group);
  p.chunk_begin = I(L.chunk_begin);
  p.chunk_end = I(L.chunk_end);
  p.chunk_row_offset = I(L.chunk_row_offset);
  p.item_desc_dense = reinterpret_cast<const psp::DenseItemDesc*>(I(L.item_desc_dense));
  p.item_chunk_dense = I(L.item_chunk_dense);
  p.item_rb_dense = I(L.item_rb_dense);
  p.item_chunk_cascade = I(L.item_chunk_cascade);
  p.item_rb_cascade = I(L.item_rb_cascade);
  p.kv_indptr = I(L.kv_indptr);
  p.kv_indices = I(L.kv_indices);
  p.o_suf = F(L.o_suf);
  p.lse_suf = F(L.lse_suf);
  p.o_pre = F(L.o_pre);
  p.lse_pre = F(L.lse_pre);
  p.status = I(L.status);
  p.done_ctas = I(L.status + 32);    // inside the status block, cleared with it at upload
  p.prefix_done = I(L.status + 48);
  {
    int64_t rows = 0;  // sum over prefix chunks of M_eff of the chunk's group, for every KV head
    for (size_t ci = 0; ci < P.chunk_group.size(); ++ci) rows += P.group_m_eff[P.chunk_group[ci]];
    p.prefix_rows_total = static_cast<int32_t>(rows * c.num_kv_heads);
  }
  p.counters = I(L.counters);
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The argument checks of a step, made before anything is copied or launched.
psp_status check_tensors(psp_handle* h, const psp_tensors* t) {
  if (!t || !t->q || !t->k_pool || !t->v_pool || !t->o)
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "q, k_pool, v_pool and o must be set");
  if (h->cfg.kv_dtype == PSP_DTYPE_FP8_E4M3 && (!t->k_scale || !t->v_scale))
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "fp8 KV needs k_scale and v_scale");
  if (!aligned16(t->q) || !aligned16(t->k_pool) || !aligned16(t->v_pool) || !aligned16(t->o))
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "tensors must be 16-byte aligned");
  return PSP_OK;
}

}  // namespace

// =================================================================== C ABI

extern "C" {

const char* psp_version(void) { return "psp 0.1 sm_103a"; }

const char* psp_status_string(psp_status s) {
  switch (s) {
    case PSP_OK: return "ok";
    case PSP_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PSP_ERR_UNSUPPORTED: return "unsupported configuration";
    case PSP_ERR_PAGE_OUT_OF_RANGE: return "page id out of range";
    case PSP_ERR_LENGTH: return "context length and page count disagree";
    case PSP_ERR_PREFIX_MISMATCH: return "prefix group members disagree";
    case PSP_ERR_NO_PLAN: return "no plan";
    case PSP_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case PSP_ERR_CUDA: return "CUDA error";
    case PSP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case PSP_ERR_HOST_ALLOC: return "host allocation failed";
    case PSP_ERR_CAPACITY: return "buffer too small";
  }
  return "unknown status";
}

psp_status psp_create(const psp_config* cfg, psp_handle** out) {
  if (!cfg || !out) return fail(nullptr, PSP_ERR_INVALID_ARGUMENT, "cfg or out is NULL");
  *out = nullptr;
  const psp_config& c = *cfg;
  if (c.num_q_heads < 1 || c.num_kv_heads < 1 || c.head_dim < 1 || c.page_size < 1 || c.num_pages < 1 ||
      c.num_sms < 0 || c.dense_threshold < 0)
    return fail(nullptr, PSP_ERR_INVALID_ARGUMENT, "non-positive size in psp_config");
  if (c.num_q_heads % c.num_kv_heads)
    return fail(nullptr, PSP_ERR_INVALID_ARGUMENT, "num_q_heads is not a multiple of num_kv_heads");
  const int G = c.num_q_heads / c.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(nullptr, PSP_ERR_UNSUPPORTED, "GQA group size must be 1, 2, 4 or 8");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(nullptr, PSP_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if ((c.page_size & (c.page_size - 1)) || c.page_size > 1024)
    return fail(nullptr, PSP_ERR_UNSUPPORTED, "page_size must be a power of two in [1, 1024]");
  const bool f32 = c.kv_dtype == PSP_DTYPE_F32 && c.q_dtype == PSP_DTYPE_F32;
  const bool low = (c.kv_dtype == PSP_DTYPE_BF16 || c.kv_dtype == PSP_DTYPE_FP8_E4M3) && c.q_dtype == PSP_DTYPE_BF16;
  if (!f32 && !low) return fail(nullptr, PSP_ERR_UNSUPPORTED, "unsupported q/kv dtype combination");
  if (c.o_dtype != PSP_DTYPE_F32 && c.o_dtype != PSP_DTYPE_BF16)
    return fail(nullptr, PSP_ERR_UNSUPPORTED, "o_dtype must be F32 or BF16");
  if (c.flags & ~(PSP_FLAG_TOKEN_FLAT | PSP_FLAG_CONCURRENT))
    return fail(nullptr, PSP_ERR_INVALID_ARGUMENT, "unknown flag");
  const int64_t slots = static_cast<int64_t>(c.num_pages) * c.page_size;
  if (slots * c.num_kv_heads * c.head_dim > (int64_t{1} << 40))
    return fail(nullptr, PSP_ERR_INVALID_ARGUMENT, "pool too large");
  if (slots > INT32_MAX) return fail(nullptr, PSP_ERR_INVALID_ARGUMENT, "pool slots exceed int32");
  psp_handle* h = new (std::nothrow) psp_handle();
  if (!h) return fail(nullptr, PSP_ERR_HOST_ALLOC, "handle allocation failed");
  h->cfg = c;
  h->group = G;
  while ((1 << h->page_shift) < c.page_size) ++h->page_shift;
  h->split_min_tiles = env_int("PSP_SPLIT_MIN_TILES", kSplitMinTiles);
  h->split_ctas_per_sm = env_int("PSP_SPLIT_CTAS_PER_SM", kSplitCtasPerSm);
  h->prefix_min_tiles = env_int("PSP_PREFIX_MIN_TILES", kPrefixMinTiles);
  h->prefix_ctas_per_sm = env_int("PSP_PREFIX_CTAS_PER_SM", kPrefixCtasPerSm);
  h->pdl_form = env_int("PSP_PDL_FORM", 0);
  h->log = env_int("PSP_LOG", 0) > 0;
  h->env_num_sms = std::max(0, env_int("PSP_NUM_SMS", 0));
  h->nvtx = env_int("PSP_NVTX", 0) > 0;
  {
    const int hw = std::max(1, static_cast<int>(std::thread::hardware_concurrency()));
    h->plan_threads = std::max(1, std::min({16, hw, env_int("PSP_PLAN_THREADS", 8)}));
  }
  if (c.dense_threshold == 0) {
    const int t = env_int("PSP_DENSE_THRESHOLD", 0);
    if (t > 0) h->cfg.dense_threshold = t;
  }
  *out = h;
  return PSP_OK;
}

void psp_destroy(psp_handle* h) {
  if (!h) return;
  if (h->staging) cudaFreeHost(h->staging);
  if (h->staging_done) cudaEventDestroy(h->staging_done);
  if (h->fork_ev) cudaEventDestroy(h->fork_ev);
  if (h->join_ev) cudaEventDestroy(h->join_ev);
  if (h->side) cudaStreamDestroy(h->side);
  for (cudaEvent_t e : h->events) cudaEventDestroy(e);
  delete h;
}

const char* psp_last_error(const psp_handle* h) {
  return h ? h->last_error.c_str() : g_create_error.c_str();
}

}  // extern "C"

namespace {

// The record of one planned step ("The 25% Page-Size Slowdown That Wasn't", "The
// workflow": log the shapes, the index and page-table lengths and what the dispatcher
// chose, per step, before reading any timing): one JSON object on one stderr line.
void log_plan(const psp_handle* h, const psp_batch* bt) {
  const psp_config& c = h->cfg;
  const HostPlan& P = h->plan;
  const psp_plan_info& I = P.info;
  static const char* kDtype[] = {"f32", "bf16", "fp8_e4m3"};
  static const char* kBranch[] = {"none", "cascade", "dense", "paged"};
  int64_t page_entries = bt->batch_size > 0 ? bt->page_indptr[bt->batch_size] : 0;
  std::string s;
  s.reserve(512 + 96 * static_cast<size_t>(P.NG));
  char buf[512];
  std::snprintf(buf, sizeof buf,
                "psp_step {\"batch\": %d, \"num_q_heads\": %d, \"num_kv_heads\": %d, \"head_dim\": %d, "
                "\"q_dtype\": \"%s\", \"kv_dtype\": \"%s\", \"o_dtype\": \"%s\", \"page_size\": %d, "
                "\"num_pages\": %d, \"token_flat\": %s, \"page_table_len\": %lld, \"kv_indices_len\": %lld, "
                "\"suffix_tokens\": %lld, \"shared_tokens\": %lld, \"num_splits\": %d, \"num_chunks\": %d, "
                "\"suffix_ctas\": %d, \"prefix_dense_ctas\": %d, \"prefix_cascade_ctas\": %d, "
                "\"dense_threshold\": %d, \"num_sms\": %d, \"workspace_bytes\": %lld, \"coerced\": false, "
                "\"groups\": [",
                P.B, c.num_q_heads, c.num_kv_heads, c.head_dim, kDtype[c.q_dtype], kDtype[c.kv_dtype],
                kDtype[c.o_dtype], c.page_size, c.num_pages, (c.flags & PSP_FLAG_TOKEN_FLAT) ? "true" : "false",
                static_cast<long long>(page_entries), static_cast<long long>(I.kv_indices_len),
                static_cast<long long>(I.suffix_tokens), static_cast<long long>(I.shared_tokens), I.num_splits,
                I.num_chunks, I.suffix_ctas, I.prefix_dense_ctas, I.prefix_cascade_ctas, I.dense_threshold,
                I.num_sms, static_cast<long long>(I.workspace_bytes));
  s += buf;
  for (int g = 0; g < P.NG; ++g) {
    std::snprintf(buf, sizeof buf,
                  "%s{\"group\": %d, \"parent\": %d, \"members\": %d, \"m_eff\": %d, \"shared_tokens\": %d, "
                  "\"branch\": \"%s\", \"chunks\": %d}",
                  g ? ", " : "", g, bt->group_parent ? bt->group_parent[g] : -1,
                  P.group_member_indptr[g + 1] - P.group_member_indptr[g], P.group_m_eff[g],
                  P.group_shared_len[g], kBranch[P.group_branch[g]],
                  P.group_chunk_indptr[g + 1] - P.group_chunk_indptr[g]);
    s += buf;
  }
  s += "]}\n";
  std::fputs(s.c_str(), stderr);
}

}  // namespace

extern "C" {

psp_status psp_plan(psp_handle* h, const psp_batch* batch) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  h->planned = false;
  h->uploaded = false;
  NvtxRange range(h->nvtx, "psp_plan");
  if (h->num_sms_resolved == 0) {
    if (h->cfg.num_sms > 0) {
      h->num_sms_resolved = h->cfg.num_sms;
    } else if (h->env_num_sms > 0) {
      h->num_sms_resolved = h->env_num_sms;
    } else {
      int dev = 0, n = 0;
      cudaError_t e = cudaGetDevice(&dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(h, e, "querying the SM count");
      h->num_sms_resolved = std::max(1, n);
    }
  }
  psp_status st = validate_batch(h, batch);
  if (st) return st;
  try {
    st = build_plan(h, batch, h->plan);
  } catch (const std::bad_alloc&) {
    return fail(h, PSP_ERR_HOST_ALLOC, "plan allocation failed");
  }
  if (st) return st;
  h->planned = true;
  h->last_error.clear();
  if (h->log) log_plan(h, batch);
  return PSP_OK;
}

psp_status psp_plan_info_get(const psp_handle* h, psp_plan_info* out) {
  if (!h || !out) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->planned) return PSP_ERR_NO_PLAN;
  *out = h->plan.info;
  return PSP_OK;
}

psp_status psp_workspace_size(const psp_handle* h, size_t* bytes) {
  if (!h || !bytes) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->planned) return PSP_ERR_NO_PLAN;
  *bytes = h->plan.layout.total;
  return PSP_OK;
}

psp_status psp_plan_query(const psp_handle* h, int32_t field, void* dst, size_t cap_bytes, size_t* needed) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->planned) return PSP_ERR_NO_PLAN;
  const std::vector<int32_t>* v = field_vector(h->plan, field);
  if (!v) return PSP_ERR_INVALID_ARGUMENT;
  const size_t bytes = v->size() * sizeof(int32_t);
  if (needed) *needed = bytes;
  if (bytes == 0) return PSP_OK;
  if (!dst || cap_bytes < bytes) return PSP_ERR_CAPACITY;
  std::memcpy(dst, v->data(), bytes);
  return PSP_OK;
}

psp_status psp_upload(psp_handle* h, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  NvtxRange range(h->nvtx, "psp_upload");
  if (!h->planned) return fail(h, PSP_ERR_NO_PLAN, "psp_upload before psp_plan");
  const HostPlan& P = h->plan;
  const PlanLayout& L = P.layout;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % psp::kWorkspaceAlign) || workspace_bytes < L.total)
    return fail(h, PSP_ERR_WORKSPACE, "workspace needs " + std::to_string(L.total) + " bytes, 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (h->staging_done) {
    e = cudaEventSynchronize(h->staging_done);   // the previous upload has left the staging
    if (e != cudaSuccess) return cuda_fail(h, e, "waiting for the previous upload");
  } else {
    e = cudaEventCreateWithFlags(&h->staging_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventCreate");
  }
  if (h->staging_bytes < L.zero_end) {
    if (h->staging) cudaFreeHost(h->staging);
    h->staging = nullptr;
    h->staging_bytes = 0;
    const size_t want = std::max<size_t>(L.zero_end, 1 << 16) * 5 / 4;
    e = cudaHostAlloc(reinterpret_cast<void**>(&h->staging), want, cudaHostAllocDefault);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaHostAlloc (plan staging)");
    h->staging_bytes = want;
  }
  // one copy: the plan's integer arrays, then the zeroed status word and merge counters
  std::memcpy(h->staging, P.image.data(), L.zero_end);
  e = cudaMemcpyAsync(workspace, h->staging, L.zero_end, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "plan upload");
  e = cudaEventRecord(h->staging_done, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventRecord");
  h->workspace = static_cast<unsigned char*>(workspace);
  h->workspace_bytes = workspace_bytes;
  h->uploaded = true;
  return PSP_OK;
}

psp_status psp_set_kernel_timing(psp_handle* h, int32_t enable) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  h->timing = enable != 0;
  h->recorded = 0;
  return PSP_OK;
}

psp_status psp_kernel_times(psp_handle* h, float* ms, const char** names, int32_t cap, int32_t* count) {
  if (!h || !count || cap < 0 || (cap > 0 && !ms)) return PSP_ERR_INVALID_ARGUMENT;
  *count = h->recorded;
  for (int i = 0; i < h->recorded && i < cap; ++i) {
    float t = 0.f;
    cudaError_t e = cudaEventElapsedTime(&t, h->events[2 * i], h->events[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventElapsedTime");
    ms[i] = t;
    if (names) names[i] = h->event_names[i];
  }
  return PSP_OK;
}

static psp_status timed_launch(psp_handle* h, cudaStream_t s, const char* name, int& slot,
                               cudaError_t (*fn)(const StepParams&, int, cudaStream_t), const StepParams& p,
                               int n) {
  cudaError_t e;
  if (h->timing) {
    while (static_cast<int>(h->events.size()) < 2 * (slot + 1)) {
      cudaEvent_t ev;
      e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventCreate");
      h->events.push_back(ev);
    }
    if (static_cast<int>(h->event_names.size()) < slot + 1) h->event_names.resize(slot + 1);
    h->event_names[slot] = name;
    e = cudaEventRecord(h->events[2 * slot], s);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventRecord");
  }
  {
    NvtxRange range(h->nvtx, name);
    e = fn(p, n, s);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, name);
  if (h->timing) {
    e = cudaEventRecord(h->events[2 * slot + 1], s);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventRecord");
    ++slot;
    h->recorded = slot;
  }
  return PSP_OK;
}

static cudaError_t expand_entry(const StepParams& p, int, cudaStream_t s) {
  return psp::launch_expand_kv_indices(p, p.kv_indices, s);
}

psp_status psp_run(psp_handle* h, const psp_tensors* t, void* stream) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  NvtxRange range(h->nvtx, "psp_run");
  if (!h->planned || !h->uploaded) return fail(h, PSP_ERR_NO_PLAN, "psp_run needs psp_plan and psp_upload first");
  const psp_status bad = check_tensors(h, t);
  if (bad) return bad;
  const HostPlan& P = h->plan;
  h->recorded = 0;  // an empty step launches nothing and reports no kernel times
  if (P.B == 0) return PSP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StepParams p = make_params(h, t);
  int slot = 0;
  psp_status st;
  const int nd = static_cast<int>(P.item_chunk_dense.size());
  const int nc = static_cast<int>(P.item_chunk_cascade.size());
  const bool fork = p.concurrent && (nd > 0 || nc > 0) && P.NS > 0;
  // The suffix kernel follows the prefix kernel as a programmatic dependent: its CTAs start
  // on the SMs the prefix kernel leaves free and never wait for it.  The two kernels then
  // run at the same time, so every part of a (request, KV head) arrives on its counter and
  // the last arrival merges (the concurrent protocol).  Not with per-kernel timing (events
  // between the launches) nor when the prefix runs on its own stream.
  p.pdl = (!fork && !h->timing && (nd > 0 || nc > 0) && P.NS > 0) ? 1 : 0;
  // Two forms (measured on GB300).  Concurrent: the suffix kernel never waits and uses the
  // concurrent merge protocol.  Sequential: the suffix CTAs wait for the prefix grid before
  // reading prefix partials.  The concurrent form wins when the prefix grid leaves at least
  // half of the SMs free (short prefixes: 76 vs 81 us) or when its CTAs run long, so that the
  // SMs it leaves free do a large share of the suffix meanwhile (16384-token chunks, e4m3
  // batch: 384 vs 395 us); with short chunks on a full GPU the sequential form is ahead
  // (1024-token chunks, agent batch: 138 vs 140 us).
  if (p.pdl) {
    int32_t longest = 0;
    for (size_t ci = 0; ci < P.chunk_begin.size(); ++ci) longest = std::max(longest, P.chunk_end[ci] - P.chunk_begin[ci]);
    if (static_cast<int64_t>(nd + nc) * p.hkv * 2 <= h->num_sms_resolved || longest >= kConcurrentChunkTokens)
      p.concurrent = 1;
  }
  // PSP_PDL_FORM overrides the choice for measurements: 1 sequential, 2 concurrent
  if (p.pdl && h->pdl_form == 1) p.concurrent = 0;
  if (p.pdl && h->pdl_form == 2) p.concurrent = 1;
  if (p.token_flat) {
    st = timed_launch(h, s, "expand_kv_indices", slot, expand_entry, p, 0);
    if (st) return st;
  }
  cudaStream_t ps = s;  // stream of the prefix kernels
  cudaError_t e;
  if (fork) {
    if (!h->side) {
      e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->fork_ev, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->join_ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(h, e, "creating the prefix stream");
    }
    e = cudaEventRecord(h->fork_ev, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->side, h->fork_ev, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "forking the prefix stream");
    ps = h->side;
  }
  if (nd > 0) {
    st = timed_launch(h, ps, "prefix_dense", slot, psp::launch_prefix_dense, p, nd);
    if (st) return st;
  }
  if (nc > 0) {
    st = timed_launch(h, ps, "prefix_cascade", slot, psp::launch_prefix_cascade, p, nc);
    if (st) return st;
  }
  if (P.NS > 0) {
    st = timed_launch(h, s, "suffix_splitkv", slot, psp::launch_suffix, p, P.NS);
    if (st) return st;
  }
  if (fork) {
    e = cudaEventRecord(h->join_ev, ps);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h->join_ev, 0);
    if (e != cudaSuccess) return cuda_fail(h, e, "joining the prefix stream");
  }
  return PSP_OK;
}

psp_status psp_step_host(psp_handle* h, const psp_batch* batch, const void* q_host, void* o_host, float* lse_host,
                         const psp_tensors* dev, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  if (!q_host || !o_host || !dev || !dev->q || !dev->o || (lse_host && !dev->lse))
    return fail(h, PSP_ERR_INVALID_ARGUMENT, "host and device staging buffers must be set");
  if (!batch || batch->batch_size < 0) return fail(h, PSP_ERR_INVALID_ARGUMENT, "batch is NULL or negative");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const psp_config& c = h->cfg;
  const size_t rows = static_cast<size_t>(batch->batch_size) * c.num_q_heads;
  // the query copy does not depend on the plan: it runs while the host plans
  cudaError_t e = cudaMemcpyAsync(const_cast<void*>(dev->q), q_host, rows * c.head_dim * dtype_bytes(c.q_dtype),
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "copying q to the device");
  psp_status st = psp_plan(h, batch);
  if (st) return st;
  st = psp_upload(h, workspace, workspace_bytes, stream);
  if (st) return st;
  st = psp_run(h, dev, stream);
  if (st) return st;
  e = cudaMemcpyAsync(o_host, dev->o, rows * c.head_dim * dtype_bytes(c.o_dtype), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "copying o to the host");
  if (lse_host) {
    e = cudaMemcpyAsync(lse_host, dev->lse, rows * sizeof(float), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "copying lse to the host");
  }
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  return PSP_OK;
}

psp_status psp_expand_kv_indices(psp_handle* h, int32_t* kv_indices, int64_t cap, void* stream) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->planned || !h->uploaded) return fail(h, PSP_ERR_NO_PLAN, "psp_expand_kv_indices needs an uploaded plan");
  if (cap < h->plan.kv_indices_len) return fail(h, PSP_ERR_CAPACITY, "kv_indices capacity too small");
  if (h->plan.kv_indices_len == 0) return PSP_OK;
  if (!kv_indices || !aligned16(kv_indices)) return fail(h, PSP_ERR_INVALID_ARGUMENT, "kv_indices NULL or misaligned");
  StepParams p = make_params(h, nullptr);
  cudaError_t e = psp::launch_expand_kv_indices(p, kv_indices, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "expand_kv_indices");
  return PSP_OK;
}

psp_status psp_wait_selftest(psp_handle* h, int32_t polls, void* stream) {
  if (!h || polls < 1) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->uploaded) return fail(h, PSP_ERR_NO_PLAN, "no workspace bound");
  int32_t* status = reinterpret_cast<int32_t*>(h->workspace + h->plan.layout.status);
  cudaError_t e = psp::launch_wait_selftest(status, static_cast<uint32_t>(polls), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(h, e, "wait self test");
  return PSP_OK;
}

psp_status psp_device_status(psp_handle* h, int32_t* code) {
  if (!h || !code) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->uploaded) return fail(h, PSP_ERR_NO_PLAN, "no workspace bound");
  cudaError_t e = cudaMemcpy(code, h->workspace + h->plan.layout.status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "reading the device status word");
  if ((*code & 0xff) == psp::kDevTimeout) return fail(h, PSP_ERR_DEVICE_TIMEOUT, "a bounded device wait ran out");
  return PSP_OK;
}

}  // extern "C"

// ------------------------------------------------- workspace-free entry point support

namespace psp {

psp_status set_error(psp_handle* h, psp_status code, const char* msg) { return fail(h, code, msg); }

// Copies the plan's host image into caller-provided device scratch without any
// allocation (pageable source, no pinned staging), clears the status word, binds
// the scratch as the handle's workspace and launches the step.  Every argument check
// of psp_run comes first, so a rejected call has written nothing into the scratch (which
// every handle shares) and leaves the handle's binding as it was; a call that fails after
// the copy restores the previous binding too.  Kernel timing events are not recorded on
// this path (creating them would allocate).
psp_status bind_image_and_run(psp_handle* h, unsigned char* ws, size_t cap, const psp_tensors* t,
                              cudaStream_t s) {
  if (!h) return PSP_ERR_INVALID_ARGUMENT;
  if (!h->planned) return fail(h, PSP_ERR_NO_PLAN, "psp_run_noalloc before psp_plan");
  const PlanLayout& L = h->plan.layout;
  if (L.total > cap)
    return fail(h, PSP_ERR_WORKSPACE,
                "the plan needs " + std::to_string(L.total) + " bytes of scratch but the static scratch holds " +
                    std::to_string(cap) + " bytes; plan a smaller batch or use psp_upload with a workspace");
  const psp_status bad = check_tensors(h, t);
  if (bad) return bad;
  unsigned char* const prev_ws = h->workspace;
  const size_t prev_bytes = h->workspace_bytes;
  const bool prev_uploaded = h->uploaded;
  // the image runs through zero_end: the status word and merge counters arrive as zeros
  cudaError_t e = cudaMemcpyAsync(ws, h->plan.image.data(), L.zero_end, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "plan copy into the static scratch");
  h->workspace = ws;
  h->workspace_bytes = cap;
  h->uploaded = true;
  const bool timing = h->timing;
  h->timing = false;
  h->allow_concurrent = false;
  const psp_status st = psp_run(h, t, s);
  h->allow_concurrent = true;
  h->timing = timing;
  if (st != PSP_OK) {
    h->workspace = prev_ws;
    h->workspace_bytes = prev_bytes;
    h->uploaded = prev_uploaded;
  }
  return st;
}

}  // namespace psp
