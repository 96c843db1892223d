/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged shared-prefix decode
 * attention.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call it; the product library never does,
 * and the two share no code.
 *
 * What it computes, and where that is defined:
 *
 *  - Attention: for one decode token of request b and query head hq, plain
 *    softmax(q K^T / sqrt(d)) V over every context token of the request, in
 *    fp64, with the keys and values gathered token by token through the
 *    block table.  Paging and sharing leave this result unchanged ("Track C
 *    Document 10 -- Shrinking the footprint", PagedAttention Q&A: the results
 *    are identical; "The 25% Page-Size Slowdown That Wasn't", "When source
 *    beats intuition": index layout changes which bytes are read, not the
 *    math).  GQA head mapping h = hq / (Hq/Hkv); no mask beyond the context
 *    length; LSE is the natural log of the softmax normaliser.
 *
 *  - kv_indices: the token-flat lowering, one pool slot per context token,
 *    slot = page[t / ps] * ps + t % ps, B x context_length entries ("The 25%
 *    Page-Size Slowdown That Wasn't", "Four meanings of page size").
 *
 *  - Plan: block-aligned prefix sharing (floor(P/ps) shared pages, the tail
 *    stays private: "Track C Document 10", block size answer: 2,003 tokens at
 *    16 share 125 blocks), M_eff = members x GQA group and the dense/cascade
 *    rule M_eff >= threshold ("GraniKV", section 3 Per-step dispatcher),
 *    nested groups (a radix tree of shared beginnings, each level matched
 *    block-aligned and read once for all requests below it), and the
 *    split-KV partition.  The pages fix neither the partition rule nor the
 *    threshold value; the rule implemented here is the library's documented
 *    rule (token units, independent of page size), restated from its
 *    description with every constant passed in.
 *
 *  - decode(): bf16 = the upper half of an IEEE binary32; fp8 = OCP e4m3
 *    ("fn": bias 7, 3 mantissa bits, subnormals at exponent 0, 0x7F/0xFF NaN,
 *    no infinities), dequantised as code value x per-head scale.
 *
 * The merge of two partial results (used only by a self-check) is the
 * log-sum-exp combination of (O1, lse1) and (O2, lse2).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_FP8_E4M3 = 2 };
enum { OR_OK = 0, OR_EARG = -1, OR_EUNSUP = -2, OR_ERANGE = -3, OR_ELEN = -4,
       OR_EPREFIX = -5, OR_ECAP = -6, OR_ENOMEM = -7 };
enum { OR_BRANCH_NONE = 0, OR_BRANCH_CASCADE = 1, OR_BRANCH_DENSE = 2, OR_BRANCH_PAGED = 3 };

/* ---------------------------------------------------------------- decode */

double oracle_decode_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double oracle_decode_fp8_e4m3(uint8_t code) {
  int sign = (code >> 7) & 1;
  int exponent = (code >> 3) & 0xF;
  int mantissa = code & 0x7;
  double v;
  if (exponent == 0xF && mantissa == 0x7) return NAN;       /* S.1111.111 */
  if (exponent == 0)
    v = ldexp((double)mantissa / 8.0, 1 - 7);                /* subnormal */
  else
    v = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
  return sign ? -v : v;
}

static double elem(const void* base, int64_t idx, int dtype) {
  switch (dtype) {
    case OR_F32: return (double)((const float*)base)[idx];
    case OR_BF16: return oracle_decode_bf16(((const uint16_t*)base)[idx]);
    case OR_FP8_E4M3: return oracle_decode_fp8_e4m3(((const uint8_t*)base)[idx]);
  }
  return NAN;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------- block table math */

/* Pool slot of token t of request b: page[b][t / ps] * ps + t % ps. */
static int64_t slot_of(const int32_t* page_indptr, const int32_t* page_indices,
                       int b, int64_t t, int ps) {
  int32_t page = page_indices[page_indptr[b] + t / ps];
  return (int64_t)page * ps + t % ps;
}

/* Checks the block table: every kv_len >= 1, ceil(kv_len/ps) pages each, ids in range. */
static int check_table(int B, const int32_t* kv_len, const int32_t* page_indptr,
                       const int32_t* page_indices, int ps, int num_pages) {
  if (B < 0 || ps < 1 || num_pages < 0) return OR_EARG;
  if (B > 0 && (!kv_len || !page_indptr)) return OR_EARG;
  if (B > 0 && page_indptr[0] != 0) return OR_EARG;
  for (int b = 0; b < B; ++b) {
    if (kv_len[b] < 1) return OR_ELEN;
    int64_t pages = page_indptr[b + 1] - page_indptr[b];
    if (pages != ((int64_t)kv_len[b] + ps - 1) / ps) return OR_ELEN;
    for (int64_t i = page_indptr[b]; i < page_indptr[b + 1]; ++i)
      if (page_indices[i] < 0 || page_indices[i] >= num_pages) return OR_ERANGE;
  }
  return OR_OK;
}

/* Token-flat lowering: kv_indptr[B+1], kv_indices[sum kv_len]. */
int oracle_expand_kv_indices(int B, const int32_t* kv_len, const int32_t* page_indptr,
                             const int32_t* page_indices, int ps, int num_pages,
                             int32_t* kv_indptr, int32_t* kv_indices, int64_t cap) {
  int rc = check_table(B, kv_len, page_indptr, page_indices, ps, num_pages);
  if (rc) return rc;
  int64_t n = 0;
  kv_indptr[0] = 0;
  for (int b = 0; b < B; ++b) {
    for (int64_t t = 0; t < kv_len[b]; ++t) {
      if (n >= cap) return OR_ECAP;
      kv_indices[n++] = (int32_t)slot_of(page_indptr, page_indices, b, t, ps);
    }
    kv_indptr[b + 1] = (int32_t)n;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------ plan */

/* Constants of the partition rule (all in the library's documented units). */
typedef struct {
  int32_t num_sms;            /* SM count the partition is sized for */
  int32_t dense_threshold;    /* M_eff >= this -> dense prefix branch */
  int32_t tile_tokens;        /* partition granule in tokens */
  int32_t split_min_tiles;    /* smallest suffix split, in granules */
  int32_t split_ctas_per_sm;  /* suffix target: this many (split, head) items per SM */
  int32_t prefix_rows_dense;  /* stacked query rows per dense prefix item */
  int32_t prefix_rows_cascade;
  int32_t prefix_min_tiles;   /* smallest prefix chunk, in granules */
  int32_t prefix_ctas_per_sm; /* prefix target: at most this many items per SM */
  int32_t read_once_min_tokens; /* shared tokens below this -> paged branch (< 0: no minimum) */
  int32_t read_once_min_mib;    /* bytes saved by reading once below this many MiB -> paged (< 0: none) */
  int32_t token_bytes;          /* K + V bytes of one token, all KV heads */
} oracle_plan_params;

/* Plan outputs; capacities in elements are given by the *_cap fields. */
typedef struct {
  /* per request */
  int32_t* suffix_start;          /* [B] first private token = shared pages * ps */
  int32_t* suffix_len;            /* [B] */
  int32_t* suffix_page_indptr;    /* [B+1] */
  int32_t* suffix_page_indices;   int64_t suffix_page_cap;
  int32_t* split_indptr;          /* [B+1] */
  int32_t* split_begin;           /* token offsets within the suffix */
  int32_t* split_end;             int64_t split_cap;
  /* per group */
  int32_t* group_shared_len;      /* [num_groups] tokens of the group's own segment read once */
  int32_t* group_page_indptr;     /* [num_groups+1] */
  int32_t* group_page_indices;    int64_t group_page_cap;
  int32_t* group_m_eff;           /* [num_groups] */
  int32_t* group_branch;          /* [num_groups] */
  int32_t* group_row_blocks;      /* [num_groups] */
  int32_t* group_chunk_indptr;    /* [num_groups+1] */
  int32_t* chunk_begin;           /* token offsets within the context (the group's own segment) */
  int32_t* chunk_end;             int64_t chunk_cap;
  /* per request: the groups whose prefix partials it merges, outermost first */
  int32_t* req_level_indptr;      /* [B+1] */
  int32_t* req_level_group;       int64_t req_level_cap;
} oracle_plan_out;

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Nested prefixes.  A group may extend the prefix of another: group_parent[g] (NULL: every
 * group is a root) is -1 or a group of lower index whose prefix is no longer than g's, so the
 * groups form a radix tree of shared beginnings ("Track C Document 10 -- Shrinking the
 * footprint": the vLLM-or-SGLang answer keeps caches in a radix tree keyed on shared
 * beginnings, and the cache table's per-user personalisation row shares per user on top of
 * what every user shares).  A request of group g is a member of g and of every ancestor of g.
 * Matching stays block-aligned at every level: g shares the first floor(P_g / ps) pages, and
 * its own segment is the pages from floor(P_parent / ps) on. */
static int parent_of(const int32_t* group_parent, int g) { return group_parent ? group_parent[g] : -1; }

/* 1 if a request of group `leaf` is a member of group a */
static int member_of(const int32_t* group_parent, int leaf, int a) {
  for (int g = leaf; g >= 0; g = parent_of(group_parent, g))
    if (g == a) return 1;
  return 0;
}

/* full pages group g shares (0 for "no group") */
static int64_t shared_pages(const int32_t* group_prefix_len, int g, int ps) {
  return g >= 0 ? group_prefix_len[g] / ps : 0;
}

/* branches whose segment is read once per step */
static int read_once(int branch) { return branch == OR_BRANCH_DENSE || branch == OR_BRANCH_CASCADE; }

int oracle_plan(int B, int Hq, int Hkv, int ps, int num_pages,
                const int32_t* kv_len, const int32_t* page_indptr, const int32_t* page_indices,
                const int32_t* prefix_group, int num_groups, const int32_t* group_prefix_len,
                const int32_t* group_parent, const oracle_plan_params* pp, oracle_plan_out* out) {
  if (Hkv < 1 || Hq < 1 || Hq % Hkv) return OR_EARG;
  if (num_groups < 0 || (num_groups > 0 && !group_prefix_len)) return OR_EARG;
  if (pp->num_sms < 1 || pp->tile_tokens < 1 || pp->split_min_tiles < 1 ||
      pp->split_ctas_per_sm < 1 || pp->prefix_rows_dense < 1 || pp->prefix_rows_cascade < 1 ||
      pp->prefix_min_tiles < 1 || pp->prefix_ctas_per_sm < 1)
    return OR_EARG;
  int rc = check_table(B, kv_len, page_indptr, page_indices, ps, num_pages);
  if (rc) return rc;
  const int G = Hq / Hkv;
  const int64_t tile = pp->tile_tokens;

  /* the group tree: a parent has a lower index and a prefix no longer than its child's */
  for (int g = 0; g < num_groups; ++g) {
    if (group_prefix_len[g] < 0) return OR_EARG;
    int par = parent_of(group_parent, g);
    if (par < -1 || par >= g) return OR_EARG;
    if (par >= 0 && group_prefix_len[par] > group_prefix_len[g]) return OR_EARG;
  }
  for (int b = 0; b < B; ++b) {
    int g = prefix_group ? prefix_group[b] : -1;
    if (g < -1 || g >= num_groups) return OR_EARG;
    if (g >= 0 && group_prefix_len[g] > kv_len[b]) return OR_EPREFIX;
  }

  /* per group: its members (its own requests and its descendants'), the first of them, and
     agreement of every member with the first on the group's shared pages */
  int32_t* first_member = (int32_t*)malloc(sizeof(int32_t) * (num_groups > 0 ? num_groups : 1));
  int32_t* members = (int32_t*)calloc(num_groups > 0 ? num_groups : 1, sizeof(int32_t));
  if (!first_member || !members) { free(first_member); free(members); return OR_ENOMEM; }
  for (int g = 0; g < num_groups; ++g) {
    first_member[g] = -1;
    int64_t n_sh = shared_pages(group_prefix_len, g, ps);
    for (int b = 0; b < B; ++b) {
      int leaf = prefix_group ? prefix_group[b] : -1;
      if (leaf < 0 || !member_of(group_parent, leaf, g)) continue;
      if (first_member[g] < 0) {
        first_member[g] = b;
      } else {
        int f = first_member[g];
        for (int64_t i = 0; i < n_sh; ++i)
          if (page_indices[page_indptr[b] + i] != page_indices[page_indptr[f] + i]) {
            rc = OR_EPREFIX; goto done;
          }
      }
      members[g] += 1;
    }
  }

  /* per group: the dispatcher's branch (GraniKV section 3: M_eff = members x G against the
     dense threshold), after the read-once test on the group's own segment: it is read once
     only if it has at least read_once_min_tokens shared tokens and reading it once saves
     (members - 1) x shared tokens x token_bytes >= read_once_min_mib MiB; otherwise every
     member reads it through its own block table (the paged branch, nothing shared).  Below a
     paged group every group is paged too, so that the tokens a request reads through its own
     block table stay one range at the end of its context. */
  for (int g = 0; g < num_groups; ++g) {
    int par = parent_of(group_parent, g);
    int64_t seg = (members[g] > 0) ? shared_pages(group_prefix_len, g, ps) - shared_pages(group_prefix_len, par, ps) : 0;
    int64_t m_eff = (int64_t)members[g] * G;
    out->group_m_eff[g] = (int32_t)m_eff;
    int below_paged = 0;
    for (int a = par; a >= 0; a = parent_of(group_parent, a))
      if (out->group_branch[a] == OR_BRANCH_PAGED) below_paged = 1;
    int branch = OR_BRANCH_NONE;
    if (m_eff > 0 && seg > 0) {
      int64_t shared = seg * ps;
      int64_t saved = (int64_t)(members[g] - 1) * shared * pp->token_bytes;
      int too_short = pp->read_once_min_tokens > 0 && shared < pp->read_once_min_tokens;
      int too_little = pp->read_once_min_mib > 0 && saved < ((int64_t)pp->read_once_min_mib << 20);
      if (below_paged || too_short || too_little) branch = OR_BRANCH_PAGED;
      else branch = (m_eff >= pp->dense_threshold) ? OR_BRANCH_DENSE : OR_BRANCH_CASCADE;
    }
    out->group_branch[g] = branch;
  }

  /* per request: the read-once groups it belongs to, outermost first (ancestors have lower
     indices), and the block-aligned split of its block table after the last of them */
  {
    int64_t np_out = 0, nl = 0;
    out->suffix_page_indptr[0] = 0;
    out->req_level_indptr[0] = 0;
    for (int b = 0; b < B; ++b) {
      int leaf = prefix_group ? prefix_group[b] : -1;
      int64_t n_sh = 0;
      for (int a = 0; a < num_groups; ++a) {
        if (leaf < 0 || !member_of(group_parent, leaf, a) || !read_once(out->group_branch[a])) continue;
        if (nl >= out->req_level_cap) { rc = OR_ECAP; goto done; }
        out->req_level_group[nl++] = a;
        n_sh = group_prefix_len[a] / ps;
      }
      out->req_level_indptr[b + 1] = (int32_t)nl;
      out->suffix_start[b] = (int32_t)(n_sh * ps);
      out->suffix_len[b] = (int32_t)(kv_len[b] - n_sh * ps);
      for (int64_t i = page_indptr[b] + n_sh; i < page_indptr[b + 1]; ++i) {
        if (np_out >= out->suffix_page_cap) { rc = OR_ECAP; goto done; }
        out->suffix_page_indices[np_out++] = page_indices[i];
      }
      out->suffix_page_indptr[b + 1] = (int32_t)np_out;
    }
  }

  /* suffix split-KV partition */
  {
    int64_t total_tiles = 0;
    for (int b = 0; b < B; ++b) total_tiles += ceil_div(out->suffix_len[b], tile);
    int64_t work = (int64_t)Hkv * total_tiles;
    int64_t target = (int64_t)pp->split_ctas_per_sm * pp->num_sms;
    int64_t per_split = ceil_div(work, target);
    if (per_split < pp->split_min_tiles) per_split = pp->split_min_tiles;
    int64_t ns = 0;
    out->split_indptr[0] = 0;
    for (int b = 0; b < B; ++b) {
      int64_t S = out->suffix_len[b];
      int64_t T = ceil_div(S, tile);
      int64_t n = ceil_div(T, per_split);
      for (int64_t s = 0; s < n; ++s) {
        if (ns >= out->split_cap) { rc = OR_ECAP; goto done; }
        int64_t lo = tile * s * per_split, hi = tile * (s + 1) * per_split;
        out->split_begin[ns] = (int32_t)lo;
        out->split_end[ns] = (int32_t)(hi < S ? hi : S);
        ++ns;
      }
      out->split_indptr[b + 1] = (int32_t)ns;
    }
  }

  /* groups: shared pages (the whole prefix, ancestors' pages first), the own segment's
     tokens, row blocks and prefix chunks over the segment */
  {
    int64_t gp = 0, nc = 0;
    out->group_page_indptr[0] = 0;
    out->group_chunk_indptr[0] = 0;
    for (int g = 0; g < num_groups; ++g) {
      int branch = out->group_branch[g];
      int64_t n_sh = read_once(branch) ? group_prefix_len[g] / ps : 0;
      int64_t seg0 = read_once(branch) ? shared_pages(group_prefix_len, parent_of(group_parent, g), ps) * ps : 0;
      out->group_shared_len[g] = (int32_t)(n_sh * ps - seg0);
      for (int64_t i = 0; i < n_sh; ++i) {
        if (gp >= out->group_page_cap) { rc = OR_ECAP; goto done; }
        out->group_page_indices[gp++] = page_indices[page_indptr[first_member[g]] + i];
      }
      out->group_page_indptr[g + 1] = (int32_t)gp;
      int64_t m_eff = out->group_m_eff[g];
      int64_t rows = 0, n_chunks = 0, per_chunk = 0;
      if (read_once(branch)) {
        int64_t rows_per = (branch == OR_BRANCH_DENSE) ? pp->prefix_rows_dense : pp->prefix_rows_cascade;
        rows = ceil_div(m_eff, rows_per);
        int64_t tiles = ceil_div(out->group_shared_len[g], tile);
        int64_t items = (int64_t)Hkv * rows;
        int64_t want = ((int64_t)pp->prefix_ctas_per_sm * pp->num_sms) / items;
        int64_t most = tiles / pp->prefix_min_tiles;
        n_chunks = want < most ? want : most;
        if (n_chunks < 1) n_chunks = 1;
        per_chunk = ceil_div(tiles, n_chunks);
        n_chunks = ceil_div(tiles, per_chunk);
      }
      out->group_row_blocks[g] = (int32_t)rows;
      for (int64_t c = 0; c < n_chunks; ++c) {
        if (nc >= out->chunk_cap) { rc = OR_ECAP; goto done; }
        int64_t lo = tile * c * per_chunk, hi = tile * (c + 1) * per_chunk;
        out->chunk_begin[nc] = (int32_t)(seg0 + lo);
        out->chunk_end[nc] = (int32_t)(seg0 + (hi < out->group_shared_len[g] ? hi : out->group_shared_len[g]));
        ++nc;
      }
      out->group_chunk_indptr[g + 1] = (int32_t)nc;
    }
  }

done:
  free(first_member);
  free(members);
  return rc;
}

/* -------------------------------------------------------------- attention */

/*
 * For each requested row r: request row_b[r], query head row_hq[r], over the
 * request's context tokens t in [row_t0[r], row_t1[r]) (row_t1 < 0 means
 * kv_len), in fp64:
 *   s_t = (q . k_t) / sqrt(d)        k_t = decode(K[slot(t), h, :]) (* k_scale[h] for fp8)
 *   m = max s_t,  w_t = exp(s_t - m),  l = sum w_t
 *   O = sum_t w_t v_t / l,  LSE = m + ln l
 * An empty token range gives O = 0, LSE = -inf.
 */
int oracle_attend(int B, int Hq, int Hkv, int d, int q_dtype, int kv_dtype, int ps, int num_pages,
                  const void* q, const void* k_pool, const void* v_pool,
                  const float* k_scale, const float* v_scale,
                  const int32_t* kv_len, const int32_t* page_indptr, const int32_t* page_indices,
                  int n_rows, const int32_t* row_b, const int32_t* row_hq,
                  const int32_t* row_t0, const int32_t* row_t1,
                  double* o_out, double* lse_out) {
  if (Hkv < 1 || Hq % Hkv || d < 1) return OR_EARG;
  if (q_dtype != OR_F32 && q_dtype != OR_BF16) return OR_EUNSUP;
  if (kv_dtype != OR_F32 && kv_dtype != OR_BF16 && kv_dtype != OR_FP8_E4M3) return OR_EUNSUP;
  if (kv_dtype == OR_FP8_E4M3 && (!k_scale || !v_scale)) return OR_EARG;
  int rc = check_table(B, kv_len, page_indptr, page_indices, ps, num_pages);
  if (rc) return rc;
  for (int r = 0; r < n_rows; ++r) {
    if (row_b[r] < 0 || row_b[r] >= B || row_hq[r] < 0 || row_hq[r] >= Hq) return OR_EARG;
    int64_t t0 = row_t0 ? row_t0[r] : 0;
    int64_t t1 = (row_t1 && row_t1[r] >= 0) ? row_t1[r] : kv_len[row_b[r]];
    if (t0 < 0 || t1 < t0 || t1 > kv_len[row_b[r]]) return OR_EARG;
  }
  const int G = Hq / Hkv;
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < n_rows; ++r) {
    int b = row_b[r], hq = row_hq[r], h = hq / G;
    int64_t t0 = row_t0 ? row_t0[r] : 0;
    int64_t t1 = (row_t1 && row_t1[r] >= 0) ? row_t1[r] : kv_len[b];
    int64_t n = t1 - t0;
    double* out = o_out + (int64_t)r * d;
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    if (n == 0) { lse_out[r] = -INFINITY; continue; }
    double* qv = (double*)malloc(sizeof(double) * d);
    double* s = (double*)malloc(sizeof(double) * n);
    if (!qv || !s) { free(qv); free(s); failed = 1; continue; }
    for (int i = 0; i < d; ++i) qv[i] = elem(q, ((int64_t)b * Hq + hq) * d + i, q_dtype);
    double ks = (kv_dtype == OR_FP8_E4M3) ? (double)k_scale[h] : 1.0;
    double vs = (kv_dtype == OR_FP8_E4M3) ? (double)v_scale[h] : 1.0;
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      int64_t slot = slot_of(page_indptr, page_indices, b, t0 + j, ps);
      int64_t base = (slot * Hkv + h) * d;
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += qv[i] * (elem(k_pool, base + i, kv_dtype) * ks);
      s[j] = acc * inv_sqrt_d;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      double w = exp(s[j] - m);
      int64_t slot = slot_of(page_indptr, page_indices, b, t0 + j, ps);
      int64_t base = (slot * Hkv + h) * d;
      for (int i = 0; i < d; ++i) out[i] += w * (elem(v_pool, base + i, kv_dtype) * vs);
      l += w;
    }
    for (int i = 0; i < d; ++i) out[i] /= l;
    lse_out[r] = m + log(l);
    free(qv);
    free(s);
  }
  return failed ? OR_ENOMEM : OR_OK;
}

/* Log-sum-exp merge of two partial results over disjoint token sets. */
void oracle_merge(int n_rows, int d, const double* o1, const double* lse1,
                  const double* o2, const double* lse2, double* o_out, double* lse_out) {
  for (int r = 0; r < n_rows; ++r) {
    double a = lse1[r], c = lse2[r];
    double m = a > c ? a : c;
    if (m == -INFINITY) {
      for (int i = 0; i < d; ++i) o_out[(int64_t)r * d + i] = 0.0;
      lse_out[r] = -INFINITY;
      continue;
    }
    double lse = m + log(exp(a - m) + exp(c - m));
    double w1 = exp(a - lse), w2 = exp(c - lse);
    for (int i = 0; i < d; ++i)
      o_out[(int64_t)r * d + i] = w1 * o1[(int64_t)r * d + i] + w2 * o2[(int64_t)r * d + i];
    lse_out[r] = lse;
  }
}
