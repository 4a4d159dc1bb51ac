/*
 * CPU ORACLE for HiSparse RESOLVE -- test infrastructure only.
 *
 * A plain, slow, sequential restatement of what RESOLVE computes for one
 * (request, layer) unit and one decode step.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this file; the product
 * path never does.  It shares no code with the CUDA library.
 *
 * What it follows (page "59188saintaubert.com ... HiSparse", section 02, and
 * page "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM",
 * section "How it works"):
 *   - a per-request page table maps a logical position either to a resident
 *     GPU block (read in place, LRU untouched, the tail is never evicted) or to
 *     a "host only" marker;
 *   - a fixed per-request, per-layer hot buffer of B slots, managed by LRU:
 *     a hit refreshes the slot's LRU entry, a miss copies one row from pinned
 *     host memory into an LRU victim slot;
 *   - the resolver hands back pool row ids; hot-buffer blocks live in the same
 *     KV tensor as resident blocks, so one stride reaches both.
 * Readings where the pages are silent (stated once here, applied below):
 *   - two phases per step: every hit is refreshed first, then misses are
 *     served, so a slot selected in the current step is never the victim;
 *   - victims are the slots with stamp < step, oldest stamp first, ties to the
 *     lowest slot; the i-th miss in selection order takes the i-th victim;
 *   - empty slots hold position -1 and stamp -1;
 *   - position -1 is padding (row id -1); a position outside [0, ctx) or a
 *     repeat of an earlier position in the same row is an input error (row id
 *     -1, error bit set); misses beyond the number of victims get row id -1
 *     and the capacity error bit.
 * Speculative decoding (page "GLM 5.3 Optimizations, Part 1", sections
 * "Composition with the rest of vLLM" and "Exploiting sparsity when needed":
 * the verify steps share the request's hot state, and the hot buffer must
 * hold every verify token's selection at once).  Reading: the T verify
 * tokens' rows are resolved as one list, token after token; the whole list's
 * hits are refreshed first and its misses served in list order, so a slot any
 * token uses is pinned for the step; a position that an earlier token also
 * selected takes no second slot -- it gets the row of its first occurrence
 * (whatever that is: resident, hot, a served miss, or -1 if that miss found
 * no slot); a repeat within one token's row stays an input error.
 */
#include "resolve_oracle.h"

#include <stdlib.h>
#include <string.h>

struct or_state {
  int32_t R, L, K, B, P, max_pages;
  int64_t blocks_per_layer;
  int32_t* ctx;          /* [R] current context length */
  int32_t* ctx_cap;      /* [R] largest context the state can hold */
  int32_t* page_table;   /* [R][max_pages]: block id, or -1 = host only */
  int32_t* hot_block;    /* [R][B/P] */
  int32_t* slot_pos;     /* [L][R][B] */
  int32_t* slot_stamp;   /* [L][R][B] */
  int32_t** where;       /* [L*R] -> [ctx_cap[r]]: slot holding a position, or -1 */
  int32_t** seen;        /* [L*R] -> [ctx_cap[r]]: call serial of last sighting */
  int32_t** seen_j;      /* [L*R] -> [ctx_cap[r]]: list index of that sighting */
  int32_t* serial;       /* [L*R] */
  /* per-call scratch */
  int32_t* cand;         /* [B] */
};

static inline int64_t unit_index(const or_state* s, int32_t layer, int32_t req) {
  return (int64_t)layer * s->R + req;
}

or_state* or_create(int32_t R, int32_t L, int32_t K, int32_t B, int32_t P,
                    int32_t max_pages, int64_t blocks_per_layer,
                    const int32_t* ctx_cap) {
  if (R <= 0 || L <= 0 || K <= 0 || B <= 0 || P <= 0 || B % P != 0) return NULL;
  or_state* s = (or_state*)calloc(1, sizeof(or_state));
  if (!s) return NULL;
  s->R = R; s->L = L; s->K = K; s->B = B; s->P = P;
  s->max_pages = max_pages;
  s->blocks_per_layer = blocks_per_layer;
  s->ctx = (int32_t*)calloc((size_t)R, sizeof(int32_t));
  s->ctx_cap = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  s->page_table = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * (size_t)max_pages);
  s->hot_block = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * (size_t)(B / P));
  s->slot_pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)L * R * B);
  s->slot_stamp = (int32_t*)malloc(sizeof(int32_t) * (size_t)L * R * B);
  s->where = (int32_t**)calloc((size_t)L * R, sizeof(int32_t*));
  s->seen = (int32_t**)calloc((size_t)L * R, sizeof(int32_t*));
  s->seen_j = (int32_t**)calloc((size_t)L * R, sizeof(int32_t*));
  s->serial = (int32_t*)calloc((size_t)L * R, sizeof(int32_t));
  s->cand = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
  if (!s->ctx || !s->ctx_cap || !s->page_table || !s->hot_block || !s->slot_pos ||
      !s->slot_stamp || !s->where || !s->seen || !s->seen_j || !s->serial || !s->cand) {
    or_destroy(s);
    return NULL;
  }
  memcpy(s->ctx_cap, ctx_cap, sizeof(int32_t) * (size_t)R);
  for (int64_t i = 0; i < (int64_t)R * max_pages; ++i) s->page_table[i] = -1;
  for (int64_t i = 0; i < (int64_t)R * (B / P); ++i) s->hot_block[i] = -1;
  for (int64_t i = 0; i < (int64_t)L * R * B; ++i) {
    s->slot_pos[i] = -1;   /* empty slot */
    s->slot_stamp[i] = -1; /* older than any step */
  }
  for (int32_t l = 0; l < L; ++l)
    for (int32_t r = 0; r < R; ++r) {
      int64_t u = unit_index(s, l, r);
      size_t n = (size_t)(ctx_cap[r] > 0 ? ctx_cap[r] : 1);
      s->where[u] = (int32_t*)malloc(sizeof(int32_t) * n);
      s->seen[u] = (int32_t*)calloc(n, sizeof(int32_t));
      s->seen_j[u] = (int32_t*)calloc(n, sizeof(int32_t));
      if (!s->where[u] || !s->seen[u] || !s->seen_j[u]) {
        or_destroy(s);
        return NULL;
      }
      for (size_t i = 0; i < n; ++i) s->where[u][i] = -1;
    }
  return s;
}

void or_destroy(or_state* s) {
  if (!s) return;
  if (s->where)
    for (int64_t u = 0; u < (int64_t)s->L * s->R; ++u) free(s->where[u]);
  if (s->seen)
    for (int64_t u = 0; u < (int64_t)s->L * s->R; ++u) free(s->seen[u]);
  if (s->seen_j)
    for (int64_t u = 0; u < (int64_t)s->L * s->R; ++u) free(s->seen_j[u]);
  free(s->where); free(s->seen); free(s->seen_j); free(s->serial);
  free(s->ctx); free(s->ctx_cap); free(s->page_table); free(s->hot_block);
  free(s->slot_pos); free(s->slot_stamp); free(s->cand);
  free(s);
}

int32_t or_set_ctx(or_state* s, int32_t req, int32_t ctx) {
  if (req < 0 || req >= s->R || ctx < 0 || ctx > s->ctx_cap[req]) return -1;
  s->ctx[req] = ctx;
  return 0;
}

int32_t or_set_page(or_state* s, int32_t req, int32_t page, int32_t block) {
  if (req < 0 || req >= s->R || page < 0 || page >= s->max_pages) return -1;
  s->page_table[(int64_t)req * s->max_pages + page] = block < 0 ? -1 : block;
  return 0;
}

int32_t or_set_hot_block(or_state* s, int32_t req, int32_t index, int32_t block) {
  if (req < 0 || req >= s->R || index < 0 || index >= s->B / s->P) return -1;
  s->hot_block[(int64_t)req * (s->B / s->P) + index] = block;
  return 0;
}

/* Pool row of hot slot `slot` of request `req`: hot blocks are ordinary blocks
 * of the same per-layer KV tensor. */
static int32_t hot_row(const or_state* s, int32_t req, int32_t slot) {
  int32_t blk = s->hot_block[(int64_t)req * (s->B / s->P) + slot / s->P];
  return blk * s->P + slot % s->P;
}

static int by_stamp_then_slot(const void* a, const void* b, void* ctx) {
  const int32_t* stamp = (const int32_t*)ctx;
  int32_t sa = *(const int32_t*)a, sb = *(const int32_t*)b;
  if (stamp[sa] != stamp[sb]) return stamp[sa] < stamp[sb] ? -1 : 1;
  return sa < sb ? -1 : (sa > sb ? 1 : 0);
}

/* Sort the candidate slots by (stamp, slot) ascending: a stable bottom-up
 * merge sort (insertion sort if no scratch can be had).  Written out rather
 * than qsort_r, whose signature differs between C libraries. */
static void sort_candidates(int32_t* cand, int32_t n, const int32_t* stamp) {
  int32_t* tmp = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  if (!tmp) { /* fall back to insertion sort */
    for (int32_t i = 1; i < n; ++i) {
      int32_t x = cand[i], j = i - 1;
      while (j >= 0 && by_stamp_then_slot(&cand[j], &x, (void*)stamp) > 0) {
        cand[j + 1] = cand[j];
        --j;
      }
      cand[j + 1] = x;
    }
    return;
  }
  for (int32_t width = 1; width < n; width *= 2) {
    for (int32_t lo = 0; lo < n; lo += 2 * width) {
      int32_t mid = lo + width < n ? lo + width : n;
      int32_t hi = lo + 2 * width < n ? lo + 2 * width : n;
      int32_t a = lo, b = mid, o = lo;
      while (a < mid && b < hi)
        tmp[o++] = by_stamp_then_slot(&cand[a], &cand[b], (void*)stamp) <= 0 ? cand[a++] : cand[b++];
      while (a < mid) tmp[o++] = cand[a++];
      while (b < hi) tmp[o++] = cand[b++];
    }
    memcpy(cand, tmp, sizeof(int32_t) * (size_t)n);
  }
  free(tmp);
}

int32_t or_resolve_tokens(or_state* s, int32_t layer, int32_t req, int32_t T,
                          const int32_t* topk, int32_t step, int32_t* out_row,
                          int32_t* miss_log, int32_t* n_miss) {
  if (layer < 0 || layer >= s->L || req < 0 || req >= s->R || T <= 0) return -1;
  const int64_t u = unit_index(s, layer, req);
  int32_t* pos_of = s->slot_pos + u * s->B;
  int32_t* stamp = s->slot_stamp + u * s->B;
  int32_t* where = s->where[u];
  int32_t* seen = s->seen[u];
  int32_t* seen_j = s->seen_j[u];
  const int32_t ctx = s->ctx[req];
  const int32_t call = ++s->serial[u];
  const int32_t n = T * s->K;  /* the list: token t's row is entries t*K .. t*K+K-1 */
  int32_t err = 0, misses = 0, n_alias = 0;
  int32_t* miss_j = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  int32_t* alias = (int32_t*)malloc(sizeof(int32_t) * 2 * (size_t)n);  /* (j, first j) */
  if (!miss_j || !alias) {
    free(miss_j);
    free(alias);
    return -1;
  }

  /* Phase 1: classify every entry; refresh hits. */
  for (int32_t j = 0; j < n; ++j) {
    const int32_t p = topk[j];
    out_row[j] = -1;
    if (p == -1) continue;                       /* padding */
    if (p < 0 || p >= ctx) { err |= OR_ERR_RANGE; continue; }
    if (seen[p] == call) {                       /* selected earlier in the list */
      if (seen_j[p] / s->K == j / s->K) { err |= OR_ERR_DUPLICATE; continue; }
      alias[2 * n_alias] = j;                    /* another token's: share its row */
      alias[2 * n_alias + 1] = seen_j[p];
      ++n_alias;
      continue;
    }
    seen[p] = call;
    seen_j[p] = j;
    const int32_t blk = s->page_table[(int64_t)req * s->max_pages + p / s->P];
    if (blk >= 0) {                               /* resident: read in place */
      if (blk >= s->blocks_per_layer) { err |= OR_ERR_BLOCK; continue; }
      out_row[j] = blk * s->P + p % s->P;
      continue;
    }
    const int32_t slot = where[p];
    if (slot >= 0) {                              /* hot hit: refresh LRU */
      stamp[slot] = step;
      out_row[j] = hot_row(s, req, slot);
      continue;
    }
    miss_j[misses++] = j;                         /* host only: a miss */
  }

  /* Phase 2: victims are slots not used in this step, least recent first. */
  int32_t ncand = 0;
  for (int32_t slot = 0; slot < s->B; ++slot)
    if (stamp[slot] < step) s->cand[ncand++] = slot;
  sort_candidates(s->cand, ncand, stamp);

  int32_t served = 0;
  for (int32_t i = 0; i < misses; ++i) {
    const int32_t j = miss_j[i], p = topk[j];
    if (i >= ncand) { err |= OR_ERR_CAPACITY; continue; }
    const int32_t slot = s->cand[i];
    if (pos_of[slot] >= 0) where[pos_of[slot]] = -1;   /* evict */
    pos_of[slot] = p;
    stamp[slot] = step;
    where[p] = slot;
    out_row[j] = hot_row(s, req, slot);   /* the row is copied from host here */
    if (miss_log) {
      miss_log[3 * served + 0] = j;
      miss_log[3 * served + 1] = p;
      miss_log[3 * served + 2] = slot;
    }
    ++served;
  }
  /* Phase 3: repeats in later tokens take their first occurrence's row. */
  for (int32_t i = 0; i < n_alias; ++i) out_row[alias[2 * i]] = out_row[alias[2 * i + 1]];
  free(miss_j);
  free(alias);
  if (n_miss) *n_miss = served;
  return err;
}

int32_t or_resolve(or_state* s, int32_t layer, int32_t req, const int32_t* topk,
                   int32_t step, int32_t* out_row, int32_t* miss_log,
                   int32_t* n_miss) {
  return or_resolve_tokens(s, layer, req, 1, topk, step, out_row, miss_log, n_miss);
}

int32_t or_get_unit(const or_state* s, int32_t layer, int32_t req,
                    int32_t* slot_pos, int32_t* slot_stamp) {
  if (layer < 0 || layer >= s->L || req < 0 || req >= s->R) return -1;
  const int64_t u = unit_index(s, layer, req);
  memcpy(slot_pos, s->slot_pos + u * s->B, sizeof(int32_t) * (size_t)s->B);
  memcpy(slot_stamp, s->slot_stamp + u * s->B, sizeof(int32_t) * (size_t)s->B);
  return 0;
}

int32_t or_row_content(const or_state* s, int32_t layer, int32_t req, int32_t row,
                       int32_t* pos) {
  /* Which logical position of `req` a pool row holds, or -1 if none. */
  *pos = -1;
  if (row < 0) return -1;
  const int32_t blk = row / s->P, off = row % s->P;
  for (int32_t page = 0; page < s->max_pages; ++page)
    if (s->page_table[(int64_t)req * s->max_pages + page] == blk) {
      *pos = page * s->P + off;
      return 0;
    }
  for (int32_t i = 0; i < s->B / s->P; ++i)
    if (s->hot_block[(int64_t)req * (s->B / s->P) + i] == blk) {
      const int64_t u = unit_index(s, layer, req);
      *pos = s->slot_pos[u * s->B + i * s->P + off];
      return 0;
    }
  return -1;
}
