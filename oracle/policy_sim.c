/*
 * Replacement-policy study for the RESOLVE hot buffer -- test infrastructure
 * only (not part of the product path; it shares no code with the CUDA library).
 *
 * Page "59188saintaubert.com ... HiSparse", section 04, compares replacement
 * policies for the hot buffer on selection traces: LRU against FIFO, random
 * and the offline optimum (Belady).  This file simulates one hot buffer of B
 * slots over a trace of top-K selections with the same step structure as
 * RESOLVE (resolve_oracle.c): hits first, so every slot the current selection
 * uses is pinned for the step, then each miss, in selection order, takes the
 * next victim among the slots not used in this step.  Empty slots are always
 * filled first, lowest slot first.  The policies differ only in which of the
 * remaining (occupied) slots go first:
 *   LRU     oldest last use first, ties to the lowest slot (RESOLVE's rule);
 *   FIFO    oldest load first, ties to the lowest slot (a hit does not renew);
 *   random  uniformly random order, from a seeded splitmix64 stream per step;
 *   Belady  the position used again furthest in the future first (never used
 *           again counts as furthest), ties to the lowest slot.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { PS_LRU = 0, PS_FIFO = 1, PS_RANDOM = 2, PS_BELADY = 3 };

typedef struct {
  int64_t key;  /* sort key: smaller goes first */
  int32_t slot;
} cand_t;

static int cand_cmp(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return x->slot < y->slot ? -1 : (x->slot > y->slot);
}

static uint64_t splitmix64(uint64_t* state) {
  uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* First step after t at which position p is selected again, or `steps` if
 * never: positions' selection steps are kept as sorted lists (CSR). */
static int32_t next_use(const int32_t* start, const int32_t* uses, int32_t p, int32_t t,
                        int32_t steps) {
  int32_t lo = start[p], hi = start[p + 1];
  while (lo < hi) {  /* first entry > t */
    const int32_t mid = lo + (hi - lo) / 2;
    if (uses[mid] <= t) lo = mid + 1; else hi = mid;
  }
  return lo < start[p + 1] ? uses[lo] : steps;
}

/* Simulate one hot buffer.  trace: [steps][K] positions in [0, ctx) or -1
 * (not selected / resident; skipped).  A position repeated within one row is
 * counted once.  misses: [steps] out.  Returns 0, or -1 for bad arguments or
 * memory. */
int32_t ps_simulate(int32_t policy, int32_t K, int32_t B, int32_t steps, int32_t ctx,
                    const int32_t* trace, uint64_t seed, int32_t* misses) {
  if (policy < PS_LRU || policy > PS_BELADY || K <= 0 || B <= 0 || steps < 0 || ctx <= 0)
    return -1;
  int32_t* where = (int32_t*)malloc(sizeof(int32_t) * (size_t)ctx);   /* position -> slot */
  int32_t* slot_pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
  int32_t* last_use = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
  int32_t* loaded = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
  int32_t* miss_p = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)B);
  int32_t* start = (int32_t*)calloc((size_t)ctx + 1, sizeof(int32_t));
  int32_t* uses = (int32_t*)malloc(sizeof(int32_t) * ((size_t)steps * K + 1));
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * ((size_t)ctx + 1));
  int32_t rc = -1;
  if (!where || !slot_pos || !last_use || !loaded || !miss_p || !cand || !start || !uses ||
      !fill)
    goto done;
  for (int32_t p = 0; p < ctx; ++p) where[p] = -1;
  for (int32_t s = 0; s < B; ++s) {
    slot_pos[s] = -1;
    last_use[s] = -1;
    loaded[s] = -1;
  }
  /* CSR of each position's selection steps (ascending) */
  for (int64_t i = 0; i < (int64_t)steps * K; ++i)
    if (trace[i] >= 0 && trace[i] < ctx) start[trace[i] + 1]++;
  for (int32_t p = 0; p < ctx; ++p) start[p + 1] += start[p];
  memcpy(fill, start, sizeof(int32_t) * (size_t)ctx);
  for (int32_t t = 0; t < steps; ++t)
    for (int32_t j = 0; j < K; ++j) {
      const int32_t p = trace[(int64_t)t * K + j];
      if (p >= 0 && p < ctx) uses[fill[p]++] = t;
    }

  for (int32_t t = 0; t < steps; ++t) {
    const int32_t* row = trace + (int64_t)t * K;
    int32_t n_miss = 0;
    /* phase 1: hits are pinned for this step; collect misses in j order */
    for (int32_t j = 0; j < K; ++j) {
      const int32_t p = row[j];
      if (p < 0 || p >= ctx) continue;
      const int32_t s = where[p];
      if (s >= 0) {
        last_use[s] = t;
        continue;
      }
      int dup = 0;
      for (int32_t i = 0; i < n_miss; ++i)
        if (miss_p[i] == p) { dup = 1; break; }
      if (!dup) miss_p[n_miss++] = p;
    }
    /* phase 2: victims among the slots not used in this step */
    int32_t nc = 0;
    uint64_t rs = seed ^ (0xD1B54A32D192ED03ull * (uint64_t)(t + 1));
    for (int32_t s = 0; s < B; ++s) {
      if (last_use[s] == t) continue;
      int64_t key;
      if (slot_pos[s] < 0) {
        key = INT64_MIN;  /* empty slots first, lowest slot first */
      } else if (policy == PS_LRU) {
        key = last_use[s];
      } else if (policy == PS_FIFO) {
        key = loaded[s];
      } else if (policy == PS_RANDOM) {
        key = (int64_t)(splitmix64(&rs) >> 1);
      } else {
        key = -(int64_t)next_use(start, uses, slot_pos[s], t, steps);
      }
      cand[nc].key = key;
      cand[nc].slot = s;
      ++nc;
    }
    qsort(cand, (size_t)nc, sizeof(cand_t), cand_cmp);
    const int32_t served = n_miss < nc ? n_miss : nc;
    for (int32_t i = 0; i < served; ++i) {
      const int32_t s = cand[i].slot;
      if (slot_pos[s] >= 0) where[slot_pos[s]] = -1;
      slot_pos[s] = miss_p[i];
      where[miss_p[i]] = s;
      last_use[s] = t;
      loaded[s] = t;
    }
    misses[t] = n_miss;
  }
  rc = 0;
done:
  free(where);
  free(slot_pos);
  free(last_use);
  free(loaded);
  free(miss_p);
  free(cand);
  free(start);
  free(uses);
  free(fill);
  return rc;
}
