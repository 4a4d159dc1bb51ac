/*
 * Seeded synthetic inputs (KV rows, queries, selection traces).
 * See synth.h for what each entry computes.  Input generation only.
 */
#include "synth.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define SY_GAMMA 0x9E3779B97F4A7C15ULL

enum {
  TAG_ROW = 0x524f57ULL,   /* "ROW" */
  TAG_Q = 0x51ULL,         /* "Q" */
  TAG_TRACE = 0x545243ULL, /* "TRC" */
  TAG_PERM = 0x5045524dULL /* "PERM" */
};

static inline uint64_t mix_(uint64_t x) {
  x += SY_GAMMA;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ULL;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBULL;
  return x ^ (x >> 31);
}
static inline uint64_t key_(uint64_t seed, uint64_t tag, uint64_t a,
                            uint64_t b, uint64_t c) {
  return mix_(mix_(mix_(mix_(seed ^ tag) + a) + b) + c);
}
static inline uint64_t draw_(uint64_t key, uint64_t i) { return mix_(key + i); }

static inline uint16_t normal_bf16_(uint64_t d) {
  /* Irwin-Hall n=4 over 16-bit uniforms: mean 2*65535, sd sqrt(4*(2^32-1)/12). */
  int32_t s = (int32_t)(d & 0xFFFF) + (int32_t)((d >> 16) & 0xFFFF) +
              (int32_t)((d >> 32) & 0xFFFF) + (int32_t)(d >> 48) - 131070;
  const float inv_sd = 0x1.bb67aep-16f; /* 1 / 37837.227 */
  float f = (float)s * inv_sd;          /* |s| < 2^24: the cast is exact */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even (no NaN possible) */
  return (uint16_t)(u >> 16);
}

uint64_t sy_mix(uint64_t x) { return mix_(x); }
uint64_t sy_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b,
                uint64_t c) {
  return key_(seed, tag, a, b, c);
}
uint64_t sy_draw(uint64_t key, uint64_t i) { return draw_(key, i); }
uint16_t sy_normal_bf16(uint64_t d) { return normal_bf16_(d); }

static inline uint64_t row_key(uint64_t seed, int32_t req, int32_t layer,
                               int64_t pos) {
  return key_(seed, TAG_ROW, (uint64_t)(uint32_t)req,
                (uint64_t)(uint32_t)layer, (uint64_t)pos);
}

static void fill_rows_serial(uint64_t seed, int32_t req, int32_t layer,
                             int64_t pos0, int64_t n, int32_t width,
                             uint16_t* dst) {
  for (int64_t i = 0; i < n; ++i) {
    uint64_t k = row_key(seed, req, layer, pos0 + i);
    uint16_t* o = dst + i * (int64_t)width;
    for (int32_t d = 0; d < width; ++d) o[d] = normal_bf16_(draw_(k, (uint64_t)d));
  }
}

typedef struct {
  uint64_t seed;
  int32_t req, layer, width;
  int64_t pos0, n;
  uint16_t* dst;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  fill_rows_serial(j->seed, j->req, j->layer, j->pos0, j->n, j->width, j->dst);
  return NULL;
}

void sy_fill_rows(uint64_t seed, int32_t req, int32_t layer, int64_t pos0,
                  int64_t n, int32_t width, uint16_t* dst, int32_t threads) {
  if (n <= 0) return;
  if (threads <= 1 || n < 4096) {
    fill_rows_serial(seed, req, layer, pos0, n, width, dst);
    return;
  }
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  fill_job jobs[256];
  int64_t per = (n + threads - 1) / threads;
  int32_t started = 0;
  for (int32_t t = 0; t < threads; ++t) {
    int64_t a = (int64_t)t * per, b = a + per;
    if (a >= n) break;
    if (b > n) b = n;
    jobs[t] = (fill_job){seed, req, layer, width, pos0 + a, b - a,
                         dst + a * (int64_t)width};
    if (pthread_create(&tid[t], NULL, fill_worker, &jobs[t]) != 0) {
      fill_worker(&jobs[t]);
      tid[t] = 0;
    }
    started = t + 1;
  }
  for (int32_t t = 0; t < started; ++t)
    if (tid[t]) pthread_join(tid[t], NULL);
}

void sy_fill_rows_at(uint64_t seed, int32_t req, int32_t layer,
                     const int32_t* pos, int64_t n, int32_t width,
                     uint16_t* dst) {
  for (int64_t i = 0; i < n; ++i) {
    uint16_t* o = dst + i * (int64_t)width;
    if (pos[i] < 0) {
      memset(o, 0, sizeof(uint16_t) * (size_t)width);
      continue;
    }
    uint64_t k = row_key(seed, req, layer, pos[i]);
    for (int32_t d = 0; d < width; ++d) o[d] = normal_bf16_(draw_(k, (uint64_t)d));
  }
}

void sy_fill_q(uint64_t seed, int32_t req, int32_t layer, int32_t step,
               int32_t heads, int32_t width, uint16_t* dst) {
  uint64_t k = key_(seed, TAG_Q, (uint64_t)(uint32_t)req,
                      (uint64_t)(uint32_t)layer, (uint64_t)(uint32_t)step);
  for (int32_t h = 0; h < heads; ++h)
    for (int32_t d = 0; d < width; ++d)
      dst[(int64_t)h * width + d] =
          normal_bf16_(draw_(k, ((uint64_t)h << 16) + (uint64_t)d));
}

/* ---------------------------------------------------------------- traces */

/* Uniform integer in [0, n) from one draw (multiply-high). */
static inline int64_t uniform_below(uint64_t d, int64_t n) {
  return (int64_t)(((unsigned __int128)d * (uint64_t)n) >> 64);
}

/* Balanced Feistel permutation of [0, 2^bits) (bits even), 4 rounds, used with
 * cycle walking to permute [0, n). */
int64_t sy_permute(uint64_t seed, int32_t req, int64_t rank, int64_t n) {
  int bits = 2;
  while (((int64_t)1 << bits) < n) bits += 2;
  const int half = bits / 2;
  const uint64_t mask = ((uint64_t)1 << half) - 1;
  uint64_t key = key_(seed, TAG_PERM, (uint64_t)(uint32_t)req, 0, 0);
  uint64_t x = (uint64_t)rank;
  do {
    uint64_t l = x >> half, r = x & mask;
    for (int round = 0; round < 4; ++round) {
      uint64_t f = draw_(key, ((uint64_t)round << 40) ^ r) & mask;
      uint64_t nl = r, nr = l ^ f;
      l = nl;
      r = nr;
    }
    x = (l << half) | r;
  } while ((int64_t)x >= n);
  return (int64_t)x;
}

/* Bounded Zipf(s) rank in [0, n) by the continuous inverse CDF of
 * p(x) ~ x^-s on [1, n+1). */
static int64_t zipf_rank(uint64_t d, int64_t n, double s) {
  double u = (double)(d >> 11) * 0x1.0p-53; /* [0, 1) */
  double one_m_s = 1.0 - s;
  double top = pow((double)n + 1.0, one_m_s);
  double x = pow((top - 1.0) * u + 1.0, 1.0 / one_m_s);
  int64_t k = (int64_t)floor(x) - 1;
  if (k < 0) k = 0;
  if (k >= n) k = n - 1;
  return k;
}

/* Small open-addressing set of non-negative positions. */
typedef struct {
  int32_t* key;
  int32_t* used; /* list of occupied buckets, to clear in O(size) */
  int32_t nused, mask;
} pos_set;

static int pos_set_init(pos_set* s, int32_t capacity) {
  int32_t cap = 16;
  while (cap < 4 * capacity) cap <<= 1;
  s->key = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  s->used = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  if (!s->key || !s->used) return -1;
  for (int32_t i = 0; i < cap; ++i) s->key[i] = -1;
  s->nused = 0;
  s->mask = cap - 1;
  return 0;
}
static void pos_set_free(pos_set* s) {
  free(s->key);
  free(s->used);
}
static void pos_set_clear(pos_set* s) {
  for (int32_t i = 0; i < s->nused; ++i) s->key[s->used[i]] = -1;
  s->nused = 0;
}
/* Returns 1 if inserted, 0 if already present. */
static int pos_set_insert(pos_set* s, int32_t p) {
  uint32_t h = ((uint32_t)p * 2654435761u) & (uint32_t)s->mask;
  for (;;) {
    if (s->key[h] == p) return 0;
    if (s->key[h] < 0) {
      s->key[h] = p;
      s->used[s->nused++] = (int32_t)h;
      return 1;
    }
    h = (h + 1) & (uint32_t)s->mask;
  }
}

/* Append up to `want` members of src (size n) chosen uniformly without
 * replacement (partial Fisher-Yates on a scratch copy), skipping members
 * already in the set.  Returns the number appended. */
static int32_t take_subset(const int32_t* src, int32_t n, int32_t want,
                           uint64_t key, uint64_t* ctr, int32_t* scratch,
                           pos_set* set, int32_t* dst) {
  memcpy(scratch, src, sizeof(int32_t) * (size_t)n);
  int32_t got = 0;
  for (int32_t i = 0; i < n && got < want; ++i) {
    int32_t j = i + (int32_t)uniform_below(draw_(key, (*ctr)++), n - i);
    int32_t t = scratch[i];
    scratch[i] = scratch[j];
    scratch[j] = t;
    if (pos_set_insert(set, scratch[i])) dst[got++] = scratch[i];
  }
  return got;
}

int32_t sy_trace_request(const sy_trace_params* prm, int32_t req,
                         const int32_t* ctx_per_step, int32_t* out) {
  const int32_t K = prm->k, L = prm->layers, T = prm->steps;
  for (int32_t t = 0; t < T; ++t)
    if (ctx_per_step[t] < K) return -1;
  pos_set set;
  if (pos_set_init(&set, K) != 0) return -2;
  int32_t* scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  int32_t* cur = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  if (!scratch || !cur) {
    pos_set_free(&set);
    free(scratch);
    free(cur);
    return -2;
  }
  const double uni_share = 1.0 - prm->reuse - prm->zipf_frac;
  for (int32_t t = 0; t < T; ++t) {
    const int64_t ctx = ctx_per_step[t];
    for (int32_t l = 0; l < L; ++l) {
      uint64_t key = key_(prm->seed, TAG_TRACE, (uint64_t)(uint32_t)req,
                            (uint64_t)(uint32_t)l, (uint64_t)(uint32_t)t);
      uint64_t ctr = 0;
      int32_t n = 0;
      pos_set_clear(&set);
      int32_t remain = K;
      /* 1. share with the layer below at this step */
      if (l > 0 && prm->layer_share > 0.0) {
        const int32_t* below = out + ((int64_t)t * L + (l - 1)) * K;
        int32_t want = (int32_t)floor(prm->layer_share * K);
        n += take_subset(below, K, want, key, &ctr, scratch, &set, cur + n);
        remain = K - n;
      }
      /* 2. split the remainder over reuse / Zipf / uniform */
      int32_t n_reuse, n_zipf;
      if (t > 0) {
        n_reuse = (int32_t)floor(prm->reuse * remain);
        n_zipf = (int32_t)floor(prm->zipf_frac * remain);
      } else {
        n_reuse = 0;
        double nz = prm->zipf_frac + uni_share;
        n_zipf = nz > 0.0 ? (int32_t)floor(prm->zipf_frac / nz * remain) : 0;
      }
      if (n_reuse > 0) {
        const int32_t* prev = out + ((int64_t)(t - 1) * L + l) * K;
        n += take_subset(prev, K, n_reuse, key, &ctr, scratch, &set, cur + n);
      }
      int32_t zipf_target = n + n_zipf;
      if (zipf_target > K) zipf_target = K;
      int32_t tries = 0;
      while (n < zipf_target && tries < 64 * K) {
        ++tries;
        int64_t rank = zipf_rank(draw_(key, ctr++), ctx, prm->zipf_s);
        int32_t p = (int32_t)sy_permute(prm->seed, req, rank, ctx);
        if (pos_set_insert(&set, p)) cur[n++] = p;
      }
      while (n < K) {
        int32_t p = (int32_t)uniform_below(draw_(key, ctr++), ctx);
        if (pos_set_insert(&set, p)) cur[n++] = p;
      }
      /* 3. shuffle the emission order */
      int32_t* row = out + ((int64_t)t * L + l) * K;
      for (int32_t i = K - 1; i > 0; --i) {
        int32_t j = (int32_t)uniform_below(draw_(key, ctr++), i + 1);
        int32_t tmp = cur[i];
        cur[i] = cur[j];
        cur[j] = tmp;
      }
      memcpy(row, cur, sizeof(int32_t) * (size_t)K);
    }
  }
  pos_set_free(&set);
  free(scratch);
  free(cur);
  return 0;
}

/* ---- FP8 rows (see synth.h) ------------------------------------------- */

uint8_t sy_e4m3_encode(float v) {
  const uint8_t sign = (v < 0.0f || (v == 0.0f && signbit(v))) ? 0x80u : 0u;
  double a = fabs((double)v);
  if (!(a < 448.0)) return (uint8_t)(sign | 0x7Eu); /* saturate (also NaN input) */
  if (a < 0x1p-6) {                                  /* subnormal range: m * 2^-9 */
    const double m = nearbyint(a * 512.0);          /* ties to even (default mode) */
    if (m >= 8.0) return (uint8_t)(sign | 0x08u);   /* rounds up to 2^-6 */
    return (uint8_t)(sign | (uint8_t)m);
  }
  int x;
  const double f = frexp(a, &x);            /* a = f * 2^x, f in [0.5, 1) */
  int e = x - 1;                            /* a = (2f) * 2^e, 2f in [1, 2) */
  double q = nearbyint(2.0 * f * 8.0);      /* significand in eighths: 8 .. 16 */
  if (q >= 16.0) {
    q = 8.0;
    ++e;
  }
  const int field = e + 7;
  const int m = (int)q - 8;
  if (field > 15 || (field == 15 && m == 7)) return (uint8_t)(sign | 0x7Eu);
  return (uint8_t)(sign | (uint8_t)(field << 3) | (uint8_t)m);
}

static float bf16_to_float_(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static void quantize_row_fp8(const uint16_t* src, uint8_t* dst) {
  for (int g = 0; g < 4; ++g) {
    float mx = 0.0f;
    for (int i = 0; i < 128; ++i) {
      const float a = fabsf(bf16_to_float_(src[128 * g + i]));
      if (a > mx) mx = a;
    }
    const float scale = mx > 0.0f ? mx / 448.0f : 1.0f;
    memcpy(dst + 512 + 4 * g, &scale, 4);
    for (int i = 0; i < 128; ++i) {
      const float y = bf16_to_float_(src[128 * g + i]) / scale;
      dst[128 * g + i] = sy_e4m3_encode(y);
    }
  }
  memcpy(dst + 528, src + 512, 64 * sizeof(uint16_t)); /* rope stays bf16 */
}

static void fill_rows_fp8_serial(uint64_t seed, int32_t req, int32_t layer, int64_t pos0,
                                 int64_t n, uint8_t* dst) {
  uint16_t row[576];
  for (int64_t i = 0; i < n; ++i) {
    fill_rows_serial(seed, req, layer, pos0 + i, 1, 576, row);
    quantize_row_fp8(row, dst + i * SY_FP8_ROW_BYTES);
  }
}

typedef struct {
  uint64_t seed;
  int32_t req, layer;
  int64_t pos0, n;
  uint8_t* dst;
} fill_fp8_job;

static void* fill_fp8_worker(void* arg) {
  fill_fp8_job* j = (fill_fp8_job*)arg;
  fill_rows_fp8_serial(j->seed, j->req, j->layer, j->pos0, j->n, j->dst);
  return NULL;
}

void sy_fill_rows_fp8(uint64_t seed, int32_t req, int32_t layer, int64_t pos0,
                      int64_t n, uint8_t* dst, int32_t threads) {
  if (n <= 0) return;
  if (threads <= 1 || n < 4096) {
    fill_rows_fp8_serial(seed, req, layer, pos0, n, dst);
    return;
  }
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  fill_fp8_job jobs[256];
  int64_t per = (n + threads - 1) / threads;
  int32_t started = 0;
  for (int32_t t = 0; t < threads; ++t) {
    int64_t a = (int64_t)t * per, b = a + per;
    if (a >= n) break;
    if (b > n) b = n;
    jobs[t] = (fill_fp8_job){seed, req, layer, pos0 + a, b - a, dst + a * SY_FP8_ROW_BYTES};
    if (pthread_create(&tid[t], NULL, fill_fp8_worker, &jobs[t]) != 0) {
      fill_fp8_worker(&jobs[t]);
      tid[t] = 0;
    }
    started = t + 1;
  }
  for (int32_t t = 0; t < started; ++t)
    if (tid[t]) pthread_join(tid[t], NULL);
}

void sy_fill_rows_fp8_at(uint64_t seed, int32_t req, int32_t layer,
                         const int32_t* pos, int64_t n, uint8_t* dst) {
  for (int64_t i = 0; i < n; ++i) {
    uint8_t* o = dst + i * SY_FP8_ROW_BYTES;
    if (pos[i] < 0) {
      memset(o, 0, SY_FP8_ROW_BYTES);
      continue;
    }
    fill_rows_fp8_serial(seed, req, layer, pos[i], 1, o);
  }
}
