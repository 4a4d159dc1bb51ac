/*
 * Seeded synthetic inputs for the HiSparse decode path: KV rows, decode
 * queries and top-K selection traces.
 *
 * This module is shared input generation only.  It holds none of the
 * method's arithmetic (no page table, no LRU, no attention): it produces the
 * data a sparse indexer and a model would hand to the decode path, so that the
 * CUDA path and the CPU oracle can be fed the same bytes.
 *
 * Every value is a pure function of (seed, coordinates), built on the
 * splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used as a counter-based generator.  All
 * arithmetic is integer except one fp32 multiply per value, so the bytes are
 * identical on every IEEE machine.
 */
#ifndef HS_SYNTH_H
#define HS_SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* splitmix64 finaliser of (x + golden gamma). */
uint64_t sy_mix(uint64_t x);

/* Key chain: mix(mix(mix(mix(seed ^ tag) + a) + b) + c). */
uint64_t sy_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b, uint64_t c);

/* The i-th draw of the stream named by key: mix(key + i). */
uint64_t sy_draw(uint64_t key, uint64_t i);

/* One approximately standard-normal bf16 value from one 64-bit draw: the
 * standardised sum of four independent uniform 16-bit integers (Irwin-Hall,
 * n = 4), scaled in fp32 and rounded to bf16 (round to nearest even).
 * Returned as raw bf16 bits. */
uint16_t sy_normal_bf16(uint64_t draw);

/* KV rows of (seed, req, layer): rows for positions pos0 .. pos0+n-1, each of
 * `width` bf16 values, written contiguously to dst (n * width values).
 * `threads` <= 1 runs on the calling thread. */
void sy_fill_rows(uint64_t seed, int32_t req, int32_t layer, int64_t pos0,
                  int64_t n, int32_t width, uint16_t* dst, int32_t threads);

/* Same rows, for an explicit list of positions (pos[i] < 0 gives a zero row). */
void sy_fill_rows_at(uint64_t seed, int32_t req, int32_t layer,
                     const int32_t* pos, int64_t n, int32_t width,
                     uint16_t* dst);

/* The same rows (576 wide) stored as FP8 rows of 656 bytes: bytes 0..511 the
 * 512 latent values as OCP E4M3 codes (bias 7, largest 448, no infinities),
 * bytes 512..527 four fp32 scales (scale g multiplies latent values
 * 128g .. 128g+127), bytes 528..655 the 64 rope values as bf16.  A group's
 * scale is its largest magnitude / 448 (1 for an all-zero group); each latent
 * value is divided by its scale in fp32 and rounded to the nearest E4M3 value
 * (ties to even, magnitudes above 448 saturate to 448). */
#define SY_FP8_ROW_BYTES 656
void sy_fill_rows_fp8(uint64_t seed, int32_t req, int32_t layer, int64_t pos0,
                      int64_t n, uint8_t* dst, int32_t threads);
void sy_fill_rows_fp8_at(uint64_t seed, int32_t req, int32_t layer,
                         const int32_t* pos, int64_t n, uint8_t* dst);
/* One fp32 value -> its E4M3 code as above (round to nearest, ties to even,
 * saturating at 448). */
uint8_t sy_e4m3_encode(float v);

/* Decode query of (seed, req, layer, step): heads x width bf16 values. */
void sy_fill_q(uint64_t seed, int32_t req, int32_t layer, int32_t step,
               int32_t heads, int32_t width, uint16_t* dst);

/* Selection-drift model of one request over all layers and steps.
 *   reuse        share of layer 0's set kept from its previous step
 *   zipf_frac    share drawn from a bounded Zipf(zipf_s) over a seeded
 *                permutation of the context (rank -> position)
 *   rest         uniform over the context
 *   layer_share  share of layer l > 0's set taken from layer l-1 at the same
 *                step; the remainder is drawn by the mixture above
 * Sets never hold a duplicate.  Each row is shuffled before it is written.
 * ctx_per_step[t] is the context length at step t (non-decreasing).
 * out is [steps][layers][k].  Returns 0, or -1 if k > ctx at some step. */
typedef struct {
  uint64_t seed;
  int32_t k;
  int32_t layers;
  int32_t steps;
  double reuse;
  double zipf_frac;
  double zipf_s;
  double layer_share;
} sy_trace_params;

int32_t sy_trace_request(const sy_trace_params* prm, int32_t req,
                         const int32_t* ctx_per_step, int32_t* out);

/* Position of Zipf rank `rank` in request req's permutation of [0, n). */
int64_t sy_permute(uint64_t seed, int32_t req, int64_t rank, int64_t n);

#ifdef __cplusplus
}
#endif
#endif
