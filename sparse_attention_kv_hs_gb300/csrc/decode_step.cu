// One decode step over several sparse layers, with the next layer's misses
// fetched while the current layer's attention runs ("precise prefetch").
//
// Page "59188saintaubert.com ... HiSparse", section 04: a synchronous resolve
// exposes 7-8 ms of host IO per token, prefetching brings that to about 3 ms,
// and what makes prefetching work is exact selection information from the
// model rather than a guess; section 03 reports prefetch alone adding 14-17%
// throughput.  Page "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading
// in vLLM", section "Exploiting sparsity when needed": with IndexShare one
// indexer layer serves four sparse-MLA layers, so the selections of the next
// layers are known before the current layer's attention runs.
//
// Schedule for layers 0 .. n-1 (all selections given):
//   stream:       RESOLVE(0)  ATTN(0)  [wait R(1)] ATTN(1)  [wait R(2)] ATTN(2) ...
//   copy_stream:  [wait S] RESOLVE(1)  RESOLVE(2)  ...
// RESOLVE launches of different layers touch disjoint state (their own
// slots, position -> slot array and pool rows), so only the data each
// attention needs orders the two streams.  The attention launches run on the
// SMs that RESOLVE does not need: a RESOLVE beside another launch takes
// clusters of 2 CTAs per unit and an attention launch beside a RESOLVE the
// SMs left.  Where the copy stream starts (S):
//  - bf16 rows (1152 B): with the step.  A RESOLVE launch, bound by the host
//    link, takes about twice an attention launch; RESOLVE(1) beside RESOLVE(0)
//    (on the SMs RESOLVE(0) leaves, then on those its clusters free) keeps the
//    link busy across both launches' start and tail.
//  - FP8 rows (656 B): after RESOLVE(0).  RESOLVE and attention launches take
//    about as long as each other, and RESOLVE(1) is best hidden beside ATTN(0).
#include "hs_internal.cuh"

// num_tokens verify tokens per request (speculative decoding; 1 otherwise):
// each layer's RESOLVE takes a unit's T lists as one (hs_resolve_tokens) and
// its attention runs one decode row per (request, token).
extern "C" hs_status hs_decode_step_tokens(hs_pool* p, int32_t layer_begin, int32_t num_layers,
                                           int32_t num_tokens, const int32_t* topk_idx,
                                           const void* q, int32_t num_heads, int32_t v_dim,
                                           float scale, const int32_t* d_step,
                                           int32_t* out_row_ids, void* out, float* lse,
                                           int32_t* miss_count, void* stream, void* copy_stream) {
  if (!p || !topk_idx || !q || !d_step || !out_row_ids || !out || num_tokens <= 0)
    return HS_ERR_INVALID;
  if (num_layers <= 0 || layer_begin < 0 || layer_begin + num_layers > p->d.num_layers)
    return HS_ERR_INVALID;
  // the attention launches' own checks, made before anything is queued
  if (num_heads <= 0 || num_heads > 128 || v_dim != 512 || p->d.row_elems != 576 ||
      !(scale > 0.f) || p->attn_max_splits < 1 || !p->attn_kv_maps)
    return HS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return HS_ERR_INVALID;
  const int64_t R = p->d.num_requests, K = p->d.top_k, H = num_heads, T = num_tokens;
  const int64_t D = p->d.row_elems;
  if (R * T > 65535) return HS_ERR_INVALID;
  auto topk_l = [&](int i) { return topk_idx + i * R * T * K; };
  auto rows_l = [&](int i) { return out_row_ids + i * R * T * K; };
  auto cnt_l = [&](int i) { return miss_count ? miss_count + i * R : nullptr; };
  auto q_l = [&](int i) { return static_cast<const char*>(q) + i * R * T * H * D * 2; };
  auto out_l = [&](int i) { return static_cast<char*>(out) + i * R * T * H * v_dim * 2; };
  auto lse_l = [&](int i) { return lse ? lse + i * R * T * H : nullptr; };
  auto resolve = [&](int i, int max_cluster, cudaStream_t st) {
    return hs_launch_resolve_tokens(p, layer_begin + i, 1, num_tokens, topk_l(i), d_step,
                                    rows_l(i), cnt_l(i), nullptr, max_cluster, st);
  };
  auto attention = [&](int i, int max_splits, cudaStream_t st) {
    return hs_launch_attention_tokens(p, layer_begin + i, num_tokens, q_l(i), rows_l(i), num_heads,
                                      v_dim, scale, out_l(i), lse_l(i), max_splits, st);
  };
  cudaStream_t s = hs_stream(stream), cs = hs_stream(copy_stream);

  hs_status st;
  if (cs == s || num_layers == 1) {  // one stream: the plain sequence
    for (int i = 0; i < num_layers; ++i) {
      if ((st = resolve(i, 0, s)) != HS_OK) return st;
      if ((st = attention(i, 0, s)) != HS_OK) return st;
    }
    return HS_OK;
  }

  // SMs while a RESOLVE runs beside an attention launch: RESOLVE clusters of
  // 2 CTAs per unit (1 if that leaves too few), attention the splits that fit
  // in the rest (at least one CTA pair per decode row)
  const int64_t sms = p->num_sms;
  const int c_side = 3 * R <= sms ? 2 : 1;
  int s_side = (int)((sms - c_side * R) / (2 * R * T));
  if (s_side < 1) s_side = 1;

  cudaEvent_t* ev = p->step_events;
  const bool together = p->d.kv_format == HS_KV_BF16;  // see the schedule above
  if (together) {  // copy_stream starts after the work queued before this step
    HS_CUDA_TRY(cudaEventRecord(ev[0], s));
    HS_CUDA_TRY(cudaStreamWaitEvent(cs, ev[0], 0));
  }
  if ((st = resolve(0, 0, s)) != HS_OK) return st;
  if (!together) {  // copy_stream starts after RESOLVE(0)
    HS_CUDA_TRY(cudaEventRecord(ev[0], s));
    HS_CUDA_TRY(cudaStreamWaitEvent(cs, ev[0], 0));
  }
  for (int i = 1; i < num_layers; ++i) {
    if ((st = resolve(i, c_side, cs)) != HS_OK) return st;
    HS_CUDA_TRY(cudaEventRecord(ev[i], cs));
  }
  for (int i = 0; i < num_layers; ++i) {
    if (i > 0) HS_CUDA_TRY(cudaStreamWaitEvent(s, ev[i], 0));
    if ((st = attention(i, i + 1 < num_layers ? s_side : 0, s)) != HS_OK) return st;
  }
  return HS_OK;
}

extern "C" hs_status hs_decode_step(hs_pool* p, int32_t layer_begin, int32_t num_layers,
                                    const int32_t* topk_idx, const void* q, int32_t num_heads,
                                    int32_t v_dim, float scale, const int32_t* d_step,
                                    int32_t* out_row_ids, void* out, float* lse,
                                    int32_t* miss_count, void* stream, void* copy_stream) {
  return hs_decode_step_tokens(p, layer_begin, num_layers, 1, topk_idx, q, num_heads, v_dim, scale,
                               d_step, out_row_ids, out, lse, miss_count, stream, copy_stream);
}
