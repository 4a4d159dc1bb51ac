// Internal definitions shared by the libhs translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hs.h"

struct hs_pool {
  hs_pool_desc d;
  int device;
  int num_sms;
  int64_t blocks_per_layer;
  int64_t hot_blocks;  // R * B / P, per layer

  void* kv_pool;  // device bf16 [L][blocks_per_layer][P][row_elems]
  size_t kv_bytes;
  void* host_pool;      // pinned host
  void* host_pool_dev;  // device alias
  size_t host_bytes;
  size_t host_map_len;  // > 0: host_pool is an mmap'd, NUMA-placed, registered region
  int host_numa_node;   // NUMA node the host pool was placed on, or -1

  int32_t* page_table;  // [R][max_pages]
  int32_t* ctx_len;     // [R]
  int64_t* host_off;    // [R]
  int32_t* hot_block;   // [R][B/P]
  int32_t* slot_pos;    // [L][R][B]
  int32_t* slot_stamp;  // [L][R][B]
  int32_t* lru_order;   // [L][R][B]
  int32_t* inv;         // [L][host_tokens]: hot slot holding each host row, or -1
  int32_t* step;        // scalar
  int32_t* error_word;  // scalar
  int32_t* resolve_counts;  // [L][R]: running miss counts of a list resolved in token groups

  // sparse MLA decode workspace (split-K partials)
  uint16_t* attn_o;  // [R][max_splits][128][512] fp16 partials
  float* attn_ml;    // [R][max_splits][128] lse
  int attn_max_splits;
  void* attn_kv_maps;  // host array of one TMA tensor map per layer (CUtensorMap)

  size_t resolve_smem;          // RESOLVE's dynamic shared memory per CTA
  int resolve_max_clusters[4];  // clusters of 1, 2, 4, 8 CTAs that run at once

  cudaEvent_t order_event;  // orders offload copies after main-stream work
  cudaEvent_t* step_events; // [L + 1] hand-offs between hs_decode_step's two streams
  int64_t* host_off_mirror; // host copy of host_off (set-up calls only)
};

#define HS_CUDA_TRY(expr)                       \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    if (e_ != cudaSuccess) return HS_ERR_CUDA;  \
  } while (0)

static inline cudaStream_t hs_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Bytes of one KV row in the pool's format (a multiple of 16).
static inline int64_t hs_row_bytes(const hs_pool_desc& d) {
  return d.kv_format == HS_KV_FP8 ? 656 : (int64_t)d.row_elems * 2;
}

// Launch wrappers implemented per translation unit.
// max_cluster > 0 caps RESOLVE's CTAs per unit (to leave SMs to a kernel that
// runs beside it); 0 = as many as fit.
hs_status hs_launch_resolve(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                            const int32_t* topk, const int32_t* d_step, int32_t* out_rows,
                            int32_t* miss_count, int32_t* miss_log, int max_cluster,
                            cudaStream_t stream);
// RESOLVE of num_tokens verify tokens per unit, taken as one list (as
// hs_resolve_tokens).
hs_status hs_launch_resolve_tokens(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                                   int32_t num_tokens, const int32_t* topk, const int32_t* d_step,
                                   int32_t* out_rows, int32_t* miss_count, int32_t* miss_log,
                                   int max_cluster, cudaStream_t stream);
// Sparse MLA decode of one layer (arguments as hs_sparse_mla_decode);
// max_splits > 0 caps the K splits per request (fewer SMs), 0 = the pool's.
hs_status hs_launch_attention(hs_pool* pool, int32_t layer, const void* q,
                              const int32_t* row_ids, int32_t num_heads, int32_t v_dim,
                              float scale, void* out, float* lse, int max_splits,
                              cudaStream_t stream);
// The same over the num_tokens verify tokens of each request (q, row_ids, out
// and lse laid out as for hs_sparse_mla_decode_tokens).
hs_status hs_launch_attention_tokens(hs_pool* pool, int32_t layer, int32_t num_tokens,
                                     const void* q, const int32_t* row_ids, int32_t num_heads,
                                     int32_t v_dim, float scale, void* out, float* lse,
                                     int max_splits, cudaStream_t stream);
// One-thread kernel: RESOLVE's bounded wait on a barrier nothing arrives on.
hs_status hs_launch_peer_wait_selftest(int32_t* gave_up, uint64_t timeout_ns,
                                       cudaStream_t stream);
hs_status hs_attn_workspace_init(hs_pool* pool);
void hs_attn_workspace_free(hs_pool* pool);
// Shared memory the RESOLVE kernel needs for these sizes; sets the kernel's
// dynamic shared-memory limit (call once per pool, outside stream capture).
// Also reports how many RESOLVE clusters of 1, 2, 4 and 8 CTAs fit at once.
hs_status hs_resolve_configure(int K, int B, int P, int max_pages, size_t* smem_bytes,
                               int max_clusters[4]);
