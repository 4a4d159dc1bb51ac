// Sparse MLA decode attention (work in progress: entry point only).
#include "hs_internal.cuh"

hs_status hs_attn_workspace_init(hs_pool* p) {
  p->attn_o = nullptr;
  p->attn_ml = nullptr;
  p->attn_max_splits = 0;
  return HS_OK;
}

extern "C" hs_status hs_sparse_mla_decode(hs_pool* pool, int32_t layer, const void* q,
                                          const int32_t* row_ids, int32_t num_heads, int32_t v_dim,
                                          float scale, void* out, float* lse, void* stream) {
  (void)pool; (void)layer; (void)q; (void)row_ids; (void)num_heads; (void)v_dim; (void)scale;
  (void)out; (void)lse; (void)stream;
  return HS_ERR_INVALID;
}
