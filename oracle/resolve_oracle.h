/*
 * CPU ORACLE for HiSparse RESOLVE -- test infrastructure only (see
 * resolve_oracle.c for what it follows).  Not part of the product path.
 */
#ifndef HS_RESOLVE_ORACLE_H
#define HS_RESOLVE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error bits returned by or_resolve (same meaning as the library's device
 * error word, restated here independently). */
#define OR_ERR_RANGE 1     /* position outside [0, ctx) and not -1 */
#define OR_ERR_DUPLICATE 2 /* position repeated within one top-K row */
#define OR_ERR_CAPACITY 4  /* more misses than victim candidates */
#define OR_ERR_BLOCK 8     /* page table names a block outside the pool */

typedef struct or_state or_state;

or_state* or_create(int32_t R, int32_t L, int32_t K, int32_t B, int32_t P,
                    int32_t max_pages, int64_t blocks_per_layer,
                    const int32_t* ctx_cap);
void or_destroy(or_state* s);
int32_t or_set_ctx(or_state* s, int32_t req, int32_t ctx);
int32_t or_set_page(or_state* s, int32_t req, int32_t page, int32_t block);
int32_t or_set_hot_block(or_state* s, int32_t req, int32_t index, int32_t block);
/* One step of one (request, layer) unit.  out_row[K]; miss_log[K][3] holds
 * (j, position, slot) per served miss in selection order (nullable).
 * Returns the OR_ERR_* bits of this call, or -1 for a bad unit. */
int32_t or_resolve(or_state* s, int32_t layer, int32_t req, const int32_t* topk,
                   int32_t step, int32_t* out_row, int32_t* miss_log,
                   int32_t* n_miss);
/* Speculative decoding: one step of one unit for T verify tokens at once.
 * topk[T*K] is token after token; out_row[T*K], miss_log[T*K][3].  A position
 * an earlier token selected shares that entry's row; a repeat within one
 * token's row is an input error. */
int32_t or_resolve_tokens(or_state* s, int32_t layer, int32_t req, int32_t T,
                          const int32_t* topk, int32_t step, int32_t* out_row,
                          int32_t* miss_log, int32_t* n_miss);
int32_t or_get_unit(const or_state* s, int32_t layer, int32_t req,
                    int32_t* slot_pos, int32_t* slot_stamp);
int32_t or_row_content(const or_state* s, int32_t layer, int32_t req,
                       int32_t row, int32_t* pos);

#ifdef __cplusplus
}
#endif
#endif
