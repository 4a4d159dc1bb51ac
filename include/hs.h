/*
 * libhs -- HiSparse decode-time hot path on one GB300 (sm_103a).
 *
 * C ABI: plain pointers and sizes only.  Streams and events are passed as
 * opaque `void*` holding a cudaStream_t / cudaEvent_t (NULL = legacy default
 * stream).  Every device pointer named "device" must point to memory of the
 * device the pool was created on.
 *
 * Sources.  Page "59188saintaubert.com ... HiSparse" (a summary of the
 * HiSparse paper), section 02: two-level KV -- pinned host DRAM holds each
 * active request's authoritative full KV, the GPU keeps a fixed hot buffer of
 * B slots per request and layer, a page table maps each logical position to a
 * cache slot or a host-only marker, LRU metadata drives replacement, and one
 * fused RESOLVE kernel per sparse layer does hit detection, LRU replacement,
 * metadata update and host fetch (logical index in, physical slot out).
 * Page "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM",
 * section "How it works": resident tokens are read in place and the tail is
 * never evicted; hot tokens are read and their LRU entry refreshed; a miss
 * copies a single row from pinned host memory into an LRU slot; hot pages are
 * ordinary blocks of the same KV tensor, so the resolver hands out row ids
 * that the sparse MLA kernel gathers with one stride; completed prefix pages
 * are copied to host in one launch covering all sparse layers.
 *
 * Data layout (all owned by the pool unless stated):
 *   KV row        row_elems bf16 values (576 = 512 latent + 64 rope), or a
 *                 656-byte FP8 row (kv_format HS_KV_FP8, below)
 *   kv_pool       device [L][blocks_per_layer][P] rows
 *                 blocks 0 .. R*B/P-1 of every layer are the hot buffers:
 *                 request r's hot slot s is block r*(B/P) + s/P, row s%P;
 *                 blocks from R*B/P on hold resident pages
 *   host_pool     pinned, mapped host [L][host_tokens] rows;
 *                 request r's position p of layer l is row host_off[r] + p
 *   row id        index of a row within one layer of kv_pool:
 *                 block * P + offset (-1 = no row)
 *   page_table    device int32 [R][max_pages]: block id, or -1 = host only
 *   LRU metadata  device int32 [L][R][B] slot_pos (-1 = empty),
 *                 slot_stamp (step of last use, -1 = never), lru_order (slots
 *                 sorted by (stamp, slot) ascending); plus an internal
 *                 position -> slot array [L][host_tokens] that RESOLVE keeps
 *                 consistent (modify LRU state only through this API)
 *
 * Errors.  Argument errors are returned synchronously.  Errors found on the
 * device (bad indices in caller data) never trap: the kernel writes row id
 * -1 for the offending entry and ORs a bit into the pool's device error word,
 * which hs_check_errors() reads and clears.
 */
#ifndef HS_H
#define HS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HS_OK = 0,
  HS_ERR_INVALID = -1,  /* bad argument (null pointer, out-of-range index, bad shape) */
  HS_ERR_CUDA = -2,     /* a CUDA runtime call failed */
  HS_ERR_OOM = -3,      /* device or pinned host allocation failed */
  HS_ERR_CAPACITY = -4, /* more misses than free slots were seen (error bit 4) */
  HS_ERR_DEVICE = -5,   /* the device error word was non-zero */
  HS_ERR_TIMEOUT = -6   /* a bounded wait gave up */
} hs_status;

/* Bits of the device error word (also returned by hs_check_errors). */
#define HS_DEV_ERR_RANGE 1     /* selected position outside [0, ctx) and not -1 */
#define HS_DEV_ERR_DUPLICATE 2 /* position repeated within one top-K row */
#define HS_DEV_ERR_CAPACITY 4  /* misses exceeded the slots not used this step */
#define HS_DEV_ERR_BLOCK 8     /* page table / row id names a block outside the pool */
#define HS_DEV_ERR_WAIT 16     /* an in-kernel bounded wait gave up */
#define HS_DEV_ERR_INTERNAL 32 /* a kernel found its own launch set-up unusable and did nothing */
#define HS_DEV_ERR_VALUE 64    /* attention: a value element (first 512 columns of a selected
                                  row) is not finite or has magnitude >= 65536; the P.V
                                  product runs in fp16 (see hs_sparse_mla_decode).  FP8
                                  rows: an operand (a latent value, a rope value or q)
                                  that fp16 cannot hold, or a NaN code */

/* KV row formats.  HS_KV_BF16: row_elems bf16 values (2 * row_elems bytes).
 * HS_KV_FP8 (row_elems must be 576): 656 bytes -- bytes 0..511 the 512 latent
 * values as OCP FP8 E4M3 codes (bias 7, largest 448, no infinities), bytes
 * 512..527 four fp32 scales (latent value i = E4M3(code i) * scale[i / 128]),
 * bytes 528..655 the 64 rope values as bf16.  The pages' benchmark runs an FP8
 * KV cache but gives no row layout; this is the one this library defines.
 * RESOLVE, gather, page loads and offload move rows as opaque bytes in
 * either format; attention dequantizes FP8 rows (see hs_sparse_mla_decode). */
enum { HS_KV_BF16 = 0, HS_KV_FP8 = 1 };

typedef struct {
  int32_t num_requests;    /* R */
  int32_t num_layers;      /* L sparse layers */
  int32_t top_k;           /* K: selections per (request, layer) and step */
  int32_t hot_slots;       /* B: hot-buffer rows per (request, layer); multiple of page_tokens */
  int32_t page_tokens;     /* P: tokens per page/block */
  int32_t row_elems;       /* bf16 values per KV row; multiple of 8 (576 here) */
  int32_t max_pages;       /* logical pages per request (page table width) */
  int32_t kv_format;       /* HS_KV_BF16 or HS_KV_FP8 (see below) */
  int64_t host_tokens;     /* rows per layer in the pinned host pool */
  int64_t resident_blocks; /* blocks per layer for resident pages (beyond the hot buffers) */
} hs_pool_desc;

typedef struct {
  void* kv_pool;          /* device, see layout above */
  void* host_pool;        /* host pointer of the pinned host pool */
  void* host_pool_device; /* device-accessible alias of the same memory */
  int32_t* page_table;    /* device [R][max_pages] */
  int32_t* ctx_len;       /* device [R] */
  int64_t* host_off;      /* device [R] */
  int32_t* hot_block;     /* device [R][B/P] */
  int32_t* slot_pos;      /* device [L][R][B] */
  int32_t* slot_stamp;    /* device [L][R][B] */
  int32_t* lru_order;     /* device [L][R][B] */
  int32_t* step;          /* device scalar: the pool's decode-step counter */
  int32_t* error_word;    /* device scalar */
  int64_t blocks_per_layer;
  int64_t kv_pool_bytes;
  int64_t host_pool_bytes;
} hs_pool_views;

typedef struct hs_pool hs_pool; /* opaque, library-owned */

/* Create a pool on the current CUDA device.  Allocates the pinned + mapped
 * host pool (cudaHostAlloc), the per-layer GPU KV pool (hot-buffer blocks
 * leased once per (request, layer), then resident blocks), the page table
 * (all host-only), LRU metadata (all slots empty, stamp -1), the step counter
 * (0) and the attention workspace.  Synchronous.  On failure *out is NULL and
 * nothing stays allocated: HS_ERR_OOM when an allocation fails, and before any
 * allocation (and any CUDA call) when the host pool is larger than the
 * machine's physical memory.  Host-pool contents are left uninitialised. */
hs_status hs_pool_create(const hs_pool_desc* desc, hs_pool** out);

/* The host NUMA node the pool's pinned host pool was placed on, or -1.
 * On a machine with several host NUMA nodes, hs_pool_create places it on the
 * node CUDA reports as nearest the device (preferred-node policy, huge pages
 * where offered, then registered pinned and mapped), so that each replica's
 * miss reads stay on its socket (page "GLM 5.3 Optimizations, Part 1",
 * section "Composition with the rest of vLLM": one pinned host pool per
 * data-parallel replica); -1 with a single node, when the device reports no
 * host node, or when the placement was refused (then cudaHostAlloc placed
 * it). */
hs_status hs_pool_host_numa_node(const hs_pool* pool, int32_t* node_out);

/* Free everything the pool owns.  Synchronises the device first. */
hs_status hs_pool_destroy(hs_pool* pool);

/* Raw pointers for inspection and bulk set-up (e.g. filling host_pool).  The
 * pool keeps ownership; pointers stay valid until hs_pool_destroy. */
hs_status hs_pool_get_views(const hs_pool* pool, hs_pool_views* out);

/* Reset the LRU metadata of every unit (slots empty, stamp -1, identity
 * order), the step counter and the error word.  Async on `stream`. */
hs_status hs_pool_reset(hs_pool* pool, void* stream);

/* Set a request's current context length and its first row in the host pool.
 * Async on `stream`, graph-capturable.  HS_ERR_INVALID if req is out of range,
 * ctx_len > max_pages * P or host_off + ctx_len > host_tokens.  A request's
 * host_off must not change while its units hold hot rows (hs_pool_reset
 * first); growing ctx_len is always allowed. */
hs_status hs_set_request(hs_pool* pool, int32_t req, int32_t ctx_len,
                         int64_t host_off, void* stream);

/* page_table[req][page] = block (block -1 marks the page host only).  Async on
 * `stream`, graph-capturable.  HS_ERR_INVALID if block is a hot-buffer block
 * or outside the pool. */
hs_status hs_map_page(hs_pool* pool, int32_t req, int32_t page, int32_t block,
                      void* stream);

/* Make a page resident: copy its rows of every layer from the host pool into
 * `block`, then map it.  Async on `stream` (set-up path). */
hs_status hs_load_page(hs_pool* pool, int32_t req, int32_t page, int32_t block,
                       void* stream);

/* RESOLVE (one launch for layers layer_begin .. layer_begin+num_layers-1,
 * one CTA per (request, layer) unit).  For every unit and j < K:
 *   p = topk_idx[i][r][j]; -1 is padding (row id -1);
 *   a resident page gives block*P + p%P, LRU untouched;
 *   a hot hit gives the slot's row and stamps it with *d_step;
 *   each miss (in j order) takes the next slot with stamp < *d_step in
 *   (stamp, slot) order, gets stamp *d_step and receives a copy of host row
 *   host_off[r] + p of layer l, loaded by the kernel from mapped pinned memory.
 * Hits are refreshed before misses are served, so a slot used in this step is
 * never a victim.
 *   topk_idx     device int32 [num_layers][R][K]          (caller-owned)
 *   d_step       device int32 scalar (e.g. views.step), read by the kernel, so
 *                a captured CUDA graph replays with the current step
 *   out_row_ids  device int32 [num_layers][R][K]          (caller-owned)
 *   miss_count   device int32 [num_layers][R] or NULL: misses served
 *   miss_log     device int32 [num_layers][R][K][3] or NULL: (j, position,
 *                slot) of each served miss in j order; later entries undefined
 * Async on `stream`; no host synchronisation, no allocation; graph-capturable.
 * Device-side errors: bits RANGE, DUPLICATE, CAPACITY, BLOCK. */
hs_status hs_resolve(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                     const int32_t* topk_idx, const int32_t* d_step,
                     int32_t* out_row_ids, int32_t* miss_count,
                     int32_t* miss_log, void* stream);

/* RESOLVE for the T verify tokens of a speculative-decoding step.  Page "GLM
 * 5.3 Optimizations, Part 1", section "Composition with the rest of vLLM":
 * speculative decoding works through a replayable per-step resolver plan and
 * the verify steps share the request's hot state; section "Exploiting
 * sparsity when needed" (note): the hot buffer must hold every verify token's
 * selection at once, (num_speculative_tokens + 2) x top-K rows.  Each unit's
 * T rows of K positions are resolved as one list, token after token, exactly
 * as hs_resolve resolves one row, except that a position an earlier token of
 * the list also selected takes no slot of its own: it gets that entry's row
 * (resident, hot or a served miss; -1 if that miss found no slot).  So the
 * whole list's hits are pinned before any miss takes a victim, which calling
 * hs_resolve once per token would not do.  A repeat within one token's row is
 * an input error (bit DUPLICATE), as in hs_resolve.  T = 1 is hs_resolve.
 *   topk_idx     device int32 [num_layers][R][T][K]
 *   out_row_ids  device int32 [num_layers][R][T][K]
 *   miss_count   device int32 [num_layers][R] or NULL: misses served
 *   miss_log     device int32 [num_layers][R][T*K][3] or NULL: (j, position,
 *                slot) per served miss, j indexing the unit's T*K list
 * Sizes: B at most 16384 slots.  A list whose tables fit one CTA's shared
 * memory (at most 8192 entries, e.g. T = 4 at K = 2048 with B up to 12288)
 * runs as one launch; a longer one as launches over groups of its tokens, in
 * order, after one pass that pins every hit of the whole list, with the same
 * row ids, slot state and miss log as one launch over the list.  HS_ERR_INVALID
 * if B is larger or even one token's tables do not fit.  Async,
 * graph-capturable, no allocation. */
hs_status hs_resolve_tokens(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                            int32_t num_tokens, const int32_t* topk_idx,
                            const int32_t* d_step, int32_t* out_row_ids,
                            int32_t* miss_count, int32_t* miss_log, void* stream);

/* Gather rows of one layer by row id ("one stride"): out_rows[i] =
 * kv_pool[layer][row_ids[i]] (one row of the pool's format: row_elems bf16,
 * or 656 bytes for HS_KV_FP8); row id -1 gives a zero row.  row_ids: device
 * int32 [n_rows]; out_rows: device [n_rows][row bytes] (caller-owned).
 * Async, graph-capturable.  A row id outside the layer writes a zero row and
 * sets error bit BLOCK. */
hs_status hs_gather(hs_pool* pool, int32_t layer, const int32_t* row_ids,
                    int64_t n_rows, void* out_rows, void* stream);

/* Sparse MLA decode attention of one layer over exactly the K rows each
 * request resolved (absorbed MLA, page "GLM 5.3 Optimizations, Part 1"
 * section "How it works": the sparse MLA kernel reads hot and resident rows
 * alike by row id):
 *   s[h][j]  = scale * sum_{d<row_elems} q[r][h][d] * kv(row_ids[r][j])[d]
 *   out[r][h][e] = sum_j softmax_j(s[h][.]) * kv(row_ids[r][j])[e],  e < v_dim
 * over the j with row_ids >= 0 (v = the first v_dim = 512 columns of each
 * row).  bf16 inputs, fp32 accumulation on the tensor cores, bf16 output.
 * Scores use bf16 q and rows as given.  The probabilities and the value
 * columns enter the P.V product as fp16, which holds every bf16 value of
 * magnitude below 65536 exactly (values below 2^-14 lose low bits, at most
 * 2^-25 each) and gives the probabilities 11 significant bits; a value
 * element that is not finite or has magnitude >= 65536 sets error bit VALUE
 * (that request's output is then not meaningful).  When K is split between
 * several CTA pairs, each pair's normalised partial output is held in fp16
 * (one more rounding, 2^-12 relative) until the bf16 combination.
 * FP8 pools (HS_KV_FP8): both products run on fp16 operands.  q is rounded
 * from bf16 to fp16; a latent value is E4M3(code) * scale formed as fp16 --
 * from the scale rounded to fp16 when every group scale of the 8 rows a
 * loader warp handles in that tile is 0 or in [2^-14, 146] (so no code can
 * overflow), else in fp32 and rounded once -- and a rope value is converted
 * from bf16.  An operand fp16 cannot hold, or a NaN code, sets VALUE.
 *   q        device bf16 [R][num_heads][row_elems]   (num_heads <= 128)
 *   row_ids  device int32 [R][K] (e.g. hs_resolve's output for this layer)
 *   out      device bf16 [R][num_heads][v_dim]
 *   lse      device float [R][num_heads] or NULL: natural-log sum of exp of
 *            the scores (-inf when a request has no valid row; out is then 0)
 * Async, graph-capturable; uses the pool's workspace (calls on one pool must
 * not overlap on the GPU). */
hs_status hs_sparse_mla_decode(hs_pool* pool, int32_t layer, const void* q,
                               const int32_t* row_ids, int32_t num_heads,
                               int32_t v_dim, float scale, void* out,
                               float* lse, void* stream);

/* One decode step over sparse layers layer_begin .. layer_begin+num_layers-1:
 * for each layer i, RESOLVE (as hs_resolve) then sparse MLA decode attention
 * over the resolved rows (as hs_sparse_mla_decode), with the same results as
 * those calls made in that order, but with "precise prefetch": RESOLVE of
 * layer i+1 -- its misses' host reads -- runs on `copy_stream` while layer i's
 * attention runs on `stream`.  Page "59188saintaubert.com ... HiSparse",
 * section 04: a synchronous resolve exposes 7-8 ms of host IO per token and
 * prefetching with exact selections brings it to about 3 ms (section 03:
 * prefetch alone adds 14-17% throughput); page "GLM 5.3 Optimizations, Part
 * 1", section "Exploiting sparsity when needed": IndexShare gives one indexer
 * layer per four sparse-MLA layers, so later layers' selections are known
 * before the current layer's attention.
 *   topk_idx     device int32 [num_layers][R][K]
 *   q            device bf16 [num_layers][R][num_heads][576]
 *   d_step       as for hs_resolve (not advanced here)
 *   out_row_ids  device int32 [num_layers][R][K]
 *   out          device bf16 [num_layers][R][num_heads][512]
 *   lse          device float [num_layers][R][num_heads] or NULL
 *   miss_count   device int32 [num_layers][R] or NULL
 * `copy_stream` starts after the work queued on `stream` before the call
 * (bf16 rows: layer 1's RESOLVE runs beside layer 0's) or, for FP8 rows, after
 * layer 0's RESOLVE; all of the step's work is ordered before later work on
 * `stream`.  With copy_stream == stream (or one layer) the calls simply run in
 * order on `stream`.
 * Attention results may differ from hs_sparse_mla_decode's in the last bits
 * (a launch beside a RESOLVE splits K into fewer parts).  Async,
 * graph-capturable (copy_stream joins the capture through events); uses the
 * pool's workspace and hand-off events, so steps on one pool must not overlap.
 * Argument errors as for the two calls, checked before anything is queued. */
hs_status hs_decode_step(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                         const int32_t* topk_idx, const void* q, int32_t num_heads,
                         int32_t v_dim, float scale, const int32_t* d_step,
                         int32_t* out_row_ids, void* out, float* lse,
                         int32_t* miss_count, void* stream, void* copy_stream);

/* hs_decode_step for a speculative-decoding step: num_tokens (T) verify
 * tokens per request.  Each layer's RESOLVE takes a unit's T lists as one
 * (as hs_resolve_tokens), and its attention runs one decode row per
 * (request, token) (as hs_sparse_mla_decode_tokens); the schedule is
 * hs_decode_step's.  Page "GLM 5.3 Optimizations, Part 1", section
 * "Composition with the rest of vLLM": the verify steps share the request's
 * hot state through a per-step resolver plan that can be replayed.
 *   topk_idx     device int32 [num_layers][R][T][K]
 *   q            device bf16 [num_layers][R][T][num_heads][576]
 *   out_row_ids  device int32 [num_layers][R][T][K]
 *   out          device bf16 [num_layers][R][T][num_heads][512]
 *   lse          device float [num_layers][R][T][num_heads] or NULL
 *   miss_count   device int32 [num_layers][R] or NULL
 * T = 1 is hs_decode_step.  HS_ERR_INVALID also when R x T > 65535 or the
 * unit's T x K list does not fit RESOLVE's shared memory (as
 * hs_resolve_tokens). */
hs_status hs_decode_step_tokens(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                                int32_t num_tokens, const int32_t* topk_idx, const void* q,
                                int32_t num_heads, int32_t v_dim, float scale,
                                const int32_t* d_step, int32_t* out_row_ids, void* out,
                                float* lse, int32_t* miss_count, void* stream,
                                void* copy_stream);

/* Sparse MLA decode attention of one layer for the T verify tokens of a
 * speculative-decoding step: each (request, token) has its own query and its
 * own K rows (hs_resolve_tokens' output), computed as hs_sparse_mla_decode
 * computes one request.
 *   q        device bf16 [R][T][num_heads][576]
 *   row_ids  device int32 [R][T][K]
 *   out      device bf16 [R][T][num_heads][512]
 *   lse      device float [R][T][num_heads] or NULL
 * The K splits are limited to what the pool's workspace holds for R*T rows;
 * HS_ERR_INVALID if even the fewest the kernel needs do not fit, or R*T >
 * 65535.  Async, graph-capturable; shares the pool's workspace with
 * hs_sparse_mla_decode (calls on one pool must not overlap). */
hs_status hs_sparse_mla_decode_tokens(hs_pool* pool, int32_t layer, int32_t num_tokens,
                                      const void* q, const int32_t* row_ids,
                                      int32_t num_heads, int32_t v_dim, float scale,
                                      void* out, float* lse, void* stream);

/* Allocation-free variant of hs_sparse_mla_decode (no counterpart on the
 * pages: it exists for callers that cannot allocate device memory when they
 * decode -- an engine that handed all free HBM to its KV cache at start-up, an
 * allocator that forbids new device allocations while serving, or a plug-in
 * that is only given raw device pointers -- and so cannot create a pool).
 * Same computation and output as hs_sparse_mla_decode, with plain pointers:
 *   kv_rows   device bf16 [num_rows][576]: the layer's KV rows, row ids index it
 *   q         device bf16 [num_requests][num_heads][576]
 *   row_ids   device int32 [num_requests][top_k] (-1 = padding; an id outside
 *             [0, num_rows) is excluded like padding and sets error bit BLOCK)
 *   out, lse  as for hs_sparse_mla_decode
 * Device-side errors go to an error word of the library's own (one per
 * device, shared by every call), which hs_noalloc_check_errors reads and
 * clears: BLOCK as above, VALUE (as for hs_sparse_mla_decode: the output of
 * that call is not meaningful), WAIT (a bounded wait gave up; the output is
 * not meaningful) and INTERNAL (the kernel found its launch set-up unusable
 * and did nothing).
 * It calls no cudaMalloc, cudaFree or other allocating routine: its split-K
 * scratch is a fixed device array of this library (8 MiB + 32 KiB, held by
 * every GPU that loads the library until the process exits), big enough for
 * 64 (request, split) partials; the call uses fewer splits to fit, and returns
 * HS_ERR_INVALID if num_requests x ceil(top_k / 2048) > 64.  The first call on
 * a device looks up that array's device address and sets the kernel's
 * shared-memory limit (no allocation); make it before any stream capture.
 * Every call shares the array, so calls whose kernels overlap on the GPU (for
 * example on two streams) race; nothing in it needs to start at zero.  Async on
 * `stream`. */
hs_status hs_sparse_mla_decode_noalloc(const void* kv_rows, int64_t num_rows, const void* q,
                                       const int32_t* row_ids, int32_t num_requests,
                                       int32_t top_k, int32_t num_heads, int32_t v_dim,
                                       float scale, void* out, float* lse, void* stream);

/* Synchronise the current device, then read and clear the error word that
 * hs_sparse_mla_decode_noalloc calls on this device OR their device-side
 * error bits into (BLOCK, VALUE, WAIT, INTERNAL; see there).  Allocates
 * nothing (a 4-byte copy each way between host and the library's fixed
 * device word).  No counterpart on the pages: it is the error channel of the
 * allocation-free call.  Returns HS_OK if the word was zero, HS_ERR_DEVICE
 * otherwise; *code_out (if not NULL) receives the bits. */
hs_status hs_noalloc_check_errors(int32_t* code_out);

/* Prefix offload: copy page `page` of request `req` (all layers, from the
 * block the page table maps it to) into its rows of the host pool.  The copy
 * is one kernel launch on `side_stream`, ordered after the work queued so far
 * on `main_stream`; `done_event` (caller-owned cudaEvent_t) is recorded on
 * `side_stream` after it.  The page stays mapped and readable on the GPU.
 * HS_ERR_INVALID for out-of-range arguments; if the page is not mapped to a
 * resident block when the copy runs, nothing is copied and the kernel sets
 * device error bit BLOCK. */
hs_status hs_offload_prefix(hs_pool* pool, int32_t req, int32_t page,
                            void* main_stream, void* side_stream,
                            void* done_event);

/* Prefix offload of several pages in one launch (e.g. every page a decode
 * step completed): as hs_offload_prefix for each (reqs[i], pages[i]),
 * i < num_pages, with one `done_event` recorded after all of them.  Page
 * "GLM 5.3 Optimizations, Part 1", section "How it works": the completed
 * prefix is copied to host memory by one launch for all sparse-MLA layers.
 * reqs and pages are host arrays; 1 <= num_pages <= HS_OFFLOAD_MAX_PAGES.
 * HS_ERR_INVALID for out-of-range arguments (nothing is launched); a pair
 * whose page is not mapped to a resident block when the copy runs is skipped
 * and sets device error bit BLOCK.  The same pair twice copies it twice. */
#define HS_OFFLOAD_MAX_PAGES 256
hs_status hs_offload_pages(hs_pool* pool, int32_t num_pages, const int32_t* reqs,
                           const int32_t* pages, void* main_stream, void* side_stream,
                           void* done_event);

/* Make `main_stream` wait for `done_event`, then mark the page host only
 * (page_table = -1).  The freed block may be mapped again afterwards. */
hs_status hs_commit_offload(hs_pool* pool, int32_t req, int32_t page,
                            void* main_stream, void* done_event);

/* Bounded wait, on the host, for an offload to finish: page "GLM 5.3
 * Optimizations, Part 1", section "How it works" -- the CPU copy of a
 * completed prefix page serves prefix reuse only once its transfer has
 * completed.  Polls `done_event` (the event hs_offload_prefix or
 * hs_offload_pages recorded) every ~20 us without synchronising any stream,
 * for at most timeout_ns of wall-clock time (0 = one poll).  Returns HS_OK once
 * the copy has completed (its host rows are then readable), HS_ERR_TIMEOUT if
 * it has not by then (nothing is cancelled; wait again or commit later),
 * HS_ERR_CUDA if the event reports an error, HS_ERR_INVALID for a NULL event or
 * a negative timeout.  An event never recorded counts as complete. */
hs_status hs_wait_offload(void* done_event, int64_t timeout_ns);

/* Copy `bytes` (a multiple of 16) from mapped pinned host memory (its device
 * alias, e.g. views.host_pool_device) to device memory `dst` with SM loads --
 * the access path RESOLVE uses for miss rows -- so its bandwidth is the
 * ceiling of the in-kernel miss copy.  Async on `stream`.  HS_ERR_INVALID for
 * null or misaligned pointers. */
hs_status hs_host_read(const void* host_device_ptr, int64_t bytes, void* dst, void* stream);

/* Have the GPU read the pool's whole host pool once (through its device
 * alias; the data is discarded).  On some machines the GPU's first read of
 * each host page is slow (a decode step's misses then took ~10x longer until
 * the pages had been read once), so a server calls this once after creating
 * the pool, before serving.  Reads p->host_bytes at the host link's rate (about
 * 23 ms for 4.8 GB at 211 GB/s); changes nothing.  Async on `stream`.
 * HS_ERR_INVALID for a NULL pool. */
hs_status hs_pool_touch_host(hs_pool* pool, void* stream);

/* Self-test of the in-kernel bounded waits that keep a stalled hand-off from
 * hanging the GPU: two one-thread kernels each wait on an mbarrier of their
 * own CTA that nothing arrives on, with the waits the attention kernel and
 * RESOLVE use, limited to timeout_ns (1 .. 1e8) instead of their 1 s.
 * result: device int32[2], set on `stream` to [the error bits the attention
 * wait raised (WAIT expected), 1 if RESOLVE's wait gave up].  HS_ERR_INVALID
 * for a null result or a timeout out of range. */
hs_status hs_selftest_bounded_waits(int64_t timeout_ns, int32_t* result, void* stream);

/* *d_step += 1 on `stream` (graph-capturable). */
hs_status hs_step_advance(int32_t* d_step, void* stream);

/* Synchronise the device, read and clear the device error word into
 * *code_out.  Returns HS_OK if it was zero, HS_ERR_DEVICE otherwise. */
hs_status hs_check_errors(hs_pool* pool, int32_t* code_out);

/* Static string naming a status. */
const char* hs_status_string(hs_status status);

/* Library version string. */
const char* hs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HS_H */
