// Row gather by row id ("one stride"): page "GLM 5.3 Optimizations, Part 1:
// Hybrid HiSparse Offloading in vLLM", section "How it works" -- whether a
// row sits in a resident page or in the hot buffer, the resolver hands out a
// row id of the same KV tensor and one stride reaches it.
//
// HBM-bound copy: each row is 1152 B (72 x 16 B).  Groups of 8 threads own a
// row and move it with 9 independent 16-byte loads each (all issued before the
// stores), so a 256-thread CTA keeps 32 rows = 36 KB in flight.  The grid is a
// multiple of the SM count and strides over the rows.
#include "hs_internal.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kLanesPerRow = 8;

template <int kVecPerLane>
__global__ void __launch_bounds__(kThreads) gather_rows_kernel(const uint4* __restrict__ layer_base,
                                                               const int32_t* __restrict__ row_ids,
                                                               int64_t n_rows, int64_t rows_in_layer,
                                                               uint4* __restrict__ out,
                                                               int32_t* error_word) {
  constexpr int rv = kVecPerLane * kLanesPerRow;
  const int sub = threadIdx.x % kLanesPerRow;
  const int64_t groups = (int64_t)gridDim.x * (kThreads / kLanesPerRow);
  int err = 0;
  for (int64_t i = (int64_t)blockIdx.x * (kThreads / kLanesPerRow) + threadIdx.x / kLanesPerRow;
       i < n_rows; i += groups) {
    const int32_t rid = __ldg(row_ids + i);
    uint4 v[kVecPerLane];
    if (rid >= 0 && rid < rows_in_layer) {
      const uint4* src = layer_base + (int64_t)rid * rv + sub;
#pragma unroll
      for (int k = 0; k < kVecPerLane; ++k) v[k] = __ldcs(src + k * kLanesPerRow);
    } else {
      if (rid != -1) err = HS_DEV_ERR_BLOCK;
#pragma unroll
      for (int k = 0; k < kVecPerLane; ++k) v[k] = make_uint4(0, 0, 0, 0);
    }
    uint4* dst = out + i * rv + sub;
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) __stcs(dst + k * kLanesPerRow, v[k]);
  }
  if (err) atomicOr(error_word, err);
}

// Any row width that is a multiple of 16 bytes.
__global__ void gather_rows_generic(const uint4* __restrict__ layer_base,
                                    const int32_t* __restrict__ row_ids, int64_t n_rows,
                                    int64_t rows_in_layer, int rv, uint4* __restrict__ out,
                                    int32_t* error_word) {
  const int64_t total = n_rows * rv;
  int err = 0;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < total;
       c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = c / rv;
    const int e = (int)(c - i * rv);
    const int32_t rid = row_ids[i];
    uint4 v = make_uint4(0, 0, 0, 0);
    if (rid >= 0 && rid < rows_in_layer)
      v = layer_base[(int64_t)rid * rv + e];
    else if (rid != -1)
      err = HS_DEV_ERR_BLOCK;
    out[c] = v;
  }
  if (err) atomicOr(error_word, err);
}

}  // namespace

extern "C" hs_status hs_gather(hs_pool* p, int32_t layer, const int32_t* row_ids, int64_t n_rows,
                               void* out_rows, void* stream) {
  if (!p || layer < 0 || layer >= p->d.num_layers || n_rows < 0) return HS_ERR_INVALID;
  if (n_rows == 0) return HS_OK;
  if (!row_ids || !out_rows || (reinterpret_cast<uintptr_t>(out_rows) & 15)) return HS_ERR_INVALID;
  const int rv = (int)(hs_row_bytes(p->d) / 16);
  const int64_t rows_in_layer = p->blocks_per_layer * p->d.page_tokens;
  const uint4* base = static_cast<const uint4*>(p->kv_pool) + (int64_t)layer * rows_in_layer * rv;
  cudaStream_t s = hs_stream(stream);
  if (rv == 72) {
    const int64_t groups_needed = (n_rows + kThreads / kLanesPerRow - 1) / (kThreads / kLanesPerRow);
    int64_t grid = (int64_t)p->num_sms * 8;  // 8 CTAs of 256 threads per SM
    if (grid > groups_needed) grid = groups_needed;
    gather_rows_kernel<9><<<(unsigned)grid, kThreads, 0, s>>>(
        base, row_ids, n_rows, rows_in_layer, static_cast<uint4*>(out_rows), p->error_word);
  } else {
    int64_t grid = (int64_t)p->num_sms * 8;
    gather_rows_generic<<<(unsigned)grid, 256, 0, s>>>(base, row_ids, n_rows, rows_in_layer, rv,
                                                       static_cast<uint4*>(out_rows),
                                                       p->error_word);
  }
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}
