// Prefix offload: page "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse
// Offloading in vLLM", section "How it works" -- when a cacheable prefix page
// completes, a copy to CPU memory is queued while the GPU keeps serving the
// page; one launch copies the page of all sparse-MLA layers; once the copy is
// stream-ordered the GPU slot may be released, and the CPU copy serves prefix
// reuse after the transfer completes.
//
// One kernel per page on a side stream: every CTA streams 16-byte vectors of
// the page's rows (P x row_elems bf16 per layer, contiguous in both pools)
// from HBM into the mapped pinned host pool.  The side stream first waits for
// the main stream (an event the pool owns), then `done` is recorded after the
// copy; committing the page waits on `done` before marking it host only.
#include "hs_internal.cuh"

namespace {

__global__ void offload_page_kernel(const uint4* __restrict__ kv_pool, uint4* __restrict__ host_dev,
                                    const int32_t* __restrict__ page_table,
                                    const int64_t* __restrict__ host_off, int32_t req, int32_t page,
                                    int32_t max_pages, int64_t blocks_per_layer,
                                    int64_t host_tokens, int32_t P, int32_t rv,
                                    int32_t* error_word) {
  const int32_t block = page_table[(int64_t)req * max_pages + page];
  if (block < 0 || block >= blocks_per_layer) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
      atomicOr(error_word, HS_DEV_ERR_BLOCK);
    return;
  }
  const int l = blockIdx.y;
  const int64_t n = (int64_t)P * rv;  // vectors per page per layer
  const uint4* src = kv_pool + ((int64_t)l * blocks_per_layer + block) * n;
  uint4* dst = host_dev + ((int64_t)l * host_tokens + host_off[req] + (int64_t)page * P) * rv;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __ldcs(src + i);
}

__global__ void unmap_page_kernel(int32_t* page_table, int64_t idx) { page_table[idx] = -1; }

// Streaming copy from mapped pinned host memory into device memory by SM loads
// (the same access path RESOLVE uses for miss rows), 4 independent 16-byte
// loads in flight per thread.
__global__ void __launch_bounds__(512) host_read_kernel(const uint4* __restrict__ src, int64_t n,
                                                        uint4* __restrict__ dst) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
    const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = __ldcs(src + i);
}

}  // namespace

extern "C" hs_status hs_offload_prefix(hs_pool* p, int32_t req, int32_t page, void* main_stream,
                                       void* side_stream, void* done_event) {
  if (!p || req < 0 || req >= p->d.num_requests || page < 0 || page >= p->d.max_pages ||
      !done_event)
    return HS_ERR_INVALID;
  cudaStream_t ms = hs_stream(main_stream), ss = hs_stream(side_stream);
  HS_CUDA_TRY(cudaEventRecord(p->order_event, ms));
  HS_CUDA_TRY(cudaStreamWaitEvent(ss, p->order_event, 0));
  const int rv = (int)(hs_row_bytes(p->d) / 16);
  const int64_t n = (int64_t)p->d.page_tokens * rv;
  int gx = (int)((n + 255) / 256);
  if (gx > 16) gx = 16;  // 16 CTAs per layer: a page is ~295 KB per layer
  dim3 grid(gx, p->d.num_layers);
  offload_page_kernel<<<grid, 256, 0, ss>>>(
      static_cast<const uint4*>(p->kv_pool), static_cast<uint4*>(p->host_pool_dev), p->page_table,
      p->host_off, req, page, p->d.max_pages, p->blocks_per_layer, p->d.host_tokens,
      p->d.page_tokens, rv, p->error_word);
  HS_CUDA_TRY(cudaGetLastError());
  HS_CUDA_TRY(cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), ss));
  return HS_OK;
}

extern "C" hs_status hs_commit_offload(hs_pool* p, int32_t req, int32_t page, void* main_stream,
                                       void* done_event) {
  if (!p || req < 0 || req >= p->d.num_requests || page < 0 || page >= p->d.max_pages ||
      !done_event)
    return HS_ERR_INVALID;
  cudaStream_t ms = hs_stream(main_stream);
  HS_CUDA_TRY(cudaStreamWaitEvent(ms, reinterpret_cast<cudaEvent_t>(done_event), 0));
  unmap_page_kernel<<<1, 1, 0, ms>>>(p->page_table, (int64_t)req * p->d.max_pages + page);
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

extern "C" hs_status hs_host_read(const void* host_device_ptr, int64_t bytes, void* dst,
                                  void* stream) {
  if (!host_device_ptr || !dst || bytes < 0 || (bytes & 15) ||
      (reinterpret_cast<uintptr_t>(host_device_ptr) & 15) || (reinterpret_cast<uintptr_t>(dst) & 15))
    return HS_ERR_INVALID;
  if (bytes == 0) return HS_OK;
  int dev = 0, sms = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  host_read_kernel<<<sms * 4, 512, 0, hs_stream(stream)>>>(
      static_cast<const uint4*>(host_device_ptr), bytes / 16, static_cast<uint4*>(dst));
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}
