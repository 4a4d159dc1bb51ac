// Prefix offload: page "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse
// Offloading in vLLM", section "How it works" -- when a cacheable prefix page
// completes, a copy to CPU memory is queued while the GPU keeps serving the
// page; one launch copies the page of all sparse-MLA layers; once the copy is
// stream-ordered the GPU slot may be released, and the CPU copy serves prefix
// reuse after the transfer completes.
//
// One kernel per call on a side stream, for one page or a batch of pages (all
// of a step's completed pages): every CTA streams 16-byte vectors of a page's
// rows (P rows per layer, contiguous in both pools) from HBM into the mapped
// pinned host pool.  The side stream first waits for the main stream (an event
// the pool owns), then `done` is recorded after the copy; committing a page
// waits on `done` before marking it host only.
#include <chrono>
#include <thread>

#include "hs_internal.cuh"

namespace {

// The pages of one offload call, passed by value (kernel parameter space).
struct PageList {
  int32_t req[HS_OFFLOAD_MAX_PAGES];
  int32_t page[HS_OFFLOAD_MAX_PAGES];
};

// blockIdx.y = (page i, layer l) segment: the page's P rows of layer l, P * rv
// contiguous 16-byte vectors in both pools.  blockIdx.x strides over the
// segment with 4 independent loads in flight per thread.
__global__ void __launch_bounds__(256) offload_pages_kernel(
    const uint4* __restrict__ kv_pool, uint4* __restrict__ host_dev,
    const int32_t* __restrict__ page_table, const int64_t* __restrict__ host_off,
    const __grid_constant__ PageList list, int32_t num_layers, int32_t max_pages,
    int64_t blocks_per_layer, int64_t host_tokens, int32_t P, int32_t rv, int32_t* error_word) {
  const int i = blockIdx.y / num_layers, l = blockIdx.y - i * num_layers;
  const int32_t req = list.req[i], page = list.page[i];
  const int32_t block = page_table[(int64_t)req * max_pages + page];
  if (block < 0 || block >= blocks_per_layer) {
    if (blockIdx.x == 0 && l == 0 && threadIdx.x == 0) atomicOr(error_word, HS_DEV_ERR_BLOCK);
    return;
  }
  const int64_t n = (int64_t)P * rv;  // vectors per page per layer
  const uint4* src = kv_pool + ((int64_t)l * blocks_per_layer + block) * n;
  uint4* dst = host_dev + ((int64_t)l * host_tokens + host_off[req] + (int64_t)page * P) * rv;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (; v + 3 * stride < n; v += 4 * stride) {
    const uint4 a = __ldcs(src + v), b = __ldcs(src + v + stride);
    const uint4 c = __ldcs(src + v + 2 * stride), d = __ldcs(src + v + 3 * stride);
    dst[v] = a;
    dst[v + stride] = b;
    dst[v + 2 * stride] = c;
    dst[v + 3 * stride] = d;
  }
  for (; v < n; v += stride) dst[v] = __ldcs(src + v);
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

// Reads every 16-byte vector of the n at src and discards it, so that the
// GPU has read each host page once (volatile loads: none may be dropped).
__global__ void __launch_bounds__(512) touch_host_kernel(const uint4* __restrict__ src, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    uint32_t a, b, c, d;
    asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(src + i));
    asm volatile("" ::"r"(a), "r"(b), "r"(c), "r"(d));
  }
}

}  // namespace

extern "C" hs_status hs_offload_pages(hs_pool* p, int32_t num_pages, const int32_t* reqs,
                                      const int32_t* pages, void* main_stream, void* side_stream,
                                      void* done_event) {
  if (!p || !reqs || !pages || !done_event || num_pages < 1 || num_pages > HS_OFFLOAD_MAX_PAGES)
    return HS_ERR_INVALID;
  PageList list;
  for (int i = 0; i < num_pages; ++i) {
    if (reqs[i] < 0 || reqs[i] >= p->d.num_requests || pages[i] < 0 ||
        pages[i] >= p->d.max_pages)
      return HS_ERR_INVALID;
    list.req[i] = reqs[i];
    list.page[i] = pages[i];
  }
  cudaStream_t ms = hs_stream(main_stream), ss = hs_stream(side_stream);
  HS_CUDA_TRY(cudaEventRecord(p->order_event, ms));
  HS_CUDA_TRY(cudaStreamWaitEvent(ss, p->order_event, 0));
  const int rv = (int)(hs_row_bytes(p->d) / 16);
  const int64_t n = (int64_t)p->d.page_tokens * rv;  // vectors per (page, layer)
  const int64_t segments = (int64_t)num_pages * p->d.num_layers;
  // about four CTAs per SM over all segments, none without work
  int64_t gx = (4 * (int64_t)p->num_sms + segments - 1) / segments;
  const int64_t gx_max = (n + 4 * 256 - 1) / (4 * 256);
  if (gx > gx_max) gx = gx_max;
  if (gx < 1) gx = 1;
  offload_pages_kernel<<<dim3((unsigned)gx, (unsigned)segments), 256, 0, ss>>>(
      static_cast<const uint4*>(p->kv_pool), static_cast<uint4*>(p->host_pool_dev), p->page_table,
      p->host_off, list, p->d.num_layers, p->d.max_pages, p->blocks_per_layer, p->d.host_tokens,
      p->d.page_tokens, rv, p->error_word);
  HS_CUDA_TRY(cudaGetLastError());
  HS_CUDA_TRY(cudaEventRecord(reinterpret_cast<cudaEvent_t>(done_event), ss));
  return HS_OK;
}

extern "C" hs_status hs_offload_prefix(hs_pool* p, int32_t req, int32_t page, void* main_stream,
                                       void* side_stream, void* done_event) {
  return hs_offload_pages(p, 1, &req, &page, main_stream, side_stream, done_event);
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

extern "C" hs_status hs_pool_touch_host(hs_pool* p, void* stream) {
  if (!p || !p->host_pool_dev) return HS_ERR_INVALID;
  int dev = 0, sms = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int64_t n = (int64_t)(p->host_bytes / 16);
  if (n == 0) return HS_OK;
  touch_host_kernel<<<sms * 4, 512, 0, hs_stream(stream)>>>(
      static_cast<const uint4*>(p->host_pool_dev), n);
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

// Bounded host-side wait for an offload's copy event: polls the event (no
// device-side wait, no stream synchronisation) until it completes or
// timeout_ns of wall-clock time have passed.
extern "C" hs_status hs_wait_offload(void* done_event, int64_t timeout_ns) {
  if (!done_event || timeout_ns < 0) return HS_ERR_INVALID;
  cudaEvent_t ev = reinterpret_cast<cudaEvent_t>(done_event);
  const auto t0 = std::chrono::steady_clock::now();
  const auto limit = std::chrono::nanoseconds(timeout_ns);
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return HS_OK;
    if (e != cudaErrorNotReady) return HS_ERR_CUDA;
    cudaGetLastError();  // "not ready" is a state, not an error: leave no trace of it
    if (std::chrono::steady_clock::now() - t0 >= limit) return HS_ERR_TIMEOUT;
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}
