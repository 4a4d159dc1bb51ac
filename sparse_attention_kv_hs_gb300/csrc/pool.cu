// Pool lifetime, set-up calls and small control kernels of libhs.
//
// The pool is the two-level KV store of page "59188saintaubert.com ...
// HiSparse", section 02: a pinned host pool with every request's full KV, and
// on the GPU a fixed hot buffer of B slots per (request, layer) plus the
// resident pages, all in one per-layer KV tensor (page "GLM 5.3
// Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM", section "How it
// works": hot pages are ordinary blocks of the same KV tensor).
#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <cstdio>
#include <cstring>
#include <new>

#include "hs_internal.cuh"

namespace {

__global__ void reset_kernel(int32_t* slot_pos, int32_t* slot_stamp, int32_t* lru_order,
                             int64_t units, int32_t B, int32_t* step, int32_t* error_word) {
  const int64_t n = units * B;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    slot_pos[i] = -1;
    slot_stamp[i] = -1;
    lru_order[i] = (int32_t)(i % B);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *step = 0;
    *error_word = 0;
  }
}

// Clear the position -> slot entries of every occupied slot (before the slots
// themselves are emptied), so the inverse array stays consistent.
__global__ void clear_inverse_kernel(const int32_t* slot_pos, int32_t* inv, const int64_t* host_off,
                                     int32_t R, int32_t B, int64_t units, int64_t host_tokens) {
  const int64_t n = units * B;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t p = slot_pos[i];
    if (p < 0) continue;
    const int64_t u = i / B;
    const int64_t l = u / R, r = u % R;
    inv[l * host_tokens + host_off[r] + p] = -1;
  }
}

__global__ void init_tables_kernel(int32_t* page_table, int64_t n_pt, int32_t* hot_block,
                                   int32_t R, int32_t hot_per_req, int32_t* ctx_len,
                                   int64_t* host_off) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_pt;
       i += (int64_t)gridDim.x * blockDim.x)
    page_table[i] = -1;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (int64_t)R * hot_per_req;
       i += (int64_t)gridDim.x * blockDim.x)
    hot_block[i] = (int32_t)i;  // request r's i-th hot block is r*(B/P)+i
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < R;
       i += (int64_t)gridDim.x * blockDim.x) {
    ctx_len[i] = 0;
    host_off[i] = 0;
  }
}

__global__ void set_request_kernel(int32_t* ctx_len, int64_t* host_off, int32_t req,
                                   int32_t ctx, int64_t off) {
  ctx_len[req] = ctx;
  host_off[req] = off;
}

__global__ void set_i32_kernel(int32_t* dst, int32_t value) { *dst = value; }

__global__ void step_advance_kernel(int32_t* step) { *step += 1; }

void free_pool(hs_pool* p) {
  if (!p) return;
  cudaFree(p->kv_pool);
  if (p->host_pool && p->host_map_len) {
    cudaHostUnregister(p->host_pool);
    munmap(p->host_pool, p->host_map_len);
  } else if (p->host_pool) {
    cudaFreeHost(p->host_pool);
  }
  cudaFree(p->page_table);
  cudaFree(p->ctx_len);
  cudaFree(p->host_off);
  cudaFree(p->hot_block);
  cudaFree(p->slot_pos);
  cudaFree(p->slot_stamp);
  cudaFree(p->lru_order);
  cudaFree(p->inv);
  cudaFree(p->step);
  cudaFree(p->error_word);
  cudaFree(p->resolve_counts);
  hs_attn_workspace_free(p);
  if (p->order_event) cudaEventDestroy(p->order_event);
  if (p->step_events) {
    for (int i = 0; i <= p->d.num_layers; ++i)
      if (p->step_events[i]) cudaEventDestroy(p->step_events[i]);
    delete[] p->step_events;
  }
  delete[] p->host_off_mirror;
  delete p;
}

// Host NUMA nodes with memory (node directories under sysfs); 0 if unknown.
int host_numa_nodes() {
  int n = 0;
  for (int i = 0; i < 1024; ++i) {
    char path[64];
    snprintf(path, sizeof path, "/sys/devices/system/node/node%d", i);
    if (access(path, F_OK) == 0) ++n;
  }
  return n;
}

// The pinned, mapped host pool.  On a machine with several host NUMA nodes it
// is placed on the node CUDA reports as nearest the device: anonymous memory
// with that node as the preferred policy (the kernel falls back to other
// nodes only when it is full) and huge pages where the system offers them,
// then registered with CUDA (pinned and mapped), so a miss's host read
// crosses no socket boundary.  With one node (or no node reported, or the
// policy call refused) cudaHostAlloc places it: with nothing to choose, its
// mapping is the faster one for the GPU's first touch of each page.
hs_status alloc_host_pool(hs_pool* p) {
  p->host_pool = nullptr;
  p->host_map_len = 0;
  p->host_numa_node = -1;
  int node = -1;
  if (cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, p->device) != cudaSuccess) {
    cudaGetLastError();
    node = -1;
  }
  const long page = sysconf(_SC_PAGESIZE);
  if (node >= 0 && node < 1024 && page > 0 && host_numa_nodes() > 1) {
    const size_t len = (p->host_bytes + (size_t)page - 1) / (size_t)page * (size_t)page;
    void* m = mmap(nullptr, len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (m != MAP_FAILED) {
      madvise(m, len, MADV_HUGEPAGE);  // advice only: ignored where unsupported
      unsigned long mask[1024 / (8 * sizeof(unsigned long))] = {0};
      mask[node / (8 * sizeof(unsigned long))] |= 1ul << (node % (8 * sizeof(unsigned long)));
      const long kPreferred = 1;  // MPOL_PREFERRED
      if (syscall(SYS_mbind, m, len, kPreferred, mask, (unsigned long)1024 + 1, 0u) == 0 &&
          cudaHostRegister(m, len, cudaHostRegisterMapped | cudaHostRegisterPortable) ==
              cudaSuccess) {
        p->host_pool = m;
        p->host_map_len = len;
        p->host_numa_node = node;
        return HS_OK;
      }
      cudaGetLastError();
      munmap(m, len);
    }
  }
  const cudaError_t e =
      cudaHostAlloc(&p->host_pool, p->host_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    p->host_pool = nullptr;
    return HS_ERR_OOM;
  }
  return HS_OK;
}

template <typename T>
hs_status dev_alloc(T** ptr, size_t count) {
  *ptr = nullptr;
  if (count == 0) count = 1;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(ptr), count * sizeof(T));
  if (e != cudaSuccess) {
    cudaGetLastError();
    *ptr = nullptr;
    return e == cudaErrorMemoryAllocation ? HS_ERR_OOM : HS_ERR_CUDA;
  }
  return HS_OK;
}

}  // namespace

extern "C" hs_status hs_pool_create(const hs_pool_desc* desc, hs_pool** out) {
  if (!out) return HS_ERR_INVALID;
  *out = nullptr;
  if (!desc) return HS_ERR_INVALID;
  const hs_pool_desc& d = *desc;
  if (d.num_requests <= 0 || d.num_layers <= 0 || d.top_k <= 0 || d.hot_slots <= 0 ||
      d.page_tokens <= 0 || d.row_elems <= 0 || d.row_elems % 8 != 0 || d.max_pages <= 0 ||
      (d.kv_format != HS_KV_BF16 && d.kv_format != HS_KV_FP8) ||
      (d.kv_format == HS_KV_FP8 && d.row_elems != 576) || d.host_tokens <= 0 ||
      d.resident_blocks < 0 ||
      d.hot_slots % d.page_tokens != 0)
    return HS_ERR_INVALID;
  // Limits of the RESOLVE kernel's shared-memory plan (one CTA per unit).
  if (d.top_k > 8192 || d.hot_slots > 16384) return HS_ERR_INVALID;
  const int64_t hot_blocks = (int64_t)d.num_requests * (d.hot_slots / d.page_tokens);
  const int64_t bpl = hot_blocks + d.resident_blocks;
  if (bpl * d.page_tokens > INT32_MAX) return HS_ERR_INVALID;  // row ids are int32
  if ((int64_t)d.max_pages * d.page_tokens > INT32_MAX) return HS_ERR_INVALID;

  {
    // A host pool larger than this machine's physical memory can never be
    // pinned: report it before anything is allocated.
    const long pages = sysconf(_SC_PHYS_PAGES), page = sysconf(_SC_PAGESIZE);
    const double host_bytes = (double)d.num_layers * (double)d.host_tokens * (double)hs_row_bytes(d);
    if (pages > 0 && page > 0 && host_bytes > (double)pages * (double)page) return HS_ERR_OOM;
  }
  hs_pool* p = new (std::nothrow) hs_pool();
  if (!p) return HS_ERR_OOM;
  std::memset(p, 0, sizeof(*p));
  p->d = d;
  p->blocks_per_layer = bpl;
  p->hot_blocks = hot_blocks;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return HS_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);

  hs_status st = HS_OK;
  const int64_t R = d.num_requests, L = d.num_layers, B = d.hot_slots;
  {
    size_t smem = 0;
    if ((st = hs_resolve_configure(d.top_k, d.hot_slots, d.page_tokens, d.max_pages, &smem,
                                   p->resolve_max_clusters)) != HS_OK) {
      delete p;
      return st;
    }
    p->resolve_smem = smem;
  }
  p->host_off_mirror = new (std::nothrow) int64_t[R]();
  if (!p->host_off_mirror) {
    delete p;
    return HS_ERR_OOM;
  }
  p->kv_bytes = (size_t)L * bpl * d.page_tokens * hs_row_bytes(d);
  if ((st = dev_alloc(reinterpret_cast<char**>(&p->kv_pool), p->kv_bytes)) != HS_OK) goto fail;
  p->host_bytes = (size_t)L * d.host_tokens * hs_row_bytes(d);
  {
    if ((st = alloc_host_pool(p)) != HS_OK) goto fail;
    if (cudaHostGetDevicePointer(&p->host_pool_dev, p->host_pool, 0) != cudaSuccess) {
      st = HS_ERR_CUDA;
      goto fail;
    }
  }
  if ((st = dev_alloc(&p->page_table, (size_t)R * d.max_pages)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->ctx_len, (size_t)R)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->host_off, (size_t)R)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->hot_block, (size_t)R * (B / d.page_tokens))) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->slot_pos, (size_t)L * R * B)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->slot_stamp, (size_t)L * R * B)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->lru_order, (size_t)L * R * B)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->inv, (size_t)L * d.host_tokens)) != HS_OK) goto fail;
  if (cudaMemset(p->inv, 0xFF, sizeof(int32_t) * (size_t)L * d.host_tokens) != cudaSuccess) {
    st = HS_ERR_CUDA;
    goto fail;
  }
  if ((st = dev_alloc(&p->step, 1)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->error_word, 1)) != HS_OK) goto fail;
  if ((st = dev_alloc(&p->resolve_counts, (size_t)L * R)) != HS_OK) goto fail;
  if ((st = hs_attn_workspace_init(p)) != HS_OK) goto fail;
  if (cudaEventCreateWithFlags(&p->order_event, cudaEventDisableTiming) != cudaSuccess) {
    p->order_event = nullptr;
    st = HS_ERR_CUDA;
    goto fail;
  }
  p->step_events = new (std::nothrow) cudaEvent_t[L + 1]();
  if (!p->step_events) {
    st = HS_ERR_OOM;
    goto fail;
  }
  for (int64_t i = 0; i <= L; ++i)
    if (cudaEventCreateWithFlags(&p->step_events[i], cudaEventDisableTiming) != cudaSuccess) {
      p->step_events[i] = nullptr;
      st = HS_ERR_CUDA;
      goto fail;
    }
  init_tables_kernel<<<64, 256>>>(p->page_table, R * d.max_pages, p->hot_block, d.num_requests,
                                  d.hot_slots / d.page_tokens, p->ctx_len, p->host_off);
  reset_kernel<<<256, 256>>>(p->slot_pos, p->slot_stamp, p->lru_order, L * R, d.hot_slots,
                             p->step, p->error_word);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    st = HS_ERR_CUDA;
    goto fail;
  }
  *out = p;
  return HS_OK;
fail:
  free_pool(p);
  return st;
}

extern "C" hs_status hs_pool_host_numa_node(const hs_pool* p, int32_t* node_out) {
  if (!p || !node_out) return HS_ERR_INVALID;
  *node_out = p->host_numa_node;
  return HS_OK;
}

extern "C" hs_status hs_pool_destroy(hs_pool* pool) {
  if (!pool) return HS_ERR_INVALID;
  cudaDeviceSynchronize();
  free_pool(pool);
  return HS_OK;
}

extern "C" hs_status hs_pool_get_views(const hs_pool* p, hs_pool_views* v) {
  if (!p || !v) return HS_ERR_INVALID;
  v->kv_pool = p->kv_pool;
  v->host_pool = p->host_pool;
  v->host_pool_device = p->host_pool_dev;
  v->page_table = p->page_table;
  v->ctx_len = p->ctx_len;
  v->host_off = p->host_off;
  v->hot_block = p->hot_block;
  v->slot_pos = p->slot_pos;
  v->slot_stamp = p->slot_stamp;
  v->lru_order = p->lru_order;
  v->step = p->step;
  v->error_word = p->error_word;
  v->blocks_per_layer = p->blocks_per_layer;
  v->kv_pool_bytes = (int64_t)p->kv_bytes;
  v->host_pool_bytes = (int64_t)p->host_bytes;
  return HS_OK;
}

extern "C" hs_status hs_pool_reset(hs_pool* p, void* stream) {
  if (!p) return HS_ERR_INVALID;
  const int64_t units = (int64_t)p->d.num_layers * p->d.num_requests;
  clear_inverse_kernel<<<256, 256, 0, hs_stream(stream)>>>(p->slot_pos, p->inv, p->host_off,
                                                           p->d.num_requests, p->d.hot_slots, units,
                                                           p->d.host_tokens);
  reset_kernel<<<256, 256, 0, hs_stream(stream)>>>(p->slot_pos, p->slot_stamp, p->lru_order,
                                                   units, p->d.hot_slots, p->step,
                                                   p->error_word);
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

extern "C" hs_status hs_set_request(hs_pool* p, int32_t req, int32_t ctx_len, int64_t host_off,
                                    void* stream) {
  if (!p || req < 0 || req >= p->d.num_requests || ctx_len < 0 || host_off < 0)
    return HS_ERR_INVALID;
  if ((int64_t)ctx_len > (int64_t)p->d.max_pages * p->d.page_tokens) return HS_ERR_INVALID;
  if (host_off + ctx_len > p->d.host_tokens) return HS_ERR_INVALID;
  set_request_kernel<<<1, 1, 0, hs_stream(stream)>>>(p->ctx_len, p->host_off, req, ctx_len,
                                                     host_off);
  p->host_off_mirror[req] = host_off;
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

extern "C" hs_status hs_map_page(hs_pool* p, int32_t req, int32_t page, int32_t block,
                                 void* stream) {
  if (!p || req < 0 || req >= p->d.num_requests || page < 0 || page >= p->d.max_pages)
    return HS_ERR_INVALID;
  if (block < -1 || (block >= 0 && (block < p->hot_blocks || block >= p->blocks_per_layer)))
    return HS_ERR_INVALID;
  set_i32_kernel<<<1, 1, 0, hs_stream(stream)>>>(
      p->page_table + (int64_t)req * p->d.max_pages + page, block);
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

extern "C" hs_status hs_load_page(hs_pool* p, int32_t req, int32_t page, int32_t block,
                                  void* stream) {
  if (!p || req < 0 || req >= p->d.num_requests || page < 0 || page >= p->d.max_pages)
    return HS_ERR_INVALID;
  if (block < p->hot_blocks || block >= p->blocks_per_layer) return HS_ERR_INVALID;
  const int64_t off = p->host_off_mirror[req];  // as last set by hs_set_request
  const int64_t P = p->d.page_tokens, RB = hs_row_bytes(p->d);
  if (off + (int64_t)(page + 1) * P > p->d.host_tokens) return HS_ERR_INVALID;
  const size_t bytes = (size_t)P * RB;
  for (int32_t l = 0; l < p->d.num_layers; ++l) {
    const char* src = static_cast<const char*>(p->host_pool) +
                      ((size_t)l * p->d.host_tokens + off + (size_t)page * P) * RB;
    char* dst = static_cast<char*>(p->kv_pool) +
                (((size_t)l * p->blocks_per_layer + block) * P) * RB;
    HS_CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, hs_stream(stream)));
  }
  return hs_map_page(p, req, page, block, stream);
}

extern "C" hs_status hs_step_advance(int32_t* d_step, void* stream) {
  if (!d_step) return HS_ERR_INVALID;
  step_advance_kernel<<<1, 1, 0, hs_stream(stream)>>>(d_step);
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

extern "C" hs_status hs_check_errors(hs_pool* p, int32_t* code_out) {
  if (!p) return HS_ERR_INVALID;
  HS_CUDA_TRY(cudaDeviceSynchronize());
  int32_t code = 0;
  HS_CUDA_TRY(cudaMemcpy(&code, p->error_word, sizeof(code), cudaMemcpyDeviceToHost));
  const int32_t zero = 0;
  HS_CUDA_TRY(cudaMemcpy(p->error_word, &zero, sizeof(zero), cudaMemcpyHostToDevice));
  if (code_out) *code_out = code;
  return code ? HS_ERR_DEVICE : HS_OK;
}

extern "C" const char* hs_status_string(hs_status s) {
  switch (s) {
    case HS_OK: return "HS_OK";
    case HS_ERR_INVALID: return "HS_ERR_INVALID: bad argument";
    case HS_ERR_CUDA: return "HS_ERR_CUDA: CUDA runtime call failed";
    case HS_ERR_OOM: return "HS_ERR_OOM: allocation failed";
    case HS_ERR_CAPACITY: return "HS_ERR_CAPACITY: more misses than free hot slots";
    case HS_ERR_DEVICE: return "HS_ERR_DEVICE: device error word set";
    case HS_ERR_TIMEOUT: return "HS_ERR_TIMEOUT: bounded wait gave up";
  }
  return "unknown hs_status";
}

extern "C" const char* hs_version(void) { return "libhs 0.1 (sm_103a)"; }
