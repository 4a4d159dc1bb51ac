// RESOLVE: logical top-K positions -> physical KV row ids, one CTA per
// (request, layer) unit, one launch per call.
//
// Page "59188saintaubert.com ... HiSparse", section 02: hit detection, LRU
// replacement, metadata update and host fetch fused in one kernel launched
// once per sparse layer; logical index in, physical slot out, like a
// software-managed TLB.  Page "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse
// Offloading in vLLM", section "How it works": resident tokens are read in
// place, hot tokens are read and their LRU entry refreshed, a miss copies a
// single row from pinned host memory into an LRU slot, and nothing on the
// decode path waits on a CPU decision (the step comes from device memory).
//
// Per unit, in shared memory:
//   1. selection hash (position -> first j) for repeat detection; hit
//      detection reads the pool's persistent position -> slot array (inv),
//      which misses keep up to date, so no per-call table is rebuilt;
//   2. classify each j: padding / error / resident / hot hit (stamp := step) /
//      miss; misses are numbered in j order by a block scan;
//   3. victims: lru_order lists the slots sorted by (stamp, slot).  Slots hit
//      in this step move to the back, so the victims are the first M entries
//      of lru_order that were not hit -- exactly "oldest stamp first, ties to
//      the lowest slot" among slots with stamp < step.  The new order is
//      (untouched non-victims, in old order) ++ (hit or refilled slots, by
//      slot number), which keeps lru_order sorted by (stamp, slot);
//   4. each miss writes slot_pos/stamp/out and its host row is copied from
//      mapped pinned host memory into the slot's pool row with 16-byte
//      vector loads and stores.
// The copies are bound by how many host reads are in flight, which is capped
// per SM, so a unit is served by a cluster of C CTAs (C = SMs / units, at most
// 8): CTA 0 runs steps 1-3 and 4's metadata, the others wait at a cluster
// barrier, fetch their share of the miss list from CTA 0's shared memory and
// every CTA copies its share of the rows.
#include "hs_internal.cuh"
#include "sm100_ptx.cuh"

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCopyUnroll = 8;

struct ResolveArgs {
  const int32_t* topk;
  const int32_t* d_step;
  int32_t* out_rows;
  int32_t* miss_count;
  int32_t* miss_log;
  const int32_t* page_table;
  const int32_t* ctx_len;
  const int64_t* host_off;
  const int32_t* hot_block;
  int32_t* slot_pos;
  int32_t* slot_stamp;
  int32_t* lru_order;
  int32_t* inv;  // [L][host_tokens]: slot holding host row (host_off[r] + p), or -1
  const uint4* host_pool;
  uint4* kv_pool;
  int32_t* error_word;
  int64_t host_tokens;
  int64_t blocks_per_layer;
  int32_t layer_begin, R, K, B, P, max_pages, row_vec;
  int32_t sel_bits, kpt, bpt;
  int32_t copy_ctas;  // C: CTAs (a cluster) per unit
};

struct SmemPlan {
  size_t order, sel_key, sel_j, miss_j, miss_p, victim, hot, flag, warp, ptab, total;
};

constexpr int kMaxSmemPages = 4096;  // page-table rows up to this width are staged in smem

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline SmemPlan smem_plan(int K, int B, int P, int sel_bits) {
  SmemPlan s;
  size_t o = 0;
  s.order = o;     o = align16(o + sizeof(int32_t) * B);
  s.sel_key = o;   o = align16(o + sizeof(int32_t) * (size_t(1) << sel_bits));
  s.sel_j = o;     o = align16(o + sizeof(int32_t) * (size_t(1) << sel_bits));
  s.miss_j = o;    o = align16(o + sizeof(int32_t) * K);
  s.miss_p = o;    o = align16(o + sizeof(int32_t) * K);
  s.victim = o;    o = align16(o + sizeof(int32_t) * K);
  s.hot = o;       o = align16(o + sizeof(int32_t) * (B / P));
  s.flag = o;      o = align16(o + B);
  s.warp = o;      o = align16(o + sizeof(int32_t) * (kWarps + 8));
  s.ptab = o;      o = align16(o + sizeof(int32_t) * kMaxSmemPages);
  s.total = o;
  return s;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t hash_pos(int32_t p, int bits) {
  return ((uint32_t)p * 0x9E3779B1u) >> (32 - bits);
}

// Exclusive scan of one value per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive per-warp prefix
  }
  __syncthreads();
  const int base = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[kWarps - 1];
  __syncthreads();  // s_warp is reused by the next scan
  return base + x - v;
}

// P_CT / RV_CT: compile-time page size and row width (16-byte vectors) for the
// common shape (256, 72 = 576 bf16); 0 = take them from the arguments.
template <int P_CT, int RV_CT>
__global__ void __launch_bounds__(kThreads, 1) resolve_kernel(const ResolveArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const SmemPlan sp = smem_plan(a.K, a.B, a.P, a.sel_bits);
  int32_t* s_order = reinterpret_cast<int32_t*>(smem + sp.order);
  int32_t* s_sel_key = reinterpret_cast<int32_t*>(smem + sp.sel_key);
  int32_t* s_sel_j = reinterpret_cast<int32_t*>(smem + sp.sel_j);
  int32_t* s_miss_j = reinterpret_cast<int32_t*>(smem + sp.miss_j);
  int32_t* s_miss_p = reinterpret_cast<int32_t*>(smem + sp.miss_p);
  int32_t* s_victim = reinterpret_cast<int32_t*>(smem + sp.victim);
  int32_t* s_hot = reinterpret_cast<int32_t*>(smem + sp.hot);
  uint8_t* s_flag = smem + sp.flag;
  int* s_warp = reinterpret_cast<int*>(smem + sp.warp);
  int32_t* s_ptab = reinterpret_cast<int32_t*>(smem + sp.ptab);
  int* s_err = s_warp + kWarps;

  const int tid = threadIdx.x;
  const int C = a.copy_ctas;
  const uint32_t crank = C > 1 ? hs_ptx::cluster_ctarank() : 0u;
  const int r = blockIdx.x / C;
  const int li = blockIdx.y;               // layer index within this call
  const int l = a.layer_begin + li;        // absolute layer
  const int64_t unit = (int64_t)l * a.R + r;
  const int64_t call_unit = (int64_t)li * a.R + r;
  const int K = a.K, B = a.B, P = P_CT ? P_CT : a.P;
  const int hot_per_req = B / P;
  const int sel_mask = (1 << a.sel_bits) - 1;

  const int32_t* topk = a.topk + call_unit * K;
  int32_t* out = a.out_rows + call_unit * K;
  int32_t* g_slot_pos = a.slot_pos + unit * B;
  int32_t* g_stamp = a.slot_stamp + unit * B;
  int32_t* g_order = a.lru_order + unit * B;
  const int32_t* ptab = a.page_table + (int64_t)r * a.max_pages;

  const int32_t step = *a.d_step;
  const int32_t ctx = a.ctx_len[r];

  int err = 0;
  int n_serve = 0;
  if (tid == 0) *s_err = 0;
  if (crank == 0) {
  // ---- 0. load unit state, clear tables ---------------------------------
  int32_t* inv_u = a.inv + (int64_t)l * a.host_tokens + a.host_off[r];
  for (int s = tid; s < B; s += kThreads) {
    s_order[s] = g_order[s];
    s_flag[s] = 0;
  }
  for (int h = tid; h <= sel_mask; h += kThreads) {
    s_sel_key[h] = -1;
    s_sel_j[h] = INT32_MAX;
  }
  for (int i = tid; i < hot_per_req; i += kThreads)
    s_hot[i] = a.hot_block[(int64_t)r * hot_per_req + i];
  const bool ptab_in_smem = a.max_pages <= kMaxSmemPages;
  if (ptab_in_smem)
    for (int i = tid; i < a.max_pages; i += kThreads) s_ptab[i] = ptab[i];
  __syncthreads();

  // ---- 1. build the selection hash ---------------------------------------
  const int j0 = tid * a.kpt;
  int32_t my_p[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int j = j0 + q;
    my_p[q] = (q < a.kpt && j < K) ? topk[j] : -1;
    const int32_t p = my_p[q];
    if (q >= a.kpt || j >= K || p < 0 || p >= ctx) continue;
    uint32_t h = hash_pos(p, a.sel_bits);
    for (int probe = 0; probe <= sel_mask; ++probe) {
      const int32_t prev = atomicCAS(&s_sel_key[h], -1, p);
      if (prev == -1 || prev == p) {
        atomicMin(&s_sel_j[h], j);
        break;
      }
      h = (h + 1) & sel_mask;
    }
  }
  __syncthreads();

  // ---- 2. classify; refresh hits ----------------------------------------
  uint32_t miss_mask = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int j = j0 + q;
    if (q >= a.kpt || j >= K) continue;
    const int32_t p = my_p[q];
    int32_t row = -1;
    if (p == -1) {
      out[j] = -1;  // padding
      continue;
    }
    if (p < 0 || p >= ctx) {
      err |= HS_DEV_ERR_RANGE;
      out[j] = -1;
      continue;
    }
    {  // first occurrence of p in this row?
      uint32_t h = hash_pos(p, a.sel_bits);
      int32_t first = -1;
      for (int probe = 0; probe <= sel_mask; ++probe) {
        if (s_sel_key[h] == p) {
          first = s_sel_j[h];
          break;
        }
        h = (h + 1) & sel_mask;
      }
      if (first != j) {
        err |= HS_DEV_ERR_DUPLICATE;
        out[j] = -1;
        continue;
      }
    }
    const int32_t blk = ptab_in_smem ? s_ptab[p / P] : ptab[p / P];
    if (blk >= 0) {  // resident page: read in place, LRU untouched
      if (blk >= a.blocks_per_layer) {
        err |= HS_DEV_ERR_BLOCK;
      } else {
        row = blk * P + p % P;
      }
      out[j] = row;
      continue;
    }
    const int32_t slot = inv_u[p];  // hot slot holding p, or -1
    if (slot >= 0) {  // hot hit: refresh the LRU entry
      s_flag[slot] = 1;
      g_stamp[slot] = step;
      out[j] = s_hot[slot / P] * P + slot % P;
    } else {
      miss_mask |= 1u << q;  // host only: a miss, served below
    }
  }

  // misses numbered in selection (j) order
  int n_miss_total;
  const int my_misses = __popc(miss_mask);
  int mi = block_exclusive_scan(my_misses, s_warp, &n_miss_total);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (miss_mask & (1u << q)) {
      s_miss_j[mi] = j0 + q;
      s_miss_p[mi] = my_p[q];
      ++mi;
    }
  // (the scan's trailing barrier also publishes s_flag from step 2)

  // ---- 3. victims: untouched slots in (stamp, slot) order ---------------
  const int i0 = tid * a.bpt;
  uint32_t cand_mask = 0;
#pragma unroll 4
  for (int q = 0; q < 16; ++q) {
    const int i = i0 + q;
    if (q < a.bpt && i < B && s_flag[s_order[i]] == 0) cand_mask |= 1u << q;
  }
  int n_cand;
  int rank = block_exclusive_scan(__popc(cand_mask), s_warp, &n_cand);
  n_serve = n_miss_total < n_cand ? n_miss_total : n_cand;
  if (n_miss_total > n_cand) err |= HS_DEV_ERR_CAPACITY;
#pragma unroll 4
  for (int q = 0; q < 16; ++q) {
    if (!(cand_mask & (1u << q))) continue;
    const int32_t s = s_order[i0 + q];
    if (rank < n_serve) {
      s_victim[rank] = s;
      s_flag[s] = 2;
    } else {
      g_order[rank - n_serve] = s;  // untouched, kept: first part of the new order
    }
    ++rank;
  }
  __syncthreads();

  // new order, second part: every slot used in this step, by slot number
  uint32_t used_mask = 0;
#pragma unroll 4
  for (int q = 0; q < 16; ++q) {
    const int s = i0 + q;
    if (q < a.bpt && s < B && s_flag[s] != 0) used_mask |= 1u << q;
  }
  int n_used;
  int upos = block_exclusive_scan(__popc(used_mask), s_warp, &n_used);
  const int kept = n_cand - n_serve;
#pragma unroll 4
  for (int q = 0; q < 16; ++q)
    if (used_mask & (1u << q)) g_order[kept + upos++] = i0 + q;

  // ---- 4. serve misses: metadata, row ids, log --------------------------
  int32_t* log = a.miss_log ? a.miss_log + call_unit * (int64_t)K * 3 : nullptr;
  for (int i = tid; i < n_miss_total; i += kThreads) {
    const int j = s_miss_j[i];
    if (i < n_serve) {
      const int32_t s = s_victim[i], p = s_miss_p[i];
      const int32_t old = g_slot_pos[s];
      if (old >= 0) inv_u[old] = -1;  // evicted (distinct from every missed position)
      inv_u[p] = s;
      g_slot_pos[s] = p;
      g_stamp[s] = step;
      out[j] = s_hot[s / P] * P + s % P;
      if (log) {
        log[3 * i + 0] = j;
        log[3 * i + 1] = p;
        log[3 * i + 2] = s;
      }
    } else {
      out[j] = -1;
    }
  }

  }  // end of CTA 0's metadata work

  // ---- 5. copy missed rows: mapped pinned host -> hot slot in HBM --------
  int* s_nserve = s_warp + kWarps + 1;
  if (C > 1) {
    if (crank == 0 && tid == 0) *s_nserve = n_serve;
    hs_ptx::cluster_sync();  // CTA 0's miss list and hot blocks are complete
    if (crank != 0) {
      auto peer = [&](const void* p) { return hs_ptx::mapa(hs_ptx::smem_u32(p), 0); };
      n_serve = (int)ld_cluster_u32(peer(s_nserve));
      const int lo = (int)((int64_t)n_serve * crank / C), hi = (int)((int64_t)n_serve * (crank + 1) / C);
      for (int i = lo + tid; i < hi; i += kThreads) {
        s_miss_p[i] = (int32_t)ld_cluster_u32(peer(s_miss_p + i));
        s_victim[i] = (int32_t)ld_cluster_u32(peer(s_victim + i));
      }
      for (int i = tid; i < hot_per_req; i += kThreads)
        s_hot[i] = (int32_t)ld_cluster_u32(peer(s_hot + i));
    }
    __syncthreads();
    hs_ptx::cluster_sync();  // every CTA holds its share: CTA 0 may run ahead and exit
  }
  const int i_lo = (int)((int64_t)n_serve * crank / C);
  const int i_hi = (int)((int64_t)n_serve * (crank + 1) / C);
  const int rv = RV_CT ? RV_CT : a.row_vec;
  const uint4* hsrc = a.host_pool + ((int64_t)l * a.host_tokens + a.host_off[r]) * rv;
  uint4* kdst = a.kv_pool + (int64_t)l * a.blocks_per_layer * P * rv;
  const int64_t total = (int64_t)(i_hi - i_lo) * rv;
  for (int64_t base = tid; base < total; base += (int64_t)kThreads * kCopyUnroll) {
    uint4 v[kCopyUnroll];
    int64_t dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = base + (int64_t)u * kThreads;
      dst[u] = -1;
      if (c < total) {
        const int ii = (int)(c / rv);
        const int e = (int)(c - (int64_t)ii * rv);
        const int i = i_lo + ii;
        const int32_t s = s_victim[i];
        v[u] = __ldcs(hsrc + (int64_t)s_miss_p[i] * rv + e);
        dst[u] = ((int64_t)s_hot[s / P] * P + s % P) * rv + e;
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u] >= 0) kdst[dst[u]] = v[u];
  }

  if (crank == 0 && tid == 0 && a.miss_count) a.miss_count[call_unit] = n_serve;
  if (err) atomicOr(s_err, err);
  __syncthreads();
  if (tid == 0 && *s_err) atomicOr(a.error_word, *s_err);
}

int ceil_log2(int64_t x) {
  int b = 0;
  while ((int64_t(1) << b) < x) ++b;
  return b;
}

}  // namespace

hs_status hs_resolve_configure(int K, int B, int P, size_t* smem_bytes) {
  const int sel_bits = ceil_log2(2 * (int64_t)K) < 5 ? 5 : ceil_log2(2 * (int64_t)K);
  const size_t smem = smem_plan(K, B, P, sel_bits).total;
  *smem_bytes = smem;
  int dev = 0, optin = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  if (smem > (size_t)optin) return HS_ERR_INVALID;  // K and B too large for one CTA
  HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<256, 72>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<0, 0>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  return HS_OK;
}

hs_status hs_launch_resolve(hs_pool* p, int32_t layer_begin, int32_t num_layers,
                            const int32_t* topk, const int32_t* d_step, int32_t* out_rows,
                            int32_t* miss_count, int32_t* miss_log, cudaStream_t stream) {
  ResolveArgs a;
  a.topk = topk;
  a.d_step = d_step;
  a.out_rows = out_rows;
  a.miss_count = miss_count;
  a.miss_log = miss_log;
  a.page_table = p->page_table;
  a.ctx_len = p->ctx_len;
  a.host_off = p->host_off;
  a.hot_block = p->hot_block;
  a.slot_pos = p->slot_pos;
  a.slot_stamp = p->slot_stamp;
  a.lru_order = p->lru_order;
  a.inv = p->inv;
  a.host_pool = static_cast<const uint4*>(p->host_pool_dev);
  a.kv_pool = static_cast<uint4*>(p->kv_pool);
  a.error_word = p->error_word;
  a.host_tokens = p->d.host_tokens;
  a.blocks_per_layer = p->blocks_per_layer;
  a.layer_begin = layer_begin;
  a.R = p->d.num_requests;
  a.K = p->d.top_k;
  a.B = p->d.hot_slots;
  a.P = p->d.page_tokens;
  a.max_pages = p->d.max_pages;
  a.row_vec = p->d.row_elems / 8;
  a.sel_bits = ceil_log2(2 * (int64_t)a.K) < 5 ? 5 : ceil_log2(2 * (int64_t)a.K);
  a.kpt = (a.K + kThreads - 1) / kThreads;
  a.bpt = (a.B + kThreads - 1) / kThreads;
  if (a.kpt > 8 || a.bpt > 16) return HS_ERR_INVALID;
  // The kernel's dynamic shared-memory limit was raised by hs_pool_create
  // (hs_resolve_configure): nothing here may call outside the stream.
  const size_t smem = smem_plan(a.K, a.B, a.P, a.sel_bits).total;
  // copy helpers per unit: enough CTAs to put every SM to work on the copies
  int C = p->num_sms / (a.R * num_layers);
  C = C >= 8 ? 8 : C >= 4 ? 4 : C >= 2 ? 2 : 1;
  a.copy_ctas = C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.R * C, num_layers);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = C > 1 ? 1 : 0;
  if (a.P == 256 && a.row_vec == 72)
    HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, resolve_kernel<256, 72>, a));
  else
    HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, resolve_kernel<0, 0>, a));
  return HS_OK;
}

extern "C" hs_status hs_resolve(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                                const int32_t* topk_idx, const int32_t* d_step,
                                int32_t* out_row_ids, int32_t* miss_count, int32_t* miss_log,
                                void* stream) {
  if (!pool || !topk_idx || !d_step || !out_row_ids) return HS_ERR_INVALID;
  if (num_layers <= 0 || layer_begin < 0 || layer_begin + num_layers > pool->d.num_layers)
    return HS_ERR_INVALID;
  return hs_launch_resolve(pool, layer_begin, num_layers, topk_idx, d_step, out_row_ids,
                           miss_count, miss_log, hs_stream(stream));
}
