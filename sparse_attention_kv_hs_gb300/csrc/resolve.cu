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
// The copies are bound by the host link and by how many host reads each SM
// keeps in flight, so a unit is served by a cluster of C CTAs (C = SMs /
// units, at most 8).  CTA 0 runs steps 1-4 for the whole selection; the
// others start the host reads of their share of the misses while CTA 0 is
// still choosing victims (see resolve_kernel), so the link does not wait for
// the metadata.
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
  // K is the length of a unit's list: T verify tokens' rows of ktok entries
  // each, token after token (T = 1 outside speculative decoding)
  int32_t ktok;
  int32_t sel_bits, kpt, bpt;
  int32_t copy_ctas;  // C: CTAs (a cluster) per unit
  int32_t smem_bytes; // dynamic shared memory per CTA (tables + staging)
  // A list longer than one CTA's tables runs as several launches over groups
  // of its tokens: this launch's K entries start at entry j_base of each
  // unit's list of list_stride entries; with `accumulate`, miss_count already
  // holds the earlier groups' misses (their log entries come first) and this
  // launch adds its own.
  int64_t list_stride;
  int32_t j_base, accumulate;
};

// Both layouts start with one mbarrier at offset 0, so each CTA of a cluster
// can address its peers' barrier without knowing their layout.
struct SmemPlan {
  size_t bar, order, sel, miss_j, miss_p, victim, hot, flag, warp, ptab, alias, total;
};

constexpr int kMaxSmemPages = 4096;  // page-table rows up to this width are staged in smem

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// ptab_pages: page-table entries staged (min(max_pages, kMaxSmemPages)).
__host__ __device__ inline SmemPlan smem_plan(int K, int B, int P, int sel_bits, int ptab_pages) {
  SmemPlan s;
  size_t o = 0;
  s.bar = o;       o = 16;
  s.order = o;     o = align16(o + sizeof(int32_t) * B);
  s.sel = o;       o = align16(o + sizeof(int32_t) * (size_t(1) << sel_bits));
  s.miss_j = o;    o = align16(o + sizeof(int32_t) * K);
  s.miss_p = o;    o = align16(o + sizeof(int32_t) * K);
  s.victim = o;    o = align16(o + sizeof(int32_t) * K);
  s.hot = o;       o = align16(o + sizeof(int32_t) * (B / P));
  s.flag = o;      o = align16(o + B);
  s.warp = o;      o = align16(o + sizeof(int32_t) * (kWarps + 8));
  s.ptab = o;      o = align16(o + sizeof(int32_t) * ptab_pages);
  s.alias = o;     o = align16(o + sizeof(uint32_t) * kThreads);
  s.total = o;
  return s;
}

// Fetch CTAs: their share's misses (j, position, destination row id), the
// scan scratch, then staging for as many rows as fit.
// With several verify tokens (dedup_bits > 0) a fetch CTA also holds its own
// selection hash, so that a position several tokens select is fetched once.
struct FetchPlan {
  size_t bar, j, p, dst, warp, sel, stage;
};

__host__ __device__ inline FetchPlan fetch_plan(int S, int dedup_bits) {
  FetchPlan f;
  size_t o = 0;
  f.bar = o;   o = 16;
  f.j = o;     o = align16(o + sizeof(int32_t) * S);
  f.p = o;     o = align16(o + sizeof(int32_t) * S);
  f.dst = o;   o = align16(o + sizeof(int32_t) * S);
  f.warp = o;  o = align16(o + sizeof(int32_t) * (kWarps + 8));
  const size_t hash = dedup_bits > 0 ? sizeof(int32_t) * (size_t(1) << dedup_bits) : 0;
  f.sel = o;   o = align16(o + hash);
  f.stage = o;
  return f;
}

constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait before giving up

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait (acquire, cluster scope) for phase `parity` of a local mbarrier
// that peers arrive on remotely; false after timeout_ns of the global timer.
__device__ __forceinline__ bool wait_peer_bar(uint32_t bar, uint32_t parity,
                                              uint64_t timeout_ns = kWaitNs) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (hs_ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 15) == 15) {
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > timeout_ns) {
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t hash_pos(int32_t p, int bits) {
  return ((uint32_t)p * 0x9E3779B1u) >> (32 - bits);
}

// Selection hash over a list (open addressing, linear probing): a slot holds
// the first index j of the list whose entry is the slot's position, or -1;
// the position itself is read back from the list.  Inserts may run
// concurrently; lookups run after every insert.
__device__ __forceinline__ void sel_insert(int32_t* slot, int bits, int32_t p, int j,
                                           const int32_t* list) {
  const int mask = (1 << bits) - 1;
  uint32_t h = hash_pos(p, bits);
  for (int probe = 0; probe <= mask; ++probe) {
    const int32_t prev = atomicCAS(&slot[h], -1, j);
    if (prev == -1) return;
    if (__ldg(list + prev) == p) {  // p's slot: keep the smallest j
      atomicMin(&slot[h], j);
      return;
    }
    h = (h + 1) & mask;
  }
}
// The first j whose entry is p, or -1.  `hint`: an index known to hold p (no
// list read when the slot holds it), or -1.
__device__ __forceinline__ int32_t sel_first(const int32_t* slot, int bits, int32_t p,
                                             const int32_t* list, int hint) {
  const int mask = (1 << bits) - 1;
  uint32_t h = hash_pos(p, bits);
  for (int probe = 0; probe <= mask; ++probe) {
    const int32_t v = slot[h];
    if (v < 0) return -1;
    if (v == hint || __ldg(list + v) == p) return v;
    h = (h + 1) & mask;
  }
  return -1;
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

// Copy rows from mapped pinned host memory into their pool rows: row i of the
// list goes from host row src(i) to pool row dst(i) (dst < 0: skip).  Each
// thread keeps kCopyUnroll 16-byte loads in flight before it stores them; the
// addresses are formed again for the stores rather than held in registers.
// hook() runs once per thread while its first loads are in flight (or at the
// end when it has none), for work that should overlap their latency.
template <typename SrcF, typename DstF, typename HookF>
__device__ __forceinline__ void copy_host_rows(const uint4* hsrc, uint4* kdst, int rv, int i_lo,
                                               int i_hi, SrcF src, DstF dst, HookF hook) {
  const int total = (i_hi - i_lo) * rv;
  bool hooked = false;
  for (int base = threadIdx.x; base < total; base += kThreads * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int c = base + u * kThreads;
      if (c < total) {
        const int i = i_lo + c / rv, e = c % rv;
        if (dst(i) >= 0) v[u] = __ldcs(hsrc + (int64_t)src(i) * rv + e);
      }
    }
    if (!hooked) {  // once, while the first loads are in flight
      hook();
      hooked = true;
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int c = base + u * kThreads;
      if (c < total) {
        const int i = i_lo + c / rv, e = c % rv;
        const int32_t row = dst(i);
        if (row >= 0) kdst[(int64_t)row * rv + e] = v[u];
      }
    }
  }
  if (!hooked) hook();
}

// Host rows i_lo .. i_hi-1 of a list -> shared-memory staging (row i at stage
// + i * rv * 16), kCopyUnroll 16-byte loads in flight per thread.  (Vector loads
// through registers: asynchronous cp.async copies from mapped host memory keep
// far fewer reads in flight per SM.)
template <typename SrcF>
__device__ __forceinline__ void stage_host_rows(const uint4* hsrc, unsigned char* stage, int rv,
                                                int i_lo, int i_hi, SrcF src) {
  uint4* st = reinterpret_cast<uint4*>(stage);
  const int total = i_hi * rv;
  for (int base = i_lo * rv + (int)threadIdx.x; base < total; base += kThreads * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int c = base + u * kThreads;
      if (c < total) {
        const int i = c / rv, e = c - i * rv;
        v[u] = __ldcs(hsrc + (int64_t)src(i) * rv + e);
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int c = base + u * kThreads;
      if (c < total) st[c] = v[u];
    }
  }
}

// Staged rows -> their pool rows.
template <typename DstF>
__device__ __forceinline__ void unstage_rows(const unsigned char* stage, uint4* kdst, int rv,
                                             int n, DstF dst) {
  for (int v = threadIdx.x; v < n * rv; v += kThreads) {
    const int i = v / rv, e = v - i * rv;
    const int32_t row = dst(i);
    if (row >= 0) kdst[(int64_t)row * rv + e] = reinterpret_cast<const uint4*>(stage)[v];
  }
}

// P_CT / RV_CT: compile-time page size and row width (16-byte vectors) for the
// common shapes (256, 72 = 576 bf16; 256, 41 = a 656-byte FP8 row); 0 = take
// them from the arguments (the row split c / rv then costs a division).
//
// A unit is served by a cluster of C CTAs.  CTA 0 ("metadata") runs steps 1-4
// for the whole selection.  With C > 1 the other C - 1 CTAs ("fetch") split
// the selection between them, classify their share themselves (page table and
// the position -> slot array answer "miss" without any unit-wide state; a
// repeated position is served by its first occurrence only, which CTA 0
// decides) and start the host reads of their misses into shared-memory
// staging at once, so the host link is busy while CTA 0 is still choosing
// victims.  Two signals, each a remote arrival on one mbarrier, order the
// phases: (1) each fetch CTA tells CTA 0 it has read the position -> slot
// array, which CTA 0 updates only after all have; (2) CTA 0 tells each fetch
// CTA that every miss's row id is written, which says where its staged rows
// go.  A fetch CTA waits for CTA 0 alone, never for another fetch CTA.  It
// stages rows only until (2) has arrived (checked after each round of loads)
// or its staging is full; the rest of its misses go straight from host memory
// to their slots after (2), the staged rows being written out while the first
// of those loads are in flight.  With C == 1, CTA 0 starts the host reads of a first
// small batch (one 16-byte load per thread, held in registers) before it
// chooses victims.
template <int P_CT, int RV_CT>
__global__ void __launch_bounds__(kThreads, 1) resolve_kernel(const ResolveArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x;
  const int C = a.copy_ctas;
  const uint32_t crank = C > 1 ? hs_ptx::cluster_ctarank() : 0u;
  const int r = blockIdx.x / C;
  const int li = blockIdx.y;               // layer index within this call
  const int l = a.layer_begin + li;        // absolute layer
  const int64_t unit = (int64_t)l * a.R + r;
  const int64_t call_unit = (int64_t)li * a.R + r;
  const int K = a.K, B = a.B, P = P_CT ? P_CT : a.P;
  const int rv = RV_CT ? RV_CT : a.row_vec;
  const int32_t* topk = a.topk + call_unit * a.list_stride + a.j_base;
  int32_t* out = a.out_rows + call_unit * a.list_stride + a.j_base;
  const int32_t* ptab = a.page_table + (int64_t)r * a.max_pages;
  int32_t* inv_u = a.inv + (int64_t)l * a.host_tokens + a.host_off[r];
  const uint4* hsrc = a.host_pool + ((int64_t)l * a.host_tokens + a.host_off[r]) * rv;
  uint4* kdst = a.kv_pool + (int64_t)l * a.blocks_per_layer * P * rv;
  const int32_t ctx = a.ctx_len[r];
  const int row_bytes = rv * 16;
  const uint32_t my_bar = hs_ptx::smem_u32(smem);  // offset 0 in both layouts
  if (C > 1) {
    if (tid == 0) {
      // CTA 0's barrier collects one arrival per fetch CTA; a fetch CTA's, one from CTA 0
      hs_ptx::mbar_init(my_bar, crank == 0 ? C - 1 : 1);
      hs_ptx::fence_mbar_init_cluster();
    }
    hs_ptx::cluster_sync();  // every barrier exists before any remote arrival
  }

  if (crank != 0) {
    // ======================= fetch CTA (C > 1) =======================
    const int F = C - 1, f = (int)crank - 1;
    const int S = (K + F - 1) / F;
    const int j_lo = f * S, j_hi = min(K, j_lo + S);
    const int kptf = (S + kThreads - 1) / kThreads;  // <= kpt <= 8
    const bool dedup = a.K != a.ktok;  // several verify tokens: fetch each position once
    const FetchPlan fp = fetch_plan(S, dedup ? a.sel_bits : 0);
    int32_t* f_j = reinterpret_cast<int32_t*>(smem + fp.j);
    int32_t* f_p = reinterpret_cast<int32_t*>(smem + fp.p);
    int32_t* f_dst = reinterpret_cast<int32_t*>(smem + fp.dst);
    int* s_warp = reinterpret_cast<int*>(smem + fp.warp);
    const int cap = (int)((a.smem_bytes - (int64_t)fp.stage) / row_bytes);

    int32_t* f_sel = reinterpret_cast<int32_t*>(smem + fp.sel);
    if (dedup) {  // the whole list's selection hash, as CTA 0 builds it
      for (int h = tid; h < (1 << a.sel_bits); h += kThreads) f_sel[h] = -1;
      __syncthreads();
      for (int j = tid; j < K; j += kThreads) {
        const int32_t p = topk[j];
        if (p >= 0 && p < ctx) sel_insert(f_sel, a.sel_bits, p, j, topk);
      }
      __syncthreads();
    }

    // classify this CTA's share: a miss is a valid position that is neither
    // resident nor in the hot buffer (with several tokens: at its first entry)
    const int j0 = j_lo + tid * kptf;
    int32_t my_p[8];
    uint32_t miss_mask = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + q;
      my_p[q] = -1;
      if (q >= kptf || j >= j_hi) continue;
      const int32_t p = topk[j];
      my_p[q] = p;
      if (p < 0 || p >= ctx) continue;
      if (ptab[p / P] >= 0) continue;
      if (inv_u[p] < 0) miss_mask |= 1u << q;
    }
    if (dedup) {  // a position an earlier entry selected is fetched for that entry only
      for (int q = 0; q < kptf; ++q)  // (topk re-read: no array indexed at run time)
        if ((miss_mask >> q) & 1u &&
            sel_first(f_sel, a.sel_bits, topk[j0 + q], topk, j0 + q) != j0 + q)
          miss_mask &= ~(1u << q);
    }
    int n_local;
    int mi = block_exclusive_scan(__popc(miss_mask), s_warp, &n_local);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (miss_mask & (1u << q)) {
        f_j[mi] = j0 + q;
        f_p[mi] = my_p[q];
        ++mi;
      }
    __syncthreads();
    // (1) this CTA is done reading the position -> slot array
    if (tid == 0) hs_ptx::mbar_arrive_remote(hs_ptx::mapa(my_bar, 0));
    // Host rows go to shared-memory staging one round of loads at a time
    // (kCopyUnroll per thread) only until CTA 0 has written the row ids (or the
    // staging is full); the rest go straight to their slots afterwards.
    int n_stage = 0;
    int* s_go = s_warp + kWarps + 1;
    for (;;) {
      const int n_next = min(n_local, min(cap, n_stage + kThreads * kCopyUnroll / rv));
      if (n_next <= n_stage) break;
      stage_host_rows(hsrc, smem + fp.stage, rv, n_stage, n_next, [&](int i) { return f_p[i]; });
      n_stage = n_next;
      if (tid == 0) *s_go = hs_ptx::mbar_test_wait_cluster(my_bar, 0) ? 1 : 0;
      __syncthreads();
      const bool go = *s_go != 0;
      __syncthreads();  // before thread 0 writes s_go again
      if (go) break;
    }
    // (2) CTA 0 has written the row id of every miss
    int* s_ok = s_warp + kWarps;
    if (tid < 32) {  // the whole warp polls, so that it sees the phase at once
      const bool got = wait_peer_bar(my_bar, 0);
      if (tid == 0) *s_ok = got ? 1 : 0;
    }
    __syncthreads();
    const bool ok = *s_ok != 0;
    if (ok) {
      for (int i = tid; i < n_local; i += kThreads) f_dst[i] = __ldcg(out + f_j[i]);
      __syncthreads();
      copy_host_rows(hsrc, kdst, rv, n_stage, n_local, [&](int i) { return f_p[i]; },
                     [&](int i) { return f_dst[i]; }, [&] {
                       unstage_rows(smem + fp.stage, kdst, rv, n_stage,
                                    [&](int i) { return f_dst[i]; });
                     });
    } else if (tid == 0) {
      atomicOr(a.error_word, HS_DEV_ERR_WAIT);
    }
    hs_ptx::cluster_sync();  // no CTA leaves while a peer may still address it
    return;
  }

  // ======================= metadata CTA =======================
  const bool ptab_in_smem = a.max_pages <= kMaxSmemPages;
  const SmemPlan sp = smem_plan(a.K, a.B, a.P, a.sel_bits, ptab_in_smem ? a.max_pages : 0);
  int32_t* s_order = reinterpret_cast<int32_t*>(smem + sp.order);
  int32_t* s_sel = reinterpret_cast<int32_t*>(smem + sp.sel);
  int32_t* s_miss_j = reinterpret_cast<int32_t*>(smem + sp.miss_j);
  int32_t* s_miss_p = reinterpret_cast<int32_t*>(smem + sp.miss_p);
  int32_t* s_victim = reinterpret_cast<int32_t*>(smem + sp.victim);
  int32_t* s_hot = reinterpret_cast<int32_t*>(smem + sp.hot);
  uint8_t* s_flag = smem + sp.flag;
  int* s_warp = reinterpret_cast<int*>(smem + sp.warp);
  int32_t* s_ptab = reinterpret_cast<int32_t*>(smem + sp.ptab);
  uint32_t* s_alias = reinterpret_cast<uint32_t*>(smem + sp.alias);
  int* s_err = s_warp + kWarps;
  const int hot_per_req = B / P;
  const int sel_mask = (1 << a.sel_bits) - 1;
  int32_t* g_slot_pos = a.slot_pos + unit * B;
  int32_t* g_stamp = a.slot_stamp + unit * B;
  int32_t* g_order = a.lru_order + unit * B;
  const int32_t step = *a.d_step;
  // earlier token groups' misses come first in the log and the count (read
  // here, before the block barriers that precede this launch's own count)
  const int32_t log_base = a.accumulate ? __ldcg(a.miss_count + call_unit) : 0;

  int err = 0;
  if (tid == 0) *s_err = 0;
  // ---- 0. load unit state, clear tables ---------------------------------
  // a slot already stamped with this step (a hit of a later token group, or a
  // slot an earlier group used) counts as used: it is no victim, and it moves
  // to the back of the order with this launch's hits and refills
  for (int s = tid; s < B; s += kThreads) {
    s_order[s] = g_order[s];
    s_flag[s] = g_stamp[s] == step ? 1 : 0;
  }
  for (int h = tid; h <= sel_mask; h += kThreads) s_sel[h] = -1;
  for (int i = tid; i < hot_per_req; i += kThreads)
    s_hot[i] = a.hot_block[(int64_t)r * hot_per_req + i];
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
    sel_insert(s_sel, a.sel_bits, p, j, topk);
  }
  __syncthreads();

  // ---- 2. classify; refresh hits ----------------------------------------
  uint32_t miss_mask = 0;
  uint32_t alias_mask = 0;  // repeats of a position an earlier verify token selected
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
    {  // first occurrence of p in the list?
      const int32_t first = sel_first(s_sel, a.sel_bits, p, topk, j);
      if (first != j) {
        if (first / a.ktok == j / a.ktok) {  // a repeat within one token's row
          err |= HS_DEV_ERR_DUPLICATE;
          out[j] = -1;
        } else {  // another token's position: its row, once served (below)
          alias_mask |= 1u << q;
        }
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

  s_alias[tid] = alias_mask;  // read back once the misses are served
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
  // Alone on the unit: start the host reads of a first batch of misses, one
  // 16-byte load per thread held in registers until the victims are known.
  int n_early = 0;
  uint4 early_v = make_uint4(0u, 0u, 0u, 0u);
  if (C == 1) {
    __syncthreads();  // s_miss_p complete
    n_early = min(n_miss_total, kThreads / rv);
    if (tid < n_early * rv) {
      const int i = tid / rv, e = tid - i * rv;
      early_v = __ldcs(hsrc + (int64_t)s_miss_p[i] * rv + e);
    }
  }

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
  int n_serve = n_miss_total < n_cand ? n_miss_total : n_cand;
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
  if (C > 1) {  // (1) every fetch CTA has read the position -> slot array
    if (tid < 32) {  // the whole warp polls, so that it sees the phase at once
      const bool got = wait_peer_bar(my_bar, 0);
      if (tid == 0) s_warp[kWarps + 1] = got ? 1 : 0;
    }
    __syncthreads();
    if (!s_warp[kWarps + 1]) {  // never updated under a reader: serve nothing
      err |= HS_DEV_ERR_WAIT;
      n_serve = 0;
    }
  }
  int32_t* log = a.miss_log ? a.miss_log + (call_unit * a.list_stride + log_base) * 3 : nullptr;
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
        log[3 * i + 0] = a.j_base + j;
        log[3 * i + 1] = p;
        log[3 * i + 2] = s;
      }
    } else {
      out[j] = -1;
    }
  }
  if (tid == 0 && a.miss_count) a.miss_count[call_unit] = log_base + n_serve;
  if (err) atomicOr(s_err, err);
  __syncthreads();
  if (tid == 0 && *s_err) atomicOr(a.error_word, *s_err);
  if (const uint32_t alias_mask = s_alias[tid]) {  // a later token's repeat: its first entry's row
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (alias_mask & (1u << q)) {
        const int j = j0 + q;
        out[j] = __ldcg(out + sel_first(s_sel, a.sel_bits, topk[j], topk, -1));
      }
  }

  if (C > 1) {  // (2) every miss's row id is written
    if (tid == 0)
      for (int c = 1; c < C; ++c) hs_ptx::mbar_arrive_remote(hs_ptx::mapa(my_bar, (uint32_t)c));
    hs_ptx::cluster_sync();  // no CTA leaves while a peer may still address it
    return;
  }
  // ---- 5. alone: copy the missed rows into their slots ------------------
  auto slot_row = [&](int i) -> int32_t {
    if (i >= n_serve) return -1;
    const int32_t s = s_victim[i];
    return s_hot[s / P] * P + s % P;
  };
  if (tid < n_early * rv) {
    const int i = tid / rv, e = tid - i * rv;
    const int32_t row = slot_row(i);
    if (row >= 0) kdst[(int64_t)row * rv + e] = early_v;
  }
  copy_host_rows(hsrc, kdst, rv, n_early, n_serve, [&](int i) { return s_miss_p[i]; }, slot_row,
                 [] {});
}

// Self-test of wait_peer_bar's time limit: one thread waits on a barrier of
// its CTA that nothing arrives on; *gave_up = 1 once the wait returns false.
__global__ void peer_wait_selftest_kernel(int32_t* gave_up, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) hs_ptx::mbar_init(hs_ptx::smem_u32(&bar), 1);
  __syncthreads();
  if (threadIdx.x == 0) *gave_up = wait_peer_bar(hs_ptx::smem_u32(&bar), 0, timeout_ns) ? 0 : 1;
}

int ceil_log2(int64_t x) {
  int b = 0;
  while ((int64_t(1) << b) < x) ++b;
  return b;
}

}  // namespace

hs_status hs_resolve_configure(int K, int B, int P, int max_pages, size_t* smem_bytes,
                               int max_clusters[4]) {
  const int sel_bits = ceil_log2(2 * (int64_t)K) < 5 ? 5 : ceil_log2(2 * (int64_t)K);
  const size_t tables =
      smem_plan(K, B, P, sel_bits, max_pages <= kMaxSmemPages ? max_pages : 0).total;
  int dev = 0, optin = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  HS_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  if (tables > (size_t)optin || fetch_plan(K, 0).stage > (size_t)optin)
    return HS_ERR_INVALID;  // K and B too large for one CTA
  // One CTA per SM either way (1024 threads): what the tables leave is staging.
  const size_t smem = (size_t)optin;
  *smem_bytes = smem;
  HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<256, 72>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<256, 41>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<0, 0>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  // How many clusters of 1, 2, 4 and 8 CTAs can run at once: a launch whose
  // clusters do not all fit runs in waves, so the launch picks a size that fits.
  int sms = 0, per_sm = 0;
  HS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  HS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, resolve_kernel<256, 72>,
                                                            kThreads, smem));
  max_clusters[0] = sms * per_sm;
  for (int i = 1; i < 4; ++i) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(1 << i) * 64u);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1u << i;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, resolve_kernel<256, 72>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    max_clusters[i] = n;
  }
  return HS_OK;
}

namespace {

// Before a list runs as several token groups: every hot hit of the whole list
// gets this step's stamp, so that no group takes another group's hit as a
// victim (the groups then resolve exactly as one launch over the whole list).
__global__ void __launch_bounds__(kThreads) protect_hits_kernel(const ResolveArgs a,
                                                                int32_t list_len) {
  const int r = blockIdx.x, li = blockIdx.y, l = a.layer_begin + li;
  const int64_t unit = (int64_t)l * a.R + r, call_unit = (int64_t)li * a.R + r;
  const int32_t* topk = a.topk + call_unit * a.list_stride;
  const int32_t* inv_u = a.inv + (int64_t)l * a.host_tokens + a.host_off[r];
  int32_t* g_stamp = a.slot_stamp + unit * a.B;
  const int32_t ctx = a.ctx_len[r], step = *a.d_step;
  for (int j = threadIdx.x; j < list_len; j += kThreads) {
    const int32_t p = topk[j];
    if (p < 0 || p >= ctx) continue;
    const int32_t slot = inv_u[p];
    if (slot >= 0) g_stamp[slot] = step;
  }
}

// RESOLVE of `num_tokens` verify tokens per unit (1 outside speculative
// decoding): the unit's list is their num_tokens * K entries, token after token.
hs_status launch_resolve(hs_pool* p, int32_t layer_begin, int32_t num_layers, int32_t num_tokens,
                         const int32_t* topk, const int32_t* d_step, int32_t* out_rows,
                         int32_t* miss_count, int32_t* miss_log, int max_cluster,
                         cudaStream_t stream) {
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
  a.ktok = p->d.top_k;
  a.B = p->d.hot_slots;
  a.P = p->d.page_tokens;
  a.max_pages = p->d.max_pages;
  a.row_vec = (int32_t)(hs_row_bytes(p->d) / 16);
  a.bpt = (a.B + kThreads - 1) / kThreads;
  if (a.bpt > 16) return HS_ERR_INVALID;
  // The kernel's dynamic shared-memory limit was raised by hs_pool_create
  // (hs_resolve_configure): nothing here may call outside the stream.
  const size_t smem = p->resolve_smem;
  const int ptab_pages = a.max_pages <= kMaxSmemPages ? a.max_pages : 0;
  // Tokens per launch: all of them when their list's tables fit one CTA (at
  // most 8 entries per thread, the tables and fetch lists in shared memory);
  // otherwise groups of the most tokens that fit, in token order.
  auto set_list = [&](int tokens) {
    a.K = tokens * a.ktok;
    a.sel_bits = ceil_log2(2 * (int64_t)a.K) < 5 ? 5 : ceil_log2(2 * (int64_t)a.K);
    a.kpt = (a.K + kThreads - 1) / kThreads;
  };
  auto fits = [&](int tokens) {
    set_list(tokens);
    if (a.kpt > 8) return false;
    return tokens == 1 || (smem_plan(a.K, a.B, a.P, a.sel_bits, ptab_pages).total <= smem &&
                           fetch_plan(a.K, a.sel_bits).stage <= smem);
  };
  int group = num_tokens;
  while (group >= 1 && !fits(group)) --group;
  if (group < 1) return HS_ERR_INVALID;
  a.list_stride = (int64_t)num_tokens * a.ktok;
  a.j_base = 0;
  a.accumulate = 0;
  a.smem_bytes = (int32_t)smem;
  // CTAs per unit: the largest cluster size (8, 4, 2) whose clusters, one per
  // unit, all run at once; else one CTA per unit
  const int64_t units = (int64_t)a.R * num_layers;
  int C = 1;
  for (int i = 3; i >= 1; --i)
    if ((max_cluster <= 0 || (1 << i) <= max_cluster) && units * (1 << i) <= p->num_sms &&
        units <= p->resolve_max_clusters[i]) {
      C = 1 << i;
      break;
    }
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
  auto launch = [&]() -> hs_status {
    if (a.P == 256 && a.row_vec == 72)  // bf16 [576] rows
      HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, resolve_kernel<256, 72>, a));
    else if (a.P == 256 && a.row_vec == 41)  // FP8 rows (656 bytes)
      HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, resolve_kernel<256, 41>, a));
    else
      HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, resolve_kernel<0, 0>, a));
    return HS_OK;
  };
  if (group == num_tokens) return launch();
  // Token groups, in order, after every hit of the whole list is stamped; the
  // miss count (the pool's scratch when the caller passes none) carries each
  // group's log offset to the next.
  if (!a.miss_count) a.miss_count = p->resolve_counts + (int64_t)layer_begin * a.R;
  protect_hits_kernel<<<dim3(a.R, num_layers), kThreads, 0, stream>>>(a, (int32_t)a.list_stride);
  HS_CUDA_TRY(cudaGetLastError());
  for (int t0 = 0; t0 < num_tokens; t0 += group) {
    set_list(num_tokens - t0 < group ? num_tokens - t0 : group);
    a.j_base = t0 * a.ktok;
    a.accumulate = t0 > 0 ? 1 : 0;
    const hs_status st = launch();
    if (st != HS_OK) return st;
  }
  return HS_OK;
}

}  // namespace

hs_status hs_launch_resolve(hs_pool* p, int32_t layer_begin, int32_t num_layers,
                            const int32_t* topk, const int32_t* d_step, int32_t* out_rows,
                            int32_t* miss_count, int32_t* miss_log, int max_cluster,
                            cudaStream_t stream) {
  return launch_resolve(p, layer_begin, num_layers, 1, topk, d_step, out_rows, miss_count,
                        miss_log, max_cluster, stream);
}

hs_status hs_launch_peer_wait_selftest(int32_t* gave_up, uint64_t timeout_ns,
                                       cudaStream_t stream) {
  peer_wait_selftest_kernel<<<1, 32, 0, stream>>>(gave_up, timeout_ns);
  HS_CUDA_TRY(cudaGetLastError());
  return HS_OK;
}

hs_status hs_launch_resolve_tokens(hs_pool* p, int32_t layer_begin, int32_t num_layers,
                                   int32_t num_tokens, const int32_t* topk, const int32_t* d_step,
                                   int32_t* out_rows, int32_t* miss_count, int32_t* miss_log,
                                   int max_cluster, cudaStream_t stream) {
  return launch_resolve(p, layer_begin, num_layers, num_tokens, topk, d_step, out_rows,
                        miss_count, miss_log, max_cluster, stream);
}

extern "C" hs_status hs_resolve(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                                const int32_t* topk_idx, const int32_t* d_step,
                                int32_t* out_row_ids, int32_t* miss_count, int32_t* miss_log,
                                void* stream) {
  if (!pool || !topk_idx || !d_step || !out_row_ids) return HS_ERR_INVALID;
  if (num_layers <= 0 || layer_begin < 0 || layer_begin + num_layers > pool->d.num_layers)
    return HS_ERR_INVALID;
  return hs_launch_resolve(pool, layer_begin, num_layers, topk_idx, d_step, out_row_ids,
                           miss_count, miss_log, 0, hs_stream(stream));
}

extern "C" hs_status hs_resolve_tokens(hs_pool* pool, int32_t layer_begin, int32_t num_layers,
                                       int32_t num_tokens, const int32_t* topk_idx,
                                       const int32_t* d_step, int32_t* out_row_ids,
                                       int32_t* miss_count, int32_t* miss_log, void* stream) {
  if (!pool || !topk_idx || !d_step || !out_row_ids || num_tokens <= 0) return HS_ERR_INVALID;
  if (num_layers <= 0 || layer_begin < 0 || layer_begin + num_layers > pool->d.num_layers)
    return HS_ERR_INVALID;
  return launch_resolve(pool, layer_begin, num_layers, num_tokens, topk_idx, d_step, out_row_ids,
                        miss_count, miss_log, 0, hs_stream(stream));
}
