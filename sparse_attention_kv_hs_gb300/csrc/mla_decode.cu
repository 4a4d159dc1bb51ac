// Sparse MLA decode attention over the K rows RESOLVE handed out, on the
// sm_100-family tensor cores (tcgen05, fp32 accumulators in tensor memory).
//
// What it computes (absorbed MLA decode; the sparse MLA kernel of page "GLM
// 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM", section "How
// it works", reads hot-buffer and resident rows alike by row id): for each
// request r and head h < 128,
//   s_j = scale * q[h] . kv(row_ids[r][j])            (576-wide rows)
//   out[h] = sum_j softmax(s)_j * kv(row_ids[r][j])[0:512]
// over the j with a valid row id.
//
// Work split.  The fp32 output accumulator O (128 heads x 512) fills a whole
// SM's tensor memory, so each (request, split-of-K) is handled by a CTA pair
// (a cluster of 2):
//   CTA 0 ("score"): Q lives in tensor memory (the A operand); 64-row KV
//     tiles are gathered by TMA (tile::gather4, 4 rows per instruction, 128B
//     swizzle); S = Q K^T (M=128, N=64, K=576) goes to a double-buffered TMEM
//     accumulator; 4 warps run the online softmax (one thread per head) and
//     write P as two bf16 parts (hi + lo, so P carries ~16 bits: bf16 P alone
//     would cost ~1e-3 relative error), which one bulk copy sends into CTA 1.
//   CTA 1 ("value"): gathers the V part (first 512 columns) of the same rows
//     the same way and accumulates O += P_hi V + P_lo V (M=128, N=256 x 2, V
//     as an MN-major operand).  Its 4 epilogue warps rescale O when the
//     running max moved (lazily: only when it grew by more than 2^8, so the
//     rescale is rare and off the common path) and write the normalised output.
// Q reaches CTA 0 by TMA (swizzled, then TMEM), each split's row ids are staged
// in shared memory once, MMA descriptors are computed once and advanced by
// constants, and every hand-off is an mbarrier.  With several splits per
// request, each pair writes a normalised fp32 partial and its log-sum-exp; a
// small merge kernel combines them.
//
// Every wait is bounded: a wait that times out sets HS_DEV_ERR_WAIT in the
// pool's error word and the CTA winds down (no further MMAs), frees its tensor
// memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>

#include <new>

#include "hs_internal.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace hs_ptx;

constexpr int kHeads = 128;        // MMA M (heads, zero-padded)
constexpr int kD = 576;            // row width (latent 512 + rope 64)
constexpr int kDV = 512;           // value width
constexpr int kTile = 64;          // KV rows per tile
constexpr int kStages = 2;         // KV tile ring depth
constexpr int kThreads = 384;
constexpr int kLoadWarps = 7;      // warps 1..7 issue the TMA row gathers
constexpr int kMathWarp0 = 8;      // warps 8..11: softmax (CTA 0) / rescale + epilogue (CTA 1)
constexpr int kCbK = kD / 64;      // 9 swizzled 128-byte column blocks per K row
constexpr int kCbV = kDV / 64;     // 8 for V

constexpr uint32_t kBlockBytes = kTile * 128;              // one column block of a tile: 8192
constexpr uint32_t kStageBytes = kCbK * kBlockBytes;       // 73728
constexpr uint32_t kQBlockBytes = kHeads * 128;            // 16384
constexpr uint32_t kPBytes = kHeads * kTile * 2;           // 16384 per part
constexpr uint32_t kPMetaBytes = 528;                      // alpha[128] floats + 4 flag words
constexpr uint32_t kPCopyBytes = 2 * kPBytes + kPMetaBytes;    // 33296 (multiple of 16)
constexpr uint32_t kPBufBytes = 2 * kPBytes + 1024;        // 33792

// Shared-memory layout, identical offsets in both CTAs of a pair (the bulk
// copy and remote barrier operations address the peer by offset).  Swizzled
// regions are 1024-byte aligned.
constexpr int kMaxSplitRows = 2048;  // row ids of one split, staged in shared memory
constexpr uint32_t OFF_STAGE = 0;    // CTA 0 first holds Q here (9 x 16384 B)
constexpr uint32_t OFF_P = OFF_STAGE + kStages * kStageBytes;  // 147456
constexpr uint32_t OFF_ML = OFF_P + 2 * kPBufBytes;            // 215040: m[128], l[128]
constexpr uint32_t OFF_RID = OFF_ML + 1024;                    // 216064: int32 [2048]
constexpr uint32_t OFF_BAR = OFF_RID + 4 * kMaxSplitRows;      // 224256
constexpr uint32_t OFF_MISC = OFF_BAR + 256;
constexpr uint32_t kSmemBytes = OFF_MISC + 64;                 // 224576
static_assert(kCbK * kQBlockBytes <= kStages * kStageBytes, "Q must fit the stage region");

// barrier indices (8 bytes each at OFF_BAR)
enum {
  B_KV_FULL = 0,     // [2] TMA complete_tx -> MMA (both CTAs: K tile / V tile)
  B_KV_EMPTY = 2,    // [2] MMA commit -> loaders
  B_S_FULL = 4,      // [2] score MMA commit -> softmax
  B_S_EMPTY = 6,     // [2] softmax -> score MMA
  B_P_EMPTY = 8,     // [2] (CTA 0) value MMA commit (multicast) -> softmax
  B_Q_SMEM = 10,     // (CTA 0) TMA of Q landed in shared memory
  B_Q_READY = 11,    // (CTA 0) softmax warps put Q in TMEM -> score MMA, loader
  B_P_FULL = 12,     // [2] (CTA 1) bulk copy complete_tx -> value MMA
  B_RID = 14,        // loader warp staged this split's row ids
  B_CORR_REQ = 15,   // (CTA 1) value MMA -> rescale warps
  B_CORR_DONE = 16,  // (CTA 1) rescale warps -> value MMA
  B_MMA_IDLE = 17,   // (CTA 1) commit: earlier P.V MMAs finished
  B_ML_FULL = 18,    // (CTA 1) softmax's final m, l -> epilogue
  B_FINAL = 19,      // MMA issuer's last commit
  B_P_READY = 20,    // [2] (CTA 0) softmax threads wrote P -> bulk-copy issuer
  B_COUNT = 22
};
static_assert(B_COUNT * 8 <= 256, "barrier area");

// TMEM columns
constexpr uint32_t TM_Q = 0;     // CTA 0: Q, 288 columns (bf16 pairs)
constexpr uint32_t TM_S = 288;   // CTA 0: S, 2 x 64 columns
constexpr uint32_t TM_O = 0;     // CTA 1: O, 512 columns

constexpr uint32_t kIdescS = idesc_bf16(128, kTile, false, false);  // A (TMEM), B K-major
constexpr uint32_t kIdescPV = idesc_bf16(128, 256, false, true);    // A K-major, B MN-major

constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait before giving up

struct AttnArgs {
  const int32_t* row_ids;   // [R][K]
  uint16_t* out;            // [R][H][512] bf16 (splits == 1)
  float* lse;               // [R][H] or null (splits == 1)
  float* ws_o;              // [R][splits][128][512] (splits > 1)
  float* ws_lse;            // [R][splits][128]
  int32_t* error_word;
  int32_t rows_in_layer;    // also the out-of-range row coordinate (TMA fills zeros)
  int32_t K, H, splits, rows_per_split;
  float scale_log2;         // scale * log2(e)
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on a local mbarrier; on timeout (or if the CTA is already
// aborting) returns false and raises the abort flag.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* error_word, bool cluster_scope = false) {
  if (*abort) return false;
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    const bool ok = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (ok) return true;
    if ((i & 63) == 63) {
      if (*abort) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitNs) {
        *abort = 1;
        atomicOr(error_word, HS_DEV_ERR_WAIT);
        return false;
      }
    }
  }
}

// Same, for roles run by whole warps: every lane gets the same answer, so
// warp-collective tcgen05 instructions after it are executed uniformly.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort,
                                              int32_t* error_word, bool cluster_scope = false) {
  const bool ok = wait_bar(bar, parity, abort, error_word, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}

// 2^x (hardware approximation, relative error ~2^-22; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Shared-memory descriptor of a 128B-swizzled operand (atoms of 8 rows x 128 B).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(addr, lbo, sbo) | ((uint64_t)2 << 61);
}

// TMA: 4 rows (y0..y3) x 64 columns from x, into 512 swizzled bytes at dst.
// A row coordinate past the tensor reads zeros.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0,
                                            int y1, int y2, int y3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
      : "memory");
}
// (unused: both CTAs gather their own rows, see the loader role)
// Same 4 rows, delivered to the same shared-memory offset (and completing
// bytes on the same barrier offset) in every CTA of cta_mask.
__device__ __forceinline__ void tma_gather4_mc(uint32_t dst, const CUtensorMap* map, int x, int y0,
                                               int y1, int y2, int y3, uint32_t bar,
                                               uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar),
      "h"(cta_mask)
      : "memory");
}
// TMA: one box (64 columns x box rows) from (x, y) into dst.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map,
                      const __grid_constant__ CUtensorMap q_map, const AttnArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* corr_tile = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
  volatile int* corr_exit = reinterpret_cast<volatile int*>(smem + OFF_MISC + 12);
  int32_t* s_rid = reinterpret_cast<int32_t*>(smem + OFF_RID);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int split = blockIdx.x >> 1;
  const int r = blockIdx.y;
  const int j_begin = split * a.rows_per_split;
  int j_end = j_begin + a.rows_per_split;
  if (j_end > a.K) j_end = a.K;
  const int n_tiles = j_end > j_begin ? (j_end - j_begin + kTile - 1) / kTile : 0;

  // ---- set-up: barriers, tensor memory ---------------------------------
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_KV_FULL + i), 1);
      mbar_init(bar(B_KV_EMPTY + i), 1);
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_S_EMPTY + i), 128);
      mbar_init(bar(B_P_EMPTY + i), 1);
      mbar_init(bar(B_P_FULL + i), 1);
      mbar_init(bar(B_P_READY + i), 128);
    }
    mbar_init(bar(B_Q_SMEM), 1);
    mbar_init(bar(B_Q_READY), 128);
    mbar_init(bar(B_RID), 32);
    mbar_init(bar(B_CORR_REQ), 1);
    mbar_init(bar(B_CORR_DONE), 128);
    mbar_init(bar(B_MMA_IDLE), 1);
    mbar_init(bar(B_ML_FULL), 128);
    mbar_init(bar(B_FINAL), 1);
    // swizzled TMA destinations and descriptors assume a 1024-byte aligned base
    *abort_flag = (sbase & 1023u) ? 1 : 0;
    if (sbase & 1023u) atomicOr(a.error_word, HS_DEV_ERR_INTERNAL);
    *corr_tile = 0;
    *corr_exit = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote operation
  const uint32_t tm = *tmem_holder;
  int err = 0;

  if (warp >= 1 && warp <= kLoadWarps) {
    // ================= loader warps (both CTAs): TMA issue =================
    // Each CTA gathers its own copy of the rows (CTA 0: all 9 column blocks,
    // CTA 1: the 8 value blocks), so a stage is released by that CTA's MMA
    // alone.  The row gathers are spread over 7 warps: TMA issue throughput
    // grows with the number of issuing warps.
    const int lw = warp - 1;
    if (rank == 0 && lw == 0 && lane == 0 && !*abort_flag) {  // Q[r] (128 rows) -> smem
      mbar_arrive_expect_tx(bar(B_Q_SMEM), kCbK * kQBlockBytes);
      for (int cb = 0; cb < kCbK; ++cb)
        tma_load_2d(sbase + OFF_STAGE + cb * kQBlockBytes, &q_map, cb * 64, r * a.H,
                    bar(B_Q_SMEM));
    }
    if (lw == 0) {  // this split's row ids -> shared memory, validated once (-1 = no row)
      const int32_t* g_rows = a.row_ids + (int64_t)r * a.K;
      for (int i = lane; i < n_tiles * kTile; i += 32) {
        const int j = j_begin + i;
        int32_t v = j < j_end ? __ldg(g_rows + j) : -1;
        if (v < -1 || v >= a.rows_in_layer) {
          err |= HS_DEV_ERR_BLOCK;
          v = -1;
        }
        s_rid[i] = v;
      }
      __syncwarp();
      mbar_arrive(bar(B_RID));
    }
    bool ok = wait_bar_warp(bar(B_RID), 0, abort_flag, a.error_word);
    // CTA 0: Q occupies the stage region until it has moved to TMEM
    if (rank == 0) ok = ok && wait_bar_warp(bar(B_Q_READY), 0, abort_flag, a.error_word);
    const int ncb = rank == 0 ? kCbK : kCbV;
    const int n_items = ncb * (kTile / 4);  // (column block, 4-row group) pairs
    for (int t = 0; ok && t < n_tiles; ++t) {
      const int s = t % kStages;
      const uint32_t ph = (uint32_t)(t / kStages) & 1u;
      if (!wait_bar_warp(bar(B_KV_EMPTY + s), ph ^ 1u, abort_flag, a.error_word)) break;
      if (lw == 0 && lane == 0)
        mbar_arrive_expect_tx(bar(B_KV_FULL + s), (uint32_t)ncb * kBlockBytes);
      if (lane < kTile / 4) {
        const int32_t* rid = s_rid + t * kTile + 4 * lane;  // lane g moves rows 4g .. 4g+3
        const int y0 = rid[0] >= 0 ? rid[0] : a.rows_in_layer;
        const int y1 = rid[1] >= 0 ? rid[1] : a.rows_in_layer;
        const int y2 = rid[2] >= 0 ? rid[2] : a.rows_in_layer;
        const int y3 = rid[3] >= 0 ? rid[3] : a.rows_in_layer;
        const uint32_t dst = sbase + OFF_STAGE + s * kStageBytes + lane * 512;
        for (int item = lw * 16 + lane; item < n_items; item += kLoadWarps * 16) {
          const int cb = item >> 4;
          tma_gather4(dst + cb * kBlockBytes, &kv_map, cb * 64, y0, y1, y2, y3, bar(B_KV_FULL + s));
        }
      }
    }
  } else if (warp == 0) {
    // ================= MMA issuer =================
    if (lane == 0) {
      if (rank == 0) {
        // B = K tile, K-major, 128B swizzle: column block cb at +cb*8192, K step
        // kk at +(kk%4)*32 inside the block; 8-row groups 1024 B apart
        const uint64_t kdesc0 = desc_sw128(sbase + OFF_STAGE, 16, 1024);
        if (wait_bar(bar(B_Q_READY), 0, abort_flag, a.error_word)) {
          tc_fence_after();
          for (int t = 0; t < n_tiles; ++t) {
            const int s = t % kStages, b = t & 1;
            const uint32_t ph = (uint32_t)(t / kStages) & 1u, pb = (uint32_t)(t >> 1) & 1u;
            if (!wait_bar(bar(B_KV_FULL + s), ph, abort_flag, a.error_word)) break;
            if (!wait_bar(bar(B_S_EMPTY + b), pb ^ 1u, abort_flag, a.error_word)) break;
            tc_fence_after();
            const uint64_t kd = kdesc0 + ((s * kStageBytes) >> 4);
            const uint32_t dS = tm + TM_S + b * kTile;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ts(dS, tm + TM_Q + kk * 8,
                     kd + (uint64_t)((((kk >> 2) * kBlockBytes) + (kk & 3) * 32) >> 4), kIdescS,
                     kk > 0);
            mma_commit(bar(B_KV_EMPTY + s));
            mma_commit(bar(B_S_FULL + b));
          }
        }
      } else {
        // A = P (interleaved core matrices: K step kk at +kk*256, 8-head groups
        // 1024 B apart); B = V, MN-major, 128B swizzle: 64-column blocks
        // 8192 B apart, 8-row groups 1024 B apart, K step kk at +kk*2048
        const uint64_t pdesc0 = smem_desc(sbase + OFF_P, 128, 1024);
        const uint64_t vdesc0 = desc_sw128(sbase + OFF_STAGE, kBlockBytes, 1024);
        uint32_t corr = 0;
        for (int t = 0; t < n_tiles; ++t) {
          const int s = t % kStages, b = t & 1;
          const uint32_t ph = (uint32_t)(t / kStages) & 1u, pb = (uint32_t)(t >> 1) & 1u;
          mbar_arrive_expect_tx(bar(B_P_FULL + b), kPCopyBytes);
          if (!wait_bar(bar(B_KV_FULL + s), ph, abort_flag, a.error_word)) break;
          if (!wait_bar(bar(B_P_FULL + b), pb, abort_flag, a.error_word, true)) break;
          const uint32_t* flags =
              reinterpret_cast<const uint32_t*>(smem + OFF_P + b * kPBufBytes + 2 * kPBytes + 512);
          if (t > 0 && (flags[0] | flags[1] | flags[2] | flags[3])) {
            // the running max moved for some head: rescale O before adding tile t
            mma_commit(bar(B_MMA_IDLE));
            if (!wait_bar(bar(B_MMA_IDLE), corr & 1u, abort_flag, a.error_word)) break;
            *corr_tile = t;
            mbar_arrive(bar(B_CORR_REQ));
            if (!wait_bar(bar(B_CORR_DONE), corr & 1u, abort_flag, a.error_word)) break;
            ++corr;
          }
          tc_fence_after();
          const uint64_t pd = pdesc0 + ((b * kPBufBytes) >> 4);
          const uint64_t vd = vdesc0 + ((s * kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
              for (int half = 0; half < 2; ++half)
                mma_ss(tm + TM_O + half * 256, pd + (uint64_t)((part * kPBytes + kk * 256) >> 4),
                       vd + (uint64_t)((half * 4 * kBlockBytes + kk * 2048) >> 4), kIdescPV,
                       (t > 0 || kk > 0 || part > 0) ? 1u : 0u);
            }
          }
          mma_commit(bar(B_KV_EMPTY + s));
          mma_commit_multicast(bar(B_P_EMPTY + b), (uint16_t)0x1);  // P buffer b free (CTA 0)
        }
        *corr_exit = 1;
        mbar_arrive(bar(B_CORR_REQ));  // releases the rescale warps
      }
      mma_commit(bar(B_FINAL));
      wait_bar(bar(B_FINAL), 0, abort_flag, a.error_word);
    }
    __syncwarp();
  } else if (warp >= kMathWarp0 && rank == 0) {
    // ================= softmax (CTA 0, warps 4..7, one thread per head) =================
    const int h = tid - kMathWarp0 * 32;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = wait_bar_warp(bar(B_Q_SMEM), 0, abort_flag, a.error_word);
    if (ok) {  // Q[h] -> TMEM columns TM_Q .. TM_Q+287 (bf16 pairs), zero for padded heads
      // swizzled rows: column block cb holds [128 rows][128 B]; 16-byte chunk c
      // of row h sits at chunk position c ^ (h % 8) (conflict-free reads)
      const unsigned char* qrow = smem + OFF_STAGE + h * 128;
      for (int c0 = 0; c0 < kD / 2; c0 += 16) {
        uint32_t v[16];
        const unsigned char* blk = qrow + (c0 / 32) * kQBlockBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = (c0 % 32) / 4 + i;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (h < a.H) x = *reinterpret_cast<const uint4*>(blk + ((c ^ (h & 7)) * 16));
          v[4 * i + 0] = x.x;
          v[4 * i + 1] = x.y;
          v[4 * i + 2] = x.z;
          v[4 * i + 3] = x.w;
        }
        tmem_st16(tm + lane_off + TM_Q + c0, v);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    mbar_arrive(bar(B_Q_READY));
    ok = ok && wait_bar_warp(bar(B_RID), 0, abort_flag, a.error_word);
    const uint32_t peer_p = mapa(sbase + OFF_P, 1);
    const uint32_t peer_pfull = mapa(bar(B_P_FULL), 1);
    float m_used = -INFINITY, l_sum = 0.f;
    for (int t = 0; ok && t < n_tiles; ++t) {
      const int b = t & 1;
      const uint32_t pb = (uint32_t)(t >> 1) & 1u;
      const uint64_t valid =
          (uint64_t)__ballot_sync(0xffffffffu, s_rid[t * kTile + lane] >= 0) |
          ((uint64_t)__ballot_sync(0xffffffffu, s_rid[t * kTile + lane + 32] >= 0) << 32);
      if (!wait_bar_warp(bar(B_S_FULL + b), pb, abort_flag, a.error_word)) break;
      tc_fence_after();
      float x[kTile];
#pragma unroll
      for (int c = 0; c < kTile; c += 16) {
        uint32_t u[16];
        tmem_ld16(tm + lane_off + TM_S + b * kTile + c, u);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) x[c + i] = __uint_as_float(u[i]);
      }
      tc_fence_before();
      mbar_arrive(bar(B_S_EMPTY + b));
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < kTile; ++i) {
        x[i] = ((valid >> i) & 1) ? x[i] * a.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, x[i]);
      }
      // lazy rescale: move the reference max only when it grew by > 2^8
      const bool rescale = tmax > m_used + 8.f;
      float alpha = 1.f;
      if (rescale) {
        alpha = fast_exp2(m_used - tmax);  // 0 when m_used is -inf
        l_sum *= alpha;
        m_used = tmax;
      }
      // P buffer b is free once the value CTA finished tile t-2
      if (!wait_bar_warp(bar(B_P_EMPTY + b), pb ^ 1u, abort_flag, a.error_word)) break;
      unsigned char* pbuf = smem + OFF_P + b * kPBufBytes;
#pragma unroll
      for (int kb = 0; kb < kTile / 8; ++kb) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = x[kb * 8 + 2 * i], x1 = x[kb * 8 + 2 * i + 1];
          const float p0 = x0 == -INFINITY ? 0.f : fast_exp2(x0 - m_used);
          const float p1 = x1 == -INFINITY ? 0.f : fast_exp2(x1 - m_used);
          l_sum += p0 + p1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          const float2 hf = __bfloat1622float2(h2);
          hi[i] = *reinterpret_cast<const uint32_t*>(&h2);
          lo[i] = pack_bf16x2(p0 - hf.x, p1 - hf.y);
        }
        // P [128 heads x 64 rows], K-major core matrices (head group, row group)
        const uint32_t off = (uint32_t)(((h >> 3) * (kTile / 8) + kb) * 128 + (h & 7) * 16);
        *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(pbuf + kPBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      float* meta = reinterpret_cast<float*>(pbuf + 2 * kPBytes);
      meta[h] = alpha;
      const uint32_t any = __ballot_sync(0xffffffffu, rescale && t > 0);
      if (lane == 0) reinterpret_cast<uint32_t*>(meta + 128)[warp & 3] = any;
      fence_proxy_async_smem();  // generic-proxy writes -> visible to the bulk copy
      mbar_arrive(bar(B_P_READY + b));
      if (h == 0) {
        if (!wait_bar(bar(B_P_READY + b), pb, abort_flag, a.error_word)) break;
        bulk_copy_s2cluster(peer_p + b * kPBufBytes, sbase + OFF_P + b * kPBufBytes, kPCopyBytes,
                            peer_pfull + 8u * b);
      }
    }
    // final m, l for this head -> value CTA
    st_cluster_f32(mapa(sbase + OFF_ML + 4 * h, 1), m_used);
    st_cluster_f32(mapa(sbase + OFF_ML + 512 + 4 * h, 1), l_sum);
    mbar_arrive_remote(mapa(bar(B_ML_FULL), 1));
    // wait until the value CTA released the last P buffers (its commits landed)
    for (int t = n_tiles - 2; t < n_tiles; ++t) {
      if (t < 0) continue;
      wait_bar(bar(B_P_EMPTY + (t & 1)), (uint32_t)(t >> 1) & 1u, abort_flag, a.error_word);
    }
  } else if (warp >= kMathWarp0) {
    // ================= rescale + epilogue (CTA 1, warps 4..7) =================
    const int h = tid - kMathWarp0 * 32;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    for (uint32_t k = 0;; ++k) {  // rare: only tiles where some head's max moved
      if (!wait_bar_warp(bar(B_CORR_REQ), k & 1u, abort_flag, a.error_word)) break;
      if (*corr_exit) break;
      tc_fence_after();
      const int t = *corr_tile;
      const float alpha =
          reinterpret_cast<const float*>(smem + OFF_P + (t & 1) * kPBufBytes + 2 * kPBytes)[h];
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        for (int c = 0; c < kDV; c += 16) {
          uint32_t u[16];
          tmem_ld16(tm + lane_off + TM_O + c, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st16(tm + lane_off + TM_O + c, u);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(B_CORR_DONE));
    }
    // epilogue: O / l
    bool ok = wait_bar_warp(bar(B_FINAL), 0, abort_flag, a.error_word) && n_tiles > 0;
    const bool have_ml = wait_bar_warp(bar(B_ML_FULL), 0, abort_flag, a.error_word, true);
    ok = ok && have_ml;  // warp-uniform: gates the warp-collective TMEM loads below
    tc_fence_after();
    const float m = have_ml ? reinterpret_cast<const float*>(smem + OFF_ML)[h] : -INFINITY;
    const float l = have_ml ? reinterpret_cast<const float*>(smem + OFF_ML + 512)[h] : 0.f;
    const bool has_rows = ok && l > 0.f;  // per head (lane)
    const float inv_l = has_rows ? 1.f / l : 0.f;
    const float lse = has_rows ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    const bool write = h < a.H;
    if (a.splits == 1) {
      uint16_t* orow = a.out + ((int64_t)r * a.H + (write ? h : 0)) * kDV;
      for (int c = 0; c < kDV; c += 16) {
        uint32_t u[16];
        if (ok) {
          tmem_ld16(tm + lane_off + TM_O + c, u);
          tmem_ld_wait();
        }
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = has_rows ? pack_bf16x2(__uint_as_float(u[2 * i]) * inv_l,
                                         __uint_as_float(u[2 * i + 1]) * inv_l)
                           : 0u;
        if (write) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
          dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if (write && a.lse) a.lse[(int64_t)r * a.H + h] = lse;
    } else {
      float* orow = a.ws_o + (((int64_t)r * a.splits + split) * kHeads + h) * kDV;
      for (int c = 0; c < kDV; c += 16) {
        uint32_t u[16];
        if (ok) {
          tmem_ld16(tm + lane_off + TM_O + c, u);
          tmem_ld_wait();
        }
        float4* dst = reinterpret_cast<float4*>(orow + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = has_rows ? make_float4(__uint_as_float(u[4 * i]) * inv_l,
                                          __uint_as_float(u[4 * i + 1]) * inv_l,
                                          __uint_as_float(u[4 * i + 2]) * inv_l,
                                          __uint_as_float(u[4 * i + 3]) * inv_l)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      a.ws_lse[((int64_t)r * a.splits + split) * kHeads + h] = lse;
    }
  }

  if (err) atomicOr(a.error_word, err);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 512);
  cluster_sync();
}

// Combine per-split normalised partials: o = sum_c w_c o_c / sum_c w_c with
// w_c = exp(lse_c - max lse).  One CTA per (request, head), 128 threads x 4.
__global__ void __launch_bounds__(128) merge_splits_kernel(const float* __restrict__ ws_o,
                                                           const float* __restrict__ ws_lse,
                                                           int splits, int H,
                                                           uint16_t* __restrict__ out,
                                                           float* __restrict__ lse_out) {
  const int r = blockIdx.y, h = blockIdx.x;
  float mx = -INFINITY;
  for (int c = 0; c < splits; ++c) mx = fmaxf(mx, ws_lse[((int64_t)r * splits + c) * kHeads + h]);
  float wsum = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int e0 = threadIdx.x * 4;
  for (int c = 0; c < splits; ++c) {
    const float lc = ws_lse[((int64_t)r * splits + c) * kHeads + h];
    const float w = lc == -INFINITY ? 0.f : expf(lc - mx);
    wsum += w;
    const float4 o = *reinterpret_cast<const float4*>(
        ws_o + (((int64_t)r * splits + c) * kHeads + h) * kDV + e0);
    acc[0] += w * o.x;
    acc[1] += w * o.y;
    acc[2] += w * o.z;
    acc[3] += w * o.w;
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2 pk;
  pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(out + ((int64_t)r * H + h) * kDV + e0) = pk;
  if (lse_out && threadIdx.x == 0)
    lse_out[(int64_t)r * H + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// Splits of K per request: enough CTA pairs to cover the SMs once.
// At most kMaxSplitRows rows per split (their ids are staged in shared memory).
int choose_splits(int num_sms, int R, int K) {
  const int tiles = (K + kTile - 1) / kTile;
  int s = num_sms / (2 * R);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  const int min_s = (tiles * kTile + kMaxSplitRows - 1) / kMaxSplitRows;
  if (s < min_s) s = min_s;
  return s;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

hs_status get_encoder() {
  if (g_encode) return HS_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return HS_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return HS_OK;
}

// 2-D bf16 tensor map over [rows][576], 128B swizzle, box = 64 columns x box_rows.
hs_status encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  if (get_encoder() != HS_OK) return HS_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult cr = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return cr == CUDA_SUCCESS ? HS_OK : HS_ERR_INVALID;
}

}  // namespace

hs_status hs_attn_workspace_init(hs_pool* p) {
  p->attn_o = nullptr;
  p->attn_ml = nullptr;
  p->attn_kv_maps = nullptr;
  p->attn_max_splits = 0;
  if (p->d.row_elems != kD) return HS_OK;  // attention needs 576-wide rows; decode call rejects
  HS_CUDA_TRY(cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemBytes));
  const int64_t rows_in_layer = p->blocks_per_layer * p->d.page_tokens;
  CUtensorMap* maps = new (std::nothrow) CUtensorMap[p->d.num_layers];
  if (!maps) return HS_ERR_OOM;
  p->attn_kv_maps = maps;
  for (int l = 0; l < p->d.num_layers; ++l) {
    const void* base = static_cast<const uint16_t*>(p->kv_pool) + (int64_t)l * rows_in_layer * kD;
    const hs_status st = encode_rows_map(&maps[l], base, (uint64_t)rows_in_layer, 1);
    if (st != HS_OK) return st;
  }
  const int splits = choose_splits(p->num_sms, p->d.num_requests, p->d.top_k);
  p->attn_max_splits = splits;
  if (splits > 1) {
    const size_t n = (size_t)p->d.num_requests * splits * kHeads;
    if (cudaMalloc(&p->attn_o, n * kDV * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&p->attn_ml, n * sizeof(float)) != cudaSuccess) {
      cudaGetLastError();
      return HS_ERR_OOM;
    }
  }
  return HS_OK;
}

void hs_attn_workspace_free(hs_pool* p) {
  cudaFree(p->attn_o);
  cudaFree(p->attn_ml);
  delete[] static_cast<CUtensorMap*>(p->attn_kv_maps);
  p->attn_o = nullptr;
  p->attn_ml = nullptr;
  p->attn_kv_maps = nullptr;
}

extern "C" hs_status hs_sparse_mla_decode(hs_pool* p, int32_t layer, const void* q,
                                          const int32_t* row_ids, int32_t num_heads, int32_t v_dim,
                                          float scale, void* out, float* lse, void* stream) {
  if (!p || !q || !row_ids || !out) return HS_ERR_INVALID;
  if (layer < 0 || layer >= p->d.num_layers || num_heads <= 0 || num_heads > kHeads ||
      v_dim != kDV || p->d.row_elems != kD || !(scale > 0.f) || p->attn_max_splits < 1 ||
      !p->attn_kv_maps)
    return HS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return HS_ERR_INVALID;
  const int64_t rows_in_layer = p->blocks_per_layer * p->d.page_tokens;
  CUtensorMap q_map;  // host-side encode only: safe inside stream capture
  if (encode_rows_map(&q_map, q, (uint64_t)p->d.num_requests * num_heads, kHeads) != HS_OK)
    return HS_ERR_INVALID;
  AttnArgs a;
  a.row_ids = row_ids;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.ws_o = p->attn_o;
  a.ws_lse = p->attn_ml;
  a.error_word = p->error_word;
  a.rows_in_layer = (int32_t)rows_in_layer;
  a.K = p->d.top_k;
  a.H = num_heads;
  a.splits = p->attn_max_splits;
  const int tiles = (a.K + kTile - 1) / kTile;
  a.rows_per_split = ((tiles + a.splits - 1) / a.splits) * kTile;
  a.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = hs_stream(stream);
  dim3 grid(2 * a.splits, p->d.num_requests);
  mla_decode_kernel<<<grid, kThreads, kSmemBytes, s>>>(
      static_cast<const CUtensorMap*>(p->attn_kv_maps)[layer], q_map, a);
  HS_CUDA_TRY(cudaGetLastError());
  if (a.splits > 1) {
    merge_splits_kernel<<<dim3(num_heads, p->d.num_requests), 128, 0, s>>>(
        p->attn_o, p->attn_ml, a.splits, num_heads, a.out, lse);
    HS_CUDA_TRY(cudaGetLastError());
  }
  return HS_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the decode call.
//
// Some callers cannot allocate device memory at the point where they decode:
// an engine that reserved all free HBM for its KV cache up front, code running
// under an allocator that forbids new device allocations once serving starts,
// or a plug-in that only receives raw device pointers from its host.  For
// them, hs_sparse_mla_decode_noalloc() takes the KV rows, queries, row ids and
// outputs as plain pointers and keeps its split-K scratch (per-split partial
// outputs and their log-sum-exp) in the fixed device array below, which every
// GPU that loads this library holds until the process exits.  It calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// Capacity: partials for at most kNoAllocMaxUnits (request, split) pairs.  The
// call picks splits = min(its usual choice, kNoAllocMaxUnits / R), and rejects
// the call (HS_ERR_INVALID) when even the fewest splits the kernel allows
// (ceil(K / 2048)) need more.  With one split no scratch is used at all.
// Every call overwrites the scratch it uses before reading it, so nothing has
// to start at zero; calls whose kernels overlap on the GPU (e.g. on two
// streams) share the array and race.
constexpr int kNoAllocMaxUnits = 64;  // 64 x 128 x 512 fp32 = 16 MiB (+ 32 KiB lse)
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocMaxUnits * kHeads * (kDV + 1)];
static __device__ int32_t g_noalloc_error_word;

namespace {
constexpr int kMaxDevices = 64;
float* g_noalloc_ptr[kMaxDevices];       // device address of the scratch, per device
int32_t* g_noalloc_err_ptr[kMaxDevices];
int g_noalloc_sms[kMaxDevices];

// Once per device, with that device current: resolve the scratch's device
// address (in host code the array's name is only a stand-in, not an address)
// and raise the kernel's shared-memory limit.
hs_status noalloc_setup(int dev) {
  if (g_noalloc_ptr[dev]) return HS_OK;
  void* scratch = nullptr;
  void* errw = nullptr;
  HS_CUDA_TRY(cudaGetSymbolAddress(&scratch, g_noalloc_scratch));
  HS_CUDA_TRY(cudaGetSymbolAddress(&errw, g_noalloc_error_word));
  HS_CUDA_TRY(cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemBytes));
  int sms = 0;
  HS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  g_noalloc_sms[dev] = sms;
  g_noalloc_err_ptr[dev] = static_cast<int32_t*>(errw);
  g_noalloc_ptr[dev] = static_cast<float*>(scratch);
  return HS_OK;
}
}  // namespace

extern "C" hs_status hs_sparse_mla_decode_noalloc(const void* kv_rows, int64_t num_rows,
                                                  const void* q, const int32_t* row_ids,
                                                  int32_t num_requests, int32_t top_k,
                                                  int32_t num_heads, int32_t v_dim, float scale,
                                                  void* out, float* lse, void* stream) {
  if (!kv_rows || !q || !row_ids || !out) return HS_ERR_INVALID;
  if (num_rows <= 0 || num_rows > INT32_MAX || num_requests <= 0 || top_k <= 0 ||
      num_heads <= 0 || num_heads > kHeads || v_dim != kDV || !(scale > 0.f))
    return HS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(kv_rows) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15))
    return HS_ERR_INVALID;
  const int tiles = (top_k + kTile - 1) / kTile;
  const int min_splits = (tiles * kTile + kMaxSplitRows - 1) / kMaxSplitRows;
  if (min_splits > 1 && (int64_t)num_requests * min_splits > kNoAllocMaxUnits)
    return HS_ERR_INVALID;  // the fixed scratch cannot hold this many partials
  int dev = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_INVALID;
  const hs_status st = noalloc_setup(dev);
  if (st != HS_OK) return st;
  int splits = choose_splits(g_noalloc_sms[dev], num_requests, top_k);
  if (splits > 1 && (int64_t)num_requests * splits > kNoAllocMaxUnits)
    splits = kNoAllocMaxUnits / num_requests;
  if (splits < min_splits) splits = min_splits;
  CUtensorMap kv_map, q_map;  // host-side encodes only
  if (encode_rows_map(&kv_map, kv_rows, (uint64_t)num_rows, 1) != HS_OK ||
      encode_rows_map(&q_map, q, (uint64_t)num_requests * num_heads, kHeads) != HS_OK)
    return HS_ERR_INVALID;
  float* scratch = g_noalloc_ptr[dev];
  AttnArgs a;
  a.row_ids = row_ids;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.ws_o = scratch;
  a.ws_lse = scratch + (size_t)kNoAllocMaxUnits * kHeads * kDV;
  a.error_word = g_noalloc_err_ptr[dev];
  a.rows_in_layer = (int32_t)num_rows;
  a.K = top_k;
  a.H = num_heads;
  a.splits = splits;
  a.rows_per_split = ((tiles + splits - 1) / splits) * kTile;
  a.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = hs_stream(stream);
  mla_decode_kernel<<<dim3(2 * splits, num_requests), kThreads, kSmemBytes, s>>>(kv_map, q_map, a);
  HS_CUDA_TRY(cudaGetLastError());
  if (splits > 1) {
    merge_splits_kernel<<<dim3(num_heads, num_requests), 128, 0, s>>>(a.ws_o, a.ws_lse, splits,
                                                                      num_heads, a.out, lse);
    HS_CUDA_TRY(cudaGetLastError());
  }
  return HS_OK;
}
