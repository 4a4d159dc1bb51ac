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
//   CTA 0 ("score"): Q lives in tensor memory (the A operand); S = Q K^T
//     (M=128, N=64, K=576) over 64-row tiles goes to one of three TMEM
//     accumulators; 4 warps run the online softmax (one thread per head) and
//     write P in fp16 (11 significant bits; bf16 P would cost ~1.5e-3 relative
//     error) straight into CTA 1's P ring by remote st.async stores, which
//     count their bytes on that buffer's mbarrier in CTA 1.
//   CTA 1 ("value"): accumulates O += P V (M=128, N=256 x 2, V as an MN-major
//     operand) with V in fp16 as well.  Its 4 rescale warps rescale O when the
//     running max moved (lazily: only when it grew by more than 2^8, so the
//     rescale is rare and off the common path).  After the last tile they and
//     the 8 loader warps (three warps per TMEM lane quarter) write the output
//     through shared memory in coalesced rows.
// Row loads.  Each CTA loads the tile rows it needs itself, so the two stage
// rings never wait on each other: CTA 0's K tiles come by TMA (tile::gather4,
// 128-byte swizzle, straight into the operand layout) into a 3-stage ring,
// the rope block from CTA 1's otherwise idle TMA unit (multicast to CTA 0),
// the rest from CTA 0's own;
// CTA 1's eight loader warps move the 512 value columns with 16-byte vector
// loads, converting them to fp16 through registers, with the loads for the
// next tile issued before the stage frees up.  Pools of FP8 rows (656 bytes:
// E4M3 latent codes with one scale per 128 values, bf16 rope) are read by
// vector loads in both CTAs and dequantized to fp16 operands on the way into
// shared memory (Fp8Loader); the score MMA then runs on fp16, with Q
// converted from bf16 as it moves to tensor memory.  Q reaches CTA 0 by TMA
// (swizzled, then TMEM), each split's row ids are staged in shared memory
// once, MMA descriptors are computed once and advanced by constants, and
// every hand-off is an mbarrier.  With several splits per request, each pair
// writes a normalised fp16 partial and its log-sum-exp; a small merge kernel
// combines them.
//
// Every wait is bounded: a wait that times out sets HS_DEV_ERR_WAIT in the
// pool's error word and the CTA winds down (no further MMAs), frees its tensor
// memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <new>
#include <string.h>

#include "hs_internal.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace hs_ptx;

constexpr int kHeads = 128;        // MMA M (heads, zero-padded)
constexpr int kD = 576;            // row width (latent 512 + rope 64)
constexpr int kDV = 512;           // value width
constexpr int kTile = 64;          // KV rows per tile
// KV tile ring depth: 3 in the score CTA (a stage is held from its gathers'
// issue, ~2 us of TMA latency, through its score MMA, so two stages kept the
// gathers idle a third of the time), 2 in the value CTA (whose loader threads
// hold two more tiles in registers)
constexpr int kStagesS = 3, kStagesV = 2;
constexpr int kThreads = 512;
// Warp roles (four warpgroups of four warps):
//   warp 0       MMA issuer               warp 1 (CTA 0)  Q load
//   warp 2 (CTA 1) rope-block gathers      warps 4..11     row loaders (CTA 0: TMA
//     into CTA 0; other warps 2..3 idle    gathers; CTA 1: vector loads + fp16)
//   warps 12..15 softmax (CTA 0) / rescale + epilogue (CTA 1; the loader
//     warps join the epilogue)
constexpr int kLoadWarp0 = 4;
constexpr int kLoadWarps = 8;
constexpr int kLoadThreads = kLoadWarps * 32;
static_assert(kLoadThreads == 4 * 64, "loader mapping: 64 value chunks x 4 groups of 16 rows");
constexpr int kQWarp = 1;
constexpr int kMathWarp0 = 12;
// Registers per thread after the split (setmaxnreg, per warpgroup): the loader
// warps hold two tiles of loads in flight.  The kernel launches with 128 per
// thread (512 threads x 128 = the SM's 65536); 64 + 168 + 168 + 112 sums to
// 4 x 128, so every increase can be granted.
constexpr int kRegsWG0 = 64, kRegsLoad = 168, kRegsMath = 112;
static_assert(kRegsWG0 + 2 * kRegsLoad + kRegsMath == 4 * 128, "register split");
static_assert(65536 / 512 == 128, "launch allocation per thread");
constexpr int kCbK = kD / 64;      // 9 swizzled 128-byte column blocks per K row
constexpr int kFp8RowBytes = 656;  // an FP8 KV row (HS_KV_FP8)

constexpr uint32_t kBlockBytes = kTile * 128;              // one column block of a tile: 8192
constexpr uint32_t kStageBytes = kCbK * kBlockBytes;       // 73728
constexpr uint32_t kQBlockBytes = kHeads * 128;            // 16384
constexpr uint32_t kPBytes = kHeads * kTile * 2;           // 16384 (fp16)
// P buffer (value CTA): P [128 heads x 64 rows] fp16, then alpha[128] (fp32),
// then one 16-byte flag record per softmax warp.  The softmax threads store
// them from registers into the value CTA's buffer (st.async, counted by the
// buffer's barrier): a head's 128 B of P and its alpha, and each warp's flag.
constexpr int kPBufs = 4;                                  // P ring depth
constexpr uint32_t kPAlphaOff = kPBytes;                   // alpha[128]
constexpr uint32_t kPFlagOff = kPBytes + 512;              // 4 x 16-byte flag records
constexpr uint32_t kPCopyBytes = kHeads * (kTile * 2 + 4) + 4 * 16;  // 16960 per tile
constexpr uint32_t kPBufBytes = kPBytes + 1024;            // 17408

// Shared-memory layout.  The score CTA holds 3 K stages; the value CTA 2 V
// stages, the P ring and m/l in the same bytes.  Row ids, barriers and the
// scalars sit at the same offsets in both CTAs (remote barrier operations
// address the peer by offset), as do the value CTA's P buffers and m/l, which
// the score CTA writes.  Swizzled regions are 1024-byte aligned.
constexpr int kMaxSplitRows = 2048;  // row ids of one split, staged in shared memory
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_P = OFF_STAGE + kStagesV * kStageBytes;  // 147456 (value CTA)
constexpr uint32_t OFF_ML = OFF_P + kPBufs * kPBufBytes;        // 217088: m[128], l[128]
constexpr uint32_t OFF_RID = OFF_STAGE + kStagesS * kStageBytes;  // 221184: int32 [2048]
constexpr uint32_t OFF_BAR = OFF_RID + 4 * kMaxSplitRows;       // 229376
constexpr uint32_t OFF_MISC = OFF_BAR + 256;
constexpr uint32_t kSmemBytes = OFF_MISC + 64;                  // 229696
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(OFF_ML + 1024 <= OFF_RID, "value CTA layout");
// CTA 0 stages Q (9 column blocks of 16 KB) in stages 1 and 2, so that stage 0
// is free for the first tile's rows from the start.
static_assert(kStagesS == 3 && kCbK * kQBlockBytes == 2 * kStageBytes, "Q staging");
__host__ __device__ constexpr uint32_t q_block_off(int cb) {
  return OFF_STAGE + kStageBytes + (uint32_t)cb * kQBlockBytes;
}
static_assert(q_block_off(0) % 1024 == 0 && kQBlockBytes % 1024 == 0, "swizzled Q blocks");
// epilogue staging (12 warps x 8 KiB) reuses the stage region once the last tile is consumed
static_assert(12 * 8192 <= kStagesV * kStageBytes, "epilogue staging");

// barrier indices (8 bytes each at OFF_BAR)
enum {
  B_KV_FULL = 0,     // [3] loader warps stored a tile -> MMA (both CTAs: K tile / V tile)
  B_KV_EMPTY = 3,    // [3] MMA commit -> loaders
  B_S_FULL = 6,      // [3] score MMA commit -> softmax
  B_S_EMPTY = 9,     // [3] softmax -> score MMA
  B_P_EMPTY = 12,    // [4] (CTA 0) value MMA commit (multicast) -> softmax
  B_P_FULL = 16,     // [4] (CTA 1) the softmax's remote stores complete_tx -> value MMA
  B_Q_SMEM = 20,     // (CTA 0) TMA of Q landed in shared memory
  B_Q_READY = 21,    // (CTA 0) softmax warps put Q in TMEM -> score MMA, loaders
  B_RID = 22,        // loader warps staged this split's row ids
  B_CORR_REQ = 23,   // (CTA 1) value MMA -> rescale warps
  B_CORR_DONE = 24,  // (CTA 1) rescale warps -> value MMA
  B_MMA_IDLE = 25,   // (CTA 1) commit: earlier P.V MMAs finished
  B_ML_FULL = 26,    // (CTA 1) softmax's final m, l -> epilogue
  B_FINAL = 27,      // MMA issuer's last commit
  B_XEMPTY = 28,     // [3] (CTA 1) score MMA commit (multicast): a K stage is free for CTA 1's gathers
  B_XQ = 31,         // (CTA 1) CTA 0's Q has left stages 1-2
  B_COUNT = 32
};
// Column blocks of each bf16 K tile (the last ones: the rope block) that CTA
// 1's TMA unit gathers into CTA 0's stage.  The loop is bound by CTA 0's TMA
// gather rate (~23 B/clk); CTA 1's TMA unit is otherwise idle.  One block: 41
// us per call of 32 x 2048 rows against 44 with none; two or three: 47.6 (CTA
// 1's own intake becomes the bound).
constexpr int kXBlocks = 1;
static_assert(kXBlocks >= 1 && kXBlocks * 16 <= 32, "one warp issues CTA 1's gathers");
constexpr int kSBufs = 3;  // S accumulators in TMEM (CTA 0)
static_assert(B_COUNT * 8 <= 256, "barrier area");

// TMEM columns
constexpr uint32_t TM_Q = 0;     // CTA 0: Q, 288 columns (bf16 pairs)
constexpr uint32_t TM_S = 288;   // CTA 0: S, 3 x 64 columns
constexpr uint32_t TM_O = 0;     // CTA 1: O, 512 columns

constexpr uint32_t kIdescS = idesc_bf16(128, kTile, false, false);  // A (TMEM), B K-major
// the same with fp16 A and B (format code 0): FP8 rows
constexpr uint32_t kIdescS16 = (1u << 4) | ((uint32_t)(kTile >> 3) << 17) |
                               ((uint32_t)(128 >> 4) << 24);
// kind::f16 with fp16 A and B (format code 0), fp32 D; A K-major, B MN-major
constexpr uint32_t kIdescPV = (1u << 4) | (1u << 16) | ((uint32_t)(256 >> 3) << 17) |
                              ((uint32_t)(128 >> 4) << 24);

constexpr uint32_t kWaitNs = 1000000000u;  // 1 s per wait before giving up (< 2^32 ns)
constexpr uint32_t kSuspendNs = 200;          // longest sleep of one try_wait

struct AttnArgs {
  const uint4* kv;          // this layer's rows: [rows_in_layer][576] bf16 as 16-byte chunks,
                            // or [rows_in_layer][656 bytes] FP8 rows
  const int32_t* row_ids;   // [R][K]
  uint16_t* out;            // [R][H][512] bf16 (splits == 1)
  float* lse;               // [R][H] or null (splits == 1)
  uint16_t* ws_o;           // [R][splits][128][512] fp16 partials (splits > 1)
  float* ws_lse;            // [R][splits][128]
  int32_t* error_word;
  int32_t rows_in_layer;
  int32_t K, H, splits, rows_per_split;
  float scale_log2;         // scale * log2(e)
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on a local mbarrier; on timeout (timeout_ns of the global
// timer, or at once if the CTA is already aborting) returns false, raises the
// abort flag and sets error bit WAIT.  After one non-blocking probe the thread
// waits with mbarrier.try_wait, which suspends it until the phase completes
// (or a hardware time limit passes), so a waiting warp takes no issue slots
// or shared-memory bandwidth from the warps that do the work.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort,
                                         int32_t* error_word, bool cluster_scope = false,
                                         uint32_t timeout_ns = kWaitNs) {
  if (*abort) return false;
  if (cluster_scope ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity))
    return true;
  // the low 32 bits of the timer suffice: they wrap after 4.29 s, longer than
  // any time limit used here
  const uint32_t t0 = (uint32_t)globaltimer();
  for (;;) {
    if (cluster_scope ? mbar_try_wait_cluster_hint(bar, parity, kSuspendNs)
                      : mbar_try_wait_hint(bar, parity, kSuspendNs))
      return true;
    if (*abort) return false;
    if ((uint32_t)globaltimer() - t0 > timeout_ns) {
      *abort = 1;
      atomicOr(error_word, HS_DEV_ERR_WAIT);
      return false;
    }
  }
}

// Same, for roles run by whole warps: every lane polls and the warp agrees
// on the answer, so warp-collective instructions after it (tcgen05, shuffles)
// run uniformly.  (With lane 0 polling alone while the other lanes waited at a
// shuffle, each hand-off took 0.25-0.5 us longer to be seen: 3 us per call
// of the 32 x 2048-row workload, 6 us with FP8 rows.)
__device__ __forceinline__ bool wait_bar_all(uint32_t bar, uint32_t parity, volatile int* abort,
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
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Two bf16 values (one 32-bit word) -> the same two values as fp16, exact for
// magnitudes in [2^-14, 65536).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
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
// The same, multicast: the rows land at the same offset in the shared memory
// of every CTA in cta_mask, each completing its own barrier at bar's offset.
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
// Register budget of this warpgroup from here on (all four of its warps run
// it).  The launch gives every thread kLaunchRegs; a budget above that is an
// increase, one below a release (setmaxnreg.inc may only grow the allocation
// and .dec may only shrink it).
constexpr int kLaunchRegs = 65536 / kThreads;
template <int N>
__device__ __forceinline__ void regs_set() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
  if constexpr (N > kLaunchRegs)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
  else if constexpr (N < kLaunchRegs)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
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

// 16-byte global load at row_base + row * 1152 bytes (one KV row), row >= 0,
// through the read-only path and not kept in L1 (each row is read once per
// CTA; the pair's second read of it hits L2).  The address is formed inside
// the statement so it occupies no register beyond the load.
__device__ __forceinline__ uint4 ld_row_chunk(const uint4* row_base, int row) {
  uint4 v;
  asm volatile(
      "{\n .reg .u64 a;\n mad.wide.s32 a, %4, 1152, %5;\n"
      " ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [a];\n}"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(row), "l"(row_base));
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// per-halfword unsigned max
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Value-column loaders: move the first 512 columns of the tile rows into the
// stage ring, 16-byte chunks in the 128B-swizzled K-major layout the MMAs read
// (column block c/8 at +8192 each, row at +128, chunk c%8 at position
// (c%8) ^ (row%8)).  Loader thread lt owns chunk c = lt % 64 of rows
// 16*(lt/64) .. +15 of every tile, so its shared-memory offsets are fixed and
// its row ids come in 16-byte reads.  Each thread keeps two tiles of loads in
// flight (the loads for tile t+2 are issued as soon as tile t is stored).
// The bf16 values are converted to fp16 on the way.  A row id of -1 stores
// zeros.
struct ValueLoader {
  static constexpr int kNst = kStagesV;  // stage ring depth (value CTA)
  struct Regs {
    uint4 v[16];
  };
  const uint4* col;  // chunk c of row 0
  const int32_t* s_rid;
  uint32_t stage0, soff, c7s;
  int r0;

  __device__ __forceinline__ ValueLoader(const uint4* kv, const int32_t* s_rid_, uint32_t stage0_,
                                         int lt)
      : s_rid(s_rid_), stage0(stage0_) {
    r0 = (lt >> 6) * 16;
    const int c = lt & 63;
    col = kv + c;
    soff = (uint32_t)((c >> 3) * kBlockBytes + r0 * 128);
    c7s = (uint32_t)(c & 7) << 4;
  }
  __device__ __forceinline__ void issue(int t, Regs& R) const {
    const int32_t* rid = s_rid + t * kTile + r0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int4 w = *reinterpret_cast<const int4*>(rid + 4 * i);
      const int32_t ids[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        R.v[4 * i + j] = ids[j] >= 0 ? ld_row_chunk(col, ids[j]) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __device__ __forceinline__ void store(int t, Regs& R, uint32_t& vmax) const {
    const uint32_t stage = stage0 + (uint32_t)(t % kNst) * kStageBytes;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      uint4 x = R.v[k];
      vmax = max_u16x2(vmax, x.x & 0x7fff7fffu);
      vmax = max_u16x2(vmax, x.y & 0x7fff7fffu);
      vmax = max_u16x2(vmax, x.z & 0x7fff7fffu);
      vmax = max_u16x2(vmax, x.w & 0x7fff7fffu);
      x.x = bf16x2_to_f16x2(x.x);
      x.y = bf16x2_to_f16x2(x.y);
      x.z = bf16x2_to_f16x2(x.z);
      x.w = bf16x2_to_f16x2(x.w);
      // row r0 + k: r0 % 8 == 0, so its swizzle phase is k % 8
      st_shared_v4(stage + soff + (uint32_t)k * 128u + (c7s ^ ((uint32_t)(k & 7) << 4)), x);
    }
  }
  // vmax holds bf16 magnitudes: 0x4780 is bf16 65536, from which up (inf and
  // NaN included) fp16 cannot hold the value
  __device__ __forceinline__ static bool overflow(uint32_t vmax) {
    return (vmax & 0xffffu) >= 0x4780u || (vmax >> 16) >= 0x4780u;
  }
};

// ---- FP8 rows (656 bytes: 512 E4M3 latent codes, 4 fp32 scales for groups of
// 128 latent values, 64 bf16 rope values).  Both CTAs turn them into fp16
// operands on the way into shared memory: latent value = E4M3 * scale, in
// fp32, rounded once to fp16; rope bf16 -> fp16.

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ uint4 ld_nc_v4(const unsigned char* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
// Four E4M3 codes (one 32-bit word, lowest byte first) times `scale` -> two
// fp16x2 words.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t w, float scale) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  return make_uint2(pack_f16x2(a.x * scale, a.y * scale), pack_f16x2(b.x * scale, b.y * scale));
}
// Two E4M3 codes (low byte first) -> the same two values as fp16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  uint32_t r;
  asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}" : "=r"(r) : "r"(codes));
  return r;
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Lane-wise maximum that returns NaN where either input is NaN.
__device__ __forceinline__ uint32_t max_nan_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void max_f16(uint32_t& vmax, uint4 x) {
  vmax = max_u16x2(vmax, x.x & 0x7fff7fffu);
  vmax = max_u16x2(vmax, x.y & 0x7fff7fffu);
  vmax = max_u16x2(vmax, x.z & 0x7fff7fffu);
  vmax = max_u16x2(vmax, x.w & 0x7fff7fffu);
}
// vmax holds fp16 magnitudes: 0x7C00 and up is inf or NaN (the value overflowed)
__device__ __forceinline__ bool f16_overflow(uint32_t vmax) {
  return (vmax & 0xffffu) >= 0x7C00u || (vmax >> 16) >= 0x7C00u;
}

// FP8 rows into the stage ring as fp16, for either CTA: ROPE (score CTA) the
// whole 576 columns, else (value CTA) the 512 latent columns.  Warp lw owns
// rows 8lw .. 8lw+7 of every tile, lane (rs, k) = (lane / 8, lane % 8) rows
// 8lw+rs and 8lw+4+rs; for each row it reads latent bytes 128j+16k .. +15
// (j = 0..3: group j, so one warp instruction covers four rows' 128-byte runs),
// the row's four scales (16 bytes shared by its 8 lanes) and rope bytes
// 528+16k .. +15.  16 codes make two 8-column fp16 chunks: columns 128j+16k+8h
// sit in column block 2j + k/4 at chunk position 2(k%4)+h; rope chunk k in
// block 8 at position k (positions swizzled with row % 8; the eight lanes of
// a row, which the shared-memory pipe serves together, hit eight different
// positions in every store).
template <bool ROPE>
struct Fp8Loader {
  static constexpr int kNst = ROPE ? kStagesS : kStagesV;  // score CTA : value CTA
  struct Regs {
    uint4 lat[2][4];
    uint4 sc[2];
    uint4 rope[ROPE ? 2 : 1];
  };
  const unsigned char* kv;  // the layer's rows, 656 bytes each
  const int32_t* s_rid;
  uint32_t stage0;
  int row0, k, lt, n_tiles;

  __device__ __forceinline__ Fp8Loader(const unsigned char* kv_, const int32_t* s_rid_,
                                       uint32_t stage0_, int lt_, int n_tiles_)
      : kv(kv_), s_rid(s_rid_), stage0(stage0_), lt(lt_), n_tiles(n_tiles_) {
    const int lane = lt & 31;
    row0 = (lt >> 5) * 8 + (lane >> 3);
    k = lane & 7;
  }
  // Loads tile t into registers, and asks L2 for the rows of tile t+2 (the
  // next loads of this register set): loader thread lt, the 128-byte lines
  // 128 (lt % 4) and 128 (lt % 4) + 512 (the latter for lt % 4 < 2) of row
  // lt / 4, six lines per row.
  __device__ __forceinline__ void issue(int t, Regs& R) const {
    if (t + 2 < n_tiles) {
      const int32_t pid = s_rid[(t + 2) * kTile + (lt >> 2)];
      if (pid >= 0) {
        const unsigned char* pb = kv + (int64_t)pid * kFp8RowBytes + 128 * (lt & 3);
        prefetch_l2(pb);
        if ((lt & 3) < 2) prefetch_l2(pb + 512);
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int32_t id = s_rid[t * kTile + row0 + 4 * rr];
      if (id >= 0) {
        const unsigned char* b = kv + (int64_t)id * kFp8RowBytes;
#pragma unroll
        for (int j = 0; j < 4; ++j) R.lat[rr][j] = ld_nc_v4(b + 128 * j + 16 * k);
        R.sc[rr] = ld_nc_v4(b + 512);
        if (ROPE) R.rope[rr] = ld_nc_v4(b + 528 + 16 * k);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) R.lat[rr][j] = make_uint4(0u, 0u, 0u, 0u);
        R.sc[rr] = make_uint4(0u, 0u, 0u, 0u);
        if (ROPE) R.rope[rr] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  // A scale for which E4M3 x scale is formed in fp16: 0, or a normal fp16
  // value small enough that no finite code (|E4M3| <= 448) passes fp16's
  // largest value (448 x 146 = 65408).  NaN and infinity fail the test.
  __device__ __forceinline__ static bool fp16_scale(uint32_t bits) {
    const float s = fabsf(__uint_as_float(bits));
    return s == 0.f || (s >= 0x1p-14f && s <= 146.f);
  }
  // FAST: the products in fp16 (scale rounded to fp16, then one rounding of
  // the product), with only NaN codes to detect.  Otherwise in fp32 (one
  // rounding to fp16) with a range check of every value.
  template <bool FAST>
  __device__ __forceinline__ void store_rows(int t, Regs& R, uint32_t& vmax) const {
    const uint32_t stage = stage0 + (uint32_t)(t % kNst) * kStageBytes;
    uint32_t nan0 = 0, nan1 = 0;  // NaN-propagating maxima (fp16x2)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = row0 + 4 * rr;
      const uint32_t base = stage + (uint32_t)row * 128u, ph = (uint32_t)(row & 7);
      const float sc[4] = {__uint_as_float(R.sc[rr].x), __uint_as_float(R.sc[rr].y),
                           __uint_as_float(R.sc[rr].z), __uint_as_float(R.sc[rr].w)};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 src = R.lat[rr][j];
        const uint32_t cb = (uint32_t)(2 * j + (k >> 2));
        uint4 half[2];
        if (FAST) {
          const uint32_t s2 = pack_f16x2(sc[j], sc[j]);
          const uint32_t w[4] = {src.x, src.y, src.z, src.w};
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            o[2 * q] = mul_f16x2(e4m3x2_to_f16x2(w[q] & 0xffffu), s2);
            o[2 * q + 1] = mul_f16x2(e4m3x2_to_f16x2(w[q] >> 16), s2);
            if (!ROPE) {  // the score CTA forms the same values: one check suffices
              nan0 = max_nan_f16x2(nan0, o[2 * q]);
              nan1 = max_nan_f16x2(nan1, o[2 * q + 1]);
            }
          }
          half[0] = make_uint4(o[0], o[1], o[2], o[3]);
          half[1] = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint2 lo = e4m3x4_to_f16x4(h ? src.z : src.x, sc[j]);
            const uint2 hi = e4m3x4_to_f16x4(h ? src.w : src.y, sc[j]);
            half[h] = make_uint4(lo.x, lo.y, hi.x, hi.y);
            max_f16(vmax, half[h]);
          }
        }
        // 16-byte stores are served eight lanes at a time: lanes k and k+4
        // of a row share chunk positions, so they store the two halves in
        // opposite orders
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int h = i ^ (k >> 2);
          const uint32_t c = (uint32_t)(2 * (k & 3) + h);
          st_shared_v4(base + cb * kBlockBytes + ((c ^ ph) << 4), h ? half[1] : half[0]);
        }
      }
      if (ROPE) {
        uint4 x = R.rope[rr];
        x.x = bf16x2_to_f16x2(x.x);
        x.y = bf16x2_to_f16x2(x.y);
        x.z = bf16x2_to_f16x2(x.z);
        x.w = bf16x2_to_f16x2(x.w);
        max_f16(vmax, x);
        st_shared_v4(base + 8u * kBlockBytes + (((uint32_t)k ^ ph) << 4), x);
      }
    }
    if (FAST && !ROPE) {
      const uint32_t n = max_nan_f16x2(nan0, nan1);
      if ((n & 0x7fffu) > 0x7c00u || (n & 0x7fff0000u) > 0x7c000000u) vmax |= 0x7C00u;
    }
  }
  // The fp16 products are taken when every scale of the warp's rows allows
  // them (one branch per warp and tile).
  __device__ __forceinline__ void store(int t, Regs& R, uint32_t& vmax) const {
    bool fast = true;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
      fast = fast && fp16_scale(R.sc[rr].x) && fp16_scale(R.sc[rr].y) &&
             fp16_scale(R.sc[rr].z) && fp16_scale(R.sc[rr].w);
    if (__all_sync(0xffffffffu, fast))
      store_rows<true>(t, R, vmax);
    else
      store_rows<false>(t, R, vmax);
  }
  __device__ __forceinline__ static bool overflow(uint32_t vmax) { return f16_overflow(vmax); }
};

// The loader warps' loop, for any of the loaders above.  If q_ready_bar is
// non-zero, the store of tile 1 waits for it (stages 1 and 2 hold Q until Q
// has moved to TMEM).  Returns error bits (VALUE if a value overflowed fp16).
template <typename Loader>
__device__ __forceinline__ int load_tiles(const Loader& L, int n_tiles, uint32_t bar_full0,
                                          uint32_t bar_empty0, uint32_t q_ready_bar,
                                          volatile int* abort_flag, int32_t* error_word) {
  uint32_t vmax = 0;  // per-halfword max of the magnitudes seen (see Loader::overflow)
  bool need_q = q_ready_bar != 0;
  const int lane = threadIdx.x & 31;
  auto put = [&](int t, typename Loader::Regs& v) -> bool {
    if (need_q && t >= 1) {
      if (!wait_bar_all(q_ready_bar, 0, abort_flag, error_word)) return false;
      need_q = false;
    }
    constexpr int kNst = Loader::kNst;
    const int s = t % kNst;
    if (!wait_bar_all(bar_empty0 + 8u * s, ((uint32_t)(t / kNst) & 1u) ^ 1u, abort_flag,
                      error_word))
      return false;
    L.store(t, v, vmax);
    fence_proxy_async_smem();  // generic-proxy stores -> visible to the MMA
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_full0 + 8u * s);
    return true;
  };
  typename Loader::Regs va, vb;  // two tiles of loads in flight
  if (n_tiles > 0) L.issue(0, va);
  for (int t = 0; t < n_tiles; t += 2) {
    if (t + 1 < n_tiles) L.issue(t + 1, vb);
    if (!put(t, va)) break;
    if (t + 2 < n_tiles) L.issue(t + 2, va);
    if (t + 1 < n_tiles && !put(t + 1, vb)) break;
  }
  return Loader::overflow(vmax) ? HS_DEV_ERR_VALUE : 0;
}

// FP8: the pool holds 656-byte FP8 rows (see Fp8Loader); both CTAs load
// them with vector loads and the MMAs run on fp16 operands (Q converted from
// bf16 as it moves to tensor memory).  Otherwise the rows are bf16 [576]; CTA
// 0 gathers them by TMA and the score MMA runs on bf16.
template <bool FP8>
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
    for (int i = 0; i < (rank == 0 ? kStagesS : kStagesV); ++i) {
      // TMA (CTA 0, bf16 rows): one arm (+ the bytes); else one arrival per loader warp
      mbar_init(bar(B_KV_FULL + i), (rank == 0 && !FP8) ? 1 : kLoadWarps);
      mbar_init(bar(B_KV_EMPTY + i), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(bar(B_S_FULL + i), 1);
      mbar_init(bar(B_S_EMPTY + i), 128);
    }
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(bar(B_P_EMPTY + i), 1);
      mbar_init(bar(B_P_FULL + i), 1);
    }
    mbar_init(bar(B_Q_SMEM), 1);
    mbar_init(bar(B_Q_READY), 128);
    mbar_init(bar(B_RID), kLoadWarps);
    mbar_init(bar(B_CORR_REQ), 1);
    mbar_init(bar(B_CORR_DONE), 128);
    mbar_init(bar(B_MMA_IDLE), 1);
    mbar_init(bar(B_ML_FULL), 128);
    mbar_init(bar(B_FINAL), 1);
    for (int i = 0; i < kStagesS; ++i) mbar_init(bar(B_XEMPTY + i), 1);
    mbar_init(bar(B_XQ), 1);
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
  // The merge kernel (launched as a programmatic dependent) may be scheduled
  // from now on; its griddepcontrol.wait still waits for this grid to finish
  // and its writes to be visible.
  asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t tm = *tmem_holder;
  int err = 0;

  // Common exit: report errors, free tensor memory once every role is done, and
  // keep the CTA alive until its peer no longer addresses it.  Each role runs
  // it at its own end.
  auto finish = [&]() {
    if (err) atomicOr(a.error_word, err);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tm, 512);
    cluster_sync();
  };

  // Value CTA epilogue: O / l to global memory.  Three warps per TMEM lane
  // quarter share the 512 columns once the last P.V is done: part 0 (loader
  // warps 4..7) columns 0..191, part 1 (loader warps 8..11) 192..351, part 2
  // (the rescale warps 12..15, which also write lse) 352..511.
  auto epilogue = [&](int part) {
    const int wq = warp & 3;
    const int h = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const int c_begin = part == 0 ? 0 : part == 1 ? 192 : 352;
    const int c_end = part == 0 ? 192 : part == 1 ? 352 : kDV;
    // 32 columns at a time, through this warp's 8 KiB of the (now idle) stage
    // region so that the global stores are whole 64-byte runs of a head's row
    bool ok = wait_bar_all(bar(B_FINAL), 0, abort_flag, a.error_word) && n_tiles > 0;
    const bool have_ml = wait_bar_all(bar(B_ML_FULL), 0, abort_flag, a.error_word, true);
    ok = ok && have_ml;  // warp-uniform: gates the warp-collective TMEM loads below
    tc_fence_after();
    const float m = have_ml ? reinterpret_cast<const float*>(smem + OFF_ML)[h] : -INFINITY;
    const float l = have_ml ? reinterpret_cast<const float*>(smem + OFF_ML + 512)[h] : 0.f;
    const bool has_rows = ok && l > 0.f;  // per head (lane)
    const float inv_l = has_rows ? 1.f / l : 0.f;
    const float lse = has_rows ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    const uint32_t stg = sbase + OFF_STAGE + (uint32_t)(warp - kLoadWarp0) * 8192u;
    // One split: the bf16 output.  Several: this split's partial O / l in fp16
    // (|O / l| is at most the largest |value|, which the loaders hold below
    // 65536, so fp16 keeps it; 11 significant bits, against bf16's 8 in the
    // final output) for the merge kernel.  Both are 16-bit: 64 B per head per
    // 32 columns.
    const bool partial = a.splits > 1;
    uint16_t* dst = partial ? a.ws_o + (((int64_t)r * a.splits + split) * kHeads + wq * 32) * kDV
                            : a.out + ((int64_t)r * a.H + wq * 32) * kDV;
    for (int c0 = c_begin; c0 < c_end; c0 += 32) {  // 32 columns at a time (few live registers)
      uint32_t u[32];
      if (ok) {
        const uint32_t oa = tm + lane_off + TM_O + c0;
        tmem_ld16p(oa, u);
        tmem_ld16p(oa + 16, u + 16);
        tmem_ld_wait();
      }
      // a head's 32 columns are 4 chunks of 16 B, chunk k at k ^ (lane % 4)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x = __uint_as_float(u[8 * k + 2 * i]) * inv_l;
          const float y = __uint_as_float(u[8 * k + 2 * i + 1]) * inv_l;
          pk[i] = !has_rows ? 0u : partial ? pack_f16x2(x, y) : pack_bf16x2(x, y);
        }
        st_shared_v4(stg + lane * 64 + ((k ^ (lane & 3)) << 4),
                     make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // 8 heads x 64 B per instruction
        const int row = 8 * i + (lane >> 2), k = lane & 3;
        const uint4 v = ld_shared_v4(stg + row * 64 + ((k ^ (row & 3)) << 4));
        if (wq * 32 + row < a.H)
          *reinterpret_cast<uint4*>(dst + (int64_t)row * kDV + c0 + 8 * k) = v;
      }
      __syncwarp();
    }
    if (part == 2) {  // lse, one per head
      if (a.splits == 1) {
        if (h < a.H && a.lse) a.lse[(int64_t)r * a.H + h] = lse;
      } else {
        a.ws_lse[((int64_t)r * a.splits + split) * kHeads + h] = lse;
      }
    }
  };

  // Each role first sets its warpgroup's register budget (kRegsWG0 ...); the
  // four warps of a warpgroup always take the same budget.
  if (warp >= kLoadWarp0 && warp < kLoadWarp0 + kLoadWarps) {
    // ================= value-column loaders (both CTAs) =================
    regs_set<kRegsLoad>();
    const int lt = tid - kLoadWarp0 * 32;
    {  // this split's row ids -> shared memory, validated once (-1 = no row)
      constexpr int kRidPer = (kMaxSplitRows + kLoadThreads - 1) / kLoadThreads;
      const int32_t* g_rows = a.row_ids + (int64_t)r * a.K;
      const int n_rows = n_tiles * kTile;
      int32_t v[kRidPer];
#pragma unroll
      for (int k = 0; k < kRidPer; ++k) {
        const int i = lt + k * kLoadThreads, j = j_begin + i;
        v[k] = (i < n_rows && j < j_end) ? __ldg(g_rows + j) : -1;
      }
#pragma unroll
      for (int k = 0; k < kRidPer; ++k) {
        const int i = lt + k * kLoadThreads;
        if (i < n_rows) {
          int32_t x = v[k];
          if (x < -1 || x >= a.rows_in_layer) {
            err |= HS_DEV_ERR_BLOCK;
            x = -1;
          }
          s_rid[i] = x;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_RID));
    }
    if (FP8) {
      // FP8 rows, both CTAs by vector loads: CTA 0 the whole rows, CTA 1 the
      // 512 value columns
      const unsigned char* kv8 = reinterpret_cast<const unsigned char*>(a.kv);
      if (wait_bar_all(bar(B_RID), 0, abort_flag, a.error_word)) {
        if (rank == 0) {
          const Fp8Loader<true> L(kv8, s_rid, sbase + OFF_STAGE, lt, n_tiles);
          err |= load_tiles(L, n_tiles, bar(B_KV_FULL), bar(B_KV_EMPTY), bar(B_Q_READY),
                            abort_flag, a.error_word);
        } else {
          const Fp8Loader<false> L(kv8, s_rid, sbase + OFF_STAGE, lt, n_tiles);
          err |= load_tiles(L, n_tiles, bar(B_KV_FULL), bar(B_KV_EMPTY), 0u, abort_flag,
                            a.error_word);
        }
      }
    } else if (rank == 0) {
      // CTA 0: the 576-column rows by TMA (written straight into the swizzled
      // stage, one shared-memory pass).  Lanes 0..15 of the eight warps issue
      // the (9 - kXBlocks) x 16 gathers of 4 rows (CTA 1 gathers the rest into
      // this stage); a row id of -1 reads past the tensor, which fills zeros.
      // Tile 1 waits for Q to leave stages 1-2.
      const int lw = warp - kLoadWarp0;
      if (wait_bar_all(bar(B_RID), 0, abort_flag, a.error_word)) {
        for (int t = 0; t < n_tiles; ++t) {
          const int s = t % kStagesS;
          if (t == 1 && !wait_bar_all(bar(B_Q_READY), 0, abort_flag, a.error_word)) break;
          if (!wait_bar_all(bar(B_KV_EMPTY + s), ((uint32_t)(t / kStagesS) & 1u) ^ 1u,
                            abort_flag, a.error_word))
            break;
          if (lw == 0 && lane == 0) mbar_arrive_expect_tx(bar(B_KV_FULL + s), kStageBytes);
          if (lane < kTile / 4) {
            const int32_t* rid = s_rid + t * kTile + 4 * lane;
            const int y0 = rid[0] >= 0 ? rid[0] : a.rows_in_layer;
            const int y1 = rid[1] >= 0 ? rid[1] : a.rows_in_layer;
            const int y2 = rid[2] >= 0 ? rid[2] : a.rows_in_layer;
            const int y3 = rid[3] >= 0 ? rid[3] : a.rows_in_layer;
            const uint32_t dst = sbase + OFF_STAGE + s * kStageBytes + lane * 512;
            for (int cb = lw; cb < kCbK - kXBlocks; cb += kLoadWarps)
              tma_gather4(dst + cb * kBlockBytes, &kv_map, cb * 64, y0, y1, y2, y3,
                          bar(B_KV_FULL + s));
          }
          __syncwarp();
        }
      }
    } else if (wait_bar_all(bar(B_RID), 0, abort_flag, a.error_word)) {
      // CTA 1: the 512 value columns by vector loads, converted to fp16
      const ValueLoader L(a.kv, s_rid, sbase + OFF_STAGE, lt);
      err |= load_tiles(L, n_tiles, bar(B_KV_FULL), bar(B_KV_EMPTY), 0u, abort_flag,
                        a.error_word);
    }
    if (rank == 1) epilogue((warp - kLoadWarp0) >> 2);
    finish();
    return;
  } else if (warp == kQWarp && rank == 0) {
    // ================= Q load (CTA 0) =================
    regs_set<kRegsWG0>();
    if (lane == 0 && !*abort_flag) {  // Q[r] (128 rows) -> stages 1 and 2 by TMA
      mbar_arrive_expect_tx(bar(B_Q_SMEM), kCbK * kQBlockBytes);
      for (int cb = 0; cb < kCbK; ++cb)
        tma_load_2d(sbase + q_block_off(cb), &q_map, cb * 64, r * a.H, bar(B_Q_SMEM));
    }
    finish();
    return;
  } else if (warp == 0) {
    // ================= MMA issuer (the whole warp runs it; one elected lane issues) =================
    regs_set<kRegsWG0>();
    if (rank == 0) {
      // B = K tile, K-major, 128B swizzle: column block cb at +cb*8192, K step
      // kk at +(kk%4)*32 inside the block; 8-row groups 1024 B apart
      const uint64_t kdesc0 = desc_sw128(sbase + OFF_STAGE, 16, 1024);
      if (wait_bar_all(bar(B_Q_READY), 0, abort_flag, a.error_word)) {
        tc_fence_after();
        if (!FP8 && lane == 0) mbar_arrive_remote(mapa(bar(B_XQ), 1));  // CTA 1 may fill stages 1-2
        __syncwarp();
        for (int t = 0; t < n_tiles; ++t) {
          const int s = t % kStagesS, b = t % kSBufs;
          const uint32_t ph = (uint32_t)(t / kStagesS) & 1u, pb = (uint32_t)(t / kSBufs) & 1u;
          if (!wait_bar_all(bar(B_KV_FULL + s), ph, abort_flag, a.error_word)) break;
          if (!wait_bar_all(bar(B_S_EMPTY + b), pb ^ 1u, abort_flag, a.error_word)) break;
          tc_fence_after();
          const uint64_t kd = kdesc0 + ((s * kStageBytes) >> 4);
          const uint32_t dS = tm + TM_S + b * kTile;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_ts_elect(dS, tm + TM_Q + kk * 8,
                         kd + (uint64_t)((((kk >> 2) * kBlockBytes) + (kk & 3) * 32) >> 4),
                         FP8 ? kIdescS16 : kIdescS, kk > 0);
          mma_commit_elect(bar(B_KV_EMPTY + s));
          if (!FP8) mma_commit_multicast_elect(bar(B_XEMPTY + s), (uint16_t)(1u << 1));
          mma_commit_elect(bar(B_S_FULL + b));
        }
      }
    } else {
      // A = P, fp16 (interleaved core matrices: K step kk at +kk*256, 8-head
      // groups 1024 B apart); B = V, fp16, MN-major, 128B swizzle: 64-column
      // blocks 8192 B apart, 8-row groups 1024 B apart, K step kk at +kk*2048
      const uint64_t pdesc0 = smem_desc(sbase + OFF_P, 128, 1024);
      const uint64_t vdesc0 = desc_sw128(sbase + OFF_STAGE, kBlockBytes, 1024);
      uint32_t corr = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kStagesV, b = t % kPBufs;
        const uint32_t ph = (uint32_t)(t / kStagesV) & 1u, pb = (uint32_t)(t / kPBufs) & 1u;
        if (lane == 0) mbar_arrive_expect_tx(bar(B_P_FULL + b), kPCopyBytes);
        __syncwarp();
        if (!wait_bar_all(bar(B_KV_FULL + s), ph, abort_flag, a.error_word)) break;
        if (!wait_bar_all(bar(B_P_FULL + b), pb, abort_flag, a.error_word, true)) break;
        // P arrived by the score CTA's stores (generic proxy): order them before
        // this thread's MMAs, which read shared memory through the async proxy
        fence_proxy_async_smem();
        const uint32_t* flags =
            reinterpret_cast<const uint32_t*>(smem + OFF_P + b * kPBufBytes + kPFlagOff);
        if (t > 0 && (flags[0] | flags[4] | flags[8] | flags[12])) {
          // the running max moved for some head: rescale O before adding tile t
          mma_commit_elect(bar(B_MMA_IDLE));
          if (!wait_bar_all(bar(B_MMA_IDLE), corr & 1u, abort_flag, a.error_word)) break;
          if (lane == 0) {
            *corr_tile = t;
            mbar_arrive(bar(B_CORR_REQ));
          }
          if (!wait_bar_all(bar(B_CORR_DONE), corr & 1u, abort_flag, a.error_word)) break;
          ++corr;
        }
        tc_fence_after();
        const uint64_t pd = pdesc0 + ((b * kPBufBytes) >> 4);
        const uint64_t vd = vdesc0 + ((s * kStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
#pragma unroll
          for (int half = 0; half < 2; ++half)
            mma_ss_elect(tm + TM_O + half * 256, pd + (uint64_t)((kk * 256) >> 4),
                         vd + (uint64_t)((half * 4 * kBlockBytes + kk * 2048) >> 4), kIdescPV,
                         (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit_elect(bar(B_KV_EMPTY + s));
        mma_commit_multicast_elect(bar(B_P_EMPTY + b), (uint16_t)0x1);  // P buffer b free (CTA 0)
      }
      if (lane == 0) {
        *corr_exit = 1;
        mbar_arrive(bar(B_CORR_REQ));  // releases the rescale warps
      }
      __syncwarp();
    }
    mma_commit_elect(bar(B_FINAL));
    wait_bar_all(bar(B_FINAL), 0, abort_flag, a.error_word);
    finish();
    return;
  } else if (warp >= kMathWarp0 && rank == 0) {
    // ================= softmax (CTA 0, warps 12..15, one thread per head) =================
    regs_set<kRegsMath>();
    const int h = tid - kMathWarp0 * 32;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // Q[h] -> TMEM columns TM_Q .. TM_Q+287 (pairs), zero for padded heads.
    // Swizzled rows: column block cb holds [128 rows][128 B]; 16-byte chunk c
    // of row h sits at chunk position c ^ (h % 8) (conflict-free reads).
    uint32_t qmax = 0;  // bf16 magnitudes seen (FP8 rows: Q must fit fp16)
    bool ok = wait_bar_all(bar(B_Q_SMEM), 0, abort_flag, a.error_word);
    if (ok) {
      for (int c0 = 0; c0 < kD / 2; c0 += 16) {
        uint32_t v[16];
        const unsigned char* blk = smem + q_block_off(c0 / 32) + h * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = (c0 % 32) / 4 + i;
          uint4 x = make_uint4(0, 0, 0, 0);
          if (h < a.H) x = *reinterpret_cast<const uint4*>(blk + ((c ^ (h & 7)) * 16));
          if (FP8) {  // the score MMA's operands are fp16
            qmax = max_u16x2(qmax, x.x & 0x7fff7fffu);
            qmax = max_u16x2(qmax, x.y & 0x7fff7fffu);
            qmax = max_u16x2(qmax, x.z & 0x7fff7fffu);
            qmax = max_u16x2(qmax, x.w & 0x7fff7fffu);
            x.x = bf16x2_to_f16x2(x.x);
            x.y = bf16x2_to_f16x2(x.y);
            x.z = bf16x2_to_f16x2(x.z);
            x.w = bf16x2_to_f16x2(x.w);
          }
          v[4 * i + 0] = x.x;
          v[4 * i + 1] = x.y;
          v[4 * i + 2] = x.z;
          v[4 * i + 3] = x.w;
        }
        tmem_st16(tm + lane_off + TM_Q + c0, v);
      }
      tmem_st_wait();
      if (FP8 && ValueLoader::overflow(qmax)) err |= HS_DEV_ERR_VALUE;
    }
    tc_fence_before();
    mbar_arrive(bar(B_Q_READY));
    ok = ok && wait_bar_all(bar(B_RID), 0, abort_flag, a.error_word);
    const uint32_t peer_p = mapa(sbase + OFF_P, 1);
    const uint32_t peer_pfull = mapa(bar(B_P_FULL), 1);
    const int wq = warp & 3;  // this warp's heads: 32 wq .. 32 wq + 31
    float m_used = -INFINITY, l_sum = 0.f;
    for (int t = 0; ok && t < n_tiles; ++t) {
      const int b = t % kSBufs;  // S buffer
      const uint32_t pb = (uint32_t)(t / kSBufs) & 1u;
      const int pbuf_i = t % kPBufs;  // P buffer
      const uint32_t ppar = (uint32_t)(t / kPBufs) & 1u;
      const uint64_t valid =
          (uint64_t)__ballot_sync(0xffffffffu, s_rid[t * kTile + lane] >= 0) |
          ((uint64_t)__ballot_sync(0xffffffffu, s_rid[t * kTile + lane + 32] >= 0) << 32);
      if (!wait_bar_all(bar(B_S_FULL + b), pb, abort_flag, a.error_word)) break;
      tc_fence_after();
      const uint32_t sa = tm + lane_off + TM_S + b * kTile;
      // One read of the tile's 64 scores from tensor memory: the tile max of
      // the raw scores (scale > 0 keeps the order; rows without a valid id do
      // not count), then the exponents from the same registers.
      uint32_t u[64];
      tmem_ld16p(sa, u);
      tmem_ld16p(sa + 16, u + 16);
      tmem_ld16p(sa + 32, u + 32);
      tmem_ld16p(sa + 48, u + 48);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(B_S_EMPTY + b));  // S buffer b read out
      float tmax = -INFINITY;
      if (valid == ~0ull) {
#pragma unroll
        for (int i = 0; i < 64; ++i) tmax = fmaxf(tmax, __uint_as_float(u[i]));
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if ((valid >> i) & 1) tmax = fmaxf(tmax, __uint_as_float(u[i]));
      }
      tmax *= a.scale_log2;
      // lazy rescale: move the reference max only when it grew by > 2^8
      const bool rescale = tmax > m_used + 8.f;
      float alpha = 1.f;
      if (rescale) {
        alpha = fast_exp2(m_used - tmax);  // 0 when m_used is -inf
        l_sum *= alpha;
        m_used = tmax;
      }
      // P buffer t % kPBufs is free once the value CTA finished tile t - kPBufs
      if (!wait_bar_all(bar(B_P_EMPTY + pbuf_i), ppar ^ 1u, abort_flag, a.error_word)) break;
      // the value CTA's P buffer and its barrier (cluster addresses)
      const uint32_t pbuf = peer_p + pbuf_i * kPBufBytes;
      const uint32_t pbar = peer_pfull + 8u * pbuf_i;
      // p = 2^(scale_log2 * x - m_used); invalid rows give p = 0.  m_used is -inf
      // only while no valid row has been seen, and then every p is 0.
      const float neg_m = -m_used;
      const uint64_t vb = m_used == -INFINITY ? 0ull : valid;
#pragma unroll
      for (int kbg = 0; kbg < 8; ++kbg) {
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = kbg * 8 + 2 * i;
          float p0 = fast_exp2(fmaf(__uint_as_float(u[j]), a.scale_log2, neg_m));
          float p1 = fast_exp2(fmaf(__uint_as_float(u[j + 1]), a.scale_log2, neg_m));
          p0 = ((vb >> j) & 1) ? p0 : 0.f;
          p1 = ((vb >> (j + 1)) & 1) ? p1 : 0.f;
          l_sum += p0 + p1;
          pk[i] = pack_f16x2(p0, p1);
        }
        // P [128 heads x 64 rows], K-major core matrices (head group, row group)
        const uint32_t off = (uint32_t)(((h >> 3) * (kTile / 8) + kbg) * 128 + (h & 7) * 16);
        st_async_v4(pbuf + off, make_uint4(pk[0], pk[1], pk[2], pk[3]), pbar);
      }
      st_async_b32(pbuf + kPAlphaOff + 4u * (uint32_t)h, __float_as_uint(alpha), pbar);
      const uint32_t any = __ballot_sync(0xffffffffu, rescale && t > 0);
      if (lane == 0) st_async_v4(pbuf + kPFlagOff + 16u * (uint32_t)wq, make_uint4(any, 0u, 0u, 0u), pbar);
    }
    // final m, l for this head -> value CTA
    st_cluster_f32(mapa(sbase + OFF_ML + 4 * h, 1), m_used);
    st_cluster_f32(mapa(sbase + OFF_ML + 512 + 4 * h, 1), l_sum);
    mbar_arrive_remote(mapa(bar(B_ML_FULL), 1));
    // wait until the value CTA released the last P buffers (its commits landed)
    for (int t = n_tiles - kPBufs; t < n_tiles; ++t) {
      if (t < 0) continue;
      wait_bar_all(bar(B_P_EMPTY + t % kPBufs), (uint32_t)(t / kPBufs) & 1u, abort_flag,
                   a.error_word);
    }
    finish();
    return;
  } else if (warp >= kMathWarp0) {
    // ================= rescale + epilogue (CTA 1, warps 12..15) =================
    regs_set<kRegsMath>();
    const int h = tid - kMathWarp0 * 32;  // head = TMEM lane
    const int wq = warp & 3;              // this warp's TMEM lane quarter (heads 32wq ..)
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    for (uint32_t k = 0;; ++k) {  // rare: only tiles where some head's max moved
      if (!wait_bar_all(bar(B_CORR_REQ), k & 1u, abort_flag, a.error_word)) break;
      if (*corr_exit) break;
      tc_fence_after();
      const int t = *corr_tile;
      const float alpha =
          reinterpret_cast<const float*>(smem + OFF_P + (t % kPBufs) * kPBufBytes + kPAlphaOff)[h];
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        for (int c = 0; c < kDV; c += 64) {
          uint32_t u0[16], u1[16], u2[16], u3[16];
          const uint32_t oa = tm + lane_off + TM_O + c;
          tmem_ld16(oa, u0);
          tmem_ld16(oa + 16, u1);
          tmem_ld16(oa + 32, u2);
          tmem_ld16(oa + 48, u3);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            u0[i] = __float_as_uint(__uint_as_float(u0[i]) * alpha);
            u1[i] = __float_as_uint(__uint_as_float(u1[i]) * alpha);
            u2[i] = __float_as_uint(__uint_as_float(u2[i]) * alpha);
            u3[i] = __float_as_uint(__uint_as_float(u3[i]) * alpha);
          }
          tmem_st16(oa, u0);
          tmem_st16(oa + 16, u1);
          tmem_st16(oa + 32, u2);
          tmem_st16(oa + 48, u3);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(B_CORR_DONE));
    }
    epilogue(2);
    finish();
    return;
  } else if (rank == 1 && !FP8 && warp == 2) {
    // ===== CTA 1, warp 2: the last kXBlocks column blocks of each K tile, gathered into CTA 0 =====
    // (multicast to CTA 0 alone; each lane 4 rows of one block, completing
    // CTA 0's KV_FULL barrier, once CTA 0's score MMAs released the stage)
    regs_set<kRegsWG0>();
    const int g = lane & 15, cbx = kCbK - kXBlocks + (lane >> 4);
    const bool issuer = (lane >> 4) < kXBlocks;
    if (wait_bar_all(bar(B_RID), 0, abort_flag, a.error_word)) {
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kStagesS;
        if (t == 1 && !wait_bar_all(bar(B_XQ), 0, abort_flag, a.error_word, true)) break;
        if (!wait_bar_all(bar(B_XEMPTY + s), ((uint32_t)(t / kStagesS) & 1u) ^ 1u, abort_flag,
                          a.error_word, true))
          break;
        if (issuer) {
          const int32_t* rid = s_rid + t * kTile + 4 * g;
          const int y0 = rid[0] >= 0 ? rid[0] : a.rows_in_layer;
          const int y1 = rid[1] >= 0 ? rid[1] : a.rows_in_layer;
          const int y2 = rid[2] >= 0 ? rid[2] : a.rows_in_layer;
          const int y3 = rid[3] >= 0 ? rid[3] : a.rows_in_layer;
          tma_gather4_mc(sbase + OFF_STAGE + s * kStageBytes + cbx * kBlockBytes + g * 512, &kv_map,
                         cbx * 64, y0, y1, y2, y3, bar(B_KV_FULL + s), (uint16_t)(1u << 0));
        }
        __syncwarp();
      }
    }
    finish();
    return;
  } else {
    regs_set<kRegsWG0>();  // idle warps of warpgroup 0
    finish();
    return;
  }
}

// Self-test of wait_bar's time limit: one thread waits on a barrier of its
// CTA that nothing arrives on, and gives up after timeout_ns.
__global__ void wait_selftest_kernel(int32_t* error_word, uint32_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bar(smem_u32(&bar), 0, &abort_flag, error_word, false, timeout_ns);
}

// Combine per-split normalised partials: o = sum_c w_c o_c / sum_c w_c with
// w_c = exp(lse_c - max lse).  A CTA covers four heads of one request, 64
// threads per head, each thread 8 columns (one 16-byte fp16 load per split).
constexpr int kMergeHeads = 4;
__global__ void __launch_bounds__(64 * kMergeHeads) merge_splits_kernel(
    const uint16_t* __restrict__ ws_o, const float* __restrict__ ws_lse, int splits, int H,
    uint16_t* __restrict__ out, float* __restrict__ lse_out) {
  // launched as a programmatic dependent of the decode kernel: wait for that
  // grid to complete and its partials to be visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int r = blockIdx.y, h = blockIdx.x * kMergeHeads + (threadIdx.x >> 6);
  if (h >= H) return;
  const int e0 = (threadIdx.x & 63) * 8;
  const float* lse_rh = ws_lse + (int64_t)r * splits * kHeads + h;
  const uint16_t* o_rh = ws_o + ((int64_t)r * splits * kHeads + h) * kDV + e0;
  // Splits in groups of four, each group's loads issued together: a running
  // max with the sums rescaled when it grows (with at most four splits, one
  // group: the plain max-then-weights sum).
  float mx = -INFINITY, wsum = 0.f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int c0 = 0; c0 < splits; c0 += 4) {
    float lc[4];
    uint4 o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u;
      lc[u] = c < splits ? lse_rh[(int64_t)c * kHeads] : -INFINITY;
      o[u] = c < splits ? __ldg(reinterpret_cast<const uint4*>(o_rh + (int64_t)c * kHeads * kDV))
                        : make_uint4(0u, 0u, 0u, 0u);
    }
    float m_new = mx;
#pragma unroll
    for (int u = 0; u < 4; ++u) m_new = fmaxf(m_new, lc[u]);
    if (mx != -INFINITY && m_new > mx) {  // rescale what earlier groups summed
      const float k = expf(mx - m_new);
      wsum *= k;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= k;
    }
    mx = m_new;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = lc[u] == -INFINITY ? 0.f : expf(lc[u] - mx);
      wsum += w;
      const uint32_t wd[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wd[i]));
        acc[2 * i] += w * f.x;
        acc[2 * i + 1] += w * f.y;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint4 pk;
  pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
  pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(out + ((int64_t)r * H + h) * kDV + e0) = pk;
  if (lse_out && (threadIdx.x & 63) == 0)
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

// TMA tensor map over bf16 [rows][576], 128B swizzle, box = 64 columns x
// box_rows (128: one request's queries; 1: KV rows for the 4-row gathers).
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

// Launch the decode kernel (+ the merge when splits > 1).  Arguments checked by
// the caller; kv_map is not read for FP8 rows.
hs_status launch_decode(AttnArgs& a, const CUtensorMap& kv_map, const void* q, int R,
                        cudaStream_t s, bool fp8 = false) {
  CUtensorMap q_map;  // host-side encode only: safe inside stream capture
  if (encode_rows_map(&q_map, q, (uint64_t)R * a.H, kHeads) != HS_OK) return HS_ERR_INVALID;
  const int tiles = (a.K + kTile - 1) / kTile;
  a.rows_per_split = ((tiles + a.splits - 1) / a.splits) * kTile;
  if (fp8)
    mla_decode_kernel<true><<<dim3(2 * a.splits, R), kThreads, kSmemBytes, s>>>(kv_map, q_map, a);
  else
    mla_decode_kernel<false><<<dim3(2 * a.splits, R), kThreads, kSmemBytes, s>>>(kv_map, q_map, a);
  HS_CUDA_TRY(cudaGetLastError());
  if (a.splits > 1) {
    // programmatic dependent launch: the merge grid is set up while the
    // decode kernel runs (1.5 us per call of 32 requests x 2048 rows)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.H + kMergeHeads - 1) / kMergeHeads, R);
    cfg.blockDim = dim3(64 * kMergeHeads);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    HS_CUDA_TRY(cudaLaunchKernelEx(&cfg, merge_splits_kernel, (const uint16_t*)a.ws_o,
                                   (const float*)a.ws_lse, a.splits, a.H, a.out, a.lse));
    HS_CUDA_TRY(cudaGetLastError());
  }
  return HS_OK;
}

// First row of `layer` in the device pool (rows of hs_row_bytes each).
const uint4* layer_rows(const hs_pool* p, int32_t layer, int64_t rows_in_layer) {
  return reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(p->kv_pool) +
                                        (int64_t)layer * rows_in_layer * hs_row_bytes(p->d));
}

}  // namespace

hs_status hs_attn_workspace_init(hs_pool* p) {
  p->attn_o = nullptr;
  p->attn_ml = nullptr;
  p->attn_max_splits = 0;
  p->attn_kv_maps = nullptr;
  // attention needs 576-wide rows (bf16, or FP8 whose pool validation fixes
  // 576); the decode calls reject other pools
  if (p->d.row_elems != kD) return HS_OK;
  const bool fp8 = p->d.kv_format == HS_KV_FP8;
  if (fp8)
    HS_CUDA_TRY(cudaFuncSetAttribute(mla_decode_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
  else
    HS_CUDA_TRY(cudaFuncSetAttribute(mla_decode_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
  const int64_t rows_in_layer = p->blocks_per_layer * p->d.page_tokens;
  CUtensorMap* maps = new (std::nothrow) CUtensorMap[p->d.num_layers];
  if (!maps) return HS_ERR_OOM;
  p->attn_kv_maps = maps;
  if (fp8) memset(maps, 0, sizeof(CUtensorMap) * p->d.num_layers);  // FP8 rows need no maps
  for (int l = 0; !fp8 && l < p->d.num_layers; ++l) {
    const void* base = static_cast<const uint16_t*>(p->kv_pool) + (int64_t)l * rows_in_layer * kD;
    const hs_status st = encode_rows_map(&maps[l], base, (uint64_t)rows_in_layer, 1);
    if (st != HS_OK) return st;
  }
  const int splits = choose_splits(p->num_sms, p->d.num_requests, p->d.top_k);
  p->attn_max_splits = splits;
  if (splits > 1) {
    const size_t n = (size_t)p->d.num_requests * splits * kHeads;
    if (cudaMalloc(&p->attn_o, n * kDV * sizeof(uint16_t)) != cudaSuccess ||
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

// Decode rows of one layer: the T verify tokens of R requests are R * T
// independent decode rows of the same kernel (T = 1 outside speculative
// decoding), each with its own query and its own K rows.  Their K splits are
// the kernel's choice for R * T rows, capped so that the partials fit the
// pool's workspace (R x its splits) and, if max_splits > 0, at max_splits.
hs_status hs_launch_attention_tokens(hs_pool* p, int32_t layer, int32_t num_tokens, const void* q,
                                     const int32_t* row_ids, int32_t num_heads, int32_t v_dim,
                                     float scale, void* out, float* lse, int max_splits,
                                     cudaStream_t stream) {
  if (!p || !q || !row_ids || !out || num_tokens <= 0) return HS_ERR_INVALID;
  if (layer < 0 || layer >= p->d.num_layers || num_heads <= 0 || num_heads > kHeads ||
      v_dim != kDV || p->d.row_elems != kD || !(scale > 0.f) || p->attn_max_splits < 1 ||
      !p->attn_kv_maps)
    return HS_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return HS_ERR_INVALID;
  const int64_t rows_in_layer = p->blocks_per_layer * p->d.page_tokens;
  const int64_t n = (int64_t)p->d.num_requests * num_tokens;  // decode rows
  if (rows_in_layer > INT32_MAX || n > 65535) return HS_ERR_INVALID;
  const int tiles = (p->d.top_k + kTile - 1) / kTile;
  const int min_splits = (tiles * kTile + kMaxSplitRows - 1) / kMaxSplitRows;
  int splits = choose_splits(p->num_sms, (int)n, p->d.top_k);
  const int fit = p->attn_max_splits / num_tokens;  // partials the workspace holds per row
  if (splits > 1 && splits > fit) splits = fit > min_splits ? fit : min_splits;
  if (max_splits > 0 && max_splits < splits) splits = max_splits > min_splits ? max_splits : min_splits;
  if (splits > 1 && n * splits > (int64_t)p->d.num_requests * p->attn_max_splits)
    return HS_ERR_INVALID;  // K too long for this many rows in the workspace
  AttnArgs a;
  a.kv = layer_rows(p, layer, rows_in_layer);
  a.row_ids = row_ids;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.ws_o = p->attn_o;
  a.ws_lse = p->attn_ml;
  a.error_word = p->error_word;
  a.rows_in_layer = (int32_t)rows_in_layer;
  a.K = p->d.top_k;
  a.H = num_heads;
  a.splits = splits;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_decode(a, static_cast<const CUtensorMap*>(p->attn_kv_maps)[layer], q, (int)n,
                       stream, p->d.kv_format == HS_KV_FP8);
}

hs_status hs_launch_attention(hs_pool* p, int32_t layer, const void* q, const int32_t* row_ids,
                              int32_t num_heads, int32_t v_dim, float scale, void* out, float* lse,
                              int max_splits, cudaStream_t stream) {
  return hs_launch_attention_tokens(p, layer, 1, q, row_ids, num_heads, v_dim, scale, out, lse,
                                    max_splits, stream);
}

extern "C" hs_status hs_sparse_mla_decode(hs_pool* p, int32_t layer, const void* q,
                                          const int32_t* row_ids, int32_t num_heads, int32_t v_dim,
                                          float scale, void* out, float* lse, void* stream) {
  return hs_launch_attention(p, layer, q, row_ids, num_heads, v_dim, scale, out, lse, 0,
                             hs_stream(stream));
}

extern "C" hs_status hs_sparse_mla_decode_tokens(hs_pool* p, int32_t layer, int32_t num_tokens,
                                                 const void* q, const int32_t* row_ids,
                                                 int32_t num_heads, int32_t v_dim, float scale,
                                                 void* out, float* lse, void* stream) {
  return hs_launch_attention_tokens(p, layer, num_tokens, q, row_ids, num_heads, v_dim, scale, out,
                                    lse, 0, hs_stream(stream));
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
// outputs and their log-sum-exp) in the fixed device arrays below, which every
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
constexpr int kNoAllocMaxUnits = 64;  // 64 x 128 x 512 fp16 = 8 MiB, + 32 KiB of lse
static __device__ __align__(256) uint16_t g_noalloc_o[kNoAllocMaxUnits * kHeads * kDV];
static __device__ __align__(256) float g_noalloc_lse[kNoAllocMaxUnits * kHeads];
static __device__ int32_t g_noalloc_error_word;

namespace {
constexpr int kMaxDevices = 64;
uint16_t* g_noalloc_o_ptr[kMaxDevices];  // device addresses of the scratch, per device
float* g_noalloc_lse_ptr[kMaxDevices];
int32_t* g_noalloc_err_ptr[kMaxDevices];
int g_noalloc_sms[kMaxDevices];

// Once per device, with that device current: resolve the scratch's device
// address (in host code the array's name is only a stand-in, not an address)
// and raise the kernel's shared-memory limit.
hs_status noalloc_setup(int dev) {
  if (g_noalloc_o_ptr[dev]) return HS_OK;
  void* scratch_o = nullptr;
  void* scratch_lse = nullptr;
  void* errw = nullptr;
  HS_CUDA_TRY(cudaGetSymbolAddress(&scratch_o, g_noalloc_o));
  HS_CUDA_TRY(cudaGetSymbolAddress(&scratch_lse, g_noalloc_lse));
  HS_CUDA_TRY(cudaGetSymbolAddress(&errw, g_noalloc_error_word));
  HS_CUDA_TRY(cudaFuncSetAttribute(mla_decode_kernel<false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
  int sms = 0;
  HS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  g_noalloc_sms[dev] = sms;
  g_noalloc_err_ptr[dev] = static_cast<int32_t*>(errw);
  g_noalloc_lse_ptr[dev] = static_cast<float*>(scratch_lse);
  g_noalloc_o_ptr[dev] = static_cast<uint16_t*>(scratch_o);
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
  CUtensorMap kv_map;  // host-side encode only
  if (encode_rows_map(&kv_map, kv_rows, (uint64_t)num_rows, 1) != HS_OK) return HS_ERR_INVALID;
  AttnArgs a;
  a.kv = static_cast<const uint4*>(kv_rows);
  a.row_ids = row_ids;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.ws_o = g_noalloc_o_ptr[dev];
  a.ws_lse = g_noalloc_lse_ptr[dev];
  a.error_word = g_noalloc_err_ptr[dev];
  a.rows_in_layer = (int32_t)num_rows;
  a.K = top_k;
  a.H = num_heads;
  a.splits = splits;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_decode(a, kv_map, q, num_requests, hs_stream(stream));
}

extern "C" hs_status hs_noalloc_check_errors(int32_t* code_out) {
  int dev = 0;
  HS_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_INVALID;
  const hs_status st = noalloc_setup(dev);
  if (st != HS_OK) return st;
  HS_CUDA_TRY(cudaDeviceSynchronize());
  int32_t code = 0;
  HS_CUDA_TRY(cudaMemcpy(&code, g_noalloc_err_ptr[dev], sizeof(code), cudaMemcpyDeviceToHost));
  const int32_t zero = 0;
  HS_CUDA_TRY(cudaMemcpy(g_noalloc_err_ptr[dev], &zero, sizeof(zero), cudaMemcpyHostToDevice));
  if (code_out) *code_out = code;
  return code ? HS_ERR_DEVICE : HS_OK;
}

extern "C" hs_status hs_selftest_bounded_waits(int64_t timeout_ns, int32_t* result, void* stream) {
  if (!result || timeout_ns <= 0 || timeout_ns > 100000000) return HS_ERR_INVALID;
  cudaStream_t st = hs_stream(stream);
  HS_CUDA_TRY(cudaMemsetAsync(result, 0, 2 * sizeof(int32_t), st));
  wait_selftest_kernel<<<1, 32, 0, st>>>(result, (uint32_t)timeout_ns);
  HS_CUDA_TRY(cudaGetLastError());
  return hs_launch_peer_wait_selftest(result + 1, (uint64_t)timeout_ns, st);
}
