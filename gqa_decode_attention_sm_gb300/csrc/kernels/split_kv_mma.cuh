// Stage 1 of GQA decode with the QK^T and P.V contractions on the tensor cores.
//
// Work comes in pieces: tokens [t_begin, t_end) of one (batch row b, KV head g)
// row, served for the 4 query heads of that KV head, so every K/V byte below
// the length is read from HBM exactly once.  Two schedules:
//   one piece per CTA — grid (8, B, splits), CTA (g, b, s) takes chunk s of
//     row (b, g); batches above kBalMaxBatch and grids of at most one wave;
//   balanced — one CTA per resident slot; the tiles of all rows (each row
//     start weighing one more tile when some row is shorter than a run)
//     form one stream and each CTA takes an equal run of it (lengths read on
//     the device), cut into pieces at row ends.
// A piece that is its row's only one writes the normalised output; the
// others write FP32 partials that stage 2 merges, or, in a one-wave grid of
// 2..8 splits launched as thread-block clusters, merge on chip through
// distributed shared memory (cluster_merge_tail).  A producer warp streams
// 16 KB K and V tiles with 1-D bulk copies (TMA unit) into an mbarrier ring,
// copying only rows below the length, straight from one piece into the next.
// The contractions run on the tensor cores because ncu showed an
// FP32 CUDA-core version of the same kernel to be instruction-bound (about 75
// warp instructions per token and KV head; on e4m3 KV, short-scoreboard stalls
// held DRAM throughput near a quarter of peak); this version executes about
// 21, and the kernel streams at the HBM roofline.
//
// Consumers: 4 warps, each owning 16-token slabs of the tile.  Per slab:
//   scores  S^T[16 tokens x 8] = K[16 x 128] . Q^T[128 x 8] as 8 mma.sync
//           m16n8k16 (FP32 accumulate).  Tokens are the M dimension and the 4
//           query heads fill half of N = 8 (columns 4..7 are zero padding).
//           The dims are permuted consistently in K and Q so each lane reads
//           whole 16-byte chunks of its K rows straight from the row-major
//           tile (no swizzle, no transpose).
//   softmax online, in the log2 domain (ex2), per head; the running max is
//           shared by the 8 lanes that hold a head (xor shuffles); the
//           accumulator is rescaled only when a max grows (warp vote).
//   output  O^T[128 dims x 8] += V^T[128 x 16 tokens] . P^T[16 x 8] as 8 mma
//           (one per 16-dim m-tile).  Each lane reads 16 contiguous dims of 4
//           token rows and pairs tokens with byte permutes; P^T reaches the
//           B-fragment layout by two 8x8 transposes (movmatrix).  bf16 P is split into a
//           high and a low bf16 part (two mma) so the weights keep ~16 bits.
// e4m3 K/V are widened with the hardware cvt (e4m3x2 -> f16x2, exact), int8
// codes with byte permutes to the f16 integer code + 1152 (exact); the
// offset comes off the scores (1152 * sum_d q_d per column, in the scale
// step) and off the output accumulator (1152 * the column's summed f16
// weights, every 16 tiles and at the piece's end); the tensor-core
// type is then f16 and a bf16 q is converted to f16 once per piece after a
// power-of-two scaling per query column (its largest magnitude brought to
// [2^14, 2^15), the inverse folded into that column's score scale), so any
// finite bf16 q is taken exactly down to 2^-31 of its column's maximum and
// nothing saturates.  fp16 and bf16 KV use their own type.  For the int8
// cache ("Qwen3-VL official BF16 on Jetson Orin (SM87)" docs, "INT8 KV cache
// (kv_mode)": a bf16 scale for each (position, KV head) row) the K row scale
// multiplies that token's scores and the V row scale joins that token's
// weight in P; the scales of slots past the length are never read.
//
// Sources: "FlashInfer sm110_gqa_decode" article ("Convenience API": log2-domain
// softmax with the host-folded scale q_scale/sqrt(128)/ln 2 and ex2;
// "num_splits": FP32 split partials merged by a separate step); "FP8 KV cache
// port on Jetson AGX Thor" blog, section 1 patch 2 (fp8 tile promoted before
// the dot product, k_scale on scores, v_scale on the output).
#pragma once

#include "common.cuh"

namespace gqa {

constexpr int kStageBytes = 2 * 16384;  // one K tile + one V tile (16 KB each)

struct SplitParams {
  const void* q;          // [B,32,128] fp16/bf16
  const void* kv;         // [B,2,8,C,128] fp16/bf16/e4m3/int8
  const uint16_t* kv_scales;  // int8 cache: bf16 [B or num_pages, 2, 8, C or page size], one scale per row
  const int32_t* lens;    // [B]
  void* out;              // [B,32,128], written by pieces that are their row's only one
  float* part_o;          // [B,32,S,128] unnormalised accumulator
  float* part_m;          // [B,32,S]  running max, log2 domain
  float* part_l;          // [B,32,S]  softmax denominator
  uint32_t* flags;        // workspace status word
  int batch, capacity, num_splits, chunk, splits_eff;
  // q and out are [B, q_len, 32, 128]; query j attends slots [0, len - q_len + j]
  // (q_len = 1: plain decode); partials are indexed by (b * q_len + j, head)
  float scale_log2;       // q_scale * k_scale * log2(e) / sqrt(128)
  float v_scale;
  uint64_t wait_budget_ns;  // every pipeline wait gives up after this long
  int skip_tile;            // test hook: tile index whose copies are never issued (-1: none)
  // paged cache (block_table != nullptr): kv is a pool [num_pages, 2, 8, 2^page_log2, 128];
  // slot t of batch row b lives in page block_table[b * max_pages + (t >> page_log2)]
  const int32_t* block_table;
  int page_log2, max_pages, num_pages;
  // balanced schedule: the least number of tiles a CTA takes (so that no row
  // is cut into more pieces than the workspace has split slots)
  int bal_q_min;
  // byte extents of the cache (or page pool) and of its int8 row scales, for
  // the range checks of checked builds
  size_t kv_bytes, scales_bytes;
};

// Row r of q, out or the partials ((b * q_len + j) * 32 + head): checked
// builds report a row outside the batch and redirect it to row 0.
__device__ __forceinline__ size_t checked_row(const SplitParams& p, int nq, size_t row) {
  if constexpr (kChecked) {
    if (row >= (size_t)p.batch * nq * kHq) {
      atomicOr(p.flags, GQA_FLAG_BOUNDS);
      return 0;
    }
  }
  return row;
}

template <int QF>
__device__ __forceinline__ uint32_t pack_out(float a, float b) {
  if constexpr (QF == kQF16) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

constexpr int kMmaConsumerWarps = 4;
constexpr int kMmaThreads = (kMmaConsumerWarps + 1) * 32;
// Ring depth and residency: 8-bit KV does twice the arithmetic per byte, and
// with one or two query tokens (8 mma columns) it fits in <= 128 registers
// without spills, so 3 CTAs of 2 stages share an SM (more warps to hide
// latency); 16-bit KV and longer verify windows use 3 stages at 2 CTAs per
// SM (measured: bf16 streams fastest so, e4m3 is 2-3 % faster at 3 CTAs).
// (A warp's registers come from one quarter of the SM's register file: 3
// CTAs of 5 warps put 4 warps on some quarter, 128 registers each at most;
// 2 CTAs put 3, 168 at most.)
__host__ __device__ constexpr int mma_stages(int kvf, int nq) { return is_8bit(kvf) && nq <= 2 ? 2 : 3; }
__host__ __device__ constexpr int mma_ctas_per_sm(int kvf, int nq) { return is_8bit(kvf) && nq <= 2 ? 3 : 2; }
constexpr int kMaxQLen = 4;  // query tokens per request (a verify window when > 1)
constexpr int kScaleStageBytes = 2 * 128 * 2;  // int8 cache: K and V row scales of one 128-token tile
// Balanced schedule: batches up to this size (every CTA's prologue scans the
// lengths).  Its merge area sits outside the ring, which keeps streaming the
// next piece while the consumers merge the last: [4 warps][4 heads][128 + 2],
// one query token of a window at a time.
constexpr int kBalMaxBatch = 1024;
constexpr int kBalMergeBytes = kMmaConsumerWarps * kGroup * (kD + 2) * 4;
static_assert((kMmaThreads + 3 + kBalMaxBatch) * 4 <= kBalMergeBytes, "the length scan uses the merge area");
// the balanced cursor's slot of 16 ints per warp (its state and the current
// piece's output coordinates), after the merge area
constexpr int kBalRunBytes = (kMmaConsumerWarps + 1) * 16 * 4;
// 3- and 4-token windows over 8-bit caches keep their Q^T fragments in
// shared memory, one copy per CTA ([k-step][lane][n-tile][2 words]; in the
// balanced schedule's merge area, idle while a piece streams, else after the
// ring's barriers): 32 registers fewer, so each warp can take two slabs of a
// tile together without spills.
__host__ __device__ constexpr bool mma_q_in_smem(int kvf, int nq) { return is_8bit(kvf) && nq > 2; }
constexpr int kQSmemBytes = 8 * 32 * 2 * 2 * 4;
__host__ __device__ constexpr int mma_smem_bytes(int kvf, int nq, bool bal = false) {
  return mma_stages(kvf, nq) * (kStageBytes + kScaleStageBytes + 2 * 8) + (bal ? kBalMergeBytes + kBalRunBytes : 0) +
         (!bal && mma_q_in_smem(kvf, nq) ? kQSmemBytes : 0);
}
static_assert(kQSmemBytes <= kBalMergeBytes, "the Q^T fragments fit the merge area");
// 228 KB of shared memory per SM, 1 KB of it reserved per resident CTA
static_assert(2 * (mma_smem_bytes(kKvF16, kMaxQLen, true) + 1024) <= 228 * 1024 &&
                  2 * (mma_smem_bytes(kKvF16, 1, true) + 1024) <= 228 * 1024 &&
                  3 * (mma_smem_bytes(kKvE4M3, 1, true) + 1024) <= 228 * 1024 &&
                  3 * (mma_smem_bytes(kKvE4M3, 2, true) + 1024) <= 228 * 1024 &&
                  2 * (mma_smem_bytes(kKvE4M3, kMaxQLen, true) + 1024) <= 228 * 1024,
              "the balanced schedule keeps its residency");
// With one piece per CTA the epilogue merges the 4 warps' states in the ring
// (idle by then): [warp][column][128] accumulators + [warp][column] max and
// denominator.
static_assert(kMmaConsumerWarps * kGroup * 2 * (kD + 2) * 4 <= mma_stages(kKvE4M3, 2) * kStageBytes &&
                  kMmaConsumerWarps * kGroup * kMaxQLen * (kD + 2) * 4 <= mma_stages(kKvF16, kMaxQLen) * kStageBytes,
              "merge area must fit in the ring");

// ... and the cluster merge's state [column][128] + max + denominator after it.
static_assert(kMmaConsumerWarps * kGroup * kMaxQLen * (kD + 2) * 4 + kGroup * kMaxQLen * (kD + 2) * 4 <=
                      mma_stages(kKvF16, kMaxQLen) * kStageBytes &&
                  kMmaConsumerWarps * kGroup * 2 * (kD + 2) * 4 + kGroup * 2 * (kD + 2) * 4 <=
                      mma_stages(kKvE4M3, 2) * kStageBytes,
              "cluster merge state must fit in the ring");

// ---------------------------------------------------------------- mma.sync

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Transpose of an 8x8 matrix of 16-bit elements spread over the warp, lane i
// holding row i/4, columns 2(i%4) and 2(i%4)+1 (low half first): lane i gets
// row i/4 of the transpose.  The score accumulator's packed weights (rows =
// tokens, columns = query columns) become the P^T B-fragment this way.
__device__ __forceinline__ uint32_t transpose8x8_b16(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// 16 bytes of this CTA's shared memory, loaded where the code reads them
// (volatile: never hoisted into registers held across the loop)
__device__ __forceinline__ uint4 ld_shared_u4(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (lo, hi) -> packed pair, round to nearest even.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16_satfinite(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float bf16_lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Four 8-bit KV elements (bytes b0..b3 of w) -> f16x2 pairs (b0,b1), (b2,b3),
// exactly: hardware cvt for e4m3, byte-permute + subtract for int8 codes.
template <int KVF>
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (KVF == kKvI8) {
    i8x4_to_f16x2x2(w, lo, hi);
  } else {
    lo = e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
    hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
  }
}

// Tensor-core operands from 8-bit K and V: int8 codes enter as code + 1152
// (one f16 subtraction per pair saved); the consumer takes the offset off
// the scores (1152 * sum_d q_d per column, in the scale step) and off the
// output accumulator (1152 * the column's summed weights, take_v_bias).  e4m3
// as widen4.
template <int KVF>
__device__ __forceinline__ void widen4_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (KVF == kKvI8) i8x4_to_f16x2x2_biased(w, lo, hi);
  else widen4<KVF>(w, lo, hi);
}

// int8 V: o holds O + 1152 * (summed weights) per column; vw[nt][c] is this
// lane's share of the weights of column 2cq + c (its tokens gq, gq + 8 of
// every slab since the last call).  Sum the shares over the 8 lanes holding
// each column, take 1152 times that off every accumulator of the column and
// start again.
template <int kNT>
__device__ __forceinline__ void take_v_bias(float (&o)[kNT][8][4], float (&vw)[kNT][2]) {
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    float s0 = vw[nt][0], s1 = vw[nt][1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, off);
      s1 += __shfl_xor_sync(0xffffffffu, s1, off);
    }
    const float c0 = -kI8Bias * s0, c1 = -kI8Bias * s1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[nt][mt][0] += c0;
      o[nt][mt][2] += c0;
      o[nt][mt][1] += c1;
      o[nt][mt][3] += c1;
    }
    vw[nt][0] = vw[nt][1] = 0.f;
  }
}

// Tensor-core element type: bf16 for bf16 KV, f16 otherwise (8-bit KV widens to f16).
template <int KVF>
constexpr bool kMmaBF16 = KVF == kKvBF16;

// ------------------------------------------------------------ dim mapping
//
// Lane (gq = lane/4, cq = lane%4).  QK A-fragment registers for k-step ks:
//   a0 = K[row gq][kp = 2cq, 2cq+1], a2 = K[row gq][kp = 2cq+8, 2cq+9]
//   (a1, a3: row gq+8).  Logical (ks, kp) maps to physical dims:
//   2-byte KV: lane cq reads 16-byte chunks cq + 4i (i = 0..3, 8 dims each);
//              ks = 2i + h covers chunk dims 4h..4h+3 (a0 <- 4h,4h+1; a2 <- 4h+2,4h+3)
//   e4m3 KV:   lane cq reads 16-byte chunks cq + 4i (i = 0..1, 16 dims each);
//              ks = 4i + s covers chunk dims 4s..4s+3 (a0 <- 4s,4s+1; a2 <- 4s+2,4s+3)
// The Q^T B-fragment (b0 = Q[head gq][kp 2cq,2cq+1], b1 = [2cq+8, 2cq+9]) uses
// the same map, so the dot products are unchanged.
template <int KVF>
__device__ __forceinline__ int qk_dim(int cq, int ks, int pair /*0: a0/b0, 1: a2/b1*/) {
  if constexpr (is_8bit(KVF)) return 16 * (cq + 4 * (ks >> 2)) + 4 * (ks & 3) + 2 * pair;
  else return 8 * (cq + 4 * (ks >> 1)) + 4 * (ks & 1) + 2 * pair;
}

// ------------------------------------------------------------ work pieces

// Tokens [t_begin, t_end) of row (b, KV head g) (L = the row's length).  Its
// FP32 partials go to split slot `slot`; a piece that is its row's only one
// (`direct`) writes the normalised output itself.
struct Piece {
  int b, g, L, t_begin, t_end, slot;
  bool direct;
};

template <int kTile, bool BAL>
struct PieceCursor;

// One piece per CTA (grid = KV heads x batch x splits).
template <int kTile>
struct PieceCursor<kTile, false> {
  Piece one;
  bool pending = false;
  __device__ void start_single(int b, int g, int L, int t_begin, int t_end, int slot, bool direct) {
    one = Piece{b, g, L, t_begin, t_end, slot, direct};
    pending = true;
  }
  __device__ bool next(Piece& pc, const SplitParams&) {
    if (!pending) return false;
    pc = one;
    pending = false;
    return true;
  }
  __device__ void reload(Piece&) const {}
};

// Balanced schedule: the CTA's positions [x, x1) of the global stream.  Rows
// r = 8b + g come in order; a row of n tiles occupies w = n + rc positions
// (none without tokens), the first rc (the row cost) for the fixed cost of a
// piece, so a CTA whose run crosses many row starts takes fewer tiles.  Row
// r's first tile sits at stream position tf = 8 pb + g w + rc (pb: positions
// per KV head of the rows before b); CTA c holds its piece number
// c - floor(tf / q), and the row has floor((tf + n - 1) / q) - floor(tf / q) + 1
// pieces.

// The cursor rests on rows that hold tokens, so the row cost is wb - nb.
// The lengths, batch and capacity are read from the kernel parameters.  Each
// warp walks its own copy, kept in the warp's slot of shared memory and read
// and written only when the warp moves to its next piece, not in registers
// held through the streaming loop; every lane of the warp calls start and
// next with the same values and writes the same words.  The slot also holds
// the current piece's output coordinates, so a consumer warp drops them
// from its registers while it streams the piece and reads them back for the
// epilogue (reload).
//
// At the 168-register cap of the 3-4-token window kernels this took their
// spills from 4-68 bytes to 0-8.  Cold on GB300, us per call, before ->
// after: e4m3 64 x U[16k, 32k] with 3 / 4 tokens 503.8 / 505.9 -> 483.3 /
// 491.5, int8 of that shape 602.1 / 616.5 -> 577.5 / 598.0, bf16 256 x
// U[1, 4096] 346.1 / 358.4 -> 333.8 / 344.1; 1- and 2-token kernels (no
// spills either way) within 1 %.  With the state alone in shared memory and
// the coordinates in registers, the int8 3-token window was slower (614.4).
enum {
  kCurB, kCurG, kCurJ, kCurNb, kCurWb, kCurL, kCurLNext, kCurPb, kCurX, kCurX1, kCurQ,
  kCurPcB, kCurPcG, kCurPcSlot, kCurPcDirect,  // the current piece's fields the epilogue needs
  kCurSlotInts = 16
};
static_assert(kBalRunBytes == (kMmaConsumerWarps + 1) * kCurSlotInts * 4, "one cursor slot per warp");

template <int kTile>
struct PieceCursor<kTile, true> {
  enum { kB = kCurB, kG = kCurG, kJ = kCurJ, kNb = kCurNb, kWb = kCurWb, kL = kCurL, kLNext = kCurLNext,
         kPb = kCurPb, kX = kCurX, kX1 = kCurX1, kQ = kCurQ };
  volatile int* st;  // this warp's slot
  __device__ void start(int b0, int pb0, int L0, int L1, int x0, int x1, int q, int rc, int* slot) {
    st = slot;
    const int nb = (L0 + kTile - 1) / kTile, wb = bal_row_positions(nb, rc);
    const int within = x0 - kHkv * pb0;
    const int g = within / wb;
    st[kB] = b0;
    st[kG] = g;
    st[kJ] = within - g * wb;  // position in the row; [0, rc) stand for the piece cost
    st[kNb] = nb;
    st[kWb] = wb;
    st[kL] = L0;
    st[kLNext] = L1;  // clamped length of row b0 + 1 (0 past the batch)
    st[kPb] = pb0;
    st[kX] = x0;
    st[kX1] = x1;
    st[kQ] = q;
  }
  __device__ bool next(Piece& pc, const SplitParams& p) {
    const int cta = blockIdx.x;
    int b = st[kB], g = st[kG], j = st[kJ], nb = st[kNb], wb = st[kWb], L = st[kL], L_next = st[kLNext],
        pb = st[kPb], x = st[kX];
    const int x1 = st[kX1], q = st[kQ];
    __syncwarp();  // every lane has read the slot before any lane writes it
    bool found = false;
    while (x < x1) {
      const int rc = wb - nb;
      const int cnt = min(wb - j, x1 - x);
      const int r0 = max(j, rc), r1 = j + cnt;  // tile positions [r0, r1) of this run
      const bool has_tiles = r1 > r0;
      if (has_tiles) {
        const int tf = kHkv * pb + g * wb + rc;
        const int fq = tf / q;
        pc = Piece{b, g, L, (r0 - rc) * kTile, min(L, (r1 - rc) * kTile), cta - fq, (tf + nb - 1) / q == fq};
        st[kCurPcB] = pc.b;
        st[kCurPcG] = pc.g;
        st[kCurPcSlot] = pc.slot;
        st[kCurPcDirect] = pc.direct;
      }
      x += cnt;
      j += cnt;
      if (j == wb) {
        j = 0;
        if (++g == kHkv) {
          g = 0;
          pb += wb;
          while (x < x1) {  // the next row that holds tokens; its successor's
            ++b;              // length is loaded a whole piece ahead of its use
            L = L_next;
            nb = (L + kTile - 1) / kTile;
            wb = bal_row_positions(nb, rc);
            L_next = b + 1 < p.batch ? min(max(__ldg(p.lens + b + 1), 0), p.capacity) : 0;
            if (wb > 0) break;
          }
        }
      }
      if (has_tiles) {
        found = true;
        break;
      }
    }
    st[kB] = b;
    st[kG] = g;
    st[kJ] = j;
    st[kNb] = nb;
    st[kWb] = wb;
    st[kL] = L;
    st[kLNext] = L_next;
    st[kPb] = pb;
    st[kX] = x;
    return found;
  }
  __device__ void reload(Piece& pc) const {
    pc.b = st[kCurPcB];
    pc.g = st[kCurPcG];
    pc.slot = st[kCurPcSlot];
    pc.direct = st[kCurPcDirect] != 0;
  }
};

// Cluster merge (one-piece grid whose splits form one thread-block cluster
// per (b, KV head)): each CTA has left its merged state — unnormalised output
// st[col][128], running max st_m[col], denominator st_l[col], column
// col = 4 * query token + head — in its own shared memory.  After a cluster
// barrier, CTA r of the S in the cluster merges the (column, 4-dim) units
// u = r, r + S, ... by reading every CTA's state through distributed shared
// memory, in rank order (deterministic), and writes the output; a second
// barrier keeps every state alive until all reads are done.  All threads of
// every CTA call this exactly once.
template <int QF, int NQ>
__device__ __forceinline__ void cluster_merge_tail(const SplitParams& p, const float* st) {
  constexpr int kCols = kGroup * NQ;
  __syncwarp();  // the barrier's .aligned form wants each warp converged
  cluster_sync_all();
  if (threadIdx.x < kMmaConsumerWarps * 32) {
    const int S = (int)cluster_size(), r = (int)cluster_rank();
    const int b = blockIdx.y, g = blockIdx.x;
    const uint32_t base = smem_addr(st);
    for (int u = r + S * (int)threadIdx.x; u < kCols * 32; u += S * kMmaConsumerWarps * 32) {
      const int col = u >> 5, d0 = 4 * (u & 31);
      const uint32_t a_o = base + (uint32_t)(col * kD + d0) * 4u;
      const uint32_t a_m = base + (uint32_t)(kCols * kD + col) * 4u;
      const uint32_t a_l = a_m + (uint32_t)kCols * 4u;
      float M = -INFINITY;
      for (int k = 0; k < S; ++k) M = fmaxf(M, cluster_ld(cluster_map(a_m, k)));
      float Ls = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < S; ++k) {
        const float mk = cluster_ld(cluster_map(a_m, k));
        const float a = mk == -INFINITY ? 0.f : ex2(mk - M);  // a split without slots adds nothing
        Ls = fmaf(cluster_ld(cluster_map(a_l, k)), a, Ls);
        const float4 v = cluster_ld4(cluster_map(a_o, k));
        acc.x = fmaf(v.x, a, acc.x);
        acc.y = fmaf(v.y, a, acc.y);
        acc.z = fmaf(v.z, a, acc.z);
        acc.w = fmaf(v.w, a, acc.w);
      }
      const float inv = Ls > 0.f ? p.v_scale / Ls : 0.f;  // a query with no slot gets zeros
      const size_t row = checked_row(p, NQ, (size_t)(b * NQ + col / kGroup) * kHq + g * kGroup + col % kGroup);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + (row * kD + d0) * 2) =
          make_uint2(pack_out<QF>(acc.x * inv, acc.y * inv), pack_out<QF>(acc.z * inv, acc.w * inv));
    }
  }
  __syncwarp();
  cluster_sync_all();
}

// CL: the one-piece grid launched as clusters of its splits, merged on chip
// (cluster_merge_tail) instead of through partials and the combine kernel.
template <int KVF, int QF, int NQ, bool BAL, bool CL>
__global__ void __launch_bounds__(kMmaThreads, mma_ctas_per_sm(KVF, NQ))
    split_kv_mma_kernel(const __grid_constant__ SplitParams p) {
  constexpr int kMmaStages = mma_stages(KVF, NQ);
  using T = KvTraits<KVF>;
  constexpr bool kBF16 = kMmaBF16<KVF>;
  constexpr int kSlabs = T::kTile / (16 * kMmaConsumerWarps);  // 16-token slabs per warp per tile
  // Slabs taken together: two for 3- and 4-token windows over 8-bit caches,
  // which are latency-bound (more independent work between the max
  // reductions, half as many of them).  With the Q^T fragments in shared
  // memory (kQS) they fit the 168 registers with small spills; measured cold
  // at 64 x U[16k, 32k] on GB300, one slab -> pairs, us per call: e4m3 3 / 4
  // tokens 507.9 / 540.7 -> 503.8 / 507.9, int8 618.5 / 620.5 -> 602.1 /
  // 616.4 (pairs with Q in registers spilled more and made all but the e4m3
  // 4-token window slower).
  constexpr int kSG = is_8bit(KVF) && NQ > 2 ? 2 : 1;
  constexpr bool kQS = mma_q_in_smem(KVF, NQ);
  static_assert(kSlabs % kSG == 0, "whole slab groups");
  constexpr int kCols = kGroup * NQ;                            // (query token, head) columns
  constexpr int kNT = (kCols + 7) / 8;                          // 8-column mma n-tiles
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint16_t* scl = reinterpret_cast<uint16_t*>(smem + kMmaStages * kStageBytes);  // [stage][K|V][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(scl) + kMmaStages * kScaleStageBytes);
  uint64_t* empty = full + kMmaStages;
  static_assert(!(BAL && CL), "the cluster merge serves the one-piece grid");
  // epilogue merge area [4 warps][kRC][128] + max + denominator: in the idle
  // ring with one piece per CTA (all kCols columns in one round), after the
  // barriers with several (the ring is then still streaming the next piece;
  // one query token's 4 columns per round)
  constexpr int kRounds = BAL ? NQ : 1;
  constexpr int kRC = kCols / kRounds;  // columns merged per round
  float* mrg_acc = BAL ? reinterpret_cast<float*>(empty + kMmaStages) : reinterpret_cast<float*>(ring);
  float* mrg_m = mrg_acc + kMmaConsumerWarps * kRC * kD;             // [4][kRC]
  float* mrg_l = mrg_m + kMmaConsumerWarps * kRC;                    // [4][kRC]
  // cluster merge: this CTA's merged state [kCols][128] + max + denominator,
  // after the merge area in the idle ring
  float* cl_state = mrg_l + kMmaConsumerWarps * kRC;
  // balanced schedule: the cursor's slot of each warp
  int* cur_sm = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(mrg_acc) + kBalMergeBytes);
  uint32_t* qfr = reinterpret_cast<uint32_t*>(empty + kMmaStages);  // Q^T fragments (kQS)

  // Every CTA of this grid is resident or done: let the next grid in the
  // stream (stage 2, or the next launch after an on-chip merge) be scheduled;
  // it waits for this grid's completion before reading what this grid writes.
  pdl_launch_dependents();
  const int C = p.capacity;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {  // ring barriers first: the prologue below hides their initialisation
    for (int i = 0; i < kMmaStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kMmaConsumerWarps);
    }
    fence_barrier_init();
  }
  // Launched as a programmatic dependent of the previous grid in the stream:
  // wait for it (its writes, e.g. an appended token, must be visible) before
  // the first read of any input.  A no-op otherwise.
  pdl_wait_prior_grid();

  // ---- this CTA's pieces
  PieceCursor<T::kTile, BAL> cur;
  if constexpr (BAL) {
    // Balanced schedule: the positions of every (b, KV head) row, rows in
    // order, form one stream of 8 * sum_b w_b positions (w = tiles + rc for a
    // row that holds tokens); CTA c takes positions [c * Q, (c + 1) * Q) with
    // Q = max(ceil(total / grid), q_min).
    // Prefix sums of tiles and of rows with tokens over the batch, by all
    // threads, each over a contiguous block of rows, and the shortest row.
    // Scratch: the merge area, idle until the first epilogue — warp sums at
    // [0, 15), the first row and its prefix at [161, 163), the clamped lengths
    // from 163 on.
    int* scan = reinterpret_cast<int*>(mrg_acc);
    int* lsh = scan + kMmaThreads + 3;
    const int B = p.batch;
    const int per_t = (B + kMmaThreads - 1) / kMmaThreads;
    const int rb0 = min(B, (int)threadIdx.x * per_t), rb1 = min(B, rb0 + per_t);
    int mine_n = 0, mine_r = 0, mn = INT_MAX;
    bool clamped = false;
    for (int bb = rb0; bb < rb1; ++bb) {
      const int lr = __ldg(p.lens + bb);
      clamped |= lr < NQ || lr > C;  // a window of NQ queries needs NQ slots
      lsh[bb] = min(max(lr, 0), C);
      const int nb = (lsh[bb] + T::kTile - 1) / T::kTile;
      mine_n += nb;
      mine_r += nb > 0;
      if (nb > 0) mn = min(mn, nb);
    }
    if (clamped && blockIdx.x == 0) atomicOr(p.flags, GQA_FLAG_LENGTH_CLAMPED);
    // exclusive prefixes of the per-thread sums: scans within each warp, then
    // the sums of the warps before
    int incl_n = mine_n, incl_r = mine_r;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int tn = __shfl_up_sync(0xffffffffu, incl_n, off);
      const int tr = __shfl_up_sync(0xffffffffu, incl_r, off);
      if (lane >= off) {
        incl_n += tn;
        incl_r += tr;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    constexpr int kW = kMmaThreads / 32;
    if (lane == 31) {
      scan[warp] = incl_n;
      scan[kW + warp] = incl_r;
      scan[2 * kW + warp] = mn;
    }
    __syncthreads();
    int pre_n = incl_n - mine_n, pre_r = incl_r - mine_r, sum_n = 0, sum_r = 0, min_n = INT_MAX;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      if (w < warp) {
        pre_n += scan[w];
        pre_r += scan[kW + w];
      }
      sum_n += scan[w];
      sum_r += scan[kW + w];
      min_n = min(min_n, scan[2 * kW + w]);
    }
    const int rc = bal_row_cost(sum_n, min_n, (int)gridDim.x, p.bal_q_min);
    const int total = kHkv * (sum_n + rc * sum_r);
    const int q = max((total + (int)gridDim.x - 1) / (int)gridDim.x, p.bal_q_min);
    const int x0 = (int)blockIdx.x * q;
    int pre = pre_n + rc * pre_r;
    // the thread whose rows hold position x0 records the first row and its prefix
    if (x0 < total && kHkv * pre <= x0 && x0 < kHkv * (pre + mine_n + rc * mine_r)) {
      for (int bb = rb0; bb < rb1; ++bb) {
        const int wb = bal_row_positions((lsh[bb] + T::kTile - 1) / T::kTile, rc);
        if (x0 < kHkv * (pre + wb)) {
          scan[kMmaThreads + 1] = bb;
          scan[kMmaThreads + 2] = pre;
          break;
        }
        pre += wb;
      }
    }
    __syncthreads();
    if (x0 >= total) return;  // more CTAs than work
    const int b0 = scan[kMmaThreads + 1];
    cur.start(b0, scan[kMmaThreads + 2], lsh[b0], b0 + 1 < B ? lsh[b0 + 1] : 0, x0, min(x0 + q, total), q, rc,
              cur_sm + warp * kCurSlotInts);
    if constexpr (kQS) __syncthreads();  // every thread has read the scratch the Q^T fragments overwrite
  } else {
    // one piece per CTA: split s of row (b, g)
    const int g = blockIdx.x, b = blockIdx.y, s = blockIdx.z;
    // The chunk's first K and V tile into L2 while the length loads: where
    // it starts does not depend on the length.  A hint only (a row that ends
    // before the chunk costs one tile read); a paged cache needs its block
    // table first.  Cold / warm in a CUDA graph on GB300, us per call: bf16
    // 1 x 4096 8.7 -> 7.9 / 7.6 -> 7.3, bf16 4 x 4096 16.0 -> 15.2 / 15.2 ->
    // 14.6, e4m3 1 x 16384 13.8 -> 13.2 / 12.7 -> 11.9, int8 2 x 8192 12.9 ->
    // 12.5 / 11.9 -> 11.2.  Prefetching every ring stage's tile was slower
    // (bf16 4 x 4096 cold 15.2 -> 16.8, bf16 32 x U[1, 512] 12.6 -> 14.1).
    if (threadIdx.x == kMmaConsumerWarps * 32 && p.block_table == nullptr) {
      const int t0 = s * p.chunk, n = min(T::kTile, C - t0);
      if (n > 0) {
        const uint32_t bytes = (uint32_t)n * T::kRowBytes;
        const uint8_t* src = static_cast<const uint8_t*>(p.kv) + ((size_t)(b * 2 * kHkv + g) * C + t0) * T::kRowBytes;
        const uint8_t* srcV = src + (size_t)kHkv * C * T::kRowBytes;
        if (!kChecked || (in_extent(p.kv, p.kv_bytes, src, bytes) && in_extent(p.kv, p.kv_bytes, srcV, bytes))) {
          bulk_prefetch_l2(src, bytes);
          bulk_prefetch_l2(srcV, bytes);
        }
      }
    }
    const int len_raw = __ldg(p.lens + b);
    const int L = min(max(len_raw, 0), C);
    if (s == 0 && g == 0 && threadIdx.x == 0 && (len_raw < NQ || len_raw > C))
      atomicOr(p.flags, GQA_FLAG_LENGTH_CLAMPED);
    const int t_begin = s * p.chunk;
    const int t_end = min(L, t_begin + p.chunk);
    // (a cluster member keeps going with no tiles: it must reach the merge)
    if (!CL && t_begin >= t_end) {
      if (p.splits_eff == 1 && threadIdx.x < kMmaConsumerWarps * 32) {
        // one-split launch with length 0: the output rows are zero
        const int hh = threadIdx.x / 32, d0 = 4 * (threadIdx.x % 32);
#pragma unroll
        for (int jq = 0; jq < NQ; ++jq) {
          const size_t row = checked_row(p, NQ, (size_t)(b * NQ + jq) * kHq + g * kGroup + hh);
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + (row * kD + d0) * 2) = make_uint2(0u, 0u);
        }
      }
      return;
    }
    cur.start_single(b, g, L, t_begin, max(t_begin, t_end), s, !CL && p.splits_eff == 1);
  }

  // the barriers' initialisation is visible to every thread (the balanced
  // prologue has synchronised the CTA already)
  if constexpr (!BAL) __syncthreads();
  const uint64_t deadline = global_timer_ns() + p.wait_budget_ns;

  if (warp == kMmaConsumerWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (its lanes fetch block-table entries 32 at
    // a time); lane 0 waits on the barriers and issues the copies.  `it`
    // counts this CTA's tiles over all its pieces: it sets the ring stage and
    // barrier phase, so the ring streams straight from one piece to the next.
    const bool paged = p.block_table != nullptr;
    const size_t page_rows = paged ? ((size_t)1 << p.page_log2) : (size_t)C;
    const size_t head_bytes = page_rows * T::kRowBytes;  // one (page, plane, KV head) block
    const uint8_t* base = static_cast<const uint8_t*>(p.kv);
    const uint64_t pol = policy_evict_first();
    int last[kMmaStages];  // last tile issued into each stage (-1: none)
#pragma unroll
    for (int k = 0; k < kMmaStages; ++k) last[k] = -1;
    bool ok = true;
    int it = 0;
    Piece pc;
    while (ok && cur.next(pc, p)) {
      const int b = pc.b, g = pc.g, t_begin = pc.t_begin, t_end = pc.t_end;
      const int n_tiles = (t_end - t_begin + T::kTile - 1) / T::kTile;
      int bt_first = -1, bt_val = 0;  // paged: entry bt_first + lane of this row's block table
      for (int i = 0; i < n_tiles; ++i, ++it) {
        const int st = it % kMmaStages;
        if (it >= kMmaStages) {
          int got = 1;
          if (lane == 0) got = mbar_wait(&empty[st], ((it / kMmaStages) & 1) ^ 1, deadline);
          if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
          }
        }
        if (it == p.skip_tile) continue;  // test hook: the consumers' wait on this tile runs out
        const int t0 = t_begin + i * T::kTile;
        const int rows = min(T::kTile, t_end - t0);
        uint8_t* dK = ring + st * kStageBytes;
        uint8_t* dV = dK + T::kTileBytes;
        uint16_t* dsk = scl + st * (kScaleStageBytes / 2);
        // The page of slot t (all lanes take part: they fetch block-table
        // entries 32 at a time): its id, the row in it, and the end of the
        // segment [t, seg_end) that stays in it.  A contiguous cache is one
        // page per batch row.
        const auto seg_of = [&](int t, size_t& page, int& in_page, int& seg_end) {
          page = (size_t)b;
          in_page = t;
          seg_end = t0 + rows;
          if (paged) {
            const int pg = t >> p.page_log2;
            // (the int8 scale tail looks up a tile's last page before its
            // first, so the window may have to move back as well as forward)
            if (bt_first < 0 || pg < bt_first || pg >= bt_first + 32) {
              bt_first = pg;
              const int e = pg + lane;
              bt_val = e < p.max_pages ? __ldg(p.block_table + (size_t)b * p.max_pages + e) : 0;
            }
            int id = __shfl_sync(0xffffffffu, bt_val, pg - bt_first);
            if (id < 0 || id >= p.num_pages) {  // out-of-contract page id: clamp, flag, never fault
              if (lane == 0) atomicOr(p.flags, GQA_FLAG_PAGE_CLAMPED);
              id = min(max(id, 0), p.num_pages - 1);
            }
            page = (size_t)id;
            in_page = t - (pg << p.page_log2);
            seg_end = min(t0 + rows, (pg + 1) << p.page_log2);
          }
        };
        // int8 row scales ([page or b][2][8][rows] bf16): whole 16-byte groups
        // of 8 rows by bulk copy with their page segment, the ragged tail
        // (< 8 rows, all in the last page) by plain loads before the arrive
        const int n8 = rows & ~7;
        if constexpr (KVF == kKvI8) {
          if (n8 < rows) {
            size_t page;
            int in_page, seg_end;
            seg_of(t0 + n8, page, in_page, seg_end);
            if (lane == 0) {
              const uint16_t* gs = p.kv_scales + (page * 2 * kHkv + g) * page_rows + in_page;
              for (int r = 0; r < rows - n8; ++r) {
                const uint16_t* sk = gs + r;
                const uint16_t* sv = gs + (size_t)kHkv * page_rows + r;
                if constexpr (kChecked) {
                  if (!in_extent(p.kv_scales, p.scales_bytes, sk, 2) || !in_extent(p.kv_scales, p.scales_bytes, sv, 2)) {
                    atomicOr(p.flags, GQA_FLAG_BOUNDS);
                    sk = sv = p.kv_scales;
                  }
                }
                dsk[n8 + r] = *sk;
                dsk[T::kTile + n8 + r] = *sv;
              }
            }
          }
        }
        const uint32_t scale_bytes = KVF == kKvI8 ? 4u * (uint32_t)n8 : 0u;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], 2u * (uint32_t)rows * T::kRowBytes + scale_bytes);
        for (int t = t0; t < t0 + rows;) {
          size_t page;
          int in_page, seg_end;
          seg_of(t, page, in_page, seg_end);
          if (lane == 0) {
            const uint32_t seg_bytes = (uint32_t)(seg_end - t) * T::kRowBytes;
            const uint8_t* src = base + (page * 2 * kHkv + g) * head_bytes + (size_t)in_page * T::kRowBytes;
            const uint8_t* srcV = src + kHkv * head_bytes;
            if constexpr (kChecked) {  // both source ranges in the cache, the destination in the stage
              if (!in_extent(p.kv, p.kv_bytes, src, seg_bytes) || !in_extent(p.kv, p.kv_bytes, srcV, seg_bytes) ||
                  (uint32_t)(t - t0) * T::kRowBytes + seg_bytes > (uint32_t)T::kTileBytes) {
                atomicOr(p.flags, GQA_FLAG_BOUNDS);
                src = base;
                srcV = base + kHkv * head_bytes;
              }
            }
            bulk_load(dK + (t - t0) * T::kRowBytes, src, seg_bytes, &full[st], pol);
            bulk_load(dV + (t - t0) * T::kRowBytes, srcV, seg_bytes, &full[st], pol);
            if constexpr (KVF == kKvI8) {
              const int s_end = min(seg_end, t0 + n8);
              if (s_end > t) {
                const uint16_t* gs = p.kv_scales + (page * 2 * kHkv + g) * page_rows + in_page;
                const uint16_t* gsv = gs + (size_t)kHkv * page_rows;
                const uint32_t sb = (uint32_t)(s_end - t) * 2u;
                if constexpr (kChecked) {
                  if (!in_extent(p.kv_scales, p.scales_bytes, gs, sb) || !in_extent(p.kv_scales, p.scales_bytes, gsv, sb)) {
                    atomicOr(p.flags, GQA_FLAG_BOUNDS);
                    gs = p.kv_scales;
                    gsv = p.kv_scales + (size_t)kHkv * page_rows;
                  }
                }
                bulk_load(dsk + (t - t0), gs, sb, &full[st], pol);
                bulk_load(dsk + T::kTile + (t - t0), gsv, sb, &full[st], pol);
              }
            }
          }
          t = seg_end;
        }
  #pragma unroll
        for (int k = 0; k < kMmaStages; ++k)
          if (k == st) last[k] = it;
      }
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.flags, GQA_FLAG_WAIT_TIMEOUT);
      // Never leave the CTA with copies in flight: wait (bounded) for the last
      // copy issued into every stage to land.
#pragma unroll
      for (int k = 0; k < kMmaStages; ++k)
        if (last[k] >= 0) mbar_wait(&full[k], (last[k] / kMmaStages) & 1, deadline + p.wait_budget_ns);
    }
    if constexpr (CL) cluster_merge_tail<QF, NQ>(p, cl_state);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gq = lane >> 2, cq = lane & 3;
  const float sl2 = p.scale_log2;
  // P^T shuffle sources: tokens 2cq and 2cq+1 of the slab, column pair gq/2
  bool alive = true;  // false once a wait has run out: the remaining tiles are skipped
  int it = 0;         // this CTA's tiles over all its pieces (ring stage and phase)
  Piece pc;
  while (cur.next(pc, p)) {
    const int b = pc.b, g = pc.g, L = pc.L, t_begin = pc.t_begin, t_end = pc.t_end;
    const int n_tiles = (t_end - t_begin + T::kTile - 1) / T::kTile;
    // Column n of n-tile nt is (query token 2nt + n/4, head n%4).  This lane's
    // score/output columns are n = 2cq, 2cq+1: query token 2nt + cq/2, heads
    // 2(cq%2) and 2(cq%2)+1.  A column past the window is zero padding.
    // (Q^T in shared memory: the previous piece's merge has read its area)
    if constexpr (kQS && BAL) named_barrier_sync(1, kMmaConsumerWarps * 32);
    int lim[kNT];  // slots below lim[nt] are attended by this lane's columns
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int jq = 2 * nt + (cq >> 1);
      lim[nt] = jq < NQ ? min(t_end, L - NQ + 1 + jq) : 0;
    }

    // Q^T B-fragments: column gq of each n-tile (zero for padding).  A bf16 q
    // meeting f16 tensor cores (8-bit KV) is first scaled by a power of two
    // 2^e per column, chosen so that the column's largest |q| lands in
    // [2^14, 2^15): every element of magnitude >= 2^-31 of that maximum is
    // then exact in f16, the rest round on the f16 subnormal grid (2^-39 of
    // the maximum at most), and nothing saturates.  The column's score scale
    // takes 2^-e (sl2c below); power-of-two scaling commutes with FP32
    // rounding, so a q already in f16 range scores bit for bit as unscaled.
    constexpr bool kQPow2 = is_8bit(KVF) && QF == kQBF16;
    uint32_t qb[kNT][8][2];
    float sl2c[kNT][2];  // score scale of this lane's columns 2cq, 2cq+1 (scale_log2 * 2^-e)
  #pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      const int jq = 2 * nt + (gq >> 2);
      const bool real = jq < NQ;
      const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                             checked_row(p, NQ, (size_t)((b * NQ + (real ? jq : 0)) * kHq) + g * kGroup + (gq & 3)) *
                                 kD;
  #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
  #pragma unroll
        for (int pr = 0; pr < 2; ++pr)
          qb[nt][ks][pr] = __ldg(reinterpret_cast<const uint32_t*>(qrow + qk_dim<KVF>(cq, ks, pr)));
      sl2c[nt][0] = sl2c[nt][1] = sl2;
      if constexpr (kQPow2) {
        // the column's largest magnitude, as bf16 bits (monotone in the value)
        uint32_t amax = 0;
  #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
  #pragma unroll
          for (int pr = 0; pr < 2; ++pr)
            amax = max(amax, max(qb[nt][ks][pr] & 0x7fffu, (qb[nt][ks][pr] >> 16) & 0x7fffu));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // lanes 4gq..4gq+3 hold column gq
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // e = 14 - floor(log2 amax) from the biased exponent; amax below
        // 2^-126 (bf16 subnormal) takes the largest e, 126; all zero takes 0
        const int ebits = (int)(amax >> 7);
        const int e = ebits > 0 ? min(141 - ebits, 126) : (amax ? 126 : 0);
        const float up = __uint_as_float((uint32_t)(127 + e) << 23);    // 2^e
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
  #pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
            const uint32_t w = qb[nt][ks][pr];
            qb[nt][ks][pr] = pack_f16_satfinite(bf16_lo_to_f32(w) * up, bf16_hi_to_f32(w) * up);
          }
        const float mine = sl2 * down;  // column gq's score scale
        sl2c[nt][0] = __shfl_sync(0xffffffffu, mine, 8 * cq);      // column 2cq
        sl2c[nt][1] = __shfl_sync(0xffffffffu, mine, 8 * cq + 4);  // column 2cq + 1
      }
  #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
  #pragma unroll
        for (int pr = 0; pr < 2; ++pr)
          if (!real) qb[nt][ks][pr] = 0u;
    }
    // int8 K: score offset of each of this lane's columns (2cq, 2cq+1),
    // -1152 * sum_d q_d * scale_log2, added in the scale step (the K operand
    // is code + 1152, see widen4_biased).
    float kb[kNT][2];
  #pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      kb[nt][0] = kb[nt][1] = 0.f;
      if constexpr (KVF == kKvI8) {
        float qs = 0.f;  // this lane's part of column gq's sum
  #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
  #pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&qb[nt][ks][pr]));
            qs += f.x + f.y;
          }
        qs += __shfl_xor_sync(0xffffffffu, qs, 1);  // lanes 4n..4n+3 hold column n
        qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        kb[nt][0] = -kI8Bias * sl2c[nt][0] * __shfl_sync(0xffffffffu, qs, 8 * cq);
        kb[nt][1] = -kI8Bias * sl2c[nt][1] * __shfl_sync(0xffffffffu, qs, 8 * cq + 4);
      }
    }
    if constexpr (kQS) {
      static_assert(kNT == 2, "the shared Q^T layout holds two n-tiles");
      if (warp == 0) {  // every consumer warp holds the same fragments
  #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          *reinterpret_cast<uint4*>(qfr + (ks * 32 + lane) * 4) =
              make_uint4(qb[0][ks][0], qb[0][ks][1], qb[1][ks][0], qb[1][ks][1]);
      }
      named_barrier_sync(1, kMmaConsumerWarps * 32);
    }

    float o[kNT][8][4];
    float m[kNT][2], l[kNT][2];  // per column: running max (log2 domain), this lane's denominator share
    float vw[kNT][2];            // int8: this lane's share of the V weights since take_v_bias
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
      vw[nt][0] = vw[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][mt][e] = 0.f;
    }

    for (int i = 0; i < n_tiles; ++i, ++it) {
      const int st = it % kMmaStages;
      if (alive && !mbar_wait(&full[st], (it / kMmaStages) & 1, deadline)) {
        if (lane == 0) atomicOr(p.flags, GQA_FLAG_WAIT_TIMEOUT);
        alive = false;
      }
      if (!alive) continue;
      const uint8_t* sK = ring + st * kStageBytes;
      const uint8_t* sV = sK + T::kTileBytes;
      const int tile_t0 = t_begin + i * T::kTile;
      const int rows = min(T::kTile, t_end - tile_t0);
      // int8: the bf16 row scale of tile row r (plane 0: K, 1: V), read where
      // it is used (fewer live registers); 0 past the tile's rows
      const uint16_t* tsk = scl + st * (kScaleStageBytes / 2);
      const auto row_scale = [&](int r, int plane) {
        return r < rows ? __uint_as_float((uint32_t)tsk[plane * T::kTile + r] << 16) : 0.f;
      };

  #pragma unroll
      for (int sg = 0; sg < kSlabs; sg += kSG) {
        // this warp's slabs sg .. sg + kSG - 1 of the tile (kSG = 2: both QK
        // products, one max reduction over their 32 tokens, both P.V products)
        if ((warp * kSlabs + sg) * 16 >= rows) break;  // warp-uniform
        float x[kSG][kNT][4];      // scaled, masked scores
        float vsa[kSG], vsb[kSG];  // int8: V row scales of this lane's tokens
  #pragma unroll
        for (int sj = 0; sj < kSG; ++sj) {
        const int R = (warp * kSlabs + sg + sj) * 16;  // first tile row of this slab
        vsa[sj] = vsb[sj] = 0.f;
        if (sj > 0 && R >= rows) {  // warp-uniform: past the tile's rows, no token
  #pragma unroll
          for (int nt = 0; nt < kNT; ++nt) x[sj][nt][0] = x[sj][nt][1] = x[sj][nt][2] = x[sj][nt][3] = -INFINITY;
          continue;
        }

        // ---- scores: S^T[16 tokens x 8] = K . Q^T for each n-tile
        float sc[kNT][4];
  #pragma unroll
        for (int nt = 0; nt < kNT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        {
          const uint8_t* k0 = sK + (R + gq) * T::kRowBytes;
          const uint8_t* k1 = k0 + 8 * T::kRowBytes;
          if constexpr (is_8bit(KVF)) {
  #pragma unroll
            for (int ci = 0; ci < 2; ++ci) {
              const uint4 x = *reinterpret_cast<const uint4*>(k0 + 16 * (cq + 4 * ci));
              const uint4 y = *reinterpret_cast<const uint4*>(k1 + 16 * (cq + 4 * ci));
              const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  #pragma unroll
              for (int s4 = 0; s4 < 4; ++s4) {
                const int ks = 4 * ci + s4;
                uint32_t a0, a1, a2, a3;
                widen4_biased<KVF>(xs[s4], a0, a2);  // row gq: dims (4s,4s+1), (4s+2,4s+3)
                widen4_biased<KVF>(ys[s4], a1, a3);  // row gq+8
                if constexpr (kQS) {
                  const uint4 qv = ld_shared_u4(qfr + (ks * 32 + lane) * 4);
                  mma16816<false>(sc[0], a0, a1, a2, a3, qv.x, qv.y);
                  mma16816<false>(sc[kNT - 1], a0, a1, a2, a3, qv.z, qv.w);
                } else {
  #pragma unroll
                  for (int nt = 0; nt < kNT; ++nt)
                    mma16816<false>(sc[nt], a0, a1, a2, a3, qb[nt][ks][0], qb[nt][ks][1]);
                }
              }
            }
          } else {
  #pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
              const uint4 x = *reinterpret_cast<const uint4*>(k0 + 16 * (cq + 4 * ci));
              const uint4 y = *reinterpret_cast<const uint4*>(k1 + 16 * (cq + 4 * ci));
  #pragma unroll
              for (int nt = 0; nt < kNT; ++nt) {
                mma16816<kBF16>(sc[nt], x.x, y.x, x.y, y.y, qb[nt][2 * ci][0], qb[nt][2 * ci][1]);
                mma16816<kBF16>(sc[nt], x.z, y.z, x.w, y.w, qb[nt][2 * ci + 1][0], qb[nt][2 * ci + 1][1]);
              }
            }
          }
        }
        // int8 row scales of this lane's tokens, read once per slab: inside the
        // n-tile loops below they were read again for each n-tile (3-4-token
        // windows of the int8 cache of 64 x U[16k, 32k] on GB300, us per call
        // back to back: 638.7 -> 612.2, 640.4 -> 613.3; the same output)
        float ks_a = 0.f, ks_b = 0.f;
        if constexpr (KVF == kKvI8) {
          ks_a = row_scale(R + gq, 0);
          ks_b = row_scale(R + gq + 8, 0);
          vsa[sj] = row_scale(R + gq, 1);
          vsb[sj] = row_scale(R + gq + 8, 1);
        }
        // sc[nt]: [0] token R+gq column 2cq, [1] token R+gq column 2cq+1, [2]/[3] token R+gq+8
        const int ta = tile_t0 + R + gq, tb = ta + 8;
  #pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
  #pragma unroll
          for (int e = 0; e < 4; ++e) {
            if constexpr (KVF == kKvI8) x[sj][nt][e] = fmaf(sc[nt][e], sl2c[nt][e & 1], kb[nt][e & 1]);
            else x[sj][nt][e] = sc[nt][e] * sl2c[nt][e & 1];
          }
          if constexpr (KVF == kKvI8) {  // per-row K scale multiplies that token's scores
            x[sj][nt][0] *= ks_a;
            x[sj][nt][1] *= ks_a;
            x[sj][nt][2] *= ks_b;
            x[sj][nt][3] *= ks_b;
          }
          if (ta >= lim[nt]) x[sj][nt][0] = x[sj][nt][1] = -INFINITY;  // select, never multiply
          if (tb >= lim[nt]) x[sj][nt][2] = x[sj][nt][3] = -INFINITY;
        }
        }

        // ---- online softmax per column (max over the slab's 16 tokens)
        float nm[kNT][2];
        bool grow = false;
  #pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          float h0 = fmaxf(x[0][nt][0], x[0][nt][2]), h1 = fmaxf(x[0][nt][1], x[0][nt][3]);
  #pragma unroll
          for (int sj = 1; sj < kSG; ++sj) {
            h0 = fmaxf(h0, fmaxf(x[sj][nt][0], x[sj][nt][2]));
            h1 = fmaxf(h1, fmaxf(x[sj][nt][1], x[sj][nt][3]));
          }
  #pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            h0 = fmaxf(h0, __shfl_xor_sync(0xffffffffu, h0, off));
            h1 = fmaxf(h1, __shfl_xor_sync(0xffffffffu, h1, off));
          }
          nm[nt][0] = fmaxf(m[nt][0], h0);
          nm[nt][1] = fmaxf(m[nt][1], h1);
          grow |= nm[nt][0] > m[nt][0] || nm[nt][1] > m[nt][1];
        }
        if (__any_sync(0xffffffffu, grow)) {
  #pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            // 0 when the old max was -inf; 1 when unchanged (also covers -inf == -inf)
            const float a0 = nm[nt][0] == m[nt][0] ? 1.f : ex2(m[nt][0] - nm[nt][0]);
            const float a1 = nm[nt][1] == m[nt][1] ? 1.f : ex2(m[nt][1] - nm[nt][1]);
            l[nt][0] *= a0;
            l[nt][1] *= a1;
            vw[nt][0] *= a0;
            vw[nt][1] *= a1;
  #pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[nt][mt][0] *= a0;
              o[nt][mt][2] *= a0;
              o[nt][mt][1] *= a1;
              o[nt][mt][3] *= a1;
            }
            m[nt][0] = nm[nt][0];
            m[nt][1] = nm[nt][1];
          }
        }

        // ---- P^T B-fragments per n-tile: lane (gq, cq) needs column gq of tokens
        // 2cq, 2cq+1 (b0) and 2cq+8, 2cq+9 (b1); the packed weights hold
        // (token gq, columns 2cq, 2cq+1) and (token gq+8, ...): one 8x8
        // transpose each.
        uint32_t bh[kSG][kNT][2], bl[kSG][kNT][2];
  #pragma unroll
        for (int sj = 0; sj < kSG; ++sj) {
  #pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const float p0 = x[sj][nt][0] == -INFINITY ? 0.f : ex2(x[sj][nt][0] - m[nt][0]);
          const float p1 = x[sj][nt][1] == -INFINITY ? 0.f : ex2(x[sj][nt][1] - m[nt][1]);
          const float p2 = x[sj][nt][2] == -INFINITY ? 0.f : ex2(x[sj][nt][2] - m[nt][0]);
          const float p3 = x[sj][nt][3] == -INFINITY ? 0.f : ex2(x[sj][nt][3] - m[nt][1]);
          bl[sj][nt][0] = bl[sj][nt][1] = 0u;
          if constexpr (kBF16) {
            const uint32_t ph_a = pack_bf16(p0, p1), ph_b = pack_bf16(p2, p3);
            const uint32_t pl_a = pack_bf16(p0 - bf16_lo_to_f32(ph_a), p1 - bf16_hi_to_f32(ph_a));
            const uint32_t pl_b = pack_bf16(p2 - bf16_lo_to_f32(ph_b), p3 - bf16_hi_to_f32(ph_b));
            l[nt][0] += bf16_lo_to_f32(ph_a) + bf16_lo_to_f32(pl_a) + bf16_lo_to_f32(ph_b) + bf16_lo_to_f32(pl_b);
            l[nt][1] += bf16_hi_to_f32(ph_a) + bf16_hi_to_f32(pl_a) + bf16_hi_to_f32(ph_b) + bf16_hi_to_f32(pl_b);
            bh[sj][nt][0] = transpose8x8_b16(ph_a);
            bh[sj][nt][1] = transpose8x8_b16(ph_b);
            bl[sj][nt][0] = transpose8x8_b16(pl_a);
            bl[sj][nt][1] = transpose8x8_b16(pl_b);
          } else if constexpr (KVF == kKvI8) {
            // the per-row V scale joins the weight of its token; the denominator
            // keeps the unscaled weights
            const uint32_t pa = pack_f16(p0 * vsa[sj], p1 * vsa[sj]);
            const uint32_t pb = pack_f16(p2 * vsb[sj], p3 * vsb[sj]);
            l[nt][0] += p0 + p2;
            l[nt][1] += p1 + p3;
            // the weights exactly as the tensor core multiplies them (V offset)
            const float2 fa = f16x2_to_f32x2(pa), fb = f16x2_to_f32x2(pb);
            vw[nt][0] += fa.x + fb.x;
            vw[nt][1] += fa.y + fb.y;
            bh[sj][nt][0] = transpose8x8_b16(pa);
            bh[sj][nt][1] = transpose8x8_b16(pb);
          } else {
            const uint32_t pa = pack_f16(p0, p1), pb = pack_f16(p2, p3);
            // the denominator sums the same rounded weights the tensor core multiplies
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pa));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&pb));
            l[nt][0] += fa.x + fb.x;
            l[nt][1] += fa.y + fb.y;
            bh[sj][nt][0] = transpose8x8_b16(pa);
            bh[sj][nt][1] = transpose8x8_b16(pb);
          }
        }
        }

        // ---- O^T[128 dims x 8] += V^T . P^T per n-tile: lane (gq, cq) reads dims
        // 16gq..16gq+15 of tokens R+2cq, R+2cq+1, R+2cq+8, R+2cq+9.
  #pragma unroll
        for (int sj = 0; sj < kSG; ++sj) {
        const int R = (warp * kSlabs + sg + sj) * 16;
        if (sj > 0 && R >= rows) break;  // warp-uniform
        const bool partial = R + 16 > rows;
        const int r0 = R + 2 * cq;
        const uint8_t* v0 = sV + r0 * T::kRowBytes;
        const bool ok0 = !partial || r0 < rows, ok1 = !partial || r0 + 1 < rows;
        const bool ok2 = !partial || r0 + 8 < rows, ok3 = !partial || r0 + 9 < rows;
        if constexpr (is_8bit(KVF)) {
          uint4 w0 = *reinterpret_cast<const uint4*>(v0 + 16 * gq);
          uint4 w1 = *reinterpret_cast<const uint4*>(v0 + T::kRowBytes + 16 * gq);
          uint4 w2 = *reinterpret_cast<const uint4*>(v0 + 8 * T::kRowBytes + 16 * gq);
          uint4 w3 = *reinterpret_cast<const uint4*>(v0 + 9 * T::kRowBytes + 16 * gq);
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          if (!ok0) w0 = z;
          if (!ok1) w1 = z;
          if (!ok2) w2 = z;
          if (!ok3) w3 = z;
          const uint32_t a[4] = {w0.x, w0.y, w0.z, w0.w}, bq[4] = {w1.x, w1.y, w1.z, w1.w};
          const uint32_t c[4] = {w2.x, w2.y, w2.z, w2.w}, d[4] = {w3.x, w3.y, w3.z, w3.w};
  #pragma unroll
          for (int j = 0; j < 4; ++j) {  // word j: dims 16gq+4j .. +3 -> m-tiles 2j, 2j+1
            // pair the two tokens of each k-step: bytes [r0.d, r1.d, r0.d', r1.d']
            uint32_t A0, A1, A2, A3;
            widen4_biased<KVF>(prmt(a[j], bq[j], 0x5140u), A0, A1);  // dims 4j, 4j+1 of tokens r0, r0+1
            widen4_biased<KVF>(prmt(c[j], d[j], 0x5140u), A2, A3);   // tokens r0+8, r0+9
  #pragma unroll
            for (int nt = 0; nt < kNT; ++nt) mma16816<false>(o[nt][2 * j], A0, A1, A2, A3, bh[sj][nt][0], bh[sj][nt][1]);
            widen4_biased<KVF>(prmt(a[j], bq[j], 0x7362u), A0, A1);  // dims 4j+2, 4j+3
            widen4_biased<KVF>(prmt(c[j], d[j], 0x7362u), A2, A3);
  #pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
              mma16816<false>(o[nt][2 * j + 1], A0, A1, A2, A3, bh[sj][nt][0], bh[sj][nt][1]);
          }
        } else {
          const uint8_t* v1 = v0 + T::kRowBytes;
          const uint8_t* v2 = v0 + 8 * T::kRowBytes;
          const uint8_t* v3 = v0 + 9 * T::kRowBytes;
  #pragma unroll
          for (int half = 0; half < 2; ++half) {  // dims 16gq + 8half .. +7 -> m-tiles 4half..4half+3
            uint4 w0 = *reinterpret_cast<const uint4*>(v0 + 32 * gq + 16 * half);
            uint4 w1 = *reinterpret_cast<const uint4*>(v1 + 32 * gq + 16 * half);
            uint4 w2 = *reinterpret_cast<const uint4*>(v2 + 32 * gq + 16 * half);
            uint4 w3 = *reinterpret_cast<const uint4*>(v3 + 32 * gq + 16 * half);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            if (!ok0) w0 = z;
            if (!ok1) w1 = z;
            if (!ok2) w2 = z;
            if (!ok3) w3 = z;
            const uint32_t a[4] = {w0.x, w0.y, w0.z, w0.w}, bq[4] = {w1.x, w1.y, w1.z, w1.w};
            const uint32_t c[4] = {w2.x, w2.y, w2.z, w2.w}, d[4] = {w3.x, w3.y, w3.z, w3.w};
  #pragma unroll
            for (int j = 0; j < 4; ++j) {  // word j: dims 16gq + 8half + 2j, +1 -> m-tile 4half + j
              const uint32_t A0 = prmt(a[j], bq[j], 0x5410u), A1 = prmt(a[j], bq[j], 0x7632u);
              const uint32_t A2 = prmt(c[j], d[j], 0x5410u), A3 = prmt(c[j], d[j], 0x7632u);
  #pragma unroll
              for (int nt = 0; nt < kNT; ++nt) {
                mma16816<kBF16>(o[nt][4 * half + j], A0, A1, A2, A3, bh[sj][nt][0], bh[sj][nt][1]);
                if constexpr (kBF16) mma16816<kBF16>(o[nt][4 * half + j], A0, A1, A2, A3, bl[sj][nt][0], bl[sj][nt][1]);
              }
            }
          }
        }
        }
      }
      // int8 V offset: taken off every 16 tiles, so the accumulator never
      // carries more than 16 tiles' worth of it
      if constexpr (KVF == kKvI8) {
        if ((i & 15) == 15) take_v_bias(o, vw);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if constexpr (KVF == kKvI8) take_v_bias(o, vw);
    cur.reload(pc);  // the piece's output coordinates (the balanced cursor keeps them in shared memory)

    // ---- per-warp denominators: sum over the 8 lanes holding each column
  #pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
  #pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
        l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
      }
    // every consumer warp is done with the piece (and, with one piece per CTA,
    // with the ring, which then holds the merge area); with several pieces this
    // also keeps the previous piece's merge reads ahead of these writes
    named_barrier_sync(1, kMmaConsumerWarps * 32);
    // The 4 warps' states merge through shared memory in rounds of kRC
    // columns: all of them at once in the idle ring with one piece per CTA,
    // one query token (4 heads) per round in the balanced schedule's smaller
    // merge area outside the ring.
    // O^T fragment: o[nt][mt][0] = O[dim 16gq+2mt][column 2cq], [1] = [..][2cq+1],
    //               o[nt][mt][2] = O[dim 16gq+2mt+1][2cq],  [3] = [..+1][2cq+1]
    const int ctid = threadIdx.x;
    const int d0 = 4 * (ctid & 31);
  #pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
      if (rd > 0) named_barrier_sync(1, kMmaConsumerWarps * 32);  // the last round's reads are done
  #pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int col = 8 * nt + 2 * cq;  // this lane's first column in the n-tile
        if (col < kCols && col / kRC == rd) {
          const int lc = col - rd * kRC;
          float* ha = mrg_acc + (warp * kRC + lc) * kD + 16 * gq;
          float* hb = ha + kD;
  #pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            *reinterpret_cast<float2*>(ha + 2 * mt) = make_float2(o[nt][mt][0], o[nt][mt][2]);
            *reinterpret_cast<float2*>(hb + 2 * mt) = make_float2(o[nt][mt][1], o[nt][mt][3]);
          }
          if (gq == 0) {
            mrg_m[warp * kRC + lc] = m[nt][0];
            mrg_m[warp * kRC + lc + 1] = m[nt][1];
            mrg_l[warp * kRC + lc] = l[nt][0];
            mrg_l[warp * kRC + lc + 1] = l[nt][1];
          }
        }
      }
      named_barrier_sync(1, kMmaConsumerWarps * 32);

      // ---- merge the 4 warps: thread -> (column, dims d0..d0+3)
  #pragma unroll
      for (int il = 0; il < kRC / kGroup; ++il) {
        const int lc = (ctid >> 5) + kGroup * il;  // column in this round
        const int col = rd * kRC + lc;             // query token col / 4, head ctid / 32
        float M = -INFINITY;
  #pragma unroll
        for (int w = 0; w < kMmaConsumerWarps; ++w) M = fmaxf(M, mrg_m[w * kRC + lc]);
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  #pragma unroll
        for (int w = 0; w < kMmaConsumerWarps; ++w) {
          const float mw = mrg_m[w * kRC + lc];
          const float a = mw == -INFINITY ? 0.f : ex2(mw - M);
          Ls = fmaf(mrg_l[w * kRC + lc], a, Ls);
          const float4 v = *reinterpret_cast<const float4*>(&mrg_acc[(w * kRC + lc) * kD + d0]);
          acc.x = fmaf(v.x, a, acc.x);
          acc.y = fmaf(v.y, a, acc.y);
          acc.z = fmaf(v.z, a, acc.z);
          acc.w = fmaf(v.w, a, acc.w);
        }
        const int row = (pc.b * NQ + col / kGroup) * kHq + pc.g * kGroup + (ctid >> 5);  // (b, query token, head)
        if constexpr (CL) {
          *reinterpret_cast<float4*>(cl_state + col * kD + d0) = acc;
          if (d0 == 0) {
            cl_state[kCols * kD + col] = M;
            cl_state[kCols * kD + kCols + col] = Ls;
          }
        } else if (pc.direct) {
          const float inv = Ls > 0.f ? p.v_scale / Ls : 0.f;  // a query with no slot gets zeros
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + (checked_row(p, NQ, row) * kD + d0) * 2) =
              make_uint2(pack_out<QF>(acc.x * inv, acc.y * inv), pack_out<QF>(acc.z * inv, acc.w * inv));
        } else {
          int slot = pc.slot;
          if constexpr (kChecked) {
            if (slot < 0 || slot >= p.num_splits) {
              atomicOr(p.flags, GQA_FLAG_BOUNDS);
              slot = 0;
            }
          }
          const size_t idx = checked_row(p, NQ, row) * p.num_splits + slot;
          *reinterpret_cast<float4*>(p.part_o + idx * kD + d0) = acc;
          if (d0 == 0) {
            p.part_m[idx] = M;
            p.part_l[idx] = Ls;
          }
        }
      }
    }
  }
  if constexpr (CL) cluster_merge_tail<QF, NQ>(p, cl_state);
}

}  // namespace gqa
