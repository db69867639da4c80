// The step before decode: normalise and rotate the new token's query and key
// heads and write its key and value into the cache.
//
// "Qwen3-VL official BF16 on Jetson Thor (SM110)" docs, "Runtime
// architecture": fused kernels that normalise Q and K, rotate them and
// write the cache (q staged for attention, k and v written at the cache
// position); decode graphs are keyed
// by (cache_pos, rope_pos), so the rotary position and the cache slot are
// separate inputs.  For each head vector x of 128 (32 query heads, 8 KV heads):
//   y_d = x_d / sqrt(mean(x^2) + eps) * w_d      (w = q_norm_w or k_norm_w)
//   z_i = y_i cos a_i - y_{i+64} sin a_i,  z_{i+64} = y_{i+64} cos a_i + y_i sin a_i,
//   a_i = pos * theta^(-i/64)                    (rotate-half RoPE)
// q -> q_out (q's dtype, RNE); k -> K plane at `slot`; v is written unchanged
// to the V plane.  The cache format decides the write: fp16/bf16 (RNE),
// e4m3 (value / scale, RNE, saturating), int8 (one bf16 scale amax/127 per
// row, codes round-to-nearest-even, clipped to +-127).
//
// One CTA per batch row, 8 warps; each warp takes six whole head vectors (all
// their loads issued together) and lane l holds dims l, l+32, l+64, l+96, so
// every RoPE pair (i, i+64) stays in one lane.  The 64 angles are formed
// and reduced in FP64 (pos * theta^(-i/64) reaches 1e5 radians at long
// contexts, beyond FP32's reach) once per CTA: the inverse frequencies
// theta^(-i/64) come from the host (FP64, once per call), and the sine and
// cosine are evaluated by sincos_series below in double-float arithmetic
// (FP64 is slow on sm_103a: forming the frequencies with pow and the
// library's sincos of angles up to 1e6 rad took about two thirds of the
// kernel's time).
//
// Precision: the result before its one rounding is within about 2^-21 of the
// exact value relative to itself, so the stored fp16/bf16 value is the
// correctly rounded one or its neighbour.  The rotation is linear, so it runs
// on a = x * w (exact in FP32: two 16-bit significands) and the norm factor
// r = 1/sqrt(mean(x^2) + eps) multiplies last.  The rotation would lose that
// bound wherever a_i cos and a_{i+64} sin nearly cancel; it keeps it with cos
// and sin held as FP32 hi + lo pairs and the rounding error of one product
// recovered exactly by an FMA (rotate_pair).
#pragma once

#include "common.cuh"

namespace gqa {

constexpr int kAppendThreads = 256;

struct AppendParams {
  const void* q_proj;      // [B,32,128] q/out dtype
  const void* k_proj;      // [B,8,128]
  const void* v_proj;      // [B,8,128]
  const void* q_norm_w;    // [128]
  const void* k_norm_w;    // [128]
  const int32_t* positions;  // [B] rotary positions
  const int32_t* slots;      // [B] cache slots to write
  void* q_out;             // [B,32,128]
  void* kv;                // [B,2,8,C,128] in the cache format (paged: [num_pages,2,8,page,128])
  uint16_t* kv_scales;     // int8 cache: [B,2,8,C] bf16 (paged: [num_pages,2,8,page])
  uint32_t* flags;         // optional status word
  int batch, capacity;     // capacity: C, or max_pages * page size for a paged cache
  // paged cache (block_table != nullptr): slot s of row b is row s % page of
  // page block_table[b * max_pages + s / page]
  const int32_t* block_table;
  int max_pages, num_pages, page_log2;
  float eps, k_inv_scale, v_inv_scale;  // e4m3: 1/k_scale, 1/v_scale
  double inv_freq[kD / 2];  // theta^(-i/64), i = 0..63, formed on the host in FP64
  size_t kv_rows;  // rows of 128 in the cache (units x 2 x 8 x rows per unit), for checked builds
};

template <int QF>
__device__ __forceinline__ float load_elem(const void* base, size_t i) {
  const uint16_t h = static_cast<const uint16_t*>(base)[i];
  if constexpr (QF == kQF16) return __half2float(__ushort_as_half(h));
  else return __uint_as_float((uint32_t)h << 16);
}

template <int QF>
__device__ __forceinline__ uint16_t round_elem(float x) {
  if constexpr (QF == kQF16) return __half_as_ushort(__float2half_rn(x));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// pi / 2 as the double nearest to it plus the double nearest to the rest
// (together within about 2^-107 of pi / 2, relative), and 2 / pi.
constexpr double kHalfPiHi = 0x1.921fb54442d18p+0;
constexpr double kHalfPiLo = 0x1.1a62633145c07p-54;
constexpr double kTwoOverPi = 0x1.45f306dc9c883p-1;

// Double-float arithmetic: a value as an unevaluated sum hi + lo of two
// floats with |lo| <= ulp(hi) / 2 (Dekker; Knuth's two-sum), about 48 bits.
// The sums and products below are the error-free transformations, so they
// use the _rn intrinsics, which the compiler never fuses into FMAs.
struct Float2 {
  float hi, lo;
};
__device__ __forceinline__ Float2 fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ Float2 df_mul(Float2 a, Float2 b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = fmaf(a.hi, b.hi, -p);  // the product's rounding error, exactly
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return fast_two_sum(p, e);
}
__device__ __forceinline__ Float2 df_add(Float2 a, Float2 c) {
  const float s = __fadd_rn(a.hi, c.hi);
  const float bb = __fsub_rn(s, a.hi);
  float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(c.hi, bb));  // two-sum error
  err = __fadd_rn(err, __fadd_rn(a.lo, c.lo));
  return fast_two_sum(s, err);
}
__device__ __forceinline__ constexpr Float2 df_const(double d) { return {(float)d, (float)(d - (double)(float)d)}; }

// sin a and cos a for an angle below 2^31 radians as double-float pairs,
// from the mathematics rather than the library routine.  FP64 issues at a
// small fraction of the FP32 rate on sm_103a, and the same series in FP64
// cost about 1 us of this kernel, so only the reduction stays in FP64:
// a = q pi/2 + x with q the integer nearest 2a/pi, q pi/2 taken off in FP64
// by two FMAs, after Cody and Waite's reduction with pi/2 split in two
// constants (the first FMA with the product exact and one rounding of a
// result below 1, the second taking off q times the rest of pi/2), so
// |x| <= pi/4 within about 2^-52; then the Taylor series of sin x and cos x
// about 0 to the x^17 and x^16 terms by Horner's rule in x^2, in
// double-float arithmetic, with the coefficients (-1)^k/(2k+1)! and
// (-1)^k/(2k)! rounded to doubles and split into pairs (the first terms left
// out are below 2^-60 for |x| <= pi/4); q mod 4 picks the quadrant: the swap
// of sin and cos and their signs.  Within about 2^-47 of the exact values at
// the given a (checked against libm on the CPU by an emulation of the same
// float operations over |x| <= pi/4).
__device__ __forceinline__ void sincos_series(double a, Float2& s, Float2& c) {
  constexpr Float2 kSin[9] = {df_const(0x1p+0), df_const(-0x1.5555555555555p-3), df_const(0x1.1111111111111p-7),
                              df_const(-0x1.a01a01a01a01ap-13), df_const(0x1.71de3a556c734p-19),
                              df_const(-0x1.ae64567f544e4p-26), df_const(0x1.6124613a86d09p-33),
                              df_const(-0x1.ae7f3e733b81fp-41), df_const(0x1.952c77030ad4ap-49)};
  constexpr Float2 kCos[9] = {df_const(0x1p+0), df_const(-0x1p-1), df_const(0x1.5555555555555p-5),
                              df_const(-0x1.6c16c16c16c17p-10), df_const(0x1.a01a01a01a01ap-16),
                              df_const(-0x1.27e4fb7789f5cp-22), df_const(0x1.1eed8eff8d898p-29),
                              df_const(-0x1.93974a8c07c9dp-37), df_const(0x1.ae7f3e733b81fp-45)};
  const double q = rint(a * kTwoOverPi);
  double xd = fma(-q, kHalfPiHi, a);
  xd = fma(-q, kHalfPiLo, xd);
  const float xh = (float)xd;
  const Float2 x = {xh, (float)(xd - (double)xh)};
  const float p = __fmul_rn(xh, xh);
  float e = fmaf(xh, xh, -p);
  e = fmaf(__fadd_rn(xh, xh), x.lo, e);  // + 2 xh xl (xl^2 is below 2^-48 x^2)
  const Float2 x2 = fast_two_sum(p, e);
  Float2 ps = kSin[8], pc = kCos[8];
#pragma unroll
  for (int k = 7; k >= 0; --k) {
    ps = df_add(df_mul(ps, x2), kSin[k]);
    pc = df_add(df_mul(pc, x2), kCos[k]);
  }
  const Float2 sx = df_mul(ps, x), cx = pc;
  const Float2 nsx = {-sx.hi, -sx.lo}, ncx = {-cx.hi, -cx.lo};
  switch ((int)((long long)q & 3)) {
    case 0: s = sx; c = cx; break;
    case 1: s = cx; c = nsx; break;
    case 2: s = nsx; c = ncx; break;
    default: s = ncx; c = sx; break;
  }
}

__device__ __forceinline__ uint8_t to_e4m3(float x) {
  uint16_t two;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.f), "f"(x));
  return (uint8_t)(two & 0xffu);
}

// a * c + b * s with c = ch + cl and s = sh + sl (FP32 hi/lo pairs of FP64
// values): b * sh = pb + eb exactly (FMA), h = a * ch + pb rounded once, and
// the small terms a * cl + b * sl + eb added last.  Error about 2^-23 of the
// result, even when the two products nearly cancel.
__device__ __forceinline__ float rotate_pair(float a, float ch, float cl, float b, float sh, float sl) {
  const float pb = b * sh;
  const float eb = fmaf(b, sh, -pb);
  const float h = fmaf(a, ch, pb);
  return h + fmaf(a, cl, fmaf(b, sl, eb));
}

template <int KVF, int QF>
__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const __grid_constant__ AppendParams p) {
  __shared__ float cs[kD / 2], cs_lo[kD / 2], sn[kD / 2], sn_lo[kD / 2];
  // the decode that follows may be scheduled now (it waits for this grid);
  // this grid waits for the previous one before its first read
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  const int b = blockIdx.x;
  const int pos = __ldg(p.positions + b);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dims[4] = {lane, lane + 32, lane + 64, lane + 96};
  // Every load of this warp's head vectors (vectors 0..31: query heads;
  // 32..39: key heads; 40..47: value heads; warp w takes w, w + 8, ...) and
  // of both norm weights is issued here, before the angles: they overlap one
  // another and the FP64 work, instead of one round of latency per vector.
  constexpr int kVecs = kHq + 2 * kHkv, kWarps = kAppendThreads / 32, kPerWarp = kVecs / kWarps;
  static_assert(kVecs % kWarps == 0, "whole vectors per warp");
  float zz[kPerWarp][4], wq[4], wk[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    wq[k] = load_elem<QF>(p.q_norm_w, dims[k]);
    wk[k] = load_elem<QF>(p.k_norm_w, dims[k]);
  }
#pragma unroll
  for (int j = 0; j < kPerWarp; ++j) {
    const int v = warp + kWarps * j;
    const bool is_q = v < kHq, is_k = v >= kHq && v < kHq + kHkv;
    const int g = is_q ? 0 : (v - kHq) % kHkv;
    const void* src = is_q ? p.q_proj : (is_k ? p.k_proj : p.v_proj);
    const size_t row = is_q ? ((size_t)b * kHq + v) * kD : ((size_t)b * kHkv + g) * kD;
#pragma unroll
    for (int k = 0; k < 4; ++k) zz[j][k] = load_elem<QF>(src, row + dims[k]);
  }
  if (threadIdx.x < kD / 2) {
    // a = pos * theta^(-i/64)
    const double a = (double)pos * p.inv_freq[threadIdx.x];
    Float2 sv, cv;
    sincos_series(a, sv, cv);
    cs[threadIdx.x] = cv.hi;
    cs_lo[threadIdx.x] = cv.lo;
    sn[threadIdx.x] = sv.hi;
    sn_lo[threadIdx.x] = sv.lo;
  }
  __syncthreads();
  const int C = p.capacity;
  const int slot = __ldg(p.slots + b);
  bool slot_ok = slot >= 0 && slot < C;
  if (!slot_ok && threadIdx.x == 0 && p.flags) atomicOr(p.flags, GQA_FLAG_SLOT_CLAMPED);
  // where the slot's row lives: (unit, row) in [units][2][8][unit_rows][128],
  // unit = the batch row of a contiguous cache or a page of a paged one
  size_t unit = (size_t)b, row_in = (size_t)max(slot, 0), unit_rows = (size_t)C;
  if (p.block_table != nullptr && slot_ok) {
    const int id = __ldg(p.block_table + (size_t)b * p.max_pages + (slot >> p.page_log2));
    if (id < 0 || id >= p.num_pages) {  // never write through an out-of-range entry
      slot_ok = false;
      if (threadIdx.x == 0 && p.flags) atomicOr(p.flags, GQA_FLAG_PAGE_CLAMPED);
    }
    unit = (size_t)max(id, 0);
    unit_rows = (size_t)1 << p.page_log2;
    row_in = (size_t)(slot & ((1 << p.page_log2) - 1));
  }
#pragma unroll
  for (int j = 0; j < kPerWarp; ++j) {
    const int v = warp + kWarps * j;
    const bool is_q = v < kHq, is_k = v >= kHq && v < kHq + kHkv;
    const int g = is_q ? 0 : (v - kHq) % kHkv;
    const size_t row = is_q ? ((size_t)b * kHq + v) * kD : ((size_t)b * kHkv + g) * kD;
    float z[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) z[k] = zz[j][k];
    if (!is_q && !is_k && !slot_ok) continue;
    if (is_q || is_k) {
      float ss = z[0] * z[0] + z[1] * z[1] + z[2] * z[2] + z[3] * z[3];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float r = 1.f / sqrtf(ss / kD + p.eps);
      float a[4];  // x * w, exact
#pragma unroll
      for (int k = 0; k < 4; ++k) a[k] = z[k] * (is_q ? wq[k] : wk[k]);
      // pairs (lane, lane+64) with angle lane, (lane+32, lane+96) with angle lane+32
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int i = lane + 32 * k;
        const float ch = cs[i], cl = cs_lo[i], sh = sn[i], sl = sn_lo[i];
        z[k] = r * rotate_pair(a[k], ch, cl, a[k + 2], -sh, -sl);
        z[k + 2] = r * rotate_pair(a[k + 2], ch, cl, a[k], sh, sl);
      }
    }
    if (is_q) {
      uint16_t* out = static_cast<uint16_t*>(p.q_out) + row;
#pragma unroll
      for (int k = 0; k < 4; ++k) out[dims[k]] = round_elem<QF>(z[k]);
      continue;
    }
    if (!slot_ok) continue;  // never write outside the cache
    const int plane = is_k ? 0 : 1;
    const size_t srow = ((unit * 2 + plane) * kHkv + g) * unit_rows + row_in;  // the scale's index
    if constexpr (kChecked) {  // the row inside the cache (and its scale inside the scale array)
      if (srow >= p.kv_rows) {
        if (lane == 0 && p.flags) atomicOr(p.flags, GQA_FLAG_BOUNDS);
        continue;
      }
    }
    const size_t crow = srow * kD;
    if constexpr (KVF == kKvE4M3) {
      const float inv = is_k ? p.k_inv_scale : p.v_inv_scale;
      uint8_t* dst = static_cast<uint8_t*>(p.kv) + crow;
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[dims[k]] = to_e4m3(z[k] * inv);
    } else if constexpr (KVF == kKvI8) {
      float amax = fmaxf(fmaxf(fabsf(z[0]), fabsf(z[1])), fmaxf(fabsf(z[2]), fabsf(z[3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      uint16_t sb = __bfloat16_as_ushort(__float2bfloat16_rn(amax / 127.f));
      if (sb == 0) sb = 0x3f80;  // an all-zero row keeps scale 1
      const float scale = __uint_as_float((uint32_t)sb << 16);
      int8_t* dst = reinterpret_cast<int8_t*>(p.kv) + crow;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int code = max(-127, min(127, __float2int_rn(z[k] / scale)));
        dst[dims[k]] = (int8_t)code;
      }
      if (lane == 0) p.kv_scales[srow] = sb;
    } else {
      uint16_t* dst = static_cast<uint16_t*>(p.kv) + crow;
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[dims[k]] = round_elem<QF>(z[k]);
    }
  }
}

}  // namespace gqa
