// Stage 2 of GQA decode: log-sum-exp merge of the split-KV partials.
//
// For each (b, query head h) the splits that hold tokens (n = ceil(len/chunk)
// of them; later splits are skipped, never read) carry an unnormalised
// accumulator O_s, a running max m_s (log2 domain) and a denominator l_s.
// With M = max_s m_s and w_s = 2^(m_s - M):
//   out = v_scale * (sum_s w_s O_s) / (sum_s w_s l_s)
// rounded once to fp16/bf16 (nearest even).  This is the merge of the
// "FlashInfer sm110_gqa_decode" article's "num_splits" section, written as a
// separate kernel so stage 1 needs no inter-CTA ticket; it is launched as a
// programmatic dependent of stage 1, so its launch overlaps stage 1's tail.  One warp per
// (b, h), each lane owning 4 dims; the splits are merged in a fixed order, so
// the result is bitwise deterministic.  With stage 1's balanced schedule the
// "splits" of a row are its pieces (their number follows from the lengths);
// a row of one piece was written by stage 1, a row without tokens is zeroed
// here.
#pragma once

#include "common.cuh"

namespace gqa {

constexpr int kCombineThreads = kGroup * 32;  // one warp per query head of a KV head

struct CombineParams {
  const int32_t* lens;
  void* out;
  const float* part_o;
  const float* part_m;
  const float* part_l;
  int capacity, num_splits, chunk;
  int q_len;  // rows are (b * q_len + j, head); query j attends len - q_len + 1 + j slots
  float v_scale;
  // balanced schedule of stage 1 (bal_ctas > 0, q_len = 1): pieces per row
  // follow from the lengths, the CTA count, q_min and the tile size
  int bal_ctas, bal_q_min, tile, batch;
};

// Merge of the first n split partials of one (b, query head) row by one warp
// (lane l owns dims 4l..4l+3) into out row `row`; n = 0 writes zeros.
// Splits are handled 32 at a time: lane k loads the max / denominator of
// split s0 + k, the weights 2^(m_s - M) are formed once per split and
// broadcast with shuffles, and the partial-output loads are independent.
template <int QF>
__device__ __forceinline__ void merge_splits(const CombineParams& p, size_t row, int n) {
  const int lane = threadIdx.x & 31;
  const size_t base = row * p.num_splits;
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, p.part_m[base + s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float Ls = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + base * (kD / 4) + lane;
  for (int s0 = 0; s0 < n; s0 += 32) {
    const int cnt = min(32, n - s0);
    float w = 0.f, lw = 0.f;
    if (lane < cnt) {
      // a piece without slots for this query (a window's causal limit) adds nothing
      const float ms = p.part_m[base + s0 + lane];
      w = ms == -INFINITY ? 0.f : ex2(ms - M);
      lw = w * p.part_l[base + s0 + lane];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
    Ls += lw;
#pragma unroll 8
    for (int k = 0; k < cnt; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      const float4 v = po[(size_t)(s0 + k) * (kD / 4)];
      o.x = fmaf(wk, v.x, o.x);
      o.y = fmaf(wk, v.y, o.y);
      o.z = fmaf(wk, v.z, o.z);
      o.w = fmaf(wk, v.w, o.w);
    }
  }
  const float inv = Ls > 0.f ? p.v_scale / Ls : 0.f;  // a query with no slot gets zeros
  uint2 packed;
  if constexpr (QF == kQF16) {
    const __half2 a = __floats2half2_rn(o.x * inv, o.y * inv);
    const __half2 c = __floats2half2_rn(o.z * inv, o.w * inv);
    packed = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&c));
  } else {
    const __nv_bfloat162 a = __floats2bfloat162_rn(o.x * inv, o.y * inv);
    const __nv_bfloat162 c = __floats2bfloat162_rn(o.z * inv, o.w * inv);
    packed = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&c));
  }
  *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + (row * kD + 4 * lane) * 2) = packed;
}

template <int QF>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ CombineParams p) {
  const int g = blockIdx.x, bq = blockIdx.y;  // bq = b * q_len + query token
  const int b = bq / p.q_len, jq = bq % p.q_len;
  const size_t row = (size_t)bq * kHq + g * kGroup + (threadIdx.x >> 5);
  int n;      // splits or pieces to merge
  bool zero = false;  // a row without tokens
  if (p.bal_ctas > 0) {
    // The stream positions stage 1 used (integers, so both kernels agree
    // exactly), read while stage 1 still runs: tiles and rows with tokens
    // before row b and in all, and the shortest row.
    constexpr int kW = kCombineThreads / 32;
    __shared__ int red[5][kW];
    int v[5] = {0, 0, 0, 0, INT_MAX};  // tiles before b, rows before b, all tiles, all rows, min
    for (int bb = threadIdx.x; bb < p.batch; bb += kCombineThreads) {
      const int nb = (min(max(__ldg(p.lens + bb), 0), p.capacity) + p.tile - 1) / p.tile;
      if (bb < b) {
        v[0] += nb;
        v[1] += nb > 0;
      }
      v[2] += nb;
      v[3] += nb > 0;
      if (nb > 0) v[4] = min(v[4], nb);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], off);
      v[4] = min(v[4], __shfl_xor_sync(0xffffffffu, v[4], off));
    }
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
      for (int k = 0; k < 5; ++k) red[k][threadIdx.x >> 5] = v[k];
    }
    __syncthreads();
    v[0] = v[1] = v[2] = v[3] = 0;
    v[4] = INT_MAX;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] += red[k][w];
      v[4] = min(v[4], red[4][w]);
    }
    const int nb = (min(max(__ldg(p.lens + b), 0), p.capacity) + p.tile - 1) / p.tile;
    const int rc = bal_row_cost(v[2], v[4], p.bal_ctas, p.bal_q_min);
    const int total = kHkv * (v[2] + rc * v[3]);
    const int q = max((total + p.bal_ctas - 1) / p.bal_ctas, p.bal_q_min);
    const int tf = kHkv * (v[0] + rc * v[1]) + g * bal_row_positions(nb, rc) + rc;  // the row's first tile
    n = nb > 0 ? (tf + nb - 1) / q - tf / q + 1 : 0;
    zero = nb == 0;  // no tokens: a zero row (stage 1 holds no piece of it)
  } else {
    const int L = min(max(__ldg(p.lens + b), 0), p.capacity) - p.q_len + 1 + jq;
    n = L > 0 ? (L + p.chunk - 1) / p.chunk : 0;
  }
  // Launched as a programmatic dependent of stage 1: wait for its partials.
  // Every CTA waits, also those with nothing to merge, so that this grid
  // completes after stage 1 and work later in the stream sees all of `out`.
  pdl_wait_prior_grid();
  // Stage 1 is complete: the next grid in the stream may be scheduled now (it
  // waits for this one before it reads or writes anything).  Triggering
  // earlier let the next split kernel take SM slots during this split's tail.
  pdl_launch_dependents();
  if (p.bal_ctas > 0 && n == 1 && !zero) return;  // one piece: stage 1 wrote the row itself
  merge_splits<QF>(p, row, n);
}

}  // namespace gqa
