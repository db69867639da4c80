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
// programmatic dependent of stage 1, so its launch overlaps stage 1's tail.
// W warps per (b, h) (W from the expected pieces per row), each lane owning 4
// dims; the splits are merged in a fixed order, so the result is bitwise
// deterministic.  With stage 1's balanced schedule the
// "splits" of a row are its pieces (their number follows from the lengths);
// a row of one piece was written by stage 1, a row without tokens is zeroed
// here.
#pragma once

#include "common.cuh"

namespace gqa {

// W warps per query head of a KV head (W = 1, 2 or 4; blockDim = 128 W),
// each merging every W-th piece of the head's row, then the W shares merged
// through shared memory: more loads in flight when rows have many pieces.
constexpr int kCombineMaxWarpsPerHead = 4;

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
  int warps_per_head;  // W (1, 2 or 4): blockDim.x = 4 * 32 * W
  uint32_t* flags;     // workspace status word (range checks of checked builds)
};

// One warp's share of the merge of one (b, query head) row: pieces j, j + W,
// j + 2W, ... of the first n (lane l owns dims 4l..4l+3).  Returns the share's
// max M (-inf without pieces), its denominator Ls and unnormalised output o,
// both relative to M.  The loads are issued in few rounds, not one per group
// of pieces (the merge runs after stage 1 and before the next launch, so its
// latency is the step's): every piece's max and denominator (lane k holds
// the share's pieces k, k + 32, ...), then, per 32 pieces, all partial-output
// vectors before any is accumulated; a share of up to 8 (or 16) pieces
// issues both in one round.  Weights 2^(m_s - M) are formed once
// per piece and broadcast with shuffles; pieces are accumulated in order
// (deterministic).
constexpr int kCombineChunks = 8;  // 32-piece chunks: 256 split slots, the most a workspace holds

// o += sum_k w_k v_k over the pieces k = 0..last of a 32-piece chunk (pc:
// lane l's float4 of piece 0, pieces `stride` float4 apart; w: this lane's
// piece weight, broadcast by shuffles).  kN >= last + 1 loads are issued
// before any is used.
template <int kN>
__device__ __forceinline__ void accumulate_pieces(float4& o, const float4* pc, size_t stride, int k0, int last,
                                                  float w) {
  float4 v[kN];
#pragma unroll
  for (int k = 0; k < kN; ++k) v[k] = pc[(size_t)min(k0 + k, last) * stride];
#pragma unroll
  for (int k = 0; k < kN; ++k) {
    const float wk = __shfl_sync(0xffffffffu, w, (k0 + k) & 31);  // past `last` the weight is 0
    o.x = fmaf(wk, v[k].x, o.x);
    o.y = fmaf(wk, v[k].y, o.y);
    o.z = fmaf(wk, v[k].z, o.z);
    o.w = fmaf(wk, v[k].w, o.w);
  }
}

// A share of at most kN pieces in a single round of loads: the partial
// vectors go out with the maxima and denominators, before the weights exist.
// The same arithmetic in the same order as the general path below, so the
// result is the same bit for bit.
template <int kN>
__device__ __forceinline__ void merge_pieces_one_round(const CombineParams& p, size_t base, int cnt, int j, int W,
                                                       float& M, float& Ls, float4& o) {
  const int lane = threadIdx.x & 31;
  const size_t stride = (size_t)W * (kD / 4);
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + (base + j) * (kD / 4) + lane;
  float4 v[kN];
#pragma unroll
  for (int k = 0; k < kN; ++k) v[k] = po[(size_t)min(k, cnt - 1) * stride];
  float m = -INFINITY, l = 0.f;
  if (lane < cnt) {
    m = p.part_m[base + j + (size_t)W * lane];
    l = p.part_l[base + j + (size_t)W * lane];
  }
  M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w = m == -INFINITY ? 0.f : ex2(m - M);
  Ls = fmaf(w, l, 0.f);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
  o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kN; ++k) {
    const float wk = __shfl_sync(0xffffffffu, w, k);  // past the share's last piece the weight is 0
    o.x = fmaf(wk, v[k].x, o.x);
    o.y = fmaf(wk, v[k].y, o.y);
    o.z = fmaf(wk, v[k].z, o.z);
    o.w = fmaf(wk, v[k].w, o.w);
  }
}

// kMaxN: the most vectors one round may hold in registers (the kernel's
// thread count sets the budget).
template <int kMaxN>
__device__ __forceinline__ void merge_pieces(const CombineParams& p, size_t row, int n, int j, int W, float& M,
                                             float& Ls, float4& o) {
  const int lane = threadIdx.x & 31;
  const size_t base = row * p.num_splits;
  const int cnt = n > j ? (n - j + W - 1) / W : 0;  // this warp's pieces
  // few pieces (warp-uniform): one round of loads instead of two
  if (cnt >= 1 && cnt <= 8) {
    merge_pieces_one_round<8>(p, base, cnt, j, W, M, Ls, o);
    return;
  }
  if (kMaxN >= 16 && cnt > 8 && cnt <= 16) {
    merge_pieces_one_round<(kMaxN >= 16 ? 16 : 8)>(p, base, cnt, j, W, M, Ls, o);
    return;
  }
  float wc[kCombineChunks];  // share piece 32c + lane: its max, then its weight
  float lc[kCombineChunks];  // its denominator
  M = -INFINITY;
#pragma unroll
  for (int c = 0; c < kCombineChunks; ++c) {
    const int k = 32 * c + lane;
    wc[c] = -INFINITY;
    lc[c] = 0.f;
    if (32 * c < cnt && k < cnt) {  // (chunks past cnt are skipped by the whole warp)
      wc[c] = p.part_m[base + j + (size_t)W * k];
      lc[c] = p.part_l[base + j + (size_t)W * k];
    }
    M = fmaxf(M, wc[c]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  Ls = 0.f;
#pragma unroll
  for (int c = 0; c < kCombineChunks; ++c) {
    // a piece without slots for this query (max -inf: a window's causal
    // limit, or past the share) adds nothing
    wc[c] = wc[c] == -INFINITY ? 0.f : ex2(wc[c] - M);
    Ls = fmaf(wc[c], lc[c], Ls);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);

  o = make_float4(0.f, 0.f, 0.f, 0.f);
  const size_t stride = (size_t)W * (kD / 4);  // float4s from one piece of the share to the next
  const float4* po = reinterpret_cast<const float4*>(p.part_o) + (base + j) * (kD / 4) + lane;
#pragma unroll
  for (int c = 0; c < kCombineChunks; ++c) {
    if (32 * c >= cnt) break;  // warp-uniform
    const int last = min(32, cnt - 32 * c) - 1;
    const float4* pc = po + (size_t)(32 * c) * stride;
    // unconditional loads, issued together: 8, 16 or 32 vectors (at most
    // kMaxN per round), whichever first covers the chunk's pieces (past the
    // last one the index repeats it, and its weight there is 0)
    if (last < 8) {
      accumulate_pieces<8>(o, pc, stride, 0, last, wc[c]);
    } else if (kMaxN >= 16 && last < 16) {
      accumulate_pieces<(kMaxN >= 16 ? 16 : 8)>(o, pc, stride, 0, last, wc[c]);
    } else {
      for (int k0 = 0; k0 <= last; k0 += kMaxN) accumulate_pieces<kMaxN>(o, pc, stride, k0, last, wc[c]);
    }
  }
}

// out row `row`, this lane's 4 dims: v_scale * o / Ls, rounded once (zeros
// for a query with no slot).
template <int QF>
__device__ __forceinline__ void write_merged(const CombineParams& p, size_t row, float Ls, const float4& o) {
  const int lane = threadIdx.x & 31;
  const float inv = Ls > 0.f ? p.v_scale / Ls : 0.f;
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

// W warps per query head (blockDim.x = 128 W); the register budget of 128 W
// threads per CTA bounds the vectors a warp keeps in flight.
template <int QF, int W>
__global__ void __launch_bounds__(kGroup * 32 * W) combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr int kMaxN = W <= 2 ? 32 : 16;  // 158 / 122 registers, no spills
  const int g = blockIdx.x, bq = blockIdx.y;  // bq = b * q_len + query token
  const int b = bq / p.q_len, jq = bq % p.q_len;
  const int warp = threadIdx.x >> 5, h = warp % kGroup, share = warp / kGroup;  // head, its warp's share
  size_t row = (size_t)bq * kHq + g * kGroup + h;
  int n;      // splits or pieces to merge
  bool zero = false;  // a row without tokens
  if (p.bal_ctas > 0) {
    // The stream positions stage 1 used (integers, so both kernels agree
    // exactly), read while stage 1 still runs: tiles and rows with tokens
    // before row b and in all, and the shortest row.
    constexpr int nw = kGroup * W;
    __shared__ int red[5][nw];
    int v[5] = {0, 0, 0, 0, INT_MAX};  // tiles before b, rows before b, all tiles, all rows, min
    for (int bb = threadIdx.x; bb < p.batch; bb += nw * 32) {
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
    for (int w = 0; w < nw; ++w) {
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
  if constexpr (kChecked) {  // the row in the batch, its pieces in the workspace's split slots
    if (row >= (size_t)p.batch * p.q_len * kHq || n < 0 || n > p.num_splits) {
      atomicOr(p.flags, GQA_FLAG_BOUNDS);
      row = 0;
      n = min(max(n, 0), p.num_splits);
    }
  }
  float M, Ls;
  float4 o;
  merge_pieces<kMaxN>(p, row, n, share, W, M, Ls, o);
  if constexpr (W == 1) {
    write_merged<QF>(p, row, Ls, o);
  } else {
    // the W shares of each head through shared memory, merged in share order
    __shared__ float4 sh_o[kGroup][W][kD / 4];
    __shared__ float sh_m[kGroup][W], sh_l[kGroup][W];
    const int lane = threadIdx.x & 31;
    sh_o[h][share][lane] = o;
    if (lane == 0) {
      sh_m[h][share] = M;
      sh_l[h][share] = Ls;
    }
    __syncthreads();
    if (share != 0) return;
    float Mt = -INFINITY;
#pragma unroll
    for (int k = 0; k < W; ++k) Mt = fmaxf(Mt, sh_m[h][k]);
    float Lt = 0.f;
    float4 ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float mk = sh_m[h][k];
      const float a = mk == -INFINITY ? 0.f : ex2(mk - Mt);
      Lt = fmaf(sh_l[h][k], a, Lt);
      const float4 v = sh_o[h][k][lane];
      ot.x = fmaf(v.x, a, ot.x);
      ot.y = fmaf(v.y, a, ot.y);
      ot.z = fmaf(v.z, a, ot.z);
      ot.w = fmaf(v.w, a, ot.w);
    }
    write_merged<QF>(p, row, Lt, ot);
  }
}

}  // namespace gqa
