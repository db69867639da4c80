// Stage 1 of GQA decode: one CTA per (split s, KV head g, batch row b).
//
// Each CTA serves all 4 query heads of its KV head, so every K/V byte of the
// chunk [s*chunk, min((s+1)*chunk, len[b])) is read from HBM exactly once.
// The computation restates the "FlashInfer sm110_gqa_decode" article
// ("Convenience API": softmax in the log2 domain with the host-folded scale
// q_scale/sqrt(128)/ln 2, evaluated with ex2; "num_splits": split-KV chunks
// write FP32 partials that a merge step combines) and, for e4m3 KV, the
// "FP8 KV cache port on Jetson AGX Thor" blog (section 1, patch 2: the fp8 tile
// is promoted before the dot product; k_scale multiplies the scores, v_scale
// the output).
//
// Structure on sm_103a:
//   warp 8 (producer): one lane streams K and V tiles (16 KB per plane per
//     tile) with 1-D bulk copies through the TMA unit into a kStages-deep
//     shared-memory ring, signalling "full" mbarriers by transaction bytes and
//     waiting on "empty" mbarriers before reusing a stage.  Only rows below
//     the length are copied: slots >= len[b] are never read.
//   warps 0-7 (consumers): 32 token groups of 8 lanes.  A group owns one token
//     of the tile at a time; each lane owns 16 of the 128 dims (16-byte
//     conflict-free shared loads), holds q (pre-scaled into the log2 domain)
//     for the 4 heads in registers, forms partial dot products, and a 3-step
//     xor butterfly gives every lane the 4 full scores.  Each group keeps its
//     own running max / denominator / 4x16 accumulator (online softmax), so no
//     block-wide synchronisation happens inside the loop.  At the end the 32
//     group states are merged (log-sum-exp) through shuffles and shared memory.
//   Epilogue: with one split the CTA writes out = acc / l * v_scale rounded to
//     fp16/bf16; otherwise it writes the unnormalised accumulator, the max
//     (log2 domain) and the denominator to the workspace for stage 2.
// Every wait is bounded (kWaitBudgetNs): on timeout the CTA sets
// GQA_FLAG_WAIT_TIMEOUT, the producer waits (bounded) for its own copies in
// flight, and the CTA returns.
#pragma once

#include "common.cuh"

namespace gqa {

constexpr int kConsumerWarps = 8;
constexpr int kSplitThreads = (kConsumerWarps + 1) * 32;  // + 1 producer warp
constexpr int kStages = 4;
constexpr int kStageBytes = 2 * 16384;                          // K tile + V tile
constexpr int kMergeBytes = kConsumerWarps * kGroup * kD * 4 + 2 * kConsumerWarps * kGroup * 4;
constexpr int kSplitSmemBytes = kStages * kStageBytes + kMergeBytes + 2 * kStages * 8;

struct SplitParams {
  const void* q;          // [B,32,128] fp16/bf16
  const void* kv;         // [B,2,8,C,128] fp16/bf16/e4m3
  const int32_t* lens;    // [B]
  void* out;              // [B,32,128], written when the effective split count is 1
  float* part_o;          // [B,32,S,128]
  float* part_m;          // [B,32,S]  running max, log2 domain
  float* part_l;          // [B,32,S]  softmax denominator
  uint32_t* flags;        // workspace status word
  int batch, capacity, num_splits, chunk, splits_eff;
  float scale_log2;       // q_scale * k_scale * log2(e) / sqrt(128)
  float v_scale;
};

// Owned dims of lane c (0..7) of a token group, i = 0..15.  2-byte formats:
// 16-byte chunks c and c+8 of the row (dims 8c..8c+7 and 64+8c..64+8c+7);
// e4m3: chunk c (dims 16c..16c+15).  Each quarter-warp reads 128 contiguous
// bytes of one row: no bank conflicts.
template <int KVF>
__device__ __forceinline__ int owned_dim(int c, int i) {
  if constexpr (KVF == kKvE4M3) return 16 * c + i;
  else return i < 8 ? 8 * c + i : 64 + 8 * c + (i - 8);
}

// Load the 16 owned elements of one row from shared memory as fp32.
template <int KVF>
__device__ __forceinline__ void load_row(const uint8_t* row, int c, float (&x)[16]) {
  if constexpr (KVF == kKvE4M3) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(ws[k] & 0xffffu)));
      const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(ws[k] >> 16)));
      x[4 * k + 0] = lo.x;
      x[4 * k + 1] = lo.y;
      x[4 * k + 2] = hi.x;
      x[4 * k + 3] = hi.y;
    }
  } else {
    const uint4 a = *reinterpret_cast<const uint4*>(row + 16 * c);
    const uint4 b = *reinterpret_cast<const uint4*>(row + 16 * (c + 8));
    const uint32_t ws[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 f = KVF == kKvF16 ? f16x2_to_f32x2(ws[k]) : bf16x2_to_f32x2(ws[k]);
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  }
}

template <int QF>
__device__ __forceinline__ float2 q_pair_to_f32(uint32_t w) {
  return QF == kQF16 ? f16x2_to_f32x2(w) : bf16x2_to_f32x2(w);
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

template <int KVF, int QF>
__global__ void __launch_bounds__(kSplitThreads, 1)
    split_kv_kernel(const __grid_constant__ SplitParams p) {
  using T = KvTraits<KVF>;
  constexpr int kTpg = T::kTile / 32;  // tokens per group per tile (2 or 4)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* mrg_acc = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [8][4][128]
  float* mrg_m = mrg_acc + kConsumerWarps * kGroup * kD;                      // [8][4]
  float* mrg_l = mrg_m + kConsumerWarps * kGroup;                             // [8][4]
  uint64_t* full = reinterpret_cast<uint64_t*>(mrg_l + kConsumerWarps * kGroup);
  uint64_t* empty = full + kStages;

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int C = p.capacity;
  const int len_raw = __ldg(p.lens + b);
  const int L = min(max(len_raw, 0), C);
  if (s == 0 && g == 0 && threadIdx.x == 0 && (len_raw < 1 || len_raw > C))
    atomicOr(p.flags, GQA_FLAG_LENGTH_CLAMPED);
  const int t_begin = s * p.chunk;
  const int t_end = min(L, t_begin + p.chunk);

  if (t_begin >= t_end) {
    // Nothing to attend to.  Split 0 of a one-split launch owns the output
    // (length clamped to 0): write zeros.  Other splits are skipped by stage 2.
    if (p.splits_eff == 1 && threadIdx.x < kGroup * kD / 2) {
      const int j = threadIdx.x / (kD / 2), d0 = 2 * (threadIdx.x % (kD / 2));
      uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.out) +
                                                ((size_t)(b * kHq + g * kGroup + j) * kD + d0) * 2);
      *o = 0u;
    }
    return;
  }
  const int n_tiles = (t_end - t_begin + T::kTile - 1) / T::kTile;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t deadline = global_timer_ns() + kWaitBudgetNs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const size_t plane = (size_t)kHkv * C * T::kRowBytes;
      const uint8_t* gK = static_cast<const uint8_t*>(p.kv) +
                          ((size_t)b * 2 * kHkv + g) * (size_t)C * T::kRowBytes;
      const uint8_t* gV = gK + plane;
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1, deadline)) {
          ok = false;
          break;
        }
        const int t0 = t_begin + i * T::kTile;
        const uint32_t bytes = (uint32_t)min(T::kTile, t_end - t0) * T::kRowBytes;
        mbar_arrive_expect_tx(&full[st], 2 * bytes);
        bulk_load(ring + st * kStageBytes, gK + (size_t)t0 * T::kRowBytes, bytes, &full[st], pol);
        bulk_load(ring + st * kStageBytes + T::kTileBytes, gV + (size_t)t0 * T::kRowBytes, bytes,
                  &full[st], pol);
        ++issued;
      }
      if (!ok) atomicOr(p.flags, GQA_FLAG_WAIT_TIMEOUT);
      // Never leave the CTA with copies in flight: wait (bounded) for the
      // last use of every stage to land.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(&full[i % kStages], (i / kStages) & 1, deadline + kWaitBudgetNs);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;  // 0..255
  const int grp = ctid >> 3, c = ctid & 7;

  float qr[kGroup][16];
  {
    const uint8_t* qbase =
        static_cast<const uint8_t*>(p.q) + ((size_t)b * kHq + g * kGroup) * kD * 2;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const uint8_t* qrow = qbase + (size_t)j * kD * 2;
      uint32_t w[8];
      if constexpr (KVF == kKvE4M3) {  // dims 16c..16c+15: 32 contiguous bytes
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(qrow + 32 * c));
        const uint4 bb = __ldg(reinterpret_cast<const uint4*>(qrow + 32 * c + 16));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = bb.x; w[5] = bb.y; w[6] = bb.z; w[7] = bb.w;
      } else {  // dims 8c..8c+7 and 64+8c..64+8c+7
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(qrow + 16 * c));
        const uint4 bb = __ldg(reinterpret_cast<const uint4*>(qrow + 128 + 16 * c));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = bb.x; w[5] = bb.y; w[6] = bb.z; w[7] = bb.w;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 f = q_pair_to_f32<QF>(w[k]);
        qr[j][2 * k] = f.x * p.scale_log2;
        qr[j][2 * k + 1] = f.y * p.scale_log2;
      }
    }
  }

  float acc[kGroup][16];
  float m[kGroup], l[kGroup];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[j][i] = 0.f;
  }

  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&full[st], (i / kStages) & 1, deadline)) {
      if (lane == 0) atomicOr(p.flags, GQA_FLAG_WAIT_TIMEOUT);
      break;
    }
    const uint8_t* sK = ring + st * kStageBytes;
    const uint8_t* sV = sK + T::kTileBytes;
    const int rows = min(T::kTile, t_end - (t_begin + i * T::kTile));

    // scores of this group's tokens (rows grp, grp+32, ...) for the 4 heads
    float sc[kTpg][kGroup];
#pragma unroll
    for (int u = 0; u < kTpg; ++u) {
      float kf[16];
      load_row<KVF>(sK + (u * 32 + grp) * T::kRowBytes, c, kf);
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        float e = 0.f, o = 0.f;
#pragma unroll
        for (int d = 0; d < 16; d += 2) {
          e = fmaf(qr[j][d], kf[d], e);
          o = fmaf(qr[j][d + 1], kf[d + 1], o);
        }
        sc[u][j] = e + o;
      }
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1)
#pragma unroll
      for (int u = 0; u < kTpg; ++u)
#pragma unroll
        for (int j = 0; j < kGroup; ++j) sc[u][j] += __shfl_xor_sync(0xffffffffu, sc[u][j], off);

    // online softmax update (identical in all 8 lanes of the group)
    float mx[kGroup];
    bool grow = false;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      mx[j] = m[j];
#pragma unroll
      for (int u = 0; u < kTpg; ++u) {
        if (u * 32 + grp >= rows) sc[u][j] = -INFINITY;  // select, never multiply
        mx[j] = fmaxf(mx[j], sc[u][j]);
      }
      grow |= mx[j] > m[j];
    }
    if (grow) {
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        const float a = ex2(m[j] - mx[j]);  // 0 when m was -inf
        l[j] *= a;
#pragma unroll
        for (int d = 0; d < 16; ++d) acc[j][d] *= a;
        m[j] = mx[j];
      }
    }
    float pr[kTpg][kGroup];
#pragma unroll
    for (int u = 0; u < kTpg; ++u)
#pragma unroll
      for (int j = 0; j < kGroup; ++j) {
        pr[u][j] = sc[u][j] == -INFINITY ? 0.f : ex2(sc[u][j] - m[j]);
        l[j] += pr[u][j];
      }
#pragma unroll
    for (int u = 0; u < kTpg; ++u) {
      if (u * 32 + grp < rows) {
        float vf[16];
        load_row<KVF>(sV + (u * 32 + grp) * T::kRowBytes, c, vf);
#pragma unroll
        for (int j = 0; j < kGroup; ++j)
#pragma unroll
          for (int d = 0; d < 16; ++d) acc[j][d] = fmaf(pr[u][j], vf[d], acc[j][d]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- merge the 4 token groups of this warp (lanes with equal c)
#pragma unroll
  for (int off = 8; off < 32; off <<= 1) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[j], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[j], off);
      const float mn = fmaxf(m[j], mo);
      const float a = m[j] == -INFINITY ? 0.f : ex2(m[j] - mn);
      const float bb = mo == -INFINITY ? 0.f : ex2(mo - mn);
      l[j] = l[j] * a + lo * bb;
#pragma unroll
      for (int d = 0; d < 16; ++d)
        acc[j][d] = acc[j][d] * a + __shfl_xor_sync(0xffffffffu, acc[j][d], off) * bb;
      m[j] = mn;
    }
  }
  if (lane < 8) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
#pragma unroll
      for (int d = 0; d < 16; ++d) mrg_acc[(warp * kGroup + j) * kD + owned_dim<KVF>(c, d)] = acc[j][d];
      if (c == 0) {
        mrg_m[warp * kGroup + j] = m[j];
        mrg_l[warp * kGroup + j] = l[j];
      }
    }
  }
  named_barrier_sync(1, kConsumerWarps * 32);

  // ---- merge the 8 warps: thread -> (head j, dims d0, d0+1)
  const int j = ctid / (kD / 2), d0 = 2 * (ctid % (kD / 2));
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg_m[w * kGroup + j]);
  float Ls = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) {
    const float mw = mrg_m[w * kGroup + j];
    const float a = mw == -INFINITY ? 0.f : ex2(mw - M);
    Ls = fmaf(mrg_l[w * kGroup + j], a, Ls);
    const float2 v = *reinterpret_cast<const float2*>(&mrg_acc[(w * kGroup + j) * kD + d0]);
    o0 = fmaf(v.x, a, o0);
    o1 = fmaf(v.y, a, o1);
  }
  const int h = g * kGroup + j;
  if (p.splits_eff == 1) {
    const float inv = p.v_scale / Ls;
    uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.out) +
                                              ((size_t)(b * kHq + h) * kD + d0) * 2);
    *o = pack_out<QF>(o0 * inv, o1 * inv);
  } else {
    const size_t idx = (size_t)(b * kHq + h) * p.num_splits + s;
    *reinterpret_cast<float2*>(p.part_o + idx * kD + d0) = make_float2(o0, o1);
    if (d0 == 0) {
      p.part_m[idx] = M;
      p.part_l[idx] = Ls;
    }
  }
}

}  // namespace gqa
