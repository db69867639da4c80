// Device-side building blocks shared by the decode kernels: the fixed head
// geometry, the KV formats, and thin inline-PTX wrappers for the sm_90+ async
// machinery used on sm_103a (mbarrier, 1-D bulk copies through the TMA unit,
// L2 eviction policies, the global nanosecond timer) and the ex2 instruction.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace gqa {

// 32 query heads share 8 KV heads (4 per KV head), head_dim 128, one query
// token per request ("FlashInfer sm110_gqa_decode" article, "Input contract").
constexpr int kHq = 32;
constexpr int kHkv = 8;
constexpr int kGroup = kHq / kHkv;
constexpr int kD = 128;

enum KvFormat : int { kKvF16 = 0, kKvBF16 = 1, kKvE4M3 = 2, kKvI8 = 3 };
enum QFormat : int { kQF16 = 0, kQBF16 = 1 };

__host__ __device__ constexpr bool is_8bit(int kv_format) {
  return kv_format == kKvE4M3 || kv_format == kKvI8;
}

// Tokens per pipeline tile: one tile of one plane is 16 KB for every format.
__host__ __device__ constexpr int tile_tokens(int kv_format) {
  return is_8bit(kv_format) ? 128 : 64;
}

// Balanced schedule of the split kernel: the stream positions a row of n tiles
// occupies, rc for the fixed cost of a piece (loading q, the epilogue: about
// one tile's streaming time) and then one per tile; none for a row without
// tokens.  The split and combine kernels both count with these functions.
constexpr int kBalRowCost = 1;
__host__ __device__ constexpr int bal_row_positions(int n_tiles, int rc) {
  return n_tiles > 0 ? n_tiles + rc : 0;
}
// The row cost in use: kBalRowCost when some row holding tokens is shorter
// than a CTA's run without it (CTAs then differ in how many pieces they hold),
// else 0 (every CTA holds one or two pieces; counting the cost would only move
// the cuts off the run length's multiples, which measured slower on GB300 for
// bf16 8 x 131072).  sum_tiles: tiles over all rows of one KV head; min_tiles:
// the fewest tiles of a row that holds tokens.
__host__ __device__ inline int bal_row_cost(int sum_tiles, int min_tiles, int ctas, int q_min) {
  const int q0 = (kHkv * sum_tiles + ctas - 1) / ctas;
  return min_tiles < (q0 > q_min ? q0 : q_min) ? kBalRowCost : 0;
}

template <int KVF>
struct KvTraits {
  static constexpr int kElemBytes = is_8bit(KVF) ? 1 : 2;
  static constexpr int kRowBytes = kD * kElemBytes;  // one token of one KV head
  static constexpr int kTile = tile_tokens(KVF);
  static constexpr int kTileBytes = kTile * kRowBytes;
};

// Split geometry shared by the split and combine kernels: chunk = tokens per
// split, rounded up to whole tiles; effective split count = ceil(C / chunk).
__host__ __device__ inline int split_chunk(int capacity, int num_splits, int kv_format) {
  const int tile = tile_tokens(kv_format);
  const int per = (capacity + num_splits - 1) / num_splits;
  return (per + tile - 1) / tile * tile;
}
__host__ __device__ inline int split_count(int capacity, int num_splits, int kv_format) {
  const int chunk = split_chunk(capacity, num_splits, kv_format);
  return (capacity + chunk - 1) / chunk;
}

// Checked builds (compiled with -DGQA_CHECKED; the product library is not):
// every global-memory access of the kernels is tested against the extent of
// its buffer first.  One outside it sets GQA_FLAG_BOUNDS in the status word
// and is redirected to an address inside the buffer, so a bad index is
// reported and nothing faults.  The tests run their cases through such a
// build and require the flag never to be set.
#ifdef GQA_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
// [p, p + bytes) lies inside [base, base + extent)
__device__ __forceinline__ bool in_extent(const void* base, size_t extent, const void* p, size_t bytes) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(base), a = reinterpret_cast<uintptr_t>(p);
  return a >= b && bytes <= extent && a - b <= extent - bytes;
}

// Default bound of a pipeline wait (a healthy wait lasts microseconds).
constexpr uint64_t kWaitBudgetNs = 4000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the phase with the given parity has completed, or until the
// global timer passes `deadline_ns`; returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t deadline_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 63u) == 0 && global_timer_ns() > deadline_ns) return false;
  }
}

// L2 policy for data streamed exactly once (the KV cache).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared through the TMA unit; completion is counted
// in bytes on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
// Bulk prefetch of global memory into L2: a hint with no completion to
// track.  `src` 16-byte aligned, `bytes` a multiple of 16, the range inside
// the allocation.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: allow the next kernel in the stream (launched
// with programmatic stream serialization) to be scheduled now; and, in that
// kernel, wait until the preceding grid has completed and its writes are
// visible.  Both are no-ops when the launch did not opt in.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- thread-block clusters: barrier and distributed shared memory ----------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
// Every thread of every CTA in the cluster arrives, then waits for all of
// them; shared-memory writes before it are visible cluster-wide after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_address, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_address), "r"(rank));
  return d;
}
__device__ __forceinline__ float cluster_ld(uint32_t address) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(address) : "memory");
  return v;
}
__device__ __forceinline__ float4 cluster_ld4(uint32_t address) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(address)
               : "memory");
  return v;
}

// 2^x with the hardware approximation (subnormal results flushed to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- element conversions (exact) -------------------------------------------

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// bf16 is the upper half of an fp32 bit pattern.
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Two e4m3 bytes (low byte = first element) -> f16x2 with the hardware
// conversion; every e4m3 value is exact in fp16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  return h2;
}

// Two int8 codes (low byte = first element) -> exact f16x2 of code + 1152.
// With b = code + 128 (flip the sign bit), the f16 pattern 0x6400 | b is
// 1024 + b, an integer in [1024, 1279], exact in f16.  Four codes of a word
// give two pairs.  A dot product with these exceeds the codes' by
// kI8Bias times the sum of the other operand.
constexpr float kI8Bias = 1152.f;
__device__ __forceinline__ void i8x4_to_f16x2x2_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(x), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(x), "r"(0x64646464u));
}
// The codes themselves: subtracting 1152 is exact.
__device__ __forceinline__ void i8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  i8x4_to_f16x2x2_biased(w, a, b);
  const uint32_t bias = 0x64806480u;  // (1152, 1152)
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

}  // namespace gqa
