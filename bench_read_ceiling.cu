// Read ceiling of this GPU for the split kernel's access pattern: every CTA
// streams one contiguous run of a 4.3 GB buffer (the size of the bf16
// 8 x 131072 cache) through a shared-memory ring with 1-D bulk copies
// (cp.async.bulk, mbarrier complete_tx) and discards it — the split kernel's
// data movement without its arithmetic.  Prints one JSON object: GB/s per
// ring geometry and the best.  Built and run by `bench.py --read-ceiling`.
// Every wait is bounded (2 s); a run that gives up reports an error.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

namespace {

__device__ __forceinline__ uint32_t shared_address(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void barrier_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(shared_address(bar)), "r"(count));
}
__device__ __forceinline__ void barrier_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(shared_address(bar)) : "memory");
}
__device__ __forceinline__ void barrier_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(shared_address(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool barrier_wait(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  for (;;) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(shared_address(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (timer_ns() > deadline) return false;
  }
}

// CTA c reads chunks [c * per, min((c + 1) * per, chunks)); warp 0 lane 0
// issues the copies into `stages` ring slots, warp 1 lane 0 releases them.
__global__ void __launch_bounds__(64) stream_read(const uint8_t* buf, long long chunks, int chunk_bytes, int stages,
                                                  long long per, unsigned* error) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * chunk_bytes);
  uint64_t* empty = full + stages;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      barrier_init(&full[i], 1);
      barrier_init(&empty[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const long long c0 = (long long)blockIdx.x * per;
  const long long c1 = c0 + per < chunks ? c0 + per : chunks;
  const uint64_t deadline = timer_ns() + 2000000000ull;
  if (threadIdx.x == 0) {
    for (long long i = c0; i < c1; ++i) {
      const int k = (int)(i - c0), slot = k % stages;
      if (k >= stages && !barrier_wait(&empty[slot], ((k / stages) & 1) ^ 1, deadline)) {
        atomicOr(error, 1u);
        break;
      }
      barrier_expect(&full[slot], (uint32_t)chunk_bytes);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              shared_address(smem + (size_t)slot * chunk_bytes)),
          "l"(buf + i * chunk_bytes), "r"(chunk_bytes), "r"(shared_address(&full[slot]))
          : "memory");
    }
    // never leave with copies in flight: wait (bounded) for each slot's last copy
    const long long n = c1 - c0;
    for (int slot = 0; slot < stages && slot < n; ++slot) {
      const long long last = ((n - 1 - slot) / stages) * stages + slot;
      if (!barrier_wait(&full[slot], (uint32_t)((last / stages) & 1), deadline + 1000000000ull)) atomicOr(error, 4u);
    }
  } else if (threadIdx.x == 32) {
    for (long long i = c0; i < c1; ++i) {
      const int k = (int)(i - c0), slot = k % stages;
      if (!barrier_wait(&full[slot], (k / stages) & 1, deadline)) {
        atomicOr(error, 2u);
        break;
      }
      barrier_arrive(&empty[slot]);
    }
  }
}

struct Geometry {
  int chunk_bytes, ctas_per_sm, stages;
};

}  // namespace

int main() {
  const size_t bytes = 4295098368ull;  // 65,538 x 64 KB: the bf16 8 x 131072 cache, rounded to 64 KB
  uint8_t* buf = nullptr;
  unsigned* error = nullptr;
  if (cudaMalloc(&buf, bytes) != cudaSuccess || cudaMalloc(&error, sizeof(unsigned)) != cudaSuccess) {
    printf("{\"error\": \"cudaMalloc failed\"}\n");
    return 1;
  }
  cudaMemset(buf, 1, bytes);
  cudaMemset(error, 0, sizeof(unsigned));
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaFuncSetAttribute(stream_read, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  cudaEvent_t start, stop;
  cudaEventCreate(&start);
  cudaEventCreate(&stop);
  // the split kernel's own ring (16 KB per plane, 2 CTAs x 3 stages per SM),
  // and deeper or coarser rings
  const Geometry geos[] = {{16384, 2, 3}, {16384, 3, 4}, {16384, 4, 3}, {32768, 2, 2}, {32768, 1, 7}, {65536, 1, 2}};
  printf("{\"bytes\": %zu, \"sms\": %d, \"geometries\": [", bytes, sms);
  double best = 0.0;
  bool first = true;
  for (const Geometry& geo : geos) {
    const size_t smem = (size_t)geo.stages * geo.chunk_bytes + 2 * geo.stages * sizeof(uint64_t);
    const long long chunks = (long long)(bytes / geo.chunk_bytes);
    const int grid = sms * geo.ctas_per_sm;
    const long long per = (chunks + grid - 1) / grid;
    std::vector<float> ms;
    for (int rep = 0; rep < 10; ++rep) {
      cudaEventRecord(start);
      stream_read<<<grid, 64, smem>>>(buf, chunks, geo.chunk_bytes, geo.stages, per, error);
      cudaEventRecord(stop);
      cudaEventSynchronize(stop);
      float t = 0.f;
      cudaEventElapsedTime(&t, start, stop);
      if (rep >= 3) ms.push_back(t);
    }
    unsigned flags = 0;
    cudaMemcpy(&flags, error, sizeof(unsigned), cudaMemcpyDeviceToHost);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || flags != 0) {
      printf("], \"error\": \"%s, wait flags %u\"}\n", cudaGetErrorString(e), flags);
      return 1;
    }
    std::sort(ms.begin(), ms.end());
    const double t = ms[ms.size() / 2];
    const double gbps = (double)chunks * geo.chunk_bytes / (t * 1e-3) / 1e9;
    best = std::max(best, gbps);
    printf("%s{\"chunk_bytes\": %d, \"ctas_per_sm\": %d, \"stages\": %d, \"us\": %.1f, \"GBps\": %.1f}",
           first ? "" : ", ", geo.chunk_bytes, geo.ctas_per_sm, geo.stages, t * 1e3, gbps);
    first = false;
  }
  printf("], \"best_GBps\": %.1f}\n", best);
  return 0;
}
