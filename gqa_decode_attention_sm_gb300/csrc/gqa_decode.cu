// Host side of libgqa_decode.so: argument validation, the one-time device
// check, the split planner, workspace layout and kernel launches behind the C
// ABI declared in include/gqa_decode.h.
//
// The API shape follows the "FlashInfer sm110_gqa_decode" article: a
// convenience call, a prepared call that allocates nothing and reads nothing
// back (capturable in a CUDA graph), fail-fast validation before any launch
// (its "prepare" step: contiguous/aligned tensors, output not aliasing an
// input, finite positive q_scale, a compatible device), and a split-KV
// workspace owned by the caller.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "gqa_decode.h"
#include "kernels/append_kv.cuh"
#include "kernels/combine.cuh"
#include "kernels/common.cuh"
#include "kernels/split_kv_mma.cuh"

static_assert(GQA_MAX_SPLITS <= 32 * gqa::kCombineChunks, "the combine's chunks cover every split slot");

namespace {

using namespace gqa;

thread_local std::string g_last_error;

gqa_status_t fail(gqa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

gqa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(GQA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- devices

constexpr int kMaxDevices = 64;
constexpr int kClusterMaxSplits = 8;  // the on-chip merge: clusters of 2..8 splits (portable sizes)

// Per-device result of the one-time check.  Kept once known for good: the
// device is ready (sm_count set) or is not a compute capability 10.3 part.  A
// CUDA error during the check is not kept, so a later call retries it.
struct DeviceState {
  std::mutex mu;
  std::atomic<int> state{0};  // 0 unknown, 1 ready, 2 unsupported
  gqa_status_t status = GQA_ERR_UNSUPPORTED_DEVICE;
  int sm_count = 0;
  std::string message;
  // The most clusters of s CTAs of the cluster-merge split kernel that can be
  // resident at once, by [KV format][q format][q_len - 1][s]
  // (cudaOccupancyMaxActiveClusters).  A cluster's CTAs share one GPC, so a
  // grid that nearly fills the SMs can hold fewer clusters than slots / s.
  int cluster_fit[4][2][kMaxQLen][kClusterMaxSplits + 1] = {};
};
DeviceState g_devices[kMaxDevices];

template <int KVF, int QF>
cudaError_t set_split_attributes() {
  cudaError_t e = cudaSuccess;
  const auto set = [&](auto kernel, int bytes) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  };
  set(split_kv_mma_kernel<KVF, QF, 1, false, false>, mma_smem_bytes(KVF, 1));
  set(split_kv_mma_kernel<KVF, QF, 2, false, false>, mma_smem_bytes(KVF, 2));
  set(split_kv_mma_kernel<KVF, QF, 3, false, false>, mma_smem_bytes(KVF, 3));
  set(split_kv_mma_kernel<KVF, QF, 4, false, false>, mma_smem_bytes(KVF, 4));
  set(split_kv_mma_kernel<KVF, QF, 1, true, false>, mma_smem_bytes(KVF, 1, true));
  set(split_kv_mma_kernel<KVF, QF, 2, true, false>, mma_smem_bytes(KVF, 2, true));
  set(split_kv_mma_kernel<KVF, QF, 3, true, false>, mma_smem_bytes(KVF, 3, true));
  set(split_kv_mma_kernel<KVF, QF, 4, true, false>, mma_smem_bytes(KVF, 4, true));
  set(split_kv_mma_kernel<KVF, QF, 1, false, true>, mma_smem_bytes(KVF, 1));
  set(split_kv_mma_kernel<KVF, QF, 2, false, true>, mma_smem_bytes(KVF, 2));
  set(split_kv_mma_kernel<KVF, QF, 3, false, true>, mma_smem_bytes(KVF, 3));
  set(split_kv_mma_kernel<KVF, QF, 4, false, true>, mma_smem_bytes(KVF, 4));
  return e;
}

template <int KVF, int QF, int NQ>
cudaError_t query_cluster_fit(DeviceState& st) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMmaThreads, 1, 1);
  cfg.dynamicSmemBytes = mma_smem_bytes(KVF, NQ);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int s = 2; s <= kClusterMaxSplits; ++s) {
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)s;
    cfg.gridDim = dim3(kHkv, 1, (unsigned)s);
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, split_kv_mma_kernel<KVF, QF, NQ, false, true>, &cfg);
    if (e != cudaSuccess) return e;
    st.cluster_fit[KVF][QF][NQ - 1][s] = n;
  }
  return cudaSuccess;
}

template <int KVF, int QF>
cudaError_t query_cluster_fits(DeviceState& st) {
  cudaError_t e = query_cluster_fit<KVF, QF, 1>(st);
  if (e == cudaSuccess) e = query_cluster_fit<KVF, QF, 2>(st);
  if (e == cudaSuccess) e = query_cluster_fit<KVF, QF, 3>(st);
  if (e == cudaSuccess) e = query_cluster_fit<KVF, QF, 4>(st);
  return e;
}

// One-time per-device check (compute capability 10.3), opt-in to the split
// kernel's dynamic shared memory, and the cluster occupancy table.  Runs
// with `dev` current.
void init_device(int dev, DeviceState& st) {
  int major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    st.status = GQA_ERR_CUDA;
    st.message = std::string("device query failed: ") + cudaGetErrorString(e);
    return;
  }
  if (major != 10 || minor != 3) {
    st.status = GQA_ERR_UNSUPPORTED_DEVICE;
    char buf[160];
    snprintf(buf, sizeof buf, "GQA decode requires compute capability 10.3 (sm_103); device %d is %d.%d",
             dev, major, minor);
    st.message = buf;
    return;
  }
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != dev) cudaSetDevice(dev);
  cudaError_t a = set_split_attributes<kKvF16, kQF16>();
  if (a == cudaSuccess) a = set_split_attributes<kKvBF16, kQBF16>();
  if (a == cudaSuccess) a = set_split_attributes<kKvE4M3, kQBF16>();
  if (a == cudaSuccess) a = set_split_attributes<kKvE4M3, kQF16>();
  if (a == cudaSuccess) a = set_split_attributes<kKvI8, kQBF16>();
  if (a == cudaSuccess) a = set_split_attributes<kKvI8, kQF16>();
  const char* what = "cudaFuncSetAttribute";
  if (a == cudaSuccess) {
    what = "cudaOccupancyMaxActiveClusters";
    a = query_cluster_fits<kKvF16, kQF16>(st);
    if (a == cudaSuccess) a = query_cluster_fits<kKvBF16, kQBF16>(st);
    if (a == cudaSuccess) a = query_cluster_fits<kKvE4M3, kQBF16>(st);
    if (a == cudaSuccess) a = query_cluster_fits<kKvE4M3, kQF16>(st);
    if (a == cudaSuccess) a = query_cluster_fits<kKvI8, kQBF16>(st);
    if (a == cudaSuccess) a = query_cluster_fits<kKvI8, kQF16>(st);
  }
  if (prev >= 0 && prev != dev) cudaSetDevice(prev);
  if (a != cudaSuccess) {
    st.status = GQA_ERR_CUDA;
    st.message = std::string(what) + " failed: " + cudaGetErrorString(a);
    return;
  }
  st.sm_count = sms;
  st.status = GQA_OK;
}

gqa_status_t device_ready(int dev, int* sm_count) {
  if (dev < 0 || dev >= kMaxDevices) return fail(GQA_ERR_UNSUPPORTED_DEVICE, "device %d out of range", dev);
  DeviceState& st = g_devices[dev];
  int known = st.state.load(std::memory_order_acquire);
  if (known == 0) {
    std::lock_guard<std::mutex> lock(st.mu);
    known = st.state.load(std::memory_order_relaxed);
    if (known == 0) {
      init_device(dev, st);
      if (st.status == GQA_OK) known = 1;
      else if (st.status == GQA_ERR_UNSUPPORTED_DEVICE) known = 2;
      else return fail(st.status, "%s", st.message.c_str());  // not kept: retried next call
      st.state.store(known, std::memory_order_release);
    }
  }
  if (known == 2) return fail(GQA_ERR_UNSUPPORTED_DEVICE, "%s", st.message.c_str());
  if (sm_count) *sm_count = st.sm_count;
  return GQA_OK;
}

gqa_status_t current_device_ready(int* sm_count) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  return device_ready(dev, sm_count);
}

// ------------------------------------------------------------- validation

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

size_t kv_elem_bytes(int fmt) { return is_8bit(fmt) ? 1 : 2; }

size_t partial_o_bytes(int batch, int splits) {
  return align_up((size_t)batch * kHq * splits * kD * sizeof(float), 256);
}
size_t partial_ml_bytes(int batch, int splits) {
  return align_up((size_t)batch * kHq * splits * sizeof(float), 256);
}

size_t workspace_bytes_for(int batch, int splits) {
  if (splits <= 1) return GQA_WORKSPACE_HEADER_BYTES;
  return GQA_WORKSPACE_HEADER_BYTES + partial_o_bytes(batch, splits) + 2 * partial_ml_bytes(batch, splits);
}

struct Call {
  const void* q;
  int q_dtype;
  const void* kv;
  int kv_format;
  const int32_t* lens;
  void* out;
  int batch, capacity;
  float q_scale, k_scale, v_scale;
  int num_splits;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  uint64_t wait_budget_ns = kWaitBudgetNs;
  int skip_tile = -1;
  const uint16_t* kv_scales = nullptr;  // int8 cache only
  const int32_t* block_table = nullptr;  // paged cache only
  int page_log2 = 0, max_pages = 0, num_pages = 0;
  int q_len = 1;  // query tokens per request (verify window)
  int sms = 0;    // SM count of the current device (set once validated)
};

gqa_status_t validate_shape(int batch, int capacity) {
  if (batch < 1 || batch > 65535) return fail(GQA_ERR_INVALID_ARGUMENT, "batch %d outside [1, 65535]", batch);
  if (capacity < 1 || capacity > (1 << 30))
    return fail(GQA_ERR_INVALID_ARGUMENT, "capacity %d outside [1, 2^30]", capacity);
  return GQA_OK;
}

// Checks that need no CUDA call.  `q_scale_min_exclusive`: the prepared entry
// requires q_scale > 0, the others q_scale >= 0.
gqa_status_t validate(const Call& c, bool q_scale_positive, bool need_q) {
  if ((need_q && !c.q) || !c.kv || !c.lens || !c.out || !c.workspace)
    return fail(GQA_ERR_INVALID_ARGUMENT, "null pointer argument");
  gqa_status_t st = validate_shape(c.batch, c.capacity);
  if (st != GQA_OK) return st;
  if (c.q_dtype != GQA_F16 && c.q_dtype != GQA_BF16)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown q/out dtype %d", c.q_dtype);
  if (c.kv_format != kKvF16 && c.kv_format != kKvBF16 && c.kv_format != kKvE4M3 && c.kv_format != kKvI8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", c.kv_format);
  if (!is_8bit(c.kv_format) && c.kv_format != c.q_dtype)
    return fail(GQA_ERR_INVALID_ARGUMENT, "fp16/bf16 KV must have the dtype of q");
  if (c.kv_format == kKvI8 && (!c.kv_scales || !aligned(c.kv_scales, 16) || c.capacity % 8 != 0))
    return fail(GQA_ERR_INVALID_ARGUMENT,
                "an int8 cache needs a 16-byte aligned bf16 scale array and a capacity that is a multiple of 8");
  if (!std::isfinite(c.q_scale) || c.q_scale < 0.f || (q_scale_positive && c.q_scale == 0.f))
    return fail(GQA_ERR_INVALID_ARGUMENT, "q_scale must be finite and %s 0", q_scale_positive ? ">" : ">=");
  if (!std::isfinite(c.k_scale) || c.k_scale <= 0.f || !std::isfinite(c.v_scale) || c.v_scale <= 0.f)
    return fail(GQA_ERR_INVALID_ARGUMENT, "k_scale and v_scale must be finite and > 0");
  if (c.num_splits < 1 || c.num_splits > GQA_MAX_SPLITS)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits %d outside [1, %d]", c.num_splits, GQA_MAX_SPLITS);
  if ((need_q && !aligned(c.q, 16)) || !aligned(c.kv, 16) || !aligned(c.out, 16) ||
      !aligned(c.workspace, 16) || !aligned(c.lens, 4))
    return fail(GQA_ERR_INVALID_ARGUMENT, "q, kv, out, workspace must be 16-byte aligned, lens 4-byte");
  const size_t need = workspace_bytes_for(c.batch * c.q_len, c.num_splits);
  if (c.workspace_bytes < need)
    return fail(GQA_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", c.workspace_bytes, need);
  const size_t qo_bytes = (size_t)c.batch * c.q_len * kHq * kD * 2;
  const size_t kv_bytes =
      c.block_table ? (size_t)c.num_pages * 2 * kHkv * ((size_t)1 << c.page_log2) * kD * kv_elem_bytes(c.kv_format)
                    : (size_t)c.batch * 2 * kHkv * (size_t)c.capacity * kD * kv_elem_bytes(c.kv_format);
  const size_t lens_bytes = (size_t)c.batch * 4;
  if ((need_q && overlap(c.out, qo_bytes, c.q, qo_bytes)) || overlap(c.out, qo_bytes, c.kv, kv_bytes) ||
      overlap(c.out, qo_bytes, c.lens, lens_bytes) || overlap(c.out, qo_bytes, c.workspace, need))
    return fail(GQA_ERR_ALIASING, "out overlaps q, kv, lens or the workspace");
  if ((need_q && overlap(c.workspace, need, c.q, qo_bytes)) || overlap(c.workspace, need, c.kv, kv_bytes) ||
      overlap(c.workspace, need, c.lens, lens_bytes))
    return fail(GQA_ERR_ALIASING, "workspace overlaps q, kv or lens");
  if (c.block_table) {
    const size_t bt_bytes = (size_t)c.batch * c.max_pages * 4;
    if (overlap(c.out, qo_bytes, c.block_table, bt_bytes) || overlap(c.workspace, need, c.block_table, bt_bytes))
      return fail(GQA_ERR_ALIASING, "out or the workspace overlaps the block table");
  }
  if (c.kv_format == kKvI8) {
    const size_t sc_bytes = c.block_table ? (size_t)c.num_pages * 2 * kHkv * ((size_t)1 << c.page_log2) * 2
                                          : (size_t)c.batch * 2 * kHkv * (size_t)c.capacity * 2;
    if (overlap(c.out, qo_bytes, c.kv_scales, sc_bytes) || overlap(c.workspace, need, c.kv_scales, sc_bytes))
      return fail(GQA_ERR_ALIASING, "out or the workspace overlaps the int8 scales");
  }
  return GQA_OK;
}

// ------------------------------------------------ static (no-alloc) scratch

// Scratch for gqa_decode_noalloc.  In host code this name is only a stand-in
// for the device symbol: its device address comes from cudaGetSymbolAddress,
// once per device, with that device current.
constexpr size_t kStaticWorkspaceBytes = GQA_STATIC_WORKSPACE_BYTES;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

struct StaticWorkspace {
  std::mutex mu;
  std::atomic<void*> ptr{nullptr};  // set once set-up has succeeded on the device
};
StaticWorkspace g_static_ws[kMaxDevices];

// Device address of the static scratch on the current device `dev`.  Set-up
// (the first successful call per device): look the address up and zero the
// header (the status word) on `stream`.  Only a successful set-up is kept: a
// failed lookup (no context yet, a transient error) is retried by the next
// call.  The address stays valid for the life of the device's primary
// context; it goes stale after cudaDeviceReset.
gqa_status_t static_workspace(int dev, cudaStream_t stream, void** ptr) {
  if (dev < 0 || dev >= kMaxDevices) return fail(GQA_ERR_UNSUPPORTED_DEVICE, "device %d out of range", dev);
  StaticWorkspace& s = g_static_ws[dev];
  void* p = s.ptr.load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(s.mu);
    p = s.ptr.load(std::memory_order_relaxed);
    if (!p) {
      cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
      e = cudaMemsetAsync(p, 0, GQA_WORKSPACE_HEADER_BYTES, stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static workspace header)");
      s.ptr.store(p, std::memory_order_release);
    }
  }
  *ptr = p;
  return GQA_OK;
}

// --------------------------------------------------------------- planning

int plan_splits(int batch, int capacity, int kv_format, int sm_count) {
  const long long tile = tile_tokens(kv_format);
  const long long units = (long long)batch * kHkv;
  const long long ctas_per_sm = mma_ctas_per_sm(kv_format, 1);
  const long long slots = ctas_per_sm * (sm_count > 0 ? sm_count : 148);
  const long long nmax = (capacity + tile - 1) / tile;
  long long per;
  if (units * nmax <= 16 * slots) {
    // Latency-bound sizes (at most 16 tiles per resident slot over the worst
    // case): one wave of work items at most, about sqrt(6 nmax) splits per
    // row — fewer leave each CTA more tiles to stream, more leave the merge
    // more partials.  Measured in CUDA graphs on GB300 (us per call, the
    // 8-wave rule -> this): bf16 1 x 4096 10.7 -> 9.0, 1 x 16384 20.6 -> 17.1,
    // 4 x 4096 16.4 -> 14.6, e4m3 1 x 8192 11.5 -> 10.3, fp16 1 x 1024 6.3.
    //
    // Batches of 8 or more rows of 4096 slots or more are not capped at one
    // wave, so they run the balanced schedule: a decode batch's lengths are
    // ragged, and only the balanced schedule spreads the actual tokens over
    // all the resident CTAs (a one-wave grid waits for the CTAs of its
    // longest rows).  Warm, in a CUDA graph, us per call, one wave ->
    // balanced, lengths U[C/4, C] and all = C: bf16 8 x 4096 22.7 -> 18.9 and
    // 24.2 -> 25.7, e4m3 16 x 4096 24.8 -> 21.2 and 26.4 -> 27.1, e4m3 8 x
    // 4096 15.6 -> 14.7 and 17.2 -> 17.6, int8 8 x 8192 26.8 -> 22.6 and 28.3
    // -> 28.3.  Shorter rows or smaller batches keep the one-wave grid: there
    // the balanced grid's extra pieces and combine cost more than it
    // balances (bf16 32 x 512 12.8 -> 14.9 and 13.7 -> 18.3, e4m3 16 x 1024
    // 10.4 -> 12.6 and 11.1 -> 14.3; bf16 4 x 8192 22.2 -> 20.2 but 24.1 ->
    // 26.1).
    long long s = (long long)std::llround(std::sqrt(6.0 * (double)nmax));
    const long long wave = slots / units;
    if (s > wave && !(batch >= 8 && capacity >= 4096)) s = wave;
    if (s < 1) s = 1;
    per = (capacity + s - 1) / s;
  } else {
    // Otherwise about 8 waves of work items over the worst case (every
    // length = capacity); such grids run the balanced schedule, where the
    // split count only bounds the pieces of a row.
    const long long target_ctas = 8LL * slots;
    per = (units * capacity + target_ctas - 1) / target_ctas;
  }
  per = (per + tile - 1) / tile * tile;
  // at least two tiles per split: a one-tile split costs more in fixed
  // prologue/epilogue than it streams (measured on the 1 x 1024 fp16 case)
  if (per < 2 * tile) per = 2 * tile;
  long long s = (capacity + per - 1) / per;
  if (s < 1) s = 1;
  if (s > GQA_MAX_SPLITS) s = GQA_MAX_SPLITS;
  return (int)s;
}

// ---------------------------------------------------------------- launches

// `bal_ctas` > 0: the balanced schedule on that many CTAs (single token).
// `cluster`: the one-piece grid as clusters of its `cluster` splits, merged
// on chip (no combine kernel).
template <int KVF, int QF, bool BAL, bool CL>
cudaError_t launch_nq(cudaLaunchConfig_t& cfg, const SplitParams& sp, int q_len) {
  switch (q_len) {
    case 1: return cudaLaunchKernelEx(&cfg, split_kv_mma_kernel<KVF, QF, 1, BAL, CL>, sp);
    case 2: return cudaLaunchKernelEx(&cfg, split_kv_mma_kernel<KVF, QF, 2, BAL, CL>, sp);
    case 3: return cudaLaunchKernelEx(&cfg, split_kv_mma_kernel<KVF, QF, 3, BAL, CL>, sp);
    default: return cudaLaunchKernelEx(&cfg, split_kv_mma_kernel<KVF, QF, 4, BAL, CL>, sp);
  }
}

template <int KVF, int QF>
cudaError_t launch_split_t(const SplitParams& sp, int q_len, int bal_ctas, int cluster, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMmaThreads, 1, 1);
  cfg.stream = stream;
  // programmatic dependent launch: CTAs may become resident while the
  // previous grid in the stream drains; they wait (griddepcontrol.wait)
  // before reading any input
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bal_ctas > 0) {
    cfg.gridDim = dim3(bal_ctas, 1, 1);
    cfg.dynamicSmemBytes = mma_smem_bytes(KVF, q_len, true);
    return launch_nq<KVF, QF, true, false>(cfg, sp, q_len);
  }
  cfg.gridDim = dim3(kHkv, sp.batch, sp.splits_eff);
  cfg.dynamicSmemBytes = mma_smem_bytes(KVF, q_len);
  if (cluster > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = (unsigned)cluster;
    cfg.numAttrs = 2;
    return launch_nq<KVF, QF, false, true>(cfg, sp, q_len);
  }
  return launch_nq<KVF, QF, false, false>(cfg, sp, q_len);
}

template <int QF>
cudaError_t launch_combine_t(const CombineParams& cp, int batch_rows, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kHkv, batch_rows, 1);
  cfg.blockDim = dim3(kGroup * 32 * cp.warps_per_head, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // programmatic dependent launch: may be scheduled while stage 1 drains; the
  // kernel waits (griddepcontrol.wait) before it reads the partials
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (cp.warps_per_head) {
    case 1: return cudaLaunchKernelEx(&cfg, combine_kernel<QF, 1>, cp);
    case 2: return cudaLaunchKernelEx(&cfg, combine_kernel<QF, 2>, cp);
    default: return cudaLaunchKernelEx(&cfg, combine_kernel<QF, 4>, cp);
  }
}

struct Layout {
  float* part_o;
  float* part_m;
  float* part_l;
  uint32_t* flags;
};

Layout layout_of(void* ws, int batch, int splits) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  Layout l;
  l.flags = reinterpret_cast<uint32_t*>(base);
  uint8_t* p = base + GQA_WORKSPACE_HEADER_BYTES;
  l.part_o = reinterpret_cast<float*>(p);
  p += partial_o_bytes(batch, splits);
  l.part_m = reinterpret_cast<float*>(p);
  p += partial_ml_bytes(batch, splits);
  l.part_l = reinterpret_cast<float*>(p);
  return l;
}

// Checked builds: how far the extents given to the split kernel's range
// checks are cut short (gqa_decode_debug_cut_extents), so a test can make
// the checks fire while every redirected access stays in the real buffers.
std::atomic<uint64_t> g_cut_kv_bytes{0}, g_cut_scales_bytes{0};

// The balanced schedule serves decode and verify windows of batches up to
// kBalMaxBatch whose rows can be split (two or more tiles of capacity) and
// whose one-piece-per-CTA grid would take more than one wave, as long as the
// global stream (n + kBalRowCost positions for a row of n tiles, the first
// ones standing for the piece's fixed cost) fits an int.  q_min keeps every
// row within the workspace's split slots: a row of n <= nmax tiles meets at
// most ceil(n / q) + 1 <= num_splits CTAs.  Measured on GB300 (us per call,
// back to back): fp16 32 x U[1,8192] 96.4 -> 89.9, e4m3 64 x U[16k,32k]
// 459.4 -> 443.7, bf16 8 x 131072 589.4 -> 584.3.
struct BalPlan {
  int ctas = 0;  // 0: the one-piece-per-CTA grid
  int q_min = 0;
};

BalPlan bal_plan(const Call& c) {
  BalPlan bp;
  const int tile = tile_tokens(c.kv_format);
  const long long nmax = ((long long)c.capacity + tile - 1) / tile;
  if (c.batch > kBalMaxBatch || c.num_splits < 2 || c.sms < 1) return bp;
  const int splits_eff = split_count(c.capacity, c.num_splits, c.kv_format);
  if (splits_eff < 2) return bp;
  if ((long long)kHkv * c.batch * (nmax + kBalRowCost) > 0x7fffffffLL) return bp;
  const long long slots = (long long)mma_ctas_per_sm(c.kv_format, c.q_len) * c.sms;
  // one wave of pieces or less: nothing to balance, the plain grid starts sooner
  if ((long long)kHkv * c.batch * splits_eff <= slots) return bp;
  // One CTA per resident slot for a contiguous cache.  A paged 16-bit cache
  // runs 4 waves of smaller runs: its per-CTA rates vary more (pages
  // scattered over HBM), and the later waves let the hardware even them out
  // (bf16 8 x 131072 in shuffled 256-token pages, GB300: 586 us back to back
  // with one wave, 580 with four).  A paged 8-bit cache keeps one wave: at 3
  // CTAs per SM its issue-heavier CTAs pay more for the extra prologues and
  // pieces (64 x U[16k, 32k] in 256-token pages: int8 461 us with one wave,
  // 469 with four; e4m3 444 against 451).
  const bool waves4 = c.block_table != nullptr && !is_8bit(c.kv_format);
  bp.ctas = (int)((waves4 ? 4 : 1) * slots);
  bp.q_min = (int)((nmax + c.num_splits - 2) / (c.num_splits - 1));
  return bp;
}

// The one-piece grid merges on chip when its 2..8 splits that hold slots fit
// one portable thread-block cluster (distributed shared memory) and the grid
// is one wave at most: latency-bound launches, where the combine launch and
// the partials' round trip through HBM are a large share of the time.
// Measured on GB300: clusters of 9..16 (a non-portable size) were slower when
// warm (e4m3 1 x 8192 in a graph 10.3 -> 12.2 us, a 4-token window at
// 1 x 4096 9.6 -> 13.7), and so were multi-wave grids of clusters (int8
// 64 x U[16k, 32k] with a 2-token window, 8 splits, 4096 CTAs: 530 -> 760 us).
// The clusters must also all be resident at once (the device's occupancy
// table): a cluster's CTAs share one GPC, and near full occupancy clusters
// of some sizes pack into fewer than the slots allow, leaving the rest for a
// second wave.  Measured on GB300: e4m3 8 x 4096 (7 splits, 448 CTAs in
// clusters of 7, 456 slots) took 24.8 us per cold call, against 18.4 with 6
// splits.  Such a grid runs as the plain grid with the combine kernel.
// Returns the cluster size, or 0 for the combine kernel.
int cluster_fit(const Call& c, int s) {
  // the current device's table, once it has been set up with this SM count
  // (0: unknown, e.g. host-only planning without a device)
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();  // (no device here: clear the error)
    return 0;
  }
  const DeviceState& st = g_devices[dev];
  if (st.state.load(std::memory_order_acquire) != 1 || st.sm_count != c.sms) return 0;
  const auto& row = st.cluster_fit[c.kv_format];
  const int nq = c.q_len - 1;
  if (!is_8bit(c.kv_format)) return row[c.kv_format == kKvF16 ? kQF16 : kQBF16][nq][s];
  // an 8-bit cache with either q format when the call does not say which
  if (c.q_dtype == GQA_F16 || c.q_dtype == GQA_BF16) return row[c.q_dtype][nq][s];
  return std::min(row[kQF16][nq][s], row[kQBF16][nq][s]);
}

int cluster_splits(const Call& c) {
  if (bal_plan(c).ctas > 0 || c.sms < 1) return 0;
  const int s = split_count(c.capacity, c.num_splits, c.kv_format);
  if (s < 2 || s > kClusterMaxSplits) return 0;
  const long long slots = (long long)mma_ctas_per_sm(c.kv_format, c.q_len) * c.sms;
  if ((long long)kHkv * c.batch * s > slots) return 0;
  const int fit = cluster_fit(c, s);
  return fit > 0 && (long long)kHkv * c.batch > fit ? 0 : s;
}

gqa_status_t run_split(const Call& c) {
  const Layout lay = layout_of(c.workspace, c.batch * c.q_len, c.num_splits);
  SplitParams sp;
  sp.q = c.q;
  sp.kv = c.kv;
  sp.lens = c.lens;
  sp.out = c.out;
  sp.part_o = lay.part_o;
  sp.part_m = lay.part_m;
  sp.part_l = lay.part_l;
  sp.flags = lay.flags;
  sp.batch = c.batch;
  sp.capacity = c.capacity;
  sp.num_splits = c.num_splits;
  sp.chunk = split_chunk(c.capacity, c.num_splits, c.kv_format);
  sp.splits_eff = split_count(c.capacity, c.num_splits, c.kv_format);
  // log2(e) / sqrt(128): the softmax runs in the exp2 domain
  sp.scale_log2 = (float)((double)c.q_scale * (double)c.k_scale * 1.4426950408889634 / std::sqrt(128.0));
  sp.v_scale = c.v_scale;
  sp.wait_budget_ns = c.wait_budget_ns;
  sp.skip_tile = c.skip_tile;
  sp.kv_scales = c.kv_scales;
  sp.block_table = c.block_table;
  sp.page_log2 = c.page_log2;
  sp.max_pages = c.max_pages;
  sp.num_pages = c.num_pages;
  const BalPlan bp = bal_plan(c);
  sp.bal_q_min = bp.q_min;
  const size_t page_rows = c.block_table ? ((size_t)1 << c.page_log2) : (size_t)c.capacity;
  const size_t units = c.block_table ? (size_t)c.num_pages : (size_t)c.batch;
  sp.kv_bytes = units * 2 * kHkv * page_rows * kD * kv_elem_bytes(c.kv_format);
  sp.scales_bytes = c.kv_format == kKvI8 ? units * 2 * kHkv * page_rows * 2 : 0;
  if (kChecked) {
    sp.kv_bytes -= std::min<size_t>(sp.kv_bytes, g_cut_kv_bytes.load());
    sp.scales_bytes -= std::min<size_t>(sp.scales_bytes, g_cut_scales_bytes.load());
  }
  cudaError_t e;
  const int ql = c.q_len, nb = bp.ctas, cl = cluster_splits(c);
  if (c.kv_format == kKvF16) e = launch_split_t<kKvF16, kQF16>(sp, ql, nb, cl, c.stream);
  else if (c.kv_format == kKvBF16) e = launch_split_t<kKvBF16, kQBF16>(sp, ql, nb, cl, c.stream);
  else if (c.kv_format == kKvE4M3)
    e = c.q_dtype == GQA_BF16 ? launch_split_t<kKvE4M3, kQBF16>(sp, ql, nb, cl, c.stream)
                              : launch_split_t<kKvE4M3, kQF16>(sp, ql, nb, cl, c.stream);
  else
    e = c.q_dtype == GQA_BF16 ? launch_split_t<kKvI8, kQBF16>(sp, ql, nb, cl, c.stream)
                              : launch_split_t<kKvI8, kQF16>(sp, ql, nb, cl, c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "split kernel launch");
  return GQA_OK;
}

gqa_status_t run_combine(const Call& c) {
  const int splits_eff = split_count(c.capacity, c.num_splits, c.kv_format);
  if (splits_eff == 1 || cluster_splits(c) > 0) return GQA_OK;  // merged by stage 1
  const Layout lay = layout_of(c.workspace, c.batch * c.q_len, c.num_splits);
  CombineParams cp;
  cp.lens = c.lens;
  cp.out = c.out;
  cp.part_o = lay.part_o;
  cp.part_m = lay.part_m;
  cp.part_l = lay.part_l;
  cp.capacity = c.capacity;
  cp.num_splits = c.num_splits;
  cp.chunk = split_chunk(c.capacity, c.num_splits, c.kv_format);
  cp.q_len = c.q_len;
  cp.v_scale = c.v_scale;
  const BalPlan bp = bal_plan(c);
  cp.bal_ctas = bp.ctas;
  cp.bal_q_min = bp.q_min;
  cp.tile = tile_tokens(c.kv_format);
  cp.batch = c.batch;
  cp.flags = lay.flags;
  // Warps per query head: enough that each merges at most about 8 pieces of
  // its row in one round of loads (up to 4).  Pieces per row: the splits
  // that hold slots, or under the balanced schedule about CTAs / rows + 2 (a
  // row meets that many runs, plus the partial ones at its ends).
  const long long expected =
      bp.ctas > 0 ? std::min<long long>(c.num_splits, bp.ctas / (kHkv * (long long)c.batch) + 2) : splits_eff;
  int W = 1;
  while (W < kCombineMaxWarpsPerHead && expected > 8LL * W) W *= 2;
  cp.warps_per_head = W;
  cudaError_t e = c.q_dtype == GQA_F16 ? launch_combine_t<kQF16>(cp, c.batch * c.q_len, c.stream)
                                       : launch_combine_t<kQBF16>(cp, c.batch * c.q_len, c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
  return GQA_OK;
}

// Resolve num_splits = 0 (auto) and validate; then the device check.
gqa_status_t prepare_call(Call& c, bool q_scale_positive, bool need_q) {
  int sms = 0;
  if (c.num_splits == 0) {
    // validate everything that does not depend on the split count first
    Call probe = c;
    probe.num_splits = 1;
    probe.workspace_bytes = (size_t)-1;
    gqa_status_t st = validate(probe, q_scale_positive, need_q);
    if (st != GQA_OK) return st;
    st = current_device_ready(&sms);
    if (st != GQA_OK) return st;
    c.num_splits = plan_splits(c.batch, c.capacity, c.kv_format, sms);
  }
  gqa_status_t st = validate(c, q_scale_positive, need_q);
  if (st != GQA_OK) return st;
  st = current_device_ready(&sms);
  c.sms = sms;
  return st;
}

// The append step on a contiguous cache (block_table = nullptr; `units` =
// batch, `unit_rows` = capacity) or a paged one (units = num_pages, unit_rows
// = page size, capacity = max_pages * page size).
gqa_status_t append_kv(const void* q_proj, const void* k_proj, const void* v_proj, const void* q_norm_w,
                       const void* k_norm_w, gqa_dtype_t dtype, const int32_t* positions, const int32_t* slots,
                       int batch, void* q_out, void* kv, gqa_kv_format_t kv_format, uint16_t* kv_scales_bf16,
                       int capacity, const int32_t* block_table, int max_pages, int num_pages, int page_log2,
                       size_t units, size_t unit_rows, float eps, float rope_theta, float k_scale, float v_scale,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!q_proj || !k_proj || !v_proj || !q_norm_w || !k_norm_w || !positions || !slots || !q_out || !kv)
    return fail(GQA_ERR_INVALID_ARGUMENT, "null pointer argument");
  gqa_status_t st = validate_shape(batch, capacity);
  if (st != GQA_OK) return st;
  if (dtype != GQA_F16 && dtype != GQA_BF16) return fail(GQA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dtype);
  const int fmt = (int)kv_format;
  if (fmt != kKvF16 && fmt != kKvBF16 && fmt != kKvE4M3 && fmt != kKvI8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", fmt);
  if (!is_8bit(fmt) && fmt != (int)dtype)
    return fail(GQA_ERR_INVALID_ARGUMENT, "fp16/bf16 KV must have the dtype of the projections");
  if (fmt == kKvI8 && !kv_scales_bf16) return fail(GQA_ERR_INVALID_ARGUMENT, "an int8 cache needs kv_scales_bf16");
  if (!std::isfinite(eps) || eps < 0.f) return fail(GQA_ERR_INVALID_ARGUMENT, "eps must be finite and >= 0");
  if (!std::isfinite(rope_theta) || rope_theta <= 0.f)
    return fail(GQA_ERR_INVALID_ARGUMENT, "rope_theta must be finite and > 0");
  if (!std::isfinite(k_scale) || k_scale <= 0.f || !std::isfinite(v_scale) || v_scale <= 0.f)
    return fail(GQA_ERR_INVALID_ARGUMENT, "k_scale and v_scale must be finite and > 0");
  if (workspace && workspace_bytes < GQA_WORKSPACE_HEADER_BYTES)
    return fail(GQA_ERR_WORKSPACE_TOO_SMALL, "workspace smaller than its %d-byte header", GQA_WORKSPACE_HEADER_BYTES);
  const void* h16[] = {q_proj, k_proj, v_proj, q_norm_w, k_norm_w, q_out};
  for (const void* ptr : h16)
    if (!aligned(ptr, 2)) return fail(GQA_ERR_INVALID_ARGUMENT, "16-bit arrays must be 2-byte aligned");
  if (!aligned(positions, 4) || !aligned(slots, 4) || (workspace && !aligned(workspace, 4)) ||
      (!is_8bit(fmt) && !aligned(kv, 2)) || (kv_scales_bf16 && !aligned(kv_scales_bf16, 2)))
    return fail(GQA_ERR_INVALID_ARGUMENT, "misaligned argument");
  const size_t qb = (size_t)batch * kHq * kD * 2, kvb_in = (size_t)batch * kHkv * kD * 2;
  const size_t cache = units * 2 * kHkv * unit_rows * kD * kv_elem_bytes(fmt);
  const void* ins[] = {q_proj, k_proj, v_proj};
  const size_t in_bytes[] = {qb, kvb_in, kvb_in};
  for (int i = 0; i < 3; ++i)
    if (overlap(q_out, qb, ins[i], in_bytes[i]) || overlap(kv, cache, ins[i], in_bytes[i]))
      return fail(GQA_ERR_ALIASING, "q_out or kv overlaps an input projection");
  if (overlap(q_out, qb, kv, cache)) return fail(GQA_ERR_ALIASING, "q_out overlaps kv");
  int dev_sms = 0;
  st = current_device_ready(&dev_sms);
  if (st != GQA_OK) return st;
  AppendParams ap;
  ap.q_proj = q_proj;
  ap.k_proj = k_proj;
  ap.v_proj = v_proj;
  ap.q_norm_w = q_norm_w;
  ap.k_norm_w = k_norm_w;
  ap.positions = positions;
  ap.slots = slots;
  ap.q_out = q_out;
  ap.kv = kv;
  ap.kv_scales = kv_scales_bf16;
  ap.flags = static_cast<uint32_t*>(workspace);
  ap.batch = batch;
  ap.capacity = capacity;
  ap.block_table = block_table;
  ap.max_pages = max_pages;
  ap.num_pages = num_pages;
  ap.page_log2 = page_log2;
  ap.eps = eps;
  ap.k_inv_scale = 1.f / k_scale;
  ap.v_inv_scale = 1.f / v_scale;
  for (int i = 0; i < kD / 2; ++i) ap.inv_freq[i] = std::pow((double)rope_theta, -(double)i / (kD / 2));
  ap.kv_rows = units * 2 * kHkv * unit_rows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch, 1, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  // programmatic dependent launch, as the split kernel: the kernel waits for
  // the previous grid before its first read
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  const bool bf = dtype == GQA_BF16;
  if (fmt == kKvF16) e = cudaLaunchKernelEx(&cfg, append_kv_kernel<kKvF16, kQF16>, ap);
  else if (fmt == kKvBF16) e = cudaLaunchKernelEx(&cfg, append_kv_kernel<kKvBF16, kQBF16>, ap);
  else if (fmt == kKvE4M3)
    e = bf ? cudaLaunchKernelEx(&cfg, append_kv_kernel<kKvE4M3, kQBF16>, ap)
           : cudaLaunchKernelEx(&cfg, append_kv_kernel<kKvE4M3, kQF16>, ap);
  else
    e = bf ? cudaLaunchKernelEx(&cfg, append_kv_kernel<kKvI8, kQBF16>, ap)
           : cudaLaunchKernelEx(&cfg, append_kv_kernel<kKvI8, kQF16>, ap);
  if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
  return GQA_OK;
}

}  // namespace

extern "C" {

const char* gqa_status_string(gqa_status_t status) {
  switch (status) {
    case GQA_OK: return "GQA_OK";
    case GQA_ERR_INVALID_ARGUMENT: return "GQA_ERR_INVALID_ARGUMENT";
    case GQA_ERR_UNSUPPORTED_DEVICE: return "GQA_ERR_UNSUPPORTED_DEVICE";
    case GQA_ERR_WORKSPACE_TOO_SMALL: return "GQA_ERR_WORKSPACE_TOO_SMALL";
    case GQA_ERR_ALIASING: return "GQA_ERR_ALIASING";
    case GQA_ERR_CUDA: return "GQA_ERR_CUDA";
  }
  return "GQA_ERR_UNKNOWN";
}

const char* gqa_last_error(void) { return g_last_error.c_str(); }

size_t gqa_decode_workspace_size(int batch, int capacity, int num_splits) {
  if (batch < 1 || capacity < 1 || num_splits < 1 || num_splits > GQA_MAX_SPLITS) return 0;
  return workspace_bytes_for(batch, num_splits);
}

gqa_status_t gqa_decode_plan(int batch, int capacity, gqa_kv_format_t kv_format, int device,
                             int* num_splits_out) {
  if (!num_splits_out) return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits_out is null");
  gqa_status_t st = validate_shape(batch, capacity);
  if (st != GQA_OK) return st;
  if (kv_format != GQA_KV_F16 && kv_format != GQA_KV_BF16 && kv_format != GQA_KV_E4M3 &&
      kv_format != GQA_KV_I8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", (int)kv_format);
  int sms = 0;
  st = device_ready(device, &sms);
  if (st != GQA_OK) return st;
  *num_splits_out = plan_splits(batch, capacity, kv_format, sms);
  return GQA_OK;
}

gqa_status_t gqa_decode_plan_for(int batch, int capacity, gqa_kv_format_t kv_format, int sm_count,
                                 int* num_splits_out) {
  if (!num_splits_out) return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits_out is null");
  gqa_status_t st = validate_shape(batch, capacity);
  if (st != GQA_OK) return st;
  if (kv_format != GQA_KV_F16 && kv_format != GQA_KV_BF16 && kv_format != GQA_KV_E4M3 &&
      kv_format != GQA_KV_I8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", (int)kv_format);
  if (sm_count < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "sm_count %d < 1", sm_count);
  *num_splits_out = plan_splits(batch, capacity, kv_format, sm_count);
  return GQA_OK;
}

gqa_status_t gqa_decode_split_geometry(int capacity, int num_splits, gqa_kv_format_t kv_format,
                                       int* chunk_tokens_out, int* splits_effective_out) {
  if (!chunk_tokens_out || !splits_effective_out) return fail(GQA_ERR_INVALID_ARGUMENT, "null output pointer");
  gqa_status_t st = validate_shape(1, capacity);
  if (st != GQA_OK) return st;
  if (kv_format != GQA_KV_F16 && kv_format != GQA_KV_BF16 && kv_format != GQA_KV_E4M3 &&
      kv_format != GQA_KV_I8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", (int)kv_format);
  if (num_splits < 1 || num_splits > GQA_MAX_SPLITS)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits %d outside [1, %d]", num_splits, GQA_MAX_SPLITS);
  *chunk_tokens_out = split_chunk(capacity, num_splits, (int)kv_format);
  *splits_effective_out = split_count(capacity, num_splits, (int)kv_format);
  return GQA_OK;
}

gqa_status_t gqa_decode_launch_count_for(int batch, int capacity, gqa_kv_format_t kv_format, int q_len,
                                        int num_splits, int sm_count, int* launches_out) {
  if (!launches_out) return fail(GQA_ERR_INVALID_ARGUMENT, "launches_out is null");
  gqa_status_t st = validate_shape(batch, capacity);
  if (st != GQA_OK) return st;
  if (kv_format != GQA_KV_F16 && kv_format != GQA_KV_BF16 && kv_format != GQA_KV_E4M3 &&
      kv_format != GQA_KV_I8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", (int)kv_format);
  if (q_len < 1 || q_len > kMaxQLen) return fail(GQA_ERR_INVALID_ARGUMENT, "q_len %d outside [1, %d]", q_len, kMaxQLen);
  if (num_splits < 1 || num_splits > GQA_MAX_SPLITS)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits %d outside [1, %d]", num_splits, GQA_MAX_SPLITS);
  if (sm_count < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "sm_count %d < 1", sm_count);
  // the same rules run_split / run_combine apply to a launch of these sizes
  Call c{};
  c.kv_format = (int)kv_format;
  c.q_dtype = -1;  // (either q format)
  c.batch = batch;
  c.capacity = capacity;
  c.num_splits = num_splits;
  c.q_len = q_len;
  c.sms = sm_count;
  const bool merged = split_count(capacity, num_splits, (int)kv_format) == 1 || cluster_splits(c) > 0;
  *launches_out = merged ? 1 : 2;
  return GQA_OK;
}

gqa_status_t gqa_decode_prepared(const void* q, const void* kv, const int32_t* lens, void* out, int batch,
                                 int capacity, gqa_dtype_t dtype, float q_scale, int num_splits,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  Call c{q, (int)dtype, kv, (int)dtype, lens, out, batch, capacity, q_scale, 1.f, 1.f, num_splits,
         workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  gqa_status_t st = prepare_call(c, /*q_scale_positive=*/true, true);
  if (st != GQA_OK) return st;
  st = run_split(c);
  if (st != GQA_OK) return st;
  return run_combine(c);
}

gqa_status_t gqa_decode_fp8kv(const void* q_bf16, const uint8_t* kv_e4m3, const int32_t* lens, void* out_bf16,
                              int batch, int capacity, float q_scale, float k_scale, float v_scale,
                              int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  Call c{q_bf16, GQA_BF16, kv_e4m3, kKvE4M3, lens, out_bf16, batch, capacity, q_scale, k_scale, v_scale,
         num_splits, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  gqa_status_t st = prepare_call(c, false, true);
  if (st != GQA_OK) return st;
  st = run_split(c);
  if (st != GQA_OK) return st;
  return run_combine(c);
}

gqa_status_t gqa_decode_int8kv(const void* q, const int8_t* kv_i8, const uint16_t* kv_scales_bf16,
                               const int32_t* lens, void* out, int batch, int capacity, gqa_dtype_t dtype,
                               float q_scale, int num_splits, void* workspace, size_t workspace_bytes,
                               void* stream) {
  Call c{q, (int)dtype, kv_i8, kKvI8, lens, out, batch, capacity, q_scale, 1.f, 1.f, num_splits, workspace,
         workspace_bytes, static_cast<cudaStream_t>(stream)};
  c.kv_scales = kv_scales_bf16;
  gqa_status_t st = prepare_call(c, false, true);
  if (st != GQA_OK) return st;
  st = run_split(c);
  if (st != GQA_OK) return st;
  return run_combine(c);
}

gqa_status_t gqa_decode_paged(const void* q, gqa_dtype_t q_dtype, const void* kv_pages, gqa_kv_format_t kv_format,
                              const uint16_t* kv_scales_pages, const int32_t* block_table, int max_pages_per_seq,
                              int num_pages, int page_size, const int32_t* lens, void* out, int batch, int q_len,
                              float q_scale, float k_scale, float v_scale, int num_splits, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!block_table) return fail(GQA_ERR_INVALID_ARGUMENT, "block_table is null");
  if (page_size < 16 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
    return fail(GQA_ERR_INVALID_ARGUMENT, "page_size %d is not a power of two in [16, 65536]", page_size);
  if (num_pages < 1 || max_pages_per_seq < 1)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_pages and max_pages_per_seq must be >= 1");
  if (q_len < 1 || q_len > kMaxQLen)
    return fail(GQA_ERR_INVALID_ARGUMENT, "q_len %d outside [1, %d]", q_len, kMaxQLen);
  const long long cap = (long long)max_pages_per_seq * page_size;
  if (cap > (1LL << 30)) return fail(GQA_ERR_INVALID_ARGUMENT, "max_pages_per_seq * page_size exceeds 2^30");
  if (!aligned(block_table, 4)) return fail(GQA_ERR_INVALID_ARGUMENT, "block_table must be 4-byte aligned");
  if (kv_format == GQA_KV_I8) {
    if (!kv_scales_pages) return fail(GQA_ERR_INVALID_ARGUMENT, "an int8 cache needs its row scales");
    if (!aligned(kv_scales_pages, 16))
      return fail(GQA_ERR_INVALID_ARGUMENT, "the int8 scale pool must be 16-byte aligned");
  }
  Call c{q, (int)q_dtype, kv_pages, (int)kv_format, lens, out, batch, (int)cap, q_scale, k_scale, v_scale,
         num_splits, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  c.block_table = block_table;
  c.max_pages = max_pages_per_seq;
  c.num_pages = num_pages;
  c.q_len = q_len;
  if (kv_format == GQA_KV_I8) c.kv_scales = kv_scales_pages;
  int lg = 0;
  while ((1 << lg) < page_size) ++lg;
  c.page_log2 = lg;
  gqa_status_t st = prepare_call(c, false, true);
  if (st != GQA_OK) return st;
  st = run_split(c);
  if (st != GQA_OK) return st;
  return run_combine(c);
}

gqa_status_t gqa_decode_verify(const void* q, gqa_dtype_t q_dtype, const void* kv, gqa_kv_format_t kv_format,
                               const uint16_t* kv_scales_bf16, const int32_t* lens, void* out, int batch,
                               int capacity, int q_len, float q_scale, float k_scale, float v_scale,
                               int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (q_len < 1 || q_len > kMaxQLen)
    return fail(GQA_ERR_INVALID_ARGUMENT, "q_len %d outside [1, %d]", q_len, kMaxQLen);
  Call c{q, (int)q_dtype, kv, (int)kv_format, lens, out, batch, capacity, q_scale, k_scale, v_scale,
         num_splits, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  c.q_len = q_len;
  c.kv_scales = kv_scales_bf16;
  gqa_status_t st = prepare_call(c, false, true);
  if (st != GQA_OK) return st;
  st = run_split(c);
  if (st != GQA_OK) return st;
  return run_combine(c);
}


gqa_status_t gqa_append_kv(const void* q_proj, const void* k_proj, const void* v_proj, const void* q_norm_w,
                           const void* k_norm_w, gqa_dtype_t dtype, const int32_t* positions, const int32_t* slots,
                           int batch, void* q_out, void* kv, gqa_kv_format_t kv_format, uint16_t* kv_scales_bf16,
                           int capacity, float eps, float rope_theta, float k_scale, float v_scale, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (capacity < 1) return fail(GQA_ERR_INVALID_ARGUMENT, "capacity %d < 1", capacity);
  return append_kv(q_proj, k_proj, v_proj, q_norm_w, k_norm_w, dtype, positions, slots, batch, q_out, kv, kv_format,
                   kv_scales_bf16, capacity, nullptr, 0, 0, 0, batch > 0 ? (size_t)batch : 0, (size_t)capacity,
                   eps, rope_theta, k_scale, v_scale, workspace, workspace_bytes, stream);
}

gqa_status_t gqa_append_kv_paged(const void* q_proj, const void* k_proj, const void* v_proj,
                                 const void* q_norm_w, const void* k_norm_w, gqa_dtype_t dtype,
                                 const int32_t* positions, const int32_t* slots, int batch, void* q_out,
                                 void* kv_pages, gqa_kv_format_t kv_format, uint16_t* kv_scales_pages,
                                 const int32_t* block_table, int max_pages_per_seq, int num_pages, int page_size,
                                 float eps, float rope_theta, float k_scale, float v_scale, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!block_table) return fail(GQA_ERR_INVALID_ARGUMENT, "block_table is null");
  if (page_size < 16 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
    return fail(GQA_ERR_INVALID_ARGUMENT, "page_size %d is not a power of two in [16, 65536]", page_size);
  if (num_pages < 1 || max_pages_per_seq < 1)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_pages and max_pages_per_seq must be >= 1");
  const long long cap = (long long)max_pages_per_seq * page_size;
  if (cap > (1LL << 30)) return fail(GQA_ERR_INVALID_ARGUMENT, "max_pages_per_seq * page_size exceeds 2^30");
  if (!aligned(block_table, 4)) return fail(GQA_ERR_INVALID_ARGUMENT, "block_table must be 4-byte aligned");
  int lg = 0;
  while ((1 << lg) < page_size) ++lg;
  return append_kv(q_proj, k_proj, v_proj, q_norm_w, k_norm_w, dtype, positions, slots, batch, q_out, kv_pages,
                   kv_format, kv_scales_pages, (int)cap, block_table, max_pages_per_seq, num_pages, lg,
                   (size_t)num_pages, (size_t)page_size, eps, rope_theta, k_scale, v_scale, workspace,
                   workspace_bytes, stream);
}

gqa_status_t gqa_decode_split_stage(const void* q, gqa_dtype_t q_dtype, const void* kv,
                                    gqa_kv_format_t kv_format, const int32_t* lens, void* out, int batch,
                                    int capacity, float q_scale, float k_scale, float v_scale, int num_splits,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (kv_format == GQA_KV_I8)
    return fail(GQA_ERR_INVALID_ARGUMENT, "an int8 cache needs its scales: use gqa_decode_int8kv");
  Call c{q, (int)q_dtype, kv, (int)kv_format, lens, out, batch, capacity, q_scale, k_scale, v_scale,
         num_splits, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  gqa_status_t st = prepare_call(c, false, true);
  if (st != GQA_OK) return st;
  return run_split(c);
}

gqa_status_t gqa_decode_debug_skip_tile(const void* q, gqa_dtype_t q_dtype, const void* kv,
                                        gqa_kv_format_t kv_format, const int32_t* lens, void* out, int batch,
                                        int capacity, float q_scale, float k_scale, float v_scale,
                                        int num_splits, void* workspace, size_t workspace_bytes,
                                        int skip_tile, uint64_t wait_budget_ns, void* stream) {
  Call c{q, (int)q_dtype, kv, (int)kv_format, lens, out, batch, capacity, q_scale, k_scale, v_scale,
         num_splits, workspace, workspace_bytes, static_cast<cudaStream_t>(stream)};
  if (skip_tile < 0) return fail(GQA_ERR_INVALID_ARGUMENT, "skip_tile must be >= 0");
  if (wait_budget_ns < 1000000ull || wait_budget_ns > kWaitBudgetNs)
    return fail(GQA_ERR_INVALID_ARGUMENT, "wait_budget_ns must be in [1 ms, 4 s]");
  c.skip_tile = skip_tile;
  c.wait_budget_ns = wait_budget_ns;
  gqa_status_t st = prepare_call(c, false, true);
  if (st != GQA_OK) return st;
  return run_split(c);
}

gqa_status_t gqa_decode_combine_stage(const int32_t* lens, void* out, gqa_dtype_t out_dtype,
                                      gqa_kv_format_t kv_format, int batch, int capacity, float v_scale,
                                      int num_splits, const void* workspace, size_t workspace_bytes,
                                      void* stream) {
  // kv and q are not read by stage 2; stand in a dummy aligned address for
  // the checks (a null kv would be rejected) and skip the q checks.
  static const uint4 dummy = {0, 0, 0, 0};
  const int fmt = (int)kv_format;
  Call c{nullptr, (int)out_dtype, &dummy, is_8bit(fmt) ? fmt : (int)out_dtype, lens, out, batch,
         capacity, 1.f, 1.f, v_scale, num_splits, const_cast<void*>(workspace), workspace_bytes,
         static_cast<cudaStream_t>(stream)};
  if (fmt != kKvE4M3 && fmt != kKvI8 && fmt != kKvF16 && fmt != kKvBF16)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown KV format %d", fmt);
  c.kv_format = fmt;
  if (!is_8bit(fmt) && fmt != (int)out_dtype)
    return fail(GQA_ERR_INVALID_ARGUMENT, "fp16/bf16 KV must have the dtype of out");
  // the dummy kv range (batch*capacity*...) would spuriously overlap out; check
  // only what stage 2 touches
  if (!lens || !out || !workspace) return fail(GQA_ERR_INVALID_ARGUMENT, "null pointer argument");
  gqa_status_t st = validate_shape(batch, capacity);
  if (st != GQA_OK) return st;
  if (out_dtype != GQA_F16 && out_dtype != GQA_BF16)
    return fail(GQA_ERR_INVALID_ARGUMENT, "unknown out dtype %d", (int)out_dtype);
  if (!std::isfinite(v_scale) || v_scale <= 0.f)
    return fail(GQA_ERR_INVALID_ARGUMENT, "v_scale must be finite and > 0");
  if (num_splits < 1 || num_splits > GQA_MAX_SPLITS)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits %d outside [1, %d]", num_splits, GQA_MAX_SPLITS);
  if (!aligned(out, 16) || !aligned(workspace, 16) || !aligned(lens, 4))
    return fail(GQA_ERR_INVALID_ARGUMENT, "out, workspace must be 16-byte aligned, lens 4-byte");
  const size_t need = workspace_bytes_for(batch, num_splits);
  if (workspace_bytes < need)
    return fail(GQA_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (overlap(out, (size_t)batch * kHq * kD * 2, workspace, need))
    return fail(GQA_ERR_ALIASING, "out overlaps the workspace");
  int sms = 0;
  st = current_device_ready(&sms);
  if (st != GQA_OK) return st;
  c.sms = sms;
  return run_combine(c);
}

gqa_status_t gqa_decode(const void* q, const void* kv, const int32_t* lens, void* out, int batch, int capacity,
                        gqa_dtype_t dtype, float q_scale, void* stream) {
  static const uint4 dummy_ws = {0, 0, 0, 0};
  Call c{q, (int)dtype, kv, (int)dtype, lens, out, batch, capacity, q_scale, 1.f, 1.f, 0,
         const_cast<uint4*>(&dummy_ws), (size_t)-1, static_cast<cudaStream_t>(stream)};
  // validate with a stand-in workspace, then allocate the real one
  Call probe = c;
  probe.num_splits = 1;
  gqa_status_t st = validate(probe, false, true);
  if (st != GQA_OK) return st;
  int sms = 0;
  st = current_device_ready(&sms);
  if (st != GQA_OK) return st;
  c.num_splits = plan_splits(batch, capacity, (int)dtype, sms);
  c.sms = sms;
  const size_t bytes = workspace_bytes_for(batch, c.num_splits);
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, bytes, c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
  c.workspace = ws;
  c.workspace_bytes = bytes;
  e = cudaMemsetAsync(ws, 0, GQA_WORKSPACE_HEADER_BYTES, c.stream);
  if (e != cudaSuccess) st = cuda_fail(e, "cudaMemsetAsync(workspace header)");
  if (st == GQA_OK) st = validate(c, false, true);
  if (st == GQA_OK) st = run_split(c);
  if (st == GQA_OK) st = run_combine(c);
  e = cudaFreeAsync(ws, c.stream);
  if (st == GQA_OK && e != cudaSuccess) st = cuda_fail(e, "cudaFreeAsync(workspace)");
  return st;
}

gqa_status_t gqa_decode_noalloc(const void* q, const void* kv, const int32_t* lens, void* out, int batch,
                                int capacity, gqa_dtype_t dtype, float q_scale, int num_splits, void* stream) {
  static const uint4 dummy_ws = {0, 0, 0, 0};
  Call c{q, (int)dtype, kv, (int)dtype, lens, out, batch, capacity, q_scale, 1.f, 1.f, 1,
         const_cast<uint4*>(&dummy_ws), (size_t)-1, static_cast<cudaStream_t>(stream)};
  gqa_status_t st = validate(c, false, true);  // everything but the split count and scratch
  if (st != GQA_OK) return st;
  if (num_splits < 0 || num_splits > GQA_MAX_SPLITS)
    return fail(GQA_ERR_INVALID_ARGUMENT, "num_splits %d outside [0, %d]", num_splits, GQA_MAX_SPLITS);
  if (num_splits > 0 && workspace_bytes_for(batch, num_splits) > kStaticWorkspaceBytes)
    return fail(GQA_ERR_WORKSPACE_TOO_SMALL,
                "batch %d with %d splits needs %zu bytes of scratch; the static scratch holds %zu",
                batch, num_splits, workspace_bytes_for(batch, num_splits), kStaticWorkspaceBytes);
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  st = device_ready(dev, &sms);
  if (st != GQA_OK) return st;
  void* ws = nullptr;
  st = static_workspace(dev, c.stream, &ws);
  if (st != GQA_OK) return st;
  int S = num_splits;
  if (S == 0) {
    S = plan_splits(batch, capacity, (int)dtype, sms);
    while (S > 1 && workspace_bytes_for(batch, S) > kStaticWorkspaceBytes) --S;
  }
  c.num_splits = S;
  c.sms = sms;
  c.workspace = ws;
  c.workspace_bytes = kStaticWorkspaceBytes;
  st = validate(c, false, true);
  if (st != GQA_OK) return st;
  // the status word (zeroed at set-up) accumulates over calls until
  // gqa_decode_noalloc_get_status reads and clears it
  st = run_split(c);
  if (st != GQA_OK) return st;
  return run_combine(c);
}

gqa_status_t gqa_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < GQA_WORKSPACE_HEADER_BYTES)
    return fail(GQA_ERR_INVALID_ARGUMENT, "workspace must be non-null and hold the %d-byte header",
                GQA_WORKSPACE_HEADER_BYTES);
  cudaError_t e = cudaMemsetAsync(workspace, 0, GQA_WORKSPACE_HEADER_BYTES, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace header)");
  return GQA_OK;
}

gqa_status_t gqa_decode_get_status(void* workspace, size_t workspace_bytes, void* stream, uint32_t* flags) {
  if (!workspace || !flags || workspace_bytes < GQA_WORKSPACE_HEADER_BYTES)
    return fail(GQA_ERR_INVALID_ARGUMENT, "workspace and flags must be non-null; workspace >= header");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status word");
  *flags = host;
  return GQA_OK;
}

gqa_status_t gqa_decode_debug_cut_extents(uint64_t kv_cut_bytes, uint64_t scales_cut_bytes) {
  if (!kChecked && (kv_cut_bytes || scales_cut_bytes))
    return fail(GQA_ERR_INVALID_ARGUMENT, "extent cuts exist only in the range-checked build (GQA_CHECKED)");
  g_cut_kv_bytes = kv_cut_bytes;
  g_cut_scales_bytes = scales_cut_bytes;
  return GQA_OK;
}

gqa_status_t gqa_decode_noalloc_get_status(void* stream, uint32_t* flags) {
  if (!flags) return fail(GQA_ERR_INVALID_ARGUMENT, "flags must be non-null");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  gqa_status_t st = device_ready(dev, nullptr);
  if (st != GQA_OK) return st;
  void* ws = nullptr;
  st = static_workspace(dev, static_cast<cudaStream_t>(stream), &ws);
  if (st != GQA_OK) return st;
  return gqa_decode_get_status(ws, GQA_WORKSPACE_HEADER_BYTES, stream, flags);
}

}  // extern "C"
