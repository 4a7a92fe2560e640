// cq_internal.cuh -- internal definitions shared by the libcq translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "cq.h"

namespace cq {

// Derived problem sizes, computed once on the host per call.
struct Dims {
  int32_t W, M, S_eff, S_r, R_rep;  // R_rep: replicas per shared expert (S_r / S)
  int32_t Z, C, Q, BS, K, H, L, NS, G;  // G = S_r + M global expert slots
  int32_t mode, etn_type, mask_ndim;
  int32_t x_dtype;                // 0 bf16, 1 fp16
  int32_t y_dtype;                // fp8 codes of modes 3-5: 0 e4m3fn, 1 e5m2
  int32_t SC;                     // mx scale columns: Align2(Ceil(H, 32))
  int32_t G3;                     // mode-3 groups per row: Ceil(H, 128)
  int32_t CH, TC;                 // routing: each source's tokens in CH chunks of TC
  int64_t R_max;
};

// Workspace layout (byte offsets, each segment 256-byte aligned).
//   hdr       : uint32 status, uint32 done counter, int32 total rows, pad
//   counts_t  : int32 [G][W][CH]  rows per (global expert slot, source rank,
//                             chunk of the source's tokens)
//   local_off : int32 [G][W][CH]  first row of each (slot, source, chunk)
//                             block, counted from the start of its destination rank
//   eidx      : int32 [W*BS*NS] arrival ordinal of each slot within its
//                             (slot, source, chunk) block, or a CQ_INV code
//   rank_tot  : int32 [W]     rows received by each destination rank
//   rank_base : int32 [W+1]   first global row of each destination rank
//   row_src   : int2 [R_max]  (source token index r*BS+i, smooth-table row) of
//                             each dispatched row (per-expert smooth path only)
struct Workspace {
  uint32_t* status;
  uint32_t* done;
  int32_t* total;
  int32_t* counts_t;
  int32_t* local_off;
  int32_t* eidx;
  int32_t* rank_tot;
  int32_t* rank_base;
  int2* row_src;
};

constexpr size_t kHdrBytes = 256;
inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

inline size_t workspace_bytes(const Dims& d) {
  size_t b = kHdrBytes;
  b += align256(sizeof(int32_t) * (size_t)d.G * d.W * d.CH);
  b += align256(sizeof(int32_t) * (size_t)d.G * d.W * d.CH);
  b += align256(sizeof(int32_t) * (size_t)d.W * d.BS * d.NS);
  b += align256(sizeof(int32_t) * (size_t)d.W);
  b += align256(sizeof(int32_t) * (size_t)(d.W + 1));
  b += align256(sizeof(int2) * (size_t)d.R_max);
  return b;
}

inline Workspace carve(void* base, const Dims& d) {
  char* p = static_cast<char*>(base);
  Workspace w;
  w.status = reinterpret_cast<uint32_t*>(p);
  w.done = reinterpret_cast<uint32_t*>(p + 4);
  w.total = reinterpret_cast<int32_t*>(p + 8);
  p += kHdrBytes;
  w.counts_t = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (size_t)d.G * d.W * d.CH);
  w.local_off = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (size_t)d.G * d.W * d.CH);
  w.eidx = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (size_t)d.W * d.BS * d.NS);
  w.rank_tot = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (size_t)d.W);
  w.rank_base = reinterpret_cast<int32_t*>(p);
  p += align256(sizeof(int32_t) * (size_t)(d.W + 1));
  w.row_src = reinterpret_cast<int2*>(p);
  return w;
}

// assist_info layout: [R_max][4] rows, then inv [W*BS*NS], then rank_row_base [W+1].
inline int64_t assist_rows_off(const Dims&) { return 0; }
inline int64_t assist_inv_off(const Dims& d) { return 4 * d.R_max; }
inline int64_t assist_base_off(const Dims& d) { return 4 * d.R_max + (int64_t)d.W * d.BS * d.NS; }
inline int64_t assist_size(const Dims& d) { return assist_base_off(d) + d.W + 1; }

struct RouteArgs {
  Dims d;
  const int32_t* expert_ids;
  const uint8_t* mask;
  const int32_t* bs_per_rank;
  int32_t* ep_recv_count;
  int64_t* expert_token_nums;
  int32_t* rank_row_base;  // inside assist_info
  Workspace ws;
};

struct PermuteArgs {
  Dims d;
  const uint16_t* x;
  const int32_t* expert_ids;
  const uint8_t* mask;          // only to skip prefetching rows of inactive tokens
  const int32_t* bs_per_rank;   // idem
  const float* smooth;
  int32_t smooth_kind;          // 0 per-expert rows, 1 one row for all, 2 one scalar
  const float* expert_scales;
  void* expand_x;
  void* dynamic_scales;
  int32_t* assist_rows;  // [R_max][4]
  int32_t* inv;          // [W*BS*NS]
  float* expand_scales;
  int32_t scale_rows_bulk;  // modes 3-5: scale rows are 16-byte sized and aligned (bulk stores)
  Workspace ws;
};

struct CombineArgs {
  Dims d;
  const uint16_t* ffn;         // bf16 expert outputs [R_max, H] (bf16 combine, quantiser input)
  int8_t* ffn_q;               // int8 expert outputs [R_max, H] (int8 combine input, quantiser output)
  float* ffn_scales;           // their block scales [R_max, H/8]
  const int32_t* total_rows;   // rank_row_base[W] inside assist_info (quantiser)
  const int32_t* inv;
  const float* expert_scales;
  const uint16_t* ori_x;
  const float* alpha1;
  const float* alpha2;
  const uint16_t* const_v;
  void* y;
  int32_t out_f32;
  uint32_t* status;  // CQ_ST_* word of this call (a workspace's), or NULL: the device's own
};

// The two 16-bit token types. In a packed 32-bit word element 2t is the low
// half. Conversions to fp32 are exact; pack2 rounds to nearest even.
struct BF16 {
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
};
struct F16 {
  static __device__ __forceinline__ float lo(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
  }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
  }
  static __device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
  }
};

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream is still running. Every kernel launched
// this way executes griddep_wait() before it reads anything an earlier kernel
// wrote, which waits for that kernel to complete and its writes to be visible.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// Once per device and kernel: ask for the largest shared-memory carveout,
// and allow `smem` bytes of dynamic shared memory (raised when a later call
// needs more). Kernels chained with programmatic dependent launch share SMs
// while one ends and the next starts; an SM set up with a small carveout for
// one kernel cannot take the next kernel's CTAs that need a large one until
// it drains, which turns a one-wave grid into two.
constexpr int kMaxDevices = 64;
template <auto Kernel>
cudaError_t prepare_kernel(size_t smem) {
  static std::mutex mu;
  static size_t allowed[kMaxDevices];
  static bool carved[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!carved[dev]) {
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    carved[dev] = true;
  }
  if (smem > allowed[dev]) {
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    allowed[dev] = smem;
  }
  return cudaSuccess;
}

// Number of SMs of the current device (cached per device; 0 on error).
inline int sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Resident CTAs per SM of `Kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device. The last query of each
// device is cached (the launchers ask with the same sizes call after call).
template <auto Kernel>
cudaError_t occupancy_blocks(int threads, size_t smem, int* blocks) {
  struct Entry {
    int threads;
    size_t smem;
    int blocks;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  Entry& c = cache[dev];
  if (c.threads != threads || c.smem != smem || c.blocks <= 0) {
    int b = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, Kernel, threads, smem);
    if (e != cudaSuccess) return e;
    c = Entry{threads, smem, b};
  }
  *blocks = c.blocks;
  return cudaSuccess;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Every host-side check of cq_dispatch's arguments (both halves), with
// nothing enqueued: CQ_OK or the error code cq_dispatch would return.
int dispatch_check(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                   const float* smooth_scales, const uint8_t* x_active_mask, const void* expand_x,
                   const void* dynamic_scales, const int32_t* assist_info,
                   const int32_t* ep_recv_count, const int64_t* expert_token_nums,
                   const void* workspace, size_t workspace_bytes);

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s);
// The whole dispatch of a small batch in one kernel (cq_dispatch_small.cu):
// whether the problem qualifies, and the launch (cudaErrorNotSupported for a
// mode it does not cover).
bool dispatch_small_fits(const Dims& d, bool per_expert_smooth);
cudaError_t launch_dispatch_small(const PermuteArgs& a, int32_t* ep_recv_count,
                                  int64_t* expert_token_nums, int32_t* rank_row_base,
                                  cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);     // from bf16 rows
cudaError_t launch_combine_q8(const CombineArgs& a, cudaStream_t s);  // from int8 rows
cudaError_t launch_combine_quant(const CombineArgs& a, cudaStream_t s);
cudaError_t read_combine_status(uint32_t* status, cudaStream_t s);

}  // namespace cq
