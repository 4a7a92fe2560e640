// cq_noalloc.cu -- cq_dispatch_noalloc: cq_dispatch with a built-in scratch
// buffer, for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code running under an
// allocator that is frozen after start-up (a serving process that reserves
// all device memory once and must not call cudaMalloc on the request path,
// because cudaMalloc can synchronise the device and fragment the pool), a
// plugin that is handed only its input and output tensors by a host
// framework that owns every allocation, or an embedded deployment with a
// fixed, pre-planned memory map. This entry point lets them dispatch by
// using a scratch area compiled into the library instead.
//
// The scratch is one file-scope device array of CQ_NOALLOC_SCRATCH_BYTES. Every
// GPU that loads libcq holds it until the process exits. Host code only ever
// sees a stand-in symbol for it, so its device address is looked up with
// cudaGetSymbolAddress once per device (on the first call made while that
// device is current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "cq_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up once).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return CQ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CQ_OK;
}

}  // namespace

extern "C" int cq_dispatch_noalloc(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                                   const float* smooth_scales, const uint8_t* x_active_mask,
                                   const int32_t* bs_per_rank, const float* expert_scales,
                                   void* expand_x, void* dynamic_scales, int32_t* assist_info,
                                   int32_t* ep_recv_count, int64_t* expert_token_nums,
                                   float* expand_scales, void* stream) {
  const int rc = cq_check_config(cfg);
  if (rc != CQ_OK) return rc;
  const size_t need = cq_workspace_size(cfg);
  if (need == 0 || need > (size_t)CQ_NOALLOC_SCRATCH_BYTES) return CQ_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int arc = scratch_address(&scratch);
  if (arc != CQ_OK) return arc;
  // Every argument check of cq_dispatch runs before the header is cleared,
  // so an argument error returns with nothing enqueued.
  const int crc = cq::dispatch_check(cfg, x, expert_ids, smooth_scales, x_active_mask, expand_x,
                                     dynamic_scales, assist_info, ep_recv_count,
                                     expert_token_nums, scratch, CQ_NOALLOC_SCRATCH_BYTES);
  if (crc != CQ_OK) return crc;
  // The array keeps whatever the previous call left. Only the header (status
  // word and the routing kernel's completion counter) has to start at zero;
  // every other byte the kernels read is written earlier in the same call.
  if (cudaMemsetAsync(scratch, 0, cq::kHdrBytes, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return CQ_ERR_CUDA;
  return cq_dispatch(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                     expert_scales, expand_x, dynamic_scales, assist_info, ep_recv_count,
                     expert_token_nums, expand_scales, scratch, CQ_NOALLOC_SCRATCH_BYTES, stream);
}
