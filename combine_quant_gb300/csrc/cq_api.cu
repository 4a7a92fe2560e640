// cq_api.cu -- host entry points of libcq (see include/cq.h for the contract).
//
// Every argument rule is checked on the host before anything is enqueued.
// The ranges follow "CANN ops-transformer 算子解析：MoeDistributeDispatchV3 的
// EP 域 Token 分发与动态量化通信实现" (约束说明, 参数说明, 前置校验) and
// "low_latency_dispatch" (shape variables: local_expert_num * W <= 2048).
// Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
// top of include/cq.h.
#include <cuda_runtime.h>

#include <chrono>

#include "cq_async.cuh"
#include "cq_internal.cuh"

using cq::Dims;

namespace {

int validate(const cq_config* c) {
  if (!c) return CQ_ERR_ARG;
  const int32_t W = c->ep_world_size, M = c->moe_expert_num;
  const int32_t S = c->shared_expert_num, Sr = c->shared_expert_rank_num;
  if (W < 2 || W > 768) return CQ_ERR_ARG;
  if (c->hidden < 1024 || c->hidden > 8192) return CQ_ERR_ARG;
  if (c->max_bs < 1 || c->max_bs > 512) return CQ_ERR_ARG;
  if (M < 1 || M > 1024) return CQ_ERR_ARG;
  if (c->topk < 1 || c->topk > 16) return CQ_ERR_ARG;
  if (S < 0 || S > 4) return CQ_ERR_ARG;
  if (Sr < 0 || Sr >= W) return CQ_ERR_ARG;
  if (Sr == 0 && S > 1) return CQ_ERR_ARG;
  if (Sr > 0 && (S == 0 || Sr % S != 0 || W % Sr != 0)) return CQ_ERR_ARG;
  if (M % (W - Sr) != 0) return CQ_ERR_ARG;
  if ((int64_t)(M / (W - Sr)) * W > 2048) return CQ_ERR_ARG;
  if (c->zero_expert_num < 0 || c->copy_expert_num < 0 || c->const_expert_num < 0)
    return CQ_ERR_ARG;
  const int64_t all =
      (int64_t)M + c->zero_expert_num + c->copy_expert_num + c->const_expert_num;
  if (all >= 2147483647LL || c->topk > all) return CQ_ERR_ARG;
  if (c->global_bs != 0 && c->global_bs != c->max_bs * W) return CQ_ERR_ARG;
  if (c->expert_token_nums_type != 0 && c->expert_token_nums_type != 1) return CQ_ERR_ARG;
  if (c->mask_ndim < 0 || c->mask_ndim > 2) return CQ_ERR_ARG;
  if (c->quant_mode < 0 || c->quant_mode > 5) return CQ_ERR_ARG;
  if (c->x_dtype != 0 && c->x_dtype != 1) return CQ_ERR_ARG;
  if (c->smooth_kind < 0 || c->smooth_kind > 2) return CQ_ERR_ARG;
  if (c->y_dtype != 0 && c->y_dtype != 1) return CQ_ERR_ARG;
  if (c->y_dtype == 1 && c->quant_mode < 3) return CQ_ERR_ARG;  // e5m2 codes: modes 3-5
  // Vector paths: 16-element units (16-byte stores of int8 / e4m3 rows); mx
  // blocks of 32 never straddle two threads' units.
  if (c->hidden % 16 != 0) return CQ_ERR_UNSUPPORTED;
  if ((c->quant_mode == 4 || c->quant_mode == 5) && c->hidden % 32 != 0)
    return CQ_ERR_UNSUPPORTED;
  return CQ_OK;
}

Dims dims_of(const cq_config* c) {
  Dims d;
  d.W = c->ep_world_size;
  d.M = c->moe_expert_num;
  d.S_r = c->shared_expert_rank_num;
  d.S_eff = d.S_r > 0 ? c->shared_expert_num : 0;
  d.R_rep = d.S_r > 0 ? d.S_r / c->shared_expert_num : 1;
  d.Z = c->zero_expert_num;
  d.C = c->copy_expert_num;
  d.Q = c->const_expert_num;
  d.BS = c->max_bs;
  d.K = c->topk;
  d.H = c->hidden;
  d.L = d.M / (d.W - d.S_r);
  d.NS = d.K + d.S_eff;
  d.G = d.S_r + d.M;
  d.mode = c->quant_mode;
  d.etn_type = c->expert_token_nums_type;
  d.mask_ndim = c->mask_ndim;
  d.x_dtype = c->x_dtype;
  d.y_dtype = c->y_dtype;
  const int32_t blocks = (d.H + 31) / 32;
  d.SC = (blocks + 1) / 2 * 2;
  d.G3 = (d.H + 127) / 128;
  d.R_max = (int64_t)d.W * d.BS * d.NS;
  // Routing chunks: CH count CTAs per source, chunks of about
  // kRouteChunkTokens tokens (16 warps of 4 tokens), at most kRouteCtas
  // count CTAs in all, and at most 2048 (local expert, source, chunk) entries
  // per destination rank (L * W <= 2048 holds already). Measured best among
  // 32-512 tokens a chunk and 64-256 CTAs on the DSV3, skew, mxfp8, special
  // and perf256 workloads.
  constexpr int kRouteCtas = 128, kRouteChunkTokens = 64;
  int ch = d.BS / kRouteChunkTokens;
  if (ch > kRouteCtas / d.W) ch = kRouteCtas / d.W;
  if (ch > 2048 / (d.L * d.W)) ch = 2048 / (d.L * d.W);
  if (ch < 1) ch = 1;
  d.CH = ch;
  d.TC = (d.BS + ch - 1) / ch;
  return d;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_ws(const Dims& d, const void* ws, size_t bytes) {
  if (!ws || !aligned(ws, 256) || bytes < cq::workspace_bytes(d)) return CQ_ERR_WORKSPACE;
  return CQ_OK;
}

// Host-only checks of the route half's arguments (nothing is enqueued).
int check_route(const cq_config* cfg, const int32_t* expert_ids, const uint8_t* mask,
                const int32_t* assist_info, const int32_t* ep_recv_count,
                const int64_t* expert_token_nums, const void* workspace,
                size_t workspace_bytes) {
  int rc = validate(cfg);
  if (rc != CQ_OK) return rc;
  const Dims d = dims_of(cfg);
  if (!expert_ids || !assist_info || !ep_recv_count || !expert_token_nums) return CQ_ERR_ARG;
  if (d.mask_ndim != 0 && !mask) return CQ_ERR_ARG;
  return check_ws(d, workspace, workspace_bytes);
}

// Host-only checks of the permute half's arguments (nothing is enqueued).
int check_permute(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                  const float* smooth, const void* expand_x, const void* dynamic_scales,
                  const int32_t* assist_info, const void* workspace, size_t workspace_bytes) {
  int rc = validate(cfg);
  if (rc != CQ_OK) return rc;
  const Dims d = dims_of(cfg);
  if (!x || !expert_ids || !expand_x || !assist_info) return CQ_ERR_ARG;
  if (d.mode >= 2 && !dynamic_scales) return CQ_ERR_ARG;
  // [LLD] quant_mode 相关约束: mx modes take no scales; static quantisation needs them.
  if (smooth && (d.mode == 0 || d.mode == 4 || d.mode == 5)) return CQ_ERR_ARG;
  if (!smooth && d.mode == 1) return CQ_ERR_ARG;
  if (!aligned(x, 16) || !aligned(expand_x, 16) ||
      (smooth && cfg->smooth_kind != 2 && !aligned(smooth, 16)) || !aligned(assist_info, 16) ||
      (smooth && !aligned(smooth, 4)) ||
      ((d.mode == 2 || d.mode == 3) && !aligned(dynamic_scales, 4)))
    return CQ_ERR_ARG;
  return check_ws(d, workspace, workspace_bytes);
}

int route_impl(const cq_config* cfg, const int32_t* expert_ids, const uint8_t* mask,
               const int32_t* bs_per_rank, int32_t* assist_info, int32_t* ep_recv_count,
               int64_t* expert_token_nums, void* workspace, size_t workspace_bytes,
               void* stream) {
  const int rc = check_route(cfg, expert_ids, mask, assist_info, ep_recv_count,
                             expert_token_nums, workspace, workspace_bytes);
  if (rc != CQ_OK) return rc;
  const Dims d = dims_of(cfg);
  cq::RouteArgs a;
  a.d = d;
  a.expert_ids = expert_ids;
  a.mask = d.mask_ndim ? mask : nullptr;
  a.bs_per_rank = bs_per_rank;
  a.ep_recv_count = ep_recv_count;
  a.expert_token_nums = expert_token_nums;
  a.rank_row_base = assist_info + cq::assist_base_off(d);
  a.ws = cq::carve(workspace, d);
  return cq::launch_route(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CQ_OK
                                                                                 : CQ_ERR_CUDA;
}

// The permute half's argument block (arguments already checked).
cq::PermuteArgs permute_args(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                             const float* smooth, const uint8_t* mask, const int32_t* bs_per_rank,
                             const float* expert_scales, void* expand_x, void* dynamic_scales,
                             int32_t* assist_info, float* expand_scales, void* workspace) {
  const Dims d = dims_of(cfg);
  cq::PermuteArgs a;
  a.d = d;
  a.x = static_cast<const uint16_t*>(x);
  a.expert_ids = expert_ids;
  a.mask = d.mask_ndim ? mask : nullptr;
  a.bs_per_rank = bs_per_rank;
  a.smooth = smooth;
  a.smooth_kind = cfg->smooth_kind;
  a.expert_scales = expert_scales;
  a.expand_x = expand_x;
  a.dynamic_scales = dynamic_scales;
  a.assist_rows = assist_info + cq::assist_rows_off(d);
  a.inv = assist_info + cq::assist_inv_off(d);
  a.expand_scales = expand_scales;
  const int scale_row_bytes = d.mode == 3 ? 4 * d.G3 : d.SC;
  a.scale_rows_bulk = scale_row_bytes % 16 == 0 && aligned(dynamic_scales, 16);
  a.ws = cq::carve(workspace, d);
  return a;
}

int permute_impl(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                 const float* smooth, const uint8_t* mask, const int32_t* bs_per_rank,
                 const float* expert_scales, void* expand_x, void* dynamic_scales,
                 int32_t* assist_info, float* expand_scales, void* workspace,
                 size_t workspace_bytes, void* stream) {
  const int rc = check_permute(cfg, x, expert_ids, smooth, expand_x, dynamic_scales,
                               assist_info, workspace, workspace_bytes);
  if (rc != CQ_OK) return rc;
  const cq::PermuteArgs a = permute_args(cfg, x, expert_ids, smooth, mask, bs_per_rank,
                                         expert_scales, expand_x, dynamic_scales, assist_info,
                                         expand_scales, workspace);
  return cq::launch_permute(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CQ_OK
                                                                                   : CQ_ERR_CUDA;
}

}  // namespace

namespace cq {

int dispatch_check(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                   const float* smooth_scales, const uint8_t* x_active_mask, const void* expand_x,
                   const void* dynamic_scales, const int32_t* assist_info,
                   const int32_t* ep_recv_count, const int64_t* expert_token_nums,
                   const void* workspace, size_t workspace_bytes) {
  const int rc = check_route(cfg, expert_ids, x_active_mask, assist_info, ep_recv_count,
                             expert_token_nums, workspace, workspace_bytes);
  if (rc != CQ_OK) return rc;
  return check_permute(cfg, x, expert_ids, smooth_scales, expand_x, dynamic_scales, assist_info,
                       workspace, workspace_bytes);
}

}  // namespace cq

extern "C" {

int cq_check_config(const cq_config* cfg) { return validate(cfg); }

int cq_dispatch_one_kernel(const cq_config* cfg, int with_smooth_scales) {
  const int rc = validate(cfg);
  if (rc != CQ_OK) return rc;
  return cq::dispatch_small_fits(dims_of(cfg), with_smooth_scales && cfg->smooth_kind == 0) ? 1
                                                                                              : 0;
}

int32_t cq_local_expert_num(const cq_config* c) {
  if (!c || c->ep_world_size <= c->shared_expert_rank_num) return 0;
  return c->moe_expert_num / (c->ep_world_size - c->shared_expert_rank_num);
}

int32_t cq_num_slots(const cq_config* c) {
  if (!c) return 0;
  return c->topk + (c->shared_expert_rank_num > 0 ? c->shared_expert_num : 0);
}

int64_t cq_max_rows(const cq_config* c) {
  if (!c) return 0;
  return (int64_t)c->ep_world_size * c->max_bs * cq_num_slots(c);
}

int32_t cq_scale_cols(const cq_config* c) {
  if (!c) return 0;
  const int32_t blocks = (c->hidden + 31) / 32;
  return (blocks + 1) / 2 * 2;
}

int64_t cq_assist_info_size(const cq_config* c) {
  if (validate(c) != CQ_OK) return -1;
  return cq::assist_size(dims_of(c));
}

size_t cq_workspace_size(const cq_config* c) {
  if (validate(c) != CQ_OK) return 0;
  return cq::workspace_bytes(dims_of(c));
}

size_t cq_dispatch_workspace_size(const cq_config* c) { return cq_workspace_size(c); }

int cq_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || !aligned(workspace, 256)) return CQ_ERR_ARG;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? CQ_OK
             : CQ_ERR_CUDA;
}

int cq_dispatch_route(const cq_config* cfg, const int32_t* expert_ids,
                      const uint8_t* x_active_mask, const int32_t* bs_per_rank,
                      int32_t* assist_info, int32_t* ep_recv_count, int64_t* expert_token_nums,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return route_impl(cfg, expert_ids, x_active_mask, bs_per_rank, assist_info, ep_recv_count,
                    expert_token_nums, workspace, workspace_bytes, stream);
}

int cq_dispatch_permute(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                        const float* smooth_scales, const uint8_t* x_active_mask,
                        const int32_t* bs_per_rank, const float* expert_scales, void* expand_x,
                        void* dynamic_scales, int32_t* assist_info, float* expand_scales,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return permute_impl(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                      expert_scales, expand_x, dynamic_scales, assist_info, expand_scales,
                      workspace, workspace_bytes, stream);
}

int cq_dispatch(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                const float* smooth_scales, const uint8_t* x_active_mask,
                const int32_t* bs_per_rank, const float* expert_scales, void* expand_x,
                void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                int64_t* expert_token_nums, float* expand_scales, void* workspace,
                size_t workspace_bytes, void* stream) {
  // Every argument of both halves is checked before the route half is
  // enqueued, so an argument error leaves the outputs untouched.
  int rc = cq::dispatch_check(cfg, x, expert_ids, smooth_scales, x_active_mask, expand_x,
                             dynamic_scales, assist_info, ep_recv_count, expert_token_nums,
                             workspace, workspace_bytes);
  if (rc != CQ_OK) return rc;
  // A small batch: routing and permute in one kernel.
  const Dims d = dims_of(cfg);
  if (cq::dispatch_small_fits(d, smooth_scales && cfg->smooth_kind == 0)) {
    const cq::PermuteArgs a = permute_args(cfg, x, expert_ids, smooth_scales, x_active_mask,
                                           bs_per_rank, expert_scales, expand_x, dynamic_scales,
                                           assist_info, expand_scales, workspace);
    const cudaError_t e = cq::launch_dispatch_small(a, ep_recv_count, expert_token_nums,
                                                    assist_info + cq::assist_base_off(d),
                                                    static_cast<cudaStream_t>(stream));
    if (e != cudaErrorNotSupported) return e == cudaSuccess ? CQ_OK : CQ_ERR_CUDA;
  }
  rc = route_impl(cfg, expert_ids, x_active_mask, bs_per_rank, assist_info, ep_recv_count,
                  expert_token_nums, workspace, workspace_bytes, stream);
  if (rc != CQ_OK) return rc;
  return permute_impl(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                      expert_scales, expand_x, dynamic_scales, assist_info, expand_scales,
                      workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Checks and argument block shared by the two combine entry points.
int combine_args(const cq_config* cfg, const int32_t* assist_info, const float* expert_scales,
                 const void* ori_x, const float* const_alpha1, const float* const_alpha2,
                 const void* const_v, int32_t out_dtype, void* y, cq::CombineArgs* a) {
  int rc = validate(cfg);
  if (rc != CQ_OK) return rc;
  const Dims d = dims_of(cfg);
  if (!assist_info || !expert_scales || !y) return CQ_ERR_ARG;
  if ((d.C + d.Q) > 0 && !ori_x) return CQ_ERR_ARG;
  if (d.Q > 0 && (!const_alpha1 || !const_alpha2 || !const_v)) return CQ_ERR_ARG;
  if (out_dtype != 0 && out_dtype != 1) return CQ_ERR_ARG;
  if (!aligned(y, 16) || (ori_x && !aligned(ori_x, 16)) || (const_v && !aligned(const_v, 16)))
    return CQ_ERR_ARG;
  *a = cq::CombineArgs{};
  a->d = d;
  a->inv = assist_info + cq::assist_inv_off(d);
  a->expert_scales = expert_scales;
  a->ori_x = static_cast<const uint16_t*>(ori_x);
  a->alpha1 = const_alpha1;
  a->alpha2 = const_alpha2;
  a->const_v = static_cast<const uint16_t*>(const_v);
  a->y = y;
  a->out_f32 = out_dtype;
  return CQ_OK;
}

}  // namespace

extern "C" {

int cq_combine(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
               const int32_t* ep_recv_count, const float* expert_scales, const void* ori_x,
               const float* const_alpha1, const float* const_alpha2, const void* const_v,
               int32_t out_dtype, void* y, void* stream) {
  (void)ep_recv_count;  // the inverse map inside assist_info locates every row
  cq::CombineArgs a;
  int rc = combine_args(cfg, assist_info, expert_scales, ori_x, const_alpha1, const_alpha2,
                        const_v, out_dtype, y, &a);
  if (rc != CQ_OK) return rc;
  if (!expand_x_ffn || !aligned(expand_x_ffn, 16)) return CQ_ERR_ARG;
  a.ffn = static_cast<const uint16_t*>(expand_x_ffn);
  return cq::launch_combine(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CQ_OK
                                                                                   : CQ_ERR_CUDA;
}

int cq_combine_ws(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
                  const int32_t* ep_recv_count, const float* expert_scales, const void* ori_x,
                  const float* const_alpha1, const float* const_alpha2, const void* const_v,
                  int32_t out_dtype, void* y, void* workspace, size_t workspace_bytes,
                  void* stream) {
  (void)ep_recv_count;
  cq::CombineArgs a;
  int rc = combine_args(cfg, assist_info, expert_scales, ori_x, const_alpha1, const_alpha2,
                        const_v, out_dtype, y, &a);
  if (rc != CQ_OK) return rc;
  if (!expand_x_ffn || !aligned(expand_x_ffn, 16)) return CQ_ERR_ARG;
  if ((rc = check_ws(a.d, workspace, workspace_bytes)) != CQ_OK) return rc;
  a.ffn = static_cast<const uint16_t*>(expand_x_ffn);
  a.status = cq::carve(workspace, a.d).status;
  return cq::launch_combine(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CQ_OK
                                                                                   : CQ_ERR_CUDA;
}

int cq_combine_quant(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
                     int8_t* ffn_codes, float* ffn_scales, void* stream) {
  int rc = validate(cfg);
  if (rc != CQ_OK) return rc;
  const Dims d = dims_of(cfg);
  if (!expand_x_ffn || !assist_info || !ffn_codes || !ffn_scales) return CQ_ERR_ARG;
  if (!aligned(expand_x_ffn, 16) || !aligned(ffn_codes, 16) || !aligned(ffn_scales, 4))
    return CQ_ERR_ARG;
  cq::CombineArgs a{};
  a.d = d;
  a.ffn = static_cast<const uint16_t*>(expand_x_ffn);
  a.ffn_q = ffn_codes;
  a.ffn_scales = ffn_scales;
  a.total_rows = assist_info + cq::assist_base_off(d) + d.W;
  return cq::launch_combine_quant(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CQ_OK
             : CQ_ERR_CUDA;
}

int cq_combine_q8(const cq_config* cfg, const int8_t* ffn_codes, const float* ffn_scales,
                  const int32_t* assist_info, const int32_t* ep_recv_count,
                  const float* expert_scales, const void* ori_x, const float* const_alpha1,
                  const float* const_alpha2, const void* const_v, int32_t out_dtype, void* y,
                  void* stream) {
  (void)ep_recv_count;
  cq::CombineArgs a;
  int rc = combine_args(cfg, assist_info, expert_scales, ori_x, const_alpha1, const_alpha2,
                        const_v, out_dtype, y, &a);
  if (rc != CQ_OK) return rc;
  if (!ffn_codes || !ffn_scales || !aligned(ffn_codes, 16) || !aligned(ffn_scales, 4))
    return CQ_ERR_ARG;
  a.ffn_q = const_cast<int8_t*>(ffn_codes);
  a.ffn_scales = const_cast<float*>(ffn_scales);
  return cq::launch_combine_q8(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CQ_OK
             : CQ_ERR_CUDA;
}

int moe_dispatch(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                 const float* smooth_scales, const uint8_t* x_active_mask,
                 const int32_t* bs_per_rank, const float* expert_scales, void* expand_x,
                 void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                 int64_t* expert_token_nums, float* expand_scales, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return cq_dispatch(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                     expert_scales, expand_x, dynamic_scales, assist_info, ep_recv_count,
                     expert_token_nums, expand_scales, workspace, workspace_bytes, stream);
}

int moe_combine(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
                const int32_t* ep_recv_count, const float* expert_scales, const void* ori_x,
                const float* const_alpha1, const float* const_alpha2, const void* const_v,
                int32_t out_dtype, void* y, void* stream) {
  return cq_combine(cfg, expand_x_ffn, assist_info, ep_recv_count, expert_scales, ori_x,
                    const_alpha1, const_alpha2, const_v, out_dtype, y, stream);
}

int cq_read_status(void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status) return CQ_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CQ_ERR_CUDA;
  *status = v;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return CQ_ERR_CUDA;
  return CQ_OK;
}

int cq_read_combine_status(uint32_t* status, void* stream) {
  if (!status) return CQ_ERR_ARG;
  return cq::read_combine_status(status, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CQ_OK
             : CQ_ERR_CUDA;
}

namespace {
// One thread waits, with the limits every kernel of the library uses, on an
// mbarrier phase that nothing completes, and records whether it gave up.
__device__ uint32_t g_wait_probe;
__global__ void bounded_wait_probe() {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  cq::async::mbar_init(&bar, 1);
  cq::async::mbar_fence_init();
  g_wait_probe = cq::async::mbar_wait(&bar, 0) ? 0u : 1u;
}
}  // namespace

int cq_check_bounded_wait(uint32_t* gave_up, double* seconds, void* stream) {
  if (!gave_up || !seconds) return CQ_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbolAsync(g_wait_probe, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return CQ_ERR_CUDA;
  const auto t0 = std::chrono::steady_clock::now();
  bounded_wait_probe<<<1, 32, 0, s>>>();
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return CQ_ERR_CUDA;
  *seconds = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  uint32_t v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_wait_probe, sizeof v, 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return CQ_ERR_CUDA;
  *gave_up = v;
  return CQ_OK;
}

const char* cq_strerror(int code) {
  switch (code) {
    case CQ_OK: return "ok";
    case CQ_ERR_ARG: return "invalid argument (range, divisibility, null or misaligned pointer)";
    case CQ_ERR_UNSUPPORTED: return "unsupported hidden size (needs H % 16 == 0, H % 32 for mx modes)";
    case CQ_ERR_CUDA: return "CUDA launch or query failed";
    case CQ_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CQ_ERR_TOO_LARGE: return "problem needs more scratch than the built-in no-alloc buffer";
    default: return "unknown error";
  }
}

}  // extern "C"
