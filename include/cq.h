/*
 * cq.h -- C ABI of libcq: MoE dispatch / combine with pre-communication
 * quantisation, for one GB300 (sm_103a) holding every logical EP rank.
 *
 * The operation is the one described by these pages (cited by title and
 * section throughout):
 *   [DV3]  "CANN ops-transformer 算子解析：MoeDistributeDispatchV3 的 EP 域
 *           Token 分发与动态量化通信实现"
 *   [DSN]  "MoeDistributeDispatch和MoeDistributeCombine算子设计介绍"
 *   [LLD]  "low_latency_dispatch" (CANN API reference page)
 *   [PERF] "CANN MoE Dispatch/Combine 通信算子性能优化实践：Kernel 直调与
 *           ACL SHMEM 实现专家分发与聚合"
 *
 * Logical ranks. ep_world_size = W ranks share one device. Every per-rank
 * tensor of the pages gains a leading rank axis, and the all-to-all exchange
 * becomes an on-device scatter: the rows received by rank d occupy the
 * global row range [rank_row_base[d], rank_row_base[d+1]) of expand_x.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major, contiguous, owned
 *     by the caller. The library never allocates or frees memory.
 *   - `stream` is a cudaStream_t passed as void*, created on the device that
 *     is current when the call is made (the library sizes launches, caches
 *     per-device state and finds its built-in arrays by the current device),
 *     and every pointer refers to that device's memory. Work is enqueued on
 *     it and the call returns without synchronising (except cq_read_status
 *     and cq_read_combine_status).
 *   - Return 0 (CQ_OK) or a negative CQ_ERR_* code. Argument errors are found
 *     on the host before anything is enqueued; nothing is enqueued then.
 *   - Data-dependent problems found on the device (an out-of-range expert
 *     id, a 1-D mask that is not a prefix, a bounded wait that gave up) never
 *     trap: they set sticky bits in the workspace status word, read with
 *     cq_read_status (the combine calls that take no workspace, in a
 *     per-device word read with cq_read_combine_status).
 *
 * Notation: W = ep_world_size, M = moe_expert_num, S = shared_expert_num,
 * S_r = shared_expert_rank_num, L = M / (W - S_r) experts per MoE rank,
 * BS = max_bs, K = topk, H = hidden, NS = K + (S_r > 0 ? S : 0) slots per
 * token, R_max = W * BS * NS (bound on dispatched rows, all ranks together),
 * SC = Align2(Ceil(H, 32)) mx scale columns.
 */
#ifndef CQ_H
#define CQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Operator attributes, [DV3] 参数说明 / [LLD] parameter list. */
typedef struct cq_config {
  int32_t ep_world_size;          /* W in [2, 768] */
  int32_t moe_expert_num;         /* M in [1, 1024], M % (W - S_r) == 0, L * W <= 2048 */
  int32_t shared_expert_num;      /* S in [0, 4]; with S_r == 0 only 0 or 1 (ignored) */
  int32_t shared_expert_rank_num; /* S_r in [0, W); S_r % S == 0 and W % S_r == 0 */
  int32_t zero_expert_num;        /* Z >= 0: ids [M, M+Z) give Moe(x) = 0 */
  int32_t copy_expert_num;        /* C >= 0: ids [M+Z, M+Z+C) give Moe(x) = x */
  int32_t const_expert_num;       /* Q >= 0: ids [M+Z+C, M+Z+C+Q) give a1*x + a2*v */
  int32_t max_bs;                 /* BS in [1, 512], tokens per rank (maximum) */
  int32_t topk;                   /* K in [1, 16], K <= M + Z + C + Q */
  int32_t hidden;                 /* H in [1024, 8192]; the library needs H % 16 == 0
                                     (H % 32 == 0 for quant_mode 4 and 5) */
  int32_t global_bs;              /* 0 or BS * W ([DV3] global_bs) */
  int32_t quant_mode;             /* 0 none, 1 static int8, 2 per-token int8, 3 per-128-group
                                     fp8, 4 mx fp8, 5 mx-clip fp8 ([LLD] 计算公式) */
  int32_t expert_token_nums_type; /* 0 cumulative sums, 1 counts */
  int32_t mask_ndim;              /* 0 none, 1 per token [W,BS], 2 per pair [W,BS,K] */
  int32_t x_dtype;                /* 0 bf16, 1 fp16: x, ori_x, const_v, expert outputs, y */
  int32_t smooth_kind;            /* shape of smooth_scales ("scales"): 0 one row per expert
                                     [(S_r>0 ? S : 0) + M, H], 1 one row [H] for every
                                     expert, 2 one scalar [1] */
  int32_t y_dtype;                /* fp8 code type of modes 3-5 ([LLD] y_dtype): 0 e4m3fn
                                     (largest value 448, emax 8), 1 e5m2 (57344, emax 15);
                                     must be 0 in modes 0-2 */
} cq_config;

enum {
  CQ_OK = 0,
  CQ_ERR_ARG = -1,         /* a range or divisibility rule broken, or a required pointer NULL */
  CQ_ERR_UNSUPPORTED = -2, /* H not a multiple of 16 (32 for quant_mode 4 and 5) */
  CQ_ERR_CUDA = -3,        /* a CUDA launch or query failed */
  CQ_ERR_WORKSPACE = -4,   /* workspace smaller than cq_workspace_size() or misaligned */
  CQ_ERR_TOO_LARGE = -5    /* cq_dispatch_noalloc: the problem needs more scratch than
                              CQ_NOALLOC_SCRATCH_BYTES */
};

/* Sticky device status bits (cq_read_status). */
enum {
  CQ_ST_BAD_ID = 1,  /* an active pair named an id outside [0, M+Z+C+Q); it was skipped */
  CQ_ST_BAD_MASK = 2, /* a 1-D x_active_mask had a true entry after a false one
                         ([DV3] x_active_mask_optional); entries were honoured as given */
  CQ_ST_INTERNAL = 4,  /* a computed row or code fell outside its buffer (an internal
                          consistency guard); the access was skipped */
  CQ_ST_TIMEOUT = 8    /* a kernel's bounded wait for its own bulk copies gave up (about
                          one second); the kernel stopped early and its outputs are
                          incomplete */
};

/* Codes stored in the inverse map for slots that own no dispatched row. */
enum { CQ_INV_NONE = -1, CQ_INV_COPY = -2, CQ_INV_CONST_BASE = -3 /* const c -> -3 - c */ };

/* Validate a config; CQ_OK or CQ_ERR_ARG / CQ_ERR_UNSUPPORTED. */
int cq_check_config(const cq_config* cfg);

/* Derived sizes (no validation beyond what they need; 0 or -1 on NULL). */
int32_t cq_local_expert_num(const cq_config* cfg); /* L */
int32_t cq_num_slots(const cq_config* cfg);        /* NS */
int64_t cq_max_rows(const cq_config* cfg);         /* R_max */
int32_t cq_scale_cols(const cq_config* cfg);       /* SC */
int64_t cq_assist_info_size(const cq_config* cfg); /* int32 elements of assist_info */
size_t cq_workspace_size(const cq_config* cfg);    /* bytes */
size_t cq_dispatch_workspace_size(const cq_config* cfg); /* the same size, by its other name */

/* Zero-fill a freshly allocated workspace (enqueued on `stream`). Required
 * once before its first use; the library keeps it consistent afterwards.
 * Returns CQ_ERR_ARG if workspace is NULL. */
int cq_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * cq_dispatch -- routing scan + permute + pre-communication quantisation.
 * [DSN] §2.2 (sendStatus scan, expandIdx, MoePermute), §2.4 (ep_recv_count as
 * the transposed received-count matrix prefix-summed row-major, expert token
 * numbers), [DV3] 功能说明 情形 1 / 情形 2 and [LLD] 计算公式 quant_mode 0-5.
 *
 * Inputs ("the token type" is bf16, or fp16 when x_dtype is 1):
 *   x              token type [W, BS, H]  tokens of every logical rank
 *   expert_ids     int32 [W, BS, K] routed expert ids (MoE, zero, copy, const ranges)
 *   smooth_scales  the "scales" of [LLD]: required in mode 1, optional in
 *                  modes 2 and 3, NULL in modes 0, 4, 5. Shape by
 *                  smooth_kind: 0 f32 [(S_r>0 ? S : 0) + M, H] (shared expert s
 *                  uses row s, MoE expert e row (S_r>0 ? S : 0) + e), 1 f32 [H]
 *                  for every expert, 2 f32 [1].
 *   x_active_mask  uint8 [W, BS] (mask_ndim 1) or [W, BS, K] (2), or NULL
 *   bs_per_rank    int32 [W] tokens of each rank (<= BS), or NULL for all BS
 *   expert_scales  f32 [W, BS, K] routing weights, or NULL (expand_scales
 *                  then unused)
 * Outputs (rows past the true total are left untouched):
 *   expand_x       [R_max, H]: the token type (mode 0), int8 (modes 1, 2),
 *                  fp8 bytes (modes 3, 4, 5: e4m3fn, or e5m2 when y_dtype is 1).
 *                  Rank d's rows, expert-contiguous
 *                  (local expert ascending, then source rank ascending, then
 *                  arrival order).
 *   dynamic_scales dequantisation multipliers: f32 [R_max] (mode 2), f32
 *                  [R_max, Ceil(H,128)] one per 128-group (mode 3), uint8 e8m0
 *                  [R_max, SC] block scales 2^e stored as e+127 (modes 4, 5,
 *                  pad column 0); not used in modes 0 and 1 (may be NULL).
 *   assist_info    int32 [cq_assist_info_size()]: pass unchanged to cq_combine.
 *                  Layout: [R_max][4] rows (src_rank, src_token, slot, 0);
 *                  then inv [W, BS, NS] (row of each slot or a CQ_INV_* code);
 *                  then rank_row_base [W + 1].
 *   ep_recv_count  int32 [W, W * L]: per destination rank d, the inclusive
 *                  running row count over (local expert, source rank),
 *                  local-expert major; a shared-expert rank fills W entries.
 *   expert_token_nums int64 [W, L]: per rank, rows per local expert (type 1)
 *                  or their running sum (type 0); shared ranks fill 1 entry.
 *   expand_scales  f32 [R_max] or NULL: the routing weight of each row
 *                  (1.0 on shared-expert rows).
 *   workspace      >= cq_workspace_size() bytes, 256-byte aligned, zero-filled
 *                  once by cq_workspace_init before first use.
 * Alignment (else CQ_ERR_ARG): x, expand_x, assist_info and a smooth_scales
 * row table (smooth_kind 0, 1) 16 bytes; a scalar smooth_scales and f32
 * dynamic_scales (modes 2, 3) 4 bytes.
 */
int cq_dispatch(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                const float* smooth_scales, const uint8_t* x_active_mask,
                const int32_t* bs_per_rank, const float* expert_scales, void* expand_x,
                void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                int64_t* expert_token_nums, float* expand_scales, void* workspace,
                size_t workspace_bytes, void* stream);

/* The two halves of cq_dispatch, same arguments; calling cq_dispatch_route
 * then cq_dispatch_permute on one stream gives exactly cq_dispatch's outputs
 * and status. (For a small batch, W * BS * K <= 2048 pairs and
 * (S_r + M) * W <= 2048 with quant_mode 0, 2 or 5 with e4m3 codes, and with
 * one smooth row per expert W * BS * NS * H <= 2^23, cq_dispatch itself runs
 * both halves in one kernel.)
 * route: scan, counts, prefix sums (writes ep_recv_count, expert_token_nums,
 *        the rank_row_base part of assist_info, and the workspace);
 * permute: row placement and quantisation (writes expand_x, dynamic_scales,
 *        the rows and inv parts of assist_info, expand_scales). It may start
 *        while the route kernel still runs and prefetch token rows; the mask
 *        and bs_per_rank (nullable, as given to route) only stop it from
 *        prefetching rows of inactive tokens. */
int cq_dispatch_route(const cq_config* cfg, const int32_t* expert_ids,
                      const uint8_t* x_active_mask, const int32_t* bs_per_rank,
                      int32_t* assist_info, int32_t* ep_recv_count, int64_t* expert_token_nums,
                      void* workspace, size_t workspace_bytes, void* stream);
int cq_dispatch_permute(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                        const float* smooth_scales, const uint8_t* x_active_mask,
                        const int32_t* bs_per_rank, const float* expert_scales,
                        void* expand_x, void* dynamic_scales, int32_t* assist_info,
                        float* expand_scales, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * cq_combine -- inverse permute + top-K weighted sum.
 * [DSN] §3.4 (locate each expert output of token i, weighted sum), [PERF]
 * Combine 计算步骤 (multiply by expert_scales, sum in float, add the shared
 * outputs), [LLD] 特殊专家场景 (zero / copy / const experts).
 *
 *   y[r,i,:] = cast( sum_{j<K} w[r,i,j] * v_j  +  sum_{s<S} shared_s )
 * accumulated in fp32 with one fused multiply-add per j, j ascending, then
 * the shared rows added in s order. v_j is expand_x_ffn[row] for a MoE
 * expert, 0 for a zero expert, ori_x[r,i] for a copy expert, and
 * alpha1[c]*ori_x + alpha2[c]*const_v[c] (products then sum, each rounded)
 * for const expert c. Inactive tokens give 0.
 *
 *   expand_x_ffn   token type [R_max, H] expert outputs, row-aligned with expand_x
 *   assist_info    as written by cq_dispatch
 *   ep_recv_count  as written by cq_dispatch, or NULL (the row map inside
 *                  assist_info already locates every row)
 *   expert_scales  f32 [W, BS, K]
 *   ori_x          token type [W, BS, H]; required when C + Q > 0, else may be NULL
 *   const_alpha1, const_alpha2  f32 [Q]; const_v token type [Q, H]; required when Q > 0
 *   out_dtype      0: y is the token type [W, BS, H]; 1: y is f32 [W, BS, H]
 */
int cq_combine(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
               const int32_t* ep_recv_count, const float* expert_scales, const void* ori_x,
               const float* const_alpha1, const float* const_alpha2, const void* const_v,
               int32_t out_dtype, void* y, void* stream);

/* cq_combine reporting to a workspace: the same operation and arguments, plus
 * the dispatch workspace of the same config (>= cq_workspace_size() bytes,
 * 256-byte aligned; CQ_ERR_WORKSPACE otherwise). A bounded wait that gave up
 * sets CQ_ST_TIMEOUT in that workspace's status word, read and cleared with
 * cq_read_status, instead of the per-device word of cq_read_combine_status;
 * so pipelines on different streams, each with its own workspace, see only
 * their own status. Only the status word of the workspace is touched. */
int cq_combine_ws(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
                  const int32_t* ep_recv_count, const float* expert_scales, const void* ori_x,
                  const float* const_alpha1, const float* const_alpha2, const void* const_v,
                  int32_t out_dtype, void* y, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * Combine with int8 expert outputs ("CANN MoE Dispatch/Combine 通信算子性能
 * 优化实践", 通信前量化: Combine 发送前按 block 量化为 int8, Int8QuantProcess /
 * Int8DequantProcess). The expert side quantises each output row before it is
 * sent back, in blocks of 8 values (32 bytes of fp32): scale = max|v| times
 * fl(1/127), and the binary32 quotient v / scale is cast float -> fp16 ->
 * int8 as the page writes it, each cast rounding to nearest even, the int8
 * one saturating (an all-zero block has scale 0 and codes 0). The receiving
 * side casts int8 -> fp16 -> float (exact), multiplies by the scale (one
 * binary32 rounding) and then forms exactly the sum of cq_combine.
 *
 * cq_combine_quant: expand_x_ffn token type [R_max, H] -> ffn_codes int8 [R_max, H]
 *   and ffn_scales f32 [R_max, H/8]; only the dispatched rows (the total in
 *   assist_info) are written. A producer that fuses this quantisation into
 *   its own epilogue can skip this call.
 * cq_combine_q8: as cq_combine, reading ffn_codes / ffn_scales instead of
 *   16-bit rows (0.5 fewer bytes per value).
 */
int cq_combine_quant(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
                     int8_t* ffn_codes, float* ffn_scales, void* stream);
int cq_combine_q8(const cq_config* cfg, const int8_t* ffn_codes, const float* ffn_scales,
                  const int32_t* assist_info, const int32_t* ep_recv_count,
                  const float* expert_scales, const void* ori_x, const float* const_alpha1,
                  const float* const_alpha2, const void* const_v, int32_t out_dtype, void* y,
                  void* stream);

/* The operators under their MoE names: identical to cq_dispatch / cq_combine. */
int moe_dispatch(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                 const float* smooth_scales, const uint8_t* x_active_mask,
                 const int32_t* bs_per_rank, const float* expert_scales, void* expand_x,
                 void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                 int64_t* expert_token_nums, float* expand_scales, void* workspace,
                 size_t workspace_bytes, void* stream);
int moe_combine(const cq_config* cfg, const void* expand_x_ffn, const int32_t* assist_info,
                const int32_t* ep_recv_count, const float* expert_scales, const void* ori_x,
                const float* const_alpha1, const float* const_alpha2, const void* const_v,
                int32_t out_dtype, void* y, void* stream);

/*
 * cq_dispatch_noalloc -- cq_dispatch for callers that cannot allocate device
 * memory. The pages have no counterpart: it exists for this library's users.
 *
 * Who needs it: a caller that is handed only its input and output buffers and
 * has no way to obtain a workspace -- a plugin inside a framework that owns
 * every allocation, a serving process whose memory plan is fixed at start-up
 * (cudaMalloc on the request path can synchronise the device and fragment the
 * pool), an embedded deployment with a pre-planned memory map.
 *
 * Same arguments and outputs as cq_dispatch, minus the workspace: the scratch
 * lives in a device array of CQ_NOALLOC_SCRATCH_BYTES built into libcq, which
 * every GPU that loads the library holds until the process exits. The call
 * allocates nothing and calls no allocating routine.
 *   - Problems whose cq_workspace_size() exceeds CQ_NOALLOC_SCRATCH_BYTES are
 *     rejected with CQ_ERR_TOO_LARGE before anything is enqueued (4 MiB covers
 *     e.g. W=64, BS=512, K=8, M=256).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it; make that
 *     first call before any stream capture.
 *   - All calls share the one array, and each call clears its header itself.
 *     Calls that overlap on the GPU (other streams, other threads) race on it;
 *     serialise them.
 *   - The device status word of this variant is not reported; use cq_dispatch
 *     with a workspace and cq_read_status when the status bits are needed.
 */
#define CQ_NOALLOC_SCRATCH_BYTES (4u << 20)
int cq_dispatch_noalloc(const cq_config* cfg, const void* x, const int32_t* expert_ids,
                        const float* smooth_scales, const uint8_t* x_active_mask,
                        const int32_t* bs_per_rank, const float* expert_scales, void* expand_x,
                        void* dynamic_scales, int32_t* assist_info, int32_t* ep_recv_count,
                        int64_t* expert_token_nums, float* expand_scales, void* stream);

/* Synchronise `stream`, copy the workspace status word into *status and clear
 * it. One of the two calls in this library that wait for the device. */
int cq_read_status(void* workspace, uint32_t* status, void* stream);

/* cq_combine and cq_combine_q8 take no workspace; their status word
 * (CQ_ST_TIMEOUT only: a bounded wait for the kernel's own bulk loads gave
 * up) is one word per device inside the library, shared by all such combine
 * calls on that device (cq_combine_ws reports to its workspace instead).
 * Synchronise `stream`, copy the word of the current device into *status and
 * clear it. Returns CQ_ERR_ARG if status is NULL, CQ_ERR_CUDA on a CUDA
 * error. */
int cq_read_combine_status(uint32_t* status, void* stream);

/* Diagnostic (no counterpart in the pages): every wait of a kernel in this
 * library on its own bulk copies gives up after about one second (or a cap on
 * polls), sets CQ_ST_TIMEOUT and lets the kernel end, instead of hanging the
 * device. This call runs that same wait on a barrier phase that nothing
 * completes, on `stream`, and synchronises: *gave_up = 1 when the wait ended
 * by its limit, *seconds = the host-measured duration of the launch. The
 * device stays usable afterwards. CQ_ERR_ARG for NULL outputs. */
int cq_check_bounded_wait(uint32_t* gave_up, double* seconds, void* stream);

/* Which kernels cq_dispatch runs for a config (no counterpart in the pages;
 * host only, nothing is enqueued): 1 when it runs routing and permute as one
 * kernel (a small batch: W * BS * K <= 2048, (S_r + M) * W <= 2048,
 * quant_mode 0, 2 or 5 with e4m3 codes, and with one smooth row per expert
 * W * BS * NS * H <= 2^23), 0 when it runs the routing kernels and the
 * permute kernels, or a negative CQ_ERR_* code for an invalid config.
 * with_smooth_scales: nonzero when the call passes smooth_scales. */
int cq_dispatch_one_kernel(const cq_config* cfg, int with_smooth_scales);

/* Static description of an error code. */
const char* cq_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* CQ_H */
