/*
 * cq_oracle.h -- plain CPU oracle for the MoE dispatch / combine hot path
 * with pre-communication quantisation.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers. The CUDA library never includes,
 * links or calls this code, and this code shares nothing with it.
 *
 * Sources, cited by page title and section:
 *   [DV3]  "CANN ops-transformer 算子解析：MoeDistributeDispatchV3 的 EP 域
 *           Token 分发与动态量化通信实现"
 *   [DSN]  "MoeDistributeDispatch和MoeDistributeCombine算子设计介绍"
 *   [LLD]  "low_latency_dispatch" (CANN API reference page)
 *   [PERF] "CANN MoE Dispatch/Combine 通信算子性能优化实践：Kernel 直调与
 *           ACL SHMEM 实现专家分发与聚合"
 *
 * Array conventions (all host memory, row-major, caller-owned):
 *   x, ori_x, ffn rows, const_v and 16-bit outputs are bf16 (x_dtype 0) or fp16
 *   (x_dtype 1), stored as raw uint16 bit patterns.
 *   NS  = K + (shared_expert_rank_num > 0 ? shared_expert_num : 0) slots per token.
 *   R_max = W * BS * NS is the bound on dispatched rows over all logical ranks.
 */
#ifndef CQ_ORACLE_H
#define CQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cqo_config {
  int32_t ep_world_size;          /* W */
  int32_t moe_expert_num;         /* M */
  int32_t shared_expert_num;      /* S */
  int32_t shared_expert_rank_num; /* S_r */
  int32_t zero_expert_num;        /* Z */
  int32_t copy_expert_num;        /* C */
  int32_t const_expert_num;       /* Q */
  int32_t max_bs;                 /* BS */
  int32_t topk;                   /* K */
  int32_t hidden;                 /* H */
  int32_t global_bs;              /* 0 or BS * W */
  int32_t quant_mode;             /* 0 .. 5 */
  int32_t expert_token_nums_type; /* 0 = cumulative sum, 1 = counts */
  int32_t mask_ndim;              /* 0 = no mask, 1 = [W,BS], 2 = [W,BS,K] */
  int32_t x_dtype;                /* 0 = bf16, 1 = fp16 (x, ori_x, const_v, ffn rows, y) */
  int32_t smooth_kind;            /* scales shape: 0 = per expert rows [(S)+M, H],
                                     1 = one row [H] for every expert, 2 = one scalar */
  int32_t y_dtype;                /* fp8 code type of modes 3-5: 0 = e4m3fn, 1 = e5m2 */
} cqo_config;

/* Return codes. */
#define CQO_OK 0
#define CQO_ERR_ARG (-1)
#define CQO_ERR_UNSUPPORTED (-2)
#define CQO_ERR_NOMEM (-3)

/* Status bits (data-dependent conditions found while scanning). */
#define CQO_ST_BAD_ID 1u   /* an expert id outside [0, M+Z+C+Q) */
#define CQO_ST_BAD_MASK 2u /* a 1-D mask whose true entries do not all precede the false ones */

/* Codes stored in inv[] for slots that own no dispatched row. */
#define CQO_INV_NONE (-1)       /* zero expert, masked pair, invalid id, inactive token */
#define CQO_INV_COPY (-2)       /* copy expert */
#define CQO_INV_CONST_BASE (-3) /* const expert c is stored as -3 - c */

int cqo_check_config(const cqo_config* c);
int32_t cqo_local_expert_num(const cqo_config* c);
int32_t cqo_num_slots(const cqo_config* c);
int64_t cqo_max_rows(const cqo_config* c);
int32_t cqo_scale_cols(const cqo_config* c); /* mode 5: Align2(Ceil(H, 32)) */

/* Routing: scan, counts, receive-side prefix sums, row placement.
 * Outputs (sizes):
 *   expand_idx        int32 [W*BS*NS]   arrival ordinal at the target expert, -1 if none
 *   ep_recv_count     int32 [W * W*L]   per destination rank, inclusive prefix, zero-padded
 *   expert_token_nums int64 [W * L]     per destination rank, zero-padded
 *   rank_row_base     int64 [W+1]       first global row of each destination rank
 *   assist            int32 [R_max*4]   (src_rank, src_token, slot, 0) per row
 *   inv               int32 [W*BS*NS]   row of each slot, or a CQO_INV_* code
 * Returns the number of rows placed, or a negative error code. */
int64_t cqo_route(const cqo_config* c, const int32_t* expert_ids, const uint8_t* mask,
                  const int32_t* bs_per_rank, int32_t* expand_idx, int32_t* ep_recv_count,
                  int64_t* expert_token_nums, int64_t* rank_row_base, int32_t* assist,
                  int32_t* inv, uint32_t* status);

/* Quantise one row of H bf16 values (x_dtype 0) or fp16 values (x_dtype 1).
 * smooth_row: H floats, or NULL; smooth_scalar: used instead when not NULL.
 *   mode 0: codes = the H 16-bit values, no scale.
 *   mode 1: codes = H int8 (static: x * smooth), no scale.
 *   mode 2: codes = H int8; scale = one float (the dequantisation multiplier).
 *   mode 3: codes = H e4m3; scale = Ceil(H,128) floats (per 128-group multipliers).
 *   mode 4: codes = H e4m3; scale = Align2(Ceil(H,32)) e8m0 bytes (floor rule).
 *   mode 5: codes = H e4m3; scale = Align2(Ceil(H,32)) e8m0 bytes (clip rule). */
int cqo_quant_row2(int32_t mode, int32_t x_dtype, int32_t hidden, const uint16_t* x_row,
                   const float* smooth_row, const float* smooth_scalar, void* codes,
                   void* scale);

/* cqo_quant_row2 with the fp8 code type of modes 3-5 chosen by y_dtype
 * (0 = e4m3fn, dst_type_max 448, emax 8; 1 = e5m2, 57344, emax 15). */
int cqo_quant_row3(int32_t mode, int32_t x_dtype, int32_t y_dtype, int32_t hidden,
                   const uint16_t* x_row, const float* smooth_row, const float* smooth_scalar,
                   void* codes, void* scale);
/* bf16 input, per-element smooth row or none (the original entry point). */
int cqo_quant_row(int32_t mode, int32_t hidden, const uint16_t* x_row, const float* smooth_row,
                  void* codes, void* scale);
int32_t cqo_group_cols(const cqo_config* c); /* mode 3: Ceil(H, 128) */
float cqo_f16_to_f32(uint16_t h);
uint16_t cqo_f16_from_f32(float f); /* round to nearest even */
int32_t cqo_floor_log2(float a);    /* exact floor(log2(a)) for finite a > 0 */

/* Whole dispatch: routing plus quantisation of every placed row.
 * expand_x is [R_max, H] of the mode's code type; dynamic_scales is [R_max] float
 * (mode 2), [R_max, group_cols] float (mode 3), [R_max, scale_cols] bytes
 * (modes 4, 5) or unused (modes 0, 1); smooth follows smooth_kind;
 * expand_scales (nullable) is [R_max] float. */
int64_t cqo_dispatch(const cqo_config* c, const uint16_t* x, const int32_t* expert_ids,
                     const float* smooth, const uint8_t* mask, const int32_t* bs_per_rank,
                     const float* expert_scales, void* expand_x, void* dynamic_scales,
                     float* expand_scales, int32_t* expand_idx, int32_t* ep_recv_count,
                     int64_t* expert_token_nums, int64_t* rank_row_base, int32_t* assist,
                     int32_t* inv, uint32_t* status);

/* Combine one token (r, i) into y_row (H values; 16-bit bits of x_dtype if
 * out_f32 == 0, else float). ffn is [rows, H] of x_dtype. */
int cqo_combine_token(const cqo_config* c, int32_t r, int32_t i, const uint16_t* ffn,
                      const int32_t* inv, const float* expert_scales, const uint16_t* ori_x,
                      const float* const_alpha1, const float* const_alpha2,
                      const uint16_t* const_v, int32_t out_f32, void* y_row);

/* Combine every token: y is [W, BS, H]. */
int cqo_combine(const cqo_config* c, const uint16_t* ffn, const int32_t* inv,
                const float* expert_scales, const uint16_t* ori_x, const float* const_alpha1,
                const float* const_alpha2, const uint16_t* const_v, int32_t out_f32, void* y);

/* Combine-side int8 block quantisation of one expert-output row of H 16-bit
 * values: blocks of 8 elements, scale = max|v| * fl(1/127), codes = the
 * quotient v / scale cast float -> fp16 -> int8 (each cast round-to-nearest-
 * even, the int8 one saturating). codes [H], scales [H/8] (H % 8 == 0). */
int cqo_combine_quant_row(int32_t hidden, int32_t x_dtype, const uint16_t* row, int8_t* codes,
                          float* scales);

/* Combine one token from int8 expert outputs: each routed / shared row is
 * dequantised (code * block scale) before the weighted sum. ffn_codes is
 * [rows, H] int8, ffn_scales [rows, H/8]. Otherwise as cqo_combine_token. */
int cqo_combine_token_q8(const cqo_config* c, int32_t r, int32_t i, const int8_t* ffn_codes,
                         const float* ffn_scales, const int32_t* inv, const float* expert_scales,
                         const uint16_t* ori_x, const float* const_alpha1,
                         const float* const_alpha2, const uint16_t* const_v, int32_t out_f32,
                         void* y_row);

/* Format helpers, exposed so the tests can pin them on their own. */
uint8_t cqo_e4m3_encode(float v);  /* round to nearest even, saturate to +-448 */
float cqo_e4m3_decode(uint8_t b);
uint8_t cqo_e5m2_encode(float v);  /* round to nearest even, saturate to +-57344 */
float cqo_e5m2_decode(uint8_t b);
uint16_t cqo_bf16_from_f32(float f); /* round to nearest even */
float cqo_bf16_to_f32(uint16_t b);
int32_t cqo_ceil_log2(float q);     /* exact ceil(log2(q)) for finite q > 0 */
/* Array forms of the helpers above (n elements). */
void cqo_e4m3_encode_n(const float* in, uint8_t* out, int64_t n);
void cqo_e5m2_encode_n(const float* in, uint8_t* out, int64_t n);
void cqo_bf16_from_f32_n(const float* in, uint16_t* out, int64_t n);
void cqo_ceil_log2_n(const float* in, int32_t* out, int64_t n);

#ifdef __cplusplus
}
#endif
#endif
