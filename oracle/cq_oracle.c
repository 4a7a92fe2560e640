/*
 * cq_oracle.c -- plain CPU oracle for the MoE dispatch / combine hot path.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers; the CUDA library shares no code with
 * this file. Single-threaded, sequential loops, in the order the pages give.
 * Page titles behind the short tags [DV3] [DSN] [LLD] [PERF] are listed in
 * cq_oracle.h.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math), so
 * every float operation below is one IEEE binary32 operation rounded to
 * nearest-even, and fmaf() is the single-rounding fused multiply-add.
 */
/* Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
 * top of cq_oracle.h. */
#include "cq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Configuration rules.                                                      */
/* ------------------------------------------------------------------------ */

int32_t cqo_local_expert_num(const cqo_config* c) {
  /* [DV3] Shape 格式说明: on an MoE-expert rank,
   * local_expert_num = moe_expert_num / (ep_world_size - shared_expert_rank_num). */
  return c->moe_expert_num / (c->ep_world_size - c->shared_expert_rank_num);
}

int32_t cqo_num_slots(const cqo_config* c) {
  /* Each token has K routed slots, plus one slot per shared expert when
   * shared-expert ranks exist ([DV3] 参数说明 shared_expert_num /
   * shared_expert_rank_num). */
  return c->topk + (c->shared_expert_rank_num > 0 ? c->shared_expert_num : 0);
}

int64_t cqo_max_rows(const cqo_config* c) {
  return (int64_t)c->ep_world_size * c->max_bs * cqo_num_slots(c);
}

int32_t cqo_scale_cols(const cqo_config* c) {
  /* [LLD] quant_mode 相关约束: mx modes give dynamic_scales shape (A, Align2(Ceil(H, 32))). */
  int32_t blocks = (c->hidden + 31) / 32;
  return (blocks + 1) / 2 * 2;
}

int cqo_check_config(const cqo_config* c) {
  /* Ranges: [DV3] 约束说明 (Atlas A3 constraints and the torch._check list in
   * the Python wrapper) and [LLD] shape variables. */
  const int32_t W = c->ep_world_size, M = c->moe_expert_num;
  const int32_t S = c->shared_expert_num, Sr = c->shared_expert_rank_num;
  if (W < 2 || W > 768) return CQO_ERR_ARG;
  if (c->hidden < 1024 || c->hidden > 8192) return CQO_ERR_ARG;
  if (c->max_bs < 1 || c->max_bs > 512) return CQO_ERR_ARG;
  if (M < 1 || M > 1024) return CQO_ERR_ARG;
  if (c->topk < 1 || c->topk > 16) return CQO_ERR_ARG;
  if (S < 0 || S > 4) return CQO_ERR_ARG;
  /* [DV3] 参数说明 shared_expert_rank_num: in [0, W); zero requires S in {0, 1},
   * non-zero requires S_r % S == 0. [DV3] 前置校验: W a multiple of S_r. */
  if (Sr < 0 || Sr >= W) return CQO_ERR_ARG;
  if (Sr == 0 && S > 1) return CQO_ERR_ARG;
  if (Sr > 0 && (S == 0 || Sr % S != 0 || W % Sr != 0)) return CQO_ERR_ARG;
  /* [DV3] 前置校验: moe_expert_num a multiple of W - S_r. */
  if (M % (W - Sr) != 0) return CQO_ERR_ARG;
  /* [LLD] local_expert_num * ep_world_size <= 2048. */
  if ((int64_t)cqo_local_expert_num(c) * W > 2048) return CQO_ERR_ARG;
  if (c->zero_expert_num < 0 || c->copy_expert_num < 0 || c->const_expert_num < 0)
    return CQO_ERR_ARG;
  /* [DV3] Shape 格式说明: 0 < K <= M + Z + C + Q, and that sum < MAX_INT32. */
  int64_t all = (int64_t)M + c->zero_expert_num + c->copy_expert_num + c->const_expert_num;
  if (all >= 2147483647LL) return CQO_ERR_ARG;
  if (c->topk > all) return CQO_ERR_ARG;
  /* [DV3] 参数说明 global_bs: 0 or max_bs * ep_world_size. */
  if (c->global_bs != 0 && c->global_bs != c->max_bs * W) return CQO_ERR_ARG;
  if (c->expert_token_nums_type != 0 && c->expert_token_nums_type != 1) return CQO_ERR_ARG;
  if (c->mask_ndim < 0 || c->mask_ndim > 2) return CQO_ERR_ARG;
  /* [LLD] quant_mode 0..5; x as float16 or bfloat16 ([DV3] 参数说明 x). */
  if (c->quant_mode < 0 || c->quant_mode > 5) return CQO_ERR_ARG;
  if (c->x_dtype != 0 && c->x_dtype != 1) return CQO_ERR_ARG;
  if (c->smooth_kind < 0 || c->smooth_kind > 2) return CQO_ERR_ARG;
  /* y_dtype ([LLD] y_dtype: float8_e4m3fn or float8_e5m2 codes): the fp8
   * type of modes 3-5; modes 0-2 have no choice (16-bit or int8). */
  if (c->y_dtype != 0 && c->y_dtype != 1) return CQO_ERR_ARG;
  if (c->y_dtype == 1 && c->quant_mode < 3) return CQO_ERR_ARG;
  return CQO_OK;
}

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                           */
/* ------------------------------------------------------------------------ */

float cqo_bf16_to_f32(uint16_t b) {
  /* bfloat16 is the upper half of a binary32. */
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t cqo_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  /* Round to nearest, ties to even, on the 16 discarded bits. */
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

float cqo_f16_to_f32(uint16_t h) {
  /* IEEE binary16: 1 sign, 5 exponent bits (bias 15), 10 mantissa bits. */
  const int sign = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  float mag;
  if (e == 0) mag = ldexpf((float)m, -24);
  else if (e == 31) mag = m ? NAN : INFINITY;
  else mag = ldexpf(1.0f + (float)m / 1024.0f, e - 15);
  return sign ? -mag : mag;
}

uint16_t cqo_f16_from_f32(float f) {
  /* Round to nearest even; magnitudes from 65520 up overflow to infinity. */
  if (isnan(f)) return 0x7e00;
  const uint16_t sign = signbit(f) ? 0x8000 : 0;
  const float a = fabsf(f);
  if (a >= 65520.0f) return sign | 0x7c00;
  if (a < 0x1p-14f) {
    /* subnormal: value = m * 2^-24, m = 0..1023; m = 1024 is the smallest normal */
    return sign | (uint16_t)rintf(a * 0x1p24f);
  }
  int e;
  frexpf(a, &e);
  int ex = e - 1; /* -14 .. 15 */
  const float t = ldexpf(a, -ex);
  float mq = rintf((t - 1.0f) * 1024.0f);
  if (mq == 1024.0f) {
    mq = 0.0f;
    ex += 1;
  }
  if (ex > 15) return sign | 0x7c00;
  return sign | (uint16_t)(((ex + 15) << 10) | (int)mq);
}

int32_t cqo_floor_log2(float a) {
  /* a = m * 2^e with m in [0.5, 1)  =>  floor(log2(a)) = e - 1 (exact, also
   * for subnormal a). */
  int e;
  frexpf(a, &e);
  return e - 1;
}

int32_t cqo_group_cols(const cqo_config* c) {
  /* [LLD] quant_mode 相关约束: pergroup scales have shape (A, Ceil(H, 128)). */
  return (c->hidden + 127) / 128;
}

int32_t cqo_ceil_log2(float q) {
  /* frexpf gives q = m * 2^e with m in [0.5, 1); q is a power of two exactly
   * when m == 0.5, and then log2(q) = e - 1; otherwise ceil(log2(q)) = e. */
  int e;
  float m = frexpf(q, &e);
  return (m == 0.5f) ? e - 1 : e;
}

float cqo_e4m3_decode(uint8_t b) {
  /* FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits with bias 7, 3 mantissa
   * bits, no infinities, only S.1111.111 is NaN; largest finite 448. */
  int sign = b >> 7, e = (b >> 3) & 0xf, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  float mag = (e == 0) ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return sign ? -mag : mag;
}

uint8_t cqo_e4m3_encode(float v) {
  /* Round to nearest even; magnitudes beyond 448 saturate to 448
   * (satfinite); NaN maps to the NaN code. */
  if (isnan(v)) return 0x7f;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  float a = fabsf(v);
  if (a >= 448.0f) return sign | 0x7e;
  if (a < 0x1p-6f) {
    /* Subnormal range: value = m * 2^-9, m = 0..7; m == 8 is the smallest
     * normal, whose code is also 8. a * 512 is exact. */
    float m = rintf(a * 512.0f);
    return sign | (uint8_t)m;
  }
  int e;
  frexpf(a, &e); /* a = f * 2^e, f in [0.5, 1)  =>  a = (2f) * 2^(e-1) */
  int ex = e - 1;  /* unbiased exponent, -6..8 */
  float t = ldexpf(a, -ex);            /* in [1, 2), exact */
  float mq = rintf((t - 1.0f) * 8.0f); /* 0..8, ties to even */
  if (mq == 8.0f) {
    mq = 0.0f;
    ex += 1;
  }
  int code = ((ex + 7) << 3) | (int)mq;
  if (code > 0x7e) code = 0x7e; /* rounding up past 448 saturates */
  return sign | (uint8_t)code;
}

float cqo_e5m2_decode(uint8_t b) {
  /* FP8 E5M2: 1 sign, 5 exponent bits with bias 15, 2 mantissa bits; the
   * all-ones exponent holds infinity (mantissa 0) and NaN; largest finite
   * 1.75 * 2^15 = 57344. */
  int sign = b >> 7, e = (b >> 2) & 0x1f, m = b & 3;
  float mag;
  if (e == 31) {
    mag = m == 0 ? INFINITY : NAN;
  } else {
    mag = (e == 0) ? ldexpf((float)m, -16) : ldexpf(1.0f + (float)m / 4.0f, e - 15);
  }
  return sign ? -mag : mag;
}

uint8_t cqo_e5m2_encode(float v) {
  /* Round to nearest even; magnitudes beyond 57344 (infinity included)
   * saturate to 57344 (satfinite); NaN maps to the NaN code 0x7f. */
  if (isnan(v)) return 0x7f;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  float a = fabsf(v);
  if (a >= 57344.0f) return sign | 0x7b;
  if (a < 0x1p-14f) {
    /* Subnormal range: value = m * 2^-16, m = 0..3; m == 4 is the smallest
     * normal, whose code is also 4. a * 65536 is exact. */
    float m = rintf(a * 65536.0f);
    return sign | (uint8_t)m;
  }
  int e;
  frexpf(a, &e);                       /* a = f * 2^e, f in [0.5, 1) */
  int ex = e - 1;                      /* unbiased exponent, -14..15 */
  float t = ldexpf(a, -ex);            /* in [1, 2), exact */
  float mq = rintf((t - 1.0f) * 4.0f); /* 0..4, ties to even */
  if (mq == 4.0f) {
    mq = 0.0f;
    ex += 1;
  }
  int code = ((ex + 15) << 2) | (int)mq;
  if (code > 0x7b) code = 0x7b; /* rounding up past 57344 saturates */
  return sign | (uint8_t)code;
}

void cqo_e5m2_encode_n(const float* in, uint8_t* out, int64_t n) {
  for (int64_t t = 0; t < n; ++t) out[t] = cqo_e5m2_encode(in[t]);
}

void cqo_e4m3_encode_n(const float* in, uint8_t* out, int64_t n) {
  for (int64_t t = 0; t < n; ++t) out[t] = cqo_e4m3_encode(in[t]);
}

void cqo_bf16_from_f32_n(const float* in, uint16_t* out, int64_t n) {
  for (int64_t t = 0; t < n; ++t) out[t] = cqo_bf16_from_f32(in[t]);
}

void cqo_ceil_log2_n(const float* in, int32_t* out, int64_t n) {
  for (int64_t t = 0; t < n; ++t) out[t] = cqo_ceil_log2(in[t]);
}

static int8_t sat_rne_int8(float v) {
  /* Round to nearest, ties to even (rintf under the default rounding mode),
   * then saturate to the int8 range; NaN gives 0. */
  if (isnan(v)) return 0;
  float r = rintf(v);
  if (r > 127.0f) r = 127.0f;
  if (r < -128.0f) r = -128.0f;
  return (int8_t)r;
}

/* ------------------------------------------------------------------------ */
/* Quantisation of one row, [LLD] 计算公式 and [DV3] 功能说明 情形 1 / 情形 2. */
/* ------------------------------------------------------------------------ */

static float in16(int32_t dtype, uint16_t v) {
  return dtype ? cqo_f16_to_f32(v) : cqo_bf16_to_f32(v);
}

static uint16_t out16(int32_t dtype, float f) {
  return dtype ? cqo_f16_from_f32(f) : cqo_bf16_from_f32(f);
}

int cqo_quant_row2(int32_t mode, int32_t dt, int32_t H, const uint16_t* x, const float* smooth,
                   const float* smooth_scalar, void* codes, void* scale) {
  return cqo_quant_row3(mode, dt, 0, H, x, smooth, smooth_scalar, codes, scale);
}

int cqo_quant_row3(int32_t mode, int32_t dt, int32_t yt, int32_t H, const uint16_t* x,
                   const float* smooth, const float* smooth_scalar, void* codes, void* scale) {
  /* The fp8 code type of modes 3-5: its largest finite value (dst_type_max)
   * and the exponent of that value (emax). */
  if (yt != 0 && yt != 1) return CQO_ERR_ARG;
  if (yt == 1 && mode < 3) return CQO_ERR_ARG;
  const float fp8_max = yt ? 57344.0f : 448.0f; /* 1.75 * 2^15, 1.75 * 2^8 */
  const int32_t emax = yt ? 15 : 8;
  uint8_t (*fp8_encode)(float) = yt ? cqo_e5m2_encode : cqo_e4m3_encode;
  if (mode == 0) {
    /* quant_out = x: the 16-bit row travels unchanged. */
    memcpy(codes, x, (size_t)H * sizeof(uint16_t));
    return CQO_OK;
  }
  /* [LLD] quant_mode 相关约束: mx modes take no smooth scales; static
   * quantisation (mode 1) needs them. */
  const int has_smooth = smooth != NULL || smooth_scalar != NULL;
  if ((mode == 4 || mode == 5) && has_smooth) return CQO_ERR_ARG;
  if (mode == 1 && !has_smooth) return CQO_ERR_ARG;
  if (mode < 1 || mode > 5) return CQO_ERR_UNSUPPORTED;
  /* x_fp32 = CastToFp32(x) * scales (when given). */
  float* xf = (float*)malloc((size_t)H * sizeof(float));
  if (!xf) return CQO_ERR_NOMEM;
  for (int32_t h = 0; h < H; ++h) {
    const float v = in16(dt, x[h]);
    xf[h] = smooth_scalar ? v * *smooth_scalar : (smooth ? v * smooth[h] : v);
  }
  if (mode == 1) {
    /* static: quant_out = Cast(CastToFp32(x) * scales, int8) */
    int8_t* q = (int8_t*)codes;
    for (int32_t h = 0; h < H; ++h) q[h] = sat_rne_int8(xf[h]);
  } else if (mode == 2) {
    /* dynamic_scales_value = 127 / max|x_fp32|;
     * quant_out = Cast(x_fp32 * dynamic_scales_value, int8);
     * carried scale = 1.0 / dynamic_scales_value. */
    float amax = 0.0f;
    for (int32_t h = 0; h < H; ++h) {
      const float a = fabsf(xf[h]);
      if (a > amax) amax = a;
    }
    const float s = 127.0f / amax; /* +inf for an all-zero row */
    int8_t* q = (int8_t*)codes;
    for (int32_t h = 0; h < H; ++h) q[h] = sat_rne_int8(xf[h] * s);
    *(float*)scale = 1.0f / s;
  } else if (mode == 3) {
    /* pergroup: the mode-2 formulas on each group of 128 values, into
     * the fp8 type (dst_type_max 448 for e4m3, 57344 for e5m2); one carried
     * scale per group. An all-zero group gives codes 0 and scale 0. */
    uint8_t* q = (uint8_t*)codes;
    float* sc = (float*)scale;
    for (int32_t g = 0; g * 128 < H; ++g) {
      const int32_t h0 = g * 128, h1 = (h0 + 128 < H) ? h0 + 128 : H;
      float amax = 0.0f;
      for (int32_t h = h0; h < h1; ++h) {
        const float a = fabsf(xf[h]);
        if (a > amax) amax = a;
      }
      const float s = fp8_max / amax;
      const float mult = amax == 0.0f ? 0.0f : s;
      for (int32_t h = h0; h < h1; ++h) q[h] = fp8_encode(xf[h] * mult);
      sc[g] = 1.0f / s;
    }
  } else {
    /* mode 4 (mx): shared_exp = floor(log2(max|x|)) - emax, emax = 8 for
     *   e4m3 (448 = 1.75 * 2^8), 15 for e5m2 (57344 = 1.75 * 2^15); an
     *   all-zero block uses the smallest scale;
     * mode 5 (mx clip): shared_exp = ceil(log2(max(max|x|, 1e-4) / fp8_max)).
     * Both: quant_out = CastToFp8(x / 2^shared_exp), the block scale
     * 2^shared_exp stored as e8m0 (shared_exp + 127), blocks of 32. */
    uint8_t* q = (uint8_t*)codes;
    uint8_t* sc = (uint8_t*)scale;
    const int32_t nblk = (H + 31) / 32;
    const int32_t cols = (nblk + 1) / 2 * 2;
    for (int32_t b = 0; b < nblk; ++b) {
      const int32_t h0 = b * 32, h1 = (h0 + 32 < H) ? h0 + 32 : H;
      float amax = 0.0f;
      for (int32_t h = h0; h < h1; ++h) {
        const float a = fabsf(xf[h]);
        if (a > amax) amax = a;
      }
      int32_t e;
      if (mode == 4) {
        e = amax == 0.0f ? -127 : cqo_floor_log2(amax) - emax;
        if (e < -127) e = -127;
      } else {
        if (amax < 1e-4f) amax = 1e-4f;
        e = cqo_ceil_log2(amax / fp8_max);
      }
      for (int32_t h = h0; h < h1; ++h) {
        /* x / 2^e; 2^-e is a normal binary32 here, so ldexpf is exact. */
        q[h] = fp8_encode(ldexpf(xf[h], -e));
      }
      sc[b] = (uint8_t)(e + 127);
    }
    for (int32_t b = nblk; b < cols; ++b) sc[b] = 0; /* Align2 padding column */
  }
  free(xf);
  return CQO_OK;
}

int cqo_quant_row(int32_t mode, int32_t H, const uint16_t* x, const float* smooth, void* codes,
                  void* scale) {
  return cqo_quant_row2(mode, 0, H, x, smooth, NULL, codes, scale);
}

/* ------------------------------------------------------------------------ */
/* Routing: [DSN] §2.2.2 (sendStatus scan and expandIdx), §2.4 (receive-side  */
/* metadata), [DV3] 参数说明 / Shape 格式说明 (shared ranks first, special     */
/* expert id ranges, masks, expert_token_nums_type).                          */
/* ------------------------------------------------------------------------ */

/* Is pair (r, i, j) of an in-range token switched on by the mask? */
static int pair_active(const cqo_config* c, const uint8_t* mask, int32_t r, int32_t i, int32_t j) {
  if (c->mask_ndim == 0 || mask == NULL) return 1;
  if (c->mask_ndim == 1) return mask[(int64_t)r * c->max_bs + i] != 0;
  return mask[((int64_t)r * c->max_bs + i) * c->topk + j] != 0;
}

int64_t cqo_route(const cqo_config* c, const int32_t* expert_ids, const uint8_t* mask,
                  const int32_t* bs_per_rank, int32_t* expand_idx, int32_t* ep_recv_count,
                  int64_t* expert_token_nums, int64_t* rank_row_base, int32_t* assist,
                  int32_t* inv, uint32_t* status) {
  int rc = cqo_check_config(c);
  if (rc != CQO_OK) return rc;
  const int32_t W = c->ep_world_size, M = c->moe_expert_num, K = c->topk, BS = c->max_bs;
  const int32_t Sr = c->shared_expert_rank_num;
  const int32_t Seff = (Sr > 0) ? c->shared_expert_num : 0;
  const int32_t L = cqo_local_expert_num(c);
  const int32_t NS = K + Seff;
  const int32_t R = (Sr > 0) ? Sr / c->shared_expert_num : 0; /* replicas per shared expert */
  const int64_t z0 = M, c0 = z0 + c->zero_expert_num, q0 = c0 + c->copy_expert_num;
  const int64_t q1 = q0 + c->const_expert_num;
  const int64_t nslot = (int64_t)W * BS * NS;
  uint32_t st = 0;

  /* dest[] / local[] record, for every slot, the (destination rank, local
   * expert) it is sent to, or -1. */
  int32_t* dest = (int32_t*)malloc((size_t)nslot * sizeof(int32_t));
  int32_t* local = (int32_t*)malloc((size_t)nslot * sizeof(int32_t));
  int32_t* send_status = (int32_t*)malloc((size_t)(M + (Seff > 0 ? Seff : 1)) * sizeof(int32_t));
  if (!dest || !local || !send_status) {
    free(dest);
    free(local);
    free(send_status);
    return CQO_ERR_NOMEM;
  }

  /* Step 1, per source rank r: traverse expertIds in row-major (token, then
   * k) order. For a MoE expert id e the target rank is S_r + e / L (integer
   * division; shared-expert ranks come first), the local index is e % L, and
   * expandIdx is the running count of earlier pairs of this source sent to
   * e, which is then incremented. Shared expert s is replicated on R ranks
   * s*R .. s*R+R-1; source r uses replica r % R, in slot K + s. */
  for (int32_t r = 0; r < W; ++r) {
    const int32_t n_r = bs_per_rank ? bs_per_rank[r] : BS;
    for (int32_t e = 0; e < M; ++e) send_status[e] = 0;
    for (int32_t s = 0; s < Seff; ++s) send_status[M + s] = 0;
    int seen_false = 0;
    for (int32_t i = 0; i < BS; ++i) {
      const int64_t tok = (int64_t)r * BS + i;
      for (int32_t k = 0; k < NS; ++k) {
        expand_idx[tok * NS + k] = -1;
        inv[tok * NS + k] = CQO_INV_NONE;
        dest[tok * NS + k] = -1;
        local[tok * NS + k] = -1;
      }
      if (i >= n_r) continue;
      if (c->mask_ndim == 1 && mask) {
        /* [DV3] x_active_mask: in 1-D form the true entries must precede the false ones. */
        int on = mask[tok] != 0;
        if (!on) seen_false = 1;
        else if (seen_false) st |= CQO_ST_BAD_MASK;
      }
      int any = 0;
      for (int32_t j = 0; j < K; ++j) {
        if (!pair_active(c, mask, r, i, j)) continue;
        any = 1;
        const int64_t sl = tok * NS + j;
        const int64_t id = expert_ids[tok * K + j];
        if (id >= 0 && id < M) {
          expand_idx[sl] = send_status[id]++;
          dest[sl] = Sr + (int32_t)(id / L);
          local[sl] = (int32_t)(id % L);
        } else if (id >= z0 && id < c0) {
          inv[sl] = CQO_INV_NONE; /* zero expert: contributes nothing */
        } else if (id >= c0 && id < q0) {
          inv[sl] = CQO_INV_COPY;
        } else if (id >= q0 && id < q1) {
          inv[sl] = CQO_INV_CONST_BASE - (int32_t)(id - q0);
        } else {
          st |= CQO_ST_BAD_ID;
        }
      }
      /* [DV3] x_active_mask: a token whose entries are all false does not
       * take part, so it reaches no shared expert either. */
      if (any) {
        for (int32_t s = 0; s < Seff; ++s) {
          const int64_t sl = tok * NS + K + s;
          expand_idx[sl] = send_status[M + s]++;
          dest[sl] = s * R + r % R;
          local[sl] = 0;
        }
      }
    }
  }

  /* Step 2, per destination rank d: the received rows are laid out expert by
   * expert (local index ascending), within an expert source rank ascending,
   * within a source in arrival order (expandIdx ascending, which is the scan
   * order). The placement is written out literally, row by row.
   * ep_recv_count[d] is the received-count matrix (source x local expert),
   * transposed and prefix-summed in row-major order ([DSN] §2.4.1), i.e. the
   * running row count at the end of each (local expert, source) block. */
  const int32_t recv_stride = W * L;
  for (int64_t t = 0; t < (int64_t)W * recv_stride; ++t) ep_recv_count[t] = 0;
  for (int64_t t = 0; t < (int64_t)W * L; ++t) expert_token_nums[t] = 0;
  int64_t row = 0;
  for (int32_t d = 0; d < W; ++d) {
    rank_row_base[d] = row;
    const int32_t Ld = (d < Sr) ? 1 : L; /* a shared-expert rank hosts one expert */
    int64_t cum = 0;
    for (int32_t le = 0; le < Ld; ++le) {
      int64_t expert_rows = 0;
      for (int32_t src = 0; src < W; ++src) {
        for (int32_t i = 0; i < BS; ++i) {
          for (int32_t k = 0; k < NS; ++k) {
            const int64_t sl = ((int64_t)src * BS + i) * NS + k;
            if (dest[sl] != d || local[sl] != le) continue;
            assist[row * 4 + 0] = src;
            assist[row * 4 + 1] = i;
            assist[row * 4 + 2] = k;
            assist[row * 4 + 3] = 0;
            inv[sl] = (int32_t)row;
            ++row;
            ++expert_rows;
          }
        }
        ep_recv_count[(int64_t)d * recv_stride + (int64_t)le * W + src] =
            (int32_t)(row - rank_row_base[d]);
      }
      cum += expert_rows;
      /* [DV3] expert_token_nums_type: 0 = prefix sum, 1 = per-expert count. */
      expert_token_nums[(int64_t)d * L + le] = (c->expert_token_nums_type == 0) ? cum : expert_rows;
    }
  }
  rank_row_base[W] = row;

  free(dest);
  free(local);
  free(send_status);
  if (status) *status |= st;
  return row;
}

/* ------------------------------------------------------------------------ */
/* Dispatch = routing + quantisation of each placed row.                     */
/* ------------------------------------------------------------------------ */

int64_t cqo_dispatch(const cqo_config* c, const uint16_t* x, const int32_t* expert_ids,
                     const float* smooth, const uint8_t* mask, const int32_t* bs_per_rank,
                     const float* expert_scales, void* expand_x, void* dynamic_scales,
                     float* expand_scales, int32_t* expand_idx, int32_t* ep_recv_count,
                     int64_t* expert_token_nums, int64_t* rank_row_base, int32_t* assist,
                     int32_t* inv, uint32_t* status) {
  /* [LLD] quant_mode 相关约束: mx modes take no smooth scales; static
   * quantisation (mode 1) needs them. */
  if ((c->quant_mode == 4 || c->quant_mode == 5) && smooth) return CQO_ERR_ARG;
  if (c->quant_mode == 1 && !smooth) return CQO_ERR_ARG;
  int64_t rows = cqo_route(c, expert_ids, mask, bs_per_rank, expand_idx, ep_recv_count,
                           expert_token_nums, rank_row_base, assist, inv, status);
  if (rows < 0) return rows;
  const int32_t H = c->hidden, K = c->topk, BS = c->max_bs;
  const int32_t Seff = (c->shared_expert_rank_num > 0) ? c->shared_expert_num : 0;
  const int32_t cols = cqo_scale_cols(c), gcols = cqo_group_cols(c);
  for (int64_t row = 0; row < rows; ++row) {
    const int32_t src = assist[row * 4 + 0], i = assist[row * 4 + 1], k = assist[row * 4 + 2];
    const int64_t tok = (int64_t)src * BS + i;
    const uint16_t* xr = x + tok * H;
    /* [LLD] quant_mode 相关约束: scales are one scalar (1,), one row (H,)
     * shared by every expert, or per expert: (S + M, H) when shared experts
     * exist, else (M, H); shared expert s uses row s, MoE expert e row S + e. */
    const float* sm = NULL;
    const float* sm_scalar = NULL;
    if (smooth) {
      if (c->smooth_kind == 2) {
        sm_scalar = smooth;
      } else if (c->smooth_kind == 1) {
        sm = smooth;
      } else {
        int64_t srow = (k < K) ? (int64_t)Seff + expert_ids[tok * K + k] : (int64_t)(k - K);
        sm = smooth + srow * H;
      }
    }
    void* codes;
    void* scale = NULL;
    if (c->quant_mode == 0) {
      codes = (uint16_t*)expand_x + row * H;
    } else if (c->quant_mode == 1) {
      codes = (int8_t*)expand_x + row * H;
    } else if (c->quant_mode == 2) {
      codes = (int8_t*)expand_x + row * H;
      scale = (float*)dynamic_scales + row;
    } else if (c->quant_mode == 3) {
      codes = (uint8_t*)expand_x + row * H;
      scale = (float*)dynamic_scales + row * gcols;
    } else {
      codes = (uint8_t*)expand_x + row * H;
      scale = (uint8_t*)dynamic_scales + row * cols;
    }
    int rc = cqo_quant_row3(c->quant_mode, c->x_dtype, c->y_dtype, H, xr, sm, sm_scalar, codes,
                            scale);
    if (rc != CQO_OK) return rc;
    /* [DV3] expand_scales: the routing weight travels with its row; a shared
     * expert row carries weight 1 (its output is added unweighted). */
    if (expand_scales)
      expand_scales[row] = (k < K) ? (expert_scales ? expert_scales[tok * K + k] : 0.0f) : 1.0f;
  }
  return rows;
}

/* ------------------------------------------------------------------------ */
/* Combine: [DSN] §3.4 (locate each expert output of token i, weighted sum),  */
/* [PERF] Combine 计算步骤 (multiply each MoE output by its expert scale, sum  */
/* in float, then add the shared-expert outputs), [LLD] 特殊专家场景.          */
/* ------------------------------------------------------------------------ */

int cqo_combine_token(const cqo_config* c, int32_t r, int32_t i, const uint16_t* ffn,
                      const int32_t* inv, const float* expert_scales, const uint16_t* ori_x,
                      const float* const_alpha1, const float* const_alpha2,
                      const uint16_t* const_v, int32_t out_f32, void* y_row) {
  const int32_t H = c->hidden, K = c->topk, BS = c->max_bs;
  const int32_t Seff = (c->shared_expert_rank_num > 0) ? c->shared_expert_num : 0;
  const int32_t NS = K + Seff;
  const int64_t tok = (int64_t)r * BS + i;
  const int32_t* slots = inv + tok * NS;
  for (int32_t h = 0; h < H; ++h) {
    float acc = 0.0f;
    /* Routed slots in j order: acc = fma(w_j, v_j, acc). */
    for (int32_t j = 0; j < K; ++j) {
      const int32_t code = slots[j];
      const float w = expert_scales[tok * K + j];
      float v;
      if (code >= 0) {
        v = in16(c->x_dtype, ffn[(int64_t)code * H + h]);
      } else if (code == CQO_INV_COPY) {
        v = in16(c->x_dtype, ori_x[tok * H + h]); /* Moe(ori_x) = ori_x */
      } else if (code <= CQO_INV_CONST_BASE) {
        /* Moe(ori_x) = alpha1 * ori_x + alpha2 * v: two rounded products, one rounded sum. */
        const int32_t q = CQO_INV_CONST_BASE - code;
        const float p1 = const_alpha1[q] * in16(c->x_dtype, ori_x[tok * H + h]);
        const float p2 = const_alpha2[q] * in16(c->x_dtype, const_v[(int64_t)q * H + h]);
        v = p1 + p2;
      } else {
        continue; /* zero expert, masked pair, invalid id: Moe(ori_x) = 0 */
      }
      acc = fmaf(w, v, acc);
    }
    /* Shared experts, added unweighted after the routed ones. */
    for (int32_t s = 0; s < Seff; ++s) {
      const int32_t code = slots[K + s];
      if (code >= 0) acc = acc + in16(c->x_dtype, ffn[(int64_t)code * H + h]);
    }
    if (out_f32) ((float*)y_row)[h] = acc;
    else ((uint16_t*)y_row)[h] = out16(c->x_dtype, acc);
  }
  return CQO_OK;
}

int cqo_combine(const cqo_config* c, const uint16_t* ffn, const int32_t* inv,
                const float* expert_scales, const uint16_t* ori_x, const float* const_alpha1,
                const float* const_alpha2, const uint16_t* const_v, int32_t out_f32, void* y) {
  const int32_t H = c->hidden;
  for (int32_t r = 0; r < c->ep_world_size; ++r) {
    for (int32_t i = 0; i < c->max_bs; ++i) {
      const int64_t tok = (int64_t)r * c->max_bs + i;
      void* yr = out_f32 ? (void*)((float*)y + tok * H) : (void*)((uint16_t*)y + tok * H);
      int rc = cqo_combine_token(c, r, i, ffn, inv, expert_scales, ori_x, const_alpha1,
                                 const_alpha2, const_v, out_f32, yr);
      if (rc != CQO_OK) return rc;
    }
  }
  return CQO_OK;
}

/* ------------------------------------------------------------------------ */
/* Combine-side int8 quantisation, [PERF] 通信前量化 / Int8QuantProcess and   */
/* Int8DequantProcess: before an expert output row is sent back it is cut     */
/* into 32-byte blocks of 8 float values; per block the scale is the largest  */
/* magnitude times 1/SCALE_PARAM (SCALE_PARAM = 127), each value is divided by */
/* the scale and the quotient is cast float -> fp16 -> int8; the receiver     */
/* casts int8 -> fp16 -> float (exact) and multiplies back by the scale.      */
/* The page names the two casts but not their rounding: both are taken as     */
/* round-to-nearest-even, the second one saturating to [-128, 127].           */
/* ------------------------------------------------------------------------ */

int cqo_combine_quant_row(int32_t H, int32_t dt, const uint16_t* row, int8_t* codes,
                          float* scales) {
  if (H % 8 != 0) return CQO_ERR_ARG;
  const float inv_param = 1.0f / 127.0f; /* the constant 1/SCALE_PARAM, rounded once */
  for (int32_t b = 0; b < H / 8; ++b) {
    float m = 0.0f;
    for (int32_t t = 0; t < 8; ++t) {
      float a = fabsf(in16(dt, row[b * 8 + t]));
      if (a > m) m = a;
    }
    const float scale = m * inv_param; /* Muls(1/SCALE_PARAM) */
    for (int32_t t = 0; t < 8; ++t) {
      /* Div, then Cast(float -> fp16 -> int8): the binary32 quotient rounded
       * to binary16 (nearest even; beyond 65504 it becomes infinity), that
       * value rounded to an integer (nearest even) and saturated. 0/0 = NaN
       * stays NaN in fp16 and gives 0. */
      const float q = in16(dt, row[b * 8 + t]) / scale;
      codes[b * 8 + t] = sat_rne_int8(cqo_f16_to_f32(cqo_f16_from_f32(q)));
    }
    scales[b] = scale;
  }
  return CQO_OK;
}

int cqo_combine_token_q8(const cqo_config* c, int32_t r, int32_t i, const int8_t* ffn_codes,
                         const float* ffn_scales, const int32_t* inv, const float* expert_scales,
                         const uint16_t* ori_x, const float* const_alpha1,
                         const float* const_alpha2, const uint16_t* const_v, int32_t out_f32,
                         void* y_row) {
  const int32_t H = c->hidden, K = c->topk, BS = c->max_bs;
  if (H % 8 != 0) return CQO_ERR_ARG;
  const int32_t Seff = (c->shared_expert_rank_num > 0) ? c->shared_expert_num : 0;
  const int32_t NS = K + Seff;
  const int64_t tok = (int64_t)r * BS + i;
  const int32_t* slots = inv + tok * NS;
  for (int32_t h = 0; h < H; ++h) {
    float acc = 0.0f;
    for (int32_t j = 0; j < K; ++j) {
      const int32_t code = slots[j];
      const float w = expert_scales[tok * K + j];
      float v;
      if (code >= 0) {
        /* received row: dequantise first (int8 value times its block scale) */
        v = (float)ffn_codes[(int64_t)code * H + h] * ffn_scales[(int64_t)code * (H / 8) + h / 8];
      } else if (code == CQO_INV_COPY) {
        v = in16(c->x_dtype, ori_x[tok * H + h]);
      } else if (code <= CQO_INV_CONST_BASE) {
        const int32_t q = CQO_INV_CONST_BASE - code;
        const float p1 = const_alpha1[q] * in16(c->x_dtype, ori_x[tok * H + h]);
        const float p2 = const_alpha2[q] * in16(c->x_dtype, const_v[(int64_t)q * H + h]);
        v = p1 + p2;
      } else {
        continue;
      }
      acc = fmaf(w, v, acc);
    }
    for (int32_t s = 0; s < Seff; ++s) {
      const int32_t code = slots[K + s];
      if (code >= 0)
        acc = acc + (float)ffn_codes[(int64_t)code * H + h] *
                        ffn_scales[(int64_t)code * (H / 8) + h / 8];
    }
    if (out_f32) ((float*)y_row)[h] = acc;
    else ((uint16_t*)y_row)[h] = out16(c->x_dtype, acc);
  }
  return CQO_OK;
}
