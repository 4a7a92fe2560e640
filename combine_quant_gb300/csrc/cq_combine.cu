// cq_combine.cu -- inverse permute + top-K weighted sum.
//
// One CTA per (token, 1024-element chunk). The slot table of the token (row
// of each expert output, or a zero / copy / const code) is read into shared
// memory; every thread then owns one 8-element unit of the chunk, gathers the
// expert rows with 128-bit loads (a batch of 8 routed slots issued before the
// first multiply, so 8 loads are in flight per thread), and sums
// in binary32: one fused multiply-add per routed slot in slot order, then the
// shared-expert rows added unweighted, then one rounding to the output type.
// This is the weighted sum of "MoeDistributeDispatch和MoeDistributeCombine
// 算子设计介绍" §3.4.2 and of the combine steps of "CANN MoE Dispatch/Combine
// 通信算子性能优化实践" (multiply by expert scale, sum in float, add the shared
// expert output, cast back), with the special experts of "low_latency_dispatch"
// 特殊专家场景.
#include <cuda_bf16.h>

#include "cq_internal.cuh"

namespace cq {
namespace {

constexpr int kMaxSlots = 32;
constexpr int kBatch = 8;  // routed slots whose rows are loaded together

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    acc[2 * t] = __fmaf_rn(w, bf_lo(p[t]), acc[2 * t]);
    acc[2 * t + 1] = __fmaf_rn(w, bf_hi(p[t]), acc[2 * t + 1]);
  }
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4& v) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    acc[2 * t] = __fadd_rn(acc[2 * t], bf_lo(p[t]));
    acc[2 * t + 1] = __fadd_rn(acc[2 * t + 1], bf_hi(p[t]));
  }
}

// const expert: acc += w * (a1 * x + a2 * v), each product and the sum rounded.
__device__ __forceinline__ void fma8_const(float (&acc)[8], float w, float a1, float a2,
                                           const uint4& x, const uint4& v) {
  const uint32_t* px = reinterpret_cast<const uint32_t*>(&x);
  const uint32_t* pv = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float t0 = __fadd_rn(__fmul_rn(a1, bf_lo(px[t])), __fmul_rn(a2, bf_lo(pv[t])));
    const float t1 = __fadd_rn(__fmul_rn(a1, bf_hi(px[t])), __fmul_rn(a2, bf_hi(pv[t])));
    acc[2 * t] = __fmaf_rn(w, t0, acc[2 * t]);
    acc[2 * t + 1] = __fmaf_rn(w, t1, acc[2 * t + 1]);
  }
}

template <bool OUT_F32>
__device__ __forceinline__ void store8(void* y, int64_t elem, const float (&acc)[8]) {
  if (OUT_F32) {
    float* p = static_cast<float*>(y) + elem;
    st_v4(p, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                        __float_as_uint(acc[2]), __float_as_uint(acc[3])));
    st_v4(p + 4, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                            __float_as_uint(acc[6]), __float_as_uint(acc[7])));
  } else {
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * t], acc[2 * t + 1]);
      o[t] = *reinterpret_cast<const uint32_t*>(&b);
    }
    st_v4(static_cast<uint16_t*>(y) + elem, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// One CTA per (token, chunk of kThreads 8-element units); one unit per thread.
constexpr int kThreads = 128;

template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads) combine_kernel(CombineArgs a, int nchunk) {
  __shared__ int s_code[kMaxSlots];
  __shared__ float s_w[kMaxSlots];

  const Dims& d = a.d;
  const int64_t tok = blockIdx.x / nchunk;
  const int chunk = blockIdx.x - (int)(tok * nchunk);
  griddep_wait();  // the inverse map comes from the permute kernel
  if (threadIdx.x < d.NS) {
    const int k = threadIdx.x;
    int code = a.inv[tok * d.NS + k];
    // Consistency guard: a row outside the buffer, a const index outside
    // [0, Q), or a special code on a shared slot is treated as "no row".
    const bool bad_row = code >= 0 && (int64_t)code >= d.R_max;
    const bool bad_const =
        code <= CQ_INV_CONST_BASE && (CQ_INV_CONST_BASE - code >= d.Q || k >= d.K);
    const bool bad_copy = code == CQ_INV_COPY && (d.C == 0 || k >= d.K);
    if (bad_row || bad_const || bad_copy) code = CQ_INV_NONE;
    s_code[k] = code;
    s_w[k] = k < d.K ? a.expert_scales[tok * d.K + k] : 1.f;
  }
  __syncthreads();

  const int H = d.H;
  const int u = chunk * kThreads + threadIdx.x;
  if (u >= (H >> 3)) return;
  float acc[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t] = 0.f;

  const int64_t col = 8 * (int64_t)u;
  const uint16_t* xrow = a.ori_x ? a.ori_x + tok * H : nullptr;

  for (int k0 = 0; k0 < d.K; k0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = k0 + b;
      const int code = k < d.K ? s_code[k] : CQ_INV_NONE;
      const uint16_t* src = nullptr;
      if (code >= 0) src = a.ffn + (int64_t)code * H;
      else if (code == CQ_INV_COPY) src = xrow;
      v[b] = src ? ld_nc_v4(src + col) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = k0 + b;
      if (k >= d.K) break;
      const int code = s_code[k];
      const float w = s_w[k];
      if (code >= 0 || code == CQ_INV_COPY) {
        fma8(acc, w, v[b]);
      } else if (code <= CQ_INV_CONST_BASE) {
        const int c = CQ_INV_CONST_BASE - code;
        fma8_const(acc, w, a.alpha1[c], a.alpha2[c], ld_nc_v4(xrow + col),
                   ld_nc_v4(a.const_v + (int64_t)c * H + col));
      }
      // CQ_INV_NONE: zero expert, masked pair or inactive token adds nothing.
    }
  }
  for (int k = d.K; k < d.NS; ++k) {
    const int code = s_code[k];
    if (code >= 0) add8(acc, ld_nc_v4(a.ffn + (int64_t)code * H + col));
  }
  store8<OUT_F32>(a.y, tok * H + col, acc);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  const int units = a.d.H >> 3;
  const int nchunk = (units + kThreads - 1) / kThreads;
  const int64_t grid = (int64_t)a.d.W * a.d.BS * nchunk;
  if (a.out_f32)
    return launch_pdl(combine_kernel<true>, dim3((unsigned)grid), dim3(kThreads), 0, s, a, nchunk);
  return launch_pdl(combine_kernel<false>, dim3((unsigned)grid), dim3(kThreads), 0, s, a, nchunk);
}

}  // namespace cq
