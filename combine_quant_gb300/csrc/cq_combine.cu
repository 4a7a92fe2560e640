// cq_combine.cu -- inverse permute + top-K weighted sum, and the combine-side
// int8 quantisation of the expert outputs.
//
// One CTA per (token, 1024-element chunk). The slot table of the token (row
// of each expert output, or a zero / copy / const code) is read into shared
// memory; every thread then owns one 8-element unit of the chunk, gathers the
// expert rows with vector loads (a batch of 8 routed slots issued before the
// first multiply), and sums in binary32: one fused multiply-add per routed
// slot in slot order, then the shared-expert rows added unweighted, then one
// rounding to the output type. This is the weighted sum of
// "MoeDistributeDispatch和MoeDistributeCombine算子设计介绍" §3.4.2 and of the
// combine steps of "CANN MoE Dispatch/Combine 通信算子性能优化实践" (multiply by
// expert scale, sum in float, add the shared expert output, cast back), with
// the special experts of "low_latency_dispatch" 特殊专家场景. Token, expert
// output and result rows are bf16 or fp16 (the T template parameter).
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

__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ float ld_nc_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// 8 fp32 values of an 8-element unit of 16-bit values.
template <class T>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    f[2 * t] = T::lo(p[t]);
    f[2 * t + 1] = T::hi(p[t]);
  }
}

__device__ __forceinline__ void fma8f(float (&acc)[8], float w, const float (&v)[8]) {
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t] = __fmaf_rn(w, v[t], acc[t]);
}

__device__ __forceinline__ void add8f(float (&acc)[8], const float (&v)[8]) {
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t] = __fadd_rn(acc[t], v[t]);
}

// const expert: acc += w * (a1 * x + a2 * v), each product and the sum rounded.
template <class T>
__device__ __forceinline__ void fma8_const(float (&acc)[8], float w, float a1, float a2,
                                           const uint4& x, const uint4& v) {
  float fx[8], fv[8];
  unpack8<T>(x, fx);
  unpack8<T>(v, fv);
#pragma unroll
  for (int t = 0; t < 8; ++t)
    acc[t] = __fmaf_rn(w, __fadd_rn(__fmul_rn(a1, fx[t]), __fmul_rn(a2, fv[t])), acc[t]);
}

template <class T, bool OUT_F32>
__device__ __forceinline__ void store8(void* y, int64_t elem, const float (&acc)[8]) {
  if (OUT_F32) {
    float* p = static_cast<float*>(y) + elem;
    st_v4(p, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                        __float_as_uint(acc[2]), __float_as_uint(acc[3])));
    st_v4(p + 4, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                            __float_as_uint(acc[6]), __float_as_uint(acc[7])));
  } else {
    st_v4(static_cast<uint16_t*>(y) + elem,
          make_uint4(T::pack2(acc[0], acc[1]), T::pack2(acc[2], acc[3]),
                     T::pack2(acc[4], acc[5]), T::pack2(acc[6], acc[7])));
  }
}

// Expert-output rows as 16-bit values: 8 per 16-byte load.
template <class T>
struct Src16 {
  const uint16_t* ffn;
  struct Item {
    uint4 v;
  };
  __device__ Item load(int64_t row, int H, int u) const {
    return {ld_nc_v4(ffn + row * H + 8 * (int64_t)u)};
  }
  __device__ void floats(const Item& it, float (&f)[8]) const { unpack8<T>(it.v, f); }
};

// Expert-output rows as int8 with one scale per 8 values ("CANN MoE
// Dispatch/Combine 通信算子性能优化实践", Int8DequantProcess): each value is
// dequantised (code times block scale, one rounding) before it is summed.
struct SrcQ8 {
  const int8_t* codes;
  const float* scales;
  struct Item {
    uint2 q;
    float s;
  };
  __device__ Item load(int64_t row, int H, int u) const {
    return {ld_nc_v2(codes + row * H + 8 * (int64_t)u), ld_nc_f32(scales + row * (H >> 3) + u)};
  }
  __device__ void floats(const Item& it, float (&f)[8]) const {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t word = t < 4 ? it.q.x : it.q.y;
      const int c = (int)(int8_t)(word >> (8 * (t & 3)));
      f[t] = __fmul_rn((float)c, it.s);
    }
  }
};

// One CTA per (token, chunk of kThreads 8-element units); one unit per thread.
constexpr int kThreads = 128;

template <class T, bool OUT_F32, class Src>
__global__ void __launch_bounds__(kThreads) combine_kernel(CombineArgs a, Src src, int nchunk) {
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
    // Issue the loads of a batch of routed rows before the first multiply.
    typename Src::Item v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = k0 + b;
      const int code = k < d.K ? s_code[k] : CQ_INV_NONE;
      if (code >= 0) v[b] = src.load(code, H, u);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = k0 + b;
      if (k >= d.K) break;
      const int code = s_code[k];
      const float w = s_w[k];
      if (code >= 0) {
        float f[8];
        src.floats(v[b], f);
        fma8f(acc, w, f);
      } else if (code == CQ_INV_COPY) {
        float f[8];
        unpack8<T>(ld_nc_v4(xrow + col), f);  // Moe(ori_x) = ori_x
        fma8f(acc, w, f);
      } else if (code <= CQ_INV_CONST_BASE) {
        const int c = CQ_INV_CONST_BASE - code;
        fma8_const<T>(acc, w, a.alpha1[c], a.alpha2[c], ld_nc_v4(xrow + col),
                      ld_nc_v4(a.const_v + (int64_t)c * H + col));
      }
      // CQ_INV_NONE: zero expert, masked pair or inactive token adds nothing.
    }
  }
  for (int k = d.K; k < d.NS; ++k) {
    const int code = s_code[k];
    if (code >= 0) {
      float f[8];
      src.floats(src.load(code, H, u), f);
      add8f(acc, f);
    }
  }
  store8<T, OUT_F32>(a.y, tok * H + col, acc);
}

// Combine-side int8 quantisation of the expert outputs before they are sent
// back ("CANN MoE Dispatch/Combine 通信算子性能优化实践", Int8QuantProcess):
// per block of 8 values, scale = max|v| * fl(1/127), code = RNE(v / scale).
// One CTA per (row, chunk); rows past the dispatched total are skipped.
template <class T>
__global__ void __launch_bounds__(kThreads) combine_quant_kernel(CombineArgs a, int nchunk) {
  griddep_wait();  // the rows may come from the preceding kernel
  const Dims& d = a.d;
  const int64_t row = blockIdx.x / nchunk;
  const int chunk = blockIdx.x - (int)(row * nchunk);
  if (row >= (int64_t)*a.total_rows) return;
  const int H = d.H;
  const int u = chunk * kThreads + threadIdx.x;
  if (u >= (H >> 3)) return;
  float f[8];
  unpack8<T>(ld_nc_v4(a.ffn + row * H + 8 * (int64_t)u), f);
  float m = 0.f;
#pragma unroll
  for (int t = 0; t < 8; ++t) m = fmaxf(m, fabsf(f[t]));
  const float s = __fmul_rn(m, __fdiv_rn(1.f, 127.f));
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    int c = __float2int_rn(__fdiv_rn(f[t], s));  // 0/0 is NaN, which converts to 0
    c = max(-128, min(127, c));
    w[t >> 2] |= ((uint32_t)c & 0xffu) << (8 * (t & 3));
  }
  int8_t* dst = a.ffn_q + row * H + 8 * (int64_t)u;
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(dst), "r"(w[0]), "r"(w[1]) : "memory");
  a.ffn_scales[row * (H >> 3) + u] = s;
}

template <class T, class Src>
cudaError_t launch_combine_t(const CombineArgs& a, const Src& src, cudaStream_t s) {
  const int units = a.d.H >> 3;
  const int nchunk = (units + kThreads - 1) / kThreads;
  const dim3 grid((unsigned)((int64_t)a.d.W * a.d.BS * nchunk));
  if (a.out_f32)
    return launch_pdl(combine_kernel<T, true, Src>, grid, dim3(kThreads), 0, s, a, src, nchunk);
  return launch_pdl(combine_kernel<T, false, Src>, grid, dim3(kThreads), 0, s, a, src, nchunk);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.d.x_dtype == 1) return launch_combine_t<F16>(a, Src16<F16>{a.ffn}, s);
  return launch_combine_t<BF16>(a, Src16<BF16>{a.ffn}, s);
}

cudaError_t launch_combine_q8(const CombineArgs& a, cudaStream_t s) {
  const SrcQ8 src{a.ffn_q, a.ffn_scales};
  if (a.d.x_dtype == 1) return launch_combine_t<F16>(a, src, s);
  return launch_combine_t<BF16>(a, src, s);
}

cudaError_t launch_combine_quant(const CombineArgs& a, cudaStream_t s) {
  const int units = a.d.H >> 3;
  const int nchunk = (units + kThreads - 1) / kThreads;
  const dim3 grid((unsigned)(a.d.R_max * nchunk));
  if (a.d.x_dtype == 1)
    return launch_pdl(combine_quant_kernel<F16>, grid, dim3(kThreads), 0, s, a, nchunk);
  return launch_pdl(combine_quant_kernel<BF16>, grid, dim3(kThreads), 0, s, a, nchunk);
}

}  // namespace cq
