// cq_combine.cu -- inverse permute + top-K weighted sum, and the combine-side
// int8 quantisation of the expert outputs.
//
// The sum for token (r, i) gathers the expert output row of each of its
// slots and adds them in binary32: one fused multiply-add per routed slot in
// slot order, then the shared-expert rows added unweighted, then one rounding
// to the output type. This is the weighted sum of
// "MoeDistributeDispatch和MoeDistributeCombine算子设计介绍" §3.4.2 and of the
// combine steps of "CANN MoE Dispatch/Combine 通信算子性能优化实践" (multiply by
// expert scale, sum in float, add the shared expert output, cast back), with
// the special experts of "low_latency_dispatch" 特殊专家场景. Token, expert
// output and result rows are bf16 or fp16 (the T template parameter).
//
// Three kernels:
// - combine_staged_kernel (16-bit expert outputs): persistent CTAs; a
//   producer warp streams each token's expert rows into a shared-memory ring
//   with bulk (TMA) loads, consumer warps sum them.
// - combine_kernel (int8 expert outputs + per-8 scales): one CTA per (token,
//   1024 values), each thread gathering its 8 values of a batch of slots.
// - combine_quant_kernel: the expert-side int8 block quantiser.
#include <mutex>

#include "cq_async.cuh"
#include "cq_internal.cuh"

namespace cq {
namespace {

using namespace async;

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

// Two binary32 fused multiply-adds (a * b + c, one rounding each) in one
// packed instruction: each lane is exactly __fmaf_rn of its operands.
__device__ __forceinline__ void fma2(float& c0, float& c1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%0, %1};\n fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Two binary32 products in one packed instruction, each lane rounded to
// nearest even on its own (as two __fmul_rn).
__device__ __forceinline__ void mul2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma8f(float (&acc)[8], float w, const float (&v)[8]) {
#pragma unroll
  for (int t = 0; t < 8; t += 2) fma2(acc[t], acc[t + 1], w, w, v[t], v[t + 1]);
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
    float c[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t word = t < 4 ? it.q.x : it.q.y;
      c[t] = (float)(int)(int8_t)(word >> (8 * (t & 3)));
    }
#pragma unroll
    for (int t = 0; t < 8; t += 2) mul2(f[t], f[t + 1], c[t], c[t + 1], it.s, it.s);
  }
};

// Expert-output rows of the token type (bf16 or fp16), read directly.
template <class T>
struct Src16 {
  const uint16_t* rows;
  struct Item {
    uint4 v;
  };
  __device__ Item load(int64_t row, int H, int u) const {
    return {ld_nc_v4(rows + row * H + 8 * (int64_t)u)};
  }
  __device__ void floats(const Item& it, float (&f)[8]) const { unpack8<T>(it.v, f); }
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

// ---------------------------------------------------------------------------
// Combine from 16-bit expert rows with staged gathers. Persistent CTAs (one
// wave) take tokens blockIdx.x, blockIdx.x + gridDim.x, ... One producer
// warp walks the same (token, slot) sequence as the consumers and streams
// every dispatched row it meets into a ring of shared-memory slots with bulk
// (TMA) loads, running up to the ring size ahead (a full and an empty
// mbarrier per slot). The consumer warps sum the rows from shared memory in
// slot order, exactly as combine_kernel does; copy and const slots read
// ori_x / const_v directly. Every wait gives up after about a second
// (CQ_ST_TIMEOUT) and the producer then waits (bounded again) for its loads
// in flight before the CTA ends.
constexpr int kRingMax = 16;

// Sticky status of the combine kernels of this device (CQ_ST_* bits), read
// and cleared by cq_read_combine_status; a call given a workspace reports to
// that workspace's status word instead.
__device__ uint32_t g_combine_status;

constexpr int kUnitsPerThread = 2;  // 8-element units per consumer thread

// Slot k's inverse-map code `code`, with the consistency guard of
// combine_kernel (a row outside the buffer, a const index outside [0, Q), or
// a special code on a shared slot counts as "no row").
__device__ __forceinline__ int guard_code(const Dims& d, int code, int k) {
  const bool bad_row = code >= 0 && (int64_t)code >= d.R_max;
  const bool bad_const =
      code <= CQ_INV_CONST_BASE && (CQ_INV_CONST_BASE - code >= d.Q || k >= d.K);
  const bool bad_copy = code == CQ_INV_COPY && (d.C == 0 || k >= d.K);
  return (bad_row || bad_const || bad_copy) ? CQ_INV_NONE : code;
}

// Lane k's raw slot code of token tok (CQ_INV_NONE past NS or past the last
// token): loaded one token ahead, guarded when used.
__device__ __forceinline__ int raw_code(const CombineArgs& a, int tok, int n_tok, int k) {
  return (tok < n_tok && k < a.d.NS) ? __ldg(a.inv + (int64_t)tok * a.d.NS + k) : CQ_INV_NONE;
}

// Position in a ring of nslots slots: the slot and the parity of the lap
// (the mbarrier phase a wait on that slot names). Advanced by one per
// streamed row, with no division.
struct RingPos {
  int slot = 0;
  uint32_t lap = 0;
  __device__ __forceinline__ void next(int nslots) {
    if (++slot == nslots) {
      slot = 0;
      lap ^= 1u;
    }
  }
};

// Work item = (token, column chunk of `cw` elements); item i is token
// i / nchunk, chunk i % nchunk. CTA b takes items b, b + gridDim.x, ...
// (fewer than 2^31 items: W * BS * nchunk <= 768 * 512 * 2).
template <class T, bool OUT_F32>
__global__ void __launch_bounds__(288) combine_staged_kernel(CombineArgs a, int nslots, int nchunk,
                                                            int cw) {
  extern __shared__ __align__(128) uint8_t s_ring[];  // nslots chunks of 2*cw bytes
  __shared__ uint64_t s_full[kRingMax];
  __shared__ uint64_t s_empty[kRingMax];
  __shared__ volatile int s_fail;

  const Dims& d = a.d;
  const int H = d.H;
  const uint32_t slot_bytes = 2u * (uint32_t)cw;
  uint32_t* const st_word = a.status ? a.status : &g_combine_status;
  const int ncons = (int)blockDim.x - 32;  // consumer threads
  const int nwc = ncons >> 5;              // consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tok = d.W * d.BS;
  const int n_items = n_tok * nchunk;
  const unsigned uchunk = (unsigned)nchunk;
  auto token_of = [&](int it) { return (int)((unsigned)it / uchunk); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], (uint32_t)nwc);
    }
    mbar_fence_init();
    s_fail = 0;
  }
  __syncthreads();
  griddep_wait();  // the inverse map and the expert rows come from earlier kernels

  if (warp == nwc) {
    // Producer warp: lane 0 issues; the warp reads each item's slot codes.
    int issued = 0;
    RingPos pos;
    bool ok = true;
    int next = raw_code(a, token_of(blockIdx.x), n_tok, lane);
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int tok = token_of(it);
      const int c0 = (it - tok * nchunk) * cw;
      const uint32_t bytes = 2u * (uint32_t)min(cw, H - c0);
      const int code = guard_code(d, next, lane);
      next = raw_code(a, token_of(it + gridDim.x), n_tok, lane);
      for (int k = 0; k < d.NS; ++k) {
        const int ck = __shfl_sync(0xffffffffu, code, k);
        if (ck < 0) continue;
        if (lane == 0) {
          // the slot's previous row (one lap earlier) must have been consumed
          if (issued >= nslots && !mbar_wait(&s_empty[pos.slot], pos.lap ^ 1u)) {
            s_fail = 1;
            atomicOr(st_word, (uint32_t)CQ_ST_TIMEOUT);
          }
          if (!s_fail) {
            mbar_arrive_expect_tx(&s_full[pos.slot], bytes);
            bulk_load(s_ring + (size_t)pos.slot * slot_bytes, a.ffn + (int64_t)ck * H + c0,
                      bytes, &s_full[pos.slot]);
            ++issued;
            pos.next(nslots);
          }
        }
        ok = __shfl_sync(0xffffffffu, s_fail, 0) == 0;
        if (!ok) break;
      }
    }
    // Wait (bounded) for the last loads to land before this warp ends, so
    // that no copy is in flight once the consumers are gone.
    if (lane == 0)
      for (int i = issued > nslots ? issued - nslots : 0; i < issued; ++i)
        mbar_wait(&s_full[i % nslots], (uint32_t)(i / nslots) & 1u);
    return;
  }

  // Consumer warps.
  RingPos pos;
  auto raw_w = [&](int t) {
    return (t < n_tok && lane < d.K) ? __ldg(a.expert_scales + (int64_t)t * d.K + lane) : 1.f;
  };
  int next = raw_code(a, token_of(blockIdx.x), n_tok, lane);
  float next_w = raw_w(token_of(blockIdx.x));
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int tok = token_of(it);
    const int c0 = (it - tok * nchunk) * cw;
    const int cu = min(cw, H - c0) >> 3;  // 8-element units in this chunk
    const int code = guard_code(d, next, lane);
    const float wl = next_w;
    const int tok_next = token_of(it + gridDim.x);
    next = raw_code(a, tok_next, n_tok, lane);
    next_w = raw_w(tok_next);
    float acc[kUnitsPerThread][8];
#pragma unroll
    for (int i = 0; i < kUnitsPerThread; ++i)
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[i][t] = 0.f;
    const int64_t tok_h = (int64_t)tok * H;
    const uint16_t* xrow = a.ori_x ? a.ori_x + tok_h + c0 : nullptr;
    for (int k = 0; k < d.NS; ++k) {
      const int ck = __shfl_sync(0xffffffffu, code, k);
      const float w = __shfl_sync(0xffffffffu, wl, k);
      if (ck >= 0) {
        // The whole warp leaves together if any lane gave up.
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[pos.slot], pos.lap))) {
          s_fail = 1;
          if (lane == 0) atomicOr(st_word, (uint32_t)CQ_ST_TIMEOUT);
          return;
        }
        const uint8_t* rowp = s_ring + (size_t)pos.slot * slot_bytes;
#pragma unroll
        for (int i = 0; i < kUnitsPerThread; ++i) {
          const int u = threadIdx.x + i * ncons;
          if (u < cu) {
            float f[8];
            unpack8<T>(ld_shared_v4(rowp + 16 * u), f);
            if (k < d.K) {
              fma8f(acc[i], w, f);
            } else {
              add8f(acc[i], f);  // shared-expert rows: added unweighted
            }
          }
        }
        release_slot(&s_empty[pos.slot]);
        pos.next(nslots);
      } else if (ck == CQ_INV_COPY || ck <= CQ_INV_CONST_BASE) {
#pragma unroll
        for (int i = 0; i < kUnitsPerThread; ++i) {
          const int u = threadIdx.x + i * ncons;
          if (u < cu) {
            const int col = 8 * u;
            if (ck == CQ_INV_COPY) {
              float f[8];
              unpack8<T>(ld_nc_v4(xrow + col), f);  // Moe(ori_x) = ori_x
              fma8f(acc[i], w, f);
            } else {
              const int cc = CQ_INV_CONST_BASE - ck;
              fma8_const<T>(acc[i], w, a.alpha1[cc], a.alpha2[cc], ld_nc_v4(xrow + col),
                            ld_nc_v4(a.const_v + (int64_t)cc * H + c0 + col));
            }
          }
        }
      }
      // CQ_INV_NONE: zero expert, masked pair or inactive token adds nothing.
    }
#pragma unroll
    for (int i = 0; i < kUnitsPerThread; ++i) {
      const int u = threadIdx.x + i * ncons;
      if (u < cu) store8<T, OUT_F32>(a.y, tok_h + c0 + 8 * u, acc[i]);
    }
  }
}

// Combine-side int8 quantisation of the expert outputs before they are sent
// back ("CANN MoE Dispatch/Combine 通信算子性能优化实践", Int8QuantProcess):
// per block of 8 values, scale = max|v| * fl(1/127), and the quotient
// v / scale cast float -> fp16 -> int8, each cast to nearest even, the int8
// one saturating.
// One wave of CTAs; CTA b takes rows b, b + gridDim.x, ... below the
// dispatched total, each thread up to kQUnits 8-element units of the row with
// all its loads issued before the first division.
constexpr int kQThreads = 256;
constexpr int kQUnits = 4;  // kQThreads * kQUnits * 8 >= the largest H (8192)

// fl(v / s) from y = RN(1 / s) by Markstein's correction step: q0 = RN(v*y),
// the remainder r = v - s*q0 exact in one fused multiply-add, then
// RN(q0 + r*y). For a normal s and no overflow this is the correctly rounded
// quotient (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990); the tests
// compare it with IEEE division on every bf16 mantissa pair at every exponent
// offset that can round to a non-zero code. A zero or infinite s gives NaN
// or 0 exactly where v / s does.
__device__ __forceinline__ float div_by(float v, float s, float y) {
  const float q0 = __fmul_rn(v, y);
  return __fmaf_rn(__fmaf_rn(-s, q0, v), y, q0);
}

// fl(v / s) for a block whose scale s is normal or infinite, or whose max is
// 0 (y = RN(1 / s)): every quotient is then NaN or lies in [-128, 128], and
// max(q, -256) maps NaN (0/0, inf/inf) to -256.
__device__ __forceinline__ float q_div(float v, float s, float y) {
  return fmaxf(div_by(v, s, y), -256.f);
}

// The page's cast chain float -> fp16 -> int8 for two quotients in
// [-256, 128]: cvt.rn.f16x2.f32 rounds each to the nearest binary16 (ties to
// even); adding 1536 = 1.5 * 2^10 in binary16 rounds the sum to an integer
// (the spacing is 1 in [1024, 2048)), so the low byte of each 16-bit sum is
// the nearest-even integer of the binary16 value in two's complement (-256
// gives 0). Byte 0 holds lo's code, byte 2 hi's.
__device__ __forceinline__ uint32_t q8x2_via_f16(float lo, float hi) {
  uint32_t h, r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x66006600u));
  return r;
}

template <class T>
__global__ void __launch_bounds__(kQThreads) combine_quant_kernel(CombineArgs a) {
  griddep_wait();  // the rows may come from the preceding kernel
  const Dims& d = a.d;
  const int H = d.H;
  const int units = H >> 3;
  int64_t total = *a.total_rows;
  if (total > d.R_max) total = d.R_max;  // never read or write past the buffers
  for (int64_t row = blockIdx.x; row < total; row += gridDim.x) {
    uint4 v[kQUnits];
#pragma unroll
    for (int i = 0; i < kQUnits; ++i) {
      const int u = threadIdx.x + i * kQThreads;
      if (u < units) v[i] = ld_nc_v4(a.ffn + row * H + 8 * (int64_t)u);
    }
#pragma unroll
    for (int i = 0; i < kQUnits; ++i) {
      const int u = threadIdx.x + i * kQThreads;
      if (u >= units) continue;
      float f[8];
      unpack8<T>(v[i], f);
      float m = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) m = fmaxf(m, fabsf(f[t]));
      const float s = __fmul_rn(m, __fdiv_rn(1.f, 127.f));
      uint32_t w[2];
      if (m == 0.f || s >= 1.17549435e-38f) {
        const float y = __frcp_rn(s);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          w[h] = __byte_perm(
              q8x2_via_f16(q_div(f[4 * h], s, y), q_div(f[4 * h + 1], s, y)),
              q8x2_via_f16(q_div(f[4 * h + 2], s, y), q_div(f[4 * h + 3], s, y)), 0x6420);
      } else {
        // A subnormal or zero scale of a non-zero block: quotients may leave
        // the int8 range (beyond 65504 the fp16 value is infinite) and
        // saturate.
        w[0] = w[1] = 0u;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          int c = __float2int_rn(__half2float(__float2half_rn(__fdiv_rn(f[t], s))));
          c = max(-128, min(127, c));
          w[t >> 2] |= ((uint32_t)c & 0xffu) << (8 * (t & 3));
        }
      }
      int8_t* dst = a.ffn_q + row * H + 8 * (int64_t)u;
      asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(dst), "r"(w[0]), "r"(w[1]) : "memory");
      a.ffn_scales[row * units + u] = s;
    }
  }
}

// Column chunks of at most kChunkCols elements; a ring of at most
// kRingBytes (several CTAs per SM), 2..kRingMax chunks; one CTA per item
// (kPersistent false) or one wave of CTAs looping over the items.
constexpr int kChunkCols = 4096;
// Below this many work items per SM the direct gathers beat the staged
// ring (measured: 512 items on 152 SMs direct by 0.8-1.7 us, 1024 staged by
// up to 1.5 us, on the performance-table, special and DSV3 shapes).
constexpr int kDirectItemsPerSm = 5;
constexpr size_t kRingBytes = 36u << 10;
constexpr bool kPersistent = true;

template <class T, bool OUT_F32>
cudaError_t launch_staged(const CombineArgs& a, cudaStream_t s) {
  const int H = a.d.H;
  const int nchunk = (H + kChunkCols - 1) / kChunkCols;
  const int cw = ((H + nchunk - 1) / nchunk + 7) / 8 * 8;
  const int per = (cw / 8 + kUnitsPerThread - 1) / kUnitsPerThread;
  const int ncons = (per + 31) / 32 * 32;
  const int threads = ncons + 32;
  const size_t slot_bytes = 2 * (size_t)cw;
  int nslots = (int)(kRingBytes / slot_bytes);
  if (nslots > kRingMax) nslots = kRingMax;
  if (nslots < 2) nslots = 2;
  const size_t smem = (size_t)nslots * slot_bytes;
  auto* kern = combine_staged_kernel<T, OUT_F32>;
  cudaError_t e = prepare_kernel<combine_staged_kernel<T, OUT_F32>>(smem);
  if (e != cudaSuccess) return e;
  int blocks = 0;
  if ((e = occupancy_blocks<combine_staged_kernel<T, OUT_F32>>(threads, smem, &blocks)) !=
      cudaSuccess)
    return e;
  const int n_sm = sm_count();
  if (blocks < 1 || n_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t items = (int64_t)a.d.W * a.d.BS * nchunk;
  int64_t grid = kPersistent ? (int64_t)n_sm * blocks : items;
  if (grid > items) grid = items;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(threads), smem, s, a, nslots, nchunk, cw);
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

// A batch of fewer than kDirectItemsPerSm work items per SM runs one CTA per
// (token, 1024 columns) instead of the staged ring, each thread loading its
// unit of every routed row at once (one round trip instead of the ring's
// laps). Both sum in the same order.
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  const int64_t items = (int64_t)a.d.W * a.d.BS * ((a.d.H + kChunkCols - 1) / kChunkCols);
  if (items < (int64_t)kDirectItemsPerSm * sm_count()) {
    if (a.d.x_dtype == 1) return launch_combine_t<F16>(a, Src16<F16>{a.ffn}, s);
    return launch_combine_t<BF16>(a, Src16<BF16>{a.ffn}, s);
  }
  if (a.d.x_dtype == 1)
    return a.out_f32 ? launch_staged<F16, true>(a, s) : launch_staged<F16, false>(a, s);
  return a.out_f32 ? launch_staged<BF16, true>(a, s) : launch_staged<BF16, false>(a, s);
}

cudaError_t read_combine_status(uint32_t* status, cudaStream_t s) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_combine_status, sizeof(v), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_combine_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *status = v;
  return e;
}

cudaError_t launch_combine_q8(const CombineArgs& a, cudaStream_t s) {
  const SrcQ8 src{a.ffn_q, a.ffn_scales};
  if (a.d.x_dtype == 1) return launch_combine_t<F16>(a, src, s);
  return launch_combine_t<BF16>(a, src, s);
}

cudaError_t launch_combine_quant(const CombineArgs& a, cudaStream_t s) {
  int blocks_per_sm = 0;  // the kernels' occupancy (the same for both types)
  const cudaError_t e = occupancy_blocks<combine_quant_kernel<BF16>>(kQThreads, 0, &blocks_per_sm);
  if (e != cudaSuccess) return e;
  if (blocks_per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)sm_count() * blocks_per_sm;
  if (grid > a.d.R_max) grid = a.d.R_max;
  if (grid < 1) grid = 1;
  if (a.d.x_dtype == 1)
    return launch_pdl(combine_quant_kernel<F16>, dim3((unsigned)grid), dim3(kQThreads), 0, s, a);
  return launch_pdl(combine_quant_kernel<BF16>, dim3((unsigned)grid), dim3(kQThreads), 0, s, a);
}

}  // namespace cq
