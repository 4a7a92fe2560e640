// cq_permute_impl.cuh -- fused gather-quantise-scatter (MoePermute + pre-send
// quantisation), templated on the 16-bit token type; instantiated for bf16
// and fp16 by cq_permute_bf16.cu / cq_permute_f16.cu.
//
// permute_kernel: one CTA per source token (r, i). Warp 0 turns each slot's arrival ordinal
// into its global row (rank base + first row of the (expert slot, source,
// chunk of the source's tokens) block within the rank + ordinal within the
// chunk: the address rule of "MoeDistributeDispatch和MoeDistributeCombine算子
// 设计介绍" §3.4.2 with the source block folded into the expert offset),
// writes the inverse map, the (src, token, slot) row record and
// the carried weight. All threads load the token row once with 128-bit loads
// (started before the routing kernels finish), quantise it in registers and
// stage the code row in shared memory; one thread then writes it to every
// routed row with bulk (TMA) stores.
//
// Quantisation ("low_latency_dispatch" 计算公式, [DV3] 功能说明 情形 1 / 情形 2):
//   mode 0  the 16-bit row travels unchanged
//   mode 1  static: int8 = RNE(x * scales)
//   mode 2  per token: s = 127 / max|x*scales|, int8 = RNE(x*scales * s), carry 1/s
//   mode 3  per 128-group: s = F / max|x*scales|, fp8 = RNE(x*scales * s), carry 1/s
//   mode 4  mx: per 32-block, e = floor(log2 max|x|) - emax, fp8 of x / 2^e, e8m0 e+127
//   mode 5  mx clip: per 32-block, e = ceil(log2(max(max|x|, 1e-4) / F)), idem
// with fp8 = e4m3fn (F = 448, emax = 8) or e5m2 (F = 57344, emax = 15).
// "scales" (smooth) is one row per expert, one row for all, or one scalar.
// With one smooth row per expert the rows are quantised expert by expert
// instead (index_kernel + smooth_rows_kernel, further down).
// Arithmetic is single IEEE binary32 operations (explicit _rn intrinsics, no
// contraction), so codes and scales are reproducible bit for bit.
// Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
// top of include/cq.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <climits>
#include <mutex>

#include "cq_async.cuh"
#include "cq_internal.cuh"

namespace cq {
namespace permute_detail {

using namespace async;

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxSlots = 32;  // NS <= 16 + 4

using BF16 = cq::BF16;
using F16 = cq::F16;

// Smooth-scale shapes ([LLD] quant_mode 相关约束).
enum SmoothKind { kNoSmooth = 0, kRowPerSlot = 1, kSharedRow = 2, kScalar = 3 };

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_shared_v4(void* p, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(p)),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Bulk (TMA) stores of staged rows: shared memory -> global, issued by one
// thread, completion tracked in bulk groups. Both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> bulk reads
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"((uint32_t)__cvta_generic_to_shared(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Streaming 128-bit global store (written once, not read again here).
__device__ __forceinline__ void st_global_cs_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Round to nearest even, saturate to int8 (a NaN product gives 0).
__device__ __forceinline__ uint32_t q8(float v) {
  int c = __float2int_rn(v);
  c = max(-128, min(127, c));
  return (uint32_t)c & 0xffu;
}

// Two binary32 values to two e4m3 bytes (lo in the low byte), round to
// nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The same into two e5m2 bytes, saturating to +-57344.
__device__ __forceinline__ uint32_t e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantisation variant Q: quant_mode Q % 10; Q >= 10 selects e5m2 codes for
// modes 3-5 (e4m3fn otherwise).
__host__ __device__ constexpr int q_mode(int q) { return q % 10; }
__host__ __device__ constexpr bool q_e5m2(int q) { return q >= 10; }

// Exact ceil(log2(q)) for a positive normal binary32 q.
__device__ __forceinline__ int ceil_log2_bits(float q) {
  const uint32_t b = __float_as_uint(q);
  return (int)((b >> 23) & 0xffu) - 127 + ((b & 0x7fffffu) != 0u ? 1 : 0);
}

// Exact floor(log2(a)) for a positive finite binary32 a (also subnormal).
__device__ __forceinline__ int floor_log2_bits(float a) {
  const uint32_t b = __float_as_uint(a);
  const int ex = (int)((b >> 23) & 0xffu);
  if (ex != 0) return ex - 127;
  const uint32_t m = b & 0x7fffffu;  // a = m * 2^-149
  return (31 - __clz((int)m)) - 149;
}

// 2^k as a binary32, for k in [-126, 127].
__device__ __forceinline__ float pow2(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// max(0, |v_t|) over the 16 values, NaN ignored, as a balanced tree (max is
// exact and associative; the final max with 0 turns an all-NaN unit into 0).
// Three-operand max: NaN operands ignored, or (NAN) propagated.
template <bool NAN_OUT = false>
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  if (NAN_OUT) {
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  } else {
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  }
  return r;
}
// max(0, |v_t|) over 16 values; NaN values are ignored, or (NAN_OUT) make the
// result NaN. Max is exact, so the order of the tree does not matter.
template <bool NAN_OUT = false>
__device__ __forceinline__ float max16(const float (&v)[16]) {
  float m[5];
#pragma unroll
  for (int t = 0; t < 5; ++t)
    m[t] = max3<NAN_OUT>(fabsf(v[3 * t]), fabsf(v[3 * t + 1]), fabsf(v[3 * t + 2]));
  return max3<NAN_OUT>(max3<NAN_OUT>(m[0], m[1], m[2]), max3<NAN_OUT>(m[3], m[4], fabsf(v[15])),
                       0.f);
}

__device__ __forceinline__ uint4 q8_16(const float (&v)[16], float s) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    o[t] = q8(__fmul_rn(v[4 * t], s)) | (q8(__fmul_rn(v[4 * t + 1], s)) << 8) |
           (q8(__fmul_rn(v[4 * t + 2], s)) << 16) | (q8(__fmul_rn(v[4 * t + 3], s)) << 24);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 q8_16_direct(const float (&v)[16]) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    o[t] = q8(v[4 * t]) | (q8(v[4 * t + 1]) << 8) | (q8(v[4 * t + 2]) << 16) |
           (q8(v[4 * t + 3]) << 24);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Two binary32 products in one packed instruction, each lane rounded to
// nearest even on its own (the same results as two scalar _rn products). Use
// only where no packed add follows the product: ptxas may fuse a packed
// multiply and a packed add into one multiply-add with a single rounding
// (a packed fma by 1.0 after it is not merged; a GPU test on rounding ties
// checks that).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// p + 1.5 * 2^23 for both lanes, as a packed fma by 1.0: p * 1 is exact, so
// each lane is the one rounding of the sum, as an add would give.
__device__ __forceinline__ float2 addmagic2(float2 p) {
  float2 r;
  asm("{\n .reg .b64 rp, rm, ro, rd;\n mov.b64 rp, {%2, %3};\n mov.b64 rm, {%4, %4};\n"
      " mov.b64 ro, {%5, %5};\n fma.rn.f32x2 rd, rp, ro, rm;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(p.x), "f"(p.y), "f"(12582912.f), "f"(1.0f));
  return r;
}

// Sixteen int8 codes RNE(fl(v * m)) for products that lie in [-128, 128]:
// adding 1.5 * 2^23 gives a sum whose ulp is 1, so its low mantissa bits
// hold the nearest-even integer n, and the low byte of its bit pattern is n
// in two's complement. Three byte permutes pack four codes.
// The products are packed f32x2 multiplies, each lane rounded on its own;
// the adds are packed fmas by 1.0, which ptxas keeps apart from the products.
// A multiply-add fused from the two would round v * m once, straight to an
// integer, and differ from RNE(fl(v * m)) where fl(v * m) is a tie that the
// exact product is not (a packed multiply followed by a packed add does get
// contracted; a GPU test on rounding ties checks these codes).
__device__ __forceinline__ uint4 q8_16_magic(const float (&v)[16], float m) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 p0 = mul2(make_float2(v[4 * t], v[4 * t + 1]), make_float2(m, m));
    const float2 p1 = mul2(make_float2(v[4 * t + 2], v[4 * t + 3]), make_float2(m, m));
    const float2 s0 = addmagic2(p0), s1 = addmagic2(p1);
    const uint32_t c0 = __float_as_uint(s0.x), c1 = __float_as_uint(s0.y);
    const uint32_t c2 = __float_as_uint(s1.x), c3 = __float_as_uint(s1.y);
    o[t] = __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Sixteen int8 codes RNE(v) for values of magnitude below 127.5 (codes in
// [-127, 127]), by the same add-and-pack.
__device__ __forceinline__ uint4 q8_16_add(const float (&v)[16]) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 s0 = addmagic2(make_float2(v[4 * t], v[4 * t + 1]));
    const float2 s1 = addmagic2(make_float2(v[4 * t + 2], v[4 * t + 3]));
    o[t] = __byte_perm(__byte_perm(__float_as_uint(s0.x), __float_as_uint(s0.y), 0x0040),
                       __byte_perm(__float_as_uint(s1.x), __float_as_uint(s1.y), 0x0040), 0x5410);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool E5>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  return E5 ? e5m2x2(lo, hi) : e4m3x2(lo, hi);
}

template <bool E5>
__device__ __forceinline__ uint4 fp8_16(const float (&v)[16], float mult) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 p0 = mul2(make_float2(v[4 * t], v[4 * t + 1]), make_float2(mult, mult));
    const float2 p1 = mul2(make_float2(v[4 * t + 2], v[4 * t + 3]), make_float2(mult, mult));
    o[t] = fp8x2<E5>(p0.x, p0.y) | (fp8x2<E5>(p1.x, p1.y) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Max over the 32 lanes of a warp of non-negative (or NaN) values: NaN
// propagated (NAN_OUT) or ignored, as in max3.
template <bool NAN_OUT = false>
__device__ __forceinline__ float warp_max(float v) {
  float r;
  if (NAN_OUT) {
    asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  } else {
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  }
  return r;
}

// Max of one non-negative (or NaN) float per thread over the first nt
// threads of the block (NaN-propagating when NAN_OUT); nt is a multiple of
// 32, at most 256 (8 warps). The threads meet at __syncthreads, or (NAMED,
// when other warps of the block do not take part) at named barrier 1. `buf`
// holds >= 8 floats and must not be reused by another block_max until the
// next such barrier.
template <bool NAN_OUT = false, bool NAMED = false>
__device__ __forceinline__ float block_max(float v, float* buf, int nt) {
  v = warp_max<NAN_OUT>(v);
  const int lane = threadIdx.x & 31;
  if (lane == 0) buf[threadIdx.x >> 5] = v;
  if (NAMED) {
    asm volatile("bar.sync 1, %0;" ::"r"(nt) : "memory");
  } else {
    __syncthreads();
  }
  return warp_max<NAN_OUT>(lane < (nt >> 5) ? buf[lane] : 0.f);
}

// Thread-owned part of the token row: two 16-element units (32 bytes each).
struct Units {
  uint4 v[2][2];
  bool ok[2];
};

// fp32 values of one unit, times the smooth scales when given.
template <class T, int SM>
__device__ __forceinline__ void unit_values(const uint4 (&u)[2], const float* srow, float scalar,
                                            int unit, float (&f)[16]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u[0]);
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    f[2 * t] = T::lo(w[t]);
    f[2 * t + 1] = T::hi(w[t]);
  }
  if (SM == kScalar) {
#pragma unroll
    for (int t = 0; t < 16; ++t) f[t] = __fmul_rn(f[t], scalar);
  } else if (SM == kSharedRow) {
    const float* sm = srow + 16 * unit;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 q = ld_nc_v4(sm + 4 * t);
      f[4 * t] = __fmul_rn(f[4 * t], __uint_as_float(q.x));
      f[4 * t + 1] = __fmul_rn(f[4 * t + 1], __uint_as_float(q.y));
      f[4 * t + 2] = __fmul_rn(f[4 * t + 2], __uint_as_float(q.z));
      f[4 * t + 3] = __fmul_rn(f[4 * t + 3], __uint_as_float(q.w));
    }
  }
}

// Quantise this thread's two units of one row: codes at 16 bytes per unit in
// `codes` (shared staging, or the global row when GLOBAL), the per-group (mode 3, floats) or
// per-block (modes 4/5, e8m0 bytes) scales in `scales`. Mode 2 returns the
// row's carried scale in the threads of warp 0. `red` holds 64 floats (mode 2
// only). nt threads share the row; NAMED as for block_max.
// 16 code bytes to shared (staging) or, when GLOBAL, straight to global memory.
template <bool GLOBAL>
__device__ __forceinline__ void put16(uint8_t* p, uint4 v) {
  if (GLOBAL) {
    st_global_cs_v4(p, v);
  } else {
    st_shared_v4(p, v);
  }
}

template <int Q, bool GLOBAL = false, bool NAMED = false>
__device__ __forceinline__ float quantise(const float (&f)[2][16], const Units& U,
                                          uint8_t* codes, uint8_t* scales, float* red, int nt) {
  constexpr int MODE = q_mode(Q);
  constexpr bool E5 = q_e5m2(Q);
  // The fp8 type's largest value and its exponent (emax).
  constexpr float kFp8Max = E5 ? 57344.f : 448.f;
  constexpr int kEmax = E5 ? 15 : 8;
  float carried = 0.f;
  if (MODE == 1) {
    // A thread whose values all lie below 127.5 in magnitude has codes in
    // [-127, 127]: add-and-pack. Any other value (large, infinite, NaN) sends
    // the thread to convert-and-saturate.
    const bool small = max3<true>(max16<true>(f[0]), max16<true>(f[1]), 0.f) < 127.5f;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (U.ok[q])
        put16<GLOBAL>(codes + 16 * (threadIdx.x + q * nt),
                      small ? q8_16_add(f[q]) : q8_16_direct(f[q]));
  } else if (MODE == 2) {
    // The row max with NaN propagated. A row with neither NaN nor infinity
    // whose 127/max is finite (or whose max is 0) has every product x * s in
    // [-127, 127]: add-and-pack rounding. Any other row takes the
    // convert-and-saturate path with the scale from the NaN-ignoring max.
    float amax =
        block_max<true, NAMED>(max3<true>(max16<true>(f[0]), max16<true>(f[1]), 0.f), red, nt);
    const bool clean = amax <= 3.402823466e38f;  // false for NaN and +inf
    if (!clean) amax = block_max<false, NAMED>(fmaxf(max16(f[0]), max16(f[1])), red + 32, nt);
    const float s = __fdiv_rn(127.f, amax);  // +inf for an all-zero row: codes 0, carried 0
    if (threadIdx.x < 32) carried = __fdiv_rn(1.f, s);  // only warp 0 stores it
    if (clean && (s <= 3.402823466e38f || amax == 0.f)) {
      const float mult = amax == 0.f ? 0.f : s;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (U.ok[q]) put16<GLOBAL>(codes + 16 * (threadIdx.x + q * nt), q8_16_magic(f[q], mult));
    } else {
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (U.ok[q]) put16<GLOBAL>(codes + 16 * (threadIdx.x + q * nt), q8_16(f[q], s));
    }
  } else if (MODE == 3) {
    // A 128-group is 8 units held by 8 consecutive lanes.
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float m = max16(f[q]);
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 2));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
      const float s = __fdiv_rn(kFp8Max, m);
      const float mult = m == 0.f ? 0.f : s;  // an all-zero group: codes 0, scale 0
      const int u = threadIdx.x + q * nt;
      if (U.ok[q]) {
        put16<GLOBAL>(codes + 16 * u, fp8_16<E5>(f[q], mult));
        if ((u & 7) == 0) reinterpret_cast<float*>(scales)[u >> 3] = __fdiv_rn(1.f, s);
      }
    }
  } else {
    // mx: a 32-block is 2 units held by lanes 2m, 2m+1.
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float m = max16(f[q]);
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      int e;
      if (MODE == 4) {
        e = m == 0.f ? -127 : max(floor_log2_bits(m) - kEmax, -127);
      } else {
        e = ceil_log2_bits(__fdiv_rn(fmaxf(m, 1e-4f), kFp8Max));
      }
      const int u = threadIdx.x + q * nt;
      if (U.ok[q]) {
        put16<GLOBAL>(codes + 16 * u, fp8_16<E5>(f[q], pow2(-e)));  // x / 2^e, exact scaling
        if ((u & 1) == 0) scales[u >> 1] = (uint8_t)(e + 127);
      }
    }
  }
  return carried;
}

// Slot k of token tok (source rank r): its global row = first row of the
// destination rank + first row of the (expert slot, source) block inside the
// rank + arrival ordinal. Writes the inverse-map entry and, for a dispatched
// slot, the (src, token, slot) row record and the carried weight. `e` is the
// slot's arrival ordinal (eidx), loaded by the caller. Returns the row (-1 if
// none) and the slot's smooth-table row in `srow`.
__device__ __forceinline__ int map_slot(const PermuteArgs& a, int64_t tok, int r, int k, int e,
                                        int& srow) {
  const Dims& d = a.d;
  srow = 0;
  if (k >= d.NS) return -1;
  int code = e, row = -1;
  if (e >= 0) {
    int g, dst;  // global expert slot, destination rank
    if (k < d.K) {
      const int id = a.expert_ids[tok * d.K + k];
      g = d.S_r + id;
      dst = d.S_r + id / d.L;
      srow = d.S_eff + id;
    } else {
      const int s = k - d.K;
      g = dst = s * d.R_rep + r % d.R_rep;  // a shared-expert rank hosts one slot
      srow = s;
    }
    const int i = (int)(tok - (int64_t)r * d.BS);
    row = a.ws.rank_base[dst] + a.ws.local_off[((int64_t)g * d.W + r) * d.CH + i / d.TC] + e;
    if (row < 0 || (int64_t)row >= d.R_max) {  // consistency guard: never write outside
      atomicOr(a.ws.status, (uint32_t)CQ_ST_INTERNAL);
      row = -1;
      code = CQ_INV_NONE;
    } else {
      code = row;
      reinterpret_cast<int4*>(a.assist_rows)[row] = make_int4(r, i, k, 0);
      if (a.expand_scales)
        a.expand_scales[row] =
            k < d.K ? (a.expert_scales ? a.expert_scales[tok * d.K + k] : 0.f) : 1.f;
    }
  }
  a.inv[tok * d.NS + k] = code;
  return row;
}

// Token-major permute for every smooth shape but per-expert rows.
// T: token type; Q: quantisation variant (q_mode, q_e5m2); SM: SmoothKind.
template <class T, int Q, int SM>
__global__ void __launch_bounds__(256) permute_kernel(PermuteArgs a) {
  constexpr int MODE = q_mode(Q);
  __shared__ int s_row[kMaxSlots];   // compact list of routed rows
  __shared__ int s_srow[kMaxSlots];  // their smooth-table rows
  __shared__ int s_nrows;
  __shared__ float s_red[2][64];
  extern __shared__ __align__(128) uint8_t s_stage[];  // staged code row(s) + scale row(s)

  const Dims& d = a.d;
  const int64_t tok = blockIdx.x;
  const int r = (int)(tok / d.BS), i = (int)(tok - (int64_t)r * d.BS);
  const int lane = threadIdx.x & 31;
  const int H = d.H;
  const int units = H >> 4;
  const uint16_t* xrow = a.x + tok * H;

  Units U;
  auto load_row = [&]() {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = threadIdx.x + q * blockDim.x;
      U.ok[q] = u < units;
      if (U.ok[q]) {
        U.v[q][0] = ld_nc_v4(xrow + 16 * u);
        U.v[q][1] = ld_nc_v4(xrow + 16 * u + 8);
      } else {
        U.v[q][0] = U.v[q][1] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // From the inputs alone, could this token be active? If so, start loading
  // its row now: this kernel may be running while the routing kernels end.
  bool prefetched = !a.bs_per_rank || i < a.bs_per_rank[r];
  if (prefetched && a.mask) {
    if (d.mask_ndim == 1) {
      prefetched = a.mask[tok] != 0;
    } else {
      bool any = false;
      for (int j = 0; j < d.K; ++j) any |= a.mask[tok * d.K + j] != 0;
      prefetched = any;
    }
  }
  if (prefetched) load_row();
  griddep_wait();  // routing outputs (ordinals, offsets) are read from here on
  // Warp 0 starts loading the slots' ordinals; the mapping finishes after the
  // row is staged, so its latency overlaps the quantisation.
  const int e_slot = threadIdx.x < 32 && lane < d.NS ? a.ws.eidx[tok * d.NS + lane] : CQ_INV_NONE;

  // Staged row layout: code row (2H bytes in mode 0, else H), then the scale
  // row padded to 16 bytes.
  const int code_bytes = MODE == 0 ? 2 * H : H;
  const int scale_bytes = MODE == 3 ? 4 * d.G3 : ((MODE == 4 || MODE == 5) ? d.SC : 0);
  char* const dyn = static_cast<char*>(a.dynamic_scales);
  char* const out = static_cast<char*>(a.expand_x);

  // The code row (and scale row) every routed row gets, into s_stage; mode 2
  // returns the carried scale in warp 0. All threads take part.
  auto stage = [&]() -> float {
    float carried = 0.f;
    if (MODE == 0) {
      // The 16-bit row itself travels ([DV3] 情形 1).
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * blockDim.x;
        if (U.ok[q]) {
          st_shared_v4(s_stage + 32 * u, U.v[q][0]);
          st_shared_v4(s_stage + 32 * u + 16, U.v[q][1]);
        }
      }
    } else {
      // One quantisation per token: every routed row gets the same codes.
      const float* srow = SM == kSharedRow ? a.smooth : nullptr;
      const float scalar = SM == kScalar ? a.smooth[0] : 0.f;
      float f[2][16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * blockDim.x;
        if (U.ok[q]) {
          unit_values<T, SM>(U.v[q], srow, scalar, u, f[q]);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) f[q][t] = 0.f;
        }
      }
      carried = quantise<Q>(f, U, s_stage, s_stage + code_bytes, s_red[0], blockDim.x);
      if (MODE == 5 || MODE == 4) {
        if (threadIdx.x == 0 && d.SC > (units >> 1)) s_stage[code_bytes + (units >> 1)] = 0;
      }
    }
    fence_proxy_async_smem();  // staging writes before the bulk copies read them
    return carried;
  };

  float carried = 0.f;
  if (prefetched) carried = stage();
  if (threadIdx.x < 32) {
    int srow;
    const int row = map_slot(a, tok, r, lane, e_slot, srow);
    const unsigned bal = __ballot_sync(kFull, row >= 0);
    if (row >= 0) {
      const int pos = __popc(bal & ((1u << lane) - 1u));
      s_row[pos] = row;
      s_srow[pos] = srow;
    }
    if (lane == 0) s_nrows = __popc(bal);
  }
  __syncthreads();
  const int nrows = s_nrows;
  if (nrows == 0) return;
  if (!prefetched) {  // routing found rows the inputs did not predict
    load_row();
    carried = stage();
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    for (int n = 0; n < nrows; ++n) {
      const int64_t row = s_row[n];
      bulk_store(out + row * code_bytes, s_stage, (uint32_t)code_bytes);
      if (scale_bytes && a.scale_rows_bulk)
        bulk_store(dyn + row * scale_bytes, s_stage + code_bytes, (uint32_t)scale_bytes);
    }
    bulk_commit();
    bulk_wait_read<0>();
  }
  if (MODE != 0) {
    if (MODE == 2 && threadIdx.x < nrows)
      reinterpret_cast<float*>(dyn)[s_row[threadIdx.x]] = carried;
    if (scale_bytes && !a.scale_rows_bulk) {  // scale rows not 16-byte sized / aligned
      for (int n = 0; n < nrows; ++n)
        for (int b = threadIdx.x; b < scale_bytes; b += blockDim.x)
          dyn[(int64_t)s_row[n] * scale_bytes + b] = s_stage[code_bytes + b];
    }
  }
  // This CTA's stores are issued: the combine kernel may start launching.
  griddep_launch_dependents();
}

// ---------------------------------------------------------------------------
// Per-expert smooth rows: x * smooth[expert] is quantised once per dispatched
// row, and what the rows of one expert share is the smooth row, not the token
// row. This path therefore runs expert-major, in two kernels:
//
// index_kernel: one warp per source token maps its slots to rows (map_slot)
//   and records, for every dispatched row, its token and smooth-table row.
//
// smooth_rows_kernel: each CTA takes a contiguous range of dispatched rows.
//   Rows are ordered by destination rank, then local expert, so a range spans
//   one expert or a few: the CTA keeps the expert's smooth row in registers
//   (reloaded only when the expert changes) and streams the token rows
//   through a ring of kXStages shared-memory slots, filled by bulk (TMA)
//   loads that thread 0 issues kXStages rows ahead, one mbarrier per slot.
//   Codes go straight from registers to the row with 128-bit streaming
//   stores; one barrier per row (the row max, or an explicit one) frees the
//   row's ring slot for the next load.
constexpr int kXStages = 4;

template <class T>  // T only keeps one instantiation per token-type translation unit
__global__ void __launch_bounds__(256) index_kernel(PermuteArgs a) {
  griddep_wait();
  const int64_t tok = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (tok < (int64_t)a.d.W * a.d.BS) {
    const int r = (int)(tok / a.d.BS);
    int srow;
    const int k = threadIdx.x & 31;
    const int e = k < a.d.NS ? a.ws.eidx[tok * a.d.NS + k] : CQ_INV_NONE;
    const int row = map_slot(a, tok, r, k, e, srow);
    if (row >= 0) a.ws.row_src[row] = make_int2((int)tok, srow);
  }
  griddep_launch_dependents();
}

// FULL: the consumer threads hold exactly two units each (H a multiple of
// 1024), so no unit needs a bounds check.
template <class T, int Q, bool FULL>
__global__ void __launch_bounds__(288, 2) smooth_rows_kernel(PermuteArgs a) {
  constexpr int MODE = q_mode(Q);
  __shared__ uint64_t s_full[kXStages];
  __shared__ uint64_t s_empty[kXStages];
  __shared__ int s_srow[kXStages];
  __shared__ float s_red[2][64];
  __shared__ volatile int s_pfail;  // set by the producer only
  __shared__ int s_cfail;  // 1 + the first row a consumer gave up on, or INT_MAX
  extern __shared__ __align__(128) uint8_t s_ring[];  // kXStages token rows

  const Dims& d = a.d;
  const int H = d.H;
  const int units = H >> 4;
  const uint32_t xbytes = 2u * (uint32_t)H;
  const int scale_bytes = MODE == 3 ? 4 * d.G3 : 0;
  const int ncons = (int)blockDim.x - 32;  // consumer threads; the last warp produces
  const int nwc = ncons >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* const dyn = static_cast<uint8_t*>(a.dynamic_scales);
  uint8_t* const out = static_cast<uint8_t*>(a.expand_x);

  if (threadIdx.x == 0) {
    for (int st = 0; st < kXStages; ++st) {
      mbar_init(&s_full[st], 1);
      mbar_init(&s_empty[st], (uint32_t)nwc);
    }
    mbar_fence_init();
    s_pfail = 0;
    s_cfail = INT_MAX;
  }
  __syncthreads();
  griddep_wait();  // the row table and the total come from the earlier kernels

  int64_t total = *a.ws.total;
  if (total < 0 || total > d.R_max) {  // consistency guard
    if (threadIdx.x == 0) atomicOr(a.ws.status, (uint32_t)CQ_ST_INTERNAL);
    total = 0;
  }
  const int64_t lo = total * blockIdx.x / gridDim.x;
  const int n_rows = (int)(total * (blockIdx.x + 1) / gridDim.x - lo);

  if (warp == nwc) {
    // Producer warp: reads 32 row-table entries at a time; lane 0 streams the
    // token rows into the ring, kXStages rows ahead of the slowest consumer.
    const int64_t n_tok = (int64_t)d.W * d.BS;
    int issued = 0;
    for (int j0 = 0; j0 < n_rows; j0 += 32) {
      // Stop (the whole warp) once either side gave up.
      if (__any_sync(kFull, s_pfail != 0 || *(volatile int*)&s_cfail != INT_MAX)) break;
      int2 p = make_int2(0, 0);
      if (j0 + lane < n_rows) {
        p = a.ws.row_src[lo + j0 + lane];
        if (p.x < 0 || (int64_t)p.x >= n_tok || p.y < 0 || p.y >= d.S_eff + d.M) {
          // consistency guard: never read outside x or the smooth table
          atomicOr(a.ws.status, (uint32_t)CQ_ST_INTERNAL);
          p = make_int2(0, 0);
        }
      }
      const int nb = min(32, n_rows - j0);
      for (int b = 0; b < nb; ++b) {
        const int px = __shfl_sync(kFull, p.x, b), py = __shfl_sync(kFull, p.y, b);
        if (lane == 0 && !s_pfail) {
          const int j = j0 + b, st = j % kXStages;
          if (j >= kXStages &&
              !mbar_wait(&s_empty[st], (uint32_t)((j / kXStages) - 1) & 1u)) {
            s_pfail = 1;
            atomicOr(a.ws.status, (uint32_t)CQ_ST_TIMEOUT);
          } else {
            s_srow[st] = py;
            mbar_arrive_expect_tx(&s_full[st], xbytes);
            bulk_load(s_ring + (size_t)st * xbytes, a.x + (int64_t)px * H, xbytes, &s_full[st]);
            issued = j + 1;
          }
        }
        __syncwarp();
      }
    }
    // Wait (bounded) for the last loads to land before this warp ends, so
    // that no copy is in flight once the consumers are gone.
    if (lane == 0)
      for (int jj = issued > kXStages ? issued - kXStages : 0; jj < issued; ++jj)
        mbar_wait(&s_full[jj % kXStages], (uint32_t)(jj / kXStages) & 1u);
    griddep_launch_dependents();
    return;
  }

  // Consumer warps: each row is quantised by all of them together.
  Units U;
#pragma unroll
  for (int q = 0; q < 2; ++q) U.ok[q] = FULL || (int)threadIdx.x + q * ncons < units;
  float sm[2][16];
  int cur = -1;
  for (int j = 0; j < n_rows; ++j) {
    const int st = j % kXStages;
    if (!__all_sync(kFull, mbar_wait(&s_full[st], (uint32_t)(j / kXStages) & 1u)) && lane == 0) {
      atomicMin(&s_cfail, j + 1);
      atomicOr(a.ws.status, (uint32_t)CQ_ST_TIMEOUT);
    }
    const int srow = s_srow[st];
    if (srow != cur) {
      cur = srow;
      const float* srcs = a.smooth + (int64_t)srow * H;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * ncons;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 v = U.ok[q] ? ld_nc_v4(srcs + 16 * u + 4 * t) : make_uint4(0, 0, 0, 0);
          sm[q][4 * t] = __uint_as_float(v.x);
          sm[q][4 * t + 1] = __uint_as_float(v.y);
          sm[q][4 * t + 2] = __uint_as_float(v.z);
          sm[q][4 * t + 3] = __uint_as_float(v.w);
        }
      }
    }
    float f[2][16];
    const uint8_t* xs = s_ring + (size_t)st * xbytes;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = threadIdx.x + q * ncons;
      uint4 w[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if (U.ok[q]) {
        w[0] = ld_shared_v4(xs + 32 * u);
        w[1] = ld_shared_v4(xs + 32 * u + 16);
      }
      const uint32_t* wv = reinterpret_cast<const uint32_t*>(w);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float2 p = mul2(make_float2(T::lo(wv[t]), T::hi(wv[t])),
                              make_float2(sm[q][2 * t], sm[q][2 * t + 1]));
        f[q][2 * t] = p.x;
        f[q][2 * t + 1] = p.y;
      }
    }
    // This warp is done with the slot (token row and its smooth-row index).
    release_slot(&s_empty[st]);
    const int64_t row = lo + j;
    const float carried = quantise<Q, true, true>(f, U, out + row * H, dyn + row * scale_bytes,
                                                  s_red[j & 1], ncons);
    if (MODE == 2 && threadIdx.x == 0) reinterpret_cast<float*>(dyn)[row] = carried;
    // Leave after row j if a consumer gave up on a row <= j. In mode 2 every
    // such record was written before row j's barrier and every warp reads
    // after it, so the warps leave together (a record for a later row does
    // not count yet); the other modes have no barrier and each warp leaves on
    // its own.
    if (*(volatile int*)&s_cfail <= j + 1) break;
  }
  griddep_launch_dependents();
}

// The per-expert-smooth path: index_kernel, then smooth_rows_kernel with one
// wave of CTAs (SMs x resident CTAs per SM).
template <class T, int Q>
cudaError_t launch_smooth_rows(const PermuteArgs& a, cudaStream_t s) {
  constexpr int MODE = q_mode(Q);
  const int64_t tokens = (int64_t)a.d.W * a.d.BS;
  cudaError_t e =
      launch_pdl(index_kernel<T>, dim3((unsigned)((tokens + 7) / 8)), dim3(256), 0, s, a);
  if (e != cudaSuccess) return e;
  const int units = a.d.H >> 4;
  int threads = ((units + 1) / 2 + 31) / 32 * 32;
  if (threads < 32) threads = 32;
  const bool full = units == 2 * threads;
  threads += 32;  // the producer warp
  const size_t smem = (size_t)kXStages * 2 * a.d.H;
  auto* kern = full ? smooth_rows_kernel<T, Q, true> : smooth_rows_kernel<T, Q, false>;
  if ((e = full ? prepare_kernel<smooth_rows_kernel<T, Q, true>>(smem)
                : prepare_kernel<smooth_rows_kernel<T, Q, false>>(smem)) != cudaSuccess)
    return e;
  int blocks = 0;
  e = full ? occupancy_blocks<smooth_rows_kernel<T, Q, true>>(threads, smem, &blocks)
           : occupancy_blocks<smooth_rows_kernel<T, Q, false>>(threads, smem, &blocks);
  if (e != cudaSuccess) return e;
  if (blocks < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)sm_count() * blocks;
  if (grid > a.d.R_max) grid = a.d.R_max;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(threads), smem, s, a);
}

template <class T, int Q, int SM>
cudaError_t launch_one(const PermuteArgs& a, cudaStream_t s) {
  constexpr int MODE = q_mode(Q);
  const int units = a.d.H >> 4;
  int threads = ((units + 1) / 2 + 31) / 32 * 32;
  if (threads < 32) threads = 32;
  const int64_t grid = (int64_t)a.d.W * a.d.BS;
  const size_t code_bytes = MODE == 0 ? 2 * (size_t)a.d.H : (size_t)a.d.H;
  const size_t scale_bytes =
      MODE == 3 ? 4 * (size_t)a.d.G3 : ((MODE == 4 || MODE == 5) ? (size_t)a.d.SC : 0);
  const size_t smem = code_bytes + ((scale_bytes + 15) & ~size_t(15));
  const cudaError_t e = prepare_kernel<permute_kernel<T, Q, SM>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(permute_kernel<T, Q, SM>, dim3((unsigned)grid), dim3(threads), smem, s, a);
}

// Per-128-group fp8 (Q = 3 e4m3fn, 13 e5m2) for each smooth shape.
template <class T, int Q>
cudaError_t launch_mode3(const PermuteArgs& a, cudaStream_t s, int sm) {
  if (sm == kRowPerSlot) return launch_smooth_rows<T, Q>(a, s);
  if (sm == kSharedRow) return launch_one<T, Q, kSharedRow>(a, s);
  if (sm == kScalar) return launch_one<T, Q, kScalar>(a, s);
  return launch_one<T, Q, kNoSmooth>(a, s);
}

// Choose the instantiation for the call's mode and smooth shape.
template <class T>
cudaError_t launch_typed(const PermuteArgs& a, cudaStream_t s) {
  int sm = kNoSmooth;
  if (a.smooth) sm = a.smooth_kind == 0 ? kRowPerSlot : (a.smooth_kind == 1 ? kSharedRow : kScalar);
  switch (a.d.mode) {
    case 0: return launch_one<T, 0, kNoSmooth>(a, s);
    case 1:
      if (sm == kRowPerSlot) return launch_smooth_rows<T, 1>(a, s);
      if (sm == kSharedRow) return launch_one<T, 1, kSharedRow>(a, s);
      if (sm == kScalar) return launch_one<T, 1, kScalar>(a, s);
      return cudaErrorInvalidValue;  // static quantisation needs scales
    case 2:
      if (sm == kRowPerSlot) return launch_smooth_rows<T, 2>(a, s);
      if (sm == kSharedRow) return launch_one<T, 2, kSharedRow>(a, s);
      if (sm == kScalar) return launch_one<T, 2, kScalar>(a, s);
      return launch_one<T, 2, kNoSmooth>(a, s);
    case 3: return a.d.y_dtype ? launch_mode3<T, 13>(a, s, sm) : launch_mode3<T, 3>(a, s, sm);
    case 4:
      return a.d.y_dtype ? launch_one<T, 14, kNoSmooth>(a, s) : launch_one<T, 4, kNoSmooth>(a, s);
    case 5:
      return a.d.y_dtype ? launch_one<T, 15, kNoSmooth>(a, s) : launch_one<T, 5, kNoSmooth>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace permute_detail
}  // namespace cq
