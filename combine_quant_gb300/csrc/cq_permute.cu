// cq_permute.cu -- fused gather-quantise-scatter (MoePermute + pre-send quantisation).
//
// One CTA per source token (r, i). Warp 0 turns each slot's arrival ordinal
// into its global row (row = first row of the (expert slot, source) block +
// ordinal, the address rule of "MoeDistributeDispatch和MoeDistributeCombine
// 算子设计介绍" §3.4.2 with the source block folded into the expert offset),
// writes the inverse map, the (src, token, slot) row record and the carried
// weight. All threads load the token row once with 128-bit loads (started
// before the routing kernels finish), quantise it in registers and stage the
// code row in shared memory; one thread then writes it to every routed row
// with bulk (TMA) stores. quant_mode 0 copies the bf16 row, quant_mode 2 is
// per-token dynamic int8 (optionally per-expert smoothed, then quantised once
// per slot), quant_mode 5 is mx-clip e4m3 with one power-of-two scale per 32
// elements ("low_latency_dispatch" 计算公式).
//
// Arithmetic is fixed to single IEEE binary32 operations (explicit _rn
// intrinsics, no contraction) so the codes and scales are reproducible.
#include "cq_internal.cuh"

namespace cq {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxSlots = 32;  // NS <= 16 + 4

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

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round to nearest even, saturate to int8 (a NaN product gives 0).
__device__ __forceinline__ uint32_t q8(float v) {
  int c = __float2int_rn(v);
  c = max(-128, min(127, c));
  return (uint32_t)c & 0xffu;
}

__device__ __forceinline__ uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return a | (b << 8) | (c << 16) | (d << 24);
}

// Two binary32 values to two e4m3 bytes (lo in the low byte), round to
// nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Exact ceil(log2(q)) for a positive normal binary32 q: its exponent, plus
// one unless q is a power of two.
__device__ __forceinline__ int ceil_log2_bits(float q) {
  const uint32_t b = __float_as_uint(q);
  return (int)((b >> 23) & 0xffu) - 127 + ((b & 0x7fffffu) != 0u ? 1 : 0);
}

// Per-thread view of two 16-element units of the row (32 bytes of bf16 each).
struct Units {
  uint4 v[2][2];
  bool ok[2];
};

__device__ __forceinline__ float unit_amax(const uint4 (&u)[2]) {
  float m = 0.f;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u[0]);
#pragma unroll
  for (int t = 0; t < 8; ++t) m = fmaxf(m, fmaxf(fabsf(bf_lo(w[t])), fabsf(bf_hi(w[t]))));
  return m;
}

// 16 int8 codes of x * s.
__device__ __forceinline__ uint4 unit_q8(const uint4 (&u)[2], float s) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u[0]);
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    o[t] = pack4(q8(__fmul_rn(bf_lo(w[2 * t]), s)), q8(__fmul_rn(bf_hi(w[2 * t]), s)),
                 q8(__fmul_rn(bf_lo(w[2 * t + 1]), s)), q8(__fmul_rn(bf_hi(w[2 * t + 1]), s)));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Smoothed values x * sm for one unit: 16 floats.
__device__ __forceinline__ void unit_smooth(const uint4 (&u)[2], const float* sm, float (&xf)[16]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u[0]);
  float s[16];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint4 q = ld_nc_v4(sm + 4 * t);
    s[4 * t] = __uint_as_float(q.x);
    s[4 * t + 1] = __uint_as_float(q.y);
    s[4 * t + 2] = __uint_as_float(q.z);
    s[4 * t + 3] = __uint_as_float(q.w);
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    xf[2 * t] = __fmul_rn(bf_lo(w[t]), s[2 * t]);
    xf[2 * t + 1] = __fmul_rn(bf_hi(w[t]), s[2 * t + 1]);
  }
}

__device__ __forceinline__ uint4 floats_q8(const float (&xf)[16], float s) {
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    o[t] = pack4(q8(__fmul_rn(xf[4 * t], s)), q8(__fmul_rn(xf[4 * t + 1], s)),
                 q8(__fmul_rn(xf[4 * t + 2], s)), q8(__fmul_rn(xf[4 * t + 3], s)));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 16 e4m3 codes of x * 2^-e (an exact scaling by a power of two).
__device__ __forceinline__ uint4 unit_e4m3(const uint4 (&u)[2], int e) {
  const float p = __uint_as_float((uint32_t)(127 - e) << 23);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u[0]);
  uint32_t o[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t a = e4m3x2(__fmul_rn(bf_lo(w[2 * t]), p), __fmul_rn(bf_hi(w[2 * t]), p));
    const uint32_t b =
        e4m3x2(__fmul_rn(bf_lo(w[2 * t + 1]), p), __fmul_rn(bf_hi(w[2 * t + 1]), p));
    o[t] = a | (b << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Block-wide max of one float per thread; `buf` holds >= 32 floats and must
// not be reused by another block_max until the next __syncthreads.
__device__ __forceinline__ float block_max(float v, float* buf) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0) buf[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = 0.f;
  const int nw = blockDim.x >> 5;
  for (int w = 0; w < nw; ++w) m = fmaxf(m, buf[w]);
  return m;
}

// MODE: 0, 2, 5. SMOOTH: mode 2 with per-expert smooth scales.
template <int MODE, bool SMOOTH>
__global__ void __launch_bounds__(256) permute_kernel(PermuteArgs a) {
  __shared__ int s_row[kMaxSlots];   // compact list of routed rows
  __shared__ int s_srow[kMaxSlots];  // their smooth-table rows
  __shared__ int s_nrows;
  __shared__ float s_red[2][32];
  extern __shared__ __align__(128) uint8_t s_stage[];  // staged code row(s) + mx scale row

  const Dims& d = a.d;
  const int64_t tok = blockIdx.x;
  const int r = (int)(tok / d.BS), i = (int)(tok - (int64_t)r * d.BS);
  const int lane = threadIdx.x & 31;
  const int H = d.H;
  const int units = H >> 4;
  const uint16_t* xrow = a.x + tok * H;

  // Thread t owns the 16-element units t and t + blockDim of the token row.
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
  // its row now: this kernel may be running while the routing kernel ends.
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
  griddep_wait();  // routing outputs (ordinals, block offsets) are read from here on

  if (threadIdx.x < 32) {
    const int k = lane;
    int row = -1, srow = 0;
    if (k < d.NS) {
      const int e = a.ws.eidx[tok * d.NS + k];
      int code = e;
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
        row = a.ws.rank_base[dst] + a.ws.local_off[(int64_t)g * d.W + r] + e;
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
    }
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
  if (!prefetched) load_row();  // routing found rows the inputs did not predict

  // Every mode stages its code row once in shared memory; thread 0 then
  // writes it to each routed row with one bulk (TMA) store per row, so the
  // K-fold store traffic costs no per-thread store instructions.
  uint8_t* const stage = s_stage;
  if (MODE == 0) {
    // quant_mode 0: the bf16 row itself travels ([DV3] 情形 1).
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = threadIdx.x + q * blockDim.x;
      if (U.ok[q]) {
        st_shared_v4(stage + 32 * u, U.v[q][0]);
        st_shared_v4(stage + 32 * u + 16, U.v[q][1]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int n = 0; n < nrows; ++n)
        bulk_store(static_cast<uint16_t*>(a.expand_x) + (int64_t)s_row[n] * H, stage, 2u * H);
      bulk_commit();
      bulk_wait_read<0>();
    }
  } else if (MODE == 2 && !SMOOTH) {
    // One quantisation per token: every routed row gets the same codes.
    const float amax = block_max(fmaxf(unit_amax(U.v[0]), unit_amax(U.v[1])), s_red[0]);
    const float s = __fdiv_rn(127.f, amax);
    const float deq = __fdiv_rn(1.f, s);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = threadIdx.x + q * blockDim.x;
      if (U.ok[q]) st_shared_v4(stage + 16 * u, unit_q8(U.v[q], s));
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int n = 0; n < nrows; ++n)
        bulk_store(static_cast<int8_t*>(a.expand_x) + (int64_t)s_row[n] * H, stage, (uint32_t)H);
      bulk_commit();
      bulk_wait_read<0>();
    }
    if (threadIdx.x < nrows) static_cast<float*>(a.dynamic_scales)[s_row[threadIdx.x]] = deq;
  } else if (MODE == 2 && SMOOTH) {
    // x_fp32 = x * smooth[expert]: one amax and one scale per routed row.
    // Two staging buffers: row n is built while row n-1's bulk store reads.
    for (int n = 0; n < nrows; ++n) {
      const float* sm = a.smooth + (int64_t)s_srow[n] * H;
      float xf[2][16];
      float m = 0.f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * blockDim.x;
        if (U.ok[q]) {
          unit_smooth(U.v[q], sm + 16 * u, xf[q]);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) xf[q][t] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) m = fmaxf(m, fabsf(xf[q][t]));
      }
      // block_max starts with a barrier: thread 0's wait below for the
      // store of row n-2 (same buffer) is complete before anyone writes it.
      const float amax = block_max(m, s_red[n & 1]);
      const float s = __fdiv_rn(127.f, amax);
      uint8_t* buf = stage + (n & 1) * H;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * blockDim.x;
        if (U.ok[q]) st_shared_v4(buf + 16 * u, floats_q8(xf[q], s));
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (threadIdx.x == 0) {
        bulk_store(static_cast<int8_t*>(a.expand_x) + (int64_t)s_row[n] * H, buf, (uint32_t)H);
        bulk_commit();
        bulk_wait_read<1>();
        static_cast<float*>(a.dynamic_scales)[s_row[n]] = __fdiv_rn(1.f, s);
      }
    }
    if (threadIdx.x == 0) bulk_wait_read<0>();
  } else if (MODE == 5) {
    // Lanes 2m and 2m+1 hold the two halves of one 32-element block. The
    // e8m0 scale row is staged after the code row.
    uint8_t* srow_stage = stage + H;
    const int nblk = units >> 1;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float m = unit_amax(U.v[q]);
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
      m = fmaxf(m, 1e-4f);
      const int e = ceil_log2_bits(__fdiv_rn(m, 448.f));
      const int u = threadIdx.x + q * blockDim.x;
      if (U.ok[q]) {
        st_shared_v4(stage + 16 * u, unit_e4m3(U.v[q], e));
        if ((u & 1) == 0) srow_stage[u >> 1] = (uint8_t)(e + 127);
      }
    }
    if (threadIdx.x == 0 && d.SC > nblk) srow_stage[nblk] = 0;  // Align2 padding column
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int n = 0; n < nrows; ++n) {
        const int64_t row = s_row[n];
        bulk_store(static_cast<uint8_t*>(a.expand_x) + row * H, stage, (uint32_t)H);
        if (a.scale_rows_bulk)
          bulk_store(static_cast<uint8_t*>(a.dynamic_scales) + row * d.SC, srow_stage,
                     (uint32_t)d.SC);
      }
      bulk_commit();
      bulk_wait_read<0>();
    }
    if (!a.scale_rows_bulk) {  // scale rows not 16-byte sized / aligned: plain stores
      for (int n = 0; n < nrows; ++n) {
        uint8_t* sc = static_cast<uint8_t*>(a.dynamic_scales) + (int64_t)s_row[n] * d.SC;
        for (int b = threadIdx.x; b < d.SC; b += blockDim.x) sc[b] = srow_stage[b];
      }
    }
  }
  // This CTA's stores are issued: the combine kernel may start launching.
  griddep_launch_dependents();
}

template <int MODE, bool SMOOTH>
cudaError_t launch_mode(const PermuteArgs& a, cudaStream_t s) {
  const int units = a.d.H >> 4;
  int threads = ((units + 1) / 2 + 31) / 32 * 32;
  if (threads < 32) threads = 32;
  const int64_t grid = (int64_t)a.d.W * a.d.BS;
  // Staging: one bf16 row (mode 0), one or two int8 rows (mode 2, two when
  // smoothed per slot), or an e4m3 row plus its scale row (mode 5).
  size_t smem = MODE == 0 ? 2 * (size_t)a.d.H : (size_t)a.d.H * (SMOOTH ? 2 : 1);
  if (MODE == 5) smem += ((size_t)a.d.SC + 15) & ~size_t(15);
  return launch_pdl(permute_kernel<MODE, SMOOTH>, dim3((unsigned)grid), dim3(threads), smem, s, a);
}

}  // namespace

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s) {
  switch (a.d.mode) {
    case 0: return launch_mode<0, false>(a, s);
    case 2: return a.smooth ? launch_mode<2, true>(a, s) : launch_mode<2, false>(a, s);
    case 5: return launch_mode<5, false>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cq
