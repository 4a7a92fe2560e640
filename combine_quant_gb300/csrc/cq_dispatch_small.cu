// cq_dispatch_small.cu -- the whole dispatch of a small batch in one launch.
//
// For up to 2048 (token, slot) pairs the routing scan is cheaper to
// repeat than to hand over: every CTA of dispatch_small_kernel (one per
// source token, as permute_kernel) reads all of expert_ids and builds, in
// shared memory, the rows of every (expert slot, source) block and their
// exclusive prefix in slot-major order, which is each block's first global
// row (rank base + the block's offset within the rank, "MoeDistributeDispatch
// 和MoeDistributeCombine算子设计介绍" §2.4 and §3.4.2). In the same pass over
// the pairs it counts the earlier pairs of its own source with each of its
// experts (the arrival ordinal, expandIdx of §2.2.2); it then maps its slots
// to rows and quantises and scatters its token row exactly as permute_kernel
// does. CTA 0 also writes
// the routing outputs (ep_recv_count, expert_token_nums, rank_row_base) and
// the workspace's total rows, so every output ends up as cq_dispatch_route +
// cq_dispatch_permute leave it (the routing kernels' own scratch tables in
// the workspace are neither needed nor written). One launch replaces
// three (count, offsets, permute) and their two grid hand-offs, which is
// most of the latency of a batch of a few tokens per rank.
// Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
// top of include/cq.h.
#include "cq_permute_impl.cuh"

namespace cq {
namespace permute_detail {
namespace {

constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
// W * BS * K: every CTA repeats the scan over all pairs; from about this
// many on the routing kernels (one scan) are as fast or faster.
constexpr int kSmallMaxPairs = 2048;
constexpr int kSmallMaxEntries = 2048;  // G * W (counts and prefix in shared memory)
constexpr int kSmallMaxW = 768;
// With one smooth row per expert every routed row is quantised on its own,
// one after another in its token's CTA(s): past about this many values
// (W * BS * NS * H) the expert-major kernels are faster.
constexpr int64_t kSmallMaxSmoothValues = int64_t(1) << 23;

// Is token tok (source r, index i) active, and is its pair j switched on?
__device__ __forceinline__ int tokens_of(const PermuteArgs& a, int r) {
  int n = a.d.BS;
  if (a.bs_per_rank) n = min(max(a.bs_per_rank[r], 0), a.d.BS);
  return n;
}
__device__ __forceinline__ bool pair_on(const PermuteArgs& a, int64_t tok, int j) {
  if (a.d.mask_ndim == 0 || a.mask == nullptr) return true;
  if (a.d.mask_ndim == 1) return a.mask[tok] != 0;
  return a.mask[tok * a.d.K + j] != 0;
}
__device__ __forceinline__ bool token_on(const PermuteArgs& a, int64_t tok) {
  if (a.d.mask_ndim == 0 || a.mask == nullptr) return true;
  if (a.d.mask_ndim == 1) return a.mask[tok] != 0;
  for (int j = 0; j < a.d.K; ++j)
    if (a.mask[tok * a.d.K + j] != 0) return true;
  return false;
}

// Block-wide exclusive scan of one int per thread, with one barrier: every
// warp reads all the warp totals from `buf` (kSmallWarps ints) and sums the
// ones before it. `buf` must not be written again before the caller's next
// barrier.
__device__ int small_excl_scan(int v, int* buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  const int w = lane < kSmallWarps ? buf[lane] : 0;
  *total = __reduce_add_sync(kFull, w);
  return __reduce_add_sync(kFull, lane < warp ? w : 0) + incl - v;
}

// Outputs of the routing half that no permute kernel writes.
struct RouteOut {
  int32_t* ep_recv_count;
  int64_t* expert_token_nums;
  int32_t* rank_row_base;
};

// trigger_early: every CTA of this grid is resident at once, so the next
// kernel may launch right away without starving it.
// halves (1 or 2): CTAs per token. With 2, both CTAs of a token route and
// quantise the whole row, and each writes one half of every routed row's
// bytes (so a batch of few tokens spreads its stores over twice the SMs);
// the first writes the row records and scales.
// SM == kRowPerSlot: each routed row is quantised with its own smooth row
// (one expert's, or one shared expert's), one row after another; with two
// CTAs per token each quantises and writes every other routed row whole.
template <class T, int Q, int SM>
__global__ void __launch_bounds__(kSmallThreads)
    dispatch_small_kernel(PermuteArgs a, RouteOut ro, int trigger_early, int halves) {
  constexpr int MODE = q_mode(Q);
  __shared__ int s_row[kMaxSlots];
  __shared__ int s_srow[kMaxSlots];  // the routed rows' smooth-table rows (kRowPerSlot)
  __shared__ int s_nrows;
  __shared__ float s_red[2][64];
  __shared__ int s_id[kMaxSlots];   // this token's expert ids (-1: pair off)
  __shared__ int s_on[kMaxSlots];   // its pairs switched on
  __shared__ float s_w[kMaxSlots];  // its routing weights
  __shared__ int s_ord[kMaxSlots];  // their ordinals; [K]: the token's ordinal among active ones
  __shared__ int s_act[kSmallMaxW];  // active tokens per source
  __shared__ int s_buf[kSmallWarps + 1];
  extern __shared__ __align__(128) uint8_t s_dyn[];  // staged row, then counts, then prefix

  const Dims& d = a.d;
  const int64_t tok = blockIdx.x / halves;
  const int half = blockIdx.x - (int)tok * halves;
  const int r = (int)(tok / d.BS), i = (int)(tok - (int64_t)r * d.BS);
  const int lane = threadIdx.x & 31;
  const int H = d.H, units = H >> 4, nt = blockDim.x;
  const int W = d.W, K = d.K, NS = d.NS;
  const int nE = d.G * W;  // (slot, source) entries, slot-major
  const int code_bytes = MODE == 0 ? 2 * H : H;
  const int scale_bytes = MODE == 3 ? 4 * d.G3 : ((MODE == 4 || MODE == 5) ? d.SC : 0);
  const int stage_bytes = (code_bytes + ((scale_bytes + 15) & ~15) + 15) & ~15;
  const int n_stages = SM == kRowPerSlot ? 2 : 1;  // row after row: two staging buffers
  const int cpart = code_bytes / halves, spart = scale_bytes / halves;  // this CTA's bytes of a row
  uint8_t* const s_stage = s_dyn;
  int* const cnt = reinterpret_cast<int*>(s_dyn + n_stages * stage_bytes);  // [G][W] rows per block
  int* const start = cnt + nE;                                  // [G][W] first global row
  char* const dyn = static_cast<char*>(a.dynamic_scales);
  char* const out = static_cast<char*>(a.expand_x);
  const uint16_t* xrow = a.x + tok * H;
  if (trigger_early) griddep_launch_dependents();

  // The token row, loaded first: the routing below takes a few round trips.
  const int n_r = tokens_of(a, r);
  const bool active = i < n_r && token_on(a, tok);
  Units U;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int u = threadIdx.x + q * nt;
    U.ok[q] = u < units;
    if (U.ok[q] && active) {
      U.v[q][0] = ld_nc_v4(xrow + 16 * u);
      U.v[q][1] = ld_nc_v4(xrow + 16 * u + 8);
    } else {
      U.v[q][0] = U.v[q][1] = make_uint4(0, 0, 0, 0);
    }
  }

  // This token's slots (thread k < K holds slot k): its id and weight, in
  // shared memory before the pass over all pairs below.
  const int n_pairs = W * d.BS * K;
  const bool my_on = (int)threadIdx.x < K && active && pair_on(a, tok, threadIdx.x);
  const int my_id = (int)threadIdx.x < K ? a.expert_ids[tok * K + threadIdx.x] : -1;
  const float my_w = (int)threadIdx.x < K && a.expert_scales
                         ? a.expert_scales[tok * K + threadIdx.x] : 0.f;
  for (int t = threadIdx.x; t < nE; t += nt) cnt[t] = 0;
  for (int t = threadIdx.x; t < W; t += nt) s_act[t] = 0;
  if (threadIdx.x < kMaxSlots) {
    s_ord[threadIdx.x] = 0;
    s_id[threadIdx.x] = my_on ? my_id : -1;
    s_on[threadIdx.x] = my_on;
    s_w[threadIdx.x] = my_w;
  }
  __syncthreads();

  // Every MoE pair of every source: rows per (slot, source). In the same
  // pass, the arrival ordinals of this token's MoE pairs: the earlier pairs
  // of source r (token-major, then slot) with the same expert, one
  // shared-memory count per match.
  const int p_lo = r * d.BS * K, p_hi = (int)tok * K + K;
  for (int p = threadIdx.x; p < n_pairs; p += nt) {
    const int t = p / K, j = p - t * K;
    const int rr = t / d.BS, ii = t - rr * d.BS;
    if (ii < tokens_of(a, rr) && pair_on(a, t, j)) {
      const int id = a.expert_ids[p];
      if (id >= 0 && id < d.M) atomicAdd(&cnt[(d.S_r + id) * W + rr], 1);
      if (p >= p_lo && p < p_hi) {
#pragma unroll
        for (int k = 0; k < 16; ++k)
          if (k < K && p < (int)tok * K + k && id == s_id[k]) atomicAdd(&s_ord[k], 1);
      }
    }
  }
  for (int t = threadIdx.x; t < W * d.BS; t += nt) {
    const int rr = t / d.BS, ii = t - rr * d.BS;
    if (ii < tokens_of(a, rr) && token_on(a, t)) {
      atomicAdd(&s_act[rr], 1);
      if (rr == r && ii < i) atomicAdd(&s_ord[K], 1);  // this token's shared-slot ordinal
    }
  }
  __syncthreads();
  // Shared-expert rank g hosts replica g % R_rep; source rr sends every
  // active token to replica rr % R_rep of each shared expert.
  if (d.S_r > 0) {
    for (int t = threadIdx.x; t < d.S_r * W; t += nt) {
      const int g = t / W, rr = t - g * W;
      cnt[t] = (d.S_eff > 0 && (g % d.R_rep) == (rr % d.R_rep)) ? s_act[rr] : 0;
    }
    __syncthreads();
  }
  // Exclusive prefix of the counts in slot-major order: each block's first row.
  int total = 0;
  {
    const int per = (nE + nt - 1) / nt;
    const int e0 = min((int)threadIdx.x * per, nE), e1 = min(e0 + per, nE);
    int sum = 0;
    for (int e = e0; e < e1; ++e) sum += cnt[e];
    int run = small_excl_scan(sum, s_buf, &total);
    for (int e = e0; e < e1; ++e) {
      start[e] = run;
      run += cnt[e];
    }
  }
  __syncthreads();

  // This token's slots: codes, rows, the row records and the inverse map.
  float carried = 0.f;
  if (threadIdx.x < 32) {
    const int k = lane;
    int code = CQ_INV_NONE, row = -1, ord = CQ_INV_NONE, srow = 0;
    bool bad = false;
    if (k < K) {
      const int id = s_id[k];
      if (s_on[k]) {
        const int64_t Z0 = d.M, C0 = Z0 + d.Z, Q0 = C0 + d.C, Q1 = Q0 + d.Q;
        const int64_t id64 = id;
        if (id64 >= 0 && id64 < d.M) {
          ord = s_ord[k];
          row = start[(d.S_r + id) * W + r] + ord;
          srow = d.S_eff + id;
        } else if (id64 >= Z0 && id64 < C0) {
          ord = code = CQ_INV_NONE;
        } else if (id64 >= C0 && id64 < Q0) {
          ord = code = CQ_INV_COPY;
        } else if (id64 >= Q0 && id64 < Q1) {
          ord = code = CQ_INV_CONST_BASE - (int)(id64 - Q0);
        } else {
          bad = true;
        }
      }
    } else if (k < NS && active) {
      const int s = k - K;
      const int g = s * d.R_rep + r % d.R_rep;
      ord = s_ord[K];
      row = start[g * W + r] + ord;
      srow = s;
    }
    if (__any_sync(kFull, bad) && lane == 0) atomicOr(a.ws.status, (uint32_t)CQ_ST_BAD_ID);
    if (row >= 0 && (int64_t)row >= d.R_max) {  // consistency guard: never write outside
      atomicOr(a.ws.status, (uint32_t)CQ_ST_INTERNAL);
      row = -1;
    }
    if (row >= 0) {
      code = row;
      if (half == 0) {
        reinterpret_cast<int4*>(a.assist_rows)[row] = make_int4(r, i, k, 0);
        if (a.expand_scales) a.expand_scales[row] = k < K ? s_w[k] : 1.f;
      }
    }
    if (k < NS && half == 0) a.inv[tok * NS + k] = code;
    const unsigned bal = __ballot_sync(kFull, row >= 0);
    if (row >= 0) {
      const int pos = __popc(bal & ((1u << lane) - 1u));
      s_row[pos] = row;
      s_srow[pos] = srow;
    }
    if (lane == 0) s_nrows = __popc(bal);
  }

  // The routing outputs, written once (CTA 0), as the routing kernels do.
  if (blockIdx.x == 0) {
    if (d.mask_ndim == 1 && a.mask) {  // [DV3] x_active_mask: true entries first
      for (int t = threadIdx.x; t < W * d.BS; t += nt) {
        const int rr = t / d.BS, ii = t - rr * d.BS;
        if (ii >= 1 && ii < tokens_of(a, rr) && a.mask[t] && !a.mask[t - 1])
          atomicOr(a.ws.status, (uint32_t)CQ_ST_BAD_MASK);
      }
    }
    for (int e = threadIdx.x; e < nE; e += nt) {
      const int g = e / W;
      const int dst = g < d.S_r ? g : d.S_r + (g - d.S_r) / d.L;
      const int g0 = dst < d.S_r ? dst : d.S_r + (dst - d.S_r) * d.L;
      const int base = start[g0 * W];
      const int le = g - g0, rr = e - g * W;
      ro.ep_recv_count[(int64_t)dst * W * d.L + le * W + rr] = start[e] + cnt[e] - base;
    }
    for (int t = threadIdx.x; t < d.S_r * W * d.L; t += nt) {  // shared-rank padding
      const int dst = t / (W * d.L), q = t - dst * W * d.L;
      if (q >= W) ro.ep_recv_count[t] = 0;
    }
    for (int t = threadIdx.x; t < W * d.L; t += nt) {
      const int dst = t / d.L, le = t - dst * d.L;
      const int Ld = dst < d.S_r ? 1 : d.L;
      int64_t v = 0;
      if (le < Ld) {
        const int g = dst < d.S_r ? dst : d.S_r + (dst - d.S_r) * d.L + le;
        const int g0 = dst < d.S_r ? dst : d.S_r + (dst - d.S_r) * d.L;
        const int end = start[g * W + W - 1] + cnt[g * W + W - 1] - start[g0 * W];
        v = d.etn_type == 1 ? end - (start[g * W] - start[g0 * W]) : end;  // [DV3] 1: counts, 0: cumsum
      }
      ro.expert_token_nums[t] = v;
    }
    for (int dst = threadIdx.x; dst <= W; dst += nt) {
      const int v = dst < W ? start[(dst < d.S_r ? dst : d.S_r + (dst - d.S_r) * d.L) * W] : total;
      a.ws.rank_base[dst] = v;
      ro.rank_row_base[dst] = v;
    }
    if (threadIdx.x == 0) *a.ws.total = total;
  }
  __syncthreads();

  const int nrows = s_nrows;
  if (nrows == 0) {
    if (!trigger_early) griddep_launch_dependents();
    return;
  }
  if (SM == kRowPerSlot) {
    // One quantisation per routed row, each with its own smooth row, into
    // the two staging buffers in turn: a row's bulk stores drain while the
    // next row is quantised. With two CTAs per token each takes every other
    // row and writes it whole.
    int it = 0;
    for (int n = half; n < nrows; n += halves, ++it) {
      uint8_t* const stg = s_stage + (it & 1) * stage_bytes;
      // The stores of this buffer's previous row have read it before any
      // thread passes the barrier inside quantise and writes it again.
      if (threadIdx.x == 0 && it >= 2) bulk_wait_read<1>();
      const float* srow = a.smooth + (int64_t)s_srow[n] * H;
      float f[2][16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = threadIdx.x + q * nt;
        if (U.ok[q]) {
          unit_values<T, kSharedRow>(U.v[q], srow, 0.f, u, f[q]);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) f[q][t] = 0.f;
        }
      }
      carried = quantise<Q>(f, U, stg, stg + code_bytes, s_red[0], nt);
      fence_proxy_async_smem();  // staging writes before the bulk copies read them
      __syncthreads();
      const int64_t row = s_row[n];
      if (threadIdx.x == 0) {
        bulk_store(out + row * code_bytes, stg, (uint32_t)code_bytes);
        if (scale_bytes && a.scale_rows_bulk)
          bulk_store(dyn + row * scale_bytes, stg + code_bytes, (uint32_t)scale_bytes);
        bulk_commit();
      }
      if (MODE == 2 && threadIdx.x == 0) reinterpret_cast<float*>(dyn)[row] = carried;
      if (scale_bytes && !a.scale_rows_bulk)
        for (int b = threadIdx.x; b < scale_bytes; b += nt) dyn[row * scale_bytes + b] = stg[code_bytes + b];
    }
    if (threadIdx.x == 0) bulk_wait_read<0>();
    if (!trigger_early) griddep_launch_dependents();
    return;
  }
  // The code row (and scale row) every routed row gets, into s_stage.
  if (MODE == 0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = threadIdx.x + q * nt;
      if (U.ok[q]) {
        st_shared_v4(s_stage + 32 * u, U.v[q][0]);
        st_shared_v4(s_stage + 32 * u + 16, U.v[q][1]);
      }
    }
  } else {
    const float* srow = SM == kSharedRow ? a.smooth : nullptr;
    const float scalar = SM == kScalar ? a.smooth[0] : 0.f;
    float f[2][16];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int u = threadIdx.x + q * nt;
      if (U.ok[q]) {
        unit_values<T, SM>(U.v[q], srow, scalar, u, f[q]);
      } else {
#pragma unroll
        for (int t = 0; t < 16; ++t) f[q][t] = 0.f;
      }
    }
    carried = quantise<Q>(f, U, s_stage, s_stage + code_bytes, s_red[0], nt);
    if (MODE == 5 || MODE == 4) {
      if (threadIdx.x == 0 && d.SC > (units >> 1)) s_stage[code_bytes + (units >> 1)] = 0;
    }
  }
  fence_proxy_async_smem();  // staging writes before the bulk copies read them
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int n = 0; n < nrows; ++n) {
      const int64_t row = s_row[n];
      bulk_store(out + row * code_bytes + half * cpart, s_stage + half * cpart, (uint32_t)cpart);
      if (scale_bytes && a.scale_rows_bulk)
        bulk_store(dyn + row * scale_bytes + half * spart, s_stage + code_bytes + half * spart,
                   (uint32_t)spart);
    }
    bulk_commit();
    bulk_wait_read<0>();
  }
  if (MODE != 0 && half == 0) {
    if (MODE == 2 && threadIdx.x < nrows)
      reinterpret_cast<float*>(dyn)[s_row[threadIdx.x]] = carried;
    if (scale_bytes && !a.scale_rows_bulk) {
      for (int n = 0; n < nrows; ++n)
        for (int b = threadIdx.x; b < scale_bytes; b += nt)
          dyn[(int64_t)s_row[n] * scale_bytes + b] = s_stage[code_bytes + b];
    }
  }
  if (!trigger_early) griddep_launch_dependents();
}

template <class T, int Q, int SM>
cudaError_t launch_small(const PermuteArgs& a, const RouteOut& ro, cudaStream_t s) {
  constexpr int MODE = q_mode(Q);
  const size_t code_bytes = MODE == 0 ? 2 * (size_t)a.d.H : (size_t)a.d.H;
  const size_t scale_bytes =
      MODE == 3 ? 4 * (size_t)a.d.G3 : ((MODE == 4 || MODE == 5) ? (size_t)a.d.SC : 0);
  const size_t stage = (code_bytes + ((scale_bytes + 15) & ~size_t(15)) + 15) & ~size_t(15);
  const size_t smem = (SM == kRowPerSlot ? 2 : 1) * stage + 2 * sizeof(int) * (size_t)a.d.G * a.d.W;
  cudaError_t e = prepare_kernel<dispatch_small_kernel<T, Q, SM>>(smem);
  if (e != cudaSuccess) return e;
  int blocks = 0;
  e = occupancy_blocks<dispatch_small_kernel<T, Q, SM>>(kSmallThreads, smem, &blocks);
  if (e != cudaSuccess) return e;
  const int64_t tokens = (int64_t)a.d.W * a.d.BS;
  const int64_t wave = (int64_t)sm_count() * blocks;
  // Two CTAs per token while they still fit in one wave and a row's halves
  // keep the bulk copies' 16-byte granularity.
  const bool split = 2 * tokens <= wave && code_bytes % 32 == 0 &&
                     (scale_bytes == 0 || !a.scale_rows_bulk || scale_bytes % 32 == 0);
  const int halves = split ? 2 : 1;
  const int trigger = tokens * halves <= wave ? 1 : 0;
  dispatch_small_kernel<T, Q, SM>
      <<<(unsigned)(tokens * halves), kSmallThreads, smem, s>>>(a, ro, trigger, halves);
  return cudaGetLastError();
}

template <class T>
cudaError_t launch_small_typed(const PermuteArgs& a, const RouteOut& ro, cudaStream_t s) {
  int sm = kNoSmooth;
  if (a.smooth) sm = a.smooth_kind == 0 ? kRowPerSlot : (a.smooth_kind == 1 ? kSharedRow : kScalar);
  switch (a.d.mode) {
    case 0: return launch_small<T, 0, kNoSmooth>(a, ro, s);
    case 2:
      if (sm == kNoSmooth) return launch_small<T, 2, kNoSmooth>(a, ro, s);
      if (sm == kSharedRow) return launch_small<T, 2, kSharedRow>(a, ro, s);
      if (sm == kScalar) return launch_small<T, 2, kScalar>(a, ro, s);
      return launch_small<T, 2, kRowPerSlot>(a, ro, s);
    case 5:
      return a.d.y_dtype ? cudaErrorNotSupported : launch_small<T, 5, kNoSmooth>(a, ro, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace
}  // namespace permute_detail

bool dispatch_small_fits(const Dims& d, bool per_expert_smooth) {
  using namespace permute_detail;
  if (per_expert_smooth &&
      (d.mode != 2 || (int64_t)d.W * d.BS * d.NS * d.H > kSmallMaxSmoothValues))
    return false;
  if (d.mode != 0 && d.mode != 2 && !(d.mode == 5 && d.y_dtype == 0)) return false;
  return (int64_t)d.W * d.BS * d.K <= kSmallMaxPairs && (int64_t)d.G * d.W <= kSmallMaxEntries &&
         d.W <= kSmallMaxW && d.K <= 16;
}

cudaError_t launch_dispatch_small(const PermuteArgs& a, int32_t* ep_recv_count,
                                  int64_t* expert_token_nums, int32_t* rank_row_base,
                                  cudaStream_t s) {
  using namespace permute_detail;
  const RouteOut ro{ep_recv_count, expert_token_nums, rank_row_base};
  return a.d.x_dtype == 1 ? launch_small_typed<F16>(a, ro, s) : launch_small_typed<BF16>(a, ro, s);
}

}  // namespace cq
