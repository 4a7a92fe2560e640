// cq_route.cu -- routing scan on the device: two kernels, no serial tail.
//
// count_kernel (one CTA per chunk of a source rank r's tokens; the chunks of
// a source are counted side by side and offsets_kernel chains them) walks
// its tokens in row-major (token, then k) order and gives every MoE pair its
// arrival ordinal at its expert within the chunk ("expandIdx", the sendStatus
// counter of "MoeDistributeDispatch和MoeDistributeCombine算子设计介绍" §2.2.2,
// once the chunk's first row is added) and every active token its ordinal
// among the chunk's active tokens (the shared-expert slots). A chunk's tokens
// are split into contiguous per-warp ranges (4, 16 or 32 warps by size);
// one walk with warp match_any (equal ids grouped, ranked by lane) gives
// each pair its ordinal inside its warp's range and per-warp counts; a
// per-expert scan over the warps then turns those into the serial scan's
// ordinals within the chunk and the chunk's counts.
//
// offsets_kernel (one CTA per destination rank d) prefix-sums rank d's
// received-count matrix, transposed to (local expert, source) order and summed
// row-major (§2.4.1), which is ep_recv_count[d]; the counts come per (local
// expert, source, chunk), so the same scan gives each chunk's block its first
// row counted from the start of rank d. It also writes expert_token_nums[d].
// The counts table is slot-major and the slots of a rank are contiguous, so
// rank d's first row is the sum of the table's entries before its first
// slot: for tables of up to kDirectBase entries every CTA sums them itself
// (one parallel reduction); for larger ones the last CTA (one atomic
// counter, no spin) prefix-sums the W rank totals.
// Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
// top of include/cq.h.
#include "cq_internal.cuh"

namespace cq {
namespace {

// The count kernel runs kCountWarps warps per CTA (one chunk of a source's
// tokens), kCountWarpsWide for chunks of at least kWideBS tokens (shorter
// per-warp ranges; measured faster from 256 tokens on, slower for fewer) and
// kCountWarpsSmall for chunks of at most kSmallBS.
constexpr int kCountWarps = 16;
constexpr int kCountWarpsWide = 32;
constexpr int kWideBS = 256;
constexpr int kCountWarpsSmall = 4;
constexpr int kSmallBS = 32;
// Pairs per warp are at most ceil(512 / 16) tokens x 16 slots = 512, i.e. 16
// per lane, so each lane keeps its pairs in 16 registers (8 with 32 warps).
constexpr int kMaxSteps = 16;
constexpr int kOffThreads = 256;
constexpr int kOffWarps = kOffThreads / 32;
// Largest counts table (G x W entries) whose prefix each offsets CTA sums
// itself instead of waiting for the last CTA's scan of the rank totals.
constexpr int64_t kDirectBase = 1024;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Is pair (token i, slot j) switched on by the mask? (i < n_r already checked)
__device__ __forceinline__ bool pair_on(const RouteArgs& a, int64_t tok, int j) {
  if (a.d.mask_ndim == 0 || a.mask == nullptr) return true;
  if (a.d.mask_ndim == 1) return a.mask[tok] != 0;
  return a.mask[tok * a.d.K + j] != 0;
}

__device__ __forceinline__ bool token_on(const RouteArgs& a, int64_t tok) {
  if (a.d.mask_ndim == 0 || a.mask == nullptr) return true;
  if (a.d.mask_ndim == 1) return a.mask[tok] != 0;
  for (int j = 0; j < a.d.K; ++j)
    if (a.mask[tok * a.d.K + j] != 0) return true;  // all-false tokens do not take part
  return false;
}

// Global expert slot of local expert le on destination rank d (shared ranks first).
__device__ __forceinline__ int gslot(const Dims& d, int rank, int le) {
  return rank < d.S_r ? rank : d.S_r + (rank - d.S_r) * d.L + le;
}

// Block-wide exclusive scan of one int per thread (NW <= 32 warps); returns
// the prefix and the block total. One barrier: every warp reads all the warp
// totals from `buf` (NW ints) and sums the ones before it, so `buf` must not
// be written again before the caller's next barrier.
template <int NW>
__device__ int block_excl_scan(int v, int* buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  const int w = lane < NW ? buf[lane] : 0;
  *total = __reduce_add_sync(kFull, w);
  return __reduce_add_sync(kFull, lane < warp ? w : 0) + incl - v;
}

// CTA r * CH + c counts chunk c of source r: tokens [c * TC, (c + 1) * TC).
// Its ordinals run within the chunk; offsets_kernel gives every (slot,
// source, chunk) block its first row, so the chunks of a source follow one
// another in arrival order.
// trigger_early: every CTA of this grid is resident at once (W * CH <= SM
// count), so the dependent kernels may launch right away without starving it.
// STEPS >= the 32-pair steps of a warp's range: the unrolled loops hold only
// as many steps as the problem needs (the kernel's code is fetched cold from
// DRAM when L2 holds other data, so its size shows in the latency).
template <int STEPS, int NW>
__global__ void __launch_bounds__(NW * 32) count_kernel(RouteArgs a, int trigger_early) {
  constexpr int kThreads = NW * 32;
  extern __shared__ uint16_t tbl[];  // [NW][M]: per-warp counts, then bases
  __shared__ int s_tokcnt[NW];
  __shared__ int s_tokbase[NW + 1];

  if (trigger_early) griddep_launch_dependents();
  const Dims& d = a.d;
  const int r = blockIdx.x / d.CH, chunk = blockIdx.x - r * d.CH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = d.M, K = d.K, BS = d.BS, NS = d.NS;
  int n_r = BS;
  if (a.bs_per_rank) n_r = min(max(a.bs_per_rank[r], 0), BS);
  const int lo = min(chunk * d.TC, BS), hi = min(lo + d.TC, BS);  // this CTA's tokens
  const int tpw = (hi - lo + NW - 1) / NW;
  const int t0 = min(lo + warp * tpw, hi), t1 = min(t0 + tpw, hi);
  const int p0 = t0 * K, p1 = t1 * K;
  const int nsteps = (p1 - p0 + 31) >> 5;
  uint16_t* mytbl = tbl + warp * M;

  // Classify every pair of this warp first (all id loads in flight together):
  // a MoE expert id (>= 0), or a CQ_INV code (none / copy / const c).
  const int64_t Z0 = M, C0 = Z0 + d.Z, Q0 = C0 + d.C, Q1 = Q0 + d.Q;
  bool bad_id = false;
  int cls[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int p = p0 + s * 32 + lane;
    int c = CQ_INV_NONE;
    if (s < nsteps && p < p1) {
      const int i = p / K, j = p - (p / K) * K;
      const int64_t tok = (int64_t)r * BS + i;
      if (i < n_r && pair_on(a, tok, j)) {
        const int64_t id = a.expert_ids[tok * K + j];
        if (id >= 0 && id < M) c = (int)id;
        else if (id >= Z0 && id < C0) c = CQ_INV_NONE;  // zero expert
        else if (id >= C0 && id < Q0) c = CQ_INV_COPY;
        else if (id >= Q0 && id < Q1) c = CQ_INV_CONST_BASE - (int)(id - Q0);
        else bad_id = true;
      }
    }
    cls[s] = c;
  }
  for (int t = threadIdx.x; t < NW * M; t += kThreads) tbl[t] = 0;
  // [DV3] x_active_mask: in 1-D form every true entry precedes every false one.
  if (d.mask_ndim == 1 && a.mask) {
    for (int i = max(lo, 1) + (int)threadIdx.x; i < min(hi, n_r); i += kThreads) {
      const int64_t tok = (int64_t)r * BS + i;
      if (a.mask[tok] && !a.mask[tok - 1]) atomicOr(a.ws.status, (uint32_t)CQ_ST_BAD_MASK);
    }
  }
  __syncthreads();

  // One walk: the ordinal of each pair inside its warp's range, and the
  // warp's count per expert (the group leader adds the group size).
  int ord[STEPS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    ord[s] = 0;
    if (s >= nsteps) continue;
    const int key = cls[s] >= 0 ? cls[s] : -1;
    const unsigned grp = __match_any_sync(kFull, key);
    int before = 0;
    if (key >= 0) {
      before = mytbl[key];
      ord[s] = before + __popc(grp & lanemask_lt());
    }
    __syncwarp();
    if (key >= 0 && lane == __ffs(grp) - 1) mytbl[key] = (uint16_t)(before + __popc(grp));
    __syncwarp();
  }
  int tokcnt = 0;
  for (int base = t0; base < t1; base += 32) {
    const int i = base + lane;
    const bool on = i < t1 && i < n_r && token_on(a, (int64_t)r * BS + i);
    tokcnt += __popc(__ballot_sync(kFull, on));
  }
  if (lane == 0) s_tokcnt[warp] = tokcnt;
  __syncthreads();

  // Per expert: exclusive scan over the warps (warp bases); the total is
  // this chunk's count for the expert.
  for (int e = threadIdx.x; e < M; e += kThreads) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int c = tbl[w * M + e];
      tbl[w * M + e] = (uint16_t)run;
      run += c;
    }
    a.ws.counts_t[((int64_t)(d.S_r + e) * d.W + r) * d.CH + chunk] = run;
  }
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      s_tokbase[w] = run;
      run += s_tokcnt[w];
    }
    s_tokbase[NW] = run;  // active tokens of this chunk
  }
  __syncthreads();
  // Shared-expert rank g hosts replica g % R of shared expert g / R; source r
  // sends every active token to replica r % R of each shared expert. (The
  // active tokens of this chunk.)
  const int n_act = s_tokbase[NW];
  for (int g = threadIdx.x; g < d.S_r; g += kThreads) {
    const bool mine = d.S_eff > 0 && (g % d.R_rep) == (r % d.R_rep);
    a.ws.counts_t[((int64_t)g * d.W + r) * d.CH + chunk] = mine ? n_act : 0;
  }

  // Final ordinals: the warp's base for the expert plus the in-warp ordinal.
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    if (s >= nsteps) break;
    const int p = p0 + s * 32 + lane;
    if (p < p1) {
      const int i = p / K, j = p - (p / K) * K;
      const int code = cls[s] >= 0 ? (int)mytbl[cls[s]] + ord[s] : cls[s];
      a.ws.eidx[((int64_t)r * BS + i) * NS + j] = code;
    }
  }
  if (__any_sync(kFull, bad_id) && lane == 0) atomicOr(a.ws.status, (uint32_t)CQ_ST_BAD_ID);
  // Shared slots: ordinal of the token among this chunk's active tokens.
  int run = s_tokbase[warp];
  for (int base = t0; base < t1; base += 32) {
    const int i = base + lane;
    const bool on = i < t1 && i < n_r && token_on(a, (int64_t)r * BS + i);
    const unsigned bal = __ballot_sync(kFull, on);
    const int o = run + __popc(bal & lanemask_lt());
    if (i < t1)
      for (int s = 0; s < d.S_eff; ++s)
        a.ws.eidx[((int64_t)r * BS + i) * NS + K + s] = on ? o : CQ_INV_NONE;
    run += __popc(bal);
  }
  griddep_launch_dependents();  // no-op if already triggered
}

__global__ void __launch_bounds__(kOffThreads) offsets_kernel(RouteArgs a) {
  __shared__ int s_buf[kOffWarps + 1];
  __shared__ int s_last;

  // The permute kernel may launch now and prefetch token rows; it waits for
  // this grid before reading anything the routing wrote. (Every CTA of this
  // grid is running once all have passed this point, so the early launch
  // cannot starve it.)
  griddep_launch_dependents();
  griddep_wait();  // counts from count_kernel

  const Dims& d = a.d;
  const int rank = blockIdx.x;
  const int Ld = rank < d.S_r ? 1 : d.L;
  const int WC = d.W * d.CH;
  const int n = Ld * WC;  // this rank's (local expert, source, chunk) entries, <= 2048
  const int64_t g0w = (int64_t)gslot(d, rank, 0) * WC;
  const int* cnt = a.ws.counts_t + g0w;
  int* loc = a.ws.local_off + g0w;
  int* erc = a.ep_recv_count + (int64_t)rank * d.W * d.L;

  // Small tables: this rank's first row is the sum of the counts of all
  // slots before its first one (ranks are laid out slot-major, shared ranks
  // first); those loads go out together with this rank's own.
  const bool direct = (int64_t)d.G * WC <= kDirectBase;
  int part = 0;
  if (direct) {
    const int n_before = gslot(d, rank, 0) * WC;
    for (int t = threadIdx.x; t < n_before; t += kOffThreads) part += __ldcg(a.ws.counts_t + t);
  }

  // Each thread takes <= 8 contiguous entries; one block scan of their sums.
  constexpr int kPer = 8;
  const int per = (n + kOffThreads - 1) / kOffThreads;
  const int c0 = min((int)threadIdx.x * per, n), c1 = min(c0 + per, n);
  int v[kPer];
  int sum = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    v[q] = c0 + q < c1 ? __ldcg(cnt + c0 + q) : 0;
    sum += v[q];
  }
  int tot = 0;
  int run = block_excl_scan<kOffWarps>(sum, s_buf, &tot);
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (c0 + q < c1) {
      loc[c0 + q] = run;  // exclusive: first row of the block within rank d
      run += v[q];
      // inclusive running count (ep_recv_count) at the end of a (local
      // expert, source) pair's chunks
      if ((c0 + q) % d.CH == d.CH - 1) erc[(c0 + q) / d.CH] = run;
    }
  }
  for (int t = Ld * d.W + threadIdx.x; t < d.W * d.L; t += kOffThreads) erc[t] = 0;  // shared-rank padding
  __syncthreads();
  for (int le = threadIdx.x; le < d.L; le += kOffThreads) {
    int64_t e = 0;
    if (le < Ld) {
      const int end = erc[le * d.W + d.W - 1];
      e = d.etn_type == 1 ? end - loc[le * WC] : end;  // [DV3] 1: counts, 0: cumsum
    }
    a.expert_token_nums[(int64_t)rank * d.L + le] = e;
  }
  if (direct) {
    int base = 0;
    block_excl_scan<kOffWarps>(part, s_buf, &base);
    if (threadIdx.x == 0) {
      a.ws.rank_base[rank] = base;
      a.rank_row_base[rank] = base;
      if (rank == d.W - 1) {
        a.ws.rank_base[d.W] = base + tot;
        a.rank_row_base[d.W] = base + tot;
        *a.ws.total = base + tot;
      }
    }
    return;
  }
  // Last CTA: exclusive prefix of the W rank totals gives each rank's first
  // row. Thread 0 publishes this rank's total with a release increment of the
  // counter; the CTA that completes the count acquires every total, and its
  // barrier passes them on to its other threads.
  if (threadIdx.x == 0) {
    a.ws.rank_tot[rank] = tot;
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.ws.done) : "memory");
    s_last = old == (unsigned)(d.W - 1);
  }
  __syncthreads();
  if (!s_last) return;
  constexpr int kPerRank = 3;  // W <= 768 = 3 x 256
  const int rb0 = threadIdx.x * kPerRank;
  int rv[kPerRank];
  int rsum = 0;
#pragma unroll
  for (int q = 0; q < kPerRank; ++q) {
    rv[q] = rb0 + q < d.W ? __ldcg(a.ws.rank_tot + rb0 + q) : 0;
    rsum += rv[q];
  }
  int total = 0;
  int rrun = block_excl_scan<kOffWarps>(rsum, s_buf, &total);
#pragma unroll
  for (int q = 0; q < kPerRank; ++q) {
    if (rb0 + q < d.W) {
      a.ws.rank_base[rb0 + q] = rrun;
      a.rank_row_base[rb0 + q] = rrun;
      rrun += rv[q];
    }
  }
  if (threadIdx.x == 0) {
    a.ws.rank_base[d.W] = total;
    a.rank_row_base[d.W] = total;
    *a.ws.total = total;
    *a.ws.done = 0u;  // ready for the next call
  }
}

// One count-kernel instantiation; the wide one first raises its dynamic
// shared-memory limit (its table reaches 64 KB at M = 1024).
template <int STEPS, int NW>
cudaError_t launch_count(const RouteArgs& a, size_t table, int trigger, cudaStream_t s) {
  if (NW == kCountWarpsWide) {
    const cudaError_t e = prepare_kernel<count_kernel<STEPS, NW>>(table);
    if (e != cudaSuccess) return e;
  }
  count_kernel<STEPS, NW><<<a.d.W * a.d.CH, NW * 32, table, s>>>(a, trigger);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const bool wide = a.d.TC >= kWideBS, small = a.d.TC <= kSmallBS;
  const int nw = wide ? kCountWarpsWide : small ? kCountWarpsSmall : kCountWarps;
  const size_t table = sizeof(uint16_t) * nw * (size_t)a.d.M;  // <= 64 KB
  const int sms = sm_count();
  if (sms < 1) return cudaErrorInvalidDevice;
  const int tpw = (a.d.TC + nw - 1) / nw;
  const int steps = (tpw * a.d.K + 31) / 32;
  const int trigger = a.d.W * a.d.CH <= sms ? 1 : 0;
  cudaError_t e;
  if (small) {  // at most 8 tokens x 16 slots per warp: 4 steps
    e = steps <= 2 ? launch_count<2, kCountWarpsSmall>(a, table, trigger, s)
                   : launch_count<4, kCountWarpsSmall>(a, table, trigger, s);
  } else if (wide) {
    e = steps <= 2   ? launch_count<2, kCountWarpsWide>(a, table, trigger, s)
        : steps <= 4 ? launch_count<4, kCountWarpsWide>(a, table, trigger, s)
                     : launch_count<8, kCountWarpsWide>(a, table, trigger, s);
  } else {
    e = steps <= 2   ? launch_count<2, kCountWarps>(a, table, trigger, s)
        : steps <= 4 ? launch_count<4, kCountWarps>(a, table, trigger, s)
        : steps <= 8 ? launch_count<8, kCountWarps>(a, table, trigger, s)
                     : launch_count<kMaxSteps, kCountWarps>(a, table, trigger, s);
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(offsets_kernel, dim3(a.d.W), dim3(kOffThreads), 0, s, a);
}

}  // namespace cq
