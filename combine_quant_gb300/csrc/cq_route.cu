// cq_route.cu -- routing scan on the device.
//
// One CTA per source rank r walks expert_ids[r] in row-major (token, then k)
// order and gives every MoE pair its arrival ordinal at its expert
// ("expandIdx", the sendStatus counter of the design page
// "MoeDistributeDispatch和MoeDistributeCombine算子设计介绍", §2.2.2), and every
// active token its ordinal among active tokens (the shared-expert slots).
// The last CTA to finish turns the per-(expert slot, source) counts into
// global row offsets and the per-rank outputs ep_recv_count and
// expert_token_nums (§2.4: the received-count matrix, transposed and
// prefix-summed in row-major order).
//
// Ordering stays deterministic without any host round trip: the tokens of a
// source are split into 16 contiguous per-warp ranges; pass 1 counts each
// warp's pairs per expert (warp match_any groups equal ids, the group leader
// adds the group size), a per-expert scan over the 16 warps turns counts into
// warp bases, and pass 2 repeats the walk handing out base + rank-in-group.
// There are no spin waits: the last CTA is found with one atomic counter.
#include "cq_internal.cuh"

namespace cq {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Is pair (token i, slot j) of source r switched on? (i < n_r already checked)
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

// Block-wide exclusive scan of one int per thread; returns the prefix and
// stores the block total in *total.
__device__ int block_excl_scan(int v, int* smem_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) smem_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? smem_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kWarps) smem_warp[lane] = wi - w;  // exclusive warp offsets
    if (lane == kWarps - 1) smem_warp[kWarps] = wi;
  }
  __syncthreads();
  int res = smem_warp[warp] + incl - v;
  *total = smem_warp[kWarps];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kThreads) route_kernel(RouteArgs a) {
  extern __shared__ uint16_t tbl[];  // [kWarps][M] per-warp counters, then bases
  __shared__ int s_tokcnt[kWarps];
  __shared__ int s_tokbase[kWarps];
  __shared__ int s_scan[kWarps + 1];
  __shared__ int s_last;

  const Dims& d = a.d;
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int M = d.M, K = d.K, BS = d.BS, NS = d.NS;
  int n_r = BS;
  if (a.bs_per_rank) n_r = min(max(a.bs_per_rank[r], 0), BS);

  for (int t = threadIdx.x; t < kWarps * M; t += kThreads) tbl[t] = 0;

  // [DV3] x_active_mask: in 1-D form every true entry precedes every false one.
  if (d.mask_ndim == 1 && a.mask) {
    for (int i = threadIdx.x + 1; i < n_r; i += kThreads) {
      const int64_t tok = (int64_t)r * BS + i;
      if (a.mask[tok] && !a.mask[tok - 1]) atomicOr(a.ws.status, (uint32_t)CQ_ST_BAD_MASK);
    }
  }
  __syncthreads();

  const int tpw = (BS + kWarps - 1) / kWarps;
  const int t0 = min(warp * tpw, BS), t1 = min(t0 + tpw, BS);
  const int p0 = t0 * K, p1 = t1 * K;
  uint16_t* mytbl = tbl + warp * M;

  // Pass 1: per-warp counts of MoE pairs per expert, and active tokens.
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    int key = -1;
    if (p < p1) {
      const int i = p / K, j = p - (p / K) * K;
      const int64_t tok = (int64_t)r * BS + i;
      if (i < n_r && pair_on(a, tok, j)) {
        const int id = a.expert_ids[tok * K + j];
        if (id >= 0 && id < M) key = id;
      }
    }
    const unsigned grp = __match_any_sync(kFull, key);
    if (key >= 0 && lane == __ffs(grp) - 1) mytbl[key] += (uint16_t)__popc(grp);
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

  // Per expert: exclusive scan over warps; the total is this source's count.
  for (int e = threadIdx.x; e < M; e += kThreads) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = tbl[w * M + e];
      tbl[w * M + e] = (uint16_t)run;
      run += c;
    }
    a.ws.counts_t[(int64_t)(d.S_r + e) * d.W + r] = run;
  }
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      s_tokbase[w] = run;
      run += s_tokcnt[w];
    }
    s_tokcnt[0] = run;  // reused below as the number of active tokens (read after the barrier)
  }
  __syncthreads();
  const int n_act = s_tokcnt[0];
  // Shared-expert rank g hosts replica g % R of shared expert g / R; source r
  // sends every active token to replica r % R of each shared expert.
  for (int g = threadIdx.x; g < d.S_r; g += kThreads) {
    const bool mine = d.S_eff > 0 && (g % d.R_rep) == (r % d.R_rep);
    a.ws.counts_t[(int64_t)g * d.W + r] = mine ? n_act : 0;
  }

  // Pass 2: hand out arrival ordinals; record special-expert codes.
  const int64_t Z0 = M, C0 = Z0 + d.Z, Q0 = C0 + d.C, Q1 = Q0 + d.Q;
  bool bad_id = false;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    int key = -1, code = CQ_INV_NONE, i = 0, j = 0;
    if (p < p1) {
      i = p / K;
      j = p - i * K;
      const int64_t tok = (int64_t)r * BS + i;
      if (i < n_r && pair_on(a, tok, j)) {
        const int64_t id = a.expert_ids[tok * K + j];
        if (id >= 0 && id < M) key = (int)id;
        else if (id >= Z0 && id < C0) code = CQ_INV_NONE;
        else if (id >= C0 && id < Q0) code = CQ_INV_COPY;
        else if (id >= Q0 && id < Q1) code = CQ_INV_CONST_BASE - (int)(id - Q0);
        else bad_id = true;
      }
    }
    const unsigned grp = __match_any_sync(kFull, key);
    int basecnt = 0;
    if (key >= 0) {
      basecnt = mytbl[key];
      code = basecnt + __popc(grp & lanemask_lt());
    }
    __syncwarp();
    if (key >= 0 && lane == __ffs(grp) - 1) mytbl[key] = (uint16_t)(basecnt + __popc(grp));
    __syncwarp();
    if (p < p1) a.ws.eidx[((int64_t)r * BS + i) * NS + j] = code;
  }
  if (__any_sync(kFull, bad_id) && lane == 0) atomicOr(a.ws.status, (uint32_t)CQ_ST_BAD_ID);
  // Shared slots: ordinal of the token among this source's active tokens.
  int run = s_tokbase[warp];
  for (int base = t0; base < t1; base += 32) {
    const int i = base + lane;
    const bool on = i < t1 && i < n_r && token_on(a, (int64_t)r * BS + i);
    const unsigned bal = __ballot_sync(kFull, on);
    const int ord = run + __popc(bal & lanemask_lt());
    if (i < t1)
      for (int s = 0; s < d.S_eff; ++s)
        a.ws.eidx[((int64_t)r * BS + i) * NS + K + s] = on ? ord : CQ_INV_NONE;
    run += __popc(bal);
  }

  // ---- Last CTA: global offsets and per-rank receive metadata. ----
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.ws.done, 1u) == (unsigned)(d.W - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // blockoff = exclusive prefix of counts_t flattened (slot-major, source-minor).
  const int64_t N = (int64_t)d.G * d.W;
  const int64_t chunk = (N + kThreads - 1) / kThreads;
  const int64_t c0 = min((int64_t)threadIdx.x * chunk, N), c1 = min(c0 + chunk, N);
  int local = 0;
  for (int64_t n = c0; n < c1; ++n) local += __ldcg(a.ws.counts_t + n);
  int total = 0;
  int off = block_excl_scan(local, s_scan, &total);
  for (int64_t n = c0; n < c1; ++n) {
    const int c = __ldcg(a.ws.counts_t + n);
    a.ws.blockoff[n] = off;
    off += c;
  }
  __threadfence_block();
  __syncthreads();

  // rank_row_base: first row of each destination rank.
  for (int rank = threadIdx.x; rank <= d.W; rank += kThreads)
    a.rank_row_base[rank] =
        rank == d.W ? total : __ldcg(a.ws.blockoff + (int64_t)gslot(d, rank, 0) * d.W);
  __threadfence_block();
  __syncthreads();

  const int WL = d.W * d.L;
  for (int64_t n = threadIdx.x; n < (int64_t)d.W * WL; n += kThreads) {
    const int rank = (int)(n / WL), rem = (int)(n - (int64_t)rank * WL);
    const int le = rem / d.W, src = rem - le * d.W;
    const int Ld = rank < d.S_r ? 1 : d.L;
    int v = 0;
    if (le < Ld) {
      const int64_t gi = (int64_t)gslot(d, rank, le) * d.W + src;
      v = __ldcg(a.ws.blockoff + gi) + __ldcg(a.ws.counts_t + gi) -
          __ldcg(a.rank_row_base + rank);
    }
    a.ep_recv_count[n] = v;
  }
  for (int64_t n = threadIdx.x; n < (int64_t)d.W * d.L; n += kThreads) {
    const int rank = (int)(n / d.L), le = (int)(n - (int64_t)rank * d.L);
    const int Ld = rank < d.S_r ? 1 : d.L;
    int64_t v = 0;
    if (le < Ld) {
      const int64_t g0 = (int64_t)gslot(d, rank, le) * d.W;
      const int64_t end = (int64_t)__ldcg(a.ws.blockoff + g0 + d.W - 1) +
                          __ldcg(a.ws.counts_t + g0 + d.W - 1);
      v = d.etn_type == 1 ? end - __ldcg(a.ws.blockoff + g0)
                          : end - __ldcg(a.rank_row_base + rank);
    }
    a.expert_token_nums[n] = v;
  }
  if (threadIdx.x == 0) {
    *a.ws.total = total;
    *a.ws.done = 0u;  // ready for the next call
  }
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(uint16_t) * kWarps * (size_t)a.d.M;  // <= 32 KB for M <= 1024
  route_kernel<<<a.d.W, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace cq
