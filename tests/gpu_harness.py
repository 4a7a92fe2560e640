"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the oracle on the same seeded inputs."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import combine_quant_gb300 as cq
import oracle
from combine_quant_gb300 import workloads

DEV = torch.device("cuda:0")


def dev(a, dtype):
    """numpy array (raw bits allowed) -> CUDA tensor of `dtype`."""
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(DEV).view(dtype)


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def uses_smooth(wl) -> bool:
    return wl.smooth is not None and wl.cfg["quant_mode"] in (1, 2, 3)


def one_kernel_dispatch(wl) -> bool:
    """Whether cq_dispatch runs this problem as one kernel (the library's own
    decision, cq_dispatch_one_kernel)."""
    return cq.dispatch_one_kernel(cq.Config.from_dict(wl.cfg), uses_smooth(wl))


def _same_outputs(cfg, a, b) -> None:
    """Every defined output equal (rows past the total are left untouched)."""
    rows_a, inv_a, base_a = cq.assist_views(cfg, a.assist_info)
    rows_b, inv_b, base_b = cq.assist_views(cfg, b.assist_info)
    R = int(host(base_a)[-1])
    assert torch.equal(base_a, base_b) and torch.equal(inv_a, inv_b)
    assert torch.equal(rows_a[:R], rows_b[:R])
    for name in ("ep_recv_count", "expert_token_nums"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.expand_x[:R].view(torch.uint8), b.expand_x[:R].view(torch.uint8))
    if a.expand_scales is not None:
        assert torch.equal(a.expand_scales[:R], b.expand_scales[:R])
    if a.dynamic_scales is not None:
        assert torch.equal(a.dynamic_scales[:R].view(torch.uint8),
                           b.dynamic_scales[:R].view(torch.uint8))


def gpu_dispatch(wl: workloads.Workload):
    """cq_dispatch on the workload. Where that runs as one kernel, the two
    halves (cq_dispatch_route + cq_dispatch_permute: the routing, permute and
    per-expert-smooth kernels that larger problems run) run too and must give
    the same outputs and status, so every caller's oracle comparison covers
    both paths."""
    cfg = cq.Config.from_dict(wl.cfg)
    x = dev(wl.x, cfg.token_dtype)
    ids = dev(wl.expert_ids, torch.int32)
    sm = dev(wl.smooth, torch.float32) if uses_smooth(wl) else None
    mask = dev(wl.mask, torch.uint8)
    bpr = dev(wl.bs_per_rank, torch.int32)
    w = dev(wl.expert_scales, torch.float32)
    ws = cq.alloc_workspace(cfg, DEV)
    out = cq.dispatch(cfg, x, ids, smooth_scales=sm, x_active_mask=mask, bs_per_rank=bpr,
                      expert_scales=w, workspace=ws)
    status = cq.read_status(ws)
    if one_kernel_dispatch(wl):
        ws2 = cq.alloc_workspace(cfg, DEV)
        out2 = cq.alloc_dispatch_outputs(cfg, DEV)
        cq.dispatch_route(cfg, ids, mask, bpr, workspace=ws2, out=out2)
        cq.dispatch_permute(cfg, x, ids, sm, w, mask, bpr, workspace=ws2, out=out2)
        assert cq.read_status(ws2) == status
        _same_outputs(cfg, out, out2)
    return cfg, out, status, ws


def compare_route(wl, cfg, out, ref_route):
    """Bit-exact comparison of every index / count output."""
    rows, inv, base = cq.assist_views(cfg, out.assist_info)
    R = ref_route.rows
    assert int(host(base)[-1]) == R, "total rows"
    assert np.array_equal(host(base), ref_route.rank_row_base.astype(np.int32))
    assert np.array_equal(host(out.ep_recv_count), ref_route.ep_recv_count)
    assert np.array_equal(host(out.expert_token_nums), ref_route.expert_token_nums)
    assert np.array_equal(host(inv), ref_route.inv)
    assert np.array_equal(host(rows[:R]), ref_route.assist[:R])


def smooth_args(wl, src, tok, k):
    """(row, scalar) smooth arguments of oracle.quant_row for one routed row."""
    if not uses_smooth(wl):
        return None, None
    kind = wl.cfg.get("smooth_kind", 0)
    if kind == 2:
        return None, float(wl.smooth.reshape(-1)[0])
    if kind == 1:
        return wl.smooth.reshape(-1), None
    K = wl.cfg["topk"]
    s_eff = wl.cfg["shared_expert_num"] if wl.cfg["shared_expert_rank_num"] > 0 else 0
    return (wl.smooth[s_eff + wl.expert_ids[src, tok, k]] if k < K else wl.smooth[k - K]), None


class FfnStandin:
    """Expert-output stand-in: row n of expand_x_ffn is pool[(n * 7919) % P]
    for a seeded random pool of P bf16 rows. The device copy is gathered on
    the GPU; the oracle reads the pool through a remapped row table, which
    leaves its arithmetic unchanged."""

    def __init__(self, wl, max_rows: int, pool_rows: int = 4096):
        xd = wl.cfg.get("x_dtype", 0)
        self.pool = workloads.ffn_standin(wl.seed, pool_rows, wl.cfg["hidden"], x_dtype=xd)
        self.P = pool_rows
        idx = (torch.arange(max_rows, dtype=torch.int64, device=DEV) * 7919) % pool_rows
        tdt = torch.float16 if xd == 1 else torch.bfloat16
        self.device_rows = dev(self.pool, tdt).index_select(0, idx).contiguous()

    def remap_inv(self, inv: np.ndarray) -> np.ndarray:
        inv = inv.astype(np.int64)
        return np.where(inv >= 0, (inv * 7919) % self.P, inv).astype(np.int32)


def gpu_combine(wl, cfg, out, ffn: FfnStandin, out_dtype):
    """out_dtype: torch.float32 or None (the token type)."""
    w = dev(wl.expert_scales, torch.float32)
    return cq.combine(cfg, ffn.device_rows, out.assist_info, w, out.ep_recv_count,
                      ori_x=dev(wl.x, cfg.token_dtype),
                      const_alpha1=dev(wl.const_alpha1, torch.float32),
                      const_alpha2=dev(wl.const_alpha2, torch.float32),
                      const_v=dev(wl.const_v, cfg.token_dtype), out_dtype=out_dtype)


def oracle_combine_tokens(wl, ref_route, ffn: FfnStandin, tokens, out_f32):
    return oracle.combine_tokens(wl.cfg, tokens, ffn.pool, ffn.remap_inv(ref_route.inv),
                                 wl.expert_scales, wl.x, wl.const_alpha1, wl.const_alpha2,
                                 wl.const_v, out_f32=out_f32)


def full_parity(wl):
    """Whole dispatch + combine on the GPU against the oracle, every element."""
    cfg, out, status, _ = gpu_dispatch(wl)
    ref = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, wl.smooth if uses_smooth(wl) else None,
                          wl.mask, wl.bs_per_rank, wl.expert_scales)
    assert status == ref["status"]
    route = oracle.Route(ref["rows"], ref["expand_idx"], ref["ep_recv_count"],
                         ref["expert_token_nums"], ref["rank_row_base"], ref["assist"],
                         ref["inv"], ref["status"])
    compare_route(wl, cfg, out, route)
    R = ref["rows"]
    if R:
        got = host(out.expand_x[:R])
        assert np.array_equal(got.view(ref["expand_x"].dtype), ref["expand_x"][:R])
        if ref["dynamic_scales"] is not None:
            g, r = host(out.dynamic_scales[:R]), ref["dynamic_scales"][:R]
            assert np.array_equal(g.view(np.uint8), r.view(np.uint8))
        assert np.array_equal(host(out.expand_scales[:R]), ref["expand_scales"][:R])
    ffn = FfnStandin(wl, cfg.max_rows)
    y32 = host(gpu_combine(wl, cfg, out, ffn, torch.float32))
    y16 = host(gpu_combine(wl, cfg, out, ffn, None))
    assert cq.read_combine_status() == 0, "a combine kernel's bounded wait gave up"
    inv = ffn.remap_inv(route.inv)
    args = (wl.cfg, ffn.pool, inv, wl.expert_scales, wl.x, wl.const_alpha1, wl.const_alpha2,
            wl.const_v)
    r32 = oracle.combine(*args, out_f32=True)
    r16 = oracle.combine(*args, out_f32=False)
    assert np.max(np.abs(y32 - r32)) <= 1e-5
    assert np.max(bf16_ulp_diff(y16, r16)) <= 1
    assert np.array_equal(y32.view(np.uint32), r32.view(np.uint32))
    assert np.array_equal(y16, r16)
    return cfg, out, ref


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units of last place between two arrays of 16-bit float
    bit patterns (bf16 or fp16: both order like sign-magnitude integers)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7fff), b & 0x7fff)
    return np.abs(key(a_bits) - key(b_bits))


# ---------------------------------------------------------------------------
# Element-complete comparison at full size. The oracle works token by token
# (its C calls release the GIL, so a thread pool spreads them over the host
# cores); the GPU outputs are copied back in chunks of tokens, so host memory
# stays bounded whatever the workload's size.

_POOL = None


def pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _quant_expect(wl, src, tok, k):
    sm_row, sm_scalar = smooth_args(wl, src, tok, k)
    return oracle.quant_row(wl.cfg["quant_mode"], wl.x[src, tok], sm_row,
                            wl.cfg.get("x_dtype", 0), sm_scalar, wl.cfg.get("y_dtype", 0))


def compare_rows_complete(wl, out, ref_route, tok_chunk: int = 512) -> int:
    """Every dispatched row against the oracle's quantisation of its source
    token (per routed slot when the smooth scales differ per expert, else once
    per token): codes, carried scales and routing weights bit for bit. The
    rows are reached through the inverse map, which compare_route has already
    matched with the oracle's; returns the number of rows checked (all R)."""
    cfg = wl.cfg
    mode, K = cfg["quant_mode"], cfg["topk"]
    W, BS = cfg["ep_world_size"], cfg["max_bs"]
    NS = ref_route.inv.shape[2]
    per_slot = uses_smooth(wl) and cfg.get("smooth_kind", 0) == 0
    inv = ref_route.inv.reshape(W * BS, NS)
    checked = 0
    for t0 in range(0, W * BS, tok_chunk):
        sub = inv[t0:t0 + tok_chunk]
        tt, kk = np.nonzero(sub >= 0)
        if tt.size == 0:
            continue
        rows = sub[tt, kk].astype(np.int64)
        idx = torch.from_numpy(rows).to(DEV)
        ex = host(out.expand_x.index_select(0, idx))
        dyn = host(out.dynamic_scales.index_select(0, idx)) if out.dynamic_scales is not None \
            else None
        es = host(out.expand_scales.index_select(0, idx)) if out.expand_scales is not None \
            else None
        toks = t0 + tt
        keys = list(zip(toks.tolist(), kk.tolist())) if per_slot else \
            sorted(set((t, 0) for t in toks.tolist()))
        exp = dict(zip(keys, pool().map(
            lambda key: _quant_expect(wl, key[0] // BS, key[0] % BS, key[1]), keys)))
        for n in range(rows.size):
            t, k = int(toks[n]), int(kk[n])
            codes, scale = exp[(t, k) if per_slot else (t, 0)]
            assert np.array_equal(ex[n].view(codes.dtype), codes), f"expand_x row {rows[n]}"
            if mode == 2:
                assert dyn[n].view(np.uint32) == np.float32(scale).view(np.uint32), \
                    f"dynamic_scales row {rows[n]}"
            elif mode == 3:
                assert np.array_equal(dyn[n].view(np.uint32), scale.view(np.uint32)), \
                    f"group scales row {rows[n]}"
            elif mode in (4, 5):
                assert np.array_equal(dyn[n], scale), f"mx scales row {rows[n]}"
            if es is not None:
                src, tok = divmod(t, BS)
                want = wl.expert_scales[src, tok, k] if k < K else np.float32(1.0)
                assert es[n] == want, f"expand_scales row {rows[n]}"
        checked += rows.size
    assert checked == ref_route.rows
    return checked


def _oracle_combine_chunk(fn, toks, n_parts):
    parts = [toks[i::n_parts] for i in range(n_parts)]  # some may be empty
    res = list(pool().map(fn, parts))
    out = np.empty((len(toks),) + res[0].shape[1:], res[0].dtype)
    for i, r in enumerate(res):
        out[i::n_parts][:len(r)] = r
    return out


def compare_combine_complete(wl, y32: torch.Tensor, y16: torch.Tensor, oracle_tokens,
                             tok_chunk: int = 1024) -> int:
    """Every token of y (fp32 and the token type) against the oracle:
    within 1e-5 and 1 ulp, and exactly equal (the same operation order).
    oracle_tokens(tokens, out_f32) -> [len(tokens), H]."""
    W, BS = wl.cfg["ep_world_size"], wl.cfg["max_bs"]
    g32v = y32.view(W * BS, -1)
    g16v = y16.view(W * BS, -1)
    n = max(1, min(32, os.cpu_count() or 1))
    for t0 in range(0, W * BS, tok_chunk):
        t1 = min(W * BS, t0 + tok_chunk)
        toks = [divmod(t, BS) for t in range(t0, t1)]
        g32 = host(g32v[t0:t1])
        g16 = host(g16v[t0:t1])
        r32 = _oracle_combine_chunk(lambda p: oracle_tokens(p, True), toks, n)
        r16 = _oracle_combine_chunk(lambda p: oracle_tokens(p, False), toks, n)
        assert np.max(np.abs(g32 - r32)) <= 1e-5, f"tokens {t0}..{t1}"
        assert np.max(bf16_ulp_diff(g16, r16)) <= 1, f"tokens {t0}..{t1}"
        assert np.array_equal(g32.view(np.uint32), r32.view(np.uint32)), f"tokens {t0}..{t1}"
        assert np.array_equal(g16, r16), f"tokens {t0}..{t1}"
    return W * BS
