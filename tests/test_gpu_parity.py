"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Small configurations and the full-size workloads alike are compared element
by element on every output (at full size the oracle runs token by token on a
thread pool and the GPU outputs come back in chunks).
Tolerances: index, count and code outputs bit-exact; the int8 scale and the
mx scale bytes bit-exact; combine within 1e-5 of the fp32 oracle value and
within 1 bf16 ulp after the cast (both kernels use the same fused
multiply-add order, so exact agreement is expected and counted).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_quant_gb300 import workloads

import gpu_harness as gh

pytestmark = pytest.mark.gpu


def _small_cases():
    return {
        "tiny_m0": lambda: workloads.tiny(0, 0),
        "tiny_m2": lambda: workloads.tiny(0, 2),
        "tiny_m5": lambda: workloads.tiny(0, 5),
        "dsv3_small": lambda: workloads.dsv3(seed=21, W=8, BS=37, M=64, K=8, H=2048),
        "mxfp8_small": lambda: workloads.mxfp8(seed=22, W=8, BS=33, M=32, K=8, H=1536),
        "special_small": lambda: workloads.special(seed=23, W=8, BS=20, H=1024, M=48),
        "skew_small": lambda: workloads.skew(seed=24, W=4, BS=64, M=32, K=16, H=2048),
    }


def _check_combine_full(wl, cfg, out, ref_route):
    ffn = gh.FfnStandin(wl, cfg.max_rows)
    y32 = gh.host(gh.gpu_combine(wl, cfg, out, ffn, torch.float32))
    yb = gh.host(gh.gpu_combine(wl, cfg, out, ffn, None))  # the token type
    inv = ffn.remap_inv(ref_route.inv)
    r32 = oracle.combine(wl.cfg, ffn.pool, inv, wl.expert_scales, wl.x, wl.const_alpha1,
                         wl.const_alpha2, wl.const_v, out_f32=True)
    rb = oracle.combine(wl.cfg, ffn.pool, inv, wl.expert_scales, wl.x, wl.const_alpha1,
                        wl.const_alpha2, wl.const_v, out_f32=False)
    assert np.max(np.abs(y32 - r32)) <= 1e-5
    assert np.max(gh.bf16_ulp_diff(yb, rb)) <= 1
    assert np.array_equal(y32.view(np.uint32), r32.view(np.uint32)), "fp32 combine not bit-exact"
    assert np.array_equal(yb, rb), "bf16 combine not bit-exact"


@pytest.mark.parametrize("name", list(_small_cases()))
def test_small_full_parity(name):
    wl = _small_cases()[name]()
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    ref = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, wl.smooth if gh.uses_smooth(wl)
                          else None, wl.mask, wl.bs_per_rank, wl.expert_scales)
    assert status == ref["status"]
    route = oracle.Route(ref["rows"], ref["expand_idx"], ref["ep_recv_count"],
                         ref["expert_token_nums"], ref["rank_row_base"], ref["assist"],
                         ref["inv"], ref["status"])
    gh.compare_route(wl, cfg, out, route)
    R = ref["rows"]
    assert np.array_equal(gh.host(out.expand_x[:R]).view(ref["expand_x"].dtype),
                          ref["expand_x"][:R])
    if ref["dynamic_scales"] is not None:
        assert np.array_equal(gh.host(out.dynamic_scales[:R]), ref["dynamic_scales"][:R])
    assert np.array_equal(gh.host(out.expand_scales[:R]), ref["expand_scales"][:R])
    _check_combine_full(wl, cfg, out, route)


FULL = ["tiny", "dsv3", "mxfp8", "special", "skew", "perf8", "perf256"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity_complete(name):
    """The five workloads at full size and the two shapes of the performance
    table ("CANN MoE Dispatch/Combine 通信算子性能优化实践", 性能数据): every
    routing output, every dispatched row (codes, carried scale, weight) and
    every combined token (fp32 and bf16) against the oracle."""
    wl = workloads.WORKLOADS[name]()
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    ref = oracle.route(wl.cfg, wl.expert_ids, wl.mask, wl.bs_per_rank)
    assert status == ref.status == 0
    gh.compare_route(wl, cfg, out, ref)
    assert gh.compare_rows_complete(wl, out, ref) == ref.rows
    ffn = gh.FfnStandin(wl, cfg.max_rows)
    y32 = gh.gpu_combine(wl, cfg, out, ffn, torch.float32)
    yb = gh.gpu_combine(wl, cfg, out, ffn, None)
    assert gh.cq.read_combine_status() == 0
    inv = ffn.remap_inv(ref.inv)

    def oracle_tokens(toks, out_f32):
        return oracle.combine_tokens(wl.cfg, toks, ffn.pool, inv, wl.expert_scales, wl.x,
                                     wl.const_alpha1, wl.const_alpha2, wl.const_v,
                                     out_f32=out_f32)

    assert gh.compare_combine_complete(wl, y32, yb, oracle_tokens) == \
        wl.cfg["ep_world_size"] * wl.cfg["max_bs"]


def _cfg_case(seed, **kw):
    """A small workload with explicit overrides of the generator's arrays."""
    W, M, BS, K, H = kw.pop("W", 4), kw.pop("M", 8), kw.pop("BS", 8), kw.pop("K", 2), kw.pop(
        "H", 1024)
    mode = kw.pop("mode", 2)
    rng = np.random.default_rng(seed)
    cfg = workloads.make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                                quant_mode=mode, **{k: v for k, v in kw.items()
                                                    if k in workloads.CONFIG_FIELDS})
    ids = np.stack([rng.permutation(M)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    x = workloads.to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    w = rng.uniform(0, 1, (W, BS, K)).astype(np.float32)
    return workloads.Workload("case", cfg, x, ids.astype(np.int32), w, seed=seed)


def _full_check(wl):
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    ref = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, wl.smooth, wl.mask, wl.bs_per_rank,
                          wl.expert_scales)
    assert status == ref["status"]
    route = oracle.Route(ref["rows"], ref["expand_idx"], ref["ep_recv_count"],
                         ref["expert_token_nums"], ref["rank_row_base"], ref["assist"],
                         ref["inv"], ref["status"])
    gh.compare_route(wl, cfg, out, route)
    R = ref["rows"]
    if R:
        assert np.array_equal(gh.host(out.expand_x[:R]).view(ref["expand_x"].dtype),
                              ref["expand_x"][:R])
        if ref["dynamic_scales"] is not None:
            assert np.array_equal(gh.host(out.dynamic_scales[:R]), ref["dynamic_scales"][:R])
    _check_combine_full(wl, cfg, out, route)
    return cfg, out, ref


@pytest.mark.parametrize("mode", [0, 2, 5])
def test_edge_all_tokens_masked(mode):
    wl = _cfg_case(1, mode=mode, mask_ndim=1)
    wl.mask = np.zeros((4, 8), np.uint8)
    cfg, out, ref = _full_check(wl)
    assert ref["rows"] == 0


def test_edge_ragged_and_empty_ranks():
    wl = _cfg_case(2, W=6, M=12, BS=17, K=3)
    wl.bs_per_rank = np.array([0, 17, 1, 5, 0, 16], np.int32)
    _full_check(wl)


@pytest.mark.parametrize("mode", [2, 5])
def test_edge_zero_rows_and_extremes(mode):
    wl = _cfg_case(3, mode=mode, H=2048)
    x = workloads.bf16_bits_to_f32(wl.x).copy()
    x[0, 0] = 0.0                   # all-zero token: int8 scale 0, codes 0; mx clamp 1e-4
    x[0, 1] *= 1e-30                # tiny values
    x[1, 2] *= 1e30                 # huge values
    x[2, 3, ::7] = 0.0
    x[3, 4, 100] = 3.0e38
    wl.x = workloads.to_bf16_bits(x)
    _full_check(wl)


def test_edge_mask_2d_duplicates_invalid_ids():
    wl = _cfg_case(4, W=3, M=6, BS=9, K=4, mask_ndim=2, zero_expert_num=1, copy_expert_num=1)
    rng = np.random.default_rng(4)
    wl.expert_ids = rng.integers(0, 9, (3, 9, 4)).astype(np.int32)  # 8 is out of range
    wl.mask = (rng.random((3, 9, 4)) < 0.7).astype(np.uint8)
    cfg, out, ref = _full_check(wl)
    assert ref["status"] & oracle.ST_BAD_ID


def test_edge_bad_1d_mask_flag():
    wl = _cfg_case(5, mask_ndim=1)
    wl.mask = np.ones((4, 8), np.uint8)
    wl.mask[2, 3] = 0  # a false entry before true ones
    cfg, out, ref = _full_check(wl)
    assert ref["status"] == oracle.ST_BAD_MASK


@pytest.mark.parametrize("H,mode", [(1040, 0), (1040, 2), (1056, 5), (8192, 5), (8192, 2)])
def test_edge_hidden_sizes(H, mode):
    wl = _cfg_case(6, H=H, mode=mode, W=2, M=4, BS=3, K=2)
    _full_check(wl)


def test_edge_minimal_and_maximal_k():
    _full_check(_cfg_case(7, W=2, M=2, BS=1, K=1))
    _full_check(_cfg_case(8, W=2, M=32, BS=5, K=16))


def test_edge_shared_experts_replicas():
    wl = _cfg_case(9, W=8, M=24, BS=6, K=3, shared_expert_num=2, shared_expert_rank_num=4,
                   mode=2)
    wl.smooth = np.random.default_rng(9).uniform(0.5, 1.5, (2 + 24, 1024)).astype(np.float32)
    _full_check(wl)


def test_mx_every_bf16_value():
    """Every finite bf16 value goes through the mx path once (hardware e4m3
    conversion against the oracle's codec)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xff
    bits = bits[exp != 0xff]  # drop inf / NaN
    H = 1024
    n = (bits.size + H - 1) // H
    row = np.zeros(n * H, np.uint16)
    row[:bits.size] = np.random.default_rng(10).permutation(bits)
    W, BS = 2, (n + 1) // 2
    x = np.zeros((W * BS * H,), np.uint16)
    x[:row.size] = row
    wl = _cfg_case(10, W=W, M=2, BS=BS, K=1, mode=5)
    wl.x = x.reshape(W, BS, H)
    _full_check(wl)


def test_determinism_and_split_entry_points():
    import combine_quant_gb300 as cq
    wl = workloads.dsv3(seed=31, W=8, BS=64, M=64, K=8, H=2048)
    cfg, out1, _, ws = gh.gpu_dispatch(wl)
    _, out2, _, _ = gh.gpu_dispatch(wl)
    for a, b in zip(out1, out2):
        if a is not None:
            assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    out3 = cq.alloc_dispatch_outputs(cfg, gh.DEV)
    ids = gh.dev(wl.expert_ids, torch.int32)
    cq.dispatch_route(cfg, ids, workspace=ws, out=out3)
    cq.dispatch_permute(cfg, gh.dev(wl.x, torch.bfloat16), ids,
                        expert_scales=gh.dev(wl.expert_scales, torch.float32), workspace=ws,
                        out=out3)
    R = int(gh.host(cq.assist_views(cfg, out1.assist_info)[2])[-1])
    assert torch.equal(out1.expand_x[:R], out3.expand_x[:R])
    assert torch.equal(out1.dynamic_scales[:R], out3.dynamic_scales[:R])
    assert torch.equal(out1.ep_recv_count, out3.ep_recv_count)


def test_edge_max_world_size():
    """W = 768, the largest rank count: more routing CTAs than SMs (the count
    kernel then lets its dependents launch only when it ends) and the longest
    rank-base prefix."""
    _full_check(_cfg_case(11, W=768, M=768, BS=2, K=8, H=1024))


def test_edge_max_experts_and_k():
    """M = 1024 experts (L = 128 per rank) with K = 16."""
    _full_check(_cfg_case(12, W=8, M=1024, BS=16, K=16, H=1024))


def test_edge_max_bs():
    _full_check(_cfg_case(14, W=4, M=8, BS=512, K=4, H=1024))


def test_edge_count_kernel_widths():
    """The routing scan runs 32 warps per CTA from 256 tokens a CTA on (with
    M = 1024 its per-warp table is 64 KB of shared memory: W = 2, BS = 512
    gives two chunks of 256 tokens per source) and 4 warps up to 32; both
    against the oracle at those edges."""
    _full_check(_cfg_case(15, W=2, M=1024, BS=512, K=16, H=1024))
    _full_check(_cfg_case(16, W=4, M=16, BS=32, K=16, H=1024))


@pytest.mark.parametrize("mode", [2, 3])
def test_edge_max_hidden_shared_and_smooth(mode):
    """H = 8192 with 4 shared experts on 4 ranks and one smooth row per expert:
    the per-expert-smooth kernel at its largest CTA."""
    wl = _cfg_case(13, W=8, M=16, BS=32, K=8, H=8192, mode=mode, shared_expert_num=4,
                   shared_expert_rank_num=4)
    wl.smooth = np.random.default_rng(13).uniform(0.5, 1.5, (4 + 16, 8192)).astype(np.float32)
    _full_check(wl)
