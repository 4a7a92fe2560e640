"""Pins for the oracle's whole dispatch: each placed row holds the quantised
source token (with the smooth row of its expert), and its carried weight."""
import numpy as np
import pytest

import oracle
from combine_quant_gb300 import workloads


@pytest.mark.parametrize("mode", [0, 2, 5])
def test_dispatch_rows_are_quantised_sources(oracle_lib, mode):
    wl = workloads.tiny(seed=11, quant_mode=mode)
    out = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, wl.smooth, expert_scales=wl.expert_scales)
    K = wl.cfg["topk"]
    assert out["rows"] == wl.x.shape[0] * wl.x.shape[1] * K
    for n in range(out["rows"]):
        src, tok, k = out["assist"][n, :3]
        e = wl.expert_ids[src, tok, k]
        sm = None if wl.smooth is None else wl.smooth[e]   # no shared experts: row e
        codes, scale = oracle.quant_row(mode, wl.x[src, tok], sm)
        assert np.array_equal(out["expand_x"][n], codes)
        if mode == 2:
            assert out["dynamic_scales"][n] == scale
        if mode == 5:
            assert np.array_equal(out["dynamic_scales"][n], scale)
        assert out["expand_scales"][n] == wl.expert_scales[src, tok, k]


def test_dispatch_shared_smooth_rows(oracle_lib):
    """With shared experts the smooth table is (S + M, H): shared expert s uses
    row s and MoE expert e uses row S + e; shared rows carry weight 1."""
    W, Sr, S, L, K, BS, H = 4, 2, 2, 2, 2, 3, 1024
    M = L * (W - Sr)
    cfg = workloads.make_config(ep_world_size=W, moe_expert_num=M, shared_expert_num=S,
                                shared_expert_rank_num=Sr, max_bs=BS, topk=K, hidden=H,
                                quant_mode=2)
    rng = np.random.default_rng(12)
    ids = np.stack([rng.permutation(M)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    x = workloads.to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    sm = rng.uniform(0.5, 1.5, (S + M, H)).astype(np.float32)
    w = rng.uniform(0, 1, (W, BS, K)).astype(np.float32)
    out = oracle.dispatch(cfg, x, ids, sm, expert_scales=w)
    assert out["rows"] == W * BS * (K + S)
    for n in range(out["rows"]):
        src, tok, k = out["assist"][n, :3]
        srow = S + ids[src, tok, k] if k < K else k - K
        codes, scale = oracle.quant_row(2, x[src, tok], sm[srow])
        assert np.array_equal(out["expand_x"][n], codes)
        assert out["dynamic_scales"][n] == scale
        assert out["expand_scales"][n] == (w[src, tok, k] if k < K else 1.0)


def test_mode5_rejects_smooth(oracle_lib):
    wl = workloads.tiny(seed=1, quant_mode=5)
    with pytest.raises(ValueError):
        oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, np.ones((8, 1024), np.float32))
