"""Host logic of the seeded workloads and of the bench's oracle sampling:
which smooth scales a workload carries under another quant_mode, and which
smooth argument the oracle gets for each routed slot."""
import sys
import os

import numpy as np

from combine_quant_gb300 import workloads

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_with_mode_keeps_smooth_for_modes_1_to_3():
    wl = workloads.skew(seed=4, W=4, BS=8, M=16, K=4, H=1024)
    assert wl.smooth is not None and wl.cfg["smooth_kind"] == 0
    for mode in (1, 2, 3):
        w = wl.with_mode(mode)
        assert w.cfg["quant_mode"] == mode
        assert w.smooth is wl.smooth and w.cfg["smooth_kind"] == 0
    for mode in (0, 4, 5):
        w = wl.with_mode(mode)
        assert w.smooth is None
    assert np.array_equal(wl.with_mode(0).x, wl.x)


def test_with_mode_1_without_smooth_gets_a_static_row():
    wl = workloads.tiny(seed=3, quant_mode=0)
    assert wl.smooth is None
    w = wl.with_mode(1)
    H = wl.cfg["hidden"]
    assert w.cfg["smooth_kind"] == 1
    assert w.smooth.shape == (H,) and w.smooth.dtype == np.float32
    assert np.all(w.smooth == 32.0)
    assert wl.cfg.get("smooth_kind", 0) == 0  # the original is left as it was


def test_bench_smooth_of_follows_smooth_kind_and_shared_layout():
    """Shared experts' rows come first in the per-expert table; a routed
    slot k < K with expert id e takes row S + e, shared slot K + s row s."""
    wl = workloads.special(seed=23, W=8, BS=4, H=1024, M=48).with_mode(2)
    cfg = wl.cfg
    S, K = cfg["shared_expert_num"], cfg["topk"]
    M = cfg["moe_expert_num"]
    table = np.arange((S + M) * 1024, dtype=np.float32).reshape(S + M, 1024)
    wl.smooth = table
    wl.cfg = dict(cfg, smooth_kind=0)
    r, i = 1, 2
    for k in range(K):
        e = int(wl.expert_ids[r, i, k])
        row, scalar = bench._smooth_of(wl, r, i, k)
        if e < M:
            assert scalar is None and np.array_equal(row, table[S + e])
    row, scalar = bench._smooth_of(wl, r, i, K)  # the shared slot
    assert np.array_equal(row, table[0])
    wl.cfg = dict(cfg, smooth_kind=1)
    wl.smooth = table[0]
    row, scalar = bench._smooth_of(wl, r, i, 0)
    assert np.array_equal(row, table[0]) and scalar is None
    wl.cfg = dict(cfg, smooth_kind=2)
    wl.smooth = np.array([2.5], np.float32)
    assert bench._smooth_of(wl, r, i, 0) == (None, 2.5)
    wl.cfg = dict(cfg, quant_mode=5)
    assert bench._smooth_of(wl, r, i, 0) == (None, None)
