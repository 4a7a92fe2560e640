"""Pins for the oracle's routing (scan, counts, prefix sums, placement).

Each test checks the oracle against something other than itself: values the
design page prints, a hand-worked case, a brute-force recount, a sort-based
re-derivation of the layout, or the page's own position / address formulas.
"""
# Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
# top of include/cq.h.
import json
import os

import numpy as np
import pytest

import oracle
from combine_quant_gb300.workloads import make_config

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_hand_case(oracle_lib):
    g = _gold("hand_case_w2.json")
    for etype, key in ((1, "expert_token_nums_type1"), (0, "expert_token_nums_type0")):
        cfg = make_config(**g["config"], expert_token_nums_type=etype)
        r = oracle.route(cfg, np.array(g["expert_ids"], np.int32),
                         bs_per_rank=np.array(g["bs_per_rank"], np.int32))
        assert r.rows == 10
        assert r.expand_idx.tolist() == g["expand_idx"]
        assert r.ep_recv_count.tolist() == g["ep_recv_count"]
        assert r.expert_token_nums.tolist() == g[key]
        assert r.rank_row_base.tolist() == g["rank_row_base"]
        assert r.assist[:10, :3].tolist() == g["rows_src_token_slot"]


def test_dsn_prefix_example(oracle_lib):
    """The page's prefix-sum sendCounts example, reproduced on destination rank 0."""
    g = _gold("dsn_prefix_example.json")
    W, L = g["ep_world_size"], g["local_expert_num"]
    # Per-source routing (K=1, BS=6) chosen so that rank 0's experts 0 and 1
    # receive [1,0,1,1] and [0,5,2,2] rows from sources 0..3; other tokens go
    # to experts on other ranks.
    ids = np.array([[0, 2, 2, 2, 2, 2],
                    [1, 1, 1, 1, 1, 2],
                    [0, 1, 1, 2, 2, 2],
                    [0, 1, 1, 3, 3, 3]], np.int32)[..., None]
    cfg = make_config(ep_world_size=W, moe_expert_num=W * L, max_bs=6, topk=1, hidden=1024)
    r = oracle.route(cfg, ids)
    got = r.ep_recv_count[0].reshape(L, W)
    assert got.tolist() == g["prefix_matrix"]
    d = g["derived"]
    assert got[0, 1] - got[0, 0] == d["expert0_to_rank1_rows"]
    assert got[1, 1] - got[1, 0] == d["expert1_to_rank1_rows"]
    # The first row expert 1 received from rank 1 sits at offset sendCounts(1,0).
    rows = [n for n in range(r.rows) if r.assist[n, 0] == 1 and r.assist[n, 2] == 0
            and ids[1, r.assist[n, 1], 0] == 1]
    assert min(rows) - r.rank_row_base[0] == d["expert1_rank1_start"]


def _brute(cfg, ids, mask=None, bpr=None):
    """Pure-Python restatement for tiny inputs: expandIdx by counting earlier
    equal ids, then the layout by sorting on (dest, local, src, expandIdx)."""
    W, M, K, BS = cfg["ep_world_size"], cfg["moe_expert_num"], cfg["topk"], cfg["max_bs"]
    Sr, S = cfg["shared_expert_rank_num"], cfg["shared_expert_num"]
    Seff = S if Sr > 0 else 0
    L = M // (W - Sr)
    R = Sr // S if Sr > 0 else 0
    NS = K + Seff
    eidx = -np.ones((W, BS, NS), np.int64)
    keys = []
    for r in range(W):
        n_r = BS if bpr is None else int(bpr[r])
        seen = []       # MoE ids of earlier active pairs of this source
        n_tok = 0       # earlier active tokens of this source
        for i in range(n_r):
            any_on = False
            for j in range(K):
                if mask is not None:
                    on = mask[r, i] if mask.ndim == 2 else mask[r, i, j]
                    if not on:
                        continue
                any_on = True
                e = int(ids[r, i, j])
                if 0 <= e < M:
                    eidx[r, i, j] = sum(1 for p in seen if p == e)
                    seen.append(e)
                    keys.append((Sr + e // L, e % L, r, eidx[r, i, j], (r, i, j)))
            if any_on:
                for s in range(Seff):
                    eidx[r, i, K + s] = n_tok
                    keys.append((s * R + r % R, 0, r, n_tok, (r, i, K + s)))
                n_tok += 1
    keys.sort()
    return eidx, [k[4] for k in keys]


def _rand_ids(rng, W, BS, K, n_ids):
    return np.stack([rng.permutation(n_ids)[:K] for _ in range(W * BS)]).reshape(
        W, BS, K).astype(np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_small(oracle_lib, seed):
    rng = np.random.default_rng(seed)
    W = int(rng.choice([2, 3, 4, 6]))
    Sr = int(rng.choice([0, W // 2 if W % 2 == 0 and W > 2 else 0]))
    S = 1 if Sr == 0 else int(rng.choice([s for s in (1, 2) if Sr % s == 0]))
    L = int(rng.integers(1, 4))
    M = L * (W - Sr)
    K = int(rng.integers(1, min(M, 5) + 1))
    BS = int(rng.integers(1, 9))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, shared_expert_num=S,
                      shared_expert_rank_num=Sr, max_bs=BS, topk=K, hidden=1024)
    ids = _rand_ids(rng, W, BS, K, M)
    bpr = rng.integers(0, BS + 1, W).astype(np.int32) if seed % 2 else None
    r = oracle.route(cfg, ids, bs_per_rank=bpr)
    eidx, order = _brute(cfg, ids, bpr=bpr)
    assert np.array_equal(r.expand_idx, eidx)
    assert r.rows == len(order)
    assert [tuple(a) for a in r.assist[:r.rows, :3].tolist()] == [tuple(o) for o in order]
    assert r.status == 0


@pytest.mark.parametrize("seed", range(4))
def test_brute_force_masks_and_duplicates(oracle_lib, seed):
    """2-D masks, 1-D prefix masks and duplicate ids inside one token."""
    rng = np.random.default_rng(100 + seed)
    W, L, K, BS = 3, 2, 3, 5
    M = W * L
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=1024,
                      mask_ndim=2 if seed % 2 else 1)
    ids = rng.integers(0, M, (W, BS, K)).astype(np.int32)  # duplicates allowed
    if seed % 2:
        mask = (rng.random((W, BS, K)) < 0.6).astype(np.uint8)
    else:
        mask = np.zeros((W, BS), np.uint8)
        for r in range(W):
            mask[r, :rng.integers(0, BS + 1)] = 1
    r = oracle.route(cfg, ids, mask=mask)
    eidx, order = _brute(cfg, ids, mask=mask)
    assert np.array_equal(r.expand_idx, eidx)
    assert [tuple(a) for a in r.assist[:r.rows, :3].tolist()] == [tuple(o) for o in order]
    assert r.status == 0


def test_bad_mask_and_bad_id_flags(oracle_lib):
    cfg = make_config(ep_world_size=2, moe_expert_num=4, max_bs=3, topk=1, hidden=1024,
                      mask_ndim=1)
    ids = np.zeros((2, 3, 1), np.int32)
    mask = np.array([[1, 0, 1], [1, 1, 0]], np.uint8)  # rank 0 breaks the prefix rule
    assert oracle.route(cfg, ids, mask=mask).status == oracle.ST_BAD_MASK
    ids[1, 1, 0] = 99
    r = oracle.route(cfg, ids, mask=np.ones((2, 3), np.uint8))
    assert r.status == oracle.ST_BAD_ID
    assert r.inv[1, 1, 0] == oracle.INV_NONE and r.expand_idx[1, 1, 0] == -1


def test_target_rank_is_integer_division(oracle_lib):
    """id / L is floor division, with shared-expert ranks placed first."""
    cfg = make_config(ep_world_size=4, moe_expert_num=6, shared_expert_num=1,
                      shared_expert_rank_num=1, max_bs=1, topk=6, hidden=1024)
    ids = np.tile(np.arange(6, dtype=np.int32), (4, 1, 1))
    r = oracle.route(cfg, ids)
    L = 2
    for n in range(r.rows):
        src, tok, k = r.assist[n, :3]
        d = int(np.searchsorted(r.rank_row_base, n, side="right") - 1)
        if k < 6:
            assert d == 1 + ids[src, tok, k] // L
        else:
            assert d == 0  # the single shared-expert rank


def _rank_of_row(rb, n):
    return int(np.searchsorted(rb, n, side="right") - 1)


def _check_invariants(cfg, ids, r, mask=None, bpr=None):
    W, M, K, BS = cfg["ep_world_size"], cfg["moe_expert_num"], cfg["topk"], cfg["max_bs"]
    Sr = cfg["shared_expert_rank_num"]
    L = M // (W - Sr)
    # Every placed row is owned by exactly one slot, and inv / assist invert
    # each other.
    inv = r.inv.reshape(-1)
    placed = inv[inv >= 0]
    assert np.array_equal(np.sort(placed), np.arange(r.rows))
    for n in range(r.rows):
        src, tok, k = r.assist[n, :3]
        assert r.inv[src, tok, k] == n
    # Counts: rows per destination rank sum to the number of routed slots.
    assert r.rank_row_base[-1] == r.rows == placed.size
    for d in range(W):
        Ld = 1 if d < Sr else L
        tot = r.ep_recv_count[d, Ld * W - 1]
        assert tot == r.rank_row_base[d + 1] - r.rank_row_base[d]
        assert np.all(np.diff(r.ep_recv_count[d, :Ld * W]) >= 0)
    # Within one (source, expert) the arrival ordinals are 0..n-1 in scan order.
    for src in range(W):
        for e in range(M):
            sel = (ids[src] == e) & (r.expand_idx[src, :, :K] >= 0)
            got = r.expand_idx[src, :, :K][sel]  # row-major = scan order
            assert np.array_equal(got, np.arange(got.size))


def test_invariants_special_workload_small(oracle_lib):
    from combine_quant_gb300 import workloads
    wl = workloads.special(seed=7, W=8, BS=12, H=1024)
    cfg = dict(wl.cfg, moe_expert_num=48)  # L=8 on 6 MoE ranks
    ids = np.where(wl.expert_ids >= 112, wl.expert_ids - 112 + 48, wl.expert_ids % 48)
    ids = ids.astype(np.int32)
    r = oracle.route(cfg, ids, mask=wl.mask)
    _check_invariants(cfg, ids, r)
    # Special experts own no rows and carry their codes.
    K = cfg["topk"]
    slots = r.inv[:, :, :K]
    on = (wl.mask != 0)[:, :, None]
    assert np.all(slots[(ids == 48) & on] == oracle.INV_NONE)      # zero expert
    assert np.all(slots[(ids == 49) & on] == oracle.INV_COPY)      # copy expert
    assert np.all(slots[(ids == 50) & on] == oracle.INV_CONST_BASE)  # const expert 0
    # Masked tokens own nothing, not even a shared row.
    off = wl.mask == 0
    assert np.all(r.inv[off] == oracle.INV_NONE)
    # Shared slot: ordinal of the token among active tokens of its source.
    act = wl.mask.astype(bool)
    assert np.array_equal(r.expand_idx[:, :, K][act], np.concatenate(
        [np.arange(a.sum()) for a in act]))


def test_send_window_position_formula(oracle_lib):
    """The design page's MoePermute position, expertCumsum(e) - expertCumsum(d*L)
    + expandIdx, orders each (source, destination) window exactly as the
    oracle orders that source's rows on the destination."""
    g = _gold("hand_case_w2.json")
    rng = np.random.default_rng(5)
    W, L, K, BS = 4, 3, 3, 7
    M = W * L
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=1024)
    ids = _rand_ids(rng, W, BS, K, M)
    r = oracle.route(cfg, ids)
    for src in range(W):
        cnt = np.bincount(ids[src].reshape(-1), minlength=M)
        excl = np.concatenate([[0], np.cumsum(cnt)[:-1]])
        for d in range(W):
            pos, rows = [], []
            for i in range(BS):
                for j in range(K):
                    e = ids[src, i, j]
                    if e // L != d:
                        continue
                    pos.append(excl[e] - excl[d * L] + r.expand_idx[src, i, j])
                    rows.append(r.inv[src, i, j])
            assert sorted(pos) == list(range(len(pos)))
            assert np.array_equal(np.argsort(pos), np.argsort(rows))
    # And the page's worked instance on the hand case.
    ids = np.array(g["expert_ids"], np.int32)
    cnt0 = np.bincount(ids[0].reshape(-1), minlength=4)
    excl0 = np.concatenate([[0], np.cumsum(cnt0)[:-1]])
    e = ids[0, 0, 0]
    assert excl0[e] - excl0[(e // 2) * 2] + 0 == g["send_window_position_rank0_pair00"]


def test_combine_address_formula(oracle_lib):
    """Design page §3.4.2: a row sits at the rank's window base, plus the
    offset of its expert's (and, here, its source's) block, plus expandIdx."""
    rng = np.random.default_rng(9)
    W, L, K, BS = 5, 2, 4, 9
    M = W * L
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=1024)
    ids = _rand_ids(rng, W, BS, K, M)
    r = oracle.route(cfg, ids)
    for src in range(W):
        cnt = np.bincount(ids[src].reshape(-1), minlength=M)
        for i in range(BS):
            for j in range(K):
                e = ids[src, i, j]
                d, le = e // L, e % L
                incl = r.ep_recv_count[d, le * W + src]
                block = r.rank_row_base[d] + incl - cnt[e]
                assert r.inv[src, i, j] == block + r.expand_idx[src, i, j]


def test_expert_token_nums_types(oracle_lib):
    rng = np.random.default_rng(3)
    W, L, K, BS = 4, 4, 4, 10
    cfg = make_config(ep_world_size=W, moe_expert_num=W * L, max_bs=BS, topk=K, hidden=1024)
    ids = _rand_ids(rng, W, BS, K, W * L)
    r1 = oracle.route(dict(cfg, expert_token_nums_type=1), ids)
    r0 = oracle.route(dict(cfg, expert_token_nums_type=0), ids)
    counts = np.bincount(ids.reshape(-1), minlength=W * L).reshape(W, L)
    assert np.array_equal(r1.expert_token_nums, counts)
    assert np.array_equal(r0.expert_token_nums, np.cumsum(counts, axis=1))
    # The last column of each expert's prefix row equals the cumulative count.
    for d in range(W):
        assert np.array_equal(r0.ep_recv_count[d].reshape(L, W)[:, -1], r0.expert_token_nums[d])


@pytest.mark.parametrize("bad", [
    dict(ep_world_size=1), dict(ep_world_size=769), dict(hidden=1023), dict(hidden=8193),
    dict(max_bs=0), dict(max_bs=513), dict(topk=0), dict(topk=17), dict(moe_expert_num=1025),
    dict(moe_expert_num=30),                      # not a multiple of W - S_r
    dict(shared_expert_num=2),                    # S_r == 0 needs S in {0, 1}
    dict(shared_expert_rank_num=3, shared_expert_num=2, moe_expert_num=13 * 4),
    dict(global_bs=5), dict(quant_mode=7), dict(expert_token_nums_type=2), dict(mask_ndim=3),
    dict(ep_world_size=768, moe_expert_num=768 * 3),  # L * W > 2048
])
def test_config_rejections(oracle_lib, bad):
    cfg = make_config(ep_world_size=16, moe_expert_num=64, max_bs=8, topk=4, hidden=1024)
    cfg.update(bad)
    assert oracle.check_config(cfg) != 0


def test_config_modes_and_types(oracle_lib):
    """quant_mode 0..5 ([LLD] 计算公式), x as bf16 / fp16, three scales shapes."""
    cfg = make_config(ep_world_size=16, moe_expert_num=64, max_bs=8, topk=4, hidden=1024)
    for m in range(6):
        assert oracle.check_config(dict(cfg, quant_mode=m)) == 0
    assert oracle.check_config(dict(cfg, quant_mode=6)) == oracle.ERR_ARG
    assert oracle.check_config(dict(cfg, x_dtype=1)) == 0
    assert oracle.check_config(dict(cfg, x_dtype=2)) == oracle.ERR_ARG
    for k in range(3):
        assert oracle.check_config(dict(cfg, smooth_kind=k)) == 0
    assert oracle.check_config(dict(cfg, smooth_kind=3)) == oracle.ERR_ARG
