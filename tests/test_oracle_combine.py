"""Pins for the oracle's combine (top-K weighted sum plus shared and special experts).

Checked against closed forms computed independently in float64 (within the
binary32 error bound of a K-step fused multiply-add chain), against single
binary32 products computed by numpy for the copy / const / zero experts, and
against torch's bf16 cast for the final rounding.
"""
import numpy as np
import pytest

import oracle
from combine_quant_gb300.workloads import bf16_bits_to_f32, make_config, to_bf16_bits


def _setup(seed, W=4, L=2, K=3, BS=6, H=1024, Sr=0, S=0, Z=0, C=0, Q=0):
    rng = np.random.default_rng(seed)
    M = L * (W - Sr)
    cfg = make_config(ep_world_size=W, moe_expert_num=M, shared_expert_num=S,
                      shared_expert_rank_num=Sr, zero_expert_num=Z, copy_expert_num=C,
                      const_expert_num=Q, max_bs=BS, topk=K, hidden=H)
    n_ids = M + Z + C + Q
    ids = np.stack([rng.permutation(n_ids)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    ids = ids.astype(np.int32)
    w = rng.uniform(-1, 1, (W, BS, K)).astype(np.float32)
    x = to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    a1 = rng.uniform(0.5, 1.5, Q).astype(np.float32)
    a2 = rng.uniform(0.5, 1.5, Q).astype(np.float32)
    v = to_bf16_bits(rng.standard_normal((Q, H)).astype(np.float32))
    r = oracle.route(cfg, ids)
    ffn = to_bf16_bits(rng.standard_normal((max(r.rows, 1), H)).astype(np.float32))
    return cfg, ids, w, x, a1, a2, v, r, ffn


def _exact(cfg, ids, w, x, a1, a2, v, r, ffn):
    """Float64 value of the weighted sum each token should approximate, and
    the sum of magnitudes that bounds the binary32 rounding error."""
    W, BS, K, H = cfg["ep_world_size"], cfg["max_bs"], cfg["topk"], cfg["hidden"]
    NS = r.inv.shape[2]
    M, Z, C = cfg["moe_expert_num"], cfg["zero_expert_num"], cfg["copy_expert_num"]
    xf = bf16_bits_to_f32(x).astype(np.float64)
    ff = bf16_bits_to_f32(ffn).astype(np.float64)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    exact = np.zeros((W, BS, H))
    mag = np.zeros((W, BS, H))
    for rr in range(W):
        for i in range(BS):
            for j in range(K):
                e = ids[rr, i, j]
                if e < M:
                    t = ff[r.inv[rr, i, j]]
                elif e < M + Z:
                    continue
                elif e < M + Z + C:
                    t = xf[rr, i]
                else:
                    q = e - (M + Z + C)
                    # the const expert's own two products and sum are binary32
                    t = (np.float32(a1[q]) * xf[rr, i].astype(np.float32)
                         + np.float32(a2[q]) * vf[q].astype(np.float32)).astype(np.float64)
                exact[rr, i] += np.float64(w[rr, i, j]) * t
                mag[rr, i] += np.abs(np.float64(w[rr, i, j]) * t)
            for s in range(K, NS):
                t = ff[r.inv[rr, i, s]]
                exact[rr, i] += t
                mag[rr, i] += np.abs(t)
    return exact, mag


@pytest.mark.parametrize("seed,kw", [
    (0, {}),
    (1, dict(K=4, L=3)),
    (2, dict(W=4, Sr=2, S=2, L=2, K=2)),             # two shared experts, one replica each
    (3, dict(W=6, Sr=3, S=1, L=2, K=3, Z=1, C=1, Q=2)),  # shared + every special kind
])
def test_combine_matches_float64_within_bound(oracle_lib, seed, kw):
    cfg, ids, w, x, a1, a2, v, r, ffn = _setup(seed, **kw)
    y32 = oracle.combine(cfg, ffn, r.inv, w, x, a1, a2, v, out_f32=True)
    exact, mag = _exact(cfg, ids, w, x, a1, a2, v, r, ffn)
    NS = r.inv.shape[2]
    bound = NS * 2.0 ** -24 * mag * (1 + 1e-6) + 1e-38
    assert np.all(np.abs(y32.astype(np.float64) - exact) <= bound)
    # the bf16 output is the round-to-nearest-even of the binary32 sum
    yb = oracle.combine(cfg, ffn, r.inv, w, x, a1, a2, v, out_f32=False)
    assert np.array_equal(yb, to_bf16_bits(y32))


def test_identity_ffn_closed_form(oracle_lib):
    """Mode 0 with an identity FFN: every row is its token, so
    y = x * sum_j w_j up to the fma-chain rounding."""
    cfg, ids, w, x, a1, a2, v, r, _ = _setup(4, K=4, L=3)
    ffn = np.zeros((r.rows, cfg["hidden"]), np.uint16)
    for n in range(r.rows):
        src, tok, _k = r.assist[n, :3]
        ffn[n] = x[src, tok]
    y32 = oracle.combine(cfg, ffn, r.inv, w, x, out_f32=True)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    wsum = w.astype(np.float64).sum(axis=2, keepdims=True)
    mag = np.abs(w.astype(np.float64)).sum(axis=2, keepdims=True) * np.abs(xf)
    assert np.all(np.abs(y32 - xf * wsum) <= 4 * 2.0 ** -24 * mag + 1e-38)


def test_single_special_expert_tokens(oracle_lib):
    """One routed slot per token: copy gives fl(w*x), const gives
    fl(w*fl(fl(a1*x)+fl(a2*v))), zero gives 0, all computed by numpy in binary32."""
    W, BS, H = 2, 3, 1024
    cfg = make_config(ep_world_size=W, moe_expert_num=2, zero_expert_num=1, copy_expert_num=1,
                      const_expert_num=1, max_bs=BS, topk=1, hidden=H)
    ids = np.array([[[2], [3], [4]], [[4], [2], [3]]], np.int32)
    rng = np.random.default_rng(6)
    w = rng.uniform(0.1, 1, (W, BS, 1)).astype(np.float32)
    x = to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    a1 = np.array([0.75], np.float32)
    a2 = np.array([1.25], np.float32)
    v = to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))
    r = oracle.route(cfg, ids)
    assert r.rows == 0
    y = oracle.combine(cfg, np.zeros((1, H), np.uint16), r.inv, w, x, a1, a2, v, out_f32=True)
    xf, vf = bf16_bits_to_f32(x), bf16_bits_to_f32(v)[0]
    for rr in range(W):
        for i in range(BS):
            e = ids[rr, i, 0]
            if e == 2:
                want = np.zeros(H, np.float32)
            elif e == 3:
                want = w[rr, i, 0] * xf[rr, i]
            else:
                want = w[rr, i, 0] * (a1[0] * xf[rr, i] + a2[0] * vf)
            assert np.array_equal(y[rr, i], want.astype(np.float32))


def test_inactive_tokens_are_zero(oracle_lib):
    cfg, ids, w, x, a1, a2, v, r, ffn = _setup(7, W=4, Sr=2, S=1, L=2, K=2)
    cfg = dict(cfg, mask_ndim=1)
    mask = np.ones((4, 6), np.uint8)
    mask[:, 4:] = 0
    r = oracle.route(cfg, ids, mask=mask)
    y = oracle.combine(cfg, ffn, r.inv, w, x, out_f32=True)
    assert np.all(y[:, 4:] == 0)
    assert np.all(np.abs(y[:, :4]).sum(axis=2) > 0)


def test_combine_tokens_matches_full(oracle_lib):
    cfg, ids, w, x, a1, a2, v, r, ffn = _setup(8, W=6, Sr=3, S=1, L=2, K=3, Z=1, C=1, Q=2)
    y = oracle.combine(cfg, ffn, r.inv, w, x, a1, a2, v)
    toks = [(0, 0), (5, 5), (3, 2)]
    ys = oracle.combine_tokens(cfg, toks, ffn, r.inv, w, x, a1, a2, v)
    for n, (rr, i) in enumerate(toks):
        assert np.array_equal(ys[n], y[rr, i])
