"""Pins for the oracle's combine-side int8 block quantisation and the
dequantising combine ([PERF] Int8QuantProcess / Int8DequantProcess)."""
# Page tags ([DV3], [DSN], [LLD], [PERF]) name the source pages listed at the
# top of include/cq.h.
import json
import os

import numpy as np
import torch

import oracle
from combine_quant_gb300.workloads import bf16_bits_to_f32, make_config, to_bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_block(oracle_lib):
    g = json.load(open(os.path.join(GOLD, "combine_int8_block.json")))
    row = np.zeros(1024, np.float32)
    row[:8] = g["block"]
    codes, scales = oracle.combine_quant_row(to_bf16_bits(row))
    assert codes[:8].tolist() == g["codes"] and scales[0] == g["scale"]
    assert np.all(codes[8:] == 0) and np.all(scales[1:] == 0)  # zero blocks


def test_golden_block_fp16_hop(oracle_lib):
    """[PERF] casts the quotient float -> fp16 -> int8: a hand-worked block whose
    quotients all sit within half an fp16 spacing of a .5 tie, so the two-step
    cast and a single rounding disagree on every value but the block max."""
    g = json.load(open(os.path.join(GOLD, "combine_int8_fp16_hop.json")))
    row = np.zeros(1024, np.float32)
    row[:8] = g["block"]
    bits = to_bf16_bits(row)
    assert np.array_equal(bf16_bits_to_f32(bits)[:8], np.float32(g["block"]))  # exact in bf16
    codes, scales = oracle.combine_quant_row(bits)
    assert hex(int(np.float32(scales[0]).view(np.uint32))) == g["scale_hex"]
    assert codes[:8].tolist() == g["codes"]
    assert codes[:8].tolist() != g["codes_one_rounding"]


def test_matches_torch_composition_and_bound(oracle_lib):
    """The chain Div -> fp16 -> int8 composed from torch's own casts (binary32
    division, .half() rounds to nearest even, torch.round is half-to-even)."""
    rng = np.random.default_rng(0)
    H = 2048
    inv_param = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(127.0, dtype=torch.float32)
    n_hop = 0
    for t in range(10):
        v = (rng.standard_normal(H) * np.exp(rng.normal(0, 3))).astype(np.float32)
        v[rng.integers(0, H, 30)] = 0.0
        bits = to_bf16_bits(v)
        codes, scales = oracle.combine_quant_row(bits)
        x = torch.from_numpy(bf16_bits_to_f32(bits)).view(-1, 8)
        s = x.abs().amax(dim=1) * inv_param
        quot = x / s[:, None]
        q = torch.nan_to_num(torch.round(quot.half().float()), nan=0.0).clamp(-128, 127)
        one = torch.nan_to_num(torch.round(quot), nan=0.0).clamp(-128, 127)
        n_hop += int((q != one).sum())
        assert np.array_equal(scales, s.numpy())
        assert np.array_equal(codes.reshape(-1, 8), q.to(torch.int8).numpy())
        # the fp16 step moves a quotient by at most half an fp16 spacing
        # (2^-5 for |q| < 128), so a code is within 0.5 + 2^-5 steps of v
        deq = codes.astype(np.float64).reshape(-1, 8) * scales[:, None].astype(np.float64)
        err = np.abs(deq - x.numpy().astype(np.float64))
        assert np.all(err <= (0.5 + 2.0 ** -5) * scales[:, None] * (1 + 1e-5) + 1e-38)
    assert n_hop > 0  # the inputs reach quotients where the fp16 step matters


def test_dequantising_combine_float64_bound(oracle_lib):
    rng = np.random.default_rng(1)
    W, L, K, BS, H, Sr, S = 6, 2, 3, 5, 1024, 3, 1
    M = L * (W - Sr)
    cfg = make_config(ep_world_size=W, moe_expert_num=M, shared_expert_num=S,
                      shared_expert_rank_num=Sr, copy_expert_num=1, max_bs=BS, topk=K, hidden=H)
    ids = np.stack([rng.permutation(M + 1)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    ids = ids.astype(np.int32)
    w = rng.uniform(-1, 1, (W, BS, K)).astype(np.float32)
    x = to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    r = oracle.route(cfg, ids)
    ffn = to_bf16_bits(rng.standard_normal((r.rows, H)).astype(np.float32))
    codes, scales = oracle.combine_quant_rows(ffn)
    toks = [(a, b) for a in range(W) for b in range(BS)]
    y = oracle.combine_tokens_q8(cfg, toks, codes, scales, r.inv, w, x, out_f32=True)
    deq = codes.astype(np.float64) * np.repeat(scales.astype(np.float64), 8, axis=1)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    NS = r.inv.shape[2]
    for n, (a, b) in enumerate(toks):
        exact = np.zeros(H)
        mag = np.zeros(H)
        for k in range(NS):
            code = r.inv[a, b, k]
            wk = np.float64(w[a, b, k]) if k < K else 1.0
            if code >= 0:
                t = deq[code].astype(np.float32).astype(np.float64)  # dequantised in binary32
            elif code == oracle.INV_COPY:
                t = xf[a, b]
            else:
                continue
            exact += wk * t
            mag += np.abs(wk * t)
        assert np.all(np.abs(y[n] - exact) <= NS * 2.0 ** -24 * mag * (1 + 1e-6) + 1e-38)
    # bf16 output is the rounding of the float32 one
    yb = oracle.combine_tokens_q8(cfg, toks, codes, scales, r.inv, w, x, out_f32=False)
    assert np.array_equal(yb, to_bf16_bits(y))
