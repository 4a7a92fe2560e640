"""Pins for the oracle's quantisation (modes 0, 2, 5) and its number formats.

The e4m3 codec is checked against torch's float8_e4m3fn type (a library
decode table and cast) and a brute-force nearest-even search; bf16 rounding
against torch's cast; int8 quantisation against a hand-worked row, a torch
composition and its error bound; the mx block scale against the definition of
ceil(log2) checked with exact float64 comparisons.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from combine_quant_gb300.workloads import bf16_bits_to_f32, to_bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3_table():
    """Decoded value of every e4m3fn code, from torch's own type."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _brute_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 code by exhaustive search, ties to the even code,
    magnitudes above 448 saturated to 448."""
    table = _torch_e4m3_table()
    pos = np.arange(0, 0x7f)          # finite non-negative codes 0x00..0x7e
    vals = table[pos]
    out = np.empty(v.shape, np.uint8)
    for s in range(0, v.size, 50_000):
        a = np.minimum(np.abs(v[s:s + 50_000].astype(np.float64)), 448.0)
        d = np.abs(a[:, None] - vals[None, :])
        cand = d == d.min(axis=1, keepdims=True)
        # among equally near codes prefer the one with an even mantissa (code & 1 == 0)
        even = cand & ((pos[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[s:s + 50_000] = pos[pick]
    return np.where(np.signbit(v), out | 0x80, out).astype(np.uint8)


def test_e4m3_decode_matches_torch(oracle_lib):
    table = _torch_e4m3_table()
    for b in range(256):
        got = oracle.e4m3_decode(b)
        if np.isnan(table[b]):
            assert np.isnan(got)
        else:
            assert got == table[b], b


def test_e4m3_encode_every_bf16(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bf16_bits_to_f32(bits)
    v = v[~np.isnan(v)]
    got = oracle.e4m3_encode_array(v)
    want = _brute_e4m3(np.where(np.isinf(v), np.sign(v) * 1e30, v).astype(np.float32))
    assert np.array_equal(got, want)


def test_e4m3_encode_ties_and_random_f32(oracle_lib):
    table = _torch_e4m3_table()
    fin = np.sort(np.unique(table[:0x7f]))
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)  # exact ties in binary32
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9))])
    rng = np.random.default_rng(0)
    rnd = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-12, 9, 200_000))).astype(
        np.float32)
    v = np.concatenate([near, -near, rnd]).astype(np.float32)
    got = oracle.e4m3_encode_array(v)
    assert np.array_equal(got, _brute_e4m3(v))
    # torch's round-to-nearest-even cast agrees inside the finite range
    inr = np.abs(v) <= 448
    t = torch.from_numpy(v[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], t)


def test_e4m3_saturates(oracle_lib):
    for v, want in ((448.0, 0x7e), (449.0, 0x7e), (463.9, 0x7e), (1e9, 0x7e),
                    (float("inf"), 0x7e), (-500.0, 0xfe)):
        assert oracle.e4m3_encode(v) == want


def test_bf16_rounding_matches_torch(oracle_lib):
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(300_000).astype(np.float32),
        (rng.standard_normal(100_000) * 1e30).astype(np.float32),
        # exact halfway cases between adjacent finite bf16 values, both signs
        ((rng.integers(0x0080, 0x7f7f, 100_000).astype(np.uint32) << 16) | 0x8000
         | (rng.integers(0, 2, 100_000).astype(np.uint32) << 31)).view(np.float32),
        np.array([3.3895314e38, 3.4e38, -3.4e38], np.float32),
    ])
    assert np.array_equal(oracle.bf16_from_f32_array(v), to_bf16_bits(v))


def test_ceil_log2_definition(oracle_lib):
    """2^(e-1) < q <= 2^e, checked exactly in float64, around every power of two."""
    k = np.arange(-40, 120)
    p = np.exp2(k).astype(np.float32)
    q = np.concatenate([p, np.nextafter(p, np.float32(0)), np.nextafter(p, np.float32(np.inf)),
                        np.random.default_rng(2).uniform(1e-7, 1e30, 50_000).astype(np.float32)])
    e = oracle.ceil_log2_array(q).astype(np.float64)
    qd = q.astype(np.float64)
    assert np.all(np.exp2(e - 1) < qd) and np.all(qd <= np.exp2(e))


def test_int8_worked_row(oracle_lib):
    g = json.load(open(os.path.join(GOLD, "int8_row.json")))
    x = np.zeros(1024, np.float32)
    x[:3] = g["x"]
    codes, scale = oracle.quant_row(2, to_bf16_bits(x))
    assert codes[:3].tolist() == g["codes"]
    assert np.all(codes[3:] == 0)
    assert scale == np.float32(1.0) / np.float32(g["dynamic_scales_value"])


@pytest.mark.parametrize("with_smooth", [False, True])
def test_int8_matches_torch_composition(oracle_lib, with_smooth):
    rng = np.random.default_rng(3)
    H = 2048
    for t in range(20):
        xf = (rng.standard_normal(H) * np.exp(rng.normal(0, 2))).astype(np.float32)
        if t == 0:
            xf[7] = 1e4  # an outlier dominating the row
        xb = to_bf16_bits(xf)
        sm = rng.uniform(0.5, 1.5, H).astype(np.float32) if with_smooth else None
        codes, scale = oracle.quant_row(2, xb, sm)
        x32 = torch.from_numpy(bf16_bits_to_f32(xb))
        if sm is not None:
            x32 = x32 * torch.from_numpy(sm)
        s = torch.tensor(127.0, dtype=torch.float32) / x32.abs().max()
        want = torch.round(x32 * s).clamp(-128, 127).to(torch.int8).numpy()
        assert np.array_equal(codes, want)
        assert scale == (torch.tensor(1.0, dtype=torch.float32) / s).item()
        # dequantised values lie within half a step of x_fp32 (plus binary32 slack)
        err = np.abs(codes.astype(np.float64) * scale - x32.numpy().astype(np.float64))
        assert np.all(err <= 0.5 * scale * (1 + 1e-5) + 1e-30)
        assert np.abs(codes).max() == 127


def test_int8_all_zero_row(oracle_lib):
    codes, scale = oracle.quant_row(2, np.zeros(1024, np.uint16))
    assert np.all(codes == 0) and scale == 0.0


@pytest.mark.parametrize("amax,e", [(448.0, 0), (450.0, 1), (896.0, 1), (900.0, 2),
                                    (1.0, -8), (-2.0, -7), (1e-5, -22), (0.0, -22)])
def test_mx_block_scale_special_cases(oracle_lib, amax, e):
    """Block maxima chosen exact in bf16: 448 -> 2^0, just above 448 -> 2^1,
    tiny or zero blocks clamp to 1e-4 -> 2^-22 (1e-4/448 ~ 2^-22.09)."""
    x = np.zeros(64, np.float32)
    x[3] = amax
    x[40] = -0.5  # second block: 0.5/448 ~ 2^-9.8 -> 2^-9
    codes, sc = oracle.quant_row(5, to_bf16_bits(x))
    assert int(sc[0]) - 127 == e
    assert int(sc[1]) - 127 == -9
    assert oracle.e4m3_decode(int(codes[3])) * 2.0 ** e == pytest.approx(
        float(bf16_bits_to_f32(to_bf16_bits(np.float32(amax)).reshape(1))[0]), rel=2 ** -4,
        abs=2.0 ** (e - 10))
    assert np.all(codes[[0, 1, 2, 4, 5]] == 0)


def test_mx_row_properties(oracle_lib):
    rng = np.random.default_rng(4)
    table = _torch_e4m3_table()
    for H in (1024, 1056, 7168):
        xf = (rng.standard_normal(H) * rng.lognormal(0, 1)).astype(np.float32)
        xf[rng.integers(0, H, 5)] *= 30
        xb = to_bf16_bits(xf)
        x = bf16_bits_to_f32(xb).astype(np.float64)
        codes, sc = oracle.quant_row(5, xb)
        nblk = (H + 31) // 32
        assert sc.shape[0] == (nblk + 1) // 2 * 2
        assert np.all(sc[nblk:] == 0)
        for b in range(nblk):
            blk = slice(32 * b, min(32 * b + 32, H))
            e = int(sc[b]) - 127
            a = max(np.abs(x[blk]).max(), np.float64(np.float32(1e-4)))
            q = np.float64(np.float32(a) / np.float32(448.0))
            assert 2.0 ** (e - 1) < q <= 2.0 ** e
            v = x[blk] * 2.0 ** -e                    # exact in float64
            assert np.all(np.abs(v) <= 448.0 * (1 + 2 ** -20))
            # codes are the nearest-even e4m3 values of x / 2^e
            assert np.array_equal(codes[blk], _brute_e4m3(v.astype(np.float32)))
            deq = table[codes[blk]] * 2.0 ** e
            rel = np.abs(deq - x[blk]) <= np.maximum(np.abs(x[blk]) * 2 ** -4, 2.0 ** (e - 10))
            assert np.all(rel)


def test_mode0_is_copy(oracle_lib):
    xb = np.random.default_rng(5).integers(0, 65535, 1024).astype(np.uint16)
    codes, scale = oracle.quant_row(0, xb)
    assert np.array_equal(codes, xb) and scale is None


def test_int8_two_step_rounding_on_ties(oracle_lib):
    """The method rounds the product to binary32 first and then to an
    integer, nearest even ("low_latency_dispatch" 计算公式, quant_mode 2). For
    rows with max A the code of A/2 is RNE(fl(A/2 * fl(127/A))); wherever
    that rounded product is the tie 63.5 (exact value off by less than an
    ulp), the code is 64, while rounding the exact product once would give 63
    where it lies below 63.5. Exact ties k + 0.5 at scale 1 go to even."""
    bits = np.arange(1, 0x7f80, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    below = above = 0
    for A in vals[(vals >= 1.0) & (vals <= 127.0)]:
        s = np.float32(127.0) / A
        h = np.float32(A / 2)
        exact = np.float64(h) * np.float64(s)
        if np.float32(h * s) != np.float32(63.5) or exact == 63.5:
            continue
        row = np.zeros(256, np.float32)
        row[0], row[1], row[2] = A, h, -h
        codes, scale = oracle.quant_row(2, to_bf16_bits(row))
        assert codes[0] == 127 and codes[1] == 64 and codes[2] == -64, A
        below += exact < 63.5
        above += exact > 63.5
    assert below > 100 and above > 100  # both sides of the tie are exercised
    halves = np.arange(127, dtype=np.float32) + np.float32(0.5)
    row = np.zeros(256, np.float32)
    row[:127] = halves
    row[127] = 127.0
    codes, _ = oracle.quant_row(2, to_bf16_bits(row))
    k = np.arange(127)
    assert np.array_equal(codes[:127], np.where(k % 2 == 0, k, k + 1))  # k + 0.5 -> even
    assert codes[127] == 127
