"""Pins for the oracle's e5m2 code type (y_dtype 1) of quant_mode 3, 4, 5.

"low_latency_dispatch" lists float8_e5m2 beside float8_e4m3fn as an output
type (y_dtype) and defines emax as the exponent of the type's largest normal
value; the pergroup formula divides the type's largest value (dst_type_max)
by the group max. For e5m2 these are 57344 = 1.75 * 2^15 and 15.

The codec is checked against torch's float8_e5m2 type (its decode table and
its round-to-nearest-even cast) and a brute-force nearest-even search; the
mode formulas against a torch / float64 composition of the definitions."""
import numpy as np
import pytest
import torch

import oracle
from combine_quant_gb300 import workloads
from combine_quant_gb300.workloads import bf16_bits_to_f32, to_bf16_bits

MAX = 57344.0


def _torch_table():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e5m2).to(torch.float64).numpy()


def _brute(v: np.ndarray) -> np.ndarray:
    """Nearest finite e5m2 code by exhaustive search, ties to the even code,
    magnitudes above 57344 saturated; NaN gives 0x7f."""
    table = _torch_table()
    pos = np.arange(0, 0x7c)  # finite non-negative codes 0x00..0x7b
    vals = table[pos]
    out = np.empty(v.shape, np.uint8)
    for s in range(0, v.size, 50_000):
        a = np.minimum(np.abs(v[s:s + 50_000].astype(np.float64)), MAX)
        d = np.abs(a[:, None] - vals[None, :])
        cand = d == d.min(axis=1, keepdims=True)
        even = cand & ((pos[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[s:s + 50_000] = pos[pick]
    out = np.where(np.signbit(v), out | 0x80, out).astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(0x7f), out).astype(np.uint8)


def _torch_e5m2(v: torch.Tensor) -> np.ndarray:
    return v.clamp(-MAX, MAX).to(torch.float8_e5m2).view(torch.uint8).numpy()


def test_e5m2_decode_matches_torch(oracle_lib):
    table = _torch_table()
    for b in range(256):
        got = oracle.e5m2_decode(b)
        if np.isnan(table[b]):
            assert np.isnan(got), b
        else:
            assert got == table[b], b


def test_e5m2_encode_every_bf16(oracle_lib):
    v = bf16_bits_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    got = oracle.e5m2_encode_array(v)
    assert np.array_equal(got, _brute(v))


def test_e5m2_encode_ties_and_random_f32(oracle_lib):
    table = _torch_table()
    fin = np.sort(np.unique(table[:0x7c]))
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)  # exact ties in binary32
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9))])
    rng = np.random.default_rng(0)
    rnd = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-20, 16, 200_000))).astype(
        np.float32)
    v = np.concatenate([near, -near, rnd]).astype(np.float32)
    got = oracle.e5m2_encode_array(v)
    assert np.array_equal(got, _brute(v))
    inr = np.abs(v) <= MAX
    assert np.array_equal(got[inr], _torch_e5m2(torch.from_numpy(v[inr])))


def test_e5m2_saturates(oracle_lib):
    for v, want in ((MAX, 0x7b), (61439.0, 0x7b), (1e9, 0x7b), (float("inf"), 0x7b),
                    (-float("inf"), 0xfb), (-60000.0, 0xfb), (float("nan"), 0x7f)):
        assert oracle.e5m2_encode(v) == want, v


def test_y_dtype_config_rules(oracle_lib):
    base = workloads.tiny(0, 2).cfg
    for mode in range(6):
        rc = oracle.check_config(dict(base, quant_mode=mode, y_dtype=1))
        assert rc == (oracle.OK if mode >= 3 else oracle.ERR_ARG), mode
    assert oracle.check_config(dict(base, quant_mode=4, y_dtype=2)) == oracle.ERR_ARG


@pytest.mark.parametrize("H", [1024, 1040])
def test_mode3_e5m2_matches_torch(oracle_lib, H):
    rng = np.random.default_rng(3)
    xv = (rng.standard_normal(H) * rng.lognormal(0, 2, H)).astype(np.float32)
    xv[128:256] = 0.0
    x = to_bf16_bits(xv)
    sm = rng.uniform(0.5, 1.5, H).astype(np.float32)
    codes, scales = oracle.quant_row(3, x, sm, y_dtype=1)
    xf = torch.from_numpy(bf16_bits_to_f32(x)) * torch.from_numpy(sm)
    for g in range((H + 127) // 128):
        blk = xf[128 * g:128 * (g + 1)]
        amax = blk.abs().max()
        s = torch.tensor(MAX) / amax
        mult = torch.tensor(0.0) if amax == 0 else s
        assert np.array_equal(codes[128 * g:128 * (g + 1)], _torch_e5m2(blk * mult))
        assert scales[g] == (torch.tensor(1.0) / s).item()
    assert np.all(codes[128:256] == 0) and scales[1] == 0.0


def test_mode4_e5m2_floor_rule(oracle_lib):
    rng = np.random.default_rng(4)
    H = 2048
    xv = (rng.standard_normal(H) * rng.lognormal(0, 3, H)).astype(np.float32)
    xv[0:32] = 0.0
    xv[32:64] = 0.0
    xv[40] = MAX                       # max 57344 -> 2^0
    xv[64:96] = 1e-39                  # subnormal block -> clamped to 2^-127
    x = to_bf16_bits(xv)
    codes, sc = oracle.quant_row(4, x, y_dtype=1)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    for b in range(H // 32):
        blk = xf[32 * b:32 * (b + 1)]
        amax = np.abs(blk).max()
        e = -127 if amax == 0 else max(int(np.floor(np.log2(amax))) - 15, -127)
        if amax > 0 and e > -127:
            assert 2.0 ** (e + 15) <= amax < 2.0 ** (e + 16)
        assert sc[b] == e + 127
        v = torch.from_numpy((blk * 2.0 ** -e).astype(np.float32))
        assert np.array_equal(codes[32 * b:32 * (b + 1)], _torch_e5m2(v))
    assert sc[0] == 0 and sc[1] == 127 and sc[2] == 0


def test_mode5_e5m2_clip_rule(oracle_lib):
    rng = np.random.default_rng(5)
    H = 2048
    xv = (rng.standard_normal(H) * rng.lognormal(0, 4, H)).astype(np.float32)
    xv[0:32] = 0.0                     # max clamped to 1e-4
    xv[32:64] = 0.0
    xv[33] = MAX                       # max / 57344 = 1 -> 2^0
    x = to_bf16_bits(xv)
    codes, sc = oracle.quant_row(5, x, y_dtype=1)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    for b in range(H // 32):
        blk = xf[32 * b:32 * (b + 1)]
        q = np.float32(np.float32(max(np.abs(blk).max(), np.float32(1e-4))) / np.float32(MAX))
        e = int(sc[b]) - 127
        assert 2.0 ** (e - 1) < float(q) <= 2.0 ** e  # e = ceil(log2 q), exactly
        v = torch.from_numpy((blk * 2.0 ** -e).astype(np.float32))
        assert np.array_equal(codes[32 * b:32 * (b + 1)], _torch_e5m2(v))
    assert sc[1] == 127
