"""Pins for the oracle's quant_mode 1, 3, 4, its fp16 handling and the three
smooth-scale shapes ("low_latency_dispatch" 计算公式 / quant_mode 相关约束)."""
import numpy as np
import pytest
import torch

import oracle
from combine_quant_gb300 import workloads
from combine_quant_gb300.workloads import bf16_bits_to_f32, make_config, to_bf16_bits


def _f16_bits(a):
    return np.asarray(a, np.float32).astype(np.float16).view(np.uint16)


def test_f16_decode_every_value(oracle_lib):
    for b in range(0, 65536, 1):
        want = np.uint16(b).view(np.float16).astype(np.float32)
        got = np.float32(oracle.f16_to_f32(b))
        assert (np.isnan(want) and np.isnan(got)) or got == want, b


def test_f16_encode_matches_numpy(oracle_lib):
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 3e4).astype(np.float32),
        (rng.standard_normal(5000) * 1e-6).astype(np.float32),  # fp16 subnormals
        np.array([65504, 65519.99, 65520, 7e4, -7e4, 2 ** -25, 2 ** -24, 3 * 2 ** -26],
                 np.float32),
    ])
    # exact ties between adjacent fp16 values
    h = rng.integers(0x0001, 0x7bff, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float32).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float32).astype(np.float64)
    v = np.concatenate([v, ((lo + hi) / 2).astype(np.float32)])
    got = np.array([oracle.f16_from_f32(float(f)) for f in v], np.uint16)
    assert np.array_equal(got, v.astype(np.float16).view(np.uint16))


def test_floor_log2_definition(oracle_lib):
    rng = np.random.default_rng(1)
    a = np.concatenate([np.exp2(np.arange(-149, 128)).astype(np.float32),
                        rng.uniform(1e-40, 1e-36, 1000).astype(np.float32),  # subnormals
                        rng.uniform(0, 3e38, 5000).astype(np.float32)])
    a = a[a > 0]
    e = np.array([oracle.floor_log2(float(x)) for x in a], np.float64)
    ad = a.astype(np.float64)
    assert np.all(np.exp2(e) <= ad) and np.all(ad < np.exp2(e + 1))


@pytest.mark.parametrize("kind", ["row", "scalar"])
def test_mode1_static_matches_torch(oracle_lib, kind):
    rng = np.random.default_rng(2)
    H = 2048
    x = to_bf16_bits((rng.standard_normal(H) * 30).astype(np.float32))
    sm = rng.uniform(0.5, 3.0, H).astype(np.float32)
    sc = np.float32(2.5)
    codes, scale = (oracle.quant_row(1, x, sm) if kind == "row"
                    else oracle.quant_row(1, x, smooth_scalar=float(sc)))
    assert scale is None
    xt = torch.from_numpy(bf16_bits_to_f32(x))
    xf = xt * torch.from_numpy(sm) if kind == "row" else xt * torch.tensor(sc)
    assert np.array_equal(codes, torch.round(xf).clamp(-128, 127).to(torch.int8).numpy())
    assert codes.max() == 127 and codes.min() == -128  # saturation exercised


def _torch_e4m3(v: torch.Tensor) -> np.ndarray:
    """torch's round-to-nearest-even e4m3fn cast, with +-448 saturation."""
    return v.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("H", [1024, 1040, 7168])
def test_mode3_pergroup_matches_torch(oracle_lib, H):
    rng = np.random.default_rng(3)
    xv = (rng.standard_normal(H) * rng.lognormal(0, 2, H)).astype(np.float32)
    xv[128:256] = 0.0  # an all-zero group
    x = to_bf16_bits(xv)
    sm = rng.uniform(0.5, 1.5, H).astype(np.float32)
    codes, scales = oracle.quant_row(3, x, sm)
    xf = torch.from_numpy(bf16_bits_to_f32(x)) * torch.from_numpy(sm)
    G = (H + 127) // 128
    assert scales.shape == (G,)
    for g in range(G):
        blk = xf[128 * g:128 * (g + 1)]
        amax = blk.abs().max()
        s = torch.tensor(448.0) / amax
        mult = torch.tensor(0.0) if amax == 0 else s
        assert np.array_equal(codes[128 * g:128 * (g + 1)], _torch_e4m3(blk * mult))
        assert scales[g] == (torch.tensor(1.0) / s).item()
    assert np.all(codes[128:256] == 0) and scales[1] == 0.0


def test_mode4_mx_floor_rule(oracle_lib):
    rng = np.random.default_rng(4)
    H = 7168
    xv = (rng.standard_normal(H) * rng.lognormal(0, 3, H)).astype(np.float32)
    xv[0:32] = 0.0                     # zero block -> smallest scale (byte 0)
    xv[32:64] = 0.0
    xv[40] = 448.0                     # max 448 -> 2^0
    xv[64:96] = 1e-39                  # subnormal block -> clamped to 2^-127
    x = to_bf16_bits(xv)
    codes, sc = oracle.quant_row(4, x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    for b in range(H // 32):
        blk = xf[32 * b:32 * (b + 1)]
        amax = np.abs(blk).max()
        e = -127 if amax == 0 else max(int(np.floor(np.log2(amax))) - 8, -127)
        if amax > 0:
            assert 2.0 ** (e + 8) <= amax < 2.0 ** (e + 9) or e == -127
        assert sc[b] == e + 127
        v = torch.from_numpy((blk * 2.0 ** -e).astype(np.float32))
        assert np.array_equal(codes[32 * b:32 * (b + 1)], _torch_e4m3(v))
    assert sc[0] == 0 and sc[1] == 127 and sc[2] == 0


def test_smooth_shapes_in_dispatch(oracle_lib):
    """One row shared by every expert, or one scalar, apply to every slot."""
    wl = workloads.tiny(seed=5, quant_mode=2)
    rng = np.random.default_rng(5)
    row = rng.uniform(0.5, 1.5, wl.cfg["hidden"]).astype(np.float32)
    for kind, sm in ((1, row), (2, np.array([1.75], np.float32))):
        cfg = dict(wl.cfg, smooth_kind=kind)
        out = oracle.dispatch(cfg, wl.x, wl.expert_ids, sm, expert_scales=wl.expert_scales)
        for n in range(out["rows"]):
            src, tok, _k = out["assist"][n, :3]
            want = (oracle.quant_row(2, wl.x[src, tok], row) if kind == 1
                    else oracle.quant_row(2, wl.x[src, tok], smooth_scalar=1.75))
            assert np.array_equal(out["expand_x"][n], want[0])
            assert out["dynamic_scales"][n] == want[1]


def test_fp16_dispatch_and_combine(oracle_lib):
    """fp16 tokens: mode 0 moves the fp16 bits; combine rounds to fp16."""
    W, M, BS, K, H = 2, 4, 3, 2, 1024
    rng = np.random.default_rng(6)
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                      quant_mode=0, x_dtype=1)
    x = _f16_bits(rng.standard_normal((W, BS, H)))
    ids = np.stack([rng.permutation(M)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    w = rng.uniform(0, 1, (W, BS, K)).astype(np.float32)
    out = oracle.dispatch(cfg, x, ids.astype(np.int32), expert_scales=w)
    for n in range(out["rows"]):
        src, tok, _k = out["assist"][n, :3]
        assert np.array_equal(out["expand_x"][n], x[src, tok])
    ffn = out["expand_x"][:out["rows"]]
    y32 = oracle.combine(cfg, ffn, out["inv"], w, out_f32=True)
    y16 = oracle.combine(cfg, ffn, out["inv"], w, out_f32=False)
    assert np.array_equal(y16, y32.astype(np.float16).view(np.uint16))
    xf = x.view(np.float16).astype(np.float64)
    wsum = w.astype(np.float64).sum(axis=2, keepdims=True)
    assert np.allclose(y32, xf * wsum, rtol=1e-6, atol=1e-6)
    # the int8 quantisation of mode 2 reads fp16 values exactly
    c16, s16 = oracle.quant_row(2, x[0, 0], x_dtype=1)
    xt = torch.from_numpy(x[0, 0].view(np.float16).astype(np.float32))
    s = torch.tensor(127.0) / xt.abs().max()
    assert np.array_equal(c16, torch.round(xt * s).clamp(-128, 127).to(torch.int8).numpy())
