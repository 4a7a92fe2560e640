"""GPU parity for quant_mode 1, 3, 4, the three smooth-scale shapes and fp16
tokens ("low_latency_dispatch" 计算公式 / quant_mode 相关约束), element by
element against the oracle (codes and scales bit-exact; combine exact)."""
import numpy as np
import pytest

import gpu_harness as gh
from combine_quant_gb300 import workloads

pytestmark = pytest.mark.gpu


def _with(wl, mode, smooth=None, kind=0):
    cfg = dict(wl.cfg, quant_mode=mode, smooth_kind=kind)
    return workloads.Workload(wl.name + f"_m{mode}_k{kind}", cfg, wl.x, wl.expert_ids,
                              wl.expert_scales, smooth, wl.mask, wl.bs_per_rank,
                              wl.const_alpha1, wl.const_alpha2, wl.const_v, wl.seed)


def _smooth(wl, kind, seed=0):
    rng = np.random.default_rng(100 + seed)
    H = wl.cfg["hidden"]
    if kind == 2:
        return np.array([rng.uniform(0.5, 4.0)], np.float32)
    if kind == 1:
        return rng.uniform(0.5, 1.5, H).astype(np.float32)
    s_eff = wl.cfg["shared_expert_num"] if wl.cfg["shared_expert_rank_num"] > 0 else 0
    return rng.uniform(0.5, 1.5, (s_eff + wl.cfg["moe_expert_num"], H)).astype(np.float32)


def _base(name):
    return {
        "tiny": lambda: workloads.tiny(3, 2),
        "dsv3_small": lambda: workloads.dsv3(seed=21, W=8, BS=37, M=64, K=8, H=2048),
        "special_small": lambda: workloads.special(seed=23, W=8, BS=20, H=1024, M=48),
        "h1040": lambda: workloads.dsv3(seed=25, W=4, BS=9, M=16, K=4, H=1040),
    }[name]()


@pytest.mark.parametrize("base", ["tiny", "special_small"])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_mode1_static(base, kind):
    wl = _base(base)
    gh.full_parity(_with(wl, 1, _smooth(wl, kind), kind))


@pytest.mark.parametrize("base", ["tiny", "dsv3_small", "h1040"])
@pytest.mark.parametrize("kind", [None, 0, 1, 2])
def test_mode3_pergroup(base, kind):
    wl = _base(base)
    if kind is None:
        gh.full_parity(_with(wl, 3))
    else:
        gh.full_parity(_with(wl, 3, _smooth(wl, kind), kind))


@pytest.mark.parametrize("base", ["tiny", "dsv3_small", "special_small"])
def test_mode4_mx(base):
    gh.full_parity(_with(_base(base), 4))


@pytest.mark.parametrize("kind", [1, 2])
def test_mode2_broadcast_smooth(kind):
    wl = _base("dsv3_small")
    gh.full_parity(_with(wl, 2, _smooth(wl, kind), kind))


def test_mode4_extremes():
    wl = _with(workloads.tiny(4, 2), 4)
    x = workloads.bf16_bits_to_f32(wl.x).copy()
    x[0, 0] = 0.0            # zero blocks -> scale byte 0
    x[0, 1, :64] = 448.0     # exactly 2^8 * 1.75 -> scale 2^0
    x[1, 2] *= 1e-38         # subnormal blocks -> scale clamped to 2^-127
    x[2, 3] *= 1e30
    wl.x = workloads.to_bf16_bits(x)
    gh.full_parity(wl)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5])
def test_fp16_tokens(mode):
    wl = workloads.as_fp16(_base("tiny"))
    sm = _smooth(wl, 0) if mode in (1, 2, 3) else None
    gh.full_parity(_with(wl, mode, sm, 0))


def test_fp16_special_experts_and_masks():
    gh.full_parity(workloads.as_fp16(_base("special_small")))


def test_fp16_dsv3_small():
    gh.full_parity(workloads.as_fp16(_base("dsv3_small")))


@pytest.mark.parametrize("kind", [None, 0, 2])
def test_mode2_nonfinite_and_extreme_rows(kind):
    """Per-token int8 on rows that leave the ordinary case: all-zero and -0
    rows (scale 0, codes 0), NaN elements (code 0, scale from the NaN-ignoring
    max), infinities (max inf, scale 0), rows so small that 127/max overflows,
    and huge rows. kind None: no smooth; 0: per-expert rows; 2: one scalar."""
    wl = _base("dsv3_small")
    x = workloads.bf16_bits_to_f32(wl.x).copy()
    x[0, 0] = 0.0
    x[0, 1] = -0.0
    x[0, 2, 5] = np.nan
    x[0, 3] = 0.0
    x[0, 3, 7] = np.nan
    x[0, 4, 9] = np.inf
    x[0, 5, 11] = -np.inf
    x[0, 5, 12] = np.nan
    x[1, 0] *= 1e-38
    x[1, 1] = 0.0
    x[1, 1, 3] = 1e-39
    x[1, 2] *= 1e30
    x[1, 3, 100] = 3.0e38
    x[2, 4] = -1.0 / 3.0
    wl.x = workloads.to_bf16_bits(x)
    if kind is None:
        gh.full_parity(_with(wl, 2))
    else:
        gh.full_parity(_with(wl, 2, _smooth(wl, kind), kind))


def _e5(wl, mode, smooth=None, kind=0):
    w = _with(wl, mode, smooth, kind)
    w.cfg["y_dtype"] = 1
    return w


@pytest.mark.parametrize("base", ["tiny", "dsv3_small", "h1040"])
@pytest.mark.parametrize("kind", [None, 0, 1, 2])
def test_mode3_e5m2(base, kind):
    """Per-128-group e5m2 codes (y_dtype 1, dst_type_max 57344), with every
    smooth shape (kind 0 runs the expert-major per-expert-smooth kernel)."""
    wl = _base(base)
    gh.full_parity(_e5(wl, 3) if kind is None else _e5(wl, 3, _smooth(wl, kind), kind))


@pytest.mark.parametrize("mode", [4, 5])
@pytest.mark.parametrize("base", ["tiny", "dsv3_small", "special_small"])
def test_mx_e5m2(mode, base):
    """mx e5m2 codes (emax 15; clip against 57344)."""
    gh.full_parity(_e5(_base(base), mode))


@pytest.mark.parametrize("mode", [3, 4, 5])
def test_e5m2_extremes_and_fp16(mode):
    wl = _e5(workloads.tiny(4, 2), mode)
    x = workloads.bf16_bits_to_f32(wl.x).copy()
    x[0, 0] = 0.0
    x[0, 1, :64] = 57344.0
    x[1, 2] *= 1e-38
    x[2, 3] *= 1e30
    x[3, 4, 5] = np.nan
    wl.x = workloads.to_bf16_bits(x)
    gh.full_parity(wl)
    gh.full_parity(workloads.as_fp16(_e5(_base("tiny"), mode)))


def _tie_maxima():
    """Row maxima A (bf16, in [1, 127]) for which the product of A/2 with the
    binary32 scale s = 127/A rounds onto the tie 63.5 without being 63.5
    exactly: a single-rounding multiply-add would round that product to 63 or
    64 by its exact value, the two-step rounding of the method gives 64."""
    bits = np.arange(1, 0x7f80, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    out = []
    for A in vals[(vals >= 1.0) & (vals <= 127.0)]:
        s = np.float32(127.0) / A
        h = np.float32(A / 2)
        p = np.float32(h * s)
        if p == np.float32(63.5) and np.float64(h) * np.float64(s) != 63.5:
            out.append(float(A))
    return np.array(out, np.float32)


@pytest.mark.parametrize("kind", [None, 0, 1, 2])
def test_mode2_rounding_ties(kind):
    """Per-token int8 codes on products that sit on .5 ties: rows whose max A
    makes fl(A/2 * fl(127/A)) a tie reached by rounding (about 600 such A), and
    rows with max 127 (scale 1) holding every k + 0.5. Smooth scales are all
    ones, so every smooth shape (kind 0: the per-expert-smooth kernel) meets
    the same products; the codes must be the round-to-nearest-even of the
    rounded product, bit for bit with the oracle."""
    wl = _base("dsv3_small")
    x = workloads.bf16_bits_to_f32(wl.x).copy()
    W, BS, H = x.shape
    maxima = _tie_maxima()
    assert maxima.size > 500
    rng = np.random.default_rng(7)
    halves = (np.arange(127, dtype=np.float32) + np.float32(0.5))  # 0.5 .. 126.5, exact in bf16
    n = 0
    for r in range(W):
        for i in range(BS):
            if n % 4 == 3:
                row = np.resize(np.concatenate([halves, -halves]), H).astype(np.float32)
                row[H - 1] = 127.0
                rng.shuffle(row)
            else:
                A = maxima[n % maxima.size]
                h = np.float32(A / 2)
                row = np.where(np.arange(H) % 2 == 0, h, -h).astype(np.float32)
                # a third of the row: random values below the max
                fill = rng.integers(0, H, H // 3)
                row[fill] = (rng.uniform(-1, 1, fill.size) * A).astype(np.float32)
                row[rng.integers(0, H)] = A if n % 2 == 0 else -A
            x[r, i] = row
            n += 1
    wl.x = workloads.to_bf16_bits(x)
    if kind is None:
        gh.full_parity(_with(wl, 2))
    else:
        sm = _smooth(wl, kind)
        sm[...] = 1.0
        gh.full_parity(_with(wl, 2, sm, kind))


@pytest.mark.parametrize("kind,scale", [(0, 1.0), (1, 1.0), (2, 1.0), (2, 37.0), (0, 37.0)])
def test_mode1_extremes(kind, scale):
    """Static int8 on values that leave the ordinary range: every tie k + 0.5
    up to 127.5, the saturation boundary (+-127.5, +-128 and beyond),
    infinities, NaN and huge values, next to ordinary rows. Smooth scales are
    all `scale`, so x * scale is exact for scale 1; scale 37 pushes about a
    quarter of the values past the int8 range, mixing threads whose values
    all round into [-127, 127] with threads that saturate."""
    wl = _base("dsv3_small")
    x = workloads.bf16_bits_to_f32(wl.x).copy()
    H = x.shape[2]
    halves = np.arange(-128, 128, dtype=np.float32) + np.float32(0.5)  # -127.5 .. 127.5
    x[0, 0] = np.resize(halves, H)
    edge = np.array([127.0, 127.5, -127.5, 128.0, -128.0, 129.0, -130.0, 126.5, -126.5, 255.0],
                    np.float32)
    x[0, 1] = np.resize(edge, H)
    x[0, 2, 3] = np.inf
    x[0, 3, 5] = -np.inf
    x[0, 4, 7] = np.nan
    x[0, 5, ::17] = 1e30
    x[0, 6, ::5] = -3e38
    x[1, 0, :] = 127.5
    x[1, 1, :] = -127.5
    x[1, 2, H // 2] = 127.5  # one thread's values reach the boundary, the rest are ordinary
    wl.x = workloads.to_bf16_bits(x)
    sm = _smooth(wl, kind)
    sm[...] = scale
    gh.full_parity(_with(wl, 1, sm, kind))


@pytest.mark.parametrize("mode", [1, 2])
def test_per_expert_smooth_ragged_hidden(mode):
    """One smooth row per expert with H = 1040 (65 units of 16): the
    per-expert-smooth kernel's variant whose last consumer threads hold one
    unit or none (H = 1024 k takes the variant without bounds checks)."""
    wl = _base("h1040")
    gh.full_parity(_with(wl, mode, _smooth(wl, 0), 0))
