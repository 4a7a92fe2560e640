"""The oracle's round trip (dispatch, an identity expert FFN, combine) against
the closed form of tests/roundtrip.py: combine returns each token's
expert_scales-weighted sum of its own row (plus the shared and special
experts' terms) within the quantisation step of the rows."""
import numpy as np
import pytest

from combine_quant_gb300 import workloads

import roundtrip as rt

CASES = {
    "tiny_m0": lambda: workloads.tiny(0, 0),
    "tiny_m2_smooth": lambda: workloads.tiny(0, 2),
    "tiny_m5": lambda: workloads.tiny(0, 5),
    "dsv3_small_m2": lambda: workloads.dsv3(seed=31, W=8, BS=24, M=64, K=8, H=2048),
    "mxfp8_small_m5": lambda: workloads.mxfp8(seed=32, W=8, BS=16, M=32, K=8, H=1536),
    "special_small_m0": lambda: workloads.special(seed=33, W=8, BS=20, H=1024, M=48),
    "skew_small_m2_smooth": lambda: workloads.skew(seed=34, W=4, BS=24, M=32, K=16, H=1024),
}


@pytest.mark.parametrize("name", list(CASES))
def test_round_trip_closed_form(name):
    wl = CASES[name]()
    ref, _, row_err, y = rt.run_oracle(wl)
    assert ref["rows"] > 0
    target, bound = rt.closed_form(wl, ref, row_err)
    diff = np.abs(y.astype(np.float64) - target)
    assert np.all(diff <= bound), float(np.max(diff - bound))
    # the bound is a quantisation step, not a free pass: per token, against
    # the largest value of the token's sum, it stays near the codes'
    # resolution (exact rows in mode 0; 1/254 of the row max, times the
    # smooth scales' spread, in mode 2; e4m3's 2^-4 in mode 5)
    peak = np.max(np.abs(target), axis=2)
    on = peak > 0
    rel = float(np.median(np.max(bound, axis=2)[on] / peak[on]))
    assert rel < {0: 1e-5, 2: 0.03, 5: 0.07}[wl.cfg["quant_mode"]], rel


def test_round_trip_detects_a_wrong_weight():
    """A planted mistake in the oracle's output (one slot's weight applied
    twice to one token) falls outside the bound."""
    wl = CASES["dsv3_small_m2"]()
    ref, ffn, row_err, y = rt.run_oracle(wl)
    target, bound = rt.closed_form(wl, ref, row_err)
    K = wl.cfg["topk"]
    inv = ref["inv"].reshape(8, 24, K)
    r, i, k = 3, 5, 2
    row = inv[r, i, k]
    assert row >= 0
    bad = y.astype(np.float64).copy()
    bad[r, i] += float(wl.expert_scales[r, i, k]) * workloads.bf16_bits_to_f32(ffn[row])
    assert not np.all(np.abs(bad - target) <= bound)
