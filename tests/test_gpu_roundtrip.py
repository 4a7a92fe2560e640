"""The round trip on the GPU: cq_dispatch, the identity expert FFN of
tests/roundtrip.py, then cq_combine. The FFN rows are made on the host from
the oracle's dispatched rows, which the GPU's rows are first shown to equal
bit for bit, so the GPU's own rows go through the FFN; y is compared with the
oracle's combine of the same rows and with the closed form."""
import numpy as np
import pytest
import torch

import combine_quant_gb300 as cq
from combine_quant_gb300 import workloads

import gpu_harness as gh
import roundtrip as rt

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_m0": lambda: workloads.tiny(0, 0),
    "tiny_m2_smooth": lambda: workloads.tiny(0, 2),
    "tiny_m5": lambda: workloads.tiny(0, 5),
    "dsv3_m2": lambda: workloads.dsv3(seed=41, W=16, BS=64, M=128, K=8, H=7168),
    "mxfp8_m5": lambda: workloads.mxfp8(seed=42, W=16, BS=96, M=64, K=8, H=7168),
    "special_m0": lambda: workloads.special(seed=43, W=16, BS=64, H=4096, M=112),
    "skew_m2_smooth": lambda: workloads.skew(seed=44, W=8, BS=96, M=64, K=16, H=2048),
}


@pytest.mark.parametrize("name", list(CASES))
def test_gpu_round_trip(name):
    wl = CASES[name]()
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    ref, ffn, row_err, y_ref = rt.run_oracle(wl)
    R = ref["rows"]
    assert R > 0 and status == ref["status"]
    _, inv, _ = cq.assist_views(cfg, out.assist_info)
    assert np.array_equal(gh.host(inv), ref["inv"])
    assert np.array_equal(gh.host(out.expand_x[:R]).view(ref["expand_x"].dtype),
                          ref["expand_x"][:R])
    if ref["dynamic_scales"] is not None:
        assert np.array_equal(gh.host(out.dynamic_scales[:R]).view(np.uint8),
                              ref["dynamic_scales"][:R].view(np.uint8))
    w = gh.dev(wl.expert_scales, torch.float32)
    y = gh.host(cq.combine(cfg, gh.dev(ffn, cfg.token_dtype), out.assist_info, w,
                           out.ep_recv_count, ori_x=gh.dev(wl.x, cfg.token_dtype),
                           const_alpha1=gh.dev(wl.const_alpha1, torch.float32),
                           const_alpha2=gh.dev(wl.const_alpha2, torch.float32),
                           const_v=gh.dev(wl.const_v, cfg.token_dtype),
                           out_dtype=torch.float32))
    assert cq.read_combine_status() == 0
    assert np.max(np.abs(y - y_ref)) <= 1e-5
    assert np.array_equal(y.view(np.uint32), y_ref.view(np.uint32))
    target, bound = rt.closed_form(wl, ref, row_err)
    assert np.all(np.abs(y.astype(np.float64) - target) <= bound)
