"""Independent dispatch + combine pipelines on separate CUDA streams, each
with its own workspace and buffers, enqueued without any synchronisation
between them: every output of each matches the oracle, as when they run
alone (the library keeps no per-call state outside the caller's buffers)."""
import numpy as np
import pytest
import torch

import combine_quant_gb300 as cq
import gpu_harness as gh
import oracle
from combine_quant_gb300 import workloads

pytestmark = pytest.mark.gpu


def _prepare(wl):
    cfg = cq.Config.from_dict(wl.cfg)
    sm = gh.dev(wl.smooth, torch.float32) if gh.uses_smooth(wl) else None
    args = dict(x=gh.dev(wl.x, cfg.token_dtype), ids=gh.dev(wl.expert_ids, torch.int32), sm=sm,
                mask=gh.dev(wl.mask, torch.uint8), bpr=gh.dev(wl.bs_per_rank, torch.int32),
                w=gh.dev(wl.expert_scales, torch.float32))
    ws = cq.alloc_workspace(cfg, gh.DEV)
    ffn = gh.FfnStandin(wl, cfg.max_rows)
    return cfg, args, ws, ffn


def _run(cfg, args, ws, ffn, steps):
    out = None
    y = None
    for _ in range(steps):
        out = cq.dispatch(cfg, args["x"], args["ids"], smooth_scales=args["sm"],
                          x_active_mask=args["mask"], bs_per_rank=args["bpr"],
                          expert_scales=args["w"], workspace=ws, out=out)
        # each pipeline's combine reports to its own workspace (cq_combine_ws)
        y = cq.combine(cfg, ffn.device_rows, out.assist_info, args["w"], out.ep_recv_count, y=y,
                       workspace=ws)
    return out, y


def _check(wl, ffn, out, y, status):
    ref = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, wl.smooth if gh.uses_smooth(wl) else None,
                          wl.mask, wl.bs_per_rank, wl.expert_scales)
    assert status == ref["status"]
    R = ref["rows"]
    assert np.array_equal(gh.host(out.expand_x[:R]).view(ref["expand_x"].dtype),
                          ref["expand_x"][:R])
    if ref["dynamic_scales"] is not None:
        assert np.array_equal(gh.host(out.dynamic_scales[:R]).view(np.uint8),
                              ref["dynamic_scales"][:R].view(np.uint8))
    inv = ffn.remap_inv(ref["inv"])
    r16 = oracle.combine(wl.cfg, ffn.pool, inv, wl.expert_scales, wl.x, wl.const_alpha1,
                         wl.const_alpha2, wl.const_v, out_f32=False)
    assert np.array_equal(gh.host(y), r16)


def test_two_streams_run_independent_pipelines():
    wls = [workloads.dsv3(seed=51, W=8, BS=40, M=64, K=8, H=2048),
           workloads.skew(seed=52, W=4, BS=48, M=32, K=16, H=2048)]  # per-expert smooth path
    preps = [_prepare(wl) for wl in wls]
    streams = [torch.cuda.Stream(gh.DEV) for _ in wls]
    torch.cuda.synchronize()
    results = []
    for (cfg, args, ws, ffn), s in zip(preps, streams):
        with torch.cuda.stream(s):
            results.append(_run(cfg, args, ws, ffn, steps=4))
    torch.cuda.synchronize()
    for wl, (cfg, args, ws, ffn), (out, y), s in zip(wls, preps, results, streams):
        with torch.cuda.stream(s):
            status = cq.read_status(ws)  # this pipeline's dispatch and combine status
        _check(wl, ffn, out, y, status)
        assert status & cq.CQ_ST_TIMEOUT == 0
    assert cq.read_combine_status() == 0  # nothing went to the per-device word
