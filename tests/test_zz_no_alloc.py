"""cq_dispatch_noalloc: dispatch for callers that cannot allocate device memory.

Such callers (a plugin handed only its tensors, a server whose memory plan is
fixed at start-up, an embedded deployment with a pre-planned memory map) get
the same results as cq_dispatch without passing a workspace: the scratch is a
device array built into libcq. This file is collected last so that a run that
stops at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_quant_gb300 as cq
from combine_quant_gb300 import _lib, workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _inputs(wl):
    t = lambda a, dt: None if a is None else torch.from_numpy(  # noqa: E731
        np.ascontiguousarray(a)).to(DEV).view(dt)
    sm = t(wl.smooth, torch.float32) if wl.cfg["quant_mode"] in (1, 2, 3) else None
    return dict(x=t(wl.x, torch.bfloat16), expert_ids=t(wl.expert_ids, torch.int32),
                smooth_scales=sm, x_active_mask=t(wl.mask, torch.uint8),
                bs_per_rank=t(wl.bs_per_rank, torch.int32),
                expert_scales=t(wl.expert_scales, torch.float32))


def _noalloc(cfg, inp, out):
    """Call the no-alloc entry point through the C ABI."""
    p = lambda tt: None if tt is None else ctypes.c_void_p(tt.data_ptr())  # noqa: E731
    c = cfg.as_c()
    rc = _lib.load().cq_dispatch_noalloc(
        ctypes.byref(c), p(inp["x"]), p(inp["expert_ids"]), p(inp["smooth_scales"]),
        p(inp["x_active_mask"]), p(inp["bs_per_rank"]), p(inp["expert_scales"]),
        p(out.expand_x), p(out.dynamic_scales), p(out.assist_info), p(out.ep_recv_count),
        p(out.expert_token_nums), p(out.expand_scales),
        ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    return rc


def _same(cfg, a, b):
    """Every output of the two entry points agrees (codes, scales and all index
    outputs are exact; this is the tolerance of the parity tests)."""
    rows_a, inv_a, base_a = cq.assist_views(cfg, a.assist_info)
    rows_b, inv_b, base_b = cq.assist_views(cfg, b.assist_info)
    R = int(base_a[-1].item())
    assert torch.equal(base_a, base_b)
    assert torch.equal(inv_a, inv_b)
    assert torch.equal(rows_a[:R], rows_b[:R])  # rows past the total are left untouched
    assert torch.equal(a.ep_recv_count, b.ep_recv_count)
    assert torch.equal(a.expert_token_nums, b.expert_token_nums)
    ea, eb = a.expand_x[:R], b.expand_x[:R]
    if ea.dtype == torch.bfloat16:
        ea, eb = ea.view(torch.int16), eb.view(torch.int16)
    assert torch.equal(ea, eb)
    if a.dynamic_scales is not None:
        assert torch.equal(a.dynamic_scales[:R], b.dynamic_scales[:R])
    assert torch.equal(a.expand_scales[:R], b.expand_scales[:R])
    return R


def _check_case(wl):
    cfg = cq.Config.from_dict(wl.cfg)
    inp = _inputs(wl)
    ref = cq.dispatch(cfg, **inp)  # the existing entry point, with its own workspace
    got = cq.alloc_dispatch_outputs(cfg, DEV)
    assert _noalloc(cfg, inp, got) == _lib.CQ_OK
    torch.cuda.synchronize()
    return _same(cfg, ref, got)


def test_noalloc_matches_dispatch_on_two_calls_in_a_row():
    cases = [workloads.dsv3(seed=41, W=8, BS=40, M=64, K=8, H=2048),
             workloads.special(seed=42, W=8, BS=24, H=1024, M=48)]
    for wl in cases:  # two different problems back to back share the scratch array
        assert _check_case(wl) > 0
    # and the first problem once more, after the second left its data behind
    _check_case(cases[0])


def test_noalloc_per_expert_smooth_and_mx_after_a_larger_problem():
    """The per-expert-smooth path (its row table is the largest part of the
    scratch) and mode 5, each right after a larger problem has filled more of
    the array, so that any byte read before this call writes it would show."""
    big = workloads.skew(seed=44, W=16, BS=64, M=64, K=16, H=1024)   # mode 2, per-expert smooth
    assert cq.Config.from_dict(big.cfg).workspace_size <= _lib.NOALLOC_SCRATCH_BYTES
    smooth_small = workloads.skew(seed=45, W=4, BS=24, M=16, K=8, H=2048)
    mx_small = workloads.mxfp8(seed=46, W=4, BS=20, M=16, K=4, H=1024)
    for wl in (big, smooth_small, big, mx_small, smooth_small):
        assert _check_case(wl) > 0


def test_python_wrapper_matches_dispatch():
    """cq.dispatch_noalloc (the binding's wrapper of the same entry point)."""
    wl = workloads.dsv3(seed=43, W=8, BS=24, M=64, K=8, H=1024)
    cfg = cq.Config.from_dict(wl.cfg)
    inp = _inputs(wl)
    ref = cq.dispatch(cfg, **inp)
    got = cq.dispatch_noalloc(cfg, **inp)
    torch.cuda.synchronize()
    assert _same(cfg, ref, got) > 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    """A problem whose workspace exceeds the built-in array is refused with
    CQ_ERR_TOO_LARGE on the host. Every pointer is NULL: the size check comes
    first, and were it ever skipped, the NULL token rows would be refused too
    (CQ_ERR_ARG) before anything is enqueued."""
    cfg = cq.Config(ep_world_size=256, moe_expert_num=512, max_bs=512, topk=16, hidden=4096,
                    quant_mode=2)
    assert cfg.check() == 0 and cfg.workspace_size > _lib.NOALLOC_SCRATCH_BYTES
    inp = dict(x=None, expert_ids=None, smooth_scales=None, x_active_mask=None,
               bs_per_rank=None, expert_scales=None)
    none = cq.DispatchResult(None, None, None, None, None, None)
    assert _noalloc(cfg, inp, none) == _lib.CQ_ERR_TOO_LARGE
