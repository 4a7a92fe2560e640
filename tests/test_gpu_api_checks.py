"""The Python binding rejects output buffers and workspaces that do not fit
the config (wrong shape, type or device) before anything is enqueued: the
kernels write through raw pointers and cannot check sizes themselves."""
import pytest
import torch

import combine_quant_gb300 as cq
import gpu_harness as gh
from combine_quant_gb300 import workloads

pytestmark = pytest.mark.gpu


def _setup(mode=2):
    wl = workloads.tiny(seed=2, quant_mode=mode)
    cfg = cq.Config.from_dict(wl.cfg)
    x = gh.dev(wl.x, cfg.token_dtype)
    ids = gh.dev(wl.expert_ids, torch.int32)
    w = gh.dev(wl.expert_scales, torch.float32)
    return cfg, x, ids, w


@pytest.mark.parametrize("field,bad", [
    ("expand_x", lambda t: t[:-1]),
    ("expand_x", lambda t: t.view(torch.uint8)),
    ("dynamic_scales", lambda t: t[:-1]),
    ("assist_info", lambda t: t[:-1]),
    ("ep_recv_count", lambda t: t.reshape(-1)),
    ("expert_token_nums", lambda t: t.to(torch.int32)),
    ("expand_scales", lambda t: t[:-1]),
])
def test_dispatch_rejects_misfit_outputs(field, bad):
    cfg, x, ids, w = _setup()
    good = cq.alloc_dispatch_outputs(cfg, gh.DEV)
    out = good._replace(**{field: bad(getattr(good, field))})
    with pytest.raises(ValueError):
        cq.dispatch(cfg, x, ids, expert_scales=w, out=out)
    # the same buffers, unchanged, still work
    cq.dispatch(cfg, x, ids, expert_scales=w, out=good)
    torch.cuda.synchronize()


def test_halves_and_workspace_checks():
    cfg, x, ids, w = _setup()
    out = cq.alloc_dispatch_outputs(cfg, gh.DEV)
    ws = cq.alloc_workspace(cfg, gh.DEV)
    with pytest.raises(ValueError):
        cq.dispatch_route(cfg, ids, workspace=ws.view(torch.int32), out=out)
    with pytest.raises(ValueError):
        cq.dispatch_route(cfg, ids, workspace=ws,
                          out=out._replace(ep_recv_count=out.ep_recv_count[:1]))
    with pytest.raises(ValueError):
        cq.dispatch_permute(cfg, x, ids, expert_scales=w, workspace=ws,
                            out=out._replace(expand_x=out.expand_x[:, :-16]))
    with pytest.raises(ValueError):
        cq.dispatch(cfg, x, ids, expert_scales=w, workspace=ws.cpu(), out=out)
    cq.dispatch_route(cfg, ids, workspace=ws, out=out)
    cq.dispatch_permute(cfg, x, ids, expert_scales=w, workspace=ws, out=out)
    assert cq.read_status(ws) == 0


def test_combine_checks_ep_recv_count():
    cfg, x, ids, w = _setup()
    out = cq.dispatch(cfg, x, ids, expert_scales=w)
    ffn = torch.zeros(cfg.max_rows, cfg.hidden, dtype=cfg.token_dtype, device=gh.DEV)
    with pytest.raises(ValueError):
        cq.combine(cfg, ffn, out.assist_info, w, out.ep_recv_count[:, :-1])
    with pytest.raises(ValueError):
        cq.combine(cfg, ffn, out.assist_info, w, out.ep_recv_count,
                   y=torch.empty(1, dtype=cfg.token_dtype, device=gh.DEV))
    y = cq.combine(cfg, ffn, out.assist_info, w, out.ep_recv_count)
    assert y.shape == (cfg.ep_world_size, cfg.max_bs, cfg.hidden)
