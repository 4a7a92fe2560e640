"""cq_dispatch of a small batch runs routing and permute in one kernel
(dispatch_small_kernel); its two halves, cq_dispatch_route and
cq_dispatch_permute, always run the three-kernel path. Both must leave every
output and the status word identical. The cases sit inside the one-kernel
path's limits (W * BS * K <= 2048, (S_r + M) * W <= 2048, quant_mode 0, 2 or
5 with e4m3 codes, W * BS * NS * H <= 2^23 with per-expert smooth rows;
each case asserts it) and cover each of its branches: masks of both shapes,
per-rank batch sizes, shared, zero, copy and const experts, invalid and
duplicate ids, every smooth shape of mode 2, fp16 tokens and the extremes of
K, BS and W. The oracle parity tests cover the same path on their own small
configurations."""
import numpy as np
import pytest
import torch

import combine_quant_gb300 as cq
from combine_quant_gb300 import workloads

import gpu_harness as gh

pytestmark = pytest.mark.gpu


def _case(seed, W=4, M=8, BS=8, K=2, H=1024, mode=2, **kw):
    rng = np.random.default_rng(seed)
    cfg = workloads.make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                                quant_mode=mode, **{k: v for k, v in kw.items()
                                                    if k in workloads.CONFIG_FIELDS})
    n_all = M + cfg["zero_expert_num"] + cfg["copy_expert_num"] + cfg["const_expert_num"]
    ids = np.stack([rng.permutation(n_all)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    x = workloads.to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    w = rng.uniform(0, 1, (W, BS, K)).astype(np.float32)
    wl = workloads.Workload("small", cfg, x, ids.astype(np.int32), w, seed=seed)
    Q = cfg["const_expert_num"]
    if Q:
        wl.const_alpha1 = rng.uniform(0.5, 1.5, Q).astype(np.float32)
        wl.const_alpha2 = rng.uniform(0.5, 1.5, Q).astype(np.float32)
        wl.const_v = workloads.to_bf16_bits(rng.standard_normal((Q, H)).astype(np.float32))
    return wl, rng


def _cases():
    out = {}
    out["tiny_m0"] = workloads.tiny(0, 0)
    out["tiny_m2_per_expert_smooth"] = workloads.tiny(0, 2)
    out["tiny_m5"] = workloads.tiny(0, 5)
    out["special_small"] = workloads.special(seed=51, W=8, BS=20, H=1024, M=48)
    # at both the pair limit and the per-expert-smooth limit (W * BS * NS * H = 2^23)
    out["skew_small_per_expert_smooth"] = workloads.skew(seed=52, W=4, BS=32, M=32, K=16,
                                                         H=4096)
    wl, rng = _case(53, W=3, M=6, BS=9, K=4, mask_ndim=2, zero_expert_num=1, copy_expert_num=1)
    wl.expert_ids = rng.integers(0, 9, (3, 9, 4)).astype(np.int32)  # 8: invalid; duplicates
    wl.mask = (rng.random((3, 9, 4)) < 0.7).astype(np.uint8)
    out["mask2d_duplicates_invalid"] = wl
    wl, rng = _case(54, W=6, M=12, BS=17, K=3, mask_ndim=1)
    wl.mask = np.ones((6, 17), np.uint8)
    wl.mask[:, 12:] = 0
    wl.mask[2, 5] = 0  # a false entry before true ones: status bit
    wl.bs_per_rank = np.array([0, 17, 1, 5, 0, 16], np.int32)
    out["mask1d_ragged_bad_prefix"] = wl
    wl, rng = _case(55, W=8, M=24, BS=6, K=3, shared_expert_num=2, shared_expert_rank_num=4,
                    const_expert_num=2, copy_expert_num=1)
    wl.smooth = rng.uniform(0.5, 1.5, (2 + 24, 1024)).astype(np.float32)
    out["shared_replicas_per_expert_smooth"] = wl
    wl, rng = _case(56, W=4, M=8, BS=16, K=4, smooth_kind=1)
    wl.smooth = rng.uniform(0.5, 1.5, 1024).astype(np.float32)
    out["smooth_shared_row"] = wl
    wl, rng = _case(57, W=4, M=8, BS=16, K=4, smooth_kind=2)
    wl.smooth = np.array([3.0], np.float32)
    out["smooth_scalar"] = wl
    out["fp16_m2"] = workloads.as_fp16(workloads.dsv3(seed=58, W=8, BS=12, M=32, K=8, H=1536))
    out["K16_W2"], _ = _case(59, W=2, M=16, BS=64, K=16, H=1024, mode=5)
    out["K1_BS1"], _ = _case(60, W=16, M=32, BS=1, K=1, H=8192, mode=0)
    out["dsv3_small_at_the_limit"] = workloads.dsv3(seed=61, W=8, BS=32, M=64, K=8, H=2048)
    # both limits at once: 2048 pairs and (S_r + M) * W = 2048 block counts
    out["pairs_and_blocks_at_the_limit"], _ = _case(62, W=32, M=64, BS=8, K=8, H=7168, mode=0)
    return out


def _uses(wl):
    return wl.smooth if wl.cfg["quant_mode"] in (1, 2, 3) else None


@pytest.mark.parametrize("name", list(_cases()))
def test_one_kernel_dispatch_matches_the_two_halves(name):
    wl = _cases()[name]
    cfg = cq.Config.from_dict(wl.cfg)
    assert cfg.check() == 0
    assert gh.one_kernel_dispatch(wl), "the case lies outside the one-kernel path"
    x = gh.dev(wl.x, cfg.token_dtype)
    ids = gh.dev(wl.expert_ids, torch.int32)
    sm, mask = gh.dev(_uses(wl), torch.float32), gh.dev(wl.mask, torch.uint8)
    bpr, w = gh.dev(wl.bs_per_rank, torch.int32), gh.dev(wl.expert_scales, torch.float32)
    outs, status = [], []
    for split in (False, True):
        ws = cq.alloc_workspace(cfg, gh.DEV)
        out = cq.alloc_dispatch_outputs(cfg, gh.DEV)
        for t in out:  # the same stale contents in both output sets
            if t is not None:
                t.view(torch.uint8).fill_(0x5A)
        if split:
            cq.dispatch_route(cfg, ids, mask, bpr, workspace=ws, out=out)
            cq.dispatch_permute(cfg, x, ids, sm, w, mask, bpr, workspace=ws, out=out)
        else:
            cq.dispatch(cfg, x, ids, smooth_scales=sm, x_active_mask=mask, bs_per_rank=bpr,
                        expert_scales=w, workspace=ws, out=out)
        status.append(cq.read_status(ws))
        outs.append(out)
    assert status[0] == status[1]
    R = int(gh.host(cq.assist_views(cfg, outs[1].assist_info)[2])[-1])
    a, b = outs
    for name_ in ("assist_info", "ep_recv_count", "expert_token_nums"):
        assert torch.equal(getattr(a, name_), getattr(b, name_)), name_
    assert torch.equal(a.expand_x[:R].view(torch.uint8), b.expand_x[:R].view(torch.uint8))
    assert torch.equal(a.expand_scales[:R], b.expand_scales[:R])
    if a.dynamic_scales is not None:
        assert torch.equal(a.dynamic_scales[:R].view(torch.uint8),
                           b.dynamic_scales[:R].view(torch.uint8))
