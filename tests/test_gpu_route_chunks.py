"""The routing scan counts each source's tokens in chunks, one count CTA
per chunk (chunks of about 64 tokens, at most 128 count CTAs and at most
2048 (local expert, source, chunk) entries per rank); offsets_kernel chains the
chunks of a source. These cases put chunk boundaries where they matter and
compare every dispatch output of cq_dispatch_route + cq_dispatch_permute
(always the chunked kernels) with the oracle: per-rank batch sizes ending inside, at
and before chunks; 1-D and 2-D masks; shared experts with replicas (their
ordinal counts active tokens across chunks); zero, copy and const experts;
duplicate and invalid ids; a hot expert that every chunk of every source
sends to."""
import numpy as np
import pytest
import torch

import combine_quant_gb300 as cq
import oracle
from combine_quant_gb300 import workloads

import gpu_harness as gh

pytestmark = pytest.mark.gpu


def _case(seed, W, M, BS, K, H=1024, mode=2, **kw):
    rng = np.random.default_rng(seed)
    cfg = workloads.make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                                quant_mode=mode, **{k: v for k, v in kw.items()
                                                    if k in workloads.CONFIG_FIELDS})
    n_all = M + cfg["zero_expert_num"] + cfg["copy_expert_num"] + cfg["const_expert_num"]
    ids = np.stack([rng.permutation(n_all)[:K] for _ in range(W * BS)]).reshape(W, BS, K)
    x = workloads.to_bf16_bits(rng.standard_normal((W, BS, H)).astype(np.float32))
    w = rng.uniform(0, 1, (W, BS, K)).astype(np.float32)
    wl = workloads.Workload("chunks", cfg, x, ids.astype(np.int32), w, seed=seed)
    Q = cfg["const_expert_num"]
    if Q:
        wl.const_alpha1 = rng.uniform(0.5, 1.5, Q).astype(np.float32)
        wl.const_alpha2 = rng.uniform(0.5, 1.5, Q).astype(np.float32)
        wl.const_v = workloads.to_bf16_bits(rng.standard_normal((Q, H)).astype(np.float32))
    return wl, rng


def _cases():
    out = {}
    # 4 sources x 4 chunks of 64 tokens; batch sizes ending inside, at and
    # before chunk boundaries, and an empty source
    wl, rng = _case(71, W=4, M=16, BS=256, K=4)
    wl.bs_per_rank = np.array([77, 256, 0, 32], np.int32)
    out["ragged_batch_sizes"] = wl
    # 1-D mask whose active prefix ends mid-chunk
    wl, rng = _case(72, W=8, M=32, BS=128, K=8, mask_ndim=1, mode=0)
    wl.mask = np.zeros((8, 128), np.uint8)
    for r, n in enumerate([128, 100, 33, 31, 64, 1, 0, 96]):
        wl.mask[r, :n] = 1
    out["mask1d_prefixes"] = wl
    # 2-D mask with duplicate and invalid ids
    wl, rng = _case(73, W=4, M=12, BS=192, K=6, mask_ndim=2, zero_expert_num=1,
                    copy_expert_num=1, const_expert_num=1)
    wl.expert_ids = rng.integers(-1, 16, (4, 192, 6)).astype(np.int32)  # 15, -1: invalid
    wl.mask = (rng.random((4, 192, 6)) < 0.6).astype(np.uint8)
    out["mask2d_duplicates_invalid_special"] = wl
    # shared experts with replicas; per-rank batch sizes
    wl, rng = _case(74, W=8, M=24, BS=192, K=4, shared_expert_num=2, shared_expert_rank_num=4,
                    const_expert_num=1)
    wl.bs_per_rank = np.array([192, 150, 65, 64, 63, 1, 190, 128], np.int32)
    wl.smooth = rng.uniform(0.5, 1.5, (2 + 24, 1024)).astype(np.float32)
    out["shared_replicas_per_expert_smooth"] = wl
    # one hot expert in every pair's first slot
    wl, rng = _case(75, W=2, M=8, BS=512, K=3, mode=5)
    wl.expert_ids[:, :, 0] = 5
    wl.expert_ids[:, :, 1:] = np.where(wl.expert_ids[:, :, 1:] == 5, 6, wl.expert_ids[:, :, 1:])
    out["hot_expert_mx"] = wl
    return out


def _split_dispatch(wl):
    """cq_dispatch_route + cq_dispatch_permute: the chunked count kernel, at
    any batch size (cq_dispatch may take the one-kernel path here)."""
    cfg = cq.Config.from_dict(wl.cfg)
    ids = gh.dev(wl.expert_ids, torch.int32)
    mask, bpr = gh.dev(wl.mask, torch.uint8), gh.dev(wl.bs_per_rank, torch.int32)
    ws = cq.alloc_workspace(cfg, gh.DEV)
    out = cq.alloc_dispatch_outputs(cfg, gh.DEV)
    cq.dispatch_route(cfg, ids, mask, bpr, workspace=ws, out=out)
    cq.dispatch_permute(cfg, gh.dev(wl.x, cfg.token_dtype), ids,
                        gh.dev(wl.smooth, torch.float32) if gh.uses_smooth(wl) else None,
                        gh.dev(wl.expert_scales, torch.float32), mask, bpr, workspace=ws, out=out)
    return cfg, out, cq.read_status(ws)


@pytest.mark.parametrize("name", list(_cases()))
def test_chunked_routing_against_the_oracle(name):
    wl = _cases()[name]
    cfg, out, status = _split_dispatch(wl)
    ref = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids, wl.smooth if gh.uses_smooth(wl) else None,
                          wl.mask, wl.bs_per_rank, wl.expert_scales)
    assert status == ref["status"]
    route = oracle.Route(ref["rows"], ref["expand_idx"], ref["ep_recv_count"],
                         ref["expert_token_nums"], ref["rank_row_base"], ref["assist"],
                         ref["inv"], ref["status"])
    gh.compare_route(wl, cfg, out, route)
    R = ref["rows"]
    assert R > 0
    assert np.array_equal(gh.host(out.expand_x[:R]).view(ref["expand_x"].dtype), ref["expand_x"][:R])
    if ref["dynamic_scales"] is not None:
        assert np.array_equal(gh.host(out.dynamic_scales[:R]).view(np.uint8),
                              ref["dynamic_scales"][:R].view(np.uint8))
    assert np.array_equal(gh.host(out.expand_scales[:R]), ref["expand_scales"][:R])
