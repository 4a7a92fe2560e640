"""GPU parity on seeded random configurations drawn over the valid parameter
space (W, shared-expert ranks and replicas, local experts, zero / copy /
const experts, K, BS and per-rank BS, H, quant_mode 0-5 with every smooth
shape, e5m2 codes, fp16 tokens, 1-D / 2-D masks, duplicate and out-of-range
ids, both expert_token_nums types): every output of dispatch and combine
against the oracle, element by element, and the status words."""
import numpy as np
import pytest

import gpu_harness as gh
from combine_quant_gb300 import workloads

pytestmark = pytest.mark.gpu


def _divisors(n):
    return [d for d in range(1, n + 1) if n % d == 0]


def random_workload(seed):
    rng = np.random.default_rng(1000 + seed)
    W = int(rng.choice([2, 3, 4, 6, 8, 12, 16]))
    Sr = 0
    S = 0
    if rng.random() < 0.4:
        Sr = int(rng.choice([d for d in _divisors(W) if d < W]))
        S = int(rng.choice([d for d in _divisors(Sr) if d <= 4]))
    L = int(rng.choice([1, 2, 3, 4, 8]))
    M = L * (W - Sr)
    Z, C, Q = (int(rng.random() < 0.3) * int(rng.integers(1, 3)) for _ in range(3))
    n_ids = M + Z + C + Q
    K = int(rng.integers(1, min(16, n_ids) + 1))
    BS = int(rng.integers(1, 25))
    mode = int(rng.integers(0, 6))
    H = int(rng.choice([1024, 2048, 3072] + ([1040, 1056] if mode < 4 else [1056])))
    kind = int(rng.integers(0, 3))
    smooth_given = mode == 1 or (mode in (2, 3) and rng.random() < 0.6)
    mask_ndim = int(rng.choice([0, 0, 1, 2]))
    cfg = workloads.make_config(
        ep_world_size=W, moe_expert_num=M, shared_expert_num=S, shared_expert_rank_num=Sr,
        zero_expert_num=Z, copy_expert_num=C, const_expert_num=Q, max_bs=BS, topk=K, hidden=H,
        global_bs=int(rng.choice([0, BS * W])), quant_mode=mode,
        expert_token_nums_type=int(rng.integers(0, 2)), mask_ndim=mask_ndim,
        smooth_kind=kind if smooth_given else 0,
        y_dtype=int(rng.random() < 0.5) if mode >= 3 else 0)
    # ids: K distinct per token, sometimes a duplicate or an out-of-range id
    keys = rng.random((W * BS, n_ids))
    ids = np.argsort(keys, axis=1)[:, :K].astype(np.int32)
    if K >= 2 and rng.random() < 0.3:
        t = rng.integers(0, W * BS, max(1, W * BS // 8))
        ids[t, 1] = ids[t, 0]
    if rng.random() < 0.15:
        t = rng.integers(0, W * BS, 2)
        ids[t, K - 1] = n_ids + 3
    ids = ids.reshape(W, BS, K)
    x = rng.standard_normal((W, BS, H)).astype(np.float32)
    x *= np.exp(rng.normal(0, 1.5, (W, BS, 1))).astype(np.float32)
    x = workloads.to_bf16_bits(x)
    w = rng.uniform(0, 1, (W, BS, K)).astype(np.float32)
    smooth = None
    if smooth_given:
        s_eff = S if Sr > 0 else 0
        if kind == 0:
            smooth = rng.uniform(0.5, 1.5, (s_eff + M, H)).astype(np.float32)
        elif kind == 1:
            smooth = rng.uniform(0.5, 1.5, H).astype(np.float32)
        else:
            smooth = np.array([rng.uniform(0.5, 4.0)], np.float32)
        if mode == 1:
            smooth *= np.float32(24.0)  # static scales that use the int8 range
    mask = None
    if mask_ndim == 1:
        n_on = rng.integers(0, BS + 1, W)
        mask = (np.arange(BS)[None, :] < n_on[:, None]).astype(np.uint8)
        if rng.random() < 0.2 and BS >= 3:
            mask[0, 1] = 0  # not a prefix: the status bit, rows as the oracle says
            mask[0, 2] = 1
    elif mask_ndim == 2:
        mask = (rng.random((W, BS, K)) < 0.8).astype(np.uint8)
    bpr = rng.integers(0, BS + 1, W).astype(np.int32) if rng.random() < 0.4 else None
    a1 = rng.uniform(0.5, 1.5, Q).astype(np.float32) if Q else None
    a2 = rng.uniform(0.5, 1.5, Q).astype(np.float32) if Q else None
    v = workloads.to_bf16_bits(rng.standard_normal((Q, H)).astype(np.float32)) if Q else None
    wl = workloads.Workload(f"random{seed}", cfg, x, ids, w, smooth, mask, bpr, a1, a2, v,
                            seed=seed)
    if rng.random() < 0.25:
        wl = workloads.as_fp16(wl)
    return wl


@pytest.mark.parametrize("seed", range(24))
def test_random_config_parity(seed):
    gh.full_parity(random_workload(seed))
