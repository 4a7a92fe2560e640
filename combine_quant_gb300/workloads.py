"""Seeded synthetic inputs for the MoE dispatch / combine path.

This module only draws inputs. It holds none of the method's arithmetic (no
routing scan, no quantisation, no weighted sum), so the CPU oracle and the
CUDA path can both consume what it produces.

Five workloads follow the shapes the pages use (DeepSeek-V3 MoE shape, hidden
7168, top-8; the sample on the performance page uses the same H and K):

  tiny     W=4,  M=8 (L=2),   BS=8,   K=2,  H=1024, modes 0 and 2 (+smooth)
  dsv3     W=32, M=256 (L=8), BS=128, K=8,  H=7168, mode 2, counts
  mxfp8    W=64, M=256 (L=4), BS=512, K=8,  H=7168, mode 5 (e4m3, 32-blocks)
  special  W=16, S_r=2, S=1, M=112 (L=8), Z=C=Q=1, K=6, BS=256, H=4096,
           mode 0, 1-D mask (last quarter false), cumulative sums
  skew     W=16, M=128 (L=8), K=16, H=8192, per-rank BS ~ U[1,512], Zipf(1.2)
           expert popularity, mode 2 with smooth scales

Every array is produced by numpy's PCG64 generator from the workload's seed.
x and other bf16 tensors are returned as uint16 bit patterns, rounded from
float32 by torch's CPU cast (round to nearest even).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

CONFIG_FIELDS = (
    "ep_world_size", "moe_expert_num", "shared_expert_num", "shared_expert_rank_num",
    "zero_expert_num", "copy_expert_num", "const_expert_num", "max_bs", "topk", "hidden",
    "global_bs", "quant_mode", "expert_token_nums_type", "mask_ndim", "x_dtype", "smooth_kind",
    "y_dtype",
)


def make_config(**kw) -> dict:
    """A config dict with every field present (defaults 0, etn type 1)."""
    cfg = {f: 0 for f in CONFIG_FIELDS}
    cfg["expert_token_nums_type"] = 1
    for k, v in kw.items():
        if k not in cfg:
            raise KeyError(k)
        cfg[k] = int(v)
    return cfg


@dataclass
class Workload:
    name: str
    cfg: dict
    x: np.ndarray                       # uint16 bf16 bits [W, BS, H]
    expert_ids: np.ndarray              # int32 [W, BS, K]
    expert_scales: np.ndarray           # float32 [W, BS, K]
    smooth: Optional[np.ndarray] = None  # float32 [S_eff + M, H]
    mask: Optional[np.ndarray] = None   # uint8 [W, BS] or [W, BS, K]
    bs_per_rank: Optional[np.ndarray] = None  # int32 [W]
    const_alpha1: Optional[np.ndarray] = None  # float32 [Q]
    const_alpha2: Optional[np.ndarray] = None  # float32 [Q]
    const_v: Optional[np.ndarray] = None       # uint16 bf16 bits [Q, H]
    seed: int = 0
    notes: dict = field(default_factory=dict)

    def with_mode(self, mode: int) -> "Workload":
        """The same inputs under another quant_mode. Modes 1-3 keep the smooth
        scales; mode 1 (static scales) without any takes one (H,) row of 32.0,
        which spreads N(0, 1) tokens over the int8 range."""
        cfg = dict(self.cfg)
        cfg["quant_mode"] = int(mode)
        smooth = self.smooth if mode in (1, 2, 3) else None
        if mode == 1 and smooth is None:
            smooth = np.full(cfg["hidden"], 32.0, np.float32)
            cfg["smooth_kind"] = 1
        return Workload(self.name + f"_m{mode}", cfg, self.x, self.expert_ids,
                        self.expert_scales, smooth, self.mask, self.bs_per_rank,
                        self.const_alpha1, self.const_alpha2, self.const_v, self.seed,
                        dict(self.notes))

    @property
    def tokens(self) -> int:
        """Active-range tokens (sum of per-rank BS)."""
        if self.bs_per_rank is not None:
            return int(self.bs_per_rank.sum())
        return self.cfg["ep_world_size"] * self.cfg["max_bs"]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_f16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def as_fp16(wl: "Workload") -> "Workload":
    """The same workload with fp16 tokens: x and const_v re-rounded from
    their bf16 values to fp16 (round to nearest even), x_dtype = 1."""
    cfg = dict(wl.cfg, x_dtype=1)
    f16 = lambda b: None if b is None else to_f16_bits(bf16_bits_to_f32(b))  # noqa: E731
    return Workload(wl.name + "_f16", cfg, f16(wl.x), wl.expert_ids, wl.expert_scales,
                    wl.smooth, wl.mask, wl.bs_per_rank, wl.const_alpha1, wl.const_alpha2,
                    f16(wl.const_v), wl.seed, dict(wl.notes))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _softmax(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def _distinct_uniform(rng, n_tok: int, n_choices: int, k: int) -> np.ndarray:
    """k distinct ids per token, uniform over [0, n_choices)."""
    keys = rng.random((n_tok, n_choices))
    return np.argsort(keys, axis=1)[:, :k].astype(np.int32)


def _normal_bf16(rng, shape) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def tiny(seed: int = 0, quant_mode: int = 2) -> Workload:
    W, M, BS, K, H = 4, 8, 8, 2, 1024
    rng = np.random.Generator(np.random.PCG64(seed))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                      quant_mode=quant_mode, expert_token_nums_type=1)
    x = _normal_bf16(rng, (W, BS, H))
    ids = _distinct_uniform(rng, W * BS, M, K).reshape(W, BS, K)
    w = _softmax(rng.standard_normal((W, BS, K), dtype=np.float32))
    smooth = rng.uniform(0.5, 1.5, (M, H)).astype(np.float32)
    return Workload("tiny", cfg, x, ids, w, smooth if quant_mode == 2 else None, seed=seed)


def _router_topk(rng, n_tok: int, M: int, K: int, bias_sd: float):
    logits = rng.standard_normal((n_tok, M), dtype=np.float32)
    if bias_sd > 0:
        logits = logits + rng.normal(0.0, bias_sd, (M,)).astype(np.float32)[None, :]
    ids = np.argsort(-logits, axis=1, kind="stable")[:, :K].astype(np.int32)
    sel = np.take_along_axis(logits, ids, axis=1)
    return ids, _softmax(sel)


def dsv3(seed: int = 1, W: int = 32, BS: int = 128, M: int = 256, K: int = 8,
         H: int = 7168) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                      quant_mode=2, expert_token_nums_type=1)
    xf = rng.standard_normal((W, BS, H), dtype=np.float32)
    n_out = max(1, int(round(0.01 * xf.size)))
    pos = rng.choice(xf.size, n_out, replace=False)
    xf.reshape(-1)[pos] *= 20.0  # 1 % outliers x20
    ids, w = _router_topk(rng, W * BS, M, K, bias_sd=0.5)
    return Workload("dsv3", cfg, to_bf16_bits(xf), ids.reshape(W, BS, K),
                    w.reshape(W, BS, K), seed=seed)


def mxfp8(seed: int = 2, W: int = 64, BS: int = 512, M: int = 256, K: int = 8,
          H: int = 7168) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                      quant_mode=5, expert_token_nums_type=1)
    xf = rng.standard_normal((W, BS, H), dtype=np.float32)
    xf *= rng.lognormal(0.0, 1.0, (W, BS, 1)).astype(np.float32)  # one scale per row
    ids, w = _router_topk(rng, W * BS, M, K, bias_sd=0.0)
    return Workload("mxfp8", cfg, to_bf16_bits(xf), ids.reshape(W, BS, K),
                    w.reshape(W, BS, K), seed=seed)


def special(seed: int = 3, W: int = 16, BS: int = 256, H: int = 4096, M: int = 112) -> Workload:
    Sr, S, Z, C, Q, K = 2, 1, 1, 1, 1, 6
    rng = np.random.Generator(np.random.PCG64(seed))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, shared_expert_num=S,
                      shared_expert_rank_num=Sr, zero_expert_num=Z, copy_expert_num=C,
                      const_expert_num=Q, max_bs=BS, topk=K, hidden=H, quant_mode=0,
                      expert_token_nums_type=0, mask_ndim=1)
    x = _normal_bf16(rng, (W, BS, H))
    ids = _distinct_uniform(rng, W * BS, M + Z + C + Q, K).reshape(W, BS, K)
    w = _softmax(rng.standard_normal((W, BS, K), dtype=np.float32))
    mask = np.ones((W, BS), np.uint8)
    mask[:, BS - BS // 4:] = 0  # last quarter of every rank inactive
    a1 = rng.uniform(0.5, 1.5, (Q,)).astype(np.float32)
    a2 = rng.uniform(0.5, 1.5, (Q,)).astype(np.float32)
    v = _normal_bf16(rng, (Q, H))
    return Workload("special", cfg, x, ids, w, None, mask, None, a1, a2, v, seed=seed)


def skew(seed: int = 4, W: int = 16, BS: int = 512, M: int = 128, K: int = 16,
         H: int = 8192) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=BS, topk=K, hidden=H,
                      global_bs=BS * W, quant_mode=2, expert_token_nums_type=1)
    bs = rng.integers(1, BS + 1, (W,)).astype(np.int32)
    x = _normal_bf16(rng, (W, BS, H))
    # Zipf(s=1.2) popularity p_e ~ (e+1)^-1.2; K draws without replacement per
    # token by Gumbel-top-k on log p.
    logp = -1.2 * np.log(np.arange(1, M + 1, dtype=np.float64))
    g = rng.gumbel(size=(W * BS, M))
    ids = np.argsort(-(logp[None, :] + g), axis=1)[:, :K].astype(np.int32).reshape(W, BS, K)
    w = _softmax(rng.standard_normal((W, BS, K), dtype=np.float32))
    smooth = rng.uniform(0.5, 1.5, (M, H)).astype(np.float32)
    return Workload("skew", cfg, x, ids, w, smooth, None, bs, seed=seed)


def perf_table(bs: int, seed: int = 5, quant_mode: int = 0) -> Workload:
    """The shape of the performance table of "CANN MoE Dispatch/Combine 通信
    算子性能优化实践" (性能数据): 8 ranks, 4 experts per rank, K=8, H=7168,
    BS 8 or 256 per rank. Routing: top-8 of N(0,1) logits; x ~ N(0,1)."""
    W, L, K, H = 8, 4, 8, 7168
    M = W * L
    rng = np.random.Generator(np.random.PCG64(seed + bs))
    cfg = make_config(ep_world_size=W, moe_expert_num=M, max_bs=bs, topk=K, hidden=H,
                      quant_mode=quant_mode, expert_token_nums_type=1)
    x = _normal_bf16(rng, (W, bs, H))
    ids, w = _router_topk(rng, W * bs, M, K, bias_sd=0.0)
    return Workload(f"perf_table_bs{bs}", cfg, x, ids.reshape(W, bs, K), w.reshape(W, bs, K),
                    seed=seed)


WORKLOADS = {"tiny": tiny, "dsv3": dsv3, "mxfp8": mxfp8, "special": special, "skew": skew,
             "perf8": lambda: perf_table(8), "perf256": lambda: perf_table(256)}


def ffn_standin(seed: int, rows: int, H: int, chunk: int = 1 << 24,
                x_dtype: int = 0) -> np.ndarray:
    """Stand-in for the experts' FFN output, 16-bit bits [rows, H] (bf16, or
    fp16 when x_dtype == 1): values N(0,1) rounded to nearest even. Drawn in
    chunks to bound host memory spikes."""
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    conv = to_f16_bits if x_dtype == 1 else to_bf16_bits
    out = np.empty((rows, H), np.uint16)
    flat = out.reshape(-1)
    for s in range(0, flat.size, chunk):
        n = min(chunk, flat.size - s)
        flat[s:s + n] = conv(rng.standard_normal(n, dtype=np.float32))
    return out
