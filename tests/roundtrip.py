"""Dispatch, an identity expert FFN, then combine: the round trip of the
"tiny" configuration (combine with an identity FFN) and of the MXFP8 one
(full dispatch + combine round trip).

The identity FFN turns every dispatched row back into its token row: the
codes are dequantised with the row's carried scale (quant_mode 2: code times
1/scale; quant_mode 5: the e4m3 value times 2^(e - 127) of its 32-block) and,
where the row was multiplied by smooth scales, divided by them again; mode 0
rows are the token rows themselves. Combine must then give, per token, the
expert_scales-weighted sum of its token row over the routed slots, the shared
experts' rows unweighted, x for a copy expert and a1*x + a2*v for a const
expert ("MoeDistributeDispatch和MoeDistributeCombine算子设计介绍" §3.4 and
"low_latency_dispatch" 特殊专家场景), up to each row's quantisation step and
the rounding of the accumulation. closed_form() states that sum from the inputs,
with an error bound from each row's quantisation step; run_oracle() runs the
oracle's own round trip.
"""
from __future__ import annotations

import numpy as np

import oracle
from combine_quant_gb300 import workloads

INV_NONE, INV_COPY, INV_CONST_BASE = -1, -2, -3
_U = 2.0 ** -24  # unit roundoff of binary32


def _dims(cfg):
    W, BS, K, H = cfg["ep_world_size"], cfg["max_bs"], cfg["topk"], cfg["hidden"]
    S_eff = cfg["shared_expert_num"] if cfg["shared_expert_rank_num"] > 0 else 0
    return W, BS, K, H, K + S_eff


def _row_smooth(wl, ref, H):
    """Smooth scales each dispatched row was multiplied by, [R, H] float32
    (ones without smooth scales)."""
    cfg, R = wl.cfg, ref["rows"]
    if wl.smooth is None or cfg["quant_mode"] not in (1, 2, 3):
        return np.ones((R, H), np.float32)
    kind = cfg.get("smooth_kind", 0)
    if kind == 2:
        return np.full((R, H), float(wl.smooth.reshape(-1)[0]), np.float32)
    if kind == 1:
        return np.broadcast_to(wl.smooth.reshape(1, H), (R, H)).astype(np.float32)
    K = cfg["topk"]
    S_eff = cfg["shared_expert_num"] if cfg["shared_expert_rank_num"] > 0 else 0
    src, tok, k = (ref["assist"][:R, c] for c in range(3))
    k_c = np.minimum(k, K - 1)
    table_row = np.where(k < K, S_eff + wl.expert_ids[src, tok, k_c], k - K)
    return wl.smooth[table_row]


def _e4m3_table() -> np.ndarray:
    return np.array([oracle.e4m3_decode(b) for b in range(256)], np.float64)


def identity_ffn(wl, ref) -> tuple[np.ndarray, np.ndarray]:
    """The expert outputs of an identity FFN, bf16 bits [R_max, H], and the
    bound on |row - token row| per element, float64 [R, H]."""
    cfg, R = wl.cfg, ref["rows"]
    mode, H = cfg["quant_mode"], cfg["hidden"]
    out = np.zeros((ref["expand_x"].shape[0], H), np.uint16)
    src, tok = ref["assist"][:R, 0], ref["assist"][:R, 1]
    x = workloads.bf16_bits_to_f32(wl.x[src, tok]).astype(np.float64)
    if mode == 0:
        out[:R] = ref["expand_x"][:R]
        return out, np.zeros((R, H))
    if mode == 2:
        c = ref["dynamic_scales"][:R].astype(np.float32)
        sm = _row_smooth(wl, ref, H)
        deq = ref["expand_x"][:R].astype(np.float32) * c[:, None]  # binary32 products
        row = (deq / sm).astype(np.float32)
        out[:R] = workloads.to_bf16_bits(row)
        c64, s64 = c.astype(np.float64)[:, None], np.abs(sm.astype(np.float64))
        # |code * c - x * s| <= c/2 + 3u|x s| (three roundings before the code),
        # then the product, the division and the bf16 cast.
        err = (0.5 * c64 + 6 * _U * np.abs(x) * s64) / s64
        return out, err + 2.0 ** -8 * (np.abs(x) + err)
    if mode == 5:
        vals = _e4m3_table()[ref["expand_x"][:R].view(np.uint8)]
        e = ref["dynamic_scales"][:R].astype(np.int64)[:, : (H + 31) // 32] - 127
        e_col = np.repeat(e, 32, axis=1)[:, :H]
        row = np.ldexp(vals, e_col)  # exact: <= 4 significant bits
        out[:R] = workloads.to_bf16_bits(row.astype(np.float32))
        # e4m3 round to nearest: half an ulp, 2^-4 relative (normal) or
        # 2^-10 absolute (subnormal), in units of the block's 2^e.
        err = np.maximum(2.0 ** -4 * np.abs(x), np.ldexp(1.0, e_col - 10))
        return out, err
    raise ValueError(f"no identity FFN for quant_mode {mode}")


def closed_form(wl, ref, row_err) -> tuple[np.ndarray, np.ndarray]:
    """Per token, what combine of the identity FFN's rows must return, and a
    bound on the difference, both float64 [W, BS, H]."""
    cfg = wl.cfg
    W, BS, K, H, NS = _dims(cfg)
    x = workloads.bf16_bits_to_f32(wl.x).astype(np.float64)
    inv = ref["inv"].reshape(W, BS, NS)
    target = np.zeros((W, BS, H))
    err = np.zeros((W, BS, H))
    mag = np.zeros((W, BS, H))
    for k in range(NS):
        code = inv[:, :, k]
        w = (wl.expert_scales[:, :, k].astype(np.float64) if k < K
             else np.ones((W, BS)))[:, :, None]
        routed = (code >= 0)[:, :, None]
        copy = (code == INV_COPY)[:, :, None]
        term = np.where(routed | copy, w * x, 0.0)
        term_mag = np.abs(term)
        if cfg["const_expert_num"] > 0:
            cidx = np.clip(INV_CONST_BASE - code, 0, cfg["const_expert_num"] - 1)
            is_const = (code <= INV_CONST_BASE)[:, :, None]
            a1 = wl.const_alpha1.astype(np.float64)[cidx][:, :, None]
            a2 = wl.const_alpha2.astype(np.float64)[cidx][:, :, None]
            v = workloads.bf16_bits_to_f32(wl.const_v).astype(np.float64)[cidx]
            cterm = w * (a1 * x + a2 * v)
            term = np.where(is_const, cterm, term)
            term_mag = np.where(is_const, np.abs(w) * (np.abs(a1 * x) + np.abs(a2 * v)),
                                term_mag)
        target += term
        mag += term_mag
        rows = np.where(code >= 0, code, 0)
        err += np.where(routed, np.abs(w) * row_err[rows], 0.0)
    # each fused multiply-add of the fixed-order chain, and the const
    # expert's three roundings, add at most u times the magnitudes involved
    bound = err + (NS + 4) * _U * (mag + err) + 1e-30
    return target, bound


def run_oracle(wl):
    """The oracle's round trip: its dispatch, the identity FFN of its rows,
    its combine (binary32 output). Returns (dispatch dict, FFN bits, row
    error bound, y)."""
    ref = oracle.dispatch(wl.cfg, wl.x, wl.expert_ids,
                          wl.smooth if wl.cfg["quant_mode"] in (1, 2, 3) else None,
                          wl.mask, wl.bs_per_rank, wl.expert_scales)
    ffn, row_err = identity_ffn(wl, ref)
    y = oracle.combine(wl.cfg, ffn, ref["inv"], wl.expert_scales, wl.x, wl.const_alpha1,
                       wl.const_alpha2, wl.const_v, out_f32=True)
    return ref, ffn, row_err, y
