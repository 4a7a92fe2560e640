"""CPU oracle for the MoE dispatch / combine hot path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. The product path (``combine_quant_gb300``) never
imports it, and the two share no code: the arithmetic lives in
``cq_oracle.c``, a plain sequential C implementation of what the pages define
(see the citations there), and this module only moves numpy arrays in and out.

Parity status of each oracle function is pinned by ``tests/test_oracle_*.py``
against worked examples from the pages, closed forms, library cross-checks and
brute force; see the tests for the pin behind each function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cq_oracle.c")
_HDR = os.path.join(_HERE, "cq_oracle.h")
_SO = os.path.join(_HERE, "libcq_oracle.so")

OK = 0
ERR_ARG = -1
ERR_UNSUPPORTED = -2
ST_BAD_ID = 1
ST_BAD_MASK = 2
INV_NONE = -1
INV_COPY = -2
INV_CONST_BASE = -3

_FIELDS = (
    "ep_world_size", "moe_expert_num", "shared_expert_num", "shared_expert_rank_num",
    "zero_expert_num", "copy_expert_num", "const_expert_num", "max_bs", "topk", "hidden",
    "global_bs", "quant_mode", "expert_token_nums_type", "mask_ndim", "x_dtype", "smooth_kind",
    "y_dtype",
)


class _Cfg(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in _FIELDS]


def build(force: bool = False) -> str:
    """Compile cq_oracle.c into libcq_oracle.so next to it (gcc, no fast-math,
    no FP contraction, so each float operation is one IEEE rounding)."""
    stale = (not os.path.exists(_SO)) or any(
        os.path.getmtime(p) > os.path.getmtime(_SO) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-Wall", "-Werror", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        cfgp = ctypes.POINTER(_Cfg)
        L.cqo_check_config.argtypes = [cfgp]
        L.cqo_check_config.restype = ctypes.c_int
        for name in ("cqo_local_expert_num", "cqo_num_slots", "cqo_scale_cols"):
            getattr(L, name).argtypes = [cfgp]
            getattr(L, name).restype = ctypes.c_int32
        L.cqo_max_rows.argtypes = [cfgp]
        L.cqo_max_rows.restype = ctypes.c_int64
        L.cqo_route.argtypes = [cfgp] + [P] * 10
        L.cqo_route.restype = ctypes.c_int64
        L.cqo_quant_row.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P, P]
        L.cqo_quant_row.restype = ctypes.c_int
        L.cqo_quant_row2.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P]
        L.cqo_quant_row2.restype = ctypes.c_int
        L.cqo_quant_row3.argtypes = [ctypes.c_int32] * 4 + [P] * 5
        L.cqo_quant_row3.restype = ctypes.c_int
        L.cqo_group_cols.argtypes = [cfgp]
        L.cqo_group_cols.restype = ctypes.c_int32
        L.cqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.cqo_f16_to_f32.restype = ctypes.c_float
        L.cqo_f16_from_f32.argtypes = [ctypes.c_float]
        L.cqo_f16_from_f32.restype = ctypes.c_uint16
        L.cqo_floor_log2.argtypes = [ctypes.c_float]
        L.cqo_floor_log2.restype = ctypes.c_int32
        L.cqo_dispatch.argtypes = [cfgp] + [P] * 16
        L.cqo_dispatch.restype = ctypes.c_int64
        L.cqo_combine_token.argtypes = [cfgp, ctypes.c_int32, ctypes.c_int32] + [P] * 7 + [
            ctypes.c_int32, P]
        L.cqo_combine_token.restype = ctypes.c_int
        L.cqo_combine.argtypes = [cfgp] + [P] * 7 + [ctypes.c_int32, P]
        L.cqo_combine.restype = ctypes.c_int
        L.cqo_e4m3_encode.argtypes = [ctypes.c_float]
        L.cqo_e4m3_encode.restype = ctypes.c_uint8
        L.cqo_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.cqo_e4m3_decode.restype = ctypes.c_float
        L.cqo_e5m2_encode.argtypes = [ctypes.c_float]
        L.cqo_e5m2_encode.restype = ctypes.c_uint8
        L.cqo_e5m2_decode.argtypes = [ctypes.c_uint8]
        L.cqo_e5m2_decode.restype = ctypes.c_float
        L.cqo_bf16_from_f32.argtypes = [ctypes.c_float]
        L.cqo_bf16_from_f32.restype = ctypes.c_uint16
        L.cqo_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.cqo_bf16_to_f32.restype = ctypes.c_float
        L.cqo_ceil_log2.argtypes = [ctypes.c_float]
        L.cqo_ceil_log2.restype = ctypes.c_int32
        for name in ("cqo_e4m3_encode_n", "cqo_e5m2_encode_n", "cqo_bf16_from_f32_n",
                     "cqo_ceil_log2_n"):
            getattr(L, name).argtypes = [P, P, ctypes.c_int64]
            getattr(L, name).restype = None
        L.cqo_combine_quant_row.argtypes = [ctypes.c_int32, ctypes.c_int32, P, P, P]
        L.cqo_combine_quant_row.restype = ctypes.c_int
        L.cqo_combine_token_q8.argtypes = [cfgp, ctypes.c_int32, ctypes.c_int32] + [P] * 8 + [
            ctypes.c_int32, P]
        L.cqo_combine_token_q8.restype = ctypes.c_int
        _LIB = L
    return _LIB


def _cfg(cfg: dict) -> _Cfg:
    return _Cfg(**{f: int(cfg.get(f, 0)) for f in _FIELDS})


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def check_config(cfg: dict) -> int:
    return lib().cqo_check_config(ctypes.byref(_cfg(cfg)))


def local_expert_num(cfg: dict) -> int:
    return lib().cqo_local_expert_num(ctypes.byref(_cfg(cfg)))


def num_slots(cfg: dict) -> int:
    return lib().cqo_num_slots(ctypes.byref(_cfg(cfg)))


def max_rows(cfg: dict) -> int:
    return lib().cqo_max_rows(ctypes.byref(_cfg(cfg)))


def scale_cols(cfg: dict) -> int:
    return lib().cqo_scale_cols(ctypes.byref(_cfg(cfg)))


@dataclass
class Route:
    rows: int
    expand_idx: np.ndarray       # int32 [W, BS, NS]
    ep_recv_count: np.ndarray    # int32 [W, W*L]
    expert_token_nums: np.ndarray  # int64 [W, L]
    rank_row_base: np.ndarray    # int64 [W+1]
    assist: np.ndarray           # int32 [R_max, 4]
    inv: np.ndarray              # int32 [W, BS, NS]
    status: int


def _route_buffers(cfg):
    W, BS = cfg["ep_world_size"], cfg["max_bs"]
    NS, L, R = num_slots(cfg), local_expert_num(cfg), max_rows(cfg)
    return dict(
        expand_idx=np.empty((W, BS, NS), np.int32),
        ep_recv_count=np.empty((W, W * L), np.int32),
        expert_token_nums=np.empty((W, L), np.int64),
        rank_row_base=np.empty((W + 1,), np.int64),
        assist=np.zeros((R, 4), np.int32),
        inv=np.empty((W, BS, NS), np.int32),
    )


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def route(cfg: dict, expert_ids, mask=None, bs_per_rank=None) -> Route:
    rc = check_config(cfg)
    if rc != OK:
        raise ValueError(f"oracle rejects config: {rc}")
    b = _route_buffers(cfg)
    st = ctypes.c_uint32(0)
    ids = _c(expert_ids, np.int32)
    m = _c(mask, np.uint8)
    bpr = _c(bs_per_rank, np.int32)
    rows = lib().cqo_route(ctypes.byref(_cfg(cfg)), _ptr(ids), _ptr(m), _ptr(bpr),
                           _ptr(b["expand_idx"]), _ptr(b["ep_recv_count"]),
                           _ptr(b["expert_token_nums"]), _ptr(b["rank_row_base"]),
                           _ptr(b["assist"]), _ptr(b["inv"]), ctypes.byref(st))
    if rows < 0:
        raise ValueError(f"oracle route failed: {rows}")
    return Route(rows=int(rows), status=int(st.value), **b)


def _scale_buffer(mode: int, H: int):
    if mode == 2:
        return np.empty(1, np.float32)
    if mode == 3:
        return np.empty((H + 127) // 128, np.float32)
    if mode in (4, 5):
        return np.empty(((H + 31) // 32 + 1) // 2 * 2, np.uint8)
    return None


def quant_row(mode: int, x_row_bits, smooth_row=None, x_dtype: int = 0, smooth_scalar=None,
              y_dtype: int = 0):
    """Quantise one 16-bit row (uint16 bit patterns of bf16, or fp16 when
    x_dtype == 1). Returns (codes, scale): scale is a float (mode 2), a
    per-group float row (mode 3), an e8m0 byte row (modes 4, 5) or None.
    y_dtype picks the fp8 code type of modes 3-5 (0 e4m3fn, 1 e5m2)."""
    x = _c(x_row_bits, np.uint16)
    H = x.shape[0]
    sm = _c(smooth_row, np.float32)
    sc = None if smooth_scalar is None else np.asarray([smooth_scalar], np.float32)
    codes = np.empty(H, code_dtype(mode))
    scale = _scale_buffer(mode, H)
    rc = lib().cqo_quant_row3(mode, x_dtype, y_dtype, H, _ptr(x), _ptr(sm), _ptr(sc),
                              _ptr(codes), _ptr(scale))
    if rc != OK:
        raise ValueError(f"oracle quant_row failed: {rc}")
    return codes, (None if scale is None else (scale[0] if mode == 2 else scale))


def code_dtype(mode: int):
    return {0: np.uint16, 1: np.int8, 2: np.int8, 3: np.uint8, 4: np.uint8, 5: np.uint8}[mode]


def group_cols(cfg: dict) -> int:
    return lib().cqo_group_cols(ctypes.byref(_cfg(cfg)))


def dispatch(cfg: dict, x_bits, expert_ids, smooth=None, mask=None, bs_per_rank=None,
             expert_scales=None) -> dict:
    """Full dispatch (every row quantised). Returns a dict of numpy arrays."""
    rc = check_config(cfg)
    if rc != OK:
        raise ValueError(f"oracle rejects config: {rc}")
    H, mode = cfg["hidden"], cfg["quant_mode"]
    R = max_rows(cfg)
    b = _route_buffers(cfg)
    expand_x = np.zeros((R, H), code_dtype(mode))
    if mode == 2:
        dyn = np.zeros((R,), np.float32)
    elif mode == 3:
        dyn = np.zeros((R, group_cols(cfg)), np.float32)
    elif mode in (4, 5):
        dyn = np.zeros((R, scale_cols(cfg)), np.uint8)
    else:
        dyn = None
    es = np.zeros((R,), np.float32)
    st = ctypes.c_uint32(0)
    xs = _c(x_bits, np.uint16)
    ids = _c(expert_ids, np.int32)
    sm = _c(smooth, np.float32)
    m = _c(mask, np.uint8)
    bpr = _c(bs_per_rank, np.int32)
    w = _c(expert_scales, np.float32)
    rows = lib().cqo_dispatch(ctypes.byref(_cfg(cfg)), _ptr(xs), _ptr(ids), _ptr(sm), _ptr(m),
                              _ptr(bpr), _ptr(w), _ptr(expand_x), _ptr(dyn), _ptr(es),
                              _ptr(b["expand_idx"]), _ptr(b["ep_recv_count"]),
                              _ptr(b["expert_token_nums"]), _ptr(b["rank_row_base"]),
                              _ptr(b["assist"]), _ptr(b["inv"]), ctypes.byref(st))
    if rows < 0:
        raise ValueError(f"oracle dispatch failed: {rows}")
    out = dict(rows=int(rows), status=int(st.value), expand_x=expand_x, dynamic_scales=dyn,
               expand_scales=es)
    out.update(b)
    return out


def combine(cfg: dict, ffn_bits, inv, expert_scales, ori_x=None, const_alpha1=None,
            const_alpha2=None, const_v=None, out_f32=False):
    W, BS, H = cfg["ep_world_size"], cfg["max_bs"], cfg["hidden"]
    y = np.empty((W, BS, H), np.float32 if out_f32 else np.uint16)
    args = [_c(ffn_bits, np.uint16), _c(inv, np.int32), _c(expert_scales, np.float32),
            _c(ori_x, np.uint16), _c(const_alpha1, np.float32), _c(const_alpha2, np.float32),
            _c(const_v, np.uint16)]
    rc = lib().cqo_combine(ctypes.byref(_cfg(cfg)), *[_ptr(a) for a in args], int(out_f32),
                           _ptr(y))
    if rc != OK:
        raise ValueError(f"oracle combine failed: {rc}")
    return y


def combine_tokens(cfg: dict, tokens, ffn_bits, inv, expert_scales, ori_x=None,
                   const_alpha1=None, const_alpha2=None, const_v=None, out_f32=False):
    """Combine only the listed (r, i) tokens; returns [len(tokens), H]."""
    H = cfg["hidden"]
    y = np.empty((len(tokens), H), np.float32 if out_f32 else np.uint16)
    args = [_c(ffn_bits, np.uint16), _c(inv, np.int32), _c(expert_scales, np.float32),
            _c(ori_x, np.uint16), _c(const_alpha1, np.float32), _c(const_alpha2, np.float32),
            _c(const_v, np.uint16)]
    ptrs = [_ptr(a) for a in args]
    cfgc = _cfg(cfg)
    for n, (r, i) in enumerate(tokens):
        row = y[n]
        rc = lib().cqo_combine_token(ctypes.byref(cfgc), int(r), int(i), *ptrs, int(out_f32),
                                     _ptr(row))
        if rc != OK:
            raise ValueError(f"oracle combine_token failed: {rc}")
    return y


def e4m3_encode(v: float) -> int:
    return int(lib().cqo_e4m3_encode(float(v)))


def e4m3_decode(b: int) -> float:
    return float(lib().cqo_e4m3_decode(int(b)))


def e5m2_encode(v: float) -> int:
    return int(lib().cqo_e5m2_encode(float(v)))


def e5m2_decode(b: int) -> float:
    return float(lib().cqo_e5m2_decode(int(b)))


def bf16_from_f32(f: float) -> int:
    return int(lib().cqo_bf16_from_f32(float(f)))


def ceil_log2(q: float) -> int:
    return int(lib().cqo_ceil_log2(float(q)))


def floor_log2(a: float) -> int:
    return int(lib().cqo_floor_log2(float(a)))


def f16_from_f32(f: float) -> int:
    return int(lib().cqo_f16_from_f32(float(f)))


def f16_to_f32(h: int) -> float:
    return float(lib().cqo_f16_to_f32(int(h)))


def e4m3_encode_array(v) -> np.ndarray:
    a = _c(v, np.float32).reshape(-1)
    out = np.empty(a.shape, np.uint8)
    lib().cqo_e4m3_encode_n(_ptr(a), _ptr(out), a.size)
    return out


def e5m2_encode_array(v) -> np.ndarray:
    a = _c(v, np.float32).reshape(-1)
    out = np.empty(a.shape, np.uint8)
    lib().cqo_e5m2_encode_n(_ptr(a), _ptr(out), a.size)
    return out


def bf16_from_f32_array(v) -> np.ndarray:
    a = _c(v, np.float32).reshape(-1)
    out = np.empty(a.shape, np.uint16)
    lib().cqo_bf16_from_f32_n(_ptr(a), _ptr(out), a.size)
    return out


def ceil_log2_array(v) -> np.ndarray:
    a = _c(v, np.float32).reshape(-1)
    out = np.empty(a.shape, np.int32)
    lib().cqo_ceil_log2_n(_ptr(a), _ptr(out), a.size)
    return out


def combine_quant_row(row_bits, x_dtype: int = 0):
    """Combine-side int8 block quantisation of one 16-bit row: (codes, scales)."""
    x = _c(row_bits, np.uint16)
    H = x.shape[0]
    codes, scales = np.empty(H, np.int8), np.empty(H // 8, np.float32)
    rc = lib().cqo_combine_quant_row(H, x_dtype, _ptr(x), _ptr(codes), _ptr(scales))
    if rc != OK:
        raise ValueError(f"oracle combine_quant_row failed: {rc}")
    return codes, scales


def combine_quant_rows(rows_bits, x_dtype: int = 0):
    rows = _c(rows_bits, np.uint16)
    codes = np.empty(rows.shape, np.int8)
    scales = np.empty((rows.shape[0], rows.shape[1] // 8), np.float32)
    for n in range(rows.shape[0]):
        codes[n], scales[n] = combine_quant_row(rows[n], x_dtype)
    return codes, scales


def combine_tokens_q8(cfg: dict, tokens, codes, scales, inv, expert_scales, ori_x=None,
                      const_alpha1=None, const_alpha2=None, const_v=None, out_f32=False):
    """Combine the listed (r, i) tokens from int8 expert outputs."""
    H = cfg["hidden"]
    y = np.empty((len(tokens), H), np.float32 if out_f32 else np.uint16)
    args = [_c(codes, np.int8), _c(scales, np.float32), _c(inv, np.int32),
            _c(expert_scales, np.float32), _c(ori_x, np.uint16), _c(const_alpha1, np.float32),
            _c(const_alpha2, np.float32), _c(const_v, np.uint16)]
    ptrs = [_ptr(a) for a in args]
    cfgc = _cfg(cfg)
    for n, (r, i) in enumerate(tokens):
        rc = lib().cqo_combine_token_q8(ctypes.byref(cfgc), int(r), int(i), *ptrs, int(out_f32),
                                        _ptr(y[n]))
        if rc != OK:
            raise ValueError(f"oracle combine_token_q8 failed: {rc}")
    return y
