"""Torch-facing wrapper of the libcq C ABI.

PyTorch supplies device memory and the current stream; every step of the
path runs in libcq's CUDA kernels. Output tensors are allocated here (or
passed in) and handed to the C entry points as raw pointers.
"""
from __future__ import annotations

import ctypes
import functools
from dataclasses import asdict, dataclass, fields
from typing import NamedTuple, Optional

import torch

from . import _lib


@dataclass(frozen=True)
class Config:
    """Operator attributes (pages' parameter names). See include/cq.h."""
    ep_world_size: int
    moe_expert_num: int
    shared_expert_num: int = 0
    shared_expert_rank_num: int = 0
    zero_expert_num: int = 0
    copy_expert_num: int = 0
    const_expert_num: int = 0
    max_bs: int = 1
    topk: int = 1
    hidden: int = 1024
    global_bs: int = 0
    quant_mode: int = 0
    expert_token_nums_type: int = 1
    mask_ndim: int = 0
    x_dtype: int = 0       # 0 bf16, 1 fp16
    smooth_kind: int = 0   # 0 per-expert rows, 1 one row for all experts, 2 one scalar
    y_dtype: int = 0       # fp8 codes of modes 3-5: 0 e4m3fn, 1 e5m2

    @classmethod
    def from_dict(cls, d: dict) -> "Config":
        names = {f.name for f in fields(cls)}
        return cls(**{k: int(v) for k, v in d.items() if k in names})

    def as_c(self) -> _lib.CqConfig:
        return _c_config(self)

    def _q(self, name):
        c = self.as_c()
        return getattr(_lib.load(), name)(ctypes.byref(c))

    def check(self) -> int:
        return self._q("cq_check_config")

    @property
    def local_expert_num(self) -> int:
        return self._q("cq_local_expert_num")

    @property
    def num_slots(self) -> int:
        return self._q("cq_num_slots")

    @property
    def max_rows(self) -> int:
        return self._q("cq_max_rows")

    @property
    def scale_cols(self) -> int:
        return self._q("cq_scale_cols")

    @property
    def assist_info_size(self) -> int:
        return self._q("cq_assist_info_size")

    @property
    def workspace_size(self) -> int:
        return self._q("cq_workspace_size")

    @property
    def token_dtype(self) -> torch.dtype:
        return torch.float16 if self.x_dtype == 1 else torch.bfloat16

    @property
    def group_cols(self) -> int:
        return (self.hidden + 127) // 128

    def code_dtype(self) -> torch.dtype:
        return {0: self.token_dtype, 1: torch.int8, 2: torch.int8, 3: torch.uint8,
                4: torch.uint8, 5: torch.uint8}[self.quant_mode]  # fp8 codes as raw bytes


@functools.lru_cache(maxsize=256)
def _c_config(cfg: Config) -> _lib.CqConfig:
    """The C struct of a config, built once per distinct config (treat as read-only)."""
    return _lib.CqConfig(**asdict(cfg))


class DispatchResult(NamedTuple):
    expand_x: torch.Tensor          # [R_max, H] bf16 / int8 / uint8 (e4m3 bytes)
    dynamic_scales: Optional[torch.Tensor]  # f32 [R_max] or uint8 [R_max, SC]
    assist_info: torch.Tensor       # int32, opaque (pass to combine)
    ep_recv_count: torch.Tensor     # int32 [W, W*L]
    expert_token_nums: torch.Tensor  # int64 [W, L]
    expand_scales: Optional[torch.Tensor]  # f32 [R_max]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t, name, dtype, shape=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def alloc_workspace(cfg: Config, device) -> torch.Tensor:
    """A zero-filled workspace (torch allocations are 512-byte aligned)."""
    n = cfg.workspace_size
    if n == 0:
        raise _lib.CqError(_lib.CQ_ERR_ARG, "workspace size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def alloc_dispatch_outputs(cfg: Config, device, with_expand_scales: bool = True) -> DispatchResult:
    W, H, R = cfg.ep_world_size, cfg.hidden, cfg.max_rows
    L = cfg.local_expert_num
    if cfg.quant_mode == 2:
        dyn = torch.empty(R, dtype=torch.float32, device=device)
    elif cfg.quant_mode == 3:
        dyn = torch.empty(R, cfg.group_cols, dtype=torch.float32, device=device)
    elif cfg.quant_mode in (4, 5):
        dyn = torch.empty(R, cfg.scale_cols, dtype=torch.uint8, device=device)
    else:
        dyn = None
    return DispatchResult(
        torch.empty(R, H, dtype=cfg.code_dtype(), device=device), dyn,
        torch.empty(cfg.assist_info_size, dtype=torch.int32, device=device),
        torch.empty(W, W * L, dtype=torch.int32, device=device),
        torch.empty(W, L, dtype=torch.int64, device=device),
        torch.empty(R, dtype=torch.float32, device=device) if with_expand_scales else None)


def _check_outputs(cfg: Config, out: DispatchResult, dev, rows: bool = True,
                   route: bool = True) -> None:
    """The caller's output buffers must have the config's shapes and types:
    the kernels write through raw pointers and cannot check sizes. `rows`:
    the permute outputs are written; `route`: the routing outputs are."""
    W, H, R = cfg.ep_world_size, cfg.hidden, cfg.max_rows
    L = cfg.local_expert_num
    if out.assist_info is None:
        raise ValueError("assist_info is required")
    _need(out.assist_info, "assist_info", torch.int32, (cfg.assist_info_size,), dev)
    if route:
        if out.ep_recv_count is None or out.expert_token_nums is None:
            raise ValueError("ep_recv_count and expert_token_nums are required")
        _need(out.ep_recv_count, "ep_recv_count", torch.int32, (W, W * L), dev)
        _need(out.expert_token_nums, "expert_token_nums", torch.int64, (W, L), dev)
    if rows:
        if out.expand_x is None:
            raise ValueError("expand_x is required")
        _need(out.expand_x, "expand_x", cfg.code_dtype(), (R, H), dev)
        if cfg.quant_mode == 2:
            _need(out.dynamic_scales, "dynamic_scales", torch.float32, (R,), dev)
        elif cfg.quant_mode == 3:
            _need(out.dynamic_scales, "dynamic_scales", torch.float32, (R, cfg.group_cols), dev)
        elif cfg.quant_mode in (4, 5):
            _need(out.dynamic_scales, "dynamic_scales", torch.uint8, (R, cfg.scale_cols), dev)
        _need(out.expand_scales, "expand_scales", torch.float32, (R,), dev)


def _check_workspace(workspace: torch.Tensor, dev) -> None:
    _need(workspace, "workspace", torch.uint8, None, dev)


def _check_inputs(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank, expert_scales):
    W, BS, K, H = cfg.ep_world_size, cfg.max_bs, cfg.topk, cfg.hidden
    dev = expert_ids.device
    _need(expert_ids, "expert_ids", torch.int32, (W, BS, K))
    if x is not None:
        _need(x, "x", cfg.token_dtype, (W, BS, H), dev)
    if smooth_scales is not None:
        s_eff = cfg.shared_expert_num if cfg.shared_expert_rank_num > 0 else 0
        shape = {0: (s_eff + cfg.moe_expert_num, H), 1: (H,), 2: (1,)}[cfg.smooth_kind]
        _need(smooth_scales, "smooth_scales", torch.float32, shape, dev)
    if cfg.mask_ndim == 1:
        _need(x_active_mask, "x_active_mask", torch.uint8, (W, BS), dev)
    elif cfg.mask_ndim == 2:
        _need(x_active_mask, "x_active_mask", torch.uint8, (W, BS, K), dev)
    _need(bs_per_rank, "bs_per_rank", torch.int32, (W,), dev)
    _need(expert_scales, "expert_scales", torch.float32, (W, BS, K), dev)
    return dev


def dispatch(cfg: Config, x: torch.Tensor, expert_ids: torch.Tensor,
             smooth_scales: Optional[torch.Tensor] = None,
             x_active_mask: Optional[torch.Tensor] = None,
             bs_per_rank: Optional[torch.Tensor] = None,
             expert_scales: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None,
             out: Optional[DispatchResult] = None) -> DispatchResult:
    """MoE dispatch of every logical rank's tokens (cq_dispatch)."""
    dev = _check_inputs(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                        expert_scales)
    if workspace is None:
        workspace = alloc_workspace(cfg, dev)
    _check_workspace(workspace, dev)
    if out is None:
        out = alloc_dispatch_outputs(cfg, dev, expert_scales is not None)
    _check_outputs(cfg, out, dev)
    c = cfg.as_c()
    with torch.cuda.device(dev):  # the library looks up the current device
        rc = _lib.load().cq_dispatch(
            ctypes.byref(c), _ptr(x), _ptr(expert_ids), _ptr(smooth_scales), _ptr(x_active_mask),
            _ptr(bs_per_rank), _ptr(expert_scales), _ptr(out.expand_x), _ptr(out.dynamic_scales),
            _ptr(out.assist_info), _ptr(out.ep_recv_count), _ptr(out.expert_token_nums),
            _ptr(out.expand_scales), _ptr(workspace), workspace.numel(), _stream(dev))
    _lib.check(rc, "cq_dispatch")
    return out


def dispatch_noalloc(cfg: Config, x: torch.Tensor, expert_ids: torch.Tensor,
                     smooth_scales: Optional[torch.Tensor] = None,
                     x_active_mask: Optional[torch.Tensor] = None,
                     bs_per_rank: Optional[torch.Tensor] = None,
                     expert_scales: Optional[torch.Tensor] = None,
                     out: Optional[DispatchResult] = None) -> DispatchResult:
    """Dispatch through cq_dispatch_noalloc: no workspace, the library's own
    fixed scratch instead (for callers that cannot allocate device memory;
    calls must not overlap on the GPU). `out` may be preallocated."""
    dev = _check_inputs(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                        expert_scales)
    if out is None:
        out = alloc_dispatch_outputs(cfg, dev, expert_scales is not None)
    _check_outputs(cfg, out, dev)
    c = cfg.as_c()
    with torch.cuda.device(dev):  # the library looks up the current device
        rc = _lib.load().cq_dispatch_noalloc(
            ctypes.byref(c), _ptr(x), _ptr(expert_ids), _ptr(smooth_scales), _ptr(x_active_mask),
            _ptr(bs_per_rank), _ptr(expert_scales), _ptr(out.expand_x), _ptr(out.dynamic_scales),
            _ptr(out.assist_info), _ptr(out.ep_recv_count), _ptr(out.expert_token_nums),
            _ptr(out.expand_scales), _stream(dev))
    _lib.check(rc, "cq_dispatch_noalloc")
    return out


def dispatch_route(cfg: Config, expert_ids, x_active_mask=None, bs_per_rank=None, *,
                   workspace, out: DispatchResult) -> None:
    """First half of dispatch (scan, counts, prefix sums)."""
    dev = _check_inputs(cfg, None, expert_ids, None, x_active_mask, bs_per_rank, None)
    _check_workspace(workspace, dev)
    _check_outputs(cfg, out, dev, rows=False)
    c = cfg.as_c()
    with torch.cuda.device(dev):  # the library looks up the current device
        rc = _lib.load().cq_dispatch_route(
            ctypes.byref(c), _ptr(expert_ids), _ptr(x_active_mask), _ptr(bs_per_rank),
            _ptr(out.assist_info), _ptr(out.ep_recv_count), _ptr(out.expert_token_nums),
            _ptr(workspace), workspace.numel(), _stream(dev))
    _lib.check(rc, "cq_dispatch_route")


def dispatch_permute(cfg: Config, x, expert_ids, smooth_scales=None, expert_scales=None,
                     x_active_mask=None, bs_per_rank=None, *, workspace,
                     out: DispatchResult) -> None:
    """Second half of dispatch (placement and quantisation). The mask and
    per-rank BS, as given to dispatch_route, only let the kernel skip
    prefetching rows of inactive tokens."""
    dev = _check_inputs(cfg, x, expert_ids, smooth_scales, x_active_mask, bs_per_rank,
                        expert_scales)
    _check_workspace(workspace, dev)
    _check_outputs(cfg, out, dev, route=False)
    c = cfg.as_c()
    with torch.cuda.device(dev):  # the library looks up the current device
        rc = _lib.load().cq_dispatch_permute(
            ctypes.byref(c), _ptr(x), _ptr(expert_ids), _ptr(smooth_scales), _ptr(x_active_mask),
            _ptr(bs_per_rank), _ptr(expert_scales), _ptr(out.expand_x), _ptr(out.dynamic_scales),
            _ptr(out.assist_info), _ptr(out.expand_scales), _ptr(workspace), workspace.numel(),
            _stream(dev))
    _lib.check(rc, "cq_dispatch_permute")


def combine(cfg: Config, expand_x_ffn: torch.Tensor, assist_info: torch.Tensor,
            expert_scales: torch.Tensor, ep_recv_count: Optional[torch.Tensor] = None,
            ori_x: Optional[torch.Tensor] = None,
            const_alpha1: Optional[torch.Tensor] = None,
            const_alpha2: Optional[torch.Tensor] = None,
            const_v: Optional[torch.Tensor] = None,
            out_dtype: Optional[torch.dtype] = None,
            y: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """MoE combine (cq_combine): y [W, BS, H] in the token dtype (default) or
    float32. With `workspace` (the dispatch workspace of the same config) the
    call is cq_combine_ws: its status goes to that workspace (read_status)."""
    W, BS, K, H = cfg.ep_world_size, cfg.max_bs, cfg.topk, cfg.hidden
    dev = assist_info.device
    if workspace is not None:
        _check_workspace(workspace, dev)
    _need(expand_x_ffn, "expand_x_ffn", cfg.token_dtype, (cfg.max_rows, H), dev)
    _need(assist_info, "assist_info", torch.int32, (cfg.assist_info_size,), dev)
    _need(expert_scales, "expert_scales", torch.float32, (W, BS, K), dev)
    _need(ep_recv_count, "ep_recv_count", torch.int32,
          (W, W * cfg.local_expert_num), dev)
    _need(ori_x, "ori_x", cfg.token_dtype, (W, BS, H), dev)
    Q = cfg.const_expert_num
    _need(const_alpha1, "const_alpha1", torch.float32, (Q,), dev)
    _need(const_alpha2, "const_alpha2", torch.float32, (Q,), dev)
    _need(const_v, "const_v", cfg.token_dtype, (Q, H), dev)
    if out_dtype is None:
        out_dtype = cfg.token_dtype
    if out_dtype not in (cfg.token_dtype, torch.float32):
        raise ValueError("out_dtype must be the token dtype or float32")
    if y is None:
        y = torch.empty(W, BS, H, dtype=out_dtype, device=dev)
    _need(y, "y", out_dtype, (W, BS, H), dev)
    c = cfg.as_c()
    args = (ctypes.byref(c), _ptr(expand_x_ffn), _ptr(assist_info), _ptr(ep_recv_count),
            _ptr(expert_scales), _ptr(ori_x), _ptr(const_alpha1), _ptr(const_alpha2),
            _ptr(const_v), 0 if out_dtype != torch.float32 else 1, _ptr(y))
    with torch.cuda.device(dev):  # the library looks up the current device
        if workspace is None:
            rc = _lib.load().cq_combine(*args, _stream(dev))
        else:
            rc = _lib.load().cq_combine_ws(*args, _ptr(workspace), workspace.numel(), _stream(dev))
    _lib.check(rc, "cq_combine" if workspace is None else "cq_combine_ws")
    return y


def combine_ws(cfg: Config, expand_x_ffn: torch.Tensor, assist_info: torch.Tensor,
               expert_scales: torch.Tensor, workspace: torch.Tensor, **kw) -> torch.Tensor:
    """cq_combine_ws: combine whose status goes to `workspace` (read_status)."""
    return combine(cfg, expand_x_ffn, assist_info, expert_scales, workspace=workspace, **kw)


def combine_quant(cfg: Config, expand_x_ffn: torch.Tensor, assist_info: torch.Tensor,
                  codes: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None):
    """Expert-side int8 block quantisation of the FFN outputs (cq_combine_quant).
    Returns (codes int8 [R_max, H], scales f32 [R_max, H/8])."""
    R, H = cfg.max_rows, cfg.hidden
    dev = assist_info.device
    _need(expand_x_ffn, "expand_x_ffn", cfg.token_dtype, (R, H), dev)
    _need(assist_info, "assist_info", torch.int32, (cfg.assist_info_size,), dev)
    if codes is None:
        codes = torch.empty(R, H, dtype=torch.int8, device=dev)
    if scales is None:
        scales = torch.empty(R, H // 8, dtype=torch.float32, device=dev)
    _need(codes, "codes", torch.int8, (R, H), dev)
    _need(scales, "scales", torch.float32, (R, H // 8), dev)
    c = cfg.as_c()
    with torch.cuda.device(dev):  # the library looks up the current device
        rc = _lib.load().cq_combine_quant(ctypes.byref(c), _ptr(expand_x_ffn), _ptr(assist_info),
                                          _ptr(codes), _ptr(scales), _stream(dev))
    _lib.check(rc, "cq_combine_quant")
    return codes, scales


def combine_q8(cfg: Config, codes: torch.Tensor, scales: torch.Tensor, assist_info: torch.Tensor,
               expert_scales: torch.Tensor, ep_recv_count: Optional[torch.Tensor] = None,
               ori_x: Optional[torch.Tensor] = None,
               const_alpha1: Optional[torch.Tensor] = None,
               const_alpha2: Optional[torch.Tensor] = None,
               const_v: Optional[torch.Tensor] = None,
               out_dtype: Optional[torch.dtype] = None,
               y: Optional[torch.Tensor] = None) -> torch.Tensor:
    """MoE combine from int8 expert outputs (cq_combine_q8)."""
    W, BS, K, H = cfg.ep_world_size, cfg.max_bs, cfg.topk, cfg.hidden
    dev = assist_info.device
    _need(codes, "codes", torch.int8, (cfg.max_rows, H), dev)
    _need(scales, "scales", torch.float32, (cfg.max_rows, H // 8), dev)
    _need(assist_info, "assist_info", torch.int32, (cfg.assist_info_size,), dev)
    _need(expert_scales, "expert_scales", torch.float32, (W, BS, K), dev)
    _need(ep_recv_count, "ep_recv_count", torch.int32,
          (W, W * cfg.local_expert_num), dev)
    _need(ori_x, "ori_x", cfg.token_dtype, (W, BS, H), dev)
    Q = cfg.const_expert_num
    _need(const_alpha1, "const_alpha1", torch.float32, (Q,), dev)
    _need(const_alpha2, "const_alpha2", torch.float32, (Q,), dev)
    _need(const_v, "const_v", cfg.token_dtype, (Q, H), dev)
    if out_dtype is None:
        out_dtype = cfg.token_dtype
    if out_dtype not in (cfg.token_dtype, torch.float32):
        raise ValueError("out_dtype must be the token dtype or float32")
    if y is None:
        y = torch.empty(W, BS, H, dtype=out_dtype, device=dev)
    _need(y, "y", out_dtype, (W, BS, H), dev)
    c = cfg.as_c()
    with torch.cuda.device(dev):  # the library looks up the current device
        rc = _lib.load().cq_combine_q8(
            ctypes.byref(c), _ptr(codes), _ptr(scales), _ptr(assist_info), _ptr(ep_recv_count),
            _ptr(expert_scales), _ptr(ori_x), _ptr(const_alpha1), _ptr(const_alpha2), _ptr(const_v),
            0 if out_dtype != torch.float32 else 1, _ptr(y), _stream(dev))
    _lib.check(rc, "cq_combine_q8")
    return y


def read_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream, return and clear the sticky status bits."""
    st = ctypes.c_uint32(0)
    with torch.cuda.device(workspace.device):
        rc = _lib.load().cq_read_status(_ptr(workspace), ctypes.byref(st),
                                        _stream(workspace.device))
    _lib.check(rc, "cq_read_status")
    return int(st.value)


def read_combine_status(device=None) -> int:
    """Synchronise the current stream of `device`, return and clear the
    combine kernels' status bits (CQ_ST_TIMEOUT) of that device."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        rc = _lib.load().cq_read_combine_status(ctypes.byref(st), _stream(dev))
    _lib.check(rc, "cq_read_combine_status")
    return int(st.value)


def check_bounded_wait(device=None) -> tuple[int, float]:
    """Run the library's bounded wait on a barrier nothing completes
    (cq_check_bounded_wait): returns (gave_up, seconds)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    gave_up, secs = ctypes.c_uint32(0), ctypes.c_double(0.0)
    with torch.cuda.device(dev):
        rc = _lib.load().cq_check_bounded_wait(ctypes.byref(gave_up), ctypes.byref(secs),
                                               _stream(dev))
    _lib.check(rc, "cq_check_bounded_wait")
    return int(gave_up.value), float(secs.value)


def assist_views(cfg: Config, assist_info: torch.Tensor):
    """Views into assist_info: rows [R_max, 4], inv [W, BS, NS], rank_row_base [W+1]."""
    R, W, BS, NS = cfg.max_rows, cfg.ep_world_size, cfg.max_bs, cfg.num_slots
    rows = assist_info[:4 * R].view(R, 4)
    inv = assist_info[4 * R:4 * R + W * BS * NS].view(W, BS, NS)
    base = assist_info[4 * R + W * BS * NS:]
    return rows, inv, base


# The C ABI's names (include/cq.h) for the same calls.
def dispatch_workspace_size(cfg: Config) -> int:
    """Bytes of the dispatch workspace (cq_dispatch_workspace_size, the same
    as Config.workspace_size)."""
    return int(_lib.load().cq_dispatch_workspace_size(ctypes.byref(cfg.as_c())))


def dispatch_one_kernel(cfg: Config, with_smooth_scales: bool = False) -> bool:
    """Whether cq_dispatch runs this config's routing and permute as one
    kernel (cq_dispatch_one_kernel; host only)."""
    rc = _lib.load().cq_dispatch_one_kernel(ctypes.byref(cfg.as_c()), int(bool(with_smooth_scales)))
    if rc < 0:
        _lib.check(rc, "cq_dispatch_one_kernel")
    return rc == 1


cq_dispatch = moe_dispatch = dispatch
cq_dispatch_workspace_size = dispatch_workspace_size
cq_dispatch_one_kernel = dispatch_one_kernel
cq_dispatch_route = dispatch_route
cq_dispatch_permute = dispatch_permute
cq_dispatch_noalloc = dispatch_noalloc
cq_combine = moe_combine = combine
cq_combine_ws = combine_ws
cq_combine_quant = combine_quant
cq_combine_q8 = combine_q8
cq_read_status = read_status
cq_read_combine_status = read_combine_status
cq_check_bounded_wait = check_bounded_wait
