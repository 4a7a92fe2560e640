"""Host-side checks of the C ABI: the library loads, exports every symbol that
include/cq.h declares, and its host logic (argument validation, derived
sizes) behaves as specified. No call here touches a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from combine_quant_gb300 import _lib, build as cqbuild
from combine_quant_gb300.workloads import make_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cqbuild.build()
    return _lib.load()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", f)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([A-Za-z_]\w*)\s*\(",
                             txt, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert set(_lib.EXPORTS) <= declared
    for name in declared:
        assert hasattr(lib, name), f"libcq.so does not export {name}"


def test_binding_has_every_call_under_its_c_name():
    """The Python binding offers each data-path entry point of the C ABI under
    the same name (size queries are Config properties)."""
    import combine_quant_gb300 as cq
    calls = [n for n in _declared() if n.startswith(("cq_dispatch", "cq_combine", "cq_read",
                                                       "moe_"))]
    assert calls
    for name in calls:
        assert callable(getattr(cq, name, None)), f"binding lacks {name}"


def test_workspace_size_under_both_names(lib):
    """cq_dispatch_workspace_size and cq_workspace_size are one size; the
    binding's size query gives it too."""
    import combine_quant_gb300 as cq
    cfg = cq.Config(ep_world_size=32, moe_expert_num=256, max_bs=128, topk=8, hidden=7168,
                    quant_mode=2)
    assert cq.cq_dispatch_workspace_size(cfg) == cfg.workspace_size > 0


def test_dispatch_one_kernel_limits(lib):
    """cq_dispatch_one_kernel: the small-batch path's limits, on both sides of
    each (2048 pairs, 2048 block counts, 2^23 per-expert-smooth values, the
    quant modes it covers), and an invalid config's error code."""
    from combine_quant_gb300 import workloads

    def one(wl, smooth=None):
        smooth = wl.smooth is not None if smooth is None else smooth
        return lib.cq_dispatch_one_kernel(_c(wl.cfg), int(smooth))

    assert one(workloads.tiny()) == 1 and one(workloads.perf_table(8)) == 1
    assert one(workloads.perf_table(32)) == 1 and one(workloads.perf_table(64)) == 0
    assert one(workloads.dsv3(BS=2)) == 0  # (S_r + M) * W = 8192 block counts
    assert one(workloads.skew(BS=4)) == 1 and one(workloads.skew(BS=8)) == 0  # 2^23 values
    assert one(workloads.skew(BS=8), smooth=False) == 1  # the same without smooth rows
    assert one(workloads.tiny(0, 5)) == 1
    mode3 = dict(workloads.tiny().cfg, quant_mode=3)
    assert lib.cq_dispatch_one_kernel(_c(mode3), 0) == 0
    bad = dict(workloads.tiny().cfg, ep_world_size=1)
    assert lib.cq_dispatch_one_kernel(_c(bad), 0) == _lib.CQ_ERR_ARG


def _c(cfg):
    return ctypes.byref(_lib.CqConfig(**cfg))


def _random_cfg(rng):
    W = int(rng.choice([2, 3, 4, 8, 16, 32, 64, 768, 769, 1]))
    Sr = int(rng.choice([0, 0, 1, 2, W // 2, W]))
    S = int(rng.choice([0, 1, 2, 3, 5]))
    L = int(rng.choice([1, 2, 3, 8]))
    M = int(max(1, (W - Sr) * L + int(rng.choice([0, 0, 0, 1]))))
    return make_config(
        ep_world_size=W, moe_expert_num=M, shared_expert_num=S, shared_expert_rank_num=Sr,
        zero_expert_num=int(rng.choice([0, 1, -1])), copy_expert_num=int(rng.choice([0, 2])),
        const_expert_num=int(rng.choice([0, 1])), max_bs=int(rng.choice([1, 128, 512, 513, 0])),
        topk=int(rng.choice([1, 8, 16, 17])), hidden=int(rng.choice([1024, 7168, 8192, 1000, 8320])),
        global_bs=int(rng.choice([0, 0, 5])), quant_mode=int(rng.choice([0, 1, 2, 3, 4, 5, 6])),
        expert_token_nums_type=int(rng.choice([0, 1, 2])), mask_ndim=int(rng.choice([0, 1, 2, 3])),
        x_dtype=int(rng.choice([0, 1, 2])), smooth_kind=int(rng.choice([0, 1, 2, 3])),
        y_dtype=int(rng.choice([0, 0, 1, 2])))


def test_validation_agrees_with_oracle(lib, oracle_lib):
    """Two independent implementations of the pages' argument rules agree
    (the CUDA library additionally needs H % 16 == 0, and H % 32 for mode 5)."""
    rng = np.random.default_rng(0)
    n_ok = 0
    for _ in range(3000):
        cfg = _random_cfg(rng)
        want = oracle.check_config(cfg)
        got = lib.cq_check_config(_c(cfg))
        if want == 0 and (cfg["hidden"] % 16 or (cfg["quant_mode"] in (4, 5)
                                                  and cfg["hidden"] % 32)):
            want = _lib.CQ_ERR_UNSUPPORTED
        assert got == want, cfg
        n_ok += got == 0
    assert n_ok >= 5  # the sweep reaches valid configs too, not only rejections


@pytest.mark.parametrize("name", ["dsv3", "mxfp8", "special", "skew"])
def test_derived_sizes(lib, oracle_lib, name):
    from combine_quant_gb300 import workloads
    cfgs = {
        "dsv3": make_config(ep_world_size=32, moe_expert_num=256, max_bs=128, topk=8, hidden=7168,
                            quant_mode=2),
        "mxfp8": make_config(ep_world_size=64, moe_expert_num=256, max_bs=512, topk=8,
                             hidden=7168, quant_mode=5),
        "special": make_config(ep_world_size=16, moe_expert_num=112, shared_expert_num=1,
                               shared_expert_rank_num=2, zero_expert_num=1, copy_expert_num=1,
                               const_expert_num=1, max_bs=256, topk=6, hidden=4096,
                               expert_token_nums_type=0, mask_ndim=1),
        "skew": make_config(ep_world_size=16, moe_expert_num=128, max_bs=512, topk=16,
                            hidden=8192, global_bs=8192, quant_mode=2),
    }
    cfg = cfgs[name]
    assert workloads.CONFIG_FIELDS == _lib.CONFIG_FIELDS
    c = _c(cfg)
    assert lib.cq_check_config(c) == 0
    assert lib.cq_max_rows(c) == oracle.max_rows(cfg)
    assert lib.cq_num_slots(c) == oracle.num_slots(cfg)
    assert lib.cq_local_expert_num(c) == oracle.local_expert_num(cfg)
    assert lib.cq_scale_cols(c) == oracle.scale_cols(cfg)
    W, BS, NS = cfg["ep_world_size"], cfg["max_bs"], oracle.num_slots(cfg)
    assert lib.cq_assist_info_size(c) == 4 * oracle.max_rows(cfg) + W * BS * NS + W + 1
    assert lib.cq_workspace_size(c) > 0
    assert lib.cq_dispatch_workspace_size(c) == lib.cq_workspace_size(c)


def _no_gpu_visible():
    """The rejection tests below hand the library pointers into host memory;
    they run only where no GPU is visible, so that even a check that stopped
    working could not launch a kernel on them."""
    import torch
    return not torch.cuda.is_available()


needs_no_gpu = pytest.mark.skipif(not _no_gpu_visible(),
                                  reason="host-pointer rejection tests run without a GPU")


class _HostBufs:
    """Real, 256-byte aligned host buffers, one per pointer argument of
    cq_dispatch / cq_combine, each large enough for the config."""

    def __init__(self, cfg):
        W, BS, K, H = cfg["ep_world_size"], cfg["max_bs"], cfg["topk"], cfg["hidden"]
        R = oracle.max_rows(cfg)
        NS = oracle.num_slots(cfg)
        sizes = dict(x=2 * W * BS * H, ids=4 * W * BS * K, smooth=4 * (cfg["moe_expert_num"] + 4) * H,
                     mask=W * BS * K, bpr=4 * W, w=4 * W * BS * K, expand_x=2 * R * H + 16,
                     dyn=4 * R * H, assist=4 * (4 * R + W * BS * NS + W + 1), erc=4 * W * 2048,
                     etn=8 * W * 2048, es=4 * R, ws=4 << 20, ffn=2 * R * H, y=4 * W * BS * H,
                     a=64, v=2 * 16 * H)
        self._mem = {k: np.zeros(n + 256, np.uint8) for k, n in sizes.items()}

    def __getitem__(self, name):
        a = self._mem[name]
        return ctypes.c_void_p(a.ctypes.data + (-a.ctypes.data) % 256)

    def dispatch_args(self):
        return [self[k] for k in ("x", "ids", "smooth", "mask", "bpr", "w", "expand_x", "dyn",
                                  "assist", "erc", "etn", "es", "ws")]

    def combine_args(self):
        return [self[k] for k in ("ffn", "assist", "erc", "w", "x", "a", "a", "v")]


@needs_no_gpu
def test_host_errors_before_any_device_work(lib):
    """Invalid arguments are rejected on the host before anything is
    enqueued. With no GPU present, a call that got as far as a launch would
    return CQ_ERR_CUDA instead of the argument error checked here."""
    cfg = make_config(ep_world_size=4, moe_expert_num=8, max_bs=8, topk=2, hidden=1024,
                      quant_mode=2)
    hb = _HostBufs(cfg)
    args = hb.dispatch_args()
    bad = dict(cfg, topk=0)
    assert lib.cq_dispatch(_c(bad), *args, 1 << 20, None) == _lib.CQ_ERR_ARG
    assert lib.cq_dispatch(_c(dict(cfg, quant_mode=5, hidden=1040)), *args, 1 << 20, None) == \
        _lib.CQ_ERR_UNSUPPORTED  # mx blocks need H % 32 == 0 in this library
    assert lib.cq_dispatch(_c(dict(cfg, quant_mode=6)), *args, 1 << 20, None) == _lib.CQ_ERR_ARG
    a_nos = list(args)
    a_nos[2] = None  # static quantisation without scales
    assert lib.cq_dispatch(_c(dict(cfg, quant_mode=1)), *a_nos, 1 << 20, None) == _lib.CQ_ERR_ARG
    assert lib.cq_dispatch(_c(dict(cfg, x_dtype=2)), *args, 1 << 20, None) == _lib.CQ_ERR_ARG
    assert lib.cq_dispatch(_c(dict(cfg, smooth_kind=3)), *args, 1 << 20, None) == _lib.CQ_ERR_ARG
    # workspace too small
    assert lib.cq_dispatch(_c(cfg), *args, 16, None) == _lib.CQ_ERR_WORKSPACE
    # x missing
    a2 = list(args)
    a2[0] = None
    assert lib.cq_dispatch(_c(cfg), *a2, 1 << 20, None) == _lib.CQ_ERR_ARG
    # smooth scales with an mx mode
    assert lib.cq_dispatch(_c(dict(cfg, quant_mode=5)), *args, 1 << 20, None) == _lib.CQ_ERR_ARG
    # mask_ndim set without a mask
    a3 = list(args)
    a3[3] = None
    assert lib.cq_dispatch(_c(dict(cfg, mask_ndim=1)), *a3, 1 << 20, None) == _lib.CQ_ERR_ARG
    # combine: copy experts need ori_x
    cargs = hb.combine_args()
    cargs[4] = None
    assert lib.cq_combine(_c(dict(cfg, copy_expert_num=1)), *cargs, 0, hb["y"], None) == \
        _lib.CQ_ERR_ARG
    assert lib.cq_combine(_c(cfg), *hb.combine_args(), 2, hb["y"], None) == _lib.CQ_ERR_ARG
    assert lib.cq_read_status(None, None, None) == _lib.CQ_ERR_ARG
    assert lib.cq_read_combine_status(None, None) == _lib.CQ_ERR_ARG
    assert lib.cq_check_bounded_wait(None, None, None) == _lib.CQ_ERR_ARG
    assert lib.cq_workspace_init(None, 0, None) == _lib.CQ_ERR_ARG
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(lib.cq_strerror(code), bytes)


@needs_no_gpu
def test_combine_ws_checks_its_workspace(lib):
    """cq_combine_ws takes the dispatch workspace for its status word: a
    missing, misaligned or too small one is refused on the host."""
    cfg = make_config(ep_world_size=4, moe_expert_num=8, max_bs=8, topk=2, hidden=1024,
                      quant_mode=2)
    hb = _HostBufs(cfg)
    need = lib.cq_workspace_size(_c(cfg))
    args = hb.combine_args()
    y = hb["y"]
    assert lib.cq_combine_ws(_c(cfg), *args, 0, y, None, need, None) == _lib.CQ_ERR_WORKSPACE
    assert lib.cq_combine_ws(_c(cfg), *args, 0, y, hb["ws"], need - 1, None) == \
        _lib.CQ_ERR_WORKSPACE
    misaligned = ctypes.c_void_p(hb["ws"].value + 16)
    assert lib.cq_combine_ws(_c(cfg), *args, 0, y, misaligned, need, None) == \
        _lib.CQ_ERR_WORKSPACE
    # argument rules of cq_combine come first
    assert lib.cq_combine_ws(_c(dict(cfg, topk=0)), *args, 0, y, hb["ws"], need, None) == \
        _lib.CQ_ERR_ARG
    assert lib.cq_combine_ws(_c(cfg), *args, 2, y, hb["ws"], need, None) == _lib.CQ_ERR_ARG


@needs_no_gpu
@pytest.mark.parametrize("which", ["x", "expand_x", "assist", "dyn", "smooth"])
def test_permute_half_errors_before_the_route_half(lib, which):
    """An argument only the permute half uses (a misaligned token row, code
    row, assist_info, scale row or smooth table) is rejected before the route
    half is enqueued: the call returns CQ_ERR_ARG, not the CQ_ERR_CUDA that a
    route launch attempted without a GPU would give."""
    cfg = make_config(ep_world_size=4, moe_expert_num=8, max_bs=8, topk=2, hidden=1024,
                      quant_mode=2)
    hb = _HostBufs(cfg)
    args = hb.dispatch_args()
    pos = {"x": 0, "smooth": 2, "expand_x": 6, "dyn": 7, "assist": 8}[which]
    args[pos] = ctypes.c_void_p(args[pos].value + (2 if which == "dyn" else 1))
    assert lib.cq_dispatch(_c(cfg), *args, 4 << 20, None) == _lib.CQ_ERR_ARG
    assert lib.cq_dispatch_noalloc(_c(cfg), *args[:12], None) in (_lib.CQ_ERR_ARG,
                                                                  _lib.CQ_ERR_CUDA)


def test_python_config_roundtrip(lib):
    from combine_quant_gb300 import Config
    cfg = make_config(ep_world_size=16, moe_expert_num=112, shared_expert_num=1,
                      shared_expert_rank_num=2, max_bs=256, topk=6, hidden=4096)
    c = Config.from_dict(cfg)
    assert c.check() == 0
    assert c.local_expert_num == 8 and c.num_slots == 7
    assert c.max_rows == 16 * 256 * 7
