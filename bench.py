#!/usr/bin/env python
"""Benchmark of the MoE dispatch + combine hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cq|reference]

A step is one pass of the whole path over one batch: cq_dispatch (the routing
scan and the fused permute-quantise) and cq_combine, on the DeepSeek-V3-shaped
workload (32 logical EP ranks,
256 experts, 8 per rank, top-8, 128 tokens per rank, hidden 7168, per-token
dynamic int8). The expert FFN between dispatch and combine is outside the path;
combine consumes a seeded stand-in for its output.

Prints one JSON line: tokens/s over the K timed steps (device-resident inputs,
L2 flushed between steps, CUDA events on the launching stream), an end-to-end
figure through cq_dispatch / cq_combine with host buffers, the roofline of the
dominant kernel, the oracle timed on the host cores, and the SM clocks seen
during the timed region. Under torchrun (N > 1) every rank runs an independent
replica on its own GPU (no collective on the data path); the reported value is
all ranks' tokens over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import inspect
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes per launch read from an ncu capture of the named kernel, keyed by
# the SHA-256 of the code of the kernel's source files (comments left out)
# when it was captured; reported only while that code is unchanged.
NCU_TRAFFIC = {
    # profiles/dsv3_step_launch_list.md: read 470.060837 MB + write 46.038894 MB
    # per launch (mean of 7 launches of one bench run)
    "combine": {"bytes_per_launch": 516099730,
                "src_sha": "7a967fd1247cf99f86c23516ef884b53b65d3966a64784ddc2b693b602628d87"},
    # the same capture: read 59.256503 MB + write 172.054382 MB
    "permute": {"bytes_per_launch": 231310885,
                "src_sha": "3c5fdb061f4710990c312e87909514cdcdc753afa41dec103d302908e9c86e6e"},
}


def _positive_int(text: str) -> int:
    v = int(text)
    if v < 1:
        raise argparse.ArgumentTypeError(f"must be >= 1, got {v}")
    return v


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["cq", "reference"], default="cq")
    ap.add_argument("--workload", default="dsv3")
    ap.add_argument("--bs", type=_positive_int, default=None,
                    help="override the per-rank batch of dsv3, mxfp8, special or skew (a "
                         "reduced case, e.g. for a profiler capture)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-all-cores", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the oracle on every host core (spawned processes)")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--quant-mode", type=int, default=None,
                    help="override the workload's quant_mode (0-5)")
    ap.add_argument("--combine", choices=["bf16", "int8"], default="bf16",
                    help="combine from bf16 expert outputs, or from int8 ones quantised on the "
                         "expert side (the quantiser is timed separately, outside the step)")
    ap.add_argument("--flush", choices=["write+read", "write", "none"], default="write+read",
                    help="L2 flush between steps (outside the timed events)")
    ap.add_argument("--e2e-sets", type=_positive_int, default=2,
                    help="input/output buffer sets of the end-to-end leg (pipeline depth, >= 1)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch each call directly instead of replaying CUDA graphs")
    ap.add_argument("--per-workload", action=argparse.BooleanOptionalAction, default=True,
                    help="with the default workload, also time the other workloads (a few "
                         "steps each) and report them under per_workload")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="host time budget of the oracle baseline")
    return ap.parse_args(argv)


def named_workload(name: str, bs=None, quant_mode=None):
    """The named workload, with the per-rank batch and quant mode overrides."""
    from combine_quant_gb300 import workloads

    gen = workloads.WORKLOADS[name]
    if bs is not None:
        if "BS" not in inspect.signature(gen).parameters:
            raise SystemExit(f"--bs: workload {name} has a fixed batch")
        wl = gen(BS=bs)
    else:
        wl = gen()
    if quant_mode is not None:
        wl = wl.with_mode(quant_mode)
    return wl


def make_workload(args):
    return named_workload(args.workload, args.bs, args.quant_mode)


def workload_desc(wl) -> str:
    c = wl.cfg
    L = c["moe_expert_num"] // (c["ep_world_size"] - c["shared_expert_rank_num"])
    return (f"{wl.name}: W={c['ep_world_size']} logical EP ranks, M={c['moe_expert_num']} "
            f"experts (L={L}/rank), K={c['topk']}, BS={c['max_bs']}/rank, H={c['hidden']}, "
            f"quant_mode={c['quant_mode']}")


# ---------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region.
    The region starts `lead_s` seconds before the timed steps, with the GPU
    running the same step meanwhile (Bench.load_for): nvidia-smi's first
    sample comes only after its start-up, and the timed steps may last a few
    milliseconds."""
    lead_s = 0.5
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.gpu = gpu_index
        self.enabled = enabled
        self.proc = None
        self.path = None

    def start(self):
        if not self.enabled:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons),
                "window": f"the timed steps and the {self.lead_s:g} s of the same step "
                          "just before them"}


# -------------------------------------------------------- byte accounting ----

def algorithmic_bytes(cfg, rows: int, tokens_active: int, with_scales: bool,
                      combine_int8: bool = False, smooth_bytes: int = 0,
                      special_tokens: int = 0) -> dict:
    """Bytes each kernel must move per launch (reads + writes of HBM), given
    the routed row count P, the active token count, the size of the smooth
    scales the call reads (once) and the number of tokens with a copy or
    const slot (their ori_x row is read once; const_v rows once in all)."""
    W, BS, K, H = cfg.ep_world_size, cfg.max_bs, cfg.topk, cfg.hidden
    NS, L = cfg.num_slots, cfg.local_expert_num
    G = cfg.shared_expert_rank_num + cfg.moe_expert_num
    T = W * BS
    mode = cfg.quant_mode
    b_code = 2 if mode == 0 else 1
    b_scale = {0: 0, 1: 0, 2: 4, 3: 4 * cfg.group_cols, 4: cfg.scale_cols, 5: cfg.scale_cols}[mode]
    route = 4 * T * K + 4 * T * NS + 3 * 4 * G * W + 4 * W * W * L + 8 * W * L
    permute = (2 * H * tokens_active            # x, read once per active token
               + rows * (H * b_code + b_scale + 16)  # codes, scale, (src, token, slot) record
               + 4 * T * NS * 2 + 4 * T * K     # eidx read, inv write, ids read
               + (8 * rows if with_scales else 0)  # routing weight read + carried copy
               + smooth_bytes)
    ffn_row = (H + 4 * (H // 8)) if combine_int8 else 2 * H  # int8 codes + block scales
    combine = (ffn_row * rows + 2 * H * T + 4 * T * NS + 4 * T * K
               + 2 * H * (special_tokens + cfg.const_expert_num))  # ori_x rows, const_v
    out = {"route": route, "permute": permute, "combine": combine}
    if combine_int8:
        out["combine_quant"] = rows * (2 * H + H + 4 * (H // 8))  # bf16 in, codes + scales out
    return out


def kernels_per_step(cfg, smooth_given: bool) -> int:
    """libcq kernels one step launches: cq_dispatch (one kernel for a small
    batch, as the library reports through cq_dispatch_one_kernel; else
    routing (count, offsets) and the permute: index + smooth-rows kernels for
    per-expert smooth scales in modes 1-3, else one kernel) and the combine."""
    import combine_quant_gb300 as cq

    if cq.dispatch_one_kernel(cfg, smooth_given):
        return 2
    per_expert_smooth = smooth_given and cfg.smooth_kind == 0 and cfg.quant_mode in (1, 2, 3)
    return 2 + (2 if per_expert_smooth else 1) + 1


def special_token_count(wl) -> int:
    """Active tokens with at least one active copy or const slot."""
    c = wl.cfg
    lo = c["moe_expert_num"] + c["zero_expert_num"]
    hi = lo + c["copy_expert_num"] + c["const_expert_num"]
    if hi == lo:
        return 0
    W, BS, K = c["ep_world_size"], c["max_bs"], c["topk"]
    ids = wl.expert_ids.reshape(W, BS, K)
    on = np.ones((W, BS, K), bool)
    if wl.bs_per_rank is not None:
        on &= (np.arange(BS)[None, :] < wl.bs_per_rank[:, None])[:, :, None]
    if wl.mask is not None:
        m = wl.mask.reshape(W, BS, -1).astype(bool)
        on &= m if m.shape[2] == K else m[:, :, :1]
    return int((((ids >= lo) & (ids < hi)) & on).any(axis=2).sum())


def measured_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


KERNEL_SOURCES = {
    "permute": ["cq_permute_impl.cuh", "cq_permute_bf16.cu", "cq_internal.cuh", "cq_async.cuh"],
    "combine": ["cq_combine.cu", "cq_internal.cuh", "cq_async.cuh"],
}


def _code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed (the
    kernel sources hold no string literal with a comment marker in it)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_sha(kernel: str) -> str:
    """SHA-256 over the code (comments left out) of the source files that
    define the kernel."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "combine_quant_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def ncu_traffic(kernel: str):
    rec = NCU_TRAFFIC.get(kernel)
    if not rec or rec.get("src_sha") != source_sha(kernel):
        return None
    return rec["bytes_per_launch"]


# ------------------------------------------------------- oracle baseline ----

def _oracle_prepare(wl):
    """The whole-batch routing scan (timed) and the inputs of the per-token
    work: (route, inv remapped into a small expert-output pool, pool, t_route)."""
    import oracle
    from combine_quant_gb300 import workloads

    oracle.build()
    pool = workloads.ffn_standin(wl.seed, 1024, wl.cfg["hidden"])
    t0 = time.perf_counter()
    route = oracle.route(wl.cfg, wl.expert_ids, wl.mask, wl.bs_per_rank)
    t_route = time.perf_counter() - t0
    inv_pool = np.where(route.inv >= 0, route.inv.astype(np.int64) % pool.shape[0],
                        route.inv).astype(np.int32)
    return route, inv_pool, pool, t_route


def _smooth_of(wl, r, i, k):
    """(row, scalar) smooth arguments of the oracle's quantisation for slot k
    of token (r, i): the expert's row (shared experts first), the one shared
    row, or the scalar, as smooth_kind says; none outside modes 1-3."""
    cfg = wl.cfg
    if wl.smooth is None or cfg["quant_mode"] not in (1, 2, 3):
        return None, None
    kind = cfg.get("smooth_kind", 0)
    if kind == 2:
        return None, float(wl.smooth.reshape(-1)[0])
    if kind == 1:
        return wl.smooth.reshape(-1), None
    K = cfg["topk"]
    s_eff = cfg["shared_expert_num"] if cfg["shared_expert_rank_num"] > 0 else 0
    return (wl.smooth[s_eff + wl.expert_ids[r, i, k]] if k < K else wl.smooth[k - K]), None


def _oracle_tokens(wl, prep, order, budget_s: float):
    """Quantise every dispatched row of each token in `order` and combine the
    token, until the budget is spent. Returns (tokens done, seconds)."""
    import oracle

    route, inv_pool, pool, _ = prep
    cfg = wl.cfg
    K, mode = cfg["topk"], cfg["quant_mode"]
    done = 0
    t0 = time.perf_counter()
    for r, i in order:
        for k in range(route.inv.shape[2]):
            row = route.inv[r, i, k]
            if row >= 0:
                sm_row, sm_scalar = _smooth_of(wl, r, i, k)
                oracle.quant_row(mode, wl.x[r, i], sm_row, cfg.get("x_dtype", 0), sm_scalar,
                                 cfg.get("y_dtype", 0))
        oracle.combine_tokens(cfg, [(r, i)], pool, inv_pool, wl.expert_scales, wl.x,
                              wl.const_alpha1, wl.const_alpha2, wl.const_v)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def oracle_sample(wl, budget_s: float, max_tokens: int | None = None):
    """Time the oracle (single-threaded C, as it stands) on a bounded sample of
    the workload: the full routing scan, then quantisation of the rows of the
    first n tokens and the combine of those n tokens, n growing until the
    budget is spent. Returns (tokens/s, description, cores)."""
    cfg = wl.cfg
    W, BS = cfg["ep_world_size"], cfg["max_bs"]
    prep = _oracle_prepare(wl)
    order = [(r, i) for r in range(W) for i in range(BS)]
    if max_tokens:
        order = order[:max_tokens]
    done, t_tok = _oracle_tokens(wl, prep, order, budget_s)
    t_route = prep[3]
    # The routing scan is a whole-batch pass; charge it pro rata.
    per_tok = t_tok / done + t_route / (W * BS)
    desc = (f"oracle route over all {W * BS} tokens ({t_route:.3f} s) + quantise-and-combine of "
            f"the first {done} tokens in rank-major order ({t_tok:.2f} s); value = tokens / "
            f"(per-token time + route time pro rata)")
    return 1.0 / per_tok, desc, 1


def _oracle_worker(name, bs, quant_mode, wi, n, budget_s, ready, start, results):
    """One process of the all-cores oracle baseline: tokens wi, wi + n, ..."""
    sys.path.insert(0, ROOT)
    wl = named_workload(name, bs, quant_mode)
    prep = _oracle_prepare(wl)
    W, BS = wl.cfg["ep_world_size"], wl.cfg["max_bs"]
    order = [(r, i) for r in range(W) for i in range(BS)][wi::n]
    ready.put(wi)
    start.wait()
    done, secs = _oracle_tokens(wl, prep, order, budget_s)
    results.put((done, secs, prep[3]))


def oracle_all_cores(name: str, quant_mode, budget_s: float, n: int | None = None, bs=None):
    """The same oracle work on every host core: n spawned processes (started
    only after all have built their inputs) take interleaved tokens. Returns
    (tokens/s, cores): all tokens done over the slowest process's time, plus
    the single-threaded routing scan pro rata."""
    import multiprocessing as mp

    n = n or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    ready, results, start = ctx.Queue(), ctx.Queue(), ctx.Event()
    procs = [ctx.Process(target=_oracle_worker,
                         args=(name, bs, quant_mode, wi, n, budget_s, ready, start, results))
             for wi in range(n)]
    for p in procs:
        p.start()
    for _ in range(n):
        ready.get(timeout=600)
    start.set()
    out = [results.get(timeout=600 + 4 * budget_s) for _ in range(n)]
    for p in procs:
        p.join(timeout=60)
    done = sum(o[0] for o in out)
    secs = max(o[1] for o in out)
    t_route = out[0][2]
    c = named_workload(name, bs).cfg
    per_tok = secs / done + t_route / (c["ep_world_size"] * c["max_bs"])
    return 1.0 / per_tok, n


# ------------------------------------------------------------- distributed ----

def job_throughput(local_ms: float, units_per_rank: int, steps: int, dist=None, device=None):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (a max over ranks). Returns (units/s, slowest ms)."""
    slowest, world = float(local_ms), 1
    if dist is not None and dist.is_initialized():
        import torch

        t = torch.tensor([slowest], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        slowest, world = float(t.item()), dist.get_world_size()
    return world * units_per_rank * steps / (slowest / 1e3), slowest


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def emit(obj):
    print(json.dumps(obj), flush=True)


# ----------------------------------------------------------- reference arm ----

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0  # the oracle arm runs once, on rank 0
    from combine_quant_gb300 import workloads

    wl = make_workload(args)
    W, BS = wl.cfg["ep_world_size"], wl.cfg["max_bs"]
    # Each step is a bounded sample: enough tokens that K + W steps take about
    # a minute of host time in total.
    _, _, _ = oracle_sample(wl, 0.5, max_tokens=4)  # warm the library and caches
    rate0, _, _ = oracle_sample(wl, 2.0)
    per_step_tokens = max(1, min(W * BS, int(rate0 * 60.0 / max(1, args.steps + args.warmup))))
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        rate, desc, cores = oracle_sample(wl, 1e9, max_tokens=per_step_tokens)
        if s >= args.warmup:
            times.append(per_step_tokens / rate)
    total = sum(times)
    value = per_step_tokens * len(times) / total
    emit({"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
          "steps": args.steps, "warmup": args.warmup,
          "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
          "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
          "config": {"workload": workload_desc(wl), "tokens_per_step": per_step_tokens},
          "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                           "sample": f"each step: {desc}"},
          "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})
    return 0


# ------------------------------------------------------------------ cq arm ----

class Bench:
    """Device inputs, outputs and the step of one workload: route, permute and
    combine through the binding, captured into CUDA graphs (the whole step,
    and each kernel alone for the breakdown) unless --no-graph."""

    def __init__(self, args, dev, wl, flush):
        import torch

        import combine_quant_gb300 as cq
        from combine_quant_gb300 import workloads

        self.args, self.dev, self.wl, self.flush = args, dev, wl, flush
        cfg = self.cfg = cq.Config.from_dict(wl.cfg)
        tdev = lambda a, dt: None if a is None else torch.from_numpy(  # noqa: E731
            np.ascontiguousarray(a)).to(dev).view(dt)
        self.x = tdev(wl.x, torch.bfloat16)
        self.ids = tdev(wl.expert_ids, torch.int32)
        self.w = tdev(wl.expert_scales, torch.float32)
        self.sm = tdev(wl.smooth, torch.float32) if cfg.quant_mode in (1, 2, 3) else None
        self.mask = tdev(wl.mask, torch.uint8)
        self.bpr = tdev(wl.bs_per_rank, torch.int32)
        self.ws = cq.alloc_workspace(cfg, dev)
        self.out = cq.alloc_dispatch_outputs(cfg, dev)
        pool = tdev(workloads.ffn_standin(wl.seed, 4096, cfg.hidden), torch.bfloat16)
        ridx = (torch.arange(cfg.max_rows, device=dev, dtype=torch.int64) * 7919) % 4096
        self.ffn = pool.index_select(0, ridx).contiguous()
        self.y = torch.empty(cfg.ep_world_size, cfg.max_bs, cfg.hidden, dtype=torch.bfloat16,
                             device=dev)
        self.ffn_q = self.ffn_s = None
        if args.combine == "int8":
            # The expert side's int8 outputs, made once before timing (a producer
            # would emit them from its own epilogue); the quantiser is timed apart.
            self.dispatch()
            self.ffn_q, self.ffn_s = cq.combine_quant(cfg, self.ffn, self.out.assist_info)
        self.consts = dict(const_alpha1=tdev(wl.const_alpha1, torch.float32),
                           const_alpha2=tdev(wl.const_alpha2, torch.float32),
                           const_v=tdev(wl.const_v, torch.bfloat16))
        self.stream = torch.cuda.current_stream(dev)
        self.use_graph = not args.no_graph
        self.parts = [self.route, self.permute, lambda: self.combine()]
        self.run_dispatch = self.dispatch
        self.run_step = self.step
        if self.use_graph:
            side = torch.cuda.Stream(dev)
            side.wait_stream(self.stream)
            graphs = {}
            with torch.cuda.stream(side):
                for name, fn in (("step", self.step), ("route", self.route),
                                 ("permute", self.permute), ("combine", lambda: self.combine()),
                                 ("dispatch", self.dispatch)):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=side):
                        fn()
                    graphs[name] = g
            self.stream.wait_stream(side)
            torch.cuda.synchronize()
            self.graphs = graphs
            self.run_step = graphs["step"].replay
            self.run_dispatch = graphs["dispatch"].replay
            self.parts = [graphs["route"].replay, graphs["permute"].replay,
                          graphs["combine"].replay]

    def route(self):
        import combine_quant_gb300 as cq
        cq.dispatch_route(self.cfg, self.ids, self.mask, self.bpr, workspace=self.ws,
                          out=self.out)

    def permute(self):
        import combine_quant_gb300 as cq
        cq.dispatch_permute(self.cfg, self.x, self.ids, self.sm, self.w, self.mask, self.bpr,
                            workspace=self.ws, out=self.out)

    def dispatch(self, x=None, ids=None, w=None):
        import combine_quant_gb300 as cq
        return cq.dispatch(self.cfg, self.x if x is None else x, self.ids if ids is None else ids,
                           smooth_scales=self.sm, x_active_mask=self.mask, bs_per_rank=self.bpr,
                           expert_scales=self.w if w is None else w, workspace=self.ws,
                           out=self.out)

    def combine(self, assist_info=None, erc=None, w=None, x=None, y=None):
        import combine_quant_gb300 as cq
        o = self.out
        a = (o.assist_info if assist_info is None else assist_info,
             o.ep_recv_count if erc is None else erc)
        w = self.w if w is None else w
        x = self.x if x is None else x
        y = self.y if y is None else y
        if self.args.combine == "int8":
            return cq.combine_q8(self.cfg, self.ffn_q, self.ffn_s, a[0], w, a[1], ori_x=x, y=y,
                                 **self.consts)
        return cq.combine(self.cfg, self.ffn, a[0], w, a[1], ori_x=x, y=y, **self.consts)

    def step(self):
        """One pass of the path: cq_dispatch, then cq_combine. (The breakdown
        times the two dispatch halves, cq_dispatch_route and
        cq_dispatch_permute, apart; a small batch's cq_dispatch runs both in
        one kernel.)"""
        self.dispatch()
        self.combine()

    def warm(self, n):
        import torch
        for _ in range(n):
            self.flush.zero_()
            self.step()
        torch.cuda.synchronize()

    def breakdown(self, n, barrier):
        """Per-kernel times (ms lists) from n steps with events between kernels."""
        import torch
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        barrier()
        for k in range(n):
            self.flush.zero_()
            for j, part in enumerate(self.parts):
                evb[k][j].record(self.stream)
                part()
            evb[k][3].record(self.stream)
        barrier()
        return ([e[0].elapsed_time(e[1]) for e in evb], [e[1].elapsed_time(e[2]) for e in evb],
                [e[2].elapsed_time(e[3]) for e in evb])

    def dispatch_alone(self, n, barrier):
        """cq_dispatch alone, L2 flushed before each call: times (ms)."""
        import torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        barrier()
        for k in range(n):
            self.flush.zero_()
            ev[k][0].record(self.stream)
            self.run_dispatch()
            ev[k][1].record(self.stream)
        barrier()
        return [e[0].elapsed_time(e[1]) for e in ev]

    def load_for(self, seconds):
        """The step (L2 flushed between steps, as in the timed loop) repeated
        for about `seconds`, untimed."""
        import torch
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(20):
                self.flush.zero_()
                self.run_step()
            torch.cuda.synchronize()

    def timed(self, n, barrier, clocks=None):
        """n steps, L2 flushed between them outside the events: step times (ms)."""
        import torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        if clocks and clocks.enabled:
            clocks.start()
            self.load_for(clocks.lead_s)
        barrier()
        t_wall = time.perf_counter()
        for k in range(n):
            self.flush.zero_()
            ev[k][0].record(self.stream)
            self.run_step()
            ev[k][1].record(self.stream)
        barrier()
        self.t_wall = time.perf_counter() - t_wall
        return [e[0].elapsed_time(e[1]) for e in ev]

    def counts(self):
        """(dispatched rows, active tokens, smooth bytes, tokens with special slots)."""
        import combine_quant_gb300 as cq
        cfg, wl = self.cfg, self.wl
        rows = int(cq.assist_views(cfg, self.out.assist_info)[2][-1].item())
        tokens = wl.tokens
        if wl.mask is not None:
            tokens = int((wl.mask.reshape(cfg.ep_world_size, cfg.max_bs, -1).max(axis=2)
                          > 0).sum())
        smooth_bytes = int(self.sm.numel() * 4) if self.sm is not None else 0
        return rows, tokens, smooth_bytes, special_token_count(wl)


# Workloads whose figures the default run adds beside the headline (key
# "per_workload"): the other four configurations and the two shapes of the
# performance table ("CANN MoE Dispatch/Combine 通信算子性能优化实践", 性能数据).
SIDE_WORKLOADS = ("tiny", "mxfp8", "special", "skew", "perf8", "perf256")


def side_figures(args, dev, flush, barrier, peak):
    """Step and per-kernel times of the side workloads, measured as the
    headline is (graph replay, L2 flushed between steps, CUDA events), with
    fewer steps."""
    import torch

    import combine_quant_gb300 as cq
    from combine_quant_gb300 import workloads

    steps = max(10, min(args.steps, 50))
    res = {}
    for name in SIDE_WORKLOADS:
        wl = workloads.WORKLOADS[name]()
        b = Bench(args, dev, wl, flush)
        b.warm(3)
        if cq.read_status(b.ws) != 0:
            raise RuntimeError(f"device status reported a bad id or mask on {name}")
        t_route, t_perm, t_comb = b.breakdown(steps, barrier)
        t_step = b.timed(steps, barrier)
        rows, tokens, smooth_bytes, special = b.counts()
        ab = algorithmic_bytes(b.cfg, rows, tokens, with_scales=True, smooth_bytes=smooth_bytes,
                               special_tokens=special)
        us = {"route": 1e3 * statistics.mean(t_route), "permute": 1e3 * statistics.mean(t_perm),
              "combine": 1e3 * statistics.mean(t_comb)}
        step_us = 1e3 * statistics.mean(t_step)
        res[name] = {
            "workload": workload_desc(wl), "tokens_per_step": tokens, "rows_per_step": rows,
            "steps": steps, "step_us": step_us, "tokens_per_s": tokens / (step_us * 1e-6),
            "kernels": {k: {"us": us[k], "alg_bytes": ab[k],
                            "frac": ab[k] / (us[k] * 1e-6) / 1e9 / peak} for k in us}}
        if kernels_per_step(b.cfg, b.sm is not None) == 2:
            # The step's cq_dispatch is one kernel (routing and permute
            # together); the route and permute figures above time the two
            # dispatch halves, which that kernel replaces.
            t_one = b.dispatch_alone(steps, barrier)
            res[name]["dispatch_one_kernel"] = {
                "us": 1e3 * statistics.mean(t_one),
                "alg_bytes": ab["route"] + ab["permute"],
                "note": "cq_dispatch as the step runs it (dispatch_small_kernel); route and "
                        "permute above are the two dispatch halves"}
        if name == "tiny":
            # latency-bound: the same step with L2 left warm between steps
            saved = flush.mode
            flush.mode = "none"
            t_hot = b.timed(steps, barrier)
            flush.mode = saved
            res[name]["step_us_hot_l2"] = 1e3 * statistics.mean(t_hot)
        del b
        torch.cuda.empty_cache()
    return res


def cpu_model() -> str:
    """The host CPU's model name from /proc/cpuinfo (or what is known)."""
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model Name", "cpu model", "Hardware"):
        for line in txt.splitlines():
            if line.split(":")[0].strip() == key and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in txt.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            parts.setdefault(k.strip(), v.strip())
    if "CPU implementer" in parts:
        # Arm cores name no model in /proc/cpuinfo; the part numbers of a few
        # server cores (implementer 0x41 is Arm Ltd.)
        arm_parts = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2",
                     "0xd4f": "Neoverse-V2", "0xd84": "Neoverse-V3", "0xd8e": "Neoverse-N3"}
        name = arm_parts.get(parts.get("CPU part", "")) if parts.get("CPU implementer") == "0x41" \
            else None
        return ((f"Arm {name}, " if name else "")
                + f"CPU implementer {parts.get('CPU implementer')}, part {parts.get('CPU part')}, "
                f"variant {parts.get('CPU variant')}, revision {parts.get('CPU revision')}")
    return "unknown"


def run_cq(args):
    import torch

    import combine_quant_gb300 as cq
    from combine_quant_gb300 import workloads

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    class _Flush:
        """Between steps: write a buffer larger than L2, then (unless
        --flush write) read another one, so that the next step starts with
        no input resident in L2 and no dirty lines left to write back."""
        mode = args.flush

        def zero_(self):
            if self.mode == "none":  # hot-L2 figures only: not a contract number
                return
            flush_w.zero_()
            if self.mode == "write+read":
                flush_r.amax()

    flush = _Flush()
    wl = make_workload(args)
    b = Bench(args, dev, wl, flush)
    cfg, stream = b.cfg, b.stream
    b.warm(args.warmup)
    if cq.read_status(b.ws) != 0:
        raise RuntimeError("device status reported a bad id or mask on the bench workload")
    rows, tokens, smooth_bytes, special_tokens = b.counts()

    # Per-kernel breakdown: events between the kernels.
    n_bd = max(3, min(args.steps, 500))
    t_route, t_perm, t_comb = b.breakdown(n_bd, barrier)

    # The timed region: K steps, events only at step boundaries.
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    t_step = b.timed(args.steps, barrier, clocks)
    t_wall = b.t_wall
    clk = clocks.stop()
    value, total_ms = job_throughput(sum(t_step), tokens, args.steps, dist, dev)
    ms_per_step = total_ms / args.steps

    # End to end through cq_dispatch / cq_combine with host buffers: each step
    # copies x, expert_ids and expert_scales from pinned memory and reads y back.
    e2e = None
    if not args.no_e2e:
        hx = torch.from_numpy(np.ascontiguousarray(wl.x)).view(torch.bfloat16).pin_memory()
        hids = torch.from_numpy(np.ascontiguousarray(wl.expert_ids)).pin_memory()
        hw = torch.from_numpy(np.ascontiguousarray(wl.expert_scales)).pin_memory()
        n_e2e = max(10, min(args.steps, 500))
        # args.e2e_sets buffer sets: step k uploads into set k % n on the upload stream,
        # computes on the main stream, downloads y on the download stream; the
        # events keep each set's reuse ordered, so copies of neighbouring
        # steps overlap the compute of this one.
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        sets = [dict(x=torch.empty_like(b.x), ids=torch.empty_like(b.ids),
                     w=torch.empty_like(b.w), y=torch.empty_like(b.y),
                     hy=torch.empty(b.y.shape, dtype=torch.bfloat16).pin_memory(),
                     up=torch.cuda.Event(), done=torch.cuda.Event(), down=torch.cuda.Event())
                for _ in range(args.e2e_sets)]
        for s in sets:
            s["done"].record(stream)
            s["down"].record(stream)

        def e2e_step(k):
            s = sets[k % len(sets)]
            with torch.cuda.stream(s_up):
                s_up.wait_event(s["done"])  # the set's inputs are free once its last compute ended
                s["x"].copy_(hx, non_blocking=True)
                s["ids"].copy_(hids, non_blocking=True)
                s["w"].copy_(hw, non_blocking=True)
                s["up"].record(s_up)
            stream.wait_event(s["up"])
            stream.wait_event(s["down"])  # y of this set has been read back
            o = b.dispatch(s["x"], s["ids"], s["w"])
            b.combine(o.assist_info, o.ep_recv_count, s["w"], s["x"], s["y"])
            s["done"].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(s["done"])
                s["hy"].copy_(s["y"], non_blocking=True)
                s["down"].record(s_down)

        for k in range(3):
            e2e_step(k)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(s_up)
        for k in range(n_e2e):
            e2e_step(k)
        s_down.wait_event(sets[(n_e2e - 1) % len(sets)]["down"])
        e1.record(s_down)
        barrier()
        e_value, _ = job_throughput(e0.elapsed_time(e1), tokens, n_e2e, dist, dev)
        e2e = {"value": e_value, "unit": UNIT,
               "h2d_bytes_per_step": hx.nbytes + hids.nbytes + hw.nbytes,
               "d2h_bytes_per_step": sets[0]["hy"].nbytes, "steps": n_e2e,
               "api": "cq_dispatch + cq_combine (libcq C ABI via ctypes)",
               "pipelining": f"{len(sets)} buffer sets; upload, compute and download on "
                             "three streams, so neighbouring steps' copies overlap"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    ab = algorithmic_bytes(cfg, rows, tokens, with_scales=True, smooth_bytes=smooth_bytes,
                           special_tokens=special_tokens,
                           combine_int8=args.combine == "int8")
    means = {"route": statistics.mean(t_route), "permute": statistics.mean(t_perm),
             "combine": statistics.mean(t_comb)}
    if args.combine == "int8":
        # the expert-side quantiser, timed alone (not part of the step)
        eq0, eq1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_q = max(3, min(args.steps, 200))
        t_q = []
        for _ in range(n_q):
            flush.zero_()
            eq0.record(stream)
            cq.combine_quant(cfg, b.ffn, b.out.assist_info, b.ffn_q, b.ffn_s)
            eq1.record(stream)
            torch.cuda.synchronize()
            t_q.append(eq0.elapsed_time(eq1))
        means["combine_quant"] = statistics.mean(t_q)
    peak, peak_kind = measured_peaks()
    kernels = {k: {"us": 1e3 * means[k], "alg_bytes": ab[k],
                   "gbs": ab[k] / (means[k] * 1e-3) / 1e9,
                   "frac": ab[k] / (means[k] * 1e-3) / 1e9 / peak} for k in means}
    dom = max(("permute", "combine"), key=lambda k: means[k])
    traffic = None
    if args.workload == "dsv3" and args.bs is None and args.quant_mode in (None, 2) \
            and args.combine == "bf16":
        traffic = ncu_traffic(dom)  # the captured configuration
    roof = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak,
            "unit": "GB/s", "frac": kernels[dom]["frac"], "traffic": traffic,
            "peak_source": f"hbm_gbs of {peak_kind}"}

    side = None
    if world == 1 and args.per_workload and args.workload == "dsv3" and args.bs is None \
            and args.quant_mode is None and args.combine == "bf16":
        del b
        torch.cuda.empty_cache()
        side = side_figures(args, dev, flush, barrier, peak)

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, desc, cores = oracle_sample(wl, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "cpu_model": cpu_model(), "host_cores": os.cpu_count()}
        if args.cpu_all_cores:
            va, na = oracle_all_cores(args.workload, args.quant_mode, args.cpu_seconds,
                                      bs=args.bs)
            cpu["all_cores"] = {"value": va, "unit": UNIT, "cores": na,
                                "sample": f"the same per-token work on {na} spawned processes, "
                                          "interleaved tokens, each for the same time budget"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_desc(wl), "tokens_per_step": tokens,
                       "rows_per_step": rows,
                       "io": "bf16 tokens in; dispatch rows " + {
                           0: "bf16", 1: "int8 (static)", 2: "int8 + f32 per-row scale",
                           3: "fp8 + f32 per-128 scales", 4: "fp8 + e8m0 per-32 scales",
                           5: "fp8 + e8m0 per-32 scales"}[cfg.quant_mode]
                       + "; combine from " + ("int8 expert outputs + f32 per-8 scales"
                                              if args.combine == "int8"
                                              else "bf16 expert outputs")
                       + "; bf16 out",
                       "l2": ("NOT flushed between steps (--flush none: hot-L2 figures, "
                              "not a valid headline number)") if args.flush == "none" else
                             "flushed between steps: 256 MiB write" + (
                                 " then 256 MiB read (no dirty lines left)"
                                 if args.flush == "write+read" else ""),
                       "parallelism": f"{world} independent replica(s), logical ranks on-device",
                       "launch": "CUDA graph replay of the step's three libcq launches"
                                 if b_use_graph(args) else "direct launches"},
            "per_call_us": {"dispatch": 1e3 * (means["route"] + means["permute"]),
                            "combine": 1e3 * means["combine"],
                            "step_pipelined": 1e3 * ms_per_step,
                            "note": "per-kernel figures come from a separate loop of "
                                    f"{n_bd} steps with events between the kernels"},
            "kernels": kernels, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_step(cfg, smooth_bytes > 0) * args.steps,
            "clocks": clk, "wall_s": t_wall}
    if side is not None:
        line["per_workload"] = side
    emit(line)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def b_use_graph(args) -> bool:
    return not args.no_graph


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_cq(args)


if __name__ == "__main__":
    sys.exit(main())
