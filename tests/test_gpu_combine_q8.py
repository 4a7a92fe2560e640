"""GPU parity of the combine-side int8 path against the oracle: the expert-side
block quantiser (codes and scales bit-exact) and the dequantising combine
(fp32 within 1e-5 and bf16 within 1 ulp; exact agreement is also asserted,
both sides use the same operation order)."""
import numpy as np
import pytest
import torch

import gpu_harness as gh
import oracle
from combine_quant_gb300 import workloads

pytestmark = pytest.mark.gpu


def _case(name):
    return {
        "tiny": lambda: workloads.tiny(0, 2),
        "special_small": lambda: workloads.special(seed=23, W=8, BS=20, H=1024, M=48),
        "skew_small": lambda: workloads.skew(seed=24, W=4, BS=64, M=32, K=16, H=2048),
        "dsv3": lambda: workloads.dsv3(),
        # H % 32 != 0: the direct-gather combine instead of the staged one
        "h1040": lambda: workloads.dsv3(seed=25, W=4, BS=9, M=16, K=4, H=1040),
    }[name]()


@pytest.mark.parametrize("name", ["tiny", "special_small", "skew_small", "dsv3", "h1040"])
def test_combine_q8_parity(name):
    import combine_quant_gb300 as cq
    wl = _case(name)
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    ref = oracle.route(wl.cfg, wl.expert_ids, wl.mask, wl.bs_per_rank)
    ffn = gh.FfnStandin(wl, cfg.max_rows)
    codes, scales = cq.combine_quant(cfg, ffn.device_rows, out.assist_info)
    # quantiser: every dispatched row against the oracle's quantisation of its pool row
    pc, ps = oracle.combine_quant_rows(ffn.pool)
    R = ref.rows
    for a in range(0, R, 16384):
        b = min(R, a + 16384)
        src = (np.arange(a, b, dtype=np.int64) * 7919) % ffn.P
        assert np.array_equal(gh.host(codes[a:b]), pc[src]), f"int8 codes differ in {a}..{b}"
        assert np.array_equal(gh.host(scales[a:b]).view(np.uint32), ps[src].view(np.uint32)), \
            f"block scales differ in {a}..{b}"
    # dequantising combine, every token
    w = gh.dev(wl.expert_scales, torch.float32)
    kw = dict(ori_x=gh.dev(wl.x, torch.bfloat16), const_alpha1=gh.dev(wl.const_alpha1, torch.float32),
              const_alpha2=gh.dev(wl.const_alpha2, torch.float32),
              const_v=gh.dev(wl.const_v, torch.bfloat16))
    y32 = cq.combine_q8(cfg, codes, scales, out.assist_info, w, out.ep_recv_count,
                        out_dtype=torch.float32, **kw)
    yb = cq.combine_q8(cfg, codes, scales, out.assist_info, w, out.ep_recv_count, **kw)
    inv = ffn.remap_inv(ref.inv)

    def oracle_tokens(toks, out_f32):
        return oracle.combine_tokens_q8(wl.cfg, toks, pc, ps, inv, wl.expert_scales, wl.x,
                                        wl.const_alpha1, wl.const_alpha2, wl.const_v,
                                        out_f32=out_f32)

    gh.compare_combine_complete(wl, y32, yb, oracle_tokens)


def test_combine_quant_zero_rows():
    """All-zero expert rows: scale 0, codes 0, and a zero contribution."""
    import combine_quant_gb300 as cq
    wl = workloads.tiny(1, 2)
    cfg, out, _, _ = gh.gpu_dispatch(wl)
    zeros = torch.zeros(cfg.max_rows, cfg.hidden, dtype=torch.bfloat16, device=gh.DEV)
    codes, scales = cq.combine_quant(cfg, zeros, out.assist_info)
    R = int(gh.host(cq.assist_views(cfg, out.assist_info)[2])[-1])
    assert torch.count_nonzero(codes[:R]) == 0 and torch.count_nonzero(scales[:R]) == 0
    y = cq.combine_q8(cfg, codes, scales, out.assist_info, gh.dev(wl.expert_scales, torch.float32),
                      out_dtype=torch.float32)
    assert torch.count_nonzero(y) == 0


@pytest.mark.parametrize("x_dtype", [0, 1])
def test_combine_quant_extreme_blocks(x_dtype):
    """Block quantiser on blocks that leave the ordinary case, every dispatched
    row against the oracle bit for bit: all-zero and -0 blocks, NaN and +-inf
    elements, subnormal blocks (the scale max * fl(1/127) underflows to a
    subnormal or zero and the quotients saturate), huge values, and values
    whose quotients sit on .5 ties."""
    import combine_quant_gb300 as cq
    wl = workloads.tiny(5, 2)
    if x_dtype:
        wl = workloads.as_fp16(wl)
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    R = int(gh.host(cq.assist_views(cfg, out.assist_info)[2])[-1])
    H = cfg.hidden
    rng = np.random.default_rng(6)
    f = rng.standard_normal((cfg.max_rows, H)).astype(np.float32)
    f[0, :8] = 0.0
    f[0, 8:16] = -0.0
    f[0, 16:24] = 1.0
    f[0, 17] = np.nan
    f[0, 24:32] = 2.0
    f[0, 25] = np.inf
    f[0, 32:40] = -np.inf
    f[0, 40:48] = np.nan
    f[1, :64] *= 1e-39 if x_dtype == 0 else 1e-7   # subnormal in the 16-bit type
    f[1, 64:72] = 3.0e38 if x_dtype == 0 else 60000.0
    f[2, :8] = [127.0, 63.5, 0.5, 1.5, -0.5, -2.5, 31.75, 100.0]  # max 127: scale ~1, ties
    f[2, 8:16] = [-127.0, 0.25, 64.25, -63.5, 126.5, 3.5, -4.5, 12.0]
    bits = workloads.to_f16_bits(f) if x_dtype else workloads.to_bf16_bits(f)
    rows = torch.from_numpy(bits).to(gh.DEV).view(cfg.token_dtype)
    codes, scales = cq.combine_quant(cfg, rows, out.assist_info)
    pc, ps = oracle.combine_quant_rows(bits[:R], x_dtype)
    assert np.array_equal(gh.host(codes[:R]), pc), "int8 codes differ"
    assert np.array_equal(gh.host(scales[:R]).view(np.uint32), ps.view(np.uint32)), \
        "block scales differ"


def _division_blocks(x_dtype: int) -> np.ndarray:
    """Blocks [m, v1..v7] with |v| <= |m| covering the quotients v / s of the
    block quantiser (s = max * fl(1/127)) that can round to a non-zero code:
    every mantissa pair of m and v at every exponent offset d = e_m - e_v in
    0..10 (a larger offset makes |v / s| < 0.5), with m at a few exponents
    from the bottom to the top of the range; bf16 exhaustively, fp16 with
    every 3rd m and every 7th v mantissa. The quotient depends only on the mantissas and d
    while s stays normal, which the bottom exponents leave."""
    rng = np.random.default_rng(17)
    if x_dtype == 0:
        man_m, man_v = range(128), range(128)
        exps = [1, 2, 5, 6, 7, 8, 9, 12, 127, 200, 254]   # biased binary32 exponents
        to_f = lambda e, mm: np.float32(np.ldexp(1.0 + mm / 128.0, e - 127))
    else:
        man_m, man_v = range(0, 1024, 3), range(0, 1024, 7)
        exps = [1, 2, 10, 15, 25, 30]                      # biased fp16 exponents
        to_f = lambda e, mm: np.float32(np.ldexp(1.0 + mm / 1024.0, e - 15))
    blocks = []
    for e in exps:
        for mm in man_m:
            m = to_f(e, mm)
            vs = []
            for d in range(0, 11):
                if e - d < 1:
                    break
                for vm in man_v:
                    if d == 0 and vm > mm:
                        continue
                    v = to_f(e - d, vm)
                    vs += [v, -v]
            if x_dtype == 1 and e <= 10:  # fp16 subnormals below m
                vs += [np.float32(np.ldexp(k, -24)) for k in range(1, 1024, 37)]
            vs = np.array(vs, np.float32)
            vs = np.concatenate([vs, np.zeros((-len(vs)) % 7, np.float32)]).reshape(-1, 7)
            sign = np.where(rng.random(len(vs)) < 0.5, -1.0, 1.0).astype(np.float32)
            blk = np.concatenate([(m * sign)[:, None], vs], axis=1)
            blocks.append(blk)
    return np.concatenate(blocks).reshape(-1)


@pytest.mark.parametrize("x_dtype", [0, 1])
def test_combine_quant_division_exhaustive(x_dtype):
    """The quantiser's division (a reciprocal and one correction step) against
    the oracle's IEEE division on the structured block set above: codes and
    scales bit for bit."""
    import combine_quant_gb300 as cq
    wl = workloads.dsv3(seed=40, W=8, BS=128, M=64, K=8, H=1024)
    if x_dtype:
        wl = workloads.as_fp16(wl)
    cfg, out, status, _ = gh.gpu_dispatch(wl)
    R = int(gh.host(cq.assist_views(cfg, out.assist_info)[2])[-1])
    vals = _division_blocks(x_dtype)
    H = cfg.hidden
    n_rows = (vals.size + H - 1) // H
    assert n_rows <= R, (n_rows, R)
    f = np.zeros((cfg.max_rows, H), np.float32)
    f.reshape(-1)[:vals.size] = vals
    bits = workloads.to_f16_bits(f) if x_dtype else workloads.to_bf16_bits(f)
    # every value is exact in the 16-bit type
    back = workloads.bf16_bits_to_f32(bits) if x_dtype == 0 else bits.view(np.float16).astype(np.float32)
    assert np.array_equal(back.reshape(-1)[:vals.size], vals)
    rows = torch.from_numpy(bits).to(gh.DEV).view(cfg.token_dtype)
    codes, scales = cq.combine_quant(cfg, rows, out.assist_info)
    pc, ps = oracle.combine_quant_rows(bits[:n_rows], x_dtype)
    assert np.array_equal(gh.host(codes[:n_rows]), pc), "int8 codes differ"
    assert np.array_equal(gh.host(scales[:n_rows]).view(np.uint32), ps.view(np.uint32))
