"""The whole layer (moe_layer) against the oracle.

Small workloads are checked on every token; the full-size workloads are run
exactly as the benchmark runs them (same entry point, second stream for the
shared expert) and checked on a seeded sample of tokens, which the oracle can
evaluate one by one, plus properties that hold at any size.
"""
import gc

import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from combine_router_gemm_gb300 import inputs
from helpers import (F32_REL_FRO, assert_bf16_close, cuda_f32, cuda_i32, near_tie_tokens, np_,
                     rel_fro, tc_router_atol)

pytestmark = pytest.mark.gpu


def run_layer(cfg, inp, overlap=True, fused_combine=False):
    T = cfg.T
    layer = B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                       inp["w2_sh"], B.cfg_from(cfg), T, overlap=overlap,
                       fused_combine=fused_combine)
    idx, w = cuda_i32((T, cfg.k)), cuda_f32((T, cfg.k))
    scores, offs = cuda_f32((T, cfg.E)), cuda_i32(cfg.E + 1)
    out = layer.forward(inp["x"], scores_out=scores, topk_idx_out=idx, topk_w_out=w,
                        offsets_out=offs)
    rc, detail = B.moe_check_error(layer.ws)
    assert rc == B.OK, detail
    return out, idx, w, scores, offs


def oracle_tokens(oracle, cfg, inp, tok, needed_experts=None):
    """Oracle on the tokens `tok`; expert weights copied to the host only for
    the experts the oracle itself selects for them."""
    fn = oracle.SIGMOID if cfg.score_fn == "sigmoid" else oracle.SOFTMAX
    x = np_(inp["x"][tok])
    wr = np_(inp["w_router"])
    bias = np_(inp["bias"])
    sc = oracle.router_scores(x, wr, fn)
    sel = oracle.select(sc, cfg.k, bias=bias if fn == oracle.SIGMOID else None,
                        n_group=cfg.n_group, topk_group=cfg.topk_group)
    experts = np.unique(sel)
    w13 = np.empty(tuple(inp["w13"].shape), np.uint16 if cfg.dtype == "bf16" else np.float32)
    w2 = np.empty(tuple(inp["w2"].shape), w13.dtype)
    for e in experts:
        w13[e] = np_(inp["w13"][int(e)])
        w2[e] = np_(inp["w2"][int(e)])
    idx, w, out = oracle.moe_tokens(
        x, E=cfg.E, k=cfg.k, w13=w13, w2=w2, w_router=wr, bias=bias, n_group=cfg.n_group,
        topk_group=cfg.topk_group, score_fn=fn, routed_scale=cfg.routed_scale,
        w13_sh=np_(inp["w13_sh"]), w2_sh=np_(inp["w2_sh"]), round_h=cfg.dtype == "bf16")
    return sc, idx, w, out


def test_layer_tiny_fp32_all_tokens(oracle):
    cfg = inputs.CONFIGS["tiny_fp32"]
    inp = inputs.make_inputs(cfg, seed=0, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp)
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, torch.arange(cfg.T, device="cuda"))
    np.testing.assert_array_equal(np_(idx), ridx)
    np.testing.assert_allclose(np_(w), rw, rtol=1e-5)
    assert rel_fro(np_(out), rout) <= F32_REL_FRO


SMALL_BF16 = [
    inputs.MoEConfig("small_dsv3", T=700, d=256, E=32, k=4, I=128, dtype="bf16",
                     score_fn="sigmoid", n_group=4, topk_group=2, routed_scale=2.5,
                     shared_I=128, bias="normal", expert_std=0.06, router_std=0.06),
    inputs.MoEConfig("small_mixtral", T=513, d=384, E=8, k=2, I=256, dtype="bf16",
                     expert_std=0.05),
    # shared expert wider than the routed ones: separate launches (second stream)
    inputs.MoEConfig("small_dsv3_wide_shared", T=300, d=256, E=16, k=4, I=128, dtype="bf16",
                     score_fn="sigmoid", n_group=4, topk_group=2, routed_scale=2.5,
                     shared_I=256, bias="normal", expert_std=0.06, router_std=0.06),
]


@pytest.mark.parametrize("cfg", SMALL_BF16, ids=lambda c: c.name)
@pytest.mark.parametrize("overlap", [True, False])
def test_layer_small_bf16_all_tokens(oracle, cfg, overlap):
    inp = inputs.make_inputs(cfg, seed=1, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp, overlap)
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, torch.arange(cfg.T, device="cuda"))
    same = (np_(idx) == ridx).all(1)
    amb = near_tie_tokens(sc, np_(inp["bias"]), cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=tc_router_atol(cfg.d))
    assert (same | amb).all()
    assert_bf16_close(np_(out)[same], rout[same], cfg.name)


FULL = ["mixtral_bf16", "dsv3_prefill", "dsv3_decode", "dsv3_zipf"]


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size_sampled(oracle, name):
    cfg = inputs.CONFIGS[name]
    inp = inputs.make_inputs(cfg, seed=0, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp, overlap=True)
    torch.cuda.synchronize()
    # properties at full size
    assert torch.isfinite(out).all()
    o = np_(offs)
    assert o[0] == 0 and o[-1] == cfg.S and (np.diff(o) >= 0).all()
    if cfg.bias == "zipf":
        assert (np.diff(o) == 0).sum() >= cfg.zipf_zero
    # sampled tokens against the oracle
    g = torch.Generator()
    g.manual_seed(7)
    tok = torch.randperm(cfg.T, generator=g)[: min(24, cfg.T)].sort().values
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, tok.cuda())
    gidx = np_(idx[tok.cuda()])
    same = (gidx == ridx).all(1)
    amb = near_tie_tokens(sc, np_(inp["bias"]), cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=tc_router_atol(cfg.d))
    assert (same | amb).all()
    assert_bf16_close(np_(out[tok.cuda()])[same], rout[same], name)
    del inp, out
    gc.collect()
    torch.cuda.empty_cache()


def test_layer_forward_host_pipelined_matches_forward():
    """Host batches through the pipelined path give the same results as
    device-side forward() calls, batch by batch."""
    cfg = SMALL_BF16[0]
    inp = inputs.make_inputs(cfg, seed=3, device="cuda")
    layer = B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                       inp["w2_sh"], B.cfg_from(cfg), cfg.T)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    xs = [torch.randn((cfg.T, cfg.d), generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(5)]
    ref = [layer.forward(x).clone() for x in xs]
    hin = [x.cpu().pin_memory() for x in xs]
    hout = [torch.empty((cfg.T, cfg.d), dtype=torch.float32).pin_memory() for _ in xs]
    layer.forward_host(hin, hout)
    torch.cuda.synchronize()
    for r, h in zip(ref, hout):
        assert torch.equal(r.cpu(), h)
    rc, detail = B.moe_check_error(layer.ws)
    assert rc == B.OK, detail


EDGE = [
    # a single token
    (inputs.MoEConfig("edge_one_token", T=1, d=256, E=32, k=4, I=128, dtype="bf16",
                      score_fn="sigmoid", n_group=4, topk_group=2, routed_scale=2.5, shared_I=128,
                      bias="normal", expert_std=0.06, router_std=0.06), None),
    # one dense expert (E = k = 1): the layer is a single SwiGLU MLP
    (inputs.MoEConfig("edge_dense", T=257, d=128, E=1, k=1, I=256, dtype="bf16",
                      expert_std=0.06), None),
    # every token forced onto the same four experts; the other 28 have NaN
    # weights, which must never be read
    (inputs.MoEConfig("edge_forced", T=600, d=256, E=32, k=4, I=128, dtype="bf16",
                      score_fn="sigmoid", n_group=1, topk_group=1, routed_scale=1.0, shared_I=0,
                      bias="normal", expert_std=0.06, router_std=0.06), [3, 9, 17, 30]),
]


@pytest.mark.parametrize("cfg,forced", EDGE, ids=lambda v: getattr(v, "name", "f"))
def test_layer_edge_cases(oracle, cfg, forced):
    inp = inputs.make_inputs(cfg, seed=5, device="cuda")
    if forced is not None:
        inp["bias"] = torch.full((cfg.E,), -5.0, device="cuda")
        inp["bias"][forced] = 5.0
        rest = [e for e in range(cfg.E) if e not in forced]
        ref_w13, ref_w2 = inp["w13"].clone(), inp["w2"].clone()
        inp["w13"][rest] = float("nan")
        inp["w2"][rest] = float("nan")
    out, idx, w, scores, offs = run_layer(cfg, inp)
    assert torch.isfinite(out).all()
    if forced is not None:
        assert sorted(np.unique(np_(idx)).tolist()) == sorted(forced)
        counts = np.diff(np_(offs))
        assert (counts[forced] == cfg.T).all() and counts.sum() == cfg.S
        inp["w13"], inp["w2"] = ref_w13, ref_w2  # the oracle reads only selected experts anyway
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, torch.arange(cfg.T, device="cuda"))
    same = (np_(idx) == ridx).all(1)
    amb = near_tie_tokens(sc, np_(inp["bias"]), cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=tc_router_atol(cfg.d))
    assert (same | amb).all()
    assert_bf16_close(np_(out)[same], rout[same], cfg.name)


# d and I not multiples of 128: partial feature tiles in the fused epilogue
FUSED_RAGGED = inputs.MoEConfig("fused_ragged", T=333, d=200, E=12, k=3, I=136, dtype="bf16",
                                score_fn="sigmoid", n_group=1, topk_group=1, routed_scale=1.5,
                                shared_I=136, bias="normal", expert_std=0.06, router_std=0.06)


@pytest.mark.parametrize("cfg", [SMALL_BF16[0], SMALL_BF16[1], EDGE[0][0], FUSED_RAGGED],
                         ids=lambda c: c.name)
def test_layer_fused_combine(oracle, cfg):
    """The down projection adding its results straight into the output (fp32
    atomics) agrees with the oracle at the bf16 tolerances, and with the
    unfused layer to fp32 rounding of a reordered sum."""
    inp = inputs.make_inputs(cfg, seed=2, device="cuda")
    out_f, idx, w, scores, offs = run_layer(cfg, inp, fused_combine=True)
    out_u, *_ = run_layer(cfg, inp, fused_combine=False)
    assert torch.isfinite(out_f).all()
    assert rel_fro(np_(out_f), np_(out_u)) < 1e-6
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, torch.arange(cfg.T, device="cuda"))
    same = (np_(idx) == ridx).all(1)
    assert_bf16_close(np_(out_f)[same], rout[same], cfg.name)


def test_layer_fused_combine_full_size_sampled(oracle):
    cfg = inputs.CONFIGS["dsv3_prefill"]
    inp = inputs.make_inputs(cfg, seed=0, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp, fused_combine=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    g = torch.Generator()
    g.manual_seed(9)
    tok = torch.randperm(cfg.T, generator=g)[:16].sort().values
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, tok.cuda())
    same = (np_(idx[tok.cuda()]) == ridx).all(1)
    amb = near_tie_tokens(sc, np_(inp["bias"]), cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=tc_router_atol(cfg.d))
    assert (same | amb).all()
    assert_bf16_close(np_(out[tok.cuda()])[same], rout[same], cfg.name)
    del inp, out
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [SMALL_BF16[0], SMALL_BF16[2], inputs.CONFIGS["tiny_fp32"]],
                         ids=lambda c: c.name)
def test_layer_cuda_graph_replay(oracle, cfg):
    """The layer recorded into a CUDA graph (both streams) and replayed on new
    tokens gives exactly what a direct call gives, and matches the oracle."""
    inp = inputs.make_inputs(cfg, seed=4, device="cuda")
    layer = B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                       inp["w2_sh"], B.cfg_from(cfg), cfg.T)
    x = inp["x"].clone()
    graph, out = layer.capture(x)
    for seed in (5, 6):
        xn = inputs.make_inputs(cfg, seed=seed, device="cuda", experts=False)["x"]
        x.copy_(xn)
        graph.replay()
        direct = layer.forward(xn)
        torch.cuda.synchronize()
        assert torch.equal(out, direct)
    rc, detail = B.moe_check_error(layer.ws)
    assert rc == B.OK, detail
    # the last replay's tokens against the oracle
    inp["x"] = xn
    tok = torch.arange(cfg.T, device="cuda")
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, tok)
    if cfg.dtype == "f32":
        assert rel_fro(np_(out), rout) < 1e-5
    else:
        idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
        layer.forward(xn, topk_idx_out=idx)
        same = (np_(idx) == ridx).all(1)
        assert_bf16_close(np_(out)[same], rout[same], cfg.name)


def test_layer_empty_batch():
    """T = 0: nothing to compute; the call succeeds and reports every expert
    empty."""
    cfg = SMALL_BF16[0].with_(T=0)
    inp = inputs.make_inputs(cfg, seed=1, device="cuda")
    layer = B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                       inp["w2_sh"], B.cfg_from(cfg), 0)
    offs = torch.full((cfg.E + 1,), -1, dtype=torch.int32, device="cuda")
    out = layer.forward(inp["x"], offsets_out=offs)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.d)
    assert (offs == 0).all()
    rc, detail = B.moe_check_error(layer.ws)
    assert rc == B.OK, detail


@pytest.mark.parametrize("overlap", [True, False])
def test_layer_packed_weights_bit_identical(overlap):
    """The layer on tile-major packed weights gives the same output, bit for
    bit, as on the row-major weights they came from."""
    cfg = SMALL_BF16[0]
    inp = inputs.make_inputs(cfg, seed=8, device="cuda")
    args = (inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"], inp["w2_sh"],
            B.cfg_from(cfg), cfg.T)
    packed = B.MoELayer(*args, overlap=overlap, pack_weights=True)
    plain = B.MoELayer(*args, overlap=overlap, pack_weights=False)
    assert packed.packed and not plain.packed
    a = packed.forward(inp["x"])
    b = plain.forward(inp["x"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    for layer in (packed, plain):
        rc, detail = B.moe_check_error(layer.ws)
        assert rc == B.OK, detail


def test_layer_presplit_router_bit_identical():
    """The router weight split once beforehand gives the same layer output,
    bit for bit, as splitting it on every call."""
    cfg = SMALL_BF16[0]
    inp = inputs.make_inputs(cfg, seed=9, device="cuda")
    args = (inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"], inp["w2_sh"],
            B.cfg_from(cfg), cfg.T)
    once = B.MoELayer(*args, split_router=True)
    each = B.MoELayer(*args, split_router=False)
    assert once.w_router_split is not None and each.w_router_split is None
    a, b = once.forward(inp["x"]), each.forward(inp["x"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
