"""The whole layer (moe_layer) against the oracle.

Small workloads are checked on every token.  The full-size workloads are run
exactly as the benchmark runs them (same entry point, second stream for the
shared expert, tile-major weights) and checked
  * on every token: the chosen experts bit for bit and the gates, from the
    layer's own score tensor; the expert offsets bit for bit; the router
    scores within their measured rounding bound, and how many tokens the
    oracle's own scores would route differently (near ties only, bounded);
  * element by element on the output rows of a token sample that covers
    every active expert, every segment's last row and every second token tile
    (the oracle evaluates tokens one by one, given the layer's scores).
"""
import gc

import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from combine_router_gemm_gb300 import inputs
from helpers import (F32_REL_FRO, GATE_RTOL, assert_bf16_close, coverage_tokens, cuda_f32,
                     cuda_i32, near_tie_tokens, np_, rel_fro, tc_router_bound)

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


def router_margin(cfg, inp):
    """Largest rounding bound of the layer's router scores on these inputs
    (bf16: tensor cores, measured accumulator range; fp32: CUDA cores)."""
    if cfg.dtype != "bf16":
        return 2e-5
    return float(tc_router_bound(np_(inp["x"]), np_(inp["w_router"]),
                                 cfg.score_fn == "sigmoid").max())


def _host_experts(cfg, inp, experts):
    """Host copies of the expert weights, filled only for `experts` (the
    oracle reads no other expert)."""
    w13 = np.empty(tuple(inp["w13"].shape), np.uint16 if cfg.dtype == "bf16" else np.float32)
    w2 = np.empty(tuple(inp["w2"].shape), w13.dtype)
    for e in experts:
        w13[e] = np_(inp["w13"][int(e)])
        w2[e] = np_(inp["w2"][int(e)])
    return w13, w2


def oracle_tokens(oracle, cfg, inp, tok, scores=None):
    """Oracle on the tokens `tok` (its own router, or the given score rows);
    expert weights copied to the host only for the experts it selects."""
    fn = oracle.SIGMOID if cfg.score_fn == "sigmoid" else oracle.SOFTMAX
    x = np_(inp["x"][tok])
    wr = np_(inp["w_router"])
    bias = np_(inp["bias"])
    sc = oracle.router_scores(x, wr, fn) if scores is None else scores
    sel = oracle.select(sc, cfg.k, bias=bias if fn == oracle.SIGMOID else None,
                        n_group=cfg.n_group, topk_group=cfg.topk_group)
    w13, w2 = _host_experts(cfg, inp, np.unique(sel))
    idx, w, out = oracle.moe_tokens(
        x, E=cfg.E, k=cfg.k, w13=w13, w2=w2, scores=scores,
        w_router=wr if scores is None else None, bias=bias, n_group=cfg.n_group,
        topk_group=cfg.topk_group, score_fn=fn, routed_scale=cfg.routed_scale,
        w13_sh=np_(inp["w13_sh"]), w2_sh=np_(inp["w2_sh"]), round_h=cfg.dtype == "bf16")
    return sc, idx, w, out


def full_size_parity(oracle, cfg, inp, out, idx, w, scores, offs, n_sample, seed):
    """Every check of a full-size layer run; returns a one-line report."""
    fn = oracle.SIGMOID if cfg.score_fn == "sigmoid" else oracle.SOFTMAX
    bias = np_(inp["bias"]) if fn == oracle.SIGMOID else None
    T = cfg.T
    sc_gpu, gidx = np_(scores), np_(idx)
    # routing from the layer's own score tensor, every token: bit-exact
    ridx = oracle.select(sc_gpu, cfg.k, bias=bias, n_group=cfg.n_group, topk_group=cfg.topk_group)
    np.testing.assert_array_equal(gidx, ridx, err_msg="top-k from the layer's scores")
    rw = oracle.gates(sc_gpu, gidx, fn, cfg.routed_scale)
    np.testing.assert_allclose(np_(w), rw, rtol=GATE_RTOL, atol=1e-7, err_msg="gates")
    # dispatch of that routing: offsets bit-exact
    counts, roffs, s2r, r2t = oracle.dispatch(gidx, cfg.E)
    np.testing.assert_array_equal(np_(offs), roffs, err_msg="expert offsets")
    # the router on every token, against the oracle's double-precision router:
    # inside the rounding bound measured from each score's accumulator range
    x_all, wr = np_(inp["x"]), np_(inp["w_router"])
    sc_o = oracle.router_scores(x_all, wr, fn)
    err = np.abs(sc_gpu.astype(np.float64) - sc_o)
    bound = tc_router_bound(x_all, wr, fn == oracle.SIGMOID)
    ratio = float((err / bound).max())
    assert ratio <= 1.0, f"router error above its bound (max err/bound {ratio:.3f})"
    # end to end without injected scores: tokens the oracle's own scores route
    # differently must be near ties within that bound, and rare
    oidx = oracle.select(sc_o, cfg.k, bias=bias, n_group=cfg.n_group, topk_group=cfg.topk_group)
    flips = (oidx != gidx).any(1)
    amb = near_tie_tokens(sc_o, bias, cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=float(bound.max()))
    bad = np.nonzero(flips & ~amb)[0]
    assert bad.size == 0, (f"{bad.size} flips without a near tie, e.g. token {bad[0]}: layer "
                           f"{gidx[bad[0]].tolist()}, oracle {oidx[bad[0]].tolist()}")
    assert flips.sum() <= max(1, T // 500), f"{int(flips.sum())} routing flips"
    # element by element on a token sample covering every active expert,
    # every segment's last row and every second token tile, given the same
    # scores (so that no token is left out)
    tok = coverage_tokens(roffs, r2t, T, n_sample, seed)
    rows = np.nonzero(np.isin(r2t, tok))[0]
    seg = np.searchsorted(roffs, rows, side="right") - 1
    local = rows - roffs[seg]
    covered = np.unique(seg)
    assert np.array_equal(covered, np.nonzero(counts)[0]), "sample misses an active expert"
    for q in (160, 256):  # a second token tile of every expert that has one
        hit = np.zeros(cfg.E, bool)
        hit[seg[local >= q]] = True
        assert (hit | (counts <= q)).all(), f"sample misses rows past {q}"
    tt = torch.from_numpy(tok).cuda()
    _, oi, ow, rout = oracle_tokens(oracle, cfg, inp, tt, scores=sc_gpu[tok])
    np.testing.assert_array_equal(oi, gidx[tok])
    mx, rf = assert_bf16_close(np_(out[tt]), rout, cfg.name)
    return (f"{cfg.name}: routing bit-exact on {T} tokens; router max |err| {err.max():.2e} "
            f"(max err/bound {ratio:.3f}, bound <= {bound.max():.2e}); {int(flips.sum())} "
            f"end-to-end flips ({int(amb.sum())} near ties); {len(tok)} tokens / {len(rows)} "
            f"rows checked, {len(covered)} experts, max row in segment {int(local.max())}, "
            f"max-abs {mx:.2e}, rel-fro {rf:.2e}")


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
    # 512 rows per expert: both routed launches on CTA pairs (256-token tiles);
    # without a second stream the shared expert's tiles ride in them
    inputs.MoEConfig("small_pairs_shared", T=2048, d=256, E=8, k=2, I=128, dtype="bf16",
                     shared_I=128, expert_std=0.06),
]


@pytest.mark.parametrize("cfg", SMALL_BF16, ids=lambda c: c.name)
@pytest.mark.parametrize("overlap", [True, False])
def test_layer_small_bf16_all_tokens(oracle, cfg, overlap):
    inp = inputs.make_inputs(cfg, seed=1, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp, overlap)
    sc, ridx, rw, rout = oracle_tokens(oracle, cfg, inp, torch.arange(cfg.T, device="cuda"))
    same = (np_(idx) == ridx).all(1)
    amb = near_tie_tokens(sc, np_(inp["bias"]), cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=router_margin(cfg, inp))
    assert (same | amb).all()
    assert_bf16_close(np_(out)[same], rout[same], cfg.name)


FULL = ["mixtral_bf16", "dsv3_prefill", "dsv3_decode", "dsv3_zipf"]


@pytest.mark.parametrize("name,seed", [(n, 0) for n in FULL] +
                         [("dsv3_prefill", 1), ("dsv3_zipf", 1)])
def test_layer_full_size(oracle, name, seed):
    """Seed 0 is the benchmark's input; seed 1 a second draw of the same
    workload."""
    cfg = inputs.CONFIGS[name]
    inp = inputs.make_inputs(cfg, seed=seed, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp, overlap=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    o = np_(offs)
    if cfg.bias == "zipf":
        assert (np.diff(o) == 0).sum() >= cfg.zipf_zero
    print(full_size_parity(oracle, cfg, inp, out, idx, w, scores, offs, n_sample=512,
                           seed=7 + seed))
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
                          abs_margin=router_margin(cfg, inp))
    assert (same | amb).all()
    assert_bf16_close(np_(out)[same], rout[same], cfg.name)


# d and I not multiples of 128: partial feature tiles in the fused epilogue
FUSED_RAGGED = inputs.MoEConfig("fused_ragged", T=333, d=200, E=12, k=3, I=136, dtype="bf16",
                                score_fn="sigmoid", n_group=1, topk_group=1, routed_scale=1.5,
                                shared_I=136, bias="normal", expert_std=0.06, router_std=0.06)


@pytest.mark.parametrize("cfg", [SMALL_BF16[0], SMALL_BF16[1], SMALL_BF16[3], EDGE[0][0],
                                 FUSED_RAGGED], ids=lambda c: c.name)
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


def test_layer_fused_combine_full_size(oracle):
    cfg = inputs.CONFIGS["dsv3_prefill"]
    inp = inputs.make_inputs(cfg, seed=0, device="cuda")
    out, idx, w, scores, offs = run_layer(cfg, inp, fused_combine=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    print(full_size_parity(oracle, cfg, inp, out, idx, w, scores, offs, n_sample=256, seed=9))
    del inp, out
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg,split", [(SMALL_BF16[0], False), (SMALL_BF16[2], False),
                                       (SMALL_BF16[3], False), (inputs.CONFIGS["tiny_fp32"], False),
                                       (SMALL_BF16[0], True), (SMALL_BF16[1], True)],
                         ids=lambda v: getattr(v, "name", "split" if v else "one-pass"))
def test_layer_cuda_graph_replay(oracle, cfg, split):
    """The layer recorded into a CUDA graph (both streams; also with the
    dispatch split over them) and replayed on new tokens gives exactly what
    a direct call gives, and matches the oracle."""
    inp = inputs.make_inputs(cfg, seed=4, device="cuda")
    layer = B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                       inp["w2_sh"], B.cfg_from(cfg), cfg.T, split_dispatch=split)
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


def _split_vs_plain(cfg, inp):
    """The layer with the dispatch split over two streams and without it, on
    the same weights and tokens: outputs, routing and offsets."""
    args = (inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"], inp["w2_sh"],
            B.cfg_from(cfg), cfg.T)
    res = []
    for split in (True, False):
        layer = B.MoELayer(*args, split_dispatch=split)
        assert (layer.stream2 is not None) or not split
        idx, offs = cuda_i32((cfg.T, cfg.k)), cuda_i32(cfg.E + 1)
        out = layer.forward(inp["x"], topk_idx_out=idx, offsets_out=offs)
        rc, detail = B.moe_check_error(layer.ws)
        assert rc == B.OK, detail
        res.append((out, idx, offs))
        del layer
    torch.cuda.synchronize()
    (a, ia, oa), (b, ib, ob) = res
    assert torch.equal(ia, ib) and torch.equal(oa, ob)
    assert torch.equal(a, b)
    return a


@pytest.mark.parametrize("cfg", SMALL_BF16, ids=lambda c: c.name)
def test_layer_split_dispatch_bit_identical(cfg):
    """The permute of the upper half of the experts on the second stream
    beside the lower half's gate/up (then that half's gate/up): the same
    output, bit for bit, as the one-pass dispatch."""
    inp = inputs.make_inputs(cfg, seed=11, device="cuda")
    _split_vs_plain(cfg, inp)


def test_layer_split_dispatch_all_tokens(oracle):
    cfg = SMALL_BF16[0]
    inp = inputs.make_inputs(cfg, seed=12, device="cuda")
    out = _split_vs_plain(cfg, inp)
    sc, ridx, _, rout = oracle_tokens(oracle, cfg, inp, torch.arange(cfg.T, device="cuda"))
    amb = near_tie_tokens(sc, np_(inp["bias"]), cfg.k, cfg.n_group, cfg.topk_group,
                          abs_margin=router_margin(cfg, inp))
    layer = B.MoELayer(inp["w_router"], inp["bias"], inp["w13"], inp["w2"], inp["w13_sh"],
                       inp["w2_sh"], B.cfg_from(cfg), cfg.T, split_dispatch=True)
    idx = cuda_i32((cfg.T, cfg.k))
    layer.forward(inp["x"], topk_idx_out=idx)
    torch.cuda.synchronize()
    same = (np_(idx) == ridx).all(1)
    assert (same | amb).all()
    assert_bf16_close(np_(out)[same], rout[same], "split dispatch")


@pytest.mark.parametrize("name", ["mixtral_bf16", "dsv3_prefill", "dsv3_zipf"])
def test_layer_split_dispatch_full_size_bit_identical(name):
    """At full size (Zipf: uneven halves and empty experts; Mixtral: no
    shared expert, the second stream free for the permute)."""
    cfg = inputs.CONFIGS[name]
    inp = inputs.make_inputs(cfg, seed=0, device="cuda")
    out = _split_vs_plain(cfg, inp)
    assert torch.isfinite(out).all()
    del inp, out
    gc.collect()
    torch.cuda.empty_cache()


SPLIT_EDGE = [
    # an odd expert count: halves of 2 and 3 experts
    (inputs.MoEConfig("split_odd", T=333, d=256, E=5, k=2, I=128, dtype="bf16",
                      expert_std=0.06), None),
    (EDGE[0][0], None),  # a single token: one half gets at most 4 slots
    (EDGE[1][0], None),  # E = 1: runs unsplit
    # every token on experts of the upper half; the lower half's permute and
    # gate/up launch have nothing to do, and the other experts' NaN weights
    # must never be read
    (EDGE[2][0], [17, 20, 25, 30]),
]


@pytest.mark.parametrize("cfg,forced", SPLIT_EDGE, ids=lambda v: getattr(v, "name", "f"))
def test_layer_split_dispatch_edge_cases(cfg, forced):
    inp = inputs.make_inputs(cfg, seed=13, device="cuda")
    if forced is not None:
        inp["bias"] = torch.full((cfg.E,), -5.0, device="cuda")
        inp["bias"][forced] = 5.0
        rest = [e for e in range(cfg.E) if e not in forced]
        inp["w13"][rest] = float("nan")
        inp["w2"][rest] = float("nan")
    out = _split_vs_plain(cfg, inp)
    assert torch.isfinite(out).all()
