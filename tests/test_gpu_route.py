"""Routing on the GPU (moe_route_from_scores, moe_route) against the oracle.

Given the same fp32 score tensor, chosen experts must match bit for bit
(including order and tie-breaking) and gates within GATE_RTOL.
"""
import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from combine_router_gemm_gb300 import inputs
from helpers import GATE_RTOL, cuda_f32, cuda_i32, near_tie_tokens, np_, tc_router_bound

pytestmark = pytest.mark.gpu

CASES = [
    # T, E, k, n_group, topk_group, score_fn, bias, quant_bits, scale
    (4096, 8, 2, 1, 1, "softmax", False, None, 1.0),      # Mixtral routing
    (4096, 8, 2, 1, 1, "softmax", False, 2, 1.0),         # heavy ties
    (4096, 256, 8, 8, 4, "sigmoid", True, None, 2.5),     # DeepSeek-V3 routing
    (4096, 256, 8, 8, 4, "sigmoid", True, 3, 2.5),        # DeepSeek-V3 routing, ties
    (1000, 16, 4, 4, 2, "sigmoid", True, 3, 1.0),
    (7, 3, 3, 1, 1, "softmax", False, None, 1.0),         # k = E
    (1, 1, 1, 1, 1, "sigmoid", False, None, 1.0),         # single expert
    (333, 64, 6, 1, 1, "sigmoid", True, 4, 1.0),
    (128, 1024, 32, 32, 8, "sigmoid", True, None, 2.5),   # largest E and k supported
    (65, 40, 5, 1, 1, "softmax", False, 1, 1.7),          # E not a multiple of 32
    (500, 64, 6, 2, 1, "sigmoid", True, 3, 1.0),          # two groups of 32
    (500, 128, 8, 4, 2, "sigmoid", True, 3, 2.5),         # four groups of 32
]


@pytest.mark.parametrize("T,E,k,ng,tg,fn,use_bias,qb,scale", CASES)
def test_route_from_scores_bit_exact(oracle, T, E, k, ng, tg, fn, use_bias, qb, scale):
    scores = inputs.make_scores(T, E, fn, seed=T + E, quant_bits=qb, device="cuda")
    bias = None
    if use_bias:
        g = torch.Generator(device="cuda")
        g.manual_seed(E)
        bias = torch.randn(E, generator=g, device="cuda") * 0.05
        if qb is not None:
            bias = torch.round(bias * 2 ** qb) / 2 ** qb
    cfg = B.route_cfg(E, k, ng, tg, B.SIGMOID if fn == "sigmoid" else B.SOFTMAX, scale)
    idx, w = cuda_i32((T, k)), cuda_f32((T, k))
    B.moe_route_from_scores(scores, bias, cfg, idx, w)
    torch.cuda.synchronize()
    sc, bb = np_(scores), np_(bias)
    ref_idx = oracle.select(sc, k, bias=bb, n_group=ng, topk_group=tg)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    ref_w = oracle.gates(sc, ref_idx, oracle.SIGMOID if fn == "sigmoid" else oracle.SOFTMAX, scale)
    np.testing.assert_allclose(np_(w), ref_w, rtol=GATE_RTOL, atol=1e-7)


@pytest.mark.parametrize("E,k,ng,tg,fn", [(8, 2, 1, 1, "softmax"), (256, 8, 8, 4, "sigmoid"),
                                          (64, 6, 16, 3, "sigmoid")])
def test_route_signed_zero_keys_tie(oracle, E, k, ng, tg, fn):
    # +0 and -0 compare equal as fp32 keys, so every choice falls to the
    # lowest index, as it does in the oracle
    T = 300
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    neg = torch.rand((T, E), generator=g, device="cuda") < 0.5
    scores = torch.where(neg, torch.tensor(-0.0, device="cuda"), torch.tensor(0.0, device="cuda"))
    assert torch.signbit(scores).any() and not torch.signbit(scores).all()
    cfg = B.route_cfg(E, k, ng, tg, B.SIGMOID if fn == "sigmoid" else B.SOFTMAX, 1.0)
    idx, w = cuda_i32((T, k)), cuda_f32((T, k))
    B.moe_route_from_scores(scores, None, cfg, idx, w)
    torch.cuda.synchronize()
    ref_idx = oracle.select(np_(scores), k, bias=None, n_group=ng, topk_group=tg)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_array_equal(ref_idx, np.tile(np.arange(k, dtype=ref_idx.dtype), (T, 1)))


@pytest.mark.parametrize("name", ["tiny_fp32", "mixtral_bf16", "dsv3_prefill", "dsv3_zipf"])
def test_route_full_router(oracle, name):
    """moe_route on the workload's own x and router weights: scores close to the
    oracle's; expert choice identical except where the oracle's own margin is
    below fp32 rounding of the scores."""
    cfg = inputs.CONFIGS[name]
    T = min(cfg.T, 2048)
    inp = inputs.make_inputs(cfg.with_(T=T), seed=0, device="cuda", experts=False)
    rc = B.cfg_from(cfg)
    scores, idx, w = cuda_f32((T, cfg.E)), cuda_i32((T, cfg.k)), cuda_f32((T, cfg.k))
    B.moe_route(inp["x"], inp["w_router"], inp["bias"], rc, scores, idx, w)
    torch.cuda.synchronize()
    fn = oracle.SIGMOID if cfg.score_fn == "sigmoid" else oracle.SOFTMAX
    ref_sc = oracle.router_scores(np_(inp["x"]), np_(inp["w_router"]), fn)
    err = np.abs(np_(scores).astype(np.float64) - ref_sc)
    if cfg.dtype == "bf16":
        # the bound from each score's measured accumulator range, no assumed
        # magnitude; the measured error must lie inside it everywhere
        bound = tc_router_bound(np_(inp["x"]), np_(inp["w_router"]), fn == oracle.SIGMOID)
        ratio = float((err / bound).max())
        print(f"{name}: router max |err| {err.max():.3e}, max bound {bound.max():.3e}, "
              f"max err/bound {ratio:.3f}")
        assert ratio <= 1.0
        atol = float(bound.max())
    else:
        atol = 2e-5
        assert (err <= atol + 1e-5 * np.abs(ref_sc)).all()
    bias = np_(inp["bias"])
    ref_idx = oracle.select(ref_sc, cfg.k, bias=bias, n_group=cfg.n_group, topk_group=cfg.topk_group)
    got = np_(idx)
    differ = (got != ref_idx).any(1)
    amb = near_tie_tokens(ref_sc, bias, cfg.k, cfg.n_group, cfg.topk_group, rel=1e-5,
                          abs_margin=atol)
    print(f"{name}: {int(differ.sum())} of {T} tokens chose differently from the oracle's own "
          f"scores ({int(amb.sum())} near ties)")
    assert not (differ & ~amb).any(), f"{int((differ & ~amb).sum())} tokens differ without a near tie"
    assert differ.sum() <= max(2, T // 500)


@pytest.mark.parametrize("T,d,E,fn", [(333, 200, 40, "sigmoid"), (1, 64, 8, "softmax"),
                                      (1000, 1024, 130, "softmax"), (257, 7168, 256, "sigmoid")])
def test_router_tensor_core_split_weight(oracle, T, d, E, fn):
    """bf16 activations: the tensor-core router with the fp32 weight split into
    three bf16 terms matches the oracle's router within the rounding bound of
    its fp32 accumulation (tails in tokens, experts and K included)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(T + d + E)
    x = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    wr = torch.randn((E, d), generator=g, device="cuda") * (d ** -0.5)
    k = min(4, E)
    cfg = B.route_cfg(E, k, 1, 1, B.SIGMOID if fn == "sigmoid" else B.SOFTMAX, 1.0)
    scores, idx, w = cuda_f32((T, E)), cuda_i32((T, k)), cuda_f32((T, k))
    B.moe_route(x, wr, None, cfg, scores, idx, w)
    torch.cuda.synchronize()
    ofn = oracle.SIGMOID if fn == "sigmoid" else oracle.SOFTMAX
    ref = oracle.router_scores(np_(x), np_(wr), ofn)
    err = np.abs(np_(scores).astype(np.float64) - ref)
    bound = tc_router_bound(np_(x), np_(wr), fn == "sigmoid")
    assert (err <= bound).all(), f"max err/bound {(err / bound).max():.3f}"


def test_split_router_weight_terms_sum_exactly():
    """hi + mid + lo reproduces every fp32 router weight of magnitude >= 2^-110
    exactly (smaller ones to within 2^-134), each term is bf16, and the terms
    shrink by at least 2^8 each."""
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    w = torch.randn((256, 7168), generator=g, device="cuda") * 0.02
    w[0, :7] = torch.tensor([0.0, -0.0, 1.0, -3.5, 1e-30, 3.0e38, 2.0 ** -126], device="cuda")
    # an fp32 subnormal with bits below bf16's finest spacing (2^-133)
    w[0, 7] = 2.0 ** -126 / 3
    sp = B.moe_split_router_weight(w)
    torch.cuda.synchronize()
    assert sp.dtype == torch.bfloat16 and sp.shape == (3, 256, 7168)
    terms = sp.double()
    total, ref = terms.sum(0), w.double()
    exact = torch.ones_like(ref, dtype=torch.bool)
    exact[0, 7] = False
    assert torch.equal(total[exact], ref[exact])
    assert (total[0, 7] - ref[0, 7]).abs() <= 2.0 ** -134
    hi, mid, lo = terms
    assert (mid.abs() <= hi.abs() * 2.0 ** -8 + 1e-45).all()
    assert (lo.abs() <= mid.abs() * 2.0 ** -8 + 1e-45).all()
