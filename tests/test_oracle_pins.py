"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test names the fact it checks: brute-force enumeration, a closed form, a
library routine on a special case, or an invariant of the definition.  The
layer's arithmetic follows the plainest reading of the DeepSeek-V3 MoE layer
named by "CUCo: An Agentic Framework for Compute and Communication Co-design"
(abstract; Table 4, row "MoE Dispatch/Combine").
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

from combine_router_gemm_gb300 import inputs

RNG = np.random.default_rng(1234)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    return inputs.to_numpy(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_fp32_values(oracle):
    # For values exactly representable in fp32, one rounding from double equals
    # torch's fp32 -> bf16 round-to-nearest-even (a library routine).
    vals = np.concatenate([
        RNG.standard_normal(2000).astype(np.float32),
        (RNG.standard_normal(500) * 1e-30).astype(np.float32),
        # exact ties between two bf16 neighbours: 1 + (2m+1) * 2^-8
        np.array([1 + (2 * m + 1) * 2.0 ** -8 for m in range(16)], np.float32),
        np.array([-(1 + 2.0 ** -8), 3 * 2.0 ** -8 + 1], np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals])
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_single_rounding_closed_forms(oracle):
    # 1 + 2^-8 + 2^-40 lies just above the midpoint of 1 and 1 + 2^-7, so the
    # nearest bf16 is 1 + 2^-7 (rounding through fp32 would give 1).
    assert oracle.round_bf16(1 + 2.0 ** -8 + 2.0 ** -40) == 1 + 2.0 ** -7
    # exact midpoint goes to the even neighbour (mantissa 0 -> 1.0)
    assert oracle.round_bf16(1 + 2.0 ** -8) == 1.0
    # subnormal range: spacing 2^-133, 1.5 * 2^-133 ties to even 2 * 2^-133
    assert oracle.round_bf16(1.5 * 2.0 ** -133) == 2.0 ** -132
    assert oracle.round_bf16(0.0) == 0.0
    assert oracle.round_bf16(-3.0) == -3.0


# ---------------------------------------------------------------- selection

def brute_topk(keys: np.ndarray, k: int, allowed=None):
    """Best k-subset by exact key sum, ties to the lexicographically smallest
    index set, then listed by descending key / ascending index."""
    cand = [e for e in range(len(keys)) if allowed is None or allowed[e]]
    best, best_sum = None, None
    for sub in itertools.combinations(cand, k):  # lexicographic order
        s = sum(float(keys[e]) for e in sub)
        if best is None or s > best_sum:
            best, best_sum = sub, s
    return sorted(best, key=lambda e: (-float(keys[e]), e))


@pytest.mark.parametrize("E,k", [(8, 2), (8, 1), (5, 3), (6, 6)])
def test_select_softmax_brute_force(oracle, E, k):
    # Scores are multiples of 1/8 in [-1, 1]: sums are exact and ties abound.
    T = 300
    scores = np.round(RNG.uniform(-1, 1, (T, E)) * 8) / 8
    scores = scores.astype(np.float32)
    idx = oracle.select(scores, k)
    for t in range(T):
        assert list(idx[t]) == brute_topk(scores[t], k), t


def brute_grouped(key: np.ndarray, n_group: int, topk_group: int, k: int):
    E = len(key)
    gs = E // n_group
    gscore = []
    for g in range(n_group):
        members = range(g * gs, (g + 1) * gs)
        # sum of the two largest = the largest sum over distinct pairs
        gscore.append(max(float(key[a]) + float(key[b])
                          for a, b in itertools.combinations(members, 2)))
    best, best_sum = None, None
    for gsub in itertools.combinations(range(n_group), topk_group):
        s = sum(gscore[g] for g in gsub)
        if best is None or s > best_sum:
            best, best_sum = gsub, s
    allowed = [(e // gs) in best for e in range(E)]
    return brute_topk(key, k, allowed)


@pytest.mark.parametrize("E,n_group,topk_group,k", [(16, 4, 2, 4), (12, 3, 1, 2), (16, 8, 3, 5)])
def test_select_grouped_brute_force(oracle, E, n_group, topk_group, k):
    # Biased key = fp32(score + bias); both multiples of 1/8, so the fp32 sum is
    # exact and equals the real sum used by the brute force.
    T = 200
    s = (np.round(RNG.uniform(0, 1, (T, E)) * 8) / 8).astype(np.float32)
    b = (np.round(RNG.uniform(-0.5, 0.5, E) * 8) / 8).astype(np.float32)
    idx = oracle.select(s, k, bias=b, n_group=n_group, topk_group=topk_group)
    for t in range(T):
        assert list(idx[t]) == brute_grouped(s[t] + b, n_group, topk_group, k), t


def test_select_bias_changes_choice_not_gates(oracle):
    # A large bias on expert 3 forces it in; gates still use the unbiased score.
    s = np.array([[0.9, 0.8, 0.7, 0.1, 0.6, 0.5, 0.4, 0.3]], np.float32)
    b = np.zeros(8, np.float32)
    b[3] = 10.0
    idx = oracle.select(s, 2, bias=b)
    assert list(idx[0]) == [3, 0]
    w = oracle.gates(s, idx, oracle.SIGMOID, routed_scale=2.5)
    np.testing.assert_allclose(w[0], [2.5 * 0.1 / 1.0, 2.5 * 0.9 / 1.0], rtol=1e-7)


# ---------------------------------------------------------------- gates

def test_gates_softmax_top2_is_logistic_of_difference(oracle):
    # Renormalised softmax over two experts: w_1 = 1 / (1 + exp(l_2 - l_1)).
    T, E = 500, 8
    scores = RNG.standard_normal((T, E)).astype(np.float32)
    idx = oracle.select(scores, 2)
    w = oracle.gates(scores, idx, oracle.SOFTMAX)
    l1 = scores[np.arange(T), idx[:, 0]].astype(np.float64)
    l2 = scores[np.arange(T), idx[:, 1]].astype(np.float64)
    np.testing.assert_allclose(w[:, 0], scipy.special.expit(l1 - l2), rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)


def test_gates_softmax_equals_softmax_of_selected(oracle):
    # The full-softmax denominator cancels: w = softmax(selected logits) * scale.
    T, E, k = 200, 32, 6
    scores = (RNG.standard_normal((T, E)) * 3).astype(np.float32)
    idx = oracle.select(scores, k)
    w = oracle.gates(scores, idx, oracle.SOFTMAX, routed_scale=1.7)
    sel = np.take_along_axis(scores, idx, 1).astype(np.float64)
    np.testing.assert_allclose(w, 1.7 * scipy.special.softmax(sel, axis=1), rtol=1e-12)
    # shift invariance of the definition
    w2 = oracle.gates(scores + np.float32(4.0), idx, oracle.SOFTMAX, routed_scale=1.7)
    np.testing.assert_allclose(w2, w, rtol=1e-5)


def test_gates_sigmoid_sum_and_ratio(oracle):
    T, E, k = 300, 64, 8
    s = RNG.uniform(0.01, 1, (T, E)).astype(np.float32)
    idx = oracle.select(s, k)
    w = oracle.gates(s, idx, oracle.SIGMOID, routed_scale=2.5)
    np.testing.assert_allclose(w.sum(1), 2.5, rtol=1e-14)
    sel = np.take_along_axis(s, idx, 1).astype(np.float64)
    np.testing.assert_allclose(w[:, 1:] / w[:, :1], sel[:, 1:] / sel[:, :1], rtol=1e-13)


# ---------------------------------------------------------------- dispatch

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 2, 8), (1000, 8, 256), (64, 2, 8), (33, 3, 5)])
def test_dispatch_equals_stable_argsort(oracle, T, k, E):
    idx = RNG.integers(0, E, (T, k)).astype(np.int32)
    if E > 4:
        idx[idx == 3] = 4                       # expert 3 receives nothing
    counts, offsets, s2r, r2t = oracle.dispatch(idx, E)
    flat = idx.reshape(-1)
    order = np.argsort(flat, kind="stable")     # row -> slot
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    inv = np.empty_like(order)
    inv[order] = np.arange(len(order))
    np.testing.assert_array_equal(s2r, inv)
    np.testing.assert_array_equal(r2t, order // k)
    # invariants: bijection onto [0, S), counts sum to S
    assert sorted(s2r.tolist()) == list(range(T * k))
    assert counts.sum() == T * k and offsets[-1] == T * k


# ---------------------------------------------------------------- expert FFN

def silu(a):
    return a * scipy.special.expit(a)


def test_ffn_dense_special_case_numpy(oracle):
    # E=1, k=1: the layer reduces to one dense SwiGLU MLP, computed here with
    # numpy matmuls.  d != I catches transposed operands.
    T, d, I = 17, 24, 40
    x = RNG.standard_normal((T, d)).astype(np.float32)
    w13 = (RNG.standard_normal((1, 2 * I, d)) * 0.3).astype(np.float32)
    w2 = (RNG.standard_normal((1, d, I)) * 0.3).astype(np.float32)
    idx, w, out = oracle.moe_tokens(x, E=1, k=1, w13=w13, w2=w2,
                                    scores=np.zeros((T, 1), np.float32))
    assert (idx == 0).all() and np.allclose(w, 1.0)
    xd = x.astype(np.float64)
    g = xd @ w13[0, :I].astype(np.float64).T
    u = xd @ w13[0, I:].astype(np.float64).T
    ref = (silu(g) * u) @ w2[0].astype(np.float64).T
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_ffn_gate_up_order_closed_form(oracle):
    # x = e_0, W1[:,0] = +40, W3[:,0] = -40, W2 = identity (d = I):
    # h = silu(40) * (-40) = -40 * 40 / (1 + e^-40).  Swapping gate and up
    # would give 40 * silu(-40), about -1e-15.
    d = I = 4
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1
    w13 = np.zeros((1, 2 * I, d), np.float32)
    w13[0, :I, 0] = 40.0
    w13[0, I:, 0] = -40.0
    w2 = np.eye(d, dtype=np.float32)[None]
    y = oracle.expert_rows(x, np.zeros(1, np.int32), w13, w2, round_h=False)
    np.testing.assert_allclose(y[0], -1600.0 / (1 + math.exp(-40.0)), rtol=1e-15)


def test_ffn_zero_gate_gives_zero(oracle):
    # silu(0) = 0: with W1 = 0 every output is exactly zero whatever W3, W2.
    d, I = 8, 12
    x = RNG.standard_normal((5, d)).astype(np.float32)
    w13 = RNG.standard_normal((1, 2 * I, d)).astype(np.float32)
    w13[0, :I] = 0
    w2 = RNG.standard_normal((1, d, I)).astype(np.float32)
    y = oracle.expert_rows(x, np.zeros(5, np.int32), w13, w2, round_h=False)
    assert (y == 0).all()


def test_ffn_bf16_h_rounding(oracle):
    # With round_h, the result equals the unrounded one within the bf16
    # half-spacing bound on h: |dy_n| <= sum_i |W2[n,i]| |h_i| 2^-8.
    d, I = 16, 48
    x = bf16_bits(RNG.standard_normal((6, d)))
    w13 = bf16_bits(RNG.standard_normal((2, 2 * I, d)) * 0.5)
    w2 = bf16_bits(RNG.standard_normal((2, d, I)) * 0.5)
    re = np.array([0, 1, 1, 0, 1, 0], np.int32)
    y_r = oracle.expert_rows(x, re, w13, w2, round_h=True)
    y = oracle.expert_rows(x, re, w13, w2, round_h=False)
    xd, w13d, w2d = bits_to_f64(x), bits_to_f64(w13), bits_to_f64(w2)
    for r in range(6):
        e = re[r]
        h = silu(w13d[e, :I] @ xd[r]) * (w13d[e, I:] @ xd[r])
        bound = np.abs(w2d[e]) @ np.abs(h) * 2.0 ** -8 + 1e-12
        assert (np.abs(y_r[r] - y[r]) <= bound).all()
        # and it is exactly W2 applied to the once-rounded h
        hr = np.array([oracle.round_bf16(v) for v in h])
        np.testing.assert_allclose(y_r[r], w2d[e] @ hr, rtol=1e-12, atol=1e-12)
    assert not np.array_equal(y_r, y)


def test_ffn_linear_in_w2(oracle):
    d, I = 8, 8
    x = RNG.standard_normal((3, d)).astype(np.float32)
    w13 = RNG.standard_normal((1, 2 * I, d)).astype(np.float32)
    w2 = RNG.standard_normal((1, d, I)).astype(np.float32)
    re = np.zeros(3, np.int32)
    y1 = oracle.expert_rows(x, re, w13, w2, round_h=False)
    y4 = oracle.expert_rows(x, re, w13, w2 * 4, round_h=False)
    np.testing.assert_allclose(y4, 4 * y1, rtol=1e-14)


# ---------------------------------------------------------------- combine

def test_combine_identity_experts(oracle):
    # y = x on every row: out[t] = (sum_j w[t,j]) * x[t].
    T, k, d, E = 40, 3, 16, 6
    idx = np.stack([RNG.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, s2r, r2t = oracle.dispatch(idx, E)
    x = RNG.standard_normal((T, d)).astype(np.float32)
    y = x[r2t]
    w = RNG.uniform(0, 1, (T, k)).astype(np.float32)
    out = oracle.combine(y, s2r, w, None, T, k)
    np.testing.assert_allclose(out, w.astype(np.float64).sum(1, keepdims=True) * x, rtol=1e-12)
    sh = RNG.standard_normal((T, d)).astype(np.float32)
    out2 = oracle.combine(y, s2r, w, sh, T, k)
    np.testing.assert_allclose(out2 - out, sh, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- whole layer

def small_layer(E=8, k=2, d=24, I=40, T=50, score_fn="softmax", dtype=np.float32):
    x = RNG.standard_normal((T, d)).astype(np.float32)
    wr = (RNG.standard_normal((E, d)) * d ** -0.5).astype(np.float32)
    w13 = (RNG.standard_normal((E, 2 * I, d)) * 0.2).astype(np.float32)
    w2 = (RNG.standard_normal((E, d, I)) * 0.2).astype(np.float32)
    return x, wr, w13, w2


def test_layer_dense_masked_formulation(oracle):
    # out = sum over ALL experts of mask_e * gate_e * dense_FFN_e(x), with every
    # expert evaluated densely by numpy and the brute-force selection as mask.
    E, k, d, I, T = 6, 2, 12, 20, 30
    x, wr, w13, w2 = small_layer(E, k, d, I, T)
    idx, w, out = oracle.moe_tokens(x, E=E, k=k, w13=w13, w2=w2, w_router=wr)
    logits = (x.astype(np.float64) @ wr.astype(np.float64).T).astype(np.float32)
    ref = np.zeros((T, d))
    for t in range(T):
        sel = brute_topk(logits[t], k)
        assert list(idx[t]) == sel
        p = scipy.special.softmax(logits[t].astype(np.float64))
        for e in range(E):
            if e not in sel:
                continue
            gate = p[e] / p[sel].sum()
            xd = x[t].astype(np.float64)
            h = silu(w13[e, :I].astype(np.float64) @ xd) * (w13[e, I:].astype(np.float64) @ xd)
            ref[t] += gate * (w2[e].astype(np.float64) @ h)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_layer_stages_compose(oracle):
    # scores -> select -> gates -> dispatch -> grouped FFN -> combine equals the
    # token-by-token layer (with the shared expert and grouped sigmoid routing).
    E, k, d, I, T = 16, 4, 16, 24, 64
    x, wr, w13, w2 = small_layer(E, k, d, I, T)
    b = (RNG.standard_normal(E) * 0.1).astype(np.float32)
    w13s = (RNG.standard_normal((2 * I, d)) * 0.2).astype(np.float32)
    w2s = (RNG.standard_normal((d, I)) * 0.2).astype(np.float32)
    kw = dict(n_group=4, topk_group=2)
    idx, w, out = oracle.moe_tokens(x, E=E, k=k, w13=w13, w2=w2, w_router=wr, bias=b,
                                    score_fn=oracle.SIGMOID, routed_scale=2.5,
                                    w13_sh=w13s, w2_sh=w2s, **kw)
    sc = oracle.router_scores(x, wr, oracle.SIGMOID)
    idx2 = oracle.select(sc, k, bias=b, **kw)
    np.testing.assert_array_equal(idx, idx2)
    w2g = oracle.gates(sc, idx2, oracle.SIGMOID, 2.5)
    np.testing.assert_allclose(w, w2g, rtol=1e-15)
    counts, offsets, s2r, r2t = oracle.dispatch(idx2, E)
    yp = oracle.grouped_ffn(x[r2t], offsets, w13, w2, round_h=False)
    ysh = oracle.expert_rows(x, np.zeros(T, np.int32), w13s[None], w2s[None], round_h=False)
    # combine takes fp32 inputs, so this composition is accurate to fp32 rounding
    out2 = oracle.combine(yp.astype(np.float32), s2r, w2g.astype(np.float32),
                          ysh.astype(np.float32), T, k)
    np.testing.assert_allclose(out2, out, rtol=1e-5, atol=1e-6)


def test_layer_token_independence_and_relabeling(oracle):
    E, k, d, I, T = 8, 2, 16, 24, 20
    x, wr, w13, w2 = small_layer(E, k, d, I, T)
    _, _, out = oracle.moe_tokens(x, E=E, k=k, w13=w13, w2=w2, w_router=wr)
    # each token alone gives the same row
    for t in (0, 7, 19):
        _, _, o1 = oracle.moe_tokens(x[t:t + 1], E=E, k=k, w13=w13, w2=w2, w_router=wr)
        np.testing.assert_array_equal(o1[0], out[t])
    # relabelling experts (router rows and weights permuted together) changes nothing
    perm = RNG.permutation(E)
    _, _, outp = oracle.moe_tokens(x, E=E, k=k, w13=w13[perm], w2=w2[perm], w_router=wr[perm])
    np.testing.assert_allclose(outp, out, rtol=1e-12, atol=1e-14)


def test_layer_zero_token_experts_never_read(oracle):
    # Experts that no token selects may hold NaN weights: the output is finite
    # and equal to the output with those weights zeroed.
    E, k, d, I, T = 8, 2, 16, 24, 30
    x, wr, w13, w2 = small_layer(E, k, d, I, T)
    scores = oracle.router_scores(x, wr, oracle.SOFTMAX)
    scores[:, 5] = -60.0                        # experts 5 and 6 score far below the rest
    scores[:, 6] = -50.0
    idx, _, _ = oracle.moe_tokens(x, E=E, k=k, w13=w13, w2=w2, scores=scores)
    assert not np.isin(idx, [5, 6]).any()
    w13n, w2n = w13.copy(), w2.copy()
    w13n[[5, 6]] = np.nan
    w2n[[5, 6]] = np.nan
    _, _, out_nan = oracle.moe_tokens(x, E=E, k=k, w13=w13n, w2=w2n, scores=scores)
    w13z, w2z = w13.copy(), w2.copy()
    w13z[[5, 6]] = 0
    w2z[[5, 6]] = 0
    _, _, out_z = oracle.moe_tokens(x, E=E, k=k, w13=w13z, w2=w2z, scores=scores)
    assert np.isfinite(out_nan).all()
    np.testing.assert_array_equal(out_nan, out_z)


def test_router_scores_numpy(oracle):
    T, d, E = 40, 64, 16
    x = bf16_bits(RNG.standard_normal((T, d)))
    wr = (RNG.standard_normal((E, d)) * 0.1).astype(np.float32)
    logits = bits_to_f64(x) @ wr.astype(np.float64).T
    sc = oracle.router_scores(x, wr, oracle.SOFTMAX)
    np.testing.assert_allclose(sc, logits.astype(np.float32), rtol=1e-6, atol=1e-7)
    ss = oracle.router_scores(x, wr, oracle.SIGMOID)
    np.testing.assert_allclose(ss, scipy.special.expit(logits), rtol=1e-6)


# ---------------------------------------------------------------- workloads

def test_zipf_workload_routing_shape(oracle):
    # The imbalanced DeepSeek-V3 workload: 32 experts never chosen, heavy skew.
    cfg = inputs.CONFIGS["dsv3_zipf"].with_(T=256)
    inp = inputs.make_inputs(cfg, seed=0, experts=False)
    sc = oracle.router_scores(inputs.to_numpy(inp["x"]), inputs.to_numpy(inp["w_router"]),
                              oracle.SIGMOID)
    idx = oracle.select(sc, cfg.k, bias=inputs.to_numpy(inp["bias"]), n_group=cfg.n_group,
                        topk_group=cfg.topk_group)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    zero = (inputs.to_numpy(inp["bias"]) < -1e3)
    assert zero.sum() == 32 and (counts[zero] == 0).all()
    assert counts.max() > 8 * counts.mean()


# ---------------------------------------------------------------- worked examples
# Hand-derived values (tests/golden/worked_examples.json): each fixture carries
# the derivation of its expected numbers from the definitions.

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden",
                                    "worked_examples.json")


def _golden():
    import json
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("i", range(3))
def test_worked_routing_examples(oracle, i):
    ex = _golden()["routing"][i]
    sc = np.asarray([ex["scores"]], np.float32)
    bias = None if ex["bias"] is None else np.asarray(ex["bias"], np.float32)
    idx = oracle.select(sc, ex["k"], bias=bias, n_group=ex["n_group"], topk_group=ex["topk_group"])
    assert list(idx[0]) == ex["expect_idx"], ex["name"]
    fn = oracle.SIGMOID if ex["score_fn"] == "sigmoid" else oracle.SOFTMAX
    w = oracle.gates(sc, idx, fn, ex["routed_scale"])
    np.testing.assert_allclose(w[0], ex["expect_w"], rtol=1e-6, err_msg=ex["name"])


def test_worked_expert_example(oracle):
    ex = _golden()["expert"][0]
    x = np.asarray([ex["x"]], np.float32)
    w13 = np.asarray([ex["w13"]], np.float32)
    w2 = np.asarray([ex["w2"]], np.float32)
    sel = np.zeros(1, np.int32)
    y = oracle.expert_rows(x, sel, w13, w2, round_h=False)
    np.testing.assert_allclose(y[0], ex["expect_y"], rtol=1e-12)
    yb = oracle.expert_rows(x, sel, w13, w2, round_h=True)
    np.testing.assert_array_equal(yb[0], ex["expect_y_bf16_h"])
