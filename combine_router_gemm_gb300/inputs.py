"""Seeded synthetic inputs for the MoE layer: shapes, distributions, generators.

This module holds no arithmetic of the layer itself -- only workload shapes and
random draws -- so that it can feed both the CUDA path and the CPU oracle.

Workloads (the pages -- "CUCo: An Agentic Framework for Compute and
Communication Co-design", abstract and Table 4 -- name a DeepSeek-V3 MoE layer
under imbalanced sparse routing but give no shapes; the shapes below are the
public Mixtral-8x7B and DeepSeek-V3 layer shapes):

==============  =====  ====  ===  =  =====  =======  =====  ===================
name              T      d    E   k    I    shared   dtype  routing
==============  =====  ====  ===  =  =====  =======  =====  ===================
tiny_fp32          64   128    8  2    256     -      f32   softmax, top-2
mixtral_bf16     4096  4096    8  2  14336     -      bf16  softmax, top-2
dsv3_prefill     4096  7168  256  8   2048   2048     bf16  sigmoid+bias, groups
dsv3_decode       128  7168  256  8   2048   2048     bf16  as dsv3_prefill
dsv3_zipf       16384  7168  256  8   2048   2048     bf16  Zipf(1.2) bias, 32 empty
==============  =====  ====  ===  =  =====  =======  =====  ===================

DeepSeek-V3 routing: 8 contiguous groups of 32 experts, keep the best 4 groups,
top-8 experts, gate weights normalised over the 8 then scaled by 2.5.

Every tensor has its own generator seeded ``seed * 1000 + tensor_id`` so that
draws do not depend on generation order.  Values are drawn in fp32 and cast to
bf16 with round-to-nearest-even.  ``N(0, s)`` means standard deviation ``s``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from statistics import NormalDist

import torch

# tensor ids for per-tensor seeding
_TID = {"x": 1, "w_router": 2, "bias": 3, "w13": 4, "w2": 5, "w13_sh": 6, "w2_sh": 7,
        "scores": 8, "zipf_perm": 9}


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    dtype: str = "bf16"            # "f32" or "bf16": activations and expert weights
    score_fn: str = "softmax"      # "softmax" (compare logits) or "sigmoid"
    n_group: int = 1
    topk_group: int = 1
    routed_scale: float = 1.0
    shared_I: int = 0              # 0: no shared expert
    x_std: float = 1.0
    router_std: float = 0.02
    expert_std: float = 0.02
    bias: str = "none"             # "none", "normal" or "zipf"
    bias_std: float = 0.01
    zipf_s: float = 1.2
    zipf_zero: int = 32

    @property
    def S(self) -> int:
        """Number of (token, slot) pairs, T*k."""
        return self.T * self.k

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


_DSV3 = dict(d=7168, E=256, k=8, I=2048, dtype="bf16", score_fn="sigmoid", n_group=8,
             topk_group=4, routed_scale=2.5, shared_I=2048, bias="normal")

CONFIGS = {
    "tiny_fp32": MoEConfig("tiny_fp32", T=64, d=128, E=8, k=2, I=256, dtype="f32",
                           router_std=128 ** -0.5),
    "mixtral_bf16": MoEConfig("mixtral_bf16", T=4096, d=4096, E=8, k=2, I=14336, dtype="bf16"),
    "dsv3_prefill": MoEConfig("dsv3_prefill", T=4096, **_DSV3),
    "dsv3_decode": MoEConfig("dsv3_decode", T=128, **_DSV3),
    "dsv3_zipf": MoEConfig("dsv3_zipf", T=16384, **{**_DSV3, "bias": "zipf"}),
    # DeepSeek-V3 layer shapes with 32 experts and 512 tokens: the same ~128
    # tokens per expert as dsv3_prefill in 1/8 of the memory (profiling case)
    "dsv3_prefill_e32": MoEConfig("dsv3_prefill_e32", T=512, **{**_DSV3, "E": 32}),
    # the Zipf-imbalanced layer with 32 experts (4 of them empty) and 2048
    # tokens: experts of ~250 to ~2000 rows, tensor-bound grouped GEMMs as in
    # dsv3_zipf, in about 4 GB (profiling case)
    "dsv3_zipf_e32": MoEConfig("dsv3_zipf_e32", T=2048,
                               **{**_DSV3, "E": 32, "bias": "zipf", "zipf_zero": 4}),
    # DeepSeek-V3 prefill routing, dispatch and combine at full size (4096
    # tokens, 256 experts, d = 7168) with narrow experts (I = 128): the
    # router, top-k, dispatch and combine kernels see the prefill shapes in
    # about 3.5 GB (profiling case)
    "dsv3_prefill_i128": MoEConfig("dsv3_prefill_i128", T=4096,
                                   **{**_DSV3, "I": 128, "shared_I": 128}),
}


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _TID[name])
    return g


def _normal(shape, std, g, device, dtype):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(dtype)


def _expert_weights(E, rows, cols, std, g, device, dtype):
    """[E, rows, cols], drawn one expert at a time to bound fp32 temporaries."""
    w = torch.empty((E, rows, cols), dtype=dtype, device=device)
    for e in range(E):
        w[e] = _normal((rows, cols), std, g, device, dtype)
    return w


def zipf_bias(cfg: MoEConfig, seed: int = 0) -> torch.Tensor:
    """Per-expert selection bias that skews expert load towards Zipf(s).

    Construction (a distribution model, not the routing itself): ranks 1..A
    (A = E - zipf_zero) are assigned to experts by a seeded permutation and get
    target selection probabilities p_r = k r^-s / sum_r' r'^-s, capped at 0.98
    since a token picks an expert at most once.  Under the stated input
    distributions a router logit is N(0, sigma^2), sigma = x_std * router_std *
    sqrt(d), so a sigmoid score has quantile function
    F^-1(q) = 1 / (1 + exp(-sigma * Phi^-1(q))).  An expert is taken when its
    biased score clears a common threshold (set to 0); bias b_r = -F^-1(1 - p_r)
    makes that happen with probability p_r.  The zipf_zero lowest ranks get
    bias -1e4 and so are never chosen.  Group-limited selection and per-token
    thresholds make the achieved load only approximately Zipf.
    """
    E, k = cfg.E, cfg.k
    active = E - cfg.zipf_zero
    perm = torch.randperm(E, generator=_gen(seed, "zipf_perm", "cpu"))
    sigma = cfg.x_std * cfg.router_std * math.sqrt(cfg.d)
    ranks = [r ** -cfg.zipf_s for r in range(1, active + 1)]
    total = sum(ranks)
    nd = NormalDist()
    bias = torch.full((E,), -1.0e4, dtype=torch.float32)
    for r in range(active):
        p = min(k * ranks[r] / total, 0.98)
        q = 1.0 - p
        bias[perm[r]] = -1.0 / (1.0 + math.exp(-sigma * nd.inv_cdf(q)))
    return bias


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu", experts: bool = True) -> dict:
    """All layer inputs for ``cfg`` on ``device``.

    Keys: x [T,d], w_router [E,d] fp32, bias [E] fp32 or None, w13 [E,2I,d]
    (gate rows 0..I-1 then up rows I..2I-1), w2 [E,d,I], w13_sh [2I_s,d] and
    w2_sh [d,I_s] or None.  Activations/expert weights are cfg.dtype.  With
    ``experts=False`` the expert weights are left out (None).
    """
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    out = {
        "x": _normal((cfg.T, cfg.d), cfg.x_std, _gen(seed, "x", device), device, dt),
        "w_router": _normal((cfg.E, cfg.d), cfg.router_std, _gen(seed, "w_router", device),
                            device, torch.float32),
        "w13": None,
        "w2": None,
        "bias": None,
        "w13_sh": None,
        "w2_sh": None,
    }
    if experts:
        out["w13"] = _expert_weights(cfg.E, 2 * cfg.I, cfg.d, cfg.expert_std,
                                     _gen(seed, "w13", device), device, dt)
        out["w2"] = _expert_weights(cfg.E, cfg.d, cfg.I, cfg.expert_std,
                                    _gen(seed, "w2", device), device, dt)
    if cfg.bias == "normal":
        out["bias"] = _normal((cfg.E,), cfg.bias_std, _gen(seed, "bias", device), device,
                              torch.float32)
    elif cfg.bias == "zipf":
        out["bias"] = zipf_bias(cfg, seed).to(device)
    if cfg.shared_I and experts:
        out["w13_sh"] = _normal((2 * cfg.shared_I, cfg.d), cfg.expert_std,
                                _gen(seed, "w13_sh", device), device, dt)
        out["w2_sh"] = _normal((cfg.d, cfg.shared_I), cfg.expert_std,
                               _gen(seed, "w2_sh", device), device, dt)
    return out


def make_scores(T: int, E: int, score_fn: str, seed: int = 0, quant_bits: int | None = None,
                device="cpu") -> torch.Tensor:
    """A synthetic fp32 score tensor [T,E] for routing-only checks.

    softmax: logits ~ N(0,1); sigmoid: scores ~ U(0,1).  With ``quant_bits``
    every score is a multiple of 2^-quant_bits, so that many ties occur.
    """
    g = _gen(seed, "scores", device)
    s = torch.empty((T, E), dtype=torch.float32, device=device)
    if score_fn == "softmax":
        s.normal_(0.0, 1.0, generator=g)
    else:
        s.uniform_(0.0, 1.0, generator=g)
    if quant_bits is not None:
        q = float(2 ** quant_bits)
        s = torch.round(s * q) / q
    return s


def to_numpy(t: torch.Tensor | None):
    """Host numpy copy; bf16 becomes its raw uint16 bits (no value conversion)."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
