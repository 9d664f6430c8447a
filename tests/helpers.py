"""Shared test helpers: tolerances and comparisons (no layer arithmetic here)."""
import numpy as np
import torch

from combine_router_gemm_gb300 import inputs

# Layer-output tolerances: bf16 workloads (max-abs and relative Frobenius
# against the oracle's result), and the fp32 workload (relative Frobenius).
BF16_MAX_ABS = 2e-2
BF16_REL_FRO = 5e-3
F32_REL_FRO = 1e-5
# Gate weights: fp32 division and sums of k terms against the oracle's double.
GATE_RTOL = 4e-6


def as_float64(a: np.ndarray) -> np.ndarray:
    """fp32 values, or raw bf16 bits (uint16), as float64."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def router_walk_range(x: np.ndarray, w_router: np.ndarray, step: int = 16) -> np.ndarray:
    """R[t,e]: the range (max - min, 0 included) of the running dot product
    sum_{i<n} x[t,i] w[e,i] over n = 0, step, 2 step, ..., d, in float64 (each
    bf16 x fp32 product is exact there).  A tensor-core MMA adds `step`
    products to an fp32 accumulator, so every accumulator value that the
    router holds -- within any K part, whatever the split -- lies in
    [-R, R]."""
    x = torch.from_numpy(as_float64(x))
    w = torch.from_numpy(as_float64(w_router))
    T, d = x.shape
    E = w.shape[0]
    nb = (d + step - 1) // step
    if nb * step != d:
        x = torch.nn.functional.pad(x, (0, nb * step - d))
        w = torch.nn.functional.pad(w, (0, nb * step - d))
    xb = x.view(T, nb, step).transpose(0, 1).contiguous()
    wb = w.view(E, nb, step).transpose(0, 1).contiguous()
    g = torch.zeros((T, E), dtype=torch.float64)
    gmax, gmin = torch.zeros_like(g), torch.zeros_like(g)
    for b in range(nb):
        g.add_(xb[b] @ wb[b].T)
        torch.maximum(gmax, g, out=gmax)
        torch.minimum(gmin, g, out=gmin)
    return (gmax - gmin).numpy()


def tc_router_bound(x: np.ndarray, w_router: np.ndarray, sigmoid: bool) -> np.ndarray:
    """Per-element bound [T,E] on |router score from the tensor cores - the
    oracle's score|, from the measured accumulator range R (router_walk_range)
    instead of an assumed magnitude.

    The weight is split exactly into three bf16 terms and every product with
    a bf16 activation is exact, so the error comes from rounding fp32 sums:
    at most one ulp (2^-23 |value| <= 2^-23 R) per MMA of the largest term
    over its d/16 MMAs (the smaller terms' accumulators are 2^-8 and 2^-16 of
    it), plus at most six more half-ulp roundings (the three terms' sum, up to
    eight K parts added, the oracle's own fp32 rounding).  A sigmoid score
    moves by at most a quarter of its logit's error, plus the few ulps of
    the fp32 sigmoid itself."""
    d = x.shape[1]
    R = router_walk_range(x, w_router)
    logit = ((d + 15) // 16 + 6) * 2.0 ** -23 * R * (1 + 2.0 ** -7)
    if sigmoid:
        return logit / 4 + 2.0 ** -21
    return logit


def np_(t):
    return inputs.to_numpy(t)


def rel_fro(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (den if den > 0 else 1.0)


def assert_bf16_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    mx = np.abs(got - ref).max() if got.size else 0.0
    rf = rel_fro(got, ref)
    assert mx <= BF16_MAX_ABS and rf <= BF16_REL_FRO, f"{what}: max-abs {mx:.3e}, rel-fro {rf:.3e}"
    return mx, rf


def near_tie_tokens(scores: np.ndarray, bias, k: int, n_group: int = 1, topk_group: int = 1,
                    rel: float = 1e-5, abs_margin: float = 0.0):
    """Tokens whose selection is decided by a margin smaller than ``rel``
    (relative) plus twice ``abs_margin`` (the score error bound of the router
    that made the other tensor): two consecutive keys among the k+1 largest
    eligible ones (the k-th vs (k+1)-th decides which experts; the others the
    order of the output slots), or (group-limited routing) the topk_group-th
    vs next group score.  Between two score tensors that differ only by
    rounding, the choice or its order may legitimately flip on exactly these
    tokens."""
    key = scores.astype(np.float64) + (0 if bias is None else bias.astype(np.float64))
    T, E = key.shape
    amb = np.zeros(T, bool)
    if n_group > 1:
        gs = E // n_group
        top2 = -np.sort(-key.reshape(T, n_group, gs), axis=2)[:, :, :2].sum(2)
        order = np.argsort(-top2, axis=1, kind="stable")
        g_sorted = np.take_along_axis(top2, order, 1)
        if topk_group < n_group:
            gap = np.abs(g_sorted[:, topk_group - 1] - g_sorted[:, topk_group])
            amb |= gap <= rel * np.maximum(1.0, np.abs(g_sorted[:, topk_group - 1])) + 4 * abs_margin
        keep = np.zeros((T, n_group), bool)
        np.put_along_axis(keep, order[:, :topk_group], True, 1)
        key = np.where(np.repeat(keep, gs, axis=1), key, -np.inf)
    # consecutive eligible keys among the first k+1 in descending order: the
    # k-th against the (k+1)-th decides the set, the others the order of the
    # k output slots
    srt = -np.sort(-key, axis=1)[:, : k + 1]
    for j in range(min(k, srt.shape[1] - 1)):
        a, b = srt[:, j], srt[:, j + 1]
        gap = np.where(np.isfinite(b), np.abs(a - b), np.inf)
        amb |= gap <= rel * np.maximum(1.0, np.abs(a)) + 2 * abs_margin
    return amb


def coverage_tokens(offsets: np.ndarray, row_to_token: np.ndarray, T: int, n_min: int,
                    seed: int, boundaries=(128, 160, 256)) -> np.ndarray:
    """Sorted token indices to check element by element: for every expert
    with rows, the tokens of its segment's first and last row and of the
    first row past each token-tile boundary the grouped GEMMs use (so that
    every active expert, every ragged tail and every second token tile is
    covered), then seeded random tokens up to at least n_min."""
    toks = set()
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        n = b - a
        if n == 0:
            continue
        for p in {0, n - 1, *[q for q in boundaries if q < n]}:
            toks.add(int(row_to_token[a + p]))
    rng = np.random.default_rng(seed)
    for t in rng.permutation(T):
        if len(toks) >= n_min:
            break
        toks.add(int(t))
    return np.array(sorted(toks), dtype=np.int64)


def cuda_i32(shape, dev="cuda"):
    return torch.empty(shape, dtype=torch.int32, device=dev)


def cuda_f32(shape, dev="cuda"):
    return torch.empty(shape, dtype=torch.float32, device=dev)
