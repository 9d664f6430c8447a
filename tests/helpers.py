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


def tc_router_atol(d: int, magnitude: float = 4.0) -> float:
    """Error bound of router scores from the tensor cores: the fp32 accumulator
    is truncated once per MMA (16 products), so over d/16 MMAs with partial
    sums up to `magnitude` the error is at most (d/16) * 2^-23 * magnitude
    (the split-weight terms have accumulators of their own, far smaller)."""
    return (d / 16) * 2.0 ** -23 * magnitude


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
    that made the other tensor): the k-th vs (k+1)-th eligible key, or
    (group-limited routing) the topk_group-th vs next group score.  Between two
    score tensors that differ only by rounding, the choice may legitimately
    flip on exactly these tokens."""
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
    srt = -np.sort(-key, axis=1)
    if srt.shape[1] > k and np.isfinite(srt[:, k]).any():
        nxt = srt[:, k]
        gap = np.where(np.isfinite(nxt), np.abs(srt[:, k - 1] - nxt), np.inf)
        amb |= gap <= rel * np.maximum(1.0, np.abs(srt[:, k - 1])) + 2 * abs_margin
    return amb


def cuda_i32(shape, dev="cuda"):
    return torch.empty(shape, dtype=torch.int32, device=dev)


def cuda_f32(shape, dev="cuda"):
    return torch.empty(shape, dtype=torch.float32, device=dev)
