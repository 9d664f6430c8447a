"""Dispatch on the GPU (moe_dispatch) against the oracle: bit-exact.

counts, offsets, slot_to_row and row_to_token must equal the oracle's stable
counting sort, and x_perm must be x gathered by row_to_token, byte for byte.
"""
import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from helpers import cuda_i32, np_

pytestmark = pytest.mark.gpu


def run_dispatch(idx: torch.Tensor, x: torch.Tensor | None, E: int):
    T, k = idx.shape
    S = T * k
    d = x.shape[1] if x is not None else 8
    counts, offsets = cuda_i32(E), cuda_i32(E + 1)
    s2r, r2t = cuda_i32(S), cuda_i32(S)
    xp = torch.empty((S, d), dtype=x.dtype, device="cuda") if x is not None else None
    ws = torch.empty(B.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    B.moe_dispatch(idx, x, E, counts, offsets, s2r, r2t, xp, ws)
    rc, detail = B.moe_check_error(ws)
    return rc, detail, counts, offsets, s2r, r2t, xp


def distinct_topk(T, E, k, seed, probs=None):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    p = torch.ones(E, device="cuda") if probs is None else probs.to("cuda")
    return torch.multinomial(p.expand(T, E), k, replacement=False, generator=g).to(torch.int32)


CASES = [
    # T, k, E, d, dtype, skew
    (4096, 2, 8, 4096, torch.bfloat16, None),      # Mixtral shape
    (4096, 8, 256, 7168, torch.bfloat16, None),    # DeepSeek-V3 prefill shape
    (128, 8, 256, 7168, torch.bfloat16, None),     # decode: most experts get 0-4 rows
    (16384, 8, 256, 512, torch.bfloat16, "zipf"),  # imbalanced, 32 empty experts
    (64, 2, 8, 128, torch.float32, None),          # fp32 rows
    (1, 1, 1, 8, torch.bfloat16, None),            # single slot
    (5000, 3, 1000, 64, torch.bfloat16, "zipf"),   # many blocks, odd k
    (777, 1, 5, 24, torch.float32, None),
]


@pytest.mark.parametrize("T,k,E,d,dtype,skew", CASES)
def test_dispatch_bit_exact(oracle, T, k, E, d, dtype, skew):
    probs = None
    if skew == "zipf":
        r = torch.arange(1, E + 1, dtype=torch.float64) ** -1.2
        r[-min(32, E // 4):] = 0  # the lowest ranks receive nothing
        probs = r.float()
    idx = distinct_topk(T, E, k, seed=T * 31 + E, probs=probs)
    g = torch.Generator(device="cuda")
    g.manual_seed(d)
    x = torch.randn((T, d), generator=g, device="cuda").to(dtype)
    rc, detail, counts, offsets, s2r, r2t, xp = run_dispatch(idx, x, E)
    assert rc == B.OK, detail
    rc_counts, rc_offsets, rc_s2r, rc_r2t = oracle.dispatch(np_(idx), E)
    np.testing.assert_array_equal(np_(counts), rc_counts)
    np.testing.assert_array_equal(np_(offsets), rc_offsets)
    np.testing.assert_array_equal(np_(s2r), rc_s2r)
    np.testing.assert_array_equal(np_(r2t), rc_r2t)
    assert torch.equal(xp, x[torch.from_numpy(rc_r2t).long().cuda()])
    if skew == "zipf":
        assert (rc_counts == 0).sum() >= min(32, E // 4)


def test_dispatch_index_maps_only(oracle):
    idx = distinct_topk(300, 16, 4, seed=5)
    rc, _, counts, offsets, s2r, r2t, _ = run_dispatch(idx, None, 16)
    assert rc == B.OK
    c, o, a, b = oracle.dispatch(np_(idx), 16)
    np.testing.assert_array_equal(np_(s2r), a)
    np.testing.assert_array_equal(np_(r2t), b)


def test_dispatch_out_of_range_index_is_flagged():
    # The host cannot see device-side indices; the count kernel skips an index
    # outside [0, E), flags it in the error word and the permute stage is
    # skipped.  No out-of-bounds access happens.
    idx = distinct_topk(100, 8, 2, seed=9)
    idx[17, 1] = 8
    rc, detail, *_ = run_dispatch(idx, torch.zeros((100, 16), dtype=torch.bfloat16, device="cuda"), 8)
    assert rc == B.ERR_DEVICE_INPUT and detail != 0


def test_dispatch_empty_batch():
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    rc, _, counts, offsets, *_ = run_dispatch(idx, torch.empty((0, 8), dtype=torch.bfloat16, device="cuda"), 4)
    assert rc == B.OK
    assert (np_(counts) == 0).all() and (np_(offsets) == 0).all()
