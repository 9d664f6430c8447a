"""moe_dispatch_noalloc: the workspace-free dispatch for callers that may not
allocate device memory while they run (fixed memory pools, hosted plug-ins).

Its outputs must equal those of moe_dispatch and of the oracle's stable
counting sort (bit-exact: integer and byte work), on calls in a row with
different inputs, since every call reuses the same fixed scratch array inside
the library.  This file is collected last
and also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from helpers import np_

# error-word bit of an expert index outside [0, E) (moe_check_error's detail)
ERR_BAD_INDEX = 1 << 8

pytestmark = pytest.mark.gpu


def _inputs(T, k, E, d, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    w = torch.arange(1, E + 1, dtype=torch.float32, device="cuda") ** -1.1
    idx = torch.multinomial(w.expand(T, E), k, replacement=False, generator=g).to(torch.int32)
    x = torch.randn((T, d), generator=g, device="cuda").to(torch.bfloat16)
    return idx, x


def _outputs(T, k, E, d):
    S = T * k
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts=torch.full((E,), -7, **i32), offsets=torch.full((E + 1,), -7, **i32),
                slot_to_row=torch.full((S,), -7, **i32), row_to_token=torch.full((S,), -7, **i32),
                x_perm=torch.zeros((S, d), dtype=torch.bfloat16, device="cuda"))


def _with_workspace(idx, x, E):
    T, k = idx.shape
    o = _outputs(T, k, E, x.shape[1])
    ws = torch.empty(B.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    B.moe_dispatch(idx, x, E, o["counts"], o["offsets"], o["slot_to_row"], o["row_to_token"],
                   o["x_perm"], ws)
    rc, detail = B.moe_check_error(ws)
    assert rc == B.OK, detail
    return o


def _without_workspace(idx, x, E):
    T, k = idx.shape
    o = _outputs(T, k, E, x.shape[1])
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.moe_dispatch_noalloc(idx, x, E, o["counts"], o["offsets"], o["slot_to_row"],
                           o["row_to_token"], o["x_perm"], device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return o


def _check_against_oracle(oracle, got, idx, x, E):
    counts, offsets, s2r, r2t = oracle.dispatch(np_(idx), E)
    for name, ref in (("counts", counts), ("offsets", offsets), ("slot_to_row", s2r),
                      ("row_to_token", r2t)):
        np.testing.assert_array_equal(np_(got[name]), ref, err_msg=name)
    assert torch.equal(got["x_perm"], x[torch.from_numpy(r2t).long().cuda()])


def test_noalloc_matches_moe_dispatch_twice(oracle):
    # a large call then a smaller one: the second must not see the first's
    # scratch; then the largest expert count at the largest slot count (the
    # scratch array at its fullest)
    for T, k, E, d, seed in [(16384, 8, 256, 64, 1), (1000, 2, 8, 128, 2),
                             (B.DISPATCH_NOALLOC_MAX_SLOTS // 8, 8, 1024, 16, 3)]:
        idx, x = _inputs(T, k, E, d, seed)
        ref = _with_workspace(idx, x, E)
        got = _without_workspace(idx, x, E)
        for name in ref:
            assert torch.equal(got[name], ref[name]), (T, name)
        _check_against_oracle(oracle, got, idx, x, E)


def test_noalloc_error_word_and_empty_batch(oracle):
    """A bad expert index (made on the host, range-checked by the kernel: no
    out-of-bounds access) sets the error bit in device_error; the next clean
    call reports 0 again (the shared error word is cleared per call); an
    empty batch writes zero counts and offsets."""
    T, k, E, d = 300, 4, 16, 32
    idx, x = _inputs(T, k, E, d, 4)
    bad = idx.clone()
    bad[123, 2] = E
    o = _outputs(T, k, E, d)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.moe_dispatch_noalloc(bad, x, E, o["counts"], o["offsets"], o["slot_to_row"],
                           o["row_to_token"], o["x_perm"], device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ERR_BAD_INDEX
    got = _without_workspace(idx, x, E)  # asserts a zero error word
    _check_against_oracle(oracle, got, idx, x, E)
    empty = torch.empty((0, k), dtype=torch.int32, device="cuda")
    o = _outputs(0, k, E, d)
    B.moe_dispatch_noalloc(empty, torch.empty((0, d), dtype=torch.bfloat16, device="cuda"), E,
                           o["counts"], o["offsets"], None, None,
                           torch.empty((0, d), dtype=torch.bfloat16, device="cuda"),
                           device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert (o["counts"] == 0).all() and (o["offsets"] == 0).all()


def test_noalloc_refuses_sizes_beyond_its_array():
    T, k, E = B.DISPATCH_NOALLOC_MAX_SLOTS // 8 + 1, 8, 256
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    o = _outputs(1, 1, E, 8)
    with pytest.raises(B.MoEError) as e:
        B.moe_dispatch_noalloc(idx, None, E, o["counts"], o["offsets"], o["slot_to_row"],
                               o["row_to_token"], None)
    assert e.value.status == B.ERR_UNSUPPORTED
