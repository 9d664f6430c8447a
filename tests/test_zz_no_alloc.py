"""moe_dispatch_noalloc: the workspace-free dispatch for callers that may not
allocate device memory while they run (fixed memory pools, hosted plug-ins).

Its outputs must equal those of moe_dispatch (bit-exact: integer and byte
work), on two calls in a row with different inputs, since every call reuses
the same fixed scratch array inside the library.  This file is collected last
and also passes on its own in a fresh process.
"""
import pytest
import torch

from combine_router_gemm_gb300 import binding as B

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


def test_noalloc_matches_moe_dispatch_twice():
    # a large call then a smaller one: the second must not see the first's scratch
    for T, k, E, d, seed in [(16384, 8, 256, 64, 1), (1000, 2, 8, 128, 2)]:
        idx, x = _inputs(T, k, E, d, seed)
        ref = _with_workspace(idx, x, E)
        got = _without_workspace(idx, x, E)
        for name in ref:
            assert torch.equal(got[name], ref[name]), (T, name)


def test_noalloc_refuses_sizes_beyond_its_array():
    T, k, E = B.DISPATCH_NOALLOC_MAX_SLOTS // 8 + 1, 8, 256
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    o = _outputs(1, 1, E, 8)
    with pytest.raises(B.MoEError) as e:
        B.moe_dispatch_noalloc(idx, None, E, o["counts"], o["offsets"], o["slot_to_row"],
                               o["row_to_token"], None)
    assert e.value.status == B.ERR_UNSUPPORTED
