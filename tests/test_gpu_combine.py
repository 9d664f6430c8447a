"""Gate-weighted combine on the GPU (moe_combine) against the oracle."""
import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from helpers import cuda_f32, np_

pytestmark = pytest.mark.gpu


def perm_maps(T, k, seed):
    g = torch.Generator()
    g.manual_seed(seed)
    s2r = torch.randperm(T * k, generator=g).to(torch.int32)
    return s2r


@pytest.mark.parametrize("T,k,d,shared", [(4096, 8, 7168, True), (300, 2, 4096, False),
                                          (1, 1, 8, True), (77, 5, 40, False)])
def test_combine(oracle, T, k, d, shared):
    g = torch.Generator(device="cuda")
    g.manual_seed(T + d)
    y = torch.randn((T * k, d), generator=g, device="cuda")
    w = torch.rand((T, k), generator=g, device="cuda")
    sh = torch.randn((T, d), generator=g, device="cuda") if shared else None
    s2r = perm_maps(T, k, T).cuda()
    out = cuda_f32((T, d))
    B.moe_combine(y, s2r, w, sh, out)
    torch.cuda.synchronize()
    ref = oracle.combine(np_(y), np_(s2r), np_(w), np_(sh), T, k)
    np.testing.assert_allclose(np_(out), ref, rtol=2e-6, atol=2e-6)


def test_combine_identity_experts(oracle):
    # y rows are the tokens' own rows: out[t] = (sum_j w[t,j]) * x[t].
    T, k, d = 500, 4, 256
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    x = torch.randn((T, d), generator=g, device="cuda")
    s2r = perm_maps(T, k, 2).cuda()
    r2t = torch.empty(T * k, dtype=torch.long, device="cuda")
    r2t[s2r.long()] = torch.arange(T * k, device="cuda") // k
    y = x[r2t].contiguous()
    w = torch.rand((T, k), generator=g, device="cuda")
    out = cuda_f32((T, d))
    B.moe_combine(y, s2r, w, None, out)
    ref = w.double().sum(1, keepdim=True) * x.double()
    np.testing.assert_allclose(np_(out), np_(ref), rtol=1e-6, atol=1e-6)


def test_combine_out_of_range_row_is_visible():
    """A slot_to_row entry outside y poisons that token's output row (NaN) and
    no other; nothing outside y is read."""
    T, k, d = 64, 8, 256
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    y = torch.randn((T * k, d), generator=g, device="cuda")
    w = torch.rand((T, k), generator=g, device="cuda")
    s2r = perm_maps(T, k, 5).cuda()
    s2r[3 * k + 2] = T * k + 7  # token 3, slot 2
    s2r[9 * k] = -1             # token 9, slot 0
    out = cuda_f32((T, d))
    B.moe_combine(y, s2r, w, None, out)
    torch.cuda.synchronize()
    bad = torch.isnan(out).any(1)
    assert bad[3] and bad[9]
    assert not bad[[t for t in range(T) if t not in (3, 9)]].any()
