"""Grouped SwiGLU FFN on the GPU (moe_grouped_ffn) against the oracle.

bf16 runs on the tcgen05 tensor cores: compared with the oracle's double
result (h rounded to bf16 once) at the bf16 layer tolerances.  fp32 runs on
the CUDA cores: relative Frobenius 1e-5.  Segments are ragged, span several
256-token tiles, include empty experts, and feature/K sizes include tails.
"""
import numpy as np
import pytest
import torch

from combine_router_gemm_gb300 import binding as B
from helpers import F32_REL_FRO, assert_bf16_close, cuda_f32, np_, rel_fro

pytestmark = pytest.mark.gpu


def make_case(E, d, I, counts, dtype, seed, wstd=0.06, extra_rows=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    counts = torch.tensor(counts, dtype=torch.int64)
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    rows = int(offsets[-1]) + extra_rows
    x = torch.randn((rows, d), generator=g, device="cuda").to(dtype)
    w13 = (torch.randn((E, 2 * I, d), generator=g, device="cuda") * wstd).to(dtype)
    w2 = (torch.randn((E, d, I), generator=g, device="cuda") * wstd).to(dtype)
    return x, offsets.cuda(), w13, w2


def run_ffn(x, offsets, w13, w2):
    rows, d = x.shape
    I = w2.shape[2]
    dt = B.BF16 if x.dtype == torch.bfloat16 else B.F32
    y = torch.full((rows, d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.moe_grouped_ffn_workspace_size(rows, d, I, dt), dtype=torch.uint8,
                     device="cuda")
    B.moe_grouped_ffn(x, offsets, w13, w2, y, ws)
    rc, detail = B.moe_check_error(ws)
    assert rc == B.OK, detail
    return y


CASES = [
    # E, d, I, counts
    (4, 128, 128, [1, 0, 300, 17]),                 # 300 rows: two token tiles
    (8, 256, 256, [5, 40, 0, 0, 256, 257, 3, 100]),  # exact tile boundary 256 / 257
    (3, 192, 136, [33, 64, 511]),                    # I tail (136 = 128 + 8), d = 3 K-blocks
    (2, 200, 264, [16, 15]),                         # K tail (200 = 3*64 + 8), N tail
    (1, 512, 384, [1000]),                           # dense, many tiles
    (16, 64, 128, [0] * 7 + [9] + [0] * 8),          # one active expert of 16
]


@pytest.mark.parametrize("E,d,I,counts", CASES)
def test_grouped_ffn_bf16(oracle, E, d, I, counts):
    x, offsets, w13, w2 = make_case(E, d, I, counts, torch.bfloat16, seed=E * 1000 + d)
    y = run_ffn(x, offsets, w13, w2)
    torch.cuda.synchronize()
    n = int(offsets[-1])
    ref = oracle.grouped_ffn(np_(x), np_(offsets), np_(w13), np_(w2), round_h=True)
    assert_bf16_close(np_(y)[:n], ref, f"E={E} d={d} I={I}")
    assert rel_fro(np_(y)[:n], ref) < 2e-3


def test_grouped_ffn_rows_past_offsets_untouched(oracle):
    x, offsets, w13, w2 = make_case(3, 128, 128, [10, 0, 20], torch.bfloat16, seed=3,
                                    extra_rows=50)
    y = run_ffn(x, offsets, w13, w2)
    assert torch.isnan(y[30:]).all()


def test_grouped_ffn_empty_experts_never_read(oracle):
    # NaN weights on experts without rows must not reach the output.
    E, d, I = 6, 128, 128
    counts = [40, 0, 70, 0, 0, 5]
    x, offsets, w13, w2 = make_case(E, d, I, counts, torch.bfloat16, seed=11)
    w13n, w2n = w13.clone(), w2.clone()
    for e in (1, 3, 4):
        w13n[e] = float("nan")
        w2n[e] = float("nan")
    y = run_ffn(x, offsets, w13n, w2n)
    y0 = run_ffn(x, offsets, w13, w2)
    assert torch.isfinite(y[:115]).all()
    assert torch.equal(y[:115], y0[:115])


@pytest.mark.parametrize("E,d,I,counts", [(8, 128, 256, [20, 0, 7, 33, 1, 0, 50, 17]),
                                           (2, 40, 24, [3, 9])])
def test_grouped_ffn_f32(oracle, E, d, I, counts):
    x, offsets, w13, w2 = make_case(E, d, I, counts, torch.float32, seed=7, wstd=0.1)
    y = run_ffn(x, offsets, w13, w2)
    n = int(offsets[-1])
    ref = oracle.grouped_ffn(np_(x), np_(offsets), np_(w13), np_(w2), round_h=False)
    assert rel_fro(np_(y)[:n], ref) <= F32_REL_FRO


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_grouped_ffn_bad_offsets_flagged(dtype):
    # Non-monotone device offsets: the kernels do no work and flag the input
    # (tensor-core path and fp32 CUDA-core path alike).
    x, offsets, w13, w2 = make_case(2, 128, 128, [10, 10], dtype, seed=1)
    offsets[1] = 15
    offsets[2] = 12
    rows, d = x.shape
    y = cuda_f32((rows, d))
    code = B.BF16 if dtype == torch.bfloat16 else B.F32
    ws = torch.empty(B.moe_grouped_ffn_workspace_size(rows, d, 128, code), dtype=torch.uint8,
                     device="cuda")
    B.moe_grouped_ffn(x, offsets, w13, w2, y, ws)
    rc, detail = B.moe_check_error(ws)
    assert rc == B.ERR_DEVICE_INPUT and detail != 0


def torch_pack(w, pairs):
    """The tile-major layouts written out with torch view/permute."""
    if w.dim() == 2:
        return torch_pack(w[None], pairs)[0]
    E, R, K = w.shape
    if pairs:
        t = w.view(E, R // 256, 2, 128, K // 64, 64).permute(0, 1, 4, 2, 3, 5)
    else:
        t = w.view(E, R // 128, 128, K // 64, 64).permute(0, 1, 3, 2, 4)
    return t.contiguous().view(E, R, K)


@pytest.mark.parametrize("E,d,I", [(3, 256, 128), (1, 512, 384), (2, 768, 256)])
def test_pack_expert_weights_layout(E, d, I):
    g = torch.Generator(device="cuda")
    g.manual_seed(E + d)
    w13 = torch.randn((E, 2 * I, d), generator=g, device="cuda").to(torch.bfloat16)
    w2 = torch.randn((E, d, I), generator=g, device="cuda").to(torch.bfloat16)
    p13, p2 = torch.empty_like(w13), torch.empty_like(w2)
    B.moe_pack_expert_weights(w13, w2, p13, p2)
    torch.cuda.synchronize()
    assert torch.equal(p13, torch_pack(w13, False))
    assert torch.equal(p2, torch_pack(w2, True))
    # 2-D shared-expert weights
    s13, s2 = torch.empty_like(w13[0]), torch.empty_like(w2[0])
    B.moe_pack_expert_weights(w13[0], w2[0], s13, s2)
    torch.cuda.synchronize()
    assert torch.equal(s13, torch_pack(w13[0], False))
    assert torch.equal(s2, torch_pack(w2[0], True))


def test_grouped_ffn_bf16_mixed_classes_wide_tiles(oracle):
    """Many experts, 256-row token tiles (at least 384 rows per expert on
    average): compute-class experts (at least 128 rows) interleaved with
    weight-streaming ones of ragged sizes, empty experts between them."""
    E, d, I = 64, 256, 128
    rng = np.random.default_rng(5)
    counts = [2300] * 10 + [int(c) for c in rng.integers(1, 128, 40)] + [0] * 14
    counts = [counts[i] for i in rng.permutation(E)]
    assert sum(counts) >= 384 * E  # the wide-tile launch configuration
    x, offsets, w13, w2 = make_case(E, d, I, counts, torch.bfloat16, seed=77)
    y = run_ffn(x, offsets, w13, w2)
    torch.cuda.synchronize()
    n = int(offsets[-1])
    ref = oracle.grouped_ffn(np_(x), np_(offsets), np_(w13), np_(w2), round_h=True)
    assert_bf16_close(np_(y)[:n], ref, "mixed classes")


def test_grouped_ffn_bf16_two_pair_clusters_ragged(oracle):
    """At least 768 rows per expert on average: the down projection runs on
    clusters of two CTA pairs (1024 output features per cluster, the token
    tile multicast to both pairs).  d = 1160 leaves the second feature tile
    with 136 valid features (the second pair has none), and the token tiles
    end ragged (900 = 3*256 + 132, 1700 = 6*256 + 164) beside an empty
    expert; d is also a K tail for gate/up (18 K-blocks + 8)."""
    E, d, I, counts = 3, 1160, 320, [900, 0, 1700]
    assert sum(counts) >= 768 * E
    x, offsets, w13, w2 = make_case(E, d, I, counts, torch.bfloat16, seed=31)
    y = run_ffn(x, offsets, w13, w2)
    torch.cuda.synchronize()
    n = int(offsets[-1])
    ref = oracle.grouped_ffn(np_(x), np_(offsets), np_(w13), np_(w2), round_h=True)
    assert_bf16_close(np_(y)[:n], ref, "two-pair clusters")
    assert rel_fro(np_(y)[:n], ref) < 2e-3
