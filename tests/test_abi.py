"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects invalid arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

from combine_router_gemm_gb300 import binding as B
from combine_router_gemm_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert sorted(B.SYMBOLS) == declared_symbols()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes structures have the C structures' field offsets and sizes
    (a small C program built against include/moe.h prints them)."""
    fields = {"moe_route_cfg": B.RouteCfg, "moe_layer_args": B.LayerArgs}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "moe.h"', 'int main(void) {']
    for cname, py in fields.items():
        lines.append(f'printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {tuple(ln.split()[:2]): int(ln.split()[2]) for ln in out.splitlines()}
    for cname, py in fields.items():
        assert got[(cname, "sizeof")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_status_strings(lib):
    assert B.status_string(B.OK) == "ok"
    for s in range(1, 7):
        assert B.status_string(s) not in ("ok", "unknown status")
    assert B.status_string(99) == "unknown status"
    assert lib.moe_version() >= 100


def test_workspace_sizes_host_only(lib):
    assert lib.moe_dispatch_workspace_size(4096, 8, 256) > 4096 * 8 * 4
    assert lib.moe_dispatch_workspace_size(-1, 8, 256) == 0
    assert lib.moe_grouped_ffn_workspace_size(1000, 256, 128, B.BF16) >= 1000 * 128 * 2
    assert lib.moe_grouped_ffn_workspace_size(1000, 256, 128, B.F32) >= 1000 * 128 * 4
    args = B.LayerArgs(1 << 20, 1 << 20, None, 1 << 20, 1 << 20, None, None, 64, 128, 256, 0,
                       B.F32, B.route_cfg(8, 2), None, None, None, None)
    n = lib.moe_layer_workspace_size(ctypes.byref(args))
    assert n > 64 * 2 * 128 * 4 * 2


P = 1 << 20  # a 16-byte aligned fake device address; never dereferenced


def cfg(E=8, k=2, ng=1, tg=1, fn=B.SOFTMAX, scale=1.0):
    return B.route_cfg(E, k, ng, tg, fn, scale)


@pytest.mark.parametrize("c", [cfg(E=0), cfg(k=0), cfg(k=9), cfg(E=10, ng=3),
                               cfg(E=8, ng=8, tg=1, fn=B.SIGMOID), cfg(E=16, ng=4, tg=5),
                               cfg(E=16, k=9, ng=4, tg=2), cfg(fn=7), cfg(scale=float("inf"))])
def test_route_rejects_bad_config(lib, c):
    rc = lib.moe_route_from_scores(P, None, 10, ctypes.byref(c), P, P, None)
    assert rc == B.ERR_INVALID_ARG


def test_route_rejects_unsupported(lib):
    c = cfg(E=2048, k=2)
    assert lib.moe_route_from_scores(P, None, 10, ctypes.byref(c), P, P, None) == B.ERR_UNSUPPORTED
    c = cfg(E=64, k=33)
    assert lib.moe_route_from_scores(P, None, 10, ctypes.byref(c), P, P, None) == B.ERR_UNSUPPORTED


def test_route_rejects_bad_pointers(lib):
    c = cfg()
    assert lib.moe_route_from_scores(None, None, 10, ctypes.byref(c), P, P, None) == B.ERR_INVALID_ARG
    # a bias with softmax routing has no meaning
    assert lib.moe_route_from_scores(P, P, 10, ctypes.byref(c), P, P, None) == B.ERR_INVALID_ARG
    need = lib.moe_route_workspace_size(10, 8, 64, B.BF16)
    assert need >= 3 * 8 * 64 * 2 + 10 * 8 * 4
    assert lib.moe_route(P + 4, B.BF16, P, None, 10, 64, ctypes.byref(c), P, P, P, P, need, None) == B.ERR_INVALID_ARG
    assert lib.moe_route(P, B.BF16, P, None, 10, 60, ctypes.byref(c), P, P, P, P, need, None) == B.ERR_INVALID_ARG
    assert lib.moe_route(P, 5, P, None, 10, 64, ctypes.byref(c), P, P, P, P, need, None) == B.ERR_INVALID_ARG
    assert lib.moe_route(P, B.BF16, P, None, 10, 64, ctypes.byref(c), P, P, P, P, need - 1, None) == B.ERR_WORKSPACE


def test_dispatch_rejects(lib):
    ws_need = lib.moe_dispatch_workspace_size(100, 2, 8)
    args = [P, P, B.BF16, 100, 64, 2, 8, P, P, P, P, P, P, ws_need, None]
    bad_ws = list(args)
    bad_ws[13] = ws_need - 1
    assert lib.moe_dispatch(*bad_ws) == B.ERR_WORKSPACE
    no_ws = list(args)
    no_ws[12] = None
    assert lib.moe_dispatch(*no_ws) == B.ERR_WORKSPACE
    half = list(args)
    half[10] = None  # x given but no x_perm
    assert lib.moe_dispatch(*half) == B.ERR_INVALID_ARG
    bad_k = list(args)
    bad_k[5] = 0
    assert lib.moe_dispatch(*bad_k) == B.ERR_INVALID_ARG


def test_grouped_ffn_rejects(lib):
    need = lib.moe_grouped_ffn_workspace_size(100, 64, 64, B.BF16)
    ok = [P, P, 4, 100, 64, 64, P, P, B.BF16, P, P, need, None]
    for pos, val, want in [(11, need - 1, B.ERR_WORKSPACE), (4, 60, B.ERR_INVALID_ARG),
                           (5, 12, B.ERR_INVALID_ARG), (1, None, B.ERR_INVALID_ARG),
                           (2, 0, B.ERR_INVALID_ARG), (2, 4096, B.ERR_UNSUPPORTED),
                           (6, P + 8, B.ERR_INVALID_ARG)]:
        a = list(ok)
        a[pos] = val
        assert lib.moe_grouped_ffn(*a) == want, (pos, val)


def test_combine_rejects(lib):
    assert lib.moe_combine(None, P, P, None, 10, 2, 64, P, None) == B.ERR_INVALID_ARG
    assert lib.moe_combine(P, P, P, None, 10, 2, 6, P, None) == B.ERR_INVALID_ARG
    assert lib.moe_combine(P, P, P, None, 10, 40, 64, P, None) == B.ERR_UNSUPPORTED
    assert lib.moe_combine(P, P, P, P + 4, 10, 2, 64, P, None) == B.ERR_INVALID_ARG


def test_layer_rejects(lib):
    def args(**kw):
        a = dict(x=P, w_router=P, bias=None, w13=P, w2=P, w13_sh=None, w2_sh=None, T=64, d=128,
                 I=256, I_sh=0, dtype=B.F32, route=cfg(), scores_out=None, topk_idx_out=None,
                 topk_w_out=None, offsets_out=None)
        a.update(kw)
        return B.LayerArgs(**a)
    need = lib.moe_layer_workspace_size(ctypes.byref(args()))
    assert need > 0
    assert lib.moe_layer(ctypes.byref(args()), P, P, need - 1, None, None) == B.ERR_WORKSPACE
    assert lib.moe_layer(ctypes.byref(args(w13_sh=P)), P, P, need, None, None) == B.ERR_INVALID_ARG
    assert lib.moe_layer(ctypes.byref(args(I=100)), P, P, need, None, None) == B.ERR_INVALID_ARG
    assert lib.moe_layer(ctypes.byref(args()), None, P, need, None, None) == B.ERR_INVALID_ARG
    assert lib.moe_layer_workspace_size(ctypes.byref(args(dtype=3))) == 0
    # the size query needs sizes only
    assert lib.moe_layer_workspace_size(ctypes.byref(args(x=None, w13=None, w2=None,
                                                          w_router=None))) == need
    # the optional outputs replace workspace regions
    assert lib.moe_layer_workspace_size(ctypes.byref(args(scores_out=P))) < need


def test_pack_expert_weights_rejects(lib):
    # the valid form launches a kernel (tests/test_gpu_ffn.py)
    assert lib.moe_pack_expert_weights(*[P, P, 4, 200, 128, P, P, None]) == B.ERR_INVALID_ARG  # d % 256
    assert lib.moe_pack_expert_weights(*[P, P, 4, 256, 136, P, P, None]) == B.ERR_INVALID_ARG  # I % 128
    assert lib.moe_pack_expert_weights(*[P, P, 0, 256, 128, P, P, None]) == B.ERR_INVALID_ARG  # E
    assert lib.moe_pack_expert_weights(*[P, P, 4, 256, 128, None, P, None]) == B.ERR_INVALID_ARG  # pairing
    assert lib.moe_pack_expert_weights(*[P + 8, P, 4, 256, 128, P, P, None]) == B.ERR_INVALID_ARG  # alignment
    assert lib.moe_pack_expert_weights(None, None, 4, 256, 128, None, None, None) == B.OK  # nothing to do


def test_layer_packed_flag_checks(lib):
    def args(**kw):
        a = dict(x=P, w_router=P, bias=None, w13=P, w2=P, w13_sh=None, w2_sh=None, T=64, d=256,
                 I=256, I_sh=0, dtype=B.BF16, route=cfg(), scores_out=None, topk_idx_out=None,
                 topk_w_out=None, offsets_out=None, flags=B.LAYER_PACKED_WEIGHTS)
        a.update(kw)
        return B.LayerArgs(**a)
    need = lib.moe_layer_workspace_size(ctypes.byref(args()))
    assert need > 0
    for bad in (dict(d=384), dict(I=136), dict(dtype=B.F32), dict(w13_sh=P, w2_sh=P, I_sh=136)):
        a = args(**bad)
        n = lib.moe_layer_workspace_size(ctypes.byref(a)) or need
        assert lib.moe_layer(ctypes.byref(a), P, P, n, None, None) == B.ERR_UNSUPPORTED, bad
    assert lib.moe_layer(ctypes.byref(args(flags=16)), P, P, need, None, None) == B.ERR_INVALID_ARG


def test_layer_split_dispatch_checks(lib):
    """The split dispatch needs a second stream, bf16 and the unfused
    combine; each miss is refused on the host before anything is enqueued."""
    def args(**kw):
        a = dict(x=P, w_router=P, bias=None, w13=P, w2=P, w13_sh=None, w2_sh=None, T=64, d=256,
                 I=256, I_sh=0, dtype=B.BF16, route=cfg(), scores_out=None, topk_idx_out=None,
                 topk_w_out=None, offsets_out=None, flags=B.LAYER_SPLIT_DISPATCH)
        a.update(kw)
        return B.LayerArgs(**a)
    need = lib.moe_layer_workspace_size(ctypes.byref(args()))
    assert need > 0
    s2 = ctypes.c_void_p(P)  # any non-null stream handle: refused before use
    assert lib.moe_layer(ctypes.byref(args()), P, P, need, None, None) == B.ERR_UNSUPPORTED
    assert lib.moe_layer(ctypes.byref(args()), P, P, need, s2, s2) == B.ERR_UNSUPPORTED
    for bad in (dict(dtype=B.F32), dict(flags=B.LAYER_SPLIT_DISPATCH | B.LAYER_FUSED_COMBINE)):
        a = args(**bad)
        n = lib.moe_layer_workspace_size(ctypes.byref(a)) or need
        assert lib.moe_layer(ctypes.byref(a), P, P, n, None, s2) == B.ERR_UNSUPPORTED, bad


def test_split_router_weight_rejects(lib):
    assert lib.moe_split_router_weight(P, 0, 64, P, None) == B.ERR_INVALID_ARG
    assert lib.moe_split_router_weight(P, 8, 60, P, None) == B.ERR_INVALID_ARG
    assert lib.moe_split_router_weight(None, 8, 64, P, None) == B.ERR_INVALID_ARG
    assert lib.moe_split_router_weight(P, 8, 64, P + 4, None) == B.ERR_INVALID_ARG


def test_layer_presplit_router_checks(lib):
    a = B.LayerArgs(x=P, w_router=P, w13=P, w2=P, T=64, d=128, I=256, dtype=B.F32,
                    route=cfg(), w_router_split=P)
    need = lib.moe_layer_workspace_size(ctypes.byref(a))
    # an fp32 layer has no split router weight
    assert lib.moe_layer(ctypes.byref(a), P, P, need, None, None) == B.ERR_INVALID_ARG
    a.dtype, a.w_router_split = B.BF16, P + 8
    need = lib.moe_layer_workspace_size(ctypes.byref(a))
    assert lib.moe_layer(ctypes.byref(a), P, P, need, None, None) == B.ERR_INVALID_ARG


def test_layer_flag_bits(lib):
    a = B.LayerArgs(x=P, w_router=P, w13=P, w2=P, T=64, d=128, I=256, dtype=B.F32, route=cfg(),
                    flags=B.LAYER_SHARED_AFTER_ROUTER | 16)
    need = lib.moe_layer_workspace_size(ctypes.byref(a))
    assert lib.moe_layer(ctypes.byref(a), P, P, need, None, None) == B.ERR_INVALID_ARG


def test_selftest_rejects(lib):
    # host-side checks, nothing is launched
    assert lib.moe_selftest_bounded_wait(3, 1000, P, 4096, None) == B.ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(2, 0, P, 4096, None) == B.ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(2, 1000, P, 16, None) == B.ERR_WORKSPACE
