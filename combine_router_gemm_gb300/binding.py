"""Thin Python binding of ``include/moe.h`` (argument marshalling only).

Each function takes torch tensors, checks that they are contiguous CUDA
tensors of the expected dtype, passes their device pointers, sizes and the
current CUDA stream to the C entry point of the same name, and raises
``MoEError`` on a non-OK status.  All computation happens in the CUDA library
``libmoe_gb300.so``; there is no fallback of any kind.  If the library is
missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_INPUT = range(7)
F32, BF16 = 0, 1
SOFTMAX, SIGMOID = 0, 1

# every symbol include/moe.h declares
SYMBOLS = ("moe_status_string", "moe_version", "moe_route_from_scores", "moe_route",
           "moe_route_workspace_size",
           "moe_dispatch_workspace_size", "moe_dispatch", "moe_grouped_ffn_workspace_size",
           "moe_grouped_ffn", "moe_combine", "moe_layer_workspace_size", "moe_layer",
           "moe_check_error", "moe_dispatch_noalloc", "moe_selftest_bounded_wait",
           "moe_pack_expert_weights", "moe_split_router_weight")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class RouteCfg(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("routed_scale", ctypes.c_float)]


class LayerArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("w_router", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w13_sh", ctypes.c_void_p),
                ("w2_sh", ctypes.c_void_p), ("T", ctypes.c_int32), ("d", ctypes.c_int32),
                ("I", ctypes.c_int32), ("I_sh", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("route", RouteCfg), ("scores_out", ctypes.c_void_p),
                ("topk_idx_out", ctypes.c_void_p), ("topk_w_out", ctypes.c_void_p),
                ("offsets_out", ctypes.c_void_p), ("stage_events", ctypes.c_void_p),
                ("flags", ctypes.c_int32), ("w_router_split", ctypes.c_void_p),
                ("sync_events", ctypes.c_void_p)]

LAYER_FUSED_COMBINE = 1
LAYER_PACKED_WEIGHTS = 2
LAYER_SHARED_AFTER_ROUTER = 4
LAYER_SPLIT_DISPATCH = 8

LAYER_EVENTS = 7
LAYER_SYNC_EVENTS = 4


_lib = None


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run __graft_entry__.build() or combine_router_gemm_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.moe_status_string.argtypes = [i32]
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_version.argtypes = []
    lib.moe_version.restype = i32
    lib.moe_route_from_scores.argtypes = [P, P, i32, ctypes.POINTER(RouteCfg), P, P, P]
    lib.moe_route_from_scores.restype = i32
    lib.moe_route_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.moe_route_workspace_size.restype = sz
    lib.moe_route.argtypes = [P, i32, P, P, i32, i32, ctypes.POINTER(RouteCfg), P, P, P, P, sz, P]
    lib.moe_route.restype = i32
    lib.moe_dispatch_workspace_size.argtypes = [i32, i32, i32]
    lib.moe_dispatch_workspace_size.restype = sz
    lib.moe_dispatch.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, sz, P]
    lib.moe_dispatch.restype = i32
    lib.moe_grouped_ffn_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.moe_grouped_ffn_workspace_size.restype = sz
    lib.moe_grouped_ffn.argtypes = [P, P, i32, i32, i32, i32, P, P, i32, P, P, sz, P]
    lib.moe_grouped_ffn.restype = i32
    lib.moe_combine.argtypes = [P, P, P, P, i32, i32, i32, P, P]
    lib.moe_combine.restype = i32
    lib.moe_layer_workspace_size.argtypes = [ctypes.POINTER(LayerArgs)]
    lib.moe_layer_workspace_size.restype = sz
    lib.moe_layer.argtypes = [ctypes.POINTER(LayerArgs), P, P, sz, P, P]
    lib.moe_layer.restype = i32
    lib.moe_check_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.moe_check_error.restype = i32
    lib.moe_dispatch_noalloc.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
    lib.moe_dispatch_noalloc.restype = i32
    lib.moe_selftest_bounded_wait.argtypes = [i32, ctypes.c_uint32, P, sz, P]
    lib.moe_selftest_bounded_wait.restype = i32
    lib.moe_pack_expert_weights.argtypes = [P, P, i32, i32, i32, P, P, P]
    lib.moe_pack_expert_weights.restype = i32
    lib.moe_split_router_weight.argtypes = [P, i32, i32, P, P]
    lib.moe_split_router_weight.restype = i32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != OK:
        raise MoEError(rc, where)


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def route_cfg(E: int, k: int, n_group: int = 1, topk_group: int = 1, score_fn: int = SOFTMAX,
              routed_scale: float = 1.0) -> RouteCfg:
    return RouteCfg(E, k, n_group, topk_group, score_fn, routed_scale)


def cfg_from(c) -> RouteCfg:
    """RouteCfg from a workload description with E, k, n_group, topk_group, score_fn, routed_scale."""
    return route_cfg(c.E, c.k, c.n_group, c.topk_group,
                     SIGMOID if c.score_fn == "sigmoid" else SOFTMAX, c.routed_scale)


# ---------------------------------------------------------------- entry points

def moe_route_from_scores(scores, bias, cfg: RouteCfg, topk_idx, topk_w, stream=None):
    T = scores.shape[0]
    rc = load().moe_route_from_scores(_ptr(scores, torch.float32, "scores"),
                                      _ptr(bias, torch.float32, "bias"), T, ctypes.byref(cfg),
                                      _ptr(topk_idx, torch.int32, "topk_idx"),
                                      _ptr(topk_w, torch.float32, "topk_w"), _stream(stream))
    _check(rc, "moe_route_from_scores")


def moe_route_workspace_size(T: int, E: int, d: int, dtype: int) -> int:
    return load().moe_route_workspace_size(T, E, d, dtype)


def moe_route(x, w_router, bias, cfg: RouteCfg, scores, topk_idx, topk_w, ws=None, stream=None):
    T, d = x.shape
    if ws is None:
        ws = torch.empty(moe_route_workspace_size(T, cfg.num_experts, d, _dtype_code(x)),
                         dtype=torch.uint8, device=x.device)
    rc = load().moe_route(_ptr(x, None, "x"), _dtype_code(x), _ptr(w_router, torch.float32, "w_router"),
                          _ptr(bias, torch.float32, "bias"), T, d, ctypes.byref(cfg),
                          _ptr(scores, torch.float32, "scores"),
                          _ptr(topk_idx, torch.int32, "topk_idx"),
                          _ptr(topk_w, torch.float32, "topk_w"), _ptr(ws, None, "ws"),
                          ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "moe_route")


def moe_dispatch_workspace_size(T: int, k: int, E: int) -> int:
    return load().moe_dispatch_workspace_size(T, k, E)


def moe_dispatch(topk_idx, x, E: int, counts, offsets, slot_to_row, row_to_token, x_perm, ws,
                 stream=None):
    T, k = topk_idx.shape
    d = x.shape[1] if x is not None else 8
    dt = _dtype_code(x) if x is not None else BF16
    rc = load().moe_dispatch(_ptr(topk_idx, torch.int32, "topk_idx"), _ptr(x, None, "x"), dt, T, d,
                             k, E, _ptr(counts, torch.int32, "counts"),
                             _ptr(offsets, torch.int32, "offsets"),
                             _ptr(slot_to_row, torch.int32, "slot_to_row"),
                             _ptr(row_to_token, torch.int32, "row_to_token"),
                             _ptr(x_perm, None, "x_perm"), _ptr(ws, None, "ws"),
                             ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "moe_dispatch")


DISPATCH_NOALLOC_MAX_SLOTS = 131072


def moe_dispatch_noalloc(topk_idx, x, E: int, counts, offsets, slot_to_row, row_to_token, x_perm,
                         device_error=None, stream=None):
    """moe_dispatch without a workspace: for callers that may not allocate
    device memory while they run (fixed memory pools, hosted plug-ins).  The
    library keeps the scratch in a fixed device array of its own; calls must
    not overlap on the GPU.  ``device_error``: optional int32 CUDA tensor of
    one element that receives the call's error word."""
    T, k = topk_idx.shape
    d = x.shape[1] if x is not None else 8
    dt = _dtype_code(x) if x is not None else BF16
    rc = load().moe_dispatch_noalloc(_ptr(topk_idx, torch.int32, "topk_idx"), _ptr(x, None, "x"),
                                     dt, T, d, k, E, _ptr(counts, torch.int32, "counts"),
                                     _ptr(offsets, torch.int32, "offsets"),
                                     _ptr(slot_to_row, torch.int32, "slot_to_row"),
                                     _ptr(row_to_token, torch.int32, "row_to_token"),
                                     _ptr(x_perm, None, "x_perm"),
                                     _ptr(device_error, torch.int32, "device_error"),
                                     _stream(stream))
    _check(rc, "moe_dispatch_noalloc")


def moe_grouped_ffn_workspace_size(rows: int, d: int, I: int, dtype: int) -> int:
    return load().moe_grouped_ffn_workspace_size(rows, d, I, dtype)


def moe_grouped_ffn(x_perm, offsets, w13, w2, y_perm, ws, stream=None):
    rows, d = x_perm.shape
    E, I = w2.shape[0], w2.shape[2]
    rc = load().moe_grouped_ffn(_ptr(x_perm, None, "x_perm"), _ptr(offsets, torch.int32, "offsets"),
                                E, rows, d, I, _ptr(w13, x_perm.dtype, "w13"),
                                _ptr(w2, x_perm.dtype, "w2"), _dtype_code(x_perm),
                                _ptr(y_perm, torch.float32, "y_perm"), _ptr(ws, None, "ws"),
                                ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "moe_grouped_ffn")


def moe_combine(y_perm, slot_to_row, topk_w, shared, out, stream=None):
    T, k = topk_w.shape
    d = out.shape[1]
    rc = load().moe_combine(_ptr(y_perm, torch.float32, "y_perm"),
                            _ptr(slot_to_row, torch.int32, "slot_to_row"),
                            _ptr(topk_w, torch.float32, "topk_w"),
                            _ptr(shared, torch.float32, "shared"), T, k, d,
                            _ptr(out, torch.float32, "out"), _stream(stream))
    _check(rc, "moe_combine")


def layer_args(x, w_router, bias, w13, w2, w13_sh, w2_sh, cfg: RouteCfg, scores_out=None,
               topk_idx_out=None, topk_w_out=None, offsets_out=None,
               stage_events=None, flags: int = 0, w_router_split=None,
               sync_events=None) -> LayerArgs:
    """``stage_events``: None or a list of LAYER_EVENTS torch.cuda.Event (kept
    alive by the caller), recorded by the library at the stage boundaries.
    ``w_router_split``: the router weight from moe_split_router_weight, or None.
    ``sync_events``: None or a list of LAYER_SYNC_EVENTS torch.cuda.Event (kept
    alive by the caller) that fork and join the second stream."""
    T, d = x.shape
    I = w2.shape[2]
    I_sh = w2_sh.shape[1] if w2_sh is not None else 0
    return LayerArgs(_ptr(x, None, "x"), _ptr(w_router, torch.float32, "w_router"),
                     _ptr(bias, torch.float32, "bias"), _ptr(w13, x.dtype, "w13"),
                     _ptr(w2, x.dtype, "w2"), _ptr(w13_sh, x.dtype, "w13_sh"),
                     _ptr(w2_sh, x.dtype, "w2_sh"), T, d, I, I_sh, _dtype_code(x), cfg,
                     _ptr(scores_out, torch.float32, "scores_out"),
                     _ptr(topk_idx_out, torch.int32, "topk_idx_out"),
                     _ptr(topk_w_out, torch.float32, "topk_w_out"),
                     _ptr(offsets_out, torch.int32, "offsets_out"), _events(stage_events), flags,
                     _ptr(w_router_split, torch.bfloat16, "w_router_split"),
                     _events(sync_events, LAYER_SYNC_EVENTS))


_event_arrays = {}


def _events(evs, n=LAYER_EVENTS):
    """Host array of cudaEvent_t handles for torch events (cached per list)."""
    if evs is None:
        return None
    if len(evs) != n:
        raise ValueError(f"need {n} events")
    key = tuple(id(e) for e in evs)
    arr = _event_arrays.get(key)
    if arr is None:
        for e in evs:  # torch creates the CUDA event lazily on first record
            if e.cuda_event == 0:
                e.record()
        arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
        _event_arrays[key] = (arr, evs)
    else:
        arr = arr[0]
    return ctypes.cast(arr, ctypes.c_void_p).value


def moe_layer_workspace_size(args: LayerArgs) -> int:
    n = load().moe_layer_workspace_size(ctypes.byref(args))
    if n == 0:
        raise MoEError(ERR_INVALID_ARG, "moe_layer_workspace_size")
    return n


def moe_layer(args: LayerArgs, out, ws, stream=None, stream2=None):
    s2 = stream2.cuda_stream if stream2 is not None else None
    rc = load().moe_layer(ctypes.byref(args), _ptr(out, torch.float32, "out"), _ptr(ws, None, "ws"),
                          ws.numel() * ws.element_size(), _stream(stream), s2)
    _check(rc, "moe_layer")


def moe_selftest_bounded_wait(which: int, limit_us: int, ws, stream=None):
    """Run a wait that nothing signals (0: mbarrier, 1: look-back flag, 2:
    cluster-scope mbarrier in a two-CTA cluster); the kernel must give up
    after limit_us and flag a timeout in ws."""
    rc = load().moe_selftest_bounded_wait(which, limit_us, _ptr(ws, None, "ws"),
                                          ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "moe_selftest_bounded_wait")


def moe_check_error(ws, stream=None) -> tuple[int, int]:
    detail = ctypes.c_uint32(0)
    rc = load().moe_check_error(_ptr(ws, None, "ws"), _stream(stream), ctypes.byref(detail))
    return rc, detail.value


# ---------------------------------------------------------------- convenience

def moe_pack_expert_weights(w13, w2, w13_packed, w2_packed, stream=None):
    """w13 [E,2I,d] and w2 [E,d,I] bf16 (either may be None, with its output)
    into the tile-major layouts of LAYER_PACKED_WEIGHTS; 2-D shared-expert
    weights ([2I,d], [d,I]) are packed as E = 1."""
    ref = w13 if w13 is not None else w2
    if ref is None:
        return
    if ref.dim() == 2:
        E = 1
        d = w13.shape[1] if w13 is not None else w2.shape[0]
        I = w13.shape[0] // 2 if w13 is not None else w2.shape[1]
    else:
        E = ref.shape[0]
        d = w13.shape[2] if w13 is not None else w2.shape[1]
        I = w13.shape[1] // 2 if w13 is not None else w2.shape[2]
    rc = load().moe_pack_expert_weights(_ptr(w13, torch.bfloat16, "w13"),
                                        _ptr(w2, torch.bfloat16, "w2"), E, d, I,
                                        _ptr(w13_packed, torch.bfloat16, "w13_packed"),
                                        _ptr(w2_packed, torch.bfloat16, "w2_packed"),
                                        _stream(stream))
    _check(rc, "moe_pack_expert_weights")


def moe_split_router_weight(w_router, out=None, stream=None):
    """w_router [E,d] fp32 -> [3,E,d] bf16 (hi, mid, lo), the router's tensor-core
    operand, for LayerArgs.w_router_split.  Returns ``out``."""
    E, d = w_router.shape
    if out is None:
        out = torch.empty((3, E, d), dtype=torch.bfloat16, device=w_router.device)
    rc = load().moe_split_router_weight(_ptr(w_router, torch.float32, "w_router"), E, d,
                                        _ptr(out, torch.bfloat16, "out"), _stream(stream))
    _check(rc, "moe_split_router_weight")
    return out


def packable(w13, w2, w13_sh=None, w2_sh=None) -> bool:
    """Whether the tile-major layouts apply (bf16, I % 128 == 0, d % 256 == 0)."""
    if w13.dtype != torch.bfloat16:
        return False
    d, I = w13.shape[2], w2.shape[2]
    I_sh = w2_sh.shape[1] if w2_sh is not None else 0
    return d % 256 == 0 and I % 128 == 0 and I_sh % 128 == 0


class MoELayer:
    """Holds the weights of one layer plus a workspace; ``forward(x)`` -> out fp32 [T,d].

    ``x`` must have the token count the layer was built for (workspace size
    depends on it).  Allocation happens only here, in PyTorch, never in the
    library.  With ``pack_weights`` (the default) the expert weights are
    copied once into the tile-major layouts the grouped GEMMs stream fastest,
    where the shapes allow it; the layer then holds those copies.  With
    ``split_dispatch`` the permute of the upper half of the experts runs on a
    second stream beside the lower half's gate/up (MOE_LAYER_SPLIT_DISPATCH).
    """

    def __init__(self, w_router, bias, w13, w2, w13_sh, w2_sh, cfg: RouteCfg, T: int,
                 overlap: bool = True, fused_combine: bool = False, pack_weights: bool = True,
                 split_router: bool = True, split_dispatch: bool = False):
        self.cfg = cfg
        self.T = T
        dev = w13.device
        d = w13.shape[2]
        I_sh = w2_sh.shape[1] if w2_sh is not None else 0
        if split_dispatch and (w13.dtype != torch.bfloat16 or fused_combine):
            raise ValueError("split_dispatch needs bf16 weights and no fused combine")
        self.flags = LAYER_FUSED_COMBINE if fused_combine else 0
        if split_dispatch:
            self.flags |= LAYER_SPLIT_DISPATCH
        self.packed = pack_weights and packable(w13, w2, w13_sh, w2_sh)
        if self.packed:
            p13, p2 = torch.empty_like(w13), torch.empty_like(w2)
            moe_pack_expert_weights(w13, w2, p13, p2)
            w13, w2 = p13, p2
            if w13_sh is not None:
                p13s, p2s = torch.empty_like(w13_sh), torch.empty_like(w2_sh)
                moe_pack_expert_weights(w13_sh, w2_sh, p13s, p2s)
                w13_sh, w2_sh = p13s, p2s
            self.flags |= LAYER_PACKED_WEIGHTS
        self.w = dict(w_router=w_router, bias=bias, w13=w13, w2=w2, w13_sh=w13_sh, w2_sh=w2_sh)
        self._extra_flags = 0
        # the bf16 router multiplies a three-term split of its fp32 weight:
        # made once here instead of on every call
        self.w_router_split = (moe_split_router_weight(w_router)
                               if split_router and w13.dtype == torch.bfloat16 else None)
        sizes = LayerArgs(None, None, None, None, None, None, None, T, d, w2.shape[2], I_sh,
                          _dtype_code(w13), cfg, None, None, None, None, None, self.flags)
        self.ws_bytes = moe_layer_workspace_size(sizes)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.stream2 = (torch.cuda.Stream(device=dev)
                        if (overlap and w13_sh is not None) or split_dispatch else None)
        # the events that fork and join the second stream, made once
        self.sync_events = ([torch.cuda.Event() for _ in range(LAYER_SYNC_EVENTS)]
                            if self.stream2 is not None else None)

    def _args(self, x, **outs):
        w = self.w
        return layer_args(x, w["w_router"], w["bias"], w["w13"], w["w2"], w["w13_sh"],
                          w["w2_sh"], self.cfg, flags=self.flags | self._extra_flags,
                          w_router_split=self.w_router_split, sync_events=self.sync_events,
                          **outs)

    def forward(self, x, out=None, stream=None, **outs):
        """out [T,d] fp32 for x [T,d] (device tensors), enqueued on `stream`
        (default: the current stream)."""
        if x.shape[0] != self.T:
            raise ValueError(f"layer built for T={self.T}, got {x.shape[0]}")
        if out is None:
            out = torch.empty((x.shape[0], x.shape[1]), dtype=torch.float32, device=x.device)
        moe_layer(self._args(x, **outs), out, self.ws, stream=stream, stream2=self.stream2)
        return out

    def capture(self, x, out=None, shared_after_router: bool = True, **outs):
        """Record one ``forward(x)`` into a CUDA graph and return ``(graph,
        out)``.

        ``graph.replay()`` recomputes the layer from the current contents of
        the static buffer ``x`` (copy new tokens into it) into the static
        ``out``; the optional outputs (``scores_out`` ...) are static as well.
        One call runs first, outside the capture, so that the per-device
        kernel settings are made before capturing.  The second stream of the
        layer is forked from and joined back into the capture by events; with
        ``shared_after_router`` its work follows the router GEMM in the graph
        (LAYER_SHARED_AFTER_ROUTER), a fixed order that replays keep.
        """
        if out is None:
            out = torch.empty((x.shape[0], x.shape[1]), dtype=torch.float32, device=x.device)
        dev = x.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self.forward(x, out=out, **outs)
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        self._extra_flags = LAYER_SHARED_AFTER_ROUTER if shared_after_router else 0
        try:
            with torch.cuda.graph(graph, capture_error_mode="relaxed"):
                self.forward(x, out=out, **outs)
        finally:
            self._extra_flags = 0
        return graph, out

    def forward_host(self, host_inputs, host_outputs):
        """Run the layer over a sequence of host batches, pipelined.

        ``host_inputs[i]`` ([T,d], pinned host memory, the layer's dtype) is
        copied in, the layer runs, and the result lands in ``host_outputs[i]``
        ([T,d] fp32, pinned).  Copies in, compute and copies out run on three
        streams with two device buffers each way, so that batch i+1's input
        and batch i-1's output move while batch i computes.  Returns the
        (first, last) CUDA events that bracket the whole sequence; the caller
        synchronises.
        """
        n = len(host_inputs)
        if n != len(host_outputs) or n == 0:
            raise ValueError("need as many outputs as inputs (at least one)")
        dev = self.ws.device
        d = host_inputs[0].shape[1]
        if not hasattr(self, "_pipe") or self._pipe["d"] != d:
            self._pipe = dict(
                d=d, x=[torch.empty((self.T, d), dtype=host_inputs[0].dtype, device=dev) for _ in range(2)],
                out=[torch.empty((self.T, d), dtype=torch.float32, device=dev) for _ in range(2)],
                s_in=torch.cuda.Stream(device=dev), s_comp=torch.cuda.Stream(device=dev),
                s_out=torch.cuda.Stream(device=dev))
        P = self._pipe
        s_in, s_comp, s_out = P["s_in"], P["s_comp"], P["s_out"]
        first = torch.cuda.Event(enable_timing=True)
        last = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        for st in (s_in, s_comp, s_out):
            st.wait_stream(cur)
        first.record(s_in)
        s_comp.wait_event(first)
        s_out.wait_event(first)
        done_comp = [None, None]  # compute of the batch that last used buffer b
        done_out = [None, None]   # output copy of the batch that last used buffer b
        for i in range(n):
            b = i % 2
            if done_comp[b] is not None:
                s_in.wait_event(done_comp[b])  # x[b] is free once its compute ran
            with torch.cuda.stream(s_in):
                P["x"][b].copy_(host_inputs[i], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            if done_out[b] is not None:
                s_comp.wait_event(done_out[b])  # out[b] is free once it was copied out
            self.forward(P["x"][b], out=P["out"][b], stream=s_comp)
            ev_c = torch.cuda.Event()
            ev_c.record(s_comp)
            done_comp[b] = ev_c
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                host_outputs[i].copy_(P["out"][b], non_blocking=True)
            ev_o = torch.cuda.Event()
            ev_o.record(s_out)
            done_out[b] = ev_o
        last.record(s_out)
        cur.wait_stream(s_out)
        return first, last
