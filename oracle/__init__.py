"""CPU oracle of the MoE layer: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.  The arithmetic lives in
``moe_oracle.c`` (plain C, double accumulation, one OpenMP thread per token);
this module builds that file with gcc and marshals numpy arrays into it.

Reading of the method (the pages -- "CUCo: An Agentic Framework for Compute and
Communication Co-design", abstract and Table 4 row "MoE Dispatch/Combine" --
name a DeepSeek-V3 MoE layer but do not write its arithmetic down) is stated at
the top of ``moe_oracle.c``.  bf16 arrays are passed as their raw ``uint16``
bits, so no value is converted on the way in.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
SOFTMAX, SIGMOID = 0, 1


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``libmoe_oracle.so`` next to it."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, f64 = ctypes.c_int, ctypes.c_double
            lib.oracle_round_bf16.argtypes = [f64]
            lib.oracle_round_bf16.restype = f64
            lib.oracle_router_scores.argtypes = [P, i32, P, i32, i32, i32, i32, P]
            lib.oracle_router_scores.restype = None
            lib.oracle_select.argtypes = [P, P, i32, i32, i32, i32, i32, P]
            lib.oracle_select.restype = i32
            lib.oracle_gates.argtypes = [P, P, i32, i32, i32, i32, f64, P]
            lib.oracle_gates.restype = None
            lib.oracle_dispatch.argtypes = [P, i32, i32, i32, P, P, P, P]
            lib.oracle_dispatch.restype = i32
            lib.oracle_expert_rows.argtypes = [P, i32, i32, P, P, P, i32, i32, i32, i32, P]
            lib.oracle_expert_rows.restype = None
            lib.oracle_combine.argtypes = [P, P, P, P, i32, i32, i32, P]
            lib.oracle_combine.restype = None
            lib.oracle_moe_tokens.argtypes = [P, i32, i32, i32, P, P, P, i32, i32, i32, i32, i32,
                                              f64, P, P, i32, i32, P, P, i32, i32, P, P, P]
            lib.oracle_moe_tokens.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def _c(a: np.ndarray | None, dtype=None):
    """Contiguous array (optionally of ``dtype``) and its address (0 for None)."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(a if dtype is None else a.astype(dtype, copy=False))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _typed(a: np.ndarray):
    """(array, dtype code) for an fp32 array or raw bf16 bits (uint16)."""
    if a.dtype == np.uint16:
        return _c(a)[0], BF16
    return _c(a, np.float32)[0], F32


def num_threads() -> int:
    return _load().oracle_num_threads()


def round_bf16(v: float) -> float:
    """Nearest bf16 value to ``v`` (ties to even), rounded once from double."""
    return _load().oracle_round_bf16(float(v))


def router_scores(x: np.ndarray, w_router: np.ndarray, score_fn: int) -> np.ndarray:
    """fp32 score tensor [T,E]: logits (softmax) or sigmoid(logits) (sigmoid)."""
    x, xdt = _typed(x)
    T, d = x.shape
    wr, pwr = _c(w_router, np.float32)
    E = wr.shape[0]
    out = np.empty((T, E), np.float32)
    _load().oracle_router_scores(x.ctypes.data_as(ctypes.c_void_p), xdt, pwr, T, d, E, score_fn,
                                 out.ctypes.data_as(ctypes.c_void_p))
    return out


def select(scores: np.ndarray, k: int, bias: np.ndarray | None = None, n_group: int = 1,
           topk_group: int = 1) -> np.ndarray:
    """Chosen experts [T,k] int32, in selection order (ties to the lower index)."""
    sc, psc = _c(scores, np.float32)
    T, E = sc.shape
    b, pb = _c(bias, np.float32)
    idx = np.empty((T, k), np.int32)
    rc = _load().oracle_select(psc, pb, T, E, k, n_group, topk_group,
                               idx.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("fewer than k eligible experts for some token")
    return idx


def gates(scores: np.ndarray, idx: np.ndarray, score_fn: int, routed_scale: float = 1.0) -> np.ndarray:
    """Gate weights [T,k] in double."""
    sc, psc = _c(scores, np.float32)
    T, E = sc.shape
    ix, pix = _c(idx, np.int32)
    k = ix.shape[1]
    w = np.empty((T, k), np.float64)
    _load().oracle_gates(psc, pix, T, E, k, score_fn, float(routed_scale),
                         w.ctypes.data_as(ctypes.c_void_p))
    return w


def dispatch(idx: np.ndarray, E: int):
    """(counts[E], offsets[E+1], slot_to_row[T*k], row_to_token[T*k]) int32."""
    ix, pix = _c(idx, np.int32)
    T, k = ix.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    s2r = np.empty(T * k, np.int32)
    r2t = np.empty(T * k, np.int32)
    rc = _load().oracle_dispatch(pix, T, k, E, counts.ctypes.data_as(ctypes.c_void_p),
                                 offsets.ctypes.data_as(ctypes.c_void_p),
                                 s2r.ctypes.data_as(ctypes.c_void_p),
                                 r2t.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("expert index out of range")
    return counts, offsets, s2r, r2t


def expert_rows(x: np.ndarray, row_expert: np.ndarray, w13: np.ndarray, w2: np.ndarray,
                round_h: bool) -> np.ndarray:
    """y[r] = SwiGLU_{row_expert[r]}(x[r]) in double; w13 [E,2I,d], w2 [E,d,I]."""
    x, xdt = _typed(x)
    n, d = x.shape
    re, pre = _c(row_expert, np.int32)
    w13, wdt = _typed(w13)
    w2, wdt2 = _typed(w2)
    assert wdt == wdt2
    I = w2.shape[2]
    y = np.empty((n, d), np.float64)
    _load().oracle_expert_rows(x.ctypes.data_as(ctypes.c_void_p), xdt, n, pre,
                               w13.ctypes.data_as(ctypes.c_void_p),
                               w2.ctypes.data_as(ctypes.c_void_p), wdt, d, I, int(round_h),
                               y.ctypes.data_as(ctypes.c_void_p))
    return y


def grouped_ffn(x_perm: np.ndarray, offsets: np.ndarray, w13: np.ndarray, w2: np.ndarray,
                round_h: bool) -> np.ndarray:
    """Expert FFN over permuted rows: rows [offsets[e], offsets[e+1]) use expert e."""
    offsets = np.asarray(offsets, np.int64)
    counts = np.diff(offsets)
    row_expert = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    return expert_rows(x_perm[: offsets[-1]], row_expert, w13, w2, round_h)


def combine(y: np.ndarray, slot_to_row: np.ndarray, w: np.ndarray, shared: np.ndarray | None,
            T: int, k: int) -> np.ndarray:
    """out[t] = sum_j w[t,j] * y[slot_to_row[t*k+j]] (+ shared[t]) in double."""
    yy, py = _c(y, np.float32)
    d = yy.shape[1]
    s2r, ps2r = _c(slot_to_row, np.int32)
    ww, pw = _c(w, np.float32)
    sh, psh = _c(shared, np.float32)
    out = np.empty((T, d), np.float64)
    _load().oracle_combine(py, ps2r, pw, psh, T, k, d, out.ctypes.data_as(ctypes.c_void_p))
    return out


def moe_tokens(x: np.ndarray, *, E: int, k: int, w13: np.ndarray, w2: np.ndarray,
               scores: np.ndarray | None = None, w_router: np.ndarray | None = None,
               bias: np.ndarray | None = None, n_group: int = 1, topk_group: int = 1,
               score_fn: int = SOFTMAX, routed_scale: float = 1.0,
               w13_sh: np.ndarray | None = None, w2_sh: np.ndarray | None = None,
               round_h: bool = False):
    """The whole layer for each row of ``x`` independently.

    Returns (idx [n,k] int32, w [n,k] double, out [n,d] double).  ``scores``
    (fp32 [n,E]) replaces the router scores when given.
    """
    x, xdt = _typed(x)
    n, d = x.shape
    sc, psc = _c(scores, np.float32)
    wr, pwr = _c(w_router, np.float32)
    if sc is None and wr is None:
        raise ValueError("need scores or w_router")
    b, pb = _c(bias, np.float32)
    w13, wdt = _typed(w13)
    w2, _ = _typed(w2)
    I = w2.shape[2]
    I_sh = 0
    p13s = p2s = None
    if w13_sh is not None:
        w13_sh, _ = _typed(w13_sh)
        w2_sh, _ = _typed(w2_sh)
        I_sh = w2_sh.shape[1]
        p13s = w13_sh.ctypes.data_as(ctypes.c_void_p)
        p2s = w2_sh.ctypes.data_as(ctypes.c_void_p)
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    out = np.empty((n, d), np.float64)
    rc = _load().oracle_moe_tokens(
        x.ctypes.data_as(ctypes.c_void_p), xdt, n, d, psc, pwr, pb, E, k, n_group, topk_group,
        score_fn, float(routed_scale), w13.ctypes.data_as(ctypes.c_void_p),
        w2.ctypes.data_as(ctypes.c_void_p), wdt, I, p13s, p2s, I_sh, int(round_h),
        idx.ctypes.data_as(ctypes.c_void_p), w.ctypes.data_as(ctypes.c_void_p),
        out.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("fewer than k eligible experts for some token")
    return idx, w, out
