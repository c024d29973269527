"""CPU oracle of the block-quantized verify path (plain C, fp64), with numpy wrappers.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package; the product path never does. It shares no code with the CUDA library.
The C source (``strata_oracle.c``) states each function's definition and the passage it follows.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` against values the
pages and mathematics fix (hand-computed one-block cases, brute-force dense fp64 matmuls of the
dequantized operands, closed-form quantizer cases, invariants, golden fixtures).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "strata_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q4, Q8 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no fp contraction, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.or_half_to_double.argtypes = [ctypes.c_uint16]
            lib.or_half_to_double.restype = ctypes.c_double
            lib.or_quantize_act.argtypes = [P, I64, I64, P, P, P]
            lib.or_block_dots.argtypes = [P, I64, I64, I, P, I64, P]
            lib.or_mmvq.argtypes = [P, I64, I64, I, P, P, I64, P, P]
            lib.or_mmvq_rows.argtypes = [P, I64, I64, I, P, P, I64, P, I64, P, P]
            lib.or_argmax.argtypes = [P, I64, I64, P]
            lib.or_margin.argtypes = [P, I64, I64, P]
            lib.or_moe_bucket.argtypes = [P, I64, I, I, P, P, P]
            lib.or_moe_bucket.restype = I64
            lib.or_moe_rows.argtypes = [P, P, P, I, I64, I64, P, I64, I, P, P, I64, P, P, P, P, P, P, P, P,
                                        P, P, P, P]
            lib.or_set_threads.argtypes = [I]
            lib.or_get_threads.restype = I
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int) -> None:
    _load().or_set_threads(int(n))


def get_threads() -> int:
    return int(_load().or_get_threads())


def half_to_double(bits: int) -> float:
    return float(_load().or_half_to_double(int(bits) & 0xFFFF))


def quantize_act(x: np.ndarray):
    """x fp32 [n][cols] -> (q int8 [n][cols], d fp32 [n][cols/32], s int32 [n][cols/32])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    n, cols = x.shape
    assert cols % 32 == 0
    q = np.empty((n, cols), np.int8)
    d = np.empty((n, cols // 32), np.float32)
    s = np.empty((n, cols // 32), np.int32)
    _load().or_quantize_act(_p(x), n, cols, _p(q), _p(d), _p(s))
    return q, d, s


def block_dots(W, rows, cols, fmt, xq) -> np.ndarray:
    """isum int64 [T][rows][cols/32]."""
    W = _c(W, np.uint8)
    xq = _c(xq, np.int8).reshape(-1, cols)
    T = xq.shape[0]
    out = np.empty((T, rows, cols // 32), np.int64)
    _load().or_block_dots(_p(W), rows, cols, fmt, _p(xq), T, _p(out))
    return out


def mmvq(W, rows, cols, fmt, xq, xd):
    """(y fp64 [T][rows], A fp64 [T][rows]) with A = sum of |block terms|."""
    W = _c(W, np.uint8)
    xq = _c(xq, np.int8).reshape(-1, cols)
    xd = _c(xd, np.float32).reshape(-1, cols // 32)
    T = xq.shape[0]
    y = np.empty((T, rows), np.float64)
    A = np.empty((T, rows), np.float64)
    _load().or_mmvq(_p(W), rows, cols, fmt, _p(xq), _p(xd), T, _p(y), _p(A))
    return y, A


def mmvq_rows(W, rows, cols, fmt, xq, xd, sel):
    """Like mmvq for the listed rows only: (y [T][len(sel)], A [T][len(sel)])."""
    W = _c(W, np.uint8)
    xq = _c(xq, np.int8).reshape(-1, cols)
    xd = _c(xd, np.float32).reshape(-1, cols // 32)
    sel = _c(sel, np.int64)
    T = xq.shape[0]
    y = np.empty((T, sel.size), np.float64)
    A = np.empty((T, sel.size), np.float64)
    _load().or_mmvq_rows(_p(W), rows, cols, fmt, _p(xq), _p(xd), T, _p(sel), sel.size, _p(y), _p(A))
    return y, A


def argmax(v) -> np.ndarray:
    v = _c(v, np.float64)
    if v.ndim == 1:
        v = v[None, :]
    T, n = v.shape
    ids = np.empty(T, np.int32)
    _load().or_argmax(_p(v), T, n, _p(ids))
    return ids


def margin(v) -> np.ndarray:
    """Top-1 minus top-2 per row (a repeated maximum gives 0, a single value +inf), fp64 [T]."""
    v = _c(v, np.float64)
    if v.ndim == 1:
        v = v[None, :]
    T, n = v.shape
    out = np.empty(T, np.float64)
    _load().or_margin(_p(v), T, n, _p(out))
    return out


def head_argmax(W, vocab, cols, fmt, xq, xd):
    """(ids int32 [T], logits fp64 [T][vocab], A fp64 [T][vocab])."""
    y, A = mmvq(W, vocab, cols, fmt, xq, xd)
    return argmax(y), y, A


def moe_bucket(ids: np.ndarray, n_expert: int):
    ids = _c(ids, np.int32)
    n_tok, k = ids.shape
    counts = np.empty(n_expert, np.int32)
    offsets = np.empty(n_expert + 1, np.int32)
    pairs = np.full(n_tok * k, -1, np.int32)
    bad = _load().or_moe_bucket(_p(ids), n_tok, k, n_expert, _p(counts), _p(offsets), _p(pairs))
    return counts, offsets, pairs, int(bad)


def moe_rows(experts, hidden, inter, ids, x, sel, want_hidden=False, hq_in=None, hd_in=None,
             want_gate_up=False):
    """MoE output rows for the pairs ``sel`` (p = tok*k + slot).

    ``experts``: list of (gate_buf, up_buf, down_buf) uint8 planar Q4 buffers.
    Returns dict with y, A (fp64 [n_sel][hidden]) and, with want_hidden, h (fp64 [n_sel][inter])
    and its quantization hq/hd/hs. With want_gate_up also g, u (fp64 [n_sel][inter]) and their
    tolerance masses Ag, Au. With hq_in/hd_in the down projection uses those rows.
    """
    ids = _c(ids, np.int32)
    n_tok, k = ids.shape
    x = _c(x, np.float32)
    sel = _c(sel, np.int64)
    n_sel = sel.size
    bufs = [[_c(b, np.uint8) for b in ex] for ex in experts]
    n_expert = len(bufs)
    arr = [(ctypes.c_void_p * n_expert)(*[b[j].ctypes.data for b in bufs]) for j in range(3)]
    y = np.empty((n_sel, hidden), np.float64)
    A = np.empty((n_sel, hidden), np.float64)
    out = {"y": y, "A": A}
    h = hq = hd = hs = None
    if want_hidden:
        h = np.empty((n_sel, inter), np.float64)
        hq = np.empty((n_sel, inter), np.int8)
        hd = np.empty((n_sel, inter // 32), np.float32)
        hs = np.empty((n_sel, inter // 32), np.int32)
        out.update(h=h, hq=hq, hd=hd, hs=hs)
    g = u = ag = au = None
    if want_gate_up:
        g, u, ag, au = (np.empty((n_sel, inter), np.float64) for _ in range(4))
        out.update(g=g, u=u, Ag=ag, Au=au)
    hq_in = None if hq_in is None else _c(hq_in, np.int8)
    hd_in = None if hd_in is None else _c(hd_in, np.float32)
    _load().or_moe_rows(ctypes.cast(arr[0], ctypes.c_void_p), ctypes.cast(arr[1], ctypes.c_void_p),
                        ctypes.cast(arr[2], ctypes.c_void_p), n_expert, hidden, inter, _p(ids), n_tok, k,
                        _p(x), _p(sel), n_sel, _p(y), _p(A), _p(h), _p(hq), _p(hd), _p(hs),
                        _p(hq_in), _p(hd_in), _p(g), _p(u), _p(ag), _p(au))
    return out


def tolerance(A):
    """The fp32 output bound: |gpu - oracle| <= 2e-6 * sum|block terms| + 1e-6."""
    return 2e-6 * np.asarray(A) + 1e-6
