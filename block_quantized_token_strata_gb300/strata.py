"""Thin ctypes binding of libstrata (the C ABI in include/strata.h).

Argument marshalling only: every step runs in the CUDA kernels behind the C calls. Tensors are
torch CUDA tensors (torch supplies device memory and the current stream); raw-pointer variants
take integers. If the library has not been built, the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

Q4, Q8 = 0, 1
MAX_T = 8
_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libstrata.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "OK", -1: "ERR_NULL", -2: "ERR_SHAPE", -3: "ERR_T", -4: "ERR_FMT", -5: "ERR_CUDA",
          -6: "ERR_EXPERT", -7: "ERR_ALIGN", -8: "ERR_WORKSPACE"}


class GemvDesc(ctypes.Structure):
    """strata_gemv_desc of include/strata.h."""
    _fields_ = [("W", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("xq", ctypes.c_void_p), ("xd", ctypes.c_void_p), ("xs", ctypes.c_void_p),
                ("y", ctypes.c_void_p)]


class StrataError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({STATUS.get(status, '?')})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libstrata.so (in-tree). Raises if it is missing: build it with __graft_entry__.build()."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.strata_error_string.argtypes = [I]
            L.strata_error_string.restype = ctypes.c_char_p
            L.strata_weight_bytes.argtypes = [I64, I64, I]
            L.strata_weight_bytes.restype = SZ
            L.strata_quantize_act.argtypes = [P, I64, I64, P, P, P, P]
            L.strata_mmvq_multi.argtypes = [P, I64, I64, I, P, P, P, I, P, P]
            L.strata_head_argmax_workspace.argtypes = [I64, I]
            L.strata_head_argmax_workspace.restype = SZ
            L.strata_head_argmax.argtypes = [P, I64, I64, I, P, P, P, I, P, P, P, SZ, P]
            L.strata_moe_grouped_workspace.argtypes = [I, I64, I, I64, I64]
            L.strata_moe_grouped_workspace.restype = SZ
            L.strata_moe_grouped.argtypes = [P, I, I64, I64, P, I64, I, P, P, P, SZ, P, P]
            L.strata_moe_debug_views.argtypes = [I, I64, I, I64, I64, P]
            L.strata_block_dots.argtypes = [P, I64, I64, I, P, P, I, P, P]
            L.strata_mmvq_grouped.argtypes = [P, I, I, I, P]
            L.strata_device_error.argtypes = [P, I]
            L.strata_head_argmax_noalloc.argtypes = [P, I64, I64, I, P, P, P, I, P, P, P]
            L.strata_head_argmax_margin.argtypes = [P, I64, I64, I, P, P, P, I, P, P, P, P, SZ, P]
            L.strata_gemm_q4.argtypes = [P, I64, I64, P, P, I64, P, P]
            L.strata_moe_grouped_gu.argtypes = [P, I, I64, I64, P, I64, I, P, P, P, SZ, P, P, P]
            L.strata_wait_probe.argtypes = [I64, I64, P]
            L.strata_gemm_q4_dequant_workspace.argtypes = [I64, I64, I64]
            L.strata_gemm_q4_dequant_workspace.restype = SZ
            L.strata_gemm_q4_dequant.argtypes = [P, I64, I64, P, P, I64, P, P, SZ, P]
            for name in ("strata_quantize_act", "strata_mmvq_multi", "strata_head_argmax",
                         "strata_moe_grouped", "strata_moe_debug_views", "strata_block_dots",
                         "strata_mmvq_grouped", "strata_device_error", "strata_head_argmax_noalloc",
                         "strata_head_argmax_margin", "strata_gemm_q4", "strata_moe_grouped_gu",
                         "strata_wait_probe", "strata_gemm_q4_dequant"):
                getattr(L, name).restype = I
            _lib = L
    return _lib


def error_string(status: int) -> str:
    return lib().strata_error_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != 0:
        raise StrataError(status, f"{what} ({error_string(status)})")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def weight_bytes(rows: int, cols: int, fmt: int) -> int:
    return int(lib().strata_weight_bytes(rows, cols, fmt))


def quantize_act(x: torch.Tensor, xq=None, xd=None, xs=None, stream=None):
    """x fp32 [n][cols] (CUDA) -> (xq int8 [n][cols], xd fp32 [n][cols/32], xs int32 [n][cols/32])."""
    n, cols = x.shape
    dev = x.device
    xq = torch.empty((n, cols), dtype=torch.int8, device=dev) if xq is None else xq
    xd = torch.empty((n, cols // 32), dtype=torch.float32, device=dev) if xd is None else xd
    xs = torch.empty((n, cols // 32), dtype=torch.int32, device=dev) if xs is None else xs
    _check(lib().strata_quantize_act(_ptr(x), n, cols, _ptr(xq), _ptr(xd), _ptr(xs), _stream(stream)),
           "strata_quantize_act")
    return xq, xd, xs


def mmvq_multi(W, rows: int, cols: int, fmt: int, xq, xd, xs, T: int, y=None, stream=None):
    """y fp32 [T][rows] = block-quantized W [rows][cols] times T quantized activation rows."""
    if y is None:
        y = torch.empty((T, rows), dtype=torch.float32, device=xq.device)
    _check(lib().strata_mmvq_multi(_ptr(W), rows, cols, fmt, _ptr(xq), _ptr(xd), _ptr(xs), T, _ptr(y),
                                   _stream(stream)), "strata_mmvq_multi")
    return y


def gemv_descs(problems) -> ctypes.Array:
    """A strata_gemv_desc array from (W, rows, cols, xq, xd, xs, y) tuples (tensors or ints)."""
    arr = (GemvDesc * len(problems))()
    for i, (W, rows, cols, xq, xd, xs, y) in enumerate(problems):
        arr[i] = GemvDesc(_ptr(W), rows, cols, _ptr(xq), _ptr(xd), _ptr(xs), _ptr(y))
    return arr


def mmvq_grouped(descs, fmt: int, T: int, stream=None) -> None:
    """Run many independent T-column GEMVs (a gemv_descs array or a list of tuples) in one launch."""
    if not isinstance(descs, ctypes.Array):
        descs = gemv_descs(descs)
    _check(lib().strata_mmvq_grouped(ctypes.cast(descs, ctypes.c_void_p), len(descs), fmt, T, _stream(stream)),
           "strata_mmvq_grouped")


def device_error(clear: bool = True) -> int:
    """The library's device error word (bit 0: a bounded wait in a kernel ran out)."""
    out = ctypes.c_int(0)
    _check(lib().strata_device_error(ctypes.byref(out), int(clear)), "strata_device_error")
    return out.value


def wait_probe(limit_ns: int, abort_after_ns: int = -1, stream=None) -> None:
    """Enqueue the bounded-wait probe (a wait nothing completes; it must end by its limit or abort)."""
    _check(lib().strata_wait_probe(int(limit_ns), int(abort_after_ns), _stream(stream)), "strata_wait_probe")


def head_argmax_workspace(vocab: int, T: int) -> int:
    return int(lib().strata_head_argmax_workspace(vocab, T))


def head_argmax(W, vocab: int, cols: int, fmt: int, xq, xd, xs, T: int, ids=None, logits=None,
                workspace=None, stream=None):
    """ids int32 [T] (argmax per token, ties to the lowest id); logits [T][vocab] written if given."""
    dev = xq.device
    if ids is None:
        ids = torch.empty(T, dtype=torch.int32, device=dev)
    need = head_argmax_workspace(vocab, T)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else need
    _check(lib().strata_head_argmax(_ptr(W), vocab, cols, fmt, _ptr(xq), _ptr(xd), _ptr(xs), T, _ptr(ids),
                                    _ptr(logits), _ptr(workspace), ws_bytes, _stream(stream)),
           "strata_head_argmax")
    return ids


def head_argmax_margin(W, vocab: int, cols: int, fmt: int, xq, xd, xs, T: int, ids=None, margin=None,
                       logits=None, workspace=None, stream=None):
    """(ids int32 [T], margin fp32 [T]): the argmax per token and its top-1 minus top-2 logit."""
    dev = xq.device
    if ids is None:
        ids = torch.empty(T, dtype=torch.int32, device=dev)
    if margin is None:
        margin = torch.empty(T, dtype=torch.float32, device=dev)
    need = head_argmax_workspace(vocab, T)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else need
    _check(lib().strata_head_argmax_margin(_ptr(W), vocab, cols, fmt, _ptr(xq), _ptr(xd), _ptr(xs), T, _ptr(ids),
                                           _ptr(margin), _ptr(logits), _ptr(workspace), ws_bytes, _stream(stream)),
           "strata_head_argmax_margin")
    return ids, margin


def gemm_q4(W, rows: int, cols: int, xq, xd, y=None, stream=None):
    """y fp32 [n_tok][rows] = the block-quantized product of n_tok activation rows with a Q4 matrix."""
    n_tok = xq.shape[0]
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=xq.device)
    _check(lib().strata_gemm_q4(_ptr(W), rows, cols, _ptr(xq), _ptr(xd), n_tok, _ptr(y), _stream(stream)),
           "strata_gemm_q4")
    return y


def gemm_q4_dequant_workspace(rows: int, cols: int, n_tok: int) -> int:
    return int(lib().strata_gemm_q4_dequant_workspace(rows, cols, n_tok))


def gemm_q4_dequant(W, rows: int, cols: int, xq, xd, y=None, workspace=None, stream=None):
    """The dense prompt GEMM's wide-dequant arm: same result as gemm_q4, bit for bit."""
    n_tok = xq.shape[0]
    if y is None:
        y = torch.empty((n_tok, rows), dtype=torch.float32, device=xq.device)
    need = gemm_q4_dequant_workspace(rows, cols, n_tok)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=xq.device)
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else need
    _check(lib().strata_gemm_q4_dequant(_ptr(W), rows, cols, _ptr(xq), _ptr(xd), n_tok, _ptr(y), _ptr(workspace),
                                        ws_bytes, _stream(stream)), "strata_gemm_q4_dequant")
    return y


def block_dots(W, rows: int, cols: int, fmt: int, xq, xs, T: int, isum=None, stream=None):
    if isum is None:
        isum = torch.empty((T, rows, cols // 32), dtype=torch.int32, device=xq.device)
    _check(lib().strata_block_dots(_ptr(W), rows, cols, fmt, _ptr(xq), _ptr(xs), T, _ptr(isum),
                                   _stream(stream)), "strata_block_dots")
    return isum


def moe_grouped_workspace(n_expert: int, n_tok: int, k: int, hidden: int, inter: int) -> int:
    return int(lib().strata_moe_grouped_workspace(n_expert, n_tok, k, hidden, inter))


def moe_debug_views(n_expert: int, n_tok: int, k: int, hidden: int, inter: int) -> dict:
    out = (ctypes.c_size_t * 7)()
    _check(lib().strata_moe_debug_views(n_expert, n_tok, k, hidden, inter, ctypes.cast(out, ctypes.c_void_p)),
           "strata_moe_debug_views")
    return dict(zip(("counts", "offsets", "pairs", "hq", "hd", "hs", "total"), [int(v) for v in out]))


def expert_table(experts, device) -> torch.Tensor:
    """Device array of strata_expert {gate, up, down} from a list of (gate, up, down) tensors."""
    ptrs = [int(_ptr(m)) for ex in experts for m in ex]
    return torch.tensor(ptrs, dtype=torch.int64).to(device)


def moe_grouped(expert_tab, n_expert: int, hidden: int, inter: int, ids, x, y=None, workspace=None,
                err_word=None, stream=None, gu=None):
    """y fp32 [n_tok*k][hidden]: one row per (token, slot) pair, grouped expert GEMMs inside. With
    ``gu`` (fp32 [n_tok*k][2][inter]) the test-hook entry point also writes each pair's g and u."""
    n_tok, k = ids.shape
    dev = x.device
    if y is None:
        y = torch.empty((n_tok * k, hidden), dtype=torch.float32, device=dev)
    need = moe_grouped_workspace(n_expert, n_tok, k, hidden, inter)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else need
    if gu is None:
        _check(lib().strata_moe_grouped(_ptr(expert_tab), n_expert, hidden, inter, _ptr(ids), n_tok, k, _ptr(x),
                                        _ptr(y), _ptr(workspace), ws_bytes, _ptr(err_word), _stream(stream)),
               "strata_moe_grouped")
    else:
        _check(lib().strata_moe_grouped_gu(_ptr(expert_tab), n_expert, hidden, inter, _ptr(ids), n_tok, k,
                                           _ptr(x), _ptr(y), _ptr(workspace), ws_bytes, _ptr(err_word), _ptr(gu),
                                           _stream(stream)), "strata_moe_grouped_gu")
    return y
