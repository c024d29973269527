"""The C-ABI library loads, exports every call include/strata.h declares, and rejects bad arguments
on the host with the documented status codes (no GPU needed: a rejected call launches nothing)."""
import ctypes
import os
import re

import pytest

from block_quantized_token_strata_gb300 import build as strata_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "strata.h")


@pytest.fixture(scope="module")
def L():
    strata_build.build()
    from block_quantized_token_strata_gb300 import strata
    return strata.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(strata_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_error_strings(L):
    for code in range(0, -9, -1):
        s = L.strata_error_string(code)
        assert s and s != b"unknown status"
    assert L.strata_error_string(-99) == b"unknown status"


A16 = 0x10000  # fake, aligned, never dereferenced: every call below fails its host checks first


def test_weight_bytes(L):
    assert L.strata_weight_bytes(4096, 4096, 0) == 4096 * 128 * 18
    assert L.strata_weight_bytes(151936, 2048, 1) == 151936 * 64 * 34
    assert L.strata_weight_bytes(4, 33, 0) == 0
    assert L.strata_weight_bytes(4, 64, 9) == 0



@pytest.mark.parametrize("fmt,per256", [(2, 210), (3, 148), (4, 180)])
def test_superblock_formats_host_checks(L, fmt, per256):
    """Q6 / Q4K / Q5K: bytes per 256 weights, whole super-blocks only (checked before any launch),
    and the no-alloc head takes Q4 and Q8 only."""
    assert L.strata_weight_bytes(10, 512, fmt) == 10 * 2 * per256
    assert L.strata_weight_bytes(10, 288, fmt) == 0                        # 288 % 256 != 0
    assert L.strata_mmvq_multi(A16, 64, 288, fmt, A16, A16, A16, 1, A16, None) == -2
    assert L.strata_mmvq_multi(A16, 64, 512, fmt, A16, A16, A16, 9, A16, None) == -3
    assert L.strata_head_argmax_noalloc(A16, 64, 512, fmt, A16, A16, A16, 1, A16, None, None) == -4




@pytest.mark.parametrize("args,code", [
    ((0, 2048, 2048, 0, A16, A16, A16, 4, A16, None), -1),        # W NULL
    ((A16, 2048, 2048, 0, 0, A16, A16, 4, A16, None), -1),        # xq NULL
    ((A16, 2048, 2000, 0, A16, A16, A16, 4, A16, None), -2),      # cols % 32
    ((A16, 0, 2048, 0, A16, A16, A16, 4, A16, None), -2),         # rows 0
    ((A16, 2048, 2048, 0, A16, A16, A16, 0, A16, None), -3),      # T 0
    ((A16, 2048, 2048, 0, A16, A16, A16, 9, A16, None), -3),      # T 9
    ((A16, 2048, 2048, 5, A16, A16, A16, 4, A16, None), -4),      # fmt
    ((A16 + 8, 2048, 2048, 0, A16, A16, A16, 4, A16, None), -7),  # W misaligned
    ((A16, 2048, 2048, 0, A16 + 4, A16, A16, 4, A16, None), -7),  # xq misaligned
    ((A16, 2048, 65536, 0, A16, A16, A16, 4, A16, None), -2),     # T*cols above the staged maximum
])
def test_mmvq_rejects(L, args, code):
    assert L.strata_mmvq_multi(*args) == code


def test_quantize_rejects(L):
    assert L.strata_quantize_act(0, 4, 64, A16, A16, A16, None) == -1
    assert L.strata_quantize_act(A16, 4, 40, A16, A16, A16, None) == -2
    assert L.strata_quantize_act(A16, 0, 64, A16, A16, A16, None) == -2
    assert L.strata_quantize_act(A16 + 4, 4, 64, A16, A16, A16, None) == -7


def test_head_rejects(L):
    ws = L.strata_head_argmax_workspace(151936, 4)
    assert ws > 0 and L.strata_head_argmax_workspace(151936, 9) == 0
    ok = (A16, 151936, 2048, 1, A16, A16, A16, 4, A16, None, A16, ws, None)
    bad_ws = ok[:10] + (A16, ws - 1, None)
    assert L.strata_head_argmax(*bad_ws) == -8
    no_ws = ok[:10] + (None, ws, None)
    assert L.strata_head_argmax(*no_ws) == -8
    no_ids = ok[:8] + (None,) + ok[9:]
    assert L.strata_head_argmax(*no_ids) == -1
    badT = ok[:7] + (0,) + ok[8:]
    assert L.strata_head_argmax(*badT) == -3


def test_moe_rejects(L):
    ws = L.strata_moe_grouped_workspace(128, 3256, 8, 2048, 768)
    assert ws > 3256 * 8 * 768
    assert L.strata_moe_grouped_workspace(128, 3256, 8, 2000, 768) == 0
    ok = [A16, 128, 2048, 768, A16, 3256, 8, A16, A16, A16, ws, None, None]
    a = list(ok); a[0] = None
    assert L.strata_moe_grouped(*a) == -1
    a = list(ok); a[2] = 2000
    assert L.strata_moe_grouped(*a) == -2
    a = list(ok); a[6] = 17
    assert L.strata_moe_grouped(*a) == -2
    a = list(ok); a[10] = ws - 1
    assert L.strata_moe_grouped(*a) == -8
    a = list(ok); a[9] = A16 + 16
    assert L.strata_moe_grouped(*a) == -7


def test_moe_debug_views(L):
    out = (ctypes.c_size_t * 7)()
    assert L.strata_moe_debug_views(128, 3256, 8, 2048, 768, ctypes.cast(out, ctypes.c_void_p)) == 0
    vals = list(out)
    assert vals == sorted(vals) and all(v % 256 == 0 for v in vals)
    assert vals[6] == L.strata_moe_grouped_workspace(128, 3256, 8, 2048, 768)


def test_gemm_rejects(L):
    ok = [A16, 256, 512, A16, A16, 300, A16, None]
    assert L.strata_gemm_q4(*ok[:0], None, 256, 512, A16, A16, 300, A16, None) == -1
    a = list(ok); a[1] = 200
    assert L.strata_gemm_q4(*a) == -2                 # rows % 128
    a = list(ok); a[2] = 96
    assert L.strata_gemm_q4(*a) == -2                 # cols % 64
    a = list(ok); a[5] = 0
    assert L.strata_gemm_q4(*a) == -2                 # no rows of activations
    a = list(ok); a[3] = A16 + 8
    assert L.strata_gemm_q4(*a) == -7                 # xq alignment
    a = list(ok); a[6] = A16 + 4
    assert L.strata_gemm_q4(*a) == -7                 # y alignment


def test_head_vocab_limit(L):
    """The head keeps a candidate's token in bits 27-29 of its row id, so every head entry point
    rejects vocab >= 2^27 on the host (before the workspace check, before any launch)."""
    V = 1 << 27
    big = 1 << 40
    assert L.strata_head_argmax(A16, V, 2048, 1, A16, A16, A16, 4, A16, None, A16, big, None) == -2
    assert L.strata_head_argmax(A16, V + 1, 2048, 1, A16, A16, A16, 4, A16, None, A16, big, None) == -2
    assert L.strata_head_argmax_margin(A16, V, 2048, 1, A16, A16, A16, 4, A16, A16, None, A16, big, None) == -2
    assert L.strata_head_argmax_noalloc(A16, V, 2048, 1, A16, A16, A16, 4, A16, None, None) == -2


def test_head_staged_activation_limit(L):
    """Q8 with cols 16384 at T = 8: T*cols is at the staged maximum but the activation records and one
    four-row slot do not fit shared memory; both head entry points say STRATA_ERR_SHAPE."""
    ws = L.strata_head_argmax_workspace(1000, 8)
    assert L.strata_head_argmax(A16, 1000, 16384, 1, A16, A16, A16, 8, A16, None, A16, ws, None) == -2
    assert L.strata_head_argmax_noalloc(A16, 1000, 16384, 1, A16, A16, A16, 8, A16, None, None) == -2
    assert L.strata_mmvq_multi(A16, 1000, 16384, 1, A16, A16, A16, 8, A16, None) == -2


def test_wait_probe_rejects(L):
    assert L.strata_wait_probe(0, -1, None) == -2
    assert L.strata_wait_probe(2_000_000_000, -1, None) == -2
    assert L.strata_wait_probe(1_000_000, 2_000_000_000, None) == -2


def test_moe_gate_up_hook_rejects(L):
    ws = L.strata_moe_grouped_workspace(128, 3256, 8, 2048, 768)
    ok = [A16, 128, 2048, 768, A16, 3256, 8, A16, A16, A16, ws, None, A16, None]
    a = list(ok); a[12] = None
    assert L.strata_moe_grouped_gu(*a) == -1
    a = list(ok); a[12] = A16 + 4
    assert L.strata_moe_grouped_gu(*a) == -7
    a = list(ok); a[10] = ws - 1
    assert L.strata_moe_grouped_gu(*a) == -8


def test_gemm_dequant_rejects(L):
    ws = L.strata_gemm_q4_dequant_workspace(6144, 2048, 3259)
    assert ws >= 48 * 64 * 8192 + 26 * 64 * 8192
    assert L.strata_gemm_q4_dequant_workspace(200, 2048, 10) == 0
    ok = [A16, 256, 512, A16, A16, 300, A16, A16, 1 << 30, None]
    a = list(ok); a[0] = None
    assert L.strata_gemm_q4_dequant(*a) == -1
    a = list(ok); a[1] = 200
    assert L.strata_gemm_q4_dequant(*a) == -2
    a = list(ok); a[8] = 16
    assert L.strata_gemm_q4_dequant(*a) == -8
    a = list(ok); a[7] = A16 + 64
    assert L.strata_gemm_q4_dequant(*a) == -7
