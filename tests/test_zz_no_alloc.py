"""strata_head_argmax_noalloc, the head + argmax entry point for callers that cannot allocate device
memory (a plugin whose host application owns all device memory, a server that fixes its memory at
start-up): called through the C ABI twice in a row per format, each time checked against
strata_head_argmax with a caller-provided workspace. Both run the same kernels with the same
summation order, so the logits must be equal bit for bit and the ids equal; the logits are also
within the oracle's fp32 bound. This file is collected last on purpose: it passes alone in a fresh
process and after the others."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_quantized_token_strata_gb300 import strata, synth

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    from block_quantized_token_strata_gb300 import build
    build.build()
    L = strata.lib()
    fn = L.strata_head_argmax_noalloc
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [P, I64, I64, I, P, P, P, I, P, P, P]
    fn.restype = I
    return fn


@pytest.mark.parametrize("fmt,vocab", [(synth.Q8, synth.HEAD_VOCAB), (synth.Q4, 50021)])
def test_noalloc_head_matches_workspace_entry_point_twice(fmt, vocab):
    fn = _noalloc_fn()
    oracle.build()
    cols = synth.WINDOW_HIDDEN
    w = synth.make_weights(vocab, cols, fmt, "noalloc")
    W = torch.from_numpy(w.buf).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    for call, T in enumerate((4, 8)):                      # two calls in a row, different inputs
        x = synth.make_activations(T, cols, "noalloc", call)
        xq_h, xd_h, xs_h = oracle.quantize_act(x)
        xq, xd, xs = (torch.from_numpy(a).cuda() for a in (xq_h, xd_h, xs_h))
        lg_ref = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
        ids_ref = strata.head_argmax(W, vocab, cols, fmt, xq, xd, xs, T, logits=lg_ref)
        lg = torch.full((T, vocab), float("nan"), dtype=torch.float32, device="cuda")
        ids = torch.full((T,), -1, dtype=torch.int32, device="cuda")
        rc = fn(W.data_ptr(), vocab, cols, fmt, xq.data_ptr(), xd.data_ptr(), xs.data_ptr(), T,
                ids.data_ptr(), lg.data_ptr(), stream)
        assert rc == 0, strata.error_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(ids.cpu(), ids_ref.cpu())
        assert torch.equal(lg.view(torch.int32), lg_ref.view(torch.int32))   # same kernels, same order
        y_or, A = oracle.mmvq_rows(w.buf, vocab, cols, fmt, xq_h, xd_h, np.arange(0, vocab, 97))
        a = lg.cpu().numpy()[:, ::97]
        assert (np.abs(a.astype(np.float64) - y_or) <= oracle.tolerance(A)).all()


def test_noalloc_rejects_without_launch():
    fn = _noalloc_fn()
    A16 = 0x10000
    assert fn(None, 100, 64, 1, A16, A16, A16, 1, A16, None, None) == -1      # NULL W
    assert fn(A16, 100, 64, 1, A16, A16, A16, 9, A16, None, None) == -3       # T out of range
    assert fn(A16, 100, 64, 1, A16 + 1, A16, A16, 1, A16, None, None) == -7   # misaligned xq
    assert fn(A16, 1 << 27, 64, 1, A16, A16, A16, 1, A16, None, None) == -2   # vocab at the id-field limit
    assert fn(A16, 1000, 16384, 1, A16, A16, A16, 8, A16, None, None) == -2   # staged activations too big
