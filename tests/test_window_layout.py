"""The verify window's buffer layout, checked on the CPU: every projection's activation arrays are
views into one flat buffer per kind (inputs, codes, scales, sums) at matching block offsets, with
the alignment the C ABI asks for, so that ONE quantize call over the flat input produces each
projection's own quantization (the quantizer works per 32-value block)."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_token_strata_gb300 import synth, window


@pytest.fixture(scope="module")
def weights():
    return window.WindowWeights(layers=2, device="cpu")


def view_offset(view: torch.Tensor, base: torch.Tensor) -> int:
    """Element offset of ``view`` inside ``base`` (asserting that it is inside)."""
    off = (view.data_ptr() - base.data_ptr()) // base.element_size()
    assert 0 <= off and off + view.numel() <= base.numel()
    return off


@pytest.mark.parametrize("T", [1, 3, 4, 8])
def test_views_offsets_and_alignment(weights, T):
    w = window.VerifyWindow(weights, T, device="cpu")
    assert w.launches_per_step() == 4
    for i, (name, rows, cols, fmt) in enumerate(w.shapes):
        assert tuple(w.x[i].shape) == (T, cols) and tuple(w.xq[i].shape) == (T, cols)
        assert tuple(w.xd[i].shape) == (T, cols // 32) and tuple(w.xs[i].shape) == (T, cols // 32)
        ox = view_offset(w.x[i], w.x_flat)
        assert ox == w.offset[i]
        assert view_offset(w.xq[i], w.q_flat) == ox
        assert view_offset(w.xd[i], w.d_flat) == ox // 32
        assert view_offset(w.xs[i], w.s_flat) == ox // 32
        assert w.xq[i].data_ptr() % 16 == 0 and w.x[i].data_ptr() % 16 == 0
        assert w.xd[i].data_ptr() % 4 == 0 and w.xs[i].data_ptr() % 4 == 0
    # the projections tile the flat input exactly, without overlap
    spans = sorted((w.offset[i], w.offset[i] + T * c) for i, (_, _, c, _) in enumerate(w.shapes))
    assert spans[0][0] == 0 and spans[-1][1] == w.x_flat.numel()
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


def test_one_quantize_over_the_flat_input_is_each_projections_own(weights):
    T = 3
    w = window.VerifyWindow(weights, T, device="cpu")
    host = w.host_inputs()
    q, d, s = oracle.quantize_act(host[None, :])
    for i, (name, rows, cols, fmt) in enumerate(w.shapes):
        qi, di, si = oracle.quantize_act(w.proj_input(host, i))
        o = w.offset[i]
        assert np.array_equal(q[0, o:o + T * cols], qi.reshape(-1)), name
        assert np.array_equal(d[0, o // 32:(o + T * cols) // 32].view(np.uint32), di.reshape(-1).view(np.uint32)), name
        assert np.array_equal(s[0, o // 32:(o + T * cols) // 32], si.reshape(-1)), name
