"""The full verify window at its real size, in the launch configuration the benchmark times (one
CUDA graph of quantize + GEMV per projection, then the head with its argmax), against the oracle:
every matrix on sampled rows, the head's argmax on all tokens; graph replay bitwise equal to
eager launches; T = 4 columns bitwise equal to T = 1."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_token_strata_gb300 import synth
from block_quantized_token_strata_gb300.window import VerifyWindow, WindowWeights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    from block_quantized_token_strata_gb300 import build
    build.build()
    oracle.build()
    return WindowWeights(device="cuda", host_copy=True)


def test_full_window_t4_matches_oracle(weights):
    T = 4
    win = VerifyWindow(weights, T, logits=True)
    host = win.host_inputs()
    win.load_inputs(host)
    win.enqueue()
    torch.cuda.synchronize()
    eager_y = [y.clone() if y is not None else None for y in win.y]
    eager_ids = win.ids.clone()

    g = win.capture()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager_y, win.y):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(eager_ids, win.ids)

    rng = np.random.default_rng(1)
    off = 0
    for i, (name, rows, cols, fmt) in enumerate(weights.shapes):
        x = host[off: off + T * cols].reshape(T, cols)
        off += T * cols
        xq, xd, xs = oracle.quantize_act(x)
        assert np.array_equal(xq, win.xq[i].cpu().numpy())
        w = weights.host[i]
        if name == "head":
            ids_or, lg_or, A = oracle.head_argmax(w.buf, rows, cols, fmt, xq, xd)
            lg = win.y[i].cpu().numpy()
            tol = oracle.tolerance(A)
            assert (np.abs(lg - lg_or) <= tol).all()
            ids = win.ids.cpu().numpy()
            for t in range(T):
                m = ids_or[t]
                band = tol[t] + tol[t, m]
                ok = set(np.nonzero(lg_or[t] >= lg_or[t, m] - band)[0].tolist())
                assert ids[t] in ok and ids[t] == int(np.argmax(lg[t]))
            continue
        sel = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 6, replace=False)]))
        y_or, A = oracle.mmvq_rows(w.buf, rows, cols, fmt, xq, xd, sel)
        y = win.y[i].cpu().numpy()[:, sel]
        assert (np.abs(y - y_or) <= oracle.tolerance(A)).all(), name


def test_full_window_columns_equal_single_token(weights):
    """The whole window at T = 4 vs four T = 1 windows on the same per-token inputs."""
    w4 = VerifyWindow(weights, 4, logits=True)
    host4 = w4.host_inputs()
    w4.load_inputs(host4)
    g4 = w4.capture()
    g4.replay()
    w1 = VerifyWindow(weights, 1, logits=True)
    g1 = w1.capture()
    cols = [c for _, _, c, _ in weights.shapes]
    for t in range(4):
        parts, off = [], 0
        for c in cols:
            parts.append(host4[off + t * c: off + (t + 1) * c])
            off += 4 * c
        w1.load_inputs(np.concatenate(parts))
        g1.replay()
        torch.cuda.synchronize()
        for i in range(len(cols)):
            assert torch.equal(w1.y[i][0].view(torch.int32), w4.y[i][t].view(torch.int32)), (t, i)
        assert int(w1.ids[0]) == int(w4.ids[t])
