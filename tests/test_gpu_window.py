"""The full verify window at its real size, in the launch configurations the benchmark times (one
CUDA graph per window: grouped = one quantize launch + one grouped GEMV launch + head; chained =
quantize + GEMV per projection + head), against the oracle: every matrix on sampled rows, the
head's argmax on all tokens; graph replay bitwise equal to eager launches; both launch structures
bitwise equal to each other; T = 4 columns bitwise equal to T = 1."""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_token_strata_gb300 import strata, synth
from block_quantized_token_strata_gb300.window import VerifyWindow, WindowWeights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    from block_quantized_token_strata_gb300 import build
    build.build()
    oracle.build()
    return WindowWeights(device="cuda", host_copy=True)


def _bits(t):
    return t.view(torch.int32)


@pytest.mark.parametrize("mode", ["grouped", "chained"])
def test_full_window_t4_matches_oracle(weights, mode):
    T = 4
    win = VerifyWindow(weights, T, logits=True, mode=mode)
    host = win.host_inputs()
    win.load_inputs(host)
    win.enqueue()
    torch.cuda.synchronize()
    eager_y = [y.clone() for y in win.y]
    eager_ids = win.ids.clone()

    g = win.capture()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager_y, win.y):
        assert torch.equal(_bits(a), _bits(b))
    assert torch.equal(eager_ids, win.ids)
    assert strata.device_error() == 0

    rng = np.random.default_rng(1)
    for i, (name, rows, cols, fmt) in enumerate(weights.shapes):
        x = win.proj_input(host, i)
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


def test_grouped_launch_equals_separate_calls(weights):
    """strata_mmvq_grouped gives every matrix bitwise the output of its own strata_mmvq_multi."""
    wg = VerifyWindow(weights, 4, logits=True, mode="grouped")
    wc = VerifyWindow(weights, 4, logits=True, mode="chained")
    host = wg.host_inputs()
    wg.load_inputs(host)
    wc.load_inputs(host)
    wg.enqueue()
    wc.enqueue()
    torch.cuda.synchronize()
    for a, b in zip(wg.y, wc.y):
        assert torch.equal(_bits(a), _bits(b))
    assert torch.equal(wg.ids, wc.ids)


def test_full_window_columns_equal_single_token(weights):
    """The whole window at T = 4 vs four T = 1 windows on the same per-token inputs."""
    w4 = VerifyWindow(weights, 4, logits=True)
    host4 = w4.host_inputs()
    w4.load_inputs(host4)
    g4 = w4.capture()
    g4.replay()
    w1 = VerifyWindow(weights, 1, logits=True)
    g1 = w1.capture()
    n = len(weights.shapes)
    for t in range(4):
        h1 = np.empty(w1.x_flat.numel(), np.float32)
        for i, (_, _, c, _) in enumerate(weights.shapes):
            h1[w1.offset[i]: w1.offset[i] + c] = w4.proj_input(host4, i)[t]
        w1.load_inputs(h1)
        g1.replay()
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(_bits(w1.y[i][0]), _bits(w4.y[i][t])), (t, i)
        assert int(w1.ids[0]) == int(w4.ids[t])


@pytest.mark.parametrize("T", [8, 7])
def test_full_window_replays_clean_at_high_T(weights, T):
    """Many replays of the T = 7/8 grouped window (register-heavy, slow consumer warps): no bounded
    wait may run out (device error word stays 0) and every output equals the per-projection
    launches bit for bit."""
    wg = VerifyWindow(weights, T, logits=True, mode="grouped")
    host = wg.host_inputs()
    wg.load_inputs(host)
    strata.device_error(clear=True)
    g = wg.capture()
    for _ in range(40):
        g.replay()
    torch.cuda.synchronize()
    assert strata.device_error(clear=True) == 0
    wc = VerifyWindow(weights, T, logits=True, mode="chained")
    wc.load_inputs(host)
    wc.enqueue()
    torch.cuda.synchronize()
    assert strata.device_error(clear=True) == 0
    for a, b in zip(wg.y, wc.y):
        assert torch.equal(_bits(a), _bits(b))
    assert torch.equal(wg.ids, wc.ids)


def test_host_pipeline_matches_plain_runs(weights):
    """The end-to-end loop: each step's host input copy overlaps the previous window (two device
    input buffers, a graph each, a copy stream). Two input sets alternate over six steps; every
    step's ids equal those of a plain run on the same inputs."""
    from block_quantized_token_strata_gb300.window import HostPipeline
    w = VerifyWindow(weights, 4, mode="grouped")
    host = [w.host_inputs()]
    host.append(np.ascontiguousarray(host[0][::-1]))
    want = []
    for h in host:
        w.load_inputs(h)
        w.enqueue()
        torch.cuda.synchronize()
        want.append(w.ids.cpu().numpy().copy())
    pipe = HostPipeline(w)
    x_hosts = [torch.from_numpy(h).pin_memory() for h in host]
    ids_hosts = [torch.empty(4, dtype=torch.int32).pin_memory() for _ in range(6)]
    strata.device_error(clear=True)
    pipe.run([x_hosts[k & 1] for k in range(6)], ids_hosts)
    torch.cuda.synchronize()
    assert strata.device_error(clear=True) == 0
    for k in range(6):
        assert np.array_equal(ids_hosts[k].numpy(), want[k & 1]), k
