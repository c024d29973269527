"""The bounded device waits end by themselves: a wait on a pipeline barrier that nothing ever
completes returns after its time limit (or when the CTA's abort flag is raised), sets bits 0 and 4
of the device error word, leaves the context usable, and the word clears. The convention (an error
word the host reads, no trap) follows the collectives of dsv41-offload worker/tp2.py."""
import time

import numpy as np
import pytest
import torch

import oracle
from block_quantized_token_strata_gb300 import strata, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_quantized_token_strata_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    oracle.build()


def _gemv_ok():
    """A normal call after the time-outs: outputs within the bound of the oracle."""
    rows, cols, T = 256, 512, 3
    w = synth.make_weights(rows, cols, synth.Q4, "after-wait")
    x = synth.make_activations(T, cols, "after-wait")
    xq, xd, xs = strata.quantize_act(torch.from_numpy(x).cuda())
    y = strata.mmvq_multi(torch.from_numpy(w.buf).cuda(), rows, cols, synth.Q4, xq, xd, xs, T)
    q0, d0, _ = oracle.quantize_act(x)
    y_or, A = oracle.mmvq(w.buf, rows, cols, synth.Q4, q0, d0)
    assert (np.abs(y.cpu().numpy() - y_or) <= oracle.tolerance(A)).all()


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_wait_times_out_and_reports(limit_ns):
    torch.cuda.synchronize()
    strata.device_error(clear=True)
    assert strata.device_error(clear=False) == 0
    t0 = time.perf_counter()
    strata.wait_probe(limit_ns)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    assert el >= limit_ns * 1e-9 * 0.9            # it really waited (the barrier never completed)
    assert el < limit_ns * 1e-9 + 1.0             # and gave up by its limit
    word = strata.device_error(clear=True)
    assert word & 1 and word & 16
    assert strata.device_error(clear=False) == 0  # cleared
    _gemv_ok()
    assert strata.device_error(clear=False) == 0


def test_wait_ends_on_abort_flag():
    """A 1 s limit, but a second warp raises the abort flag after 2 ms: the wait returns early."""
    torch.cuda.synchronize()
    strata.device_error(clear=True)
    t0 = time.perf_counter()
    strata.wait_probe(1_000_000_000, 2_000_000)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    assert el < 0.5
    word = strata.device_error(clear=True)
    assert word & 1 and word & 16
    _gemv_ok()
    assert strata.device_error(clear=False) == 0
