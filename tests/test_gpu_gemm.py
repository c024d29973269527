"""GPU parity of the dense prompt-chunk GEMM (strata_gemm_q4, tensor cores) against the CPU oracle.

The definition is the GEMV's with one column per activation row: y[n][r] = sum_b (d_w * xd) * isum,
so the oracle's T-column product is the reference (T = the number of rows). Bar: every output within
|gpu - oracle| <= 2e-6 * sum|block terms| + 1e-6.
"""
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


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(rows, cols, n_tok, key, outliers=False):
    w = synth.make_weights(rows, cols, synth.Q4, key)
    x = synth.make_activations(n_tok, cols, key, outliers=outliers)
    xq, xd, xs = strata.quantize_act(cu(x))
    y = torch.full((n_tok, rows), float("nan"), device="cuda")
    strata.gemm_q4(cu(w.buf), rows, cols, xq, xd, y=y)
    torch.cuda.synchronize()
    return w, xq.cpu().numpy(), xd.cpu().numpy(), y.cpu().numpy()


@pytest.mark.parametrize("rows,cols,n_tok", [(256, 512, 300), (128, 64, 1), (384, 2048, 128), (128, 4096, 129)])
def test_gemm_full_parity(rows, cols, n_tok):
    """Every output of small cases: ragged M-tiles (300 = 2 x 128 + 44, 129), a one-row prompt, the
    narrowest K (2 quant blocks)."""
    w, xq, xd, y = run(rows, cols, n_tok, "gemm-full", outliers=True)
    y_or, A = oracle.mmvq(w.buf, rows, cols, synth.Q4, xq, xd)
    tol = oracle.tolerance(A)
    err = np.abs(y.astype(np.float64) - y_or)
    assert not np.isnan(y).any()
    assert (err <= tol).all(), f"{(err > tol).sum()} outside the bound"


def test_gemm_prompt_chunk_sampled_rows():
    """The 3,259-token prompt chunk against the window's FFN up projection (6144 x 2048): every token
    on a seeded sample of 96 weight rows (every N-tile touched)."""
    rows, cols, n_tok = 6144, 2048, 3259
    w, xq, xd, y = run(rows, cols, n_tok, "gemm-prompt")
    rng = np.random.default_rng(1)
    sel = np.unique(np.concatenate([rng.choice(rows, 64, replace=False), np.arange(0, rows, 128) + 127]))
    y_or, A = oracle.mmvq_rows(w.buf, rows, cols, synth.Q4, xq, xd, sel)
    err = np.abs(y[:, sel].astype(np.float64) - y_or)
    assert not np.isnan(y).any()
    assert (err <= oracle.tolerance(A)).all()


def test_gemm_agrees_with_the_gemv_within_bounds():
    """Same inputs through strata_mmvq_multi (8 columns): each within the bound of the oracle, so the
    two differ by at most twice the bound."""
    rows, cols, T = 512, 1024, 8
    w, xq, xd, y = run(rows, cols, T, "gemm-vs-gemv")
    xs = strata.quantize_act(cu(synth.make_activations(T, cols, "gemm-vs-gemv")))[2]
    yv = strata.mmvq_multi(cu(w.buf), rows, cols, synth.Q4, cu(xq), cu(xd), xs, T).cpu().numpy()
    _, A = oracle.mmvq(w.buf, rows, cols, synth.Q4, xq, xd)
    assert (np.abs(y.astype(np.float64) - yv) <= 2 * oracle.tolerance(A)).all()


def run_dequant(rows, cols, n_tok, key, outliers=False):
    """The same inputs through both arms: (w, xq, xd, y of the no-dequant arm, y of the wide-dequant arm)."""
    w = synth.make_weights(rows, cols, synth.Q4, key)
    x = synth.make_activations(n_tok, cols, key, outliers=outliers)
    xq, xd, _ = strata.quantize_act(cu(x))
    W = cu(w.buf)
    y0 = torch.full((n_tok, rows), float("nan"), device="cuda")
    y1 = torch.full((n_tok, rows), float("nan"), device="cuda")
    strata.gemm_q4(W, rows, cols, xq, xd, y=y0)
    strata.gemm_q4_dequant(W, rows, cols, xq, xd, y=y1)
    torch.cuda.synchronize()
    return w, xq.cpu().numpy(), xd.cpu().numpy(), y0, y1


@pytest.mark.parametrize("rows,cols,n_tok", [(256, 512, 300), (128, 64, 1), (384, 2048, 128), (128, 4096, 129)])
def test_gemm_dequant_arm_full_parity(rows, cols, n_tok):
    """The wide-dequant arm (fp16 operand tiles prepared once per call, streamed by bulk copies): every
    output within the oracle's bound, and bit for bit the no-dequant arm's (same block arithmetic,
    same order)."""
    w, xq, xd, y0, y1 = run_dequant(rows, cols, n_tok, "gemm-dq", outliers=True)
    assert torch.equal(y1.view(torch.int32), y0.view(torch.int32))
    y = y1.cpu().numpy()
    y_or, A = oracle.mmvq(w.buf, rows, cols, synth.Q4, xq, xd)
    err = np.abs(y.astype(np.float64) - y_or)
    assert not np.isnan(y).any()
    assert (err <= oracle.tolerance(A)).all(), f"{(err > oracle.tolerance(A)).sum()} outside the bound"


def test_gemm_dequant_arm_prompt_chunk():
    """The 3,259-token chunk x 6144 x 2048: the two arms bit for bit equal everywhere, a sample of rows
    against the oracle, and no error bit."""
    rows, cols, n_tok = 6144, 2048, 3259
    strata.device_error(clear=True)
    w, xq, xd, y0, y1 = run_dequant(rows, cols, n_tok, "gemm-dq-prompt")
    assert strata.device_error(clear=True) == 0
    assert torch.equal(y1.view(torch.int32), y0.view(torch.int32))
    rng = np.random.default_rng(2)
    sel = np.unique(np.concatenate([rng.choice(rows, 48, replace=False), np.arange(0, rows, 128) + 5]))
    y_or, A = oracle.mmvq_rows(w.buf, rows, cols, synth.Q4, xq, xd, sel)
    err = np.abs(y1.cpu().numpy()[:, sel].astype(np.float64) - y_or)
    assert (err <= oracle.tolerance(A)).all()
