"""GPU parity of the 256-weight super-block formats through the same GEMV family: Q6 (6-bit codes,
int8 sub-scale per 16 weights, fp16 d per 256), Q4K (4-bit codes, 6-bit scale and minimum per 32
weights, fp16 d and dmin per 256) and Q5K (Q4K with 5-bit codes, the fifth bits in a per-block word
after the row's nibble blocks). Bars: exact integer dots (bit for bit), outputs within the fp32
bound of the oracle, every column of a T-token launch bitwise equal to the T = 1 launch, grouped
launches equal to single calls.
"""
import numpy as np
import pytest
import torch

import oracle
from block_quantized_token_strata_gb300 import strata, synth

pytestmark = pytest.mark.gpu
FMTS = [synth.Q6, synth.Q4K, synth.Q5K]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from block_quantized_token_strata_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    oracle.build()


def cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y_gpu, y_or, A, what=""):
    tol = oracle.tolerance(A)
    err = np.abs(y_gpu.astype(np.float64) - y_or)
    assert not (err > tol).any(), f"{what}: {(err > tol).sum()} outside the bound"


@pytest.mark.parametrize("Q6", FMTS)
def test_q6_block_dots_exact(Q6):
    rows, cols, T = 37, 768, 3
    w = synth.make_weights(rows, cols, Q6, "q6dots")
    x = synth.make_activations(T, cols, "q6dots", outliers=True)
    xq, xd, xs = oracle.quantize_act(x)
    got = strata.block_dots(cu(w.buf), rows, cols, Q6, cu(xq), cu(xs), T).cpu().numpy()
    ref = oracle.block_dots(w.buf, rows, cols, Q6, xq)
    assert np.array_equal(got.astype(np.int64).reshape(ref.shape), ref)


@pytest.mark.parametrize("rows,cols,T,outl", [
    (256, 512, 4, False),       # two super-blocks a row
    (33, 768, 3, True),         # ragged rows
    (1000, 2304, 5, True),      # nine super-blocks: lanes take uneven block counts
    (4096, 4096, 1, True),      # decode
    (10240, 2560, 2, False),    # the pages' Q6 MMVQ shape at T = 2
    (1, 256, 8, False),         # one row, one super-block
])
@pytest.mark.parametrize("Q6", FMTS)
def test_q6_mmvq_matches_oracle(Q6, rows, cols, T, outl):
    w = synth.make_weights(rows, cols, Q6, "q6mmvq")
    x = synth.make_activations(T, cols, "q6mmvq", outliers=outl)
    xq, xd, xs = oracle.quantize_act(x)
    y = strata.mmvq_multi(cu(w.buf), rows, cols, Q6, cu(xq), cu(xd), cu(xs), T).cpu().numpy()
    if rows * cols * T <= 50_000_000:
        y_or, A = oracle.mmvq(w.buf, rows, cols, Q6, xq, xd)
        assert_within(y, y_or, A, f"q6 {rows}x{cols} T={T}")
    else:
        sel = np.unique(np.concatenate([np.arange(0, rows, 37), [rows - 1]]))
        y_or, A = oracle.mmvq_rows(w.buf, rows, cols, Q6, xq, xd, sel)
        assert_within(y[:, sel], y_or, A, f"q6 {rows}x{cols} T={T} (sampled)")


@pytest.mark.parametrize("rows,cols", [(10240, 2560), (3000, 4096)])
@pytest.mark.parametrize("Q6", FMTS)
def test_q6_columns_bitwise_equal_single_token(Q6, rows, cols):
    w = synth.make_weights(rows, cols, Q6, "q6inv")
    W = cu(w.buf)
    xq, xd, xs = strata.quantize_act(cu(synth.make_activations(8, cols, "q6inv")))
    single = [strata.mmvq_multi(W, rows, cols, Q6, xq[t:t + 1], xd[t:t + 1], xs[t:t + 1], 1).cpu().numpy()
              for t in range(8)]
    for T in (2, 3, 4, 5, 8):
        y = strata.mmvq_multi(W, rows, cols, Q6, xq[:T], xd[:T], xs[:T], T).cpu().numpy()
        for t in range(T):
            assert np.array_equal(y[t].view(np.uint32), single[t][0].view(np.uint32)), (T, t)


@pytest.mark.parametrize("Q6", FMTS)
def test_q6_grouped_equals_separate_calls(Q6):
    shapes, T = [(256, 512), (33, 768), (2048, 2048), (1, 256), (777, 1024)], 4
    probs, sep = [], []
    for k, (rows, cols) in enumerate(shapes):
        w = synth.make_weights(rows, cols, Q6, "q6grp", k)
        xq, xd, xs = oracle.quantize_act(synth.make_activations(T, cols, "q6grp", k, outliers=True))
        W = cu(w.buf)
        y = torch.full((T, rows), float("nan"), device="cuda")
        probs.append((W, rows, cols, cu(xq), cu(xd), cu(xs), y))
        sep.append(strata.mmvq_multi(W, rows, cols, Q6, cu(xq), cu(xd), cu(xs), T).cpu().numpy())
        y_or, A = oracle.mmvq(w.buf, rows, cols, Q6, xq, xd)
        assert_within(sep[-1], y_or, A, f"q6 grouped member {k}")
    strata.mmvq_grouped(strata.gemv_descs(probs), Q6, T)
    for (W, rows, cols, xq, xd, xs, y), s in zip(probs, sep):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_superblock_formats_reject_partial_superblocks():
    L = strata.lib()
    A16 = 0x10000
    for fmt, per256 in ((synth.Q6, 210), (synth.Q4K, 148), (synth.Q5K, 180)):
        assert L.strata_mmvq_multi(A16, 64, 288, fmt, A16, A16, A16, 1, A16, None) == -2   # 288 % 256 != 0
        assert L.strata_weight_bytes(10, 512, fmt) == 10 * 2 * per256


def test_q4k_head_argmax_matches_oracle():
    """The vocabulary head in Q4K: ids exact (outside near ties), logits within the bound."""
    vocab, cols, T = 20000, 2048, 4
    w = synth.make_weights(vocab, cols, synth.Q4K, "q4khead")
    xq, xd, xs = oracle.quantize_act(synth.make_activations(T, cols, "q4khead"))
    lg = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
    ids = strata.head_argmax(cu(w.buf), vocab, cols, synth.Q4K, cu(xq), cu(xd), cu(xs), T, logits=lg).cpu().numpy()
    ids_or, lg_or, A = oracle.head_argmax(w.buf, vocab, cols, synth.Q4K, xq, xd)
    assert_within(lg.cpu().numpy(), lg_or, A, "q4k head")
    for t in range(T):
        assert ids[t] == int(np.argmax(lg.cpu().numpy()[t]))
        top = np.sort(lg_or[t])[-2:]
        if top[1] - top[0] > 2 * oracle.tolerance(A[t]).max():
            assert ids[t] == ids_or[t]


def test_q5k_head_argmax_and_fifth_bits_matter():
    """A Q5K head: ids and logits against the oracle; and the same codes with every fifth bit cleared
    give different logits, so the kernel reads the fifth-bit words."""
    vocab, cols, T = 6000, 2048, 3
    w = synth.make_weights(vocab, cols, synth.Q5K, "q5khead")
    xq, xd, xs = oracle.quantize_act(synth.make_activations(T, cols, "q5khead"))
    lg = torch.empty((T, vocab), dtype=torch.float32, device="cuda")
    ids = strata.head_argmax(cu(w.buf), vocab, cols, synth.Q5K, cu(xq), cu(xd), cu(xs), T, logits=lg).cpu().numpy()
    ids_or, lg_or, A = oracle.head_argmax(w.buf, vocab, cols, synth.Q5K, xq, xd)
    assert_within(lg.cpu().numpy(), lg_or, A, "q5k head")
    for t in range(T):
        assert ids[t] == int(np.argmax(lg.cpu().numpy()[t]))
    cleared = w.buf.copy()
    nb = cols // 32
    for r in range(vocab):  # zero the row's fifth-bit words
        cleared[r * nb * 20 + nb * 16: (r + 1) * nb * 20] = 0
    y0 = strata.mmvq_multi(cu(cleared), vocab, cols, synth.Q5K, cu(xq), cu(xd), cu(xs), T).cpu().numpy()
    y0_or, A0 = oracle.mmvq(cleared, vocab, cols, synth.Q5K, xq, xd)
    assert_within(y0, y0_or, A0, "q5k without fifth bits")
    assert (np.abs(y0 - lg.cpu().numpy()) > oracle.tolerance(A)).mean() > 0.5
