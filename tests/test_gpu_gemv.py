"""GPU parity of the verify path through the C ABI against the CPU oracle.

Bars: bit-exact activation codes/scales/sums and integer block dots; fp32 outputs within
|gpu - oracle| <= 2e-6 * sum|block terms| + 1e-6; every column of a T-token launch bitwise equal
to the T = 1 launch (the verify window's exact mode); argmax ids equal to the oracle's except
where the oracle's top-2 gap is inside the fp32 bound.
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


def gpu_quantize(x):
    xq, xd, xs = strata.quantize_act(cu(x))
    return xq, xd, xs


def assert_within(y_gpu, y_or, A, what=""):
    tol = oracle.tolerance(A)
    err = np.abs(y_gpu.astype(np.float64) - y_or)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} outside bound, worst excess {(err - tol).max():.3g}"


# ---- a1: quantizer -------------------------------------------------------------------------------
@pytest.mark.parametrize("n,cols,outl", [(4, 512, False), (1, 4096, True), (3256, 2048, False), (8, 14336, True),
                                         (1, 32, False), (5, 96, True)])
def test_quantizer_bit_exact(n, cols, outl):
    x = synth.make_activations(n, cols, "q", outliers=outl)
    q0, d0, s0 = oracle.quantize_act(x)
    q1, d1, s1 = [t.cpu().numpy() for t in gpu_quantize(x)]
    assert np.array_equal(q0, q1)
    assert np.array_equal(d0.view(np.uint32), d1.view(np.uint32))
    assert np.array_equal(s0, s1)


def test_quantizer_special_blocks():
    x = np.zeros((4, 64), np.float32)
    x[1, :8] = [127.0, 0.5, -0.5, 1.5, 2.5, -2.5, 126.5, -0.49999997]
    x[2, :] = 1.0
    x[2, 5] = 20.0
    x[3, :] = np.float32(1e-30)
    q0, d0, s0 = oracle.quantize_act(x)
    q1, d1, s1 = [t.cpu().numpy() for t in gpu_quantize(x)]
    assert np.array_equal(q0, q1) and np.array_equal(d0.view(np.uint32), d1.view(np.uint32))
    assert np.array_equal(s0, s1)


# ---- a2/a3: integer block dots -----------------------------------------------------------------------
@pytest.mark.parametrize("fmt,rows,cols,T", [(synth.Q4, 256, 512, 4), (synth.Q8, 256, 512, 4),
                                             (synth.Q8, 4096, 4096, 1), (synth.Q4, 37, 2080, 8)])
def test_block_dots_exact(fmt, rows, cols, T):
    w = synth.make_weights(rows, cols, fmt, "dots")
    x = synth.make_activations(T, cols, "dots", outliers=True)
    xq, xd, xs = oracle.quantize_act(x)
    ref = oracle.block_dots(w.buf, rows, cols, fmt, xq)
    got = strata.block_dots(cu(w.buf), rows, cols, fmt, cu(xq), cu(xs), T).cpu().numpy()
    assert np.array_equal(got.astype(np.int64), ref)


# ---- a4/a5: T-column GEMV ------------------------------------------------------------------------------
SHAPES = [
    (synth.Q4, 256, 512, 4, False),      # Tiny
    (synth.Q4, 4096, 4096, 1, True),     # Decode GEMV, Q4
    (synth.Q8, 4096, 4096, 1, True),     # Decode GEMV, Q8
    (synth.Q4, 33, 96, 3, False),        # ragged: rows not a multiple of any row group, 3 blocks
    (synth.Q8, 1, 32, 8, False),         # one row, one block
    (synth.Q4, 1000, 2080, 5, True),     # 65 blocks: lane 0 takes three blocks, others two
    (synth.Q4, 512, 2048, 4, False),     # one row group per CTA: one half-warp group of a warp has rows, the other none
    (synth.Q4, 5120, 2048, 4, False),    # window qkv
    (synth.Q4, 2048, 6144, 4, False),    # window down
]


@pytest.mark.parametrize("fmt,rows,cols,T,outl", SHAPES)
def test_mmvq_matches_oracle(fmt, rows, cols, T, outl):
    w = synth.make_weights(rows, cols, fmt, "mmvq")
    x = synth.make_activations(T, cols, "mmvq", outliers=outl)
    xq, xd, xs = oracle.quantize_act(x)
    y_or, A = oracle.mmvq(w.buf, rows, cols, fmt, xq, xd)
    y = strata.mmvq_multi(cu(w.buf), rows, cols, fmt, cu(xq), cu(xd), cu(xs), T).cpu().numpy()
    assert_within(y, y_or, A, f"{fmt} {rows}x{cols} T={T}")


@pytest.mark.parametrize("fmt,T,cols", [(synth.Q4, 8, 16384), (synth.Q8, 4, 16384)])
def test_mmvq_widest_staged_activations(fmt, T, cols):
    """The largest activation copy the launch stages (T*cols = 131072 for Q4 at T = 8), ragged rows,
    against the oracle on every row; the T = 1 columns are the same bits."""
    rows = 257
    assert strata.lib().strata_mmvq_multi(None, rows, cols, fmt, None, None, None, T, None, None) == -1
    w = synth.make_weights(rows, cols, fmt, "widest")
    W = cu(w.buf)
    x = synth.make_activations(T, cols, "widest", outliers=True)
    xq, xd, xs = gpu_quantize(x)
    y = strata.mmvq_multi(W, rows, cols, fmt, xq, xd, xs, T).cpu().numpy()
    y_or, A = oracle.mmvq(w.buf, rows, cols, fmt, xq.cpu().numpy(), xd.cpu().numpy())
    assert_within(y, y_or, A, f"widest fmt={fmt} T={T}")
    y1 = strata.mmvq_multi(W, rows, cols, fmt, xq[T - 1:], xd[T - 1:], xs[T - 1:], 1).cpu().numpy()
    assert np.array_equal(y[T - 1].view(np.uint32), y1[0].view(np.uint32))


def test_mmvq_rejects_activations_past_the_staged_maximum():
    L = strata.lib()
    A16 = 0x10000
    # Q4 at T = 8 stages at most 131072 activation values; Q8 at T = 8 and 16384 columns does not fit
    assert L.strata_mmvq_multi(A16, 256, 16416, synth.Q4, A16, A16, A16, 8, A16, None) == -2
    assert L.strata_mmvq_multi(A16, 256, 16384, synth.Q8, A16, A16, A16, 8, A16, None) == -2


@pytest.mark.parametrize("rows,cols", [(14336, 4096), (4096, 14336), (1000, 2080)])
def test_columns_bitwise_equal_single_token(rows, cols):
    """Verify window FFN: each column at T in {2,3,4,8} is the T = 1 launch, bit for bit."""
    w = synth.make_weights(rows, cols, synth.Q4, "ffn")
    W = cu(w.buf)
    x = synth.make_activations(8, cols, "ffn")
    xq, xd, xs = gpu_quantize(x)
    single = [strata.mmvq_multi(W, rows, cols, synth.Q4, xq[t:t + 1], xd[t:t + 1], xs[t:t + 1], 1).cpu().numpy()
              for t in range(8)]
    for T in (2, 3, 4, 5, 6, 7, 8):
        y = strata.mmvq_multi(W, rows, cols, synth.Q4, xq[:T], xd[:T], xs[:T], T).cpu().numpy()
        for t in range(T):
            assert np.array_equal(y[t].view(np.uint32), single[t][0].view(np.uint32)), (T, t)
    # and the 8 columns against the oracle (sampled rows)
    sel = np.unique(np.concatenate([np.arange(0, rows, max(1, rows // 512)), [rows - 1]]))
    y_or, A = oracle.mmvq_rows(w.buf, rows, cols, synth.Q4, xq.cpu().numpy(), xd.cpu().numpy(), sel)
    y8 = strata.mmvq_multi(W, rows, cols, synth.Q4, xq, xd, xs, 8).cpu().numpy()
    assert_within(y8[:, sel], y_or, A, "ffn T=8")


def test_q8_columns_bitwise_equal_single_token():
    rows, cols = 3000, 2048
    w = synth.make_weights(rows, cols, synth.Q8, "q8inv")
    W = cu(w.buf)
    xq, xd, xs = gpu_quantize(synth.make_activations(8, cols, "q8inv"))
    y8 = strata.mmvq_multi(W, rows, cols, synth.Q8, xq, xd, xs, 8).cpu().numpy()
    for t in range(8):
        y1 = strata.mmvq_multi(W, rows, cols, synth.Q8, xq[t:t + 1], xd[t:t + 1], xs[t:t + 1], 1).cpu().numpy()
        assert np.array_equal(y8[t].view(np.uint32), y1[0].view(np.uint32))


# ---- a6: head GEMV + argmax --------------------------------------------------------------------------
def accepted_ids(logits_or, A):
    """Ids whose oracle logit is within the fp32 bound of the maximum (both sides' bounds)."""
    out = []
    for t in range(logits_or.shape[0]):
        m = np.argmax(logits_or[t])
        band = oracle.tolerance(A[t]) + oracle.tolerance(A[t, m])
        out.append(set(np.nonzero(logits_or[t] >= logits_or[t, m] - band)[0].tolist()))
    return out


@pytest.fixture(scope="module")
def head_case():
    vocab, cols = synth.HEAD_VOCAB, synth.WINDOW_HIDDEN
    w = synth.make_weights(vocab, cols, synth.Q8, "head")
    x = synth.make_activations(8, cols, "head")
    xq, xd, xs = oracle.quantize_act(x)
    ids_or, logits_or, A = oracle.head_argmax(w.buf, vocab, cols, synth.Q8, xq, xd)
    return dict(w=w, W=cu(w.buf), xq=xq, xd=xd, xs=xs, ids=ids_or, logits=logits_or, A=A, vocab=vocab, cols=cols)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_head_argmax_matches_oracle(head_case, T):
    c = head_case
    logits = torch.empty((T, c["vocab"]), dtype=torch.float32, device="cuda")
    ids = strata.head_argmax(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"][:T]), cu(c["xd"][:T]),
                             cu(c["xs"][:T]), T, logits=logits).cpu().numpy()
    lg = logits.cpu().numpy()
    assert_within(lg, c["logits"][:T], c["A"][:T], "head logits")
    acc = accepted_ids(c["logits"][:T], c["A"][:T])
    for t in range(T):
        assert ids[t] in acc[t]
        if len(acc[t]) == 1:
            assert ids[t] == c["ids"][t]
        # the GPU's own argmax of its logits, ties to the lowest id
        assert ids[t] == int(np.argmax(lg[t]))
    # without logits: same ids
    ids2 = strata.head_argmax(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"][:T]), cu(c["xd"][:T]),
                              cu(c["xs"][:T]), T).cpu().numpy()
    assert np.array_equal(ids, ids2)


def test_head_columns_bitwise_equal_single_token(head_case):
    c = head_case
    T = 8
    lg8 = torch.empty((T, c["vocab"]), dtype=torch.float32, device="cuda")
    ids8 = strata.head_argmax(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"]), cu(c["xd"]), cu(c["xs"]), T,
                              logits=lg8).cpu().numpy()
    for t in range(T):
        lg1 = torch.empty((1, c["vocab"]), dtype=torch.float32, device="cuda")
        ids1 = strata.head_argmax(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"][t:t + 1]),
                                  cu(c["xd"][t:t + 1]), cu(c["xs"][t:t + 1]), 1, logits=lg1).cpu().numpy()
        assert ids1[0] == ids8[t]
        assert torch.equal(lg1[0].view(torch.int32), lg8[t].view(torch.int32))


@pytest.mark.parametrize("pair", [(17, 200), (5, 151930), (70000, 70001)])
def test_head_planted_tie_goes_to_lower_id(pair):
    """Two byte-identical rows, every other row at scale 0: equal maxima resolve to the lower id,
    whether the rows share a CTA or sit at opposite ends of the vocabulary."""
    vocab, cols = synth.HEAD_VOCAB, 256
    lo, hi = pair
    w = synth.make_weights(vocab, cols, synth.Q8, "tie")
    buf = w.buf.copy()
    nb = w.nb
    buf[hi * nb * 32:(hi + 1) * nb * 32] = buf[lo * nb * 32:(lo + 1) * nb * 32]
    sc = buf[w.plane_bytes:].view(np.float16).reshape(vocab, nb)
    keep = sc[lo].copy()
    sc[:] = 0
    sc[lo] = keep
    sc[hi] = keep
    x = synth.make_activations(2, cols, "tie")
    xq, xd, xs = oracle.quantize_act(x)
    y, _ = oracle.mmvq_rows(buf, vocab, cols, synth.Q8, xq, xd, [lo])
    neg = y[:, 0] < 0                            # make the tied logit positive (the rest are 0)
    xq[neg] = -xq[neg]
    xs[neg] = -xs[neg]
    ids = strata.head_argmax(cu(buf), vocab, cols, synth.Q8, cu(xq), cu(xd), cu(xs), 2).cpu().numpy()
    ids_or, logits_or, _ = oracle.head_argmax(buf, vocab, cols, synth.Q8, xq, xd)
    for t in range(2):
        assert logits_or[t, lo] == logits_or[t, hi] and logits_or[t, lo] > 0
        assert ids_or[t] == lo
        assert ids[t] == lo


def test_head_all_equal_logits_pick_id_zero():
    vocab, cols = 5000, 64
    w = synth.make_weights(vocab, cols, synth.Q8, "flat")
    buf = w.buf.copy()
    buf[w.plane_bytes:] = 0                        # every scale 0: every logit is exactly 0
    xq, xd, xs = oracle.quantize_act(synth.make_activations(3, cols, "flat"))
    ids = strata.head_argmax(cu(buf), vocab, cols, synth.Q8, cu(xq), cu(xd), cu(xs), 3).cpu().numpy()
    assert list(ids) == [0, 0, 0]


# ---- top-2 margin (batch-window confidence: top-1 minus top-2 logit per token) ------------------------
def gpu_top2_margin(lg):
    """fp32 top-1 minus top-2 of the GPU's own logits (a repeated maximum gives 0)."""
    s = np.sort(lg, axis=1)
    return (s[:, -1] - s[:, -2]).astype(np.float32)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_head_margin_matches_oracle(head_case, T):
    c = head_case
    logits = torch.empty((T, c["vocab"]), dtype=torch.float32, device="cuda")
    ids, mg = strata.head_argmax_margin(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"][:T]),
                                        cu(c["xd"][:T]), cu(c["xs"][:T]), T, logits=logits)
    ids, mg, lg = ids.cpu().numpy(), mg.cpu().numpy(), logits.cpu().numpy()
    # the same ids as the plain head, and the margin from the same fp32 logits, bit for bit
    ids_plain = strata.head_argmax(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"][:T]), cu(c["xd"][:T]),
                                   cu(c["xs"][:T]), T).cpu().numpy()
    assert np.array_equal(ids, ids_plain)
    assert np.array_equal(mg.view(np.uint32), gpu_top2_margin(lg).view(np.uint32))
    # against the oracle: order statistics move by at most the largest per-logit bound, so the
    # margin by at most twice that
    mg_or = oracle.margin(c["logits"][:T])
    bound = 2 * oracle.tolerance(c["A"][:T]).max(axis=1)
    assert (np.abs(mg.astype(np.float64) - mg_or) <= bound).all()


def test_head_margin_columns_bitwise_equal_single_token(head_case):
    c = head_case
    _, mg8 = strata.head_argmax_margin(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"]), cu(c["xd"]),
                                       cu(c["xs"]), 8)
    mg8 = mg8.cpu().numpy()
    for t in range(8):
        _, mg1 = strata.head_argmax_margin(c["W"], c["vocab"], c["cols"], synth.Q8, cu(c["xq"][t:t + 1]),
                                           cu(c["xd"][t:t + 1]), cu(c["xs"][t:t + 1]), 1)
        assert mg1.cpu().numpy().view(np.uint32)[0] == mg8.view(np.uint32)[t]


def test_head_margin_planted_tie_is_zero_and_one_row_is_inf():
    """Two byte-identical rows, every other row at scale 0 (logit exactly 0), the tied logit made
    positive: ids = the lower row, margin exactly 0. With the twin's scales zeroed too the margin is
    the tied row's logit itself; a one-row head has margin +inf."""
    vocab, cols = 4000, 256
    lo, hi = 100, 3900
    w = synth.make_weights(vocab, cols, synth.Q8, "mtie")
    buf = w.buf.copy()
    nb = w.nb
    buf[hi * nb * 32:(hi + 1) * nb * 32] = buf[lo * nb * 32:(lo + 1) * nb * 32]
    sc = buf[w.plane_bytes:].view(np.float16).reshape(vocab, nb)
    keep = sc[lo].copy()
    sc[:] = 0
    sc[lo] = keep
    sc[hi] = keep
    xq, xd, xs = oracle.quantize_act(synth.make_activations(3, cols, "mtie"))
    y, _ = oracle.mmvq_rows(buf, vocab, cols, synth.Q8, xq, xd, [lo])
    neg = y[:, 0] < 0
    xq[neg] = -xq[neg]
    xs[neg] = -xs[neg]
    lg = torch.empty((3, vocab), dtype=torch.float32, device="cuda")
    ids, mg = strata.head_argmax_margin(cu(buf), vocab, cols, synth.Q8, cu(xq), cu(xd), cu(xs), 3, logits=lg)
    assert list(ids.cpu().numpy()) == [lo] * 3 and (mg.cpu().numpy() == 0.0).all()
    sc[hi] = 0                                     # the twin drops to 0: margin = the logit
    ids, mg = strata.head_argmax_margin(cu(buf), vocab, cols, synth.Q8, cu(xq), cu(xd), cu(xs), 3, logits=lg)
    assert list(ids.cpu().numpy()) == [lo] * 3
    assert np.array_equal(mg.cpu().numpy(), lg.cpu().numpy()[:, lo])
    w1 = synth.make_weights(1, cols, synth.Q8, "one")
    ids1, mg1 = strata.head_argmax_margin(cu(w1.buf), 1, cols, synth.Q8, cu(xq), cu(xd), cu(xs), 3)
    assert list(ids1.cpu().numpy()) == [0, 0, 0] and np.isinf(mg1.cpu().numpy()).all()


def test_head_margin_rejects_null_margin():
    L = strata.lib()
    A16 = 0x10000
    assert L.strata_head_argmax_margin(A16, 1000, 256, synth.Q8, A16, A16, A16, 2, A16, None, None, A16,
                                       1 << 20, None) == -1


# ---- grouped launch (many independent matrices, one persistent launch) -----------------------------
@pytest.mark.parametrize("fmt,shapes,T", [
    (synth.Q4, [(256, 512), (33, 96), (1000, 2080), (5120, 2048), (2048, 6144), (7, 4096), (1, 32)], 3),
    (synth.Q8, [(4096, 4096), (300, 2048), (1, 32), (77, 160)], 8),
    (synth.Q4, [(14336, 4096), (4096, 14336)], 2),
])
def test_grouped_equals_separate_calls_and_oracle(fmt, shapes, T):
    probs, ref = [], []
    for k, (rows, cols) in enumerate(shapes):
        w = synth.make_weights(rows, cols, fmt, "grouped", k)
        xq, xd, xs = oracle.quantize_act(synth.make_activations(T, cols, "grouped", k, outliers=True))
        W = cu(w.buf)
        y = torch.full((T, rows), float("nan"), device="cuda")
        probs.append((W, rows, cols, cu(xq), cu(xd), cu(xs), y))
        ref.append((w, xq, xd))
    strata.mmvq_grouped(probs, fmt, T)
    torch.cuda.synchronize()
    for (W, rows, cols, xq, xd, xs, y), (w, xq_h, xd_h) in zip(probs, ref):
        y1 = strata.mmvq_multi(W, rows, cols, fmt, xq, xd, xs, T)
        assert torch.equal(y.view(torch.int32), y1.view(torch.int32)), (rows, cols)
        sel = np.unique(np.concatenate([np.arange(0, rows, max(1, rows // 64)), [rows - 1]]))
        y_or, A = oracle.mmvq_rows(w.buf, rows, cols, fmt, xq_h, xd_h, sel)
        assert_within(y.cpu().numpy()[:, sel], y_or, A, f"grouped {rows}x{cols}")
    assert strata.device_error() == 0


def test_grouped_rejects_bad_descriptor():
    w = torch.zeros(synth.weight_nbytes(64, 64, synth.Q4), dtype=torch.uint8, device="cuda")
    xq = torch.zeros((1, 64), dtype=torch.int8, device="cuda")
    xd = torch.zeros((1, 2), dtype=torch.float32, device="cuda")
    xs = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    y = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    good = (w, 64, 64, xq, xd, xs, y)
    bad = (w, 64, 48, xq, xd, xs, y)
    with pytest.raises(strata.StrataError) as e:
        strata.mmvq_grouped([good, bad], synth.Q4, 1)
    assert e.value.status == -2
