"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Every oracle function is checked against something other than itself:
  * the fp16 decoder against numpy's binary16 conversion over all 65,536 patterns;
  * the activation quantizer against hand-derived closed-form blocks (ties round away from zero,
    a single outlier, all zeros) and the invariants its definition implies;
  * the integer block dots against hand-computed one-block values and a brute-force numpy int64
    matmul of codes this test packs itself;
  * the fp64 GEMV against a brute-force dense fp64 matmul of the dequantized operands;
  * the argmax tie rule against planted ties and numpy's first-occurrence argmax;
  * the top-2 margin against hand-worked rows and the pages' two-shard merge rule;
  * the MoE grouping against numpy's stable sort, and the MoE rows against a dense brute force.
Sources: Strata commit "wire multi-token kernels into Verifier and MtpDrafter CUDA graphs"
(verify.hpp header comment: exact mode, q8_1 activations, pool layout (n_tok*k, n_embd));
pull request "sm_80 (GA100) tuning" (exact integer block dots); dsv41-offload worker/tp2.py
(argmax ties to the lowest id).
"""
import json
import os

import numpy as np
import pytest

from block_quantized_token_strata_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ---- this test's own packer of the documented planar layout ------------------------------------
def pack_q4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes uint [rows][cols] in 0..15, scales float16 [rows][cols/32] -> planar bytes."""
    rows, cols = codes.shape
    nb = cols // 32
    c = codes.reshape(rows, nb, 32).astype(np.uint8)
    plane = (c[:, :, :16] | (c[:, :, 16:] << 4)).reshape(-1)
    return np.concatenate([plane, np.asarray(scales, np.float16).reshape(-1).view(np.uint8)])


def pack_q8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    plane = np.asarray(codes, np.int8).reshape(-1).view(np.uint8)
    return np.concatenate([plane, np.asarray(scales, np.float16).reshape(-1).view(np.uint8)])


# ---- fp16 decoder -------------------------------------------------------------------------------
def test_half_decoder_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---- activation quantizer -------------------------------------------------------------------------
def test_quantize_zero_block(orc):
    q, d, s = orc.quantize_act(np.zeros((2, 64), np.float32))
    assert not q.any() and not d.any() and not s.any()


def test_quantize_half_way_ties_round_away_from_zero(orc):
    # amax = 127 gives d = 127/127 = 1 and 1/d = 1 exactly, so q = roundf(x) on exact halves.
    x = np.zeros(32, np.float32)
    x[:8] = [127.0, 0.5, -0.5, 1.5, 2.5, -2.5, 126.5, -0.49999997]
    q, d, s = orc.quantize_act(x[None])
    assert d[0, 0] == np.float32(1.0)
    assert list(q[0, :8]) == [127, 1, -1, 2, 3, -3, 127, 0]
    assert s[0, 0] == 127 + 1 - 1 + 2 + 3 - 3 + 127 + 0
    # amax = 254 gives d = 2 and 1/d = 0.5 (both exact): 3 -> 1.5 -> 2, 5 -> 2.5 -> 3, -1 -> -1
    x = np.zeros(32, np.float32)
    x[:4] = [-254.0, 3.0, 5.0, -1.0]
    q, d, s = orc.quantize_act(x[None])
    assert d[0, 0] == np.float32(2.0)
    assert list(q[0, :4]) == [-127, 2, 3, -1]
    assert s[0, 0] == -127 + 2 + 3 - 1


def test_quantize_single_outlier_block(orc):
    # one x20 outlier among ones: d = fp32(20/127), q_0 = 127, the ones map to round(127/20)=6
    x = np.ones(32, np.float32)
    x[5] = 20.0
    q, d, s = orc.quantize_act(x[None])
    assert d[0, 0] == np.float32(20.0) / np.float32(127.0)
    assert q[0, 5] == 127 and (np.delete(q[0], 5) == 6).all()
    assert s[0, 0] == 127 + 31 * 6


def test_quantize_invariants_random(orc):
    x = synth.make_activations(16, 1024, "pins", outliers=True)
    q, d, s = orc.quantize_act(x)
    xb = x.reshape(16, 32, 32).astype(np.float64)
    qb = q.reshape(16, 32, 32).astype(np.int64)
    assert np.abs(qb).max() <= 127
    assert (np.abs(qb).max(axis=2) == 127).all()              # the block maximum maps to +-127
    assert np.array_equal(s, qb.sum(axis=2))                    # exact block sums
    amax = np.abs(xb).max(axis=2)
    assert np.allclose(d, amax / 127.0, rtol=2 ** -23, atol=0)  # d is amax/127 to one rounding
    err = np.abs(xb - d[:, :, None].astype(np.float64) * qb)   # reconstruction within half a step
    assert (err <= d[:, :, None] * (0.5 + 1e-5)).all()
    assert (np.sign(qb) * np.sign(xb) >= 0).all()


# ---- integer block dots ----------------------------------------------------------------------------
@pytest.fixture(scope="module")
def golden_blocks():
    with open(os.path.join(HERE, "golden", "one_block_dots.json")) as f:
        return json.load(f)["cases"]


def test_block_dots_hand_cases(orc, golden_blocks):
    for case in golden_blocks:
        fmt = synth.Q4 if case["fmt"] == "Q4" else synth.Q8
        codes = np.array(case["w_codes"], np.int64).reshape(1, 32)
        xq = np.array(case["x_codes"], np.int8).reshape(1, 32)
        scale = np.array([[case["w_scale"]]], np.float16)
        W = pack_q4(codes, scale) if fmt == synth.Q4 else pack_q8(codes, scale)
        isum = orc.block_dots(W, 1, 32, fmt, xq)
        assert isum[0, 0, 0] == case["isum"], case["name"]
        xd = np.array([[case["x_scale"]]], np.float32)
        y, A = orc.mmvq(W, 1, 32, fmt, xq, xd)
        assert y[0, 0] == case["y"], case["name"]
        assert A[0, 0] == abs(case["y"])


@pytest.mark.parametrize("fmt", [synth.Q4, synth.Q8])
def test_block_dots_brute_force(orc, fmt):
    rng = np.random.default_rng(7)
    rows, cols, T = 40, 256, 3
    if fmt == synth.Q4:
        codes = rng.integers(0, 16, (rows, cols))
        W = pack_q4(codes, rng.random((rows, cols // 32)).astype(np.float16))
        wv = codes - 8
    else:
        codes = rng.integers(-127, 128, (rows, cols))
        W = pack_q8(codes, rng.random((rows, cols // 32)).astype(np.float16))
        wv = codes
    xq = rng.integers(-127, 128, (T, cols)).astype(np.int8)
    got = orc.block_dots(W, rows, cols, fmt, xq)
    ref = np.einsum("rbj,tbj->trb", wv.reshape(rows, cols // 32, 32).astype(np.int64),
                    xq.reshape(T, cols // 32, 32).astype(np.int64))
    assert np.array_equal(got, ref)


# ---- fp64 GEMV -------------------------------------------------------------------------------------
def dense_dequant(w: synth.Weights) -> np.ndarray:
    codes = w.codes().astype(np.float64)
    if w.fmt == synth.Q4:
        codes -= 8.0
    sc = np.repeat(w.scales.astype(np.float64), 32, axis=1)
    return codes * sc


@pytest.mark.parametrize("fmt,rows,cols,T", [(synth.Q4, 256, 512, 4), (synth.Q8, 96, 1024, 3),
                                             (synth.Q4, 33, 96, 1)])
def test_mmvq_brute_force_dense(orc, fmt, rows, cols, T):
    w = synth.make_weights(rows, cols, fmt, "pin")
    x = synth.make_activations(T, cols, "pin")
    xq, xd, _ = orc.quantize_act(x)
    y, A = orc.mmvq(w.buf, rows, cols, fmt, xq, xd)
    xdeq = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
    ref = xdeq @ dense_dequant(w).T                                  # [T][rows]
    assert np.all(np.abs(y - ref) <= 1e-12 * A + 1e-300)
    assert np.all(A >= np.abs(y))
    ys, As = orc.mmvq_rows(w.buf, rows, cols, fmt, xq, xd, [rows - 1, 0, 5])
    assert np.array_equal(ys, y[:, [rows - 1, 0, 5]]) and np.array_equal(As, A[:, [rows - 1, 0, 5]])


def test_mmvq_linear_in_scales(orc):
    # doubling every weight scale (exact in fp16) doubles every output exactly
    w = synth.make_weights(64, 256, synth.Q4, "lin")
    x = synth.make_activations(2, 256, "lin")
    xq, xd, _ = orc.quantize_act(x)
    y1, _ = orc.mmvq(w.buf, 64, 256, synth.Q4, xq, xd)
    w2 = w.buf.copy()
    sc = w2[w.plane_bytes:].view(np.float16)
    sc *= np.float16(2.0)
    y2, _ = orc.mmvq(w2, 64, 256, synth.Q4, xq, xd)
    assert np.array_equal(y2, 2.0 * y1)


# ---- argmax -----------------------------------------------------------------------------------------
def test_argmax_ties_to_lowest(orc):
    v = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [-1.0, -2.0, -1.0, -1.5]])
    assert list(orc.argmax(v)) == [1, 0, 0]
    rng = np.random.default_rng(3)
    r = rng.integers(0, 5, (6, 1000)).astype(np.float64)   # many ties
    assert np.array_equal(orc.argmax(r), np.argmax(r, axis=1))


def test_head_argmax_planted_tie(orc):
    # rows 17 and 200 are byte-identical and every other row has scale 0 (logit exactly 0):
    # the two equal maxima must resolve to the lower id, 17.
    w = synth.make_weights(300, 256, synth.Q8, "tie")
    nb = w.nb
    buf = w.buf.copy()
    buf[200 * nb * 32:201 * nb * 32] = buf[17 * nb * 32:18 * nb * 32]
    sc = buf[w.plane_bytes:].view(np.float16).reshape(300, nb)
    keep = sc[17].copy()
    sc[:] = 0
    sc[17] = keep
    sc[200] = keep
    x = synth.make_activations(1, 256, "tie")
    xq, xd, _ = orc.quantize_act(x)
    y, _ = orc.mmvq(buf, 300, 256, synth.Q8, xq, xd)
    if y[0, 17] < 0:
        xq = (-xq.astype(np.int16)).astype(np.int8)
    ids, logits, _ = orc.head_argmax(buf, 300, 256, synth.Q8, xq, xd)
    assert logits[0, 17] == logits[0, 200] > 0
    assert ids[0] == 17


# ---- MoE ---------------------------------------------------------------------------------------------
def test_moe_bucket_matches_stable_sort(orc):
    ids = synth.make_routing(300, 16, 4, "bucket")
    counts, offsets, pairs, bad = orc.moe_bucket(ids, 16)
    assert bad == 0
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(pairs, order.astype(np.int32))
    assert np.array_equal(counts, np.bincount(flat, minlength=16))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)


def test_moe_bucket_skips_bad_ids(orc):
    ids = np.array([[0, 3], [-1, 1], [7, 0]], np.int32)
    counts, offsets, pairs, bad = orc.moe_bucket(ids, 4)
    assert bad == 2
    assert list(counts) == [2, 1, 0, 1]
    assert list(pairs[:4]) == [0, 5, 3, 1]


def test_moe_rows_brute_force(orc):
    n_exp, hidden, inter, n_tok, k = 4, 128, 64, 6, 2
    experts = [(synth.make_weights(inter, hidden, synth.Q4, "g", e),
                synth.make_weights(inter, hidden, synth.Q4, "u", e),
                synth.make_weights(hidden, inter, synth.Q4, "d", e)) for e in range(n_exp)]
    ids = synth.make_routing(n_tok, n_exp, k, "moe-bf")
    x = synth.make_activations(n_tok, hidden, "moe-bf")
    sel = np.arange(n_tok * k)
    out = orc.moe_rows([(g.buf, u.buf, d.buf) for g, u, d in experts], hidden, inter, ids, x, sel,
                       want_hidden=True, want_gate_up=True)
    xq, xd, _ = orc.quantize_act(x)
    xdeq = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
    for p in sel:
        tok, e = p // k, ids.reshape(-1)[p]
        g = dense_dequant(experts[e][0]) @ xdeq[tok]
        u = dense_dequant(experts[e][1]) @ xdeq[tok]
        h = g * u / (1.0 + np.exp(-g))
        assert np.allclose(out["h"][p], h, rtol=1e-12, atol=1e-300)
        # the gate and up outputs and their masses: the dense values, and A = sum |d_w d_x isum| per
        # block written out here from the unpacked codes and scales
        for name, mass, ref, wm in (("g", "Ag", g, experts[e][0]), ("u", "Au", u, experts[e][1])):
            assert np.all(np.abs(out[name][p] - ref) <= 1e-12 * out[mass][p] + 1e-300)
            qq = wm.codes().astype(np.int64).reshape(inter, hidden // 32, 32) - 8
            isum = np.einsum("rbj,bj->rb", qq, xq[tok].astype(np.int64).reshape(hidden // 32, 32))
            terms = wm.scales.astype(np.float64) * xd[tok].astype(np.float64)[None, :] * isum
            assert np.allclose(out[mass][p], np.abs(terms).sum(axis=1), rtol=1e-12, atol=0)
        hdeq = out["hq"][p].astype(np.float64) * np.repeat(out["hd"][p].astype(np.float64), 32)
        yref = dense_dequant(experts[e][2]) @ hdeq
        assert np.all(np.abs(out["y"][p] - yref) <= 1e-12 * out["A"][p] + 1e-300)
    # the hidden re-quantization is the pinned quantizer applied to fp32(h)
    q2, d2, s2 = orc.quantize_act(out["h"].astype(np.float32))
    assert np.array_equal(q2, out["hq"]) and np.array_equal(d2, out["hd"]) and np.array_equal(s2, out["hs"])
    # feeding the quantized hidden rows back reproduces y exactly
    out2 = orc.moe_rows([(g.buf, u.buf, d.buf) for g, u, d in experts], hidden, inter, ids, x, sel,
                        hq_in=out["hq"], hd_in=out["hd"])
    assert np.array_equal(out2["y"], out["y"])


def test_moe_rows_one_pair_equals_gemv(orc):
    # one token routed to one expert: the row is the down GEMV of the re-quantized hidden row
    hidden, inter = 64, 32
    g, u, d = (synth.make_weights(inter, hidden, synth.Q4, "one", 0),
               synth.make_weights(inter, hidden, synth.Q4, "one", 1),
               synth.make_weights(hidden, inter, synth.Q4, "one", 2))
    x = synth.make_activations(1, hidden, "one")
    out = orc.moe_rows([(g.buf, u.buf, d.buf)], hidden, inter, np.zeros((1, 1), np.int32), x, [0],
                       want_hidden=True)
    y, A = orc.mmvq(d.buf, hidden, inter, synth.Q4, out["hq"], out["hd"])
    assert np.array_equal(out["y"][0], y[0]) and np.array_equal(out["A"][0], A[0])


def test_margin_hand_cases(orc):
    """Top-1 minus top-2 (dsv41-offload worker/tp2.py, EmuComm.margin): worked by hand."""
    oracle = orc
    v = np.array([[1.0, 3.0, 2.0, -4.0],      # 3 - 2
                  [5.0, 5.0, 1.0, 0.0],       # the maximum twice: 0
                  [-1.0, -7.0, -2.5, -1.5],   # -1 - (-1.5)
                  [0.0, 0.0, 0.0, 0.0]])      # all equal: 0
    assert list(oracle.margin(v)) == [1.0, 0.0, 0.5, 0.0]
    assert oracle.margin(np.array([[2.5]]))[0] == np.inf    # one value: nothing to beat


def test_margin_matches_two_shard_merge(orc):
    """The pages' two-shard merge: split each row at a random point, take each shard's top-2, merge
    as EmuComm.margin does (take_a = a1 >= b1; second = max(a2, b1) or max(b2, a1)); equals the
    whole-row margin. Ties are planted so that both branches and equal maxima occur."""
    oracle = orc
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(4, 40))
        row = rng.integers(-5, 6, size=n).astype(np.float64)   # small integers: many ties
        cut = int(rng.integers(2, n - 1))
        A, B = np.sort(row[:cut])[::-1], np.sort(row[cut:])[::-1]
        a1, a2, b1, b2 = A[0], A[1], B[0], B[1]
        second = max(a2, b1) if a1 >= b1 else max(b2, a1)
        assert oracle.margin(row)[0] == max(a1, b1) - second


# ---- Q6 (6-bit codes, int8 sub-scale per 16 weights, fp16 d per 256 weights) --------------------------
def pack_q6(q: np.ndarray, sub: np.ndarray, d: np.ndarray) -> np.ndarray:
    """This test's own packer of the documented Q6 planar layout (code plane 24 B a block: bytes 0..15
    the low 4 bits of elements j and j+16, bytes 16..23 the high 2 bits of elements i, i+8, i+16,
    i+24; then int8 sub-scales, 2 a block; then fp16 d, one per 256 weights)."""
    rows, cols = q.shape
    nb = cols // 32
    out = bytearray()
    for r in range(rows):
        for b in range(nb):
            blk = [int(v) for v in q[r, 32 * b:32 * b + 32]]
            low = [blk[j] & 15 for j in range(32)]
            high = [blk[j] >> 4 for j in range(32)]
            out += bytes(low[j] | (low[j + 16] << 4) for j in range(16))
            out += bytes(high[i] | (high[i + 8] << 2) | (high[i + 16] << 4) | (high[i + 24] << 6) for i in range(8))
    out += np.asarray(sub, np.int8).tobytes()
    out += np.asarray(d, np.float16).tobytes()
    return np.frombuffer(bytes(out), np.uint8).copy()


def test_q6_one_superblock_by_hand(orc):
    """cols = 256 (one super-block, 8 blocks, 16 sub-scales); d = 1, x codes all 1 with d_x = 1:
    codes all 32 give 0; codes all 63 with sub-scales 1 give 16 halves x 16 x 31 = 7936; sub-scales
    alternating +1/-1 cancel to 0; sub-scale 3 on the first half only gives 3 x 16 x 31 = 1488."""
    xq = np.ones((1, 256), np.int8)
    xd = np.ones((1, 8), np.float32)
    d = np.ones((1, 1), np.float16)
    cases = [(32, np.ones(16), 0.0), (63, np.ones(16), 7936.0),
             (63, np.array([1, -1] * 8), 0.0), (63, np.array([3] + [0] * 15), 1488.0)]
    for code, sub, want in cases:
        W = pack_q6(np.full((1, 256), code, np.uint8), sub.reshape(1, 16).astype(np.int8), d)
        y, A = orc.mmvq(W, 1, 256, 2, xq, xd)
        assert y[0, 0] == want, (code, sub, y)


def test_q6_brute_force_dense(orc):
    """Dense fp64 dequantization w = d * s * (q - 32) against the oracle's block form."""
    rng = np.random.default_rng(17)
    rows, cols, T = 9, 768, 3
    q = rng.integers(0, 64, size=(rows, cols)).astype(np.uint8)
    sub = rng.integers(-127, 128, size=(rows, cols // 16)).astype(np.int8)
    d = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
    W = pack_q6(q, sub, d)
    assert W.size == rows * (cols // 256) * 210
    x = rng.standard_normal((T, cols)).astype(np.float32)
    xq, xd, _ = orc.quantize_act(x)
    w = (d.astype(np.float64).repeat(256, axis=1) * sub.astype(np.float64).repeat(16, axis=1)
         * (q.astype(np.float64) - 32))
    xdq = xq.astype(np.float64) * xd.astype(np.float64).repeat(32, axis=1)
    ref = xdq @ w.T
    y, A = orc.mmvq(W, rows, cols, 2, xq, xd)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # the block dots: s0 * (first 16) + s1 * (last 16), brute force in int64
    isum = orc.block_dots(W, rows, cols, 2, xq)
    qq = q.astype(np.int64).reshape(rows, cols // 32, 2, 16) - 32
    ss = sub.astype(np.int64).reshape(rows, cols // 32, 2)
    xx = xq.astype(np.int64).reshape(T, cols // 32, 2, 16)
    want = np.einsum("rbhj,tbhj,rbh->trb", qq, xx, ss)
    assert np.array_equal(isum.reshape(T, rows, cols // 32), want)
    # the generator's buffer decodes the same way
    from block_quantized_token_strata_gb300 import synth
    assert np.array_equal(synth.make_q6_buffer(q, sub, d), W)


# ---- Q4K (4-bit codes, 6-bit scale and minimum per 32 weights, fp16 d and dmin per 256) --------------
def pack_q4k(q, sc, mn, d, dmin) -> np.ndarray:
    """This test's own packer: Q4 code bytes (no offset), then (sc, m) byte pairs per block, then
    (d, dmin) fp16 pairs per super-block."""
    rows, cols = q.shape
    out = bytearray()
    for r in range(rows):
        for b in range(cols // 32):
            blk = [int(v) for v in q[r, 32 * b:32 * b + 32]]
            out += bytes(blk[j] | (blk[j + 16] << 4) for j in range(16))
    for r in range(rows):
        for b in range(cols // 32):
            out += bytes([int(sc[r, b]), int(mn[r, b])])
    for r in range(rows):
        for k in range(cols // 256):
            out += np.array([d[r, k], dmin[r, k]], np.float16).tobytes()
    return np.frombuffer(bytes(out), np.uint8).copy()


def test_q4k_one_superblock_by_hand(orc):
    """cols = 256, x codes all 1 with d_x = 1 (block sums 32), d = dmin = 1: codes 15 with sc 1 and
    m 0 give 8 blocks x 32 x 15 = 3840; adding m = 2 subtracts 8 x 2 x 32 = 512; sc 0 and m 1 give
    -8 x 32 = -256."""
    xq = np.ones((1, 256), np.int8)
    xd = np.ones((1, 8), np.float32)
    one = np.ones((1, 1), np.float16)
    for code, sc, mn, want in [(15, 1, 0, 3840.0), (15, 1, 2, 3328.0), (7, 0, 1, -256.0), (0, 63, 0, 0.0)]:
        W = pack_q4k(np.full((1, 256), code, np.uint8), np.full((1, 8), sc), np.full((1, 8), mn), one, one)
        y, A = orc.mmvq(W, 1, 256, 3, xq, xd)
        assert y[0, 0] == want, (code, sc, mn, y)


def test_q4k_brute_force_dense(orc):
    rng = np.random.default_rng(23)
    rows, cols, T = 7, 512, 3
    q = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    sc = rng.integers(0, 64, size=(rows, cols // 32)).astype(np.uint8)
    mn = rng.integers(0, 64, size=(rows, cols // 32)).astype(np.uint8)
    d = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
    dmin = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
    W = pack_q4k(q, sc, mn, d, dmin)
    assert W.size == rows * (cols // 256) * 148
    xq, xd, _ = orc.quantize_act(rng.standard_normal((T, cols)).astype(np.float32))
    w = (d.astype(np.float64).repeat(256, axis=1) * sc.astype(np.float64).repeat(32, axis=1) * q
         - dmin.astype(np.float64).repeat(256, axis=1) * mn.astype(np.float64).repeat(32, axis=1))
    ref = (xq.astype(np.float64) * xd.astype(np.float64).repeat(32, axis=1)) @ w.T
    y, A = orc.mmvq(W, rows, cols, 3, xq, xd)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # block dots are the unscaled sums of q * x
    isum = orc.block_dots(W, rows, cols, 3, xq)
    want = np.einsum("rbj,tbj->trb", q.astype(np.int64).reshape(rows, -1, 32), xq.astype(np.int64).reshape(T, -1, 32))
    assert np.array_equal(isum.reshape(T, rows, cols // 32), want)
    from block_quantized_token_strata_gb300 import synth
    assert np.array_equal(synth.make_q4k_buffer(q, sc, mn, d, dmin), W)


# ---- Q5K (5-bit codes, 6-bit scale and minimum per 32 weights, fp16 d and dmin per 256) --------------
def pack_q5k(q, sc, mn, d, dmin) -> np.ndarray:
    """This test's own packer: per row, the Q4-style nibble bytes of every block, then per block a
    little-endian 32-bit word whose bit 8k + g is the fifth bit of element 4g + k (g < 4) or
    16 + 4(g - 4) + k (g >= 4); then (sc, m) byte pairs per block and (d, dmin) fp16 pairs per 256."""
    rows, cols = q.shape
    out = bytearray()
    for r in range(rows):
        nib, words = bytearray(), bytearray()
        for b in range(cols // 32):
            blk = [int(v) for v in q[r, 32 * b:32 * b + 32]]
            nib += bytes((blk[j] & 15) | ((blk[j + 16] & 15) << 4) for j in range(16))
            word = 0
            for j in range(32):
                g = j // 4 if j < 16 else 4 + (j - 16) // 4
                word |= ((blk[j] >> 4) & 1) << (8 * (j % 4) + g)
            words += word.to_bytes(4, "little")
        out += nib + words
    for r in range(rows):
        for b in range(cols // 32):
            out += bytes([int(sc[r, b]), int(mn[r, b])])
    for r in range(rows):
        for k in range(cols // 256):
            out += np.array([d[r, k], dmin[r, k]], np.float16).tobytes()
    return np.frombuffer(bytes(out), np.uint8).copy()


def test_q5k_one_superblock_by_hand(orc):
    """cols = 256, x codes all 1 with d_x = 1, d = dmin = 1. Code 31 with sc 1 and m 0 gives
    8 blocks x 32 x 31 = 7936; code 16 (only the fifth bit set) with sc 2, m 3 gives
    8 x 32 x (2*16 - 3) = 7424; code 17 with sc 0 and m 1 gives -256; a code whose fifth bit is clear
    (15) matches Q4K's 3840."""
    xq = np.ones((1, 256), np.int8)
    xd = np.ones((1, 8), np.float32)
    one = np.ones((1, 1), np.float16)
    for code, sc, mn, want in [(31, 1, 0, 7936.0), (16, 2, 3, 7424.0), (17, 0, 1, -256.0), (15, 1, 0, 3840.0)]:
        W = pack_q5k(np.full((1, 256), code, np.uint8), np.full((1, 8), sc), np.full((1, 8), mn), one, one)
        y, A = orc.mmvq(W, 1, 256, 4, xq, xd)
        assert y[0, 0] == want, (code, sc, mn, y)


def test_q5k_fifth_bit_positions(orc):
    """One code 16 at element j, all others 0, x = one-hot at element j: the block dot is 16 exactly
    for the one matching element, 0 for every other placement (a wrong bit index shows here)."""
    for j in range(32):
        q = np.zeros((1, 256), np.uint8)
        q[0, j] = 16
        W = pack_q5k(q, np.ones((1, 8), np.uint8), np.zeros((1, 8), np.uint8),
                     np.ones((1, 1), np.float16), np.ones((1, 1), np.float16))
        for i in (j, (j + 1) % 32, (j + 4) % 32, (j + 16) % 32):
            xq = np.zeros((1, 256), np.int8)
            xq[0, i] = 1
            isum = orc.block_dots(W, 1, 256, 4, xq)
            assert isum[0, 0, 0] == (16 if i == j else 0), (j, i, isum[0, 0, 0])


def test_q5k_brute_force_dense(orc):
    rng = np.random.default_rng(29)
    rows, cols, T = 5, 768, 3
    q = rng.integers(0, 32, size=(rows, cols)).astype(np.uint8)
    sc = rng.integers(0, 64, size=(rows, cols // 32)).astype(np.uint8)
    mn = rng.integers(0, 64, size=(rows, cols // 32)).astype(np.uint8)
    d = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
    dmin = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
    W = pack_q5k(q, sc, mn, d, dmin)
    assert W.size == rows * (cols // 256) * 180
    xq, xd, _ = orc.quantize_act(rng.standard_normal((T, cols)).astype(np.float32))
    w = (d.astype(np.float64).repeat(256, axis=1) * sc.astype(np.float64).repeat(32, axis=1) * q
         - dmin.astype(np.float64).repeat(256, axis=1) * mn.astype(np.float64).repeat(32, axis=1))
    ref = (xq.astype(np.float64) * xd.astype(np.float64).repeat(32, axis=1)) @ w.T
    y, A = orc.mmvq(W, rows, cols, 4, xq, xd)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    isum = orc.block_dots(W, rows, cols, 4, xq)
    want = np.einsum("rbj,tbj->trb", q.astype(np.int64).reshape(rows, -1, 32), xq.astype(np.int64).reshape(T, -1, 32))
    assert np.array_equal(isum.reshape(T, rows, cols // 32), want)
    from block_quantized_token_strata_gb300 import synth
    assert np.array_equal(synth.make_q5k_buffer(q, sc, mn, d, dmin), W)


def test_quantizer_is_blockwise_so_inputs_concatenate(orc):
    """The quantizer sees one 32-value block at a time: quantizing inputs of different widths laid
    end to end as one row gives each input's own codes, scales and sums (the window quantizes all
    of its inputs in one call on this property)."""
    rng = np.random.default_rng(41)
    parts = [rng.standard_normal((4, c)).astype(np.float32) * s for c, s in ((2048, 1.0), (4096, 3.0), (96, 0.01))]
    parts[1][0, :32] = 0.0                                       # an all-zero block inside the row
    flat = np.concatenate([p.reshape(-1) for p in parts])[None, :]
    qf, df, sf = orc.quantize_act(flat)
    qs, ds, ss = [], [], []
    for p in parts:
        q, d, s = orc.quantize_act(p)
        qs.append(q.reshape(-1)); ds.append(d.reshape(-1)); ss.append(s.reshape(-1))
    assert np.array_equal(qf[0], np.concatenate(qs))
    assert np.array_equal(df[0].view(np.uint32), np.concatenate(ds).view(np.uint32))
    assert np.array_equal(sf[0], np.concatenate(ss))


@pytest.mark.parametrize("fmt", [0, 1, 2, 3, 4])
def test_tolerance_mass_is_sum_of_abs_terms(orc, fmt):
    """A (the tolerance's mass) is the sum of |term| over the format's terms, computed here from the
    unpacked fields: Q4 / Q8 one term per block (d_w*d_x*isum, isum = sum (q-8)x or sum qx), Q6 one
    per 16 weights (d*s*d_x*isum16), Q4K / Q5K two per block (d*sc*d_x*isum and -dmin*m*d_x*sum x).
    A too-large A (say summed twice, or summed over the signed terms' absolute total) would loosen
    every GPU comparison; rows hold many blocks with terms of both signs, so such a mistake shows."""
    rng = np.random.default_rng(53 + fmt)
    rows, cols, T = 3, 512, 2
    nb = cols // 32
    xq, xd, _ = orc.quantize_act(rng.standard_normal((T, cols)).astype(np.float32))
    x = xq.astype(np.int64).reshape(T, nb, 32)
    dx = xd.astype(np.float64)
    if fmt in (0, 1):
        q = (rng.integers(0, 16, size=(rows, cols)) if fmt == 0 else rng.integers(-127, 128, size=(rows, cols)))
        d = (np.abs(rng.standard_normal((rows, nb))) * 0.01).astype(np.float16)
        W = pack_q4(q, d) if fmt == 0 else pack_q8(q, d)
        qq = q.astype(np.int64).reshape(rows, nb, 32) - (8 if fmt == 0 else 0)
        isum = np.einsum("rbj,tbj->trb", qq, x)
        terms = d.astype(np.float64)[None] * dx[:, None, :] * isum
        assert (terms > 0).any() and (terms < 0).any()
    elif fmt == 2:
        q = rng.integers(0, 64, size=(rows, cols)).astype(np.uint8)
        sub = rng.integers(-127, 128, size=(rows, cols // 16)).astype(np.int8)
        d = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
        W = pack_q6(q, sub, d)
        qq = q.astype(np.int64).reshape(rows, nb, 2, 16) - 32
        isum16 = np.einsum("rbhj,tbhj->trbh", qq, x.reshape(T, nb, 2, 16))
        terms = (d.astype(np.float64).repeat(8, axis=1)[None, :, :, None] * sub.astype(np.float64).reshape(rows, nb, 2)[None]
                 * dx[:, None, :, None] * isum16)
    else:
        hi = 32 if fmt == 4 else 16
        q = rng.integers(0, hi, size=(rows, cols)).astype(np.uint8)
        sc = rng.integers(0, 64, size=(rows, nb)).astype(np.uint8)
        mn = rng.integers(0, 64, size=(rows, nb)).astype(np.uint8)
        d = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
        dmin = (np.abs(rng.standard_normal((rows, cols // 256))) * 0.001).astype(np.float16)
        W = (pack_q5k if fmt == 4 else pack_q4k)(q, sc, mn, d, dmin)
        isum = np.einsum("rbj,tbj->trb", q.astype(np.int64).reshape(rows, nb, 32), x)
        xsum = x.sum(axis=2)                                                   # [T][nb]
        t1 = d.astype(np.float64).repeat(8, axis=1)[None] * sc.astype(np.float64)[None] * dx[:, None, :] * isum
        t2 = -dmin.astype(np.float64).repeat(8, axis=1)[None] * mn.astype(np.float64)[None] * dx[:, None, :] * xsum[:, None, :]
        terms = np.stack([t1, t2], axis=-1)
    y, A = orc.mmvq(W, rows, cols, fmt, xq, xd)
    want_A = np.abs(terms).reshape(T, rows, -1).sum(axis=2)
    want_y = terms.reshape(T, rows, -1).sum(axis=2)
    assert np.allclose(A, want_A, rtol=1e-12, atol=0)
    assert np.allclose(y, want_y, rtol=1e-12, atol=1e-12 * np.abs(want_y).max())
