"""The seeded input generators (CPU): sizes match the documented formats, the same key gives the
same bytes on every call, another key gives other bytes, and the drawn values follow the stated
recipe (code ranges, outlier rate, routing law). Both the oracle and the CUDA path read these
inputs, so a drift here would move both sides together; these checks pin the recipe itself."""
import numpy as np
import pytest

from block_quantized_token_strata_gb300 import synth

FORMATS = [(synth.Q4, 18 * 8), (synth.Q8, 34 * 8), (synth.Q6, 210), (synth.Q4K, 148), (synth.Q5K, 180)]


@pytest.mark.parametrize("fmt,per256", FORMATS)
def test_weight_sizes_and_determinism(fmt, per256):
    rows, cols = 7, 512
    a = synth.make_weights(rows, cols, fmt, "synth-test", 1)
    b = synth.make_weights(rows, cols, fmt, "synth-test", 1)
    c = synth.make_weights(rows, cols, fmt, "synth-test", 2)
    assert a.buf.size == synth.weight_nbytes(rows, cols, fmt) == rows * (cols // 256) * per256
    assert np.array_equal(a.buf, b.buf)
    assert not np.array_equal(a.buf, c.buf)


def test_q4_q8_code_and_scale_ranges():
    rows, cols = 64, 1024
    nb = cols // 32
    w8 = synth.make_weights(rows, cols, synth.Q8, "ranges")
    codes8 = w8.buf[:rows * nb * 32].view(np.int8)
    assert codes8.min() >= -127 and codes8.max() <= 127
    d8 = w8.buf[rows * nb * 32:].view(np.float16).astype(np.float64)
    assert (d8 >= 0).all() and 0.004 < d8.mean() < 0.012      # |N(0,1)| * 0.01 has mean 0.008
    w4 = synth.make_weights(rows, cols, synth.Q4, "ranges")
    nib = np.concatenate([w4.buf[:rows * nb * 16] & 15, w4.buf[:rows * nb * 16] >> 4])
    assert nib.min() == 0 and nib.max() == 15


def test_activations_and_outlier_rate():
    x = synth.make_activations(64, 4096, "synth-test")
    assert x.dtype == np.float32 and abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    xo = synth.make_activations(64, 4096, "synth-test", outliers=True)
    big = np.abs(xo) > 8.0                                      # N(0,1) beyond 8 sigma: practically never
    assert 0.006 < big.mean() < 0.012                           # the 1% scaled x20 (most land past 8)
    assert np.array_equal(xo, synth.make_activations(64, 4096, "synth-test", outliers=True))


def test_routing_distinct_and_zipf_ordered():
    ids = synth.make_routing(3256, 128, 8, "synth-test")
    assert ids.shape == (3256, 8) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < 128
    assert all(len(set(row)) == 8 for row in ids.tolist())      # k distinct experts per token
    counts = np.bincount(ids.reshape(-1), minlength=128)
    assert counts[0] > counts[10] > counts[100]                 # lower ranks drawn more often
    assert np.array_equal(ids, synth.make_routing(3256, 128, 8, "synth-test"))


def test_window_shapes():
    shapes = synth.window_shapes(2)
    assert len(shapes) == 2 * 4 + 1 and shapes[-1] == ("head", synth.HEAD_VOCAB, synth.WINDOW_HIDDEN, synth.Q8)
    total = sum(synth.weight_nbytes(r, c, f) for _, r, c, f in synth.window_shapes())
    assert total == 1519697920                                  # the full window: 1.52 GB per step
