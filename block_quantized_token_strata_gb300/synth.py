"""Seeded synthetic inputs for the verify-window path and the prompt-chunk MoE.

This module only draws random numbers (numpy PCG64) and lays them out in the byte formats that
``include/strata.h`` documents. It holds none of the method's arithmetic: no quantisation of
activations, no dot products, no scaling. Both the CUDA path and the CPU oracle take its outputs
as plain inputs.

Distributions (the workload recipe):
  * weight block scales d = fp16(|N(0,1)| * 0.01), rounded to nearest-even by numpy;
  * Q4 codes q ~ U{0..15} (two independent codes per byte, i.e. a uniform byte);
  * Q8 codes q ~ U{-127..127};
  * Q6 (256-weight super-blocks): codes q ~ U{0..63}, sub-block scales ~ U{-127..127} (int8, one
    per 16 weights), super-block scale d = fp16(|N(0,1)| * 0.001);
  * Q4K (256-weight super-blocks with minimums): codes q ~ U{0..15}, per 32 weights a scale
    sc ~ U{0..63} and a minimum m ~ U{0..63}, per 256 weights d and dmin = fp16(|N(0,1)| * 0.001);
  * Q5K: as Q4K with codes q ~ U{0..31};
  * activations x ~ N(0,1) fp32, optionally with a Bernoulli(0.01) mask of elements scaled x20;
  * MoE routing: k distinct experts per token drawn without replacement from a Zipf(1.1)
    law over expert ranks, p_e proportional to (e+1)^-1.1, draw order = slot order.
"""
from __future__ import annotations

import hashlib

import numpy as np

QK = 32
QKS = 256  # Q6 super-block
Q4, Q8, Q6, Q4K, Q5K = 0, 1, 2, 3, 4
_QBYTES = {Q4: 16, Q8: 32, Q6: 24, Q4K: 16, Q5K: 20}


def _rng(*key) -> np.random.Generator:
    """A PCG64 stream keyed by any tuple of ints/strings (stable across machines)."""
    words = []
    for k in key:
        if isinstance(k, str):
            words.append(int.from_bytes(hashlib.sha256(k.encode()).digest()[:4], "little"))
        else:
            words.append(int(k) & 0xFFFFFFFF)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def weight_nbytes(rows: int, cols: int, fmt: int) -> int:
    nb = rows * (cols // QK)
    # per super-block: Q6 one fp16 d, Q4K / Q5K fp16 d and dmin
    extra = rows * (cols // QKS) * (2 if fmt == Q6 else 4) if fmt in (Q6, Q4K, Q5K) else 0
    return nb * (_QBYTES[fmt] + 2) + extra


class Weights:
    """One block-quantized matrix: ``buf`` is the planar byte buffer of the C ABI.

    ``codes(r0, r1)`` returns the integer codes of rows [r0, r1) as int16 [rows][cols] (Q4: 0..15,
    Q8: -127..127) and ``scales`` the fp16 scales [rows][nb]; both are views of the same bytes,
    decoded from the documented layout for tests that need them.
    """

    def __init__(self, rows: int, cols: int, fmt: int, buf: np.ndarray):
        self.rows, self.cols, self.fmt, self.buf = rows, cols, fmt, buf
        self.nb = cols // QK
        self.plane_bytes = rows * self.nb * _QBYTES[fmt]

    @property
    def scales(self) -> np.ndarray:
        return self.buf[self.plane_bytes:].view(np.float16).reshape(self.rows, self.nb)

    def codes(self, r0: int = 0, r1: int | None = None) -> np.ndarray:
        r1 = self.rows if r1 is None else r1
        qb = _QBYTES[self.fmt]
        plane = self.buf[r0 * self.nb * qb: r1 * self.nb * qb]
        if self.fmt == Q8:
            return plane.view(np.int8).astype(np.int16).reshape(r1 - r0, self.cols)
        by = plane.reshape(r1 - r0, self.nb, 16)
        out = np.empty((r1 - r0, self.nb, 32), dtype=np.int16)
        out[:, :, :16] = by & 0x0F
        out[:, :, 16:] = by >> 4
        return out.reshape(r1 - r0, self.cols)


def make_q6_buffer(q: np.ndarray, sub: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Lay out Q6 codes q uint8 [rows][cols] (0..63), sub-block scales int8 [rows][cols/16] and
    super-block scales fp16 [rows][cols/256] in the planar Q6 format of include/strata.h."""
    rows, cols = q.shape
    nb = cols // QK
    qb = q.reshape(rows, nb, 32).astype(np.uint8)
    low = (qb & 15)
    high = (qb >> 4) & 3
    code = np.empty((rows, nb, 24), np.uint8)
    code[:, :, :16] = low[:, :, :16] | (low[:, :, 16:] << 4)
    code[:, :, 16:] = high[:, :, 0:8] | (high[:, :, 8:16] << 2) | (high[:, :, 16:24] << 4) | (high[:, :, 24:32] << 6)
    return np.concatenate([code.reshape(-1), np.asarray(sub, np.int8).reshape(-1).view(np.uint8),
                           np.asarray(d, np.float16).reshape(-1).view(np.uint8)])


def make_q4k_buffer(q: np.ndarray, sc: np.ndarray, mn: np.ndarray, d: np.ndarray, dmin: np.ndarray) -> np.ndarray:
    """Lay out Q4K codes q uint8 [rows][cols] (0..15), per-32 scales sc and minimums mn uint8
    [rows][cols/32] (0..63) and per-256 fp16 d, dmin [rows][cols/256] in the planar Q4K format."""
    rows, cols = q.shape
    nb = cols // QK
    qb = q.reshape(rows, nb, 32).astype(np.uint8)
    code = (qb[:, :, :16] & 15) | ((qb[:, :, 16:] & 15) << 4)
    smp = np.stack([np.asarray(sc, np.uint8), np.asarray(mn, np.uint8)], axis=-1)
    dd = np.stack([np.asarray(d, np.float16), np.asarray(dmin, np.float16)], axis=-1)
    return np.concatenate([code.reshape(-1), smp.reshape(-1), dd.reshape(-1).view(np.uint8)])


def make_q5k_buffer(q: np.ndarray, sc: np.ndarray, mn: np.ndarray, d: np.ndarray, dmin: np.ndarray) -> np.ndarray:
    """Lay out Q5K codes q uint8 [rows][cols] (0..31), per-32 scales and minimums and per-256 fp16
    d, dmin in the planar Q5K format: per row its Q4-style nibble blocks, then one 32-bit word per
    block with the fifth bit of the k-th code of four-code group g (groups of elements 0-15, then
    16-31) at bit 8k + g; then the (sc, m) plane and the (d, dmin) plane as in Q4K."""
    rows, cols = q.shape
    nb = cols // QK
    qb = q.reshape(rows, nb, 32).astype(np.uint32)
    nib = ((qb[:, :, :16] & 15) | ((qb[:, :, 16:] & 15) << 4)).astype(np.uint8)
    fifth = (qb >> 4) & 1                                   # [rows][nb][32]
    groups = fifth.reshape(rows, nb, 8, 4)                  # group g = elements 4g..4g+3
    shifts = (8 * np.arange(4)[None, None, None, :] + np.arange(8)[None, None, :, None]).astype(np.uint32)
    words = (groups << shifts).sum(axis=(2, 3)).astype(np.uint32)  # distinct bits: the sum is an OR
    code = np.concatenate([nib.reshape(rows, nb * 16), words.view(np.uint8).reshape(rows, nb * 4)], axis=1)
    smp = np.stack([np.asarray(sc, np.uint8), np.asarray(mn, np.uint8)], axis=-1)
    dd = np.stack([np.asarray(d, np.float16), np.asarray(dmin, np.float16)], axis=-1)
    return np.concatenate([code.reshape(-1), smp.reshape(-1), dd.reshape(-1).view(np.uint8)])


def make_weights(rows: int, cols: int, fmt: int, *key) -> Weights:
    """A seeded [rows][cols] matrix in Q4, Q8, Q6, Q4K or Q5K (planar layout, see include/strata.h)."""
    if cols % QK or rows <= 0:
        raise ValueError("cols must be a multiple of 32 and rows positive")
    rng = _rng("weights", rows, cols, fmt, *key)
    if fmt == Q6:
        if cols % QKS:
            raise ValueError("Q6 needs cols % 256 == 0")
        q = rng.integers(0, 64, size=(rows, cols), dtype=np.uint8)
        sub = rng.integers(-127, 128, size=(rows, cols // 16), dtype=np.int8)
        d = (np.abs(rng.standard_normal((rows, cols // QKS))) * 0.001).astype(np.float16)
        return Weights(rows, cols, fmt, make_q6_buffer(q, sub, d))
    if fmt == Q4K:
        if cols % QKS:
            raise ValueError("Q4K needs cols % 256 == 0")
        q = rng.integers(0, 16, size=(rows, cols), dtype=np.uint8)
        sc = rng.integers(0, 64, size=(rows, cols // QK), dtype=np.uint8)
        mn = rng.integers(0, 64, size=(rows, cols // QK), dtype=np.uint8)
        d = (np.abs(rng.standard_normal((rows, cols // QKS))) * 0.001).astype(np.float16)
        dmin = (np.abs(rng.standard_normal((rows, cols // QKS))) * 0.001).astype(np.float16)
        return Weights(rows, cols, fmt, make_q4k_buffer(q, sc, mn, d, dmin))
    if fmt == Q5K:
        if cols % QKS:
            raise ValueError("Q5K needs cols % 256 == 0")
        q = rng.integers(0, 32, size=(rows, cols), dtype=np.uint8)
        sc = rng.integers(0, 64, size=(rows, cols // QK), dtype=np.uint8)
        mn = rng.integers(0, 64, size=(rows, cols // QK), dtype=np.uint8)
        d = (np.abs(rng.standard_normal((rows, cols // QKS))) * 0.001).astype(np.float16)
        dmin = (np.abs(rng.standard_normal((rows, cols // QKS))) * 0.001).astype(np.float16)
        return Weights(rows, cols, fmt, make_q5k_buffer(q, sc, mn, d, dmin))
    nb = rows * (cols // QK)
    d = (np.abs(rng.standard_normal(nb)) * 0.01).astype(np.float16)
    if fmt == Q4:
        plane = rng.integers(0, 256, size=nb * 16, dtype=np.uint8)
    elif fmt == Q8:
        plane = rng.integers(-127, 128, size=nb * 32, dtype=np.int8).view(np.uint8)
    else:
        raise ValueError("fmt")
    buf = np.empty(plane.size + 2 * nb, dtype=np.uint8)
    buf[:plane.size] = plane
    buf[plane.size:] = d.view(np.uint8)
    return Weights(rows, cols, fmt, buf)


def make_activations(n: int, cols: int, *key, outliers: bool = False) -> np.ndarray:
    """fp32 [n][cols] ~ N(0,1); with ``outliers`` 1% of the elements are scaled by 20."""
    rng = _rng("act", n, cols, int(outliers), *key)
    x = rng.standard_normal((n, cols), dtype=np.float32)
    if outliers:
        mask = rng.random((n, cols)) < 0.01
        x[mask] *= np.float32(20.0)
    return x


def make_routing(n_tok: int, n_expert: int, k: int, *key, zipf_s: float = 1.1) -> np.ndarray:
    """int32 [n_tok][k]: k distinct experts per token, Zipf(s) over ranks (rank e -> id e)."""
    rng = _rng("route", n_tok, n_expert, k, *key)
    p = (np.arange(1, n_expert + 1, dtype=np.float64)) ** (-zipf_s)
    p /= p.sum()
    ids = np.empty((n_tok, k), dtype=np.int32)
    for t in range(n_tok):
        ids[t] = rng.choice(n_expert, size=k, replace=False, p=p)
    return ids


# ---- named workloads ------------------------------------------------------------------------

# Full verify window: 48 layers x (qkv 2048->5120, o 4096->2048, FFN up 2048->6144, down 6144->2048)
# Q4, then a Q8 head 151936 x 2048. Each projection gets its own seeded input (layers not chained).
WINDOW_LAYERS = 48
WINDOW_HIDDEN = 2048
WINDOW_PROJ = (("qkv", 5120, 2048), ("o", 2048, 4096), ("up", 6144, 2048), ("down", 2048, 6144))
HEAD_VOCAB = 151936


def window_shapes(layers: int = WINDOW_LAYERS, layer_fmt: int = Q4):
    """[(name, rows, cols, fmt)] of every matrix of the verify window, in launch order (the layer
    projections in ``layer_fmt``, Q4 by default; the head in Q8)."""
    out = []
    for layer in range(layers):
        for name, rows, cols in WINDOW_PROJ:
            out.append((f"L{layer}.{name}", rows, cols, layer_fmt))
    out.append(("head", HEAD_VOCAB, WINDOW_HIDDEN, Q8))
    return out


# Prompt-chunk MoE: 128 experts, hidden 2048, inter 768, 3,256 tokens, top-8 Zipf(1.1)
MOE_EXPERTS, MOE_HIDDEN, MOE_INTER, MOE_TOKENS, MOE_TOPK = 128, 2048, 768, 3256, 8
