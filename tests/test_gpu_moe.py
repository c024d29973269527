"""GPU parity of the prompt-chunk MoE (strata_moe_grouped) against the CPU oracle.

Bars: the per-expert grouping equals the oracle's exactly; the fp32 gate and up outputs g, u (read
back through the strata_moe_grouped_gu test hook, which runs the same kernels) lie element by element
within the stated bound |gpu - oracle| <= 2e-6 * sum|block terms| + 1e-6 of the oracle's fp64 g, u;
the down projection's integer dots are pinned by feeding the GPU's own re-quantized hidden rows to
the oracle (so y must then lie within the fp32 bound); the re-quantized hidden codes equal the
oracle's up to a one-step flip where fp32 SiLU rounding moves a value across a rounding boundary;
out-of-range ids set the error word and leave their rows untouched.
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


class MoeCase:
    def __init__(self, n_exp, hidden, inter, n_tok, k, key):
        self.n_exp, self.hidden, self.inter, self.n_tok, self.k = n_exp, hidden, inter, n_tok, k
        self.host = [(synth.make_weights(inter, hidden, synth.Q4, key, "g", e),
                      synth.make_weights(inter, hidden, synth.Q4, key, "u", e),
                      synth.make_weights(hidden, inter, synth.Q4, key, "d", e)) for e in range(n_exp)]
        self.dev = [tuple(cu(m.buf) for m in ex) for ex in self.host]
        self.tab = strata.expert_table(self.dev, "cuda")
        self.ids = synth.make_routing(n_tok, n_exp, k, key)
        self.x = synth.make_activations(n_tok, hidden, key)

    def bufs(self):
        return [(g.buf, u.buf, d.buf) for g, u, d in self.host]

    def run(self, ids=None, y_init=None, with_gu=True):
        ids = self.ids if ids is None else ids
        ws = torch.empty(strata.moe_grouped_workspace(self.n_exp, self.n_tok, self.k, self.hidden, self.inter),
                         dtype=torch.uint8, device="cuda")
        err = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        y = (torch.full((self.n_tok * self.k, self.hidden), float(y_init), device="cuda")
             if y_init is not None else None)
        gu = (torch.full((self.n_tok * self.k, 2, self.inter), float("nan"), device="cuda") if with_gu else None)
        y = strata.moe_grouped(self.tab, self.n_exp, self.hidden, self.inter, cu(ids), cu(self.x), y=y,
                               workspace=ws, err_word=err, gu=gu)
        torch.cuda.synchronize()
        v = strata.moe_debug_views(self.n_exp, self.n_tok, self.k, self.hidden, self.inter)
        wsn = ws.cpu().numpy()
        n_pair = self.n_tok * self.k
        nbi = self.inter // 32
        out = dict(
            y=y.cpu().numpy(), err=int(err.item()),
            counts=wsn[v["counts"]:v["counts"] + 4 * self.n_exp].view(np.int32).copy(),
            offsets=wsn[v["offsets"]:v["offsets"] + 4 * (self.n_exp + 1)].view(np.int32).copy(),
            pairs=wsn[v["pairs"]:v["pairs"] + 4 * n_pair].view(np.int32).copy(),
            hq=wsn[v["hq"]:v["hq"] + n_pair * self.inter].view(np.int8).reshape(n_pair, self.inter).copy(),
            hd=wsn[v["hd"]:v["hd"] + 4 * n_pair * nbi].view(np.float32).reshape(n_pair, nbi).copy(),
            hs=wsn[v["hs"]:v["hs"] + 4 * n_pair * nbi].view(np.int32).reshape(n_pair, nbi).copy())
        out["gu"] = gu.cpu().numpy() if with_gu else None
        return out


def check_rows(case, out, sel):
    """y of pairs ``sel`` against the oracle fed with the GPU's own hidden codes; hidden codes
    against the oracle's own re-quantization (one-step flips only at rounding boundaries)."""
    pos_of = np.empty(case.n_tok * case.k, np.int64)
    n_valid = out["offsets"][-1]
    pos_of[out["pairs"][:n_valid]] = np.arange(n_valid)
    pos = pos_of[sel]
    ref = oracle.moe_rows(case.bufs(), case.hidden, case.inter, case.ids, case.x, sel, want_hidden=True,
                          hq_in=out["hq"][pos], hd_in=out["hd"][pos], want_gate_up=out["gu"] is not None)
    if out["gu"] is not None:
        # gate and up at the stated bound, element by element
        for plane, name, mass in ((0, "g", "Ag"), (1, "u", "Au")):
            got = out["gu"][sel, plane].astype(np.float64)
            e = np.abs(got - ref[name])
            t = oracle.tolerance(ref[mass])
            assert (e <= t).all(), f"{name}: {(e > t).sum()} of {e.size} outside the bound, worst {(e / t).max():.3g}x"
    tol = oracle.tolerance(ref["A"])
    err = np.abs(out["y"][sel].astype(np.float64) - ref["y"])
    assert (err <= tol).all(), f"{(err > tol).sum()} of {err.size} y values outside the bound"
    # hidden re-quantization
    assert np.allclose(out["hd"][pos], ref["hd"], rtol=1e-4, atol=0)
    hq_g, hq_o = out["hq"][pos].astype(np.int32), ref["hq"].astype(np.int32)
    diff = np.abs(hq_g - hq_o)
    assert diff.max() <= 1
    v = ref["h"] / np.repeat(ref["hd"].astype(np.float64), 32, axis=1)
    near = np.abs(np.abs(v) - np.floor(np.abs(v)) - 0.5) < 0.02
    assert not (diff.astype(bool) & ~near).any()
    assert np.array_equal(out["hs"][pos], hq_g.reshape(len(sel), -1, 32).sum(axis=2))


def test_moe_small_full_parity():
    case = MoeCase(16, 256, 128, 300, 4, "moe-small")
    out = case.run()
    counts, offsets, pairs, bad = oracle.moe_bucket(case.ids, case.n_exp)
    assert bad == 0 and out["err"] == 0
    assert np.array_equal(out["counts"], counts)
    assert np.array_equal(out["offsets"], offsets)
    assert np.array_equal(out["pairs"], pairs)
    check_rows(case, out, np.arange(case.n_tok * case.k))


def test_moe_one_token_one_expert():
    case = MoeCase(1, 128, 128, 1, 1, "moe-one")
    out = case.run()
    check_rows(case, out, np.array([0]))


def test_moe_bad_ids_flag_and_skip():
    case = MoeCase(8, 128, 128, 40, 2, "moe-bad")
    ids = case.ids.copy()
    ids[3, 1] = -1
    ids[17, 0] = 8
    ids[39, 1] = 1 << 20
    case.ids = ids
    out = case.run(ids=ids, y_init=123.0)
    assert out["err"] == 1
    bad = [3 * 2 + 1, 17 * 2 + 0, 39 * 2 + 1]
    assert (out["y"][bad] == 123.0).all()
    assert np.isnan(out["gu"][bad]).all()                     # the hook skips them too
    counts, offsets, pairs, nbad = oracle.moe_bucket(ids, 8)
    assert nbad == 3 and np.array_equal(out["pairs"][:offsets[-1]], pairs[:offsets[-1]])
    good = np.setdiff1d(np.arange(80), bad)
    check_rows(case, out, good)


@pytest.fixture(scope="module")
def c5():
    return MoeCase(synth.MOE_EXPERTS, synth.MOE_HIDDEN, synth.MOE_INTER, synth.MOE_TOKENS, synth.MOE_TOPK,
                   "prompt-moe")


def test_moe_prompt_chunk_sampled(c5):
    """The 3,256-token, 128-expert, top-8 chunk: grouping exact; rows of the heaviest expert and a
    seeded 3% sample of all pairs within the bound."""
    out = c5.run()
    counts, offsets, pairs, bad = oracle.moe_bucket(c5.ids, c5.n_exp)
    assert bad == 0 and out["err"] == 0
    assert np.array_equal(out["counts"], counts) and np.array_equal(out["pairs"], pairs)
    assert counts.max() > 2000 and counts.min() < 100          # the Zipf(1.1) skew is there
    rng = np.random.default_rng(0)
    heavy = pairs[offsets[0]:offsets[1]][::8]                   # every 8th pair of expert 0
    light = pairs[offsets[127]:offsets[128]]                    # all pairs of the rarest id
    sample = rng.choice(c5.n_tok * c5.k, size=(c5.n_tok * c5.k) * 3 // 100, replace=False)
    sel = np.unique(np.concatenate([heavy, light, sample]))
    check_rows(c5, out, sel)
    # every row written exactly once: a second run, through the product entry point, with a NaN-filled
    # y leaves no NaN and equals the test hook's run bit for bit (same kernels)
    out2 = c5.run(y_init=float("nan"), with_gu=False)
    assert not np.isnan(out2["y"]).any()
    assert np.array_equal(out2["y"], out["y"])
    assert not np.isnan(out["gu"]).any()


def test_moe_idle_experts_get_no_tiles():
    """Experts no pair routes to (the first, the last and some between) hold no M-tile; the rest are
    exact as usual."""
    case = MoeCase(8, 256, 128, 120, 2, "moe-idle")
    rng = np.random.default_rng(11)
    used = np.array([1, 5, 6], np.int32)
    ids = np.stack([rng.choice(used, size=2, replace=False) for _ in range(case.n_tok)]).astype(np.int32)
    case.ids = ids
    out = case.run(ids=ids)
    counts, offsets, pairs, bad = oracle.moe_bucket(ids, case.n_exp)
    assert bad == 0 and out["err"] == 0
    assert np.array_equal(out["counts"], counts) and (counts[[0, 2, 3, 4, 7]] == 0).all()
    assert np.array_equal(out["offsets"], offsets) and np.array_equal(out["pairs"], pairs)
    check_rows(case, out, np.arange(case.n_tok * case.k))


def test_moe_tile_boundaries():
    """Experts with exactly 128, 129 and 1 pairs: a full M-tile, a full tile plus a one-row tile, and
    a one-row tile; rows in a shuffled order."""
    n_tok = 258
    case = MoeCase(3, 128, 128, n_tok, 1, "moe-edges")
    ids = np.concatenate([np.zeros(128), np.ones(129), [2]]).astype(np.int32)
    np.random.default_rng(5).shuffle(ids)
    ids = ids.reshape(n_tok, 1)
    case.ids = ids
    out = case.run(ids=ids)
    counts, offsets, pairs, bad = oracle.moe_bucket(ids, 3)
    assert list(out["counts"]) == [128, 129, 1] and np.array_equal(out["pairs"], pairs)
    check_rows(case, out, np.arange(n_tok))
