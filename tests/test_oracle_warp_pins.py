"""Pins of the warped LLM distribution in the oracle's stochastic verification
(top-k, then top-p, before multi-step speculative sampling).

The warp is fixed without restating the oracle's ranking code: top-k = 1 must
reproduce greedy verification (an independent oracle function) for any
uniforms; hand-derived warped distributions are checked exactly through the
bonus draw's inverse CDF (ties included); settings that warp nothing leave the
result unchanged; and a chi-square test checks that verification with warping
emits the warped law (SpecInfer §1 Correctness: MSS preserves the distribution
it verifies against).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from test_oracle_verify_pins import _chi2_pvalue, _run_mss_markov, _softmax


def _stochastic_case(seed, V=50, B=4):
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], wid=3000 + seed, B=B, V=V)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    return trees, si


@pytest.mark.parametrize("seed", range(4))
def test_top_k_one_is_greedy_verification(seed):
    trees, si = _stochastic_case(seed)
    r = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                 si.u_accept, si.u_sample, top_k=1)
    g = oracle.verify_greedy(si.llm_logits, si.tokens, trees.parent, trees.node_offsets)
    assert np.array_equal(r["path"], g["path"])
    assert np.array_equal(r["accept_len"], g["accept_len"])
    assert np.array_equal(r["bonus"], g["bonus"])


@pytest.mark.parametrize("seed", range(2))
def test_tiny_top_p_keeps_only_the_top_token(seed):
    trees, si = _stochastic_case(seed)
    a = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                 si.u_accept, si.u_sample, top_p=1e-9)
    b = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                 si.u_accept, si.u_sample, top_k=1)
    for k in ("path", "accept_len", "bonus"):
        assert np.array_equal(a[k], b[k])


def test_settings_that_keep_everything_change_nothing():
    trees, si = _stochastic_case(7)
    base = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                    si.u_accept, si.u_sample)
    for kw in (dict(top_k=50), dict(top_k=10_000), dict(top_k=0, top_p=1.0)):
        r = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                     si.u_accept, si.u_sample, **kw)
        for k in ("path", "accept_len", "bonus", "n_tried"):
            assert np.array_equal(r[k], base[k])


def _bonus_law(logits, grid, **kw):
    """Bonus tokens of a root without children for a grid of sample uniforms."""
    V = len(logits)
    n = len(grid)
    llm = np.tile(np.asarray(logits, np.float32), (n, 1))
    r = oracle.verify_stochastic(llm, np.full((n, V), 1.0 / V, np.float32), np.zeros(n, np.int32),
                                 np.full(n, -1, np.int32), np.arange(n + 1, dtype=np.int32),
                                 np.zeros(n, np.float32), np.asarray(grid, np.float32), **kw)
    assert (r["accept_len"] == 0).all()
    return r["bonus"]


# Hand-derived: p = (0.5, 0.3, 0.15, 0.05).  top_k = 2 keeps tokens 0 and 1:
# (0.625, 0.375).  top_p = 0.7: cumulative 0.5, 0.8 -> keep two, same law.
# top_p = 0.45 -> keep one.  top_p = 0.85: 0.5, 0.8, 0.95 -> keep three:
# (0.5, 0.3, 0.15) / 0.95 = (0.5263, 0.3158, 0.1579).
P4 = np.log(np.array([0.5, 0.3, 0.15, 0.05]))


@pytest.mark.parametrize("kw,cdf", [
    (dict(top_k=2), [0.625, 1.0]),
    (dict(top_p=0.7), [0.625, 1.0]),
    (dict(top_p=0.45), [1.0]),
    (dict(top_p=0.85), [0.5 / 0.95, 0.8 / 0.95, 1.0]),
    (dict(top_k=3, top_p=0.75), [0.5 / 0.8, 1.0]),  # within top-3 (mass 0.95): 0.5/0.95, 0.8/0.95 >= 0.75
])
def test_hand_derived_warped_laws(kw, cdf):
    grid = np.linspace(0.0005, 0.9995, 400)
    got = _bonus_law(P4, grid, **kw)
    want = np.searchsorted(np.array(cdf), grid, side="right")
    # Away from the boundaries (rounding of the cumulative sums) the draw is exact.
    far = np.min(np.abs(grid[:, None] - np.array(cdf)[None, :]), axis=1) > 1e-4
    assert np.array_equal(got[far], want[far])


def test_equal_logits_at_the_cut_keep_the_lower_index():
    # Tokens 1 and 2 share the largest logit: top_k = 1 keeps token 1.
    got = _bonus_law([1.0, 2.0, 2.0, 0.0], np.linspace(0.01, 0.99, 50), top_k=1)
    assert (got == 1).all()
    # top_k = 2 keeps both (p = 1/2 each), never token 0 or 3.
    got = _bonus_law([1.0, 2.0, 2.0, 0.0], np.linspace(0.01, 0.99, 50), top_k=2)
    assert set(got.tolist()) == {1, 2}


def _warped_law(k=0, p=1.0):
    def law(A):
        out = []
        for row in _softmax(A):
            keep = np.argsort(-row, kind="stable")
            keep = keep[:k] if k else keep
            if p < 1.0:
                m = row[keep].sum()
                j = int(np.searchsorted(np.cumsum(row[keep]) / m, p - 1e-12)) + 1
                keep = keep[:j]
            w = np.zeros_like(row)
            w[keep] = row[keep]
            out.append(w / w.sum())
        return np.array(out)
    return law


@pytest.mark.parametrize("kw", [dict(k=2), dict(k=3, p=0.8)])
def test_mss_preserves_the_warped_law(kw):
    law = _warped_law(**kw)
    verify = lambda *a: oracle.verify_stochastic(*a, top_k=kw.get("k", 0), top_p=kw.get("p", 1.0))
    obs, exp = _run_mss_markov(verify, trials=60_000, seed=23, law=law)
    assert _chi2_pvalue(obs, exp) > 1e-3
