"""Pins of the temperature in the oracle's stochastic verification (the LLM
distribution is softmax(logits / T); SpecInfer §4 Token Verification samples
from the LLM's distribution, and §1 Correctness requires that MSS reproduces
whatever distribution it verifies against).

Each pin fixes T by something other than the oracle's own softmax: dividing
by a power of two is exact, so T = 2^e on logits l must give the same result,
bit for bit, as T = 1 on l / 2^e; as T goes to zero the LLM distribution is
one-hot at the argmax, so verification must reduce to greedy verification (an
independent oracle function, pinned against incremental decoding); and a
chi-square test checks that the emitted tokens follow softmax(A / T) of a
Markov toy LLM.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from test_oracle_verify_pins import _chi2_pvalue, _mutant_verify, _run_mss_markov, _softmax


def _case(seed, V=50, B=6):
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], wid=5000 + seed, B=B, V=V)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    # Make about half the children carry their parent's argmax token, so that
    # the walks go deeper than the root.
    rng = np.random.default_rng(seed)
    tok = si.tokens.copy()
    for b in range(spec.B):
        off = int(trees.node_offsets[b])
        for i in range(1, int(trees.node_offsets[b + 1]) - off):
            if rng.random() < 0.5:
                tok[off + i] = int(np.argmax(si.llm_logits[off + int(trees.parent[off + i])]))
    return trees, si, tok


def _run(verify, trees, si, tok, logits, T):
    return verify(logits, si.ssm_probs, tok, trees.parent, trees.node_offsets, si.u_accept, si.u_sample, T)


def _power_of_two_pin(verify, seed, e):
    """(holds, T matters): T = 2^e on l against T = 1 on l / 2^e, and against T = 1 on l."""
    trees, si, tok = _case(seed)
    T = 2.0 ** e
    a = _run(verify, trees, si, tok, si.llm_logits, T)
    b = _run(verify, trees, si, tok, (si.llm_logits / np.float32(T)).astype(np.float32), 1.0)
    c = _run(verify, trees, si, tok, si.llm_logits, 1.0)
    keys = ("path", "accept_len", "bonus", "n_tried")
    return (all(np.array_equal(a[k], b[k]) for k in keys),
            any(not np.array_equal(a[k], c[k]) for k in keys))


@pytest.mark.parametrize("seed,e", [(0, -1), (1, 1), (2, 2), (3, -3)])
def test_power_of_two_temperature_equals_prescaled_logits(seed, e):
    holds, matters = _power_of_two_pin(oracle.verify_stochastic, seed, e)
    assert holds
    assert matters  # the temperature changes the result here, else the pin proves nothing


def test_power_of_two_pin_rejects_a_multiplying_temperature(tmp_path):
    """Negative control, planted in a copy of the oracle on the CPU: logits
    multiplied by T instead of divided."""
    verify = _mutant_verify(tmp_path, "p[t] = exp((double)x[t] / T - m);", "p[t] = exp((double)x[t] * T - m);")
    assert not all(_power_of_two_pin(verify, seed, e)[0] for seed, e in [(0, -1), (1, 1), (2, 2)])


@pytest.mark.parametrize("seed", range(4))
def test_vanishing_temperature_is_greedy_verification(seed):
    trees, si, tok = _case(seed)
    top2 = np.sort(si.llm_logits, axis=1)[:, -2:]
    assert (top2[:, 1] > top2[:, 0]).all()  # a unique argmax in every row
    # l / 2^-60 separates any two distinct fp32 logits by far more than exp's
    # range, so every probability but the argmax's is exactly zero.
    r = _run(oracle.verify_stochastic, trees, si, tok, si.llm_logits, 2.0 ** -60)
    g = oracle.verify_greedy(si.llm_logits, tok, trees.parent, trees.node_offsets)
    assert np.array_equal(r["path"], g["path"])
    assert np.array_equal(r["accept_len"], g["accept_len"])
    assert np.array_equal(r["bonus"], g["bonus"])
    assert g["accept_len"].sum() > 0


@pytest.mark.parametrize("T", [0.6, 1.7])
def test_mss_preserves_the_tempered_law(T):
    verify = lambda *a: oracle.verify_stochastic(*a, temperature=T)
    obs, exp = _run_mss_markov(verify, trials=60_000, seed=31, law=lambda A: _softmax(A / T))
    assert _chi2_pvalue(obs, exp) > 1e-3
    # The untempered law must be rejected by the same counts.
    _, exp1 = _run_mss_markov(verify, trials=60_000, seed=31, law=_softmax)
    assert _chi2_pvalue(obs, exp1) < 1e-6
