"""Pins of the oracle's near-tie report.

The GPU kernels compute in fp32 and the oracle in fp64, so a stochastic
decision whose margin is below 1e-6 may go either way; the parity tests stop
comparing a request after the first decision the oracle reports as such.  The
report must therefore fire exactly on such decisions: an accept test with
|u - p(x)/q(x)| < 1e-6 (p(x) itself when q(x) = 0), and a bonus draw whose
target lies within 1e-6 (relative to the mass) of a cumulative sum.  Each
case places a uniform next to a boundary computed here from the definition
p = softmax(logits), and once well away from it; a copy of the oracle with
the tolerance set to zero (on the CPU) must miss the near cases.
"""
import numpy as np
import pytest

import oracle
from test_oracle_verify_pins import _mutant_verify

LOGITS = np.array([0.3, -0.2, 1.1, 0.0, -0.7], np.float32)


def _p(logits):
    z = logits.astype(np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def _verify(u_acc, u_smp, q_row, token, logits_child=LOGITS, verify=oracle.verify_stochastic):
    """Root 0 with one child 1 carrying `token`, proposed from q_row."""
    llm = np.stack([LOGITS, logits_child]).astype(np.float32)
    ssm = np.stack([np.full(5, 0.2, np.float32), np.asarray(q_row, np.float32)])
    return verify(llm, ssm, np.array([0, token], np.int32), np.array([-1, 0], np.int32),
                  np.array([0, 2], np.int32), np.array([0.0, u_acc], np.float32),
                  np.array(u_smp, np.float32))


def _mid_targets(p):
    """A uniform in the middle of every cumulative interval (far from ties)."""
    c = np.concatenate([[0.0], np.cumsum(p)])
    return (c[:-1] + c[1:]) / 2


Q = np.array([0.05, 0.05, 0.6, 0.2, 0.1], np.float32)


@pytest.mark.parametrize("delta,near", [(3e-7, True), (-3e-7, True), (1e-4, False), (-1e-4, False)])
def test_accept_test_margin(delta, near):
    p = _p(LOGITS)
    ratio = p[2] / float(Q[2])
    u = float(np.float32(ratio + delta))
    mid = _mid_targets(p)
    r = _verify(u, [mid[1], mid[3]], Q, 2)
    assert r["status"][0] == 0
    assert (r["n_near_tie"][0] > 0) == near
    assert r["tie_path_len"][0] == (1 if near else -1)
    # Away from the boundary the decision is the plain comparison.
    if not near:
        assert r["accept_len"][0] == (1 if u < ratio else 0)


@pytest.mark.parametrize("k,delta,near", [(1, 3e-7, True), (3, -3e-7, True), (1, 1e-4, False), (3, -1e-4, False)])
def test_bonus_draw_margin(k, delta, near):
    p = _p(LOGITS)
    target = float(np.float32(np.cumsum(p)[k] + delta))
    # A one-node tree: the bonus is drawn from the root's p with this target.
    r = oracle.verify_stochastic(LOGITS[None, :], np.full((1, 5), 0.2, np.float32), np.array([0], np.int32),
                                 np.array([-1], np.int32), np.array([0, 1], np.int32),
                                 np.array([0.0], np.float32), np.array([target], np.float32))
    assert (r["n_near_tie"][0] > 0) == near
    if not near:
        assert r["bonus"][0] == int(np.searchsorted(np.cumsum(p), target, side="right"))


@pytest.mark.parametrize("p_x_logit,near", [(-20.0, True), (1.1, False)])
def test_zero_proposal_margin_is_p(p_x_logit, near):
    """With q(x) = 0 the child is accepted iff p(x) > 0; p(x) itself is the margin."""
    logits = LOGITS.copy()
    logits[4] = p_x_logit
    q = np.array([0.25, 0.25, 0.25, 0.25, 0.0], np.float32)
    llm = np.stack([logits, LOGITS]).astype(np.float32)
    mid = _mid_targets(_p(LOGITS))
    r = oracle.verify_stochastic(llm, np.stack([np.full(5, 0.2, np.float32), q]), np.array([0, 4], np.int32),
                                 np.array([-1, 0], np.int32), np.array([0, 2], np.int32),
                                 np.array([0.0, 0.5], np.float32), np.array([mid[0], mid[2]], np.float32))
    assert (r["n_near_tie"][0] > 0) == near
    assert r["accept_len"][0] == 1  # p(x) > 0 either way


@pytest.mark.parametrize("delta,near", [(3e-7, True), (-3e-7, True), (1e-3, False), (-1e-3, False)])
def test_top_p_cut_margin(delta, near):
    """The top-p cut: the shortest ranked prefix whose share reaches top_p; a
    share within 1e-6 of top_p is a near tie."""
    p = _p(LOGITS)
    share = np.sort(p)[::-1][:2].sum()  # the two largest tokens
    top_p = float(share + delta)
    r = oracle.verify_stochastic(LOGITS[None, :], np.full((1, 5), 0.2, np.float32), np.array([0], np.int32),
                                 np.array([-1], np.int32), np.array([0, 1], np.int32),
                                 np.array([0.0], np.float32), np.array([0.999], np.float32),
                                 top_k=5, top_p=top_p)
    assert (r["n_near_tie"][0] > 0) == near
    if not near:
        # A uniform near 1 draws the last kept token in index order: tokens
        # {0, 2} are kept below the share, {0, 2, 3} just above it.
        assert r["bonus"][0] == (3 if delta > 0 else 2)


def test_zero_tolerance_copy_misses_the_near_cases(tmp_path):
    """Negative control, planted in a copy of the oracle on the CPU."""
    verify = _mutant_verify(tmp_path, "#define NEAR_TIE_EPS 1e-6", "#define NEAR_TIE_EPS 0.0")
    p = _p(LOGITS)
    u = float(np.float32(p[2] / float(Q[2]) + 3e-7))
    mid = _mid_targets(p)
    assert _verify(u, [mid[1], mid[3]], Q, 2, verify=verify)["n_near_tie"][0] == 0
    assert _verify(u, [mid[1], mid[3]], Q, 2)["n_near_tie"][0] > 0


def test_near_ties_are_rare_on_random_inputs():
    """About 2e-6 per decision: none expected over a few hundred decisions."""
    import workloads as W
    tried = near = 0
    for seed in range(16):
        spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], wid=9000 + seed, V=1000)
        trees = W.make_trees(spec)
        si = W.make_stochastic_inputs(spec, trees)
        r = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                     si.u_accept, si.u_sample)
        tried += int(r["n_tried"].sum()) + spec.B  # accept tests and bonus draws
        near += int(r["n_near_tie"].sum())
    assert tried > 300 and near == 0
