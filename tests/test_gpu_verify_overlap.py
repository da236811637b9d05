"""Verification in overlap mode (tsv_set_verify_overlap): the calls start
while the kernel before them on the stream still runs (in compact CTAs, or the
stochastic walk at full size) and complete after it.  The results must be
bit-identical to the default mode (itself checked against the oracle), whether
or not an attention launch precedes them, and every output must be complete
when the stream is.  (The full-size walk may run in smaller clusters, whose
sums go in another order; these seeded inputs hold no decision within rounding
of a tie, so that changes nothing here.)
"""
import numpy as np
import pytest
import torch

import workloads as W
from _util import d

pytestmark = pytest.mark.gpu

KEYS = ("path", "accept_len", "bonus", "n_tried", "status")


def _inputs(spec):
    trees, att, gi, si = W.make_trees(spec), None, None, None
    att = W.make_attention_inputs(spec, trees)
    if spec.greedy:
        gi = W.make_greedy_inputs(spec, trees)
    if spec.stochastic:
        si = W.make_stochastic_inputs(spec, trees)
    return trees, att, gi, si


def _verify(tsv, trees, gi, si, warp):
    out = {}
    if gi is not None:
        out["g"] = tsv.tree_verify_greedy(d(gi.logits), d(gi.tokens), d(trees.parent), d(trees.node_offsets))
    if si is not None:
        out["s"] = tsv.tree_verify_stochastic(d(si.llm_logits), d(si.ssm_probs), d(si.tokens), d(trees.parent),
                                              d(trees.node_offsets), d(si.u_accept), d(si.u_sample), **warp)
    return out


def _attention(tsv, spec, trees, att):
    tsv.tree_attention(d(att.q), d(att.k_cache), d(att.v_cache), trees.prefix_len, trees.node_offsets,
                       d(trees.prefix_len), d(trees.node_offsets), parent=d(trees.parent))


def _same(a, b):
    for kind in a:
        for k in KEYS:
            if k in a[kind]:
                assert torch.equal(a[kind][k], b[kind][k]), (kind, k)


COMPACT, FULL = "compact", "full"


def _kinds(tsv, form):
    return tsv.TSV_OVERLAP_GREEDY | (tsv.TSV_OVERLAP_STOCHASTIC if form == COMPACT else
                                     tsv.TSV_OVERLAP_STOCHASTIC_FULL)


@pytest.mark.parametrize("name,warp,form", [("batch32-P2048-n16", {}, COMPACT), ("batch8-ragged-merge64-mss", {}, COMPACT),
                                            ("gqa64x8-P32768-n128", {}, COMPACT), ("llama7b-layer-P1024-n20", {}, COMPACT),
                                            ("batch8-ragged-merge64-mss", {"top_k": 50, "top_p": 0.9}, COMPACT),
                                            ("gqa64x8-P32768-n128", {}, FULL), ("batch32-P2048-n16", {}, FULL),
                                            ("batch8-ragged-merge64-mss", {"top_k": 50, "top_p": 0.9}, FULL)])
def test_overlap_mode_matches_default_mode(tsv, name, warp, form):
    spec = W.SPECS[name]
    trees, att, gi, si = _inputs(spec)
    ref = _verify(tsv, trees, gi, si, warp)
    torch.cuda.synchronize()
    for s in ref.values():
        assert (s["status"].cpu() == 0).all()
    # After a running attention launch (the case the mode is for), then with
    # nothing before it on the stream.
    for precede in (True, False):
        if precede:
            _attention(tsv, spec, trees, att)
        with tsv.verify_overlap(_kinds(tsv, form)):
            got = _verify(tsv, trees, gi, si, warp)
        torch.cuda.synchronize()
        _same(ref, got)


@pytest.mark.parametrize("form", [COMPACT, FULL])
def test_overlap_mode_results_are_complete_when_a_later_kernel_runs(tsv, form):
    """A kernel launched after an overlap-mode call (in stream order) must see
    its finished outputs: the next launch here copies the stochastic call's
    path."""
    spec = W.SPECS["batch8-ragged-merge64-mss"]
    trees, att, gi, si = _inputs(spec)
    ref = _verify(tsv, trees, gi, si, {})["s"]
    torch.cuda.synchronize()
    _attention(tsv, spec, trees, att)
    with tsv.verify_overlap(_kinds(tsv, form)):
        got = _verify(tsv, trees, gi, si, {})["s"]
    later = got["path"].clone()  # an ordinary copy kernel, after the call on the stream
    torch.cuda.synchronize()
    assert torch.equal(later, ref["path"])
    assert torch.equal(got["bonus"], ref["bonus"])


def test_overlap_option_rejects_other_values(tsv):
    h = tsv.handle()
    with pytest.raises(tsv.TSVError):
        tsv.tsv_set_verify_overlap(h, 8)
    tsv.tsv_set_verify_overlap(h, tsv.TSV_OVERLAP_GREEDY | tsv.TSV_OVERLAP_STOCHASTIC |
                               tsv.TSV_OVERLAP_STOCHASTIC_FULL)
    tsv.tsv_set_verify_overlap(h, 0)


@pytest.mark.parametrize("form", [COMPACT, FULL])
def test_overlap_mode_reports_bad_requests_like_the_default_mode(tsv, form):
    """A malformed tree in one request and a token outside the vocabulary in
    another make those requests' CTAs leave early; in overlap mode they still
    wait for the kernel before them, and every output, the statuses included,
    equals the default mode's."""
    spec = W.SPECS["batch8-ragged-merge64-mss"]
    trees, att, gi, si = _inputs(spec)
    offs = trees.node_offsets
    parent = trees.parent.copy()
    parent[offs[2] + 3] = 5  # points forward (parents are local indices below the node)
    tokens = si.tokens.copy()
    tokens[offs[5] + 1] = spec.V + 7

    def run():
        return tsv.tree_verify_stochastic(d(si.llm_logits), d(si.ssm_probs), d(tokens), d(parent), d(offs),
                                          d(si.u_accept), d(si.u_sample))

    ref = run()
    torch.cuda.synchronize()
    want = [0] * spec.B
    want[2], want[5] = tsv.TSV_ERR_BAD_TREE, tsv.TSV_ERR_INVALID_ARG
    assert ref["status"].cpu().tolist() == want
    _attention(tsv, spec, trees, att)
    with tsv.verify_overlap(_kinds(tsv, form)):
        got = run()
    torch.cuda.synchronize()
    _same({"s": ref}, {"s": got})
