"""GPU parity of stochastic verification against a top-k / top-p warped LLM
distribution.  As for the unwarped call, paths, accept lengths and bonus tokens
must match the oracle bit for bit, except after a decision the oracle marks as
a near tie (an accept margin, a bonus boundary or a top-p cut within 1e-6)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import compare_stochastic, d

pytestmark = pytest.mark.gpu


def _run(tsv, trees, si, **kw):
    r = tsv.tree_verify_stochastic(d(si.llm_logits), d(si.ssm_probs), d(si.tokens), d(trees.parent),
                                   d(trees.node_offsets), d(si.u_accept), d(si.u_sample), **kw)
    torch.cuda.synchronize()
    ref = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                   si.u_accept, si.u_sample, temperature=kw.get("temperature", 1.0),
                                   top_k=kw.get("top_k", 0), top_p=kw.get("top_p", 1.0))
    return r, ref


def _propose_like_llm(si, trees, seed=0, top_k=0, top_p=1.0):
    """Proposals close to the (warped) LLM law at each node's parent, tokens
    drawn from them, so that accepted children become likely: 0.7 x the warped
    law + 0.3 x softmax of the parent's row."""
    offs = trees.node_offsets
    prow = np.concatenate([np.maximum(trees.parent[offs[b]:offs[b + 1]], 0) + offs[b]
                           for b in range(len(offs) - 1)])
    lg_par = si.llm_logits[prow]
    p = W.proposal_rows(lg_par).astype(np.float64)
    V = p.shape[1]
    if top_k or top_p < 1.0:
        w = np.zeros_like(p)
        for i, (row, lg) in enumerate(zip(p, lg_par)):
            order = np.lexsort((np.arange(V), -lg.astype(np.float64)))
            keep = order[:top_k] if 0 < top_k < V else order
            if top_p < 1.0:
                c = np.cumsum(row[keep]) / row[keep].sum()
                keep = keep[:int(np.searchsorted(c, top_p)) + 1]
            w[i, keep] = row[keep] / row[keep].sum()
        p = 0.7 * w + 0.3 * p
    si.ssm_probs[:] = p.astype(np.float32)
    rng = np.random.default_rng(seed)
    cdf = np.cumsum(si.ssm_probs.astype(np.float64), axis=1)
    u = rng.random(len(cdf))[:, None] * cdf[:, -1:]
    si.tokens[:] = np.minimum((u >= cdf).sum(1), V - 1).astype(np.int32)


def _case(name, like_llm, top_k=0, top_p=1.0, **kw):
    spec = W.spec_variant(W.SPECS[name], **kw)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    if like_llm:
        _propose_like_llm(si, trees, 0, top_k, top_p)
    return spec, trees, si


@pytest.mark.parametrize("top_k,top_p", [(50, 1.0), (50, 0.9), (3, 1.0), (1024, 0.5), (200, 0.95)])
@pytest.mark.parametrize("like_llm", [False, True])
def test_batch8_warped(tsv, top_k, top_p, like_llm):
    spec, trees, si = _case("batch8-ragged-merge64-mss", like_llm, top_k, top_p, prefix=64)
    r, ref = _run(tsv, trees, si, top_k=top_k, top_p=top_p)
    near = compare_stochastic(r, ref, trees)
    assert near <= 2
    if like_llm:
        assert ref["accept_len"].sum() > 0


def test_top_k_one_is_greedy_on_the_gpu(tsv):
    spec, trees, si = _case("batch8-ragged-merge64-mss", True, 1, 1.0, prefix=64)
    r, _ = _run(tsv, trees, si, top_k=1)
    g = tsv.tree_verify_greedy(d(si.llm_logits), d(si.tokens), d(trees.parent), d(trees.node_offsets))
    torch.cuda.synchronize()
    assert np.array_equal(r["path"].cpu().numpy(), g["path"].cpu().numpy())
    assert np.array_equal(r["bonus"].cpu().numpy(), g["bonus"].cpu().numpy())


def test_long_vocabulary_warped(tsv):
    spec, trees, si = _case("gqa64x8-P32768-n128", True, 50, 0.9, prefix=64, nodes=40)
    r, ref = _run(tsv, trees, si, top_k=50, top_p=0.9, temperature=0.7)
    compare_stochastic(r, ref, trees)


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_warped(tsv, seed):
    V = [5, 17, 300, 1000, 4099, 32000][seed]
    spec = W.spec_variant(W.fuzz_spec(400 + seed), V=V)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    top_k = [1, 50, 7, 1024, 64, 500][seed]
    top_p = [1.0, 0.8, 0.6, 0.95, 1.0, 0.3][seed]
    if seed % 2:
        _propose_like_llm(si, trees, seed, top_k, top_p)
    r, ref = _run(tsv, trees, si, top_k=top_k, top_p=top_p)
    compare_stochastic(r, ref, trees)


def test_equal_logits_at_the_boundary(tsv):
    # Logits on a coarse grid: many tokens tie at the top-k boundary, so the
    # cut by token index decides which of them stay.
    spec, trees, si = _case("batch8-ragged-merge64-mss", True, prefix=64, B=4, V=5000)
    si.llm_logits[:] = np.round(si.llm_logits * 2.0) / 2.0
    _propose_like_llm(si, trees, 5, 100, 0.9)
    for top_k, top_p in [(10, 1.0), (100, 0.9), (1000, 1.0)]:
        r, ref = _run(tsv, trees, si, top_k=top_k, top_p=top_p)
        compare_stochastic(r, ref, trees)


def test_warp_argument_checks(tsv):
    spec, trees, si = _case("batch8-ragged-merge64-mss", False, prefix=64, B=1, V=100)
    for kw, code in [(dict(top_k=1025), tsv.TSV_ERR_UNSUPPORTED), (dict(top_k=0, top_p=0.5), tsv.TSV_ERR_UNSUPPORTED),
                     (dict(top_k=5, top_p=0.0), tsv.TSV_ERR_INVALID_ARG), (dict(top_k=5, top_p=1.5), tsv.TSV_ERR_INVALID_ARG),
                     (dict(top_k=-1, top_p=0.5), tsv.TSV_ERR_INVALID_ARG)]:
        with pytest.raises(tsv.TSVError) as e:
            tsv.tree_verify_stochastic(d(si.llm_logits), d(si.ssm_probs), d(si.tokens), d(trees.parent),
                                       d(trees.node_offsets), d(si.u_accept), d(si.u_sample), **kw)
        assert e.value.code == code
