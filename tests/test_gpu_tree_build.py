"""GPU token-tree construction against the oracle, bit for bit: expansion
(top-k children of every frontier row) and merge (union of several trees by
token path)."""
import numpy as np
import pytest
import torch

import oracle
from _util import d

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("F,V,k,grid", [(7, 5, 1, 0.0), (7, 5, 5, 0.5), (33, 1000, 4, 0.0), (33, 1000, 16, 0.5),
                                        (64, 32000, 4, 0.0), (8, 32000, 1024, 0.25), (5, 128256, 8, 0.0),
                                        (300, 3000, 3, 1.0),
                                        # few long rows: each row split over a cluster of CTAs
                                        (1, 128256, 1, 0.0), (2, 50001, 7, 0.5), (3, 40000, 9, 1.0),
                                        (1, 16384, 8, 0.0), (4, 128256, 64, 0.25)])
def test_expand_matches_oracle(tsv, F, V, k, grid):
    rng = np.random.default_rng(F * 7 + k)
    z = (rng.standard_normal((F, V)) * 2).astype(np.float32)
    if grid:  # coarse logits: many ties, decided by token index
        z = (np.round(z / grid) * grid).astype(np.float32)
    got = tsv.tree_expand(d(z), k)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.tree_expand(z, k))


def test_expand_argument_checks(tsv):
    z = d(np.zeros((2, 10), np.float32))
    for k, code in [(0, tsv.TSV_ERR_INVALID_ARG), (11, tsv.TSV_ERR_INVALID_ARG)]:
        with pytest.raises(tsv.TSVError) as e:
            tsv.tree_expand(z, k)
        assert e.value.code == code
    z = d(np.zeros((1, 2000), np.float32))
    with pytest.raises(tsv.TSVError) as e:
        tsv.tree_expand(z, 1025)
    assert e.value.code == tsv.TSV_ERR_UNSUPPORTED


def _random_tree(rng, n, V, root_tok):
    par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    tok = rng.integers(0, V, n).astype(np.int32)
    tok[0] = root_tok
    return par, tok


def _batch(rng, B, V, max_trees=4, max_nodes=40):
    reqs = []
    for b in range(B):
        reqs.append([_random_tree(rng, int(rng.integers(1, max_nodes)), V, 100 + b)
                     for _ in range(int(rng.integers(1, max_trees + 1)))])
    trees = [t for r in reqs for t in r]
    tree_offsets = np.concatenate([[0], np.cumsum([len(t[0]) for t in trees])]).astype(np.int32)
    request_trees = np.concatenate([[0], np.cumsum([len(r) for r in reqs])]).astype(np.int32)
    parent = np.concatenate([t[0] for t in trees])
    tokens = np.concatenate([t[1] for t in trees])
    return reqs, parent, tokens, tree_offsets, request_trees


@pytest.mark.parametrize("seed,V", [(0, 3), (1, 8), (2, 50), (3, 1000)])
def test_merge_matches_oracle(tsv, seed, V):
    rng = np.random.default_rng(seed)
    reqs, parent, tokens, toffs, rtrees = _batch(rng, 6, V)
    r = tsv.tree_merge(d(parent), d(tokens), d(toffs), d(rtrees))
    torch.cuda.synchronize()
    gp, gt, gs = r["parent"].cpu().numpy(), r["tokens"].cpu().numpy(), r["source"].cpu().numpy()
    for b, req in enumerate(reqs):
        par, tok, src = oracle.tree_merge([t[0] for t in req], [t[1] for t in req])
        n0 = int(toffs[rtrees[b]])
        n1 = int(toffs[rtrees[b + 1]])
        cnt = int(r["count"][b])
        assert r["status"][b].item() == 0
        assert cnt == len(par)
        assert np.array_equal(gp[n0:n0 + cnt], par) and np.array_equal(gt[n0:n0 + cnt], tok)
        want_src = [int(toffs[rtrees[b] + t]) + i for t, i in src]
        assert gs[n0:n0 + cnt].tolist() == want_src
        assert (gp[n0 + cnt:n1] == -1).all()


def test_merge_reports_bad_and_oversized_inputs(tsv):
    rng = np.random.default_rng(4)
    # Request 0 fine; request 1's second tree has a forward parent; request 2's
    # union would exceed 256 nodes (five distinct chains of 60).
    good = _random_tree(rng, 10, 5, 1)
    bad = (np.array([-1, 0, 3, 1], np.int32), np.array([1, 2, 3, 4], np.int32))
    chains = [(np.arange(-1, 59, dtype=np.int32), np.full(60, 1000 + c, np.int32)) for c in range(5)]
    for c in chains:
        c[1][0] = 1
    reqs = [[good], [good, bad], chains]
    trees = [t for r in reqs for t in r]
    toffs = np.concatenate([[0], np.cumsum([len(t[0]) for t in trees])]).astype(np.int32)
    rtrees = np.concatenate([[0], np.cumsum([len(r) for r in reqs])]).astype(np.int32)
    r = tsv.tree_merge(d(np.concatenate([t[0] for t in trees])), d(np.concatenate([t[1] for t in trees])),
                       d(toffs), d(rtrees))
    torch.cuda.synchronize()
    assert r["status"].cpu().tolist() == [tsv.TSV_OK, tsv.TSV_ERR_BAD_TREE, tsv.TSV_ERR_UNSUPPORTED]
    assert r["count"].cpu().tolist()[1:] == [0, 0]


def test_expand_then_merge_builds_a_verifiable_tree(tsv):
    # Two speculators expand the same root with <2, 2> children per level;
    # the merged tree must satisfy the verification tree rules.
    rng = np.random.default_rng(11)
    V = 64
    trees = []
    for s in range(2):
        z0 = (rng.standard_normal((1, V)) * (1 + s)).astype(np.float32)
        lvl1 = tsv.tree_expand(d(z0), 2).cpu().numpy()[0]
        z1 = (rng.standard_normal((2, V)) * (1 + s)).astype(np.float32)
        lvl2 = tsv.tree_expand(d(z1), 2).cpu().numpy()
        par = np.array([-1, 0, 0, 1, 1, 2, 2], np.int32)
        tok = np.array([5, lvl1[0], lvl1[1], lvl2[0, 0], lvl2[0, 1], lvl2[1, 0], lvl2[1, 1]], np.int32)
        trees.append((par, tok))
    toffs = np.array([0, 7, 14], np.int32)
    r = tsv.tree_merge(d(np.concatenate([t[0] for t in trees])), d(np.concatenate([t[1] for t in trees])),
                       d(toffs), d(np.array([0, 2], np.int32)))
    torch.cuda.synchronize()
    cnt = int(r["count"][0])
    par = r["parent"].cpu().numpy()[:cnt]
    assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, cnt))
    ref = oracle.tree_merge([t[0] for t in trees], [t[1] for t in trees])
    assert np.array_equal(par, ref[0])
