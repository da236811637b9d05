"""Pins of the oracle's token-tree construction (SpecInfer §3: expansion-based
and merge-based token trees).

Expansion is pinned by closed forms (k = 1 is the argmax, k = V a full
ranking, a hand-worked case with ties) and by numpy's own stable ranking;
merge by what the union must contain: every root-to-node token path of every
input tree exactly once, nothing else, parents before children."""
import numpy as np
import pytest

import oracle


def test_expand_hand_worked():
    z = np.array([[0.5, 2.0, 2.0, -1.0, 3.0], [1.0, 1.0, 1.0, 1.0, 1.0]], np.float32)
    assert oracle.tree_expand(z, 3).tolist() == [[4, 1, 2], [0, 1, 2]]


def test_expand_k1_is_argmax_and_kV_is_a_full_ranking():
    rng = np.random.default_rng(0)
    z = np.round(rng.standard_normal((20, 40)), 1).astype(np.float32)  # ties likely
    assert np.array_equal(oracle.tree_expand(z, 1)[:, 0], z.argmax(1))
    full = oracle.tree_expand(z, 40)
    for f in range(20):
        assert sorted(full[f].tolist()) == list(range(40))
        assert np.all(np.diff(z[f, full[f]]) <= 0)
        assert np.array_equal(full[f], np.lexsort((np.arange(40), -z[f].astype(np.float64))))


def _paths(par, tok):
    out = {0: ()}
    for i in range(1, len(par)):
        out[i] = out[int(par[i])] + (int(tok[i]),)
    return out


def _random_tree(rng, n, V):
    par = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], np.int32)
    tok = rng.integers(0, V, n).astype(np.int32)
    tok[0] = 7
    return par, tok


@pytest.mark.parametrize("seed", range(5))
def test_merge_contains_each_path_once(seed):
    rng = np.random.default_rng(seed)
    trees = [_random_tree(rng, int(rng.integers(1, 30)), 4) for _ in range(3)]
    par, tok, src = oracle.tree_merge([t[0] for t in trees], [t[1] for t in trees])
    assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, len(par)))
    union = list(_paths(par, tok).values())
    assert len(union) == len(set(union))
    want = set()
    for p, t in trees:
        want |= set(_paths(p, t).values())
    assert set(union) == want


def test_merging_a_tree_with_itself_or_a_subtree_changes_nothing():
    rng = np.random.default_rng(9)
    par, tok = _random_tree(rng, 25, 1000)  # tokens distinct enough: no repeated sibling paths
    p2, t2, _ = oracle.tree_merge([par, par[:10]], [tok, tok[:10]])
    assert np.array_equal(p2, par) and np.array_equal(t2, tok)
