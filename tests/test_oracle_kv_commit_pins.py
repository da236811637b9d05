"""Pins of the oracle's KV commit (SpecInfer §4, Token Tree Verifier: the
accepted tokens join the verified sequence held in the one KV cache).

Each pin fixes the result by something other than the oracle's own loop: a
hand-worked case, the identity path, and the meaning of the committed cache —
ordinary attention over the committed sequence must equal tree attention of
the path's last node over the uncommitted cache.
"""
import numpy as np
import pytest

import oracle
import workloads as W


def test_hand_worked_case():
    # One request, prefix 2, five tree nodes, scalar rows holding their own
    # index.  Path 0 -> 2 -> 4: row 3 takes old row 2+2 = 4, row 4 takes old
    # row 2+4 = 6; rows 5 and 6 keep their values.
    k = np.arange(7, dtype=np.float32).reshape(1, 7, 1, 1)
    v = 10 * k
    path = np.array([0, 2, 4, -1, -1], dtype=np.int32)
    k2, v2, new_len, status = oracle.kv_commit(k, v, [2], [0, 5], path, [2])
    assert status.tolist() == [0]
    assert new_len.tolist() == [5]
    assert k2.reshape(-1).tolist() == [0, 1, 2, 4, 6, 5, 6]
    assert v2.reshape(-1).tolist() == [0, 10, 20, 40, 60, 50, 60]


def test_identity_path_leaves_the_cache_unchanged():
    rng = np.random.default_rng(1)
    k = rng.standard_normal((2, 40, 3, 8)).astype(np.float32)
    v = rng.standard_normal((2, 40, 3, 8)).astype(np.float32)
    offs = [0, 6, 10]
    path = np.array([0, 1, 2, 3, -1, -1, 0, 1, 2, 3], dtype=np.int32)
    k2, v2, new_len, status = oracle.kv_commit(k, v, [20, 30], offs, path, [3, 3])
    assert status.tolist() == [0, 0]
    assert new_len.tolist() == [24, 34]
    assert np.array_equal(k2, k) and np.array_equal(v2, v)


def _attention(q, k, v, scale):
    s = (k @ q) * scale
    w = np.exp(s - s.max())
    return (w[:, None] * v).sum(0) / w.sum()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_committed_sequence_attends_like_the_tree_node(seed):
    # After the commit, the path's last node looking at rows 0 .. new_len-1 as
    # an ordinary sequence sees exactly its tree key set: the prefix and its
    # ancestors, in order.
    rng = np.random.default_rng(seed)
    n, P, H, D = 24, 17, 2, 16
    parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], dtype=np.int32)
    leaf = int(rng.integers(1, n))
    chain = [leaf]
    while parent[chain[-1]] >= 0:
        chain.append(int(parent[chain[-1]]))
    path = np.full(n, -1, dtype=np.int32)
    path[:len(chain)] = chain[::-1]
    L = len(chain) - 1
    k = rng.standard_normal((1, P + n + 3, H, D)).astype(np.float32)
    v = rng.standard_normal((1, P + n + 3, H, D)).astype(np.float32)
    q = rng.standard_normal((n, H, D)).astype(np.float32)
    tree_out, tstat = oracle.tree_attention(q, k, v, [P], [0, n], parent)
    assert tstat[0] == 0
    k2, v2, new_len, status = oracle.kv_commit(k, v, [P], [0, n], path, [L])
    assert status[0] == 0 and new_len[0] == P + 1 + L
    scale = 1.0 / np.sqrt(D)
    for h in range(H):
        seq = _attention(q[leaf, h].astype(np.float64), k2[0, :new_len[0], h].astype(np.float64),
                         v2[0, :new_len[0], h].astype(np.float64), scale)
        np.testing.assert_allclose(seq, tree_out[leaf, h], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("path,L", [
    ([1, 2, 3, -1], 2),   # does not start at the root
    ([0, 2, 2, -1], 2),   # not rising
    ([0, 3, 1, -1], 2),   # falls back
    ([0, 1, 2, 3], 4),    # longer than the tree allows
    ([0, 1, 2, 3], -1),   # negative length
    ([0, 1, 4, -1], 2),   # past the request's nodes
])
def test_malformed_paths_are_rejected_and_leave_rows_alone(path, L):
    k = np.arange(12, dtype=np.float32).reshape(1, 12, 1, 1)
    k2, v2, new_len, status = oracle.kv_commit(k, k, [3], [0, 4], np.array(path, np.int32), [L])
    assert status.tolist() == [oracle.INVALID_ARG]
    assert new_len.tolist() == [-1]
    assert np.array_equal(k2, k)


def test_requests_are_independent():
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], B=3, Hq=2, Hkv=2, D=8, prefix=(5, 40))
    trees = W.make_trees(spec)
    rng = np.random.default_rng(5)
    Lcap = int(max(trees.prefix_len) + np.diff(trees.node_offsets).max())
    k = rng.standard_normal((3, Lcap, 2, 8)).astype(np.float32)
    paths, lens = [], []
    for b in range(3):
        off, n = int(trees.node_offsets[b]), int(trees.node_offsets[b + 1] - trees.node_offsets[b])
        node, chain = n - 1, []
        while node >= 0:
            chain.append(node)
            node = int(trees.parent[off + node])
        p = np.full(n, -1, np.int32)
        p[:len(chain)] = chain[::-1]
        paths.append(p)
        lens.append(len(chain) - 1)
    path = np.concatenate(paths)
    k_all, _, len_all, _ = oracle.kv_commit(k, k, trees.prefix_len, trees.node_offsets, path, lens)
    for b in range(3):
        off, end = int(trees.node_offsets[b]), int(trees.node_offsets[b + 1])
        kb, _, lb, _ = oracle.kv_commit(k[b:b + 1], k[b:b + 1], trees.prefix_len[b:b + 1], [0, end - off],
                                        path[off:end], lens[b:b + 1])
        assert np.array_equal(kb[0], k_all[b]) and lb[0] == len_all[b]
