"""Pins of the oracle's tree attention against things other than itself.

Each test ties the fp64 oracle to a fact the pages or plain mathematics fix:
  * a chain tree is ordinary causal attention with the prefix in front
    (SpecInfer §4 "Tree Attention": a node's output is sequence attention over
    the sequence the node stands for) — checked against torch's
    scaled_dot_product_attention on CPU in fp64 with an explicit mask;
  * each node's output equals attention over its gathered root-to-node key list
    (brute force with the library routine, one node at a time);
  * one node is plain decode attention; a star tree sees prefix + root + itself;
  * with identical keys every visible key weighs the same, so the output is the
    mean of the visible values (closed form that pins the key set exactly);
  * rows of non-ancestor tree nodes never change a node's output, bit for bit
    (SpecInfer §4, Tree-Based Parallel Decoding: shared-prefix tokens get
    identical outputs under causal masking);
  * a topological relabelling of the nodes permutes the outputs alike;
  * grouped-query heads equal the same problem with KV heads repeated;
  * the dense-mask formulation (beta) agrees with the gathered one (alpha).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W


def _problem(seed, B=2, Hq=4, Hkv=2, D=16, n=9, P=(3, 11), depth=4, tree="random"):
    spec = W.Spec(f"pin{seed}", 500 + seed, "f32", B, Hq, Hkv, D, 7, P, n, tree, max_depth=depth)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    return spec, trees, att.q.numpy(), att.k_cache.numpy(), att.v_cache.numpy()


def _sdpa(q, k, v, mask=None):
    """torch SDPA in fp64; q [Lq, D], k/v [Lk, D], mask bool [Lq, Lk] (True = attend)."""
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, None]
    kt = torch.from_numpy(np.asarray(k, np.float64))[None, None]
    vt = torch.from_numpy(np.asarray(v, np.float64))[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m)[0, 0].numpy()


def test_chain_tree_is_causal_attention():
    spec, trees, q, k, v = _problem(1, tree="chain", n=12, P=17)
    out, st = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    assert (st == 0).all()
    G = spec.Hq // spec.Hkv
    for b in range(spec.B):
        off, P = trees.node_offsets[b], trees.prefix_len[b]
        n = trees.node_offsets[b + 1] - off
        mask = np.arange(P + n)[None, :] <= (P + np.arange(n))[:, None]
        for h in range(spec.Hq):
            ref = _sdpa(q[off:off + n, h], k[b, :P + n, h // G], v[b, :P + n, h // G], mask)
            np.testing.assert_allclose(out[off:off + n, h], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_each_node_equals_attention_over_its_gathered_sequence(seed):
    spec, trees, q, k, v = _problem(seed, n=13, depth=5)
    out, st = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    assert (st == 0).all()
    G = spec.Hq // spec.Hkv
    for b in range(spec.B):
        off, P = int(trees.node_offsets[b]), int(trees.prefix_len[b])
        n = int(trees.node_offsets[b + 1]) - off
        par = trees.parent[off:off + n]
        for i in range(n):
            path = []
            a = i
            while a != -1:
                path.append(a)
                a = par[a]
            rows = list(range(P)) + [P + a for a in reversed(path)]
            for h in range(spec.Hq):
                ref = _sdpa(q[off + i, h][None], k[b, rows, h // G], v[b, rows, h // G])[0]
                np.testing.assert_allclose(out[off + i, h], ref, rtol=1e-12, atol=1e-12)


def test_single_node_is_decode_attention():
    spec, trees, q, k, v = _problem(7, B=1, n=1, P=40)
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    for h in range(spec.Hq):
        ref = _sdpa(q[0, h][None], k[0, :41, h // 2], v[0, :41, h // 2])[0]
        np.testing.assert_allclose(out[0, h], ref, rtol=1e-12, atol=1e-12)


def test_star_tree_sees_prefix_root_and_self():
    spec, trees, q, k, v = _problem(8, B=1, n=10, P=5, tree="star")
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    for i in range(10):
        rows = list(range(5)) + ([5] if i == 0 else [5, 5 + i])
        for h in range(spec.Hq):
            ref = _sdpa(q[i, h][None], k[0, rows, h // 2], v[0, rows, h // 2])[0]
            np.testing.assert_allclose(out[i, h], ref, rtol=1e-12, atol=1e-12)


def test_identical_keys_give_mean_of_visible_values():
    """Closed form: equal scores -> uniform weights over exactly J(i)."""
    spec, trees, q, k, v = _problem(9, n=15, depth=6)
    k[:] = k[:, :1]  # every row of every request holds the same key
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    G = spec.Hq // spec.Hkv
    for b in range(spec.B):
        off, P = int(trees.node_offsets[b]), int(trees.prefix_len[b])
        n = int(trees.node_offsets[b + 1]) - off
        anc, depth, _ = oracle.tree_ancestors(trees.parent[off:off + n])
        for i in range(n):
            for h in range(spec.Hq):
                g = h // G
                vv = v.astype(np.float64)
                tot = vv[b, :P, g].sum(0) + vv[b, P + np.nonzero(anc[i])[0], g].sum(0)
                np.testing.assert_allclose(out[off + i, h], tot / (P + depth[i] + 1), rtol=1e-12,
                                           atol=1e-12)


def test_non_ancestor_rows_do_not_change_output():
    spec, trees, q, k, v = _problem(10, B=1, n=16, depth=4)
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    anc, _, _ = oracle.tree_ancestors(trees.parent)
    P = int(trees.prefix_len[0])
    rng = np.random.default_rng(0)
    for i in range(16):
        k2, v2 = k.copy(), v.copy()
        others = np.nonzero(~anc[i])[0]
        k2[0, P + others] = rng.standard_normal(k2[0, P + others].shape) * 50
        v2[0, P + others] = rng.standard_normal(v2[0, P + others].shape) * 50
        out2, _ = oracle.tree_attention(q, k2, v2, trees.prefix_len, trees.node_offsets,
                                        trees.parent)
        assert np.array_equal(out2[i], out[i])
        if len(others):
            changed = [j for j in range(16) if anc[j][others].any()]
            assert all(not np.array_equal(out2[j], out[j]) for j in changed)


def test_topological_relabelling_permutes_outputs():
    spec, trees, q, k, v = _problem(11, B=1, n=14, depth=5)
    par = trees.parent
    n, P = 14, int(trees.prefix_len[0])
    # A different topological order: order by depth, ties broken by reversed index.
    depth = W.tree_depths(par)
    order = sorted(range(n), key=lambda i: (depth[i], -i))  # new position -> old node
    new_of_old = np.empty(n, dtype=np.int64)
    new_of_old[order] = np.arange(n)
    par2 = np.array([-1 if par[o] < 0 else new_of_old[par[o]] for o in order], dtype=np.int32)
    assert all(par2[i] < i for i in range(n))
    q2 = q[order]
    k2, v2 = k.copy(), v.copy()
    k2[0, P:P + n] = k[0, P + np.array(order)]
    v2[0, P:P + n] = v[0, P + np.array(order)]
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, par)
    out2, _ = oracle.tree_attention(q2, k2, v2, trees.prefix_len, trees.node_offsets, par2)
    np.testing.assert_allclose(out2, out[order], rtol=1e-12, atol=1e-12)


def test_gqa_equals_repeated_kv_heads():
    spec, trees, q, k, v = _problem(12, Hq=8, Hkv=2)
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    k_rep = np.repeat(k, 4, axis=2)
    v_rep = np.repeat(v, 4, axis=2)
    out2, _ = oracle.tree_attention(q, k_rep, v_rep, trees.prefix_len, trees.node_offsets,
                                    trees.parent)
    np.testing.assert_allclose(out, out2, rtol=0, atol=0)


def test_scale_argument():
    spec, trees, q, k, v = _problem(13)
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent,
                                   scale=0.3)
    out2, _ = oracle.tree_attention(q * np.float32(0.3 * math.sqrt(16)), k, v, trees.prefix_len,
                                    trees.node_offsets, trees.parent)
    np.testing.assert_allclose(out, out2, rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("seed", range(3))
def test_dense_mask_formulation_agrees(seed):
    spec, trees, q, k, v = _problem(20 + seed, B=3, n=21, depth=7)
    out, _ = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
    out_b = oracle.tree_attention_dense_mask(q, k, v, trees.prefix_len, trees.node_offsets,
                                             trees.parent)
    np.testing.assert_allclose(out, out_b, rtol=1e-11, atol=1e-12)


def test_forest_is_allowed_in_attention():
    """Attention accepts several roots: each node still sees prefix + its own path."""
    par = np.array([-1, 0, -1, 2, 1], dtype=np.int32)
    spec, trees, q, k, v = _problem(30, B=1, n=5, P=4)
    out, st = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, par)
    assert st[0] == 0
    rows = [0, 1, 2, 3, 4 + 2, 4 + 3]  # node 3's path: 2 -> 3
    ref = _sdpa(q[3, 0][None], k[0, rows, 0], v[0, rows, 0])[0]
    np.testing.assert_allclose(out[3, 0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bad", [[-1, 1], [-1, 0, 5], [0], [-1, -2], [-1, 0, 2]])
def test_bad_tree_sets_status(bad):
    bad = np.array(bad, dtype=np.int32)
    n = len(bad)
    spec, trees, q, k, v = _problem(31, B=1, n=n, P=3)
    out, st = oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, bad)
    assert st[0] == oracle.BAD_TREE and not out.any()


def test_ancestor_sets_invariants():
    for seed in range(5):
        par = W.random_tree(np.random.default_rng(seed), 60, 7)
        anc, depth, st = oracle.tree_ancestors(par)
        assert st == 0
        assert (anc.sum(1) == depth + 1).all()
        assert anc[np.arange(60), np.arange(60)].all()
        for i in range(1, 60):
            p = par[i]
            assert (anc[i] >= anc[p]).all() and anc[i].sum() == anc[p].sum() + 1
        assert (np.tril(np.ones((60, 60), bool)) | ~anc).all()  # ancestors have lower index
