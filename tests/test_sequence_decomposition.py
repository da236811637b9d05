"""The sequence-based baseline's decomposition, on the CPU: one width-1 request
per root-to-leaf path, each with its own copy of the prefix rows.  Every
position of every sequence must see exactly the keys its tree node sees (the
prefix, then the node's ancestors and itself, in the same order), so the
oracle's tree attention and its attention over the decomposition agree row
for row: the pages' equivalence of tree-based and sequence-based decoding,
checked without a GPU."""
import numpy as np
import pytest

import oracle
import workloads as W


@pytest.mark.parametrize("tree,nodes,max_depth", [("random", 17, 5), ("trunk_chains", 20, 8), ("star", 9, 2),
                                                  ("chain", 6, 6)])
def test_sequences_match_tree_rows(tree, nodes, max_depth):
    spec = W.Spec("seqdec", 4100 + nodes, "f32", 2, 4, 2, 16, 10, (5, 23), nodes, tree, max_depth=max_depth)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    seq = W.sequence_decomposition(trees, att)
    # One sequence per leaf, each the root-to-leaf chain of its request.
    leaves = 0
    for b in range(spec.B):
        par = trees.parent[trees.node_offsets[b]:trees.node_offsets[b + 1]]
        leaves += int(np.sum(~np.isin(np.arange(len(par)), par[par >= 0])))
    assert len(seq.trees.node_offsets) - 1 == leaves
    sizes = np.diff(seq.trees.node_offsets)
    for s in range(leaves):
        lo = seq.trees.node_offsets[s]
        assert list(seq.trees.parent[lo:lo + sizes[s]]) == list(range(-1, sizes[s] - 1))  # a chain
    out_t, st_t = oracle.tree_attention(att.q.numpy(), att.k_cache.numpy(), att.v_cache.numpy(),
                                        trees.prefix_len, trees.node_offsets, trees.parent)
    out_s, st_s = oracle.tree_attention(seq.inputs.q.numpy(), seq.inputs.k_cache.numpy(), seq.inputs.v_cache.numpy(),
                                        seq.trees.prefix_len, seq.trees.node_offsets, seq.trees.parent)
    assert (st_t == 0).all() and (st_s == 0).all()
    np.testing.assert_allclose(out_s, out_t[seq.tree_row], rtol=0, atol=1e-12)
