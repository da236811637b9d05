"""The sequence-based baseline (every root-to-leaf path as its own request,
with its own copy of the prefix) computes the same attention as the tree:
SpecInfer §4 defines a node's tree-attention output as attention over the
token sequence it stands for."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import BF16_TOL, F32_TOL, d

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,kw", [
    ("batch8-ragged-merge64-mss", dict(B=2, Hq=4, Hkv=4, prefix=(100, 700))),
    ("gqa64x8-P32768-n128", dict(Hq=16, Hkv=2, prefix=900, nodes=48)),
    ("tiny-f32-P128-n16", {}),
])
def test_sequences_reproduce_tree_outputs(tsv, name, kw):
    spec = W.spec_variant(W.SPECS[name], **kw)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    seq = W.sequence_decomposition(trees, att)
    tol = BF16_TOL if spec.dtype == "bf16" else F32_TOL
    tree_out, st = tsv.tree_attention(d(att.q), d(att.k_cache), d(att.v_cache), trees.prefix_len,
                                      trees.node_offsets, d(trees.prefix_len), d(trees.node_offsets),
                                      parent=d(trees.parent))
    s = seq.trees
    seq_out, st2 = tsv.tree_attention(d(seq.inputs.q), d(seq.inputs.k_cache), d(seq.inputs.v_cache), s.prefix_len,
                                      s.node_offsets, d(s.prefix_len), d(s.node_offsets), parent=d(s.parent))
    torch.cuda.synchronize()
    assert st.cpu().eq(0).all() and st2.cpu().eq(0).all()
    diff = (seq_out.float().cpu() - tree_out.float().cpu()[torch.as_tensor(seq.tree_row)]).abs().max().item()
    assert diff <= tol, diff
    # And the sequences against the oracle (first sequence, all heads).
    n0 = int(s.node_offsets[1])
    ref, _ = oracle.tree_attention(seq.inputs.q[:n0].float().numpy(), seq.inputs.k_cache[:1].float().numpy(),
                                   seq.inputs.v_cache[:1].float().numpy(), s.prefix_len[:1], [0, n0], s.parent[:n0])
    assert np.abs(seq_out[:n0].float().cpu().numpy() - ref).max() <= tol
