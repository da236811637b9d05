"""The bench's algorithmic bytes and FLOPs (the numerators of its roofline
fractions) against closed forms written out from each workload's shape.

Bytes: every (request, KV head) reads its K and V rows 0 .. P_b + n_b - 1
once, Q is read once and O written once; greedy reads every logits row once.
FLOPs: 4 D per query row per key the row sees (its prefix, then the node and
its ancestors).
"""
import numpy as np
import pytest

import bench
import workloads as W


def _depths(parent):
    """Strict ancestors of every node, by walking the parent links."""
    out = []
    for i in range(len(parent)):
        d, u = 0, int(parent[i])
        while u >= 0:
            d, u = d + 1, int(parent[u])
        out.append(d)
    return np.array(out)


@pytest.mark.parametrize("name,expected", [
    # 2 (K, V) x (P + n) x Hkv x D x 2 B + 2 (Q, O) x N x Hq x D x 2 B
    ("llama7b-layer-P1024-n20", 2 * 1044 * 32 * 128 * 2 + 2 * 20 * 32 * 128 * 2),          # 17,432,576
    ("gqa64x8-P32768-n128", 2 * 32896 * 8 * 128 * 2 + 2 * 128 * 64 * 128 * 2),             # 138,936,320
    ("batch32-P2048-n16", 32 * 2 * 2064 * 32 * 128 * 2 + 2 * 512 * 32 * 128 * 2),          # 1,090,519,040
    ("tiny-f32-P128-n16", 2 * 144 * 1 * 64 * 4 + 2 * 16 * 1 * 64 * 4),                     # 81,920 (fp32)
])
def test_attention_bytes_closed_forms(name, expected):
    spec = W.SPECS[name]
    assert bench.attention_bytes(spec, W.make_trees(spec)) == expected


def test_attention_bytes_ragged_prefixes():
    spec = W.SPECS["batch8-ragged-merge64-mss"]
    trees = W.make_trees(spec)
    kv = sum(2 * (int(p) + 64) * 32 * 128 * 2 for p in trees.prefix_len)
    assert bench.attention_bytes(spec, trees) == kv + 2 * 8 * 64 * 32 * 128 * 2


def test_attention_flops_default_workload():
    # Trunk 0 -> 1, then three 6-node chains under node 1: the nodes see
    # 1, 2 and 3..8 (three times) of the tree's keys, 102 in all.
    spec = W.SPECS["llama7b-layer-P1024-n20"]
    assert bench.attention_flops(spec, W.make_trees(spec)) == 4 * 128 * 32 * (20 * 1024 + 102)  # 337,215,488


@pytest.mark.parametrize("name", ["tiny-f32-P128-n16", "batch8-ragged-merge64-mss", "gqa64x8-P32768-n128"])
def test_attention_flops_random_trees(name):
    spec = W.SPECS[name]
    trees = W.make_trees(spec)
    seen = 0
    for b in range(spec.B):
        lo, hi = int(trees.node_offsets[b]), int(trees.node_offsets[b + 1])
        d = _depths(trees.parent[lo:hi])
        seen += (hi - lo) * int(trees.prefix_len[b]) + int((d + 1).sum())
    assert bench.attention_flops(spec, trees) == 4 * spec.D * spec.Hq * seen


def test_greedy_bytes():
    spec = W.SPECS["llama7b-layer-P1024-n20"]
    assert bench.verify_bytes(spec, W.make_trees(spec)) == 20 * 32000 * 4  # 2.56 MB


def test_stochastic_bytes_count_the_visited_and_rejected_rows():
    # Batch 32 x 16 nodes, V 32000, greedy + stochastic: every greedy row, then
    # the LLM rows the walk visited and the proposal rows of rejected children.
    spec = W.SPECS["batch32-P2048-n16"]
    trees = W.make_trees(spec)
    assert bench.verify_bytes(spec, trees, 40, 100) == 512 * 32000 * 4 + (40 + 100) * 32000 * 4
    assert bench.verify_bytes(spec, trees) == 2 * 512 * 32000 * 4  # no visit count: every LLM row
