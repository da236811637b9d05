"""GPU parity of the KV commit of the accepted path against the CPU oracle.

The commit is a copy, so the whole K and V caches must match the oracle bit
for bit (compared as raw 16- or 32-bit words), as must new_len and status.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import BF16_TOL, d

pytestmark = pytest.mark.gpu


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).numpy()


def _deepest_paths(trees, rng=None):
    """Per request, the root-to-node chain of a random (or the last) node."""
    offs = trees.node_offsets
    path = np.full(int(offs[-1]), -1, np.int32)
    lens = []
    for b in range(len(offs) - 1):
        off, n = int(offs[b]), int(offs[b + 1] - offs[b])
        node = int(rng.integers(0, n)) if rng is not None else n - 1
        chain = []
        while node >= 0:
            chain.append(node)
            node = int(trees.parent[off + node])
        path[off:off + len(chain)] = chain[::-1]
        lens.append(len(chain) - 1)
    return path, np.array(lens, np.int32)


def _run_and_compare(tsv, k, v, trees, path, lens):
    ref_k, ref_v, ref_len, ref_st = oracle.kv_commit(_bits(k), _bits(v), trees.prefix_len,
                                                     trees.node_offsets, path, lens)
    kg, vg = d(k), d(v)
    r = tsv.kv_commit(kg, vg, d(trees.prefix_len), d(trees.node_offsets), d(path), d(lens))
    torch.cuda.synchronize()
    assert np.array_equal(r["status"].cpu().numpy(), ref_st)
    assert np.array_equal(r["new_len"].cpu().numpy(), ref_len)
    assert np.array_equal(_bits(kg), ref_k)
    assert np.array_equal(_bits(vg), ref_v)
    return kg, vg, r


@pytest.mark.parametrize("name", ["llama7b-layer-P1024-n20", "batch8-ragged-merge64-mss", "batch32-P2048-n16",
                                  "tiny-f32-P128-n16"])
def test_workload_paths(tsv, name):
    spec = W.SPECS[name]
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    path, lens = _deepest_paths(trees, np.random.default_rng(7))
    _run_and_compare(tsv, att.k_cache, att.v_cache, trees, path, lens)


def test_paths_from_gpu_greedy_verification(tsv):
    spec = W.spec_variant(W.SPECS["batch32-P2048-n16"], V=3000, prefix=512)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    gi = W.make_greedy_inputs(spec, trees)
    g = tsv.tree_verify_greedy(d(gi.logits), d(gi.tokens), d(trees.parent), d(trees.node_offsets))
    ref = oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets)
    torch.cuda.synchronize()
    assert np.array_equal(g["path"].cpu().numpy(), ref["path"])
    assert (ref["accept_len"] > 0).any()
    _run_and_compare(tsv, att.k_cache, att.v_cache, trees, ref["path"], ref["accept_len"])


@pytest.mark.parametrize("seed", range(6))
def test_fuzz(tsv, seed):
    spec = W.fuzz_spec(seed, dtype="bf16" if seed % 2 == 0 else "f32", max_nodes=200)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    path, lens = _deepest_paths(trees, np.random.default_rng(seed))
    _run_and_compare(tsv, att.k_cache, att.v_cache, trees, path, lens)


def test_strided_cache(tsv):
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], B=3, Hq=4, Hkv=4, D=64, prefix=(20, 300))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    B, Lcap, H, D = att.k_cache.shape
    big_k = torch.zeros(B, Lcap + 5, H, D + 8, dtype=att.k_cache.dtype)
    big_v = torch.zeros_like(big_k)
    big_k[:, :Lcap, :, :D] = att.k_cache
    big_v[:, :Lcap, :, :D] = att.v_cache
    path, lens = _deepest_paths(trees)
    ref_k, ref_v, ref_len, ref_st = oracle.kv_commit(_bits(big_k), _bits(big_v), trees.prefix_len,
                                                     trees.node_offsets, path, lens)
    kg, vg = d(big_k), d(big_v)
    r = tsv.kv_commit(kg[:, :, :, :D], vg[:, :, :, :D], d(trees.prefix_len), d(trees.node_offsets), d(path),
                      d(lens))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kg), ref_k) and np.array_equal(_bits(vg), ref_v)
    assert np.array_equal(r["new_len"].cpu().numpy(), ref_len)


def test_edges(tsv):
    # Request 0: empty path (L = 0).  Request 1: a 256-node chain committed
    # whole (every copy is the identity).  Request 2: nodes i -> i-2, path
    # 0, 2, 4, ..., 254 (127 moved rows).  Request 3: a single node.
    n = [5, 256, 256, 1]
    parents = [[-1, 0, 0, 1, 1], [-1] + list(range(255)), [-1, 0] + list(range(0, 254)), [-1]]
    offs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    parent = np.concatenate([np.array(p, np.int32) for p in parents])
    prefix = np.array([3, 100, 7, 50], np.int32)
    trees = W.Trees(parent=parent, node_offsets=offs, prefix_len=prefix,
                    Lcap=int((prefix + np.array(n)).max()))
    rng = np.random.default_rng(3)
    shape = (4, trees.Lcap, 2, 64)
    k = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    path = np.full(int(offs[-1]), -1, np.int32)
    path[offs[0]] = 0
    path[offs[1]:offs[2]] = np.arange(256)
    path[offs[2]:offs[2] + 128] = np.arange(0, 256, 2)
    path[offs[3]] = 0
    lens = np.array([0, 255, 127, 0], np.int32)
    _run_and_compare(tsv, k, v, trees, path, lens)


@pytest.mark.parametrize("bad", ["not_root", "not_rising", "too_long", "outside"])
def test_malformed_paths_are_reported_and_rows_untouched(tsv, bad):
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], B=2, Hq=2, Hkv=2, D=64, prefix=(30, 60))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    path, lens = _deepest_paths(trees)
    off1 = int(trees.node_offsets[1])
    n1 = int(trees.node_offsets[2]) - off1
    if bad == "not_root":
        path[off1] = 1
    elif bad == "not_rising":
        lens[1] = max(lens[1], 2)
        path[off1 + 1:off1 + 3] = [2, 1]
    elif bad == "too_long":
        lens[1] = n1
    else:
        lens[1] = max(lens[1], 1)
        path[off1 + lens[1]] = n1
    kg, vg, r = _run_and_compare(tsv, att.k_cache, att.v_cache, trees, path, lens)
    assert r["status"].cpu().tolist() == [tsv.TSV_OK, tsv.TSV_ERR_INVALID_ARG]


def test_host_argument_checks(tsv):
    k = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(2, dtype=torch.int32, device="cuda")
    h = tsv.handle(0)
    with pytest.raises(tsv.TSVError):  # row of one head not a multiple of 16 bytes
        tsv.tsv_kv_commit(h, 1, k, k, 8 * 64, 64, 7, 1, 1, 7, z, z, z, z, z, z)
    with pytest.raises(tsv.TSVError):  # misaligned base pointer
        kb = k.view(-1)[1:]
        tsv.tsv_kv_commit(h, 1, kb, kb, 8 * 64, 64, 64, 1, 1, 64, z, z, z, z, z, z)
    with pytest.raises(tsv.TSVError):  # batch out of range
        tsv.tsv_kv_commit(h, 1, k, k, 8 * 64, 64, 64, 0, 1, 64, z, z, z, z, z, z)


def test_committed_cache_attends_like_the_tree_node(tsv):
    # At the full llama7b-layer shape: after the commit, a one-node "tree" at
    # the last committed row over prefix new_len-1 must give the output the
    # path's last node had in the tree pass (same cache keys, ordinary order).
    spec = W.SPECS["llama7b-layer-P1024-n20"]
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    path, lens = _deepest_paths(trees)  # the last node's chain: 0 1 14 15 .. 19
    leaf = int(path[lens[0]])
    tree_out, _ = tsv.tree_attention(d(att.q), d(att.k_cache), d(att.v_cache), trees.prefix_len,
                                     trees.node_offsets, d(trees.prefix_len), d(trees.node_offsets),
                                     parent=d(trees.parent))
    kg, vg, r = _run_and_compare(tsv, att.k_cache, att.v_cache, trees, path, lens)
    new_len = int(r["new_len"].cpu()[0])
    one = np.array([0, 1], np.int32)
    pl = np.array([new_len - 1], np.int32)
    out1, _ = tsv.tree_attention(d(att.q[leaf:leaf + 1]), kg, vg, pl, one, d(pl), d(one),
                                 parent=d(np.array([-1], np.int32)))
    torch.cuda.synchronize()
    diff = (out1[0].float() - tree_out[leaf].float()).abs().max().item()
    assert diff <= BF16_TOL, diff
