"""GPU parity of tree preparation and tree attention against the CPU oracle.

Every test calls the library through its C ABI (via the ctypes binding) on
seeded inputs and compares element by element with the fp64 oracle: whole
outputs where the oracle finishes in seconds, sampled (request, KV head)
sub-problems at the full workload sizes.  Tolerances (max-abs): 2e-2 for bf16
outputs, 1e-4 for fp32.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import BF16_TOL, compare_attention, d, run_attention

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ prepare


@pytest.mark.parametrize("n,depth,B", [(1, 1, 1), (7, 3, 3), (33, 5, 2), (64, 8, 4), (129, 12, 2),
                                       (256, 20, 3), (256, 255, 1)])
def test_prepare_matches_oracle(tsv, n, depth, B):
    rng = np.random.default_rng(n * 7 + depth)
    parents = [W.random_tree(rng, n, depth) for _ in range(B)]
    par = np.concatenate(parents).astype(np.int32)
    offs = (np.arange(B + 1) * n).astype(np.int32)
    anc, dep, st = tsv.tree_prepare(d(par), d(offs))
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    a = anc.cpu().numpy().view(np.uint32)
    for b in range(B):
        ref, rdep, _ = oracle.tree_ancestors(parents[b])
        bits = np.unpackbits(a[b * n:(b + 1) * n].view(np.uint8), axis=1, bitorder="little").astype(bool)
        assert np.array_equal(bits[:, :n], ref)
        assert not bits[:, n:].any()
        assert np.array_equal(dep.cpu().numpy()[b * n:(b + 1) * n], rdep)


def test_prepare_flags_bad_trees(tsv):
    par = np.array([-1, 0, 1, -1, 0, 0, -1, 0, 1], dtype=np.int32)  # three requests of 3 nodes
    par[5] = 7  # request 1: its node 2 points forward
    offs = np.array([0, 3, 6, 9], dtype=np.int32)
    anc, dep, st = tsv.tree_prepare(d(par), d(offs))
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [0, tsv.TSV_ERR_BAD_TREE, 0]
    assert not anc.cpu().numpy()[3:6].any()


# ------------------------------------------------------------------ the five workloads


def test_tiny_f32_full(tsv):
    spec = W.SPECS["tiny-f32-P128-n16"]
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att)
    assert (st.cpu() == 0).all()
    compare_attention(out, att, trees, "f32")


@pytest.mark.parametrize("flags", [0, 1])
def test_llama7b_layer_full(tsv, flags):
    spec = W.SPECS["llama7b-layer-P1024-n20"]
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att, flags=flags)
    compare_attention(out, att, trees, "bf16")


def test_batch8_ragged_sampled(tsv):
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], pad_value=float("nan"))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att)
    assert np.isfinite(out.float().cpu().numpy()).all()
    compare_attention(out, att, trees, "bf16", reqs=[0, 3, 7], kv_heads=[0, 13, 31])


def test_gqa_32k_sampled(tsv):
    spec = W.SPECS["gqa64x8-P32768-n128"]
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att)
    compare_attention(out, att, trees, "bf16", reqs=[0], kv_heads=[0, 5])


def test_batch32_sampled(tsv):
    spec = W.SPECS["batch32-P2048-n16"]
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att)
    compare_attention(out, att, trees, "bf16", reqs=[0, 17, 31], kv_heads=[0, 31])


# Batches with more (request, KV head) units than SMs and one key chunk per
# unit run as a persistent launch: one CTA per SM walks a sequence of units,
# its producer streaming the next unit's K/V while the previous one finishes.
# Every output is checked, with NaN in the cache rows no request may read.
PERSISTENT = {
    "b16-h32-ragged": dict(B=16, Hq=32, Hkv=32, D=128, nodes=16, prefix=(0, 600), max_depth=6),
    "b128-h4-d64-short": dict(B=128, Hq=4, Hkv=4, D=64, nodes=5, prefix=(0, 300), max_depth=3),
    "b64-gqa4-n16": dict(B=64, Hq=16, Hkv=4, D=128, nodes=16, prefix=(100, 1500), max_depth=5),
}


@pytest.mark.parametrize("name", list(PERSISTENT))
@pytest.mark.parametrize("use_prepare", [False, True])
def test_persistent_keys_kernel_full(tsv, name, use_prepare):
    kw = PERSISTENT[name]
    spec = W.Spec(name, 3500 + list(PERSISTENT).index(name), "bf16", kw["B"], kw["Hq"], kw["Hkv"], kw["D"],
                  10, kw["prefix"], kw["nodes"], "random", max_depth=kw["max_depth"], pad_value=float("nan"))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att, use_prepare=use_prepare)
    assert (st.cpu() == 0).all()
    compare_attention(out, att, trees, "bf16")


# ------------------------------------------------------------------ fuzz and edges


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_tensor_core(tsv, seed):
    spec = W.spec_variant(W.fuzz_spec(seed, "bf16"), pad_value=float("nan"))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att, use_prepare=bool(seed % 2))
    assert (st.cpu() == 0).all()
    compare_attention(out, att, trees, "bf16")


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fuzz_cuda_cores(tsv, seed, dtype):
    spec = W.spec_variant(W.fuzz_spec(100 + seed, dtype), pad_value=float("nan"))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att, flags=tsv.TSV_ATTN_SIMT)
    compare_attention(out, att, trees, dtype)


EDGE = {
    "root-only-no-prefix": dict(B=1, nodes=1, prefix=0, tree="chain"),
    "tree-no-prefix": dict(B=2, nodes=50, prefix=0, tree="random", max_depth=7),
    "max-nodes-gqa8": dict(B=1, Hq=16, Hkv=2, nodes=256, prefix=300, tree="random", max_depth=10),
    "deep-chain": dict(B=1, nodes=256, prefix=1000, tree="chain"),
    "star": dict(B=1, nodes=200, prefix=77, tree="star"),
    "keys-multiple-of-64": dict(B=3, nodes=64, prefix=(128, 128), tree="random"),
    "keys-64k-plus-1": dict(B=2, nodes=65, prefix=(128, 128), tree="random"),
    "keys-64k-minus-1": dict(B=2, nodes=63, prefix=(128, 128), tree="random"),
    "head-dim-64-gqa": dict(B=2, Hq=8, Hkv=1, D=64, nodes=40, prefix=(500, 900), tree="random"),
    "many-requests": dict(B=128, Hq=2, Hkv=1, nodes=3, prefix=(0, 70), tree="random"),
    "long-prefix-one-head": dict(B=1, Hq=1, Hkv=1, nodes=9, prefix=20000, tree="random"),
    # rows-on-lanes kernels: one 128-row tile per KV head (one-tile kernel), and
    # three tiles (a full pair and a pair with one tile)
    "one-row-tile-mha": dict(B=2, Hq=4, Hkv=4, nodes=100, prefix=(300, 900), tree="random", max_depth=9),
    "three-row-tiles": dict(B=2, Hq=4, Hkv=2, nodes=150, prefix=(200, 700), tree="random", max_depth=9),
    # tile pairs with prefixes of whole 128-key blocks: a block ends exactly
    # where the tree keys begin, and the next one starts with them
    "row-tiles-prefix-of-whole-blocks": dict(B=2, Hq=16, Hkv=2, nodes=100, prefix=1024, tree="random",
                                             max_depth=9),
    # head dim 64 on the one-tile rows kernel (120 rows per KV head) and on a
    # persistent keys-on-lanes launch (48 x 4 units of 40 rows, more than SMs)
    "one-row-tile-head-dim-64": dict(B=2, Hq=8, Hkv=2, D=64, nodes=30, prefix=(300, 900), tree="random",
                                     max_depth=7),
    "persistent-keys-head-dim-64": dict(B=48, Hq=8, Hkv=4, D=64, nodes=20, prefix=(100, 600), tree="random"),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_shapes(tsv, name):
    kw = dict(Hq=4, Hkv=2, D=128, V=10, max_depth=5)
    kw.update(EDGE[name])
    spec = W.Spec(name, 3000 + list(EDGE).index(name), "bf16", kw["B"], kw["Hq"], kw["Hkv"], kw["D"],
                  kw["V"], kw["prefix"], kw["nodes"], kw["tree"], max_depth=kw["max_depth"],
                  pad_value=float("nan"))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, st = run_attention(tsv, trees, att)
    assert (st.cpu() == 0).all()
    reqs = None if spec.B <= 8 else [0, 1, spec.B // 2, spec.B - 1]
    compare_attention(out, att, trees, "bf16", reqs=reqs)


def test_strided_cache_layout(tsv):
    """A cache stored [B, Hkv, Lcap, D] and passed as a strided view."""
    spec = W.spec_variant(W.fuzz_spec(7, "bf16"), Hq=4, Hkv=2, D=128)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    k = d(att.k_cache).permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    v = d(att.v_cache).permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    assert not k.is_contiguous()
    out, _ = run_attention(tsv, trees, att, k=k, v=v)
    compare_attention(out, att, trees, "bf16")


def test_explicit_scale(tsv):
    spec = W.fuzz_spec(3, "bf16")
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, _ = run_attention(tsv, trees, att, scale=0.05)
    compare_attention(out, att, trees, "bf16", scale=0.05)


def test_non_ancestor_rows_do_not_change_gpu_output(tsv):
    spec = W.spec_variant(W.SPECS["llama7b-layer-P1024-n20"], Hq=4, Hkv=4)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    out, _ = run_attention(tsv, trees, att)
    anc, _, _ = oracle.tree_ancestors(trees.parent)
    P = int(trees.prefix_len[0])
    node = 7  # in the first chain: sees 0, 1, 2 .. 7
    others = np.nonzero(~anc[node])[0]
    k2, v2 = att.k_cache.clone(), att.v_cache.clone()
    k2[0, P + others] = 9.0
    v2[0, P + others] = -7.0
    out2, _ = run_attention(tsv, trees, W.AttentionInputs(att.q, k2, v2))
    assert torch.equal(out2[node], out[node])
    assert not torch.equal(out2[8], out[8])  # node 8 (second chain) sees neither 2..7 nor 14..


def test_tensor_core_and_cuda_core_paths_agree(tsv):
    spec = W.SPECS["batch8-ragged-merge64-mss"]
    spec = W.spec_variant(spec, B=3, Hq=8, Hkv=2, prefix=(1000, 3000))
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    a, _ = run_attention(tsv, trees, att)
    b, _ = run_attention(tsv, trees, att, flags=tsv.TSV_ATTN_SIMT)
    assert (a.float() - b.float()).abs().max().item() < BF16_TOL


def test_bad_tree_reported_when_preparing_inside(tsv):
    spec = W.fuzz_spec(5, "bf16")
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    bad = trees.parent.copy()
    bad[trees.node_offsets[0]] = 3  # the first node of request 0 points forward
    trees_bad = W.Trees(trees.prefix_len, trees.node_offsets, bad, trees.Lcap)
    _, st = run_attention(tsv, trees_bad, att, use_prepare=False)
    assert st[0].item() == tsv.TSV_ERR_BAD_TREE


def test_host_side_argument_checks(tsv):
    spec = W.fuzz_spec(2, "bf16")
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    q, k, v = d(att.q), d(att.k_cache), d(att.v_cache)
    h = tsv.handle()
    B = spec.B
    N, Hq, D = q.shape
    Hkv = k.shape[2]
    out = torch.empty_like(q)
    st = torch.zeros(B, dtype=torch.int32, device=q.device)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device=q.device)
    plen, offs, par = d(trees.prefix_len), d(trees.node_offsets), d(trees.parent)
    s = k.stride()

    def call(**kw):
        a = dict(dtype_code=tsv.TSV_BF16, q=q, k_cache=k, v_cache=v, kv_stride_b=s[0], kv_stride_l=s[1],
                 kv_stride_h=s[2], out=out, prefix_len_host=trees.prefix_len,
                 node_offsets_host=trees.node_offsets, prefix_len=plen, node_offsets=offs, parent=par,
                 anc=None, B=B, Hq=Hq, Hkv=Hkv, D=D, scale=0.0, workspace=ws,
                 workspace_bytes=ws.numel(), status=st)
        a.update(kw)
        with pytest.raises(tsv.TSVError) as e:
            tsv.tsv_tree_attention(h, **a)
        return e.value.code

    assert call(D=96) == tsv.TSV_ERR_UNSUPPORTED
    assert call(Hkv=3) == tsv.TSV_ERR_INVALID_ARG
    assert call(B=0) == tsv.TSV_ERR_INVALID_ARG
    assert call(q=None) == tsv.TSV_ERR_INVALID_ARG
    big_ws_need = tsv.tsv_tree_attention_workspace_size(h, tsv.TSV_BF16, B, trees.prefix_len, trees.node_offsets, Hq, Hkv, D, False)
    if big_ws_need > 16:  # the keys-on-lanes kernel needs no workspace at all
        assert call(workspace_bytes=16) == tsv.TSV_ERR_INVALID_ARG
    assert call(kv_stride_l=s[1] + 1) == tsv.TSV_ERR_INVALID_ARG
    assert call(k_cache=k.data_ptr() + 2) == tsv.TSV_ERR_INVALID_ARG
    assert call(scale=-1.0) == tsv.TSV_ERR_INVALID_ARG
    big = np.array([0, 300], dtype=np.int32)
    assert call(B=1, node_offsets_host=big, prefix_len_host=trees.prefix_len[:1]) == \
        tsv.TSV_ERR_UNSUPPORTED
    assert call(dtype_code=7) == tsv.TSV_ERR_INVALID_ARG
