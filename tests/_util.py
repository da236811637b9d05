"""Shared helpers of the GPU tests: move seeded inputs to the device, run the
library, run the oracle on the same inputs (or on sampled sub-problems), compare."""
import numpy as np
import torch

import oracle
import workloads as W

BF16_TOL = 2e-2  # max-abs, attention outputs in bf16
F32_TOL = 1e-4   # max-abs, attention outputs in fp32


def dev():
    return torch.device("cuda:0")


def d(x, dtype=None):
    t = x if isinstance(x, torch.Tensor) else torch.as_tensor(np.ascontiguousarray(x))
    return t.to(dev()) if dtype is None else t.to(dev(), dtype)


def tol(spec_dtype):
    return BF16_TOL if spec_dtype == "bf16" else F32_TOL


def run_attention(tsv, trees, att, flags=0, use_prepare=True, scale=0.0, k=None, v=None):
    parent, offs, plen = d(trees.parent), d(trees.node_offsets), d(trees.prefix_len)
    anc = None
    if use_prepare:
        anc, _, st = tsv.tree_prepare(parent, offs)
    out, st2 = tsv.tree_attention(d(att.q), d(att.k_cache) if k is None else k,
                                  d(att.v_cache) if v is None else v, trees.prefix_len,
                                  trees.node_offsets, plen, offs, parent=parent, anc=anc,
                                  scale=scale, flags=flags)
    torch.cuda.synchronize()
    return out, st2


def oracle_attention_sub(att, trees, reqs, kv_heads, scale=None):
    """Oracle on a sub-problem: requests `reqs`, KV heads `kv_heads` (and their query heads).

    The output of (request b, node i, query head h) depends only on request b's
    cache rows of KV head h // G, so slicing requests and KV heads gives exactly
    the same values as the full problem for the kept entries.
    """
    B, _, Hkv, D = att.k_cache.shape
    Hq = att.q.shape[1]
    G = Hq // Hkv
    qh = [g * G + r for g in kv_heads for r in range(G)]
    sizes = np.diff(trees.node_offsets)
    rows = np.concatenate([np.arange(trees.node_offsets[b], trees.node_offsets[b + 1]) for b in reqs])
    offs = np.concatenate([[0], np.cumsum(sizes[reqs])]).astype(np.int32)
    q = att.q[rows][:, qh].float().numpy()
    Lsub = int((trees.prefix_len[reqs] + sizes[reqs]).max())
    k = att.k_cache[reqs][:, :Lsub][:, :, kv_heads].float().numpy()
    v = att.v_cache[reqs][:, :Lsub][:, :, kv_heads].float().numpy()
    par = np.concatenate([trees.parent[trees.node_offsets[b]:trees.node_offsets[b + 1]] for b in reqs])
    out, st = oracle.tree_attention(q, k, v, trees.prefix_len[reqs], offs, par, scale=scale)
    assert (st == 0).all()
    return out, rows, qh


def compare_attention(out_gpu, att, trees, spec_dtype, reqs=None, kv_heads=None, scale=None):
    B, _, Hkv, _ = att.k_cache.shape
    reqs = list(range(B)) if reqs is None else list(reqs)
    kv_heads = list(range(Hkv)) if kv_heads is None else list(kv_heads)
    ref, rows, qh = oracle_attention_sub(att, trees, reqs, kv_heads, scale)
    got = out_gpu.float().cpu().numpy()[rows][:, qh]
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= tol(spec_dtype), "max-abs error %g > %g" % (err, tol(spec_dtype))
    return err


def compare_stochastic(gpu, ref, trees):
    """Bit-exact per request, except after a decision the oracle marks as a near tie."""
    path = gpu["path"].cpu().numpy()
    near = 0
    for b in range(len(trees.node_offsets) - 1):
        lo, hi = trees.node_offsets[b], trees.node_offsets[b + 1]
        if ref["n_near_tie"][b]:
            near += 1
            k = ref["tie_path_len"][b]
            assert np.array_equal(path[lo:lo + k], ref["path"][lo:lo + k])
            continue
        assert np.array_equal(path[lo:hi], ref["path"][lo:hi]), "request %d path" % b
        assert gpu["accept_len"][b].item() == ref["accept_len"][b], "request %d accept_len" % b
        assert gpu["bonus"][b].item() == ref["bonus"][b], "request %d bonus" % b
        assert gpu["n_tried"][b].item() == ref["n_tried"][b], "request %d n_tried" % b
        assert gpu["status"][b].item() == 0
    return near
