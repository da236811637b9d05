"""The no-allocation greedy verification entry point.

tsv_tree_verify_greedy_noalloc serves callers that cannot hand the library a
device workspace (an engine whose allocator owns all device memory, a loop that
must never enter the allocator): its scratch is a fixed array inside the
library.  Called through the C ABI, it must give exactly what
tsv_tree_verify_greedy gives with a caller-provided workspace, on two calls in
a row (the shared scratch keeps the previous call's contents).  This file is
collected last so that a failure here stops a -x run only after every other test.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(spec):
    trees = W.make_trees(spec)
    gi = W.make_greedy_inputs(spec, trees)
    d = lambda x: torch.as_tensor(np.ascontiguousarray(x)).cuda()
    return trees, dict(logits=d(gi.logits), tokens=d(gi.tokens), parent=d(trees.parent),
                       offs=d(trees.node_offsets))


def _outputs(N, B):
    z = lambda n: torch.full((n,), -7, dtype=torch.int32, device="cuda")
    return dict(path=z(N), accept_len=z(B), bonus=z(B), status=z(B))


def _with_workspace(tsv, h, x, B, N, V):
    o = _outputs(N, B)
    ws = torch.zeros(tsv.tsv_tree_verify_greedy_workspace_size(h, B, N, V), dtype=torch.uint8,
                     device="cuda")
    tsv.tsv_tree_verify_greedy(h, x["logits"], V, x["tokens"], x["parent"], x["offs"], B, N, o["path"],
                               o["accept_len"], o["bonus"], ws, ws.numel(), o["status"])
    return o


def _no_alloc(tsv, h, x, B, N, V):
    o = _outputs(N, B)
    tsv.tsv_tree_verify_greedy_noalloc(h, x["logits"], V, x["tokens"], x["parent"], x["offs"], B, N,
                                       o["path"], o["accept_len"], o["bonus"], o["status"])
    return o


def test_no_alloc_matches_workspace_entry_on_consecutive_calls(tsv):
    h = tsv.handle()
    specs = [W.SPECS["batch32-P2048-n16"], W.SPECS["llama7b-layer-P1024-n20"]]
    for spec in specs:  # two different batches, each verified twice in a row
        trees, x = _inputs(spec)
        B, N, V = spec.B, int(trees.node_offsets[-1]), spec.V
        ref = _with_workspace(tsv, h, x, B, N, V)
        first = _no_alloc(tsv, h, x, B, N, V)
        second = _no_alloc(tsv, h, x, B, N, V)
        torch.cuda.synchronize()
        assert (ref["status"].cpu() == 0).all()
        for k in ref:  # integer outputs: bit-exact
            assert torch.equal(first[k], ref[k]), k
            assert torch.equal(second[k], ref[k]), k


def test_no_alloc_clears_counters_a_previous_call_left_nonzero(tsv):
    """Calls of different shapes in a row share the scratch: a call with one
    request has its row argmax words right after its 256 bytes of counters,
    where a later call with 128 requests has counters.  Every call leaves its
    words and counters at zero and the entry point clears them before each
    launch; a nonzero counter would keep that request's walk from running."""
    h = tsv.handle()
    small = W.SPECS["llama7b-layer-P1024-n20"]  # B = 1: counters in bytes 0..255, partials from 256
    trees, x = _inputs(small)
    first = _no_alloc(tsv, h, x, small.B, int(trees.node_offsets[-1]), small.V)
    big = W.spec_variant(W.SPECS["batch32-P2048-n16"], name="noalloc-b128", B=128, prefix=64, V=4000,
                         stochastic=False)  # B = 128: counters in bytes 0..511
    btrees, bx = _inputs(big)
    B, N, V = big.B, int(btrees.node_offsets[-1]), big.V
    ref = _with_workspace(tsv, h, bx, B, N, V)
    second = _no_alloc(tsv, h, bx, B, N, V)
    torch.cuda.synchronize()
    assert (first["status"].cpu() == 0).all() and (ref["status"].cpu() == 0).all()
    for k in ref:
        assert torch.equal(second[k], ref[k]), k


def test_no_alloc_rejects_what_the_scratch_cannot_hold(tsv):
    h = tsv.handle()
    o = _outputs(1, 1)
    # A valid batch size whose node count needs more row argmax words than the
    # fixed scratch holds: rejected on the host, before anything is launched.
    need = tsv.tsv_tree_verify_greedy_workspace_size(h, 1, 200000, 32000)
    assert need > 1 << 20
    with pytest.raises(tsv.TSVError) as e:
        tsv.tsv_tree_verify_greedy_noalloc(h, None, 32000, None, None, None, 1, 200000, None, o["accept_len"],
                                           o["bonus"], o["status"])
    assert e.value.code == tsv.TSV_ERR_SCRATCH_LIMIT
    with pytest.raises(tsv.TSVError) as e:  # B beyond the library's maximum
        tsv.tsv_tree_verify_greedy_noalloc(h, None, 10, None, None, None, 1000, 0, None, o["accept_len"],
                                           o["bonus"], o["status"])
    assert e.value.code == tsv.TSV_ERR_INVALID_ARG
