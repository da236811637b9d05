"""Failure detection on the GPU without a fault: a device-side wait that never
completes must end in TSV_ERR_TIMEOUT after its time limit (about 1 s), the
kernel must return normally, and the context must stay usable for the next
call.  Nothing here traps, faults or hangs: the self-test kernel's waits are
the library's own bounded mbarrier waits on barriers that nothing arrives on.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import d

pytestmark = pytest.mark.gpu


def test_completed_wait_returns_ok(tsv):
    status, secs = tsv.selftest_bounded_wait(arrive=1)
    assert status == tsv.TSV_OK
    assert secs < 0.1


def test_stalled_wait_reports_timeout(tsv):
    status, secs = tsv.selftest_bounded_wait(arrive=0)
    assert status == tsv.TSV_ERR_TIMEOUT
    # The limit is 1 s of wall clock per wait; the second waiting warp leaves
    # as soon as it sees the first one's abort flag.
    assert 0.9 < secs < 3.0


def test_context_usable_after_timeout(tsv):
    assert tsv.selftest_bounded_wait(arrive=0)[0] == tsv.TSV_ERR_TIMEOUT
    spec = W.SPECS["tiny-f32-P128-n16"]
    trees = W.make_trees(spec)
    gi = W.make_greedy_inputs(spec, trees)
    r = tsv.tree_verify_greedy(d(gi.logits), d(gi.tokens), d(trees.parent), d(trees.node_offsets))
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets)
    assert np.array_equal(r["path"].cpu().numpy(), ref["path"])
    assert np.array_equal(r["bonus"].cpu().numpy(), ref["bonus"])
    assert tsv.selftest_bounded_wait(arrive=1)[0] == tsv.TSV_OK


def test_selftest_rejects_null_status(tsv):
    with pytest.raises(tsv.TSVError) as e:
        tsv.tsv_selftest_bounded_wait(tsv.handle(), 1, None)
    assert e.value.code == tsv.TSV_ERR_INVALID_ARG
