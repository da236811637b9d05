"""The bench's step (what bench.py times) computes what the calls compute one
after another: with verification in overlap mode (the stochastic walk beside
attention at full size, greedy beside the walk) the attention output and
every verification output equal those of the serial step bit for bit, and
every status is OK.  The serial step's calls are themselves checked against
the oracle elsewhere."""
import pytest
import torch

import bench
import workloads as W

pytestmark = pytest.mark.gpu

GREEDY_OUT = ("path", "accept_len", "bonus", "status")  # what greedy verification writes
STOCHASTIC_OUT = ("path", "accept_len", "bonus", "n_tried", "status")


def _snapshot(w, st):
    out = {"attention": st["out"].clone(), "status": st["status"].clone()}
    for kind, keys in (("g", GREEDY_OUT if w.gi is not None else ()),
                       ("s", STOCHASTIC_OUT if w.si is not None else ())):
        out.update({kind + "." + k: st[kind][k].clone() for k in keys})
    return out


@pytest.mark.parametrize("name", list(W.SPECS))
def test_overlapped_step_matches_serial_step(tsv, name):
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    w = bench.DeviceWorkload(W.SPECS[name], tsv, dev, stream)
    c, st = w.copies[0], w.states[0]
    w.step(c, st, overlap=False)
    torch.cuda.synchronize()
    ref = _snapshot(w, st)
    assert (ref["status"].cpu() == 0).all()
    for kind in ("g", "s"):
        if kind + ".status" in ref:
            assert (ref[kind + ".status"].cpu() == 0).all(), kind
    # Poison the outputs, so that a step that skipped a write would differ.
    st["out"].fill_(float("nan"))
    for kind in ("g", "s"):
        for v in st[kind].values():
            v.fill_(-7)
    w.step(c, st, overlap=True)
    torch.cuda.synchronize()
    got = _snapshot(w, st)
    for k in ref:
        assert torch.equal(ref[k], got[k]), k
