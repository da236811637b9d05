"""The oracle against the hand-derived fixtures in tests/golden/ (derivations inside each file)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_attention_handcalc():
    g = _load("attention_handcalc.json")
    q = np.array(g["q"], np.float32)
    k = np.array(g["k_cache"], np.float32)
    v = np.array(g["v_cache"], np.float32)
    par = np.array(g["parent"], np.int32)
    out, st = oracle.tree_attention(q, k, v, np.array(g["prefix_len"], np.int32),
                                    np.array([0, len(par)], np.int32), par, scale=g["scale"])
    assert st[0] == 0
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("case", _load("greedy_walk.json")["cases"], ids=lambda c: c["name"])
def test_greedy_walk_cases(case):
    par = np.array(case["parent"], np.int32)
    r = oracle.verify_greedy(np.array(case["logits"], np.float32), np.array(case["tokens"], np.int32),
                             par, np.array([0, len(par)], np.int32))
    assert r["status"][0] == 0
    assert r["path"].tolist() == case["path"]
    assert int(r["accept_len"][0]) == case["accept_len"]
    assert int(r["bonus"][0]) == case["bonus"]


def _mss_cases():
    for case in _load("mss_closed_forms.json")["cases"]:
        for i, var in enumerate(case["variants"]):
            yield pytest.param(case, var, id=f"{case['name'][:40]}-{i}")


@pytest.mark.parametrize("case,var", list(_mss_cases()))
def test_mss_closed_forms(case, var):
    par = np.array(case["parent"], np.int32)
    logits = np.log(np.array(case["llm_probs"], np.float64)).astype(np.float32)
    r = oracle.verify_stochastic(logits, np.array(case["ssm_probs"], np.float32),
                                 np.array(case["tokens"], np.int32), par,
                                 np.array([0, len(par)], np.int32),
                                 np.array(var["u_acc"], np.float32), np.array(var["u_smp"], np.float32))
    assert r["status"][0] == 0
    assert r["path"].tolist() == var["path"]
    assert int(r["accept_len"][0]) == var["accept_len"]
    assert int(r["bonus"][0]) == var["bonus"]
    assert int(r["n_tried"][0]) == var["n_tried"]
    assert int(r["n_near_tie"][0]) == 0
