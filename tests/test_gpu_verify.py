"""GPU parity of greedy and stochastic tree verification against the CPU oracle.

Paths, accept lengths and bonus tokens must be bit-exact; for stochastic
verification a request may part from the oracle only after a decision the
oracle marks as a near tie (margin below 1e-6), which is counted.
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _util import compare_stochastic, d

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _greedy(tsv, trees, gi):
    r = tsv.tree_verify_greedy(d(gi.logits), d(gi.tokens), d(trees.parent), d(trees.node_offsets))
    torch.cuda.synchronize()
    return r


def _check_greedy(r, ref):
    assert np.array_equal(r["path"].cpu().numpy(), ref["path"])
    assert np.array_equal(r["accept_len"].cpu().numpy(), ref["accept_len"])
    assert np.array_equal(r["bonus"].cpu().numpy(), ref["bonus"])
    assert np.array_equal(r["status"].cpu().numpy(), ref["status"])


@pytest.mark.parametrize("name", ["tiny-f32-P128-n16", "llama7b-layer-P1024-n20", "gqa64x8-P32768-n128",
                                  "batch32-P2048-n16"])
def test_greedy_workloads(tsv, name):
    spec = W.SPECS[name]
    trees = W.make_trees(spec)
    gi = W.make_greedy_inputs(spec, trees)
    r = _greedy(tsv, trees, gi)
    ref = oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets)
    _check_greedy(r, ref)
    if spec.B > 1:
        assert ref["accept_len"].sum() > 0  # the recipe makes about half the children match


@pytest.mark.parametrize("seed", range(12))
def test_greedy_fuzz(tsv, seed):
    spec = W.fuzz_spec(seed)
    spec = W.spec_variant(spec, V=[5, 1000, 4097, 5001, 32003, 70000][seed % 6])
    trees = W.make_trees(spec)
    gi = W.make_greedy_inputs(spec, trees)
    # Plant ties: copy each row's maximum to a later and an earlier position.
    rng = np.random.default_rng(seed)
    for u in range(len(gi.tokens)):
        a = int(np.argmax(gi.logits[u]))
        for pos in rng.integers(0, spec.V, size=2):
            gi.logits[u, pos] = gi.logits[u, a]
    r = _greedy(tsv, trees, gi)
    _check_greedy(r, oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets))


@pytest.mark.parametrize("name", ["llama7b-layer-P1024-n20", "gqa64x8-P32768-n128", "batch32-P2048-n16"])
def test_greedy_workspace_reused_across_calls(tsv, name):
    """One workspace, zero-filled once, serves consecutive calls: each call
    must leave its completion counters (per request and, when a row is split
    into vocabulary slices, per row) at zero for the next one.  Outputs are
    refilled with -7 before every call, so a walk that does not run shows."""
    spec = W.SPECS[name]
    trees = W.make_trees(spec)
    gi = W.make_greedy_inputs(spec, trees)
    ref = oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets)
    x = [d(gi.logits), d(gi.tokens), d(trees.parent), d(trees.node_offsets)]
    N, B = len(gi.tokens), spec.B
    h = tsv.handle()
    ws = torch.zeros(tsv.tsv_tree_verify_greedy_workspace_size(h, B, N, spec.V), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        out = {k: torch.full((n,), -7, dtype=torch.int32, device="cuda")
               for k, n in (("path", N), ("accept_len", B), ("bonus", B), ("status", B))}
        r = tsv.tree_verify_greedy(*x, workspace=ws, out=out)
        torch.cuda.synchronize()
        _check_greedy(r, ref)


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "greedy_walk.json")))["cases"],
                         ids=lambda c: c["name"])
def test_greedy_golden(tsv, case):
    par = np.array(case["parent"], np.int32)
    r = tsv.tree_verify_greedy(d(np.array(case["logits"], np.float32)),
                               d(np.array(case["tokens"], np.int32)), d(par),
                               d(np.array([0, len(par)], np.int32)))
    torch.cuda.synchronize()
    assert r["path"].cpu().tolist() == case["path"]
    assert r["accept_len"].item() == case["accept_len"] and r["bonus"].item() == case["bonus"]


def test_greedy_bad_trees(tsv):
    par = np.array([-1, 0, 0, 2, 1, 5], np.int32)  # second request: node 1 points forward
    offs = np.array([0, 3, 6], np.int32)
    z = np.zeros((6, 10), np.float32)
    r = tsv.tree_verify_greedy(d(z), d(np.zeros(6, np.int32)), d(par), d(offs))
    torch.cuda.synchronize()
    assert r["status"].cpu().tolist() == [0, tsv.TSV_ERR_BAD_TREE]
    assert r["bonus"].cpu().tolist()[1] == -1 and r["path"].cpu().tolist()[3:] == [-1, -1, -1]


# ------------------------------------------------------------------ stochastic


def _stochastic(tsv, trees, si, temperature=1.0):
    r = tsv.tree_verify_stochastic(d(si.llm_logits), d(si.ssm_probs), d(si.tokens), d(trees.parent),
                                   d(trees.node_offsets), d(si.u_accept), d(si.u_sample),
                                   temperature=temperature)
    torch.cuda.synchronize()
    return r


@pytest.mark.parametrize("name", ["batch8-ragged-merge64-mss", "gqa64x8-P32768-n128", "batch32-P2048-n16"])
def test_stochastic_workloads(tsv, name):
    spec = W.SPECS[name]
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    r = _stochastic(tsv, trees, si)
    ref = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent,
                                   trees.node_offsets, si.u_accept, si.u_sample)
    near = compare_stochastic(r, ref, trees)
    assert near <= max(1, spec.B // 8)


@pytest.mark.parametrize("seed", range(12))
def test_stochastic_fuzz(tsv, seed):
    spec = W.spec_variant(W.fuzz_spec(200 + seed), V=[3, 17, 1000, 4099, 32000, 50001][seed % 6])
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    if seed % 3 == 0:  # make acceptances likely: proposals equal to the LLM rows
        z = si.llm_logits.astype(np.float64)
        si.ssm_probs[:] = W.proposal_rows(si.llm_logits)
    r = _stochastic(tsv, trees, si)
    ref = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent,
                                   trees.node_offsets, si.u_accept, si.u_sample)
    compare_stochastic(r, ref, trees)


@pytest.mark.parametrize("V,like_llm", [(160000, False), (160000, True), (137984, True), (138000, True)])
def test_stochastic_slices_staged_or_streamed(tsv, V, like_llm):
    """Vocabularies around the largest whose three slices per CTA fit in shared
    memory (137984 at eight CTAs per request): above it the slices are read
    from global memory, below it they are staged; both walks must agree with
    the oracle, through rejections (residual passes) and acceptances."""
    spec = W.spec_variant(W.fuzz_spec(310, max_nodes=24), V=V, B=2)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    if like_llm:  # proposals close to the LLM law at each parent: long accepted paths
        from test_gpu_verify_warped import _propose_like_llm
        _propose_like_llm(si, trees, seed=V)
    r = _stochastic(tsv, trees, si)
    ref = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent,
                                   trees.node_offsets, si.u_accept, si.u_sample)
    compare_stochastic(r, ref, trees)


@pytest.mark.parametrize("V,seed", [(32000, 32000), (160000, 160003)])  # seeds with no near tie
def test_stochastic_vanishing_residual_keeps_p(tsv, V, seed):
    """Proposal rows of all ones make every residual max(0, p - q) exactly zero,
    so p must survive each rejection unchanged (the staged kernel writes the
    residual over the spent proposals, never over p); a tiny accept uniform
    then accepts a later child, and the bonus is drawn from the kept p."""
    par = np.array([-1, 0, 0, 0, 0, 3, 3, 2], np.int32)
    n = len(par)
    trees = W.Trees(np.array([64], np.int32), np.array([0, n], np.int32), par, 64 + n)
    rng = np.random.default_rng(seed)
    llm = (rng.standard_normal((n, V)) * 2).astype(np.float32)
    ssm = np.ones((n, V), np.float32)
    tok = rng.integers(0, V, n).astype(np.int32)
    ua = np.full(n, 0.5, np.float32)
    ua[3] = 1e-12  # the third child of the root is accepted after two rejections;
    # its two children are rejected too, and the bonus comes from its kept p
    us = rng.random(n).astype(np.float32)
    si = W.StochasticInputs(llm, ssm, tok, ua, us)
    r = _stochastic(tsv, trees, si)
    ref = oracle.verify_stochastic(llm, ssm, tok, par, trees.node_offsets, ua, us)
    assert compare_stochastic(r, ref, trees) == 0
    assert ref["path"][1] == 3 and ref["accept_len"][0] == 1 and ref["n_tried"][0] == 5


def test_stochastic_temperature(tsv):
    spec = W.spec_variant(W.fuzz_spec(300), V=2000)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    r = _stochastic(tsv, trees, si, temperature=0.7)
    ref = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent,
                                   trees.node_offsets, si.u_accept, si.u_sample, temperature=0.7)
    compare_stochastic(r, ref, trees)


@pytest.mark.parametrize("V", [2000, 32000])
def test_stochastic_vanishing_temperature_is_greedy(tsv, V):
    """As T goes to zero the LLM distribution is one-hot at the argmax (every
    other probability underflows to exactly zero at T = 2^-60), so stochastic
    verification on the GPU must give greedy verification's result."""
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], V=V)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    rng = np.random.default_rng(V)
    tok = si.tokens.copy()
    for b in range(spec.B):
        off = int(trees.node_offsets[b])
        for i in range(1, int(trees.node_offsets[b + 1]) - off):
            if rng.random() < 0.5:
                tok[off + i] = int(np.argmax(si.llm_logits[off + int(trees.parent[off + i])]))
    top2 = np.sort(si.llm_logits, axis=1)[:, -2:]
    assert (top2[:, 1] > top2[:, 0]).all()
    r = _stochastic(tsv, trees, dataclasses.replace(si, tokens=tok), temperature=2.0 ** -60)
    g = oracle.verify_greedy(si.llm_logits, tok, trees.parent, trees.node_offsets)
    assert np.array_equal(r["path"].cpu().numpy(), g["path"])
    assert np.array_equal(r["accept_len"].cpu().numpy(), g["accept_len"])
    assert np.array_equal(r["bonus"].cpu().numpy(), g["bonus"])
    assert (r["status"].cpu().numpy() == 0).all() and g["accept_len"].sum() > 0


@pytest.mark.parametrize("B,n,V,tree", [(1, 1, 1, "random"), (1, 1, 7, "random"), (3, 5, 1, "random"),
                                        (2, 256, 64, "random"), (2, 256, 40, "chain"), (1, 256, 3, "star"),
                                        (128, 2, 100, "random"), (5, 9, 4, "random")])
def test_verify_edge_shapes(tsv, B, n, V, tree):
    """Root-only trees, V = 1 (every decision forced), the largest tree
    (256 nodes: deepest chain, widest star) and the largest batch (128)."""
    spec = W.spec_variant(W.SPECS["tiny-f32-P128-n16"], wid=7000 + n + V, B=B, nodes=n, V=V, tree=tree)
    trees = W.make_trees(spec)
    gi = W.make_greedy_inputs(spec, trees)
    si = W.make_stochastic_inputs(spec, trees)
    if tree == "chain":
        # Every node matches: both walks must run the whole 255-step chain.
        for b in range(B):
            off = int(trees.node_offsets[b])
            for i in range(1, n):
                u = off + int(trees.parent[off + i])
                gi.tokens[off + i] = int(np.argmax(gi.logits[u]))
                z = np.exp(si.llm_logits[u].astype(np.float64) - si.llm_logits[u].max())
                si.ssm_probs[off + i] = (z / z.sum()).astype(np.float32)  # q = p: accepted unless u ~ 1
    ref_g = oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets)
    _check_greedy(_greedy(tsv, trees, gi), ref_g)
    ref = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent, trees.node_offsets,
                                   si.u_accept, si.u_sample)
    compare_stochastic(_stochastic(tsv, trees, si), ref, trees)
    if tree == "chain":
        assert (ref_g["accept_len"] == n - 1).all() and (ref["accept_len"] == n - 1).all()


def _mss_golden():
    for case in json.load(open(os.path.join(GOLDEN, "mss_closed_forms.json")))["cases"]:
        for i, var in enumerate(case["variants"]):
            yield pytest.param(case, var, id="%s-%d" % (case["name"][:30], i))


@pytest.mark.parametrize("case,var", list(_mss_golden()))
def test_stochastic_golden(tsv, case, var):
    par = np.array(case["parent"], np.int32)
    logits = np.log(np.array(case["llm_probs"], np.float64)).astype(np.float32)
    r = tsv.tree_verify_stochastic(d(logits), d(np.array(case["ssm_probs"], np.float32)),
                                   d(np.array(case["tokens"], np.int32)), d(par),
                                   d(np.array([0, len(par)], np.int32)),
                                   d(np.array(var["u_acc"], np.float32)),
                                   d(np.array(var["u_smp"], np.float32)))
    torch.cuda.synchronize()
    assert r["path"].cpu().tolist() == var["path"]
    assert r["accept_len"].item() == var["accept_len"]
    assert r["bonus"].item() == var["bonus"]
    assert r["n_tried"].item() == var["n_tried"]


def test_stochastic_rejects_out_of_range_tokens(tsv):
    par = np.array([-1, 0, 0], np.int32)
    tok = np.array([0, 1, 9], np.int32)  # 9 >= V
    V = 4
    z = np.zeros((3, V), np.float32)
    r = tsv.tree_verify_stochastic(d(z), d(z + 0.25), d(tok), d(par), d(np.array([0, 3], np.int32)),
                                   d(np.zeros(3, np.float32)), d(np.zeros(3, np.float32)))
    torch.cuda.synchronize()
    assert r["status"].item() == tsv.TSV_ERR_INVALID_ARG and r["bonus"].item() == -1


def test_gpu_mss_preserves_llm_distribution(tsv):
    """The chi-square test of the oracle pins, run through the GPU kernels."""
    import test_oracle_verify_pins as pins

    def gpu_verify(llm, ssm, tok, par, offs, ua, us):
        B = len(offs) - 1
        out = {k: [] for k in ("path", "accept_len", "bonus")}
        for lo in range(0, B, 128):
            hi = min(B, lo + 128)
            r0, r1 = offs[lo], offs[hi]
            sub = offs[lo:hi + 1] - r0
            r = tsv.tree_verify_stochastic(d(llm[r0:r1]), d(ssm[r0:r1]), d(tok[r0:r1]), d(par[r0:r1]),
                                           d(sub), d(ua[r0:r1]), d(us[r0:r1]))
            for k in out:
                out[k].append(r[k].cpu().numpy())
        return {k: np.concatenate(v) for k, v in out.items()}

    obs, exp = pins._run_mss_markov(gpu_verify, trials=30_000, seed=12)
    assert pins._chi2_pvalue(obs, exp) > 1e-3


def test_greedy_equals_incremental_decoding_through_gpu(tsv):
    """Toy LM (D=64): one GPU tree-attention pass + GPU greedy verification
    reproduce token-by-token decoding (SpecInfer §6)."""
    import test_oracle_verify_pins as pins

    for seed in range(6):
        lm = pins.ToyLM(seed, V=16, d=64)
        rng = np.random.default_rng(500 + seed)
        P = 20
        prompt = rng.integers(lm.V, size=P + 1).tolist()
        cont = lm.incremental_decode(prompt, 8)
        keep = int(rng.integers(0, 7))
        par, tok = pins._tree_with_continuation(rng, cont, prompt[-1], lm.V, n_distract=12, keep=keep)
        n = len(par)
        h_pre, _, k_pre, v_pre = lm.qkv(prompt[:-1])
        h_tree, q_tree, k_tree, v_tree = lm.qkv(tok)
        kc = torch.from_numpy(np.concatenate([k_pre, k_tree])[None, :, None, :].copy())
        vc = torch.from_numpy(np.concatenate([v_pre, v_tree])[None, :, None, :].copy())
        offs = np.array([0, n], np.int32)
        o, st = tsv.tree_attention(d(q_tree[:, None, :].copy()), d(kc), d(vc), np.array([P], np.int32),
                                   offs, d(np.array([P], np.int32)), d(offs), parent=d(par))
        logits = (h_tree.astype(np.float64) + o[:, 0, :].double().cpu().numpy()) @ lm.Wo.astype(np.float64)
        r = tsv.tree_verify_greedy(d(logits.astype(np.float32)), d(tok), d(par), d(offs))
        torch.cuda.synchronize()
        a = r["accept_len"].item()
        emitted = [int(tok[c]) for c in r["path"].cpu().numpy()[1:a + 1]] + [r["bonus"].item()]
        assert emitted == cont[:a + 1]
        assert a >= keep
