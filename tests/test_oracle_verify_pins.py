"""Pins of the oracle's verification against what the pages fix.

  * Greedy token-tree verification emits exactly the tokens of incremental
    decoding (SpecInfer §6: "the exact same token sequences"), shown with a toy
    seeded one-layer LM: decode token by token with textbook causal attention,
    then score a tree holding that continuation plus distractors in ONE tree
    attention pass and verify it.
  * Multi-step speculative sampling preserves the LLM's output distribution
    (SpecInfer §1 Correctness, §4 Token Verification): chi-square over many
    seeds on a Markov toy LLM with several toy SSMs; the same test must reject a
    copy of the oracle compiled with the residual update removed.
  * Deepest fully-matching node = the greedy walk's stop node, by brute force,
    when sibling tokens are distinct.
"""
import math
import os
import subprocess

import numpy as np
import pytest
from scipy import stats

import oracle
import workloads as W

# ------------------------------------------------------------------ greedy == incremental


class ToyLM:
    """One attention layer over token embeddings, seeded; logits = (h + attn(h)) Wo."""

    def __init__(self, seed, V=16, d=8):
        r = np.random.default_rng(seed)
        self.V, self.d = V, d
        self.E = r.standard_normal((V, d)).astype(np.float32)
        self.Wq = (r.standard_normal((d, d)) * 1.5 / math.sqrt(d)).astype(np.float32)
        self.Wk = (r.standard_normal((d, d)) * 1.5 / math.sqrt(d)).astype(np.float32)
        self.Wv = (r.standard_normal((d, d)) / math.sqrt(d)).astype(np.float32)
        self.Wo = (r.standard_normal((d, V)) * 2.0).astype(np.float32)

    def qkv(self, toks):
        h = self.E[np.asarray(toks)]
        return h, (h @ self.Wq).astype(np.float32), (h @ self.Wk).astype(np.float32), \
            (h @ self.Wv).astype(np.float32)

    def logits_from(self, h, o):
        return ((h.astype(np.float64) + o) @ self.Wo.astype(np.float64)).astype(np.float32)

    def incremental_decode(self, prompt, steps):
        """Textbook greedy decoding: causal softmax attention over every earlier position."""
        seq = list(prompt)
        out = []
        for _ in range(steps):
            h, q, k, v = self.qkv(seq)
            s = (q[-1].astype(np.float64) @ k.T.astype(np.float64)) / math.sqrt(self.d)
            w = np.exp(s - s.max())
            o = (w @ v.astype(np.float64)) / w.sum()
            logit = self.logits_from(h[-1], o)
            nxt = int(np.argmax(logit))
            out.append(nxt)
            seq.append(nxt)
        return out


def _tree_with_continuation(rng, cont, root_tok, V, n_distract, keep):
    """Root + the first ``keep`` tokens of ``cont`` as one path, plus random distractors."""
    parent, tok, on_path = [-1], [root_tok], [True]
    for t in cont[:keep]:
        parent.append(len(parent) - 1)
        tok.append(t)
        on_path.append(True)
    for _ in range(n_distract):
        j = int(rng.integers(len(parent)))
        t = int(rng.integers(V))
        if on_path[j] and j < keep:  # never duplicate the stored continuation's next token
            while t == cont[j]:
                t = int(rng.integers(V))
        parent.append(j)
        tok.append(t)
        on_path.append(False)
    # Shuffle into another topological order so the true path is not always lowest-index.
    n = len(parent)
    depth = W.tree_depths(np.array(parent))
    order = sorted(range(n), key=lambda i: (depth[i], rng.random()))
    new = {o: i for i, o in enumerate(order)}
    par2 = [-1 if parent[o] < 0 else new[parent[o]] for o in order]
    return np.array(par2, np.int32), np.array([tok[o] for o in order], np.int32)


@pytest.mark.parametrize("seed", range(12))
def test_greedy_tree_verification_equals_incremental_decoding(seed):
    lm = ToyLM(seed)
    rng = np.random.default_rng(100 + seed)
    P = 6
    prompt = rng.integers(lm.V, size=P + 1).tolist()  # prefix tokens + the root token
    steps = 6
    cont = lm.incremental_decode(prompt, steps + 1)
    keep = int(rng.integers(0, steps + 1))
    par, tok = _tree_with_continuation(rng, cont, prompt[-1], lm.V, n_distract=10, keep=keep)
    n = len(par)
    # One tree-attention pass over the whole tree.
    h_pre, _, k_pre, v_pre = lm.qkv(prompt[:-1])
    h_tree, q_tree, k_tree, v_tree = lm.qkv(tok)
    kc = np.concatenate([k_pre, k_tree])[None, :, None, :]
    vc = np.concatenate([v_pre, v_tree])[None, :, None, :]
    o, st = oracle.tree_attention(q_tree[:, None, :], kc, vc, np.array([P], np.int32),
                                  np.array([0, n], np.int32), par)
    assert st[0] == 0
    logits = lm.logits_from(h_tree, o[:, 0, :])
    r = oracle.verify_greedy(logits, tok, par, np.array([0, n], np.int32))
    a = int(r["accept_len"][0])
    emitted = [int(tok[c]) for c in r["path"][1:a + 1]] + [int(r["bonus"][0])]
    assert emitted == cont[:a + 1]
    assert a >= keep  # the whole stored continuation is accepted


def test_deepest_matching_node_is_the_walk_end():
    rng = np.random.default_rng(7)
    for trial in range(30):
        n, V = 25, 6
        par = W.random_tree(rng, n, 6)
        logits = rng.standard_normal((n, V)).astype(np.float32)
        arg = logits.argmax(1)
        tok = np.zeros(n, np.int32)
        for u in range(n):  # distinct sibling tokens, half of them the parent's argmax
            kids = [c for c in range(n) if par[c] == u]
            perm = rng.permutation(V)
            if kids and rng.random() < 0.7:
                perm = np.concatenate([[arg[u]], perm[perm != arg[u]]])
            for j, c in enumerate(kids[:V]):
                tok[c] = perm[j]
        kids_ok = all(len([c for c in range(n) if par[c] == u]) <= V for u in range(n))
        if not kids_ok:
            continue
        good = np.zeros(n, bool)
        good[0] = True
        for c in range(1, n):
            good[c] = good[par[c]] and tok[c] == arg[par[c]]
        deepest = max(np.nonzero(good)[0], key=lambda i: W.tree_depths(par)[i])
        r = oracle.verify_greedy(logits, tok, par, np.array([0, n], np.int32))
        a = int(r["accept_len"][0])
        assert r["path"][a] == deepest
        assert r["bonus"][0] == arg[deepest]


@pytest.mark.parametrize("bad", [[0, 0], [-1, -1], [-1, 1], [-1, 0, 3]])
def test_verification_rejects_bad_trees(bad):
    par = np.array(bad, np.int32)
    n = len(par)
    z = np.zeros((n, 4), np.float32)
    r = oracle.verify_greedy(z, np.zeros(n, np.int32), par, np.array([0, n], np.int32))
    assert r["status"][0] == oracle.BAD_TREE and r["bonus"][0] == -1 and (r["path"] == -1).all()
    s = oracle.verify_stochastic(z, z + 0.25, np.zeros(n, np.int32), par, np.array([0, n], np.int32),
                                 np.zeros(n, np.float32), np.zeros(n, np.float32))
    assert s["status"][0] == oracle.BAD_TREE and s["bonus"][0] == -1


def test_requests_are_independent():
    """A batch gives the same per-request results as separate calls."""
    spec = W.spec_variant(W.SPECS["batch8-ragged-merge64-mss"], V=50, B=4, prefix=8)
    trees = W.make_trees(spec)
    si = W.make_stochastic_inputs(spec, trees)
    full = oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent,
                                    trees.node_offsets, si.u_accept, si.u_sample)
    for b in range(spec.B):
        lo, hi = trees.node_offsets[b], trees.node_offsets[b + 1]
        one = oracle.verify_stochastic(si.llm_logits[lo:hi], si.ssm_probs[lo:hi], si.tokens[lo:hi],
                                       trees.parent[lo:hi], np.array([0, hi - lo], np.int32),
                                       si.u_accept[lo:hi], si.u_sample[lo:hi])
        assert one["path"].tolist() == full["path"][lo:hi].tolist()
        assert one["bonus"][0] == full["bonus"][b] and one["n_tried"][0] == full["n_tried"][b]


# ------------------------------------------------------------------ MSS distribution


def _softmax(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def _run_mss_markov(lib_verify, trials, seed, V=4, n=8, max_depth=3, n_ssm=3, emit=3, law=None):
    """Iterate tree verification on a Markov toy LLM until every trial emitted `emit` tokens.
    `law(A)` gives the next-token law the emitted tokens must follow (default:
    softmax of the LLM's logits)."""
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((V, V)).astype(np.float32)  # LLM logits given the previous token
    Q = np.stack([_softmax(rng.standard_normal((V, V)) * 1.5) for _ in range(n_ssm)]).astype(np.float32)
    t0 = 0
    seqs = [[] for _ in range(trials)]
    ctx = np.full(trials, t0, np.int64)
    active = np.arange(trials)
    while len(active):
        B = len(active)
        # Random trees: parent[i] uniform over earlier nodes of depth < max_depth (vectorised).
        par = np.full((B, n), -1, np.int32)
        dep = np.zeros((B, n), np.int32)
        for i in range(1, n):
            key = rng.random((B, i))
            key[dep[:, :i] >= max_depth] = -1.0
            j = key.argmax(1)
            par[:, i] = j
            dep[:, i] = dep[np.arange(B), j] + 1
        tok = np.zeros((B, n), np.int64)
        tok[:, 0] = ctx[active]
        ssm_rows = np.zeros((B, n, V), np.float32)
        ssm_rows[:, 0] = 1.0 / V
        for i in range(1, n):
            s = rng.integers(n_ssm, size=B)
            q = Q[s, tok[np.arange(B), par[:, i]]]  # [B, V]
            cdf = np.cumsum(q.astype(np.float64), axis=1)
            x = (rng.random(B)[:, None] * cdf[:, -1:] >= cdf).sum(1)
            tok[:, i] = np.minimum(x, V - 1)
            ssm_rows[:, i] = q
        llm = A[tok]  # [B, n, V]
        u = rng.random((B, 2 * n)).astype(np.float32)
        r = lib_verify(llm.reshape(B * n, V), ssm_rows.reshape(B * n, V),
                       tok.reshape(-1).astype(np.int32), par.reshape(-1),
                       (np.arange(B + 1) * n).astype(np.int32),
                       u[:, :n].reshape(-1), u[:, n:].reshape(-1))
        path = r["path"].reshape(B, n)
        still = []
        for bi, t in enumerate(active):
            a = int(r["accept_len"][bi])
            em = [int(tok[bi, c]) for c in path[bi, 1:a + 1]] + [int(r["bonus"][bi])]
            seqs[t].extend(em)
            ctx[t] = seqs[t][-1]
            if len(seqs[t]) < emit:
                still.append(t)
        active = np.array(still, dtype=np.int64)
    P1 = _softmax(A) if law is None else law(A)  # next-token law of the LLM
    expected = np.zeros([V] * emit)
    for idx in np.ndindex(*([V] * emit)):
        pr, prev = 1.0, t0
        for y in idx:
            pr *= P1[prev, y]
            prev = y
        expected[idx] = pr
    counts = np.zeros([V] * emit)
    for s in seqs:
        counts[tuple(s[:emit])] += 1
    return counts.ravel(), expected.ravel() * trials


def _chi2_pvalue(obs, exp):
    small = exp < 5
    o = np.append(obs[~small], obs[small].sum())
    e = np.append(exp[~small], exp[small].sum())
    if e[-1] == 0:
        o, e = o[:-1], e[:-1]
    chi2 = ((o - e) ** 2 / e).sum()
    return stats.chi2.sf(chi2, len(e) - 1)


def test_mss_preserves_llm_distribution():
    obs, exp = _run_mss_markov(oracle.verify_stochastic, trials=100_000, seed=11)
    assert _chi2_pvalue(obs, exp) > 1e-3


def _mutant_verify(tmp_path, original, replacement):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(original) == 1
    mutant = src.replace(original, replacement)
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutant)
    subprocess.run(["gcc", "-O2", "-shared", "-fPIC", str(c), "-o", str(so), "-lm"], check=True)
    lib = oracle._bind(str(so))

    def verify(*args):
        saved = oracle._LIB
        oracle._LIB = lib
        try:
            return oracle.verify_stochastic(*args)
        finally:
            oracle._LIB = saved

    return verify


def test_chi_square_rejects_mss_without_residual_update(tmp_path):
    """Negative control: planted in a copy of the oracle, on the CPU."""
    verify = _mutant_verify(tmp_path, "p[t] = (r > 0.0 ? r : 0.0) / Z;", "(void)r;")
    obs, exp = _run_mss_markov(verify, trials=100_000, seed=11)
    assert _chi2_pvalue(obs, exp) < 1e-3


def test_chi_square_rejects_wrong_acceptance_ratio(tmp_path):
    """Negative control: accept with p/q replaced by q/p."""
    verify = _mutant_verify(tmp_path, "if (ua * qx < p[x]) {", "if (ua * p[x] < qx) {")
    obs, exp = _run_mss_markov(verify, trials=100_000, seed=11)
    assert _chi2_pvalue(obs, exp) < 1e-3
