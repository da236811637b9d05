"""CPU oracle for token-tree verification — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the GPU library
and never imports it; the library never imports this.

Two layers:
  * ``liboracle.so`` (``oracle.c``): fp64 plain loops for tree attention
    (formulation alpha: gather each node's root-to-node key list and run
    ordinary attention), greedy verification and multi-step speculative
    sampling.  Wrapped by :func:`tree_attention`, :func:`verify_greedy`,
    :func:`verify_stochastic`, :func:`tree_ancestors`.
  * :func:`kv_commit` (numpy, a copy): moves the accepted path's cache rows
    behind the prefix, in path order.
  * :func:`tree_attention_dense_mask` (formulation beta, numpy fp64): builds the
    full topology-aware mask as a boolean matrix from the transitive closure of
    the parent relation and runs masked attention over every cache row.  It is
    kept as an independent cross-check of formulation alpha.

Sources: "SpecInfer: Accelerating Generative Large Language Model Serving with
Tree-based Speculative Inference and Verification", §2 (tree verification),
§4 Token Tree Verifier (Tree Attention, Tree-Based Parallel Decoding with
topology-aware causal masking, Token Verification / multi-step speculative
sampling), §6 (greedy output equals incremental decoding); "Accelerating LLM
Inference with Staged Speculative Decoding", §3 Implementation (attention split
between the cached prefix and the in-batch tree).
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from .build import build_oracle

OK, INVALID_ARG, BAD_TREE, NONFINITE = 0, 1, 2, 6
NEAR_TIE_EPS = 1e-6

_LIB = None
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def _bind(path):
    """Load a compiled oracle and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_tree_ancestors.argtypes = [_i32p, ctypes.c_int32, _u8p, _i32p]
    lib.oracle_tree_attention.argtypes = [
        _f32p, _f32p, _f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        _i32p, _i32p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_double, _f64p, _i32p]
    lib.oracle_verify_greedy.argtypes = [
        _f32p, ctypes.c_int64, _i32p, _i32p, _i32p, ctypes.c_int32,
        _i32p, _i32p, _i32p, _i32p]
    lib.oracle_verify_stochastic.argtypes = [
        _f32p, _f32p, ctypes.c_int64, _i32p, _i32p, _i32p, _f32p, _f32p,
        ctypes.c_int32, ctypes.c_double, ctypes.c_int32, ctypes.c_double,
        _i32p, _i32p, _i32p, _i32p, _i32p, _i32p, _i32p]
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    for f in (lib.oracle_tree_ancestors, lib.oracle_tree_attention,
              lib.oracle_verify_greedy, lib.oracle_verify_stochastic, lib.oracle_num_threads):
        f.restype = ctypes.c_int
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = _bind(build_oracle())
    return _LIB


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's later calls from this thread (no effect on results)."""
    _lib().oracle_set_num_threads(int(n))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a, ptype):
    return a.ctypes.data_as(ptype)


def tree_ancestors(parent):
    """Dense ancestor-or-self matrix (bool [n, n]) and depth (int32 [n]) of one tree.

    Returns (anc, depth, status); status is BAD_TREE when parent[] breaks the
    topological convention (parent[i] == -1 or 0 <= parent[i] < i).
    """
    parent = _c(parent, np.int32)
    n = parent.shape[0]
    anc = np.zeros((n, n), dtype=np.uint8)
    depth = np.zeros(n, dtype=np.int32)
    st = _lib().oracle_tree_ancestors(_p(parent, _i32p), n, _p(anc, _u8p), _p(depth, _i32p))
    return anc.astype(bool), depth, st


def tree_attention(q, k_cache, v_cache, prefix_len, node_offsets, parent, scale=None):
    """Tree attention in fp64 (formulation alpha).

    q: float32 [N, Hq, D]; k_cache, v_cache: float32 [B, Lcap, Hkv, D];
    prefix_len int32 [B]; node_offsets int32 [B+1]; parent int32 [N] (local
    indices per request).  scale defaults to 1/sqrt(D).
    Returns (out float64 [N, Hq, D], status int32 [B]).
    """
    q = _c(q, np.float32)
    k_cache = _c(k_cache, np.float32)
    v_cache = _c(v_cache, np.float32)
    assert k_cache.shape == v_cache.shape
    B, _, Hkv, D = k_cache.shape
    N, Hq, Dq = q.shape
    assert Dq == D and Hq % Hkv == 0
    prefix_len = _c(prefix_len, np.int32)
    node_offsets = _c(node_offsets, np.int32)
    parent = _c(parent, np.int32)
    assert node_offsets.shape[0] == B + 1 and node_offsets[-1] == N
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((N, Hq, D), dtype=np.float64)
    status = np.zeros(B, dtype=np.int32)
    sb, sl, sh = (s // 4 for s in k_cache.strides[:3])
    _lib().oracle_tree_attention(
        _p(q, _f32p), _p(k_cache, _f32p), _p(v_cache, _f32p), sb, sl, sh,
        _p(prefix_len, _i32p), _p(node_offsets, _i32p), _p(parent, _i32p),
        B, Hq, Hkv, D, float(scale), _p(out, _f64p), _p(status, _i32p))
    return out, status


def tree_attention_dense_mask(q, k_cache, v_cache, prefix_len, node_offsets, parent, scale=None):
    """Tree attention in fp64 (formulation beta): dense boolean mask + masked softmax.

    The mask row of node i over the request's cache rows 0 .. P+n-1 is true on
    the whole prefix and on tree row P+j iff j is i or one of its ancestors.
    The ancestor relation is the reflexive-transitive closure of
    "j is the parent of i", computed by repeated boolean matrix squaring.
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    B, _, Hkv, D = k_cache.shape
    N, Hq, _ = q.shape
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((N, Hq, D), dtype=np.float64)
    for b in range(B):
        off, end = int(node_offsets[b]), int(node_offsets[b + 1])
        n, P = end - off, int(prefix_len[b])
        par = np.asarray(parent[off:end])
        reach = np.eye(n, dtype=bool)
        for i in range(n):
            if par[i] >= 0:
                reach[i, par[i]] = True
        for _ in range(max(1, int(math.ceil(math.log2(max(n, 2)))) + 1)):
            reach = reach | ((reach.astype(np.int64) @ reach.astype(np.int64)) > 0)
        mask = np.concatenate([np.ones((n, P), dtype=bool), reach], axis=1)  # [n, P+n]
        for h in range(Hq):
            g = h // G
            kk = k_cache[b, : P + n, g, :]  # [P+n, D]
            vv = v_cache[b, : P + n, g, :]
            s = scale * (q[off:end, h, :] @ kk.T)  # [n, P+n]
            s = np.where(mask, s, -np.inf)
            s = s - s.max(axis=1, keepdims=True)
            w = np.exp(s)
            out[off:end, h, :] = (w @ vv) / w.sum(axis=1, keepdims=True)
    return out


def verify_greedy(logits, tokens, parent, node_offsets):
    """Greedy token-tree verification.  Returns dict(path, accept_len, bonus, status)."""
    logits = _c(logits, np.float32)
    N, V = logits.shape
    tokens = _c(tokens, np.int32)
    parent = _c(parent, np.int32)
    node_offsets = _c(node_offsets, np.int32)
    B = node_offsets.shape[0] - 1
    path = np.full(N, -1, dtype=np.int32)
    accept_len = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    _lib().oracle_verify_greedy(
        _p(logits, _f32p), V, _p(tokens, _i32p), _p(parent, _i32p), _p(node_offsets, _i32p), B,
        _p(path, _i32p), _p(accept_len, _i32p), _p(bonus, _i32p), _p(status, _i32p))
    return dict(path=path, accept_len=accept_len, bonus=bonus, status=status)


def verify_stochastic(llm_logits, ssm_probs, tokens, parent, node_offsets, u_accept, u_sample,
                      temperature=1.0, top_k=0, top_p=1.0):
    """Multi-step speculative sampling against the LLM distribution
    softmax(logits / temperature), warped by top-k (top_k > 0) and then top-p
    (top_p < 1) when asked (see warp_row in oracle.c for the exact rule).

    Returns dict(path, accept_len, bonus, n_tried, n_near_tie, tie_path_len, status).
    """
    llm_logits = _c(llm_logits, np.float32)
    ssm_probs = _c(ssm_probs, np.float32)
    N, V = llm_logits.shape
    assert ssm_probs.shape == (N, V)
    tokens = _c(tokens, np.int32)
    parent = _c(parent, np.int32)
    node_offsets = _c(node_offsets, np.int32)
    u_accept = _c(u_accept, np.float32)
    u_sample = _c(u_sample, np.float32)
    B = node_offsets.shape[0] - 1
    path = np.full(N, -1, dtype=np.int32)
    out = {k: np.zeros(B, dtype=np.int32) for k in
           ("accept_len", "bonus", "n_tried", "n_near_tie", "tie_path_len", "status")}
    _lib().oracle_verify_stochastic(
        _p(llm_logits, _f32p), _p(ssm_probs, _f32p), V, _p(tokens, _i32p), _p(parent, _i32p),
        _p(node_offsets, _i32p), _p(u_accept, _f32p), _p(u_sample, _f32p), B, float(temperature),
        int(top_k), float(top_p), _p(path, _i32p), _p(out["accept_len"], _i32p), _p(out["bonus"], _i32p),
        _p(out["n_tried"], _i32p), _p(out["n_near_tie"], _i32p), _p(out["tie_path_len"], _i32p),
        _p(out["status"], _i32p))
    out["path"] = path
    return out


def kv_commit(k_cache, v_cache, prefix_len, node_offsets, path, accept_len):
    """Commit the accepted path to the KV cache.

    SpecInfer §4 (Token Tree Verifier) keeps one cache for the verified
    sequence and the speculated tree; once a path is accepted, its tokens
    become the next part of the verified sequence.  Tree node i of request b
    sits at cache row prefix_len[b] + i (the root, node 0, is the last verified
    token), so committing the path path[0] = 0, path[1], ..., path[L] means:
    row prefix_len[b] + k of the result holds row prefix_len[b] + path[k] of
    the input, for k = 1 .. L; every other row is unchanged.

    A path is accepted for commit when 0 <= L < n_b, path[0] == 0 and
    path[1..L] rise strictly below n_b; otherwise that request's rows are left
    as they are and its status is INVALID_ARG.  Returns (k, v, new_len,
    status) with new_len[b] = prefix_len[b] + 1 + L (-1 when rejected).
    k_cache, v_cache: [B, Lcap, Hkv, D] arrays of any dtype (values are copied).
    """
    k_in = np.asarray(k_cache)
    v_in = np.asarray(v_cache)
    k_out = k_in.copy()
    v_out = v_in.copy()
    B = len(node_offsets) - 1
    new_len = np.full(B, -1, dtype=np.int64)
    status = np.zeros(B, dtype=np.int64)
    for b in range(B):
        off = int(node_offsets[b])
        n = int(node_offsets[b + 1]) - off
        L = int(accept_len[b])
        P = int(prefix_len[b])
        ok = 0 <= L < n
        if ok:
            pth = [int(x) for x in path[off:off + L + 1]]
            ok = pth[0] == 0 and all(pth[k - 1] < pth[k] < n for k in range(1, L + 1))
        if not ok:
            status[b] = INVALID_ARG
            continue
        for k in range(1, L + 1):
            k_out[b, P + k] = k_in[b, P + pth[k]]
            v_out[b, P + k] = v_in[b, P + pth[k]]
        new_len[b] = P + 1 + L
    return k_out, v_out, new_len, status


def tree_expand(ssm_logits, k):
    """Expansion step of token-tree construction (SpecInfer §3, expansion-based
    token tree construction: each node of the frontier gets the SSM's top-k
    tokens as children).

    ssm_logits: [F, V] logits of the F frontier nodes.  Returns tokens [F, k]:
    row f lists the k tokens of largest logit, larger first, equal logits by
    lower token index (k <= V).
    """
    z = np.asarray(ssm_logits, dtype=np.float32)
    F, V = z.shape
    out = np.zeros((F, k), dtype=np.int32)
    for f in range(F):
        ranked = sorted(range(V), key=lambda t: (-float(z[f, t]), t))
        out[f] = ranked[:k]
    return out


def tree_merge(parents, tokens):
    """Merge-based token-tree construction (SpecInfer §3: the trees of several
    speculators are merged into one token tree).  Every input tree shares the
    root (node 0, the last verified token); a node is identified by the token
    path from the root, so equal paths become one node.

    parents / tokens: lists of int arrays, one pair per input tree (parent[0]
    = -1, parent[i] < i).  Returns (parent, token, source) of the union in
    creation order: input trees in order, nodes in order, a node created the
    first time its path is seen; source[j] = (tree, node) that created it.
    """
    key_to_id = {(): 0}
    par_out, tok_out, src = [-1], [int(tokens[0][0])], [(0, 0)]
    for t, (par, tok) in enumerate(zip(parents, tokens)):
        path_of = {0: ()}
        for i in range(1, len(par)):
            path = path_of[int(par[i])] + (int(tok[i]),)
            path_of[i] = path
            if path not in key_to_id:
                key_to_id[path] = len(par_out)
                par_out.append(key_to_id[path[:-1]])
                tok_out.append(int(tok[i]))
                src.append((t, i))
    return (np.array(par_out, dtype=np.int32), np.array(tok_out, dtype=np.int32), src)
