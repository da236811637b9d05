"""Seeded synthetic inputs for token-tree verification (shared by tests, smoke and bench).

This module only draws inputs; it holds none of the verified method's arithmetic.
Both the GPU library's callers and the CPU oracle's callers take their inputs
from here, so the two sides always see the same numbers.

Seeding: every array comes from its own stream,
``np.random.SeedSequence([workload_id, stream, chunk])`` with PCG64, so each
array can be regenerated alone and large arrays are drawn in fixed chunks (the
values do not depend on the number of threads).  Streams:
0 tree, 1 prefix lengths, 2 Q, 3 K, 4 V, 5 greedy logits, 6 greedy tokens,
7 LLM logits, 8 SSM logits, 9 stochastic tokens, 10 uniforms.

Value rules:
  * bf16 tensors are drawn in fp32 and rounded to nearest-even; consumers read
    the rounded values (``.float()`` gives them exactly).
  * uniforms are drawn in fp64 in [0, 1) and rounded down to fp32.
  * cache rows past a request's prefix + tree are filled with ``pad_value``
    (0 by default; tests use NaN to prove those rows never reach an output).
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple, Union

import numpy as np
import torch

CHUNK = 1 << 22

S_TREE, S_PREFIX, S_Q, S_K, S_V, S_GLOGITS, S_GTOK, S_LLM, S_SSM, S_STOK, S_UNIF = range(11)


def _rng(wid: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([wid, stream, chunk])))


def normal_f32(wid: int, stream: int, shape, sigma: float = 1.0) -> np.ndarray:
    """N(0, sigma^2) fp32 array, drawn chunk by chunk from its own stream."""
    total = int(np.prod(shape))
    out = np.empty(total, dtype=np.float32)
    nchunks = (total + CHUNK - 1) // CHUNK

    def fill(c):
        lo, hi = c * CHUNK, min(total, (c + 1) * CHUNK)
        _rng(wid, stream, c).standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=16) as ex:
            list(ex.map(fill, range(nchunks)))
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out.reshape(shape)


def uniform_f32(wid: int, stream: int, n: int) -> np.ndarray:
    """U[0,1) drawn in fp64 and rounded down to fp32."""
    u64 = _rng(wid, stream).random(n)
    u32 = u64.astype(np.float32)
    over = u32.astype(np.float64) > u64
    u32[over] = np.nextafter(u32[over], np.float32(0.0))
    return u32


# --------------------------------------------------------------------------- trees


def random_tree(rng: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """parent[0] = -1; parent[i] ~ Uniform{j < i : depth[j] < max_depth}."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int32)
    for i in range(1, n):
        cand = np.nonzero(depth[:i] < max_depth)[0]
        j = int(cand[rng.integers(len(cand))])
        parent[i] = j
        depth[i] = depth[j] + 1
    return parent


def expansion_tree_trunk_chains(trunk: int = 2, branches: int = 3, chain: int = 6) -> np.ndarray:
    """A trunk of ``trunk`` tokens, then ``branches`` children of the trunk's end,
    each extending a chain of ``chain`` tokens (20 nodes for 2/3/6)."""
    parent = [-1] + list(range(trunk - 1))
    for _ in range(branches):
        start = len(parent)
        parent.append(trunk - 1)
        parent.extend(range(start, start + chain - 1))
    return np.asarray(parent, dtype=np.int32)


def merge_tree(rng: np.random.Generator, subtrees: int = 3, sub_nodes: int = 21,
               max_depth: int = 8) -> np.ndarray:
    """Union of ``subtrees`` random-branching speculator trees under one shared root.

    Each subtree grows breadth-first from a child of the root; every expanded
    node gets k ~ U{1,2,3} children while its depth is below ``max_depth``.  The
    subtrees are concatenated in order (no token de-duplication).
    """
    parent = [-1]
    depth = [0]
    for _ in range(subtrees):
        base = len(parent)
        parent.append(0)
        depth.append(1)
        queue = [base]
        while len(parent) - base < sub_nodes:
            if not queue:  # every frontier node hit the depth cap: attach anywhere legal
                cand = [i for i in range(base, len(parent)) if depth[i] < max_depth]
                queue = [cand[int(rng.integers(len(cand)))]]
            u = queue.pop(0)
            if depth[u] >= max_depth:
                continue
            k = int(rng.integers(1, 4))
            for _ in range(k):
                if len(parent) - base >= sub_nodes:
                    break
                parent.append(u)
                depth.append(depth[u] + 1)
                queue.append(len(parent) - 1)
    return np.asarray(parent, dtype=np.int32)


def tree_depths(parent: np.ndarray) -> np.ndarray:
    depth = np.zeros(len(parent), dtype=np.int32)
    for i, p in enumerate(parent):
        depth[i] = 0 if p < 0 else depth[p] + 1
    return depth


# --------------------------------------------------------------------------- specs


@dataclass(frozen=True)
class Spec:
    """Shape and recipe of one synthetic workload."""
    name: str
    wid: int
    dtype: str  # "f32" or "bf16": type of q / K / V / out
    B: int
    Hq: int
    Hkv: int
    D: int
    V: int
    prefix: Union[int, Tuple[int, int]]  # fixed, or inclusive uniform range
    nodes: int
    tree: str  # "random", "trunk_chains", "merge", "chain", "star"
    max_depth: int = 5
    greedy_sigma: float = 1.0
    greedy: bool = True
    stochastic: bool = False
    pad_value: float = 0.0
    extra: dict = field(default_factory=dict)


SPECS = {
    # Tiny fp32 case: one request, one head, D 64, prefix 128, 16-node random tree.
    "tiny-f32-P128-n16": Spec("tiny-f32-P128-n16", 1, "f32", 1, 1, 1, 64, 1000, 128, 16,
                              "random", max_depth=5, greedy_sigma=1.0),
    # Llama-7B-shaped single layer: 32 heads, D 128, prefix 1024, 20-node expansion tree.
    "llama7b-layer-P1024-n20": Spec("llama7b-layer-P1024-n20", 2, "bf16", 1, 32, 32, 128, 32000,
                                    1024, 20, "trunk_chains", greedy_sigma=3.0),
    # Batch 8, ragged prefixes U[512, 4096], 64-node merge trees, MSS verification.
    "batch8-ragged-merge64-mss": Spec("batch8-ragged-merge64-mss", 3, "bf16", 8, 32, 32, 128,
                                      32000, (512, 4096), 64, "merge", max_depth=8,
                                      greedy=False, stochastic=True),
    # Long context GQA: 64 query / 8 KV heads, prefix 32768, 128-node random tree.
    "gqa64x8-P32768-n128": Spec("gqa64x8-P32768-n128", 4, "bf16", 1, 64, 8, 128, 128256, 32768,
                                128, "random", max_depth=12, greedy_sigma=1.0, stochastic=True),
    # Large batch: 32 requests, prefix 2048, 16-node random trees.
    "batch32-P2048-n16": Spec("batch32-P2048-n16", 5, "bf16", 32, 32, 32, 128, 32000, 2048, 16,
                              "random", max_depth=6, greedy_sigma=1.0, stochastic=True),
}
ORDER = list(SPECS)


def spec_variant(spec: Spec, **kw) -> Spec:
    return replace(spec, **kw)


# --------------------------------------------------------------------------- generation


@dataclass
class Trees:
    prefix_len: np.ndarray  # int32 [B]
    node_offsets: np.ndarray  # int32 [B+1]
    parent: np.ndarray  # int32 [N], local indices per request
    Lcap: int


def make_trees(spec: Spec) -> Trees:
    rng_t = _rng(spec.wid, S_TREE)
    parents = []
    for _ in range(spec.B):
        if spec.tree == "random":
            parents.append(random_tree(rng_t, spec.nodes, spec.max_depth))
        elif spec.tree == "trunk_chains":
            p = expansion_tree_trunk_chains()
            assert len(p) == spec.nodes
            parents.append(p)
        elif spec.tree == "merge":
            sub = (spec.nodes - 1) // 3
            assert 1 + 3 * sub == spec.nodes
            parents.append(merge_tree(rng_t, 3, sub, spec.max_depth))
        elif spec.tree == "chain":
            parents.append(np.arange(-1, spec.nodes - 1, dtype=np.int32))
        elif spec.tree == "star":
            p = np.zeros(spec.nodes, dtype=np.int32)
            p[0] = -1
            parents.append(p)
        else:
            raise ValueError(spec.tree)
    if isinstance(spec.prefix, tuple):
        lo, hi = spec.prefix
        prefix_len = _rng(spec.wid, S_PREFIX).integers(lo, hi + 1, size=spec.B).astype(np.int32)
    else:
        prefix_len = np.full(spec.B, spec.prefix, dtype=np.int32)
    sizes = np.array([len(p) for p in parents], dtype=np.int32)
    node_offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    Lcap = int((prefix_len + sizes).max())
    return Trees(prefix_len, node_offsets, np.concatenate(parents).astype(np.int32), Lcap)


def _to_dtype(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(x)
    return t.to(torch.bfloat16) if dtype == "bf16" else t.clone()


@dataclass
class AttentionInputs:
    q: torch.Tensor  # [N, Hq, D] (CPU, spec dtype)
    k_cache: torch.Tensor  # [B, Lcap, Hkv, D]
    v_cache: torch.Tensor


def make_attention_inputs(spec: Spec, trees: Trees, Lcap: Optional[int] = None) -> AttentionInputs:
    N = int(trees.node_offsets[-1])
    Lcap = trees.Lcap if Lcap is None else Lcap
    q = normal_f32(spec.wid, S_Q, (N, spec.Hq, spec.D))
    k = normal_f32(spec.wid, S_K, (spec.B, Lcap, spec.Hkv, spec.D))
    v = normal_f32(spec.wid, S_V, (spec.B, Lcap, spec.Hkv, spec.D))
    sizes = np.diff(trees.node_offsets)
    for b in range(spec.B):
        used = int(trees.prefix_len[b] + sizes[b])
        k[b, used:] = spec.pad_value
        v[b, used:] = spec.pad_value
    return AttentionInputs(_to_dtype(q, spec.dtype), _to_dtype(k, spec.dtype), _to_dtype(v, spec.dtype))


@dataclass
class GreedyInputs:
    logits: np.ndarray  # float32 [N, V]
    tokens: np.ndarray  # int32 [N]


def make_greedy_inputs(spec: Spec, trees: Trees) -> GreedyInputs:
    """Logits ~ N(0, sigma^2); a child's token equals its parent's argmax with
    probability 1/2, else it is uniform over the other V-1 tokens (V = 1:
    every token is 0)."""
    N = int(trees.node_offsets[-1])
    logits = normal_f32(spec.wid, S_GLOGITS, (N, spec.V), spec.greedy_sigma)
    rng = _rng(spec.wid, S_GTOK)
    tokens = np.zeros(N, dtype=np.int32)
    for b in range(spec.B):
        off = int(trees.node_offsets[b])
        n = int(trees.node_offsets[b + 1]) - off
        for i in range(n):
            p = int(trees.parent[off + i])
            hit = rng.random() < 0.5 or spec.V == 1  # with one token every child matches
            other = int(rng.integers(spec.V - 1)) if spec.V > 1 else 0
            if p < 0:
                tokens[off + i] = other
                continue
            top = int(np.argmax(logits[off + p]))
            tokens[off + i] = top if hit else (other if other < top else other + 1)
    return GreedyInputs(logits, tokens)


@dataclass
class StochasticInputs:
    llm_logits: np.ndarray  # float32 [N, V], ~ N(0, 2^2)
    ssm_probs: np.ndarray  # float32 [N, V], rows softmax(N(0, 2^2)) (row c = node c's proposal)
    tokens: np.ndarray  # int32 [N], token[c] ~ ssm_probs[c]
    u_accept: np.ndarray  # float32 [N]
    u_sample: np.ndarray  # float32 [N]


def proposal_rows(z: np.ndarray) -> np.ndarray:
    """Proposal distributions from raw scores (fp64 softmax per row, stored fp32)."""
    z64 = z.astype(np.float64)
    z64 -= z64.max(axis=1, keepdims=True)
    e = np.exp(z64)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def make_stochastic_inputs(spec: Spec, trees: Trees) -> StochasticInputs:
    N = int(trees.node_offsets[-1])
    llm = normal_f32(spec.wid, S_LLM, (N, spec.V), 2.0)
    ssm = proposal_rows(normal_f32(spec.wid, S_SSM, (N, spec.V), 2.0))
    rng = _rng(spec.wid, S_STOK)
    tokens = np.zeros(N, dtype=np.int32)
    for c in range(N):
        row = ssm[c].astype(np.float64)
        cdf = np.cumsum(row)
        x = int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right"))
        tokens[c] = min(x, spec.V - 1)
    u = uniform_f32(spec.wid, S_UNIF, 2 * N)
    return StochasticInputs(llm, ssm, tokens, u[:N].copy(), u[N:].copy())


def propose_near_llm(si: StochasticInputs, trees: Trees, mix: float = 0.7, seed: int = 0) -> StochasticInputs:
    """Stochastic inputs whose proposals sit close to the LLM's law at each
    node's parent (mix x softmax of the parent's LLM row + (1 - mix) x the
    drawn proposal row), with each child's token redrawn from its new row, so
    that accepted children are likely.  Returns a new StochasticInputs."""
    offs = trees.node_offsets
    prow = np.concatenate([np.maximum(trees.parent[offs[b]:offs[b + 1]], 0) + offs[b]
                           for b in range(len(offs) - 1)])
    q = (mix * proposal_rows(si.llm_logits[prow]).astype(np.float64)
         + (1.0 - mix) * si.ssm_probs.astype(np.float64)).astype(np.float32)
    rng = np.random.default_rng(seed)
    cdf = np.cumsum(q.astype(np.float64), axis=1)
    u = rng.random(len(cdf))[:, None] * cdf[:, -1:]
    tokens = np.minimum((u >= cdf).sum(1), q.shape[1] - 1).astype(np.int32)
    return StochasticInputs(si.llm_logits, q, tokens, si.u_accept, si.u_sample)


def fuzz_spec(seed: int, dtype: str = "bf16", max_nodes: int = 40) -> Spec:
    """A small random shape for parity fuzzing: random n, V, D, GQA group, prefixes."""
    r = _rng(1000 + seed, 99)
    B = int(r.integers(1, 4))
    D = int(r.choice([64, 128]))
    G = int(r.choice([1, 2, 8]))
    Hkv = int(r.integers(1, 3))
    lo = int(r.integers(0, 200))
    return Spec(f"fuzz{seed}", 1000 + seed, dtype, B, Hkv * G, Hkv, D, int(r.integers(2, 3000)),
                (lo, lo + int(r.integers(0, 300))), int(r.integers(1, max_nodes + 1)), "random",
                max_depth=int(r.integers(1, 9)), stochastic=True)


# --------------------------------------------------------------------------- sequence baseline


@dataclass
class SequenceBatch:
    """A tree batch decomposed into its root-to-leaf sequences: one request per
    leaf, a chain tree whose cache holds its own copy of the prefix followed by
    the rows of the leaf's path (the layout a sequence-based verifier uses)."""
    trees: Trees
    inputs: AttentionInputs
    tree_row: np.ndarray  # int64 [N_seq]: global tree node each sequence token stands for


def sequence_decomposition(trees: Trees, att: AttentionInputs) -> SequenceBatch:
    offs = trees.node_offsets
    chains, reqs = [], []
    for b in range(len(offs) - 1):
        off, n = int(offs[b]), int(offs[b + 1] - offs[b])
        par = trees.parent[off:off + n]
        has_child = np.zeros(n, dtype=bool)
        has_child[par[par >= 0]] = True
        for leaf in np.nonzero(~has_child)[0]:
            chain, node = [], int(leaf)
            while node >= 0:
                chain.append(node)
                node = int(par[node])
            chains.append(chain[::-1])
            reqs.append(b)
    S = len(chains)
    sizes = np.array([len(c) for c in chains], dtype=np.int32)
    prefix = np.array([int(trees.prefix_len[b]) for b in reqs], dtype=np.int32)
    Lcap = int((prefix + sizes).max())
    B, _, Hkv, D = att.k_cache.shape
    dev = att.k_cache.device  # gathers run where the cache lives (the copies can be large)
    k = torch.zeros((S, Lcap, Hkv, D), dtype=att.k_cache.dtype, device=dev)
    v = torch.zeros_like(k)
    q_rows, tree_row = [], []
    for s, (b, chain) in enumerate(zip(reqs, chains)):
        P = int(trees.prefix_len[b])
        k[s, :P] = att.k_cache[b, :P]
        v[s, :P] = att.v_cache[b, :P]
        rows = torch.as_tensor([P + c for c in chain], device=dev)
        k[s, P:P + len(chain)] = att.k_cache[b, rows]
        v[s, P:P + len(chain)] = att.v_cache[b, rows]
        tree_row.extend(int(offs[b]) + c for c in chain)
    tree_row = np.array(tree_row, dtype=np.int64)
    q = att.q[torch.as_tensor(tree_row, device=att.q.device)]
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    parent = np.concatenate([np.arange(-1, len(c) - 1, dtype=np.int32) for c in chains])
    return SequenceBatch(Trees(prefix, offsets, parent, Lcap), AttentionInputs(q, k, v), tree_row)
