"""Python binding of libtsv — token-tree speculative verification on GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libtsv.so`` (built in-tree for sm_103a by ``build.py``).  Importing
this package fails loudly when the library has not been built; there is no
fallback implementation.  PyTorch supplies device memory and the current
stream.

Two layers:
  * ``tsv_*`` functions mirror the C ABI of ``include/tsv.h`` one to one
    (tensors are passed by their data pointers, ``None`` is NULL, host arrays
    are int32 numpy arrays);
  * ``tree_prepare``, ``tree_attention``, ``tree_verify_greedy`` and
    ``tree_verify_stochastic`` allocate outputs and workspace with torch and
    call the mirror functions.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsv.so")

(TSV_OK, TSV_ERR_INVALID_ARG, TSV_ERR_BAD_TREE, TSV_ERR_UNSUPPORTED, TSV_ERR_CUDA, TSV_ERR_TIMEOUT,
 TSV_ERR_SCRATCH_LIMIT) = range(7)
TSV_F32, TSV_BF16 = 0, 1
TSV_ATTN_DEFAULT, TSV_ATTN_SIMT = 0, 1
TSV_MAX_NODES, TSV_MAX_BATCH, TSV_ANC_WORDS = 256, 128, 8

EXPORTED = (
    "tsv_status_string", "tsv_version", "tsv_create", "tsv_destroy", "tsv_tree_prepare",
    "tsv_tree_attention_workspace_size", "tsv_tree_attention",
    "tsv_tree_verify_greedy_workspace_size", "tsv_tree_verify_greedy",
    "tsv_tree_verify_stochastic_workspace_size", "tsv_tree_verify_stochastic",
    "tsv_tree_verify_greedy_noalloc", "tsv_kv_commit", "tsv_tree_verify_stochastic_warped",
    "tsv_tree_expand", "tsv_tree_merge", "tsv_selftest_bounded_wait", "tsv_set_verify_overlap",
)


class TSVError(RuntimeError):
    def __init__(self, code, where):
        super().__init__("%s: %s (status %d)" % (where, status_string(code), code))
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libtsv.so is not built: run `python tree_speculative_verification_attention_gb300/build.py`"
            " (or __graft_entry__.build()) first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                  ctypes.c_float, ctypes.c_size_t)
    i32p = ctypes.POINTER(ctypes.c_int32)
    szp = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "tsv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "tsv_version": (ctypes.c_int, []),
        "tsv_create": (ctypes.c_int, [ctypes.POINTER(vp), ctypes.c_int]),
        "tsv_destroy": (ctypes.c_int, [vp]),
        "tsv_tree_prepare": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, vp, vp]),
        "tsv_tree_attention_workspace_size": (
            ctypes.c_int, [vp, ctypes.c_int, i32, i32p, i32p, i32, i32, i32, ctypes.c_int, u32, szp]),
        "tsv_tree_attention": (
            ctypes.c_int, [vp, ctypes.c_int, vp, vp, vp, i64, i64, i64, vp, i32p, i32p, vp, vp, vp, vp,
                           i32, i32, i32, i32, f32, vp, sz, vp, u32, vp]),
        "tsv_tree_verify_greedy_workspace_size": (ctypes.c_int, [vp, i32, i32, i64, szp]),
        "tsv_tree_verify_greedy": (
            ctypes.c_int, [vp, vp, i64, vp, vp, vp, i32, i32, vp, vp, vp, vp, sz, vp, vp]),
        "tsv_tree_verify_greedy_noalloc": (
            ctypes.c_int, [vp, vp, i64, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp]),
        "tsv_tree_verify_stochastic_warped": (
            ctypes.c_int, [vp, vp, vp, i64, vp, vp, vp, vp, vp, f32, i32, f32, i32, i32, vp, vp, vp, vp, vp, sz,
                           vp, vp]),
        "tsv_tree_expand": (ctypes.c_int, [vp, vp, i64, i32, i32, vp, vp]),
        "tsv_tree_merge": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]),
        "tsv_selftest_bounded_wait": (ctypes.c_int, [vp, i32, vp, vp, vp]),
        "tsv_set_verify_overlap": (ctypes.c_int, [vp, u32]),
        "tsv_kv_commit": (
            ctypes.c_int, [vp, ctypes.c_int, vp, vp, i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]),
        "tsv_tree_verify_stochastic_workspace_size": (ctypes.c_int, [vp, i32, i32, i64, szp]),
        "tsv_tree_verify_stochastic": (
            ctypes.c_int, [vp, vp, vp, i64, vp, vp, vp, vp, vp, f32, i32, i32, vp, vp, vp, vp, vp, sz,
                           vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


_lib = _load()


def status_string(code: int) -> str:
    return _lib.tsv_status_string(int(code)).decode()


def _check(code, where):
    if code != TSV_OK:
        raise TSVError(code, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host_i32(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return TSV_BF16
    if dt == torch.float32:
        return TSV_F32
    raise TypeError("tree attention takes bfloat16 or float32 tensors, got %s" % dt)


# ----------------------------------------------------------------- C ABI mirror


def tsv_version() -> int:
    return _lib.tsv_version()


def tsv_create(device: int = 0):
    h = ctypes.c_void_p()
    _check(_lib.tsv_create(ctypes.byref(h), int(device)), "tsv_create")
    return h


def tsv_destroy(h):
    _check(_lib.tsv_destroy(h), "tsv_destroy")


def tsv_tree_prepare(h, parent, node_offsets, B, anc, depth, status, stream=None):
    _check(_lib.tsv_tree_prepare(h, _ptr(parent), _ptr(node_offsets), int(B), _ptr(anc), _ptr(depth),
                                 _ptr(status), _stream(stream)), "tsv_tree_prepare")


def tsv_tree_attention_workspace_size(h, dtype_code, B, prefix_len_host, node_offsets_host, Hq, Hkv, D,
                                      anc_given, flags=TSV_ATTN_DEFAULT) -> int:
    pl, plp = _host_i32(prefix_len_host)
    no, nop = _host_i32(node_offsets_host)
    out = ctypes.c_size_t()
    _check(_lib.tsv_tree_attention_workspace_size(h, int(dtype_code), int(B), plp, nop, int(Hq), int(Hkv),
                                                  int(D), int(bool(anc_given)), int(flags),
                                                  ctypes.byref(out)),
           "tsv_tree_attention_workspace_size")
    return out.value


def tsv_tree_attention(h, dtype_code, q, k_cache, v_cache, kv_stride_b, kv_stride_l, kv_stride_h, out,
                       prefix_len_host, node_offsets_host, prefix_len, node_offsets, parent, anc, B, Hq,
                       Hkv, D, scale, workspace, workspace_bytes, status, flags=TSV_ATTN_DEFAULT,
                       stream=None):
    pl, plp = _host_i32(prefix_len_host)
    no, nop = _host_i32(node_offsets_host)
    _check(_lib.tsv_tree_attention(
        h, int(dtype_code), _ptr(q), _ptr(k_cache), _ptr(v_cache), int(kv_stride_b), int(kv_stride_l),
        int(kv_stride_h), _ptr(out), plp, nop, _ptr(prefix_len), _ptr(node_offsets), _ptr(parent),
        _ptr(anc), int(B), int(Hq), int(Hkv), int(D), float(scale), _ptr(workspace),
        int(workspace_bytes), _ptr(status), int(flags), _stream(stream)), "tsv_tree_attention")


def tsv_tree_verify_greedy_workspace_size(h, B, N, V) -> int:
    out = ctypes.c_size_t()
    _check(_lib.tsv_tree_verify_greedy_workspace_size(h, int(B), int(N), int(V), ctypes.byref(out)),
           "tsv_tree_verify_greedy_workspace_size")
    return out.value


def tsv_tree_verify_greedy(h, logits, V, tree_tokens, parent, node_offsets, B, N, path, accept_len, bonus,
                           workspace, workspace_bytes, status, stream=None):
    _check(_lib.tsv_tree_verify_greedy(
        h, _ptr(logits), int(V), _ptr(tree_tokens), _ptr(parent), _ptr(node_offsets), int(B), int(N),
        _ptr(path), _ptr(accept_len), _ptr(bonus), _ptr(workspace), int(workspace_bytes), _ptr(status),
        _stream(stream)), "tsv_tree_verify_greedy")


def tsv_tree_verify_greedy_noalloc(h, logits, V, tree_tokens, parent, node_offsets, B, N, path, accept_len,
                                   bonus, status, stream=None):
    """Greedy verification with the library's fixed device scratch (no workspace
    argument): for callers that cannot allocate device memory.  Calls that overlap
    on the GPU share that scratch and must not run concurrently."""
    _check(_lib.tsv_tree_verify_greedy_noalloc(
        h, _ptr(logits), int(V), _ptr(tree_tokens), _ptr(parent), _ptr(node_offsets), int(B), int(N),
        _ptr(path), _ptr(accept_len), _ptr(bonus), _ptr(status), _stream(stream)),
        "tsv_tree_verify_greedy_noalloc")


def tsv_tree_verify_stochastic_warped(h, llm_logits, ssm_probs, V, tree_tokens, parent, node_offsets, u_accept,
                                      u_sample, temperature, top_k, top_p, B, N, path, accept_len, bonus,
                                      n_tried, workspace, workspace_bytes, status, stream=None):
    _check(_lib.tsv_tree_verify_stochastic_warped(
        h, _ptr(llm_logits), _ptr(ssm_probs), int(V), _ptr(tree_tokens), _ptr(parent), _ptr(node_offsets),
        _ptr(u_accept), _ptr(u_sample), float(temperature), int(top_k), float(top_p), int(B), int(N), _ptr(path),
        _ptr(accept_len), _ptr(bonus), _ptr(n_tried), _ptr(workspace), int(workspace_bytes), _ptr(status),
        _stream(stream)), "tsv_tree_verify_stochastic_warped")


def tsv_tree_expand(h, ssm_logits, V, F, k, tokens, stream=None):
    _check(_lib.tsv_tree_expand(h, _ptr(ssm_logits), int(V), int(F), int(k), _ptr(tokens), _stream(stream)),
           "tsv_tree_expand")


def tsv_tree_merge(h, parent, tokens, tree_offsets, request_trees, B, out_parent, out_tokens, out_source,
                   out_count, status, stream=None):
    _check(_lib.tsv_tree_merge(h, _ptr(parent), _ptr(tokens), _ptr(tree_offsets), _ptr(request_trees), int(B),
                               _ptr(out_parent), _ptr(out_tokens), _ptr(out_source), _ptr(out_count),
                               _ptr(status), _stream(stream)), "tsv_tree_merge")


TSV_OVERLAP_GREEDY, TSV_OVERLAP_STOCHASTIC, TSV_OVERLAP_STOCHASTIC_FULL = 1, 2, 4


def tsv_set_verify_overlap(h, kinds):
    _check(_lib.tsv_set_verify_overlap(h, int(kinds)), "tsv_set_verify_overlap")


def tsv_selftest_bounded_wait(h, arrive, status, elapsed_ns=None, stream=None):
    _check(_lib.tsv_selftest_bounded_wait(h, int(arrive), _ptr(status), _ptr(elapsed_ns), _stream(stream)),
           "tsv_selftest_bounded_wait")


def tsv_kv_commit(h, dtype_code, k_cache, v_cache, sb, sl, sh, B, Hkv, D, prefix_len, node_offsets, path,
                  accept_len, new_len, status, stream=None):
    _check(_lib.tsv_kv_commit(h, int(dtype_code), _ptr(k_cache), _ptr(v_cache), int(sb), int(sl), int(sh),
                              int(B), int(Hkv), int(D), _ptr(prefix_len), _ptr(node_offsets), _ptr(path),
                              _ptr(accept_len), _ptr(new_len), _ptr(status), _stream(stream)),
           "tsv_kv_commit")


def tsv_tree_verify_stochastic_workspace_size(h, B, N, V) -> int:
    out = ctypes.c_size_t()
    _check(_lib.tsv_tree_verify_stochastic_workspace_size(h, int(B), int(N), int(V), ctypes.byref(out)),
           "tsv_tree_verify_stochastic_workspace_size")
    return out.value


def tsv_tree_verify_stochastic(h, llm_logits, ssm_probs, V, tree_tokens, parent, node_offsets, u_accept,
                               u_sample, temperature, B, N, path, accept_len, bonus, n_tried, workspace,
                               workspace_bytes, status, stream=None):
    _check(_lib.tsv_tree_verify_stochastic(
        h, _ptr(llm_logits), _ptr(ssm_probs), int(V), _ptr(tree_tokens), _ptr(parent), _ptr(node_offsets),
        _ptr(u_accept), _ptr(u_sample), float(temperature), int(B), int(N), _ptr(path), _ptr(accept_len),
        _ptr(bonus), _ptr(n_tried), _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream)),
        "tsv_tree_verify_stochastic")


# ----------------------------------------------------------------- convenience layer

_HANDLES = {}


def handle(device=None):
    """A library handle for `device` (default: torch's current device), created once."""
    dev = torch.cuda.current_device() if device is None else int(device)
    if dev not in _HANDLES:
        _HANDLES[dev] = tsv_create(dev)
    return _HANDLES[dev]


@contextlib.contextmanager
def verify_overlap(kinds=TSV_OVERLAP_GREEDY | TSV_OVERLAP_STOCHASTIC, device=None):
    """Verification calls of the given kinds made inside the block run beside
    the kernel launched before them on their stream (tsv_set_verify_overlap):
    their inputs must be complete before that kernel began."""
    h = handle(device)
    tsv_set_verify_overlap(h, int(kinds))
    try:
        yield
    finally:
        tsv_set_verify_overlap(h, 0)


def _workspace(nbytes, device):
    """A zero-filled workspace (the library's completion counters start at zero)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def tree_prepare(parent, node_offsets, stream=None):
    """Ancestor bitsets (uint32 [N, 8] as int32), depths and per-request status."""
    N = parent.shape[0]
    B = node_offsets.shape[0] - 1
    dev = parent.device
    anc = torch.empty((N, TSV_ANC_WORDS), dtype=torch.int32, device=dev)
    depth = torch.empty(N, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    tsv_tree_prepare(handle(dev.index), parent, node_offsets, B, anc, depth, status, stream)
    return anc, depth, status


def tree_attention(q, k_cache, v_cache, prefix_len_host, node_offsets_host, prefix_len, node_offsets,
                   parent=None, anc=None, scale=0.0, flags=TSV_ATTN_DEFAULT, out=None, workspace=None,
                   status=None, stream=None):
    """Tree attention: q [N, Hq, D]; k_cache / v_cache [B, Lcap, Hkv, D] (or any view
    with D contiguous); returns out [N, Hq, D] (same dtype as q) and status [B]."""
    N, Hq, D = q.shape
    B = len(prefix_len_host)
    Hkv = k_cache.shape[2]
    assert k_cache.stride() == v_cache.stride() and k_cache.stride(3) == 1
    sb, sl, sh = k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)
    dev = q.device
    h = handle(dev.index)
    code = _dtype_code(q.dtype)
    if out is None:
        out = torch.empty_like(q)
    if status is None:
        status = torch.zeros(B, dtype=torch.int32, device=dev)
    need = tsv_tree_attention_workspace_size(h, code, B, prefix_len_host, node_offsets_host, Hq, Hkv, D,
                                             anc is not None, flags)
    if workspace is None:
        workspace = _workspace(need, dev)
    tsv_tree_attention(h, code, q, k_cache, v_cache, sb, sl, sh, out, prefix_len_host, node_offsets_host,
                       prefix_len, node_offsets, parent, anc, B, Hq, Hkv, D, scale, workspace,
                       workspace.numel(), status, flags, stream)
    return out, status


def tree_verify_greedy(logits, tree_tokens, parent, node_offsets, workspace=None, stream=None, out=None):
    """Greedy verification; returns dict(path [N], accept_len [B], bonus [B], status [B])."""
    N, V = logits.shape
    B = node_offsets.shape[0] - 1
    dev = logits.device
    h = handle(dev.index)
    o = out or dict(path=torch.empty(N, dtype=torch.int32, device=dev),
                    accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                    bonus=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = _workspace(tsv_tree_verify_greedy_workspace_size(h, B, N, V), dev)
    tsv_tree_verify_greedy(h, logits, V, tree_tokens, parent, node_offsets, B, N, o["path"],
                           o["accept_len"], o["bonus"], workspace, workspace.numel(), o["status"], stream)
    return o


def tree_verify_stochastic(llm_logits, ssm_probs, tree_tokens, parent, node_offsets, u_accept, u_sample,
                           temperature=1.0, workspace=None, stream=None, out=None, top_k=0, top_p=1.0):
    """Multi-step speculative sampling, against the top-k / top-p warped LLM
    distribution when top_k > 0 or top_p < 1; returns dict(path, accept_len,
    bonus, n_tried, status)."""
    N, V = llm_logits.shape
    B = node_offsets.shape[0] - 1
    dev = llm_logits.device
    h = handle(dev.index)
    o = out or dict(path=torch.empty(N, dtype=torch.int32, device=dev),
                    accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                    bonus=torch.empty(B, dtype=torch.int32, device=dev),
                    n_tried=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = _workspace(tsv_tree_verify_stochastic_workspace_size(h, B, N, V), dev)
    if top_k or top_p < 1.0:
        tsv_tree_verify_stochastic_warped(h, llm_logits, ssm_probs, V, tree_tokens, parent, node_offsets,
                                          u_accept, u_sample, temperature, top_k, top_p, B, N, o["path"],
                                          o["accept_len"], o["bonus"], o["n_tried"], workspace, workspace.numel(),
                                          o["status"], stream)
    else:
        tsv_tree_verify_stochastic(h, llm_logits, ssm_probs, V, tree_tokens, parent, node_offsets, u_accept,
                                   u_sample, temperature, B, N, o["path"], o["accept_len"], o["bonus"],
                                   o["n_tried"], workspace, workspace.numel(), o["status"], stream)
    return o


def kv_commit(k_cache, v_cache, prefix_len, node_offsets, path, accept_len, stream=None, out=None):
    """Moves the accepted path's K/V rows behind the prefix, in place: row
    prefix_len[b] + k takes node path[k]'s row.  k_cache / v_cache [B, Lcap,
    Hkv, D] (or views with d contiguous); the other arguments are device int32
    tensors as the verify calls write them.  Returns dict(new_len, status)."""
    B, _, Hkv, D = k_cache.shape
    assert k_cache.stride() == v_cache.stride() and k_cache.stride(3) == 1
    dev = k_cache.device
    o = out or dict(new_len=torch.empty(B, dtype=torch.int32, device=dev),
                    status=torch.empty(B, dtype=torch.int32, device=dev))
    tsv_kv_commit(handle(dev.index), _dtype_code(k_cache.dtype), k_cache, v_cache, k_cache.stride(0),
                  k_cache.stride(1), k_cache.stride(2), B, Hkv, D, prefix_len, node_offsets, path, accept_len,
                  o["new_len"], o["status"], stream)
    return o


def tree_expand(ssm_logits, k, stream=None, out=None):
    """Top-k children of every frontier row: int32 [F, k] tokens (larger logit
    first, equal logits by lower token index)."""
    F, V = ssm_logits.shape
    out = out if out is not None else torch.empty((F, k), dtype=torch.int32, device=ssm_logits.device)
    tsv_tree_expand(handle(ssm_logits.device.index), ssm_logits, V, F, k, out, stream)
    return out


def tree_merge(parent, tokens, tree_offsets, request_trees, stream=None):
    """Union of each request's input trees by token path; returns dict(parent,
    tokens, source, count, status) laid out as tsv_tree_merge describes."""
    dev = parent.device
    M = parent.shape[0]
    B = request_trees.shape[0] - 1
    o = dict(parent=torch.empty(M, dtype=torch.int32, device=dev), tokens=torch.empty(M, dtype=torch.int32, device=dev),
             source=torch.empty(M, dtype=torch.int32, device=dev), count=torch.empty(B, dtype=torch.int32, device=dev),
             status=torch.empty(B, dtype=torch.int32, device=dev))
    tsv_tree_merge(handle(dev.index), parent, tokens, tree_offsets, request_trees, B, o["parent"], o["tokens"],
                   o["source"], o["count"], o["status"], stream)
    return o


def selftest_bounded_wait(arrive, device=None, stream=None):
    """Runs the bounded-wait self-test on `device`; returns (status, elapsed
    seconds) after synchronising: (TSV_OK, ~0) with `arrive`, (TSV_ERR_TIMEOUT,
    about 1 s) without."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else int(device))
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ns = torch.zeros(1, dtype=torch.int64, device=dev)
    tsv_selftest_bounded_wait(handle(dev.index), arrive, st, ns, stream)
    torch.cuda.synchronize(dev)
    return int(st.item()), ns.item() * 1e-9
