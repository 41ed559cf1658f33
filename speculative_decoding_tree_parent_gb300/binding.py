"""Thin ctypes binding of libspecverify (include/spec_verify.h).

Functions carry the C entry points' names and argument order; they take torch
tensors (device memory) and only marshal pointers, sizes and the current CUDA
stream. All computation happens in the library's kernels. A negative status
raises SpecError; nothing here falls back to another implementation.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SPEC_OK = 0
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_GREEDY, SPEC_STOCHASTIC = 0, 1
SPEC_OP_MASK, SPEC_OP_ATTN, SPEC_OP_ACCEPT, SPEC_OP_COMMIT, SPEC_OP_TREE = 0, 1, 2, 3, 4
STATUS = {
    0: "SPEC_OK", -1: "SPEC_ERR_ARG", -2: "SPEC_ERR_PARENT", -3: "SPEC_ERR_PAGE", -4: "SPEC_ERR_CAPACITY",
    -5: "SPEC_ERR_WORKSPACE", -6: "SPEC_ERR_UNSUPPORTED", -7: "SPEC_ERR_CUDA", -8: "SPEC_ERR_TIMEOUT",
    -9: "SPEC_ERR_INDEX",
}
EXPORTS = ("spec_version", "spec_status_string", "spec_workspace_size", "spec_attn_plan", "spec_build_tree_mask",
           "spec_tree_verify_attn", "spec_accept", "spec_kv_commit", "spec_accept_commit", "spec_accept_noalloc",
           "spec_tree_init", "spec_tree_expand", "spec_tree_verify_attn_kv8", "spec_kv_commit_kv8",
           "spec_tree_verify_attn_parents", "spec_tree_expand_multi", "spec_accept_plan", "spec_set_early_reads")

_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "spec_version": (_I, []),
    "spec_status_string": (ctypes.c_char_p, [_I]),
    "spec_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "spec_attn_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "spec_accept_plan": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "spec_set_early_reads": (_I, [_I]),
    "spec_build_tree_mask": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "spec_tree_verify_attn": (_I, [_I, _P, _P, _P, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                   _I, _F, _P, _P, _P, _Z, _P, _P]),
    "spec_accept": (_I, [_I, _P, _P, _P, _P, _P, _F, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P, _P]),
    "spec_kv_commit": (_I, [_I, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "spec_accept_commit": (_I, [_I, _P, _P, _P, _P, _P, _F, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P,
                                _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _I, _P, _Z, _P, _P]),
    "spec_accept_noalloc": (_I, [_I, _P, _P, _P, _P, _P, _F, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "spec_tree_init": (_I, [_P, _I, _I, _P, _Z, _P, _P, _P, _P, _P, _P]),
    "spec_tree_expand": (_I, [_P, _I, ctypes.c_longlong, ctypes.c_longlong, _I, _I, _I, _I, ctypes.c_double, _P, _Z,
                              _P, _P, _P, _P, _P, _P, _P]),
    "spec_tree_expand_multi": (_I, [_P, _I, ctypes.c_longlong, ctypes.c_longlong, _I, _I, _I, _I, _I, ctypes.c_double,
                                    _P, _Z, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "spec_tree_verify_attn_kv8": (_I, [_P, _P, _P, _P, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                       _I, _F, _P, _P, _P, _Z, _P, _P]),
    "spec_tree_verify_attn_parents": (_I, [_P, _P, _P, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                           _I, _F, _P, _P, _P, _Z, _P, _P]),
    "spec_kv_commit_kv8": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
}

_lib = None


class SpecError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def load(path: str | None = None):
    """Open libspecverify.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libspecverify not found at {path}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().spec_status_string(int(status)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(st: int, what: str) -> int:
    if st < 0:
        raise SpecError(st, what)
    return st


def _dtype(t) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise ValueError(f"unsupported dtype {t.dtype}")


def _logits_ptr(t) -> int | None:
    """Logits may be a device tensor or a pinned host tensor (the library checks that the
    device reads it at the same address; the acceptance then reads only the rows it visits)."""
    if t is None:
        return None
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("device tensor or pinned host tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _need(t, dtype, what):
    if t.dtype != dtype:
        raise ValueError(f"{what}: {dtype} expected, got {t.dtype}")


def spec_workspace_size(op, batch=0, total_nodes=0, max_nodes=0, hq=0, hkv=0, d=0, max_prefix=0, vocab=0) -> int:
    return int(load().spec_workspace_size(op, batch, total_nodes, max_nodes, hq, hkv, d, max_prefix, vocab))


def spec_attn_plan(dtype, batch, max_nodes, hq, hkv, d, page_size, max_prefix):
    """(splits, tensor_cores) the attention call uses for these sizes."""
    s, tc = ctypes.c_int(0), ctypes.c_int(0)
    st = load().spec_attn_plan(int(dtype), batch, max_nodes, hq, hkv, d, page_size, max_prefix,
                               ctypes.addressof(s), ctypes.addressof(tc))
    _check(st, "spec_attn_plan")
    return s.value, tc.value


def spec_accept_plan(mode, batch, total_nodes, vocab, path_cap, sm_count=0):
    """1 when spec_accept reads only the visited nodes' rows (the walk), 0 when it streams
    every row (greedy only); sm_count 0: the current device's."""
    w = ctypes.c_int(0)
    st = load().spec_accept_plan(int(mode), int(batch), int(total_nodes), int(vocab), int(path_cap), int(sm_count),
                                 ctypes.addressof(w))
    _check(st, "spec_accept_plan")
    return w.value


def spec_set_early_reads(enable):
    """Let the attention and the greedy walk read their inputs before waiting for the kernel
    enqueued just before them (only where that kernel writes none of them); returns the
    previous setting. Off by default."""
    return int(load().spec_set_early_reads(1 if enable else 0))


class early_reads:
    """Context manager: spec_set_early_reads(enable) inside, the previous setting after."""

    def __init__(self, enable=True):
        self.enable = enable

    def __enter__(self):
        self.prev = spec_set_early_reads(self.enable)
        return self

    def __exit__(self, *exc):
        spec_set_early_reads(self.prev)
        return False


def spec_build_tree_mask(parent, qo_indptr, max_nodes, mask, depth=None, dev_status=None, stream=None):
    _need(parent, torch.int32, "parent")
    _need(qo_indptr, torch.int32, "qo_indptr")
    _need(mask, torch.int64, "mask (uint64 bits held in an int64 tensor)")
    st = load().spec_build_tree_mask(_ptr(parent), _ptr(qo_indptr), qo_indptr.numel() - 1, parent.numel(),
                                     int(max_nodes), _ptr(mask), _ptr(depth), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_build_tree_mask")


def spec_tree_verify_attn(q, k_pool, v_pool, page_table, prefix_len, max_prefix, k_tree, v_tree, mask,
                          qo_indptr, max_nodes, out, lse=None, ws=None, sm_scale=0.0, dev_status=None,
                          stream=None):
    """q [T,Hq,D]; k_pool/v_pool [pages,Hkv,PS,D]; page_table int32 [B,max_pages]; k_tree/v_tree [T,Hkv,D]."""
    dt = _dtype(q)
    T, hq, d = q.shape
    num_pages, hkv, ps, _ = k_pool.shape
    st = load().spec_tree_verify_attn(
        dt, _ptr(q), _ptr(k_pool), _ptr(v_pool), num_pages, ps, _ptr(page_table), page_table.shape[1],
        _ptr(prefix_len), int(max_prefix), _ptr(k_tree), _ptr(v_tree), _ptr(mask), _ptr(qo_indptr),
        qo_indptr.numel() - 1, T, int(max_nodes), hq, hkv, d, float(sm_scale), _ptr(out), _ptr(lse),
        _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_tree_verify_attn")


def spec_accept(mode, parent, draft_tokens, target_logits, qo_indptr, max_nodes, accept_len, path, out_tokens,
                ws, draft_logits=None, uniforms=None, temperature=1.0, flags=None, dev_status=None, stream=None):
    T, V = target_logits.shape
    st = load().spec_accept(
        int(mode), _ptr(parent), _ptr(draft_tokens), _logits_ptr(target_logits), _logits_ptr(draft_logits),
        _ptr(uniforms),
        float(temperature), V, _ptr(qo_indptr), qo_indptr.numel() - 1, T, int(max_nodes), path.shape[1],
        _ptr(accept_len), _ptr(path), _ptr(out_tokens), _ptr(flags), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(dev_status), _stream(stream))
    return _check(st, "spec_accept")


def spec_kv_commit(k_tree, v_tree, path, accept_len, qo_indptr, page_table, prefix_len, k_pool, v_pool,
                   seq_len_out=None, dev_status=None, stream=None):
    dt = _dtype(k_tree)
    T, hkv, d = k_tree.shape
    num_pages, _, ps, _ = k_pool.shape
    st = load().spec_kv_commit(
        dt, _ptr(k_tree), _ptr(v_tree), _ptr(path), path.shape[1], _ptr(accept_len), _ptr(qo_indptr),
        _ptr(page_table), page_table.shape[1], num_pages, ps, _ptr(prefix_len), _ptr(seq_len_out), _ptr(k_pool),
        _ptr(v_pool), qo_indptr.numel() - 1, T, hkv, d, _ptr(dev_status), _stream(stream))
    return _check(st, "spec_kv_commit")


def spec_accept_commit(mode, parent, draft_tokens, target_logits, qo_indptr, max_nodes, accept_len, path,
                       out_tokens, ws, k_tree, v_tree, page_table, prefix_len, k_pool, v_pool, seq_len_out=None,
                       draft_logits=None, uniforms=None, temperature=1.0, flags=None, dev_status=None, stream=None,
                       token_buf=None):
    """spec_accept then spec_kv_commit of the accepted paths, as one call; with `token_buf`
    ([batch][stride] int32) also the step's tokens written after each sequence's root."""
    T, V = target_logits.shape
    _, hkv, d = k_tree.shape
    num_pages, _, ps, _ = k_pool.shape
    stride = token_buf.shape[1] if token_buf is not None else 0
    st = load().spec_accept_commit(
        int(mode), _ptr(parent), _ptr(draft_tokens), _logits_ptr(target_logits), _logits_ptr(draft_logits),
        _ptr(uniforms),
        float(temperature), V, _ptr(qo_indptr), qo_indptr.numel() - 1, T, int(max_nodes), path.shape[1],
        _ptr(accept_len), _ptr(path), _ptr(out_tokens), _ptr(flags), _dtype(k_tree), _ptr(k_tree), _ptr(v_tree),
        _ptr(page_table), page_table.shape[1], num_pages, ps, _ptr(prefix_len), _ptr(seq_len_out), _ptr(k_pool),
        _ptr(v_pool), hkv, d, _ptr(token_buf), stride, _ptr(ws), ws.numel() * ws.element_size(), _ptr(dev_status),
        _stream(stream))
    return _check(st, "spec_accept_commit")


def spec_accept_noalloc(mode, parent, draft_tokens, target_logits, qo_indptr, max_nodes, accept_len, path,
                        out_tokens, draft_logits=None, uniforms=None, temperature=1.0, flags=None, dev_status=None,
                        stream=None):
    """spec_accept without a workspace argument: for callers that cannot allocate device
    memory; the scratch is a fixed array inside the library (see include/spec_verify.h)."""
    T, V = target_logits.shape
    st = load().spec_accept_noalloc(
        int(mode), _ptr(parent), _ptr(draft_tokens), _logits_ptr(target_logits), _logits_ptr(draft_logits),
        _ptr(uniforms),
        float(temperature), V, _ptr(qo_indptr), qo_indptr.numel() - 1, T, int(max_nodes), path.shape[1],
        _ptr(accept_len), _ptr(path), _ptr(out_tokens), _ptr(flags), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_accept_noalloc")


def spec_tree_init(root_tokens, max_nodes, state, parent_out, tokens_out, n_nodes_out, next_node, flags=None,
                   stream=None):
    """Start one draft tree per sequence at its root token (see include/spec_verify.h)."""
    st = load().spec_tree_init(_ptr(root_tokens), root_tokens.numel(), int(max_nodes), _ptr(state),
                               state.numel() * state.element_size(), _ptr(parent_out), _ptr(tokens_out),
                               _ptr(n_nodes_out), _ptr(next_node), _ptr(flags), _stream(stream))
    return _check(st, "spec_tree_init")


def spec_tree_expand(draft_logits, max_nodes, topk, max_depth, state, parent_out, tokens_out, n_nodes_out,
                     next_node, row_stride, node_stride, threshold=0.0, flags=None, dev_status=None, stream=None):
    """One expansion of every sequence's draft tree from the draft logits rows (vocabulary =
    the last dimension of draft_logits; strides in elements)."""
    V = draft_logits.shape[-1]
    st = load().spec_tree_expand(_ptr(draft_logits), V, int(row_stride), int(node_stride), next_node.numel(),
                                 int(max_nodes), int(topk), int(max_depth), float(threshold), _ptr(state),
                                 state.numel() * state.element_size(), _ptr(parent_out), _ptr(tokens_out),
                                 _ptr(n_nodes_out), _ptr(next_node), _ptr(flags), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_tree_expand")


def spec_tree_expand_multi(draft_rows, max_nodes, topk, max_depth, state, parent_out, tokens_out, n_nodes_out,
                           next_node, req_parent, req_token, req_n, threshold=0.0, flags=None, dev_status=None,
                           stream=None):
    """One multi-row expansion of every sequence's draft tree. draft_rows float32
    [batch][width][vocab]: row j of sequence b is the draft logits of the request listed in
    req_parent[b][j] / req_token[b][j] by the previous call (after spec_tree_init: the root
    alone, in row 0). req_parent / req_token int32 [batch][width], req_n int32 [batch] are
    written with the next call's requests."""
    Bn, W, V = draft_rows.shape
    if draft_rows.dtype != torch.float32 or draft_rows.stride(2) != 1:
        raise ValueError("draft_rows must be float32 with contiguous rows")
    st = load().spec_tree_expand_multi(_ptr(draft_rows), V, int(draft_rows.stride(0)), int(draft_rows.stride(1)), Bn,
                                       int(max_nodes), W, int(topk), int(max_depth), float(threshold), _ptr(state),
                                       state.numel() * state.element_size(), _ptr(parent_out), _ptr(tokens_out),
                                       _ptr(n_nodes_out), _ptr(next_node), _ptr(req_parent), _ptr(req_token),
                                       _ptr(req_n), _ptr(flags), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_tree_expand_multi")



def spec_tree_verify_attn_kv8(q, k_pool, v_pool, kv_scale, page_table, prefix_len, max_prefix, k_tree, v_tree,
                              mask, qo_indptr, max_nodes, out, lse=None, ws=None, sm_scale=0.0, dev_status=None,
                              stream=None):
    """Tree-verify attention over an FP8 cache: k_pool/v_pool uint8 E4M3 codes
    [pages,Hkv,16,128], kv_scale float32 [2,Hkv] (K scales, then V scales); q, k_tree,
    v_tree and out bf16."""
    _need(q, torch.bfloat16, "q")
    for t, what in ((k_tree, "k_tree"), (v_tree, "v_tree"), (out, "out")):
        _need(t, torch.bfloat16, what)
    _need(k_pool, torch.uint8, "k_pool (E4M3 codes)")
    _need(v_pool, torch.uint8, "v_pool (E4M3 codes)")
    _need(kv_scale, torch.float32, "kv_scale")
    T, hq, d = q.shape
    num_pages, hkv, ps, _ = k_pool.shape
    st = load().spec_tree_verify_attn_kv8(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_scale), num_pages, ps, _ptr(page_table), page_table.shape[1],
        _ptr(prefix_len), int(max_prefix), _ptr(k_tree), _ptr(v_tree), _ptr(mask), _ptr(qo_indptr),
        qo_indptr.numel() - 1, T, int(max_nodes), hq, hkv, d, float(sm_scale), _ptr(out), _ptr(lse),
        _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_tree_verify_attn_kv8")


def spec_kv_commit_kv8(k_tree, v_tree, kv_scale, path, accept_len, qo_indptr, page_table, prefix_len, k_pool,
                       v_pool, seq_len_out=None, dev_status=None, stream=None):
    """Commit of bf16 tree K/V rows into an FP8 cache (E4M3 codes of x / scale)."""
    _need(k_tree, torch.bfloat16, "k_tree")
    _need(v_tree, torch.bfloat16, "v_tree")
    _need(k_pool, torch.uint8, "k_pool (E4M3 codes)")
    _need(v_pool, torch.uint8, "v_pool (E4M3 codes)")
    _need(kv_scale, torch.float32, "kv_scale")
    T, hkv, d = k_tree.shape
    num_pages, _, ps, _ = k_pool.shape
    st = load().spec_kv_commit_kv8(
        _ptr(k_tree), _ptr(v_tree), _ptr(kv_scale), _ptr(path), path.shape[1], _ptr(accept_len), _ptr(qo_indptr),
        _ptr(page_table), page_table.shape[1], num_pages, ps, _ptr(prefix_len), _ptr(seq_len_out), _ptr(k_pool),
        _ptr(v_pool), qo_indptr.numel() - 1, T, hkv, d, _ptr(dev_status), _stream(stream))
    return _check(st, "spec_kv_commit_kv8")


def spec_tree_verify_attn_parents(q, k_pool, v_pool, page_table, prefix_len, max_prefix, k_tree, v_tree, parent,
                                  qo_indptr, max_nodes, out, lse=None, ws=None, sm_scale=0.0, dev_status=None,
                                  stream=None):
    """Tree-verify attention with the ancestor bits built in-kernel from the parent array
    (bf16, tensor-core shapes)."""
    _need(q, torch.bfloat16, "q")
    for t, what in ((k_tree, "k_tree"), (v_tree, "v_tree"), (out, "out"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, torch.bfloat16, what)
    _need(parent, torch.int32, "parent")
    T, hq, d = q.shape
    num_pages, hkv, ps, _ = k_pool.shape
    st = load().spec_tree_verify_attn_parents(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), num_pages, ps, _ptr(page_table), page_table.shape[1],
        _ptr(prefix_len), int(max_prefix), _ptr(k_tree), _ptr(v_tree), _ptr(parent), _ptr(qo_indptr),
        qo_indptr.numel() - 1, T, int(max_nodes), hq, hkv, d, float(sm_scale), _ptr(out), _ptr(lse),
        _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _ptr(dev_status), _stream(stream))
    return _check(st, "spec_tree_verify_attn_parents")
