"""Tree-verify step of tree speculative decoding on GB300 (sm_103a).

A thin ctypes binding over libtreeverify.so, whose C ABI is declared in
include/tree_verify.h (the verify step), include/tree_expand.h (dynamic
draft-tree expansion), include/tree_lm_head.h (fused lm_head + argmax) and
include/tree_rope.h (tree-position RoPE and the K/V scatter).  Every function here only marshals arguments (torch
tensors or raw device addresses, a stream) and raises on a non-zero status;
all work happens in the library's CUDA kernels.  There is no CPU fallback:
calling into a library that was not built raises ``LibraryNotBuilt``.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "TvDesc", "TvPlan", "TreeVerifyError", "LibraryNotBuilt", "F32", "BF16", "DEV_BITS",
    "lib", "make_desc", "tv_workspace_size", "tv_attn_plan", "tv_status_string", "tv_version",
    "tv_build_tree_mask", "tree_verify_attn", "tv_attn_partials", "tv_attn_merge", "tree_accept_commit",
    "tree_accept_commit_sampled", "TvExpandDesc", "make_expand_desc", "tv_expand_workspace_size",
    "tv_expand_steps", "tv_tree_expand_step", "TvLmHeadDesc", "make_lmhead_desc", "tv_lm_head_workspace_size",
    "tv_lm_head_argmax", "tv_tree_rope_scatter", "tree_accept_commit_argmax", "tv_check_bounded_wait",
]

F32, BF16 = 0, 1
DEV_BITS = {1: "BAD_TREE", 2: "BAD_OFFSETS", 4: "BAD_PREFIX", 8: "BAD_PAGE", 16: "CAPACITY", 32: "TIMEOUT",
            64: "BAD_LOGITS", 128: "BAD_STEP"}
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtreeverify.so")


class LibraryNotBuilt(RuntimeError):
    pass


class TreeVerifyError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {tv_status_string(code)} ({code})")


class TvDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32), ("out_f32", ctypes.c_int32),
        ("scale", ctypes.c_float), ("max_nodes", ctypes.c_int32), ("total_rows", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("capacity", ctypes.c_int64), ("num_pages", ctypes.c_int64),
        ("max_prefix", ctypes.c_int64),
    ]


class TvPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kernel", "num_splits", "chunk", "row_tiles", "rows_per_tile", "grid_ctas")]


class TvExpandDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("batch", "vocab", "top_k", "width", "max_nodes", "max_depth", "logits_dtype")]


class TvLmHeadDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("rows", "hidden", "vocab")]


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIG = {
    "tv_workspace_size": [ctypes.POINTER(TvDesc), _I, ctypes.POINTER(ctypes.c_size_t)],
    "tv_attn_plan": [ctypes.POINTER(TvDesc), ctypes.POINTER(TvPlan)],
    "tv_build_tree_mask": [ctypes.POINTER(TvDesc), _P, _P, _P, _P, _P, _P],
    "tree_verify_attn": [ctypes.POINTER(TvDesc)] + [_P] * 11 + [ctypes.c_size_t, _P, _P],
    "tv_attn_partials": [ctypes.POINTER(TvDesc)] + [_P] * 10 + [ctypes.c_size_t, _P, _P],
    "tv_attn_merge": [ctypes.POINTER(TvDesc), _P, _P, _P, _P, ctypes.c_size_t, _P, _P],
    "tree_accept_commit": [ctypes.POINTER(TvDesc), _I, _I] + [_P] * 15 + [ctypes.c_size_t, _P, _P],
    "tree_accept_commit_sampled": [ctypes.POINTER(TvDesc), _I, _I, _P, ctypes.c_float, ctypes.c_uint64,
                                   ctypes.c_uint64] + [_P] * 14 + [ctypes.c_size_t, _P, _P],
    "tv_expand_workspace_size": [ctypes.POINTER(TvExpandDesc), ctypes.POINTER(ctypes.c_size_t)],
    "tv_expand_steps": [ctypes.POINTER(TvExpandDesc), ctypes.POINTER(ctypes.c_int32)],
    "tv_tree_expand_step": [ctypes.POINTER(TvExpandDesc), _I, _P, ctypes.c_int64] + [_P] * 9
                           + [ctypes.c_size_t, _P, _P],
    "tv_lm_head_workspace_size": [ctypes.POINTER(TvLmHeadDesc), ctypes.POINTER(ctypes.c_size_t)],
    "tv_lm_head_argmax": [ctypes.POINTER(TvLmHeadDesc)] + [_P] * 5 + [ctypes.c_size_t, _P, _P],
    "tv_tree_rope_scatter": [ctypes.POINTER(TvDesc), ctypes.c_double] + [_P] * 11,
    "tree_accept_commit_argmax": [ctypes.POINTER(TvDesc)] + [_P] * 15,
    "tv_check_bounded_wait": [ctypes.c_int64, _P, _P],
}


def lib(path: str = LIB_PATH):
    """The loaded library (loaded on first use)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(path):
            raise LibraryNotBuilt(
                f"{path} is missing: build it with speculative_decoding_tree_gb300._build.build() "
                "(the tree-verify step has no CPU fallback)")
        L = ctypes.CDLL(path)
        for name, args in _SIG.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.tv_status_string.argtypes = [ctypes.c_int]
        L.tv_status_string.restype = ctypes.c_char_p
        L.tv_version.argtypes = []
        L.tv_version.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc, where):
    if rc != 0:
        raise TreeVerifyError(rc, where)


def make_desc(*, batch, num_q_heads, num_kv_heads, head_dim, dtype, max_nodes, total_rows, capacity,
              max_prefix, page_size=0, num_pages=0, out_f32=0, scale=0.0) -> TvDesc:
    return TvDesc(batch, num_q_heads, num_kv_heads, head_dim, dtype, out_f32, scale, max_nodes, total_rows,
                  page_size, capacity, num_pages, max_prefix)


def tv_status_string(code: int) -> str:
    return lib().tv_status_string(int(code)).decode()


def tv_version() -> str:
    return lib().tv_version().decode()


def tv_workspace_size(desc: TvDesc, vocab: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().tv_workspace_size(ctypes.byref(desc), int(vocab), ctypes.byref(n)), "tv_workspace_size")
    return n.value


def tv_attn_plan(desc: TvDesc) -> dict:
    p = TvPlan()
    _check(lib().tv_attn_plan(ctypes.byref(desc), ctypes.byref(p)), "tv_attn_plan")
    return {name: getattr(p, name) for name, _ in TvPlan._fields_}


def tv_build_tree_mask(desc, parents, node_offsets, anc, depth, status, stream=None):
    _check(lib().tv_build_tree_mask(ctypes.byref(desc), _ptr(parents), _ptr(node_offsets), _ptr(anc),
                                    _ptr(depth), _ptr(status), _stream(stream)), "tv_build_tree_mask")


def tree_verify_attn(desc, q, k_cache, v_cache, page_table, prefix_len, node_offsets, k_tree, v_tree, anc, out,
                     workspace, workspace_bytes, status, stream=None):
    _check(lib().tree_verify_attn(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                  _ptr(prefix_len), _ptr(node_offsets), _ptr(k_tree), _ptr(v_tree), _ptr(anc),
                                  _ptr(out), _ptr(workspace), int(workspace_bytes), _ptr(status),
                                  _stream(stream)), "tree_verify_attn")


def tv_attn_partials(desc, q, k_cache, v_cache, page_table, prefix_len, node_offsets, k_tree, v_tree, anc,
                     workspace, workspace_bytes, status, stream=None):
    _check(lib().tv_attn_partials(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                  _ptr(prefix_len), _ptr(node_offsets), _ptr(k_tree), _ptr(v_tree), _ptr(anc),
                                  _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream)),
           "tv_attn_partials")


def tv_attn_merge(desc, prefix_len, node_offsets, out, workspace, workspace_bytes, status, stream=None):
    _check(lib().tv_attn_merge(ctypes.byref(desc), _ptr(prefix_len), _ptr(node_offsets), _ptr(out),
                               _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream)),
           "tv_attn_merge")


def tree_accept_commit(desc, vocab, logits_dtype, logits, draft_tokens, parents, node_offsets, k_tree, v_tree,
                       k_cache, v_cache, page_table, prefix_len, argmax, accept_len, path, tokens, workspace,
                       workspace_bytes, status, stream=None):
    _check(lib().tree_accept_commit(ctypes.byref(desc), int(vocab), int(logits_dtype), _ptr(logits),
                                    _ptr(draft_tokens), _ptr(parents), _ptr(node_offsets), _ptr(k_tree),
                                    _ptr(v_tree), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
                                    _ptr(prefix_len), _ptr(argmax), _ptr(accept_len), _ptr(path), _ptr(tokens),
                                    _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream)),
           "tree_accept_commit")


def tree_accept_commit_sampled(desc, vocab, logits_dtype, logits, temperature, seed, offset, draft_tokens, parents,
                               node_offsets, k_tree, v_tree, k_cache, v_cache, page_table, prefix_len, sampled,
                               accept_len, path, tokens, workspace, workspace_bytes, status, stream=None):
    _check(lib().tree_accept_commit_sampled(ctypes.byref(desc), int(vocab), int(logits_dtype), _ptr(logits),
                                            float(temperature), int(seed) & (2 ** 64 - 1),
                                            int(offset) & (2 ** 64 - 1), _ptr(draft_tokens), _ptr(parents),
                                            _ptr(node_offsets), _ptr(k_tree), _ptr(v_tree), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(page_table), _ptr(prefix_len), _ptr(sampled),
                                            _ptr(accept_len), _ptr(path), _ptr(tokens), _ptr(workspace),
                                            int(workspace_bytes), _ptr(status), _stream(stream)),
           "tree_accept_commit_sampled")


def make_expand_desc(*, batch, vocab, top_k, width, max_nodes, max_depth, logits_dtype) -> TvExpandDesc:
    return TvExpandDesc(batch, vocab, top_k, width, max_nodes, max_depth, logits_dtype)


def tv_expand_workspace_size(desc: TvExpandDesc) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().tv_expand_workspace_size(ctypes.byref(desc), ctypes.byref(n)), "tv_expand_workspace_size")
    return n.value


def tv_expand_steps(desc: TvExpandDesc) -> int:
    n = ctypes.c_int32(0)
    _check(lib().tv_expand_steps(ctypes.byref(desc), ctypes.byref(n)), "tv_expand_steps")
    return n.value


def tv_tree_expand_step(desc, step, logits, seq_stride, root_tokens, token_map, tokens, parents, depths, cum,
                        n_nodes, expand_count, workspace, workspace_bytes, status, stream=None):
    _check(lib().tv_tree_expand_step(ctypes.byref(desc), int(step), _ptr(logits), int(seq_stride),
                                     _ptr(root_tokens), _ptr(token_map), _ptr(tokens), _ptr(parents), _ptr(depths),
                                     _ptr(cum), _ptr(n_nodes), _ptr(expand_count), _ptr(workspace),
                                     int(workspace_bytes), _ptr(status), _stream(stream)), "tv_tree_expand_step")


def make_lmhead_desc(*, rows, hidden, vocab) -> TvLmHeadDesc:
    return TvLmHeadDesc(rows, hidden, vocab)


def tv_lm_head_workspace_size(desc: TvLmHeadDesc) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().tv_lm_head_workspace_size(ctypes.byref(desc), ctypes.byref(n)), "tv_lm_head_workspace_size")
    return n.value


def tv_lm_head_argmax(desc, hidden, weight, argmax, max_logit, workspace, workspace_bytes, status, stream=None):
    _check(lib().tv_lm_head_argmax(ctypes.byref(desc), _ptr(hidden), _ptr(weight), _ptr(argmax), _ptr(max_logit),
                                   _ptr(workspace), int(workspace_bytes), _ptr(status), _stream(stream)),
           "tv_lm_head_argmax")


def tv_tree_rope_scatter(desc, theta, q_in, k_in, v_in, prefix_len, node_offsets, depth, q_out, k_tree, v_tree,
                         status, stream=None):
    _check(lib().tv_tree_rope_scatter(ctypes.byref(desc), float(theta), _ptr(q_in), _ptr(k_in), _ptr(v_in),
                                      _ptr(prefix_len), _ptr(node_offsets), _ptr(depth), _ptr(q_out), _ptr(k_tree),
                                      _ptr(v_tree), _ptr(status), _stream(stream)), "tv_tree_rope_scatter")


def tree_accept_commit_argmax(desc, argmax, draft_tokens, parents, node_offsets, k_tree, v_tree, k_cache, v_cache,
                              page_table, prefix_len, accept_len, path, tokens, status, stream=None):
    _check(lib().tree_accept_commit_argmax(ctypes.byref(desc), _ptr(argmax), _ptr(draft_tokens), _ptr(parents),
                                           _ptr(node_offsets), _ptr(k_tree), _ptr(v_tree), _ptr(k_cache),
                                           _ptr(v_cache), _ptr(page_table), _ptr(prefix_len), _ptr(accept_len),
                                           _ptr(path), _ptr(tokens), _ptr(status), _stream(stream)),
           "tree_accept_commit_argmax")


def tv_check_bounded_wait(limit_ns, status, stream=None):
    _check(lib().tv_check_bounded_wait(int(limit_ns), _ptr(status), _stream(stream)), "tv_check_bounded_wait")
