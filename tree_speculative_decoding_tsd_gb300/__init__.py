"""Python binding of ``libtsd.so``, the GB300 tree-speculative-decoding verify step.

Argument marshalling only: every function takes torch CUDA tensors, passes
their device pointers to the C ABI declared in ``include/tsd.h`` (same names),
and raises :class:`TsdError` on a non-OK status.  All arithmetic runs in the
library's CUDA kernels; there is no CPU fallback -- importing this package
fails if the compiled library is missing.

Typical step on one stream::

    ws = workspace(...)                      # caller-owned scratch
    tsd_tree_build(probs, root, D, tree..., ws_build, err)
    tsd_tree_verify_attn(desc, q, kcache, vcache, prefix_len, ktree, vtree,
                         tree.mask, out, lse, ws_verify, err)
    tsd_accept_walk(logits, S, tree..., walk..., ws_walk, err)
    tsd_commit_path(desc, S, ktree, vtree, walk.accept_rows, walk.accept_len,
                    kcache, vcache, prefix_len, err)
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtsd.so")

TSD_OK = 0
TSD_ERR_INVALID_ARG = 1
TSD_ERR_UNSUPPORTED = 2
TSD_ERR_CUDA = 3
TSD_ERR_DEVICE = 4
TSD_ERR_DEVICE_TIMEOUT = 5
TSD_DEV_ERR_CAPACITY = 0x01000000
TSD_DEV_ERR_BAD_TREE = 0x02000000
TSD_DEV_ERR_BAD_PAGE = 0x04000000
TSD_DEV_ERR_TIMEOUT = 0x03000000
TSD_DEV_ERR_MASK = 0x7F000000
TSD_F32 = 0
TSD_BF16 = 1

# every symbol the header declares
EXPORTED = ("tsd_status_string", "tsd_version", "tsd_tree_build_workspace_size",
            "tsd_tree_build", "tsd_tree_build_adaptive", "tsd_tree_build_conditioned",
            "tsd_verify_workspace_size",
            "tsd_tree_verify_attn", "tsd_tree_verify_attn_paged", "tsd_commit_path_paged",
            "tsd_accept_walk_workspace_size", "tsd_accept_walk", "tsd_accept_walk_static",
            "tsd_commit_path")


class TsdError(RuntimeError):
    def __init__(self, func, status):
        self.status = status
        super().__init__(f"{func}: {tsd_status_string(status)} (status {status})")


class tsd_attn_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("R", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
                ("cap", ctypes.c_int), ("dtype", ctypes.c_int), ("v_aliases_k", ctypes.c_int),
                ("scale", ctypes.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtsd.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.tsd_status_string.argtypes = [I]
    lib.tsd_status_string.restype = ctypes.c_char_p
    lib.tsd_version.restype = I
    lib.tsd_tree_build_workspace_size.argtypes = [I, I, I, I]
    lib.tsd_tree_build_workspace_size.restype = Z
    lib.tsd_tree_build.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P, P, P, Z, P, P]
    lib.tsd_tree_build.restype = I
    lib.tsd_tree_build_adaptive.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, Z,
                                            P, P]
    lib.tsd_tree_build_adaptive.restype = I
    lib.tsd_tree_build_conditioned.argtypes = [P, P, P, I, I, I, P, P, P, P, P, P, P, P, P]
    lib.tsd_tree_build_conditioned.restype = I
    lib.tsd_verify_workspace_size.argtypes = [ctypes.POINTER(tsd_attn_desc)]
    lib.tsd_verify_workspace_size.restype = Z
    lib.tsd_tree_verify_attn.argtypes = [ctypes.POINTER(tsd_attn_desc), P, P, P, P, P, P, P, P,
                                         P, P, Z, P, P]
    lib.tsd_tree_verify_attn.restype = I
    lib.tsd_accept_walk_workspace_size.argtypes = [I, I, I]
    lib.tsd_accept_walk_workspace_size.restype = Z
    lib.tsd_accept_walk.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, P, P, Z, P, P]
    lib.tsd_accept_walk.restype = I
    lib.tsd_accept_walk_static.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P]
    lib.tsd_accept_walk_static.restype = I
    lib.tsd_commit_path.argtypes = [ctypes.POINTER(tsd_attn_desc), I, P, P, P, P, P, P, P, P, P]
    lib.tsd_commit_path.restype = I
    lib.tsd_tree_verify_attn_paged.argtypes = [ctypes.POINTER(tsd_attn_desc), P, P, P, P, I, I, I,
                                               P, P, P, P, P, P, P, Z, P, P]
    lib.tsd_tree_verify_attn_paged.restype = I
    lib.tsd_commit_path_paged.argtypes = [ctypes.POINTER(tsd_attn_desc), I, P, P, P, P, P, P, P, I,
                                          I, I, P, P, P]
    lib.tsd_commit_path_paged.restype = I
    return lib


lib = _load()


def tsd_status_string(status: int) -> str:
    return lib.tsd_status_string(int(status)).decode()


def tsd_version() -> int:
    return lib.tsd_version()


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(func, status):
    if status != TSD_OK:
        raise TsdError(func, status)


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def make_desc(B, R, Hq, Hkv, dk, dv, cap, dtype, v_aliases_k, scale) -> tsd_attn_desc:
    if isinstance(dtype, torch.dtype):
        dtype = TSD_BF16 if dtype == torch.bfloat16 else TSD_F32
    return tsd_attn_desc(B, R, Hq, Hkv, dk, dv, cap, dtype, 1 if v_aliases_k else 0, scale)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Caller-owned device scratch of at least nbytes (16-byte aligned)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------ calls --

def tsd_tree_build_workspace_size(B, S, V, k) -> int:
    return lib.tsd_tree_build_workspace_size(B, S, V, k)


def tsd_tree_build(probs, k, D, root_tok, token, parent, depth, score, mask, is_leaf, ws,
                   err=None, stream=None):
    B, S, V = probs.shape
    _check("tsd_tree_build", lib.tsd_tree_build(
        _ptr(probs), B, S, V, k, D, _ptr(root_tok), _ptr(token), _ptr(parent), _ptr(depth),
        _ptr(score), _ptr(mask), _ptr(is_leaf), _ptr(ws), _nbytes(ws), _ptr(err),
        _stream(stream)))


def tsd_tree_build_adaptive(probs, k, D_max, root_tok, cost_d, cost_v, token, parent, depth,
                            score, mask, is_leaf, n_nodes, ws, err=None, stream=None):
    B, S, V = probs.shape
    _check("tsd_tree_build_adaptive", lib.tsd_tree_build_adaptive(
        _ptr(probs), B, S, V, k, D_max, _ptr(root_tok), _ptr(cost_d), _ptr(cost_v), _ptr(token),
        _ptr(parent), _ptr(depth), _ptr(score), _ptr(mask), _ptr(is_leaf), _ptr(n_nodes),
        _ptr(ws), _nbytes(ws), _ptr(err), _stream(stream)))


def tsd_tree_build_conditioned(cand_p, cand_tok, cand_parent, D, root_tok, token, parent, depth,
                               score, mask, is_leaf, err=None, stream=None):
    B, C = cand_p.shape
    _check("tsd_tree_build_conditioned", lib.tsd_tree_build_conditioned(
        _ptr(cand_p), _ptr(cand_tok), _ptr(cand_parent), B, C, D, _ptr(root_tok), _ptr(token),
        _ptr(parent), _ptr(depth), _ptr(score), _ptr(mask), _ptr(is_leaf), _ptr(err),
        _stream(stream)))


def tsd_verify_workspace_size(desc: tsd_attn_desc) -> int:
    return lib.tsd_verify_workspace_size(ctypes.byref(desc))


def tsd_tree_verify_attn(desc, q, kcache, vcache, prefix_len, ktree, vtree, mask, out, lse, ws,
                         err=None, stream=None):
    _check("tsd_tree_verify_attn", lib.tsd_tree_verify_attn(
        ctypes.byref(desc), _ptr(q), _ptr(kcache), _ptr(vcache), _ptr(prefix_len), _ptr(ktree),
        _ptr(vtree), _ptr(mask), _ptr(out), _ptr(lse), _ptr(ws), _nbytes(ws), _ptr(err),
        _stream(stream)))


def tsd_accept_walk_workspace_size(B, D, V) -> int:
    return lib.tsd_accept_walk_workspace_size(B, D, V)


def tsd_accept_walk(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus,
                    chain_id, ws, err=None, stream=None):
    B, R, V = logits.shape
    _check("tsd_accept_walk", lib.tsd_accept_walk(
        _ptr(logits), B, R - 1, S, V, _ptr(token), _ptr(parent), _ptr(mask), _ptr(is_leaf),
        _ptr(tgt), _ptr(accept_len), _ptr(accept_rows), _ptr(bonus), _ptr(chain_id), _ptr(ws),
        _nbytes(ws), _ptr(err), _stream(stream)))


def tsd_accept_walk_static(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows,
                           bonus, chain_id, err=None, stream=None):
    """tsd_accept_walk without a workspace (fixed in-library scratch; see tsd.h)."""
    B, R, V = logits.shape
    _check("tsd_accept_walk_static", lib.tsd_accept_walk_static(
        _ptr(logits), B, R - 1, S, V, _ptr(token), _ptr(parent), _ptr(mask), _ptr(is_leaf),
        _ptr(tgt), _ptr(accept_len), _ptr(accept_rows), _ptr(bonus), _ptr(chain_id), _ptr(err),
        _stream(stream)))


def tsd_tree_verify_attn_paged(desc, q, kpool, vpool, page_table, page_size, prefix_len, ktree,
                               vtree, mask, out, lse, ws, err=None, stream=None):
    """page_table [B][max_pages] int32; pools [num_pages][Hkv][page_size][d]."""
    _check("tsd_tree_verify_attn_paged", lib.tsd_tree_verify_attn_paged(
        ctypes.byref(desc), _ptr(q), _ptr(kpool), _ptr(vpool), _ptr(page_table),
        page_table.shape[1], page_size, kpool.shape[0], _ptr(prefix_len), _ptr(ktree),
        _ptr(vtree), _ptr(mask), _ptr(out), _ptr(lse), _ptr(ws), _nbytes(ws), _ptr(err),
        _stream(stream)))


def tsd_commit_path_paged(desc, S, ktree, vtree, accept_rows, accept_len, kpool, vpool,
                          page_table, page_size, prefix_len, err=None, stream=None):
    _check("tsd_commit_path_paged", lib.tsd_commit_path_paged(
        ctypes.byref(desc), S, _ptr(ktree), _ptr(vtree), _ptr(accept_rows), _ptr(accept_len),
        _ptr(kpool), _ptr(vpool), _ptr(page_table), page_table.shape[1], page_size,
        kpool.shape[0], _ptr(prefix_len), _ptr(err), _stream(stream)))


def tsd_commit_path(desc, S, ktree, vtree, accept_rows, accept_len, kcache, vcache, prefix_len,
                    err=None, stream=None):
    _check("tsd_commit_path", lib.tsd_commit_path(
        ctypes.byref(desc), S, _ptr(ktree), _ptr(vtree), _ptr(accept_rows), _ptr(accept_len),
        _ptr(kcache), _ptr(vcache), _ptr(prefix_len), _ptr(err), _stream(stream)))
