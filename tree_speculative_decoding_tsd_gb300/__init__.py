"""Python binding of ``libtsd.so``, the GB300 tree-speculative-decoding verify step.

Argument marshalling only: every function takes torch CUDA tensors, checks
their element types and shapes, passes their device pointers to the C ABI
declared in ``include/tsd.h`` (same names), and raises :class:`TsdError` on a
non-OK status.  All arithmetic runs in the library's CUDA kernels; there is no
CPU fallback.  The library is loaded on first use (``lib``), so importing the
package, or its input generators in ``workloads``, maps nothing; the first
call fails with ImportError if the compiled library is missing.

Typical step on one stream::

    ws = workspace(...)                      # caller-owned scratch
    tsd_tree_build(probs, root, D, tree..., ws_build, err)
    tsd_tree_verify_attn(desc, q, kcache, vcache, prefix_len, ktree, vtree,
                         tree.mask, out, lse, ws_verify, err)
    tsd_accept_walk(logits, S, tree..., walk..., ws_walk, err)
    tsd_commit_path(desc, S, ktree, vtree, walk.accept_rows, walk.accept_len,
                    kcache, vcache, prefix_len, err)

or the last two as one call, ``tsd_accept_commit`` (the walk's kernel commits
the path it finds).
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
TSD_DEV_ERR_BAD_PROBS = 0x05000000
TSD_DEV_ERR_TIMEOUT = 0x03000000
TSD_DEV_ERR_MASK = 0x7F000000
TSD_F32 = 0
TSD_BF16 = 1
VERIFY_PATHS = {"auto": 0, "generic": 1, "mma": 2, "tc": 3}   # TSD_PATH_* of tsd.h

# every symbol the header declares
EXPORTED = ("tsd_status_string", "tsd_version", "tsd_tree_build_workspace_size",
            "tsd_tree_build", "tsd_tree_build_adaptive", "tsd_tree_build_conditioned",
            "tsd_verify_workspace_size",
            "tsd_tree_verify_attn", "tsd_tree_verify_attn_paged", "tsd_commit_path_paged",
            "tsd_accept_walk_workspace_size", "tsd_accept_walk", "tsd_accept_walk_static",
            "tsd_commit_path", "tsd_accept_commit", "tsd_target_argmax", "tsd_walk_commit",
            "tsd_set_verify_path", "tsd_set_wait_budget")


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
    lib.tsd_accept_commit.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, P,
                                      ctypes.POINTER(tsd_attn_desc), P, P, P, P, P, I, I, I, P,
                                      P, Z, P, P]
    lib.tsd_accept_commit.restype = I
    lib.tsd_target_argmax.argtypes = [P, I, I, I, P, Z, P]
    lib.tsd_target_argmax.restype = I
    lib.tsd_walk_commit.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P,
                                    ctypes.POINTER(tsd_attn_desc), P, P, P, P, P, I, I, I, P, P,
                                    Z, P, P]
    lib.tsd_walk_commit.restype = I
    lib.tsd_set_verify_path.argtypes = [I]
    lib.tsd_set_verify_path.restype = I
    lib.tsd_set_wait_budget.argtypes = [ctypes.c_longlong]
    lib.tsd_set_wait_budget.restype = ctypes.c_longlong
    return lib


_lib = None


def _L():
    """The loaded library (loaded on first use; ImportError if it is not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def __getattr__(name):
    if name == "lib":
        return _L()
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


def tsd_set_verify_path(path) -> int:
    """Force an attention path ("auto", "generic", "mma", "tc" or a TSD_PATH_*
    value) for the verify calls that follow; returns the previous value."""
    code = VERIFY_PATHS[path] if isinstance(path, str) else int(path)
    prev = _L().tsd_set_verify_path(code)
    if prev < 0:
        raise ValueError(f"unknown verify path {path!r}")
    return prev


class verify_path:
    """Context manager: the verify calls inside use the given path."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.prev = tsd_set_verify_path(self.path)
        return self

    def __exit__(self, *exc):
        tsd_set_verify_path(self.prev)
        return False


def tsd_set_wait_budget(cycles: int) -> int:
    """Budget (SM clock cycles) of the tcgen05 verify kernel's pipeline waits
    for the calls that follow; 0 restores the default.  Returns the previous
    setting."""
    if int(cycles) < 0:
        raise ValueError("wait budget must be >= 0")
    return int(_L().tsd_set_wait_budget(int(cycles)))


class wait_budget:
    """Context manager: the verify calls inside use the given wait budget."""

    def __init__(self, cycles):
        self.cycles = cycles

    def __enter__(self):
        self.prev = tsd_set_wait_budget(self.cycles)
        return self

    def __exit__(self, *exc):
        tsd_set_wait_budget(self.prev)
        return False


def tsd_status_string(status: int) -> str:
    return _L().tsd_status_string(int(status)).decode()


def tsd_version() -> int:
    return _L().tsd_version()


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

_I32, _F32, _U8 = torch.int32, torch.float32, torch.uint8
_MASK = (torch.int64,) + ((torch.uint64,) if hasattr(torch, "uint64") else ())


def _t(t, name, dtypes, shape=None):
    """Device pointer of ``t`` after checking its element type and shape
    (None passes through as a NULL pointer)."""
    if t is None:
        return None
    if not isinstance(dtypes, tuple):
        dtypes = (dtypes,)
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: element type {t.dtype}, expected "
                        f"{' or '.join(str(d) for d in dtypes)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return _ptr(t)


def _err(err):
    return _t(err, "err", _I32)


def _tree(B, R, token, parent, depth, score, mask, is_leaf):
    return (_t(token, "token", _I32, (B, R)), _t(parent, "parent", _I32, (B, R)),
            _t(depth, "depth", _I32, (B, R)), _t(score, "score", _F32, (B, R)),
            _t(mask, "mask", _MASK, (B, R)), _t(is_leaf, "is_leaf", _U8, (B, R)))


def _attn_dtype(desc):
    return torch.bfloat16 if desc.dtype == TSD_BF16 else torch.float32


def tsd_tree_build_workspace_size(B, S, V, k) -> int:
    return _L().tsd_tree_build_workspace_size(B, S, V, k)


def tsd_tree_build(probs, k, D, root_tok, token, parent, depth, score, mask, is_leaf, ws,
                   err=None, stream=None):
    B, S, V = probs.shape
    _check("tsd_tree_build", _L().tsd_tree_build(
        _t(probs, "probs", _F32), B, S, V, k, D, _t(root_tok, "root_tok", _I32, (B,)),
        *_tree(B, D + 1, token, parent, depth, score, mask, is_leaf), _ptr(ws), _nbytes(ws),
        _err(err), _stream(stream)))


def tsd_tree_build_adaptive(probs, k, D_max, root_tok, cost_d, cost_v, token, parent, depth,
                            score, mask, is_leaf, n_nodes, ws, err=None, stream=None):
    B, S, V = probs.shape
    _check("tsd_tree_build_adaptive", _L().tsd_tree_build_adaptive(
        _t(probs, "probs", _F32), B, S, V, k, D_max, _t(root_tok, "root_tok", _I32, (B,)),
        _t(cost_d, "cost_d", _F32, (B,)), _t(cost_v, "cost_v", _F32, (B, D_max + 1)),
        *_tree(B, D_max + 1, token, parent, depth, score, mask, is_leaf),
        _t(n_nodes, "n_nodes", _I32, (B,)), _ptr(ws), _nbytes(ws), _err(err), _stream(stream)))


def tsd_tree_build_conditioned(cand_p, cand_tok, cand_parent, D, root_tok, token, parent, depth,
                               score, mask, is_leaf, err=None, stream=None):
    B, C = cand_p.shape
    _check("tsd_tree_build_conditioned", _L().tsd_tree_build_conditioned(
        _t(cand_p, "cand_p", _F32), _t(cand_tok, "cand_tok", _I32, (B, C)),
        _t(cand_parent, "cand_parent", _I32, (B, C)), B, C, D,
        _t(root_tok, "root_tok", _I32, (B,)),
        *_tree(B, D + 1, token, parent, depth, score, mask, is_leaf), _err(err),
        _stream(stream)))


def tsd_verify_workspace_size(desc: tsd_attn_desc) -> int:
    return _L().tsd_verify_workspace_size(ctypes.byref(desc))


def _verify_common(desc, q, prefix_len, ktree, vtree, mask, out, lse):
    d = desc
    dt = _attn_dtype(d)
    alias = bool(d.v_aliases_k)
    return (_t(q, "q", dt, (d.B, d.R, d.Hq, d.dk)), _t(prefix_len, "prefix_len", _I32, (d.B,)),
            _t(ktree, "ktree", dt, (d.B, d.R, d.Hkv, d.dk)),
            None if alias else _t(vtree, "vtree", dt, (d.B, d.R, d.Hkv, d.dv)),
            _t(mask, "mask", _MASK, (d.B, d.R)), _t(out, "out", dt, (d.B, d.R, d.Hq, d.dv)),
            _t(lse, "lse", _F32, (d.B, d.R, d.Hq)))


def tsd_tree_verify_attn(desc, q, kcache, vcache, prefix_len, ktree, vtree, mask, out, lse, ws,
                         err=None, stream=None):
    d = desc
    dt = _attn_dtype(d)
    pq, pl, pkt, pvt, pm, po, pls = _verify_common(d, q, prefix_len, ktree, vtree, mask, out, lse)
    pkc = _t(kcache, "kcache", dt, (d.B, d.Hkv, d.cap, d.dk))
    pvc = None if d.v_aliases_k else _t(vcache, "vcache", dt, (d.B, d.Hkv, d.cap, d.dv))
    _check("tsd_tree_verify_attn", _L().tsd_tree_verify_attn(
        ctypes.byref(d), pq, pkc, pvc, pl, pkt, pvt, pm, po, pls, _ptr(ws), _nbytes(ws),
        _err(err), _stream(stream)))


def tsd_accept_walk_workspace_size(B, D, V) -> int:
    return _L().tsd_accept_walk_workspace_size(B, D, V)


def _walk_args(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus,
               chain_id):
    B, R, V = logits.shape
    return (_t(logits, "logits", _F32), B, R - 1, S, V, _t(token, "token", _I32, (B, R)),
            _t(parent, "parent", _I32, (B, R)), _t(mask, "mask", _MASK, (B, R)),
            _t(is_leaf, "is_leaf", _U8, (B, R)), _t(tgt, "tgt", _I32, (B, R)),
            _t(accept_len, "accept_len", _I32, (B,)),
            _t(accept_rows, "accept_rows", _I32, (B, S + 1)), _t(bonus, "bonus", _I32, (B,)),
            _t(chain_id, "chain_id", _I32, (B,)))


def tsd_accept_walk(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus,
                    chain_id, ws, err=None, stream=None):
    _check("tsd_accept_walk", _L().tsd_accept_walk(
        *_walk_args(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus,
                    chain_id), _ptr(ws), _nbytes(ws), _err(err), _stream(stream)))


def tsd_accept_walk_static(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows,
                           bonus, chain_id, err=None, stream=None):
    """tsd_accept_walk without a workspace (fixed in-library scratch; see tsd.h)."""
    _check("tsd_accept_walk_static", _L().tsd_accept_walk_static(
        *_walk_args(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus,
                    chain_id), _err(err), _stream(stream)))


def tsd_tree_verify_attn_paged(desc, q, kpool, vpool, page_table, page_size, prefix_len, ktree,
                               vtree, mask, out, lse, ws, err=None, stream=None):
    """page_table [B][max_pages] int32; pools [num_pages][Hkv][page_size][d]."""
    d = desc
    dt = _attn_dtype(d)
    pq, pl, pkt, pvt, pm, po, pls = _verify_common(d, q, prefix_len, ktree, vtree, mask, out, lse)
    npg, mp = kpool.shape[0], page_table.shape[1]
    pkp = _t(kpool, "kpool", dt, (npg, d.Hkv, page_size, d.dk))
    pvp = None if d.v_aliases_k else _t(vpool, "vpool", dt, (npg, d.Hkv, page_size, d.dv))
    _check("tsd_tree_verify_attn_paged", _L().tsd_tree_verify_attn_paged(
        ctypes.byref(d), pq, pkp, pvp, _t(page_table, "page_table", _I32, (d.B, mp)), mp,
        page_size, npg, pl, pkt, pvt, pm, po, pls, _ptr(ws), _nbytes(ws), _err(err),
        _stream(stream)))


def _commit_common(desc, S, ktree, vtree, accept_rows, accept_len, prefix_len):
    d = desc
    dt = _attn_dtype(d)
    return (_t(ktree, "ktree", dt, (d.B, d.R, d.Hkv, d.dk)),
            None if d.v_aliases_k else _t(vtree, "vtree", dt, (d.B, d.R, d.Hkv, d.dv)),
            _t(accept_rows, "accept_rows", _I32, (d.B, S + 1)),
            _t(accept_len, "accept_len", _I32, (d.B,)),
            _t(prefix_len, "prefix_len", _I32, (d.B,)))


def tsd_commit_path_paged(desc, S, ktree, vtree, accept_rows, accept_len, kpool, vpool,
                          page_table, page_size, prefix_len, err=None, stream=None):
    d = desc
    dt = _attn_dtype(d)
    pkt, pvt, par, pal, ppl = _commit_common(d, S, ktree, vtree, accept_rows, accept_len,
                                             prefix_len)
    npg, mp = kpool.shape[0], page_table.shape[1]
    pkp = _t(kpool, "kpool", dt, (npg, d.Hkv, page_size, d.dk))
    pvp = None if d.v_aliases_k else _t(vpool, "vpool", dt, (npg, d.Hkv, page_size, d.dv))
    _check("tsd_commit_path_paged", _L().tsd_commit_path_paged(
        ctypes.byref(d), S, pkt, pvt, par, pal, pkp, pvp,
        _t(page_table, "page_table", _I32, (d.B, mp)), mp, page_size, npg, ppl, _err(err),
        _stream(stream)))


def tsd_commit_path(desc, S, ktree, vtree, accept_rows, accept_len, kcache, vcache, prefix_len,
                    err=None, stream=None):
    d = desc
    dt = _attn_dtype(d)
    pkt, pvt, par, pal, ppl = _commit_common(d, S, ktree, vtree, accept_rows, accept_len,
                                             prefix_len)
    pkc = _t(kcache, "kcache", dt, (d.B, d.Hkv, d.cap, d.dk))
    pvc = None if d.v_aliases_k else _t(vcache, "vcache", dt, (d.B, d.Hkv, d.cap, d.dv))
    _check("tsd_commit_path", _L().tsd_commit_path(
        ctypes.byref(d), S, pkt, pvt, par, pal, pkc, pvc, ppl, _err(err), _stream(stream)))


def _commit_targets(d, kcache, vcache, page_table, page_size):
    dt = _attn_dtype(d)
    if page_table is None:
        pkc = _t(kcache, "kcache", dt, (d.B, d.Hkv, d.cap, d.dk))
        pvc = None if d.v_aliases_k else _t(vcache, "vcache", dt, (d.B, d.Hkv, d.cap, d.dv))
        return pkc, pvc, (None, 0, 0, 0)
    npg, mp = kcache.shape[0], page_table.shape[1]
    pkc = _t(kcache, "kpool", dt, (npg, d.Hkv, page_size, d.dk))
    pvc = None if d.v_aliases_k else _t(vcache, "vpool", dt, (npg, d.Hkv, page_size, d.dv))
    return pkc, pvc, (_t(page_table, "page_table", _I32, (d.B, mp)), mp, page_size, npg)


def tsd_target_argmax(logits, ws, stream=None):
    """The argmax part of tsd_accept_commit: per-chunk candidates of every row into ws."""
    B, R, V = logits.shape
    _check("tsd_target_argmax", _L().tsd_target_argmax(
        _t(logits, "logits", _F32), B, R - 1, V, _ptr(ws), _nbytes(ws), _stream(stream)))


def tsd_walk_commit(V, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows, bonus,
                    chain_id, desc, ktree, vtree, kcache, vcache, prefix_len, ws, err=None,
                    stream=None, page_table=None, page_size=0):
    """The rest of tsd_accept_commit, from the candidates tsd_target_argmax left in ws."""
    d = desc
    B, R = token.shape
    if B != d.B or R != d.R:
        raise ValueError("tsd_walk_commit: tree batch / rows do not match desc (B, R)")
    pkt, pvt, _, _, ppl = _commit_common(d, S, ktree, vtree, accept_rows, accept_len, prefix_len)
    pkc, pvc, paging = _commit_targets(d, kcache, vcache, page_table, page_size)
    _check("tsd_walk_commit", _L().tsd_walk_commit(
        B, R - 1, S, V, _t(token, "token", _I32, (B, R)), _t(parent, "parent", _I32, (B, R)),
        _t(mask, "mask", _MASK, (B, R)), _t(is_leaf, "is_leaf", _U8, (B, R)),
        _t(tgt, "tgt", _I32, (B, R)), _t(accept_len, "accept_len", _I32, (B,)),
        _t(accept_rows, "accept_rows", _I32, (B, S + 1)), _t(bonus, "bonus", _I32, (B,)),
        _t(chain_id, "chain_id", _I32, (B,)), ctypes.byref(d), pkt, pvt, pkc, pvc, *paging, ppl,
        _ptr(ws), _nbytes(ws), _err(err), _stream(stream)))


def tsd_accept_commit(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows,
                      bonus, chain_id, desc, ktree, vtree, kcache, vcache, prefix_len, ws,
                      err=None, stream=None, page_table=None, page_size=0):
    """tsd_accept_walk, then the commit of the accepted paths, in one call.

    kcache/vcache are the contiguous cache, or with ``page_table`` [B][max_pages]
    the page pools [num_pages][Hkv][page_size][d] of tsd_commit_path_paged.
    """
    d = desc
    walk = _walk_args(logits, S, token, parent, mask, is_leaf, tgt, accept_len, accept_rows,
                      bonus, chain_id)
    if walk[1] != d.B or walk[2] + 1 != d.R:
        raise ValueError("tsd_accept_commit: logits batch / rows do not match desc (B, R)")
    pkt, pvt, _, _, ppl = _commit_common(d, S, ktree, vtree, accept_rows, accept_len, prefix_len)
    pkc, pvc, paging = _commit_targets(d, kcache, vcache, page_table, page_size)
    _check("tsd_accept_commit", _L().tsd_accept_commit(
        *walk, ctypes.byref(d), pkt, pvt, pkc, pvc, *paging, ppl, _ptr(ws), _nbytes(ws),
        _err(err), _stream(stream)))
