"""Python wrapper of the plain CPU oracle (``tsd_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the benchmark's CPU-baseline leg, never by the library.  It shares no code
with the CUDA path; the two meet only in the seeded input generators.

Every function takes and returns numpy arrays.  Attention inputs may be fp32
or bf16; bf16 arrays are passed as their raw uint16 bit patterns and widened
exactly inside the oracle.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tsd_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with g++ (-O2, no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", "-o", _LIB + ".tmp", _SRC]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def build_command() -> list:
    return ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-pthread", "-o", _LIB, _SRC]


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        _lib.oracle_hardware_threads.restype = I
        _lib.oracle_topk.argtypes = [P, I, I, I, I, P, P, I]
        _lib.oracle_topk.restype = None
        for name in ("oracle_tree_enum", "oracle_tree_beam"):
            f = getattr(_lib, name)
            f.argtypes = [P, P, I, I, I, I, P, P, P, P, P, P, P]
            f.restype = I
        _lib.oracle_verify_attn.argtypes = [I, I, I, I, I, I, I, I, I, ctypes.c_double,
                                            P, P, P, P, P, P, P, I, P, P, P, I]
        _lib.oracle_verify_attn.restype = None
        _lib.oracle_argmax.argtypes = [P, ctypes.c_long, I, P, I]
        _lib.oracle_argmax.restype = None
        _lib.oracle_accept_walk.argtypes = [P, I, I, I, P, P, P, P, P, P, P, P]
        _lib.oracle_accept_walk.restype = I
        _lib.oracle_commit.argtypes = [I, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P]
        _lib.oracle_commit.restype = I
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def hardware_threads() -> int:
    return _load().oracle_hardware_threads()


def topk(probs, k, nthreads=0):
    """probs [B][S][V] fp32 -> (top_p [B][S][k] fp32, top_id [B][S][k] int32)."""
    probs = _c(probs, np.float32)
    B, S, V = probs.shape
    if not 1 <= k <= V:
        raise ValueError("need 1 <= k <= V")
    tp = np.zeros((B, S, k), np.float32)
    ti = np.zeros((B, S, k), np.int32)
    _load().oracle_topk(_p(probs), B, S, V, k, _p(tp), _p(ti), nthreads)
    return tp, ti


def tree(top_p, top_id, D, root_tok, method="enum"):
    """Best-first tree from per-position top-k lists.

    Returns a dict of [B][1+D] arrays: token, parent, depth, score, mask, is_leaf.
    method: "enum" (all paths, the definition) or "beam" (exact level beam).
    """
    top_p = _c(top_p, np.float32)
    top_id = _c(top_id, np.int32)
    B, S, k = top_p.shape
    root_tok = _c(root_tok, np.int32)
    R = D + 1
    out = dict(token=np.zeros((B, R), np.int32), parent=np.zeros((B, R), np.int32),
               depth=np.zeros((B, R), np.int32), score=np.zeros((B, R), np.float32),
               mask=np.zeros((B, R), np.uint64), is_leaf=np.zeros((B, R), np.uint8))
    f = _load().oracle_tree_enum if method == "enum" else _load().oracle_tree_beam
    rc = f(_p(top_p), _p(top_id), B, S, k, D, _p(root_tok), _p(out["token"]),
           _p(out["parent"]), _p(out["depth"]), _p(out["score"]), _p(out["mask"]),
           _p(out["is_leaf"]))
    if rc != 0:
        raise ValueError("oracle tree build rejected the arguments")
    return out


def adaptive_count(scores, cost_d, cost_v):
    """Cost-aware node count ("Cost-Aware Diffusion Draft Trees for Speculative
    Decoding", Method items 1, 3, 4): take the best-first nodes in order and
    keep node n+1 only while it raises (1 + Phi) / (C_d + C_v(n)), Phi being
    the sum of the kept scores; stop at the first node that does not.

    scores: the D_max non-root scores of one request in row (pop) order;
    cost_d: scalar; cost_v: [D_max + 1].  Every step is one fp32 operation,
    in the order the C-ABI header fixes:
      A_0 = 1, A_{n+1} = A_n + s_{n+1}, cost_n = C_d + C_v(n),
      keep n+1 iff (A_{n+1} * cost_n) > (A_n * cost_{n+1}).
    """
    f = np.float32
    A = f(1.0)
    cd = f(cost_d)
    cost = [f(cd + f(c)) for c in np.asarray(cost_v, np.float32)]
    n = 0
    for s in np.asarray(scores, np.float32):
        A1 = f(A + s)
        if not f(A1 * cost[n]) > f(A * cost[n + 1]):
            break
        A = A1
        n += 1
    return n


def tree_adaptive(top_p, top_id, D_max, root_tok, cost_d, cost_v, method="enum"):
    """The best-first tree of tree() with each request's node count chosen by
    adaptive_count; rows past the count are inert padding (token -1, parent 0,
    depth 0, score 0, mask 0, not a leaf) and leaves are recomputed over the
    kept rows.  Returns tree() arrays plus n_nodes [B]."""
    t = tree(top_p, top_id, D_max, root_tok, method)
    cost_d = np.asarray(cost_d, np.float32)
    cost_v = np.asarray(cost_v, np.float32)
    B = t["token"].shape[0]
    n_nodes = np.zeros(B, np.int32)
    for b in range(B):
        n = adaptive_count(t["score"][b, 1:], cost_d[b], cost_v[b])
        n_nodes[b] = n
        t["token"][b, n + 1:] = -1
        t["parent"][b, n + 1:] = 0
        t["depth"][b, n + 1:] = 0
        t["score"][b, n + 1:] = 0.0
        t["mask"][b, n + 1:] = 0
        leaf = np.ones(D_max + 1, np.uint8)
        for r in range(1, n + 1):
            leaf[t["parent"][b, r]] = 0
        leaf[n + 1:] = 0
        t["is_leaf"][b] = leaf
    t["n_nodes"] = n_nodes
    return t


def tree_conditioned(cand_p, cand_tok, cand_parent, D, root_tok):
    """Best-first tree over a forest of parent-conditioned proposals (the V4
    review's toy, "How it works" steps 1-2: each node's children are that
    node's own proposals; the tree keeps the D nodes of highest cumulative
    score; "Cost-Aware Diffusion Draft Trees", Method 2).

    cand_p/cand_tok/cand_parent: [B][C], parents listed first (parent < c, -1
    for a child of the root).  Score: fp32 product along the path in depth
    order.  Rows 1..D: the first D candidates by (score desc, depth asc, index
    asc) among those within depth 65.  A malformed forest (parent out of range,
    probability outside [0, 1], too few candidates) gives a root-only tree with
    padding rows and status 1 for that request.  Returns tree() arrays plus
    "status" [B].
    """
    f = np.float32
    cand_p = np.asarray(cand_p, np.float32)
    cand_tok = np.asarray(cand_tok, np.int32)
    cand_parent = np.asarray(cand_parent, np.int32)
    B, C = cand_p.shape
    R = D + 1
    out = dict(token=np.zeros((B, R), np.int32), parent=np.zeros((B, R), np.int32),
               depth=np.zeros((B, R), np.int32), score=np.zeros((B, R), np.float32),
               mask=np.zeros((B, R), np.uint64), is_leaf=np.zeros((B, R), np.uint8),
               status=np.zeros(B, np.int32))
    for b in range(B):
        sc = [f(0)] * C
        dep = [0] * C
        bad = False
        for c in range(C):
            pp, p = int(cand_parent[b, c]), cand_p[b, c]
            if pp < -1 or pp >= c or not (0.0 <= p <= 1.0):
                bad = True
                break
            sc[c] = f(f(1.0) * p) if pp < 0 else f(sc[pp] * p)
            dep[c] = 1 if pp < 0 else dep[pp] + 1
        order = sorted((c for c in range(C) if not bad and dep[c] <= 65),
                       key=lambda c: (-float(sc[c]), dep[c], c))
        if bad or len(order) < D:
            bad = True
        out["token"][b, 0] = root_tok[b]
        out["parent"][b, 0] = -1
        out["score"][b, 0] = 1.0
        if bad:
            out["status"][b] = 1
            out["token"][b, 1:] = -1
            out["is_leaf"][b, 0] = 1
            continue
        row_of = {}
        masks = [0] * R
        has_child = [False] * R
        for i, c in enumerate(order[:D], start=1):
            row_of[c] = i
            pp = int(cand_parent[b, c])
            pr = 0 if pp < 0 else row_of[pp]   # a kept node's parent is kept earlier
            masks[i] = masks[pr] | (1 << (i - 1))
            has_child[pr] = True
            out["token"][b, i] = cand_tok[b, c]
            out["parent"][b, i] = pr
            out["depth"][b, i] = dep[c]
            out["score"][b, i] = sc[c]
            out["mask"][b, i] = masks[i]
        for i in range(R):
            out["is_leaf"][b, i] = 0 if has_child[i] else 1
    return out


def verify_attn(q, kcache, vcache, prefix_len, ktree, vtree, mask, scale,
                v_aliases_k=False, dv=None, sel=None, nthreads=0):
    """fp64 tree-verify attention.

    Arrays are numpy fp32, or uint16 bit patterns for bf16 (all the same kind).
    q [B][R][Hq][dk]; kcache [B][Hkv][cap][dk]; vcache [B][Hkv][cap][dv];
    ktree [B][R][Hkv][dk]; vtree [B][R][Hkv][dv]; mask [B][R] uint64.
    sel: optional int array [n][3] of (b, r, h).  Returns (out, lse) float64:
    out [n][dv] (or [B][R][Hq][dv] when sel is None), lse [n] (or [B][R][Hq]).
    """
    dtype = 1 if q.dtype == np.uint16 else 0
    npdt = np.uint16 if dtype else np.float32
    q = _c(q, npdt)
    kcache = _c(kcache, npdt)
    ktree = _c(ktree, npdt)
    B, R, Hq, dk = q.shape
    _, Hkv, cap, _ = kcache.shape
    if v_aliases_k:
        dv = dv if dv is not None else dk
        vcache = None
        vtree = None
    else:
        vcache = _c(vcache, npdt)
        vtree = _c(vtree, npdt)
        dv = vcache.shape[3]
    prefix_len = _c(prefix_len, np.int32)
    mask = _c(mask, np.uint64)
    if sel is None:
        n = B * R * Hq
        selp = None
        nsel = 0
    else:
        sel = _c(sel, np.int32).reshape(-1, 3)
        n = sel.shape[0]
        selp = _p(sel)
        nsel = n
    out = np.zeros((n, dv), np.float64)
    lse = np.zeros((n,), np.float64)
    _load().oracle_verify_attn(B, R, Hq, Hkv, dk, dv, cap, dtype, 1 if v_aliases_k else 0,
                               float(scale), _p(q), _p(kcache), _p(vcache), _p(prefix_len),
                               _p(ktree), _p(vtree), _p(mask), nsel, selp, _p(out), _p(lse),
                               nthreads)
    if sel is None:
        return out.reshape(B, R, Hq, dv), lse.reshape(B, R, Hq)
    return out, lse


def argmax(logits, nthreads=0):
    """logits [..., V] fp32 -> int32 [...] (ties to the lowest id)."""
    logits = _c(logits, np.float32)
    V = logits.shape[-1]
    rows = logits.size // V
    out = np.zeros(rows, np.int32)
    _load().oracle_argmax(_p(logits), rows, V, _p(out), nthreads)
    return out.reshape(logits.shape[:-1])


def accept_walk(tgt, tree_arrays, S):
    """Greedy walk.  tgt [B][R] int32; tree_arrays as returned by tree().

    Returns dict accept_len [B], accept_rows [B][S+1], bonus [B], chain_id [B]
    and status (0 ok, 1 malformed tree seen).
    """
    tgt = _c(tgt, np.int32)
    B, R = tgt.shape
    out = dict(accept_len=np.zeros(B, np.int32), accept_rows=np.zeros((B, S + 1), np.int32),
               bonus=np.zeros(B, np.int32), chain_id=np.zeros(B, np.int32))
    st = _load().oracle_accept_walk(
        _p(tgt), B, R, S, _p(_c(tree_arrays["token"], np.int32)),
        _p(_c(tree_arrays["parent"], np.int32)), _p(_c(tree_arrays["mask"], np.uint64)),
        _p(_c(tree_arrays["is_leaf"], np.uint8)), _p(out["accept_len"]),
        _p(out["accept_rows"]), _p(out["bonus"]), _p(out["chain_id"]))
    out["status"] = st
    return out


def commit(ktree, vtree, accept_rows, accept_len, kcache, vcache, prefix_len, S,
           v_aliases_k=False):
    """Byte-copy commit, in place on kcache/vcache/prefix_len (numpy arrays).

    Returns the number of requests skipped for lack of capacity.
    """
    for a in (kcache, prefix_len) + (() if v_aliases_k else (vcache,)):
        assert a.flags["C_CONTIGUOUS"]
    ktree = np.ascontiguousarray(ktree)
    B, R, Hkv, dk = ktree.shape
    cap = kcache.shape[2]
    dv = dk if v_aliases_k else vcache.shape[3]
    if not v_aliases_k:
        vtree = np.ascontiguousarray(vtree)
    eb = ktree.dtype.itemsize
    return _load().oracle_commit(B, R, Hkv, dk, dv, cap, S, eb, 1 if v_aliases_k else 0,
                                 _p(ktree), None if v_aliases_k else _p(vtree),
                                 _p(_c(accept_rows, np.int32)), _p(_c(accept_len, np.int32)),
                                 _p(kcache), None if v_aliases_k else _p(vcache),
                                 _p(prefix_len))
