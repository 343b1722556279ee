"""CPU checks of the C-ABI library: it loads, exports every function that
include/tsd.h declares, and rejects invalid arguments on the host before any
CUDA call (no GPU needed: the rejected calls never launch)."""

import ctypes
import os
import re

import pytest

import tree_speculative_decoding_tsd_gb300 as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "tsd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tsd_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_four_calls():
    names = _declared_functions()
    for n in ("tsd_tree_build", "tsd_tree_verify_attn", "tsd_accept_walk", "tsd_commit_path"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(T.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(T.EXPORTED)


def test_status_strings_and_version():
    assert T.tsd_status_string(T.TSD_OK) == "ok"
    for s in range(1, 6):
        assert T.tsd_status_string(s) != "unknown status"
    assert T.tsd_status_string(99) == "unknown status"
    assert T.tsd_version() >= 100


# fake, 16-byte-aligned addresses: validation must reject before touching them
A = ctypes.c_void_p(0x10000)
U = ctypes.c_void_p(0x10004)   # misaligned
N = None


def _build(B=1, S=3, V=32, k=2, D=4, probs=A, ws=A, ws_bytes=1 << 20, out=A):
    return T.lib.tsd_tree_build(probs, B, S, V, k, D, A, out, A, A, A, A, A, ws, ws_bytes, A, N)


@pytest.mark.parametrize("kw", [dict(B=0), dict(S=0), dict(S=17), dict(k=0), dict(k=33),
                                dict(V=1, k=2), dict(D=0), dict(D=65), dict(S=2, k=2, D=7),
                                dict(probs=N), dict(probs=U), dict(out=N), dict(ws=N),
                                dict(ws_bytes=0)])
def test_tree_build_rejects(kw):
    assert _build(**kw) == T.TSD_ERR_INVALID_ARG


def test_tree_build_budget_limit_is_sum_of_levels():
    # S=2, k=2 gives 2 + 4 = 6 possible nodes: D=6 passes validation (the launch
    # then fails without a GPU, or succeeds with one), D=7 does not
    assert _build(S=2, k=2, D=7) == T.TSD_ERR_INVALID_ARG
    assert T.tsd_tree_build_workspace_size(1, 2, 32, 2) > 0


def _desc(**kw):
    base = dict(B=2, R=5, Hq=4, Hkv=2, dk=128, dv=128, cap=64, dtype=T.TSD_BF16,
                v_aliases_k=0, scale=0.088)
    base.update(kw)
    return T.tsd_attn_desc(**base)


@pytest.mark.parametrize("kw", [dict(B=0), dict(R=0), dict(R=66), dict(Hq=3), dict(Hkv=0),
                                dict(dk=96, dv=96), dict(dk=128, dv=64), dict(dtype=7),
                                dict(scale=0.0), dict(scale=float("nan")), dict(cap=0),
                                dict(v_aliases_k=1)])
def test_verify_rejects_bad_descriptors(kw):
    d = _desc(**kw)
    assert T.lib.tsd_verify_workspace_size(ctypes.byref(d)) == 0
    st = T.lib.tsd_tree_verify_attn(ctypes.byref(d), A, A, A, A, A, A, A, A, A, A, 1 << 30, N, N)
    assert st == T.TSD_ERR_INVALID_ARG


@pytest.mark.parametrize("which", range(9))
def test_verify_rejects_bad_pointers(which):
    d = _desc()
    ptrs = [A] * 9
    ptrs[which] = U
    st = T.lib.tsd_tree_verify_attn(ctypes.byref(d), *ptrs, A, 1 << 30, N, N)
    assert st == T.TSD_ERR_INVALID_ARG


def test_verify_latent_descriptor_is_accepted_and_v_pointers_optional():
    d = _desc(Hq=128, Hkv=1, dk=576, dv=512, v_aliases_k=1)
    assert T.lib.tsd_verify_workspace_size(ctypes.byref(d)) >= 0
    # too-small workspace is rejected when one is needed
    need = T.lib.tsd_verify_workspace_size(ctypes.byref(d))
    if need > 0:
        st = T.lib.tsd_tree_verify_attn(ctypes.byref(d), A, A, N, A, A, N, A, A, A, A, need - 1,
                                        N, N)
        assert st == T.TSD_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [dict(B=0), dict(D=0), dict(D=65), dict(S=0), dict(S=17),
                                  dict(logits=N), dict(logits=U), dict(ws_bytes=0)])
def test_accept_walk_rejects(args):
    kw = dict(B=2, D=4, S=3, V=32, logits=A, ws_bytes=1 << 20)
    kw.update(args)
    st = T.lib.tsd_accept_walk(kw["logits"], kw["B"], kw["D"], kw["S"], kw["V"], A, A, A, A, N,
                               A, A, A, A, A, kw["ws_bytes"], N, N)
    assert st == T.TSD_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [dict(S=0), dict(S=17), dict(kt=N), dict(kc=U), dict(dk=3),
                                  dict(vt=N), dict(plen=N)])
def test_commit_rejects(args):
    kw = dict(S=3, kt=A, vt=A, kc=A, vc=A, plen=A, dk=128)
    kw.update(args)
    d = _desc(dk=kw["dk"], dv=kw["dk"])
    st = T.lib.tsd_commit_path(ctypes.byref(d), kw["S"], kw["kt"], kw["vt"], A, A, kw["kc"],
                               kw["vc"], kw["plen"], N, N)
    assert st == T.TSD_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [dict(), dict(B=3), dict(D=5), dict(S=0), dict(S=17),
                                  dict(logits=N), dict(ws_bytes=0), dict(kt=N), dict(kc=U),
                                  dict(plen=N), dict(page_size=-1), dict(page_size=128),
                                  dict(page_size=128, max_pages=1, table=A, num_pages=4)])
def test_accept_commit_rejects(args):
    """The walk's checks, the commit's, and the two agreeing on (B, D + 1)."""
    kw = dict(B=2, D=4, S=3, V=32, logits=A, ws_bytes=1 << 20, kt=A, kc=A, plen=A,
              table=N, max_pages=0, page_size=0, num_pages=0, dk=128)
    kw.update(args)
    d = _desc(dk=kw["dk"], dv=kw["dk"], cap=64)
    if not args:
        d.R = 9     # desc R != D + 1
    st = T.lib.tsd_accept_commit(kw["logits"], kw["B"], kw["D"], kw["S"], kw["V"], A, A, A, A, N,
                                 A, A, A, A, ctypes.byref(d), kw["kt"], A, kw["kc"], A,
                                 kw["table"], kw["max_pages"], kw["page_size"], kw["num_pages"],
                                 kw["plen"], A, kw["ws_bytes"], N, N)
    assert st == T.TSD_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [dict(B=0), dict(D=65), dict(V=0), dict(logits=N), dict(logits=U),
                                  dict(ws=N), dict(ws_bytes=0)])
def test_target_argmax_rejects(args):
    kw = dict(B=2, D=4, V=32, logits=A, ws=A, ws_bytes=1 << 20)
    kw.update(args)
    st = T.lib.tsd_target_argmax(kw["logits"], kw["B"], kw["D"], kw["V"], kw["ws"], kw["ws_bytes"],
                                 N)
    assert st == T.TSD_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [dict(), dict(B=3), dict(S=17), dict(V=0), dict(tok=N),
                                  dict(kt=N), dict(ws_bytes=0), dict(page_size=-1)])
def test_walk_commit_rejects(args):
    kw = dict(B=2, D=4, S=3, V=32, tok=A, kt=A, ws_bytes=1 << 20, page_size=0)
    kw.update(args)
    d = _desc(cap=64)
    if not args:
        d.R = 9     # desc R != D + 1
    st = T.lib.tsd_walk_commit(kw["B"], kw["D"], kw["S"], kw["V"], kw["tok"], A, A, A, N, A, A, A,
                               A, ctypes.byref(d), kw["kt"], A, A, A, N, 0, kw["page_size"], 0, A,
                               A, kw["ws_bytes"], N, N)
    assert st == T.TSD_ERR_INVALID_ARG


def test_workspace_sizes_are_deterministic_and_scale():
    a = T.tsd_tree_build_workspace_size(32, 7, 151936, 8)
    assert a == T.tsd_tree_build_workspace_size(32, 7, 151936, 8) and a > 0
    b = T.tsd_accept_walk_workspace_size(32, 32, 151936)
    assert b >= 32 * 33 * 8
    assert T.tsd_tree_build_workspace_size(0, 7, 100, 8) == 0


# (rows, V, chunks per row) of the vocabulary scans, read back from the
# workspace sizes (one k-candidate list per chunk).  Chunks minimise
# (waves of resident CTAs) x (chunk length + a fixed per-chunk cost) on 152
# SMs (4 top-k or 8 argmax CTAs each), and a row's lists hold at most 256
# candidates: e.g. 7 top-k rows take 32 chunks of k=8 (one wave of 224 CTAs),
# 224 rows take 5 (1120 CTAs, two waves of 608), 64 rows with k=10 take 9
# (576 CTAs, one wave), 17 argmax rows take 66.
@pytest.mark.parametrize("B,S,V,k,nchunk", [(1, 7, 151936, 8, 32), (32, 7, 151936, 8, 5),
                                            (8, 8, 151936, 10, 9), (1, 3, 32, 2, 1)])
def test_topk_scan_geometry(B, S, V, k, nchunk):
    ws = T.tsd_tree_build_workspace_size(B, S, V, k)
    assert ws == B * S * nchunk * k * 8
    assert nchunk * k <= 256


@pytest.mark.parametrize("B,D,V,nchunk", [(1, 16, 151936, 66), (32, 32, 151936, 8)])
def test_argmax_scan_geometry(B, D, V, nchunk):
    assert T.tsd_accept_walk_workspace_size(B, D, V) == B * (D + 1) * nchunk * 8


@pytest.mark.parametrize("args", [dict(page_size=64), dict(page_size=100), dict(max_pages=3),
                                  dict(table=N), dict(table=U), dict(num_pages=0)])
def test_paged_calls_reject(args):
    kw = dict(page_size=128, max_pages=4, num_pages=8, table=A)
    kw.update(args)
    d = _desc(cap=512)
    st = T.lib.tsd_tree_verify_attn_paged(ctypes.byref(d), A, A, A, kw["table"], kw["max_pages"],
                                          kw["page_size"], kw["num_pages"], A, A, A, A, A, A, A,
                                          1 << 30, N, N)
    assert st == T.TSD_ERR_INVALID_ARG
    # every case here also fails the commit's checks (capacity != max_pages *
    # page_size, or a bad table pointer, or no pages), so nothing is launched
    st = T.lib.tsd_commit_path_paged(ctypes.byref(d), 3, A, A, A, A, A, A, kw["table"],
                                     kw["max_pages"], kw["page_size"], kw["num_pages"], A, N, N)
    assert st == T.TSD_ERR_INVALID_ARG
