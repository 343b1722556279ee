"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the pages'
worked examples (tests/golden), textbook special cases computed by a different
formulation (dense masked softmax in numpy), library routines (numpy sort and
argmax), brute force over tiny inputs, closed forms and invariants.
"""

import itertools

import numpy as np
import pytest

import oracle
from tree_speculative_decoding_tsd_gb300 import workloads as W
from tests.conftest import load_golden

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ helpers --

def _toy_probs(g):
    return np.array([[g["p1"], g["p2"]]], np.float32)            # [1][2][3]


def _dspark_probs(g):
    V, S = g["V"][0], g["S"][0]
    p = np.full((1, S, V), 0.0625, np.float32)
    for s, tok in enumerate(g["top"]):
        p[0, s, tok] = 0.5
    return p


def _textbook_attention(q, keys, values, scale):
    """One query over an explicit key list: dense softmax(q K^T) V in float64."""
    s = scale * (keys.astype(np.float64) @ q.astype(np.float64))
    w = np.exp(s - s.max())
    return (w[:, None] * values.astype(np.float64)).sum(0) / w.sum(), s.max() + np.log(w.sum())


def _random_attn_inputs(B, R, Hq, Hkv, d, cap, P, rng=RNG):
    q = rng.standard_normal((B, R, Hq, d)).astype(np.float32)
    kc = rng.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    vc = rng.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    kt = rng.standard_normal((B, R, Hkv, d)).astype(np.float32)
    vt = rng.standard_normal((B, R, Hkv, d)).astype(np.float32)
    return q, kc, vc, np.array(P, np.int32), kt, vt


def _random_tree(B, S, k, D, V=50, quantize=None, rng=RNG):
    logits = rng.standard_normal((B, S, V)) * 2.0
    p = np.exp(logits - logits.max(-1, keepdims=True))
    p = p / p.sum(-1, keepdims=True)
    if quantize:
        p = np.round(p * quantize) / quantize                  # force ties
    probs = p.astype(np.float32)
    root = rng.integers(0, V, B).astype(np.int32)
    tp, ti = oracle.topk(probs, k)
    return probs, tp, ti, root


# ---------------------------------------------------------- worked examples --

def test_toy_tree_matches_page_example():
    g = load_golden("toy_tree.txt")
    tp, ti = oracle.topk(_toy_probs(g), g["k"][0])
    for method in ("enum", "beam"):
        t = oracle.tree(tp, ti, g["D"][0], np.array(g["root"], np.int32), method=method)
        for key in ("token", "parent", "depth", "is_leaf"):
            np.testing.assert_array_equal(t[key][0], g[key], err_msg=f"{method}:{key}")
        np.testing.assert_array_equal(t["score"][0], np.array(g["score"], np.float32))
        np.testing.assert_array_equal(t["mask"][0], np.array(g["mask"], np.uint64))


def test_toy_visibility_matches_page_example():
    """Each row's output equals plain attention over prefix + the page's visible rows."""
    g = load_golden("toy_tree.txt")
    R, Hq, Hkv, d, P, cap = 4, 2, 1, 16, 5, 8
    q, kc, vc, pl, kt, vt = _random_attn_inputs(1, R, Hq, Hkv, d, cap, [P])
    mask = np.array([g["mask"]], np.uint64)
    scale = 0.25
    out, lse = oracle.verify_attn(q, kc, vc, pl, kt, vt, mask, scale)
    for r in range(R):
        vis = g[f"visible{r}"]
        for h in range(Hq):
            keys = np.concatenate([kc[0, 0, :P], kt[0, vis, 0]])
            vals = np.concatenate([vc[0, 0, :P], vt[0, vis, 0]])
            o, l = _textbook_attention(q[0, r, h], keys, vals, scale)
            np.testing.assert_allclose(out[0, r, h], o, rtol=0, atol=1e-12)
            assert abs(lse[0, r, h] - l) < 1e-12


def test_toy_walk_and_commit_match_page_example():
    g = load_golden("toy_tree.txt")
    tp, ti = oracle.topk(_toy_probs(g), 2)
    t = oracle.tree(tp, ti, 3, np.array([0], np.int32))
    w = oracle.accept_walk(np.array([g["tgt"]], np.int32), t, g["S"][0])
    assert w["status"] == 0
    assert w["accept_len"][0] == g["accept_len"][0]
    np.testing.assert_array_equal(w["accept_rows"][0], g["accept_rows"])
    assert w["bonus"][0] == g["bonus"][0]
    assert w["chain_id"][0] == g["chain_id"][0]
    # the accepted chain is the page's A-C chain: rows of chain2
    L = w["accept_len"][0]
    assert list(w["accept_rows"][0][:L + 1]) == g["chain2"]
    # commit: only rows 0 and 2 (A, C) land in the cache, after the prefix
    Hkv, d, P, cap = 1, 8, 3, 8
    kt = RNG.standard_normal((1, 4, Hkv, d)).astype(np.float32)
    vt = RNG.standard_normal((1, 4, Hkv, d)).astype(np.float32)
    kc = RNG.standard_normal((1, Hkv, cap, d)).astype(np.float32)
    vc = RNG.standard_normal((1, Hkv, cap, d)).astype(np.float32)
    kc0, vc0 = kc.copy(), vc.copy()
    pl = np.array([P], np.int32)
    assert oracle.commit(kt, vt, w["accept_rows"], w["accept_len"], kc, vc, pl, 2) == 0
    assert pl[0] == P + 2
    np.testing.assert_array_equal(kc[0, 0, P:P + 2], kt[0, [0, 2], 0])
    np.testing.assert_array_equal(vc[0, 0, P:P + 2], vt[0, [0, 2], 0])
    np.testing.assert_array_equal(kc[0, 0, :P], kc0[0, 0, :P])
    np.testing.assert_array_equal(kc[0, 0, P + 2:], kc0[0, 0, P + 2:])
    np.testing.assert_array_equal(vc[0, 0, P + 2:], vc0[0, 0, P + 2:])


def test_dspark_cycle():
    g = load_golden("dspark_chain.txt")
    tp, ti = oracle.topk(_dspark_probs(g), 1)
    t = oracle.tree(tp, ti, g["D"][0], np.array(g["root"], np.int32))
    for key in ("token", "parent", "depth", "is_leaf"):
        np.testing.assert_array_equal(t[key][0], g[key], err_msg=key)
    np.testing.assert_array_equal(t["score"][0], np.array(g["score"], np.float32))
    np.testing.assert_array_equal(t["mask"][0], np.array(g["mask"], np.uint64))
    w = oracle.accept_walk(np.array([g["tgt"]], np.int32), t, g["S"][0])
    assert w["accept_len"][0] == g["accept_len"][0]
    np.testing.assert_array_equal(w["accept_rows"][0], g["accept_rows"])
    assert w["bonus"][0] == g["bonus"][0]
    assert w["chain_id"][0] == g["chain_id"][0]


# ------------------------------------------------------------------- top-k --

@pytest.mark.parametrize("V,k", [(7, 1), (64, 5), (1000, 32), (513, 8)])
def test_topk_matches_numpy_lexsort(V, k):
    probs = (RNG.integers(0, 40, (3, 2, V)) / 40.0).astype(np.float32)   # many ties
    tp, ti = oracle.topk(probs, k)
    for b in range(3):
        for s in range(2):
            row = probs[b, s]
            order = np.lexsort((np.arange(V), -row.astype(np.float64)))[:k]
            np.testing.assert_array_equal(ti[b, s], order)
            np.testing.assert_array_equal(tp[b, s], row[order])


# -------------------------------------------------------------------- tree --

@pytest.mark.parametrize("S,k,D,quant", [(3, 2, 4, None), (4, 3, 20, None), (5, 4, 64, 64),
                                         (7, 8, 16, None), (6, 2, 40, 16), (2, 32, 64, 8)])
def test_tree_enum_equals_beam(S, k, D, quant):
    _, tp, ti, root = _random_tree(4, S, k, D, quantize=quant)
    a = oracle.tree(tp, ti, D, root, "enum")
    b = oracle.tree(tp, ti, D, root, "beam")
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


@pytest.mark.parametrize("name,B", [("toy", None), ("qwen", None), ("batched", 4), ("mla", None)])
def test_tree_enum_equals_beam_on_workload_inputs(name, B):
    """The level beam (used where enumeration is out of reach) gives the same
    tree bytes as enumerating every path, on the workloads' own marginals
    (at most 8^7 paths per request)."""
    w = W.WORKLOADS[name] if B is None else W.WORKLOADS[name].scaled(B=B)
    probs = W.draft_probs(w, W.draft_logits(w))
    tp, ti = oracle.topk(probs.numpy(), w.k)
    root = W.root_tokens(w).numpy()
    a = oracle.tree(tp, ti, w.D, root, "enum")
    b = oracle.tree(tp, ti, w.D, root, "beam")
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def _ancestors(parent, r):
    out = []
    while r > 0:
        out.append(r)
        r = parent[r]
    return out


@pytest.mark.parametrize("S,k,D", [(3, 2, 4), (5, 3, 30), (7, 8, 16), (8, 10, 64)])
def test_tree_structure_invariants(S, k, D):
    _, tp, ti, root = _random_tree(3, S, k, D)
    t = oracle.tree(tp, ti, D, root, "beam")
    for b in range(3):
        par, dep, tok, msk = t["parent"][b], t["depth"][b], t["token"][b], t["mask"][b]
        assert par[0] == -1 and dep[0] == 0 and msk[0] == 0 and tok[0] == root[b]
        for r in range(1, D + 1):
            assert 0 <= par[r] < r                                 # parents precede children
            assert dep[r] == dep[par[r]] + 1 and dep[r] <= S
            bits = sum(1 << (int(j) - 1) for j in _ancestors(par, r))
            assert int(msk[r]) == bits                             # ancestor-or-self mask
            assert t["score"][b][r] <= t["score"][b][par[r]]
        for r in range(D + 1):
            kids = [c for c in range(1, D + 1) if par[c] == r]
            assert t["is_leaf"][b][r] == (0 if kids else 1)
            assert len(set(tok[c] for c in kids)) == len(kids)    # siblings distinct


def test_greedy_tree_is_optimal_by_brute_force():
    """CaDDTree, Method 2: for a fixed node count the greedy best-first tree
    maximizes the expected accepted length, i.e. the sum of the nodes' prefix
    probabilities over all parent-closed node sets.  Checked by enumerating
    every parent-closed set of D nodes of a tiny tree (dyadic probabilities, so
    the fp32 products are exact)."""
    S, k = 3, 2
    for trial in range(6):
        V = 6
        p = RNG.integers(1, 16, (1, S, V)).astype(np.float64)
        probs = (p / 64.0).astype(np.float32)           # dyadic, not normalised: fine
        tp, ti = oracle.topk(probs, k)
        nodes = [c for l in range(1, S + 1) for c in itertools.product(range(k), repeat=l)]
        sc = {c: np.prod([float(tp[0, i, c[i]]) for i in range(len(c))]) for c in nodes}
        for D in (1, 3, 5):
            best = -1.0
            for subset in itertools.combinations(nodes, D):
                ss = set(subset)
                if all(len(c) == 1 or c[:-1] in ss for c in subset):
                    best = max(best, sum(sc[c] for c in subset))
            t = oracle.tree(tp, ti, D, np.array([0], np.int32))
            assert abs(float(t["score"][0][1:].astype(np.float64).sum()) - best) < 1e-12


# --------------------------------------------------------------- attention --

def test_chain_equals_causal_attention():
    """A k=1 tree is a chain; its tree attention is plain causal attention over
    prefix + chain (the linear-speculation special case)."""
    S, D, Hq, Hkv, d, P = 6, 6, 4, 2, 32, 11
    probs = RNG.random((1, S, 20)).astype(np.float32)
    tp, ti = oracle.topk(probs, 1)
    t = oracle.tree(tp, ti, D, np.array([3], np.int32))
    assert list(t["parent"][0]) == [-1, 0, 1, 2, 3, 4, 5]
    R, cap = D + 1, P + 8
    q, kc, vc, pl, kt, vt = _random_attn_inputs(1, R, Hq, Hkv, d, cap, [P])
    scale = 1.0 / np.sqrt(d)
    out, lse = oracle.verify_attn(q, kc, vc, pl, kt, vt, t["mask"], scale)
    g = Hq // Hkv
    for h in range(Hq):
        K = np.concatenate([kc[0, h // g, :P], kt[0, :, h // g]]).astype(np.float64)
        Vv = np.concatenate([vc[0, h // g, :P], vt[0, :, h // g]]).astype(np.float64)
        Q = q[0, :, h].astype(np.float64)                        # positions P..P+D
        s = scale * Q @ K.T
        causal = np.arange(P + R)[None, :] <= (P + np.arange(R))[:, None]
        s = np.where(causal, s, -np.inf)
        w = np.exp(s - s.max(1, keepdims=True))
        ref = (w @ Vv) / w.sum(1, keepdims=True)
        np.testing.assert_allclose(out[0, :, h], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[0, :, h], s.max(1) + np.log(w.sum(1)), atol=1e-12)


def test_root_only_empty_prefix_returns_root_value():
    d = 24
    q, kc, vc, pl, kt, vt = _random_attn_inputs(2, 3, 2, 1, d, 4, [0, 0])
    mask = np.array([[0, 1, 3], [0, 1, 2]], np.uint64)
    out, lse = oracle.verify_attn(q, kc, vc, pl, kt, vt, mask, 0.3)
    for b in range(2):
        for h in range(2):
            np.testing.assert_array_equal(out[b, 0, h], vt[b, 0, 0].astype(np.float64))
            s = 0.3 * float(np.dot(q[b, 0, h].astype(np.float64), kt[b, 0, 0].astype(np.float64)))
            assert abs(lse[b, 0, h] - s) < 1e-12


def test_identical_keys_give_mean_of_visible_values():
    d, P, R = 16, 9, 4
    q, kc, vc, pl, kt, vt = _random_attn_inputs(1, R, 1, 1, d, 16, [P])
    key = RNG.standard_normal(d).astype(np.float32)
    kc[:] = key
    kt[:] = key
    mask = np.array([[0, 1, 2, 5]], np.uint64)                    # toy topology
    out, lse = oracle.verify_attn(q, kc, vc, pl, kt, vt, mask, 0.5)
    vis = {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3]}
    for r in range(R):
        vals = np.concatenate([vc[0, 0, :P], vt[0, vis[r], 0]]).astype(np.float64)
        np.testing.assert_allclose(out[0, r, 0], vals.mean(0), rtol=0, atol=1e-13)
        s = 0.5 * float(np.dot(q[0, r, 0].astype(np.float64), key.astype(np.float64)))
        assert abs(lse[0, r, 0] - (s + np.log(len(vals)))) < 1e-12


def test_non_ancestor_rows_are_invisible():
    """Branch isolation: changing the K/V of rows outside a node's ancestor path
    leaves its output bit-identical; changing an ancestor's K/V changes it."""
    S, k, D = 4, 3, 12
    _, tp, ti, root = _random_tree(1, S, k, D)
    t = oracle.tree(tp, ti, D, root)
    R, d, P = D + 1, 16, 7
    q, kc, vc, pl, kt, vt = _random_attn_inputs(1, R, 2, 1, d, 16, [P])
    base, _ = oracle.verify_attn(q, kc, vc, pl, kt, vt, t["mask"], 0.25)
    par = t["parent"][0]
    for j in range(1, R):
        kt2, vt2 = kt.copy(), vt.copy()
        kt2[0, j] += 1.0
        vt2[0, j] -= 1.0
        out, _ = oracle.verify_attn(q, kc, vc, pl, kt2, vt2, t["mask"], 0.25)
        for r in range(R):
            sees = j in _ancestors(par, r)
            if sees:
                assert not np.array_equal(out[0, r], base[0, r])
            else:
                np.testing.assert_array_equal(out[0, r], base[0, r])


def test_sibling_swap_invariance():
    """Relabelling tree rows (swapping two sibling subtrees' row numbers)
    permutes the outputs and changes nothing else (up to summation order)."""
    S, k, D = 3, 3, 9
    _, tp, ti, root = _random_tree(1, S, k, D)
    t = oracle.tree(tp, ti, D, root)
    par = t["parent"][0]
    R, d, P = D + 1, 8, 5
    q, kc, vc, pl, kt, vt = _random_attn_inputs(1, R, 2, 1, d, 12, [P])
    base, base_lse = oracle.verify_attn(q, kc, vc, pl, kt, vt, t["mask"], 0.4)
    perm = np.concatenate([[0], 1 + RNG.permutation(D)])         # new row -> old row
    inv = np.argsort(perm)
    new_par = np.array([-1] + [inv[par[perm[r]]] for r in range(1, R)])
    new_mask = np.zeros((1, R), np.uint64)
    for r in range(1, R):
        bits = 0
        x = r
        while x > 0:
            bits |= 1 << (int(x) - 1)
            x = new_par[x]
        new_mask[0, r] = bits
    out, lse = oracle.verify_attn(q[:, perm], kc, vc, pl, kt[:, perm], vt[:, perm],
                                  new_mask, 0.4)
    np.testing.assert_allclose(out[0], base[0, perm], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], base_lse[0, perm], rtol=0, atol=1e-12)


def test_gqa_grouping_and_latent_alias():
    """KV head of query head h is h // (Hq/Hkv); with v_aliases_k the value is
    the first dv entries of the key (latent KV)."""
    B, R, Hq, Hkv, d, P = 1, 2, 4, 2, 8, 3
    q, kc, vc, pl, kt, vt = _random_attn_inputs(B, R, Hq, Hkv, d, 6, [P])
    mask = np.array([[0, 1]], np.uint64)
    out, _ = oracle.verify_attn(q, kc, vc, pl, kt, vt, mask, 0.3)
    for h in range(Hq):
        o, _ = _textbook_attention(q[0, 1, h], np.concatenate([kc[0, h // 2, :P], kt[0, :2, h // 2]]),
                                   np.concatenate([vc[0, h // 2, :P], vt[0, :2, h // 2]]), 0.3)
        np.testing.assert_allclose(out[0, 1, h], o, atol=1e-12)
    dv = 5
    out, _ = oracle.verify_attn(q, kc, None, pl, kt, None, mask, 0.3, v_aliases_k=True, dv=dv)
    keys = np.concatenate([kc[0, 0, :P], kt[0, :2, 0]])
    o, _ = _textbook_attention(q[0, 1, 0], keys, keys[:, :dv], 0.3)
    np.testing.assert_allclose(out[0, 1, 0], o, atol=1e-12)


def test_bf16_bits_widen_exactly():
    """bf16 inputs given as bit patterns give the same result as the same values in fp32."""
    import torch
    B, R, Hq, Hkv, d, P = 1, 3, 2, 1, 16, 6
    q, kc, vc, pl, kt, vt = _random_attn_inputs(B, R, Hq, Hkv, d, 8, [P])
    mask = np.array([[0, 1, 3]], np.uint64)
    as_bf = [torch.from_numpy(a).to(torch.bfloat16) for a in (q, kc, vc, kt, vt)]
    f32 = [t.float().numpy() for t in as_bf]
    b16 = [t.view(torch.int16).numpy().view(np.uint16) for t in as_bf]
    o1, l1 = oracle.verify_attn(f32[0], f32[1], f32[2], pl, f32[3], f32[4], mask, 0.25)
    o2, l2 = oracle.verify_attn(b16[0], b16[1], b16[2], pl, b16[3], b16[4], mask, 0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ------------------------------------------------------------ argmax / walk --

def test_argmax_matches_numpy_first_occurrence():
    x = (RNG.integers(-5, 5, (7, 300))).astype(np.float32)          # many ties
    np.testing.assert_array_equal(oracle.argmax(x), np.argmax(x, axis=1))


@pytest.mark.parametrize("S,k,D", [(3, 2, 5), (5, 3, 20), (7, 8, 16), (4, 1, 4)])
def test_walk_properties(S, k, D):
    B = 16
    V = max(6, k)
    probs, tp, ti, root = _random_tree(B, S, k, D, V=V)
    t = oracle.tree(tp, ti, D, root)
    R = D + 1
    # targets that often agree with the tree's tokens
    tgt = RNG.integers(0, V, (B, R)).astype(np.int32)
    w = oracle.accept_walk(tgt, t, S)
    assert w["status"] == 0
    for b in range(B):
        par, tok = t["parent"][b], t["token"][b]
        L = w["accept_len"][b]
        rows = w["accept_rows"][b]
        assert 0 <= L <= t["depth"][b].max()
        assert rows[0] == 0 and all(x == -1 for x in rows[L + 1:])
        for i in range(1, L + 1):
            assert par[rows[i]] == rows[i - 1]
            assert tok[rows[i]] == tgt[b, rows[i - 1]]
        last = rows[L]
        assert w["bonus"][b] == tgt[b, last]
        assert not any(par[c] == last and tok[c] == tgt[b, last] for c in range(1, R))
        # brute force: the longest root path whose tokens all match is the accepted one
        best = 0
        for r in range(1, R):
            path = list(reversed(_ancestors(par, r)))
            prev = 0
            ok = True
            for x in path:
                if tok[x] != tgt[b, prev]:
                    ok = False
                    break
                prev = x
            if ok:
                best = max(best, len(path))
        assert L == best
        if L == 0:
            assert w["chain_id"][b] == -1
        else:
            c = w["chain_id"][b]
            assert t["is_leaf"][b][c] == 1 and last in _ancestors(par, c)
            assert not any(t["is_leaf"][b][x] and last in _ancestors(par, x) for x in range(1, c))


def test_commit_capacity_overflow_is_skipped():
    B, R, Hkv, d, cap, S = 2, 3, 2, 4, 6, 2
    kt = RNG.standard_normal((B, R, Hkv, d)).astype(np.float32)
    vt = RNG.standard_normal((B, R, Hkv, d)).astype(np.float32)
    kc = RNG.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    vc = RNG.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    kc0, vc0 = kc.copy(), vc.copy()
    pl = np.array([4, 3], np.int32)
    rows = np.array([[0, 1, 2], [0, 2, -1]], np.int32)
    ln = np.array([2, 1], np.int32)                               # b0: 4+3 > 6 -> skipped
    assert oracle.commit(kt, vt, rows, ln, kc, vc, pl, S) == 1
    assert list(pl) == [4, 5]
    np.testing.assert_array_equal(kc[0], kc0[0])
    np.testing.assert_array_equal(vc[0], vc0[0])
    np.testing.assert_array_equal(kc[1, :, 3:5], kt[1, [0, 2]].transpose(1, 0, 2))
    np.testing.assert_array_equal(vc[1, :, 3:5], vt[1, [0, 2]].transpose(1, 0, 2))
    np.testing.assert_array_equal(kc[1, :, :3], kc0[1, :, :3])
    np.testing.assert_array_equal(kc[1, :, 5:], kc0[1, :, 5:])


# ------------------------------------------------- cost-aware node count --
# "Cost-Aware Diffusion Draft Trees for Speculative Decoding", Method 1, 3, 4:
# keep adding best-first nodes while (1 + Phi) / (C_d + C_v(n)) rises.

def test_adaptive_toy_tree_with_linear_cost():
    """The page's toy tree (scores 0.5, 0.375, 0.3125 in best-first order) with
    C_d = 1 and C_v(n) = n / 4: the objective is 1, 1.2, 1.25, 1.25 for
    n = 0..3, so nodes 1 and 2 raise it and node 3 does not (all values exact
    binary fractions): two nodes are kept, and row 3 becomes padding."""
    tp = np.array([[[0.5, 0.375], [0.625, 0.25]]], np.float32)
    ti = np.array([[[1, 2], [1, 0]]], np.int32)
    t = oracle.tree_adaptive(tp, ti, 3, np.array([0], np.int32), [1.0], [[0.0, 0.25, 0.5, 0.75]])
    assert t["n_nodes"].tolist() == [2]
    assert t["token"][0].tolist() == [0, 1, 2, -1]
    assert t["parent"][0].tolist() == [-1, 0, 0, 0]
    assert t["mask"][0].tolist() == [0, 1, 2, 0]
    assert t["is_leaf"][0].tolist() == [0, 1, 1, 0]
    # a cheaper node lets the third one in
    t = oracle.tree_adaptive(tp, ti, 3, np.array([0], np.int32), [1.0], [[0.0, 0.25, 0.5, 0.7]])
    assert t["n_nodes"].tolist() == [3]


def _objective(scores, cost_d, cost_v, n):
    return (1.0 + float(np.sum(np.asarray(scores[:n], np.float64)))) / (cost_d + float(cost_v[n]))


def test_adaptive_stop_is_the_argmax_under_convex_cost():
    """Unimodality (Method 3): with non-increasing scores and a convex,
    non-decreasing verify cost, the first non-improving node is the global
    maximum of the objective over n = 0..D (checked against an fp64 brute
    force wherever the maximum is clear of rounding)."""
    rng = np.random.default_rng(3)
    checked = 0
    for _ in range(400):
        D = int(rng.integers(1, 40))
        s = np.sort(rng.uniform(0.0, 1.0, D) ** rng.uniform(1, 4))[::-1].astype(np.float32)
        a, b, c = rng.uniform(1, 50), rng.uniform(0, 3), rng.uniform(0, 0.2)
        n = np.arange(D + 1)
        cv = (a + b * n + c * n * n).astype(np.float32)
        cd = np.float32(rng.uniform(1, 100))
        J = np.array([_objective(s, float(cd), cv, m) for m in range(D + 1)])
        best = int(np.argmax(J))
        srt = np.sort(J)
        if D > 0 and srt[-1] - srt[-2] < 1e-5 * srt[-1]:
            continue
        assert oracle.adaptive_count(s, cd, cv) == best
        checked += 1
    assert checked > 300


def test_adaptive_extremes():
    s = np.array([0.5, 0.25, 0.125, 0.0625], np.float32)
    # no marginal verify cost: every node with a positive score helps
    assert oracle.adaptive_count(s, 10.0, np.full(5, 3.0, np.float32)) == 4
    # the first node alone costs more than it can ever return
    assert oracle.adaptive_count(s, 1.0, np.array([0, 1e9, 1e9, 1e9, 1e9], np.float32)) == 0
    # zero-probability nodes never raise the objective
    assert oracle.adaptive_count(np.zeros(4, np.float32), 1.0, np.arange(5, dtype=np.float32)) == 0


# ------------------------------------------- parent-conditioned proposals --
# "Adapting Tree-Structured Speculative Decoding to DeepSeek-V4" (review),
# "How it works" steps 1-2: A expands B and C; B proposes B and C, C proposes
# A and B; with D = 3 the kept nodes are A-B, A-C and A-B-B.

TOY_FOREST = dict(
    # candidates, parents first: B, C | B, C (children of B) | A, B (children of C)
    p=[[0.5, 0.375, 0.625, 0.25, 0.5, 0.25]],
    tok=[[1, 2, 1, 2, 0, 1]],
    parent=[[-1, -1, 0, 0, 1, 1]],
)


def test_conditioned_toy_matches_page_example():
    t = oracle.tree_conditioned(TOY_FOREST["p"], TOY_FOREST["tok"], TOY_FOREST["parent"], 3,
                                np.array([0], np.int32))
    # rows: A (root), A-B (0.5), A-C (0.375), A-B-B (0.3125); A-C-A (0.1875) is cut
    assert t["token"][0].tolist() == [0, 1, 2, 1]
    assert t["parent"][0].tolist() == [-1, 0, 0, 1]
    assert t["score"][0].tolist() == [1.0, 0.5, 0.375, 0.3125]
    assert t["mask"][0].tolist() == [0, 1, 2, 5]
    assert t["is_leaf"][0].tolist() == [0, 0, 1, 1]
    assert t["status"].tolist() == [0]


def _bfs_forest(tp, ti):
    """The full k-ary expansion of per-position marginals as a forest in BFS
    order (children in rank order), B = 1."""
    S, k = tp.shape
    p, tok, par = [], [], []
    level = [-1]
    for s in range(S):
        nxt = []
        for parent_idx in level:
            for r in range(k):
                p.append(tp[s, r]); tok.append(ti[s, r]); par.append(parent_idx)
                nxt.append(len(p) - 1)
        level = nxt
    return (np.array([p], np.float32), np.array([tok], np.int32), np.array([par], np.int32))


@pytest.mark.parametrize("S,k,D,quant", [(2, 2, 3, None), (3, 3, 12, None), (3, 4, 20, 8),
                                         (4, 2, 15, 4), (2, 5, 25, None)])
def test_conditioned_on_marginal_expansion_equals_marginal_tree(S, k, D, quant):
    """Proposals that ignore the parent (every node's children are the same
    per-position top-k) give exactly the per-position tree, ties included:
    BFS order with children in rank order is the rank-tuple order."""
    rng = np.random.default_rng(S * 100 + k * 10 + D)
    x = rng.normal(size=(1, S, 30)) * 2.0
    pr = np.exp(x) / np.exp(x).sum(-1, keepdims=True)
    if quant:
        pr = np.round(pr * quant) / quant
    tp, ti = oracle.topk(pr.astype(np.float32), k)
    ref = oracle.tree(tp, ti, D, np.array([7], np.int32), method="enum")
    cp, ct, cpar = _bfs_forest(tp[0], ti[0])
    got = oracle.tree_conditioned(cp, ct, cpar, D, np.array([7], np.int32))
    for key in ("token", "parent", "depth", "score", "mask", "is_leaf"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


def test_conditioned_tree_maximises_expected_acceptance():
    """Method 2: among all ancestor-closed sets of D candidates, the kept set
    has the largest sum of scores (brute force over small random forests)."""
    rng = np.random.default_rng(5)
    for _ in range(30):
        C = int(rng.integers(5, 11))
        par = [-1] + [int(rng.integers(-1, c)) for c in range(1, C)]
        p = rng.uniform(0.05, 1.0, C).astype(np.float32)
        D = int(rng.integers(1, min(C, 5) + 1))
        t = oracle.tree_conditioned(p[None], np.arange(C, dtype=np.int32)[None],
                                    np.array([par], np.int32), D, np.array([99], np.int32))
        sc = np.zeros(C)
        for c in range(C):
            sc[c] = p[c] * (1.0 if par[c] < 0 else sc[par[c]])
        best = 0.0
        for sub in itertools.combinations(range(C), D):
            ss = set(sub)
            if all(par[c] < 0 or par[c] in ss for c in sub):
                best = max(best, sum(sc[c] for c in sub))
        assert abs(float(np.sum(t["score"][0, 1:], dtype=np.float64)) - best) < 1e-5


def test_conditioned_rejects_malformed_forest():
    t = oracle.tree_conditioned([[0.5, 0.5]], [[1, 2]], [[-1, 1]], 2, np.array([0], np.int32))
    assert t["status"].tolist() == [1] and t["token"][0].tolist() == [0, -1, -1]
    t = oracle.tree_conditioned([[0.5, 1.5]], [[1, 2]], [[-1, 0]], 2, np.array([0], np.int32))
    assert t["status"].tolist() == [1]
