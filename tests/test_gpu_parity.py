"""GPU parity of every call of the C ABI against the CPU oracle.

Trees, argmax, walks and committed caches must match bit for bit; attention
must match within 1e-5 max abs (fp32) or 2e-2 max abs (bf16, fp32 accumulate).
Full-size workloads are checked on sampled attention rows the oracle computes
one by one; reduced sizes (several tiles plus a ragged tail) on every row.
"""

import functools

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import load_golden

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import tree_speculative_decoding_tsd_gb300 as T
    from tree_speculative_decoding_tsd_gb300 import workloads as W
    from tree_speculative_decoding_tsd_gb300.step import TreeVerifyStep
else:  # collected on CPU only to be deselected
    from tree_speculative_decoding_tsd_gb300 import workloads as W

DEV = "cuda:0"
NAMES = ["toy", "qwen", "batched", "long", "mla"]
TOL = {"f32": 1e-5, "bf16": 2e-2}


def _tol(w):
    return TOL[w.dtype]


@functools.lru_cache(maxsize=16)
def inputs(name, **over):
    """CPU inputs of a workload plus the oracle's tree (cached)."""
    w = W.WORKLOADS[name]
    if over:
        w = w.scaled(**dict(over))
    lg = W.draft_logits(w)
    probs = W.draft_probs(w, lg)
    root = W.root_tokens(w)
    tp, ti = oracle.topk(probs.numpy(), w.k)
    tree = oracle.tree(tp, ti, w.D, root.numpy(), method="beam")
    return dict(w=w, logits=lg, probs=probs, root=root, tp=tp, ti=ti, tree=tree)


def attn_inputs(w):
    q = W.queries(w)
    kc, vc = W.kv_cache(w)
    kt, vt = W.tree_kv(w)
    return q, kc, vc, W.prefix_lens(w), kt, vt


def gpu(*ts):
    return [None if t is None else t.to(DEV) for t in ts]


def run_tree(step, probs, root):
    p, r = gpu(probs, root)
    step.build(p, r)
    torch.cuda.synchronize()
    t = step.tree
    return dict(token=t.token.cpu().numpy(), parent=t.parent.cpu().numpy(),
                depth=t.depth.cpu().numpy(), score=t.score.cpu().numpy(),
                mask=t.mask.cpu().numpy().view(np.uint64), is_leaf=t.is_leaf.cpu().numpy())


def assert_tree_equal(got, ref):
    for key in ("token", "parent", "depth", "is_leaf"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    np.testing.assert_array_equal(got["score"].view(np.uint32), ref["score"].view(np.uint32))
    np.testing.assert_array_equal(got["mask"], ref["mask"])


def set_tree(step, tree):
    t = step.tree
    t.token.copy_(torch.from_numpy(tree["token"]))
    t.parent.copy_(torch.from_numpy(tree["parent"]))
    t.depth.copy_(torch.from_numpy(tree["depth"]))
    t.score.copy_(torch.from_numpy(tree["score"]))
    t.mask.copy_(torch.from_numpy(tree["mask"].view(np.int64)))
    t.is_leaf.copy_(torch.from_numpy(tree["is_leaf"]))


# --------------------------------------------------------------- smoke --

def test_smoke():
    import __graft_entry__
    __graft_entry__.smoke()


# ---------------------------------------------------------- tree build --

@pytest.mark.parametrize("name", NAMES)
def test_tree_build_full_size(name):
    d = inputs(name)
    w = d["w"]
    step = TreeVerifyStep.for_workload(w, DEV)
    got = run_tree(step, d["probs"], d["root"])
    assert_tree_equal(got, d["tree"])
    assert int(step.err[0]) == 0


@pytest.mark.parametrize("B,S,V,k,D,quant", [
    (3, 3, 1001, 3, 12, None),      # rows not 16-byte aligned
    (2, 5, 4099, 1, 5, None),       # chain (linear speculation)
    (2, 2, 3000, 32, 64, None),     # k = 32, D = 64
    (1, 16, 700, 2, 64, None),      # deepest tree
    (4, 4, 2053, 8, 40, 256),       # heavy ties in the marginals
    (2, 3, 32, 32, 40, 16),         # V == k: every token kept, ties
    (3, 2, 200000, 4, 9, None),     # long rows over many chunks
    (2, 3, 50000, 8, 20, 1),        # every probability rounds to 0: all elements tie
    # register slots of the frontier: ceil(D / 32), the frontier growing by one
    # entry per pop (a sibling and a child each time) up to D entries
    (2, 16, 600, 32, 31, None), (2, 16, 600, 32, 32, None), (2, 16, 600, 32, 33, None),
    (2, 16, 600, 32, 63, None), (2, 16, 600, 32, 64, None), (2, 16, 600, 32, 64, 64),
])
def test_tree_build_edge_cases(B, S, V, k, D, quant):
    g = torch.Generator().manual_seed(B * 1000 + S * 100 + k)
    x = torch.randn((B, S, V), generator=g, dtype=torch.float64) * 2.0
    p = torch.softmax(x, -1)
    if quant:
        p = torch.round(p * quant) / quant
    probs = p.float().contiguous()
    root = torch.randint(0, V, (B,), generator=g).int()
    tp, ti = oracle.topk(probs.numpy(), k)
    ref = oracle.tree(tp, ti, D, root.numpy(), method="beam")
    step = TreeVerifyStep(B, S, V, k, D, 2, 1, 64, 64, 8, torch.float32, False, 0.125, DEV)
    assert_tree_equal(run_tree(step, probs, root), ref)


def test_tree_build_toy_fixture():
    g = load_golden("toy_tree.txt")
    probs = torch.tensor([[g["p1"], g["p2"]]], dtype=torch.float32)
    step = TreeVerifyStep(1, 2, 3, 2, 3, 1, 1, 64, 64, 8, torch.float32, False, 0.125, DEV)
    got = run_tree(step, probs, torch.tensor(g["root"], dtype=torch.int32))
    for key in ("token", "parent", "depth", "is_leaf"):
        assert list(got[key][0]) == g[key], key
    assert list(got["mask"][0]) == g["mask"]


# ----------------------------------------------------------- attention --

def check_attention(w, q, kc, vc, plen, kt, vt, mask, sel=None):
    step = TreeVerifyStep.for_workload(w, DEV)
    step.tree.mask.copy_(torch.from_numpy(np.ascontiguousarray(mask).view(np.int64)))
    step.verify(*gpu(q, kc, vc, plen, kt, vt))
    torch.cuda.synchronize()
    assert int(step.err[0]) == 0, hex(int(step.err[0]))   # no bounded wait gave up
    out = step.out.float().cpu().numpy().astype(np.float64)
    lse = step.lse.cpu().numpy().astype(np.float64)
    ref_out, ref_lse = oracle.verify_attn(W.bits(q), W.bits(kc), None if vc is None else W.bits(vc),
                                          plen.numpy(), W.bits(kt),
                                          None if vt is None else W.bits(vt), mask, w.scale,
                                          v_aliases_k=w.v_aliases_k, dv=w.dv, sel=sel)
    if sel is not None:
        out = np.stack([out[b, r, h] for b, r, h in sel])
        lse = np.array([lse[b, r, h] for b, r, h in sel])
    err = np.abs(out - ref_out).max()
    assert err <= _tol(w), f"max abs err {err}"
    assert np.abs(lse - ref_lse).max() <= _tol(w) * 5e-2 + 1e-5
    return step


def sample_rows(w, n, seed=0):
    rng = np.random.default_rng(seed)
    n = min(n, w.B * w.R * w.Hq)
    rows = {(0, 0, 0), (w.B - 1, w.R - 1, w.Hq - 1), (0, w.R - 1, w.Hq // 2), (w.B - 1, 1, 0)}
    while len(rows) < n:
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.R)), int(rng.integers(w.Hq))))
    return np.array(sorted(rows), np.int32)


@pytest.mark.parametrize("name", NAMES)
def test_verify_attention_full_size_sampled(name):
    d = inputs(name)
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"], sel=sample_rows(w, 40))


REDUCED = {
    # all rows checked; prefixes span several KV tiles/splits and a ragged tail
    "toy": dict(),
    "qwen": dict(P=777, P_min=777),
    "batched": dict(B=5, P=1100, P_min=0, V=5000),
    "long": dict(B=2, P=1500, P_min=1500, V=3000),
    "mla": dict(B=2, P=300, P_min=300, V=2000),
    "qwen_f32": dict(dtype="f32", P=513, P_min=513),
}


@pytest.mark.parametrize("key", list(REDUCED))
def test_verify_attention_reduced_all_rows(key):
    name = key.split("_")[0]
    d = inputs(name, **REDUCED[key])
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"])


def test_verify_attention_empty_and_tiny_prefixes():
    w = W.WORKLOADS["qwen"].scaled(B=6, P=40, P_min=0, V=500)
    d = inputs("qwen", B=6, P=40, P_min=0, V=500)
    q, kc, vc, _, kt, vt = attn_inputs(w)
    plen = torch.tensor([0, 1, 2, 39, 40, 17], dtype=torch.int32)
    check_attention(w, q, kc, vc, plen, kt, vt, d["tree"]["mask"])


@pytest.mark.parametrize("B", [64, 65])
def test_verify_large_batch_longest_first_order(B):
    """Batches of 64 and more (request, KV head) units take the wave-cost split
    rule; up to 64 requests the CTAs take requests longest first (warp 0 ranks
    the prefix lengths, ties by index), 65 keeps the natural order.  Prefix
    lengths mix zero, ties and a ragged tail; every row checked."""
    over = dict(B=B, D=3, k=4, P=600, P_min=0, V=500)
    d = inputs("batched", **over)
    w = d["w"]
    q, kc, vc, _, kt, vt = attn_inputs(w)
    g = torch.Generator().manual_seed(B)
    plen = torch.randint(0, 601, (B,), generator=g).int()
    plen[::7] = 300                               # ties
    plen[3] = 0
    plen[5] = 600
    check_attention(w, q, kc, vc, plen, kt, vt, d["tree"]["mask"])


def test_verify_branch_isolation_bit_exact():
    """Changing scratch K/V of rows outside a node's ancestor path leaves the
    node's output bit-identical (research gap item 1 of the V4 review)."""
    d = inputs("qwen", P=300, P_min=300, V=4000)
    w, tree = d["w"], d["tree"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    s0 = check_attention(w, q, kc, vc, plen, kt, vt, tree["mask"])
    base = s0.out.clone()
    par = tree["parent"][0]
    j = int(w.R - 1)                        # perturb the last row (a leaf)
    kt2, vt2 = kt.clone(), vt.clone()
    kt2[0, j] += 1.0
    vt2[0, j] -= 1.0
    s1 = TreeVerifyStep.for_workload(w, DEV)
    s1.tree.mask.copy_(torch.from_numpy(tree["mask"].view(np.int64)))
    s1.verify(*gpu(q, kc, vc, plen, kt2, vt2))
    torch.cuda.synchronize()
    for r in range(w.R):
        anc, x = set(), r
        while x > 0:
            anc.add(x)
            x = par[x]
        same = torch.equal(s1.out[0, r], base[0, r])
        assert same == (j not in anc), r


def test_verify_determinism_and_batch_consistency():
    """Repeated calls are bit-identical; a request computed alone matches the
    same request inside a batch within the tolerance (the prefix split -- and
    with it the rounding -- may depend on the batch size)."""
    d = inputs("batched", B=4, P=900, P_min=100, V=3000)
    w, tree = d["w"], d["tree"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    full = check_attention(w, q, kc, vc, plen, kt, vt, tree["mask"])
    again = TreeVerifyStep.for_workload(w, DEV)
    again.tree.mask.copy_(full.tree.mask)
    again.verify(*gpu(q, kc, vc, plen, kt, vt))
    torch.cuda.synchronize()
    assert torch.equal(again.out, full.out) and torch.equal(again.lse, full.lse)
    b = 2
    w1 = w.scaled(B=1)
    one = TreeVerifyStep.for_workload(w1, DEV)
    one.tree.mask.copy_(full.tree.mask[b:b + 1])
    one.verify(*gpu(q[b:b + 1].contiguous(), kc[b:b + 1].contiguous(), vc[b:b + 1].contiguous(),
                    plen[b:b + 1].contiguous(), kt[b:b + 1].contiguous(),
                    vt[b:b + 1].contiguous()))
    torch.cuda.synchronize()
    diff = (one.out[0].float() - full.out[b].float()).abs().max().item()
    assert diff <= _tol(w)
    assert (one.lse[0] - full.lse[b]).abs().max().item() <= 1e-3


@pytest.mark.parametrize("dtype,Hq", [("bf16", 4), ("f32", 1)])
def test_verify_many_splits_per_request(dtype, Hq):
    """One request on one KV head with a 16000-key prefix: every row's result
    is merged from 63 prefix splits (several batches of partials and two
    rounds of 32 split weights in the merge), on the tcgen05 path (bf16, four
    query heads: 20 packed rows) and the CUDA-core path (fp32)."""
    over = dict(B=1, D=4, Hq=Hq, Hkv=1, P=16000, P_min=16000, V=500, dtype=dtype)
    d = inputs("qwen", **over)
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"])


# ---------------------------------------------------------- accept walk --

def run_walk(step, logits):
    (lg,) = gpu(logits)
    step.accept(lg)
    torch.cuda.synchronize()
    wk = step.walk
    return dict(tgt=wk.tgt.cpu().numpy(), accept_len=wk.accept_len.cpu().numpy(),
                accept_rows=wk.accept_rows.cpu().numpy(), bonus=wk.bonus.cpu().numpy(),
                chain_id=wk.chain_id.cpu().numpy())


def assert_walk_equal(got, ref, tgt):
    np.testing.assert_array_equal(got["tgt"], tgt)
    for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)


@pytest.mark.parametrize("name", NAMES)
def test_accept_walk_full_size(name):
    d = inputs(name)
    w, tree = d["w"], d["tree"]
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    tgt = oracle.argmax(tl.numpy())
    ref = oracle.accept_walk(tgt, tree, w.S)
    step = TreeVerifyStep.for_workload(w, DEV)
    set_tree(step, tree)
    assert_walk_equal(run_walk(step, tl), ref, tgt)
    assert int(step.err[0]) == 0


@pytest.mark.parametrize("V", [13, 1001, 4097, 150001])
def test_accept_walk_unaligned_rows_and_ties(V):
    d = inputs("qwen", V=V, P=8, P_min=8)
    w, tree = d["w"], d["tree"]
    g = torch.Generator().manual_seed(V)
    # integer-valued logits: many exact ties, argmax must take the lowest id
    tl = torch.randint(-4, 4, (w.B, w.R, w.V), generator=g).float()
    tgt = oracle.argmax(tl.numpy())
    ref = oracle.accept_walk(tgt, tree, w.S)
    step = TreeVerifyStep.for_workload(w, DEV)
    set_tree(step, tree)
    assert_walk_equal(run_walk(step, tl), ref, tgt)


def _golden_tree(g):
    R = len(g["token"])
    tree = dict(token=np.array([g["token"]], np.int32), parent=np.array([g["parent"]], np.int32),
                depth=np.array([g["depth"]], np.int32),
                score=np.array([g["score"]], np.float32),
                mask=np.array([g["mask"]], np.uint64), is_leaf=np.array([g["is_leaf"]], np.uint8))
    return tree, R


@pytest.mark.parametrize("fixture", ["toy_tree.txt", "dspark_chain.txt"])
def test_accept_walk_page_fixtures(fixture):
    g = load_golden(fixture)
    tree, R = _golden_tree(g)
    V = g["V"][0]
    tl = torch.full((1, R, V), -1.0)
    for r, t in enumerate(g["tgt"]):
        tl[0, r, t] = 1.0
    step = TreeVerifyStep(1, g["S"][0], V, g["k"][0], R - 1, 1, 1, 64, 64, 8, torch.float32,
                          False, 0.125, DEV)
    set_tree(step, tree)
    got = run_walk(step, tl)
    assert got["accept_len"][0] == g["accept_len"][0]
    assert list(got["accept_rows"][0]) == g["accept_rows"]
    assert got["bonus"][0] == g["bonus"][0] and got["chain_id"][0] == g["chain_id"][0]


def _deep_row_tree():
    """A 65-row tree whose accepted path runs through rows 40, 60, 61, 64 (all
    past the first 32 child rows) with two children of row 60 carrying the
    same token (the lower row must win) and the chain leaf in the same rows."""
    R, S, V = 65, 4, 2048
    parent = np.zeros(R, np.int32)
    parent[0] = -1
    parent[45:61] = 40
    parent[61:64] = 60
    parent[64] = 61
    token = (1000 + np.arange(R)).astype(np.int32)
    token[0] = 7
    token[61] = token[62] = 777
    depth = np.zeros(R, np.int32)
    mask = np.zeros(R, np.uint64)
    for c in range(1, R):
        depth[c] = depth[parent[c]] + 1
        mask[c] = (mask[parent[c]] if parent[c] > 0 else np.uint64(0)) | np.uint64(1 << (c - 1))
    has_child = np.zeros(R, bool)
    has_child[parent[1:]] = True
    tree = dict(token=token[None], parent=parent[None], depth=depth[None],
                score=np.linspace(1.0, 0.01, R, dtype=np.float32)[None], mask=mask[None],
                is_leaf=(~has_child).astype(np.uint8)[None])
    tgt = np.full(R, 5, np.int64)
    tgt[0], tgt[40], tgt[60], tgt[61] = token[40], token[60], 777, token[64]
    tl = torch.full((1, R, V), -1.0)
    for r in range(R):
        tl[0, r, tgt[r]] = 1.0
    return tree, tl, R, S, V


def test_accept_walk_rows_past_the_first_warp():
    """Rows 33-64 (the second chunk of the walk's row-per-lane layout): the
    accepted path, the lowest of two matching siblings, and the chain leaf
    all lie there; the separate walk and the fused walk + commit agree with
    the oracle."""
    tree, tl, R, S, V = _deep_row_tree()
    tgt = oracle.argmax(tl.numpy())
    ref = oracle.accept_walk(tgt, tree, S)
    assert list(ref["accept_rows"][0]) == [0, 40, 60, 61, 64] and ref["chain_id"][0] == 64
    step = TreeVerifyStep(1, S, V, 8, R - 1, 1, 1, 64, 64, 16, torch.float32, False, 0.125, DEV)
    set_tree(step, tree)
    assert_walk_equal(run_walk(step, tl), ref, tgt)
    # fused: also the commit of rows 0, 40, 60, 61, 64 at positions P..P+4
    g = torch.Generator().manual_seed(11)
    kt = torch.randn((1, R, 1, 64), generator=g)
    vt = torch.randn((1, R, 1, 64), generator=g)
    kc = torch.zeros((1, 1, 16, 64))
    vc = torch.zeros((1, 1, 16, 64))
    plen = torch.tensor([3], dtype=torch.int32)
    kc_ref, vc_ref, pl_ref = W.bits(kc).copy(), W.bits(vc).copy(), plen.numpy().copy()
    oracle.commit(W.bits(kt), W.bits(vt), ref["accept_rows"], ref["accept_len"], kc_ref, vc_ref,
                  pl_ref, S)
    step.walk.accept_len.zero_()
    gtl, gkt, gvt, gkc, gvc, gpl = gpu(tl, kt, vt, kc, vc, plen)
    step.accept_commit(gtl, gkt, gvt, gkc, gvc, gpl)
    torch.cuda.synchronize()
    for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(getattr(step.walk, key).cpu().numpy(), ref[key])
    np.testing.assert_array_equal(W.bits(gkc.cpu()), kc_ref)
    np.testing.assert_array_equal(W.bits(gvc.cpu()), vc_ref)
    assert int(gpl[0]) == 3 + 1 + 4 and int(step.err[0]) == 0


def test_accept_walk_reports_malformed_tree():
    d = inputs("toy")
    w, tree = d["w"], dict(d["tree"])
    tree["parent"] = tree["parent"].copy()
    tree["parent"][0, 2] = 3                         # parent after child
    step = TreeVerifyStep.for_workload(w, DEV)
    set_tree(step, tree)
    got = run_walk(step, torch.zeros((w.B, w.R, w.V)))
    e = int(step.err[0])
    assert e & T.TSD_DEV_ERR_MASK == T.TSD_DEV_ERR_BAD_TREE and e & 0xFFFFFF == 0
    assert got["accept_len"][0] == 0 and got["chain_id"][0] == -1


# -------------------------------------------------------------- commit --

def run_commit_case(w, accept_rows, accept_len, plen, seed=7):
    g = torch.Generator().manual_seed(seed)
    shape_k = (w.B, w.Hkv, w.cap, w.dk)
    kc = torch.randn(shape_k, generator=g).to(w.torch_dtype)           # canary contents
    vc = None if w.v_aliases_k else torch.randn((w.B, w.Hkv, w.cap, w.dv), generator=g).to(
        w.torch_dtype)
    kt, vt = W.tree_kv(w)
    kc_ref = W.bits(kc).copy()
    vc_ref = None if vc is None else W.bits(vc).copy()
    pl_ref = plen.numpy().copy()
    skipped = oracle.commit(W.bits(kt), None if vt is None else W.bits(vt), accept_rows,
                            accept_len, kc_ref, vc_ref, pl_ref, w.S, v_aliases_k=w.v_aliases_k)
    step = TreeVerifyStep.for_workload(w, DEV)
    step.walk.accept_rows.copy_(torch.from_numpy(accept_rows))
    step.walk.accept_len.copy_(torch.from_numpy(accept_len))
    gk, gv, gpl, gkt, gvt = gpu(kc, vc, plen, kt, vt)
    step.commit(gkt, gvt, gk, gv, gpl)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(W.bits(gk.cpu()), kc_ref)
    if vc is not None:
        np.testing.assert_array_equal(W.bits(gv.cpu()), vc_ref)
    np.testing.assert_array_equal(gpl.cpu().numpy(), pl_ref)
    return skipped, int(step.err[0])


@pytest.mark.parametrize("name", NAMES)
def test_commit_full_size(name):
    d = inputs(name)
    w, tree = d["w"], d["tree"]
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    ref = oracle.accept_walk(oracle.argmax(tl.numpy()), tree, w.S)
    skipped, err = run_commit_case(w, ref["accept_rows"], ref["accept_len"], W.prefix_lens(w))
    assert skipped == 0 and err == 0


def test_commit_deep_paths_and_capacity_overflow():
    w = W.WORKLOADS["qwen"].scaled(B=4, P=64, P_min=64, V=64)
    S = w.S
    rng = np.random.default_rng(3)
    rows = np.full((w.B, S + 1), -1, np.int32)
    ln = np.array([S, 3, 0, S], np.int32)
    for b in range(w.B):
        rows[b, 0] = 0
        rows[b, 1:ln[b] + 1] = rng.choice(np.arange(1, w.R), ln[b], replace=False)
    plen = torch.tensor([w.cap - S - 1, 10, w.cap - 1, w.cap - S], dtype=torch.int32)
    skipped, err = run_commit_case(w, rows, ln, plen)
    assert skipped == 1                                   # request 3 does not fit
    assert err & T.TSD_DEV_ERR_MASK == T.TSD_DEV_ERR_CAPACITY and err & 0xFFFFFF == 3


# ------------------------------------------------------------ full step --

@pytest.mark.parametrize("name,over", [("toy", {}), ("qwen", {}),
                                       ("batched", dict(B=6, V=20000)),
                                       ("mla", dict(B=3, P=700, P_min=700, V=9000)),
                                       ("long", dict(B=2, P=2000, P_min=2000, V=7000))])
def test_full_step_chained(name, over):
    d = inputs(name, **over)
    w, tree = d["w"], d["tree"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    tgt = oracle.argmax(tl.numpy())
    ref_walk = oracle.accept_walk(tgt, tree, w.S)
    sel = sample_rows(w, 24, seed=5)
    ref_out, _ = oracle.verify_attn(W.bits(q), W.bits(kc), None if vc is None else W.bits(vc),
                                    plen.numpy(), W.bits(kt), None if vt is None else W.bits(vt),
                                    tree["mask"], w.scale, v_aliases_k=w.v_aliases_k, dv=w.dv,
                                    sel=sel)
    kc_ref = W.bits(kc).copy()
    vc_ref = None if vc is None else W.bits(vc).copy()
    pl_ref = plen.numpy().copy()
    oracle.commit(W.bits(kt), None if vt is None else W.bits(vt), ref_walk["accept_rows"],
                  ref_walk["accept_len"], kc_ref, vc_ref, pl_ref, w.S, v_aliases_k=w.v_aliases_k)

    step = TreeVerifyStep.for_workload(w, DEV)
    g = gpu(d["probs"], d["root"], q, kc, vc, plen, kt, vt, tl)
    step.run(*g)
    torch.cuda.synchronize()
    got_tree = dict(token=step.tree.token.cpu().numpy(), parent=step.tree.parent.cpu().numpy(),
                    depth=step.tree.depth.cpu().numpy(), score=step.tree.score.cpu().numpy(),
                    mask=step.tree.mask.cpu().numpy().view(np.uint64),
                    is_leaf=step.tree.is_leaf.cpu().numpy())
    assert_tree_equal(got_tree, tree)
    out = step.out.float().cpu().numpy()
    assert np.abs(np.stack([out[b, r, h] for b, r, h in sel]) - ref_out).max() <= _tol(w)
    wk = step.walk
    np.testing.assert_array_equal(wk.tgt.cpu().numpy(), tgt)
    for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(getattr(wk, key).cpu().numpy(), ref_walk[key])
    np.testing.assert_array_equal(W.bits(g[3].cpu()), kc_ref)
    if vc is not None:
        np.testing.assert_array_equal(W.bits(g[4].cpu()), vc_ref)
    np.testing.assert_array_equal(g[5].cpu().numpy(), pl_ref)
    assert int(step.err[0]) == 0


def test_rounds_enqueued_back_to_back():
    """Three full rounds enqueued on one stream with no host synchronisation
    in between (each round's first kernel may be scheduled while the previous
    round's commit finishes): the final cache and prefix lengths equal three
    oracle rounds applied in order, and the last round's tree, attention
    (over the cache the first two rounds extended) and walk match."""
    w = W.WORKLOADS["qwen"].scaled(B=3, V=5000, P=300, P_min=100)
    base_lg = W.draft_logits(w)
    root = W.root_tokens(w)
    q, kc, vc, _, kt, vt = attn_inputs(w)
    plen = torch.tensor([50, 120, 0], dtype=torch.int32)   # room for three rounds
    kc_ref, vc_ref, pl_ref = W.bits(kc).copy(), W.bits(vc).copy(), plen.numpy().copy()
    rounds = []
    for r in range(3):
        lg = torch.roll(base_lg, shifts=101 * r, dims=-1)
        probs = W.draft_probs(w, lg)
        tp, ti = oracle.topk(probs.numpy(), w.k)
        tree = oracle.tree(tp, ti, w.D, root.numpy(), method="beam")
        tl = W.target_logits(w, torch.from_numpy(tree["depth"]), lg)
        ktr, vtr = torch.roll(kt, shifts=r, dims=1), torch.roll(vt, shifts=r, dims=1)
        walk = oracle.accept_walk(oracle.argmax(tl.numpy()), tree, w.S)
        if r == 2:
            sel = sample_rows(w, 24, seed=9)
            ref_out, _ = oracle.verify_attn(W.bits(q), kc_ref, vc_ref, pl_ref.copy(), W.bits(ktr),
                                            W.bits(vtr), tree["mask"], w.scale, sel=sel)
        oracle.commit(W.bits(ktr), W.bits(vtr), walk["accept_rows"], walk["accept_len"], kc_ref,
                      vc_ref, pl_ref, w.S)
        rounds.append((probs, tl, ktr, vtr, tree, walk))
    step = TreeVerifyStep.for_workload(w, DEV)
    gq, gkc, gvc, gpl, groot = gpu(q, kc, vc, plen, root)
    dev_rounds = [gpu(p_, tl_, kt_, vt_) for p_, tl_, kt_, vt_, _, _ in rounds]
    torch.cuda.synchronize()
    for gp, gtl, gkt, gvt in dev_rounds:
        step.run(gp, groot, gq, gkc, gvc, gpl, gkt, gvt, gtl)
    torch.cuda.synchronize()
    assert int(step.err[0]) == 0
    np.testing.assert_array_equal(W.bits(gkc.cpu()), kc_ref)
    np.testing.assert_array_equal(W.bits(gvc.cpu()), vc_ref)
    np.testing.assert_array_equal(gpl.cpu().numpy(), pl_ref)
    tree, walk = rounds[2][4], rounds[2][5]
    np.testing.assert_array_equal(step.tree.token.cpu().numpy(), tree["token"])
    np.testing.assert_array_equal(step.tree.mask.cpu().numpy().view(np.uint64), tree["mask"])
    out = step.out.float().cpu().numpy()
    assert np.abs(np.stack([out[b, r, h] for b, r, h in sel]) - ref_out).max() <= _tol(w)
    for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(getattr(step.walk, key).cpu().numpy(), walk[key])


# ------------------------------------------------- every attention path --

@pytest.fixture
def force_path(request):
    with T.verify_path(request.param):
        yield request.param


@pytest.mark.parametrize("force_path", ["tc", "mma", "generic"], indirect=True)
@pytest.mark.parametrize("key", ["qwen", "batched", "long"])
def test_verify_each_path_reduced(force_path, key):
    d = inputs(key, **REDUCED[key])
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"])


def test_verify_bounded_wait_gives_up_then_next_call_is_exact():
    """A pipeline-wait budget of a few clock cycles makes the tcgen05 kernel's
    first wait on a product give up (the waits poll instead of sleeping):
    each CTA skips its output and exits once its copies and products in flight
    have landed and its TMEM is released, and the first one records
    TSD_DEV_ERR_TIMEOUT | b.  With the default budget restored, the next call
    on the same buffers is within tolerance of the oracle, and the one after
    that on a fresh step too."""
    d = inputs("qwen", **REDUCED["qwen"])
    w = d["w"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    step = TreeVerifyStep.for_workload(w, DEV)
    step.tree.mask.copy_(torch.from_numpy(np.ascontiguousarray(d["tree"]["mask"]).view(np.int64)))
    args = gpu(q, kc, vc, plen, kt, vt)
    with T.verify_path("tc"):
        with T.wait_budget(16):
            step.verify(*args)
            torch.cuda.synchronize()
        e = int(step.err[0])
        assert e & T.TSD_DEV_ERR_MASK == T.TSD_DEV_ERR_TIMEOUT, hex(e)
        assert 0 <= (e & 0xFFFFFF) < w.B
        assert T.tsd_set_wait_budget(0) == 0           # the context manager restored it
        step.err.zero_()
        step.verify(*args)
        torch.cuda.synchronize()
        assert int(step.err[0]) == 0
        ref_out, _ = oracle.verify_attn(W.bits(q), W.bits(kc), W.bits(vc), plen.numpy(), W.bits(kt),
                                        W.bits(vt), d["tree"]["mask"], w.scale)
        err = np.abs(step.out.float().cpu().numpy().astype(np.float64) - ref_out).max()
        assert err <= _tol(w), f"max abs err {err}"
        check_attention(w, q, kc, vc, plen, kt, vt, d["tree"]["mask"])


@pytest.mark.parametrize("force_path", ["tc"], indirect=True)
@pytest.mark.parametrize("D", [3, 5, 7, 11])
def test_verify_tcgen05_small_trees(force_path, D):
    """Packed-row counts 16..48 (g = 4): MMA N of 16, 32 and 48."""
    d = inputs("qwen", D=D, P=1300, P_min=1300, V=3000)
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"])


@pytest.mark.parametrize("force_path", ["tc", "mma"], indirect=True)
@pytest.mark.parametrize("D", [15, 19, 23, 27, 31, 35, 48])
def test_verify_tensor_core_column_tiles(force_path, D):
    """Packed-row counts 64..196 (g = 4): every MMA N width and a two-group split."""
    d = inputs("qwen", D=D, P=1300, P_min=1300, V=3000)
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"])


@pytest.mark.parametrize("force_path", ["tc", "mma", "generic"], indirect=True)
def test_verify_rescale_on_late_large_scores(force_path):
    """Keys near the end of the prefix align with the queries, so the running
    max jumps on late tiles (exercises the rescale of the accumulators)."""
    d = inputs("qwen", B=2, P=1500, P_min=1500, V=3000)
    w, tree = d["w"], d["tree"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    g = w.Hq // w.Hkv
    for b in range(w.B):
        for hk in range(w.Hkv):
            qd = q[b, :, hk * g:(hk + 1) * g].float().mean(dim=(0, 1))
            qd = qd / qd.norm()
            for j, pos in enumerate(range(1100, 1500, 37)):
                kc[b, hk, pos] = (qd * (8.0 + j)).to(kc.dtype)
    check_attention(w, q, kc, vc, plen, kt, vt, tree["mask"])


@pytest.mark.parametrize("force_path", ["tc", "mma"], indirect=True)
def test_verify_paths_empty_and_tiny_prefixes(force_path):
    w = W.WORKLOADS["qwen"].scaled(B=6, P=300, P_min=0, V=500)
    d = inputs("qwen", B=6, P=300, P_min=0, V=500)
    q, kc, vc, _, kt, vt = attn_inputs(w)
    plen = torch.tensor([0, 1, 127, 128, 129, 300], dtype=torch.int32)
    check_attention(w, q, kc, vc, plen, kt, vt, d["tree"]["mask"])


# ------------------------------------------------------ latent (MLA) heads --

@pytest.mark.parametrize("force_path", ["tc", "generic"], indirect=True)
def test_verify_latent_paths_splits_and_tails(force_path):
    """Latent heads (dk 576, V = K[:, :512], 128 query heads): prefixes of
    several 128-key tiles with ragged tails, split across CTAs and merged."""
    d = inputs("mla", B=3, P=1300, P_min=200, V=2000)
    w = d["w"]
    check_attention(w, *attn_inputs(w), d["tree"]["mask"])


@pytest.mark.parametrize("force_path", ["tc", "generic"], indirect=True)
def test_verify_latent_empty_and_tiny_prefixes(force_path):
    w = W.WORKLOADS["mla"].scaled(B=6, P=300, P_min=0, V=500)
    d = inputs("mla", B=6, P=300, P_min=0, V=500)
    q, kc, vc, _, kt, vt = attn_inputs(w)
    plen = torch.tensor([0, 1, 127, 128, 129, 300], dtype=torch.int32)
    check_attention(w, q, kc, vc, plen, kt, vt, d["tree"]["mask"])


@pytest.mark.parametrize("force_path", ["tc", "generic"], indirect=True)
def test_verify_latent_rescale_on_late_large_scores(force_path):
    d = inputs("mla", B=2, P=900, P_min=900, V=2000)
    w, tree = d["w"], d["tree"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    for b in range(w.B):
        qd = q[b].float().mean(dim=(0, 1))
        qd = qd / qd.norm()
        for j, pos in enumerate(range(600, 900, 41)):
            kc[b, 0, pos] = (qd * (6.0 + j)).to(kc.dtype)
    check_attention(w, q, kc, vc, plen, kt, vt, tree["mask"])


@pytest.mark.parametrize("name,force", [("qwen", "tc"), ("qwen", "mma"), ("qwen", "generic"),
                                        ("mla", "tc"), ("mla", "generic")])
def test_verify_ignores_nonfinite_cache_rows_past_prefix(name, force):
    """Cache rows at and past prefix_len hold NaN/Inf: tiles that straddle the
    end of the prefix must not let them reach the output (0 x NaN)."""
    with T.verify_path(force):
        _nonfinite_case(name)


def _nonfinite_case(name):
    over = dict(B=3, P=700, P_min=100, V=1000)
    d = inputs(name, **over)
    w = d["w"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    kc = kc.clone()
    vc = None if vc is None else vc.clone()
    for b in range(w.B):
        p = int(plen[b])
        kc[b, :, p:] = float("nan")
        kc[b, :, p + 1::2] = float("inf")
        if vc is not None:
            vc[b, :, p:] = float("nan")
    check_attention(w, q, kc, vc, plen, kt, vt, d["tree"]["mask"])


# --------------------------------------------- cost-aware adaptive budget --

def _cost_tables(w, kind, seed=0):
    """Convex, non-decreasing verify costs (same unit as the drafting cost)
    placing the stop inside, below or above the budget."""
    rng = np.random.default_rng(seed)
    n = np.arange(w.D + 1, dtype=np.float64)
    if kind == "mid":
        cd = rng.uniform(5, 15, w.B)
        cv = np.stack([20 + rng.uniform(0.5, 3) * n + rng.uniform(0, 0.3) * n * n
                       for _ in range(w.B)])
    elif kind == "none":
        cd, cv = np.full(w.B, 1.0), np.stack([1.0 + 1e9 * (n > 0)] * w.B)
    else:  # "all": free nodes
        cd, cv = np.full(w.B, 10.0), np.full((w.B, w.D + 1), 5.0)
    return cd.astype(np.float32), cv.astype(np.float32)


def run_adaptive(step, probs, root, cd, cv):
    p, r, c1, c2 = gpu(probs, root, torch.from_numpy(cd), torch.from_numpy(cv))
    step.build_adaptive(p, r, c1, c2)
    torch.cuda.synchronize()
    t = step.tree
    got = dict(token=t.token.cpu().numpy(), parent=t.parent.cpu().numpy(),
               depth=t.depth.cpu().numpy(), score=t.score.cpu().numpy(),
               mask=t.mask.cpu().numpy().view(np.uint64), is_leaf=t.is_leaf.cpu().numpy())
    return got, step.n_nodes.cpu().numpy()


@pytest.mark.parametrize("name", ["toy", "qwen", "batched", "long", "mla"])
@pytest.mark.parametrize("kind", ["mid", "none", "all"])
def test_tree_build_adaptive_matches_oracle(name, kind):
    d = inputs(name)
    w = d["w"]
    cd, cv = _cost_tables(w, kind, seed=len(name))
    ref = oracle.tree_adaptive(d["tp"], d["ti"], w.D, d["root"].numpy(), cd, cv, method="beam")
    step = TreeVerifyStep.for_workload(w, DEV)
    got, n = run_adaptive(step, d["probs"], d["root"], cd, cv)
    np.testing.assert_array_equal(n, ref["n_nodes"])
    assert_tree_equal(got, ref)
    if kind == "none":
        assert (n == 0).all()
    if kind == "all":   # free nodes: stops only where fp32 1 + Phi stops growing
        assert (n >= min(w.D, 4)).all()


def test_adaptive_step_never_accepts_padding():
    """Verify, walk and commit on a tree with padded rows: the walk equals the
    oracle's on the padded tree and stays within the kept rows."""
    d = inputs("batched", B=6, P=700, P_min=100, V=3000)
    w = d["w"]
    cd, cv = _cost_tables(w, "mid", seed=11)
    ref = oracle.tree_adaptive(d["tp"], d["ti"], w.D, d["root"].numpy(), cd, cv, method="beam")
    step = TreeVerifyStep.for_workload(w, DEV)
    got, n = run_adaptive(step, d["probs"], d["root"], cd, cv)
    assert_tree_equal(got, ref)
    # target logits that favour the draft: most walks go deep
    tl = W.target_logits(w, torch.from_numpy(ref["depth"]), d["logits"])
    tgt = oracle.argmax(tl.numpy())
    ref_walk = oracle.accept_walk(tgt, ref, w.S)
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    g = gpu(q, kc, vc, plen, kt, vt, tl)
    step.verify(*g[:6])
    step.accept(g[6])
    step.commit(g[4], g[5], g[1], g[2], g[3])
    torch.cuda.synchronize()
    wk = step.walk
    for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(getattr(wk, key).cpu().numpy(), ref_walk[key])
    rows = wk.accept_rows.cpu().numpy()
    for b in range(w.B):
        L = int(wk.accept_len[b])
        assert all(1 <= rows[b, i] <= n[b] for i in range(1, L + 1))
    assert int(step.err[0]) == 0


def test_cost_model_calibrated_on_this_gpu():
    """Measure the step at a few budgets and prefix lengths, fit the convex
    model and drive the adaptive build with it."""
    pytest.importorskip("scipy")
    from tree_speculative_decoding_tsd_gb300 import costmodel
    w = W.WORKLOADS["qwen"].scaled(V=20000)
    cost_d, samples = costmodel.measure(w, [2, 8, 32], [512, 4096], steps=5, warmup=2, device=DEV)
    assert cost_d > 0
    m = costmodel.CostModel.from_samples(cost_d, samples)
    cv = m.verify_cost(2048, 32).astype(np.float64)
    assert np.all(np.diff(cv) >= -1e-3) and np.all(np.diff(cv, 2) >= -1e-3)
    d = inputs("qwen", D=32, V=20000)
    wq = d["w"]
    cdt, cvt = m.tables([2048] * wq.B, wq.D)
    ref = oracle.tree_adaptive(d["tp"], d["ti"], wq.D, d["root"].numpy(), cdt, cvt, method="beam")
    step = TreeVerifyStep.for_workload(wq, DEV)
    got, n = run_adaptive(step, d["probs"], d["root"], cdt, cvt)
    np.testing.assert_array_equal(n, ref["n_nodes"])
    assert_tree_equal(got, ref)


# ------------------------------------------------ one graph per round --

def _oracle_round(w, d, tree, q, kc, vc, plen, kt, vt, tl, sel):
    """The oracle's view of one whole round on these inputs: sampled attention
    rows, argmax, walk, and the cache and prefix lengths after the commit."""
    ref_out, _ = oracle.verify_attn(W.bits(q), W.bits(kc), None if vc is None else W.bits(vc),
                                    plen.numpy(), W.bits(kt), None if vt is None else W.bits(vt),
                                    tree["mask"], w.scale, v_aliases_k=w.v_aliases_k, dv=w.dv,
                                    sel=sel)
    tgt = oracle.argmax(tl.numpy())
    walk = oracle.accept_walk(tgt, tree, w.S)
    kc_ref = W.bits(kc).copy()
    vc_ref = None if vc is None else W.bits(vc).copy()
    pl_ref = plen.numpy().copy()
    oracle.commit(W.bits(kt), None if vt is None else W.bits(vt), walk["accept_rows"],
                  walk["accept_len"], kc_ref, vc_ref, pl_ref, w.S, v_aliases_k=w.v_aliases_k)
    return ref_out, tgt, walk, kc_ref, vc_ref, pl_ref


@pytest.mark.parametrize("case", ["batched", "batched_adaptive", "batched_one_stream", "qwen"])
def test_captured_round_matches_oracle(case):
    """The whole round recorded as one CUDA graph (TreeVerifyStep.capture, the
    flow the benchmark times) matches the oracle replay after replay -- tree,
    sampled attention rows, argmax, walk, committed cache and prefix lengths
    -- and is bit-identical to the eager calls.  "qwen" is the benchmark's own
    graph: the full qwen workload."""
    adaptive = case.endswith("adaptive")
    d = inputs("qwen") if case == "qwen" else inputs("batched", B=4, P=600, P_min=200, V=4000)
    w = d["w"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    if adaptive:
        cd, cv = _cost_tables(w, "mid", seed=2)
        tree = oracle.tree_adaptive(d["tp"], d["ti"], w.D, d["root"].numpy(), cd, cv,
                                    method="beam")
        extra = (torch.from_numpy(cd).to(DEV), torch.from_numpy(cv).to(DEV))
    else:
        tree = d["tree"]
        extra = (None, None)
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    sel = sample_rows(w, 24, seed=3)
    ref_out, tgt, walk, kc_ref, vc_ref, pl_ref = _oracle_round(w, d, tree, q, kc, vc, plen, kt,
                                                               vt, tl, sel)

    def fresh():
        return gpu(d["probs"], d["root"], q, kc.clone(), None if vc is None else vc.clone(),
                   plen.clone(), kt, vt, tl)

    # "batched_one_stream": the round without the second stream for the
    # target argmax (the fused walk and commit)
    ov = False if case.endswith("one_stream") else None
    eager = TreeVerifyStep.for_workload(w, DEV, overlap_argmax=ov)
    ge = fresh()
    eager._round(*ge, *extra, None)
    torch.cuda.synchronize()

    graphed = TreeVerifyStep.for_workload(w, DEV, overlap_argmax=ov)
    gg = fresh()
    g = graphed.capture(*gg, *extra)
    for _ in range(2):
        # restore the state the round started from, then replay
        gg[3].copy_(kc.to(DEV))
        if vc is not None:
            gg[4].copy_(vc.to(DEV))
        gg[5].copy_(plen.to(DEV))
        g.replay()
        torch.cuda.synchronize()
        t = graphed.tree
        got = dict(token=t.token.cpu().numpy(), parent=t.parent.cpu().numpy(),
                   depth=t.depth.cpu().numpy(), score=t.score.cpu().numpy(),
                   mask=t.mask.cpu().numpy().view(np.uint64), is_leaf=t.is_leaf.cpu().numpy())
        assert_tree_equal(got, tree)
        if adaptive:
            np.testing.assert_array_equal(graphed.n_nodes.cpu().numpy(), tree["n_nodes"])
        out = graphed.out.float().cpu().numpy()
        err = np.abs(np.stack([out[b, r, h] for b, r, h in sel]) - ref_out).max()
        assert err <= _tol(w), f"attention max abs err {err}"
        wk = graphed.walk
        np.testing.assert_array_equal(wk.tgt.cpu().numpy(), tgt)
        for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
            np.testing.assert_array_equal(getattr(wk, key).cpu().numpy(), walk[key])
        np.testing.assert_array_equal(W.bits(gg[3].cpu()), kc_ref)
        if vc is not None:
            np.testing.assert_array_equal(W.bits(gg[4].cpu()), vc_ref)
        np.testing.assert_array_equal(gg[5].cpu().numpy(), pl_ref)
        # and the same bytes as the eager calls
        for f in ("token", "parent", "depth", "score", "mask", "is_leaf"):
            assert torch.equal(getattr(eager.tree, f), getattr(graphed.tree, f)), f
        assert torch.equal(eager.out, graphed.out) and torch.equal(eager.lse, graphed.lse)
        for f in ("tgt", "accept_len", "accept_rows", "bonus", "chain_id"):
            assert torch.equal(getattr(eager.walk, f), getattr(graphed.walk, f)), f
        assert torch.equal(ge[3], gg[3]) and torch.equal(ge[5], gg[5])
    assert int(graphed.err[0]) == 0


def test_tree_build_reports_probabilities_above_one_or_nan():
    """A draft row with a value above 1 or a NaN breaks the score order the
    best-first rule needs: the build reports it in the error word (the first
    error wins) and builds the other requests' trees exactly."""
    d = inputs("qwen", B=3, V=3000)
    w = d["w"]
    for bad_b, val in [(1, 1.5), (2, float("nan")), (0, float("inf"))]:
        probs = d["probs"].clone()
        probs[bad_b, 3, 1234] = val
        step = TreeVerifyStep.for_workload(w, DEV)
        got = run_tree(step, probs, d["root"])
        assert int(step.err[0]) == (T.TSD_DEV_ERR_BAD_PROBS | bad_b), val
        for b in range(w.B):
            if b == bad_b:
                continue
            for key in ("token", "parent", "depth", "is_leaf", "mask"):
                np.testing.assert_array_equal(got[key][b], d["tree"][key][b], err_msg=key)
    step = TreeVerifyStep.for_workload(w, DEV)
    probs = d["probs"].clone()
    probs[0, 0, 7] = 1.0          # exactly 1 is allowed
    probs[1, 2, 9] = -0.0
    run_tree(step, probs, d["root"])
    assert int(step.err[0]) == 0


# ------------------------------------------- parent-conditioned proposals --

def _random_forest(B, C, seed, quant=None):
    """Random parents (any earlier candidate or the root), skewed probabilities."""
    rng = np.random.default_rng(seed)
    par = np.full((B, C), -1, np.int32)
    for b in range(B):
        for c in range(1, C):
            par[b, c] = int(rng.integers(-1, c))
    p = rng.uniform(0.0, 1.0, (B, C)) ** rng.uniform(1, 3)
    if quant:
        p = np.round(p * quant) / quant
    tok = rng.integers(0, 50000, (B, C)).astype(np.int32)
    return p.astype(np.float32), tok, par


def run_conditioned(w, cp, ct, cpar, root, D):
    step = TreeVerifyStep(w.B, w.S, w.V, w.k, D, w.Hq, w.Hkv, w.dk, w.dv, w.cap, w.torch_dtype,
                          w.v_aliases_k, w.scale, DEV)
    g = gpu(torch.from_numpy(cp), torch.from_numpy(ct), torch.from_numpy(cpar), root)
    step.err.zero_()
    step.build_conditioned(*g)
    torch.cuda.synchronize()
    t = step.tree
    got = dict(token=t.token.cpu().numpy(), parent=t.parent.cpu().numpy(),
               depth=t.depth.cpu().numpy(), score=t.score.cpu().numpy(),
               mask=t.mask.cpu().numpy().view(np.uint64), is_leaf=t.is_leaf.cpu().numpy())
    return got, int(step.err[0])


@pytest.mark.parametrize("C,D,quant", [(6, 3, None), (100, 16, None), (700, 64, 16),
                                       (2048, 64, None), (2048, 40, 4), (37, 37, None)])
def test_tree_build_conditioned_random_forests(C, D, quant):
    B = 4
    w = W.WORKLOADS["qwen"].scaled(B=B, V=50000, P=64, P_min=64)
    cp, ct, cpar = _random_forest(B, C, seed=C + D, quant=quant)
    root = torch.arange(B, dtype=torch.int32)
    ref = oracle.tree_conditioned(cp, ct, cpar, D, root.numpy())
    assert (ref["status"] == 0).all()
    got, err = run_conditioned(w, cp, ct, cpar, root, D)
    assert err == 0
    assert_tree_equal(got, ref)


def test_tree_build_conditioned_page_toy_and_marginal_equivalence():
    w = W.WORKLOADS["toy"]
    cp = np.array([[0.5, 0.375, 0.625, 0.25, 0.5, 0.25]], np.float32)
    ct = np.array([[1, 2, 1, 2, 0, 1]], np.int32)
    cpar = np.array([[-1, -1, 0, 0, 1, 1]], np.int32)
    root = torch.tensor([0], dtype=torch.int32)
    got, err = run_conditioned(w.scaled(B=1), cp, ct, cpar, root, 3)
    assert err == 0
    assert got["token"][0].tolist() == [0, 1, 2, 1] and got["parent"][0].tolist() == [-1, 0, 0, 1]
    # the full expansion of the qwen marginals equals tsd_tree_build's tree
    d = inputs("qwen", S=3, k=8, D=40, V=3000)
    wq = d["w"]
    S, k = wq.S, wq.k
    p, tok, par = [], [], []
    level = [-1]
    for s in range(S):
        nxt = []
        for pi in level:
            for r in range(k):
                p.append(d["tp"][0, s, r]); tok.append(d["ti"][0, s, r]); par.append(pi)
                nxt.append(len(p) - 1)
        level = nxt
    got, err = run_conditioned(wq, np.array([p], np.float32), np.array([tok], np.int32),
                               np.array([par], np.int32), d["root"], wq.D)
    assert err == 0
    assert_tree_equal(got, d["tree"])


def test_tree_build_conditioned_reports_malformed_forest():
    w = W.WORKLOADS["qwen"].scaled(B=2, V=50000, P=64, P_min=64)
    cp, ct, cpar = _random_forest(2, 50, seed=1)
    cpar[1, 10] = 20          # parent listed after its child: request 1 rejected
    root = torch.tensor([5, 6], dtype=torch.int32)
    got, err = run_conditioned(w, cp, ct, cpar, root, 8)
    assert err == (T.TSD_DEV_ERR_BAD_TREE | 1)
    assert got["token"][1].tolist() == [6] + [-1] * 8
    ref = oracle.tree_conditioned(cp[:1], ct[:1], cpar[:1], 8, root.numpy()[:1])
    assert got["token"][0].tolist() == ref["token"][0].tolist()


# --------------------------------------------------------- paged KV cache --

def _paged(cache, page_size, seed, spare=3):
    """Scatter a contiguous cache [B][Hkv][cap][d] (cap a multiple of
    page_size) into a shuffled page pool [num_pages][Hkv][page_size][d]."""
    B, Hkv, cap, dd = cache.shape
    mp = cap // page_size
    num_pages = B * mp + spare
    perm = np.random.default_rng(seed).permutation(num_pages)[:B * mp].reshape(B, mp)
    pool = torch.zeros((num_pages, Hkv, page_size, dd), dtype=cache.dtype)
    for b in range(B):
        for j in range(mp):
            pool[perm[b, j]] = cache[b, :, j * page_size:(j + 1) * page_size]
    return pool, torch.from_numpy(perm.astype(np.int32))


def _gather(pool, table, page_size):
    B, mp = table.shape
    return torch.cat([torch.stack([pool[int(table[b, j])] for j in range(mp)], 1)
                      .reshape(pool.shape[1], mp * page_size, pool.shape[3])[None]
                      for b in range(B)])


@pytest.mark.parametrize("name,over,page_size,force", [
    ("qwen", dict(B=3, P=900, P_min=100, V=2000), 128, "tc"),
    ("qwen", dict(B=3, P=900, P_min=100, V=2000), 256, "generic"),
    ("mla", dict(B=2, P=700, P_min=300, V=2000), 128, "tc"),
    ("toy", dict(), 128, None),
])
def test_paged_verify_equals_contiguous(name, over, page_size, force):
    """Verify through a shuffled page pool gives the same bytes as the
    contiguous cache, and matches the oracle on the gathered cache."""
    with T.verify_path(force or "auto"):
        _paged_case(name, over, page_size)


def _paged_case(name, over, page_size):
    d = inputs(name, **over)
    w = d["w"]
    cap = -(-w.cap // page_size) * page_size
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    pad = cap - kc.shape[2]
    kc = torch.nn.functional.pad(kc, (0, 0, 0, pad))
    vc = None if vc is None else torch.nn.functional.pad(vc, (0, 0, 0, pad))
    step = TreeVerifyStep(w.B, w.S, w.V, w.k, w.D, w.Hq, w.Hkv, w.dk, w.dv, cap, w.torch_dtype,
                          w.v_aliases_k, w.scale, DEV)
    step.tree.mask.copy_(torch.from_numpy(np.ascontiguousarray(d["tree"]["mask"]).view(np.int64)))
    step.verify(*gpu(q, kc, vc, plen, kt, vt))
    torch.cuda.synchronize()
    out_c, lse_c = step.out.clone(), step.lse.clone()
    kpool, table = _paged(kc, page_size, seed=7)
    vpool = None if vc is None else _paged(vc, page_size, seed=7)[0]
    g = gpu(q, kpool, vpool, table, plen, kt, vt)
    T.tsd_tree_verify_attn_paged(step.desc, g[0], g[1], g[2], g[3], page_size, g[4], g[5], g[6],
                                 step.tree.mask, step.out, step.lse, step.ws_verify, step.err)
    torch.cuda.synchronize()
    assert int(step.err[0]) == 0
    assert torch.equal(step.out, out_c) and torch.equal(step.lse, lse_c)
    kg = _gather(kpool, table, page_size)
    assert torch.equal(kg, kc)
    ref_out, _ = oracle.verify_attn(W.bits(q), W.bits(kg), None if vc is None else W.bits(vc),
                                    plen.numpy(), W.bits(kt), None if vt is None else W.bits(vt),
                                    d["tree"]["mask"], w.scale, v_aliases_k=w.v_aliases_k, dv=w.dv)
    assert np.abs(step.out.float().cpu().numpy() - ref_out).max() <= _tol(w)


@pytest.mark.parametrize("name", ["qwen", "mla"])
def test_paged_commit_equals_contiguous(name):
    d = inputs(name, B=3, P=500, P_min=100, V=2000)
    w, tree = d["w"], d["tree"]
    page_size = 128
    cap = -(-w.cap // page_size) * page_size
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    pad = cap - kc.shape[2]
    kc = torch.nn.functional.pad(kc, (0, 0, 0, pad))
    vc = None if vc is None else torch.nn.functional.pad(vc, (0, 0, 0, pad))
    step = TreeVerifyStep(w.B, w.S, w.V, w.k, w.D, w.Hq, w.Hkv, w.dk, w.dv, cap, w.torch_dtype,
                          w.v_aliases_k, w.scale, DEV)
    set_tree(step, tree)
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    step.accept(tl.to(DEV))
    kpool, table = _paged(kc, page_size, seed=3)
    vpool = None if vc is None else _paged(vc, page_size, seed=3)[0]
    gc = gpu(kt, vt, kc, vc, plen)
    step.commit(*gc)
    gp = gpu(kt, vt, kpool, vpool, table, plen)
    wk = step.walk
    T.tsd_commit_path_paged(step.desc, w.S, gp[0], gp[1], wk.accept_rows, wk.accept_len, gp[2],
                            gp[3], gp[4], page_size, gp[5], step.err)
    torch.cuda.synchronize()
    assert int(step.err[0]) == 0
    assert torch.equal(gc[4], gp[5])
    assert torch.equal(_gather(gp[2].cpu(), table, page_size), gc[2].cpu())
    if vc is not None:
        assert torch.equal(_gather(gp[3].cpu(), table, page_size), gc[3].cpu())


@pytest.mark.parametrize("name,over", [("qwen", {}), ("batched", dict(B=6, V=20000)),
                                       ("mla", dict(B=3, P=700, P_min=700, V=9000)),
                                       ("long", dict(B=2, P=2000, P_min=2000, V=7000))])
@pytest.mark.parametrize("paged", [False, True])
def test_accept_commit_matches_oracle_walk_and_commit(name, over, paged):
    """tsd_accept_commit (the walk's kernel commits the path) against the
    oracle's walk and commit; one request is placed so that its accepted path
    overflows the cache (skipped, TSD_DEV_ERR_CAPACITY)."""
    d = inputs(name, **over)
    w, tree = d["w"], d["tree"]
    page_size = 128
    cap = -(-w.cap // page_size) * page_size if paged else w.cap
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    kc = torch.nn.functional.pad(kc, (0, 0, 0, cap - kc.shape[2]))
    vc = None if vc is None else torch.nn.functional.pad(vc, (0, 0, 0, cap - vc.shape[2]))
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    tgt = oracle.argmax(tl.numpy())
    ref = oracle.accept_walk(tgt, tree, w.S)
    over_b = [b for b in range(w.B) if ref["accept_len"][b] > 0]
    if over_b:   # the last request with a non-empty path no longer fits
        b = over_b[-1]
        plen[b] = cap - int(ref["accept_len"][b])
    kc_ref = W.bits(kc).copy()
    vc_ref = None if vc is None else W.bits(vc).copy()
    pl_ref = plen.numpy().copy()
    # the oracle commit checks against the cache length it is handed
    skipped = oracle.commit(W.bits(kt), None if vt is None else W.bits(vt), ref["accept_rows"],
                            ref["accept_len"], kc_ref, vc_ref, pl_ref, w.S,
                            v_aliases_k=w.v_aliases_k)
    assert skipped == (1 if over_b else 0)

    step = TreeVerifyStep(w.B, w.S, w.V, w.k, w.D, w.Hq, w.Hkv, w.dk, w.dv, cap, w.torch_dtype,
                          w.v_aliases_k, w.scale, DEV)
    set_tree(step, tree)
    gtl, gkt, gvt, gpl = gpu(tl, kt, vt, plen)
    if paged:
        kpool, table = _paged(kc, page_size, seed=5)
        vpool = None if vc is None else _paged(vc, page_size, seed=5)[0]
        gk, gv, gtab = gpu(kpool, vpool, table)
    else:
        gk, gv = gpu(kc, vc)
        gtab = None
    t, wk = step.tree, step.walk
    T.tsd_accept_commit(gtl, w.S, t.token, t.parent, t.mask, t.is_leaf, wk.tgt, wk.accept_len,
                        wk.accept_rows, wk.bonus, wk.chain_id, step.desc, gkt, gvt, gk, gv, gpl,
                        step.ws_walk, step.err, page_table=gtab, page_size=page_size if paged else 0)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(wk.tgt.cpu().numpy(), tgt)
    for key in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(getattr(wk, key).cpu().numpy(), ref[key])
    gk_c = _gather(gk.cpu(), table, page_size) if paged else gk.cpu()
    np.testing.assert_array_equal(W.bits(gk_c), kc_ref)
    if vc is not None:
        gv_c = _gather(gv.cpu(), table, page_size) if paged else gv.cpu()
        np.testing.assert_array_equal(W.bits(gv_c), vc_ref)
    np.testing.assert_array_equal(gpl.cpu().numpy(), pl_ref)
    err = int(step.err[0])
    if over_b:
        assert err & T.TSD_DEV_ERR_MASK == T.TSD_DEV_ERR_CAPACITY and err & 0xFFFFFF == over_b[-1]
    else:
        assert err == 0


@pytest.mark.parametrize("name,over", [("qwen", {}), ("batched", dict(B=6, V=20000))])
def test_argmax_then_walk_commit_equals_the_fused_call(name, over):
    """tsd_target_argmax then tsd_walk_commit on one stream, and with the
    argmax on a second stream joined by an event, against tsd_accept_commit:
    identical outputs, cache and prefix lengths."""
    d = inputs(name, **over)
    w, tree = d["w"], d["tree"]
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    tl = W.target_logits(w, torch.from_numpy(tree["depth"]), d["logits"])
    results = []
    for mode in ("fused", "split", "two streams"):
        step = TreeVerifyStep.for_workload(w, DEV)
        set_tree(step, tree)
        gtl, gkt, gvt, gkc, gvc, gpl = gpu(tl, kt, vt, kc, vc, plen)
        t, wk = step.tree, step.walk
        main = torch.cuda.current_stream()
        if mode == "fused":
            step.accept_commit(gtl, gkt, gvt, gkc, gvc, gpl)
        else:
            side = step.side if mode == "two streams" else main
            if side is not main:
                step.ev_fork.record(main)
                side.wait_event(step.ev_fork)
            T.tsd_target_argmax(gtl, step.ws_walk, side)
            if side is not main:
                step.ev_join.record(side)
                main.wait_event(step.ev_join)
            T.tsd_walk_commit(w.V, w.S, t.token, t.parent, t.mask, t.is_leaf, wk.tgt, wk.accept_len,
                              wk.accept_rows, wk.bonus, wk.chain_id, step.desc, gkt, gvt, gkc, gvc,
                              gpl, step.ws_walk, step.err, main)
        torch.cuda.synchronize()
        results.append([x.cpu() for x in (wk.tgt, wk.accept_len, wk.accept_rows, wk.bonus,
                                          wk.chain_id, gkc, gpl, step.err)]
                       + ([] if gvc is None else [gvc.cpu()]))
    for other in results[1:]:
        for a, b in zip(results[0], other):
            assert torch.equal(a, b)


def test_paged_bad_page_is_reported_not_read():
    d = inputs("qwen", B=2, P=600, P_min=600, V=2000)
    w = d["w"]
    page_size = 128
    cap = -(-w.cap // page_size) * page_size
    q, kc, vc, plen, kt, vt = attn_inputs(w)
    kc = torch.nn.functional.pad(kc, (0, 0, 0, cap - kc.shape[2]))
    vc = torch.nn.functional.pad(vc, (0, 0, 0, cap - vc.shape[2]))
    kpool, table = _paged(kc, page_size, seed=1)
    vpool = _paged(vc, page_size, seed=1)[0]
    table[1, 2] = kpool.shape[0] + 100     # request 1, positions 256..383: outside the pool
    for force in ("tc", "generic"):
        with T.verify_path(force):
            # the workspace follows the plan of the forced path
            step = TreeVerifyStep(w.B, w.S, w.V, w.k, w.D, w.Hq, w.Hkv, w.dk, w.dv, cap,
                                  w.torch_dtype, w.v_aliases_k, w.scale, DEV)
            step.tree.mask.copy_(
                torch.from_numpy(np.ascontiguousarray(d["tree"]["mask"]).view(np.int64)))
            g = gpu(q, kpool, vpool, table, plen, kt, vt)
            T.tsd_tree_verify_attn_paged(step.desc, g[0], g[1], g[2], g[3], page_size, g[4], g[5],
                                         g[6], step.tree.mask, step.out, step.lse, step.ws_verify,
                                         step.err)
            torch.cuda.synchronize()
        assert int(step.err[0]) == (T.TSD_DEV_ERR_BAD_PAGE | 1), force
