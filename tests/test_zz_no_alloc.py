"""The allocation-free accept walk (tsd_accept_walk_static) against the CPU
oracle and against the workspace version (tsd_accept_walk).

tsd_accept_walk_static serves callers that are handed only their input and
output buffers and may not allocate device memory (for example a custom
operator inside a framework that owns the device heap).  Its scratch is a
fixed array inside the library, shared by every call, so these tests make
calls in a row and check every one against the oracle's argmax and greedy
walk and against the workspace entry point.  The file is collected last, and
its tests also pass alone in a fresh process (the first call on a device
looks up the array's address).
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LIMIT = 1 << 20          # bytes of the library's fixed scratch


def _walk(fn, logits, S, tree, ws=None, stream=None):
    B, R, _ = logits.shape
    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(tgt=torch.full((B, R), -7, **i32), accept_len=torch.full((B,), -7, **i32),
               accept_rows=torch.full((B, S + 1), -7, **i32), bonus=torch.full((B,), -7, **i32),
               chain_id=torch.full((B,), -7, **i32))
    err = torch.zeros(4, **i32)
    args = [logits, S, tree["token"], tree["parent"], tree["mask"], tree["is_leaf"], out["tgt"],
            out["accept_len"], out["accept_rows"], out["bonus"], out["chain_id"]]
    if ws is not None:
        args.append(ws)
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())
    fn(*args, err=err, stream=stream)
    if stream is not None:
        stream.synchronize()
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def _check_oracle(got, logits_cpu, tree_np, S, what):
    import oracle
    tgt = oracle.argmax(logits_cpu.numpy())
    ref = oracle.accept_walk(tgt, tree_np, S)
    np.testing.assert_array_equal(got["tgt"], tgt, err_msg=f"{what}: tgt")
    for k in ("accept_len", "accept_rows", "bonus", "chain_id"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{what}: {k}")


def _dev_tree(tree):
    return {k: torch.from_numpy(np.ascontiguousarray(
        v.view(np.int64) if k == "mask" else v)).to(DEV) for k, v in tree.items()}


def test_static_scratch_walk_matches_oracle_twice():
    import oracle
    import tree_speculative_decoding_tsd_gb300 as T
    from tree_speculative_decoding_tsd_gb300 import workloads as W

    for name, over in [("qwen", {}), ("batched", dict(B=8, V=40000))]:
        w = W.WORKLOADS[name].scaled(**over) if over else W.WORKLOADS[name]
        lg = W.draft_logits(w)
        tp, ti = oracle.topk(W.draft_probs(w, lg).numpy(), w.k)
        tree = oracle.tree(tp, ti, w.D, W.root_tokens(w).numpy(), method="beam")
        dev_tree = _dev_tree(tree)
        ws = T.workspace(T.tsd_accept_walk_workspace_size(w.B, w.D, w.V), DEV)
        first = second = None
        for call in range(2):
            # a different batch of target logits on each call
            g = torch.Generator().manual_seed(100 + call)
            tl_cpu = (W.target_logits(w, torch.from_numpy(tree["depth"]), lg)
                      + torch.randn((w.B, w.R, w.V), generator=g)).contiguous()
            tl = tl_cpu.to(DEV)
            got = _walk(T.tsd_accept_walk_static, tl, w.S, dev_tree)
            _check_oracle(got, tl_cpu, tree, w.S, f"{name} call {call}")
            ref = _walk(T.tsd_accept_walk, tl, w.S, dev_tree, ws)
            for k in ref:
                np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{name} call {call}: {k}")
            if call == 0:
                first = got
            else:
                second = got
        assert not np.array_equal(first["tgt"], second["tgt"])   # the two calls differ


def test_static_scratch_walk_at_its_size_limit_on_a_side_stream():
    """A batch whose scratch is exactly the 1 MiB the library holds (2048
    requests of 64 rows, one 8-byte candidate per row) runs on a non-default
    stream and matches the oracle; one more request is refused."""
    import oracle
    import tree_speculative_decoding_tsd_gb300 as T

    S, k, D, V = 3, 4, 63, 100
    B = LIMIT // (8 * (D + 1))
    assert T.tsd_accept_walk_workspace_size(B, D, V) == LIMIT
    assert T.tsd_accept_walk_workspace_size(B + 1, D, V) > LIMIT
    rng = np.random.default_rng(5)
    probs = rng.random((B, S, V)).astype(np.float32)
    probs /= probs.sum(-1, keepdims=True)
    tp, ti = oracle.topk(probs, k)
    tree = oracle.tree(tp, ti, D, rng.integers(0, V, B).astype(np.int32), method="beam")
    logits = rng.standard_normal((B, D + 1, V)).astype(np.float32)
    # plant the first child chain in half of the requests so walks go deep
    for b in range(0, B, 2):
        u = 0
        for _ in range(S):
            kids = np.nonzero(tree["parent"][b] == u)[0]
            if len(kids) == 0:
                break
            c = int(kids[0])
            logits[b, u, tree["token"][b, c]] = 10.0
            u = c
    tl_cpu = torch.from_numpy(logits)
    tl = tl_cpu.to(DEV)
    dev_tree = _dev_tree(tree)
    side = torch.cuda.Stream(device=DEV)
    for call in range(2):
        got = _walk(T.tsd_accept_walk_static, tl, S, dev_tree, stream=side)
        _check_oracle(got, tl_cpu, tree, S, f"limit call {call}")
    assert (got["accept_len"][::2] >= 1).all()
    # one request more than the scratch holds: refused before any launch
    big = torch.empty((B + 1, D + 1, V), dtype=torch.float32, device=DEV)
    t1 = {kk: torch.cat([v, v[:1]]) for kk, v in dev_tree.items()}
    with pytest.raises(T.TsdError) as e:
        _walk(T.tsd_accept_walk_static, big, S, t1, stream=side)
    assert e.value.status == T.TSD_ERR_UNSUPPORTED


def test_static_scratch_walk_rejects_sizes_beyond_its_scratch():
    import tree_speculative_decoding_tsd_gb300 as T
    B, D, V = 4096, 64, 151936                  # needs far more than 1 MiB of scratch
    assert T.tsd_accept_walk_workspace_size(B, D, V) > LIMIT
    A = torch.empty(16, dtype=torch.uint8, device=DEV)
    p = A.data_ptr()
    st = T.lib.tsd_accept_walk_static(p, B, D, 7, V, p, p, p, p, None, p, p, p, p, None, None)
    assert st == T.TSD_ERR_UNSUPPORTED
