"""The allocation-free accept walk (tsd_accept_walk_static) against the
workspace version (tsd_accept_walk).

tsd_accept_walk_static serves callers that are handed only their input and
output buffers and may not allocate device memory (for example a custom
operator inside a framework that owns the device heap).  Its scratch is a
fixed array inside the library, shared by every call, so this test makes two
calls in a row and checks both against the workspace entry point.  It lives in
a file of its own, collected last, and also passes alone in a fresh process
(the first call on a device looks up the array's address).
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _walk(fn, T, logits, S, tree, ws=None):
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
    fn(*args, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_static_scratch_walk_matches_workspace_walk_twice():
    import oracle
    import tree_speculative_decoding_tsd_gb300 as T
    from tree_speculative_decoding_tsd_gb300 import workloads as W

    for name, over in [("qwen", {}), ("batched", dict(B=8, V=40000))]:
        w = W.WORKLOADS[name].scaled(**over) if over else W.WORKLOADS[name]
        lg = W.draft_logits(w)
        tp, ti = oracle.topk(W.draft_probs(w, lg).numpy(), w.k)
        tree = oracle.tree(tp, ti, w.D, W.root_tokens(w).numpy(), method="beam")
        dev_tree = {k: torch.from_numpy(np.ascontiguousarray(
            v.view(np.int64) if k == "mask" else v)).to(DEV) for k, v in tree.items()}
        ws = T.workspace(T.tsd_accept_walk_workspace_size(w.B, w.D, w.V), DEV)
        first = second = None
        for call in range(2):
            # a different batch of target logits on each call
            g = torch.Generator().manual_seed(100 + call)
            tl = (W.target_logits(w, torch.from_numpy(tree["depth"]), lg)
                  + torch.randn((w.B, w.R, w.V), generator=g)).contiguous().to(DEV)
            ref = _walk(T.tsd_accept_walk, T, tl, w.S, dev_tree, ws)
            got = _walk(T.tsd_accept_walk_static, T, tl, w.S, dev_tree)
            for k in ref:
                np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{name} call {call}: {k}")
            if call == 0:
                first = got
            else:
                second = got
        assert not np.array_equal(first["tgt"], second["tgt"])   # the two calls differ


def test_static_scratch_walk_rejects_sizes_beyond_its_scratch():
    import tree_speculative_decoding_tsd_gb300 as T
    B, D, V = 4096, 64, 151936                  # needs far more than 1 MiB of scratch
    assert T.tsd_accept_walk_workspace_size(B, D, V) > (1 << 20)
    A = torch.empty(16, dtype=torch.uint8, device=DEV)
    p = A.data_ptr()
    st = T.lib.tsd_accept_walk_static(p, B, D, 7, V, p, p, p, p, None, p, p, p, p, None, None)
    assert st == T.TSD_ERR_UNSUPPORTED
