"""One tree-verify step: device buffers plus the four C-ABI calls on one stream.

``TreeVerifyStep`` owns every output and workspace buffer of the step for a
fixed configuration, so repeated steps allocate nothing.  The inputs of a
step (draft marginals, root tokens, queries, scratch-pad K/V, target logits)
and the persistent state (KV cache, prefix lengths) are caller tensors.
"""

from __future__ import annotations

import dataclasses

import torch

from . import (make_desc, tsd_accept_commit, tsd_accept_walk, tsd_accept_walk_workspace_size,
               tsd_commit_path, tsd_target_argmax, tsd_walk_commit,
               tsd_tree_build, tsd_tree_build_adaptive, tsd_tree_build_conditioned,
               tsd_tree_build_workspace_size, tsd_tree_verify_attn, tsd_verify_workspace_size,
               workspace)


@dataclasses.dataclass
class TreeBuffers:
    token: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    score: torch.Tensor
    mask: torch.Tensor
    is_leaf: torch.Tensor


@dataclasses.dataclass
class WalkBuffers:
    tgt: torch.Tensor
    accept_len: torch.Tensor
    accept_rows: torch.Tensor
    bonus: torch.Tensor
    chain_id: torch.Tensor


class TreeVerifyStep:
    def __init__(self, B, S, V, k, D, Hq, Hkv, dk, dv, cap, dtype, v_aliases_k, scale,
                 device="cuda", overlap_argmax=None):
        self.B, self.S, self.V, self.k, self.D = B, S, V, k, D
        self.R = R = D + 1
        self.Hq, self.Hkv, self.dk, self.dv, self.cap = Hq, Hkv, dk, dv, cap
        self.dtype = dtype
        self.v_aliases_k = v_aliases_k
        self.desc = make_desc(B, R, Hq, Hkv, dk, dv, cap, dtype, v_aliases_k, scale)
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.tree = TreeBuffers(
            token=torch.empty((B, R), **i32), parent=torch.empty((B, R), **i32),
            depth=torch.empty((B, R), **i32),
            score=torch.empty((B, R), dtype=torch.float32, device=dev),
            mask=torch.empty((B, R), dtype=torch.int64, device=dev),   # uint64 bit patterns
            is_leaf=torch.empty((B, R), dtype=torch.uint8, device=dev))
        self.out = torch.empty((B, R, Hq, dv), dtype=dtype, device=dev)
        self.lse = torch.empty((B, R, Hq), dtype=torch.float32, device=dev)
        self.walk = WalkBuffers(
            tgt=torch.empty((B, R), **i32), accept_len=torch.empty((B,), **i32),
            accept_rows=torch.empty((B, S + 1), **i32), bonus=torch.empty((B,), **i32),
            chain_id=torch.empty((B,), **i32))
        self.err = torch.zeros((4,), **i32)
        self.n_nodes = torch.zeros((B,), **i32)
        self.ws_build = workspace(tsd_tree_build_workspace_size(B, S, V, k), dev)
        self.ws_verify = workspace(tsd_verify_workspace_size(self.desc), dev)
        self.ws_walk = workspace(tsd_accept_walk_workspace_size(B, D, V), dev)
        # The target argmax of a round reads only the logits, so it runs on a
        # second stream and the walk waits for it (fork and join by events,
        # also inside a captured graph).  It is forked after the tree build
        # and enqueued after the attention, so the attention's CTAs go first
        # and the argmax fills the SMs its last wave leaves idle.  Measured on
        # a GB300 (captured step): 32k prefixes 430.7 -> 423.9 us, latent heads
        # 2063 -> 2010 us, qwen-sized 33.4 -> 31.6 us, 32 requests of 1-4k
        # prefixes 231.9 -> 231.3 us.  overlap_argmax=False keeps the round on
        # one stream (the fused tsd_accept_commit).
        self.overlap_argmax = True if overlap_argmax is None else bool(overlap_argmax)
        self.side = torch.cuda.Stream(device=dev)
        self.ev_fork = torch.cuda.Event()
        self.ev_join = torch.cuda.Event()

    # the four calls -------------------------------------------------------
    def build(self, probs, root_tok, stream=None):
        t = self.tree
        tsd_tree_build(probs, self.k, self.D, root_tok, t.token, t.parent, t.depth, t.score,
                       t.mask, t.is_leaf, self.ws_build, self.err, stream)

    def build_adaptive(self, probs, root_tok, cost_d, cost_v, stream=None):
        """Tree with the cost-aware node count per request (at most D); the
        kept counts land in ``self.n_nodes``, the remaining rows are padding."""
        t = self.tree
        tsd_tree_build_adaptive(probs, self.k, self.D, root_tok, cost_d, cost_v, t.token, t.parent,
                                t.depth, t.score, t.mask, t.is_leaf, self.n_nodes, self.ws_build,
                                self.err, stream)

    def build_conditioned(self, cand_p, cand_tok, cand_parent, root_tok, stream=None):
        """Tree from parent-conditioned proposals (a candidate forest [B][C])."""
        t = self.tree
        tsd_tree_build_conditioned(cand_p, cand_tok, cand_parent, self.D, root_tok, t.token,
                                   t.parent, t.depth, t.score, t.mask, t.is_leaf, self.err,
                                   stream)

    def verify(self, q, kcache, vcache, prefix_len, ktree, vtree, stream=None):
        tsd_tree_verify_attn(self.desc, q, kcache, vcache, prefix_len, ktree, vtree,
                             self.tree.mask, self.out, self.lse, self.ws_verify, self.err, stream)

    def accept(self, logits, stream=None):
        t, w = self.tree, self.walk
        tsd_accept_walk(logits, self.S, t.token, t.parent, t.mask, t.is_leaf, w.tgt,
                        w.accept_len, w.accept_rows, w.bonus, w.chain_id, self.ws_walk, self.err,
                        stream)

    def commit(self, ktree, vtree, kcache, vcache, prefix_len, stream=None):
        w = self.walk
        tsd_commit_path(self.desc, self.S, ktree, vtree, w.accept_rows, w.accept_len, kcache,
                        vcache, prefix_len, self.err, stream)

    def accept_commit(self, logits, ktree, vtree, kcache, vcache, prefix_len, stream=None):
        """accept() then commit() as one call (the walk's kernel commits the path)."""
        t, w = self.tree, self.walk
        tsd_accept_commit(logits, self.S, t.token, t.parent, t.mask, t.is_leaf, w.tgt,
                          w.accept_len, w.accept_rows, w.bonus, w.chain_id, self.desc, ktree,
                          vtree, kcache, vcache, prefix_len, self.ws_walk, self.err, stream)

    def run(self, probs, root_tok, q, kcache, vcache, prefix_len, ktree, vtree, logits,
            stream=None):
        """The whole step: build -> verify -> walk and commit, the target argmax
        on a second stream beside the attention (asynchronous)."""
        self._round(probs, root_tok, q, kcache, vcache, prefix_len, ktree, vtree, logits, None,
                    None, stream)

    def capture(self, probs, root_tok, q, kcache, vcache, prefix_len, ktree, vtree, logits,
                cost_d=None, cost_v=None, stream=None):
        """Record the whole step as one CUDA graph on the given tensors.

        Every buffer of the step is preallocated and every shape is fixed, and
        all per-round metadata (tree rows, masks, accepted path, prefix
        lengths, and with cost tables the per-request node count) lives on the
        device, so one replay runs a full round with no host work: refill the
        captured input tensors in place, then call ``replay()`` on the
        returned graph.  With ``cost_d``/``cost_v`` the tree is built by the
        cost-aware rule (rows past each request's count are padding).
        """
        import torch

        if stream is None:
            stream = torch.cuda.Stream(device=probs.device)
        # one eager warm-up: lazy set-up (function attributes, tensor-map
        # encoder lookup) must not happen during capture
        with torch.cuda.stream(stream):
            self._round(probs, root_tok, q, kcache, vcache, prefix_len, ktree, vtree, logits,
                        cost_d, cost_v, stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self._round(probs, root_tok, q, kcache, vcache, prefix_len, ktree, vtree, logits,
                        cost_d, cost_v, stream)
        return graph

    def _round(self, probs, root_tok, q, kcache, vcache, prefix_len, ktree, vtree, logits,
               cost_d, cost_v, stream):
        main = stream if stream is not None else torch.cuda.current_stream(probs.device)
        if cost_v is None:
            self.build(probs, root_tok, main)
        else:
            self.build_adaptive(probs, root_tok, cost_d, cost_v, main)
        if self.overlap_argmax:
            self.ev_fork.record(main)
        self.verify(q, kcache, vcache, prefix_len, ktree, vtree, main)
        if not self.overlap_argmax:
            self.accept_commit(logits, ktree, vtree, kcache, vcache, prefix_len, main)
            return
        self.side.wait_event(self.ev_fork)
        tsd_target_argmax(logits, self.ws_walk, self.side)
        self.ev_join.record(self.side)
        main.wait_event(self.ev_join)
        t, w = self.tree, self.walk
        tsd_walk_commit(self.V, self.S, t.token, t.parent, t.mask, t.is_leaf, w.tgt,
                        w.accept_len, w.accept_rows, w.bonus, w.chain_id, self.desc, ktree, vtree,
                        kcache, vcache, prefix_len, self.ws_walk, self.err, main)

    @classmethod
    def for_workload(cls, w, device="cuda", overlap_argmax=None):
        return cls(w.B, w.S, w.V, w.k, w.D, w.Hq, w.Hkv, w.dk, w.dv, w.cap, w.torch_dtype,
                   w.v_aliases_k, w.scale, device, overlap_argmax)
