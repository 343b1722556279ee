"""Verify-cost model for the cost-aware tree budget.

Source: "Cost-Aware Diffusion Draft Trees for Speculative Decoding", Method
items 1, 4 and 5: a round costs C_d + C_v(n; l) (drafting plus verifying n
draft nodes at context length l); C_v is estimated once, offline, by convex
regression on latencies measured over node counts and context lengths, which
keeps it convex and monotone so that the throughput objective is unimodal in
n and the greedy stop of ``tsd_tree_build_adaptive`` finds its maximum.

Here the latencies are this library's own: C_d is the draft-side call
(``tsd_tree_build``: top-k scan and tree) and C_v(n; l) the verify-side calls
(attention, argmax walk, commit) of a step with budget n at prefix length l,
timed with CUDA events.  For each measured l the fit is the least-squares
projection onto convex, non-decreasing functions of n that are piecewise
linear with knots at the measured n (non-negative coefficients on the basis
1, n, max(0, n - n_j)); between measured l the curves are interpolated
linearly, which keeps convexity and monotonicity in n.
"""

from __future__ import annotations

import numpy as np


def _basis(n, knots):
    n = np.asarray(n, np.float64)
    cols = [np.ones_like(n), n] + [np.maximum(0.0, n - k) for k in knots]
    return np.stack(cols, axis=1)


def fit_convex_nondecreasing(n, y):
    """Coefficients of the least-squares convex, non-decreasing, piecewise
    linear fit of samples (n_i, y_i), knots at the interior sample points."""
    from scipy.optimize import nnls

    n = np.asarray(n, np.float64)
    y = np.asarray(y, np.float64)
    knots = np.unique(n)[1:-1]
    coef, _ = nnls(_basis(n, knots), y)
    return coef, knots


def eval_fit(fit, n):
    coef, knots = fit
    return _basis(n, knots) @ coef


class CostModel:
    """C_d and C_v(n; l): fits at measured context lengths, linear in between."""

    def __init__(self, cost_d, ells, fits):
        order = np.argsort(ells)
        self.cost_d = float(cost_d)
        self.ells = np.asarray(ells, np.float64)[order]
        self.fits = [fits[i] for i in order]

    @classmethod
    def from_samples(cls, cost_d, samples):
        """samples: {l: (list of n, list of latency)}."""
        ells = sorted(samples)
        fits = [fit_convex_nondecreasing(*samples[l]) for l in ells]
        return cls(cost_d, ells, fits)

    def verify_cost(self, ell, D_max):
        """C_v(n; ell) for n = 0..D_max (fp32)."""
        n = np.arange(D_max + 1, dtype=np.float64)
        curves = [eval_fit(f, n) for f in self.fits]
        if ell <= self.ells[0] or len(self.ells) == 1:
            c = curves[0]
        elif ell >= self.ells[-1]:
            c = curves[-1]
        else:
            i = int(np.searchsorted(self.ells, ell)) - 1
            u = (ell - self.ells[i]) / (self.ells[i + 1] - self.ells[i])
            c = (1.0 - u) * curves[i] + u * curves[i + 1]
        return c.astype(np.float32)

    def tables(self, ells, D_max):
        """Per-request arguments of tsd_tree_build_adaptive: cost_d [B],
        cost_v [B][D_max + 1] (fp32)."""
        cost_v = np.stack([self.verify_cost(float(l), D_max) for l in ells])
        cost_d = np.full(len(ells), self.cost_d, np.float32)
        return cost_d, cost_v


def measure(workload, budgets, prefix_lens, steps=10, warmup=3, device="cuda"):
    """Time the step of `workload` at each budget n and prefix length l on the
    GPU.  Returns (C_d, {l: (ns, verify-side latencies)}) in microseconds."""
    import torch

    from . import workloads as W
    from .step import TreeVerifyStep

    dev = torch.device(device)
    samples = {}
    draft = []
    for ell in prefix_lens:
        ns, lat = [], []
        for n in budgets:
            w = workload.scaled(D=n, P=ell, P_min=ell)
            probs = W.draft_probs(w, W.draft_logits(w)).to(dev)
            root = W.root_tokens(w).to(dev)
            q = W.queries(w).to(dev)
            kc, vc = W.kv_cache(w)
            kt, vt = W.tree_kv(w)
            kc, kt = kc.to(dev), kt.to(dev)
            vc = None if vc is None else vc.to(dev)
            vt = None if vt is None else vt.to(dev)
            plen0 = W.prefix_lens(w).to(dev)
            plen = plen0.clone()
            step = TreeVerifyStep.for_workload(w, dev)
            stream = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(stream):
                step.build(probs, root, stream)
            torch.cuda.synchronize(dev)
            logits = W.target_logits(w, step.tree.depth.cpu(), W.draft_logits(w)).to(dev)
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
            with torch.cuda.stream(stream):
                for i in range(warmup + steps):
                    plen.copy_(plen0)
                    e = ev[i - warmup] if i >= warmup else None
                    if e is not None:
                        e[0].record(stream)
                    step.build(probs, root, stream)
                    if e is not None:
                        e[1].record(stream)
                    step.verify(q, kc, vc, plen, kt, vt, stream)
                    step.accept(logits, stream)
                    step.commit(kt, vt, kc, vc, plen, stream)
                    if e is not None:
                        e[2].record(stream)
            torch.cuda.synchronize(dev)
            draft += [e[0].elapsed_time(e[1]) * 1e3 for e in ev]
            ns.append(n)
            lat.append(float(np.median([e[1].elapsed_time(e[2]) * 1e3 for e in ev])))
        samples[ell] = (ns, lat)
    return float(np.median(draft)), samples
