"""Seeded synthetic inputs for the verify step.

This module generates inputs only: it performs none of the step's own
arithmetic (no top-k, no tree, no attention, no walk, no commit).  It is the
one module that both the CUDA path's tests/benchmark and the CPU oracle read
from.  All tensors are produced on the CPU with ``torch.Generator`` so that the
same bytes reach both sides.

The five workloads stand in for the public evaluation sets used on the
pages (GSM8K, MBPP, ShareGPT, MATH-500), which are not available here; none of
their items is reproduced.  Shapes follow the pages' notation s{steps}_k{topk}_d{budget}:

  toy      B=1,  V=32,     S=3, k=2,  D=4,  P=16,             Hq=2/Hkv=1,  d=64,  fp32
  qwen     B=1,  V=151936, S=7, k=8,  D=16, P=2048,           Hq=32/Hkv=8, d=128, bf16
  batched  B=32, V=151936, S=7, k=8,  D=32, P_b~U{1024..4096}, Hq=32/Hkv=8, d=128, bf16
  long     B=8,  V=151936, S=8, k=10, D=64, P=32768,          Hq=32/Hkv=8, d=128, bf16
  mla      B=64, V=129280, S=5, k=4,  D=8,  P=8192,  Hq=128/Hkv=1, dk=576, dv=512 (V=K[:512]), bf16

Draft marginals: softmax (computed once here in float64, rounded to fp32) of
N(0, sigma_draft) logits per (request, position).  Target logits for tree row r
at depth d: the draft logits of position d+1 plus N(0, sigma_target) noise
(fresh N(0, sigma_draft) logits stand in for position S+1).  Q, prefix K/V and
scratch-pad tree K/V are N(0, 1), rounded to nearest-even for bf16.
Cache capacity = max P + 1 + S.  N(mean, std) everywhere.
"""

from __future__ import annotations

import dataclasses
import math

import torch

BASE_SEED = 20260


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    V: int
    S: int
    k: int
    D: int
    P: int                 # prefix length (upper end for ragged workloads)
    P_min: int             # lower end of the uniform prefix range (== P if fixed)
    Hq: int
    Hkv: int
    dk: int
    dv: int
    dtype: str             # "f32" | "bf16"
    v_aliases_k: bool
    sigma_draft: float
    sigma_target: float

    @property
    def R(self) -> int:
        return self.D + 1

    @property
    def cap(self) -> int:
        return self.P + 1 + self.S

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def scale(self) -> float:
        # softmax scale 1/sqrt(dk), rounded to fp32 (the value both sides use)
        return float(torch.tensor(1.0 / math.sqrt(self.dk), dtype=torch.float32))

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "toy": Workload("toy", 0, B=1, V=32, S=3, k=2, D=4, P=16, P_min=16, Hq=2, Hkv=1,
                    dk=64, dv=64, dtype="f32", v_aliases_k=False,
                    sigma_draft=2.0, sigma_target=0.5),
    "qwen": Workload("qwen", 1, B=1, V=151936, S=7, k=8, D=16, P=2048, P_min=2048, Hq=32,
                     Hkv=8, dk=128, dv=128, dtype="bf16", v_aliases_k=False,
                     sigma_draft=3.0, sigma_target=1.0),
    "batched": Workload("batched", 2, B=32, V=151936, S=7, k=8, D=32, P=4096, P_min=1024,
                        Hq=32, Hkv=8, dk=128, dv=128, dtype="bf16", v_aliases_k=False,
                        sigma_draft=3.0, sigma_target=1.0),
    "long": Workload("long", 3, B=8, V=151936, S=8, k=10, D=64, P=32768, P_min=32768,
                     Hq=32, Hkv=8, dk=128, dv=128, dtype="bf16", v_aliases_k=False,
                     sigma_draft=3.0, sigma_target=1.5),
    "mla": Workload("mla", 4, B=64, V=129280, S=5, k=4, D=8, P=8192, P_min=8192, Hq=128,
                    Hkv=1, dk=576, dv=512, dtype="bf16", v_aliases_k=True,
                    sigma_draft=3.0, sigma_target=1.0),
}

# fixed sub-stream ids, so each tensor can be regenerated on its own
_STREAM = dict(draft=1, root=2, prefix=3, q=4, kcache=5, vcache=6, ktree=7, vtree=8,
               noise=9, extra=10)


def _gen(w: Workload, stream: str) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(w.seed * 1000 + _STREAM[stream])
    return g


def _normal(shape, std, gen, dtype=torch.float32):
    t = torch.empty(shape, dtype=torch.float32)
    t.normal_(0.0, std, generator=gen)
    return t if dtype == torch.float32 else t.to(dtype)


def draft_logits(w: Workload) -> torch.Tensor:
    """[B][S][V] fp32 draft logits ~ N(0, sigma_draft)."""
    return _normal((w.B, w.S, w.V), w.sigma_draft, _gen(w, "draft"))


def draft_probs(w: Workload, logits: torch.Tensor | None = None) -> torch.Tensor:
    """Per-position draft marginals [B][S][V] fp32: softmax in float64, rounded."""
    if logits is None:
        logits = draft_logits(w)
    return torch.softmax(logits.double(), dim=-1).float().contiguous()


def root_tokens(w: Workload) -> torch.Tensor:
    """[B] int32 anchor tokens, uniform over [0, V)."""
    return torch.randint(0, w.V, (w.B,), generator=_gen(w, "root"), dtype=torch.int64).int()


def prefix_lens(w: Workload) -> torch.Tensor:
    """[B] int32 prefix lengths, uniform over {P_min..P} (inclusive)."""
    if w.P_min == w.P:
        return torch.full((w.B,), w.P, dtype=torch.int32)
    return torch.randint(w.P_min, w.P + 1, (w.B,), generator=_gen(w, "prefix"),
                         dtype=torch.int64).int()


def queries(w: Workload) -> torch.Tensor:
    return _normal((w.B, w.R, w.Hq, w.dk), 1.0, _gen(w, "q"), w.torch_dtype)


def kv_cache(w: Workload):
    """(kcache [B][Hkv][cap][dk], vcache [B][Hkv][cap][dv] or None if V aliases K)."""
    k = _normal((w.B, w.Hkv, w.cap, w.dk), 1.0, _gen(w, "kcache"), w.torch_dtype)
    v = None if w.v_aliases_k else _normal((w.B, w.Hkv, w.cap, w.dv), 1.0,
                                           _gen(w, "vcache"), w.torch_dtype)
    return k, v


def tree_kv(w: Workload):
    """Scratch-pad K/V of the 1+D verified rows: [B][R][Hkv][dk] / [B][R][Hkv][dv]."""
    k = _normal((w.B, w.R, w.Hkv, w.dk), 1.0, _gen(w, "ktree"), w.torch_dtype)
    v = None if w.v_aliases_k else _normal((w.B, w.R, w.Hkv, w.dv), 1.0,
                                           _gen(w, "vtree"), w.torch_dtype)
    return k, v


def target_logits(w: Workload, depth: torch.Tensor, logits: torch.Tensor | None = None) -> torch.Tensor:
    """[B][R][V] fp32 target logits for the rows of a tree with the given depths.

    Row r at depth d gets the draft logits of position d+1 plus N(0, sigma_target)
    noise; rows at depth S get fresh N(0, sigma_draft) logits plus noise.
    ``depth`` is [B][R] (the tree's depth array).
    """
    if logits is None:
        logits = draft_logits(w)
    extra = _normal((w.B, 1, w.V), w.sigma_draft, _gen(w, "extra"))
    table = torch.cat([logits, extra], dim=1)             # [B][S+1][V]
    depth = torch.as_tensor(depth).long().clamp(0, w.S)
    base = torch.gather(table, 1, depth[:, :, None].expand(w.B, w.R, w.V))
    noise = _normal((w.B, w.R, w.V), w.sigma_target, _gen(w, "noise"))
    return (base + noise).contiguous()


def bits(t: torch.Tensor):
    """numpy view for the oracle: fp32 as float32, bf16 as raw uint16 bits."""
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
