"""Seeded synthetic inputs for the sparse MoE FFN layer.

This module is shared by the tests, the smoke check and the benchmark.  It
draws tensors and nothing else: it holds none of the layer's arithmetic
(no softmax, top-k, grouping or expert maths).  Its one computation on the
drawn values is a rejection filter: a token whose router logits have two
near-equal values among its k+1 largest is redrawn, so that "which experts
win" is decided by a margin far above fp32 rounding (ties are decided by
rounding order, not by the method, and would make an exact comparison of the
routing meaningless).

Recipe (draw order is fixed; a fresh ``torch.Generator`` on the CPU seeded
with ``seed``):

1. ``x ~ N(0, 1)`` of shape [N, H];
2. ``router ~ N(0, 0.02)`` [E, H];
3. per expert e = 0..E-1: ``w_gate[e] ~ N(0, 0.02)`` [I, H];
4. per expert: ``w_up[e]`` [I, H];  5. per expert: ``w_down[e]`` [H, I];
6. if a shared expert is configured: ``shared_gate_proj`` [I_s, H],
   ``shared_up_proj`` [I_s, H], ``shared_down_proj`` [H, I_s] (all N(0, 0.02))
   and ``shared_gate`` [1, H] (N(0, 0.02));
7. skewed routing: ``x[:, 0] = 1`` (a bias channel), ``router[hot, 0] = 2``
   for the 8 hot experts 0..7 (a +2.0 logit offset) and
   ``router[dead, 0] = -8`` for the last 10 experts (so they receive no
   tokens);
8. every value is rounded to bf16 (round to nearest even);
9. rejection: with l = x @ router^T in fp64 on the bf16 values, a row whose
   k+1 largest logits have an adjacent gap below ``margin`` (1e-3) is
   redrawn from the same generator (then step 7's bias channel and step 8
   again) until no such row remains.

Configurations whose inputs are "fp32 cast to bf16 on the GPU" return the raw
fp32 draws; ``to_device`` performs that cast (round to nearest even, the same
rounding as step 8, so the filter saw the values the GPU will hold).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

WEIGHT_STD = 0.02
HOT_EXPERTS = 8
HOT_BIAS = 2.0
DEAD_EXPERTS = 10
DEAD_BIAS = -8.0
MARGIN = 1e-3


@dataclass(frozen=True)
class MoEShape:
    """One workload of the layer: N tokens, hidden H, E experts, top-k, expert
    intermediate I, shared-expert intermediate I_s (0 = no shared expert)."""

    name: str
    N: int
    H: int
    E: int
    k: int
    I: int
    I_s: int = 0
    norm_topk_prob: bool = True
    skew: bool = False
    cast_on_gpu: bool = False

    @property
    def pairs(self) -> int:
        return self.N * self.k

    def with_tokens(self, N: int) -> "MoEShape":
        return replace(self, N=N)


CONFIGS = {
    "tiny": MoEShape("tiny", N=16, H=64, E=6, k=2, I=128, cast_on_gpu=True),
    "decode": MoEShape("decode", N=64, H=2048, E=128, k=8, I=768),
    "prefill": MoEShape("prefill", N=8192, H=2048, E=128, k=8, I=768),
    "talker": MoEShape("talker", N=2048, H=2048, E=64, k=6, I=768, I_s=2048,
                       norm_topk_prob=False),
    "skewed": MoEShape("skewed", N=16384, H=2048, E=128, k=8, I=768, skew=True),
}

WEIGHT_KEYS = ("router", "w_gate", "w_up", "w_down")
SHARED_KEYS = ("shared_gate_proj", "shared_up_proj", "shared_down_proj", "shared_gate")


def _normal(g: torch.Generator, shape, std: float) -> torch.Tensor:
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    return t * std if std != 1.0 else t


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def _apply_skew_x(x: torch.Tensor, shape: MoEShape) -> None:
    if shape.skew:
        x[:, 0] = 1.0


def _near_tie_rows(x_bf16: torch.Tensor, router_bf16: torch.Tensor, k: int,
                   margin: float) -> torch.Tensor:
    """Indices of rows whose k+1 largest fp64 logits have a gap below margin."""
    E = router_bf16.shape[0]
    m = min(k + 1, E)
    if m < 2 or x_bf16.shape[0] == 0:
        return torch.zeros(0, dtype=torch.long)
    r = router_bf16.double()
    bad = []
    for s in range(0, x_bf16.shape[0], 4096):
        lg = x_bf16[s:s + 4096].double() @ r.T
        top = torch.topk(lg, m, dim=1).values
        gap = (top[:, :-1] - top[:, 1:]).min(dim=1).values
        bad.append(torch.nonzero(gap < margin).flatten() + s)
    return torch.cat(bad)


def make_inputs(shape: MoEShape, seed: int = 0, margin: float = MARGIN,
                max_redraws: int = 1000) -> dict:
    """Draw one seeded set of inputs for ``shape`` (CPU tensors).

    Returns a dict with x, router, w_gate, w_up, w_down and, when
    ``shape.I_s > 0``, the four shared-expert tensors.  Values are bf16, or
    the raw fp32 draws when ``shape.cast_on_gpu`` (``to_device`` casts them).
    """
    N, H, E, I, I_s = shape.N, shape.H, shape.E, shape.I, shape.I_s
    if shape.skew and E < HOT_EXPERTS + DEAD_EXPERTS + shape.k:
        raise ValueError("skewed routing needs E >= 18 + k")
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)

    # bf16 storage, or the raw fp32 draws when the cast happens on the GPU
    store = torch.float32 if shape.cast_on_gpu else torch.bfloat16

    def keep(t: torch.Tensor) -> torch.Tensor:
        return t.to(store)

    x = _normal(g, (N, H), 1.0)
    router = _normal(g, (E, H), WEIGHT_STD)
    w_gate = torch.empty((E, I, H), dtype=store)
    w_up = torch.empty((E, I, H), dtype=store)
    w_down = torch.empty((E, H, I), dtype=store)
    for e in range(E):
        w_gate[e] = keep(_normal(g, (I, H), WEIGHT_STD))
    for e in range(E):
        w_up[e] = keep(_normal(g, (I, H), WEIGHT_STD))
    for e in range(E):
        w_down[e] = keep(_normal(g, (H, I), WEIGHT_STD))
    out = {}
    if I_s > 0:
        out["shared_gate_proj"] = keep(_normal(g, (I_s, H), WEIGHT_STD))
        out["shared_up_proj"] = keep(_normal(g, (I_s, H), WEIGHT_STD))
        out["shared_down_proj"] = keep(_normal(g, (H, I_s), WEIGHT_STD))
        out["shared_gate"] = keep(_normal(g, (1, H), WEIGHT_STD))

    if shape.skew:
        router[:HOT_EXPERTS, 0] = HOT_BIAS
        router[E - DEAD_EXPERTS:, 0] = DEAD_BIAS
    _apply_skew_x(x, shape)
    router_b = _bf16(router)
    xb = _bf16(x)

    for _ in range(max_redraws):
        bad = _near_tie_rows(xb, router_b, shape.k, margin)
        if bad.numel() == 0:
            break
        fresh = _normal(g, (bad.numel(), H), 1.0)
        _apply_skew_x(fresh, shape)
        x[bad] = fresh
        xb[bad] = _bf16(fresh)
    else:
        raise RuntimeError(f"{shape.name}: near-tie rows remain after {max_redraws} redraws")

    out.update(x=keep(x), router=keep(router), w_gate=w_gate, w_up=w_up, w_down=w_down)
    return out


def make_tokens(shape: MoEShape, router: torch.Tensor, n: int, seed: int,
                margin: float = MARGIN, max_redraws: int = 1000) -> torch.Tensor:
    """Fresh activations for one step of a decode loop over a layer whose
    router is already drawn: x ~ N(0, 1) of shape [n, H] from a generator
    seeded with ``seed``, the skew bias channel when ``shape.skew``, rounded
    to bf16, with near-tie rows (against ``router``, bf16 [E, H]) redrawn as
    in ``make_inputs``.  Returns a bf16 CPU tensor."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = _normal(g, (n, shape.H), 1.0)
    _apply_skew_x(x, shape)
    xb = _bf16(x)
    router_b = router.to("cpu", torch.bfloat16)
    for _ in range(max_redraws):
        bad = _near_tie_rows(xb, router_b, shape.k, margin)
        if bad.numel() == 0:
            return xb
        fresh = _normal(g, (bad.numel(), shape.H), 1.0)
        _apply_skew_x(fresh, shape)
        xb[bad] = _bf16(fresh)
    raise RuntimeError(f"{shape.name}: near-tie rows remain after {max_redraws} redraws")


def to_device(inputs: dict, device="cuda") -> dict:
    """Move inputs to ``device``; fp32 tensors are cast to bf16 there."""
    dev = {}
    for name, t in inputs.items():
        t = t.to(device)
        if t.dtype == torch.float32:
            t = t.to(torch.bfloat16)
        dev[name] = t.contiguous()
    return dev
