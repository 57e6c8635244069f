"""Seeded synthetic router inputs for the MoE route-sort workloads.

This module only draws numbers: it holds none of the routing arithmetic, so both the CUDA
path's tests/benchmark and the CPU oracle's tests can share it.  Where a workload needs a
token redrawn (a near-tie in the selection), the caller passes a ``needs_redraw`` callback
that decides which rows to redraw; the generator just draws the replacement rows from the
same random stream.

Recipe (numpy ``default_rng(seed)``, PCG64), in draw order:
  1. skewed workloads only: ``perm = rng.permutation(E)``, ``rank_e = 1 + perm[e]``,
     per-expert logit offset ``0.5 * ln(rank_e ** -1.1)`` (a few experts are hot);
  2. bias: ``rng.uniform(-h, h, E)`` in float64, rounded to float32;
  3. logits: ``rng.standard_normal((T, E)) * std + offset`` in float64, rounded to float32,
     then to bf16 by round-to-nearest-even on the float32 bit pattern;
  4. redraws: for each row the callback names (ascending), ``E`` new normals from the same
     stream with the same recipe; repeated until the callback names no row (at most
     ``max_rounds`` rounds, else an error).

Gate-projection inputs (``make_gate_inputs``: hidden states and gate rows that produce the
logits), numpy ``default_rng(seed)``, in draw order:
  1. bias as in step 2 above;
  2. gate rows ``rng.integers(-3, 4, (E, H)) / 64``;
  3. hidden rows ``rng.integers(-16, 17, (T, H)) / 16``;
  4. redraws of hidden rows as in step 4 above.
Both grids are exact in bf16, and every partial sum of a dot product is a multiple of 2^-10
below 2^9 (H <= 8192), so a float32 accumulation of it is exact in any order.  With H = 7168
the logits have a standard deviation of about 1.6.  ``grid="general"`` draws instead, in the
same order, gate rows ``rng.standard_normal((E, H)) / sqrt(H)`` and hidden rows
``rng.standard_normal((T, H))``, both rounded to bf16 (logits of standard deviation about 1,
whose float32 sums are rounded).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Callable, Iterable, Optional

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    E: int
    n_group: int
    topk_group: int
    topk: int
    routed_scale: float
    block_m: int
    logit_std: float = 1.0
    bias_half_range: float = 0.1
    skewed: bool = False
    seed: int = 0

    @property
    def routes(self) -> int:
        return self.T * self.topk


# The five workloads: Kimi-K3-shaped TP8 decode (E=896, top-16), the 512-token prefill at
# which the gfx1250 workgroup-histogram route is enabled for E=896, a skewed 8192-token
# prefill, a 4096-expert wide set, and a tiny case for the oracle.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_T4_E64", T=4, E=64, n_group=8, topk_group=4, topk=6, routed_scale=2.5,
                 block_m=16),
        Workload("decode_T1_E896_G8", T=1, E=896, n_group=8, topk_group=4, topk=16,
                 routed_scale=2.5, block_m=32),
        Workload("decode_T1_E896_G1", T=1, E=896, n_group=1, topk_group=1, topk=16,
                 routed_scale=2.5, block_m=32),
        Workload("prefill_T512_E896", T=512, E=896, n_group=8, topk_group=4, topk=16,
                 routed_scale=2.5, block_m=32, logit_std=1.5),
        Workload("skewed_T8192_E896", T=8192, E=896, n_group=8, topk_group=4, topk=16,
                 routed_scale=2.5, block_m=64, skewed=True),
        Workload("wide_T16384_E4096", T=16384, E=4096, n_group=16, topk_group=4, topk=8,
                 routed_scale=1.0, block_m=128, bias_half_range=0.05),
    ]
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


@dataclass
class RouterInputs:
    workload: Workload
    logits_bf16: np.ndarray  # uint16 [T, E], bf16 bit patterns, row-major
    bias: np.ndarray  # float32 [E]
    redrawn_rows: int = 0


class _Stream:
    def __init__(self, w: Workload):
        self.w = w
        self.rng = np.random.default_rng(w.seed)
        if w.skewed:
            perm = self.rng.permutation(w.E)
            rank = 1.0 + perm.astype(np.float64)
            self.offset = 0.5 * np.log(rank ** -1.1)
        else:
            self.offset = np.zeros(w.E, np.float64)

    def bias(self) -> np.ndarray:
        h = self.w.bias_half_range
        return self.rng.uniform(-h, h, self.w.E).astype(np.float32)

    def rows(self, n: int) -> np.ndarray:
        z = self.rng.standard_normal((n, self.w.E)) * self.w.logit_std + self.offset
        return float32_to_bf16_bits(z.astype(np.float32))


def make_inputs(
    w: Workload,
    needs_redraw: Optional[Callable[[np.ndarray, np.ndarray], Iterable[int]]] = None,
    max_rounds: int = 64,
    T: Optional[int] = None,
) -> RouterInputs:
    """Draw the inputs of workload ``w`` (optionally with ``T`` tokens instead of ``w.T``)."""
    if T is not None:
        w = replace(w, T=T)
    st = _Stream(w)
    bias = st.bias()
    logits = st.rows(w.T)
    redrawn = 0
    if needs_redraw is not None and w.T > 0:
        rows = sorted(set(int(r) for r in needs_redraw(logits, bias)))
        rounds = 0
        while rows:
            rounds += 1
            if rounds > max_rounds:
                raise RuntimeError(
                    f"{w.name}: near-tie rows remain after {max_rounds} redraw rounds: {rows[:8]}"
                )
            logits[rows] = st.rows(len(rows))
            redrawn += len(rows)
            sub = needs_redraw(logits[rows], bias)
            rows = sorted(rows[int(i)] for i in sub)
    return RouterInputs(w, logits, bias, redrawn)


@dataclass
class GateInputs:
    hidden_bf16: np.ndarray  # uint16 [T, H], bf16 bit patterns
    w_gate_bf16: np.ndarray  # uint16 [E, H], one gate row per expert
    bias: np.ndarray  # float32 [E]
    redrawn_rows: int = 0


def make_gate_inputs(
    T: int,
    E: int,
    H: int,
    bias_half_range: float = 0.1,
    seed: int = 0,
    needs_redraw: Optional[Callable[[np.ndarray, np.ndarray, np.ndarray], Iterable[int]]] = None,
    max_rounds: int = 64,
    grid: str = "coarse",
) -> GateInputs:
    """Draw hidden states and gate rows on the coarse grids of the recipe above (or, with
    ``grid="general"``, general normal values rounded to bf16)."""
    if grid not in ("coarse", "general"):
        raise ValueError(f"unknown grid {grid!r}")
    rng = np.random.default_rng(seed)
    bias = rng.uniform(-bias_half_range, bias_half_range, E).astype(np.float32)
    if grid == "coarse":
        w = float32_to_bf16_bits((rng.integers(-3, 4, (E, H)) / 64.0).astype(np.float32))
    else:
        w = float32_to_bf16_bits((rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32))

    def rows(n):
        if grid == "general":
            return float32_to_bf16_bits(rng.standard_normal((n, H)).astype(np.float32))
        return float32_to_bf16_bits((rng.integers(-16, 17, (n, H)) / 16.0).astype(np.float32))

    hidden = rows(T)
    redrawn = 0
    if needs_redraw is not None and T > 0:
        todo = sorted(set(int(r) for r in needs_redraw(hidden, w, bias)))
        rounds = 0
        while todo:
            rounds += 1
            if rounds > max_rounds:
                raise RuntimeError(f"near-tie hidden rows remain after {max_rounds} rounds")
            hidden[todo] = rows(len(todo))
            redrawn += len(todo)
            sub = needs_redraw(hidden[todo], w, bias)
            todo = sorted(todo[int(i)] for i in sub)
    return GateInputs(hidden, w, bias, redrawn)
