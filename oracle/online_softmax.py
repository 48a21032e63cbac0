"""Tiled online-softmax recurrence for one query row (fp64, pure Python).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Restates the tutorial page "research-attention", section 02: every row keeps
three pieces of state over the keys seen so far -- the running maximum m, the
sum l of exp(s - m) and the unnormalised vector u = sum exp(s - m) v. When a
new block of scores arrives the old state is moved to the new base
m' = max(m, max of block) by alpha = exp(m - m'), the block's weights
p = exp(s - m') are added, and the output is u / l once all blocks are in.
The statistic saved for the backward pass is L = m + log(l) (section 04).

Reading for a block whose scores are all -inf while m is still -inf (a fully
masked tile with no history): exp(-inf - (-inf)) is undefined, so alpha is
taken as 1 and the block's weights as 0, which leaves the state unchanged.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Sequence


@dataclass
class RowState:
    m: float = -math.inf
    l: float = 0.0
    u: List[float] = field(default_factory=list)


def _exp_shift(x: float, base: float) -> float:
    if x == -math.inf:
        return 0.0
    return math.exp(x - base)


def absorb_block(state: RowState, scores: Sequence[float], values: Sequence[Sequence[float]]) -> RowState:
    """One step of the recurrence: fold a block of (score, value) pairs in."""
    if not state.u:
        state.u = [0.0] * len(values[0])
    m_new = max([state.m] + list(scores))
    alpha = 1.0 if m_new == -math.inf else _exp_shift(state.m, m_new)
    if m_new == -math.inf:
        weights = [0.0] * len(scores)
    else:
        weights = [_exp_shift(s, m_new) for s in scores]
    l_new = alpha * state.l + sum(weights)
    u_new = []
    for c, old in enumerate(state.u):
        u_new.append(alpha * old + sum(w * values[j][c] for j, w in enumerate(weights)))
    return RowState(m=m_new, l=l_new, u=u_new)


def tiled_row(scores: Sequence[float], values: Sequence[Sequence[float]], tile: int):
    """Run the recurrence over consecutive blocks of ``tile`` keys.

    Returns (o, L, states) where o = u / l, L = m + log(l) and ``states`` is the
    state after each block (for checking intermediate values).
    """
    if tile < 1:
        raise ValueError("tile must be >= 1")
    state = RowState()
    states = []
    for start in range(0, len(scores), tile):
        state = absorb_block(state, scores[start:start + tile], values[start:start + tile])
        states.append(RowState(m=state.m, l=state.l, u=list(state.u)))
    o = [x / state.l for x in state.u]
    return o, state.m + math.log(state.l), states
