"""One FlashLoop loop on the CPU oracle, composed from the steps in ``oracle``.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``). The order of the steps is
the one the rit.work page "FlashLoop: Fast and Memory-Efficient Looped
Transformers via Lazy Updates" gives in its section "FlashLoop combines three
kinds of saving": early loops run in full; later loops rank tokens by change
and recompute only the active ones, write low-bit KV deltas for them, choose
keys from the previous loop's statistics and attend with preserved mass.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from . import DeltaLayer, attention, bits, kv_delta_append, reconstruct, token_scores, topk


@dataclasses.dataclass
class Cache:
    """Per-loop KV: bf16 layers of the dense loops, delta layers after them."""

    dense_k: List[np.ndarray] = dataclasses.field(default_factory=list)
    dense_v: List[np.ndarray] = dataclasses.field(default_factory=list)
    delta_k: List[DeltaLayer] = dataclasses.field(default_factory=list)
    delta_v: List[DeltaLayer] = dataclasses.field(default_factory=list)

    def rec(self, loop: int, which: str) -> np.ndarray:
        """K_rec^{(loop)} (or V) as bf16 bits [B,Nk,H,d]."""
        dense = self.dense_k if which == "k" else self.dense_v
        deltas = self.delta_k if which == "k" else self.delta_v
        td = len(dense)
        if loop <= td:
            return dense[loop - 1]
        _, h = reconstruct(dense[-1], deltas[: loop - td], want_f32=False)
        return h


@dataclasses.dataclass
class State:
    qhat: np.ndarray    # [B,N,H,d] bf16 bits
    o: np.ndarray       # [B,N,H,d] f32
    z: np.ndarray       # [B,H,N] f32
    c: np.ndarray       # [B,H,N] f32


def empty_state(B, N, H, d) -> State:
    return State(np.zeros((B, N, H, d), np.uint16), np.zeros((B, N, H, d), np.float32),
                 np.zeros((B, H, N), np.float32), np.zeros((B, H, N), np.float32))


def dense_loop(loop: int, q, k, v, cache: Cache, state: State, bh_mask=None) -> State:
    """A dense loop: every row, every key; stores a full bf16 KV layer."""
    q, k, v = bits(q), bits(k), bits(v)
    B, N, H, d = q.shape
    first = loop == 1
    k_old = None if first else cache.dense_k[-1]
    v_old = None if first else cache.dense_v[-1]
    cache.dense_k.append(np.array(k, copy=True))
    cache.dense_v.append(np.array(v, copy=True))
    rows = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    S = np.tile(np.arange(N, dtype=np.int32), (B, H, 1))
    qh, o, z, c, _ = attention(first, rows, rows, q, state.qhat, state.o, state.z, state.c, S,
                               k_old, v_old, k, v, bh_mask=bh_mask)
    return State(qh, o, z, c)


def exit_flags(scores: np.ndarray, threshold: float, exited: Optional[np.ndarray] = None) -> np.ndarray:
    """Early exit by state difference (the recurrent-depth overview page's
    dynamic early exit: a sequence stops looping once its state stops
    changing): a sequence is flagged once its largest token change score
    falls below ``threshold``, and stays flagged. The comparison is made in
    fp32, on the fp32 rounding of the largest score."""
    B = scores.shape[0]
    ex = np.zeros(B, bool) if exited is None else np.asarray(exited, bool).copy()
    if threshold > 0:
        ex |= np.float32(scores.max(axis=-1)) < np.float32(threshold)
    return ex


def lazy_loop(loop: int, h_prev, h_cur, q, k, v, cache: Cache, state: State, R: int, K: int,
              A: Optional[np.ndarray] = None, S: Optional[np.ndarray] = None, bh_mask=None,
              exit_threshold: float = 0.0, exited: Optional[np.ndarray] = None):
    """A lazy loop. ``A``/``S`` override the selections (teacher forcing).
    With ``exited`` (per-sequence flags) or ``exit_threshold`` > 0, a flagged
    sequence stops looping: its delta entries hold zero deltas (scale 0,
    codes 0) and its rows keep their state; the flags come back as the last
    element of the result.

    Returns (A, S, scores, new_state, new_k_layer, new_v_layer[, flags]).
    """
    q, k, v = bits(q), bits(k), bits(v)
    B, N, H, d = q.shape
    scores = token_scores(h_prev, h_cur)
    use_exit = exited is not None or exit_threshold > 0
    flags = exit_flags(scores, exit_threshold, exited) if use_exit else np.zeros(B, bool)
    if A is None:
        A = topk(scores, R)
    if S is None:
        S = topk(state.c.astype(np.float64), K)
    td = len(cache.dense_k)
    lk = kv_delta_append(k, cache.dense_k[-1], cache.delta_k[: loop - 1 - td], A)
    lv = kv_delta_append(v, cache.dense_v[-1], cache.delta_v[: loop - 1 - td], A)
    for lay in (lk, lv):          # a sequence that stopped looping keeps its K/V
        lay.codes[flags] = 0
        lay.scales[flags] = 0
    k_old, v_old = cache.rec(loop - 1, "k"), cache.rec(loop - 1, "v")
    del cache.delta_k[loop - 1 - td:], cache.delta_v[loop - 1 - td:]
    cache.delta_k.append(lk)
    cache.delta_v.append(lv)
    k_new, v_new = cache.rec(loop, "k"), cache.rec(loop, "v")
    qh, o, z, c, _ = attention(False, A, A, q, state.qhat, state.o, state.z, state.c, S,
                               k_old, v_old, k_new, v_new, bh_mask=bh_mask)
    # rows of a sequence that stopped looping keep their state
    qh[flags], o[flags], z[flags], c[flags] = state.qhat[flags], state.o[flags], state.z[flags], state.c[flags]
    if use_exit:
        return A, S, scores, State(qh, o, z, c), lk, lv, flags
    return A, S, scores, State(qh, o, z, c), lk, lv
