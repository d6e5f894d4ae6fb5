"""The synthetic looped block around the lazy loop, on the CPU oracle.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``). The rit.work page
"FlashLoop: Fast and Memory-Efficient Looped Transformers via Lazy Updates",
section "FlashLoop combines three kinds of saving", says a later loop
recomputes only its active tokens while the rest reuse their state; it gives
no block. The block here is reading R9 of ``flashloop_oracle.c``: one
weight-shared block of attention and a ReLU MLP with residuals and no
normalisation, applied every loop,

    q, k, v = bf16(x W_q), bf16(x W_k), bf16(x W_v)       x = H_{l-1}[i]
    (the loop's attention, ``loop.dense_loop`` / ``loop.lazy_loop``)  -> O_i
    y = bf16(x + bf16(O_i) W_o)
    u = bf16(relu(y W_1))
    H_l[i] = bf16(y + u W_2)

for every token of a dense loop and the active tokens of a lazy loop; the
other tokens keep H_l[i] = H_{l-1}[i]. Weights are stored transposed,
[out features, in features] bf16 bits, with w_qkv's rows 0..D-1 giving q,
D..2D-1 k and 2D..3D-1 v. Products are summed exactly (numpy's float64
matmul of bf16 values; its rounding error is far below bf16's) and each
output is rounded once to bf16 by ``round_bf16``.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import bf16_values, bits, key_scores_per_row, round_bf16, token_scores, topk
from .loop import Cache, State, dense_loop, lazy_loop


def project(x, w_t, residual=None, relu: bool = False) -> np.ndarray:
    """bf16(act(x W + residual)) with W given as w_t = W^T [N_out, K_in]:
    x [..., K_in] bf16 bits -> [..., N_out] bf16 bits."""
    acc = bf16_values(x) @ bf16_values(w_t).T
    if residual is not None:
        acc = acc + bf16_values(residual)
    if relu:
        acc = np.maximum(acc, 0.0)
    return round_bf16(acc)


def split_qkv(qkv: np.ndarray, H: int, d: int):
    """The q, k, v parts of a projection by w_qkv, each [..., H, d]."""
    D = H * d
    lead = qkv.shape[:-1]
    return tuple(np.ascontiguousarray(qkv[..., i * D:(i + 1) * D]).reshape(lead + (H, d)) for i in range(3))


def mlp(x, a, weights):
    """The block after the attention, for input rows x and attention outputs
    a = bf16(O) (bf16 bits, [..., D]): y = bf16(x + a W_o),
    u = bf16(relu(y W_1)), h = bf16(y + u W_2); returns h."""
    _, w_o, w_1, w_2 = weights
    y = project(a, w_o, residual=x)
    u = project(y, w_1, relu=True)
    return project(u, w_2, residual=y)


def block_loop(loop: int, weights: Sequence[np.ndarray], h_prev, h_cur, cache: Cache, state: State,
               T_dense: int, H: int, d: int, R: int = 0, K: int = 0, A: Optional[np.ndarray] = None,
               S: Optional[np.ndarray] = None, key_rank: int = 0):
    """One loop of the block. h_prev = H_{l-2} (lazy loops), h_cur = H_{l-1},
    both [B, N, D] bf16 bits. ``A``/``S`` override the token and key
    selections (teacher forcing); key_rank 1 ranks keys by column mass per
    causal row. Returns (h_out, state, A, S) with A, S None for a dense loop.
    """
    h_cur = bits(h_cur)
    B, N, D = h_cur.shape
    w_qkv = weights[0]
    if loop <= T_dense:
        q, k, v = split_qkv(project(h_cur, w_qkv), H, d)
        state = dense_loop(loop, q, k, v, cache, state)
        a = round_bf16(state.o.astype(np.float64)).reshape(B, N, D)
        return mlp(h_cur, a, weights), state, None, None
    if A is None:
        A = topk(token_scores(h_prev, h_cur), R)
    if S is None:
        col = state.c.astype(np.float64) if key_rank == 0 else key_scores_per_row(state.c, N)
        S = topk(col, K)
    bi = np.arange(B)[:, None]
    x = h_cur[bi, A]                                        # [B, R, D]
    qa, ka, va = split_qkv(project(x, w_qkv), H, d)        # [B, R, H, d]
    q, k, v = (np.zeros((B, N, H, d), np.uint16) for _ in range(3))
    q[bi, A], k[bi, A], v[bi, A] = qa, ka, va
    _, _, _, state, _, _ = lazy_loop(loop, h_prev, h_cur, q, k, v, cache, state, R, K, A=A, S=S)
    a = round_bf16(state.o[bi, A].astype(np.float64)).reshape(B, -1, D)
    h_out = np.array(h_cur, copy=True)
    h_out[bi, A] = mlp(x, a, weights)
    return h_out, state, A, S
