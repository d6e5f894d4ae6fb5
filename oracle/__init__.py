"""CPU oracle of the FlashLoop lazy loop step -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product path (the CUDA library and its
binding) never does; it shares no code with this package.

The arithmetic lives in ``flashloop_oracle.c`` (plain C, built with
``-O2 -ffp-contract=off -fopenmp``); this module only builds it and marshals
numpy arrays. Method: the rit.work page "FlashLoop: Fast and
Memory-Efficient Looped Transformers via Lazy Updates", sections "Later loops
change only part of the state" and "FlashLoop combines three kinds of
saving"; the readings taken where the page is silent are listed at the top of
the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "flashloop_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_flashloop_oracle.so")
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_flashloop_oracle.so``."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.orc_bf16_to_f32.restype = ctypes.c_float
        _lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        _lib.orc_f32_to_bf16.restype = ctypes.c_uint16
        _lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        _lib.orc_f16_to_f32.restype = ctypes.c_float
        _lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        _lib.orc_f32_to_f16.restype = ctypes.c_uint16
        _lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
        _lib.orc_token_scores.argtypes = [P, P, I64, I64, I64, P]
        _lib.orc_topk_rows.argtypes = [P, I64, I64, I64, P]
        _lib.orc_kv_delta_append.argtypes = [P, P, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P,
                                             I64, I64, I64, I64, P, I64, P, P, P]
        _lib.orc_reconstruct.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P, P, P, P, I64, I64, I64, I64, P, P]
        _lib.orc_quantize_base.argtypes = [P, I64, I64, I64, I64, P, P]
        _lib.orc_attention.argtypes = [ctypes.c_int, I64, I64, I64, I64, I64, I64, P, P,
                                       P, P, P, P, P, I64, P, P, P, P, P, P, P]
        _lib.orc_softmax_attention.argtypes = [P, P, P, I64, I64, I64, I64, P, P]
        _lib.orc_round_bf16.argtypes = [P, I64, P]
        if hasattr(_lib, "orc_set_threads"):   # timing control; absent from older builds
            _lib.orc_set_threads.argtypes = [ctypes.c_int]
            _lib.orc_get_threads.restype = ctypes.c_int
    return _lib


def set_threads(n: int) -> None:
    """OpenMP threads of the oracle's parallel regions (for timing it)."""
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(P)


def bits(t) -> np.ndarray:
    """uint16 bit pattern of a bf16 or fp16 torch tensor (or pass numpy through)."""
    if isinstance(t, np.ndarray):
        return t
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# scalar formats

def bf16_to_f32(h: int) -> float:
    return lib().orc_bf16_to_f32(h)


def f32_to_bf16(x: float) -> int:
    return lib().orc_f32_to_bf16(x)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 bit patterns, nearest even, in one step
    (reading R9 of the C file)."""
    a = _c(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(a.shape, np.uint16)
    lib().orc_round_bf16(_ptr(a), a.size, _ptr(out))
    return out


def bf16_values(h) -> np.ndarray:
    """float64 values of bf16 bit patterns (exact)."""
    u = np.asarray(bits(h), dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f16_to_f32(h: int) -> float:
    return lib().orc_f16_to_f32(h)


def f32_to_f16(x: float) -> int:
    return lib().orc_f32_to_f16(x)


# ---------------------------------------------------------------------------
# steps of the lazy loop

def token_scores(h_prev, h_cur) -> np.ndarray:
    """Squared L2 norm of the hidden-state change per token: [B, N] float64."""
    a, b = _c(bits(h_prev), np.uint16), _c(bits(h_cur), np.uint16)
    B, N, D = a.shape
    out = np.empty((B, N), np.float64)
    lib().orc_token_scores(_ptr(a), _ptr(b), B, N, D, _ptr(out))
    return out


def topk(score: np.ndarray, k: int) -> np.ndarray:
    """Top-k per row (ties to the lower index), ascending: [..., k] int32."""
    s = _c(np.asarray(score, dtype=np.float64), np.float64)
    lead, n = s.shape[:-1], s.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (k,), np.int32)
    lib().orc_topk_rows(_ptr(s), rows, n, k, _ptr(out))
    return out


class DeltaLayer:
    """One delta layer: idx [B,cnt] i32, codes [B,cnt,H,d*bits/8] u8, scales [B,cnt,H,d/32] u16 (fp16 bits)."""

    def __init__(self, idx, codes, scales):
        self.idx = _c(np.asarray(idx), np.int32)
        self.codes = _c(np.asarray(codes), np.uint8)
        self.scales = _c(np.asarray(scales), np.uint16)
        self.cnt = self.idx.shape[1]

    def concat(self, other: "DeltaLayer") -> "DeltaLayer":
        return DeltaLayer(np.concatenate([self.idx, other.idx], 1),
                          np.concatenate([self.codes, other.codes], 1),
                          np.concatenate([self.scales, other.scales], 1))


class CompressedBase:
    """An int8 base (the page's compressed base; reading R8 of the C file):
    codes [B,Nk,H,d] int8 and fp16 scales [B,Nk,H,d/32] (uint16 bits)."""

    def __init__(self, codes, scales):
        self.codes = _c(np.asarray(codes), np.int8)
        self.scales = _c(np.asarray(scales), np.uint16)
        self.shape = self.codes.shape


def quantize_base(x) -> CompressedBase:
    """The int8 compressed base of a bf16 layer x [B,Nk,H,d]."""
    xb = _c(bits(x), np.uint16)
    B, Nk, H, d = xb.shape
    codes = np.empty((B, Nk, H, d), np.int8)
    scales = np.empty((B, Nk, H, d // 32), np.uint16)
    lib().orc_quantize_base(_ptr(xb), B, Nk, H, d, _ptr(codes), _ptr(scales))
    return CompressedBase(codes, scales)


def _base_args(base):
    """(bf16 base, base codes, base scales) pointers and the base's shape."""
    if isinstance(base, CompressedBase):
        return None, base, (None, _ptr(base.codes), _ptr(base.scales)), base.shape
    bs = _c(bits(base), np.uint16)
    return bs, None, (_ptr(bs), None, None), bs.shape


def _layer_arrays(layers: Sequence[DeltaLayer]):
    n = len(layers)
    assert n <= 64
    idx = (P * max(n, 1))(*[_ptr(l.idx) for l in layers])
    codes = (P * max(n, 1))(*[_ptr(l.codes) for l in layers])
    scales = (P * max(n, 1))(*[_ptr(l.scales) for l in layers])
    cnt = (I64 * max(n, 1))(*[l.cnt for l in layers])
    return n, idx, codes, scales, cnt


def kv_delta_append(x_l, base, layers: Sequence[DeltaLayer], active, code_bits: int = 4) -> DeltaLayer:
    """New delta layer (``code_bits``-bit codes) for the active tokens of loop-l
    tensor ``x_l`` [B,Nk,H,d]; ``base`` is a bf16 layer or a CompressedBase."""
    assert code_bits in (2, 3, 4)
    x = _c(bits(x_l), np.uint16)
    keep_bs, keep_cb, (pb, pc, ps), _ = _base_args(base)
    act = _c(np.asarray(active, dtype=np.int32), np.int32)
    B, Nk, H, d = x.shape
    R = act.shape[1]
    idx = np.empty((B, R), np.int32)
    codes = np.zeros((B, R, H, d * code_bits // 8), np.uint8)
    scales = np.empty((B, R, H, d // 32), np.uint16)
    n, li, lc, ls, cnt = _layer_arrays(layers)
    lib().orc_kv_delta_append(_ptr(x), pb, pc, ps, code_bits, n, li, lc, ls, cnt, B, Nk, H, d,
                              _ptr(act), R, _ptr(idx), _ptr(codes), _ptr(scales))
    return DeltaLayer(idx, codes, scales)


def reconstruct(base, layers: Sequence[DeltaLayer], want_f32: bool = True, want_bf16: bool = True,
                code_bits: int = 4):
    """(fp32 [B,Nk,H,d] or None, bf16-bits uint16 [B,Nk,H,d] or None); ``base``
    is a bf16 layer or a CompressedBase, the layers hold ``code_bits``-bit codes."""
    keep_bs, keep_cb, (pb, pc, ps), shape = _base_args(base)
    B, Nk, H, d = shape
    f = np.empty(shape, np.float32) if want_f32 else None
    h = np.empty(shape, np.uint16) if want_bf16 else None
    n, li, lc, ls, cnt = _layer_arrays(layers)
    lib().orc_reconstruct(pb, pc, ps, code_bits, n, li, lc, ls, cnt, B, Nk, H, d, _ptr(f), _ptr(h))
    return f, h


def attention(first: bool, pos, slot, q, qhat, o, z, c, S, k_old, v_old, k_new, v_new,
              bh_mask=None, want_m: bool = False):
    """Lazy mass-preserving attention; updates copies of (qhat, o, z, c).

    pos/slot [B,R] i32; q/qhat [B,Ns,H,d] bf16 bits; o [B,Ns,H,d] f32;
    z [B,H,Ns] f32; c [B,H,Nk] f32; S [B,H,K] i32; k/v [B,Nk,H,d] bf16 bits
    (old ones may be None when ``first``). Returns (qhat, o, z, c, m).
    """
    q = _c(bits(q), np.uint16)
    qhat = np.array(bits(qhat), dtype=np.uint16, copy=True, order="C")
    o = np.array(o, dtype=np.float32, copy=True, order="C")
    z = np.array(z, dtype=np.float32, copy=True, order="C")
    c = np.array(c, dtype=np.float32, copy=True, order="C")
    pos = _c(np.asarray(pos, dtype=np.int32), np.int32)
    slot = _c(np.asarray(slot, dtype=np.int32), np.int32)
    S = _c(np.asarray(S, dtype=np.int32), np.int32)
    kn, vn = _c(bits(k_new), np.uint16), _c(bits(v_new), np.uint16)
    ko = None if k_old is None else _c(bits(k_old), np.uint16)
    vo = None if v_old is None else _c(bits(v_old), np.uint16)
    if not first:
        assert ko is not None and vo is not None
    B, Ns, H, d = q.shape
    Nk = kn.shape[1]
    R = pos.shape[1]
    K = S.shape[2]
    mask = None if bh_mask is None else _c(np.asarray(bh_mask, dtype=np.uint8).reshape(B * H), np.uint8)
    m = np.full((B, H, R), np.nan) if want_m else None
    lib().orc_attention(int(first), B, H, d, Nk, Ns, R, _ptr(pos), _ptr(slot),
                        _ptr(q), _ptr(qhat), _ptr(o), _ptr(z), _ptr(c), K, _ptr(S),
                        _ptr(ko), _ptr(vo), _ptr(kn), _ptr(vn), _ptr(mask), _ptr(m))
    return qhat, o, z, c, m


def key_scores_per_row(c, n_rows: int) -> np.ndarray:
    """Column mass per causal row that sees the key: c_j / (n_rows - j), as the
    IEEE fp32 quotient (another reading of "keys chosen from the previous
    loop's statistics", rit.work page, section "FlashLoop combines three kinds
    of saving"; in a prefill of n_rows tokens, n_rows - j rows see key j).
    c [..., N] fp32 -> float64 scores for ``topk``."""
    c = np.asarray(c, dtype=np.float32)
    n = c.shape[-1]
    assert n <= n_rows
    den = (n_rows - np.arange(n)).astype(np.float32)
    return (c / den).astype(np.float32).astype(np.float64)


def column_recovery(o_lazy, o_full, o_prev):
    """How much of the exact loop-l attention result the lazy update over a
    key subset recovers (the synthetic analogue of the rit.work page's
    observation, section "Later loops change only part of the state", that
    updating 10% of the attention columns in a late loop recovers more than
    90% of the exact result), over the rows given (float64):
      recovered = 1 - ||o_lazy - o_full|| / ||o_prev - o_full||
      rel_err   = ||o_lazy - o_full|| / ||o_full||
    with o_full the same rows updated over every key (exact softmax of the
    loop-l reconstruction) and o_prev the rows before the loop."""
    a, f, p = (np.asarray(x, dtype=np.float64) for x in (o_lazy, o_full, o_prev))
    miss = np.linalg.norm((a - f).ravel())
    change = np.linalg.norm((p - f).ravel())
    return {"recovered": 1.0 - miss / change if change > 0 else 1.0,
            "rel_err": miss / np.linalg.norm(f.ravel()) if np.any(f) else 0.0}


def softmax_attention(q, k, v):
    """Textbook causal softmax attention in double: (o [B,N,H,d], lse [B,H,N])."""
    q, k, v = (_c(bits(t), np.uint16) for t in (q, k, v))
    B, N, H, d = q.shape
    o = np.empty((B, N, H, d), np.float64)
    lse = np.empty((B, H, N), np.float64)
    lib().orc_softmax_attention(_ptr(q), _ptr(k), _ptr(v), B, N, H, d, _ptr(o), _ptr(lse))
    return o, lse
