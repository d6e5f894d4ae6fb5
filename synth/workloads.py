"""Seeded synthetic workloads shaped like the FlashLoop pages' settings.

This module draws random numbers and arranges them into per-loop tensors. It
holds none of the method's arithmetic: no change scores, no selections, no
quantisation and no attention. Both the CUDA path (tests, benchmark) and the
CPU oracle (tests) take their inputs from here, so neither can lean on the
other for data.

Structure reproduced from the rit.work page "FlashLoop: Fast and
Memory-Efficient Looped Transformers via Lazy Updates", section "Later loops
change only part of the state": as loops repeat, most tokens change less and
less, a small group keeps changing, and that group narrows and nests (tokens
active late were usually active the loop before).

Recipe (per workload):
  * loop 1: every tensor X in {H, Q, K, V} is N(0,1), rounded RNE to bf16;
  * loop l >= 2: X_l = bf16(float(X_{l-1}) + eps_{l,i} * z), z ~ N(0,1) drawn
    independently per element, eps_{l,i} = eps_hi * gamma**(l-2) for tokens in
    the loop's heavy set and eps_lo * gamma**(l-2) for the rest
    (eps_hi = 0.5, eps_lo = 0.01);
  * heavy set: a fixed seeded subset, or (nested workloads) 90% carried over
    from the previous loop's heavy set plus 10% fresh tokens.
Every draw comes from its own torch.Generator seeded from (workload id, loop,
tensor tag), so any loop can be regenerated on its own and the result does
not depend on the device order of other draws.
"""
from __future__ import annotations

import dataclasses
import math
from fractions import Fraction
from typing import Dict, Iterator, Optional

import torch

EPS_HI = 0.5
EPS_LO = 0.01
SEED_BASE = 0xF1A51000

_TAGS = {"H": 1, "Q": 2, "K": 3, "V": 4, "heavy": 5, "carry": 6, "fresh": 7,
         "dq": 8, "dk": 9, "dv": 10, "ctx": 11, "wqkv": 12, "wo": 13, "w1": 14, "w2": 15}

# Synthetic looped block: MLP width and the gains of its random weights.
BLOCK_FF_MULT = 4
BLOCK_GAINS = {"wqkv": 1.0, "wo": 0.5, "w1": 1.0, "w2": 0.5}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and drift recipe of one synthetic workload."""

    name: str
    cid: int            # workload id, feeds the seed
    B: int              # sequences
    N: int              # tokens per sequence (prefill) / cached context (decode)
    H: int              # heads
    d: int              # head dim
    T: int              # loops
    T_dense: int        # leading dense loops
    r: Fraction         # active token fraction of a lazy loop
    k: Fraction         # key column fraction of a lazy loop
    heavy_frac: Fraction
    gamma: float
    nested: bool        # heavy set carries 90% over from the previous loop
    decode: bool        # a decode workload: context cache + one new token
    decode_after_prefill: bool = False

    @property
    def D(self) -> int:
        return self.H * self.d

    @property
    def seed(self) -> int:
        return SEED_BASE + self.cid


def _ceil_frac(f: Fraction, n: int) -> int:
    v = math.ceil(f * n)
    return max(1, min(n, v))


def active_count(w: Workload, n: Optional[int] = None) -> int:
    """R = ceil(r * N), clamped to [1, N]."""
    return _ceil_frac(w.r, w.N if n is None else n)


def key_count(w: Workload, n: Optional[int] = None) -> int:
    """K = ceil(k * N_keys), clamped to [1, N_keys]."""
    return _ceil_frac(w.k, w.N if n is None else n)


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 0, 1, 1024, 4, 64, 4, 1, Fraction(1, 4), Fraction(1, 10),
                     Fraction(1, 5), 0.5, False, False),
    "8k": Workload("8k", 1, 1, 8192, 16, 128, 4, 1, Fraction(1, 4), Fraction(1, 10),
                   Fraction(1, 5), 0.5, False, False),
    "32k": Workload("32k", 2, 1, 32768, 16, 128, 4, 1, Fraction(15, 100), Fraction(1, 10),
                    Fraction(15, 100), 0.5, True, False),
    "decode": Workload("decode", 3, 64, 16384, 16, 128, 4, 1, Fraction(1, 4), Fraction(1, 10),
                       Fraction(1, 4), 0.5, True, True),
    "deep": Workload("deep", 4, 8, 16384, 32, 96, 16, 2, Fraction(1, 10), Fraction(1, 20),
                     Fraction(1, 5), 0.8, False, False, decode_after_prefill=True),
}


def _gen(w: Workload, loop: int, tag: str, device, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((w.seed * 1000003 + loop * 1009 + _TAGS[tag] + 65537 * sub) & ((1 << 62) - 1))
    return g


def normal_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) draws rounded RNE to bf16."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _drift(x: torch.Tensor, eps_tok: torch.Tensor, gen: torch.Generator) -> torch.Tensor:
    """bf16(float(x) + eps_tok * z); eps_tok broadcasts over the token axis 1."""
    z = torch.randn(x.shape, generator=gen, device=x.device, dtype=torch.float32)
    shape = list(eps_tok.shape) + [1] * (x.dim() - eps_tok.dim())
    return (x.float() + eps_tok.view(shape) * z).to(torch.bfloat16)


def _heavy_sets(w: Workload, n_tok: int, device) -> Dict[int, torch.Tensor]:
    """Boolean heavy mask [B, n_tok] for every lazy loop l = 2..T.

    Fixed workloads draw one subset per sequence and keep it for every loop.
    Nested workloads draw loop 2's subset, then build loop l from 90% of loop
    l-1's subset plus fresh tokens from outside it.
    """
    n_heavy = int(round(float(w.heavy_frac) * n_tok))
    n_keep = int(round(0.9 * n_heavy))
    out: Dict[int, torch.Tensor] = {}
    prev = None
    for l in range(2, w.T + 1):
        mask = torch.zeros(w.B, n_tok, dtype=torch.bool)
        for b in range(w.B):
            if prev is None or not w.nested:
                sel = torch.randperm(n_tok, generator=_gen(w, 2 if w.nested else 0, "heavy", "cpu", b))
                mask[b, sel[:n_heavy]] = True
            else:
                old = torch.nonzero(prev[b]).flatten()
                rest = torch.nonzero(~prev[b]).flatten()
                keep = old[torch.randperm(old.numel(), generator=_gen(w, l, "carry", "cpu", b))[:n_keep]]
                fresh = rest[torch.randperm(rest.numel(), generator=_gen(w, l, "fresh", "cpu", b))[:n_heavy - n_keep]]
                mask[b, keep] = True
                mask[b, fresh] = True
        out[l] = mask
        prev = mask
    return {l: m.to(device) for l, m in out.items()}


def prefill_loops(w: Workload, device="cpu", last: Optional[int] = None) -> Iterator[Dict[str, torch.Tensor]]:
    """Yield {"loop", "H" [B,N,D], "Q","K","V" [B,N,H,d], "heavy"} for l = 1..T.

    Each yielded dict is fresh; the generator only keeps the previous loop.
    """
    T = w.T if last is None else last
    heavy = _heavy_sets(w, w.N, device)
    cur = {
        "H": normal_bf16((w.B, w.N, w.D), _gen(w, 1, "H", device), device),
        "Q": normal_bf16((w.B, w.N, w.H, w.d), _gen(w, 1, "Q", device), device),
        "K": normal_bf16((w.B, w.N, w.H, w.d), _gen(w, 1, "K", device), device),
        "V": normal_bf16((w.B, w.N, w.H, w.d), _gen(w, 1, "V", device), device),
    }
    yield dict(cur, loop=1, heavy=None)
    for l in range(2, T + 1):
        scale = w.gamma ** (l - 2)
        hv = heavy[l]
        eps = torch.where(hv, torch.tensor(EPS_HI * scale, device=device),
                          torch.tensor(EPS_LO * scale, device=device)).float()
        cur = {name: _drift(cur[name], eps, _gen(w, l, name, device)) for name in ("H", "Q", "K", "V")}
        yield dict(cur, loop=l, heavy=hv)


def decode_context(w: Workload, device="cpu") -> Dict[str, object]:
    """Context of a decode workload: base K/V and, per lazy loop, the drifted
    K/V of a nested random 25% of the context tokens.

    Returns {"K1","V1": [B,N,H,d] bf16, "loops": {l: {"K","V","active"}}}
    where "active" is the ascending [B, R_ctx] int32 token list that loop l
    appends deltas for.
    """
    k1 = normal_bf16((w.B, w.N, w.H, w.d), _gen(w, 1, "K", device), device)
    v1 = normal_bf16((w.B, w.N, w.H, w.d), _gen(w, 1, "V", device), device)
    heavy = _heavy_sets(w, w.N, device)
    loops = {}
    kc, vc = k1, v1
    for l in range(2, w.T + 1):
        hv = heavy[l]
        eps = torch.where(hv, torch.tensor(EPS_HI * 0.5 ** (l - 2), device=device),
                          torch.tensor(0.0, device=device)).float()
        kc = _drift(kc, eps, _gen(w, l, "K", device))
        vc = _drift(vc, eps, _gen(w, l, "V", device))
        act = torch.stack([torch.nonzero(hv[b]).flatten() for b in range(w.B)]).to(torch.int32)
        loops[l] = {"K": kc, "V": vc, "active": act.contiguous()}
    return {"K1": k1, "V1": v1, "loops": loops}


def decode_token_loops(w: Workload, device="cpu") -> Iterator[Dict[str, torch.Tensor]]:
    """The new token's q/k/v [B,1,H,d] per loop l = 1..T: N(0,1) at loop 1,
    then drift 0.5 * gamma**(l-2) on every element."""
    shape = (w.B, 1, w.H, w.d)
    cur = {n: normal_bf16(shape, _gen(w, 1, t, device), device)
           for n, t in (("q", "dq"), ("k", "dk"), ("v", "dv"))}
    yield dict(cur, loop=1)
    for l in range(2, w.T + 1):
        eps = torch.full((w.B, 1), EPS_HI * w.gamma ** (l - 2), device=device)
        cur = {n: _drift(cur[n], eps, _gen(w, l, t, device))
               for n, t in (("q", "dq"), ("k", "dk"), ("v", "dv"))}
        yield dict(cur, loop=l)


def block_weights(w: Workload, F: Optional[int] = None, device="cpu"):
    """Random weights of the synthetic looped block, each stored transposed
    [out features, in features] as bf16: (w_qkv [3D, D], w_o [D, D],
    w_1 [F, D], w_2 [D, F]), entries N(0, (gain / sqrt(in features))^2)
    rounded RNE to bf16 (F = 4 D by default). The gains below one on the two
    projections back into the residual stream keep the state's scale moderate
    over the loops."""
    D = w.D
    F = BLOCK_FF_MULT * D if F is None else F
    shapes = {"wqkv": (3 * D, D), "wo": (D, D), "w1": (F, D), "w2": (D, F)}
    out = []
    for tag in ("wqkv", "wo", "w1", "w2"):
        n_out, n_in = shapes[tag]
        z = torch.randn((n_out, n_in), generator=_gen(w, 0, tag, device), device=device, dtype=torch.float32)
        out.append((z * (BLOCK_GAINS[tag] / math.sqrt(n_in))).to(torch.bfloat16))
    return tuple(out)


def block_input(w: Workload, device="cpu") -> torch.Tensor:
    """H_0 of the synthetic looped block: [B, N, D], N(0,1) rounded to bf16
    (the same draw as loop 1's H of the prefill workload)."""
    return normal_bf16((w.B, w.N, w.D), _gen(w, 1, "H", device), device)
