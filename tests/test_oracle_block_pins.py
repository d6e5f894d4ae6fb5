"""Pins of the oracle's synthetic looped block (reading R9 of the oracle's C
file) against definitions it does not share code with: exact rational
arithmetic with a textbook round-to-nearest-even, library bf16 conversion,
and closed forms of the block's wiring (zero output weights, a single token).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import block as ob
from oracle.loop import Cache, empty_state


def _rne_bf16_exact(v: Fraction) -> Fraction:
    """Nearest bf16 value to the rational v, ties to an even significand
    (8 significant bits; normal range only)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    assert -126 <= e <= 127
    spacing = Fraction(2) ** (e - 7)
    lo = (abs(v) // spacing) * spacing
    hi = lo + spacing
    dl, dh = abs(v) - lo, hi - abs(v)
    if dl < dh or (dl == dh and (lo / spacing) % 2 == 0):
        r = lo
    else:
        r = hi
    return sign * r


def _to_bits(x: Fraction) -> int:
    return int(oracle.round_bf16(np.array([float(x)]))[0])   # float(x) exact: x is a bf16 value


def _frac_bits(b) -> Fraction:
    return Fraction(float(oracle.bf16_values(np.array([b], np.uint16))[0]))


def test_round_bf16_matches_library_conversion_of_binary32():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp2(torch.randint(-20, 20, (20000,),
                                                                                          generator=g).float())
    ties = (1 + (2 * torch.arange(0, 64, dtype=torch.float32) + 1) * 2.0 ** -8) * 2.0 ** torch.arange(-8, 56) \
        .float()[:64]
    x = torch.cat([x, ties, -ties])
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(x.double().numpy())
    assert np.array_equal(got, want)


@pytest.mark.parametrize("value, expect", [
    (1 + 2 ** -8, 0x3F80),                 # tie -> even (1.0)
    (1 + 3 * 2 ** -8, 0x3F82),             # tie -> even (1 + 2^-6)
    (1 + 2 ** -8 + 2 ** -40, 0x3F81),      # just above the tie: up, although binary32 would land on the tie
    (-(1 + 2 ** -8 + 2 ** -40), 0xBF81),
    (1.3 * 2.0 ** -130, 10),               # subnormal: 10.4 steps of 2^-133
    (3.5e38, 0x7F80),                      # overflow
    (0.0, 0x0000),
])
def test_round_bf16_single_rounding_cases(value, expect):
    assert int(oracle.round_bf16(np.array([value]))[0]) == expect


@pytest.mark.parametrize("relu", [False, True])
def test_project_equals_exact_rational_brute_force(relu):
    rng = np.random.default_rng(3)
    M, K, N = 3, 5, 4
    x = oracle.round_bf16(rng.standard_normal((M, K)))
    w_t = oracle.round_bf16(rng.standard_normal((N, K)))
    res = oracle.round_bf16(rng.standard_normal((M, N)))
    got = ob.project(x, w_t, residual=res, relu=relu)
    for m in range(M):
        for n in range(N):
            acc = sum(_frac_bits(x[m, kk]) * _frac_bits(w_t[n, kk]) for kk in range(K)) + _frac_bits(res[m, n])
            if relu:
                acc = max(acc, Fraction(0))
            want = _rne_bf16_exact(acc)
            assert _frac_bits(got[m, n]) == want, (m, n)


def _tiny_weights(D, F, seed, zero_out=False):
    rng = np.random.default_rng(seed)
    w = [oracle.round_bf16(rng.standard_normal(s) / np.sqrt(s[1])) for s in ((3 * D, D), (D, D), (F, D), (D, F))]
    if zero_out:
        w[1][:] = 0
        w[3][:] = 0
    return w


def test_zero_output_weights_leave_the_state_unchanged():
    # y = bf16(x + 0) = x and h = bf16(y + 0) = y: every loop is the identity
    B, N, H, d, F = 1, 24, 2, 8, 32
    D = H * d
    w = _tiny_weights(D, F, 11, zero_out=True)
    h0 = oracle.round_bf16(np.random.default_rng(5).standard_normal((B, N, D)))
    cache, st = Cache(), empty_state(B, N, H, d)
    h1, st, _, _ = ob.block_loop(1, w, None, h0, cache, st, T_dense=1, H=H, d=d)
    assert np.array_equal(h1, h0)
    h2, st, A, S = ob.block_loop(2, w, h0, h1, cache, st, T_dense=1, H=H, d=d, R=6, K=5)
    assert np.array_equal(h2, h0) and A.shape == (B, 6) and S.shape == (B, H, 5)


def test_single_token_block_is_the_mlp_of_its_value():
    # one token, one key: its attention output is v exactly, so the loop is
    # h = bf16(y + bf16(relu(y W_1)) W_2) with y = bf16(x + v W_o), v = bf16(x W_v)
    B, N, H, d, F = 1, 1, 1, 8, 16
    D = H * d
    w_qkv, w_o, w_1, w_2 = _tiny_weights(D, F, 21)
    x = oracle.round_bf16(np.random.default_rng(9).standard_normal((B, N, D)))
    h1, _, _, _ = ob.block_loop(1, (w_qkv, w_o, w_1, w_2), None, x, Cache(), empty_state(B, N, H, d),
                                T_dense=1, H=H, d=d)
    X = [_frac_bits(b) for b in x[0, 0]]

    def proj(vec, wt, rows, res=None, relu=False):
        out = []
        for n in rows:
            acc = sum(vec[kk] * _frac_bits(wt[n, kk]) for kk in range(len(vec)))
            if res is not None:
                acc += res[len(out)]
            if relu:
                acc = max(acc, Fraction(0))
            out.append(_rne_bf16_exact(acc) if acc != 0 else Fraction(0))
        return out

    v = proj(X, w_qkv, range(2 * D, 3 * D))
    y = proj(v, w_o, range(D), res=X)
    u = proj(y, w_1, range(F), relu=True)
    h = proj(u, w_2, range(D), res=y)
    assert [_frac_bits(b) for b in h1[0, 0]] == h


def test_lazy_block_recomputes_only_the_active_rows():
    # inactive rows keep H_{l-1} bit for bit; active rows are the MLP of
    # (x = H_{l-1}[i], bf16(O_i)) with the loop's own attention output
    B, N, H, d, F, R, K = 2, 40, 2, 8, 32, 9, 12
    D = H * d
    w = _tiny_weights(D, F, 31)
    h0 = oracle.round_bf16(np.random.default_rng(2).standard_normal((B, N, D)))
    cache, st = Cache(), empty_state(B, N, H, d)
    h1, st, _, _ = ob.block_loop(1, w, None, h0, cache, st, T_dense=1, H=H, d=d)
    h2, st, A, S = ob.block_loop(2, w, h0, h1, cache, st, T_dense=1, H=H, d=d, R=R, K=K)
    assert np.array_equal(A, oracle.topk(oracle.token_scores(h0, h1), R))
    for b in range(B):
        inactive = np.setdiff1d(np.arange(N), A[b])
        assert np.array_equal(h2[b, inactive], h1[b, inactive])
        for r in (0, R - 1):
            i = A[b, r]
            X = [_frac_bits(v) for v in h1[b, i]]
            a = [Fraction(float(np.float32(o))) for o in st.o[b, i].reshape(-1)]
            a = [_rne_bf16_exact(t) if t != 0 else Fraction(0) for t in a]

            def proj(vec, wt, rows, res=None, relu=False):
                out = []
                for n in rows:
                    acc = sum(vec[kk] * _frac_bits(wt[n, kk]) for kk in range(len(vec)))
                    if res is not None:
                        acc += res[len(out)]
                    if relu:
                        acc = max(acc, Fraction(0))
                    out.append(_rne_bf16_exact(acc) if acc != 0 else Fraction(0))
                return out

            y = proj(a, w[1], range(D), res=X)
            u = proj(y, w[2], range(F), relu=True)
            h = proj(u, w[3], range(D), res=y)
            assert [_frac_bits(v) for v in h2[b, i]] == h, (b, i)
