"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against a closed form, a library routine, a
hand-worked example under tests/golden/, brute force on tiny inputs, or an
invariant of the method (rit.work page "FlashLoop: Fast and Memory-Efficient
Looped Transformers via Lazy Updates", sections "Later loops change only part
of the state" and "FlashLoop combines three kinds of saving").
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read(path):
    with open(path) as f:
        return f.read()


def bf16_bits(x):
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float().numpy()


# --------------------------------------------------------------------------
# number formats: the oracle's own converters against numpy / torch

def test_f16_decode_every_pattern(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(p)) for p in pats], np.float32)
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.isnan(got[~fin]).all()


def test_f16_encode_matches_numpy_rne(orc):
    rng = np.random.default_rng(7)
    vals = [rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000)]
    h = np.arange(0, 0x7C00, 37, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    vals.append((h[:-1] + h[1:]) / 2)                        # exact midpoints: ties to even
    vals.append(np.array([65504.0, 65519.0, 65520.0, 7e4, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                          2.0 ** -14 - 2.0 ** -30, 0.0, -0.0]))
    x = np.concatenate(vals).astype(np.float32)
    x = np.concatenate([x, -x])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_roundtrip_matches_torch(orc):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    b = np.arange(0, 0x7F80, 13, dtype=np.uint32).astype(np.uint16)
    mids = (bits_to_f32(b[:-1]).astype(np.float64) + bits_to_f32(b[1:])) / 2
    x = np.concatenate([x, mids.astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)
    back = np.array([orc.bf16_to_f32(int(v)) for v in ref[:2000]], np.float32)
    assert np.array_equal(back, bits_to_f32(ref[:2000]))


# --------------------------------------------------------------------------
# token change score: squared L2 norm of the hidden-state change

def test_scores_closed_forms(orc):
    rng = np.random.default_rng(1)
    B, N, D = 2, 9, 64
    a = bf16_bits(rng.standard_normal((B, N, D)))
    assert np.array_equal(orc.token_scores(a, a), np.zeros((B, N)))
    z = np.zeros((1, 2, 8), np.float32)
    c = np.zeros((1, 2, 8), np.float32)
    c[0, 0, 1], c[0, 0, 6] = 3.0, 4.0                     # 3-4-5 triangle
    c[0, 1, 2] = -0.375
    s = orc.token_scores(bf16_bits(z), bf16_bits(c))
    assert s[0, 0] == 25.0 and s[0, 1] == 0.140625


def test_scores_match_library_norm(orc):
    rng = np.random.default_rng(2)
    a = bf16_bits(rng.standard_normal((3, 50, 256)))
    b = bf16_bits(rng.standard_normal((3, 50, 256)))
    ref = np.linalg.norm(bits_to_f32(b).astype(np.float64) - bits_to_f32(a), axis=-1) ** 2
    np.testing.assert_allclose(orc.token_scores(a, b), ref, rtol=1e-13)


# --------------------------------------------------------------------------
# top-k with lower-index tie-break, ascending output

def test_topk_golden():
    import oracle
    g = json.loads(_read(os.path.join(GOLD, "topk_ties.json")))
    for case in g["cases"]:
        got = oracle.topk(np.array([g["scores"]]), case["k"])[0]
        assert got.tolist() == case["expect"], case


@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (64, 64), (300, 17), (1000, 999)])
def test_topk_brute_force(orc, n, k):
    rng = np.random.default_rng(n * 31 + k)
    s = np.round(rng.standard_normal((4, n)) * 3) / 2          # many ties
    got = orc.topk(s, k)
    for r in range(4):
        order = sorted(range(n), key=lambda j: (-s[r, j], j))[:k]
        assert got[r].tolist() == sorted(order)


# --------------------------------------------------------------------------
# base + int4 delta cache

def _quant_one(orc, delta):
    x = bf16_bits(np.asarray(delta, np.float32).reshape(1, 1, 1, 32))
    base = np.zeros_like(x)
    return orc.kv_delta_append(x, base, [], np.array([[0]], np.int32))


def test_quantiser_golden(orc):
    g = json.loads(_read(os.path.join(GOLD, "quantiser_groups.json")))
    for grp in g["groups"]:
        layer = _quant_one(orc, grp["delta"])
        assert int(layer.scales[0, 0, 0, 0]) == grp["scale_bits"], grp["why"]
        assert layer.codes[0, 0, 0].tolist() == grp["bytes"], grp["why"]
        lo = (layer.codes[0, 0, 0] & 0xF).astype(np.int8)
        hi = (layer.codes[0, 0, 0] >> 4).astype(np.int8)
        codes = np.stack([lo, hi], 1).reshape(-1)
        codes = np.where(codes >= 8, codes - 16, codes)
        assert codes.tolist() == grp["codes"], grp["why"]


def _random_cache(orc, B=2, N=40, H=3, d=64, loops=3, seed=3):
    rng = np.random.default_rng(seed)
    base = bf16_bits(rng.standard_normal((B, N, H, d)))
    xs, layers, acts = [base], [], []
    for l in range(loops):
        x = bits_to_f32(xs[-1]) + rng.standard_normal((B, N, H, d)) * (0.3 / (l + 1))
        x[0, 5] = bits_to_f32(xs[-1])[0, 5]                      # an unchanged token
        x = bf16_bits(x)
        act = np.stack([np.sort(rng.choice(N, N // 3, replace=False)) for _ in range(B)]).astype(np.int32)
        if 5 not in act[0]:
            act[0, 0] = 5
            act[0] = np.sort(act[0])
        layers.append(orc.kv_delta_append(x, base, layers, act))
        xs.append(x)
        acts.append(act)
    return base, xs, layers, acts


def test_delta_roundtrip_error_within_half_scale(orc):
    base, xs, layers, acts = _random_cache(orc)
    B, N, H, d = base.shape
    for l in range(len(layers)):
        new, _ = orc.reconstruct(base, layers[: l + 1], want_bf16=False)
        x = bits_to_f32(xs[l + 1])
        lay = layers[l]
        for b in range(B):
            for e, i in enumerate(lay.idx[b]):
                s = np.array([orc.f16_to_f32(int(v)) for v in lay.scales[b, e].reshape(-1)], np.float32)
                s = np.repeat(s.reshape(H, d // 32), 32, axis=1)
                err = np.abs(new[b, i] - x[b, i])
                assert np.all(err <= s / 2 * (1 + 2.0 ** -20) + 1e-30), (l, b, i)


def test_delta_zero_change_gives_zero_entry(orc):
    rng = np.random.default_rng(4)
    base = bf16_bits(rng.standard_normal((1, 6, 2, 64)))
    lay = orc.kv_delta_append(base, base, [], np.array([[1, 4]], np.int32))
    assert not lay.codes.any() and not lay.scales.any()


def test_inactive_tokens_reconstruct_bit_identically(orc):
    base, xs, layers, acts = _random_cache(orc)
    B, N = base.shape[:2]
    for l in range(len(layers)):
        prev, _ = orc.reconstruct(base, layers[:l], want_bf16=False)
        new, _ = orc.reconstruct(base, layers[: l + 1], want_bf16=False)
        for b in range(B):
            inactive = np.setdiff1d(np.arange(N), acts[l][b])
            assert np.array_equal(prev[b, inactive].view(np.uint32), new[b, inactive].view(np.uint32))


def test_layer_holds_entries_only_for_active_tokens(orc):
    base, xs, layers, acts = _random_cache(orc)
    B, N, H, d = base.shape
    for lay, act in zip(layers, acts):
        assert np.array_equal(lay.idx, act)
        R = act.shape[1]
        assert lay.codes.nbytes + lay.scales.nbytes == B * R * H * (d // 2 + 2 * d // 32)
        assert np.all(np.abs(np.where((lay.codes & 0xF) >= 8, (lay.codes & 0xF) - 16.0, lay.codes & 0xF)) <= 7)
        assert np.all((lay.codes >> 4) != 8) and np.all((lay.codes & 0xF) != 8)


def test_unchanged_active_token_gets_zero_delta(orc):
    base, xs, layers, acts = _random_cache(orc)
    # token 5 of sequence 0 is active but its K never changes
    for lay in layers:
        e = int(np.where(lay.idx[0] == 5)[0][0])
        assert not lay.codes[0, e].any()


# --------------------------------------------------------------------------
# attention

def _sdpa(qb, kb, vb):
    q, k, v = (torch.from_numpy(bits_to_f32(t).astype(np.float64)).permute(0, 2, 1, 3) for t in (qb, kb, vb))
    d = q.shape[-1]
    logits = q @ k.transpose(-1, -2) / math.sqrt(d)
    N = q.shape[2]
    mask = torch.ones(N, N, dtype=torch.bool).tril()
    logits = logits.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(logits, -1)
    p = torch.softmax(logits, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy(), p.sum(2).numpy()


def _tensors(seed, B=2, N=48, H=2, d=64):
    rng = np.random.default_rng(seed)
    return [bf16_bits(rng.standard_normal((B, N, H, d))) for _ in range(3)]


def _dense_first(orc, q, k, v):
    from oracle import loop
    B, N, H, d = q.shape
    st = loop.empty_state(B, N, H, d)
    cache = loop.Cache()
    return loop.dense_loop(1, q, k, v, cache, st), cache


def test_first_dense_is_softmax_attention(orc):
    q, k, v = _tensors(11)
    st, _ = _dense_first(orc, q, k, v)
    o_ref, lse_ref, col_ref = _sdpa(q, k, v)
    np.testing.assert_allclose(st.o, o_ref, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(st.z, lse_ref, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(st.c, col_ref, rtol=1e-6, atol=1e-6)
    o2, lse2 = orc.softmax_attention(q, k, v)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse2, lse_ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(st.qhat, q)


def test_first_dense_has_unit_mass_and_no_old_term(orc):
    q, k, v = _tensors(12, B=1, N=20)
    B, N, H, d = q.shape
    rows = np.arange(N, dtype=np.int32)[None]
    S = np.tile(np.arange(N, dtype=np.int32), (B, H, 1))
    zero = np.zeros((B, N, H, d), np.float32)
    junk = np.full((B, N, H, d), 5.0, np.float32)           # old O must be ignored
    _, o1, _, _, m = orc.attention(True, rows, rows, q, q, junk, np.zeros((B, H, N), np.float32),
                                   np.zeros((B, H, N), np.float32), S, None, None, k, v, want_m=True)
    _, o2, _, _, _ = orc.attention(True, rows, rows, q, q, zero, np.zeros((B, H, N), np.float32),
                                   np.zeros((B, H, N), np.float32), S, None, None, k, v)
    assert np.all(m == 1.0)
    assert np.array_equal(o1, o2)


def test_lazy_full_sets_reduce_to_softmax(orc):
    """S = all keys and A = all tokens: the lazy step is exact softmax attention."""
    from oracle import loop
    q1, k1, v1 = _tensors(13)
    q2, k2, v2 = _tensors(14)
    st, cache = _dense_first(orc, q1, k1, v1)
    B, N, H, d = q1.shape
    rows = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    S = np.tile(np.arange(N, dtype=np.int32), (B, H, 1))
    qh, o, z, c, m = orc.attention(False, rows, rows, q2, st.qhat, st.o, st.z, st.c, S,
                                   k1, v1, k2, v2, want_m=True)
    o_ref, lse_ref, col_ref = _sdpa(q2, k2, v2)
    np.testing.assert_allclose(m, 1.0, rtol=0, atol=2e-6)
    np.testing.assert_allclose(o, o_ref, rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(z, lse_ref, rtol=0, atol=5e-6)
    np.testing.assert_allclose(c, col_ref, rtol=1e-5, atol=2e-6)
    assert np.array_equal(qh, q2)


def test_lazy_step_with_unchanged_inputs_is_identity(orc):
    """Nothing changed (same q, same K/V): with any key subset, the preserved
    mass makes m * softmax_S equal the old probabilities, so O, Z, c stay."""
    q, k, v = _tensors(15)
    st, _ = _dense_first(orc, q, k, v)
    B, N, H, d = q.shape
    rng = np.random.default_rng(5)
    S = np.stack([np.stack([np.sort(rng.choice(N, 11, replace=False)) for _ in range(H)])
                  for _ in range(B)]).astype(np.int32)
    S[..., 0] = 0
    S.sort(-1)
    A = np.stack([np.sort(rng.choice(N, 17, replace=False)) for _ in range(B)]).astype(np.int32)
    qh, o, z, c, m = orc.attention(False, A, A, q, st.qhat, st.o, st.z, st.c, S, k, v, k, v, want_m=True)
    np.testing.assert_allclose(o, st.o, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(z, st.z, rtol=0, atol=1e-5)
    np.testing.assert_allclose(c, st.c, rtol=1e-5, atol=1e-6)
    mm = m[~np.isnan(m)]
    assert mm.size > 0 and np.all(mm > 0) and np.all(mm <= 1 + 1e-6)


def test_no_active_rows_leaves_state_bit_identical(orc):
    q, k, v = _tensors(16)
    st, _ = _dense_first(orc, q, k, v)
    q2, k2, v2 = _tensors(17)
    B, N, H, d = q.shape
    A = np.zeros((B, 0), np.int32)
    S = np.tile(np.arange(N, dtype=np.int32), (B, H, 1))
    qh, o, z, c, _ = orc.attention(False, A, A, q2, st.qhat, st.o, st.z, st.c, S, k, v, k2, v2)
    assert np.array_equal(o, st.o) and np.array_equal(z, st.z)
    assert np.array_equal(c, st.c) and np.array_equal(qh, st.qhat)


def test_rows_before_every_selected_key_are_unchanged(orc):
    q, k, v = _tensors(18)
    st, _ = _dense_first(orc, q, k, v)
    q2, k2, v2 = _tensors(19)
    B, N, H, d = q.shape
    S = np.tile(np.arange(30, 40, dtype=np.int32), (B, H, 1))      # every key >= 30
    A = np.tile(np.arange(0, N, 2, dtype=np.int32), (B, 1))
    qh, o, z, c, m = orc.attention(False, A, A, q2, st.qhat, st.o, st.z, st.c, S, k, v, k2, v2, want_m=True)
    early = A[0][A[0] < 30]
    assert np.array_equal(o[:, early], st.o[:, early]) and np.array_equal(qh[:, early], st.qhat[:, early])
    assert np.array_equal(z[:, :, early], st.z[:, :, early])
    assert np.isnan(m[:, :, : early.size]).all()
    late = A[0][A[0] >= 30]
    assert not np.array_equal(o[:, late], st.o[:, late])
    assert np.array_equal(c[..., :30], st.c[..., :30]) and np.array_equal(c[..., 40:], st.c[..., 40:])


def _prefix_softmax(q_rows, k, v, pos):
    """Per (sequence, head, row): textbook softmax of q.k_j/sqrt(d) over keys
    j <= pos in float64, giving (o, lse, p) with p over all keys (0 past pos)."""
    q, k, v = (bits_to_f32(t).astype(np.float64) for t in (q_rows, k, v))
    B, R, H, d = q.shape
    Nk = k.shape[1]
    o = np.zeros((B, R, H, d))
    lse = np.zeros((B, H, R))
    p = np.zeros((B, H, R, Nk))
    for b in range(B):
        for h in range(H):
            for r in range(R):
                n = pos[b, r] + 1
                x = k[b, :n, h] @ q[b, r, h] / math.sqrt(d)
                mx = x.max()
                e = np.exp(x - mx)
                p[b, h, r, :n] = e / e.sum()
                lse[b, h, r] = mx + math.log(e.sum())
                o[b, r, h] = p[b, h, r, :n] @ v[b, :n, h]
    return o, lse, p


def _decode_rows(seed, B=2, N=37, H=2, d=64):
    """Two state slots per sequence whose rows sit at key positions N - 5 and
    N (slots stored in the opposite order), over N + 1 keys: the decode form,
    where a row's state slot is not its key position."""
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((B, 2, H, d)))
    k, v = (bf16_bits(rng.standard_normal((B, N + 1, H, d))) for _ in range(2))
    pos = np.tile(np.array([N - 5, N], np.int32), (B, 1))
    slot = np.tile(np.array([1, 0], np.int32), (B, 1))
    S = np.tile(np.arange(N + 1, dtype=np.int32), (B, H, 1))
    return q, k, v, pos, slot, S


def _by_slot(x_rows, slot, axis):
    """Rows of x (row order) placed at their state slots along `axis`."""
    out = np.empty_like(x_rows)
    for r in range(slot.shape[1]):
        idx = [slice(None)] * x_rows.ndim
        src = list(idx)
        idx[axis], src[axis] = int(slot[0, r]), r
        out[tuple(idx)] = x_rows[tuple(src)]
    return out


def test_decode_rows_first_dense_is_prefix_softmax(orc):
    """First dense loop on rows whose state slot differs from their key
    position: each row gets softmax attention over its own causal prefix, and
    c starts afresh as the sum of the rows' probabilities (any earlier c is
    discarded, as the first dense loop has no previous state)."""
    q, k, v, pos, slot, S = _decode_rows(21)
    B, R, H, d = q.shape
    Nk = k.shape[1]
    q_slots = _by_slot(q, slot, 1)
    c0 = np.random.default_rng(3).random((B, H, Nk)).astype(np.float32)
    qh, o, z, c, m = orc.attention(True, pos, slot, q_slots, q_slots, np.full((B, R, H, d), 9.0, np.float32),
                                   np.zeros((B, H, R), np.float32), c0, S, None, None, k, v, want_m=True)
    o_ref, lse_ref, p_ref = _prefix_softmax(q, k, v, pos)
    np.testing.assert_allclose(o, _by_slot(o_ref, slot, 1), rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(z, _by_slot(lse_ref, slot, 2), rtol=0, atol=5e-6)
    np.testing.assert_allclose(c, p_ref.sum(2), rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(m, 1.0, rtol=0, atol=0)
    assert np.array_equal(qh, q_slots)


def test_decode_rows_lazy_full_set_is_softmax_of_new_keys(orc):
    """A lazy loop over every key, after a dense loop on the previous keys, on
    the decode-form rows: m = 1 and the result is softmax attention over the
    new keys, each row over its own prefix."""
    q1, k1, v1, pos, slot, S = _decode_rows(22)
    q2, k2, v2, _, _, _ = _decode_rows(23)
    B, R, H, d = q1.shape
    Nk = k1.shape[1]
    q1s, q2s = _by_slot(q1, slot, 1), _by_slot(q2, slot, 1)
    zeros_c = np.zeros((B, H, Nk), np.float32)
    qh1, o1, z1, c1, _ = orc.attention(True, pos, slot, q1s, q1s, np.zeros((B, R, H, d), np.float32),
                                       np.zeros((B, H, R), np.float32), zeros_c, S, None, None, k1, v1)
    qh2, o2, z2, c2, m = orc.attention(False, pos, slot, q2s, qh1, o1, z1, c1, S, k1, v1, k2, v2, want_m=True)
    o_ref, lse_ref, p_ref = _prefix_softmax(q2, k2, v2, pos)
    np.testing.assert_allclose(m, 1.0, rtol=0, atol=2e-6)
    np.testing.assert_allclose(o2, _by_slot(o_ref, slot, 1), rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(z2, _by_slot(lse_ref, slot, 2), rtol=0, atol=5e-6)
    np.testing.assert_allclose(c2, p_ref.sum(2), rtol=1e-5, atol=2e-6)
    assert np.array_equal(qh2, q2s)


def test_chain_preserves_mass_and_bounds_m(orc):
    """Tiny workload through loops 1..T on the oracle alone: every row keeps
    unit mass, so the column masses always sum to the causal row count N."""
    from oracle import loop
    w = synth.WORKLOADS["tiny"]
    w = synth.Workload(**{**w.__dict__, "N": 256})
    R, K = synth.active_count(w), synth.key_count(w)
    cache, st, prev = loop.Cache(), None, None
    for x in synth.prefill_loops(w):
        l = x["loop"]
        if l == 1:
            st = loop.empty_state(w.B, w.N, w.H, w.d)
            st = loop.dense_loop(1, x["Q"], x["K"], x["V"], cache, st)
        else:
            A, S, scores, st2, lk, lv = loop.lazy_loop(l, prev, x["H"], x["Q"], x["K"], x["V"],
                                                       cache, st, R, K)
            assert A.shape == (w.B, R) and S.shape == (w.B, w.H, K)
            assert np.all(np.diff(A, axis=-1) > 0) and np.all(np.diff(S, axis=-1) > 0)
            # the heavy tokens (large drift) are the ones selected
            assert np.isin(np.nonzero(x["heavy"][0].numpy())[0], A[0]).mean() > 0.95
            rows = A
            _, _, _, _, m = orc.attention(False, rows, rows, x["Q"], st.qhat, st.o, st.z, st.c, S,
                                          cache.rec(l - 1, "k"), cache.rec(l - 1, "v"),
                                          cache.rec(l, "k"), cache.rec(l, "v"), want_m=True)
            mm = m[~np.isnan(m)]
            assert np.all(mm > 0) and np.all(np.isfinite(mm))
            if l == 2:
                # every row's state was computed against the loop-1 keys, so its
                # tracked probabilities over any subset sum to at most one
                assert np.all(mm <= 1 + 1e-6)
            st = st2
        np.testing.assert_allclose(st.c.sum(-1), w.N, rtol=1e-6)
        prev = x["H"]


# ---------------------------------------------------------------------------
# key ranking by column mass per causal row, and the column-recovery measure

def test_key_scores_per_row_hand_worked(orc):
    """c = [8, 3, 4, 3] over N = 4 rows: rows 4, 3, 2, 1 see keys 0..3, so the
    scores are [2, 1, 2, 3]; the top two are key 3 and, of the tie at 2, key 0."""
    s = orc.key_scores_per_row(np.array([[8.0, 3.0, 4.0, 3.0]], np.float32), 4)
    assert s.tolist() == [[2.0, 1.0, 2.0, 3.0]]
    assert orc.topk(s, 2).tolist() == [[0, 3]]
    # more rows than columns (a prefix of a longer prefill): rows 6..3 see keys 0..3
    s = orc.key_scores_per_row(np.array([6.0, 5.0, 4.0, 3.0], np.float32), 6)
    assert s.tolist() == [1.0, 1.0, 1.0, 1.0]


def test_key_scores_per_row_is_the_fp32_quotient(orc):
    """The quotient is rounded once to fp32 (as a kernel's IEEE fp32 division
    would), checked against exact rational arithmetic on random values."""
    from fractions import Fraction
    rng = np.random.default_rng(5)
    c = (rng.random(300) * 50).astype(np.float32)
    s = orc.key_scores_per_row(c, 1000)
    for j in range(0, 300, 7):
        exact = Fraction(float(c[j])) / (1000 - j)
        # s[j] is the fp32 nearest to the exact quotient: no fp32 lies strictly closer
        up, dn = np.nextafter(np.float32(s[j]), np.float32(np.inf)), np.nextafter(np.float32(s[j]), np.float32(-np.inf))
        err = abs(Fraction(float(s[j])) - exact)
        assert err <= abs(Fraction(float(up)) - exact) and err <= abs(Fraction(float(dn)) - exact)


def test_column_recovery_closed_forms(orc):
    prev = np.zeros((3, 4))
    full = np.ones((3, 4))
    assert orc.column_recovery(full, full, prev)["recovered"] == 1.0          # exact result
    assert orc.column_recovery(prev, full, prev)["recovered"] == 0.0          # no update at all
    half = orc.column_recovery(0.5 * full, full, prev)
    assert half["recovered"] == 0.5 and half["rel_err"] == 0.5


def test_full_key_set_recovers_everything(orc):
    """The lazy step over every key of a (tiny) loop is the exact result: its
    recovery is 1 by the mass-preserving identity, whatever the previous state."""
    rng = np.random.default_rng(9)
    B, N, H, d = 1, 40, 1, 64
    bf = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q1, k1, v1, q2, k2, v2 = (bf(rng.standard_normal((B, N, H, d))) for _ in range(6))
    rows = np.arange(N, dtype=np.int32)[None]
    S_all = np.arange(N, dtype=np.int32)[None, None]
    zero = (np.zeros((B, N, H, d), np.uint16), np.zeros((B, N, H, d), np.float32),
            np.zeros((B, H, N), np.float32), np.zeros((B, H, N), np.float32))
    st = orc.attention(True, rows, rows, q1, *zero, S_all, None, None, k1, v1)[:4]
    A = np.array([[3, 10, 22, 39]], np.int32)
    full = orc.attention(False, A, A, q2, *st, S_all, k1, v1, k2, v2)[1]
    some = orc.attention(False, A, A, q2, *st, np.array([[[0, 5, 10, 22]]], np.int32), k1, v1, k2, v2)[1]
    rec_full = orc.column_recovery(full[:, A[0]], full[:, A[0]], st[1][:, A[0]])
    assert rec_full["recovered"] == 1.0
    rec = orc.column_recovery(some[:, A[0]], full[:, A[0]], st[1][:, A[0]])
    assert rec["recovered"] < 1.0 and rec["rel_err"] > 0


# ---------------------------------------------------------------------------
# early exit by state difference

def _exit_case(orc, B=3, N=64, H=2, d=64, seed=21):
    from oracle import loop as oloop
    rng = np.random.default_rng(seed)
    bf = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    h1 = rng.standard_normal((B, N, H * d))
    h2 = h1 + rng.standard_normal((B, N, H * d)) * np.array([0.5, 0.0, 0.01])[:, None, None]   # seq 1 frozen
    q1, k1, v1, q2, k2, v2 = (bf(rng.standard_normal((B, N, H, d))) for _ in range(6))
    cache = oloop.Cache()
    st = oloop.dense_loop(1, q1, k1, v1, cache, oloop.empty_state(B, N, H, d))
    return oloop, bf(h1), bf(h2), (q2, k2, v2), cache, st


def test_exit_threshold_zero_changes_nothing(orc):
    oloop, h1, h2, (q2, k2, v2), cache, st = _exit_case(orc)
    import copy
    plain = oloop.lazy_loop(2, h1, h2, q2, k2, v2, copy.deepcopy(cache), st, 16, 8)
    ex = oloop.lazy_loop(2, h1, h2, q2, k2, v2, copy.deepcopy(cache), st, 16, 8, exit_threshold=0.0,
                         exited=np.zeros(3, bool))
    assert not ex[6].any()
    for a, b in zip(plain[3].__dict__.values(), ex[3].__dict__.values()):
        assert np.array_equal(a, b)
    assert np.array_equal(plain[4].codes, ex[4].codes) and np.array_equal(plain[4].scales, ex[4].scales)


def test_frozen_sequence_exits_and_keeps_its_state(orc):
    """Sequence 1 did not change between the loops (every score 0), so any
    positive threshold stops it: its rows keep O, Z, qhat and c bit for bit and
    its delta entries are zero; the other sequences loop as usual."""
    oloop, h1, h2, (q2, k2, v2), cache, st = _exit_case(orc)
    import copy
    plain = oloop.lazy_loop(2, h1, h2, q2, k2, v2, copy.deepcopy(cache), st, 16, 8)
    A, S, scores, new, lk, lv, flags = oloop.lazy_loop(2, h1, h2, q2, k2, v2, copy.deepcopy(cache), st, 16, 8,
                                                       exit_threshold=1e-6)
    assert flags.tolist() == [False, True, False]
    assert scores[1].max() == 0.0
    for name in ("qhat", "o", "z", "c"):
        assert np.array_equal(getattr(new, name)[1], getattr(st, name)[1])        # exited: unchanged
        assert np.array_equal(getattr(new, name)[[0, 2]], getattr(plain[3], name)[[0, 2]])   # others: as usual
    assert not lk.codes[1].any() and not lk.scales[1].any() and not lv.scales[1].any()
    assert lk.scales[0].any()


def test_exit_is_strict_and_sticky(orc):
    from oracle import loop as oloop
    scores = np.array([[0.5, 2.0], [1.0, 0.25], [3.0, 3.0]])
    # largest scores 2.0, 1.0, 3.0: a threshold equal to a maximum does not stop it
    assert oloop.exit_flags(scores, 1.0).tolist() == [False, False, False]
    assert oloop.exit_flags(scores, 1.0 + 1e-6).tolist() == [False, True, False]
    # a flag once set stays set, whatever the scores
    assert oloop.exit_flags(scores, 0.5, np.array([True, False, False])).tolist() == [True, False, False]
    assert oloop.exit_flags(scores, float("inf")).tolist() == [True, True, True]


# ---------------------------------------------------------------------------
# narrower deltas (int3, int2) and the int8 compressed base

def _bf(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _one_group_append(orc, delta32, code_bits, d=32):
    """A single-token, single-head layer whose delta against a zero base is `delta32`."""
    x = np.zeros((1, 1, 1, d), np.float32)
    x[0, 0, 0, :32] = delta32
    return orc.kv_delta_append(_bf(x), _bf(np.zeros_like(x)), [], np.array([[0]], np.int32), code_bits=code_bits)


def test_int3_group_hand_worked(orc):
    """amax 3 -> scale fp16(3/3) = 1; codes rint(3, -1.5, 0.75, 0) = 3, -2
    (the tie goes to even), 1, 0; 3-bit two's complement from bit 0 upward:
    011, 110, 001 -> byte 0 = 0b01110011 = 0x73, byte 1 bit 0 = 0."""
    delta = np.zeros(32, np.float32)
    delta[:4] = [3.0, -1.5, 0.75, 0.0]
    lay = _one_group_append(orc, delta, 3)
    assert lay.codes.shape == (1, 1, 1, 12) and lay.scales.tolist() == [[[[0x3C00]]]]   # fp16 1.0
    assert lay.codes[0, 0, 0, 0] == 0x73 and (lay.codes[0, 0, 0, 1] & 1) == 0
    assert not lay.codes[0, 0, 0, 2:].any()


def test_int2_group_hand_worked(orc):
    """amax 0.625 (exact in bf16 and fp16) -> scale 0.625; codes rint(1, -0.32, -0.8, 0.8) = 1, 0, -1, 1
    -> 2-bit fields 01, 00, 11, 01 -> byte 0 = 0b01110001 = 0x71."""
    delta = np.zeros(32, np.float32)
    delta[:4] = [0.625, -0.2, -0.5, 0.5]
    lay = _one_group_append(orc, delta, 2)
    assert lay.codes.shape == (1, 1, 1, 8) and lay.scales.tolist() == [[[[0x3900]]]]   # fp16 0.625
    assert lay.codes[0, 0, 0, 0] == 0x71 and not lay.codes[0, 0, 0, 1:].any()


@pytest.mark.parametrize("code_bits", [2, 3, 4])
def test_narrow_deltas_round_trip_within_half_a_scale(orc, code_bits):
    """|delta - s q| <= s/2 wherever the code is not clamped, for every width, and
    codes stay in [-qmax, qmax]; the reconstruction reads back the same codes."""
    rng = np.random.default_rng(40 + code_bits)
    B, N, H, d = 1, 40, 2, 96
    base = _bf(rng.standard_normal((B, N, H, d)))
    x = _bf((np.asarray(base, np.uint32) << 16).view(np.float32) + 0.1 * rng.standard_normal((B, N, H, d)))
    A = np.array([np.sort(rng.choice(N, 15, replace=False))], np.int32)
    lay = orc.kv_delta_append(x, base, [], A, code_bits=code_bits)
    qmax = (1 << (code_bits - 1)) - 1
    rec, _ = orc.reconstruct(base, [lay], want_bf16=False, code_bits=code_bits)
    xf = (np.asarray(x, np.uint32) << 16).view(np.float32)
    bf = (np.asarray(base, np.uint32) << 16).view(np.float32)
    s = np.repeat(lay.scales.view(np.float16).astype(np.float32), 32, axis=-1)[0]
    delta = (xf - bf)[0][A[0]]
    q = (rec[0][A[0]] - bf[0][A[0]]) / np.where(s > 0, s, 1)
    assert np.all(np.abs(np.round(q)) <= qmax) and np.allclose(q, np.round(q))
    inside = np.abs(delta) <= s * qmax
    assert np.all(np.abs(delta - s * np.round(q))[inside] <= s[inside] / 2 + 1e-12)
    others = np.setdiff1d(np.arange(N), A[0])
    assert np.array_equal(rec[0][others], bf[0][others])


def test_int8_base_round_trip_and_reconstruction(orc):
    rng = np.random.default_rng(44)
    x = _bf(rng.standard_normal((2, 30, 3, 64)) * 3)
    cb = orc.quantize_base(x)
    xf = (np.asarray(x, np.uint32) << 16).view(np.float32)
    s = np.repeat(cb.scales.view(np.float16).astype(np.float32), 32, axis=-1)
    assert np.all(np.abs(cb.codes.astype(np.int32)) <= 127)
    assert np.all(np.abs(xf - s * cb.codes) <= s / 2 + 1e-12)
    # the group's largest element maps to +-127 exactly when the scale is amax/127 in fp16
    rec, _ = orc.reconstruct(cb, [], want_bf16=False)
    assert np.array_equal(rec, (s * cb.codes.astype(np.float32)).astype(np.float32))
    zero = orc.quantize_base(np.zeros((1, 2, 1, 32), np.uint16))
    assert not zero.codes.any() and not zero.scales.any()
