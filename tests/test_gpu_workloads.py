"""The five workloads end to end through flashloop_loop_step, compared with the
CPU oracle loop by loop (teacher forcing: the oracle starts every loop from
the GPU's previous state, selections and cache, so legitimate near-threshold
differences cannot cascade). Large workloads are compared on a seeded subset
of sequences, heads and (for dense loops) rows; every token still takes part
in the selections."""
import numpy as np
import pytest
import torch

import oracle
import synth
import lazy_sparse_attention_token_b300 as fl
from lazy_sparse_attention_token_b300 import build as flbuild
from gpu_helpers import (C_ATOL, C_RTOL, O_ATOL, O_RTOL, Z_ATOL, State, assert_close, assert_layer,
                         assert_selection, bits, check_slot_map, delta_over_scale, dims_for, f32,
                         layers_from_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    flbuild.build()
    fl.lib()
    oracle.build()


def _sample_rows(N, seed, n_rand=24):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 2, 127, 128, 129, N // 2, N - 129, N - 128, N - 1]
    rows = set(r for r in fixed if 0 <= r < N) | set(rng.choice(N, min(N, n_rand), replace=False).tolist())
    return np.array(sorted(rows), np.int32)


def _check_append(cache, l, x_l, name, base, prev_layers, A, bsel, rows_are_tokens=True, entry0=0):
    idx, slot, kc, ks, vc, vs = cache.delta_layer(l)
    codes, scales = (kc, ks) if name == "K" else (vc, vs)
    g_codes = codes[bsel][:, entry0:].cpu().numpy()
    g_scales = scales[bsel][:, entry0:].cpu().numpy().view(np.uint16)
    orc = oracle.kv_delta_append(x_l, base, prev_layers, A)
    if np.array_equal(g_codes, orc.codes) and np.array_equal(g_scales, orc.scales):
        return
    rec, _ = oracle.reconstruct(base, prev_layers, want_bf16=False)
    rows = np.stack([rec[i, A[i]] for i in range(len(bsel))])
    xb = np.stack([x_l[i, A[i]] for i in range(len(bsel))])
    assert_layer(g_codes, g_scales, orc.codes, orc.scales, delta_over_scale(xb, rows, orc.scales), f"{name} layer {l}")


def _pick_heads(H, n, seed):
    """n heads of H for the attention comparison: the first, the last, and a
    seeded draw of the rest (every head still takes part in the selections
    and the delta appends, which are compared on all heads)."""
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, H - 1), size=max(0, min(n, H) - 2), replace=False).tolist()
    return sorted({0, H - 1, *mid})


def _dense_full_rows(name, l, first, x, bsel, head, before_full, cache, w):
    """Dense loop l on every row of one (sequence, head): O, Z, q_hat and the
    column masses c, all of them, against the oracle on the same inputs."""
    sl = lambda t: bits(t[bsel][:, :, [head]])
    q, k_new, v_new = sl(x["Q"]), sl(x["K"]), sl(x["V"])
    k_old = v_old = None
    if not first:
        ko, vo = cache.dense_layer(l - 1)
        k_old, v_old = bits(ko[bsel][:, :w.N][:, :, [head]]), bits(vo[bsel][:, :w.N][:, :, [head]])
    rows = np.tile(np.arange(w.N, dtype=np.int32), (len(bsel), 1))
    S = np.tile(np.arange(w.N, dtype=np.int32), (len(bsel), 1, 1))
    qh, o, z, c, _ = oracle.attention(first, rows, rows, q, *before_full, S, k_old, v_old, k_new, v_new)
    return qh, o, z, c


def run_prefill(name, bsel, hsel, full_dense=False, loops_to_check=None, keep=False, full_rows_loop=None):
    w = synth.WORKLOADS[name]
    extra = 1 if w.decode_after_prefill else 0
    dm = dims_for(w, extra_tokens=extra, R_extra=extra)
    R, K = dm.R, dm.K
    cache = fl.Cache(dm)
    cache.n_tokens = w.N
    ws = fl.workspace_for(dm)
    st = State(w.B, w.N, w.H, w.d, w.N)
    active = torch.empty(w.B, R, dtype=torch.int32, device="cuda")
    keys = torch.empty(w.B, w.H, K, dtype=torch.int32, device="cuda")
    scores = torch.empty(w.B, w.N, dtype=torch.float32, device="cuda")
    prev = None
    for x in synth.prefill_loops(w, device="cuda"):
        l = x["loop"]
        check = loops_to_check is None or l in loops_to_check
        before = st.snapshot(bsel, hsel) if check else None
        full_rows = check and l == full_rows_loop
        before_full = st.snapshot(bsel, [hsel[0]]) if full_rows else None
        if check and l > w.T_dense:
            prev_k, prev_v = layers_from_gpu(cache, range(w.T_dense + 1, l), bsel)
            c_full_before = f32(st.c[bsel])
        fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], st.q_hat, st.o, st.z, st.c, ws,
                               h_prev=prev, h_cur=x["H"], active_idx=active, key_idx=keys, scores=scores)
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        if check:
            sl = lambda t: bits(t[bsel][:, :, hsel])
            q = sl(x["Q"])
            if l <= w.T_dense:
                k_new, v_new = sl(x["K"]), sl(x["V"])
                k_old = v_old = None
                if l > 1:
                    ko, vo = cache.dense_layer(l - 1)
                    k_old, v_old = bits(ko[bsel][:, :w.N][:, :, hsel]), bits(vo[bsel][:, :w.N][:, :, hsel])
                rows = np.arange(w.N, dtype=np.int32) if full_dense else _sample_rows(w.N, l)
                rr = np.tile(rows, (len(bsel), 1))
                S = np.tile(np.arange(w.N, dtype=np.int32), (len(bsel), len(hsel), 1))
                qh, o, z, c, _ = oracle.attention(l == 1, rr, rr, q, *before, S, k_old, v_old, k_new, v_new)
                after = st.snapshot(bsel, hsel)
                assert_close(after[1][:, rows], o[:, rows], O_ATOL, O_RTOL, f"{name} loop {l} O")
                assert_close(after[2][:, :, rows], z[:, :, rows], Z_ATOL, 0, f"{name} loop {l} Z")
                assert np.array_equal(after[0][:, rows], qh[:, rows])
                if full_dense:
                    assert_close(after[3], c, C_ATOL, C_RTOL, f"{name} loop {l} c")
                if full_rows:
                    # every row of the first sampled head, and its complete column masses
                    qh1, o1, z1, c1 = _dense_full_rows(name, l, l == 1, x, bsel, hsel[0], before_full, cache, w)
                    got = st.snapshot(bsel, [hsel[0]])
                    what = f"{name} loop {l} head {hsel[0]} all {w.N} rows"
                    assert_close(got[1], o1, O_ATOL, O_RTOL, what + " O")
                    assert_close(got[2], z1, Z_ATOL, 0, what + " Z")
                    assert np.array_equal(got[0], qh1), what + " q_hat"
                    assert_close(got[3], c1, C_ATOL, C_RTOL, what + " c")
            else:
                # (1) token selection on the full hidden state of each sequence
                sc = oracle.token_scores(bits(prev[bsel]), bits(x["H"][bsel]))
                assert_close(f32(scores[bsel]), sc, 1e-30, 2e-6, f"{name} loop {l} scores")
                A_orc = oracle.topk(sc, R)
                A = active[bsel].cpu().numpy()
                for i in range(len(bsel)):
                    assert_selection(A[i], A_orc[i], sc[i], f"{name} loop {l} active set")
                # (3) delta append of every head, from the GPU's previous cache
                base_k, base_v = (bits(t[bsel][:, :w.N]) for t in cache.dense_layer(w.T_dense))
                _check_append(cache, l, bits(x["K"][bsel]), "K", base_k, prev_k, A, bsel)
                _check_append(cache, l, bits(x["V"][bsel]), "V", base_v, prev_v, A, bsel)
                check_slot_map(cache, l, w.N)
                # (4) key columns from the previous loop's column mass
                S = keys[bsel].cpu().numpy()
                S_orc = oracle.topk(c_full_before.astype(np.float64), K)
                assert np.array_equal(S, S_orc), f"{name} loop {l} key columns"
                # attention over the reconstructed cache
                lk, lv = layers_from_gpu(cache, range(w.T_dense + 1, l + 1), bsel, hsel)
                bk, bv = base_k[:, :, hsel], base_v[:, :, hsel]
                k_old = oracle.reconstruct(bk, lk[:-1], want_f32=False)[1]
                v_old = oracle.reconstruct(bv, lv[:-1], want_f32=False)[1]
                k_new = oracle.reconstruct(bk, lk, want_f32=False)[1]
                v_new = oracle.reconstruct(bv, lv, want_f32=False)[1]
                qh, o, z, c, _ = oracle.attention(False, A, A, q, *before, S[:, hsel], k_old, v_old, k_new, v_new)
                after = st.snapshot(bsel, hsel)
                assert_close(after[1], o, O_ATOL, O_RTOL, f"{name} loop {l} O")
                assert_close(after[2], z, Z_ATOL, 0, f"{name} loop {l} Z")
                assert_close(after[3], c, C_ATOL, C_RTOL, f"{name} loop {l} c")
                assert np.array_equal(after[0], qh), f"{name} loop {l} q_hat"
        # every row keeps unit mass: column masses sum to the row count
        np.testing.assert_allclose(f32(st.c).sum(-1), w.N, rtol=1e-3)
        prev = x["H"]
    if keep:
        return w, dm, cache, ws
    return None


def test_tiny_every_output():
    run_prefill("tiny", [0], [0, 1, 2, 3], full_dense=True)


def test_8k_prefill():
    w = synth.WORKLOADS["8k"]
    run_prefill("8k", [0], _pick_heads(w.H, 4, 8), full_rows_loop=1)


def test_32k_prefill():
    w = synth.WORKLOADS["32k"]
    run_prefill("32k", [0], _pick_heads(w.H, 4, 32), full_rows_loop=1)


def _decode_loops(w, dm, cache, ws, bsel, hsel):
    """One new token per sequence through loops 1..T, checked on sequences
    bsel (appends: every head; attention: heads hsel)."""
    N = cache.n_tokens - 1   # the new token's key position
    Nk = N + 1
    K = dm.K
    st = State(w.B, 1, w.H, w.d, Nk)
    keys = torch.empty(w.B, w.H, K, dtype=torch.int32, device="cuda")
    pos = np.full((len(bsel), 1), N, np.int32)
    slot = np.zeros((len(bsel), 1), np.int32)
    for t in synth.decode_token_loops(w, device="cuda"):
        l = t["loop"]
        before = st.snapshot(bsel, hsel)
        td = w.T_dense
        if l > td:
            prev_k, prev_v = layers_from_gpu(cache, range(td + 1, l), bsel)
            m = l - td - 1
            entry0 = cache.c.count[m]
        fl.flashloop_loop_step(cache, l, t["q"], t["k"], t["v"], st.q_hat, st.o, st.z, st.c, ws, key_idx=keys,
                               decode=True)
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        q = bits(t["q"][bsel][:, :, hsel])
        if l <= td:
            kn, vn = (bits(x[bsel][:, :Nk][:, :, hsel]) for x in cache.dense_layer(l))
            ko = vo = None
            if l > 1:
                ko, vo = (bits(x[bsel][:, :Nk][:, :, hsel]) for x in cache.dense_layer(l - 1))
            S = np.tile(np.arange(Nk, dtype=np.int32), (len(bsel), len(hsel), 1))
            qh, o, z, c, _ = oracle.attention(l == 1, pos, slot, q, *before, S, ko, vo, kn, vn)
        else:
            S = keys[bsel][:, hsel].cpu().numpy()
            S_orc = oracle.topk(before[3].astype(np.float64), K)
            assert np.array_equal(S, S_orc), f"decode loop {l} key columns"
            base_k, base_v = (bits(x[bsel][:, :Nk]) for x in cache.dense_layer(td))
            xk = np.zeros_like(base_k)
            xk[:, N] = bits(t["k"][bsel])[:, 0]
            xv = np.zeros_like(base_v)
            xv[:, N] = bits(t["v"][bsel])[:, 0]
            _check_append(cache, l, xk, "K", base_k, prev_k, pos, bsel, entry0=entry0)
            _check_append(cache, l, xv, "V", base_v, prev_v, pos, bsel, entry0=entry0)
            lk, lv = layers_from_gpu(cache, range(td + 1, l + 1), bsel, hsel)
            bk, bv = base_k[:, :, hsel], base_v[:, :, hsel]
            ko = oracle.reconstruct(bk, lk[:-1], want_f32=False)[1]
            vo = oracle.reconstruct(bv, lv[:-1], want_f32=False)[1]
            kn = oracle.reconstruct(bk, lk, want_f32=False)[1]
            vn = oracle.reconstruct(bv, lv, want_f32=False)[1]
            qh, o, z, c, _ = oracle.attention(False, pos, slot, q, *before, S, ko, vo, kn, vn)
        after = st.snapshot(bsel, hsel)
        assert_close(after[1], o, O_ATOL, O_RTOL, f"decode loop {l} O")
        assert_close(after[2], z, Z_ATOL, 0, f"decode loop {l} Z")
        assert_close(after[3], c, C_ATOL, C_RTOL, f"decode loop {l} c")
        assert np.array_equal(after[0], qh)
        np.testing.assert_allclose(f32(st.c).sum(-1), 1.0, rtol=1e-3)


def test_decode():
    w = synth.WORKLOADS["decode"]
    ctx = synth.decode_context(w, device="cuda")
    R_ctx = ctx["loops"][2]["active"].shape[1]
    Nk = w.N + 1
    dm = fl.make_dims(w.B, Nk, w.H, w.d, R_ctx, synth.key_count(w, Nk), w.T, w.T_dense, R_cap=R_ctx + 1)
    cache = fl.Cache(dm)
    cache.n_tokens = w.N
    ws = fl.workspace_for(dm)
    bsel = [0, 37]
    fl.flashloop_kv_dense_store(cache, 1, ctx["K1"], ctx["V1"])
    for l in range(2, w.T + 1):
        L = ctx["loops"][l]
        prev_k, prev_v = layers_from_gpu(cache, range(2, l), bsel)
        fl.flashloop_kv_delta_append(cache, l, L["K"], L["V"], L["active"])
        torch.cuda.synchronize()
        base_k, base_v = (bits(x[bsel][:, :w.N]) for x in cache.dense_layer(1))
        A = L["active"][bsel].cpu().numpy()
        _check_append(cache, l, bits(L["K"][bsel]), "K", base_k, prev_k, A, bsel)
        _check_append(cache, l, bits(L["V"][bsel]), "V", base_v, prev_v, A, bsel)
    cache.n_tokens = Nk
    _decode_loops(w, dm, cache, ws, bsel, [0, 7, 15])


def test_deep_prefill_then_decode():
    """Two sequences x two heads (the first and the last) through the prefill;
    the second dense loop (previous state in use, m and u computed) on every
    row of one head; then a decode token on two more sequences and heads."""
    w = synth.WORKLOADS["deep"]
    w, dm, cache, ws = run_prefill("deep", [0, 5], [0, w.H - 1], loops_to_check={1, 2, 3, 4, 9, 16}, keep=True,
                                   full_rows_loop=2)
    cache.n_tokens = w.N + 1
    _decode_loops(w, dm, cache, ws, [3, 7], [5, 30])
