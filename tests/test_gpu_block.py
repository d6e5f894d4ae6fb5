"""GPU parity of the tensor-core GEMM and of the synthetic looped block
(projections and MLP around the lazy step) against the CPU oracle.

The GEMM rounds an fp32 accumulation to bf16 where the oracle rounds the exact
sum, so outputs agree bit for bit except where the exact value lies within
the accumulation error of a bf16 rounding boundary. The error of a K-term
fp32 sum is at most K * 2^-24 * S, with S the sum of the terms' magnitudes
(plus the residual's): an output may differ from the oracle's by one bf16 ulp
plus that bound (more than one ulp only where the sum cancels), in a small
fraction of the elements. The block's hidden states also inherit the attention's fp32/bf16-probability deviations
(the attention tolerances of the other parity tests), propagated through
W_o and the MLP: the dense loop and the first lazy loop are compared with
each side running on its own; every loop is compared with the oracle started
from the GPU's previous state, as in the workload tests, because a 4-bit delta
code on a rounding boundary may round either way on the two sides (both
correct) and move a reconstructed K or V element by a whole quantisation step,
which later loops would carry on.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import lazy_sparse_attention_token_b300 as fl
from oracle import block as ob
from oracle.loop import Cache as OCache, empty_state
from gpu_helpers import (C_ATOL, C_RTOL, O_ATOL, O_RTOL, Z_ATOL, State, assert_close, assert_layer,
                         assert_selection, bits, delta_over_scale, f32, layers_from_gpu)
from oracle.loop import State as OState, dense_loop, lazy_loop

pytestmark = pytest.mark.gpu

H_ATOL, H_RTOL = 4e-2, 2e-2    # hidden states after the attention-dependent steps
MLP_ATOL, MLP_RTOL = 1e-2, 1e-2  # the MLP from the same attention output (three GEMMs' roundings)


def gemm_max_frac(K: int) -> float:
    """Fraction of outputs allowed to differ from the exactly rounded value.
    A K-term fp32 sum typically errs by about sqrt(K) 2^-24 of its magnitude,
    and a bf16 ulp is 2^-8 (to 2^-7) of it, so about 2 sqrt(K) 2^-16 of the
    outputs lie that close to a rounding boundary; four times that is allowed."""
    return 8.0 * np.sqrt(K) * 2.0 ** -16


def _ulp(v: np.ndarray) -> np.ndarray:
    """bf16 unit in the last place at |v| (normal range)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def gemm_bound(a_bits, w_bits, res_bits=None):
    """K * 2^-24 * S: the fp32 accumulation error bound of each output, with S
    = |A| |W|^T (+ |residual|) the sum of the terms' magnitudes."""
    s = np.abs(oracle.bf16_values(a_bits)) @ np.abs(oracle.bf16_values(w_bits)).T
    if res_bits is not None:
        s = s + np.abs(oracle.bf16_values(res_bits))
    return (a_bits.shape[-1] + 1) * 2.0 ** -24 * s


def assert_gemm(gpu_bits, orc_bits, bound, what, K):
    max_frac = gemm_max_frac(K)
    g, o = oracle.bf16_values(gpu_bits), oracle.bf16_values(orc_bits)
    assert g.shape == o.shape, what
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    err = np.abs(g - o)
    bad = err > _ulp(o) + bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond one ulp plus the accumulation bound"
    frac = float((err > 0).mean()) if err.size else 0.0
    assert frac <= max_frac, f"{what}: {frac:.2e} of the elements differ (allowed {max_frac:.0e})"


def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _dev(t):
    return t.contiguous().cuda()


# ---------------------------------------------------------------------------
# GEMM

@pytest.mark.parametrize("M, K, N, with_res, relu", [
    (1, 64, 256, False, False),       # one row, one K slice
    (129, 192, 768, True, False),     # ragged rows, fewer K slices than ring slots
    (300, 1024, 512, True, True),     # several tiles, the ring wraps four times
    (513, 2048, 256, False, True),
])
def test_gemm_matches_oracle(M, K, N, with_res, relu):
    a = _rand_bf16((M, K), 1 + M)
    w = _rand_bf16((N, K), 2 + K, 1.0 / np.sqrt(K))
    res = _rand_bf16((M, N), 3 + N) if with_res else None
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fl.flashloop_gemm(_dev(a), _dev(w), [c], residual=None if res is None else _dev(res), relu=relu)
    torch.cuda.synchronize()
    rb = None if res is None else bits(res)
    want = ob.project(bits(a), bits(w), residual=rb, relu=relu)
    assert_gemm(bits(c), want, gemm_bound(bits(a), bits(w), rb), f"gemm {M}x{K}x{N}", K)


@pytest.mark.parametrize("n_split", [2, 3])
def test_gemm_split_and_scatter_to_token_rows(n_split):
    B, R, n_rows, K, D = 2, 150, 400, 256, 256
    g = torch.Generator().manual_seed(17)
    rows = torch.stack([torch.sort(torch.randperm(n_rows, generator=g)[:R]).values for _ in range(B)]).int()
    a = _rand_bf16((B * R, K), 5)
    w = _rand_bf16((n_split * D, K), 6, 1.0 / 16)
    sentinel = torch.tensor(0x7F7F, dtype=torch.int16).view(torch.bfloat16)
    outs = [torch.full((B * n_rows, D), float(sentinel), dtype=torch.bfloat16, device="cuda") for _ in range(n_split)]
    fl.flashloop_gemm(_dev(a), _dev(w), outs, c_rows=_dev(rows), rows_per_seq=R, seq_rows=n_rows)
    torch.cuda.synchronize()
    want = ob.project(bits(a), bits(w)).reshape(B, R, n_split, D)
    bound = gemm_bound(bits(a), bits(w)).reshape(B, R, n_split, D)
    for s in range(n_split):
        got = bits(outs[s]).reshape(B, n_rows, D)
        listed = np.zeros((B, n_rows), bool)
        for b in range(B):
            listed[b, rows[b].numpy()] = True
            assert_gemm(got[b, rows[b].numpy()], want[b, :, s], bound[b, :, s], f"output {s}, sequence {b}", K)
        assert np.all(got[~listed] == 0x7F7F), "rows not listed were written"


def test_gemm_out_of_range_row_is_reported_not_stored():
    M, K, N, n_rows = 8, 64, 256, 16
    rows = torch.arange(M, dtype=torch.int32) * 2
    rows[3] = n_rows                                  # outside [0, n_rows)
    a, w = _rand_bf16((M, K), 8), _rand_bf16((N, K), 9, 0.125)
    c = torch.zeros((n_rows + 1, N), dtype=torch.bfloat16, device="cuda")   # a spare row past the end
    fl.flashloop_gemm(_dev(a), _dev(w), [c], c_rows=_dev(rows), rows_per_seq=M, seq_rows=n_rows)
    assert fl.flashloop_device_status() == 0x101    # the GEMM's out-of-range row code
    assert fl.flashloop_device_status() == 0        # read and cleared
    got = bits(c)
    assert np.all(got[n_rows] == 0), "the out-of-range row was stored"
    want = ob.project(bits(a), bits(w))
    ok = [m for m in range(M) if m != 3]
    assert_gemm(got[rows[ok].numpy()], want[ok], gemm_bound(bits(a), bits(w))[ok], "rows in range", K)


def test_gemm_rejects_bad_shapes():
    a = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 96), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fl.FlashLoopError):
        fl.flashloop_gemm(a, w, [c])                    # K % 64 != 0
    a = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((384, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fl.FlashLoopError):
        fl.flashloop_gemm(a, w, [c])                    # N % 256 != 0


def test_gemm_full_size_projection_sampled_rows():
    # the projection shapes of the 32K workload's lazy loop: M = B R active
    # rows, D = 2048, 3D outputs; rows sampled for the oracle
    w32 = synth.WORKLOADS["32k"]
    M, D = synth.active_count(w32) * w32.B, w32.D
    a = _rand_bf16((M, D), 41)
    w = _rand_bf16((3 * D, D), 42, 1.0 / np.sqrt(D))
    outs = [torch.empty((M, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    fl.flashloop_gemm(_dev(a), _dev(w), outs)
    torch.cuda.synchronize()
    sample = np.array([0, 1, 127, 128, 2047, M // 2, M - 2, M - 1])
    want = ob.project(bits(a)[sample], bits(w))
    got = np.concatenate([bits(o)[sample] for o in outs], axis=1)
    assert_gemm(got, want, gemm_bound(bits(a)[sample], bits(w)), "32K projection, sampled rows", D)


# ---------------------------------------------------------------------------
# the looped block

CONFIGS = {
    "tiny": dict(B=2, N=384, H=2, d=128, F=512, T=4, T_dense=1, R=96, K=77),
    "wide": dict(B=1, N=1024, H=16, d=128, F=8192, T=3, T_dense=1, R=160, K=103),
    # a ragged sequence (not a multiple of the 128-row tiles), head dim 96, two dense
    # loops (the second one attends with a previous state)
    "ragged": dict(B=1, N=300, H=8, d=96, F=1024, T=4, T_dense=2, R=70, K=50),
}
# the 8K prefill workload's shapes (B=1, N=8192, H=16, d=128, T=4, r=25%,
# k=10%) with F = 4D; the attention state is compared on 4 seeded heads
# (the first, the last and two drawn), everything else on all of them
_W8 = synth.WORKLOADS["8k"]
CONFIGS["8k"] = dict(B=_W8.B, N=_W8.N, H=_W8.H, d=_W8.d, F=synth.BLOCK_FF_MULT * _W8.D, T=_W8.T,
                     T_dense=_W8.T_dense, R=synth.active_count(_W8), K=synth.key_count(_W8), heads=4)


def _heads(cfg, seed=5):
    """Heads on which the attention state is compared (all unless cfg["heads"])."""
    H = cfg["H"]
    n = cfg.get("heads")
    if not n or n >= H:
        return np.arange(H)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, H - 1), size=n - 2, replace=False).tolist()
    return np.array(sorted({0, H - 1, *mid}))


def _weights(cfg, seed):
    D, F = cfg["H"] * cfg["d"], cfg["F"]
    shapes = ((3 * D, D), (D, D), (F, D), (D, F))
    gains = (1.0, 0.5, 1.0, 0.5)
    return [_rand_bf16(s, seed + i, gains[i] / np.sqrt(s[1])) for i, s in enumerate(shapes)]


def _oracle_chain(cfg, w_bits, h0_bits, T=None):
    B, N, H, d = cfg["B"], cfg["N"], cfg["H"], cfg["d"]
    cache, st = OCache(), empty_state(B, N, H, d)
    hs, sel, states = [h0_bits], {}, {}
    for l in range(1, (cfg["T"] if T is None else T) + 1):
        h_prev = hs[-2] if l >= 2 else None
        h, st, A, S = ob.block_loop(l, w_bits, h_prev, hs[-1], cache, st, cfg["T_dense"], H, d, cfg["R"], cfg["K"])
        hs.append(h)
        sel[l] = (A, S)
        states[l] = st
    return hs, sel, states


class GpuBlock:
    """The block on the GPU, loop by loop, with two alternating H buffers
    (the loop's output overwrites H_{l-2}; only its stale rows are copied)."""

    def __init__(self, cfg, w_dev, h0):
        B, N, H, d, F = (cfg[k] for k in ("B", "N", "H", "d", "F"))
        self.cfg = cfg
        self.w = w_dev
        self.dims = fl.make_dims(B, N, H, d, cfg["R"], cfg["K"], cfg["T"], cfg["T_dense"])
        self.cache = fl.Cache(self.dims)
        self.cache.n_tokens = N
        self.ws = fl.block_workspace_for(self.dims, F)
        self.st = State(B, N, H, d, N)
        self.buf = [h0.clone(), torch.empty((B, N, H * d), dtype=torch.bfloat16, device="cuda")]
        self.cur, self.prev_idx = 0, None
        self.hs = [bits(h0)]

    def state(self):
        return OState(bits(self.st.q_hat), f32(self.st.o), f32(self.st.z), f32(self.st.c))

    def run(self, l, forced=None, qkv=None, key_rank=0):
        cfg = self.cfg
        B, N, H = cfg["B"], cfg["N"], cfg["H"]
        out = 1 - self.cur
        lazy = l > cfg["T_dense"]
        act = torch.empty((B, cfg["R"]), dtype=torch.int32, device="cuda")
        keys = torch.empty((B, H, cfg["K"]), dtype=torch.int32, device="cuda")
        sc = torch.empty((B, N), dtype=torch.float32, device="cuda")
        if forced is not None:
            act.copy_(torch.from_numpy(forced[0]))
            keys.copy_(torch.from_numpy(forced[1]))
        st = self.st
        fl.flashloop_block_loop(self.cache, l, self.w, self.buf[self.cur], self.buf[out], st.q_hat, st.o, st.z, st.c,
                                self.ws, h_prev=self.buf[out] if lazy else None,
                                stale_idx=self.prev_idx if lazy else None,
                                active_idx=act if lazy else None, key_idx=keys if lazy else None,
                                force_selection=forced is not None, key_rank=key_rank, scores=sc if lazy else None,
                                q=None if qkv is None else qkv[0], k=None if qkv is None else qkv[1],
                                v=None if qkv is None else qkv[2])
        torch.cuda.synchronize()
        self.hs.append(bits(self.buf[out]))
        self.cur = out
        if not lazy:
            return None
        self.prev_idx = act
        return act.cpu().numpy(), keys.cpu().numpy(), sc.cpu().numpy()

    def oracle_cache(self, l):
        """The GPU's cache as the oracle's, as loop l finds it."""
        td = self.cfg["T_dense"]
        oc = OCache()
        for t in range(1, min(l - 1, td) + 1):
            k, v = self.cache.dense_layer(t)
            oc.dense_k.append(bits(k))
            oc.dense_v.append(bits(v))
        if l - 1 > td:
            oc.delta_k, oc.delta_v = layers_from_gpu(self.cache, range(td + 1, l), np.arange(self.cfg["B"]))
        return oc


def _bf16_vals(b):
    return oracle.bf16_values(b)


def assert_mostly_close(gpu, orc, atol, rtol, what, max_frac=1e-3, max_rel=5e-3):
    """For a loop whose 4-bit codes come from K/V that each side rounded on its
    own: a code on a rounding boundary may round either way (both correct) and
    move a reconstructed element by a whole quantisation step, so a few
    elements may leave the elementwise tolerance; the share of them and the
    relative Frobenius error stay small."""
    gpu = np.asarray(gpu, np.float64)
    orc = np.asarray(orc, np.float64)
    assert gpu.shape == orc.shape and np.all(np.isfinite(gpu)), what
    err = np.abs(gpu - orc)
    frac = float((err > atol + rtol * np.abs(orc)).mean())
    rel = float(np.linalg.norm(err.ravel()) / np.linalg.norm(orc.ravel()))
    assert frac <= max_frac, f"{what}: {frac:.2e} of the elements outside tolerance"
    assert rel <= max_rel, f"{what}: relative Frobenius error {rel:.2e}"


@pytest.mark.parametrize("name", ["tiny", "wide", "ragged"])
def test_block_chain_independent(name):
    # the dense loops and the first lazy loop, the oracle and the GPU each on
    # their own from the same inputs (the lazy loop's selections are the
    # oracle's, passed in): H of every dense loop and the state after them
    # elementwise, then the first lazy loop's H (mostly close, see above). The
    # state after the lazy loop is compared in the loop-by-loop test.
    cfg = CONFIGS[name]
    D, l2 = cfg["H"] * cfg["d"], cfg["T_dense"] + 1
    w = _weights(cfg, 100)
    h0 = _rand_bf16((cfg["B"], cfg["N"], D), 7)
    hs_o, sel_o, st_o = _oracle_chain(cfg, [bits(t) for t in w], bits(h0), T=l2)
    g = GpuBlock(cfg, [_dev(t) for t in w], _dev(h0))
    for l in range(1, l2 + 1):
        g.run(l, forced=sel_o[l] if l > cfg["T_dense"] else None)
        check = assert_close if l <= cfg["T_dense"] else assert_mostly_close
        check(_bf16_vals(g.hs[l]), _bf16_vals(hs_o[l]), H_ATOL, H_RTOL, f"{name}: H_{l}")
        if l == cfg["T_dense"]:
            o = g.state()
            assert_close(o.o, st_o[l].o, O_ATOL, O_RTOL, f"{name}: O after loop {l}")
            assert_close(o.z, st_o[l].z, Z_ATOL, 0, f"{name}: Z after loop {l}")
            assert_close(o.c, st_o[l].c, C_ATOL, C_RTOL, f"{name}: c after loop {l}")
    assert fl.flashloop_device_status() == 0


@pytest.mark.parametrize("name, key_rank", [("tiny", 0), ("tiny", 1), ("wide", 0), ("ragged", 0), ("8k", 0)])
def test_block_loop_by_loop(name, key_rank):
    # every loop with the GPU's own selections, each part against the oracle
    # started from the GPU's values before that part (the teacher forcing of
    # the workload tests): the projections of the loop's input rows, the
    # lazy step on the GPU's q/k/v, cache and row state, and the MLP on the
    # GPU's attention output
    cfg = CONFIGS[name]
    B, N, H, d, R, K = (cfg[k] for k in ("B", "N", "H", "d", "R", "K"))
    D = H * d
    w = _weights(cfg, 300)
    wb = [bits(t) for t in w]
    h0 = _rand_bf16((B, N, D), 9)
    g = GpuBlock(cfg, [_dev(t) for t in w], _dev(h0))
    qkv = [torch.zeros((B, N, H, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    bi = np.arange(B)[:, None]
    hs = _heads(cfg)
    mask = np.zeros((B, H), bool)
    mask[:, hs] = True
    for l in range(1, cfg["T"] + 1):
        before = g.state()
        oc = g.oracle_cache(l)
        h_prev = g.hs[-2] if l >= 2 else None
        h_cur = g.hs[-1]
        got = g.run(l, qkv=qkv, key_rank=key_rank)
        q_g, k_g, v_g = (bits(t) for t in qkv)
        A = S = None
        if got is not None:
            A, S, scores = got
            sc_o = oracle.token_scores(h_prev, h_cur)
            assert_close(scores, sc_o, 0, 1e-5, f"{name}: change scores of loop {l}")
            A_o = oracle.topk(sc_o, R)
            col = before.c.astype(np.float64) if key_rank == 0 else oracle.key_scores_per_row(before.c, N)
            S_o = oracle.topk(col, K)
            for b in range(B):
                assert_selection(A[b], A_o[b], sc_o[b], f"{name}: active tokens of loop {l}, sequence {b}")
                for h in range(H):
                    assert_selection(S[b, h], S_o[b, h], col[b, h], f"{name}: keys of loop {l}, sequence {b}, head {h}")
        rows = np.tile(np.arange(N), (B, 1)) if A is None else A
        x = h_cur[bi, rows]
        # (1) projections of the loop's input rows
        want = ob.project(x, wb[0])
        gotp = np.concatenate([t[bi, rows].reshape(B, rows.shape[1], D) for t in (q_g, k_g, v_g)], axis=-1)
        assert_gemm(gotp, want, gemm_bound(x, wb[0]), f"{name}: q/k/v of loop {l}", D)
        # (2) the loop's step on the GPU's projections
        if A is None:
            st_o = dense_loop(l, q_g, k_g, v_g, oc, before, bh_mask=mask)
        else:
            # the append against the oracle's own (codes exact except at rounding
            # boundaries), then the attention over the GPU's layers, as in the workload
            # tests: a boundary code that rounded the other way would move a
            # reconstructed element by a whole quantisation step
            _, _, _, _, lk, lv = lazy_loop(l, h_prev, h_cur, q_g, k_g, v_g, oc, before, R, K, A=A, S=S,
                                           bh_mask=mask)
            _check_layers(g.cache, l, lk, lv, oc, k_g, v_g, A, f"{name}: loop {l}")
            og = g.oracle_cache(l + 1)   # the GPU's cache after this loop
            qh, oo, zz, cc, _ = oracle.attention(False, A, A, q_g, before.qhat, before.o, before.z, before.c, S,
                                                 og.rec(l - 1, "k"), og.rec(l - 1, "v"), og.rec(l, "k"),
                                                 og.rec(l, "v"), bh_mask=mask)
            st_o = OState(qh, oo, zz, cc)
        after = g.state()
        assert_close(after.o[:, :, hs], st_o.o[:, :, hs], O_ATOL, O_RTOL, f"{name}: O after loop {l}")
        assert_close(after.z[:, hs], st_o.z[:, hs], Z_ATOL, 0, f"{name}: Z after loop {l}")
        assert_close(after.c[:, hs], st_o.c[:, hs], C_ATOL, C_RTOL, f"{name}: c after loop {l}")
        assert np.array_equal(after.qhat[:, :, hs], st_o.qhat[:, :, hs]), f"{name}: q_hat after loop {l}"
        # (3) the MLP on the GPU's attention output; untouched rows keep H_{l-1}
        a = oracle.round_bf16(after.o[bi, rows].astype(np.float64)).reshape(B, rows.shape[1], D)
        h_rows = ob.mlp(x, a, wb)
        assert_close(_bf16_vals(g.hs[l][bi, rows]), _bf16_vals(h_rows), MLP_ATOL, MLP_RTOL, f"{name}: H_{l} rows")
        if A is not None:
            for b in range(B):
                keep = np.setdiff1d(np.arange(N), A[b])
                assert np.array_equal(g.hs[l][b, keep], h_cur[b, keep]), f"{name}: loop {l} changed inactive rows"
    assert fl.flashloop_device_status() == 0


def _check_layers(cache, l, lk, lv, oc, k_g, v_g, A, what):
    """The loop's K and V delta layers against the oracle's from the same
    inputs: scales bit-exact, codes bit-exact except at rounding boundaries."""
    idx, _, kc, ks, vc, vs = cache.delta_layer(l)
    assert np.array_equal(idx.cpu().numpy(), A), f"{what}: entry tokens"
    B = A.shape[0]
    for name, x_g, lay, codes, scales in (("K", k_g, lk, kc, ks), ("V", v_g, lv, vc, vs)):
        base = oc.dense_k[-1] if name == "K" else oc.dense_v[-1]
        prev = (oc.delta_k if name == "K" else oc.delta_v)[: l - 1 - len(oc.dense_k)]
        rec, _ = oracle.reconstruct(base, prev, want_bf16=False)
        rows = np.stack([rec[b, A[b]] for b in range(B)])
        xb = np.stack([x_g[b, A[b]] for b in range(B)])
        assert_layer(codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16), lay.codes, lay.scales,
                     delta_over_scale(xb, rows, lay.scales), f"{what}: {name} layer")
