"""Per-step parity of the CUDA path against the CPU oracle, through the C ABI,
on seeded inputs at sizes that span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

import oracle
import lazy_sparse_attention_token_b300 as fl
from lazy_sparse_attention_token_b300 import build as flbuild
from gpu_helpers import (C_ATOL, C_RTOL, O_ATOL, O_RTOL, Z_ATOL, State, assert_close, assert_layer,
                         assert_selection, bits, check_slot_map, delta_over_scale, f32, layers_from_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    flbuild.build()
    fl.lib()
    oracle.build()


def gen(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed, scale=1.0):
    return (torch.randn(shape, generator=gen(seed), device="cuda") * scale).to(torch.bfloat16)


# --------------------------------------------------------------------------
# token selection

@pytest.mark.parametrize("B,N,D,R", [(1, 1000, 256, 250), (3, 4097, 2048, 615), (1, 32768, 2048, 4916),
                                     (2, 50, 64, 50), (1, 7, 8, 1), (2, 70000, 64, 9000),
                                     (1, 400000, 8, 40000)])   # cluster segments too long to stage
def test_select_tokens(B, N, D, R):
    hp = randn_bf16((B, N, D), 1)
    drift = torch.rand((B, N, 1), generator=gen(2), device="cuda") ** 4
    hc = (hp.float() + drift * torch.randn((B, N, D), generator=gen(3), device="cuda")).to(torch.bfloat16)
    scores = torch.empty(B, N, device="cuda")
    act = fl.flashloop_select_tokens(hp, hc, R, scores=scores)
    torch.cuda.synchronize()
    sc = oracle.token_scores(bits(hp), bits(hc))
    assert_close(f32(scores), sc, atol=1e-30, rtol=2e-6, what="token scores")
    orc = oracle.topk(sc, R)
    a = act.cpu().numpy()
    for b in range(B):
        assert_selection(a[b], orc[b], sc[b], f"active set b={b}")


def test_select_tokens_ties_go_to_lower_index():
    B, N, D, R = 2, 3000, 64, 1000
    hp = torch.zeros(B, N, D, dtype=torch.bfloat16, device="cuda")
    hc = hp.clone()
    hc[:, :, 0] = 1.0                    # every token changed by exactly the same amount
    hc[1, 2500:, 0] = 2.0                # sequence 1: the last 500 changed more
    act = fl.flashloop_select_tokens(hp, hc, R, scores=torch.empty(B, N, device="cuda")).cpu().numpy()
    assert np.array_equal(act[0], np.arange(R))
    assert np.array_equal(act[1], np.concatenate([np.arange(500), np.arange(2500, 3000)]))


@pytest.mark.parametrize("B,H,N,K", [(1, 4, 1024, 103), (2, 16, 8192, 820), (1, 3, 129, 129), (4, 2, 5, 1),
                                     (1, 16, 32768, 3277),
                                     (2, 64, 3001, 300),        # one CTA per row, staged, ragged tail
                                     (1, 128, 50000, 5000)])    # one CTA per row, row too long to stage
def test_select_keys_exact(B, H, N, K):
    c = torch.randn(B, H, N, generator=gen(4), device="cuda").abs() * 3
    c = torch.where(torch.rand(B, H, N, generator=gen(5), device="cuda") < 0.2, torch.round(c), c)   # ties
    c[..., : min(N, 3)] = -0.0
    idx = fl.flashloop_select_keys(c, K).cpu().numpy()
    orc = oracle.topk(f32(c).astype(np.float64), K)
    assert np.array_equal(idx, orc)


# --------------------------------------------------------------------------
# gather

@pytest.mark.parametrize("row_shape,dtype", [((8,), torch.bfloat16), ((16, 128), torch.bfloat16),
                                             ((16, 128), torch.float32), ((3,), torch.float32)])
def test_gather_is_exact(row_shape, dtype):
    B, N, R = 3, 777, 130
    src = torch.randn((B, N) + row_shape, generator=gen(6), device="cuda").to(dtype)
    idx = torch.stack([torch.sort(torch.randperm(N, device="cuda")[:R]).values for _ in range(B)]).to(torch.int32)
    if src[0, 0].numel() * src.element_size() % 16:
        with pytest.raises(fl.FlashLoopError):
            fl.flashloop_gather(src, idx)
        return
    out = fl.flashloop_gather(src, idx)
    ref = torch.stack([src[b, idx[b].long()] for b in range(B)])
    assert torch.equal(out, ref)


def test_gather_skips_rows_outside_the_sequence():
    B, N, R = 2, 100, 5
    src = torch.randn((B, N, 8), generator=gen(7), device="cuda")
    idx = torch.tensor([[0, 3, 100, 50, 99], [-1, 2, 4, 1 << 30, 7]], dtype=torch.int32, device="cuda")
    out = torch.full((B, R, 8), 7.0, device="cuda")
    fl.flashloop_gather(src, idx, dst=out)
    torch.cuda.synchronize()
    for b in range(B):
        for r in range(R):
            i = int(idx[b, r])
            want = src[b, i] if 0 <= i < N else torch.full((8,), 7.0, device="cuda")
            assert torch.equal(out[b, r], want), (b, r)


# --------------------------------------------------------------------------
# base + int4 delta cache

@pytest.mark.parametrize("d", [64, 96, 128])
def test_delta_append_and_reconstruct_bit_exact(d):
    B, N, H, T = 2, 300, 3, 4
    R = 101
    dm = fl.make_dims(B, N, H, d, R, 77, T, 1, R_cap=R + 1)
    cache = fl.Cache(dm)
    cache.n_tokens = N
    xs_k = [randn_bf16((B, N, H, d), 10)]
    xs_v = [randn_bf16((B, N, H, d), 11)]
    fl.flashloop_kv_dense_store(cache, 1, xs_k[0], xs_v[0])
    bsel = [0, 1]
    base_k, base_v = (bits(t[bsel]) for t in cache.dense_layer(1))
    for l in range(2, T + 1):
        scale = 0.5 ** l
        k_l = (xs_k[-1].float() + scale * torch.randn(xs_k[-1].shape, generator=gen(20 + l), device="cuda")).to(torch.bfloat16)
        v_l = (xs_v[-1].float() + scale * torch.randn(xs_v[-1].shape, generator=gen(40 + l), device="cuda")).to(torch.bfloat16)
        act = torch.stack([torch.sort(torch.randperm(N, generator=gen(60 + l + b), device="cuda")[:R]).values
                           for b in range(B)]).to(torch.int32)
        prev_k, prev_v = layers_from_gpu(cache, range(2, l), bsel)
        fl.flashloop_kv_delta_append(cache, l, k_l, v_l, act)
        torch.cuda.synchronize()
        check_slot_map(cache, l, N)
        idx, slot, kc, ks, vc, vs = cache.delta_layer(l)
        a = act.cpu().numpy()
        assert np.array_equal(idx.cpu().numpy(), a)
        for x_l, base, prev, codes, scales, name in ((k_l, base_k, prev_k, kc, ks, "K"), (v_l, base_v, prev_v, vc, vs, "V")):
            orc = oracle.kv_delta_append(bits(x_l), base, prev, a)
            g_codes, g_scales = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
            if not (np.array_equal(g_codes, orc.codes) and np.array_equal(g_scales, orc.scales)):
                rec, _ = oracle.reconstruct(base, prev, want_bf16=False)
                rows = np.stack([rec[b, a[b]] for b in range(B)])
                xb = np.stack([bits(x_l)[b, a[b]] for b in range(B)])
                dos = delta_over_scale(xb, rows, orc.scales)
                assert_layer(g_codes, g_scales, orc.codes, orc.scales, dos, f"{name} layer {l}")
        xs_k.append(k_l)
        xs_v.append(v_l)
        # reconstruct-gather of a key list, old and new loop, bit for bit
        K = 77
        key_idx = torch.stack([torch.stack([torch.sort(torch.randperm(N, generator=gen(80 + l + 7 * b + h), device="cuda")[:K]).values
                                            for h in range(H)]) for b in range(B)]).to(torch.int32)
        ko, vo, kn, vn = fl.flashloop_reconstruct_keys(cache, l, key_idx)
        lk, lv = layers_from_gpu(cache, range(2, l + 1), bsel)
        S = key_idx.cpu().numpy()
        for got, base, lays, which in ((ko, base_k, lk[:-1], "k_old"), (kn, base_k, lk, "k_new"),
                                       (vo, base_v, lv[:-1], "v_old"), (vn, base_v, lv, "v_new")):
            _, ref = oracle.reconstruct(base, lays, want_f32=False)
            exp = np.stack([np.stack([ref[b, S[b, h], h] for h in range(H)]) for b in range(B)])
            assert np.array_equal(bits(got), exp), f"{which} loop {l}"


def test_decode_style_append_at_offset():
    B, N, H, d = 2, 200, 2, 64
    dm = fl.make_dims(B, N + 1, H, d, 50, 20, 2, 1, R_cap=51)
    cache = fl.Cache(dm)
    cache.n_tokens = N
    k1, v1 = randn_bf16((B, N, H, d), 90), randn_bf16((B, N, H, d), 91)
    fl.flashloop_kv_dense_store(cache, 1, k1, v1)
    act = torch.stack([torch.arange(0, 200, 4, device="cuda")] * B).to(torch.int32)
    k2 = (k1.float() * 1.01).to(torch.bfloat16)
    fl.flashloop_kv_delta_append(cache, 2, k2, k2, act)
    # one more token at position N, appended after the 50 context entries
    kn, vn = randn_bf16((B, 1, H, d), 92), randn_bf16((B, 1, H, d), 93)
    fl.flashloop_kv_dense_store(cache, 1, kn, vn, pos0=N)
    tok = torch.full((B, 1), N, dtype=torch.int32, device="cuda")
    kn2 = (kn.float() + 0.25).to(torch.bfloat16)
    fl.flashloop_kv_delta_append(cache, 2, kn2, kn2, tok, at=50, rows_are_tokens=False)
    torch.cuda.synchronize()
    check_slot_map(cache, 2, N + 1)
    idx, slot, kc, ks, vc, vs = cache.delta_layer(2)
    assert idx.shape[1] == 51 and (idx[:, 50] == N).all()
    base = bits(cache.dense_layer(1)[0])
    x = np.zeros((B, N + 1, H, d), np.uint16)
    x[:, N] = bits(kn2)[:, 0]
    orc = oracle.kv_delta_append(x, base, [], np.full((B, 1), N, np.int32))
    assert np.array_equal(kc[:, 50:].cpu().numpy(), orc.codes)
    assert np.array_equal(ks[:, 50:].cpu().numpy().view(np.uint16), orc.scales)
    with pytest.raises(fl.FlashLoopError):     # the layer is full
        fl.flashloop_kv_delta_append(cache, 2, kn2, kn2, tok, at=51, rows_are_tokens=False)


def test_refused_append_leaves_slot_map_and_count():
    """A delta append refused on the host (here: a token-indexed append while
    the cache counts no tokens) touches nothing: the layer's slot map, entries
    and count stay those of the previous append."""
    B, N, H, d = 2, 300, 2, 64
    dm = fl.make_dims(B, N, H, d, 40, 20, 2, 1, R_cap=40)
    cache = fl.Cache(dm)
    cache.n_tokens = N
    k1, v1 = randn_bf16((B, N, H, d), 94), randn_bf16((B, N, H, d), 95)
    fl.flashloop_kv_dense_store(cache, 1, k1, v1)
    act = torch.stack([torch.arange(3, 300, 7, device="cuda")[:40]] * B).to(torch.int32)
    k2 = (k1.float() * 1.02).to(torch.bfloat16)
    fl.flashloop_kv_delta_append(cache, 2, k2, k2, act)
    torch.cuda.synchronize()
    idx0, slot0, kc0, *_ = (t.clone() for t in cache.delta_layer(2))
    cache.n_tokens = 0
    with pytest.raises(fl.FlashLoopError):
        fl.flashloop_kv_delta_append(cache, 2, k2, k2, act[:, :10].contiguous())
    torch.cuda.synchronize()
    cache.n_tokens = N
    assert cache.c.count[0] == 40
    idx1, slot1, kc1, *_ = cache.delta_layer(2)
    assert torch.equal(slot0, slot1) and torch.equal(idx0, idx1) and torch.equal(kc0, kc1)
    check_slot_map(cache, 2, N)


# --------------------------------------------------------------------------
# attention

def _setup_first(B, N, H, d, seed):
    dm = fl.make_dims(B, N, H, d, max(1, N // 4), max(1, N // 10), 2, 1, R_cap=N)
    cache = fl.Cache(dm)
    cache.n_tokens = N
    q, k, v = (randn_bf16((B, N, H, d), seed + i) for i in range(3))
    st = State(B, N, H, d, N)
    fl.flashloop_kv_dense_store(cache, 1, k, v)
    fl.flashloop_lazy_attention(cache, fl.FIRST_DENSE, 1, q, st.q_hat, st.o, st.z, st.c)
    torch.cuda.synchronize()
    assert fl.flashloop_device_status() == 0
    return dm, cache, st, q, k, v


@pytest.mark.parametrize("B,N,H,d", [(1, 300, 2, 64), (2, 257, 3, 96), (1, 400, 2, 128), (1, 128, 1, 128),
                                     (1, 1, 1, 64)])
def test_first_dense_attention(B, N, H, d):
    dm, cache, st, q, k, v = _setup_first(B, N, H, d, 100)
    rows = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    S = np.tile(np.arange(N, dtype=np.int32), (B, H, 1))
    z0 = np.zeros((B, H, N), np.float32)
    qh, o, z, c, _ = oracle.attention(True, rows, rows, bits(q), np.zeros((B, N, H, d), np.uint16),
                                      np.zeros((B, N, H, d), np.float32), z0, z0, S, None, None, bits(k), bits(v))
    assert_close(f32(st.o), o, O_ATOL, O_RTOL, "O")
    assert_close(f32(st.z), z, Z_ATOL, 0, "Z")
    assert_close(f32(st.c), c, C_ATOL, C_RTOL, "c")
    assert np.array_equal(bits(st.q_hat), qh)
    np.testing.assert_allclose(f32(st.c).sum(-1), N, rtol=1e-4)


@pytest.mark.parametrize("B,N,H,d,R,K", [(1, 300, 2, 64, 77, 41), (2, 520, 2, 96, 130, 200), (1, 700, 3, 128, 300, 129),
                                         (1, 256, 2, 128, 256, 256), (1, 300, 1, 128, 5, 300),
                                         # more (row tile, head) items than SMs: the items past the last full
                                         # wave are split over clusters by key tiles (some parts get none)
                                         (1, 2048, 16, 128, 1280, 600), (2, 1024, 16, 64, 640, 90)])
def test_lazy_attention(B, N, H, d, R, K):
    dm, cache, st, q1, k1, v1 = _setup_first(B, N, H, d, 200)
    dm2 = fl.make_dims(B, N, H, d, R, K, 2, 1, R_cap=R)
    cache2 = fl.Cache(dm2)
    cache2.n_tokens = N
    fl.flashloop_kv_dense_store(cache2, 1, k1, v1)
    q2 = (q1.float() + 0.3 * torch.randn(q1.shape, generator=gen(210), device="cuda")).to(torch.bfloat16)
    k2 = (k1.float() + 0.3 * torch.randn(k1.shape, generator=gen(211), device="cuda")).to(torch.bfloat16)
    v2 = (v1.float() + 0.3 * torch.randn(v1.shape, generator=gen(212), device="cuda")).to(torch.bfloat16)
    A = torch.stack([torch.sort(torch.randperm(N, generator=gen(220 + b), device="cuda")[:R]).values
                     for b in range(B)]).to(torch.int32)
    fl.flashloop_kv_delta_append(cache2, 2, k2, v2, A)
    S = fl.flashloop_select_keys(st.c, K)
    before = (bits(st.q_hat), f32(st.o), f32(st.z), f32(st.c))
    ws = fl.workspace_for(dm2)
    fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S, workspace=ws)
    torch.cuda.synchronize()
    assert fl.flashloop_device_status() == 0
    base_k, base_v = (bits(t) for t in cache2.dense_layer(1))
    lk, lv = layers_from_gpu(cache2, [2], list(range(B)))
    kn = oracle.reconstruct(base_k, lk, want_f32=False)[1]
    vn = oracle.reconstruct(base_v, lv, want_f32=False)[1]
    a, s = A.cpu().numpy(), S.cpu().numpy()
    qh, o, z, c, _ = oracle.attention(False, a, a, bits(q2), *before, s, base_k, base_v, kn, vn)
    assert_close(f32(st.o), o, O_ATOL, O_RTOL, "O")
    assert_close(f32(st.z), z, Z_ATOL, 0, "Z")
    assert_close(f32(st.c), c, C_ATOL, C_RTOL, "c")
    assert np.array_equal(bits(st.q_hat), qh)
    inactive = np.ones(N, bool)
    inactive[a[0]] = False
    assert np.array_equal(f32(st.o)[0, inactive], before[1][0, inactive])
    np.testing.assert_allclose(f32(st.c).sum(-1), N, rtol=1e-4)


def _lazy_case(seed, B=1, N=520, H=2, d=128, R=200, K=150):
    """A lazy attention call (by default small: two row tiles, two key tiles) and its inputs."""
    dm, cache, st, q1, k1, v1 = _setup_first(B, N, H, d, seed)
    dm2 = fl.make_dims(B, N, H, d, R, K, 2, 1, R_cap=R)
    cache2 = fl.Cache(dm2)
    cache2.n_tokens = N
    fl.flashloop_kv_dense_store(cache2, 1, k1, v1)
    q2, k2, v2 = ((x.float() + 0.3 * torch.randn(x.shape, generator=gen(seed + 10 + i), device="cuda")).to(torch.bfloat16)
                  for i, x in enumerate((q1, k1, v1)))
    A = torch.stack([torch.sort(torch.randperm(N, generator=gen(seed + 20 + b), device="cuda")[:R]).values
                     for b in range(B)]).to(torch.int32)
    fl.flashloop_kv_delta_append(cache2, 2, k2, v2, A)
    S = fl.flashloop_select_keys(st.c, K)
    torch.cuda.synchronize()
    return dm2, cache2, st, q2, A, S


def test_bounded_wait_gives_up_and_the_context_recovers():
    """Failure path of the attention kernel's bounded waits, made to run out on
    purpose by setting the limit to zero (a wait then gives up unless its phase
    has already completed; nothing is withheld, and every copy and MMA issued
    before the give-up still lands). The launch completes, the device status
    reports the failure with one of the kernel's wait codes, and once the limit
    is restored the same call on fresh state matches the oracle."""
    dm2, cache2, st, q2, A, S = _lazy_case(500)
    ws = fl.workspace_for(dm2)
    assert fl.flashloop_device_status() == 0
    fl.flashloop_set_wait_limit_ns(0)
    try:
        fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S,
                                    workspace=ws)
        torch.cuda.synchronize()                    # the launch returned
        word = fl.flashloop_device_status()
    finally:
        fl.flashloop_set_wait_limit_ns(fl.flashloop.WAIT_LIMIT_DEFAULT_NS)
    assert word in (1, 2, 5, 6, 7, 8, 9, 10, 11, 12, 13), word
    assert fl.flashloop_device_status() == 0        # read and cleared
    # a fresh state through the same call, with the default limit
    dm2, cache2, st, q2, A, S = _lazy_case(500)
    before = (bits(st.q_hat), f32(st.o), f32(st.z), f32(st.c))
    fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S,
                                workspace=fl.workspace_for(dm2))
    torch.cuda.synchronize()
    assert fl.flashloop_device_status() == 0
    base_k, base_v = (bits(t) for t in cache2.dense_layer(1))
    lk, lv = layers_from_gpu(cache2, [2], [0])
    kn = oracle.reconstruct(base_k, lk, want_f32=False)[1]
    vn = oracle.reconstruct(base_v, lv, want_f32=False)[1]
    a, s_ = A.cpu().numpy(), S.cpu().numpy()
    qh, o, z, c, _ = oracle.attention(False, a, a, bits(q2), *before, s_, base_k, base_v, kn, vn)
    assert_close(f32(st.o), o, O_ATOL, O_RTOL, "O after recovery")
    assert_close(f32(st.c), c, C_ATOL, C_RTOL, "c after recovery")


def test_bounded_wait_gives_up_on_split_items():
    """The same failure path with more (row tile, head) items than SMs, so that the
    items past the last full wave run split over clusters, whose CTAs also wait on
    one another (bounded, like every other wait) and meet at two cluster barriers
    that every CTA reaches. The launch completes and reports a wait code; with the
    limit restored the same call on fresh state matches the oracle."""
    case = dict(B=1, N=2048, H=16, d=128, R=1280, K=600)
    dm2, cache2, st, q2, A, S = _lazy_case(510, **case)
    ws = fl.workspace_for(dm2)
    assert fl.flashloop_device_status() == 0
    fl.flashloop_set_wait_limit_ns(0)
    try:
        fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S,
                                    workspace=ws)
        torch.cuda.synchronize()                    # the launches returned
        word = fl.flashloop_device_status()
    finally:
        fl.flashloop_set_wait_limit_ns(fl.flashloop.WAIT_LIMIT_DEFAULT_NS)
    assert word in (1, 2, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15), word
    assert fl.flashloop_device_status() == 0
    dm2, cache2, st, q2, A, S = _lazy_case(510, **case)
    before = (bits(st.q_hat), f32(st.o), f32(st.z), f32(st.c))
    fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S,
                                workspace=fl.workspace_for(dm2))
    torch.cuda.synchronize()
    assert fl.flashloop_device_status() == 0
    base_k, base_v = (bits(t) for t in cache2.dense_layer(1))
    lk, lv = layers_from_gpu(cache2, [2], [0])
    kn = oracle.reconstruct(base_k, lk, want_f32=False)[1]
    vn = oracle.reconstruct(base_v, lv, want_f32=False)[1]
    a, s_ = A.cpu().numpy(), S.cpu().numpy()
    qh, o, z, c, _ = oracle.attention(False, a, a, bits(q2), *before, s_, base_k, base_v, kn, vn)
    assert_close(f32(st.o), o, O_ATOL, O_RTOL, "O after recovery")
    assert_close(f32(st.z), z, Z_ATOL, 0, "Z after recovery")
    assert_close(f32(st.c), c, C_ATOL, C_RTOL, "c after recovery")


def test_lazy_full_sets_match_softmax_of_new_loop():
    """A = all rows, S = all keys: the lazy step is softmax attention over the
    loop-2 reconstruction (compared with torch's attention in float64)."""
    B, N, H, d = 1, 384, 2, 128
    dm, cache, st, q1, k1, v1 = _setup_first(B, N, H, d, 300)
    dm2 = fl.make_dims(B, N, H, d, N, N, 2, 1, R_cap=N)
    cache2 = fl.Cache(dm2)
    cache2.n_tokens = N
    fl.flashloop_kv_dense_store(cache2, 1, k1, v1)
    q2, k2, v2 = (randn_bf16((B, N, H, d), 310 + i) for i in range(3))
    A = torch.arange(N, dtype=torch.int32, device="cuda")[None]
    S = torch.arange(N, dtype=torch.int32, device="cuda").expand(B, H, N).contiguous()
    fl.flashloop_kv_delta_append(cache2, 2, k2, v2, A)
    fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S,
                                workspace=fl.workspace_for(dm2))
    _, _, kn, vn = fl.flashloop_reconstruct_keys(cache2, 2, S)
    torch.cuda.synchronize()
    qd = q2.double().permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kn.double(), vn.double(), is_causal=True)
    assert_close(f32(st.o), ref.permute(0, 2, 1, 3).cpu().numpy(), O_ATOL, O_RTOL, "O vs softmax")
    lse = torch.logsumexp((qd @ kn.double().transpose(-1, -2) / d ** 0.5).masked_fill(
        ~torch.ones(N, N, dtype=torch.bool, device="cuda").tril(), float("-inf")), -1)
    assert_close(f32(st.z), lse.cpu().numpy(), Z_ATOL, 0, "Z vs logsumexp")


def test_rows_before_every_key_keep_state():
    B, N, H, d = 1, 512, 2, 64
    dm, cache, st, q1, k1, v1 = _setup_first(B, N, H, d, 400)
    dm2 = fl.make_dims(B, N, H, d, 256, 64, 2, 1, R_cap=256)
    cache2 = fl.Cache(dm2)
    cache2.n_tokens = N
    fl.flashloop_kv_dense_store(cache2, 1, k1, v1)
    A = torch.arange(0, N, 2, dtype=torch.int32, device="cuda")[None]
    fl.flashloop_kv_delta_append(cache2, 2, k1, v1, A)
    S = torch.arange(300, 364, dtype=torch.int32, device="cuda").expand(B, H, 64).contiguous()
    before = (bits(st.q_hat), f32(st.o), f32(st.z))
    q2 = randn_bf16((B, N, H, d), 410)
    fl.flashloop_lazy_attention(cache2, fl.LAZY, 2, q2, st.q_hat, st.o, st.z, st.c, row_pos=A, key_idx=S,
                                workspace=fl.workspace_for(dm2))
    torch.cuda.synchronize()
    early = np.arange(0, 300)
    assert np.array_equal(bits(st.q_hat)[0, early], before[0][0, early])
    assert np.array_equal(f32(st.o)[0, early], before[1][0, early])
    assert np.array_equal(f32(st.z)[0][:, early], before[2][0][:, early])
    assert not np.array_equal(f32(st.o)[0, 300:], before[1][0, 300:])
