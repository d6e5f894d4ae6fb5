"""Cache variants (beyond the main setting; the rit.work page: "a compressed
base plus a sequence of compressed deltas", 4-bit deltas in the main
experiments, quality dropping at lower widths): delta codes of 3 and 2 bits
and an int8 base, through the C ABI, against the oracle on the same inputs.
Codes and scales bit-exact except where a quotient lies within 1e-3 of a
rounding boundary; attention state within the usual tolerances."""
import numpy as np
import pytest
import torch

import oracle
import synth
import lazy_sparse_attention_token_b300 as fl
from lazy_sparse_attention_token_b300 import build as flbuild
from gpu_helpers import (C_ATOL, C_RTOL, CODE_BOUNDARY, O_ATOL, O_RTOL, Z_ATOL, State, assert_close, bits, f32,
                         check_slot_map)

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


def unpack_codes(codes, code_bits, d):
    """[..., d*bits/8] u8 rows -> [..., d] int codes (little-endian bit strings)."""
    c = np.asarray(codes, np.uint8)
    bitsarr = np.unpackbits(c, axis=-1, bitorder="little")
    bitsarr = bitsarr.reshape(c.shape[:-1] + (d, code_bits)).astype(np.int64)
    v = (bitsarr * (1 << np.arange(code_bits))).sum(-1)
    return np.where(v >= (1 << (code_bits - 1)), v - (1 << code_bits), v)


def assert_codes(g_codes, g_scales, o_codes, o_scales, quotient, code_bits, d, what):
    """Scales bit-exact; codes exact except within CODE_BOUNDARY of n + 1/2."""
    g_scales = np.asarray(g_scales).view(np.uint16)
    assert np.array_equal(g_scales, np.asarray(o_scales).view(np.uint16)), f"{what}: scales differ"
    if np.array_equal(g_codes, o_codes):
        return
    ge, oe = unpack_codes(g_codes, code_bits, d), unpack_codes(o_codes, code_bits, d)
    frac = np.abs(quotient - np.floor(quotient) - 0.5)
    bad = (ge != oe) & (frac >= CODE_BOUNDARY)
    assert not bad.any(), f"{what}: {int(bad.sum())} codes differ away from a rounding boundary"


def f32_of(bits16):
    return (np.asarray(bits16, np.uint32) << 16).view(np.float32)


def gpu_base(cache, bsel, hsel=None):
    """The base the lazy loops read, as the oracle takes it: the bf16 base layer
    or the int8 base (CompressedBase)."""
    i8 = cache.base_int8()
    td = cache.dims.T_dense
    N = cache.dims.N_cap
    sl = (lambda a: a[bsel]) if hsel is None else (lambda a: a[bsel][:, :, hsel])
    if i8 is None:
        kb, vb = cache.dense_layer(td)
        return bits(sl(kb)), bits(sl(vb))
    kc, ks, vc, vs = (sl(t).cpu().numpy() for t in i8)
    return (oracle.CompressedBase(kc, ks.view(np.uint16)), oracle.CompressedBase(vc, vs.view(np.uint16)))


def layers(cache, loops, bsel, hsel=None):
    out_k, out_v = [], []
    for l in loops:
        idx, slot, kc, ks, vc, vs = cache.delta_layer(l)
        sl = (lambda a: a[bsel]) if hsel is None else (lambda a: a[bsel][:, :, hsel])
        out_k.append(oracle.DeltaLayer(idx[bsel].cpu().numpy(), sl(kc).cpu().numpy(), sl(ks).cpu().numpy().view(np.uint16)))
        out_v.append(oracle.DeltaLayer(idx[bsel].cpu().numpy(), sl(vc).cpu().numpy(), sl(vs).cpu().numpy().view(np.uint16)))
    return out_k, out_v


def check_base(cache, k1, v1, what):
    """The int8 base against the oracle's quantiser of the stored bf16 layer."""
    i8 = cache.base_int8()
    if i8 is None:
        return
    d = cache.dims.d
    for x, codes, scales, name in ((k1, i8[0], i8[1], "K"), (v1, i8[2], i8[3], "V")):
        n = x.shape[1]
        ref = oracle.quantize_base(bits(x))
        g_codes = codes[:, :n].cpu().numpy()
        g_scales = scales[:, :n].cpu().numpy().view(np.uint16)
        assert np.array_equal(g_scales, ref.scales), f"{what} {name} base scales"
        if not np.array_equal(g_codes, ref.codes):
            s = np.repeat(ref.scales.view(np.float16).astype(np.float32), 32, -1)
            qt = np.where(s > 0, f32_of(bits(x)) / np.where(s > 0, s, 1), 0)
            frac = np.abs(qt - np.floor(qt) - 0.5)
            assert not ((g_codes != ref.codes) & (frac >= CODE_BOUNDARY)).any(), f"{what} {name} base codes"


def check_append(cache, l, x_l, base, prev, A, bsel, name, code_bits, d, entry0=0):
    idx, slot, kc, ks, vc, vs = cache.delta_layer(l)
    codes, scales = (kc, ks) if name == "K" else (vc, vs)
    g_codes = codes[bsel][:, entry0:].cpu().numpy()
    g_scales = scales[bsel][:, entry0:].cpu().numpy().view(np.uint16)
    orc = oracle.kv_delta_append(x_l, base, prev, A, code_bits=code_bits)
    rec, _ = oracle.reconstruct(base, prev, want_bf16=False, code_bits=code_bits)
    rows = np.stack([rec[i, A[i]] for i in range(len(bsel))])
    xb = np.stack([f32_of(x_l[i, A[i]]) for i in range(len(bsel))])
    s = np.repeat(orc.scales.view(np.float16).astype(np.float32), 32, -1)
    qt = np.where(s > 0, (xb - rows).astype(np.float32) / np.where(s > 0, s, 1), 0)
    assert_codes(g_codes, g_scales, orc.codes, orc.scales, qt, code_bits, d, f"{name} layer {l}")


@pytest.mark.parametrize("d,code_bits,base_bits", [(128, 3, 16), (96, 2, 16), (64, 3, 8), (128, 4, 8), (96, 2, 8),
                                                   (64, 2, 16), (128, 2, 8)])
def test_variant_append_and_reconstruct(d, code_bits, base_bits):
    B, N, H, T, R, K = 2, 300, 3, 4, 101, 77
    dm = fl.make_dims(B, N, H, d, R, K, T, 1, R_cap=R, delta_bits=code_bits, base_bits=base_bits)
    cache = fl.Cache(dm)
    cache.n_tokens = N
    k1, v1 = randn_bf16((B, N, H, d), 10, 2.0), randn_bf16((B, N, H, d), 11, 2.0)
    fl.flashloop_kv_dense_store(cache, 1, k1, v1)
    torch.cuda.synchronize()
    check_base(cache, k1, v1, "store")
    bsel = [0, 1]
    base_k, base_v = gpu_base(cache, bsel)
    ks_, vs_ = k1, v1
    for l in range(2, T + 1):
        k_l = (ks_.float() + 0.5 ** l * torch.randn(ks_.shape, generator=gen(20 + l), device="cuda")).to(torch.bfloat16)
        v_l = (vs_.float() + 0.5 ** l * torch.randn(vs_.shape, generator=gen(40 + l), device="cuda")).to(torch.bfloat16)
        act = torch.stack([torch.sort(torch.randperm(N, generator=gen(60 + l + b), device="cuda")[:R]).values
                           for b in range(B)]).to(torch.int32)
        prev_k, prev_v = layers(cache, range(2, l), bsel)
        fl.flashloop_kv_delta_append(cache, l, k_l, v_l, act)
        torch.cuda.synchronize()
        check_slot_map(cache, l, N)
        A = act.cpu().numpy()
        check_append(cache, l, bits(k_l), base_k, prev_k, A, bsel, "K", code_bits, d)
        check_append(cache, l, bits(v_l), base_v, prev_v, A, bsel, "V", code_bits, d)
        ks_, vs_ = k_l, v_l
        key_idx = torch.stack([torch.stack([torch.sort(torch.randperm(N, generator=gen(80 + l + 7 * b + h),
                                                                      device="cuda")[:K]).values
                                            for h in range(H)]) for b in range(B)]).to(torch.int32)
        ko, vo, kn, vn = fl.flashloop_reconstruct_keys(cache, l, key_idx)
        lk, lv = layers(cache, range(2, l + 1), bsel)
        S = key_idx.cpu().numpy()
        for got, base, lays, which in ((ko, base_k, lk[:-1], "k_old"), (kn, base_k, lk, "k_new"),
                                       (vo, base_v, lv[:-1], "v_old"), (vn, base_v, lv, "v_new")):
            _, ref = oracle.reconstruct(base, lays, want_f32=False, code_bits=code_bits)
            exp = np.stack([np.stack([ref[b, S[b, h], h] for h in range(H)]) for b in range(B)])
            assert np.array_equal(bits(got), exp), f"{which} loop {l}"


@pytest.mark.parametrize("code_bits,base_bits", [(3, 8), (2, 16)])
def test_variant_tiny_workload_chain(code_bits, base_bits):
    """The tiny workload through flashloop_loop_step with a narrow or compressed
    cache, every loop compared with the oracle on every head (teacher forcing),
    then one decode token through every loop."""
    w = synth.WORKLOADS["tiny"]
    R, K = synth.active_count(w), synth.key_count(w, w.N + 1)
    dm = fl.make_dims(w.B, w.N + 1, w.H, w.d, R, K, w.T, w.T_dense, R_cap=R + 1, delta_bits=code_bits,
                      base_bits=base_bits)
    cache = fl.Cache(dm)
    cache.n_tokens = w.N
    ws = fl.workspace_for(dm)
    st = State(w.B, w.N, w.H, w.d, w.N)
    act = torch.empty(w.B, R, dtype=torch.int32, device="cuda")
    keys = torch.empty(w.B, w.H, K, dtype=torch.int32, device="cuda")
    hs = list(range(w.H))
    prev = None
    for x in synth.prefill_loops(w, device="cuda"):
        l = x["loop"]
        before = st.snapshot([0], hs)
        prev_k, prev_v = layers(cache, range(2, l), [0]) if l > 1 else ([], [])
        fl.flashloop_loop_step(cache, l, x["Q"], x["K"], x["V"], st.q_hat, st.o, st.z, st.c, ws, h_prev=prev,
                               h_cur=x["H"], active_idx=act, key_idx=keys)
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        if l == 1:
            check_base(cache, x["K"], x["V"], "loop 1")
        else:
            A, S = act.cpu().numpy(), keys.cpu().numpy()
            base_k, base_v = gpu_base(cache, [0])
            base_k = base_k if isinstance(base_k, oracle.CompressedBase) else base_k[:, :w.N]
            base_v = base_v if isinstance(base_v, oracle.CompressedBase) else base_v[:, :w.N]
            if isinstance(base_k, oracle.CompressedBase):
                base_k = oracle.CompressedBase(base_k.codes[:, :w.N], base_k.scales[:, :w.N])
                base_v = oracle.CompressedBase(base_v.codes[:, :w.N], base_v.scales[:, :w.N])
            check_append(cache, l, bits(x["K"]), base_k, prev_k, A, [0], "K", code_bits, w.d)
            check_append(cache, l, bits(x["V"]), base_v, prev_v, A, [0], "V", code_bits, w.d)
            lk, lv = layers(cache, range(2, l + 1), [0])
            ko = oracle.reconstruct(base_k, lk[:-1], want_f32=False, code_bits=code_bits)[1]
            vo = oracle.reconstruct(base_v, lv[:-1], want_f32=False, code_bits=code_bits)[1]
            kn = oracle.reconstruct(base_k, lk, want_f32=False, code_bits=code_bits)[1]
            vn = oracle.reconstruct(base_v, lv, want_f32=False, code_bits=code_bits)[1]
            qh, o, z, c, _ = oracle.attention(False, A, A, bits(x["Q"]), *before, S, ko, vo, kn, vn)
            after = st.snapshot([0], hs)
            assert_close(after[1], o, O_ATOL, O_RTOL, f"loop {l} O")
            assert_close(after[2], z, Z_ATOL, 0, f"loop {l} Z")
            assert_close(after[3], c, C_ATOL, C_RTOL, f"loop {l} c")
        prev = x["H"]
    # one decode token at key position N through every loop
    N = w.N
    cache.n_tokens = N + 1
    dst = State(w.B, 1, w.H, w.d, N + 1)
    dkeys = torch.empty(w.B, w.H, K, dtype=torch.int32, device="cuda")
    pos, slot = np.full((1, 1), N, np.int32), np.zeros((1, 1), np.int32)
    for t in synth.decode_token_loops(w, device="cuda"):
        l = t["loop"]
        before = dst.snapshot([0], hs)
        if l > w.T_dense:
            prev_k, prev_v = layers(cache, range(2, l), [0])
            entry0 = cache.c.count[l - w.T_dense - 1]
        fl.flashloop_loop_step(cache, l, t["q"], t["k"], t["v"], dst.q_hat, dst.o, dst.z, dst.c, ws, key_idx=dkeys,
                               decode=True)
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        q = bits(t["q"])
        if l <= w.T_dense:
            kn, vn = (bits(y[:, :N + 1]) for y in cache.dense_layer(l))
            S = np.tile(np.arange(N + 1, dtype=np.int32), (1, w.H, 1))
            qh, o, z, c, _ = oracle.attention(True, pos, slot, q, *before, S, None, None, kn, vn)
            if base_bits == 8:   # the new token's row of the int8 base
                i8 = cache.base_int8()
                ref = oracle.quantize_base(bits(t["k"]))
                assert np.array_equal(i8[1][:, N:N + 1].cpu().numpy().view(np.uint16), ref.scales)
        else:
            S = dkeys.cpu().numpy()
            assert np.array_equal(S, oracle.topk(before[3].astype(np.float64), K))
            base_k, base_v = gpu_base(cache, [0])
            xk = np.zeros((1, N + 1, w.H, w.d), np.uint16)
            xk[:, N] = bits(t["k"])[:, 0]
            xv = np.zeros_like(xk)
            xv[:, N] = bits(t["v"])[:, 0]
            check_append(cache, l, xk, base_k, prev_k, pos, [0], "K", code_bits, w.d, entry0=entry0)
            check_append(cache, l, xv, base_v, prev_v, pos, [0], "V", code_bits, w.d, entry0=entry0)
            lk, lv = layers(cache, range(2, l + 1), [0])
            ko = oracle.reconstruct(base_k, lk[:-1], want_f32=False, code_bits=code_bits)[1]
            vo = oracle.reconstruct(base_v, lv[:-1], want_f32=False, code_bits=code_bits)[1]
            kn = oracle.reconstruct(base_k, lk, want_f32=False, code_bits=code_bits)[1]
            vn = oracle.reconstruct(base_v, lv, want_f32=False, code_bits=code_bits)[1]
            qh, o, z, c, _ = oracle.attention(False, pos, slot, q, *before, S, ko, vo, kn, vn)
        after = dst.snapshot([0], hs)
        assert_close(after[1], o, O_ATOL, O_RTOL, f"decode loop {l} O")
        assert_close(after[2], z, Z_ATOL, 0, f"decode loop {l} Z")
        assert_close(after[3], c, C_ATOL, C_RTOL, f"decode loop {l} c")
