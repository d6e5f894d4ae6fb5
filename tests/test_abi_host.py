"""CPU checks of the C-ABI library: it builds, loads, exports every entry
point the header declares, and rejects bad arguments on the host before
touching a device."""
import ctypes
import os
import re

import pytest

import lazy_sparse_attention_token_b300 as fl
from lazy_sparse_attention_token_b300 import build as flbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flashloop.h")

OK, INVALID, UNSUPPORTED, CAPACITY, CUDA, WORKSPACE = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def L():
    flbuild.build()
    return fl.lib()


def _header_text():
    with open(HEADER) as f:
        return f.read()


def declared_functions():
    text = _header_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flashloop_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert set(names) <= set(fl.flashloop.EXPORTS) | set(names)


def test_every_declaration_has_its_own_comment():
    """Each entry point of the header is directly preceded by a comment of its
    own (its operation, arguments, ownership and errors)."""
    text = _header_text()
    blank = re.sub(r"/\*.*?\*/", lambda m: " " * len(m.group(0)), text, flags=re.S)
    for n in declared_functions():
        m = re.search(r"^[^\n]*\b" + n + r"\s*\(", blank, re.M)
        assert m, n
        assert text[:m.start()].rstrip().endswith("*/"), f"{n} has no comment of its own"


def test_binding_covers_every_entry_point():
    for n in declared_functions():
        assert n in fl.flashloop.EXPORTS, n


def dims(**kw):
    base = dict(B=1, N_cap=1024, H=4, d=64, R=256, K=103, T=4, T_dense=1, R_cap=256)
    base.update(kw)
    return fl.Dims(**base)


def test_sizes(L):
    dm = dims()
    ws = fl.flashloop_workspace_bytes(dm)
    assert ws >= 1024 * 4 + 4 * 1 * 4 * 103 * 64 * 2
    cb = fl.flashloop_kv_cache_bytes(dm)
    dense = 1 * 1024 * 4 * 64 * 2
    per_delta_min = 256 * 4 + 1024 * 4 + 2 * 256 * 4 * (64 // 2 + 2 * 64 // 32)
    assert cb >= 2 * dense + 3 * per_delta_min
    assert cb <= 2 * dense + 3 * (per_delta_min + 6 * 256)
    for bad in (dict(d=80), dict(R=0), dict(K=2000), dict(T_dense=5), dict(R_cap=10), dict(T=40)):
        assert fl.flashloop_workspace_bytes(dims(**bad)) == 0
        assert fl.flashloop_kv_cache_bytes(dims(**bad)) == 0


def test_status_strings(L):
    for s in (OK, INVALID, UNSUPPORTED, CAPACITY, CUDA, WORKSPACE, -6):
        assert L.flashloop_status_string(s)
    assert L.flashloop_status_string(123) == b"unknown status"


P = ctypes.c_void_p


def test_select_tokens_rejects_bad_args(L):
    a, b, out = P(0x1000), P(0x2000), P(0x3000)
    assert L.flashloop_select_tokens(None, b, 1, 8, 16, 2, out, None, None, 0, None) == INVALID
    assert L.flashloop_select_tokens(P(0x1001), b, 1, 8, 16, 2, out, None, None, 0, None) == INVALID
    assert L.flashloop_select_tokens(a, b, 1, 8, 12, 2, out, None, None, 0, None) == INVALID   # D % 8
    assert L.flashloop_select_tokens(a, b, 1, 8, 16, 9, out, None, None, 0, None) == INVALID   # R > N
    assert L.flashloop_select_tokens(a, b, 1, 8, 16, 0, out, None, None, 0, None) == INVALID
    assert L.flashloop_select_tokens(a, b, 1, 8, 16, 2, out, None, None, 0, None) == WORKSPACE  # no scores buffer
    assert b"workspace" in L.flashloop_last_error()


def test_select_tokens_noalloc_rejects_bad_args(L):
    """Checked on the host before any device call: pointers, alignment, sizes,
    and B*N against the fixed scratch of 1,048,576 scores. Every call here is
    rejected by the host, so the placeholder pointers never reach a kernel."""
    a, b, out = P(0x1000), P(0x2000), P(0x3000)
    f = L.flashloop_select_tokens_noalloc
    assert f(None, b, 1, 8, 16, 2, out, None) == INVALID
    assert f(a, b, 1, 8, 16, 2, None, None) == INVALID
    assert f(a, P(0x2008), 1, 8, 16, 2, out, None) == INVALID      # misaligned
    assert f(a, b, 1, 8, 12, 2, out, None) == INVALID              # D % 8
    assert f(a, b, 1, 8, 16, 9, out, None) == INVALID              # R > N
    assert f(a, b, 0, 8, 16, 2, out, None) == INVALID              # B < 1
    assert f(a, b, 4, (1 << 18) + 1, 16, 2, out, None) == CAPACITY
    assert b"fixed scratch" in L.flashloop_last_error()
    assert f(a, b, 1 << 11, 1 << 11, 16, 2, out, None) == CAPACITY  # 4,194,304 scores


def test_binding_refuses_strided_and_host_tensors(L):
    """The binding hands the library only dense CUDA buffers: a strided or a
    host tensor is refused in Python, before any library call."""
    import torch
    from lazy_sparse_attention_token_b300 import flashloop as F
    assert F._ptr(None) is None
    with pytest.raises(ValueError, match="contiguous"):
        F._ptr(torch.zeros(4, 4).t())
    with pytest.raises(ValueError, match="CUDA"):
        F._ptr(torch.zeros(4))
    n0 = fl.flashloop_launch_count()
    with pytest.raises(ValueError, match="CUDA"):
        fl.flashloop_select_keys(torch.zeros(1, 2, 8), 2)
    assert fl.flashloop_launch_count() == n0


def test_gather_and_keys_reject_bad_args(L):
    assert L.flashloop_gather(P(0x1000), 1, 8, 24, P(0x2000), 2, P(0x3000), None) == INVALID      # row_bytes % 16
    assert L.flashloop_gather(P(0x1008), 1, 8, 32, P(0x2000), 2, P(0x3000), None) == INVALID      # misaligned
    assert L.flashloop_select_keys(P(0x1000), 1, 4, 8, 9, P(0x2000), None, 0, None) == INVALID    # K > N
    assert L.flashloop_select_keys(None, 1, 4, 8, 2, P(0x2000), None, 0, None) == INVALID


def test_cache_init_rejects_bad_args(L):
    c = fl.KVCache()
    dm = dims()
    need = fl.flashloop_kv_cache_bytes(dm)
    assert L.flashloop_kv_cache_init(ctypes.byref(c), P(0x10000), need - 1, ctypes.byref(dm), None) == CAPACITY
    assert L.flashloop_kv_cache_init(ctypes.byref(c), P(0x10010), need, ctypes.byref(dm), None) == INVALID
    bad = dims(d=80)
    assert L.flashloop_kv_cache_init(ctypes.byref(c), P(0x10000), need, ctypes.byref(bad), None) == UNSUPPORTED


def fake_cache(dm):
    """A descriptor with fake (never dereferenced) pointers for host-side checks."""
    c = fl.KVCache()
    c.dims = dm
    c.n_tokens = dm.N_cap
    for t in range(dm.T_dense):
        c.k_dense[t] = 0x100000 * (t + 1)
        c.v_dense[t] = 0x100000 * (t + 1) + 0x80000
    return c


def test_append_and_attention_reject_bad_args(L):
    dm = dims()
    c = fake_cache(dm)
    k, v, act = P(0x200000), P(0x300000), P(0x400000)
    # loop 1 is dense: no delta layer
    assert L.flashloop_kv_delta_append(ctypes.byref(c), 1, k, v, 1, act, 4, 0, None) == INVALID
    # appending past the layer's capacity
    assert L.flashloop_kv_delta_append(ctypes.byref(c), 2, k, v, 1, act, 300, 0, None) == CAPACITY
    # appending at an offset that is neither 0 nor the current count
    assert L.flashloop_kv_delta_append(ctypes.byref(c), 2, k, v, 1, act, 4, 7, None) == INVALID
    # dense store of a lazy loop
    assert L.flashloop_kv_dense_store(ctypes.byref(c), 2, k, v, 0, 4, None) == INVALID
    assert L.flashloop_kv_dense_store(ctypes.byref(c), 1, k, v, 1020, 8, None) == CAPACITY
    # reconstruct-gather of selected keys: lazy loops only, pointers, alignment, K
    rk = L.flashloop_reconstruct_keys
    kidx, o1, o2, o3, o4 = P(0x700000), P(0x710000), P(0x720000), P(0x730000), P(0x740000)
    assert rk(ctypes.byref(c), 1, kidx, 8, o1, o2, o3, o4, None) == INVALID           # loop 1 is dense
    assert rk(ctypes.byref(c), dm.T + 1, kidx, 8, o1, o2, o3, o4, None) == INVALID    # past the last loop
    assert rk(ctypes.byref(c), 2, None, 8, o1, o2, o3, o4, None) == INVALID
    assert rk(ctypes.byref(c), 2, kidx, 8, o1, o2, P(0x730008), o4, None) == INVALID  # misaligned output
    assert rk(ctypes.byref(c), 2, kidx, 0, o1, o2, o3, o4, None) == INVALID
    assert rk(ctypes.byref(c), 2, kidx, dm.N_cap + 1, o1, o2, o3, o4, None) == INVALID
    a = fl.AttnArgs()
    a.mode, a.loop, a.n_keys, a.n_state, a.R = fl.LAZY, 2, 1024, 1024, 4
    a.q = a.q_hat = a.o = 0x500000
    a.z = a.c = 0x600000
    a.cache = ctypes.pointer(c)
    assert L.flashloop_lazy_attention(ctypes.byref(a), None) == INVALID       # no key_idx
    a.mode = fl.DENSE
    assert L.flashloop_lazy_attention(ctypes.byref(a), None) == INVALID       # loop 2 is lazy
    a.mode, a.loop = fl.FIRST_DENSE, 2
    assert L.flashloop_lazy_attention(ctypes.byref(a), None) == INVALID
    s = fl.StepArgs()
    s.loop = 2
    s.cache = ctypes.pointer(c)
    assert L.flashloop_loop_step(ctypes.byref(s), None) == WORKSPACE


def test_rejected_calls_launch_nothing(L):
    """The launch counter (the source of the bench's launch figure) moves only
    when a kernel is enqueued: calls the host rejects leave it unchanged."""
    n0 = fl.flashloop_launch_count()
    a, b, out = P(0x1000), P(0x2000), P(0x3000)
    L.flashloop_select_tokens(a, b, 1, 8, 16, 9, out, None, None, 0, None)
    L.flashloop_select_tokens_noalloc(a, b, 4, (1 << 18) + 1, 16, 2, out, None)
    L.flashloop_gather(P(0x1000), 1, 8, 24, P(0x2000), 2, P(0x3000), None)
    L.flashloop_select_keys(P(0x1000), 1, 4, 8, 9, P(0x2000), None, 0, None)
    c = fake_cache(dims())
    L.flashloop_kv_delta_append(ctypes.byref(c), 2, P(0x200000), P(0x300000), 1, P(0x400000), 300, 0, None)
    s = fl.StepArgs()
    s.loop = 2
    s.cache = ctypes.pointer(c)
    L.flashloop_loop_step(ctypes.byref(s), None)
    assert fl.flashloop_launch_count() == n0


def kv_layout_bytes(B, N_cap, H, d, R_cap, T, T_dense):
    """The cache layout the header documents, summed without alignment padding:
    a bf16 K and V layer per dense loop; per lazy loop an entry list [B, R_cap]
    and slot map [B, N_cap] (int32) and, for K and V, int4 codes
    [B, R_cap, H, d/2] with fp16 scales [B, R_cap, H, d/32]."""
    dense = B * N_cap * H * d * 2
    delta = B * R_cap * 4 + B * N_cap * 4 + 2 * (B * R_cap * H * (d // 2) + B * R_cap * H * (d // 32) * 2)
    return 2 * T_dense * dense + (T - T_dense) * delta


@pytest.mark.parametrize("shape, ratio_lo", [
    # 32K prefill: 1 dense loop + 3 lazy loops of 15% active tokens
    (dict(B=1, N_cap=32768, H=16, d=128, R=4916, K=3277, T=4, T_dense=1, R_cap=4916), 3.4),
    # deep recurrence: 2 dense loops + 14 lazy loops of 10% active tokens
    (dict(B=8, N_cap=16384, H=32, d=96, R=1639, K=820, T=16, T_dense=2, R_cap=1639), 6.5),
])
def test_cache_against_a_bf16_cache_per_loop(L, shape, ratio_lo):
    """The base + int4-delta cache against one bf16 K/V cache per loop (a looped
    model without lazy updates): the library's size is the documented layout up
    to 256-byte alignment per section, and the ratio is what the deltas save."""
    cb = fl.flashloop_kv_cache_bytes(dims(**shape))
    want = kv_layout_bytes(shape["B"], shape["N_cap"], shape["H"], shape["d"], shape["R_cap"], shape["T"],
                           shape["T_dense"])
    sections = 2 * shape["T_dense"] + 6 * (shape["T"] - shape["T_dense"])
    assert want <= cb <= want + 256 * sections
    per_loop = shape["T"] * 2 * shape["B"] * shape["N_cap"] * shape["H"] * shape["d"] * 2
    assert per_loop / cb >= ratio_lo


def test_rejected_append_leaves_the_layer_as_it_was(L):
    """Every argument check of the delta append runs before its slot map is
    reset: a call refused for its token count returns INVALID_ARG without a
    device call (here on a host without a GPU it would otherwise report the
    missing device), and the layer's count stays where it was."""
    dm = dims()
    c = fake_cache(dm)
    c.count[0] = 5
    n0 = fl.flashloop_launch_count()
    for n_tokens in (0, dm.N_cap + 1):
        c.n_tokens = n_tokens
        st = L.flashloop_kv_delta_append(ctypes.byref(c), 2, P(0x200000), P(0x300000), 1, P(0x400000), 4, 0, None)
        assert st == INVALID
        assert b"n_tokens" in L.flashloop_last_error()
        assert c.count[0] == 5
    assert fl.flashloop_launch_count() == n0


def test_wait_limit_can_only_be_shortened(L):
    """The hook that shortens the attention kernel's bounded waits refuses a
    limit above the default on the host, before any device call."""
    n0 = fl.flashloop_launch_count()
    assert L.flashloop_set_wait_limit_ns(fl.flashloop.WAIT_LIMIT_DEFAULT_NS + 1) == INVALID
    assert b"exceeds the default" in L.flashloop_last_error()
    assert L.flashloop_set_wait_limit_ns(2 ** 63) == INVALID
    assert fl.flashloop_launch_count() == n0


def test_gemm_rejects_bad_args(L):
    """Shapes, pointers and alignment are checked on the host; the placeholder
    pointers never reach a kernel."""
    a, w, r = P(0x1000), P(0x2000), P(0x3000)
    outs = (P * 3)(P(0x10000), P(0x20000), P(0x30000))
    g = L.flashloop_gemm
    assert g(a, 8, 96, w, 256, None, 0, outs, 1, None, 0, 0, None) == INVALID       # K % 64
    assert g(a, 8, 64, w, 384, None, 0, outs, 1, None, 0, 0, None) == INVALID       # N % 256
    assert g(a, 8, 64, w, 512, None, 0, outs, 3, None, 0, 0, None) == INVALID       # N % (256 * 3)
    assert g(a, 8, 64, w, 256, None, 0, outs, 4, None, 0, 0, None) == INVALID       # n_split > 3
    assert g(a, -1, 64, w, 256, None, 0, outs, 1, None, 0, 0, None) == INVALID      # M < 0
    assert g(P(0x1008), 8, 64, w, 256, None, 0, outs, 1, None, 0, 0, None) == INVALID   # misaligned A
    assert g(a, 8, 64, w, 256, P(0x3004), 0, outs, 1, None, 0, 0, None) == INVALID   # misaligned residual
    assert g(a, 8, 64, w, 256, None, 0, None, 1, None, 0, 0, None) == INVALID       # no outputs
    assert g(a, 8, 64, w, 256, None, 0, outs, 1, r, 3, 16, None) == INVALID         # 3 does not divide M
    assert g(a, 0, 64, w, 256, None, 0, outs, 1, None, 0, 0, None) == OK            # M = 0: nothing to do


def test_block_sizes_and_rejects(L):
    dm = dims(H=4, d=64)                       # D = 256
    ws = fl.flashloop_block_workspace_bytes(dm, 1024)
    D, rows = 256, 1024
    assert ws >= fl.flashloop_workspace_bytes(dm) + 5 * rows * D * 2 + rows * 1024 * 2 + 256 * D * 2
    assert L.flashloop_block_workspace_bytes(ctypes.byref(dm), 1000) == 0      # F % 256
    assert L.flashloop_block_workspace_bytes(ctypes.byref(dims(H=3, d=64)), 1024) == 0   # D % 256
    assert L.flashloop_block_loop(None, None) == INVALID
    c = fake_cache(dm)
    wt = fl.BlockWeights(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 1024)
    a = fl.BlockArgs()
    a.loop, a.cache, a.weights = 2, ctypes.pointer(c), ctypes.pointer(wt)
    a.h_cur, a.h_out, a.h_prev = P(0x5000), P(0x5000), P(0x6000)
    a.workspace, a.workspace_bytes = P(0x100000), ws
    a.active_idx, a.key_idx = P(0x7000), P(0x8000)
    assert L.flashloop_block_loop(ctypes.byref(a), None) == INVALID           # h_out == h_cur
    a.h_out = P(0x9000)
    a.workspace_bytes = ws - 1
    assert L.flashloop_block_loop(ctypes.byref(a), None) == WORKSPACE
    a.workspace_bytes = ws
    wt.F = 1000
    assert L.flashloop_block_loop(ctypes.byref(a), None) == INVALID           # F % 256
    wt.F = 1024
    a.h_prev = None
    assert L.flashloop_block_loop(ctypes.byref(a), None) == INVALID           # lazy loop without h_prev


def test_lazy_loop_needs_r_and_k_within_the_tokens(L):
    """A lazy prefill loop whose R or K exceeds the cache's token count is refused
    on the host (the selections would have fewer candidates than picks)."""
    dm = dims(H=4, d=64)                       # R = 256, K = 103
    c = fake_cache(dm)
    c.n_tokens = 200                           # fewer tokens than R
    ws = fl.flashloop_block_workspace_bytes(dm, 1024)
    wt = fl.BlockWeights(P(0x1000), P(0x2000), P(0x3000), P(0x4000), 1024)
    a = fl.BlockArgs()
    a.loop, a.cache, a.weights = 2, ctypes.pointer(c), ctypes.pointer(wt)
    a.h_cur, a.h_out, a.h_prev = P(0x5000), P(0x9000), P(0x6000)
    a.workspace, a.workspace_bytes = P(0x100000), ws
    a.active_idx, a.key_idx = P(0x7000), P(0x8000)
    assert L.flashloop_block_loop(ctypes.byref(a), None) == INVALID
    assert b"must not exceed" in L.flashloop_last_error()
    st = fl.StepArgs()
    st.loop, st.cache = 2, ctypes.pointer(c)
    st.h_prev, st.h_cur, st.q, st.k, st.v = P(0x5000), P(0x6000), P(0x7000), P(0x8000), P(0x9000)
    st.q_hat, st.o, st.z, st.c = P(0xA000), P(0xB000), P(0xC000), P(0xD000)
    st.active_idx, st.key_idx = P(0xE000), P(0xF000)
    st.workspace, st.workspace_bytes = P(0x100000), fl.flashloop_workspace_bytes(dm)
    assert L.flashloop_loop_step(ctypes.byref(st), None) == INVALID
    assert b"must not exceed" in L.flashloop_last_error()
