"""Early exit by state difference (beyond the main setting; the recurrent-depth
overview page's per-sequence dynamic early exit): through flashloop_loop_step,
a sequence whose largest token change score falls below the threshold stops
looping, and is compared with the oracle's loop on the same inputs and sets."""
import copy

import numpy as np
import pytest
import torch

import oracle
from oracle import loop as oloop
import lazy_sparse_attention_token_b300 as fl
from lazy_sparse_attention_token_b300 import build as flbuild
from gpu_helpers import C_ATOL, C_RTOL, O_ATOL, O_RTOL, Z_ATOL, State, assert_close, bits, f32, layers_from_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    flbuild.build()
    fl.lib()
    oracle.build()


def _inputs(B, N, H, d, drift, seed=70):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    rn = lambda *s: torch.randn(*s, generator=g, device="cuda")
    h1 = rn(B, N, H * d).to(torch.bfloat16)
    scale = torch.tensor(drift, device="cuda").view(B, 1, 1)
    h2 = (h1.float() + scale * rn(B, N, H * d)).to(torch.bfloat16)
    h3 = (h2.float() + scale * rn(B, N, H * d)).to(torch.bfloat16)
    qkv = [[rn(B, N, H, d).to(torch.bfloat16) for _ in range(3)] for _ in range(3)]
    return (h1, h2, h3), qkv


def test_loop_step_stops_a_frozen_sequence():
    B, N, H, d, T = 3, 700, 2, 64, 3
    R, K = 175, 70
    (h1, h2, h3), qkv = _inputs(B, N, H, d, [0.5, 0.0, 0.01])   # sequence 1 does not change at all
    dm = fl.make_dims(B, N, H, d, R, K, T, 1, R_cap=R)
    cache = fl.Cache(dm)
    cache.n_tokens = N
    ws = fl.workspace_for(dm)
    st = State(B, N, H, d, N)
    flags = torch.zeros(B, dtype=torch.int32, device="cuda")
    act = torch.empty(B, R, dtype=torch.int32, device="cuda")
    keys = torch.empty(B, H, K, dtype=torch.int32, device="cuda")
    fl.flashloop_loop_step(cache, 1, *qkv[0], st.q_hat, st.o, st.z, st.c, ws)
    ocache = oloop.Cache()
    ocache.dense_k.append(bits(qkv[0][1]))
    ocache.dense_v.append(bits(qkv[0][2]))
    hs = [h1, h2, h3]
    exited = np.zeros(B, bool)
    for l, thr in ((2, 1e-6), (3, 0.0)):     # loop 3: no new threshold, the flag stays
        before = oloop.State(*st.snapshot(list(range(B)), list(range(H))))
        fl.flashloop_loop_step(cache, l, *qkv[l - 1], st.q_hat, st.o, st.z, st.c, ws, h_prev=hs[l - 2],
                               h_cur=hs[l - 1], active_idx=act, key_idx=keys, exit_threshold=thr, seq_exit=flags)
        torch.cuda.synchronize()
        assert fl.flashloop_device_status() == 0
        assert flags.cpu().tolist() == [0, 1, 0], (l, flags)
        A, S = act.cpu().numpy(), keys.cpu().numpy()
        res = oloop.lazy_loop(l, bits(hs[l - 2]), bits(hs[l - 1]), *qkv[l - 1], copy.deepcopy(ocache), before, R, K,
                              A=A, S=S, exit_threshold=thr, exited=exited)
        exited = res[6]
        assert exited.tolist() == [False, True, False]
        after = st.snapshot(list(range(B)), list(range(H)))
        assert_close(after[1], res[3].o, O_ATOL, O_RTOL, f"loop {l} O")
        assert_close(after[2], res[3].z, Z_ATOL, 0, f"loop {l} Z")
        assert_close(after[3], res[3].c, C_ATOL, C_RTOL, f"loop {l} c")
        assert np.array_equal(after[0], res[3].qhat)
        for name, i in (("q_hat", 0), ("o", 1), ("z", 2), ("c", 3)):   # the stopped sequence, bit for bit
            assert np.array_equal(after[i][1], before.__dict__[("qhat", "o", "z", "c")[i]][1]), name
        lk, lv = layers_from_gpu(cache, [l], list(range(B)))
        assert not lk[0].codes[1].any() and not lk[0].scales[1].any() and not lv[0].scales[1].any()
        assert np.array_equal(lk[0].scales, res[4].scales) and np.array_equal(lv[0].scales, res[5].scales)
        # the oracle's cache follows the GPU's layers (teacher forcing)
        ocache.delta_k.append(lk[0])
        ocache.delta_v.append(lv[0])
