"""flashloop_select_tokens_noalloc: token selection for callers that may not
allocate device memory (code inside a memory arena it does not own, or on a
path where an allocation could stall or fail). It keeps the change scores
in a fixed array of the library; its result must equal the workspace-based
flashloop_select_tokens on the same inputs, call after call. The file is
named to run last so that a failure here never hides another test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import lazy_sparse_attention_token_b300 as fl
from lazy_sparse_attention_token_b300 import build as flbuild
from gpu_helpers import assert_selection, bits

pytestmark = pytest.mark.gpu

CAPACITY = -3


def _inputs(seed, B, N, D):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    hp = torch.randn(B, N, D, generator=g, device="cuda").to(torch.bfloat16)
    drift = torch.rand(B, N, 1, generator=g, device="cuda") ** 3
    hc = (hp.float() + drift * torch.randn(B, N, D, generator=g, device="cuda")).to(torch.bfloat16)
    return hp, hc


def test_no_alloc_selection_matches_workspace_selection_twice():
    flbuild.build()
    L = fl.lib()
    B, N, D, R = 3, 20000, 256, 2500
    for call, seed in enumerate((101, 202)):      # two calls in a row share the fixed scratch
        hp, hc = _inputs(seed, B, N, D)
        ref = fl.flashloop_select_tokens(hp, hc, R, scores=torch.empty(B, N, device="cuda"))
        out = torch.full((B, R), -1, dtype=torch.int32, device="cuda")
        st = L.flashloop_select_tokens_noalloc(ctypes.c_void_p(hp.data_ptr()), ctypes.c_void_p(hc.data_ptr()),
                                               B, N, D, R, ctypes.c_void_p(out.data_ptr()),
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, fl.flashloop._last_error()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy()), f"call {call}"
        # and both against the oracle's ranking of the same hidden states
        sc = oracle.token_scores(bits(hp), bits(hc))
        A_orc = oracle.topk(sc, R)
        got = out.cpu().numpy()
        for b in range(B):
            assert_selection(got[b], A_orc[b], sc[b], f"call {call}, sequence {b}")


def test_no_alloc_selection_at_its_full_scratch():
    L = fl.lib()
    B, N, D, R = 4, (1 << 20) // 4, 8, 30000      # B*N exactly fills the fixed scratch
    hp, hc = _inputs(303, B, N, D)
    ref = fl.flashloop_select_tokens(hp, hc, R, scores=torch.empty(B, N, device="cuda"))
    out = torch.full((B, R), -1, dtype=torch.int32, device="cuda")
    st = L.flashloop_select_tokens_noalloc(ctypes.c_void_p(hp.data_ptr()), ctypes.c_void_p(hc.data_ptr()),
                                           B, N, D, R, ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, fl.flashloop._last_error()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref.cpu().numpy())


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    L = fl.lib()
    hp, hc = _inputs(7, 1, 8, 8)
    out = torch.empty(1, 1, dtype=torch.int32, device="cuda")
    st = L.flashloop_select_tokens_noalloc(ctypes.c_void_p(hp.data_ptr()), ctypes.c_void_p(hc.data_ptr()),
                                           2, (1 << 20) // 2 + 1, 8, 1, ctypes.c_void_p(out.data_ptr()), None)
    assert st == CAPACITY
    assert b"fixed scratch" in L.flashloop_last_error()
