"""Shared helpers of the GPU parity tests: running the CUDA path loop by loop
and comparing each step with the CPU oracle on the same inputs (teacher
forcing: the oracle starts every loop from the GPU's previous state)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
import lazy_sparse_attention_token_b300 as fl

# tolerances: attention outputs (bf16 operands, fp32 accumulation) and the
# proposed state tolerances for Z and the column mass c
O_ATOL, O_RTOL = 2e-2, 1e-2
Z_ATOL = 2e-2
C_ATOL, C_RTOL = 1e-3, 2e-2
SET_REL = 1e-5          # selection differences allowed within this of the k-th score
CODE_BOUNDARY = 1e-3    # int4 codes may differ this close to a rounding boundary


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


def assert_close(gpu: np.ndarray, orc: np.ndarray, atol: float, rtol: float, what: str):
    gpu = np.asarray(gpu, np.float64)
    orc = np.asarray(orc, np.float64)
    assert gpu.shape == orc.shape, (what, gpu.shape, orc.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - orc)
    bad = err > atol + rtol * np.abs(orc)
    if bad.any():
        i = np.unravel_index(np.argmax(err - atol - rtol * np.abs(orc)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} oracle={orc[i]!r}")


def assert_selection(gpu_idx: np.ndarray, orc_idx: np.ndarray, score: np.ndarray, what: str):
    """Same size, ascending; elements may differ only where the oracle's score
    lies within SET_REL of the k-th largest score."""
    assert gpu_idx.shape == orc_idx.shape, what
    assert np.all(np.diff(gpu_idx.astype(np.int64)) > 0), f"{what}: not strictly ascending"
    k = orc_idx.shape[0]
    thr = np.sort(score)[::-1][k - 1]
    diff = np.setxor1d(gpu_idx, orc_idx)
    if diff.size:
        far = np.abs(score[diff] - thr) > SET_REL * abs(thr)
        assert not far.any(), f"{what}: {int(far.sum())} elements differ away from the threshold"


def assert_layer(g_codes, g_scales, o_codes, o_scales, delta_over_scale, what):
    """Scales bit-exact; codes bit-exact except within CODE_BOUNDARY of a
    rounding boundary (delta/scale = n + 1/2)."""
    g_scales = np.asarray(g_scales).view(np.uint16)
    assert np.array_equal(g_scales, o_scales), f"{what}: fp16 scales differ in {int((g_scales != o_scales).sum())} places"
    if np.array_equal(g_codes, o_codes):
        return
    lo_g, hi_g = g_codes & 0xF, g_codes >> 4
    lo_o, hi_o = o_codes & 0xF, o_codes >> 4
    ge = np.stack([lo_g, hi_g], -1).reshape(delta_over_scale.shape)
    oe = np.stack([lo_o, hi_o], -1).reshape(delta_over_scale.shape)
    frac = np.abs(delta_over_scale - np.floor(delta_over_scale) - 0.5)
    bad = (ge != oe) & (frac >= CODE_BOUNDARY)
    assert not bad.any(), f"{what}: {int(bad.sum())} int4 codes differ away from a rounding boundary"


def delta_over_scale(x_l_bits, rec_f32, scales_bits):
    """(x - rec) / scale per element, in fp32 as the quantiser divides."""
    x = torch.from_numpy(x_l_bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    dl = (x - rec_f32).astype(np.float32)
    s = np.array(scales_bits, np.uint16).view(np.float16).astype(np.float32)
    s = np.repeat(s, 32, axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(s > 0, dl / np.where(s > 0, s, 1), 0).astype(np.float32)


def layers_from_gpu(cache: fl.Cache, loops, bsel, hsel=None):
    """Oracle DeltaLayers (sliced to sequences bsel and heads hsel) of the GPU's delta layers."""
    out_k, out_v = [], []
    for l in loops:
        idx, slot, kc, ks, vc, vs = cache.delta_layer(l)
        sl = (lambda a: a[bsel] if hsel is None else a[bsel][:, :, hsel])
        out_k.append(oracle.DeltaLayer(idx[bsel].cpu().numpy(), sl(kc).cpu().numpy(),
                                       sl(ks).cpu().numpy().view(np.uint16)))
        out_v.append(oracle.DeltaLayer(idx[bsel].cpu().numpy(), sl(vc).cpu().numpy(),
                                       sl(vs).cpu().numpy().view(np.uint16)))
    return out_k, out_v


def check_slot_map(cache: fl.Cache, loop: int, n_tokens: int):
    idx, slot, *_ = cache.delta_layer(loop)
    idx = idx.cpu().numpy()
    slot = slot.cpu().numpy()[:, :n_tokens]
    for b in range(idx.shape[0]):
        expect = np.full(n_tokens, -1, np.int64)
        expect[idx[b]] = np.arange(idx.shape[1])
        assert np.array_equal(slot[b], expect), f"slot map of loop {loop}, sequence {b}"


class State:
    """Row state of the CUDA path, on the device."""

    def __init__(self, B, n_state, H, d, n_keys, device="cuda"):
        self.q_hat = torch.zeros(B, n_state, H, d, dtype=torch.bfloat16, device=device)
        self.o = torch.zeros(B, n_state, H, d, dtype=torch.float32, device=device)
        self.z = torch.zeros(B, H, n_state, dtype=torch.float32, device=device)
        self.c = torch.zeros(B, H, n_keys, dtype=torch.float32, device=device)

    def snapshot(self, bsel, hsel):
        """Host copies sliced to sequences bsel and heads hsel (oracle layout)."""
        return (bits(self.q_hat[bsel][:, :, hsel]), f32(self.o[bsel][:, :, hsel]),
                f32(self.z[bsel][:, hsel]), f32(self.c[bsel][:, hsel]))


def dims_for(w: synth.Workload, extra_tokens: int = 0, R_extra: int = 0):
    R, K = synth.active_count(w), synth.key_count(w, w.N + extra_tokens)
    return fl.make_dims(w.B, w.N + extra_tokens, w.H, w.d, R, K, w.T, w.T_dense, R_cap=R + R_extra)
