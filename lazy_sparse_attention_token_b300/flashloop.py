"""Thin ctypes binding of libflashloop.so (the C ABI in include/flashloop.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream. Functions carry the
C names; each raises FlashLoopError on a non-OK status. There is no other
implementation behind these calls: without the built library on an sm_103
device they fail.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflashloop.so")
MAX_LOOPS = 32

I32, SZ, P = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p

FIRST_DENSE, DENSE, LAZY = 0, 1, 2


class FlashLoopError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({_status_string(status)}): {_last_error()}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("B", I32), ("N_cap", I32), ("H", I32), ("d", I32), ("R", I32), ("K", I32),
                ("T", I32), ("T_dense", I32), ("R_cap", I32), ("delta_bits", I32), ("base_bits", I32)]


class KVCache(ctypes.Structure):
    _fields_ = [("dims", Dims), ("n_tokens", I32),
                ("k_dense", P * MAX_LOOPS), ("v_dense", P * MAX_LOOPS),
                ("idx", P * MAX_LOOPS), ("slot", P * MAX_LOOPS),
                ("k_codes", P * MAX_LOOPS), ("k_scales", P * MAX_LOOPS),
                ("v_codes", P * MAX_LOOPS), ("v_scales", P * MAX_LOOPS),
                ("count", I32 * MAX_LOOPS),
                ("k_base_codes", P), ("v_base_codes", P), ("k_base_scales", P), ("v_base_scales", P)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("mode", I32), ("loop", I32), ("n_keys", I32), ("n_state", I32), ("R", I32),
                ("row_pos", P), ("row_slot", P), ("K", I32), ("key_idx", P),
                ("q", P), ("q_hat", P), ("o", P), ("z", P), ("c", P),
                ("cache", ctypes.POINTER(KVCache)), ("workspace", P), ("workspace_bytes", SZ)]


class StepArgs(ctypes.Structure):
    _fields_ = [("loop", I32), ("decode", I32), ("h_prev", P), ("h_cur", P), ("q", P), ("k", P), ("v", P),
                ("q_hat", P), ("o", P), ("z", P), ("c", P), ("cache", ctypes.POINTER(KVCache)),
                ("active_idx", P), ("key_idx", P), ("scores", P), ("workspace", P), ("workspace_bytes", SZ),
                ("key_rank", I32), ("exit_threshold", ctypes.c_float), ("seq_exit", P)]


class BlockWeights(ctypes.Structure):
    _fields_ = [("w_qkv", P), ("w_o", P), ("w_1", P), ("w_2", P), ("F", I32)]


class BlockArgs(ctypes.Structure):
    _fields_ = [("loop", I32), ("h_prev", P), ("h_cur", P), ("h_out", P), ("stale_idx", P), ("n_stale", I32),
                ("q_hat", P), ("o", P), ("z", P), ("c", P), ("cache", ctypes.POINTER(KVCache)),
                ("active_idx", P), ("key_idx", P), ("force_selection", I32), ("key_rank", I32), ("scores", P),
                ("weights", ctypes.POINTER(BlockWeights)), ("q", P), ("k", P), ("v", P),
                ("workspace", P), ("workspace_bytes", SZ)]


_lib = None

EXPORTS = [
    "flashloop_workspace_bytes", "flashloop_kv_cache_bytes", "flashloop_kv_cache_init",
    "flashloop_select_tokens", "flashloop_gather", "flashloop_kv_delta_append", "flashloop_kv_dense_store",
    "flashloop_select_keys", "flashloop_reconstruct_keys", "flashloop_lazy_attention", "flashloop_loop_step",
    "flashloop_status_string", "flashloop_last_error", "flashloop_device_status", "flashloop_launch_count",
    "flashloop_timing_enable", "flashloop_timing_read", "flashloop_select_tokens_noalloc",
    "flashloop_set_wait_limit_ns", "flashloop_select_keys_per_row", "flashloop_block_workspace_bytes",
    "flashloop_gemm", "flashloop_block_loop",
]
KEYS_BY_MASS, KEYS_BY_MASS_PER_ROW = 0, 1
WAIT_LIMIT_DEFAULT_NS = 1_000_000_000


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FileNotFoundError(f"{LIB_PATH} is missing: run lazy_sparse_attention_token_b300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        L.flashloop_workspace_bytes.restype = SZ
        L.flashloop_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
        L.flashloop_kv_cache_bytes.restype = SZ
        L.flashloop_kv_cache_bytes.argtypes = [ctypes.POINTER(Dims)]
        L.flashloop_kv_cache_init.argtypes = [ctypes.POINTER(KVCache), P, SZ, ctypes.POINTER(Dims), P]
        L.flashloop_select_tokens.argtypes = [P, P, I32, I32, I32, I32, P, P, P, SZ, P]
        L.flashloop_select_tokens_noalloc.argtypes = [P, P, I32, I32, I32, I32, P, P]
        L.flashloop_gather.argtypes = [P, I32, I32, I32, P, I32, P, P]
        L.flashloop_kv_delta_append.argtypes = [ctypes.POINTER(KVCache), I32, P, P, I32, P, I32, I32, P]
        L.flashloop_kv_dense_store.argtypes = [ctypes.POINTER(KVCache), I32, P, P, I32, I32, P]
        L.flashloop_select_keys.argtypes = [P, I32, I32, I32, I32, P, P, SZ, P]
        L.flashloop_select_keys_per_row.argtypes = [P, I32, I32, I32, I32, I32, P, P]
        L.flashloop_reconstruct_keys.argtypes = [ctypes.POINTER(KVCache), I32, P, I32, P, P, P, P, P]
        L.flashloop_lazy_attention.argtypes = [ctypes.POINTER(AttnArgs), P]
        L.flashloop_loop_step.argtypes = [ctypes.POINTER(StepArgs), P]
        L.flashloop_block_workspace_bytes.restype = SZ
        L.flashloop_block_workspace_bytes.argtypes = [ctypes.POINTER(Dims), I32]
        L.flashloop_gemm.argtypes = [P, I32, I32, P, I32, P, I32, ctypes.POINTER(P), I32, P, I32, I32, P]
        L.flashloop_block_loop.argtypes = [ctypes.POINTER(BlockArgs), P]
        L.flashloop_status_string.restype = ctypes.c_char_p
        L.flashloop_status_string.argtypes = [ctypes.c_int]
        L.flashloop_last_error.restype = ctypes.c_char_p
        L.flashloop_device_status.argtypes = [ctypes.POINTER(I32)]
        L.flashloop_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.flashloop_launch_count.restype = ctypes.c_int64
        L.flashloop_timing_enable.argtypes = [I32]
        L.flashloop_timing_read.restype = I32
        L.flashloop_timing_read.argtypes = [ctypes.c_char_p, I32, ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_int64), I32]
        for name in EXPORTS:
            if name not in ("flashloop_workspace_bytes", "flashloop_kv_cache_bytes", "flashloop_status_string",
                            "flashloop_block_workspace_bytes",
                            "flashloop_last_error", "flashloop_launch_count", "flashloop_timing_read"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _status_string(s: int) -> str:
    return lib().flashloop_status_string(s).decode()


def _last_error() -> str:
    return lib().flashloop_last_error().decode()


def _check(status: int, what: str):
    if status != 0:
        raise FlashLoopError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    """Device address of a contiguous CUDA tensor (None passes NULL). The
    library reads every buffer as dense row-major device memory, so a strided
    or host tensor is refused here rather than handed to a kernel."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must be in CUDA device memory")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_dims(B, N_cap, H, d, R, K, T, T_dense, R_cap=None, delta_bits=4, base_bits=16) -> Dims:
    return Dims(B, N_cap, H, d, R, K, T, T_dense, R if R_cap is None else R_cap, delta_bits, base_bits)


def flashloop_workspace_bytes(dims: Dims) -> int:
    return int(lib().flashloop_workspace_bytes(ctypes.byref(dims)))


def flashloop_kv_cache_bytes(dims: Dims) -> int:
    return int(lib().flashloop_kv_cache_bytes(ctypes.byref(dims)))


class Cache:
    """A KV cache in one device buffer, with torch views of its layers."""

    def __init__(self, dims: Dims, device="cuda", stream=None):
        self.dims = dims
        self.nbytes = flashloop_kv_cache_bytes(dims)
        if self.nbytes == 0:
            raise FlashLoopError(-1, "flashloop_kv_cache_bytes")
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.base = self.buf[off:off + self.nbytes]
        self.c = KVCache()
        _check(lib().flashloop_kv_cache_init(ctypes.byref(self.c), _ptr(self.base), self.nbytes,
                                              ctypes.byref(dims), _stream(stream)), "flashloop_kv_cache_init")

    @property
    def n_tokens(self) -> int:
        return self.c.n_tokens

    @n_tokens.setter
    def n_tokens(self, v: int):
        self.c.n_tokens = int(v)

    def _view(self, addr: int, shape, dtype) -> torch.Tensor:
        off = addr - self.base.data_ptr()
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.base[off:off + nbytes].view(dtype).view(shape)

    def dense_layer(self, loop: int):
        d = self.dims
        shape = (d.B, d.N_cap, d.H, d.d)
        return (self._view(self.c.k_dense[loop - 1], shape, torch.bfloat16),
                self._view(self.c.v_dense[loop - 1], shape, torch.bfloat16))

    @property
    def code_bits(self) -> int:
        return self.dims.delta_bits or 4

    def base_int8(self):
        """(k_codes, k_scales, v_codes, v_scales) of the int8 base (base_bits = 8), or None."""
        d = self.dims
        if d.base_bits != 8:
            return None
        shape, sshape = (d.B, d.N_cap, d.H, d.d), (d.B, d.N_cap, d.H, d.d // 32)
        return (self._view(self.c.k_base_codes, shape, torch.int8), self._view(self.c.k_base_scales, sshape, torch.int16),
                self._view(self.c.v_base_codes, shape, torch.int8), self._view(self.c.v_base_scales, sshape, torch.int16))

    def delta_layer(self, loop: int):
        """(idx, slot, k_codes, k_scales, v_codes, v_scales) of lazy loop `loop`, the first count entries."""
        d = self.dims
        m = loop - d.T_dense - 1
        cnt = self.c.count[m]
        row = d.d * self.code_bits // 8
        idx = self._view(self.c.idx[m], (d.B, d.R_cap), torch.int32)[:, :cnt]
        slot = self._view(self.c.slot[m], (d.B, d.N_cap), torch.int32)
        kc = self._view(self.c.k_codes[m], (d.B, d.R_cap, d.H, row), torch.uint8)[:, :cnt]
        ks = self._view(self.c.k_scales[m], (d.B, d.R_cap, d.H, d.d // 32), torch.int16)[:, :cnt]
        vc = self._view(self.c.v_codes[m], (d.B, d.R_cap, d.H, row), torch.uint8)[:, :cnt]
        vs = self._view(self.c.v_scales[m], (d.B, d.R_cap, d.H, d.d // 32), torch.int16)[:, :cnt]
        return idx, slot, kc, ks, vc, vs


def flashloop_select_tokens(h_prev, h_cur, R: int, active_idx=None, scores=None, workspace=None, stream=None):
    B, N, D = h_prev.shape
    if active_idx is None:
        active_idx = torch.empty(B, R, dtype=torch.int32, device=h_prev.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().flashloop_select_tokens(_ptr(h_prev), _ptr(h_cur), B, N, D, R, _ptr(active_idx), _ptr(scores),
                                         _ptr(workspace), ws_bytes, _stream(stream)), "flashloop_select_tokens")
    return active_idx


def flashloop_select_tokens_noalloc(h_prev, h_cur, R: int, active_idx=None, stream=None):
    """flashloop_select_tokens with the library's fixed scratch (no workspace, no allocation)."""
    B, N, D = h_prev.shape
    if active_idx is None:
        active_idx = torch.empty(B, R, dtype=torch.int32, device=h_prev.device)
    _check(lib().flashloop_select_tokens_noalloc(_ptr(h_prev), _ptr(h_cur), B, N, D, R, _ptr(active_idx),
                                                 _stream(stream)), "flashloop_select_tokens_noalloc")
    return active_idx


def flashloop_gather(src, idx, dst=None, stream=None):
    """dst[b, r] = src[b, idx[b, r]] over the trailing dims of src [B, N, ...]."""
    B, N = src.shape[:2]
    R = idx.shape[1]
    if dst is None:
        dst = torch.empty((B, R) + tuple(src.shape[2:]), dtype=src.dtype, device=src.device)
    row_bytes = src[0, 0].numel() * src.element_size()
    _check(lib().flashloop_gather(_ptr(src), B, N, row_bytes, _ptr(idx), R, _ptr(dst), _stream(stream)),
           "flashloop_gather")
    return dst


def flashloop_kv_delta_append(cache: Cache, loop: int, k_l, v_l, active_idx, at: int = 0,
                              rows_are_tokens: bool = True, stream=None):
    R = active_idx.shape[1]
    _check(lib().flashloop_kv_delta_append(ctypes.byref(cache.c), loop, _ptr(k_l), _ptr(v_l), int(rows_are_tokens),
                                           _ptr(active_idx), R, at, _stream(stream)), "flashloop_kv_delta_append")


def flashloop_kv_dense_store(cache: Cache, loop: int, k, v, pos0: int = 0, stream=None):
    _check(lib().flashloop_kv_dense_store(ctypes.byref(cache.c), loop, _ptr(k), _ptr(v), pos0, k.shape[1],
                                          _stream(stream)), "flashloop_kv_dense_store")


def flashloop_select_keys(col_stats, K: int, key_idx=None, stream=None):
    B, H, N = col_stats.shape
    if key_idx is None:
        key_idx = torch.empty(B, H, K, dtype=torch.int32, device=col_stats.device)
    _check(lib().flashloop_select_keys(_ptr(col_stats), B, H, N, K, _ptr(key_idx), None, 0, _stream(stream)),
           "flashloop_select_keys")
    return key_idx


def flashloop_select_keys_per_row(col_stats, K: int, n_rows: Optional[int] = None, key_idx=None, stream=None):
    """Top-K of col_stats[b, h, j] / (n_rows - j) per (b, h) (n_rows defaults to N)."""
    B, H, N = col_stats.shape
    if key_idx is None:
        key_idx = torch.empty(B, H, K, dtype=torch.int32, device=col_stats.device)
    _check(lib().flashloop_select_keys_per_row(_ptr(col_stats), B, H, N, K, N if n_rows is None else n_rows,
                                               _ptr(key_idx), _stream(stream)), "flashloop_select_keys_per_row")
    return key_idx


def flashloop_reconstruct_keys(cache: Cache, loop: int, key_idx, stream=None):
    d = cache.dims
    B, H, K = key_idx.shape
    outs = [torch.empty(B, H, K, d.d, dtype=torch.bfloat16, device=key_idx.device) for _ in range(4)]
    _check(lib().flashloop_reconstruct_keys(ctypes.byref(cache.c), loop, _ptr(key_idx), K, *[_ptr(o) for o in outs],
                                            _stream(stream)), "flashloop_reconstruct_keys")
    return outs


def flashloop_lazy_attention(cache: Cache, mode: int, loop: int, q, q_hat, o, z, c, row_pos=None, row_slot=None,
                             key_idx=None, n_keys: Optional[int] = None, workspace=None, stream=None):
    a = AttnArgs()
    a.mode, a.loop = mode, loop
    a.n_keys = c.shape[2] if n_keys is None else n_keys
    a.n_state = q.shape[1]
    a.R = a.n_state if row_pos is None else row_pos.shape[1]
    a.row_pos, a.row_slot = _ptr(row_pos), _ptr(row_slot)
    a.K = 0 if key_idx is None else key_idx.shape[2]
    a.key_idx = _ptr(key_idx)
    a.q, a.q_hat, a.o, a.z, a.c = _ptr(q), _ptr(q_hat), _ptr(o), _ptr(z), _ptr(c)
    a.cache = ctypes.pointer(cache.c)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().flashloop_lazy_attention(ctypes.byref(a), _stream(stream)), "flashloop_lazy_attention")


def flashloop_loop_step(cache: Cache, loop: int, q, k, v, q_hat, o, z, c, workspace, h_prev=None, h_cur=None,
                        active_idx=None, key_idx=None, scores=None, decode: bool = False, key_rank: int = 0,
                        exit_threshold: float = 0.0, seq_exit=None, stream=None):
    a = StepArgs()
    a.loop, a.decode = loop, int(decode)
    a.key_rank = key_rank
    a.exit_threshold, a.seq_exit = float(exit_threshold), _ptr(seq_exit)
    a.h_prev, a.h_cur = _ptr(h_prev), _ptr(h_cur)
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.q_hat, a.o, a.z, a.c = _ptr(q_hat), _ptr(o), _ptr(z), _ptr(c)
    a.cache = ctypes.pointer(cache.c)
    a.active_idx, a.key_idx, a.scores = _ptr(active_idx), _ptr(key_idx), _ptr(scores)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().flashloop_loop_step(ctypes.byref(a), _stream(stream)), "flashloop_loop_step")


def flashloop_gemm(a, w_t, c: Sequence[torch.Tensor], residual=None, relu: bool = False, c_rows=None,
                   rows_per_seq: int = 0, seq_rows: int = 0, stream=None):
    """C = act(a @ w_t.T + residual) into the outputs ``c`` (a column split
    of N into len(c) parts), rows scattered by ``c_rows`` when given."""
    M, K = a.shape
    N = w_t.shape[0]
    outs = (P * len(c))(*[_ptr(t) for t in c])
    _check(lib().flashloop_gemm(_ptr(a), M, K, _ptr(w_t), N, _ptr(residual), int(relu), outs, len(c), _ptr(c_rows),
                                rows_per_seq, seq_rows, _stream(stream)), "flashloop_gemm")


def flashloop_block_workspace_bytes(dims: Dims, F: int) -> int:
    return int(lib().flashloop_block_workspace_bytes(ctypes.byref(dims), F))


def block_workspace_for(dims: Dims, F: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned workspace of flashloop_block_workspace_bytes(dims, F)."""
    n = flashloop_block_workspace_bytes(dims, F)
    if n == 0:
        raise FlashLoopError(-1, "flashloop_block_workspace_bytes")
    buf = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def flashloop_block_loop(cache: Cache, loop: int, weights: Sequence[torch.Tensor], h_cur, h_out, q_hat, o, z, c,
                         workspace, h_prev=None, stale_idx=None, active_idx=None, key_idx=None,
                         force_selection: bool = False, key_rank: int = 0, scores=None, q=None, k=None, v=None,
                         stream=None):
    """One loop of the synthetic looped block; ``weights`` = (w_qkv, w_o, w_1, w_2), each [out, in] bf16."""
    w_qkv, w_o, w_1, w_2 = weights
    wt = BlockWeights(_ptr(w_qkv), _ptr(w_o), _ptr(w_1), _ptr(w_2), w_1.shape[0])
    a = BlockArgs()
    a.loop = loop
    a.h_prev, a.h_cur, a.h_out = _ptr(h_prev), _ptr(h_cur), _ptr(h_out)
    a.stale_idx = _ptr(stale_idx)
    a.n_stale = 0 if stale_idx is None else stale_idx.shape[-1]
    a.q_hat, a.o, a.z, a.c = _ptr(q_hat), _ptr(o), _ptr(z), _ptr(c)
    a.cache = ctypes.pointer(cache.c)
    a.active_idx, a.key_idx = _ptr(active_idx), _ptr(key_idx)
    a.force_selection, a.key_rank, a.scores = int(force_selection), key_rank, _ptr(scores)
    a.weights = ctypes.pointer(wt)
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().flashloop_block_loop(ctypes.byref(a), _stream(stream)), "flashloop_block_loop")


def flashloop_device_status() -> int:
    w = I32(0)
    lib().flashloop_device_status(ctypes.byref(w))
    return w.value


def flashloop_set_wait_limit_ns(ns: int):
    """Limit of the attention kernel's bounded waits (may only shorten the default; synchronises)."""
    _check(lib().flashloop_set_wait_limit_ns(int(ns)), "flashloop_set_wait_limit_ns")


def flashloop_launch_count() -> int:
    return int(lib().flashloop_launch_count())


def flashloop_timing_enable(on: bool = True):
    _check(lib().flashloop_timing_enable(int(on)), "flashloop_timing_enable")


def flashloop_timing_read(max_kinds: int = 32):
    """{kernel family: (total ms, launches)} since the previous read (synchronises)."""
    name_len = 64
    names = ctypes.create_string_buffer(name_len * max_kinds)
    ms = (ctypes.c_double * max_kinds)()
    cnt = (ctypes.c_int64 * max_kinds)()
    n = lib().flashloop_timing_read(names, name_len, ms, cnt, max_kinds)
    if n < 0:
        raise FlashLoopError(-4, "flashloop_timing_read")
    return {names.raw[k * name_len:(k + 1) * name_len].split(b"\0")[0].decode(): (ms[k], cnt[k]) for k in range(n)}


def workspace_for(dims: Dims, device="cuda") -> torch.Tensor:
    """A 256-byte aligned workspace of flashloop_workspace_bytes(dims)."""
    n = flashloop_workspace_bytes(dims)
    buf = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]
