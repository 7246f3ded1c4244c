"""Thin ctypes binding of libkda (include/kda.h), same names as the C entry points.

Argument marshalling only: every step of the KDA mixer runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (PyTorch supplies device memory and streams); this module
checks their dtype, shape, device and contiguity (the C side only sees pointers), allocates
outputs the caller did not pass, and forwards raw pointers and the current stream of the
tensors' device, with that device current.  ``prepare_decode`` / ``prepare_verify`` do the
checks once for a loop over fixed buffers.  If the library is missing or fails to load,
importing this module raises: there is no other path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_DEVICE = range(5)
KDA_STATE_F32, KDA_STATE_BF16 = 0, 1
KDA_W_BF16, KDA_W_FP8_E4M3 = 0, 1
KDA_DEVERR_SLOT, KDA_DEVERR_ACCEPTED, KDA_DEVERR_TIMEOUT, KDA_DEVERR_DECAY = 0x1, 0x2, 0x4, 0x8
KDA_DEVERR_TOKENS, KDA_DEVERR_SEQLEN = 0x10, 0x20
DK = DV = RANK = 128
CONV_K = 4
PREFILL_CHUNK = 64


class KdaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class _Layer(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32), ("head_k_dim", ctypes.c_int32),
        ("head_v_dim", ctypes.c_int32), ("fa_rank", ctypes.c_int32),
        ("conv_size", ctypes.c_int32),
        ("W_fb", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
        ("l2_eps", ctypes.c_float), ("norm_eps", ctypes.c_float),
        ("w_fb_dtype", ctypes.c_int32), ("W_fb_scale", ctypes.c_void_p),
    ]


class _Pool(ctypes.Structure):
    _fields_ = [
        ("state", ctypes.c_void_p), ("state_dtype", ctypes.c_int32),
        ("conv_state", ctypes.c_void_p), ("num_slots", ctypes.c_int32),
        ("err_word", ctypes.c_void_p),
    ]


def _load() -> ctypes.CDLL:
    path = _build.LIB if _build.up_to_date() else _build.build()
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "kda_decode": [P, P, P, I32, P, P, P, P, P, P, P, P],
        "kda_verify": [P, P, P, I32, I32, P, P, P, P, P, P, P, P, P, P],
        "kda_commit": [P, I32, I32, I32, I32, P, P, I32, I32, P, P, P],
        "kda_decode_resume": [P, P, P, I32, P, I32, P, P, P, P, P, P, P, P, P, P],
        "kda_verify_resume": [P, P, P, I32, I32, P, P, I32, P, P, P, P, P, P, P, P, P, P, P, P],
        "kda_prefill": [P, P, P, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P],
        "kda_get_error": [P, P, P],
        "kda_prefill_noalloc": [P, P, P, I32, I32, I32, P, P, P, P, P, P, P, P],
        "kda_prefill_varlen": [P, P, P, I32, P, I32, I32, I32, P, P, P, P, P, P, P, P, SZ, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.kda_prefill_workspace_size.argtypes = [P, I32, I32, I32]
    lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
    lib.kda_prefill_varlen_workspace_size.argtypes = [P, I32, I32, I32]
    lib.kda_prefill_varlen_workspace_size.restype = ctypes.c_size_t
    lib.kda_prefill_noalloc_max_bytes.argtypes = []
    lib.kda_prefill_noalloc_max_bytes.restype = ctypes.c_size_t
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_abi_version.restype = ctypes.c_int32
    return lib


_lib = _load()

EXPORTS = ("kda_decode", "kda_verify", "kda_commit", "kda_decode_resume", "kda_verify_resume",
           "kda_prefill", "kda_prefill_workspace_size", "kda_prefill_varlen",
           "kda_prefill_varlen_workspace_size",
           "kda_get_error", "kda_status_string", "kda_last_error", "kda_abi_version",
           "kda_prefill_noalloc", "kda_prefill_noalloc_max_bytes")


def library() -> ctypes.CDLL:
    return _lib


def _raise(status: int):
    if status != KDA_OK:
        name = _lib.kda_status_string(status).decode()
        raise KdaError(status, f"{name}: {_lib.kda_last_error().decode()}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device: torch.device) -> int:
    """The cudaStream_t to launch on: the given stream (a torch.cuda.Stream or a raw handle), or
    the current stream of the tensors' device."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(device: torch.device, fn, *args) -> None:
    """Calls a C entry point with the tensors' device current: the library launches on the
    current device (and takes per-device set-up from it), which must be the one that owns the
    pointers."""
    if torch.cuda.current_device() == device.index:
        _raise(fn(*args))
    else:
        with torch.cuda.device(device):
            _raise(fn(*args))


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape, device):
    if (isinstance(t, torch.Tensor) and t.dtype == dtype and t.shape == shape and t.device == device
            and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


@dataclass
class KdaLayer:
    """Weights of one KDA layer on the device (see kda_layer in include/kda.h).  W_fb is bf16,
    or float8_e4m3fn codes with W_fb_scale (f32 [H*128], one scale per row): the FP8 path."""
    W_fb: torch.Tensor      # bf16 or float8_e4m3fn [H*128, 128]
    A_log: torch.Tensor     # f32 [H]
    dt_bias: torch.Tensor   # f32 [H*128]
    conv_w: torch.Tensor    # bf16 [3, H*128, 4]
    norm_w: torch.Tensor    # f32 [128]
    l2_eps: float = 1e-6
    norm_eps: float = 1e-5
    W_fb_scale: Optional[torch.Tensor] = None   # f32 [H*128] with float8_e4m3fn W_fb

    @property
    def H(self) -> int:
        return self.A_log.shape[0]

    @property
    def device(self) -> torch.device:
        return self.W_fb.device

    def c_struct(self) -> _Layer:
        # the struct is cached while the same tensors (same storage and shape) are attached
        ts = (self.W_fb, self.A_log, self.dt_bias, self.conv_w, self.norm_w)
        sc = self.W_fb_scale
        key = tuple((id(t), t.data_ptr(), t.shape, t.dtype) for t in ts) + (self.l2_eps, self.norm_eps) + \
            ((id(sc), sc.data_ptr(), sc.shape) if sc is not None else (None,))
        cached = self.__dict__.get("_c_struct")
        if cached is not None and cached[0] == key:
            return cached[1]
        H, dev = self.H, self.device
        fp8 = self.W_fb.dtype == torch.float8_e4m3fn
        _need(self.W_fb, "W_fb", torch.float8_e4m3fn if fp8 else torch.bfloat16, (H * DK, RANK), dev)
        if fp8:
            if sc is None:
                raise ValueError("W_fb_scale is required with float8_e4m3fn W_fb")
            _need(sc, "W_fb_scale", torch.float32, (H * DK,), dev)
        _need(self.A_log, "A_log", torch.float32, (H,), dev)
        _need(self.dt_bias, "dt_bias", torch.float32, (H * DK,), dev)
        _need(self.conv_w, "conv_w", torch.bfloat16, (3, H * DK, CONV_K), dev)
        _need(self.norm_w, "norm_w", torch.float32, (DV,), dev)
        st = _Layer(H, DK, DV, RANK, CONV_K, _ptr(self.W_fb), _ptr(self.A_log),
                    _ptr(self.dt_bias), _ptr(self.conv_w), _ptr(self.norm_w),
                    float(self.l2_eps), float(self.norm_eps),
                    KDA_W_FP8_E4M3 if fp8 else KDA_W_BF16, _ptr(sc) if fp8 else None)
        self.__dict__["_c_struct"] = (key, st)
        return st


@dataclass
class KdaPool:
    """Caller-owned slot pool (see kda_pool in include/kda.h)."""
    state: torch.Tensor        # f32 or bf16 [num_slots, H, 128, 128]
    conv_state: torch.Tensor   # bf16 [num_slots, 3, 3, H*128]
    err_word: torch.Tensor     # int32 [1], zeroed

    @staticmethod
    def zeros(num_slots: int, H: int, state_dtype=torch.float32, device="cuda") -> "KdaPool":
        return KdaPool(torch.zeros(num_slots, H, DK, DV, dtype=state_dtype, device=device),
                       torch.zeros(num_slots, 3, CONV_K - 1, H * DK, dtype=torch.bfloat16, device=device),
                       torch.zeros(1, dtype=torch.int32, device=device))

    @property
    def num_slots(self) -> int:
        return self.state.shape[0]

    @property
    def H(self) -> int:
        return self.state.shape[1]

    def c_struct(self) -> _Pool:
        ts = (self.state, self.conv_state, self.err_word)
        key = tuple((id(t), t.data_ptr(), t.shape, t.dtype) for t in ts)
        cached = self.__dict__.get("_c_struct")
        if cached is not None and cached[0] == key:
            return cached[1]
        dev = self.state.device
        if self.state.dtype == torch.float32:
            dt = KDA_STATE_F32
        elif self.state.dtype == torch.bfloat16:
            dt = KDA_STATE_BF16
        else:
            raise TypeError(f"state dtype {self.state.dtype}: expected float32 or bfloat16")
        n, H = self.num_slots, self.H
        _need(self.state, "state", self.state.dtype, (n, H, DK, DV), dev)
        _need(self.conv_state, "conv_state", torch.bfloat16, (n, 3, CONV_K - 1, H * DK), dev)
        _need(self.err_word, "err_word", torch.int32, (1,), dev)
        st = _Pool(_ptr(self.state), dt, _ptr(self.conv_state), n, _ptr(self.err_word))
        self.__dict__["_c_struct"] = (key, st)
        return st


def _token_args(layer: KdaLayer, pool: KdaPool, slot_ids, lead, q, k, v, f_a, beta_logit, gate):
    H, dev = layer.H, layer.device
    if pool.H != H:
        raise ValueError(f"pool has {pool.H} heads, layer {H}")
    B = lead[0]
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    for name, t, c in (("q", q, H * DK), ("k", k, H * DK), ("v", v, H * DV), ("f_a", f_a, RANK),
                       ("beta_logit", beta_logit, H), ("gate", gate, H * DV)):
        _need(t, name, torch.bfloat16, tuple(lead) + (c,), dev)


def kda_decode(layer: KdaLayer, pool: KdaPool, slot_ids, q, k, v, f_a, beta_logit, gate,
               out=None, stream=None) -> torch.Tensor:
    """Single-token decode for B sequences; inputs [B, C].  Returns out bf16 [B, H*128]."""
    B = q.shape[0]
    _token_args(layer, pool, slot_ids, (B,), q, k, v, f_a, beta_logit, gate)
    if out is None:
        out = torch.empty(B, layer.H * DV, dtype=torch.bfloat16, device=layer.device)
    _need(out, "out", torch.bfloat16, (B, layer.H * DV), layer.device)
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_decode, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B, _ptr(q), _ptr(k),
                           _ptr(v), _ptr(f_a), _ptr(beta_logit), _ptr(gate), _ptr(out),
                           _stream(stream, layer.device))
    return out


def kda_verify(layer: KdaLayer, pool: KdaPool, slot_ids, q, k, v, f_a, beta_logit, gate,
               out=None, rec_state=None, rec_conv=None, stream=None):
    """T draft tokens per sequence; inputs [B, T, C].  Returns (out [B,T,H*128],
    rec_state f32 [B,T,H,128,128], rec_conv bf16 [B,T,3,3,H*128])."""
    B, T = q.shape[0], q.shape[1]
    H, dev = layer.H, layer.device
    _token_args(layer, pool, slot_ids, (B, T), q, k, v, f_a, beta_logit, gate)
    if out is None:
        out = torch.empty(B, T, H * DV, dtype=torch.bfloat16, device=dev)
    if rec_state is None:
        rec_state = torch.empty(B, T, H, DK, DV, dtype=torch.float32, device=dev)
    if rec_conv is None:
        rec_conv = torch.empty(B, T, 3, CONV_K - 1, H * DK, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, T, H * DV), dev)
    _need(rec_state, "rec_state", torch.float32, (B, T, H, DK, DV), dev)
    _need(rec_conv, "rec_conv", torch.bfloat16, (B, T, 3, CONV_K - 1, H * DK), dev)
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_verify, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B, T, _ptr(q),
                           _ptr(k), _ptr(v), _ptr(f_a), _ptr(beta_logit), _ptr(gate), _ptr(out),
                           _ptr(rec_state), _ptr(rec_conv), _stream(stream, layer.device))
    return out, rec_state, rec_conv


def kda_commit(pool: KdaPool, slot_ids, accepted, rec_state, rec_conv, stream=None) -> None:
    """Commit accepted lengths (int32 [B], each in [0, T]) after kda_verify."""
    B, T, H = rec_state.shape[0], rec_state.shape[1], pool.H
    dev = pool.state.device
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(accepted, "accepted", torch.int32, (B,), dev)
    _need(rec_state, "rec_state", torch.float32, (B, T, H, DK, DV), dev)
    _need(rec_conv, "rec_conv", torch.bfloat16, (B, T, 3, CONV_K - 1, H * DK), dev)
    P = pool.c_struct()
    _call(dev, _lib.kda_commit, ctypes.byref(P), H, DK, DV, CONV_K, _ptr(slot_ids), _ptr(accepted), B, T,
                           _ptr(rec_state), _ptr(rec_conv), _stream(stream, dev))


def _prev_args(pool: KdaPool, B: int, prev):
    """(prev_accepted, prev_T, prev_rec_state, prev_rec_conv) pointers from a
    (accepted, rec_state, rec_conv) triple, or all empty for None."""
    if prev is None:
        return None, 0, None, None
    accepted, rec_state, rec_conv = prev
    H, dev = pool.H, pool.state.device
    Tp = rec_state.shape[1]
    _need(accepted, "prev_accepted", torch.int32, (B,), dev)
    _need(rec_state, "prev_rec_state", torch.float32, (B, Tp, H, DK, DV), dev)
    _need(rec_conv, "prev_rec_conv", torch.bfloat16, (B, Tp, 3, CONV_K - 1, H * DK), dev)
    return _ptr(accepted), Tp, _ptr(rec_state), _ptr(rec_conv)


def kda_decode_resume(layer: KdaLayer, pool: KdaPool, slot_ids, prev, q, k, v, f_a, beta_logit,
                      gate, out=None, stream=None) -> torch.Tensor:
    """Decode that first commits the previous step's drafts: prev = (accepted int32 [B],
    rec_state, rec_conv) of the previous verify, or None.  Equals kda_commit + kda_decode."""
    B = q.shape[0]
    _token_args(layer, pool, slot_ids, (B,), q, k, v, f_a, beta_logit, gate)
    if out is None:
        out = torch.empty(B, layer.H * DV, dtype=torch.bfloat16, device=layer.device)
    _need(out, "out", torch.bfloat16, (B, layer.H * DV), layer.device)
    pa, Tp, prs, prc = _prev_args(pool, B, prev)
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_decode_resume, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B, pa, Tp, prs,
                                  prc, _ptr(q), _ptr(k), _ptr(v), _ptr(f_a), _ptr(beta_logit),
                                  _ptr(gate), _ptr(out), _stream(stream, layer.device))
    return out


def kda_verify_resume(layer: KdaLayer, pool: KdaPool, slot_ids, prev, q, k, v, f_a, beta_logit,
                      gate, n_tokens=None, out=None, rec_state=None, rec_conv=None, stream=None):
    """Draft verify that first commits the previous step's drafts (prev as in
    kda_decode_resume) and runs n_tokens[b] (int32 [B] in [1, T], or None for T) tokens of
    sequence b.  Inputs [B, T, C].  Returns (out, rec_state, rec_conv) as kda_verify; entries
    past n_tokens[b] are left as they were."""
    B, T = q.shape[0], q.shape[1]
    H, dev = layer.H, layer.device
    _token_args(layer, pool, slot_ids, (B, T), q, k, v, f_a, beta_logit, gate)
    if n_tokens is not None:
        _need(n_tokens, "n_tokens", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty(B, T, H * DV, dtype=torch.bfloat16, device=dev)
    if rec_state is None:
        rec_state = torch.empty(B, T, H, DK, DV, dtype=torch.float32, device=dev)
    if rec_conv is None:
        rec_conv = torch.empty(B, T, 3, CONV_K - 1, H * DK, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, T, H * DV), dev)
    _need(rec_state, "rec_state", torch.float32, (B, T, H, DK, DV), dev)
    _need(rec_conv, "rec_conv", torch.bfloat16, (B, T, 3, CONV_K - 1, H * DK), dev)
    pa, Tp, prs, prc = _prev_args(pool, B, prev)
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_verify_resume, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B, T,
                                  _ptr(n_tokens), pa, Tp, prs, prc, _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(f_a), _ptr(beta_logit), _ptr(gate), _ptr(out),
                                  _ptr(rec_state), _ptr(rec_conv), _stream(stream, layer.device))
    return out, rec_state, rec_conv


def kda_prefill_workspace_size(layer: KdaLayer, B: int, L: int, chunk: int = PREFILL_CHUNK) -> int:
    Ls = layer.c_struct()
    return int(_lib.kda_prefill_workspace_size(ctypes.byref(Ls), B, L, chunk))


def kda_prefill(layer: KdaLayer, pool: KdaPool, slot_ids, q, k, v, f_a, beta_logit, gate,
                chunk: int = PREFILL_CHUNK, out=None, workspace=None, stream=None) -> torch.Tensor:
    """Prefill of L tokens per sequence from the slots' state; inputs [B, L, C].
    Returns out bf16 [B, L, H*128]; final state and conv window are left in the slots."""
    B, Ltok = q.shape[0], q.shape[1]
    H, dev = layer.H, layer.device
    _token_args(layer, pool, slot_ids, (B, Ltok), q, k, v, f_a, beta_logit, gate)
    if out is None:
        out = torch.empty(B, Ltok, H * DV, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, Ltok, H * DV), dev)
    need = kda_prefill_workspace_size(layer, B, Ltok, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_prefill, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B, Ltok, chunk,
                            _ptr(q), _ptr(k), _ptr(v), _ptr(f_a), _ptr(beta_logit), _ptr(gate),
                            _ptr(out), ws_ptr, ws_bytes, _stream(stream, layer.device))
    return out


def kda_prefill_varlen_workspace_size(layer: KdaLayer, B: int, total_tokens: int,
                                      chunk: int = PREFILL_CHUNK) -> int:
    Ls = layer.c_struct()
    return int(_lib.kda_prefill_varlen_workspace_size(ctypes.byref(Ls), B, total_tokens, chunk))


def kda_prefill_varlen(layer: KdaLayer, pool: KdaPool, slot_ids, cu_seqlens, max_len: int, q, k, v,
                       f_a, beta_logit, gate, chunk: int = PREFILL_CHUNK, out=None, workspace=None,
                       stream=None) -> torch.Tensor:
    """Variable-length prefill: sequence b is rows cu_seqlens[b]..cu_seqlens[b+1]-1 of the packed
    inputs [total_tokens, C] and continues from slot slot_ids[b].  max_len bounds every length
    (host int; no device read).  Returns out bf16 [total_tokens, H*128]."""
    H, dev = layer.H, layer.device
    B, total = slot_ids.shape[0], q.shape[0]
    if pool.H != H:
        raise ValueError(f"pool has {pool.H} heads, layer {H}")
    _need(slot_ids, "slot_ids", torch.int32, (B,), dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, (B + 1,), dev)
    for name, t, c in (("q", q, H * DK), ("k", k, H * DK), ("v", v, H * DV), ("f_a", f_a, RANK),
                       ("beta_logit", beta_logit, H), ("gate", gate, H * DV)):
        _need(t, name, torch.bfloat16, (total, c), dev)
    if out is None:
        out = torch.empty(total, H * DV, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (total, H * DV), dev)
    need = kda_prefill_varlen_workspace_size(layer, B, total, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel() * workspace.element_size())
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_prefill_varlen, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B,
                                   _ptr(cu_seqlens), total, int(max_len), chunk, _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(f_a), _ptr(beta_logit), _ptr(gate), _ptr(out),
                                   ws_ptr, ws_bytes, _stream(stream, layer.device))
    return out


def kda_prefill_noalloc(layer: KdaLayer, pool: KdaPool, slot_ids, q, k, v, f_a, beta_logit, gate,
                        chunk: int = PREFILL_CHUNK, out=None, stream=None) -> torch.Tensor:
    """kda_prefill without a caller workspace: the scratch lives in a fixed region inside the
    library (kda_prefill_noalloc_max_bytes(); larger requests raise KdaError).  For callers
    that cannot allocate device memory around the call.  `out` is allocated here only when the
    caller does not pass one."""
    B, Ltok = q.shape[0], q.shape[1]
    H, dev = layer.H, layer.device
    _token_args(layer, pool, slot_ids, (B, Ltok), q, k, v, f_a, beta_logit, gate)
    if out is None:
        out = torch.empty(B, Ltok, H * DV, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, Ltok, H * DV), dev)
    L, P = layer.c_struct(), pool.c_struct()
    _call(layer.device, _lib.kda_prefill_noalloc, ctypes.byref(L), ctypes.byref(P), _ptr(slot_ids), B, Ltok, chunk,
                                    _ptr(q), _ptr(k), _ptr(v), _ptr(f_a), _ptr(beta_logit), _ptr(gate),
                                    _ptr(out), _stream(stream, layer.device))
    return out


def kda_prefill_noalloc_max_bytes() -> int:
    return int(_lib.kda_prefill_noalloc_max_bytes())


def kda_get_error(pool: KdaPool, stream=None) -> int:
    """Reads and clears the pool's device error word (synchronises the stream)."""
    P = pool.c_struct()
    v = ctypes.c_int32(0)
    dev = pool.state.device
    if torch.cuda.current_device() == dev.index:
        st = _lib.kda_get_error(ctypes.byref(P), ctypes.byref(v), _stream(stream, dev))
    else:
        with torch.cuda.device(dev):
            st = _lib.kda_get_error(ctypes.byref(P), ctypes.byref(v), _stream(stream, dev))
    if st not in (KDA_OK, KDA_ERR_DEVICE):
        _raise(st)
    return int(v.value)


class PreparedCall:
    """One checked call of a C entry point, bound to fixed device buffers.

    ``prepare_decode`` / ``prepare_verify`` validate every argument once and keep the raw
    pointers as ctypes values; calling the object re-issues the same launch on the stream chosen
    when it was prepared, without re-checking or allocating anything.  Between calls the caller
    rewrites the bound input buffers in place, as a serving loop with static buffers (or a CUDA
    graph) does.  The object holds references to the bound tensors."""
    __slots__ = ("_fn", "_args", "_keep", "_dev")

    def __init__(self, fn, args, keep, device: torch.device):
        self._fn, self._args, self._keep, self._dev = fn, tuple(args), keep, device

    def __call__(self) -> None:
        if torch.cuda.current_device() == self._dev.index:
            st = self._fn(*self._args)
        else:
            with torch.cuda.device(self._dev):
                st = self._fn(*self._args)
        if st != KDA_OK:
            _raise(st)


def _c_ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(None if t is None else t.data_ptr())


def prepare_decode(layer: KdaLayer, pool: KdaPool, slot_ids, q, k, v, f_a, beta_logit, gate, out,
                   stream=None) -> PreparedCall:
    """kda_decode bound to these buffers (inputs [B, C], out [B, H*128]); see PreparedCall.
    `stream` defaults to the device's current stream at preparation."""
    B = q.shape[0]
    _token_args(layer, pool, slot_ids, (B,), q, k, v, f_a, beta_logit, gate)
    _need(out, "out", torch.bfloat16, (B, layer.H * DV), layer.device)
    L, P = layer.c_struct(), pool.c_struct()
    args = (ctypes.byref(L), ctypes.byref(P), _c_ptr(slot_ids), ctypes.c_int32(B), _c_ptr(q), _c_ptr(k),
            _c_ptr(v), _c_ptr(f_a), _c_ptr(beta_logit), _c_ptr(gate), _c_ptr(out),
            ctypes.c_void_p(_stream(stream, layer.device)))
    keep = (layer, pool, L, P, slot_ids, q, k, v, f_a, beta_logit, gate, out, stream)
    return PreparedCall(_lib.kda_decode, args, keep, layer.device)


def prepare_verify(layer: KdaLayer, pool: KdaPool, slot_ids, q, k, v, f_a, beta_logit, gate, out,
                   rec_state, rec_conv, stream=None) -> PreparedCall:
    """kda_verify bound to these buffers (inputs [B, T, C]); see PreparedCall."""
    B, T = q.shape[0], q.shape[1]
    H, dev = layer.H, layer.device
    _token_args(layer, pool, slot_ids, (B, T), q, k, v, f_a, beta_logit, gate)
    _need(out, "out", torch.bfloat16, (B, T, H * DV), dev)
    _need(rec_state, "rec_state", torch.float32, (B, T, H, DK, DV), dev)
    _need(rec_conv, "rec_conv", torch.bfloat16, (B, T, 3, CONV_K - 1, H * DK), dev)
    L, P = layer.c_struct(), pool.c_struct()
    args = (ctypes.byref(L), ctypes.byref(P), _c_ptr(slot_ids), ctypes.c_int32(B), ctypes.c_int32(T),
            _c_ptr(q), _c_ptr(k), _c_ptr(v), _c_ptr(f_a), _c_ptr(beta_logit), _c_ptr(gate), _c_ptr(out),
            _c_ptr(rec_state), _c_ptr(rec_conv), ctypes.c_void_p(_stream(stream, dev)))
    keep = (layer, pool, L, P, slot_ids, q, k, v, f_a, beta_logit, gate, out, rec_state, rec_conv, stream)
    return PreparedCall(_lib.kda_verify, args, keep, dev)
