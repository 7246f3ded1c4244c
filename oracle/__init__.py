"""FP64 CPU oracle for the KDA mixer step (ctypes wrapper around ``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the product path (``verify_kda_decode_gb300``) never does,
and this package never imports the product.  The two share nothing but the seeded input
generators in ``kda_inputs``.

Every array crossing into C is a contiguous numpy array: BF16 tensors travel as their raw
``uint16`` bit patterns and are decoded exactly inside the oracle; everything else is float64.
The method's arithmetic lives only in ``kda_oracle.c`` (see its header for the sources and the
readings of the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")

STORE_F64, STORE_F32, STORE_BF16 = 0, 1, 2

_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_u16_p = ctypes.POINTER(ctypes.c_uint16)


class _Layer(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("r", ctypes.c_int),
        ("K", ctypes.c_int),
        ("W_fb", _c_u16_p), ("A_log", _c_double_p), ("dt_bias", _c_double_p),
        ("conv_w", _c_u16_p), ("norm_w", _c_double_p),
        ("l2_eps", ctypes.c_double), ("norm_eps", ctypes.c_double),
        ("W_fb8", ctypes.POINTER(ctypes.c_uint8)), ("W_fb_scale", _c_double_p),
    ]


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` to ``libkda_oracle.so`` with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.kdo_f32_to_bf16.restype = ctypes.c_uint16
        _lib.kdo_f32_to_bf16.argtypes = [ctypes.c_float]
        _lib.kdo_e4m3_to_f64.restype = ctypes.c_double
        _lib.kdo_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    return _lib


def _p(a: np.ndarray, dtype) -> ctypes.c_void_p:
    assert a.dtype == dtype and a.flags["C_CONTIGUOUS"], (a.dtype, dtype)
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


@dataclass
class Layer:
    """Layer weights in oracle form (BF16 as uint16 bits, the rest float64)."""
    H: int
    dk: int
    dv: int
    r: int
    K: int
    W_fb: np.ndarray      # uint16 [H*dk, r]
    A_log: np.ndarray     # f64 [H]
    dt_bias: np.ndarray   # f64 [H*dk]
    conv_w: np.ndarray    # uint16 [2*H*dk + H*dv, K]  (q, k, v channels)
    norm_w: np.ndarray    # f64 [dv]
    l2_eps: float = 1e-6
    norm_eps: float = 1e-5
    W_fb8: Optional[np.ndarray] = None       # uint8 [H*dk, r] E4M3 codes (FP8 input path)
    W_fb_scale: Optional[np.ndarray] = None  # f64 [H*dk] per-row scales (FP8 input path)

    def window_len(self) -> int:
        return (self.K - 1) * (2 * self.H * self.dk + self.H * self.dv)

    def _c(self):
        self._keep = [_u16(self.W_fb), _f64(self.A_log), _f64(self.dt_bias), _u16(self.conv_w),
                      _f64(self.norm_w)]
        w, a, d, c, n = self._keep
        w8 = sc = None
        if self.W_fb8 is not None:
            w8 = np.ascontiguousarray(self.W_fb8, dtype=np.uint8)
            sc = _f64(self.W_fb_scale)
            self._keep += [w8, sc]
        s = _Layer(self.H, self.dk, self.dv, self.r, self.K,
                   w.ctypes.data_as(_c_u16_p), a.ctypes.data_as(_c_double_p),
                   d.ctypes.data_as(_c_double_p), c.ctypes.data_as(_c_u16_p),
                   n.ctypes.data_as(_c_double_p), float(self.l2_eps), float(self.norm_eps),
                   None if w8 is None else w8.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                   None if sc is None else sc.ctypes.data_as(_c_double_p))
        return s


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed (rc={rc})")


def decode(layer: Layer, state, window, q, k, v, f_a, beta, gate, storage=STORE_F64):
    """n_steps single-token steps.  state [B,H,dk,dv], window [B,wl] (float64, copied);
    inputs [n_steps,B,...] uint16.  Returns (out [n_steps,B,H*dv], state, window)."""
    state, window = _f64(state).copy(), _f64(window).copy()
    q, k, v, f_a, beta, gate = map(_u16, (q, k, v, f_a, beta, gate))
    n_steps, B = q.shape[0], q.shape[1]
    out = np.zeros((n_steps, B, layer.H * layer.dv), np.float64)
    cl = layer._c()
    _check(lib().kdo_decode(ctypes.byref(cl), B, n_steps, storage, _p(state, np.float64),
                            _p(window, np.float64), _p(q, np.uint16), _p(k, np.uint16),
                            _p(v, np.uint16), _p(f_a, np.uint16), _p(beta, np.uint16),
                            _p(gate, np.uint16), _p(out, np.float64)), "decode")
    return out, state, window


def verify(layer: Layer, state, window, q, k, v, f_a, beta, gate):
    """T draft tokens.  inputs [B,T,...].  Returns (out [B,T,H*dv], rec_state [B,T,H,dk,dv],
    rec_window [B,T,wl]); state and window are not modified."""
    state, window = _f64(state), _f64(window)
    q, k, v, f_a, beta, gate = map(_u16, (q, k, v, f_a, beta, gate))
    B, T = q.shape[0], q.shape[1]
    out = np.zeros((B, T, layer.H * layer.dv), np.float64)
    rec = np.zeros((B, T, layer.H, layer.dk, layer.dv), np.float64)
    recw = np.zeros((B, T, layer.window_len()), np.float64)
    cl = layer._c()
    _check(lib().kdo_verify(ctypes.byref(cl), B, T, _p(state, np.float64), _p(window, np.float64),
                            _p(q, np.uint16), _p(k, np.uint16), _p(v, np.uint16),
                            _p(f_a, np.uint16), _p(beta, np.uint16), _p(gate, np.uint16),
                            _p(rec, np.float64), _p(recw, np.float64), _p(out, np.float64)),
           "verify")
    return out, rec, recw


def commit(H, dk, dv, K, storage, pool_state, pool_window, slot_ids, accepted, rec_state,
           rec_window):
    """Commit accepted draft lengths on raw pool bytes (returns new copies and the rc)."""
    pool_state = np.ascontiguousarray(pool_state).copy()
    pool_window = _u16(pool_window).copy()
    slot_ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    accepted = np.ascontiguousarray(accepted, dtype=np.int32)
    rec_state = np.ascontiguousarray(rec_state, dtype=np.float32)
    rec_window = _u16(rec_window)
    if storage == STORE_F32:
        assert pool_state.dtype == np.float32
    else:
        assert pool_state.dtype == np.uint16
    B, T = rec_state.shape[0], rec_state.shape[1]
    num_slots = pool_state.shape[0]
    rc = lib().kdo_commit(B, T, H, dk, dv, K, storage, num_slots,
                          pool_state.ctypes.data_as(ctypes.c_void_p), _p(pool_window, np.uint16),
                          _p(slot_ids, np.int32), _p(accepted, np.int32),
                          _p(rec_state, np.float32), _p(rec_window, np.uint16))
    return pool_state, pool_window, rc


def prefill(layer: Layer, state, window, q, k, v, f_a, beta, gate, storage=STORE_F64):
    """Token-by-token prefill.  inputs [B,L,...].  Returns (out [B,L,H*dv], state, window)."""
    state, window = _f64(state).copy(), _f64(window).copy()
    q, k, v, f_a, beta, gate = map(_u16, (q, k, v, f_a, beta, gate))
    B, L = q.shape[0], q.shape[1]
    out = np.zeros((B, L, layer.H * layer.dv), np.float64)
    cl = layer._c()
    _check(lib().kdo_prefill(ctypes.byref(cl), B, L, storage, _p(state, np.float64),
                             _p(window, np.float64), _p(q, np.uint16), _p(k, np.uint16),
                             _p(v, np.uint16), _p(f_a, np.uint16), _p(beta, np.uint16),
                             _p(gate, np.uint16), _p(out, np.float64)), "prefill")
    return out, state, window


def prefill_chunked(layer: Layer, state, window, q, k, v, f_a, beta, gate, chunk,
                    storage=STORE_F64):
    """Chunk-form prefill (FP64), for the recurrent = chunked pin."""
    state, window = _f64(state).copy(), _f64(window).copy()
    q, k, v, f_a, beta, gate = map(_u16, (q, k, v, f_a, beta, gate))
    B, L = q.shape[0], q.shape[1]
    out = np.zeros((B, L, layer.H * layer.dv), np.float64)
    cl = layer._c()
    _check(lib().kdo_prefill_chunked(ctypes.byref(cl), B, L, int(chunk), storage,
                                     _p(state, np.float64), _p(window, np.float64),
                                     _p(q, np.uint16), _p(k, np.uint16), _p(v, np.uint16),
                                     _p(f_a, np.uint16), _p(beta, np.uint16), _p(gate, np.uint16),
                                     _p(out, np.float64)), "prefill_chunked")
    return out, state, window


def recurrence_step(S, alpha, k, v, q, beta):
    """a6 alone on explicit vectors: returns (S_new, o)."""
    S = _f64(S).copy()
    dk, dv = S.shape
    alpha, k, v, q = map(_f64, (alpha, k, v, q))
    o = np.zeros(dv, np.float64)
    lib().kdo_recurrence_step(dk, dv, _p(S, np.float64), _p(alpha, np.float64), _p(k, np.float64),
                              _p(v, np.float64), _p(q, np.float64), ctypes.c_double(beta),
                              _p(o, np.float64))
    return S, o


def decay(layer: Layer, h: int, f_a) -> np.ndarray:
    """a1 + a2 for head h and one token's f_a (uint16 [r])."""
    f_a = _u16(f_a)
    alpha = np.zeros(layer.dk, np.float64)
    cl = layer._c()
    lib().kdo_decay(ctypes.byref(cl), h, _p(f_a, np.uint16), _p(alpha, np.float64))
    return alpha


def gated_rmsnorm(o, norm_w, eps, gate_bits):
    o, norm_w = _f64(o), _f64(norm_w)
    gate_bits = _u16(gate_bits)
    y = np.zeros_like(o)
    lib().kdo_gated_rmsnorm(o.shape[0], _p(o, np.float64), _p(norm_w, np.float64),
                            ctypes.c_double(eps), _p(gate_bits, np.uint16), _p(y, np.float64))
    return y


def conv_sequence(w_bits, w0, x_bits):
    """a4 on one channel over a sequence: returns (y [n], final window [K-1])."""
    w_bits, x_bits = _u16(w_bits), _u16(x_bits)
    w0 = _f64(w0)
    K = w_bits.shape[0]
    y = np.zeros(x_bits.shape[0], np.float64)
    w_end = np.zeros(K - 1, np.float64)
    lib().kdo_conv_sequence(K, _p(w_bits, np.uint16), _p(w0, np.float64), _p(x_bits, np.uint16),
                            x_bits.shape[0], _p(y, np.float64), _p(w_end, np.float64))
    return y, w_end


def l2_norms(q, k, eps):
    q, k = _f64(q).copy(), _f64(k).copy()
    lib().kdo_l2_norms(q.shape[0], ctypes.c_double(eps), _p(q, np.float64), _p(k, np.float64))
    return q, k


def store_round(x, storage):
    x = _f64(x).copy()
    lib().kdo_store_round(_p(x, np.float64), ctypes.c_size_t(x.size), storage)
    return x


def e4m3_to_f64(codes) -> np.ndarray:
    """FP8 E4M3 codes (uint8) -> values, by the oracle's decoding of the format."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    f = lib().kdo_e4m3_to_f64
    return np.array([f(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def f32_to_bf16(x) -> np.ndarray:
    """float32 array -> bf16 bits (uint16), round to nearest even, by the oracle's definition."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    f = lib().kdo_f32_to_bf16
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def max_threads() -> int:
    return int(lib().kdo_max_threads())


def set_threads(n: int) -> None:
    lib().kdo_set_threads(int(n))
