"""Test plumbing: turn a ``kda_inputs.Case`` into oracle arguments and compare results.

Gathering a pool's rows by slot id, decoding BF16 bit patterns and the error metrics live
here; none of the method's arithmetic does.
"""
from __future__ import annotations

import numpy as np

import oracle
from kda_inputs import Case, bf16_bits_to_f32


def oracle_layer(case: Case) -> oracle.Layer:
    lw = case.layer
    return oracle.Layer(
        H=lw.H, dk=lw.dk, dv=lw.dv, r=lw.r, K=lw.K,
        W_fb=lw.W_fb, A_log=lw.A_log.astype(np.float64), dt_bias=lw.dt_bias.astype(np.float64),
        conv_w=np.ascontiguousarray(lw.conv_w.reshape(3 * lw.H * lw.dk, lw.K)),
        norm_w=lw.norm_w.astype(np.float64), l2_eps=lw.l2_eps, norm_eps=lw.norm_eps,
        W_fb8=lw.W_fb_fp8,
        W_fb_scale=None if lw.W_fb_scale is None else lw.W_fb_scale.astype(np.float64))


def pool_state_f64(case: Case, state=None) -> np.ndarray:
    """Whole pool state as float64 (exact decode of FP32 / BF16 storage)."""
    st = case.pool.state if state is None else state
    if case.pool.state_dtype == "bf16":
        return bf16_bits_to_f32(st).astype(np.float64)
    return np.asarray(st, np.float32).astype(np.float64)


def gathered_state(case: Case, sel=None) -> np.ndarray:
    ids = case.slot_ids if sel is None else case.slot_ids[sel]
    st = case.pool.state[ids]
    if case.pool.state_dtype == "bf16":
        return bf16_bits_to_f32(st).astype(np.float64)
    return st.astype(np.float64)


def gathered_window(case: Case, sel=None) -> np.ndarray:
    ids = case.slot_ids if sel is None else case.slot_ids[sel]
    w = bf16_bits_to_f32(case.pool.conv[ids]).astype(np.float64)
    return np.ascontiguousarray(w.reshape(w.shape[0], -1))


def storage_mode(case: Case) -> int:
    return oracle.STORE_BF16 if case.pool.state_dtype == "bf16" else oracle.STORE_F32


def bf16_half_ulp(a) -> np.ndarray:
    """Half the spacing of BF16 numbers (8 significant bits) at |a| (binary32 exponent range)."""
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def bf16_out_err(x, ref) -> float:
    """Error of BF16 outputs x against unrounded reference values, beyond the output rounding
    itself: max_i max(0, |x_i - ref_i| - half_ulp_bf16(max(|x_i|, |ref_i|))) / max_i |ref_i|.
    Rounding a result to BF16 moves it by up to half a BF16 ulp (up to 2^-8 = 3.9e-3 of the
    value), which no BF16 output can avoid; the tolerance applies to what remains."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if not ref.size:
        return 0.0
    slack = bf16_half_ulp(np.maximum(np.abs(x), np.abs(ref)))
    excess = np.maximum(np.abs(x - ref) - slack, 0.0)
    den = float(np.max(np.abs(ref)))
    return float(np.max(excess) / den) if den > 0 else float(np.max(excess))


def bf16_pair_err(x, y) -> float:
    """Error between two BF16-rounded results of the same quantity, beyond one BF16 spacing
    (two roundings of nearly equal values can land one spacing apart)."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    if not x.size:
        return 0.0
    slack = 2.0 * bf16_half_ulp(np.maximum(np.abs(x), np.abs(y)))
    excess = np.maximum(np.abs(x - y) - slack, 0.0)
    den = float(np.max(np.abs(y)))
    return float(np.max(excess) / den) if den > 0 else float(np.max(excess))


def normwise_err(x, ref) -> float:
    """max_i |x_i - ref_i| / max_i |ref_i| (error relative to the largest reference value)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if den == 0.0:
        return float(np.max(np.abs(x - ref))) if ref.size else 0.0
    return float(np.max(np.abs(x - ref)) / den)
