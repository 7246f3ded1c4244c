"""Numerical premise of the chunked prefill's tensor-core operand encoding (CPU only).

The chunked prefill computes its products (the decay-weighted Gram of the keys, X = T [βKΓ | βV],
[W; Q̃]·S and [K̄ᵀ; A_qk]·Ũ) on the tensor cores, while the recurrence is an FP32 one
("vsabavat/TensorRT-LLM pull request 1: NVFP4 Kimi K3 targets", Description: FP32 recurrence).
The kernels encode every FP32 operand x as two bf16 values, hi = bf16(x) and lo = bf16(x − hi),
and form hi·hi + hi·lo + lo·hi with FP32 accumulation (two MMA passes: A hi against [B hi | B lo],
then A lo against B hi).  This test emulates the chunk form with that encoding and with the
alternatives of the same or lower shared-memory cost: one TF32 pass (rounded to nearest, or the
low mantissa bits dropped) and TF32 with only the A operand split.  It checks that the
encoding the kernels use stays well inside the 1e-4 final-state bar of the parity tests while
the TF32 alternatives do not, on the prefill workload's value distributions (unit q and k after
SiLU, per-channel decay −e^{A_log}·softplus(f_b) with f_b of standard deviation 0.02·√128).
A TF32 form that passes needs three passes over 4-byte operands, twice the operand bytes that
bound these small-N products.
"""
from __future__ import annotations

import numpy as np
import pytest

STATE_BAR = 1e-4   # the final-state tolerance of the FP32 prefill parity tests
DK = DV = 128
CHUNK = 64


def _f32(x):
    return np.asarray(x, np.float32).astype(np.float64)


def _keep_bits(x, drop: int, nearest: bool):
    """FP32 value with the low `drop` mantissa bits cleared: rounded to nearest-even, or cut."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    if nearest:
        b = b + ((1 << (drop - 1)) - 1) + ((b >> drop) & 1)
    b = b & (0xFFFFFFFF ^ ((1 << drop) - 1))
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16(x):
    return _keep_bits(x, 16, True)


def tf32(x, nearest=True):
    return _keep_bits(x, 13, nearest)


def product(a, b, enc: str):
    """a @ b with both operands encoded as `enc`, products exact, sums in FP32 at the end."""
    if enc == "fp32":
        return _f32(_f32(a) @ _f32(b))
    if enc == "bf16_split":
        ah, bh = bf16(a), bf16(b)
        al, bl = bf16(a - ah), bf16(b - bh)
        return _f32(ah @ bh + ah @ bl + al @ bh)
    if enc == "tf32":
        return _f32(tf32(a) @ tf32(b))
    if enc == "tf32_cut":
        return _f32(tf32(a, False) @ tf32(b, False))
    if enc == "tf32_split_a":
        ah = tf32(a)
        return _f32(ah @ tf32(b) + tf32(a - ah) @ tf32(b))
    if enc == "tf32_split":
        ah, bh = tf32(a), tf32(b)
        al, bl = tf32(a - ah), tf32(b - bh)
        return _f32(ah @ bh + ah @ bl + al @ bh)
    raise ValueError(enc)


def workload(seed: int, L: int):
    rng = np.random.default_rng(seed)
    silu = lambda x: x / (1.0 + np.exp(-x))
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = unit(silu(rng.standard_normal((L, DK))))
    k = unit(silu(rng.standard_normal((L, DK))))
    v = silu(rng.standard_normal((L, DV)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    f_b = rng.normal(0.0, 0.02 * np.sqrt(128.0), size=(L, DK))
    log_alpha = -np.exp(rng.uniform(-1.0, 1.0)) * np.log1p(np.exp(f_b))
    return q, k, v, beta, log_alpha


def token_by_token(q, k, v, beta, log_alpha):
    """S_t = (I − β_t k_t k_tᵀ) diag(α_t) S_{t−1} + β_t k_t v_tᵀ, o_t = S_tᵀ q_t, in FP64."""
    S = np.zeros((DK, DV))
    out = np.empty((len(q), DV))
    for t in range(len(q)):
        S = np.exp(log_alpha[t])[:, None] * S
        S = S + beta[t] * np.outer(k[t], v[t] - k[t] @ S)
        out[t] = q[t] @ S
    return S, out


def chunked(q, k, v, beta, log_alpha, enc: str):
    """The chunk (WY) form with every contraction through `product`; the decay exponents are
    taken relative to the middle token of the chunk, the triangular solve in FP64 rounded to FP32.
    Entries above the diagonal of the Gram products may overflow; np.tril discards them, as the
    kernels' read-outs do."""
    S = np.zeros((DK, DV))
    out = np.empty((len(q), DV))
    with np.errstate(over="ignore", invalid="ignore"):
        for c0 in range(0, len(q), CHUNK):
            s = slice(c0, min(len(q), c0 + CHUNK))
            n = s.stop - s.start
            g = np.cumsum(log_alpha[s], axis=0)
            ref = g[n // 2]
            k_up, k_dn = k[s] * np.exp(g - ref), k[s] * np.exp(ref - g)
            A = np.tril(beta[s][:, None] * product(k_up, k_dn.T, enc), -1)
            A_qk = np.tril(product(q[s] * np.exp(g - ref), k_dn.T, enc))
            T = _f32(np.linalg.inv(np.eye(n) + A))
            R = np.concatenate([beta[s][:, None] * k[s] * np.exp(g), beta[s][:, None] * v[s]], axis=1)
            X = product(T, R, enc)
            W, U = X[:, :DK], X[:, DK:]
            WQ_S = product(np.concatenate([W, q[s] * np.exp(g)]), S, enc)
            U_t = _f32(U - WQ_S[:n])
            out[s] = _f32(WQ_S[n:] + product(A_qk, U_t, enc))
            S = _f32(np.exp(g[-1])[:, None] * S + product((k[s] * np.exp(g[-1] - g)).T, U_t, enc))
    return S, out


def rel(x, ref):
    return float(np.max(np.abs(x - ref)) / np.max(np.abs(ref)))


@pytest.fixture(scope="module", params=[0, 1])
def case(request):
    w = workload(request.param, 1024)
    return w, token_by_token(*w)


def test_fp32_chunk_form_equals_recurrence(case):
    """Control: with FP32 operands the chunk form reproduces the recurrence to FP32 rounding, so
    the errors below come from the operand encoding."""
    w, (S, out) = case
    S_c, out_c = chunked(*w, "fp32")
    assert rel(S_c, S) < 1e-6 and rel(out_c, out) < 1e-6


def test_bf16_split_meets_the_state_bar_with_margin(case):
    w, (S, out) = case
    S_c, out_c = chunked(*w, "bf16_split")
    assert rel(S_c, S) < STATE_BAR / 4
    assert rel(out_c, out) < STATE_BAR / 4


@pytest.mark.parametrize("enc", ["tf32", "tf32_cut", "tf32_split_a"])
def test_tf32_forms_of_equal_operand_bytes_miss_the_state_bar(case, enc):
    w, (S, _) = case
    S_c, _ = chunked(*w, enc)
    assert rel(S_c, S) > 2 * STATE_BAR


def test_three_pass_tf32_would_pass(case):
    """TF32 meets the bar only with three passes (twice the operand bytes of the bf16 split)."""
    w, (S, _) = case
    S_c, _ = chunked(*w, "tf32_split")
    assert rel(S_c, S) < 1e-6
