"""Pins of the FP64 oracle to facts that do not come from the oracle itself.

The pages print no KDA values, so the oracle's absolute numbers cannot be pinned to them.
Instead each part is pinned by a closed form, an invariant, a special case that reduces to a
library routine (numpy / scipy / torch), brute force through a differently-written formula on
tiny inputs, or the recurrent-equals-chunked identity.  A dropped term, a wrong sign or index,
or a transposed operand in any step fails at least one test here.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from case_io import oracle_layer
from kda_inputs import bf16_bits_to_f32, make_decode, make_prefill, to_bf16_bits

RNG = np.random.default_rng(1234)
NEG_INF_BF16 = np.uint16(0xFF80)
POS_INF_BF16 = np.uint16(0x7F80)


def bits(x):
    return to_bf16_bits(np.asarray(x, np.float32))


def vals(b):
    return bf16_bits_to_f32(b).astype(np.float64)


# --------------------------------------------------------------------------- BF16 rounding

def test_bf16_rounding_matches_torch():
    """The oracle's RNE float32->BF16 equals torch's conversion (library routine), including
    ties, subnormals, the largest finite values and infinities."""
    x = RNG.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** RNG.integers(-30, 30, 20000).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130,
                     3.3895e38, 3.39e38, -3.4e38, 1e-45, 0.0, -0.0, np.inf, -np.inf], np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(x)
    np.testing.assert_array_equal(got, ref)


def test_store_round_matches_bf16_of_float32():
    x = RNG.standard_normal(5000).astype(np.float32)
    got = oracle.store_round(x.astype(np.float64), oracle.STORE_BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)
    got32 = oracle.store_round(np.array([1.0 + 2.0 ** -30, np.pi]), oracle.STORE_F32)
    np.testing.assert_array_equal(got32, np.array([1.0, np.float32(np.pi)], np.float64))


# --------------------------------------------------------------------------- FP8 input path

def test_e4m3_decoding_matches_torch():
    """The oracle's decoding of the FP8 E4M3 format equals torch's float8_e4m3fn conversion on
    all 256 codes (normal, subnormal, zero, the largest value 448, and the NaN codes)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_fp8_decay_against_dequantised_projection():
    """FP8 input path: the decay equals the plain formula with the projection done by numpy on
    W = scale_row * E4M3 code (codes decoded by torch)."""
    case = make_decode(seed=17, B=1, H=2, n_steps=1, dk=8, dv=8, r=16, random_dt_bias=True, fp8_w_fb=True)
    lw = case.layer
    L = oracle_layer(case)
    W = lw.W_fb_scale.astype(np.float64)[:, None] * torch.from_numpy(lw.W_fb_fp8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    f_a = vals(case.inputs["f_a"][0, 0])
    for h in range(2):
        sl = slice(h * 8, (h + 1) * 8)
        graw = W[sl] @ f_a + lw.dt_bias[sl]
        ref = np.exp(-np.exp(np.float64(lw.A_log[h])) * np.logaddexp(0.0, graw))
        np.testing.assert_allclose(oracle.decay(L, h, case.inputs["f_a"][0, 0]), ref, rtol=1e-13)
    # and it differs from the BF16 weights' decay (the FP8 path is really taken)
    L16 = oracle_layer(case)
    L16.W_fb8 = L16.W_fb_scale = None
    assert not np.allclose(oracle.decay(L16, 0, case.inputs["f_a"][0, 0]), oracle.decay(L, 0, case.inputs["f_a"][0, 0]), rtol=0, atol=0)


# --------------------------------------------------------------------------- recurrence a6

def test_recurrence_beta0_alpha1_leaves_state_unchanged():
    S0 = RNG.standard_normal((7, 5))
    q, k = RNG.standard_normal(7), RNG.standard_normal(7)
    v = RNG.standard_normal(5)
    S1, o = oracle.recurrence_step(S0, np.ones(7), k, v, q, 0.0)
    np.testing.assert_array_equal(S1, S0)
    np.testing.assert_allclose(o, S0.T @ q, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("seed", range(5))
def test_recurrence_beta1_unit_key_writes_value(seed):
    """After a beta = 1 update with a unit key, S^T k = v exactly (delta rule), whatever the decay."""
    rng = np.random.default_rng(seed)
    dk, dv = 6, 4
    S0 = rng.standard_normal((dk, dv))
    k = rng.standard_normal(dk)
    k /= np.linalg.norm(k)
    alpha = rng.uniform(0.1, 1.0, dk)
    v, q = rng.standard_normal(dv), rng.standard_normal(dk)
    S1, _ = oracle.recurrence_step(S0, alpha, k, v, q, 1.0)
    np.testing.assert_allclose(S1.T @ k, v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_recurrence_matches_projection_form(seed):
    """Brute force with dk != dv: S' = (I - beta k k^T) Diag(alpha) S + beta k v^T, o = S'^T q."""
    rng = np.random.default_rng(100 + seed)
    dk, dv = 3, 5
    S0 = rng.standard_normal((dk, dv))
    k, q = rng.standard_normal(dk), rng.standard_normal(dk)
    v = rng.standard_normal(dv)
    alpha = rng.uniform(0.05, 1.0, dk)
    beta = float(rng.uniform(0, 1))
    P = np.eye(dk) - beta * np.outer(k, k)
    S_ref = P @ np.diag(alpha) @ S0 + beta * np.outer(k, v)
    S1, o = oracle.recurrence_step(S0, alpha, k, v, q, beta)
    np.testing.assert_allclose(S1, S_ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, S_ref.T @ q, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- a1, a2: decay

def test_decay_half_when_projection_is_zero():
    """W_fb = 0, dt_bias = 0, A_log = 0 => g = -softplus(0) = -ln 2, alpha = 1/2."""
    case = make_decode(seed=5, B=1, H=2, n_steps=1, dk=8, dv=8, r=4)
    case.layer.W_fb[:] = 0
    case.layer.A_log[:] = 0
    L = oracle_layer(case)
    alpha = oracle.decay(L, 1, case.inputs["f_a"][0, 0])
    np.testing.assert_allclose(alpha, 0.5, rtol=1e-15)


def test_decay_against_library_softplus():
    case = make_decode(seed=6, B=1, H=3, n_steps=1, dk=8, dv=8, r=16, random_dt_bias=True)
    L = oracle_layer(case)
    fa = case.inputs["f_a"][0, 0]
    W = vals(case.layer.W_fb)
    for h in range(3):
        graw = W[h * 8:(h + 1) * 8] @ vals(fa)
        g = -np.exp(np.float64(case.layer.A_log[h])) * np.logaddexp(0.0, graw + case.layer.dt_bias[h * 8:(h + 1) * 8])
        np.testing.assert_allclose(oracle.decay(L, h, fa), np.exp(g), rtol=1e-13)


# --------------------------------------------------------------------------- a4: conv

def test_conv_identity_tap_is_silu():
    w = bits([0, 0, 0, 1])
    x = bits(RNG.standard_normal(20))
    y, _ = oracle.conv_sequence(w, np.zeros(3), x)
    xv = vals(x)
    np.testing.assert_allclose(y, xv * expit(xv), rtol=1e-15)


def test_conv_impulse_reproduces_taps():
    w = bits(RNG.uniform(-0.5, 0.5, 4))
    x = bits([1, 0, 0, 0, 0, 0])
    y, _ = oracle.conv_sequence(w, np.zeros(3), x)
    pre = np.concatenate([vals(w)[::-1], [0, 0]])  # tap K-1 multiplies the current token
    np.testing.assert_allclose(y, pre * expit(pre), rtol=1e-15)


def test_conv_matches_numpy_convolve_with_window():
    w = bits(RNG.uniform(-0.5, 0.5, 4))
    w0 = vals(bits(RNG.standard_normal(3)))
    x = bits(RNG.standard_normal(50))
    y, w_end = oracle.conv_sequence(w, w0, x)
    full = np.concatenate([w0, vals(x)])
    pre = np.convolve(full, vals(w)[::-1], mode="valid")
    np.testing.assert_allclose(y, pre * expit(pre), rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(w_end, vals(x)[-3:])
    # split into two calls: the window carries the history
    y1, we1 = oracle.conv_sequence(w, w0, x[:17])
    y2, _ = oracle.conv_sequence(w, we1, x[17:])
    np.testing.assert_array_equal(np.concatenate([y1, y2]), y)


# --------------------------------------------------------------------------- a5, a7

def test_l2_norms():
    q, k = RNG.standard_normal(16), RNG.standard_normal(16)
    qn, kn = oracle.l2_norms(q, k, 0.0)
    np.testing.assert_allclose(np.linalg.norm(kn), 1.0, rtol=1e-15)
    np.testing.assert_allclose(np.linalg.norm(qn), 0.25, rtol=1e-15)   # 1/sqrt(16)
    np.testing.assert_allclose(kn, k / np.linalg.norm(k), rtol=1e-15)
    qe, _ = oracle.l2_norms(np.full(4, 1e-4), np.full(4, 1e-4), 1e-6)
    np.testing.assert_allclose(qe, 1e-4 / np.sqrt(4e-8 + 1e-6) / 2.0, rtol=1e-14)


def test_gated_rmsnorm_constant_and_random():
    gate = bits([0.0] * 6)
    y = oracle.gated_rmsnorm(np.full(6, -3.0), np.arange(1, 7, dtype=np.float64), 0.0, gate)
    np.testing.assert_allclose(y, -0.5 * np.arange(1, 7), rtol=1e-15)
    o = RNG.standard_normal(32)
    w = RNG.uniform(0.5, 1.5, 32)
    g = bits(RNG.standard_normal(32))
    y = oracle.gated_rmsnorm(o, w, 1e-5, g)
    rms = np.sqrt(np.mean(np.square(o)) + 1e-5)
    np.testing.assert_allclose(y, o / rms * w * expit(vals(g)), rtol=1e-14)


# --------------------------------------------------------------------------- whole step, brute force

def _bruteforce_decode(case, n_steps):
    """Every step written with library primitives and the projection form of the update."""
    lw = case.layer
    H, dk, dv, K = lw.H, lw.dk, lw.dv, lw.K
    W = vals(lw.W_fb)
    cw = vals(lw.conv_w)                      # [3, H*dk, K]
    S = np.zeros((H, dk, dv))
    hist = {n: np.zeros((K - 1, H * dk)) for n in ("q", "k", "v")}
    outs = []
    for s in range(n_steps):
        inp = {n: vals(case.inputs[n][s, 0]) for n in ("q", "k", "v", "f_a", "beta", "gate")}
        conv = {}
        for ti, n in enumerate(("q", "k", "v")):
            seq = np.vstack([hist[n], inp[n][None]])          # [K, C], oldest first
            pre = np.einsum("kc,ck->c", seq, cw[ti])
            conv[n] = pre * expit(pre)
            hist[n] = seq[1:]
        y = np.zeros(H * dv)
        for h in range(H):
            sl = slice(h * dk, (h + 1) * dk)
            graw = W[sl] @ inp["f_a"] + lw.dt_bias[sl]
            alpha = np.exp(-np.exp(np.float64(lw.A_log[h])) * np.logaddexp(0.0, graw))
            k = conv["k"][sl] / np.sqrt(np.sum(conv["k"][sl] ** 2) + lw.l2_eps)
            q = conv["q"][sl] / np.sqrt(np.sum(conv["q"][sl] ** 2) + lw.l2_eps) / np.sqrt(dk)
            v = conv["v"][h * dv:(h + 1) * dv]
            beta = expit(inp["beta"][h])
            S[h] = (np.eye(dk) - beta * np.outer(k, k)) @ np.diag(alpha) @ S[h] + beta * np.outer(k, v)
            o = S[h].T @ q
            g = inp["gate"][h * dv:(h + 1) * dv]
            y[h * dv:(h + 1) * dv] = o / np.sqrt(np.mean(o ** 2) + lw.norm_eps) * lw.norm_w * expit(g)
        outs.append(y)
    return np.array(outs), S


def test_full_step_bruteforce_tiny():
    case = make_decode(seed=7, B=1, H=2, n_steps=6, dk=4, dv=4, r=5, random_norm=True,
                       random_dt_bias=True)
    L = oracle_layer(case)
    wl = L.window_len()
    out, S, _ = oracle.decode(L, np.zeros((1, 2, 4, 4)), np.zeros((1, wl)), *(case.inputs[n] for n in ("q", "k", "v", "f_a", "beta", "gate")))
    ref_out, ref_S = _bruteforce_decode(case, 6)
    np.testing.assert_allclose(out[:, 0], ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S[0], ref_S, rtol=1e-12, atol=1e-12)


def test_decode_beta0_closed_form():
    """beta = 0 (logit -inf): the state only decays, S_t = Diag(prod alpha) S0, so each output is
    the gated RMSNorm of (Diag(prod alpha) S0)^T q_t."""
    case = make_decode(seed=8, B=1, H=2, n_steps=5, dk=8, dv=6, r=8, state_std=0.5,
                       random_conv=True)
    case.inputs["beta"][:] = NEG_INF_BF16
    L = oracle_layer(case)
    S0 = case.pool.state[case.slot_ids].astype(np.float64)
    win0 = bf16_bits_to_f32(case.pool.conv[case.slot_ids]).astype(np.float64).reshape(1, -1)
    ins = [case.inputs[n] for n in ("q", "k", "v", "f_a", "beta", "gate")]
    out, S, _ = oracle.decode(L, S0, win0, *ins)
    cumalpha = np.ones((2, 8))
    for s in range(5):
        for h in range(2):
            cumalpha[h] *= oracle.decay(L, h, case.inputs["f_a"][s, 0])
    np.testing.assert_allclose(S[0], cumalpha[:, :, None] * S0[0], rtol=1e-13)


def test_alpha1_beta0_state_bitwise_unchanged():
    case = make_decode(seed=9, B=2, H=2, n_steps=4, dk=8, dv=8, r=8, state_std=0.3, num_slots=2)
    case.inputs["beta"][:] = NEG_INF_BF16
    case.layer.A_log[:] = -np.inf                      # exp(A_log) = 0 => g = 0, alpha = 1
    L = oracle_layer(case)
    S0 = case.pool.state[case.slot_ids].astype(np.float64)
    win0 = np.zeros((2, L.window_len()))
    out, S, _ = oracle.decode(L, S0, win0, *(case.inputs[n] for n in ("q", "k", "v", "f_a", "beta", "gate")))
    np.testing.assert_array_equal(S, S0)


# --------------------------------------------------------------------------- forms agree

def _ins(case):
    return [case.inputs[n] for n in ("q", "k", "v", "f_a", "beta", "gate")]


def test_verify_records_equal_decode_steps():
    case = make_decode(seed=10, B=3, H=2, n_steps=5, dk=8, dv=8, r=8, state_std=0.2, num_slots=5,
                       random_conv=True)
    L = oracle_layer(case)
    S0 = case.pool.state[case.slot_ids].astype(np.float64)
    w0 = bf16_bits_to_f32(case.pool.conv[case.slot_ids]).astype(np.float64).reshape(3, -1)
    ins = _ins(case)
    outs, recs, recw = oracle.verify(L, S0, w0, *[np.ascontiguousarray(np.swapaxes(a, 0, 1)) for a in ins])
    for t in range(1, 6):
        o_d, S_d, w_d = oracle.decode(L, S0, w0, *[a[:t] for a in ins])
        np.testing.assert_array_equal(recs[:, t - 1], S_d)
        np.testing.assert_array_equal(recw[:, t - 1], w_d)
        np.testing.assert_array_equal(outs[:, t - 1], o_d[t - 1])


def test_prefill_equals_decode_loop():
    case = make_prefill(seed=11, B=2, L=9, H=2, dk=8, dv=8, r=8, random_conv=True, state_std=0.1)
    L = oracle_layer(case)
    S0 = case.pool.state[case.slot_ids].astype(np.float64)
    w0 = bf16_bits_to_f32(case.pool.conv[case.slot_ids]).astype(np.float64).reshape(2, -1)
    ins = _ins(case)
    out_p, S_p, w_p = oracle.prefill(L, S0, w0, *ins)
    out_d, S_d, w_d = oracle.decode(L, S0, w0, *[np.ascontiguousarray(np.swapaxes(a, 0, 1)) for a in ins])
    np.testing.assert_array_equal(out_p, np.swapaxes(out_d, 0, 1))
    np.testing.assert_array_equal(S_p, S_d)
    np.testing.assert_array_equal(w_p, w_d)


@pytest.mark.parametrize("storage", [oracle.STORE_F32, oracle.STORE_BF16])
def test_decode_rounds_state_to_storage_after_every_step(storage):
    """FP32 recurrence with FP32 or BF16 storage between steps: an n-step decode with a storage
    dtype equals n one-step decodes in full precision with the storage rounding (pinned above
    against torch) applied to the state between them, and to nothing else.  Rounding only at
    the end, never, or to the wrong dtype breaks the equality."""
    case = make_decode(seed=14, B=2, H=2, n_steps=5, dk=8, dv=8, r=8, state_std=0.4, num_slots=3,
                       random_conv=True, random_norm=True)
    L = oracle_layer(case)
    S0 = oracle.store_round(case.pool.state[case.slot_ids].astype(np.float64), storage)
    w0 = bf16_bits_to_f32(case.pool.conv[case.slot_ids]).astype(np.float64).reshape(2, -1)
    ins = _ins(case)
    out_n, S_n, w_n = oracle.decode(L, S0, w0, *ins, storage=storage)
    S, w = S0, w0
    for s in range(5):
        o1, S, w = oracle.decode(L, S, w, *[a[s:s + 1] for a in ins], storage=oracle.STORE_F64)
        S = oracle.store_round(S, storage)
        np.testing.assert_array_equal(out_n[s], o1[0])
    np.testing.assert_array_equal(S_n, S)
    np.testing.assert_array_equal(w_n, w)
    # the rounding is not a no-op on these values (so the equality above sees where it falls)
    _, S_full, _ = oracle.decode(L, S0, w0, *ins, storage=oracle.STORE_F64)
    assert not np.array_equal(oracle.store_round(S_full, storage), S_n)


@pytest.mark.parametrize("storage", [oracle.STORE_F32, oracle.STORE_BF16])
def test_prefill_rounds_state_to_storage_once_at_the_end(storage):
    """Prefill keeps the state in full precision across its tokens and rounds it to the storage
    dtype once, at the end: outputs equal the full-precision prefill's exactly, and the final
    state is the storage rounding of the full-precision final state."""
    case = make_prefill(seed=15, B=2, L=11, H=2, dk=8, dv=8, r=8, random_conv=True, state_std=0.3)
    L = oracle_layer(case)
    S0 = oracle.store_round(case.pool.state[case.slot_ids].astype(np.float64), storage)
    w0 = bf16_bits_to_f32(case.pool.conv[case.slot_ids]).astype(np.float64).reshape(2, -1)
    ins = _ins(case)
    out_s, S_s, w_s = oracle.prefill(L, S0, w0, *ins, storage=storage)
    out_f, S_f, w_f = oracle.prefill(L, S0, w0, *ins, storage=oracle.STORE_F64)
    np.testing.assert_array_equal(out_s, out_f)
    np.testing.assert_array_equal(S_s, oracle.store_round(S_f, storage))
    np.testing.assert_array_equal(w_s, w_f)
    assert not np.array_equal(S_s, S_f)


@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
@pytest.mark.parametrize("strong_decay", [False, True])
def test_recurrent_equals_chunked(chunk, strong_decay):
    case = make_prefill(seed=12, B=2, L=77, H=2, dk=16, dv=12, r=8, state_std=0.3,
                        random_conv=True, random_norm=True, random_dt_bias=True)
    if strong_decay:
        case.layer.A_log[:] = np.float32(1.5)          # per-token log-decay around -3
    L = oracle_layer(case)
    S0 = case.pool.state[case.slot_ids].astype(np.float64)
    w0 = bf16_bits_to_f32(case.pool.conv[case.slot_ids]).astype(np.float64).reshape(2, -1)
    ins = _ins(case)
    out_r, S_r, w_r = oracle.prefill(L, S0, w0, *ins)
    out_c, S_c, w_c = oracle.prefill_chunked(L, S0, w0, *ins, chunk=chunk)
    np.testing.assert_allclose(out_c, out_r, rtol=0, atol=1e-10 * np.abs(out_r).max())
    np.testing.assert_allclose(S_c, S_r, rtol=0, atol=1e-10 * np.abs(S_r).max())
    np.testing.assert_array_equal(w_c, w_r)


# --------------------------------------------------------------------------- commit

@pytest.mark.parametrize("storage", [oracle.STORE_F32, oracle.STORE_BF16])
def test_commit_copies_accepted_record(storage):
    rng = np.random.default_rng(13)
    B, T, H, dk, dv, K, slots = 5, 4, 2, 4, 4, 4, 9
    wl = (K - 1) * 3 * H * dk
    if storage == oracle.STORE_F32:
        pool = rng.standard_normal((slots, H, dk, dv)).astype(np.float32)
    else:
        pool = bits(rng.standard_normal((slots, H, dk, dv)))
    pool_w = bits(rng.standard_normal((slots, wl)))
    ids = rng.permutation(slots)[:B].astype(np.int32)
    acc = np.array([0, 1, 4, 2, 3], np.int32)
    rec = rng.standard_normal((B, T, H, dk, dv)).astype(np.float32)
    rec_w = bits(rng.standard_normal((B, T, wl)))
    new, new_w, rc = oracle.commit(H, dk, dv, K, storage, pool, pool_w, ids, acc, rec, rec_w)
    assert rc == 0
    exp, exp_w = pool.copy(), pool_w.copy()
    for b in range(B):
        if acc[b] == 0:
            continue
        src = rec[b, acc[b] - 1]
        exp[ids[b]] = src if storage == oracle.STORE_F32 else torch.from_numpy(src).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        exp_w[ids[b]] = rec_w[b, acc[b] - 1]
    np.testing.assert_array_equal(new, exp)
    np.testing.assert_array_equal(new_w, exp_w)
    # out-of-range accepted length or slot id: reported, that sequence left alone
    bad_acc = acc.copy()
    bad_acc[2] = T + 1
    new2, _, rc2 = oracle.commit(H, dk, dv, K, storage, pool, pool_w, ids, bad_acc, rec, rec_w)
    assert rc2 == 2
    np.testing.assert_array_equal(new2[ids[2]], pool[ids[2]])
