"""GPU prefill vs the token-by-token FP64 oracle.

Outputs at every token within 2e-3 beyond the BF16 output rounding and the final FP32 state within 1e-4 (errors relative to
the largest reference value, per sequence); final conv window bit-exact; other slots untouched.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from case_io import bf16_out_err, bf16_pair_err, gathered_state, gathered_window, normwise_err, oracle_layer, storage_mode
from gpu_io import NAMES, bf16_bits, bf16_vals, device_inputs, device_layer, device_pool, pool_state_host, pool_state_raw
from kda_inputs import bf16_bits_to_f32, make, make_prefill

OUT_TOL = 2e-3
STATE_F32_TOL = 1e-4
STATE_BF16_TOL = 5e-3

pytestmark = pytest.mark.gpu


def check_prefill(case):
    import verify_kda_decode_gb300 as K

    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    out = K.kda_prefill(layer, pool, slots, *(ins[n] for n in NAMES), chunk=case.chunk)
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == 0
    ref_out, ref_S, ref_w = oracle.prefill(oracle_layer(case), gathered_state(case),
                                           gathered_window(case), *(case.inputs[n] for n in NAMES),
                                           storage=storage_mode(case))
    got = bf16_vals(out)
    st = pool_state_host(pool)[case.slot_ids]
    tol = STATE_BF16_TOL if case.pool.state_dtype == "bf16" else STATE_F32_TOL
    for b in range(case.B):
        e = bf16_out_err(got[b], ref_out[b])
        assert e <= OUT_TOL, f"seq {b}: output err {e:.3e}"
        e = normwise_err(st[b], ref_S[b])
        assert e <= tol, f"seq {b}: state err {e:.3e}"
    got_w = bf16_bits_to_f32(bf16_bits(pool.conv_state)).astype(np.float64)[case.slot_ids]
    np.testing.assert_array_equal(got_w.reshape(case.B, -1), ref_w)
    untouched = np.setdiff1d(np.arange(case.pool.num_slots), case.slot_ids)
    if untouched.size:
        np.testing.assert_array_equal(pool_state_raw(pool)[untouched], case.pool.state[untouched])
    return out


def test_prefill_b4_full():
    """B=4, L=4096, H=8, chunk 64, FP32 state from zero (seed 4), checked against the
    token-by-token recurrence at every token."""
    check_prefill(make("prefill_b4"))


@pytest.mark.parametrize("L", [1, 63, 64, 65, 150, 200])
def test_prefill_ragged_lengths(L):
    """One chunk, exact chunks, and 2, 3 and 4 chunks with a ragged last one (the scan alternates
    its output accumulator from chunk to chunk and reads a chunk's outputs during the next)."""
    case = make_prefill(seed=80 + L, B=3, L=L, H=2, num_slots=5, state_std=0.2, random_conv=True,
                        random_norm=True, random_dt_bias=True)
    check_prefill(case)


def test_prefill_more_clusters_than_fit_at_once():
    """B x H = 80 (sequence, head) pairs: 80 clusters of four scan CTAs, about twice what one
    GB300 holds at once, so the clusters run in more than one wave (each on its own pair)."""
    case = make_prefill(seed=95, B=10, L=130, H=8, num_slots=12, state_std=0.2, random_conv=True)
    check_prefill(case)


@pytest.mark.parametrize("a_log", [(-2.0, -2.0), (1.9, 1.9), (-2.0, 1.9)])
def test_prefill_weak_and_strong_decay(a_log):
    """Weak decay keeps a chunk's log-decay within the one-reference range of the Gram staging;
    strong decay (|log alpha| ~ 4.6 per token) takes the per-block form (block-boundary
    references below the diagonal, exact exponent differences on it).  Both forms, and both in
    one launch (one head of each), against the oracle."""
    case = make_prefill(seed=95, B=2, L=200, H=2, num_slots=4, state_std=0.2, random_conv=True)
    case.layer.A_log[:] = np.array(a_log, np.float32)
    check_prefill(case)


def test_prefill_bf16_pool_from_existing_state():
    case = make_prefill(seed=90, B=2, L=150, H=3, num_slots=4, state_dtype="bf16", state_std=0.2,
                        random_conv=True)
    check_prefill(case)


def test_prefill_then_decode_matches_longer_prefill():
    """Prefill of L tokens followed by one decode equals prefill of L+1 tokens (FP32 pool)."""
    import verify_kda_decode_gb300 as K

    case = make_prefill(seed=91, B=2, L=97, H=2, num_slots=4, state_std=0.0)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_a = device_pool(case)
    out_a = K.kda_prefill(layer, pool_a, slots, *(ins[n] for n in NAMES))
    pool_b = device_pool(case)
    K.kda_prefill(layer, pool_b, slots, *(ins[n][:, :96].contiguous() for n in NAMES))
    o = K.kda_decode(layer, pool_b, slots, *(ins[n][:, 96].contiguous() for n in NAMES))
    torch.cuda.synchronize()
    ref = bf16_vals(out_a[:, 96])
    # both sides are BF16-rounded: a rounding that falls the other way costs up to one ulp
    assert bf16_pair_err(bf16_vals(o), ref) <= OUT_TOL
    assert normwise_err(pool_state_host(pool_b), pool_state_host(pool_a)) <= STATE_F32_TOL


# softplus(W_fb . f_a + 0) is about log 2 for these weights, so A_log = log(x / log 2) gives a
# per-token log-decay of about -x
def _a_log_for(x):
    return np.float32(np.log(x / np.log(2.0)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("neg_log_decay", [12.0, 40.0])
def test_prefill_very_strong_decay(neg_log_decay, dtype):
    """Per-token log-decay around -12 and -40 (alpha ~ 6e-6 and 4e-18): any decay the method
    can produce is handled, with no range limit, against the token-by-token oracle; the second
    head decays weakly in the same launch."""
    case = make_prefill(seed=96, B=2, L=200, H=2, num_slots=4, state_dtype=dtype, state_std=0.2,
                        random_conv=True)
    case.layer.A_log[:] = np.array([_a_log_for(neg_log_decay), -2.0], np.float32)
    check_prefill(case)


def test_prefill_decay_spread_over_channels():
    """Channels of one head from almost no decay to log-decay ~ -53 per token (dt_bias spread
    over [-6, 3]): within every chunk the fast channels span thousands in log-decay while the
    slow ones stay near zero."""
    case = make_prefill(seed=97, B=2, L=300, H=2, num_slots=4, state_std=0.2, random_conv=True)
    rng = np.random.default_rng(97)
    case.layer.A_log[:] = _a_log_for(12.0)
    case.layer.dt_bias[:] = rng.uniform(-6.0, 3.0, case.layer.dt_bias.shape).astype(np.float32)
    check_prefill(case)


def test_prefill_nonfinite_decay_sets_the_decay_flag():
    """A non-finite log-decay (here from a NaN f_a row made on the host) is the one case the
    chunked form reports: KDA_DEVERR_DECAY, read and cleared by kda_get_error."""
    import verify_kda_decode_gb300 as K

    case = make_prefill(seed=98, B=1, L=70, H=2, num_slots=2)
    case.inputs["f_a"][0, 5, :] = np.uint16(0x7FC0)     # BF16 quiet NaN
    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    K.kda_prefill(layer, pool, slots, *(ins[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) & K.kda.KDA_DEVERR_DECAY
    assert K.kda_get_error(pool) == 0
