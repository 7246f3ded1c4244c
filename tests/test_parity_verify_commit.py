"""GPU draft verify + commit vs the FP64 oracle.

Verify keeps the state in FP32 across the draft tokens whatever the storage dtype, so its
records are compared against the oracle's full-precision records at 1e-4 (error relative to
the largest value), outputs at 2e-3 beyond the BF16 output rounding, conv-window records
bit-exact.  Commit is checked bit for
bit against the oracle's commit applied to the GPU's own records (bit copy into an FP32 pool,
round-to-nearest-even into a BF16 pool), including every slot the call does not name.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from case_io import bf16_half_ulp, bf16_out_err, gathered_state, gathered_window, normwise_err, oracle_layer, storage_mode
from gpu_io import (NAMES, bf16_bits, bf16_vals, device_inputs, device_layer, device_pool,
                    pool_state_raw)
from kda_inputs import bf16_bits_to_f32, make, make_verify

OUT_TOL = 2e-3
REC_TOL = 1e-4

pytestmark = pytest.mark.gpu


def run_verify(case):
    import verify_kda_decode_gb300 as K

    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    out, rec, recw = K.kda_verify(layer, pool, slots, *(ins[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == 0
    return layer, pool, slots, out, rec, recw


def check_verify(case, sel=None):
    layer, pool, slots, out, rec, recw = run_verify(case)
    sel_idx = np.arange(case.B) if sel is None else np.asarray(sel)
    ins = [np.ascontiguousarray(case.inputs[n][sel_idx]) for n in NAMES]
    ref_out, ref_rec, ref_w = oracle.verify(oracle_layer(case), gathered_state(case, sel_idx),
                                            gathered_window(case, sel_idx), *ins)
    got_out = bf16_vals(out)[sel_idx]
    got_rec = rec.cpu().numpy().astype(np.float64)[sel_idx]
    T = case.inputs["q"].shape[1]
    for t in range(T):
        e = bf16_out_err(got_out[:, t], ref_out[:, t])
        assert e <= OUT_TOL, f"token {t}: output err {e:.3e}"
        e = normwise_err(got_rec[:, t], ref_rec[:, t])
        assert e <= REC_TOL, f"token {t}: record err {e:.3e}"
    got_w = bf16_bits_to_f32(bf16_bits(recw)).astype(np.float64)[sel_idx]
    np.testing.assert_array_equal(got_w.reshape(ref_w.shape), ref_w)
    # verify leaves the pool untouched
    np.testing.assert_array_equal(pool_state_raw(pool), case.pool.state)
    np.testing.assert_array_equal(bf16_bits(pool.conv_state), case.pool.conv)
    return layer, pool, slots, out, rec, recw


def check_commit(case, pool, slots, rec, recw, accepted):
    import verify_kda_decode_gb300 as K

    acc = torch.from_numpy(accepted).cuda()
    before_raw = pool_state_raw(pool)
    before_w = bf16_bits(pool.conv_state)
    K.kda_commit(pool, slots, acc, rec, recw)
    torch.cuda.synchronize()
    err = K.kda_get_error(pool)
    lw = case.layer
    exp_state, exp_w, rc = oracle.commit(lw.H, lw.dk, lw.dv, lw.K, storage_mode(case), before_raw,
                                         before_w.reshape(before_w.shape[0], -1), case.slot_ids,
                                         accepted, rec.cpu().numpy(),
                                         bf16_bits(recw).reshape(rec.shape[0], rec.shape[1], -1))
    np.testing.assert_array_equal(pool_state_raw(pool), exp_state)
    np.testing.assert_array_equal(bf16_bits(pool.conv_state).reshape(exp_w.shape), exp_w)
    return err, rc


def test_verify_b64_commit_full():
    """B=64, H=8, T=4, FP32 pool of 256 slots (seed 3): records, outputs, then commit of the
    drawn accepted lengths, bit-exact."""
    case = make("verify_b64")
    layer, pool, slots, out, rec, recw = check_verify(case)
    err, rc = check_commit(case, pool, slots, rec, recw, case.accepted)
    assert err == 0 and rc == 0


@pytest.mark.parametrize("T", [1, 3, 8, 11, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_commit_shapes(T, dtype):
    """T = 8 fills one 8-token projection chain exactly, T = 11 leaves a ragged second one."""
    case = make_verify(seed=60 + T, B=5, H=3, T=T, num_slots=11, state_dtype=dtype, state_std=0.2,
                       random_conv=True, random_norm=True, random_dt_bias=True)
    layer, pool, slots, out, rec, recw = check_verify(case)
    acc = case.accepted.copy()
    acc[0], acc[-1] = 0, T                      # both ends of the range
    err, rc = check_commit(case, pool, slots, rec, recw, acc)
    assert err == 0 and rc == 0


def test_commit_out_of_range_length_flags_and_skips():
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=70, B=4, H=2, T=4, num_slots=8, state_std=0.1)
    layer, pool, slots, out, rec, recw = run_verify(case)
    acc = np.array([2, 5, -1, 4], np.int32)          # 5 and -1 are out of range
    err, rc = check_commit(case, pool, slots, rec, recw, acc)
    assert err == K.kda.KDA_DEVERR_ACCEPTED and rc == 2


def test_commit_then_decode_continues_from_accepted_state():
    """After committing n of T draft tokens, the next decode starts from the record n-1: with
    FP32 storage its output equals the verify output of draft token n (same inputs) to one BF16
    rounding step plus 1e-5 of the largest output (verify projects f_b on the tensor cores,
    decode with FMA chains)."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=71, B=6, H=2, T=4, num_slots=9, state_std=0.1, random_conv=True)
    layer, pool, slots, out, rec, recw = run_verify(case)
    acc = np.array([1, 2, 3, 1, 2, 3], np.int32)
    K.kda_commit(pool, slots, torch.from_numpy(acc).cuda(), rec, recw)
    ins = device_inputs(case)
    idx = torch.from_numpy(acc).long().cuda()
    step = [ins[n][torch.arange(6, device="cuda"), idx].contiguous() for n in NAMES]
    o = K.kda_decode(layer, pool, slots, *step)
    torch.cuda.synchronize()
    ref = out[torch.arange(6, device="cuda"), idx]
    a, b = bf16_vals(o).astype(np.float64), bf16_vals(ref).astype(np.float64)
    assert np.all(np.abs(a - b) <= 2.0 * bf16_half_ulp(np.maximum(np.abs(a), np.abs(b))) + 1e-5 * np.max(np.abs(b)))


def test_verify_many_waves_sampled():
    """B*H = 960 tiles, three resident waves and more: each verify CTA prefetches the tile and
    window of the CTA one wave later at its start.  Sampled sequences against the oracle, then
    the commit of every sequence bit-exact."""
    case = make_verify(seed=75, B=120, H=8, T=2, num_slots=130, state_std=0.2, random_conv=True)
    layer, pool, slots, out, rec, recw = check_verify(case, sel=[0, 1, 59, 60, 118, 119])
    err, rc = check_commit(case, pool, slots, rec, recw, case.accepted)
    assert err == 0 and rc == 0
