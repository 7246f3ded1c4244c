"""GPU variable-length prefill (kda_prefill_varlen) vs the token-by-token FP64 oracle.

Sequences of different lengths (zero, shorter than the conv window, ragged multi-chunk, exact
chunk multiples) are packed one after another and continue from slots holding a nonzero state
and conv window.  Each sequence is checked against the oracle's prefill of that sequence alone:
outputs within 2e-3 beyond the BF16 rounding, final FP32 state within 1e-4 (BF16 pools 5e-3),
final conv window bit-exact, every other slot untouched.  Equal lengths must reproduce
kda_prefill bit for bit, and inconsistent offsets are flagged and skipped.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from case_io import bf16_out_err, gathered_state, gathered_window, normwise_err, oracle_layer, storage_mode
from gpu_io import NAMES, bf16_bits, bf16_dev, bf16_vals, device_inputs, device_layer, device_pool, pool_state_host, pool_state_raw
from kda_inputs import bf16_bits_to_f32, make_prefill, to_bf16_bits

OUT_TOL = 2e-3
STATE_F32_TOL = 1e-4
STATE_BF16_TOL = 5e-3

pytestmark = pytest.mark.gpu


def varlen_case(seed, lens, H=3, dtype="f32", num_slots=None):
    B = len(lens)
    case = make_prefill(seed=seed, B=B, L=max(max(lens), 1), H=H,
                        num_slots=num_slots or B + 3, state_dtype=dtype, state_std=0.2,
                        random_conv=True, random_norm=True, random_dt_bias=True)
    # the sequences continue earlier prompts: nonzero conv windows in every slot
    rng = np.random.default_rng(seed + 1000)
    case.pool.conv[...] = to_bf16_bits(rng.standard_normal(case.pool.conv.shape, dtype=np.float32))
    packed = {n: np.ascontiguousarray(np.concatenate([case.inputs[n][b, :lens[b]] for b in range(B)], axis=0))
              for n in NAMES}
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return case, packed, cu


def run_varlen(case, packed, cu, max_len):
    import verify_kda_decode_gb300 as K

    layer, pool = device_layer(case), device_pool(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    ins = {n: bf16_dev(packed[n]) for n in NAMES}
    out = K.kda_prefill_varlen(layer, pool, slots, torch.from_numpy(cu).cuda(), max_len,
                               *(ins[n] for n in NAMES))
    torch.cuda.synchronize()
    return layer, pool, out, K.kda_get_error(pool)


def check_sequences(case, pool, out, cu, seqs):
    """Sequences `seqs` against the oracle's prefill of each alone."""
    L = oracle_layer(case)
    got = bf16_vals(out)
    st = pool_state_host(pool)
    tol = STATE_BF16_TOL if case.pool.state_dtype == "bf16" else STATE_F32_TOL
    for b in seqs:
        n = int(cu[b + 1] - cu[b])
        slot = case.slot_ids[b]
        S0 = gathered_state(case, [b])
        W0 = gathered_window(case, [b])
        got_w = bf16_bits_to_f32(bf16_bits(pool.conv_state[slot])).astype(np.float64).reshape(1, -1)
        if n == 0:
            np.testing.assert_array_equal(pool_state_raw(pool)[slot], case.pool.state[slot])
            np.testing.assert_array_equal(got_w, W0)
            continue
        ref_out, ref_S, ref_w = oracle.prefill(L, S0, W0, *(case.inputs[nm][b:b + 1, :n] for nm in NAMES),
                                               storage=storage_mode(case))
        e = bf16_out_err(got[cu[b]:cu[b + 1]], ref_out[0])
        assert e <= OUT_TOL, f"seq {b} (L={n}): output err {e:.3e}"
        e = normwise_err(st[slot], ref_S[0])
        assert e <= tol, f"seq {b} (L={n}): state err {e:.3e}"
        np.testing.assert_array_equal(got_w, ref_w)


def untouched_slots_keep_bytes(case, pool, skip=()):
    named = [s for b, s in enumerate(case.slot_ids) if b not in skip]
    untouched = np.setdiff1d(np.arange(case.pool.num_slots), named)
    np.testing.assert_array_equal(pool_state_raw(pool)[untouched], case.pool.state[untouched])
    np.testing.assert_array_equal(bf16_bits(pool.conv_state)[untouched], case.pool.conv[untouched])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_mixed_lengths_continue_from_slots(dtype):
    lens = [0, 1, 70, 200, 64, 2, 129]
    case, packed, cu = varlen_case(110, lens, dtype=dtype)
    layer, pool, out, err = run_varlen(case, packed, cu, max(lens))
    assert err == 0
    check_sequences(case, pool, out, cu, range(len(lens)))
    untouched_slots_keep_bytes(case, pool)


def test_varlen_loose_max_len_and_many_sequences():
    """max_len well above every length (extra prep CTAs exit at once); 12 short sequences."""
    lens = [5, 64, 1, 0, 33, 65, 7, 128, 2, 3, 90, 17]
    case, packed, cu = varlen_case(111, lens, H=2)
    layer, pool, out, err = run_varlen(case, packed, cu, 1000)
    assert err == 0
    check_sequences(case, pool, out, cu, range(len(lens)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_varlen_equal_lengths_is_prefill_bitwise(dtype):
    import verify_kda_decode_gb300 as K

    lens = [150, 150, 150]
    case, packed, cu = varlen_case(112, lens, dtype=dtype)
    layer, pool_a, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    out_a = K.kda_prefill(layer, pool_a, slots, *(ins[n] for n in NAMES))
    _, pool_b, out_b, err = run_varlen(case, packed, cu, 150)
    assert err == 0
    assert torch.equal(out_a.reshape(-1, out_a.shape[-1]).view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(pool_a.state.view(torch.int16), pool_b.state.view(torch.int16))
    assert torch.equal(pool_a.conv_state.view(torch.int16), pool_b.conv_state.view(torch.int16))


def test_varlen_inconsistent_offsets_flag_and_skip():
    import verify_kda_decode_gb300 as K

    lens = [5, 4, 7, 2]
    case, packed, _ = varlen_case(113, lens, H=2)
    # sequence 1 ends before it starts; sequence 2 starts before sequence 1's start
    cu = np.array([0, 5, 3, 10, 12], np.int32)
    packed = {n: np.ascontiguousarray(np.concatenate([case.inputs[n][0, :5], case.inputs[n][2, :5],
                                                      case.inputs[n][3, :2]], axis=0)) for n in NAMES}
    # rows: seq 0 = 0..4 (its own first 5 tokens), seq 3 = 10..11 (its own first 2 tokens)
    layer, pool, out, err = run_varlen(case, packed, cu, 8)
    assert err == K.kda.KDA_DEVERR_SEQLEN
    check_sequences(case, pool, out, cu, [0, 3])
    untouched_slots_keep_bytes(case, pool, skip=(1, 2))
    # a sequence longer than max_len is skipped, the others run
    lens = [9, 3]
    case, packed, cu = varlen_case(114, lens, H=2)
    layer, pool, out, err = run_varlen(case, packed, cu, 8)
    assert err == K.kda.KDA_DEVERR_SEQLEN
    check_sequences(case, pool, out, cu, [1])
    untouched_slots_keep_bytes(case, pool, skip=(0,))


def test_varlen_graph_replay_bitwise():
    """kda_prefill_varlen captured once in a CUDA graph and replayed twice (the second replay
    continuing from the states the first left) equals two eager calls bit for bit."""
    import verify_kda_decode_gb300 as K

    lens = [70, 0, 5, 130]
    case, packed, cu = varlen_case(115, lens, H=2)
    layer, ins = device_layer(case), {n: bf16_dev(packed[n]) for n in NAMES}
    slots = torch.from_numpy(case.slot_ids).cuda()
    cu_d = torch.from_numpy(cu).cuda()
    total, max_len = int(cu[-1]), 200
    ws = torch.empty(K.kda_prefill_varlen_workspace_size(layer, len(lens), total), dtype=torch.uint8, device="cuda")
    pool_e, pool_g = device_pool(case), device_pool(case)
    out_e = K.kda_prefill_varlen(layer, pool_e, slots, cu_d, max_len, *(ins[n] for n in NAMES), workspace=ws)
    out_e = K.kda_prefill_varlen(layer, pool_e, slots, cu_d, max_len, *(ins[n] for n in NAMES), workspace=ws)
    out_g = torch.empty_like(out_e)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            K.kda_prefill_varlen(layer, pool_g, slots, cu_d, max_len, *(ins[n] for n in NAMES), out=out_g, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_g) == 0
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16))
    assert torch.equal(pool_g.state, pool_e.state)
    assert torch.equal(pool_g.conv_state.view(torch.int16), pool_e.conv_state.view(torch.int16))
