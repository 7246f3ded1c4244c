"""GPU decode vs the FP64 oracle, element by element, on the same seeded inputs.

Tolerances (error relative to the largest reference value of the tensor):
  outputs (BF16)              2e-3  against the unrounded FP64 oracle, beyond the output
                                    rounding itself: rounding to BF16 moves a value by up to
                                    half a BF16 spacing (2^-8 = 3.9e-3 of the value), which no
                                    BF16 result avoids, so each element gets that much slack
                                    first (case_io.bf16_out_err).  FP32 arithmetic adds ~1e-6.
  state, FP32 storage         1e-4  against the oracle with FP32 storage rounding per step.
  state, BF16 storage         5e-3  against the oracle with BF16 storage rounding per step
                                    (one BF16 ulp is 2^-8 = 3.9e-3 of a value; a rounding that
                                    falls the other way on the GPU than in FP64 costs one ulp).
  conv windows, slot mapping  bit-exact (the window holds copies of the BF16 inputs; slots
                                    not named in the call keep their bytes).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from case_io import (bf16_half_ulp, bf16_out_err, gathered_state, gathered_window, normwise_err, oracle_layer,
                     storage_mode)
from gpu_io import (NAMES, bf16_bits, bf16_vals, device_inputs, device_layer, device_pool,
                    pool_state_host, pool_state_raw)
from kda_inputs import bf16_bits_to_f32, make, make_decode

OUT_TOL = 2e-3
STATE_F32_TOL = 1e-4
STATE_BF16_TOL = 5e-3

pytestmark = pytest.mark.gpu


def run_decode_gpu(case, n_steps=None):
    import verify_kda_decode_gb300 as K

    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    n_steps = ins["q"].shape[0] if n_steps is None else n_steps
    outs = []
    for s in range(n_steps):
        outs.append(K.kda_decode(layer, pool, slots, *(ins[n][s] for n in NAMES)))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == 0
    return pool, torch.stack(outs)


def run_decode_oracle(case, n_steps=None, sel=None):
    L = oracle_layer(case)
    ins = [case.inputs[n] for n in NAMES]
    if n_steps is not None:
        ins = [a[:n_steps] for a in ins]
    if sel is not None:
        ins = [np.ascontiguousarray(a[:, sel]) for a in ins]
    return oracle.decode(L, gathered_state(case, sel), gathered_window(case, sel), *ins,
                         storage=storage_mode(case))


def check_decode(case, n_steps=None, sel=None):
    pool, outs = run_decode_gpu(case, n_steps)
    sel_idx = np.arange(case.B) if sel is None else np.asarray(sel)
    ref_out, ref_S, ref_w = run_decode_oracle(case, n_steps, None if sel is None else sel_idx)
    got_out = bf16_vals(outs)[:, sel_idx]
    for s in range(got_out.shape[0]):
        e = bf16_out_err(got_out[s], ref_out[s])
        assert e <= OUT_TOL, f"step {s}: output err {e:.3e}"
    st = pool_state_host(pool)
    got_S = st[case.slot_ids[sel_idx]]
    tol = STATE_BF16_TOL if case.pool.state_dtype == "bf16" else STATE_F32_TOL
    e = normwise_err(got_S, ref_S)
    assert e <= tol, f"state err {e:.3e}"
    got_w = bf16_bits_to_f32(bf16_bits(pool.conv_state)).astype(np.float64)[case.slot_ids[sel_idx]]
    np.testing.assert_array_equal(got_w.reshape(len(sel_idx), -1), ref_w)
    # slots not named by the call keep their bytes
    untouched = np.setdiff1d(np.arange(case.pool.num_slots), case.slot_ids)
    if untouched.size:
        raw = pool_state_raw(pool)
        np.testing.assert_array_equal(raw[untouched], case.pool.state[untouched])
        np.testing.assert_array_equal(bf16_bits(pool.conv_state)[untouched], case.pool.conv[untouched])
    return pool, outs


def test_decode_small_full():
    """1 sequence, H=2, 8 steps, FP32 state from zero (seed 0)."""
    check_decode(make("decode_small"))


def test_decode_b64_full():
    """B=64, H=8, FP32 pool of 256 slots, 64 steps (seed 1)."""
    check_decode(make("decode_b64"))


def test_decode_b256_bf16_full():
    """B=256, H=32, BF16 pool of 512 slots, 16 steps (seed 2): every sequence, head and step
    against the oracle, and the untouched slots bit for bit."""
    check_decode(make("decode_b256"))


@pytest.mark.parametrize("H,B,slots", [(1, 3, 7), (3, 5, 5), (5, 1, 9)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_ragged_shapes_random_extras(H, B, slots, dtype):
    case = make_decode(seed=40 + H, B=B, H=H, n_steps=6, num_slots=slots, state_dtype=dtype,
                       state_std=0.2, random_conv=True, random_norm=True, random_dt_bias=True)
    check_decode(case)


def test_decode_zero_batch_is_noop():
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=50, B=2, H=2, n_steps=1, num_slots=4, state_std=0.1)
    layer, pool = device_layer(case), device_pool(case)
    before = pool.state.clone()
    e = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    K.kda_decode(layer, pool, torch.empty(0, dtype=torch.int32, device="cuda"), e, e, e,
                 torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"),
                 torch.empty(0, 2, dtype=torch.bfloat16, device="cuda"), e)
    torch.cuda.synchronize()
    assert torch.equal(before, pool.state)


def test_decode_bad_slot_sets_error_and_skips_tile():
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=51, B=3, H=2, n_steps=1, num_slots=4, state_std=0.1)
    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.tensor([1, 4, -1], dtype=torch.int32, device="cuda")   # 4 and -1 are out of range
    before = pool.state.clone()
    K.kda_decode(layer, pool, slots, *(ins[n][0] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == K.kda.KDA_DEVERR_SLOT
    assert K.kda_get_error(pool) == 0          # read-and-clear
    assert torch.equal(before[[0, 2, 3]], pool.state[[0, 2, 3]])
    assert not torch.equal(before[1], pool.state[1])


def within_one_bf16_step(x, y):
    """BF16 outputs of values that differ by FP32 rounding: each pair at most one BF16 rounding
    step apart, plus 1e-5 of the largest output (near zero a BF16 step is finer than the FP32
    differences of the unnormalised values)."""
    a = x.float().cpu().numpy().astype(np.float64)
    b = y.float().cpu().numpy().astype(np.float64)
    ulp = 2.0 * bf16_half_ulp(np.maximum(np.abs(a), np.abs(b)))
    return bool(np.all(np.abs(a - b) <= ulp + 1e-5 * np.max(np.abs(b))))


def test_decode_steps_match_verify_records():
    """FP32 storage: T decode launches and one T-token verify run the same recurrence.  The
    verify projects f_b on the tensor cores (FP32 accumulation in the MMA's order), decode with
    FMA chains, so the records equal the decode states to FP32 rounding (1e-6 of the largest
    entry), the outputs to one BF16 rounding step (plus 1e-5 of the largest), and the windows
    bit for bit."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=52, B=4, H=3, n_steps=5, num_slots=6, state_std=0.1, random_conv=True)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_v = device_pool(case)
    vin = [ins[n].transpose(0, 1).contiguous() for n in NAMES]
    out_v, rec, recw = K.kda_verify(layer, pool_v, slots, *vin)
    pool_d = device_pool(case)
    for s in range(5):
        o = K.kda_decode(layer, pool_d, slots, *(ins[n][s] for n in NAMES))
        assert within_one_bf16_step(o, out_v[:, s])
        assert normwise_err(pool_d.state[slots.long()].cpu().numpy(), rec[:, s].cpu().numpy()) <= 1e-6
        assert torch.equal(pool_d.conv_state[slots.long()], recw[:, s])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cluster_decode_equals_tile_kernel_bitwise(dtype):
    """B*H = 38 tiles: single-token decode splits each tile's columns over a cluster of four
    CTAs.  It equals the one-tile-per-CTA decode (kda_decode_resume with nothing to commit runs
    the tile kernel) bit for bit: outputs, state and window; and it matches the oracle."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=57, B=19, H=2, n_steps=2, num_slots=23, state_dtype=dtype, state_std=0.2,
                       random_conv=True, random_norm=True, random_dt_bias=True)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_d, pool_t = device_pool(case), device_pool(case)
    B, H = case.B, case.layer.H
    none = (torch.zeros(B, dtype=torch.int32, device="cuda"),
            torch.zeros(B, 1, H, 128, 128, dtype=torch.float32, device="cuda"),
            torch.zeros(B, 1, 3, 3, H * 128, dtype=torch.bfloat16, device="cuda"))
    for s in range(2):
        o = K.kda_decode(layer, pool_d, slots, *(ins[n][s] for n in NAMES))
        o_t = K.kda_decode_resume(layer, pool_t, slots, none, *(ins[n][s] for n in NAMES))
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_t.view(torch.int16))
        got, want = pool_d.state[slots.long()], pool_t.state[slots.long()]
        assert torch.equal(got.view(torch.int16) if dtype == "bf16" else got.view(torch.int32),
                           want.view(torch.int16) if dtype == "bf16" else want.view(torch.int32))
        assert torch.equal(pool_d.conv_state.view(torch.int16), pool_t.conv_state.view(torch.int16))
    assert K.kda_get_error(pool_d) == 0 and K.kda_get_error(pool_t) == 0
    check_decode(case)


def test_cluster_decode_bad_slot_sets_error_and_skips_tile():
    """Few tiles (cluster kernel): an out-of-range slot id is flagged and its cluster skips the
    tile without any CTA of the cluster waiting on another; the other tiles are updated."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=58, B=3, H=2, n_steps=1, num_slots=4, state_std=0.1)
    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.tensor([2, 7, 0], dtype=torch.int32, device="cuda")
    before = pool.state.clone()
    K.kda_decode(layer, pool, slots, *(ins[n][0] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == K.kda.KDA_DEVERR_SLOT
    assert torch.equal(before[[1, 3]], pool.state[[1, 3]])
    assert not torch.equal(before[2], pool.state[2]) and not torch.equal(before[0], pool.state[0])


def test_decode_graph_replay_bitwise_and_deterministic():
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=53, B=8, H=4, n_steps=3, num_slots=16, state_std=0.1)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pools = [device_pool(case) for _ in range(3)]
    outs = []
    for pool in pools[:2]:
        for s in range(3):
            o = K.kda_decode(layer, pool, slots, *(ins[n][s] for n in NAMES))
        outs.append(o)
    # graph: capture one step with static inputs, replay three times feeding new inputs
    static = {n: ins[n][0].clone() for n in NAMES}
    out_g = torch.empty_like(outs[0])
    g = torch.cuda.CUDAGraph()
    s_ = torch.cuda.Stream()
    s_.wait_stream(torch.cuda.current_stream())
    pool_g = pools[2]
    snapshot = (pool_g.state.clone(), pool_g.conv_state.clone())
    with torch.cuda.stream(s_):
        K.kda_decode(layer, pool_g, slots, *(static[n] for n in NAMES), out=out_g)   # warm
    torch.cuda.current_stream().wait_stream(s_)
    pool_g.state.copy_(snapshot[0])
    pool_g.conv_state.copy_(snapshot[1])
    with torch.cuda.graph(g):
        K.kda_decode(layer, pool_g, slots, *(static[n] for n in NAMES), out=out_g)
    for s in range(3):
        for n in NAMES:
            static[n].copy_(ins[n][s])
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(pools[0].state, pools[1].state)
    assert torch.equal(out_g, outs[0])
    assert torch.equal(pool_g.state, pools[0].state)


def test_prepared_decode_and_verify_equal_the_checked_calls_bitwise():
    """prepare_decode / prepare_verify bind fixed buffers once; each call re-issues the launch
    with the inputs rewritten in place between calls, and equals kda_decode / kda_verify."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=55, B=6, H=3, n_steps=3, num_slots=9, state_std=0.1, random_conv=True)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_a, pool_b = device_pool(case), device_pool(case)
    static = {n: ins[n][0].clone() for n in NAMES}
    out_b = torch.empty(case.B, layer.H * 128, dtype=torch.bfloat16, device="cuda")
    step = K.prepare_decode(layer, pool_b, slots, *(static[n] for n in NAMES), out=out_b)
    for s in range(3):
        o = K.kda_decode(layer, pool_a, slots, *(ins[n][s] for n in NAMES))
        for n in NAMES:
            static[n].copy_(ins[n][s])
        step()
        torch.cuda.synchronize()
        assert torch.equal(o, out_b)
    assert torch.equal(pool_a.state, pool_b.state)
    assert torch.equal(pool_a.conv_state, pool_b.conv_state)
    vin = {n: ins[n].transpose(0, 1).contiguous() for n in NAMES}   # [B, T, ...]
    o_v, r_v, w_v = K.kda_verify(layer, pool_a, slots, *(vin[n] for n in NAMES))
    o_p, r_p, w_p = torch.empty_like(o_v), torch.empty_like(r_v), torch.empty_like(w_v)
    K.prepare_verify(layer, pool_a, slots, *(vin[n] for n in NAMES), out=o_p, rec_state=r_p, rec_conv=w_p)()
    torch.cuda.synchronize()
    assert torch.equal(o_v, o_p) and torch.equal(r_v, r_p) and torch.equal(w_v, w_p)
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs a second GPU")
def test_decode_on_a_device_that_is_not_current():
    """Tensors on cuda:1 with cuda:0 current: the binding makes their device current for the
    call, so the result equals the same decode run with cuda:1 current."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=56, B=4, H=2, n_steps=2, num_slots=5, state_std=0.1)
    dev = torch.device("cuda", 1)
    layer, ins = device_layer(case, dev), device_inputs(case, dev)
    slots = torch.from_numpy(case.slot_ids).to(dev)
    pool_a, pool_b = device_pool(case, dev), device_pool(case, dev)
    with torch.cuda.device(0):
        o_a = K.kda_decode(layer, pool_a, slots, *(ins[n][0] for n in NAMES))
    with torch.cuda.device(1):
        o_b = K.kda_decode(layer, pool_b, slots, *(ins[n][0] for n in NAMES))
    torch.cuda.synchronize(dev)
    assert torch.equal(o_a, o_b) and torch.equal(pool_a.state, pool_b.state)
    assert K.kda_get_error(pool_a) == 0


def decode_in_parts(K, layer, pool, slots, step_inputs, parts):
    """kda_decode over sub-batches of at most 240 tiles (one tile per CTA); the outputs joined."""
    outs = [K.kda_decode(layer, pool, slots[lo:hi], *(x[lo:hi] for x in step_inputs)) for lo, hi in parts]
    return torch.cat(outs)


def test_decode_paired_tiles_equal_one_tile_decode_bitwise():
    """Many FP32 tiles (B*H = 644, B odd): decode takes two tiles per CTA.  Its steps must equal
    the same decode run on sub-batches of one tile per CTA bit for bit (outputs, states,
    windows), match the records of one multi-token verify to FP32 rounding, and a sample of the
    sequences must match the oracle."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=54, B=161, H=4, n_steps=3, num_slots=170, state_std=0.2, random_conv=True,
                       random_norm=True, random_dt_bias=True)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_v = device_pool(case)
    vin = [ins[n].transpose(0, 1).contiguous() for n in NAMES]
    out_v, rec, recw = K.kda_verify(layer, pool_v, slots, *vin)
    pool_d, pool_t = device_pool(case), device_pool(case)
    parts = [(0, 60), (60, 120), (120, case.B)]
    for s in range(3):
        o = K.kda_decode(layer, pool_d, slots, *(ins[n][s] for n in NAMES))
        o_t = decode_in_parts(K, layer, pool_t, slots, [ins[n][s] for n in NAMES], parts)
        assert torch.equal(o.view(torch.int16), o_t.view(torch.int16))
        assert torch.equal(pool_d.state.view(torch.int32), pool_t.state.view(torch.int32))
        assert torch.equal(pool_d.conv_state.view(torch.int16), pool_t.conv_state.view(torch.int16))
        assert within_one_bf16_step(o, out_v[:, s])
        assert normwise_err(pool_d.state[slots.long()].cpu().numpy(), rec[:, s].cpu().numpy()) <= 1e-6
        assert torch.equal(pool_d.conv_state[slots.long()], recw[:, s])
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_d) == 0 and K.kda_get_error(pool_t) == 0
    check_decode(case, sel=np.array([0, 1, 2, 79, 80, 158, 159, 160]))


def test_decode_paired_tiles_bad_slots():
    """Two tiles per CTA with a bad slot in the first, the second, both, or neither tile of a
    CTA: the bad ones are flagged and skipped, the others equal a one-tile-per-CTA decode of
    them alone, bit for bit."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=55, B=160, H=4, n_steps=1, num_slots=200, state_std=0.2, random_conv=True)
    layer, ins = device_layer(case), device_inputs(case)
    bad = {0: -1, 3: 200, 4: -7, 5: 1 << 20}
    good = np.array([b for b in range(case.B) if b not in bad])
    slots_h = case.slot_ids.copy()
    for b, s in bad.items():
        slots_h[b] = s
    pool_d = device_pool(case)
    out = K.kda_decode(layer, pool_d, torch.from_numpy(slots_h).cuda(), *(ins[n][0] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_d) == K.kda.KDA_DEVERR_SLOT
    pool_t = device_pool(case)
    g = torch.from_numpy(good).cuda()
    gslots = torch.from_numpy(case.slot_ids[good]).cuda()
    parts = [(lo, min(lo + 60, len(good))) for lo in range(0, len(good), 60)]
    out_t = decode_in_parts(K, layer, pool_t, gslots, [ins[n][0][g].contiguous() for n in NAMES], parts)
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_t) == 0
    assert torch.equal(out[g].view(torch.int16), out_t.view(torch.int16))
    gs = gslots.long()
    assert torch.equal(pool_d.state[gs].view(torch.int32), pool_t.state[gs].view(torch.int32))
    assert torch.equal(pool_d.conv_state[gs].view(torch.int16), pool_t.conv_state[gs].view(torch.int16))
    named = case.slot_ids[good]
    untouched = np.setdiff1d(np.arange(case.pool.num_slots), named)
    np.testing.assert_array_equal(pool_state_raw(pool_d)[untouched], case.pool.state[untouched])
    np.testing.assert_array_equal(bf16_bits(pool_d.conv_state)[untouched], case.pool.conv[untouched])
