"""GPU fused commit-into-next-step (kda_decode_resume, kda_verify_resume) and mixed steps.

Each resume entry replaces an unfused pair of calls (kda_commit, then kda_decode or kda_verify)
and must reproduce it bit for bit: outputs, records and every byte of the pool.  A three-step
serving loop (verify, mixed verify-resume, decode-resume) is also checked against the FP64
oracle running the same commits on its own pool, with the tolerances of the single steps.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from case_io import bf16_out_err, bf16_pair_err, normwise_err, oracle_layer, storage_mode
from gpu_io import NAMES, bf16_bits, bf16_vals, device_inputs, device_layer, device_pool, pool_state_raw
from kda_inputs import bf16_bits_to_f32, make_verify

OUT_TOL = 2e-3
STATE_F32_TOL = 1e-4
STATE_BF16_TOL = 5e-3

pytestmark = pytest.mark.gpu


def copy_pool(pool):
    from verify_kda_decode_gb300 import KdaPool

    return KdaPool(pool.state.clone(), pool.conv_state.clone(), torch.zeros_like(pool.err_word))


def same_pool(a, b):
    assert torch.equal(a.state.view(torch.int16) if a.state.dtype == torch.bfloat16 else a.state.view(torch.int32),
                       b.state.view(torch.int16) if b.state.dtype == torch.bfloat16 else b.state.view(torch.int32))
    assert torch.equal(a.conv_state.view(torch.int16), b.conv_state.view(torch.int16))


def token_inputs(seed, B, H, T):
    """Fresh per-token inputs [B, T, ...] for a later step (same draw recipe as the workloads)."""
    return make_verify(seed=seed, B=B, H=H, T=T, num_slots=B).inputs


def dev(inputs):
    from gpu_io import bf16_dev

    return {n: bf16_dev(inputs[n]) for n in NAMES}


def first_step(case):
    import verify_kda_decode_gb300 as K

    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    out, rec, recw = K.kda_verify(layer, pool, slots, *(ins[n] for n in NAMES))
    return layer, pool, slots, out, rec, recw


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_resume_equals_commit_then_decode(dtype):
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=80, B=7, H=3, T=4, num_slots=12, state_dtype=dtype, state_std=0.2,
                       random_conv=True, random_norm=True, random_dt_bias=True)
    layer, pool, slots, out, rec, recw = first_step(case)
    acc = torch.from_numpy(np.array([0, 1, 2, 3, 4, 0, 2], np.int32)).cuda()
    step = dev({n: a[:, 0] for n, a in token_inputs(81, case.B, case.layer.H, 1).items()})
    pool_a, pool_b = copy_pool(pool), copy_pool(pool)
    K.kda_commit(pool_a, slots, acc, rec, recw)
    out_a = K.kda_decode(layer, pool_a, slots, *(step[n] for n in NAMES))
    out_b = K.kda_decode_resume(layer, pool_b, slots, (acc, rec, recw), *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    same_pool(pool_a, pool_b)


def test_decode_resume_without_previous_step_is_decode():
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=82, B=4, H=2, T=1, num_slots=6, state_std=0.1)
    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    step = {n: ins[n][:, 0].contiguous() for n in NAMES}
    pool_b = copy_pool(pool)
    out_a = K.kda_decode(layer, pool, slots, *(step[n] for n in NAMES))
    out_b = K.kda_decode_resume(layer, pool_b, slots, None, *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    same_pool(pool, pool_b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 4, 16])
def test_verify_resume_equals_commit_then_verify(dtype, T):
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=83 + T, B=6, H=2, T=4, num_slots=9, state_dtype=dtype, state_std=0.2,
                       random_conv=True)
    layer, pool, slots, out, rec, recw = first_step(case)
    acc = torch.from_numpy(np.array([4, 0, 1, 3, 2, 4], np.int32)).cuda()
    step = dev(token_inputs(90 + T, case.B, case.layer.H, T))
    pool_a, pool_b = copy_pool(pool), copy_pool(pool)
    K.kda_commit(pool_a, slots, acc, rec, recw)
    oa, ra, wa = K.kda_verify(layer, pool_a, slots, *(step[n] for n in NAMES))
    ob, rb, wb = K.kda_verify_resume(layer, pool_b, slots, (acc, rec, recw), *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(ra.view(torch.int32), rb.view(torch.int32))
    assert torch.equal(wa.view(torch.int16), wb.view(torch.int16))
    same_pool(pool_a, pool_b)


@pytest.mark.parametrize("dtype,T", [("f32", 5), ("bf16", 5), ("f32", 13)])
def test_mixed_step_token_counts(dtype, T):
    """Per-sequence token counts: tokens t < n_tokens[b] equal a full-length verify_resume bit
    for bit; the entries past n_tokens[b] keep what the caller put there.  With T = 13 the
    counts fall on both sides of the 8-token projection chains (1 to 13 tokens)."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=95, B=8, H=3, T=3, num_slots=11, state_dtype=dtype, state_std=0.2)
    layer, pool, slots, out, rec, recw = first_step(case)
    acc = torch.from_numpy(np.array([1, 3, 0, 2, 3, 1, 0, 2], np.int32)).cuda()
    ntok_h = (np.array([1, 5, 2, 1, 3, 5, 4, 1], np.int32) if T == 5
              else np.array([1, 13, 8, 9, 7, 12, 4, 10], np.int32))
    step = dev(token_inputs(96, case.B, case.layer.H, T))
    pool_a, pool_b = copy_pool(pool), copy_pool(pool)
    oa, ra, wa = K.kda_verify_resume(layer, pool_a, slots, (acc, rec, recw), *(step[n] for n in NAMES))
    H = case.layer.H
    ob = torch.full((case.B, T, H * 128), 7.0, dtype=torch.bfloat16, device="cuda")
    rb = torch.full((case.B, T, H, 128, 128), -3.0, dtype=torch.float32, device="cuda")
    wb = torch.full((case.B, T, 3, 3, H * 128), 5.0, dtype=torch.bfloat16, device="cuda")
    K.kda_verify_resume(layer, pool_b, slots, (acc, rec, recw), *(step[n] for n in NAMES),
                        n_tokens=torch.from_numpy(ntok_h).cuda(), out=ob, rec_state=rb, rec_conv=wb)
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_b) == 0
    for b, n in enumerate(ntok_h):
        assert torch.equal(oa[b, :n].view(torch.int16), ob[b, :n].view(torch.int16))
        assert torch.equal(ra[b, :n].view(torch.int32), rb[b, :n].view(torch.int32))
        assert torch.equal(wa[b, :n].view(torch.int16), wb[b, :n].view(torch.int16))
        assert bool((ob[b, n:] == 7.0).all()) and bool((rb[b, n:] == -3.0).all()) and bool((wb[b, n:] == 5.0).all())
    same_pool(pool_a, pool_b)   # both committed the same records; verify leaves the rest


def test_resume_out_of_range_lengths_flag_and_skip():
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=97, B=4, H=2, T=4, num_slots=8, state_std=0.1)
    layer, pool, slots, out, rec, recw = first_step(case)
    step = dev(token_inputs(98, case.B, case.layer.H, 2))
    before = copy_pool(pool)
    bad_acc = torch.tensor([5, -1, 5, -2], dtype=torch.int32, device="cuda")   # all out of range
    K.kda_verify_resume(layer, pool, slots, (bad_acc, rec, recw), *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == K.kda.KDA_DEVERR_ACCEPTED
    same_pool(pool, before)
    one = {n: step[n][:, 0].contiguous() for n in NAMES}
    K.kda_decode_resume(layer, pool, slots, (bad_acc, rec, recw), *(one[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == K.kda.KDA_DEVERR_ACCEPTED
    same_pool(pool, before)
    zero = torch.zeros(4, dtype=torch.int32, device="cuda")
    bad_n = torch.tensor([0, 3, 2, 1], dtype=torch.int32, device="cuda")      # 0 and 3 > T = 2
    K.kda_verify_resume(layer, pool, slots, (zero, rec, recw), *(step[n] for n in NAMES), n_tokens=bad_n)
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == K.kda.KDA_DEVERR_TOKENS
    same_pool(pool, before)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_serving_loop_matches_oracle(dtype):
    """verify (T=4) -> accept -> mixed verify_resume (1..4 tokens per sequence) -> accept ->
    decode_resume, against the oracle's verify / commit / decode on its own pool."""
    import verify_kda_decode_gb300 as K

    B, H, T = 6, 2, 4
    case = make_verify(seed=99, B=B, H=H, T=T, num_slots=10, state_dtype=dtype, state_std=0.2,
                       random_conv=True, random_norm=True, random_dt_bias=True)
    acc1 = np.array([2, 0, 4, 1, 3, 4], np.int32)
    ntok = np.array([1, 4, 2, 4, 3, 1], np.int32)
    acc2 = np.array([1, 3, 0, 4, 2, 1], np.int32)     # each <= ntok
    in2 = token_inputs(100, B, H, T)
    in3 = {n: a[:, 0] for n, a in token_inputs(101, B, H, 1).items()}

    # GPU
    layer, pool, slots, o1, r1, w1 = first_step(case)
    cu = lambda a: torch.from_numpy(a).cuda()
    o2, r2, w2 = K.kda_verify_resume(layer, pool, slots, (cu(acc1), r1, w1), *(dev(in2)[n] for n in NAMES),
                                     n_tokens=cu(ntok))
    o3 = K.kda_decode_resume(layer, pool, slots, (cu(acc2), r2, w2), *(dev(in3)[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == 0

    # oracle, on its own copy of the pool bytes
    L, lw, mode = oracle_layer(case), case.layer, storage_mode(case)
    raw = case.pool.state.copy()
    win = case.pool.conv.reshape(case.pool.num_slots, -1).copy()
    ids = case.slot_ids

    def slot_state(raw_state):
        st = raw_state[ids]
        return (bf16_bits_to_f32(st) if dtype == "bf16" else st).astype(np.float64)

    def slot_window(w):
        return bf16_bits_to_f32(w[ids]).astype(np.float64)

    def f32_bits_to_bf16_bits(x):
        return oracle.f32_to_bf16(np.asarray(x, np.float32))

    ro1, rr1, rw1 = oracle.verify(L, slot_state(raw), slot_window(win), *(case.inputs[n] for n in NAMES))
    raw, win, rc = oracle.commit(lw.H, lw.dk, lw.dv, lw.K, mode, raw, win, ids, acc1,
                                 rr1.astype(np.float32), f32_bits_to_bf16_bits(rw1))
    assert rc == 0
    ro2, rr2, rw2 = oracle.verify(L, slot_state(raw), slot_window(win), *(in2[n] for n in NAMES))
    raw, win, rc = oracle.commit(lw.H, lw.dk, lw.dv, lw.K, mode, raw, win, ids, acc2,
                                 rr2.astype(np.float32), f32_bits_to_bf16_bits(rw2))
    assert rc == 0
    ro3, rS3, rW3 = oracle.decode(L, slot_state(raw), slot_window(win),
                                  *(np.ascontiguousarray(in3[n][None]) for n in NAMES), storage=mode)

    got1, got2 = bf16_vals(o1), bf16_vals(o2)
    for t in range(T):
        assert bf16_out_err(got1[:, t], ro1[:, t]) <= OUT_TOL
    for b in range(B):
        for t in range(ntok[b]):
            assert bf16_out_err(got2[b, t], ro2[b, t]) <= OUT_TOL, (b, t)
            got_r = r2[b, t].cpu().numpy().astype(np.float64)
            if dtype == "bf16" and acc1[b] > 0:
                # started from a record committed into BF16: the GPU rounds its FP32 record, the
                # oracle its own; near a tie the two land one BF16 spacing apart, which the FP32
                # record carries on (the commit itself is pinned bit for bit elsewhere)
                assert bf16_pair_err(got_r, rr2[b, t]) <= STATE_BF16_TOL, (b, t)
            else:
                assert normwise_err(got_r, rr2[b, t]) <= STATE_F32_TOL, (b, t)
    assert bf16_out_err(bf16_vals(o3), ro3[0]) <= OUT_TOL
    got_S = pool.state.float().cpu().numpy().astype(np.float64)[ids]
    if dtype == "bf16":
        assert bf16_pair_err(got_S, rS3) <= STATE_BF16_TOL
    else:
        assert normwise_err(got_S, rS3) <= STATE_F32_TOL
    got_w = bf16_bits_to_f32(bf16_bits(pool.conv_state)).astype(np.float64)[ids].reshape(B, -1)
    np.testing.assert_array_equal(got_w, rW3)
    untouched = np.setdiff1d(np.arange(case.pool.num_slots), ids)
    np.testing.assert_array_equal(pool_state_raw(pool)[untouched], case.pool.state[untouched])


def test_serving_step_graph_replay_bitwise():
    """A whole speculative step (verify_resume of the previous step's records with per-sequence
    token counts, then the accepted lengths rewritten in place) captured once as a CUDA graph
    and replayed with new inputs equals the same calls issued eagerly, bit for bit."""
    import verify_kda_decode_gb300 as K

    B, H, T = 5, 2, 3
    case = make_verify(seed=120, B=B, H=H, T=T, num_slots=8, state_std=0.2, random_conv=True)
    layer, pool_e, slots, o0, r0, w0 = first_step(case)
    pool_g = copy_pool(pool_e)
    steps = [dev(token_inputs(121 + i, B, H, T)) for i in range(3)]
    # step i commits accs[i] tokens of step i - 1: at most the 3 of the first verify, then at
    # most the n_tokens each sequence ran (records past them are never written)
    ntok = torch.tensor([1, 3, 2, 3, 3], dtype=torch.int32, device="cuda")
    accs = [np.array([1, 3, 0, 2, 3], np.int32), np.array([1, 1, 2, 0, 3], np.int32),
            np.array([1, 3, 2, 1, 1], np.int32)]
    # double-buffered records: step i reads buffer i % 2 and writes buffer (i + 1) % 2
    def bufs():
        return [(torch.empty_like(r0), torch.empty_like(w0)) for _ in range(2)]
    rec_e, rec_g = bufs(), bufs()
    for rb in (rec_e, rec_g):
        rb[0][0].copy_(r0)
        rb[0][1].copy_(w0)
    acc_e, acc_g = torch.zeros(B, dtype=torch.int32, device="cuda"), torch.zeros(B, dtype=torch.int32, device="cuda")
    out_e = [torch.empty(B, T, H * 128, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    for i in range(3):   # eager
        acc_e.copy_(torch.from_numpy(accs[i]))
        src, dst = rec_e[i % 2], rec_e[(i + 1) % 2]
        K.kda_verify_resume(layer, pool_e, slots, (acc_e, src[0], src[1]), *(steps[i][n] for n in NAMES),
                            n_tokens=ntok, out=out_e[i], rec_state=dst[0], rec_conv=dst[1])
    # graph: two captured steps (one per record-buffer parity), inputs and lengths rewritten in place
    static = {n: torch.empty_like(steps[0][n]) for n in NAMES}
    out_g = torch.empty_like(out_e[0])
    graphs = []
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for par in range(2):
        src, dst = rec_g[par], rec_g[1 - par]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                K.kda_verify_resume(layer, pool_g, slots, (acc_g, src[0], src[1]), *(static[n] for n in NAMES),
                                    n_tokens=ntok, out=out_g, rec_state=dst[0], rec_conv=dst[1])
        graphs.append(g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for i in range(3):
        acc_g.copy_(torch.from_numpy(accs[i]))
        for n in NAMES:
            static[n].copy_(steps[i][n])
        graphs[i % 2].replay()
        torch.cuda.synchronize()
        for b, n in enumerate(ntok.tolist()):
            assert torch.equal(out_g[b, :n].view(torch.int16), out_e[i][b, :n].view(torch.int16)), (i, b)
    assert K.kda_get_error(pool_g) == 0 and K.kda_get_error(pool_e) == 0
    same_pool(pool_g, pool_e)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_resume_many_waves_equals_commit_then_decode(dtype):
    """B*H = 960 tiles: decode_resume (one tile per CTA, each prefetching the record or tile of
    the CTA one wave later at its start) against commit + decode (tile pairs for FP32, the BF16
    decode kernel's many-wave path) bit for bit."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=121, B=120, H=8, T=2, num_slots=130, state_dtype=dtype, state_std=0.2,
                       random_conv=True)
    layer, pool, slots, out, rec, recw = first_step(case)
    acc = torch.from_numpy(np.random.default_rng(5).integers(0, 3, case.B).astype(np.int32)).cuda()
    step = dev({n: a[:, 0] for n, a in token_inputs(122, case.B, case.layer.H, 1).items()})
    pool_a, pool_b = copy_pool(pool), copy_pool(pool)
    K.kda_commit(pool_a, slots, acc, rec, recw)
    out_a = K.kda_decode(layer, pool_a, slots, *(step[n] for n in NAMES))
    out_b = K.kda_decode_resume(layer, pool_b, slots, (acc, rec, recw), *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    same_pool(pool_a, pool_b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_many_waves_equal_one_wave_bitwise(dtype):
    """B*H = 644 tiles, more than two resident waves: verify, a mixed verify_resume and a
    decode_resume (each CTA prefetching the tile or record of the CTA one wave later) must equal
    the same calls made on sub-batches that fit one wave, bit for bit: outputs, records,
    windows and every byte of the pool."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=131, B=161, H=4, T=3, num_slots=170, state_dtype=dtype, state_std=0.2,
                       random_conv=True)
    B, H = case.B, case.layer.H
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    parts = [(0, 60), (60, 120), (120, B)]   # at most 240 tiles: one wave of one-tile CTAs
    pool_a, pool_b = device_pool(case), device_pool(case)

    def bits(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)

    def same(x, y):
        for a, b in zip(x, y):
            assert torch.equal(bits(a), bits(b))

    # 1. verify
    va = K.kda_verify(layer, pool_a, slots, *(ins[n] for n in NAMES))
    vb = [torch.empty_like(t) for t in va]
    for lo, hi in parts:
        K.kda_verify(layer, pool_b, slots[lo:hi], *(ins[n][lo:hi] for n in NAMES), out=vb[0][lo:hi],
                     rec_state=vb[1][lo:hi], rec_conv=vb[2][lo:hi])
    torch.cuda.synchronize()
    same(va, vb)
    # 2. mixed step: commit the drawn lengths, then 1..4 tokens per sequence
    rng = np.random.default_rng(131)
    acc = torch.from_numpy(rng.integers(0, 4, B).astype(np.int32)).cuda()
    ntok_h = rng.integers(1, 5, B).astype(np.int32)
    ntok = torch.from_numpy(ntok_h).cuda()
    step = dev(token_inputs(132, B, H, 4))
    ma = [torch.full((B, 4, H * 128), 3.0, dtype=torch.bfloat16, device="cuda"),
          torch.full((B, 4, H, 128, 128), -1.0, dtype=torch.float32, device="cuda"),
          torch.full((B, 4, 3, 3, H * 128), 2.0, dtype=torch.bfloat16, device="cuda")]
    mb = [t.clone() for t in ma]
    K.kda_verify_resume(layer, pool_a, slots, (acc, va[1], va[2]), *(step[n] for n in NAMES), n_tokens=ntok,
                        out=ma[0], rec_state=ma[1], rec_conv=ma[2])
    for lo, hi in parts:
        K.kda_verify_resume(layer, pool_b, slots[lo:hi], (acc[lo:hi], vb[1][lo:hi], vb[2][lo:hi]),
                            *(step[n][lo:hi] for n in NAMES), n_tokens=ntok[lo:hi], out=mb[0][lo:hi],
                            rec_state=mb[1][lo:hi], rec_conv=mb[2][lo:hi])
    torch.cuda.synchronize()
    same(ma, mb)
    same_pool(pool_a, pool_b)
    # 3. decode resuming from the mixed step's records
    acc2 = torch.from_numpy((rng.integers(0, 5, B) % (ntok_h + 1)).astype(np.int32)).cuda()
    one = dev({n: a[:, 0] for n, a in token_inputs(133, B, H, 1).items()})
    oa = K.kda_decode_resume(layer, pool_a, slots, (acc2, ma[1], ma[2]), *(one[n] for n in NAMES))
    ob = torch.empty_like(oa)
    for lo, hi in parts:
        K.kda_decode_resume(layer, pool_b, slots[lo:hi], (acc2[lo:hi], mb[1][lo:hi], mb[2][lo:hi]),
                            *(one[n][lo:hi] for n in NAMES), out=ob[lo:hi])
    torch.cuda.synchronize()
    assert torch.equal(bits(oa), bits(ob))
    same_pool(pool_a, pool_b)
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0


def test_many_waves_resume_bad_lengths_equal_one_wave():
    """A mixed verify_resume of 644 tiles (several waves) with out-of-range accepted lengths,
    token counts and slot ids: the same error bits as the calls on sub-batches that fit one
    wave, and every output, record, window and pool byte equal to theirs, including the records
    of the skipped sequences (filled beforehand), which no call may touch."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=137, B=161, H=4, T=4, num_slots=170, state_std=0.2, random_conv=True)
    B, H = case.B, case.layer.H
    layer, pool, slots, out, rec, recw = first_step(case)
    rng = np.random.default_rng(137)
    acc = rng.integers(0, 5, B).astype(np.int32)
    ntok = rng.integers(1, 5, B).astype(np.int32)
    acc[[7, 90]] = [5, -2]          # out of range: skipped, slot untouched
    ntok[[30, 150]] = [0, 6]        # out of range: committed, then skipped
    bad_slots = slots.clone()
    bad_slots[100] = -1
    acc_d, ntok_d = torch.from_numpy(acc).cuda(), torch.from_numpy(ntok).cuda()
    step = dev(token_inputs(138, B, H, 4))
    parts = [(0, 60), (60, 120), (120, B)]
    pool_a, pool_b = copy_pool(pool), copy_pool(pool)
    ma = [torch.full((B, 4, H * 128), 3.0, dtype=torch.bfloat16, device="cuda"),
          torch.full((B, 4, H, 128, 128), -1.0, dtype=torch.float32, device="cuda"),
          torch.full((B, 4, 3, 3, H * 128), 2.0, dtype=torch.bfloat16, device="cuda")]
    mb = [t.clone() for t in ma]
    K.kda_verify_resume(layer, pool_a, bad_slots, (acc_d, rec, recw), *(step[n] for n in NAMES),
                        n_tokens=ntok_d, out=ma[0], rec_state=ma[1], rec_conv=ma[2])
    err_a = K.kda_get_error(pool_a)
    errs_b = 0
    for lo, hi in parts:
        K.kda_verify_resume(layer, pool_b, bad_slots[lo:hi], (acc_d[lo:hi], rec[lo:hi], recw[lo:hi]),
                            *(step[n][lo:hi] for n in NAMES), n_tokens=ntok_d[lo:hi], out=mb[0][lo:hi],
                            rec_state=mb[1][lo:hi], rec_conv=mb[2][lo:hi])
        errs_b |= K.kda_get_error(pool_b)
    torch.cuda.synchronize()
    assert err_a == errs_b == K.kda.KDA_DEVERR_ACCEPTED | K.kda.KDA_DEVERR_TOKENS | K.kda.KDA_DEVERR_SLOT
    for x, y in zip(ma, mb):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))
    same_pool(pool_a, pool_b)
    for b in (7, 90, 100, 30, 150):   # skipped: nothing of theirs written
        assert bool((ma[1][b] == -1.0).all()) and bool((ma[0][b].float() == 3.0).all())


def test_many_waves_bad_slot_skips_only_its_tiles():
    """Two bad slot ids in a verify of several waves: the error bit is set, those sequences are
    skipped, and every other sequence equals a call without the bad ids."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=134, B=161, H=4, T=2, num_slots=170, state_std=0.2, random_conv=True)
    layer, ins = device_layer(case), device_inputs(case)
    good = torch.from_numpy(case.slot_ids).cuda()
    bad = good.clone()
    bad[5], bad[6] = -1, 170
    pool_a, pool_b = device_pool(case), device_pool(case)
    oa, ra, wa = K.kda_verify(layer, pool_a, good, *(ins[n] for n in NAMES))
    ob, rb, wb = K.kda_verify(layer, pool_b, bad, *(ins[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_b) == K.kda.KDA_DEVERR_SLOT
    keep = [b for b in range(case.B) if b not in (5, 6)]
    assert torch.equal(oa[keep].view(torch.int16), ob[keep].view(torch.int16))
    assert torch.equal(ra[keep], rb[keep]) and torch.equal(wa[keep].view(torch.int16), wb[keep].view(torch.int16))
    same_pool(pool_a, pool_b)   # verify writes no slot


def test_paired_resume_flags_and_skips_bad_lengths():
    """decode_resume of 40 x 8 FP32 tiles (two tiles per CTA): out-of-range accepted lengths and
    slot ids are flagged and skip their tiles (also when the partner tile in the CTA is fine);
    every other sequence equals commit + decode bit for bit."""
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=135, B=40, H=8, T=3, num_slots=44, state_std=0.2, random_conv=True)
    layer, pool, slots, out, rec, recw = first_step(case)
    acc_h = np.random.default_rng(135).integers(0, 4, case.B).astype(np.int32)
    bad_acc = acc_h.copy()
    bad_acc[[3, 10, 11]] = [4, -1, 9]          # out of range (T = 3); 10 and 11 share a CTA
    bad_slots = slots.clone()
    bad_slots[20] = 44                          # out of range; its partner 21 is fine
    keep = [b for b in range(case.B) if b not in (3, 10, 11, 20)]
    step = dev({n: a[:, 0] for n, a in token_inputs(136, case.B, case.layer.H, 1).items()})
    pool_a, pool_b = copy_pool(pool), copy_pool(pool)
    K.kda_commit(pool_a, slots, torch.from_numpy(acc_h).cuda(), rec, recw)
    out_a = K.kda_decode(layer, pool_a, slots, *(step[n] for n in NAMES))
    out_b = K.kda_decode_resume(layer, pool_b, bad_slots, (torch.from_numpy(bad_acc).cuda(), rec, recw),
                                *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert K.kda_get_error(pool_a) == 0
    assert K.kda_get_error(pool_b) == K.kda.KDA_DEVERR_ACCEPTED | K.kda.KDA_DEVERR_SLOT
    assert torch.equal(out_a[keep].view(torch.int16), out_b[keep].view(torch.int16))
    ks = slots[keep].long()
    assert torch.equal(pool_a.state[ks], pool_b.state[ks])
    assert torch.equal(pool_a.conv_state[ks].view(torch.int16), pool_b.conv_state[ks].view(torch.int16))
    skipped = slots[[3, 10, 11]].long()        # the skipped sequences' slots keep their bytes
    assert torch.equal(pool_b.state[skipped], pool.state[skipped])
