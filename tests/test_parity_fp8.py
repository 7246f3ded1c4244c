"""FP8 input path on the GPU: W_fb as FP8 E4M3 codes with one FP32 scale per row, against the
FP64 oracle that dequantises the same codes exactly.  Every kernel that computes the f_b
projection runs here: the tile kernel (small decode, verify, resume), the BF16 decode kernel,
the paired-tile decode kernel and the chunked prefill.  Tolerances are those of the BF16-weight
tests (outputs 2e-3 beyond the BF16 output rounding, FP32 state / records 1e-4, BF16 state
5e-3, windows and commit bit-exact)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_io import NAMES, device_inputs, device_layer, device_pool
from kda_inputs import make, make_decode, make_prefill, make_verify
from test_parity_decode import check_decode
from test_parity_prefill import check_prefill
from test_parity_verify_commit import check_commit, check_verify

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,B,H", [("f32", 3, 2), ("bf16", 5, 3), ("f32", 40, 8)])
def test_fp8_decode(dtype, B, H):
    """One tile per CTA (FP32, few tiles), the BF16 decode kernel, and tile pairs (FP32, 320
    tiles, more than one resident wave of single tiles)."""
    case = make_decode(seed=200 + B, B=B, H=H, n_steps=5, num_slots=B + 3, state_dtype=dtype,
                       state_std=0.2, random_conv=True, random_dt_bias=True, fp8_w_fb=True)
    check_decode(case)


def test_fp8_decode_b64_full():
    """The decode_b64 workload (B=64, H=8, 64 steps, FP32 pool) with FP8 W_fb."""
    check_decode(make("decode_b64", fp8_w_fb=True))


def test_fp8_verify_b64_commit():
    case = make("verify_b64", fp8_w_fb=True)
    layer, pool, slots, out, rec, recw = check_verify(case)
    err, rc = check_commit(case, pool, slots, rec, recw, case.accepted)
    assert err == 0 and rc == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fp8_resume_equals_commit_then_decode(dtype):
    import verify_kda_decode_gb300 as K

    case = make_verify(seed=210, B=6, H=2, T=3, num_slots=9, state_dtype=dtype, state_std=0.2,
                       random_conv=True, fp8_w_fb=True)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_a = device_pool(case)
    out, rec, recw = K.kda_verify(layer, pool_a, slots, *(ins[n] for n in NAMES))
    pool_b = device_pool(case)
    acc = torch.from_numpy(case.accepted).cuda()
    step = {n: ins[n][:, 0].contiguous() for n in NAMES}
    K.kda_commit(pool_a, slots, acc, rec, recw)
    o_a = K.kda_decode(layer, pool_a, slots, *(step[n] for n in NAMES))
    o_b = K.kda_decode_resume(layer, pool_b, slots, (acc, rec, recw), *(step[n] for n in NAMES))
    torch.cuda.synchronize()
    assert torch.equal(o_a.view(torch.int16), o_b.view(torch.int16))
    assert torch.equal(pool_a.state, pool_b.state) and torch.equal(pool_a.conv_state, pool_b.conv_state)
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0


@pytest.mark.parametrize("L", [70, 300])
def test_fp8_prefill(L):
    case = make_prefill(seed=220 + L, B=2, L=L, H=3, num_slots=4, state_std=0.2, random_conv=True,
                        random_dt_bias=True, fp8_w_fb=True)
    check_prefill(case)


def test_fp8_prefill_b4_full():
    """The prefill_b4 workload (B=4, L=4096, H=8) with FP8 W_fb, at every token."""
    check_prefill(make("prefill_b4", fp8_w_fb=True))


def test_fp8_weights_change_the_result():
    """The FP8 path is really taken: the same inputs with the BF16 weights give other outputs."""
    import verify_kda_decode_gb300 as K

    case = make_decode(seed=230, B=2, H=2, n_steps=1, num_slots=2, state_std=0.2, fp8_w_fb=True)
    ins = device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    outs = []
    for fp8 in (True, False):
        lw = case.layer
        saved = (lw.W_fb_fp8, lw.W_fb_scale)
        if not fp8:
            lw.W_fb_fp8 = lw.W_fb_scale = None
        outs.append(K.kda_decode(device_layer(case), device_pool(case), slots, *(ins[n][0] for n in NAMES)))
        lw.W_fb_fp8, lw.W_fb_scale = saved
    torch.cuda.synchronize()
    assert not torch.equal(outs[0], outs[1])


def test_fp8_prefill_varlen():
    """Variable-length prefill with FP8 weights: mixed lengths continuing from their slots."""
    from kda_inputs import quantize_w_fb_fp8
    from test_parity_prefill_varlen import check_sequences, run_varlen, untouched_slots_keep_bytes, varlen_case

    lens = [0, 3, 70, 130, 64]
    case, packed, cu = varlen_case(240, lens)
    quantize_w_fb_fp8(case.layer)
    layer, pool, out, err = run_varlen(case, packed, cu, max(lens))
    assert err == 0
    check_sequences(case, pool, out, cu, range(len(lens)))
    untouched_slots_keep_bytes(case, pool)


def test_fp8_prefill_noalloc_equals_prefill_bitwise():
    import verify_kda_decode_gb300 as K

    case = make_prefill(seed=241, B=2, L=150, H=2, num_slots=4, state_std=0.2, random_conv=True, fp8_w_fb=True)
    layer, ins = device_layer(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    pool_a, pool_b = device_pool(case), device_pool(case)
    oa = K.kda_prefill(layer, pool_a, slots, *(ins[n] for n in NAMES))
    ob = K.kda_prefill_noalloc(layer, pool_b, slots, *(ins[n] for n in NAMES))
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and torch.equal(pool_a.state, pool_b.state)
    assert K.kda_get_error(pool_a) == 0 and K.kda_get_error(pool_b) == 0
