"""kda_prefill_noalloc: the prefill entry point for callers that cannot allocate device memory.

Such callers (code running inside a CUDA-graph capture, serving runtimes that reserve their
whole memory budget up front, hosts without an allocator of their own) cannot hand kda_prefill
a scratch workspace; kda_prefill_noalloc uses a fixed scratch region built into the library.
This file checks it against kda_prefill, through the C ABI, on two calls in a row (the second
call reuses the region the first one left behind).  It is collected last so that a run that
stops at the first failure has run every other test first.
"""
from __future__ import annotations

import pytest
import torch

from gpu_io import NAMES, device_inputs, device_layer, device_pool
from kda_inputs import make_prefill

pytestmark = pytest.mark.gpu


def _run(case, entry):
    import verify_kda_decode_gb300 as K

    layer, pool, ins = device_layer(case), device_pool(case), device_inputs(case)
    slots = torch.from_numpy(case.slot_ids).cuda()
    args = [ins[n] for n in NAMES]
    if entry == "noalloc":
        out = K.kda_prefill_noalloc(layer, pool, slots, *args)
    else:
        out = K.kda_prefill(layer, pool, slots, *args)
    torch.cuda.synchronize()
    assert K.kda_get_error(pool) == 0
    return out, pool


@pytest.mark.parametrize("seed,L", [(101, 300), (102, 197)])
def test_noalloc_prefill_matches_prefill_twice(seed, L):
    case = make_prefill(seed=seed, B=2, L=L, H=4, num_slots=4, state_std=0.2, random_conv=True)
    ref_out, ref_pool = _run(case, "workspace")
    for _ in range(2):   # two calls in a row on the shared scratch region
        out, pool = _run(case, "noalloc")
        # the same kernels on the same inputs: equal bit for bit, so that scratch left over
        # from the previous call cannot hide inside a tolerance
        assert torch.equal(out, ref_out)
        assert torch.equal(pool.state, ref_pool.state)
        assert torch.equal(pool.conv_state, ref_pool.conv_state)


def test_noalloc_prefill_rejects_sizes_beyond_the_region():
    import verify_kda_decode_gb300 as K

    case = make_prefill(seed=103, B=1, L=64, H=32, num_slots=1)
    layer, pool = device_layer(case), device_pool(case)
    limit = K.kda_prefill_noalloc_max_bytes()
    L = 64 * 64   # far beyond the region for 32 heads
    assert K.kda_prefill_workspace_size(layer, 1, L) > limit
    z = lambda c: torch.zeros(1, L, c, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(K.KdaError) as ei:
        K.kda_prefill_noalloc(layer, pool, torch.zeros(1, dtype=torch.int32, device="cuda"),
                              z(32 * 128), z(32 * 128), z(32 * 128), z(128), z(32), z(32 * 128))
    assert ei.value.status == K.kda.KDA_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
