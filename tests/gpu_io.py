"""Test plumbing for the CUDA path: move a ``kda_inputs.Case`` onto the device and back.

BF16 tensors travel as their bit patterns (uint16 -> int16 view -> bfloat16 view), so the
device holds exactly the values the oracle decodes.
"""
from __future__ import annotations

import numpy as np
import torch

from kda_inputs import Case

NAMES = ("q", "k", "v", "f_a", "beta", "gate")


def bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_vals(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def device_layer(case: Case, device="cuda"):
    from verify_kda_decode_gb300 import KdaLayer

    lw = case.layer
    if lw.W_fb_fp8 is not None:   # FP8 input path: E4M3 codes and per-row scales
        return KdaLayer(W_fb=torch.from_numpy(lw.W_fb_fp8).view(torch.float8_e4m3fn).to(device),
                        W_fb_scale=torch.from_numpy(lw.W_fb_scale).to(device),
                        A_log=torch.from_numpy(lw.A_log).to(device),
                        dt_bias=torch.from_numpy(lw.dt_bias).to(device),
                        conv_w=bf16_dev(lw.conv_w, device),
                        norm_w=torch.from_numpy(lw.norm_w).to(device),
                        l2_eps=lw.l2_eps, norm_eps=lw.norm_eps)
    return KdaLayer(W_fb=bf16_dev(lw.W_fb, device),
                    A_log=torch.from_numpy(lw.A_log).to(device),
                    dt_bias=torch.from_numpy(lw.dt_bias).to(device),
                    conv_w=bf16_dev(lw.conv_w, device),
                    norm_w=torch.from_numpy(lw.norm_w).to(device),
                    l2_eps=lw.l2_eps, norm_eps=lw.norm_eps)


def device_pool(case: Case, device="cuda"):
    from verify_kda_decode_gb300 import KdaPool

    if case.pool.state_dtype == "bf16":
        st = bf16_dev(case.pool.state, device)
    else:
        st = torch.from_numpy(case.pool.state).to(device)
    return KdaPool(state=st, conv_state=bf16_dev(case.pool.conv, device),
                   err_word=torch.zeros(1, dtype=torch.int32, device=device))


def device_inputs(case: Case, device="cuda"):
    return {n: bf16_dev(case.inputs[n], device) for n in NAMES}


def pool_state_host(pool) -> np.ndarray:
    """Pool state as float64 (exact)."""
    return pool.state.detach().float().cpu().numpy().astype(np.float64)


def pool_state_raw(pool) -> np.ndarray:
    if pool.state.dtype == torch.bfloat16:
        return bf16_bits(pool.state)
    return pool.state.detach().cpu().numpy().copy()
