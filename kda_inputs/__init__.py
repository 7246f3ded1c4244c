"""Seeded synthetic inputs for the KDA mixer step.

This module is the only code that the CUDA path and the FP64 oracle share.  It draws random
numbers and lays them out; it holds none of the method's arithmetic.  Arrays are numpy: BF16
tensors are returned as their raw ``uint16`` bit patterns (converted from float32 draws with
round-to-nearest-even by torch), everything else as float32 / int32.

Workloads (the five shapes the KDA decode / verify / prefill paths are measured on):

  decode_small   B=1,   H=2,  8 steps,  FP32 state from zero                      (seed 0)
  decode_b64     B=64,  H=8,  64 steps, FP32 pool of 256 slots, S0 ~ N(0, 0.1)   (seed 1)
  decode_b256    B=256, H=32, 16 steps, BF16 pool of 512 slots, S0 ~ N(0, 0.1)   (seed 2)
  verify_b64     B=64,  H=8,  T=4 draft tokens, FP32 pool of 256 slots, accepted
                 lengths uniform in {0..4}                                         (seed 3)
  prefill_b4     B=4,   L=4096, H=8, chunk 64, FP32 state from zero              (seed 4)

Common to all: dk = dv = 128, f_a rank r = 128, conv taps K = 4.

Draw order with ``numpy.random.default_rng(seed)`` (PCG64), each draw float32 unless noted:
  1. W_fb        N(0, 0.02)  [H*dk, r]            -> BF16
  2. A_log       U(-1, 1)    [H]
  3. dt_bias     zeros       [H*dk]               (no draw)
  4. conv_w      U(-0.5, 0.5) [3, H*dk, K]        -> BF16   (q, k, v convolutions)
  5. norm_w      ones        [dv]                 (no draw)
  6. slot_ids    first B entries of a permutation of range(num_slots), int32
  7. pool state  N(0, 0.1) [num_slots, H, dk, dv] (or zeros) -> BF16 for a BF16 pool
  8. pool conv   zeros [num_slots, 3, K-1, H*dk] BF16 (no draw)
  9. per-token inputs, each over all steps/tokens at once, in this order:
     q, k, v [.., H*dk], f_a [.., r], beta_logit [.., H], gate [.., H*dv], all N(0, 1) -> BF16
 10. (verify only) accepted lengths, integers uniform in {0..T}, int32
Options ``random_conv`` / ``random_norm`` / ``random_dt_bias`` replace the fixed zeros / ones of
steps 3, 5 and 8 with draws appended after step 10 (used by extra parity cases only).
Option ``fp8_w_fb`` also stores W_fb as FP8 E4M3 with one FP32 scale per row (no draw): the
scale is the row's largest |W| / 448 (448 = the largest E4M3 value), and the codes are torch's
round-to-nearest-even conversion of W / scale.

Standard deviations are written N(mean, std).  Conv weights follow the default PyTorch Conv1d
bound 1/sqrt(fan_in) = 0.5 for fan_in = 4.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

DK = DV = 128
RANK = 128
CONV_K = 4


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (round to nearest even), via torch's conversion."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class LayerWeights:
    H: int
    dk: int
    dv: int
    r: int
    K: int
    W_fb: np.ndarray       # uint16 [H*dk, r]
    A_log: np.ndarray      # float32 [H]
    dt_bias: np.ndarray    # float32 [H*dk]
    conv_w: np.ndarray     # uint16 [3, H*dk, K]
    norm_w: np.ndarray     # float32 [dv]
    l2_eps: float = 1e-6
    norm_eps: float = 1e-5
    W_fb_fp8: Optional[np.ndarray] = None    # uint8 [H*dk, r] E4M3 codes (FP8 input path)
    W_fb_scale: Optional[np.ndarray] = None  # float32 [H*dk] per-row scales (FP8 input path)


@dataclass
class Pool:
    num_slots: int
    state_dtype: str                 # "f32" | "bf16"
    state: np.ndarray                # float32 or uint16 [num_slots, H, dk, dv]
    conv: np.ndarray                 # uint16 [num_slots, 3, K-1, H*dk]


@dataclass
class Case:
    name: str
    kind: str                        # "decode" | "verify" | "prefill"
    seed: int
    layer: LayerWeights
    pool: Pool
    slot_ids: np.ndarray             # int32 [B]
    # decode: [n_steps, B, ...];  verify / prefill: [B, T or L, ...]
    inputs: Dict[str, np.ndarray]
    accepted: Optional[np.ndarray] = None   # verify only, int32 [B]
    chunk: int = 64                          # prefill only
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.slot_ids.shape[0])

    @property
    def n_tokens(self) -> int:
        q = self.inputs["q"]
        return int(q.shape[0] * q.shape[1])


def _layer(rng, H, dk=DK, dv=DV, r=RANK, K=CONV_K) -> LayerWeights:
    W_fb = to_bf16_bits(rng.normal(0.0, 0.02, size=(H * dk, r)).astype(np.float32))
    A_log = rng.uniform(-1.0, 1.0, size=(H,)).astype(np.float32)
    dt_bias = np.zeros((H * dk,), np.float32)
    conv_w = to_bf16_bits(rng.uniform(-0.5, 0.5, size=(3, H * dk, K)).astype(np.float32))
    norm_w = np.ones((dv,), np.float32)
    return LayerWeights(H, dk, dv, r, K, W_fb, A_log, dt_bias, conv_w, norm_w)


E4M3_MAX = 448.0


def quantize_w_fb_fp8(layer: LayerWeights) -> None:
    """Adds the FP8 E4M3 form of W_fb with one FP32 scale per row: scale = max|W_row| / 448,
    codes = E4M3(W / scale) by torch's conversion (round to nearest even)."""
    import torch

    W = torch.from_numpy(bf16_bits_to_f32(layer.W_fb))
    amax = W.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (W / scale[:, None]).to(torch.float8_e4m3fn)
    layer.W_fb_fp8 = codes.view(torch.uint8).numpy().copy()
    layer.W_fb_scale = scale.numpy().astype(np.float32)


def e4m3_codes_to_f32(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) -> float32 values by torch's conversion (exact)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _pool(rng, num_slots, H, dk, dv, K, state_dtype, state_std) -> Pool:
    shape = (num_slots, H, dk, dv)
    if state_std > 0:
        st = rng.standard_normal(size=shape, dtype=np.float32)
        st *= np.float32(state_std)
    else:
        st = np.zeros(shape, np.float32)
    if state_dtype == "bf16":
        st = to_bf16_bits(st)
    conv = np.zeros((num_slots, 3, K - 1, H * dk), np.uint16)
    return Pool(num_slots, state_dtype, st, conv)


def _token_inputs(rng, lead, H, dk, dv, r) -> Dict[str, np.ndarray]:
    def n(*shape):
        return to_bf16_bits(rng.standard_normal(size=lead + shape, dtype=np.float32))

    out = {}
    out["q"] = n(H * dk)
    out["k"] = n(H * dk)
    out["v"] = n(H * dv)
    out["f_a"] = n(r)
    out["beta"] = n(H)
    out["gate"] = n(H * dv)
    return out


def _extras(rng, layer: LayerWeights, pool: Pool, random_conv, random_norm, random_dt_bias):
    if random_conv:
        pool.conv = to_bf16_bits(rng.standard_normal(size=pool.conv.shape, dtype=np.float32))
    if random_norm:
        layer.norm_w = (1.0 + 0.25 * rng.standard_normal(size=layer.norm_w.shape)).astype(np.float32)
    if random_dt_bias:
        layer.dt_bias = (0.5 * rng.standard_normal(size=layer.dt_bias.shape)).astype(np.float32)


def make_decode(name="decode", seed=0, B=1, H=2, n_steps=8, num_slots=None, state_dtype="f32",
                state_std=0.0, dk=DK, dv=DV, r=RANK, K=CONV_K, random_conv=False,
                random_norm=False, random_dt_bias=False, fp8_w_fb=False) -> Case:
    num_slots = B if num_slots is None else num_slots
    rng = np.random.default_rng(seed)
    layer = _layer(rng, H, dk, dv, r, K)
    slot_ids = rng.permutation(num_slots)[:B].astype(np.int32)
    pool = _pool(rng, num_slots, H, dk, dv, K, state_dtype, state_std)
    inputs = _token_inputs(rng, (n_steps, B), H, dk, dv, r)
    _extras(rng, layer, pool, random_conv, random_norm, random_dt_bias)
    if fp8_w_fb:
        quantize_w_fb_fp8(layer)
    return Case(name, "decode", seed, layer, pool, slot_ids, inputs)


def make_verify(name="verify", seed=3, B=64, H=8, T=4, num_slots=256, state_dtype="f32",
                state_std=0.1, dk=DK, dv=DV, r=RANK, K=CONV_K, random_conv=False,
                random_norm=False, random_dt_bias=False, fp8_w_fb=False) -> Case:
    rng = np.random.default_rng(seed)
    layer = _layer(rng, H, dk, dv, r, K)
    slot_ids = rng.permutation(num_slots)[:B].astype(np.int32)
    pool = _pool(rng, num_slots, H, dk, dv, K, state_dtype, state_std)
    inputs = _token_inputs(rng, (B, T), H, dk, dv, r)
    accepted = rng.integers(0, T + 1, size=(B,)).astype(np.int32)
    _extras(rng, layer, pool, random_conv, random_norm, random_dt_bias)
    if fp8_w_fb:
        quantize_w_fb_fp8(layer)
    return Case(name, "verify", seed, layer, pool, slot_ids, inputs, accepted=accepted)


def make_prefill(name="prefill", seed=4, B=4, L=4096, H=8, chunk=64, num_slots=None,
                 state_dtype="f32", state_std=0.0, dk=DK, dv=DV, r=RANK, K=CONV_K,
                 random_conv=False, random_norm=False, random_dt_bias=False, fp8_w_fb=False) -> Case:
    num_slots = 2 * B if num_slots is None else num_slots
    rng = np.random.default_rng(seed)
    layer = _layer(rng, H, dk, dv, r, K)
    slot_ids = rng.permutation(num_slots)[:B].astype(np.int32)
    pool = _pool(rng, num_slots, H, dk, dv, K, state_dtype, state_std)
    inputs = _token_inputs(rng, (B, L), H, dk, dv, r)
    _extras(rng, layer, pool, random_conv, random_norm, random_dt_bias)
    if fp8_w_fb:
        quantize_w_fb_fp8(layer)
    return Case(name, "prefill", seed, layer, pool, slot_ids, inputs, chunk=chunk)


# The five measured workloads.  Pool sizes not fixed by the workload descriptions are readings:
# decode_small uses a one-slot pool, prefill_b4 a pool of 2*B slots.
WORKLOADS = {
    "decode_small": dict(kind="decode", seed=0, B=1, H=2, n_steps=8, num_slots=1,
                         state_dtype="f32", state_std=0.0),
    "decode_b64": dict(kind="decode", seed=1, B=64, H=8, n_steps=64, num_slots=256,
                       state_dtype="f32", state_std=0.1),
    "decode_b256": dict(kind="decode", seed=2, B=256, H=32, n_steps=16, num_slots=512,
                        state_dtype="bf16", state_std=0.1),
    "verify_b64": dict(kind="verify", seed=3, B=64, H=8, T=4, num_slots=256,
                       state_dtype="f32", state_std=0.1),
    "prefill_b4": dict(kind="prefill", seed=4, B=4, L=4096, H=8, chunk=64, num_slots=8,
                       state_dtype="f32", state_std=0.0),
}


def make(name: str, **overrides) -> Case:
    """Build one of the named workloads; keyword overrides change sizes for smaller cases."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    kind = spec.pop("kind")
    fn = {"decode": make_decode, "verify": make_verify, "prefill": make_prefill}[kind]
    return fn(name=name, **spec)
