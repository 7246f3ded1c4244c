"""Negative controls: plant a plausible mistake in a copy of the oracle, on the CPU, and check
that at least one pin in ``test_oracle_pins`` fails for it.  The planted copies are built in a
temporary directory; the committed oracle is never modified."""
from __future__ import annotations

import ctypes
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

MUTATIONS = {
    "u_sign": ("double u = v[j] - stk;", "double u = v[j] + stk;"),
    "decay_dropped": ("S[(size_t)i * dv + j] *= alpha[i];", "S[(size_t)i * dv + j] *= 1.0;"),
    "q_scale_dropped": ("/ sqrt((double)L->dk);", ";"),
    "conv_taps_reversed": ("acc += bf16_to_f64(w[j]) * win", "acc += bf16_to_f64(w[K - 2 - j]) * win"),
    "softplus_dropped": ("-a * softplus(graw + L->dt_bias[h * L->dk + i]);",
                         "-a * (graw + L->dt_bias[h * L->dk + i]);"),
    "rms_sum_not_mean": ("ss / dv + eps", "ss + eps"),
    "gate_not_sigmoid": ("norm_w[j] * sigmoid(bf16_to_f64(gate[j]))", "norm_w[j] * bf16_to_f64(gate[j])"),
    "beta_dropped": ("S[(size_t)i * dv + j] += beta * k[i] * u;", "S[(size_t)i * dv + j] += k[i] * u;"),
    "output_reads_key": ("acc += S[(size_t)i * dv + j] * q[i];", "acc += S[(size_t)i * dv + j] * k[i];"),
    "chunk_M_sign": ("M[(size_t)t * C + s] = bet[t] * acc;", "M[(size_t)t * C + s] = -bet[t] * acc;"),
    "commit_wrong_record": ("rec_state + ((size_t)b * T + (n - 1)) * sz",
                            "rec_state + ((size_t)b * T + n % T) * sz"),
    "bf16_truncates": ("nearbyint(scaled)", "trunc(scaled)"),
    # where the storage rounding falls: decode rounds after every token, prefill once at the end
    "decode_rounds_only_at_end": (
        "out + tb * H * dv + (size_t)h * dv, scr);\n"
        "                for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);\n"
        "            }\n",
        "out + tb * H * dv + (size_t)h * dv, scr);\n"
        "            }\n"
        "            for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);\n"),
    "decode_never_rounds": (
        "out + tb * H * dv + (size_t)h * dv, scr);\n"
        "                for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);\n",
        "out + tb * H * dv + (size_t)h * dv, scr);\n"),
    "prefill_rounds_every_token": (
        "out + bt * H * dv + (size_t)h * dv, scr);\n"
        "            }\n"
        "            for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);\n",
        "out + bt * H * dv + (size_t)h * dv, scr);\n"
        "                for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);\n"
        "            }\n"),
    "prefill_never_rounds": (
        "out + bt * H * dv + (size_t)h * dv, scr);\n"
        "            }\n"
        "            for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);\n",
        "out + bt * H * dv + (size_t)h * dv, scr);\n"
        "            }\n"),
    "e4m3_wrong_bias": ("else v = ldexp(8.0 + m, e - 10);", "else v = ldexp(8.0 + m, e - 11);"),
    "e4m3_subnormal_as_normal": ("if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp(8.0 + m, -10);"),
    "fp8_scale_dropped": ("graw += L->W_fb_scale[row] * kdo_e4m3_to_f64(w8[j])", "graw += kdo_e4m3_to_f64(w8[j])"),
    "bf16_storage_rounds_to_f32": ("if (storage == KDO_STORE_BF16) return round_to_bf16(x);",
                                   "if (storage == KDO_STORE_BF16) return (double)(float)x;"),
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        combos = [{}]
        for m in params:          # every combination of the parametrize values
            combos = [dict(c, **{m.args[0]: v}) for c in combos for v in m.args[1]]
        out.extend((name, fn, kw) for kw in combos)
    return out


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, tmp_path, monkeypatch):
    before, after = MUTATIONS[mutation]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor not found exactly once: {before}"
    mutated = tmp_path / "kda_oracle_mut.c"
    mutated.write_text(src.replace(before, after))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(mutated), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(so))
    lib.kdo_f32_to_bf16.restype = ctypes.c_uint16
    lib.kdo_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.kdo_e4m3_to_f64.restype = ctypes.c_double
    lib.kdo_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for name, fn, kwargs in _pin_functions():
        try:
            fn(**kwargs)
        except AssertionError:
            failed.append(name)
        except RuntimeError:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mutation}"
