"""The C-ABI library (no GPU needed): it loads, exports every entry point include/kda.h
declares, and rejects bad arguments on the host before launching anything.

Every call here fails host-side validation (or is a documented no-op), so no kernel is ever
launched with the fake pointers used below."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def K():
    import verify_kda_decode_gb300 as K
    return K


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kda_decode", "kda_verify", "kda_commit", "kda_decode_resume", "kda_verify_resume",
              "kda_prefill", "kda_prefill_workspace_size", "kda_prefill_varlen",
              "kda_get_error", "kda_status_string", "kda_last_error", "kda_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(K):
    lib = K.library()
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) <= set(K.kda.EXPORTS)
    assert lib.kda_abi_version() == 3


def _layer(K, H=2, dk=128, ptr=0x10000, w_dtype=0, scale=None):
    return K.kda._Layer(H, dk, 128, 128, 4, ptr, ptr, ptr, ptr, ptr, 1e-6, 1e-5, w_dtype, scale)


def _pool(K, slots=4, dtype=0, ptr=0x20000):
    return K.kda._Pool(ptr, dtype, ptr, slots, ptr)


def _decode(K, L, P, B, ptr=0x30000):
    lib = K.library()
    return lib.kda_decode(ctypes.byref(L) if L is not None else None,
                          ctypes.byref(P) if P is not None else None,
                          ptr, B, ptr, ptr, ptr, ptr, ptr, ptr, ptr, None)


def msg(K):
    return K.library().kda_last_error().decode()


def test_fp8_weights_need_a_valid_dtype_and_scales(K):
    kk = K.kda
    assert _decode(K, _layer(K, w_dtype=7), _pool(K), 1) == kk.KDA_ERR_INVALID_ARG
    assert "w_fb_dtype" in msg(K)
    assert _decode(K, _layer(K, w_dtype=kk.KDA_W_FP8_E4M3), _pool(K), 1) == kk.KDA_ERR_INVALID_ARG
    assert "W_fb_scale" in msg(K)
    assert _decode(K, _layer(K, w_dtype=kk.KDA_W_FP8_E4M3, scale=0x10008), _pool(K), 1) == kk.KDA_ERR_INVALID_ARG
    assert "W_fb_scale" in msg(K)   # not 16-byte aligned


def test_decode_rejects_bad_arguments(K):
    kk = K.kda
    assert _decode(K, None, _pool(K), 1) == kk.KDA_ERR_INVALID_ARG
    assert "layer" in msg(K)
    assert _decode(K, _layer(K), None, 1) == kk.KDA_ERR_INVALID_ARG
    assert _decode(K, _layer(K, dk=64), _pool(K), 1) == kk.KDA_ERR_UNSUPPORTED
    assert _decode(K, _layer(K, H=0), _pool(K), 1) == kk.KDA_ERR_INVALID_ARG
    assert _decode(K, _layer(K, ptr=0x10008), _pool(K), 1) == kk.KDA_ERR_INVALID_ARG
    assert "aligned" in msg(K)
    assert _decode(K, _layer(K), _pool(K, dtype=7), 1) == kk.KDA_ERR_INVALID_ARG
    assert _decode(K, _layer(K), _pool(K, slots=0), 1) == kk.KDA_ERR_INVALID_ARG
    assert _decode(K, _layer(K), _pool(K, slots=4), 5) == kk.KDA_ERR_INVALID_ARG
    assert "num_slots" in msg(K)
    assert _decode(K, _layer(K), _pool(K), -1) == kk.KDA_ERR_INVALID_ARG
    assert _decode(K, _layer(K), _pool(K), 1, ptr=0x30004) == kk.KDA_ERR_INVALID_ARG
    # B == 0 is a documented no-op (nothing launched)
    assert _decode(K, _layer(K), _pool(K), 0) == kk.KDA_OK


def test_verify_commit_prefill_reject_bad_sizes(K):
    kk, lib = K.kda, K.library()
    L, P, p = _layer(K), _pool(K), 0x30000
    for T in (0, 17, -3):
        assert lib.kda_verify(ctypes.byref(L), ctypes.byref(P), p, 1, T, p, p, p, p, p, p, p, p, p,
                              None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_verify(ctypes.byref(L), ctypes.byref(P), p, 1, 4, p, p, p, p, p, p, p, 0x30008, p,
                          None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_commit(ctypes.byref(P), 2, 128, 128, 4, p, p, 1, 0, p, p, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_commit(ctypes.byref(P), 2, 64, 128, 4, p, p, 1, 4, p, p, None) == kk.KDA_ERR_UNSUPPORTED
    assert lib.kda_commit(ctypes.byref(P), 2, 128, 128, 4, p, None, 1, 4, p, p, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill(ctypes.byref(L), ctypes.byref(P), p, 1, 10, 32, p, p, p, p, p, p, p, None, 0,
                           None) == kk.KDA_ERR_UNSUPPORTED
    assert lib.kda_prefill(ctypes.byref(L), ctypes.byref(P), p, 1, -1, 64, p, p, p, p, p, p, p, None, 0,
                           None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill(ctypes.byref(L), ctypes.byref(P), p, 1, 0, 64, p, p, p, p, p, p, p, None, 0,
                           None) == kk.KDA_OK
    assert lib.kda_prefill_workspace_size(ctypes.byref(L), 4, 4096, 32) == 0


def test_resume_entries_reject_bad_arguments(K):
    kk, lib = K.kda, K.library()
    L, P, p = ctypes.byref(_layer(K)), ctypes.byref(_pool(K)), 0x30000
    ins = (p, p, p, p, p, p, p)   # q, k, v, f_a, beta_logit, gate, out
    for Tp in (0, 17):   # previous step's T out of range
        assert lib.kda_decode_resume(L, P, p, 1, p, Tp, p, p, *ins, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_resume(L, P, p, 1, 0x30002, 4, p, p, *ins, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_resume(L, P, p, 1, p, 4, None, p, *ins, None) == kk.KDA_ERR_INVALID_ARG
    assert "prev_rec_state" in msg(K)
    assert lib.kda_decode_resume(L, P, p, 0, None, 0, None, None, *ins, None) == kk.KDA_OK
    assert lib.kda_verify_resume(L, P, p, 1, 0, None, None, 0, None, None, *ins, p, p, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_verify_resume(L, P, p, 1, 4, 0x30002, None, 0, None, None, *ins, p, p, None) == kk.KDA_ERR_INVALID_ARG
    assert "n_tokens" in msg(K)
    # the previous records may not be this step's records
    assert lib.kda_verify_resume(L, P, p, 1, 4, None, p, 4, 0x40000, 0x50000, *ins, 0x40000, 0x60000,
                                 None) == kk.KDA_ERR_INVALID_ARG
    assert "different buffers" in msg(K)
    assert lib.kda_verify_resume(L, P, p, 0, 4, None, None, 0, None, None, *ins, p, p, None) == kk.KDA_OK


def test_prefill_varlen_rejects_bad_arguments(K):
    kk, lib = K.kda, K.library()
    L, P, p = ctypes.byref(_layer(K)), ctypes.byref(_pool(K)), 0x30000
    ins = (p, p, p, p, p, p, p)   # q, k, v, f_a, beta_logit, gate, out
    ws = 0x40000
    need = lib.kda_prefill_varlen_workspace_size(L, 2, 100, 64)
    assert need > 0 and lib.kda_prefill_varlen_workspace_size(L, 2, 100, 32) == 0
    # args: layer, pool, slot_ids, B, cu_seqlens, total_tokens, max_len, chunk, ins..., ws, bytes
    assert lib.kda_prefill_varlen(L, P, p, 2, p, 100, 64, 32, *ins, ws, need, None) == kk.KDA_ERR_UNSUPPORTED
    assert lib.kda_prefill_varlen(L, P, p, 2, p, -1, 64, 64, *ins, ws, need, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_varlen(L, P, p, 2, p, 100, 0, 64, *ins, ws, need, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_varlen(L, P, p, 2, None, 100, 64, 64, *ins, ws, need, None) == kk.KDA_ERR_INVALID_ARG
    assert "cu_seqlens" in msg(K)
    assert lib.kda_prefill_varlen(L, P, p, 2, p, 100, 64, 64, *ins, ws, need - 1, None) == kk.KDA_ERR_INVALID_ARG
    assert "workspace_bytes" in msg(K)
    assert lib.kda_prefill_varlen(L, P, p, 2, p, 100, 64, 64, *ins, ws + 16, need, None) == kk.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_varlen(L, P, p, 0, p, 100, 64, 64, *ins, None, 0, None) == kk.KDA_OK
    assert lib.kda_prefill_varlen(L, P, p, 2, p, 0, 64, 64, *ins, None, 0, None) == kk.KDA_OK


def test_status_strings(K):
    lib = K.library()
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(4) == b"KDA_ERR_DEVICE"
    assert lib.kda_status_string(99) == b"KDA_ERR_UNKNOWN"


def test_python_binding_checks_shapes_before_calling(K):
    import torch

    lay = K.KdaLayer(W_fb=torch.zeros(256, 128, dtype=torch.bfloat16),
                     A_log=torch.zeros(2), dt_bias=torch.zeros(256),
                     conv_w=torch.zeros(3, 256, 4, dtype=torch.bfloat16), norm_w=torch.ones(128))
    with pytest.raises(ValueError):
        K.KdaLayer(W_fb=lay.W_fb, A_log=lay.A_log, dt_bias=torch.zeros(255), conv_w=lay.conv_w,
                   norm_w=lay.norm_w).c_struct()
    with pytest.raises(TypeError):
        K.KdaLayer(W_fb=lay.W_fb.float(), A_log=lay.A_log, dt_bias=lay.dt_bias, conv_w=lay.conv_w,
                   norm_w=lay.norm_w).c_struct()
    assert lay.c_struct().num_heads == 2
    pool = K.KdaPool.zeros(4, 2, device="cpu")
    ok = torch.zeros(2, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):   # q has the wrong width: caught before anything is bound
        K.prepare_decode(lay, pool, torch.zeros(2, dtype=torch.int32), ok[:, :255].contiguous(), ok, ok,
                         torch.zeros(2, 128, dtype=torch.bfloat16), torch.zeros(2, 2, dtype=torch.bfloat16),
                         ok, out=ok)
