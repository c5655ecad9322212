"""C-ABI checks that need no GPU: the library loads, exports what the header
declares, struct layouts agree, and argument errors come back before any CUDA call.

Regression cases follow the "SuperKittens PR #7" review: a caller struct
shorter than the library's must be rejected (not read past), and errors must
be reported, not returned as success.
"""
import ctypes as C
import os
import subprocess

import pytest

import workload as W
from sequence_decode_step_gb300 import _binding as B


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(B.LIB_PATH):
        from sequence_decode_step_gb300 import build_lib
        build_lib.build()
    return B.lib()


def test_exports_every_header_symbol(L):
    names = B.header_symbols()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)


def test_struct_layouts_match(L):
    assert L.qw_abi_version() == B.QW_ABI_VERSION
    assert L.qw_sizeof_config() == C.sizeof(B.qw_config) == 72
    assert L.qw_sizeof_weights() == C.sizeof(B.qw_weights) == 208
    assert L.qw_sizeof_lora() == C.sizeof(B.qw_lora) == 48
    assert B.qw_weights.lm_head.offset == 24 and B.qw_weights.attn_norm.offset == 40


def test_short_config_struct_rejected(L):
    cfg = B.make_config(W.TINY, 64)
    cfg.struct_size = C.sizeof(B.qw_config) - 4      # a caller built against an older header
    h = C.c_void_p()
    assert L.qw_create(C.byref(cfg), None, C.byref(h)) == B.QW_ERR_ABI
    assert h.value is None
    assert "struct_size" in B.last_error()
    cfg = B.make_config(W.TINY, 64)
    cfg.abi_version = 99
    assert L.qw_create(C.byref(cfg), None, C.byref(h)) == B.QW_ERR_ABI


@pytest.mark.parametrize("field,value", [("head_dim", 96), ("n_kv_heads", 3), ("hidden", 0),
                                         ("max_ctx", 0), ("hidden", 250), ("weight_format", 3),
                                         ("kv_format", 2)])
def test_bad_config_rejected_before_cuda(L, field, value):
    cfg = B.make_config(W.TINY, 64)
    setattr(cfg, field, value)
    h = C.c_void_p()
    assert L.qw_create(C.byref(cfg), None, C.byref(h)) == B.QW_ERR_ARG
    assert B.last_error()


def test_null_arguments_rejected(L):
    assert L.qw_create(None, None, None) == B.QW_ERR_ARG
    assert L.qw_load_weights(None, None) == B.QW_ERR_ARG
    assert L.qw_decode_step(None, 0, None, None) == B.QW_ERR_ARG
    assert L.qw_quantize_int4_g128(None, 4, 128, None, None, None) == B.QW_ERR_ARG
    assert L.qw_quantize_int4_g128(1, 4, 100, 1, 1, None) == B.QW_ERR_ARG   # cols % 128
    assert L.qw_attention_workspace_bytes(16, 8, 128, 19) > 16 * 19 * 128 * 4
    assert L.qw_lm_head_workspace_bytes() >= 256 + 8 * 1024
    L.qw_destroy(None)


def test_sample_arguments_checked_before_cuda(L):
    # qw_sample validates its arguments on the host: no device is touched here
    V = 151936
    ws = L.qw_sample_workspace_bytes(V, 64)
    assert ws >= (V // 1024) * 64 * 8
    assert L.qw_sample_workspace_bytes(0, 8) == 0
    assert L.qw_sample(None, V, 1.0, 8, 0.9, 0.5, None, None, 0, None) == B.QW_ERR_ARG
    bad = [(V, 1.0, 0, 0.9, 0.5),      # top_k below 1
           (V, 1.0, 257, 0.9, 0.5),    # top_k above 256
           (V, 1.0, 8, 0.0, 0.5),      # top_p not above 0
           (V, 1.0, 8, 0.9, 1.0),      # u not below 1
           (V, 1.0, 8, 0.9, -0.1),     # u below 0
           (0, 1.0, 8, 0.9, 0.5),      # empty row
           (1 << 22, 1.0, 256, 0.9, 0.5)]  # final sort would exceed one CTA
    for vocab, t, k, p, u in bad:
        assert L.qw_sample(1, vocab, t, k, p, u, 1, 1, 1 << 30, None) == B.QW_ERR_ARG, (vocab, k, p, u)
    assert L.qw_sample(1, V, 1.0, 64, 0.9, 0.5, 1, 1, ws - 8, None) == B.QW_ERR_ARG  # workspace
    assert L.qw_sample_last(None, 1.0, 8, 0.9, 0.5, None) == B.QW_ERR_ARG


def test_attention_arguments_checked_before_any_launch(L):
    # every case returns from the host checks: no kernel runs on these dummy pointers
    a = (1, None, None, 1, 1)
    # nq = 0 is an empty shape, not a zero-size workspace
    assert L.qw_attention_decode(*a, 0, 8, 128, 16, 3, 1e-6, 1e6, 4, 1, 1, 1 << 30,
                                 None) == B.QW_ERR_ARG
    # head_dim 64, one query head per KV head: 20000 splits overflow the combine's buffers
    assert L.qw_attention_decode(*a, 1, 1, 64, 40000, 39999, 1e-6, 1e6, 20000, 1, 1, 1 << 34,
                                 None) == B.QW_ERR_ARG
    assert "n_splits" in B.last_error()
    assert L.qw_attention_decode_noalloc(*a, 2, 2, 64, 20000, 19999, 1e-6, 1e6, 13000, 1,
                                         None) == B.QW_ERR_ARG
    assert "n_splits" in B.last_error()
    assert L.qw_attention_decode_noalloc(*a, 0, 2, 64, 8, 3, 1e-6, 1e6, 4, 1, None) == B.QW_ERR_ARG
    assert "shape" in B.last_error()
    assert L.qw_attention_decode_noalloc(None, None, None, 1, 1, 2, 2, 64, 8, 3, 1e-6, 1e6, 4, 1,
                                         None) == B.QW_ERR_ARG
    assert "null" in B.last_error()
    # 16 heads x 1000 splits x (128 + 2) floats is about 8 MB, beyond the 1 MiB array
    assert L.qw_attention_decode_noalloc(*a, 16, 8, 128, 10, 0, 1e-6, 1e6, 1000, 1,
                                         None) == B.QW_ERR_SIZE
    assert "1 MiB" in B.last_error()


def test_int4_gemv_arguments_checked_before_any_launch(L):
    assert L.qw_gemv_int4_workspace_bytes(3, 256) == 256 + 3 * (128 + 16)
    assert L.qw_gemv_int4_workspace_bytes(3, 100) == 0
    ws = L.qw_gemv_int4_workspace_bytes(8, 384)
    assert L.qw_gemv_int4_g128(None, 1, 8, 384, 1, 1, 16, ws, None) == B.QW_ERR_ARG
    assert L.qw_gemv_int4_g128(1, 1, 8, 200, 1, 1, 16, 1 << 20, None) == B.QW_ERR_ARG  # cols % 128
    assert L.qw_gemv_int4_g128(1, 1, 8, 384, 1, 1, 16, ws - 16, None) == B.QW_ERR_ARG  # short
    assert L.qw_gemv_int4_g128(1, 1, 8, 384, 1, 1, 8, ws, None) == B.QW_ERR_ARG       # unaligned
    assert "workspace" in B.last_error()


def test_q8_0_arguments_checked_before_any_launch(L):
    assert L.qw_quantize_q8_0(None, 4, 64, 1, 1, None) == B.QW_ERR_ARG
    assert L.qw_quantize_q8_0(1, 4, 48, 1, 1, None) == B.QW_ERR_ARG          # cols % 32
    assert L.qw_gemv_q8_0_workspace_bytes(3, 64) == 256 + 3 * (64 + 16)
    assert L.qw_gemv_q8_0_workspace_bytes(3, 40) == 0
    ws = L.qw_gemv_q8_0_workspace_bytes(8, 96)
    assert L.qw_gemv_q8_0(None, 1, 8, 96, 1, 1, 16, ws, None) == B.QW_ERR_ARG
    assert L.qw_gemv_q8_0(1, 1, 8, 96, 1, 1, 16, ws - 16, None) == B.QW_ERR_ARG   # short
    assert L.qw_gemv_q8_0(1, 1, 8, 96, 1, 1, 8, ws, None) == B.QW_ERR_ARG         # unaligned
    # a Q8_0 model needs hidden, q width and intermediate in multiples of 32
    cfg = B.make_config(W.TINY.replace(weight_format="q8_0", hidden=248), 64)
    h = C.c_void_p()
    assert L.qw_create(C.byref(cfg), None, C.byref(h)) == B.QW_ERR_ARG
    assert "32 for Q8_0" in B.last_error()
