"""ctypes binding of include/qw.h: the same names, argument marshalling only.

Every computation runs in libqw.so; nothing here falls back to CPU code. If the
library is missing, ``lib()`` raises instead of silently degrading.
"""
from __future__ import annotations

import ctypes as C
import os
import re
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqw.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "qw.h")

QW_ABI_VERSION = 2
QW_OK = 0
QW_ERR_ABI = -1
QW_ERR_ARG = -2
QW_ERR_CTX = -3
QW_ERR_NOT_CAPTURED = -4
QW_ERR_SIZE = -5
QW_ERR_CUDA = -6
QW_ERR_DEVICE_TIMEOUT = -7
QW_ERR_STATE = -8
QW_ERR_NUMERIC = -9
QW_WEIGHTS_BF16 = 0
QW_WEIGHTS_INT4_G128 = 1
QW_WEIGHTS_Q8_0 = 2
QW_KV_F32 = 0
QW_KV_BF16 = 1
QW_CAPTURE_EMBEDDING = 0
QW_CAPTURE_BLOCK0 = 1
QW_CAPTURE_FINAL_NORM = 2
QW_CAPTURE_LOGITS = 3

_ERR_NAMES = {v: k for k, v in globals().items() if k.startswith("QW_ERR_")}


class QwError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} -> {_ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


PP = C.POINTER(C.c_void_p)  # host array of device pointers


class qw_config(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("abi_version", C.c_uint32),
                ("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("intermediate", C.c_int32),
                ("vocab", C.c_int32), ("eps", C.c_float), ("rope_theta", C.c_float),
                ("tie_word_embeddings", C.c_uint32), ("qk_norm", C.c_uint32),
                ("qkv_bias", C.c_uint32), ("max_ctx", C.c_int32), ("max_prefill_t", C.c_int32),
                ("weight_format", C.c_uint32), ("kv_format", C.c_uint32)]


_WEIGHT_LISTS = ["attn_norm", "q", "k", "v", "o", "mlp_norm", "gate", "up", "down", "q_norm",
                 "k_norm", "q_bias", "k_bias", "v_bias", "q_scales", "k_scales", "v_scales",
                 "o_scales", "gate_scales", "up_scales", "down_scales"]


class qw_weights(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("reserved0", C.c_uint32),
                ("embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("lm_head_scales", C.c_void_p)] + [(n, PP) for n in _WEIGHT_LISTS]


class qw_lora(C.Structure):
    _fields_ = [("struct_size", C.c_uint32), ("rank", C.c_int32), ("alpha", C.c_float),
                ("reserved0", C.c_uint32), ("q_a", PP), ("q_b", PP), ("v_a", PP), ("v_b", PP)]


_SIG = {
    "qw_abi_version": (C.c_uint32, []),
    "qw_sizeof_config": (C.c_size_t, []),
    "qw_sizeof_weights": (C.c_size_t, []),
    "qw_sizeof_lora": (C.c_size_t, []),
    "qw_create": (C.c_int, [C.POINTER(qw_config), C.c_void_p, C.POINTER(C.c_void_p)]),
    "qw_load_weights": (C.c_int, [C.c_void_p, C.POINTER(qw_weights)]),
    "qw_prefill": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_int32, C.c_void_p,
                             C.POINTER(C.c_int32)]),
    "qw_decode_step": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.POINTER(C.c_int32)]),
    "qw_decode_greedy": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.POINTER(C.c_int32)]),
    "qw_reset": (C.c_int, [C.c_void_p]),
    "qw_set_lora": (C.c_int, [C.c_void_p, C.POINTER(qw_lora)]),
    "qw_kv_cache": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_void_p),
                              C.POINTER(C.c_void_p)]),
    "qw_set_pos": (C.c_int, [C.c_void_p, C.c_int32]),
    "qw_get_pos": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32)]),
    "qw_set_capture": (C.c_int, [C.c_void_p, C.c_int32]),
    "qw_capture_size": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_size_t)]),
    "qw_get_capture": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_size_t]),
    "qw_set_wait_limit_ns": (C.c_int, [C.c_void_p, C.c_uint64]),
    "qw_set_decode_path": (C.c_int, [C.c_void_p, C.c_int32]),
    "qw_get_decode_path": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32)]),
    "qw_last_error": (C.c_char_p, [C.c_void_p]),
    "qw_destroy": (None, [C.c_void_p]),
    "qw_quantize_int4_g128": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p,
                                        C.c_void_p, C.c_void_p]),
    "qw_attention_workspace_bytes": (C.c_size_t, [C.c_int32] * 4),
    "qw_attention_decode": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                      C.c_int32, C.c_float, C.c_float, C.c_int32, C.c_void_p,
                                      C.c_void_p, C.c_size_t, C.c_void_p]),
    "qw_attention_noalloc_max_bytes": (C.c_size_t, []),
    "qw_attention_decode_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                              C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                              C.c_int32, C.c_int32, C.c_float, C.c_float,
                                              C.c_int32, C.c_void_p, C.c_void_p]),
    "qw_gemm_bf16": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                               C.c_int32, C.c_void_p, C.c_int32, C.c_void_p]),
    "qw_sample_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "qw_sample": (C.c_int, [C.c_void_p, C.c_int32, C.c_float, C.c_int32, C.c_float, C.c_float,
                            C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "qw_sample_last": (C.c_int, [C.c_void_p, C.c_float, C.c_int32, C.c_float, C.c_float,
                                 C.POINTER(C.c_int32)]),
    "qw_gemv_int4_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "qw_gemv_int4_g128": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "qw_quantize_q8_0": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                   C.c_void_p]),
    "qw_gemv_q8_0_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "qw_gemv_q8_0": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p,
                               C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "qw_lm_head_workspace_bytes": (C.c_size_t, []),
    "qw_lm_head_argmax": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                    C.c_float, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t,
                                    C.c_void_p]),
}

_lib: Optional[C.CDLL] = None


def header_symbols() -> list:
    """Names of the functions include/qw.h declares."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"\b(qw_[a-z0-9_]+)\s*\(", txt)))


def lib() -> C.CDLL:
    """Load libqw.so (built by build_lib.build()); raises if it is not there."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                               "(nvcc, sm_103a) first; there is no fallback")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        for name, st in (("qw_sizeof_config", qw_config), ("qw_sizeof_weights", qw_weights),
                         ("qw_sizeof_lora", qw_lora)):
            if getattr(L, name)() != C.sizeof(st):
                raise RuntimeError(f"ctypes {st.__name__} ({C.sizeof(st)} B) does not match "
                                   f"the library ({getattr(L, name)()} B)")
        _lib = L
    return _lib


def last_error(h=None) -> str:
    m = lib().qw_last_error(h)
    return m.decode() if m else ""


def check(fn: str, rc: int, h=None) -> None:
    if rc != QW_OK:
        raise QwError(fn, rc, last_error(h))


def ptr_array(ptrs) -> C.Array:
    """Host array of device pointers (ints or None)."""
    return (C.c_void_p * len(ptrs))(*[p if p else None for p in ptrs])


def make_config(shape, max_ctx: int, max_prefill_t: int = 0) -> qw_config:
    """qw_config from a workload shape (fields named as in include/qw.h)."""
    return qw_config(
        struct_size=C.sizeof(qw_config), abi_version=QW_ABI_VERSION,
        n_layers=shape.n_layers, hidden=shape.hidden, n_q_heads=shape.n_q_heads,
        n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, intermediate=shape.intermediate,
        vocab=shape.vocab, eps=shape.eps, rope_theta=shape.rope_theta,
        tie_word_embeddings=int(shape.tie_word_embeddings), qk_norm=int(shape.qk_norm),
        qkv_bias=int(shape.qkv_bias), max_ctx=max_ctx, max_prefill_t=max_prefill_t,
        weight_format={"int4_g128": QW_WEIGHTS_INT4_G128,
                       "q8_0": QW_WEIGHTS_Q8_0}.get(shape.weight_format, QW_WEIGHTS_BF16),
        kv_format=QW_KV_BF16 if getattr(shape, "kv_format", "f32") == "bf16" else QW_KV_F32)


# -- thin wrappers with the C names (raise QwError on a non-zero status) --------
def qw_create(cfg: qw_config, stream=None) -> C.c_void_p:
    h = C.c_void_p()
    check("qw_create", lib().qw_create(C.byref(cfg), stream, C.byref(h)))
    return h


def qw_load_weights(h, w: qw_weights) -> None:
    check("qw_load_weights", lib().qw_load_weights(h, C.byref(w)), h)


def qw_prefill(h, ids, logits_dev=None, want_argmax=True) -> Optional[int]:
    arr = (C.c_int32 * len(ids))(*[int(i) for i in ids])
    out = C.c_int32(-1)
    check("qw_prefill", lib().qw_prefill(h, arr, len(ids), logits_dev,
                                         C.byref(out) if want_argmax else None), h)
    return out.value if want_argmax else None


def qw_decode_step(h, token: int, logits_dev=None, want_argmax=True) -> Optional[int]:
    out = C.c_int32(-1)
    check("qw_decode_step", lib().qw_decode_step(h, int(token), logits_dev,
                                                 C.byref(out) if want_argmax else None), h)
    return out.value if want_argmax else None


def qw_decode_greedy(h, token: int, n_steps: int) -> list:
    ids = (C.c_int32 * n_steps)()
    check("qw_decode_greedy", lib().qw_decode_greedy(h, int(token), n_steps, ids), h)
    return list(ids)


def qw_reset(h) -> None:
    check("qw_reset", lib().qw_reset(h), h)


def qw_set_lora(h, lora: Optional[qw_lora]) -> None:
    check("qw_set_lora", lib().qw_set_lora(h, C.byref(lora) if lora is not None else None), h)


def qw_kv_cache(h, layer: int):
    k, v = C.c_void_p(), C.c_void_p()
    check("qw_kv_cache", lib().qw_kv_cache(h, layer, C.byref(k), C.byref(v)), h)
    return k.value, v.value


def qw_set_pos(h, pos: int) -> None:
    check("qw_set_pos", lib().qw_set_pos(h, pos), h)


def qw_get_pos(h) -> int:
    p = C.c_int32()
    check("qw_get_pos", lib().qw_get_pos(h, C.byref(p)), h)
    return p.value


def qw_set_capture(h, enable: bool) -> None:
    check("qw_set_capture", lib().qw_set_capture(h, int(enable)), h)


def qw_get_capture(h, which: int):
    import numpy as np
    n = C.c_size_t()
    check("qw_capture_size", lib().qw_capture_size(h, which, C.byref(n)), h)
    out = np.empty(n.value, dtype=np.float32)
    check("qw_get_capture", lib().qw_get_capture(h, which, out.ctypes.data, n.value), h)
    return out


def qw_set_wait_limit_ns(h, ns: int) -> None:
    check("qw_set_wait_limit_ns", lib().qw_set_wait_limit_ns(h, int(ns)), h)


def qw_destroy(h) -> None:
    lib().qw_destroy(h)


def qw_set_decode_path(h, path: int) -> None:
    check("qw_set_decode_path", lib().qw_set_decode_path(h, int(path)), h)


def qw_sample_last(h, temperature: float, top_k: int, top_p: float, u: float) -> int:
    """Sampled id from the handle's last logits (temperature / top-k / top-p, draw u)."""
    t = C.c_int32()
    check("qw_sample_last", lib().qw_sample_last(h, float(temperature), int(top_k), float(top_p),
                                                 float(u), C.byref(t)), h)
    return t.value


def qw_sample(logits_ptr: int, vocab: int, temperature: float, top_k: int, top_p: float,
              u: float, token_ptr: int, workspace_ptr: int, workspace_bytes: int,
              stream: Optional[int] = None) -> None:
    """Queue one sampling of a device logits row; the id lands in device memory."""
    check("qw_sample", lib().qw_sample(logits_ptr, int(vocab), float(temperature), int(top_k),
                                       float(top_p), float(u), token_ptr, workspace_ptr,
                                       int(workspace_bytes), stream))


def qw_get_decode_path(h) -> int:
    p = C.c_int32()
    check("qw_get_decode_path", lib().qw_get_decode_path(h, C.byref(p)), h)
    return p.value
