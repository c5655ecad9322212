"""Put a drawn workload on the GPU and drive it through the qw_* C ABI.

PyTorch is used only for device memory (uploading the weight tensors, viewing
the library's KV cache); every computation is a libqw.so kernel.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

import numpy as np

from . import _binding as B


class _CudaArray:
    """Minimal __cuda_array_interface__ wrapper over a raw device pointer."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3,
                                         "strides": None}


def device_view(ptr: int, shape, dtype: str = "<f4"):
    import torch
    return torch.as_tensor(_CudaArray(ptr, shape, dtype), device="cuda")


def _to_dev(arr: np.ndarray):
    import torch
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


class DeviceModel:
    """One qw handle with its weights loaded from a dict of drawn arrays.

    ``weights`` maps the workload's names to uint16 bf16 bits (or float32 for
    tensors an int4 model quantises on the device with qw_quantize_int4_g128).
    """

    def __init__(self, shape, weights: Dict[str, np.ndarray], max_ctx: int,
                 max_prefill_t: int = 0, stream=None):
        import torch
        self.shape = shape
        self.max_ctx = max_ctx
        self.cfg = B.make_config(shape, max_ctx, max_prefill_t)
        self.h = B.qw_create(self.cfg, stream)
        self._lora_keep = None
        try:
            self.load(weights)
        except Exception:
            B.qw_destroy(self.h)
            raise
        torch.cuda.synchronize()

    # -- weights -----------------------------------------------------------------------
    def load(self, weights: Dict[str, np.ndarray]) -> None:
        import torch
        s = self.shape
        keep = []

        def up(name):
            t = _to_dev(weights[name])
            keep.append(t)
            return t.data_ptr()

        L = s.n_layers
        lists = {}

        def per_layer(nm, present=True):
            if not present:
                return None
            return B.ptr_array([up(f"layers.{l}.{nm}") for l in range(L)])

        w = B.qw_weights()
        w.struct_size = C.sizeof(B.qw_weights)
        w.embed = up("embed")
        w.final_norm = up("final_norm")
        w.lm_head = None if s.tie_word_embeddings else up("lm_head")
        for nm in ("attn_norm", "q", "k", "v", "o", "mlp_norm", "gate", "up", "down"):
            lists[nm] = per_layer(nm)
        lists["q_norm"] = per_layer("q_norm", s.qk_norm)
        lists["k_norm"] = per_layer("k_norm", s.qk_norm)
        for nm in ("q_bias", "k_bias", "v_bias"):
            lists[nm] = per_layer(nm, s.qkv_bias)
        for nm, arr in lists.items():
            if arr is not None:
                setattr(w, nm, C.cast(arr, B.PP))
        self._arrays = lists
        torch.cuda.synchronize()
        B.qw_load_weights(self.h, w)
        del keep
        torch.cuda.synchronize()

    # -- stepping ----------------------------------------------------------------------
    def prefill(self, ids, logits: bool = False):
        lg = self._logits_buf() if logits else None
        am = B.qw_prefill(self.h, list(ids), lg.data_ptr() if lg is not None else None)
        return (am, lg.cpu().numpy()) if logits else am

    def decode(self, token: int, logits: bool = False):
        lg = self._logits_buf() if logits else None
        am = B.qw_decode_step(self.h, token, lg.data_ptr() if lg is not None else None)
        return (am, lg.cpu().numpy()) if logits else am

    def greedy(self, token: int, n: int):
        return B.qw_decode_greedy(self.h, token, n)

    def _logits_buf(self):
        import torch
        if not hasattr(self, "_lg"):
            self._lg = torch.empty(self.shape.vocab, dtype=torch.float32, device="cuda")
        return self._lg

    # -- state hooks -------------------------------------------------------------------
    def kv(self, layer: int):
        k, v = B.qw_kv_cache(self.h, layer)
        shp = (self.shape.n_kv_heads, self.max_ctx, self.shape.head_dim)
        return device_view(k, shp), device_view(v, shp)

    def set_kv(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        import torch
        kd, vd = self.kv(layer)
        n = k.shape[1]
        kd[:, :n].copy_(torch.from_numpy(np.ascontiguousarray(k)))
        vd[:, :n].copy_(torch.from_numpy(np.ascontiguousarray(v)))
        torch.cuda.synchronize()

    def set_pos(self, pos: int) -> None:
        B.qw_set_pos(self.h, pos)

    def pos(self) -> int:
        return B.qw_get_pos(self.h)

    def reset(self) -> None:
        B.qw_reset(self.h)

    def set_capture(self, on: bool) -> None:
        B.qw_set_capture(self.h, on)

    def capture(self, which: int) -> np.ndarray:
        return B.qw_get_capture(self.h, which)

    def close(self) -> None:
        if self.h is not None:
            B.qw_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
