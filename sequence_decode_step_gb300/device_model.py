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


def _to_dev(arr):
    """A host array (uint16 bf16 bits become int16) on the device; device tensors pass."""
    import torch
    if isinstance(arr, torch.Tensor):
        return arr
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to("cuda")


class DeviceModel:
    """One qw handle with its weights loaded from a dict of drawn arrays.

    ``weights`` maps the workload's names to uint16 bf16 bits (or float32 for
    tensors an int4 or Q8_0 model quantises on the device with qw_quantize_int4_g128 or
    qw_quantize_q8_0), as host arrays or as device tensors (int16 for bf16 bits).
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

        int4 = s.weight_format == "int4_g128"
        q8 = s.weight_format == "q8_0"
        L_ = B.lib()

        def up(name):
            t = _to_dev(weights[name])
            keep.append(t)
            return t.data_ptr()

        def up_q(name):
            """float32 [rows, K] -> int4 g128 (packed nibbles, bf16 scales) or Q8_0 (int8,
            fp16 scales) on the device, with the library's quantiser."""
            src = weights[name]
            w32 = src if isinstance(src, torch.Tensor) else \
                _to_dev(np.ascontiguousarray(src, dtype=np.float32))
            rows, K = w32.shape
            if q8:
                packed = torch.empty((rows, K), dtype=torch.int8, device="cuda")
                scales = torch.empty((rows, K // 32), dtype=torch.int16, device="cuda")
                B.check("qw_quantize_q8_0",
                        L_.qw_quantize_q8_0(w32.data_ptr(), rows, K, packed.data_ptr(),
                                            scales.data_ptr(), None))
            else:
                packed = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
                scales = torch.empty((rows, K // 128), dtype=torch.int16, device="cuda")
                B.check("qw_quantize_int4_g128",
                        L_.qw_quantize_int4_g128(w32.data_ptr(), rows, K, packed.data_ptr(),
                                                 scales.data_ptr(), None))
            keep.extend([packed, scales])
            torch.cuda.synchronize()
            del w32
            return packed.data_ptr(), scales.data_ptr()

        L = s.n_layers
        lists = {}

        def per_layer(nm, present=True):
            if not present:
                return None
            return B.ptr_array([up(f"layers.{l}.{nm}") for l in range(L)])

        def per_layer_q(nm):
            ps = [up_q(f"layers.{l}.{nm}") for l in range(L)]
            return B.ptr_array([p for p, _ in ps]), B.ptr_array([q for _, q in ps])

        w = B.qw_weights()
        w.struct_size = C.sizeof(B.qw_weights)
        w.embed = up("embed")
        w.final_norm = up("final_norm")
        if s.tie_word_embeddings:
            w.lm_head = None
        elif int4 or q8:
            w.lm_head, w.lm_head_scales = up_q("lm_head")
        else:
            w.lm_head = up("lm_head")
        for nm in ("attn_norm", "mlp_norm"):
            lists[nm] = per_layer(nm)
        for nm in ("q", "k", "v", "o", "gate", "up", "down"):
            if int4 or q8:
                lists[nm], lists[nm + "_scales"] = per_layer_q(nm)
            else:
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

    def sample(self, temperature: float, top_k: int, top_p: float, u: float) -> int:
        """Sampled id from the logits of the last step (the row stays on the device)."""
        return B.qw_sample_last(self.h, temperature, top_k, top_p, u)

    def _logits_buf(self):
        import torch
        if not hasattr(self, "_lg"):
            self._lg = torch.empty(self.shape.vocab, dtype=torch.float32, device="cuda")
        return self._lg

    # -- state hooks -------------------------------------------------------------------
    def _kv_raw(self, layer: int):
        """Live device views of one layer's K and V cache (f32, or int16-typed bf16 bits)."""
        k, v = B.qw_kv_cache(self.h, layer)
        shp = (self.shape.n_kv_heads, self.max_ctx, self.shape.head_dim)
        dt = "<i2" if getattr(self.shape, "kv_format", "f32") == "bf16" else "<f4"
        return device_view(k, shp, dt), device_view(v, shp, dt)

    def kv(self, layer: int):
        """K and V of one layer as f32 tensors: live views of an f32 cache, widened
        copies of a bf16 one."""
        import torch
        k, v = self._kv_raw(layer)
        if k.dtype == torch.int16:
            widen = lambda t: (t.to(torch.int32) << 16).view(torch.float32)
            return widen(k), widen(v)
        return k, v

    def set_lora(self, lora, alpha: float = 0.0) -> None:
        """Set (dict 'lora.{l}.q_a' ... of bf16 bits) or clear (None) the adapter; the
        uploaded tensors are kept alive here because the library borrows them."""
        if lora is None:
            B.qw_set_lora(self.h, None)
            self._lora_keep = None
            return
        L = self.shape.n_layers
        keep = {}
        arrays = {}
        for nm in ("q_a", "q_b", "v_a", "v_b"):
            ts = [_to_dev(lora[f"lora.{l}.{nm}"]) for l in range(L)]
            keep[nm] = ts
            arrays[nm] = B.ptr_array([t.data_ptr() for t in ts])
        rank = lora["lora.0.q_a"].shape[0]
        st = B.qw_lora(struct_size=C.sizeof(B.qw_lora), rank=rank, alpha=alpha)
        for nm, arr in arrays.items():
            setattr(st, nm, C.cast(arr, B.PP))
        B.qw_set_lora(self.h, st)
        self._lora_keep = (keep, arrays)

    def set_kv(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        """Write f32 K, V [n_kv_heads, n, head_dim] into positions 0..n-1 (rounded to the
        nearest bf16 for a bf16 cache)."""
        import torch
        kd, vd = self._kv_raw(layer)
        n = k.shape[1]
        for dst, src in ((kd, k), (vd, v)):
            t = src if isinstance(src, torch.Tensor) else \
                torch.from_numpy(np.ascontiguousarray(src, dtype=np.float32))
            if dst.dtype == torch.int16:
                t = t.to(torch.bfloat16).view(torch.int16)
            dst[:, :n].copy_(t)
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
