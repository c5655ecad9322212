"""Oracle for the batch-1 Qwen-style decode step and its causal prefill.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module. The CUDA
path (``sequence_decode_step_gb300``) never imports it and shares no code with it.

It is the plain definition of the network, written out step by step:

  * "Failed Star / fs, M2" page, "One prefill, all shapes visible": ids are
    gathered from the embedding table, pass x28 blocks, a row-wise final
    RMSNorm, then the last row is projected by the tied table used as a [V,H]
    linear.
  * Same page, residual-bus paragraph: each sublayer reads a normalised copy of
    the bus and adds its output back; a block is RMSNorm -> QK-norm, RoPE, GQA
    causal attention -> o_proj (+bus) -> RMSNorm -> SwiGLU -> down (+bus).
  * Same page, "Correct before fast": linear layers dot the input with stored
    [out, in] weight rows; bf16 weights are widened once.
  * "flashmoon demo" page, Performance: the KV cache is f32 and RoPE is applied
    before keys are written to it.
  * "Emberglass" README, "Why it's hard": int4 group-128 weights; LoRA applied
    live as an additive branch.

Precision: every tensor between two operations is float32 (f32 activations and
f32 KV cache, as on the flashmoon page). Inside one operation the products and
sums are formed in float64 and rounded to float32 once.

Readings of points the pages leave open (each listed in the design notes):
  * RMSNorm: y = g * x / sqrt(mean(x^2) + eps), eps inside the root, gain
    multiplies directly.
  * QK-norm: RMSNorm over head_dim of every q and k head with gains [head_dim]
    shared by all heads, applied before RoPE.
  * RoPE: rotate-half pairing (j, j + hd/2); inv_freq_j = theta^(-2j/hd);
    angle = p * inv_freq_j with 0-based positions; cos/sin formed in float64
    and rounded to float32.
  * GQA: query head h reads kv head h // (n_q_heads / n_kv_heads).
  * Attention: scale 1/sqrt(head_dim); query at position p sees keys 0..p.
  * SiLU(z) = z / (1 + exp(-z)).
  * q/k/v bias (Qwen2.5) is added after the projection, before RoPE.
  * LoRA on q_proj and v_proj: y = W x + b + (alpha / rank) * B (A x).
  * int4 g128: see ``int4_quantize``; Q8_0: see ``q8_0_quantize``.
  * Greedy argmax: ties go to the lowest index; a NaN logit is an error.
  * bf16 KV cache (option): keys (after QK-norm and RoPE) and values are rounded
    to the nearest bf16 when stored, and attention reads the stored values.
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

F32 = np.float32
F64 = np.float64


# ----------------------------------------------------------------------------- dtype helpers
def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32. Exact: a bf16 is the top half of an f32
    ("Failed Star / fs, M2", Correct before fast: BF16 weights widen once)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(F32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (ties to even), returned as float32.

    Used for the bf16 KV cache ("Emberglass" README, Context window & prefill sizes:
    the f32 cache could be quantised to roughly half its size): keys and values are
    stored, and read back, at bf16 precision. Finite inputs only."""
    u = np.ascontiguousarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(F32)


# ----------------------------------------------------------------------------- basic ops
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """Row-wise RMSNorm over the last axis: g * x / sqrt(mean(x^2) + eps).

    "Failed Star / fs, M2", FINAL NORM ("Row-wise RMSNorm") and the
    residual-bus paragraph; also used per head for QK-norm.
    """
    x64 = x.astype(F64)
    ms = np.mean(x64 * x64, axis=-1, keepdims=True)
    return (g.astype(F64) * x64 / np.sqrt(ms + eps)).astype(F32)


def linear(x: np.ndarray, w64: np.ndarray, b: Optional[np.ndarray] = None) -> np.ndarray:
    """y = x . W^T (+ b) with W stored [out, in] ("Failed Star / fs, M2",
    Correct before fast). ``w64`` is the float64 view of the weight."""
    y = x.astype(F64) @ w64.T
    if b is not None:
        y = y + b.astype(F64)
    return y.astype(F32)


def rope_cos_sin(positions: Sequence[int], head_dim: int, theta: float
                 ) -> Tuple[np.ndarray, np.ndarray]:
    """Rotary tables for the given 0-based positions: float32 [P, head_dim/2].

    inv_freq_j = theta^(-2j/head_dim), angle = p * inv_freq_j, formed in float64.
    """
    half = head_dim // 2
    j = np.arange(half, dtype=F64)
    inv_freq = theta ** (-2.0 * j / head_dim)
    ang = np.asarray(positions, dtype=F64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE. x [P, n_heads, hd]; cos/sin [P, hd/2].

    Pair (j, j + hd/2) is rotated by its angle: (a, b) -> (a cos - b sin, b cos + a sin)
    ("flashmoon demo", Performance: RoPE fused on the KV write; "Failed Star /
    fs, M2": QK-norm then RoPE inside the block).
    """
    half = x.shape[-1] // 2
    a = x[..., :half].astype(F64)
    b = x[..., half:].astype(F64)
    c = cos.astype(F64)[:, None, :]
    s = sin.astype(F64)[:, None, :]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1).astype(F32)


def silu_mul(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SwiGLU core: silu(gate) * up with silu(z) = z / (1 + e^-z)."""
    g = gate.astype(F64)
    return (g / (1.0 + np.exp(-g)) * up.astype(F64)).astype(F32)


def causal_gqa_attention(q: np.ndarray, q_pos: np.ndarray, k: np.ndarray, v: np.ndarray,
                         k_pos: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention.

    q [Tq, nq, hd] at positions q_pos; k, v [nkv, Tk, hd] at positions k_pos.
    Query head h uses kv head h // (nq / nkv); a query at position p sees the
    keys whose position is <= p; scores are scaled by 1/sqrt(hd) and
    soft-maxed with the row maximum subtracted. Returns float32 [Tq, nq, hd].
    """
    Tq, nq, hd = q.shape
    nkv = k.shape[0]
    group = nq // nkv
    out = np.empty((Tq, nq, hd), dtype=F32)
    mask = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]  # [Tq, Tk]
    scale = 1.0 / math.sqrt(hd)
    for h in range(nq):
        if h % group == 0:                    # widen each kv head once per group
            kh = k[h // group].astype(F64)
            vh = v[h // group].astype(F64)
        s = (q[:, h, :].astype(F64) @ kh.T) * scale
        s = np.where(mask, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = (p @ vh).astype(F32)
    return out


def greedy_argmax(logits: np.ndarray) -> int:
    """Index of the largest logit; ties go to the lowest index; NaN is an error."""
    if np.isnan(logits).any():
        raise FloatingPointError("NaN logit")
    return int(np.argmax(logits))


def sample_logits(logits: np.ndarray, temperature: float, top_k: int, top_p: float, u: float):
    """Temperature / top-k / top-p sampling of one logits row with the draw u in [0, 1).

    "flashmoon demo" page: greedy plus temperature/top-k/top-p sampling, temp = 0
    meaning greedy. The page gives no formula; the reading used here:
      candidates: the top_k largest logits (top_k clamped to the row), ordered by
        logit descending, index ascending;
      w_i = exp((l_i - l_0) / T) in float64, l_0 the largest;
      nucleus: the shortest prefix whose running sum (in candidate order) reaches
        top_p times the sum over all candidates (top_p >= 1: all of them);
      token: the first candidate of the nucleus whose running sum exceeds u times
        the nucleus sum.
      T <= 0 or top_k == 1: the greedy argmax.
    Returns (token, margin): margin is the smallest relative distance between a
    running sum and either threshold it was compared with near the decision, so a
    test can tell a decision that float rounding could flip. NaN -> FloatingPointError;
    no finite logit -> FloatingPointError.
    """
    x = np.asarray(logits, dtype=np.float32)
    if np.isnan(x).any():
        raise FloatingPointError("NaN logit")
    k = min(int(top_k), x.size)
    order = np.lexsort((np.arange(x.size), -x.astype(np.float64)))[:k]  # logit desc, index asc
    l = x[order].astype(np.float64)
    if not np.isfinite(l[0]) or l[0] == -np.inf:
        raise FloatingPointError("no finite logit")
    if not temperature > 0 or k == 1:
        return int(order[0]), np.inf
    w = np.exp((l - l[0]) / float(temperature))
    run = np.empty(k)
    acc = 0.0
    for i in range(k):                       # running sums in candidate order
        acc += w[i]
        run[i] = acc
    need = float(np.float32(top_p)) * run[-1]
    cut = k - 1
    for i in range(k):
        if run[i] >= need:
            cut = i
            break
    target = float(np.float32(u)) * run[cut]
    pick = cut
    for i in range(cut + 1):
        if run[i] > target:
            pick = i
            break
    # decision margins (relative to the total): how far the running sums on either
    # side of each decision sit from its threshold (the last candidate always
    # meets the nucleus threshold, so it is no margin)
    near = [np.inf]
    if cut < k - 1:
        near.append(run[cut] - need)
    if cut > 0:
        near.append(need - run[cut - 1])
    near.append(run[pick] - target)
    if pick > 0:
        near.append(target - run[pick - 1])
    return int(order[pick]), float(min(near) / run[-1])


# ----------------------------------------------------------------------------- int4 group-128
INT4_GROUP = 128


def int4_quantize(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Symmetric int4, one bf16 scale per 128 consecutive inputs of a row.

    "Emberglass" README, "Why it's hard": int4 group-128 weights, quantised on
    the way to the GPU. The page gives no formula; the reading used here:
      s = bf16(max|w| / 7)     (division in float32, then round-to-nearest-even to bf16)
      q = clamp(rint(w / s), -7, 7)   (division in float32, rint ties to even); q = 0 if s = 0
      stored nibble = q + 8; element 2i in the low nibble of byte i.
    w: float32 [N, K] with K % 128 == 0. Returns (packed uint8 [N, K/2],
    scale bits uint16 [N, K/128]).
    """
    w = np.ascontiguousarray(w, dtype=F32)
    N, K = w.shape
    assert K % INT4_GROUP == 0
    G = K // INT4_GROUP
    wg = w.reshape(N, G, INT4_GROUP)
    m = np.max(np.abs(wg), axis=2)                                   # f32 [N, G]
    s32 = (m / F32(7.0)).astype(F32)
    u = s32.view(np.uint32).astype(np.uint64)                        # f32 -> bf16, RNE
    s_bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    s = widen_bf16(s_bits)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (wg / s[:, :, None]).astype(F32)
    q = np.where(s[:, :, None] == 0, 0, np.clip(np.rint(r), -7, 7)).astype(np.int32)
    nib = (q + 8).astype(np.uint8).reshape(N, K)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return packed, s_bits


def int4_dequantize(packed: np.ndarray, s_bits: np.ndarray) -> np.ndarray:
    """w' = (nibble - 8) * scale, exact in float32 (a 4-bit integer times a bf16)."""
    N, Kh = packed.shape
    nib = np.empty((N, Kh * 2), dtype=np.int32)
    nib[:, 0::2] = packed & 0x0F
    nib[:, 1::2] = packed >> 4
    s = widen_bf16(s_bits)
    return ((nib - 8).astype(F32).reshape(N, -1, INT4_GROUP) * s[:, :, None]).reshape(N, -1)


# ----------------------------------------------------------------------------- Q8_0 (block-32 int8)
Q8_BLOCK = 32


def q8_0_quantize(w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Symmetric int8, one fp16 scale per 32 consecutive inputs of a row (Q8_0).

    "SuperKittens PR #7" page, the Q8_0 commit: Q8_0 weights (GGUF type 8: blocks
    of 32 int8 values with one scale) read by a q8_0 matvec for decode and for the
    LM head (quantised from the embedding table when the head is tied). The page
    gives no formula; the reading used here (the int4 reading with 127 levels):
      s = fp16(max|w| / 127)    (division in float32, then round-to-nearest-even to fp16)
      q = clamp(rint(w / s), -127, 127)   (division in float32, ties to even); q = 0 if s = 0
    w: float32 [N, K] with K % 32 == 0. Returns (q int8 [N, K], scale bits uint16 [N, K/32]).
    """
    w = np.ascontiguousarray(w, dtype=F32)
    N, K = w.shape
    assert K % Q8_BLOCK == 0
    wg = w.reshape(N, K // Q8_BLOCK, Q8_BLOCK)
    m = np.max(np.abs(wg), axis=2)
    with np.errstate(over="ignore"):
        s16 = (m / F32(127.0)).astype(F32).astype(np.float16)      # IEEE round to nearest even
    s = s16.astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (wg / s[:, :, None]).astype(F32)
    q = np.where(s[:, :, None] == 0, 0, np.clip(np.rint(r), -127, 127)).astype(np.int8)
    return q.reshape(N, K), s16.view(np.uint16)


def q8_0_dequantize(q: np.ndarray, s_bits: np.ndarray) -> np.ndarray:
    """w' = q * scale, exact in float32 (a 7-bit integer times an fp16)."""
    N, K = q.shape
    s = np.ascontiguousarray(s_bits, dtype=np.uint16).view(np.float16).astype(F32)
    return (q.astype(F32).reshape(N, -1, Q8_BLOCK) * s[:, :, None]).reshape(N, K)


# ----------------------------------------------------------------------------- model
@dataclass
class Config:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    eps: float = 1e-6
    rope_theta: float = 1e6
    tie_word_embeddings: bool = True
    qk_norm: bool = True
    qkv_bias: bool = False
    weight_format: str = "bf16"
    int4_lm_head: bool = False
    kv_format: str = "f32"       # "f32" or "bf16": precision of the stored keys and values

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @classmethod
    def from_shape(cls, s) -> "Config":
        return cls(**{f: getattr(s, f) for f in cls.__dataclass_fields__})


def kv_cache_bytes(cfg: Config, n_positions: int) -> int:
    """f32 K and V for every layer and kv head ("Emberglass" README, Context
    window & prefill sizes: the KV cache grows linearly with context, f32)."""
    return cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 4 * n_positions


_LINEAR = ("q", "k", "v", "o", "gate", "up", "down")


class OracleModel:
    """The network with its own f32 KV cache.

    ``weights`` maps names (see the workload draw order) to uint16 bf16 bits,
    or, for an int4 model's linear weights, to float32 values which are
    quantised here with ``int4_quantize`` and widened back exactly.
    """

    def __init__(self, cfg: Config, weights: Dict[str, np.ndarray], max_ctx: int,
                 lora: Optional[Dict[str, np.ndarray]] = None, lora_alpha: float = 0.0,
                 cache_f64: Optional[bool] = None):
        self.cfg = cfg
        self.max_ctx = max_ctx
        self.w: Dict[str, np.ndarray] = {}
        self.int4: Dict[str, Tuple[np.ndarray, np.ndarray]] = {}
        self.q8: Dict[str, Tuple[np.ndarray, np.ndarray]] = {}
        int4_names, q8_names = set(), set()
        if cfg.weight_format == "int4_g128":
            int4_names = {f"layers.{l}.{n}" for l in range(cfg.n_layers) for n in _LINEAR}
            if not cfg.tie_word_embeddings and cfg.int4_lm_head:
                int4_names.add("lm_head")
        elif cfg.weight_format == "q8_0":
            q8_names = {f"layers.{l}.{n}" for l in range(cfg.n_layers) for n in _LINEAR}
            if not cfg.tie_word_embeddings:
                q8_names.add("lm_head")
        for name, arr in weights.items():
            if name.startswith("lora."):
                continue
            if name in int4_names:
                packed, sb = int4_quantize(arr)
                self.int4[name] = (packed, sb)
                self.w[name] = int4_dequantize(packed, sb)
            elif name in q8_names:
                q, sb = q8_0_quantize(arr)
                self.q8[name] = (q, sb)
                self.w[name] = q8_0_dequantize(q, sb)
            else:
                self.w[name] = widen_bf16(arr)
        if cfg.weight_format == "q8_0" and cfg.tie_word_embeddings:
            # the tied head reads a Q8_0 copy of the table; the gather keeps bf16 rows
            q, sb = q8_0_quantize(self.w["embed"])
            self.q8["lm_head"] = (q, sb)
            self.w["lm_head_q8"] = q8_0_dequantize(q, sb)
        self.lora: Optional[Dict[str, np.ndarray]] = None
        self.lora_scale = 0.0
        if lora is not None:
            self.set_lora(lora, lora_alpha)
        n_params = sum(a.size for a in self.w.values())
        if cache_f64 is None:
            cache_f64 = n_params * 8 < 0.4 * _mem_available()
        self._cache_f64 = cache_f64
        self._w64: Dict[str, np.ndarray] = {}
        self.reset()

    # -- state --------------------------------------------------------------------------
    def reset(self) -> None:
        c = self.cfg
        self.pos = 0
        self.k_cache = [np.zeros((c.n_kv_heads, self.max_ctx, c.head_dim), F32)
                        for _ in range(c.n_layers)]
        self.v_cache = [np.zeros((c.n_kv_heads, self.max_ctx, c.head_dim), F32)
                        for _ in range(c.n_layers)]

    def set_kv(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        n = k.shape[1]
        self.k_cache[layer][:, :n] = k
        self.v_cache[layer][:, :n] = v

    def set_lora(self, lora: Optional[Dict[str, np.ndarray]], alpha: float = 0.0) -> None:
        """LoRA on q_proj and v_proj ("Emberglass" README: hot-swap; clearing it
        restores the base output). A/B arrive as bf16 bits, keyed 'lora.{l}.q_a' etc."""
        if lora is None:
            self.lora, self.lora_scale = None, 0.0
            return
        self.lora = {k: widen_bf16(v).astype(F64) for k, v in lora.items()}
        rank = self.lora["lora.0.q_a"].shape[0]
        self.lora_scale = alpha / rank

    # -- helpers ------------------------------------------------------------------------
    def W(self, name: str) -> np.ndarray:
        if name in self._w64:
            return self._w64[name]
        w = self.w[name].astype(F64)
        if self._cache_f64:
            self._w64[name] = w
        return w

    def _gain(self, name: str) -> np.ndarray:
        return self.w[name]

    def _bias(self, name: str) -> Optional[np.ndarray]:
        return self.w[name] if self.cfg.qkv_bias else None

    def _proj_qkv(self, l: int, xn: np.ndarray):
        p = f"layers.{l}."
        if self.lora is None:
            q = linear(xn, self.W(p + "q"), self._bias(p + "q_bias"))
            k = linear(xn, self.W(p + "k"), self._bias(p + "k_bias"))
            v = linear(xn, self.W(p + "v"), self._bias(p + "v_bias"))
            return q, k, v
        x64 = xn.astype(F64)
        lp = f"lora.{l}."

        def with_lora(wname, bname, a, b):
            y = x64 @ self.W(p + wname).T
            bias = self._bias(p + bname)
            if bias is not None:
                y = y + bias.astype(F64)
            if a is not None:
                y = y + self.lora_scale * ((x64 @ self.lora[lp + a].T) @ self.lora[lp + b].T)
            return y.astype(F32)

        return (with_lora("q", "q_bias", "q_a", "q_b"), with_lora("k", "k_bias", None, None),
                with_lora("v", "v_bias", "v_a", "v_b"))

    def _qkv_heads(self, l: int, xn: np.ndarray, positions: np.ndarray):
        """Projection, QK-norm, RoPE for T rows. Returns q [T,nq,hd], k,v [T,nkv,hd]."""
        c = self.cfg
        T = xn.shape[0]
        q, k, v = self._proj_qkv(l, xn)
        q = q.reshape(T, c.n_q_heads, c.head_dim)
        k = k.reshape(T, c.n_kv_heads, c.head_dim)
        v = v.reshape(T, c.n_kv_heads, c.head_dim)
        if c.qk_norm:
            q = rmsnorm(q, self._gain(f"layers.{l}.q_norm"), c.eps)
            k = rmsnorm(k, self._gain(f"layers.{l}.k_norm"), c.eps)
        cos, sin = rope_cos_sin(positions, c.head_dim, c.rope_theta)
        k, v = apply_rope(k, cos, sin), v
        if c.kv_format == "bf16":          # what the cache stores is what attention reads
            k, v = round_bf16(k), round_bf16(v)
        return apply_rope(q, cos, sin), k, v

    def _mlp(self, l: int, x: np.ndarray) -> np.ndarray:
        p = f"layers.{l}."
        xn = rmsnorm(x, self._gain(p + "mlp_norm"), self.cfg.eps)
        m = silu_mul(linear(xn, self.W(p + "gate")), linear(xn, self.W(p + "up")))
        return (x.astype(F64) + linear(m, self.W(p + "down")).astype(F64)).astype(F32)

    def _head(self, x_last: np.ndarray):
        c = self.cfg
        h = rmsnorm(x_last, self._gain("final_norm"), c.eps)
        table = "embed" if c.tie_word_embeddings else "lm_head"
        if c.tie_word_embeddings and c.weight_format == "q8_0":
            table = "lm_head_q8"
        logits = linear(h, self.W(table))
        return h, logits

    # -- the two entry points -------------------------------------------------------------
    def prefill(self, ids: Sequence[int], keep_cache: bool = True) -> Dict[str, np.ndarray]:
        """No-cache causal forward of T ids at positions 0..T-1.

        Returns the four checkpoints of the "Failed Star / fs, M2" page
        (embedding [T,H], block 0 [T,H], final norm [T,H], last-row logits [V])
        and, with ``keep_cache``, leaves K/V of every position in the cache with
        pos = T so that decoding can continue.
        """
        c = self.cfg
        ids = np.asarray(ids, dtype=np.int64)
        T = ids.shape[0]
        assert 0 < T <= self.max_ctx
        positions = np.arange(T)
        x = self.w["embed"][ids].astype(F32)                        # gather, not a matmul
        cp = {"embedding": x.copy()}
        for l in range(c.n_layers):
            p = f"layers.{l}."
            xn = rmsnorm(x, self._gain(p + "attn_norm"), c.eps)
            q, k, v = self._qkv_heads(l, xn, positions)
            kt, vt = k.transpose(1, 0, 2), v.transpose(1, 0, 2)      # [nkv, T, hd]
            o = causal_gqa_attention(q, positions, kt, vt, positions).reshape(T, c.q_dim)
            x = (x.astype(F64) + linear(o, self.W(p + "o")).astype(F64)).astype(F32)
            x = self._mlp(l, x)
            if keep_cache:
                self.k_cache[l][:, :T] = kt
                self.v_cache[l][:, :T] = vt
            if l == 0:
                cp["block0"] = x.copy()
        h_all = rmsnorm(x, self._gain("final_norm"), c.eps)
        cp["final_norm"] = h_all
        _, logits = self._head(x[-1:])
        cp["logits"] = logits[0]
        if keep_cache:
            self.pos = T
        return cp

    def decode_step(self, token: int) -> Dict[str, np.ndarray]:
        """One cached step at position ``pos``: append k/v, attend to 0..pos, pos += 1."""
        c = self.cfg
        p0 = self.pos
        assert 0 <= token < c.vocab and p0 < self.max_ctx
        x = self.w["embed"][[token]].astype(F32)
        cp = {"embedding": x.copy()}
        positions = np.array([p0])
        for l in range(c.n_layers):
            p = f"layers.{l}."
            xn = rmsnorm(x, self._gain(p + "attn_norm"), c.eps)
            q, k, v = self._qkv_heads(l, xn, positions)
            self.k_cache[l][:, p0] = k[0]
            self.v_cache[l][:, p0] = v[0]
            kpos = np.arange(p0 + 1)
            o = causal_gqa_attention(q, positions, self.k_cache[l][:, :p0 + 1],
                                     self.v_cache[l][:, :p0 + 1], kpos).reshape(1, c.q_dim)
            x = (x.astype(F64) + linear(o, self.W(p + "o")).astype(F64)).astype(F32)
            x = self._mlp(l, x)
            if l == 0:
                cp["block0"] = x.copy()
        h, logits = self._head(x)
        cp["final_norm"] = h
        cp["logits"] = logits[0]
        self.pos = p0 + 1
        return cp


def build_oracle(drawn, max_ctx: Optional[int] = None, lora_on: bool = False,
                 cache_f64: Optional[bool] = None) -> OracleModel:
    """An OracleModel for a drawn workload (weights, optional KV prefill)."""
    w = drawn.workload
    cfg = Config.from_shape(w.shape)
    lora = None
    if lora_on and w.lora is not None:
        lora = {k: v for k, v in drawn.weights.items() if k.startswith("lora.")}
    m = OracleModel(cfg, drawn.weights, max_ctx or w.max_ctx, lora=lora,
                    lora_alpha=w.lora.alpha if w.lora else 0.0, cache_f64=cache_f64)
    for l, (k, v) in enumerate(drawn.kv):
        m.set_kv(l, k, v)
    if drawn.kv:
        m.pos = drawn.kv[0][0].shape[1]
    return m


def _mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 8 << 30
