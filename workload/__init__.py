"""Seeded synthetic workloads for the batch-1 Qwen-style decode step.

This module only *draws* inputs. It holds none of the method's arithmetic: no
normalisation, no projection, no attention, no quantisation. Both the oracle
(under ``oracle/``) and the CUDA path are fed from here, and neither one is
imported by this module.

Shapes follow the models the source pages run:
  * "flashmoon demo" page, Components / Performance: Qwen3-0.6B (28 layers,
    bf16 weights, f32 KV cache).
  * "Failed Star / fs, M2" page, "One prefill, all shapes visible":
    residual [seq, 1024], vocab 151936, tied embedding table.
  * "Emberglass" README, "What this is" / "Context window & prefill sizes":
    Qwen2.5-3B, int4 group-128 weights, LoRA hot-swap, 36 layers.

Draw recipe (numpy ``default_rng(seed)``, PCG64):
  weights ~ N(0, 0.02) drawn as float32 ``standard_normal * 0.02`` in a fixed
  tensor order (embed; per layer attn_norm, q, k, v, [q/k/v bias], q_norm,
  k_norm, o, mlp_norm, gate, up, down; final_norm; [lm_head]; [LoRA A/B for q
  then v, per layer]); norm gains are 1.0 unless a test asks for drawn gains
  (1 + N(0, 0.1)). bf16 tensors are the float32 draw rounded to nearest-even
  bf16. Tensors bound for int4 or Q8_0 stay float32 (each side quantises them itself).
  After the weights: the KV prefill (N(0,1) rounded to bf16, stored as f32, in
  order layer -> K then V -> kv head -> position -> dim), then token ids,
  uniform in [0, vocab).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, Iterator, List, Optional, Tuple

import numpy as np

WEIGHT_STD = 0.02
LORA_STD = 0.01
GAIN_JITTER_STD = 0.1


@dataclass(frozen=True)
class ModelShape:
    """Architecture of one Qwen-style decoder (names as in HF configs)."""

    name: str
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
    weight_format: str = "bf16"  # "bf16", "int4_g128" or "q8_0"
    int4_lm_head: bool = False   # untied lm_head quantised too (int4 models)
    kv_format: str = "f32"       # "f32" or "bf16" KV cache

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def replace(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class LoraShape:
    rank: int = 16
    alpha: float = 32.0


@dataclass(frozen=True)
class Workload:
    """One seeded workload: a model shape plus what is fed to it."""

    name: str
    shape: ModelShape
    seed: int
    prompt_len: int = 0          # ids fed through prefill
    decode_steps: int = 0        # greedy steps after the prompt
    kv_prefill: int = 0          # positions of the KV cache pre-filled with N(0,1)
    lora: Optional[LoraShape] = None
    max_ctx: int = 0             # KV capacity the handle is created with
    description: str = ""


TINY = ModelShape("tiny-qwen3", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2,
                  head_dim=64, intermediate=768, vocab=4096)
QWEN3_0_6B = ModelShape("qwen3-0.6b", n_layers=28, hidden=1024, n_q_heads=16, n_kv_heads=8,
                        head_dim=128, intermediate=3072, vocab=151936)
QWEN25_3B_INT4 = ModelShape("qwen2.5-3b-int4g128", n_layers=36, hidden=2048, n_q_heads=16,
                            n_kv_heads=2, head_dim=128, intermediate=11008, vocab=151936,
                            tie_word_embeddings=False, qk_norm=False, qkv_bias=True,
                            weight_format="int4_g128", int4_lm_head=True)
# Qwen3-0.6B with Q8_0 weights ("SuperKittens PR #7" page, Q8_0 commit: decode of the
# same model with GGUF Q8_0 projections and LM head)
QWEN3_0_6B_Q8 = QWEN3_0_6B.replace(name="qwen3-0.6b-q8_0", weight_format="q8_0")

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", TINY, seed=0, prompt_len=8, decode_steps=16, max_ctx=64,
                     description="tiny Qwen3-style decoder: 8-id prompt, 16 greedy steps"),
    "qwen3_0.6b_decode": Workload("qwen3_0.6b_decode", QWEN3_0_6B, seed=1, prompt_len=5,
                                  decode_steps=128, max_ctx=2048,
                                  description="Qwen3-0.6B shape, 5-id prompt then 128 greedy "
                                              "batch-1 decode steps (positions 5..132)"),
    "qwen3_0.6b_longctx": Workload("qwen3_0.6b_longctx", QWEN3_0_6B, seed=2, kv_prefill=8192,
                                   decode_steps=32, max_ctx=8192 + 32,
                                   description="Qwen3-0.6B shape, KV cache 0..8191 pre-filled, "
                                               "32 greedy steps from position 8192"),
    "qwen3_0.6b_prefill": Workload("qwen3_0.6b_prefill", QWEN3_0_6B, seed=3, prompt_len=1024,
                                   max_ctx=1024 + 8,
                                   description="Qwen3-0.6B shape, one causal prefill of T=1024"),
    "qwen2.5_3b_int4_lora": Workload("qwen2.5_3b_int4_lora", QWEN25_3B_INT4, seed=4,
                                     kv_prefill=4096, decode_steps=64, lora=LoraShape(16, 32.0),
                                     max_ctx=4096 + 64,
                                     description="Qwen2.5-3B shape, int4 g128, q/k/v bias, untied "
                                                 "head, KV pre-filled to 4096, 64 greedy steps with "
                                                 "a rank-16 LoRA on q/v and 64 without"),
    "qwen3_0.6b_longctx_bf16kv": Workload("qwen3_0.6b_longctx_bf16kv",
                                          QWEN3_0_6B.replace(kv_format="bf16"), seed=2,
                                          kv_prefill=8192, decode_steps=32, max_ctx=8192 + 32,
                                          description="the long-context workload with a bf16 "
                                                      "KV cache (the pre-filled values are "
                                                      "bf16 already)"),
    "qwen3_0.6b_q8_0_decode": Workload("qwen3_0.6b_q8_0_decode", QWEN3_0_6B_Q8, seed=5,
                                       prompt_len=5, decode_steps=64, max_ctx=256,
                                       description="Qwen3-0.6B shape with Q8_0 projections and "
                                                   "LM head, 5-id prompt then 64 greedy steps"),
}


# ----------------------------------------------------------------------------- bf16 bits
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return the uint16 bits.

    Input synthesis only: it turns a float32 draw into a bf16 *input tensor*.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> float32 (exact); used by the generator for bf16-valued f32 data."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- weights
def _linear_shapes(s: ModelShape) -> List[Tuple[str, Tuple[int, int]]]:
    H, I = s.hidden, s.intermediate
    return [("q", (s.q_dim, H)), ("k", (s.kv_dim, H)), ("v", (s.kv_dim, H)),
            ("o", (H, s.q_dim)), ("gate", (I, H)), ("up", (I, H)), ("down", (H, I))]


def weight_draw_order(s: ModelShape, lora: Optional[LoraShape] = None,
                      drawn_gains: bool = False) -> List[Tuple[str, Tuple[int, ...], str]]:
    """(name, shape, kind) in draw order. kind: 'bf16', 'f32q' (float32 bound for int4 or
    Q8_0 quantisation), 'gain'."""
    lin_kind = "f32q" if s.weight_format in ("int4_g128", "q8_0") else "bf16"
    out: List[Tuple[str, Tuple[int, ...], str]] = [("embed", (s.vocab, s.hidden), "bf16")]
    for l in range(s.n_layers):
        p = f"layers.{l}."
        out.append((p + "attn_norm", (s.hidden,), "gain"))
        for nm, shp in _linear_shapes(s)[:3]:
            out.append((p + nm, shp, lin_kind))
        if s.qkv_bias:
            out += [(p + "q_bias", (s.q_dim,), "bf16"), (p + "k_bias", (s.kv_dim,), "bf16"),
                    (p + "v_bias", (s.kv_dim,), "bf16")]
        if s.qk_norm:
            out += [(p + "q_norm", (s.head_dim,), "gain"), (p + "k_norm", (s.head_dim,), "gain")]
        out.append((p + "o", _linear_shapes(s)[3][1], lin_kind))
        out.append((p + "mlp_norm", (s.hidden,), "gain"))
        for nm, shp in _linear_shapes(s)[4:]:
            out.append((p + nm, shp, lin_kind))
    out.append(("final_norm", (s.hidden,), "gain"))
    if not s.tie_word_embeddings:
        out.append(("lm_head", (s.vocab, s.hidden),
                    "f32q" if ((s.int4_lm_head and s.weight_format == "int4_g128")
                               or s.weight_format == "q8_0") else "bf16"))
    if lora is not None:
        r = lora.rank
        for l in range(s.n_layers):
            p = f"lora.{l}."
            out += [(p + "q_a", (r, s.hidden), "lora"), (p + "q_b", (s.q_dim, r), "lora"),
                    (p + "v_a", (r, s.hidden), "lora"), (p + "v_b", (s.kv_dim, r), "lora")]
    return out


def iter_weights(s: ModelShape, rng: np.random.Generator, lora: Optional[LoraShape] = None,
                 drawn_gains: bool = False) -> Iterator[Tuple[str, np.ndarray]]:
    """Yield (name, array) in draw order.

    bf16 tensors come back as uint16 bit arrays; int4-bound tensors as float32;
    gains as uint16 bf16 bits (1.0 = 0x3F80 unless ``drawn_gains``).
    """
    for name, shape, kind in weight_draw_order(s, lora, drawn_gains):
        if kind == "gain":
            if drawn_gains:
                g = 1.0 + rng.standard_normal(shape, dtype=np.float32) * np.float32(GAIN_JITTER_STD)
                yield name, f32_to_bf16_bits(g)
            else:
                yield name, np.full(shape, 0x3F80, dtype=np.uint16)
            continue
        std = LORA_STD if kind == "lora" else WEIGHT_STD
        w = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
        if kind == "f32q":
            yield name, w
        else:
            yield name, f32_to_bf16_bits(w)


def draw_kv_prefill(s: ModelShape, n_pos: int, rng: np.random.Generator
                    ) -> Iterator[Tuple[int, np.ndarray, np.ndarray]]:
    """Yield (layer, K, V) with K, V float32 [n_kv_heads, n_pos, head_dim], values N(0,1)
    rounded to bf16. K is taken to be already position-rotated (it is data)."""
    for l in range(s.n_layers):
        k = bf16_bits_to_f32(f32_to_bf16_bits(
            rng.standard_normal((s.n_kv_heads, n_pos, s.head_dim), dtype=np.float32)))
        v = bf16_bits_to_f32(f32_to_bf16_bits(
            rng.standard_normal((s.n_kv_heads, n_pos, s.head_dim), dtype=np.float32)))
        yield l, k, v


@dataclass
class DrawnWorkload:
    """Everything a workload feeds the model, drawn in the documented order."""

    workload: Workload
    weights: Dict[str, np.ndarray] = field(default_factory=dict)
    kv: List[Tuple[np.ndarray, np.ndarray]] = field(default_factory=list)
    prompt: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    start_token: int = -1


def draw(w: Workload, drawn_gains: bool = False, with_kv: bool = True) -> DrawnWorkload:
    """Draw the full input set of workload ``w`` (weights, KV prefill, token ids)."""
    rng = np.random.default_rng(w.seed)
    out = DrawnWorkload(w)
    for name, arr in iter_weights(w.shape, rng, w.lora, drawn_gains):
        out.weights[name] = arr
    if w.kv_prefill:
        if with_kv:
            for _, k, v in draw_kv_prefill(w.shape, w.kv_prefill, rng):
                out.kv.append((k, v))
        else:  # advance the stream exactly as the draw would
            for _ in range(w.shape.n_layers * 2):
                rng.standard_normal((w.shape.n_kv_heads, w.kv_prefill, w.shape.head_dim),
                                    dtype=np.float32)
    if w.prompt_len:
        out.prompt = rng.integers(0, w.shape.vocab, size=w.prompt_len).astype(np.int32)
    if w.kv_prefill:
        out.start_token = int(rng.integers(0, w.shape.vocab))
    return out


def random_ids(vocab: int, n: int, seed: int) -> np.ndarray:
    """Uniform token ids in [0, vocab) for ad-hoc test cases."""
    return np.random.default_rng(seed).integers(0, vocab, size=n).astype(np.int32)
