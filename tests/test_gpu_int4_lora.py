"""Qwen2.5-style decode: int4 group-128 weights (quantised on the device), q/k/v
biases, no QK-norm, untied int4 LM head, and a LoRA on q_proj and v_proj that is
set and cleared live ("Emberglass" README: int4 g128, LoRA hot-swap, perfect
restore on clear).

The GPU quantiser and the oracle's quantiser are separate implementations of the
same rule (checked bit-exact in test_gpu_ops); each side quantises the same f32
draws itself. Clearing the adapter must give bit-identical logits to a handle
that never had one.
"""
import numpy as np
import pytest

import workload as W
from oracle import qwen_ref as R
from sequence_decode_step_gb300 import _binding as B
from sequence_decode_step_gb300.device_model import DeviceModel

from gpu_util import MARGIN, top2_margin, violation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TINY_INT4 = W.TINY.replace(weight_format="int4_g128", tie_word_embeddings=False,
                           int4_lm_head=True, qk_norm=False, qkv_bias=True, n_kv_heads=1)


def _lora(d):
    return {k: v for k, v in d.weights.items() if k.startswith("lora.")}


def _run(m, o, tok, steps, check_ids=True):
    """Teacher-forced steps; returns the GPU logits of every step and the next token."""
    out = []
    for i in range(steps):
        want = o.decode_step(tok)["logits"]
        got_id, got = m.decode(tok, logits=True)
        assert violation(got, want) <= 0, f"step {i}: off by {violation(got, want)}"
        if check_ids and top2_margin(want) > MARGIN:
            assert got_id == R.greedy_argmax(want)
        out.append(got)
        tok = R.greedy_argmax(want)
    return out, tok


# 0: the persistent kernel (its wide-input build takes int4 weights), 1: the graph
@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("shape", [TINY_INT4, TINY_INT4.replace(kv_format="bf16"),
                                   TINY_INT4.replace(intermediate=3584)],
                         ids=["f32kv", "bf16kv", "wide"])
def test_tiny_int4_decode(shape, path):
    wl = W.Workload("t4", shape, seed=5, prompt_len=8, decode_steps=16, max_ctx=64)
    d = W.draw(wl, drawn_gains=True)
    m = DeviceModel(wl.shape, d.weights, 64, max_prefill_t=0)    # prompt as sequential steps
    o = R.build_oracle(d)
    try:
        assert B.qw_get_decode_path(m.h) == 0
        B.qw_set_decode_path(m.h, path)
        assert B.qw_get_decode_path(m.h) == path
        am, lg = m.prefill(d.prompt, logits=True)
        ref = o.prefill(d.prompt)["logits"]
        assert violation(lg, ref) <= 0
        _run(m, o, R.greedy_argmax(ref), 16)
    finally:
        m.close()


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("shape", [TINY_INT4, W.TINY.replace(qkv_bias=True),
                                   W.TINY.replace(qkv_bias=False),
                                   W.TINY.replace(qkv_bias=True, kv_format="bf16")],
                         ids=["int4", "bf16", "bf16_nobias", "bf16_kvbf16"])
def test_tiny_lora_on_then_cleared(shape, path):
    wl = W.Workload("tl", shape, seed=6, prompt_len=6, decode_steps=12, max_ctx=64,
                    lora=W.LoraShape(4, 8.0))
    d = W.draw(wl, drawn_gains=True)
    m = DeviceModel(shape, d.weights, 64, max_prefill_t=64)
    fresh = DeviceModel(shape, d.weights, 64, max_prefill_t=64)
    try:
        # 0: the persistent kernel adds the LoRA update in its QKV phase; 1: the graph
        B.qw_set_decode_path(m.h, path)
        B.qw_set_decode_path(fresh.h, path)
        # phase A: adapter on (prefill falls back to the sequential path; int4 prompts
        # without an adapter take the batched pass)
        m.set_lora(_lora(d), 8.0)
        assert B.qw_get_decode_path(m.h) == path
        o = R.build_oracle(d, lora_on=True)
        am, lg = m.prefill(d.prompt, logits=True)
        ref = o.prefill(d.prompt)["logits"]
        assert violation(lg, ref) <= 0
        base = R.build_oracle(d).prefill(d.prompt)["logits"]
        assert np.abs(ref - base).max() > 1e-3          # the adapter changes the output
        _run(m, o, R.greedy_argmax(ref), wl.decode_steps)
        # phase B: cleared; same inputs as a handle that never had an adapter
        m.set_lora(None)
        assert B.qw_get_decode_path(m.h) == path
        m.reset()
        o2 = R.build_oracle(d)
        am, lg = m.prefill(d.prompt, logits=True)
        am_f, lg_f = fresh.prefill(d.prompt, logits=True)
        np.testing.assert_array_equal(lg, lg_f)
        ref2 = o2.prefill(d.prompt)["logits"]
        tok = R.greedy_argmax(ref2)
        for _ in range(wl.decode_steps):
            want = o2.decode_step(tok)["logits"]
            _, a = m.decode(tok, logits=True)
            _, b = fresh.decode(tok, logits=True)
            np.testing.assert_array_equal(a, b)
            assert violation(a, want) <= 0
            tok = R.greedy_argmax(want)
    finally:
        m.close()
        fresh.close()


def test_qwen25_3b_int4_lora_4k():
    wl = W.WORKLOADS["qwen2.5_3b_int4_lora"]
    d = W.draw(wl)
    lora = _lora(d)
    o = R.build_oracle(d, lora_on=True)
    m = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    fresh = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    d.weights = {}                                            # the oracle keeps its own copies
    P = wl.kv_prefill
    try:
        assert B.qw_get_decode_path(fresh.h) == 0     # int4 on the persistent kernel
        for l, (k, v) in enumerate(d.kv):
            m.set_kv(l, k, v)
            fresh.set_kv(l, k, v)
        m.set_pos(P)
        fresh.set_pos(P)
        # phase A: 64 steps with the adapter, the last 8 on the multi-kernel graph
        m.set_lora(lora, wl.lora.alpha)
        assert B.qw_get_decode_path(m.h) == 0         # the adapter on the persistent kernel
        n0 = wl.decode_steps - 8
        tok = d.start_token
        for path, n in ((0, n0), (1, 8)):
            B.qw_set_decode_path(m.h, path)
            assert B.qw_get_decode_path(m.h) == path
            _, tok = _run(m, o, tok, n)
        B.qw_set_decode_path(m.h, 0)
        # phase B: cleared, cache and position restored, 64 steps; bit-identical to a
        # handle that never had the adapter, and within tolerance of the oracle
        m.set_lora(None)
        assert B.qw_get_decode_path(m.h) == 0         # back on the persistent kernel
        o.set_lora(None)
        o.reset()
        for l, (k, v) in enumerate(d.kv):
            m.set_kv(l, k, v)
            o.set_kv(l, k, v)
        m.set_pos(P)
        o.pos = P
        tok = d.start_token
        for i in range(wl.decode_steps):
            want = o.decode_step(tok)["logits"]
            ga, a = m.decode(tok, logits=True)
            gb, b = fresh.decode(tok, logits=True)
            np.testing.assert_array_equal(a, b)
            assert violation(a, want) <= 0, f"step {i}"
            if top2_margin(want) > MARGIN:
                assert ga == R.greedy_argmax(want)
            tok = R.greedy_argmax(want)
    finally:
        m.close()
        fresh.close()


def _int4_prefill_check(shape, seed, T, max_ctx, kv_layers, chunks=None):
    """Batched int4 prefill ("Emberglass" README, Context window & prefill sizes: a
    prompt up to maxPrefillT ids runs as one tiled int4-GEMM pass) against the oracle's
    no-cache prefill and against the same ids as sequential steps on the GPU."""
    wl = W.Workload("p4", shape, seed=seed, max_ctx=max_ctx)
    d = W.draw(wl, drawn_gains=True)
    ids = list(W.random_ids(shape.vocab, T, seed=seed + 1))
    m = DeviceModel(shape, d.weights, max_ctx, max_prefill_t=max(chunks or [T]))
    seq = DeviceModel(shape, d.weights, max_ctx, max_prefill_t=0)
    o = R.build_oracle(d, cache_f64=False)
    d.weights = {}
    try:
        if chunks:
            t0 = 0
            for n in chunks:
                am, lg = m.prefill(ids[t0:t0 + n], logits=True)
                t0 += n
        else:
            am, lg = m.prefill(ids, logits=True)
        cp = o.prefill(ids)
        assert violation(lg, cp["logits"]) <= 0
        am_s, lg_s = seq.prefill(ids, logits=True)
        assert violation(lg, lg_s) <= 0
        if top2_margin(cp["logits"]) > MARGIN:
            assert am == am_s == R.greedy_argmax(cp["logits"])
        for l in kv_layers:
            kd, vd = m.kv(l)
            kd, vd = kd.cpu().numpy()[:, :T], vd.cpu().numpy()[:, :T]
            assert violation(kd, o.k_cache[l][:, :T]) <= 0
            assert violation(vd, o.v_cache[l][:, :T]) <= 0
        assert m.pos() == T
        _run(m, o, R.greedy_argmax(cp["logits"]), 3)
    finally:
        m.close()
        seq.close()


def test_tiny_int4_batched_prefill():
    _int4_prefill_check(TINY_INT4, 25, 45, 64, [0, 1], chunks=[20, 25])


def test_qwen25_3b_int4_batched_prefill_512():
    _int4_prefill_check(W.QWEN25_3B_INT4, 26, 512, 520, [0, 17, 35])
