"""bf16 KV cache ("Emberglass" README, Context window & prefill sizes: the f32 cache
could be quantised to roughly half its size).

Keys (after QK-norm and RoPE) and values are stored rounded to the nearest bf16 and
attention reads the stored values; the oracle applies the same rounding, so the GPU
is checked at the model tolerance on every path that writes or reads the cache: the
persistent decode kernel (7- and 11-warp builds), the multi-kernel graph, batched and
sequential prefill.
"""
import numpy as np
import pytest

import workload as W
from oracle import qwen_ref as R
from sequence_decode_step_gb300 import _binding as B
from sequence_decode_step_gb300.device_model import DeviceModel

from gpu_util import ATOL, MARGIN, top2_margin, violation

# Stored keys and values are bf16: a value the GPU computes a hair away from the
# oracle's can round to the neighbouring bf16, one unit in the last place (2^-7 of
# the value at most) apart; the cache rows are compared with that allowance.
KV_RTOL = 2.0 ** -7

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _steps(m, o, tok, n):
    compared = 0
    for i in range(n):
        want = o.decode_step(tok)["logits"]
        got_id, got = m.decode(tok, logits=True)
        assert violation(got, want) <= 0, f"step {i}: off by {violation(got, want)}"
        if top2_margin(want) > MARGIN:
            assert got_id == R.greedy_argmax(want)
            compared += 1
        tok = R.greedy_argmax(want)
    return compared


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("prefill", ["batched", "sequential"])
def test_tiny_bf16_kv_prefill_and_decode(path, prefill):
    shape = W.TINY.replace(kv_format="bf16")
    wl = W.Workload("kvb", shape, seed=41, prompt_len=11, max_ctx=64)
    d = W.draw(wl, drawn_gains=True)
    m = DeviceModel(shape, d.weights, 64, max_prefill_t=64 if prefill == "batched" else 0)
    o = R.build_oracle(d)
    try:
        B.qw_set_decode_path(m.h, path)
        assert B.qw_get_decode_path(m.h) == path
        am, lg = m.prefill(d.prompt, logits=True)
        cp = o.prefill(d.prompt)
        assert violation(lg, cp["logits"]) <= 0
        assert _steps(m, o, R.greedy_argmax(cp["logits"]), 12) > 0
        n = len(d.prompt) + 12
        for l in range(shape.n_layers):
            kd, vd = m.kv(l)
            kd, vd = kd.cpu().numpy()[:, :n], vd.cpu().numpy()[:, :n]
            np.testing.assert_array_equal(R.round_bf16(kd), kd)     # bf16 values stored
            assert violation(kd, o.k_cache[l][:, :n], ATOL, KV_RTOL) <= 0
            assert violation(vd, o.v_cache[l][:, :n], ATOL, KV_RTOL) <= 0
    finally:
        m.close()


@pytest.mark.parametrize("start", [8192, 1532])
def test_qwen3_06b_longctx_bf16_kv(start):
    # the pre-filled keys and values are bf16 already, so both caches hold the same
    # context; from 1532 the steps cross the switch to the 11-warp kernel build
    wl = W.WORKLOADS["qwen3_0.6b_longctx_bf16kv"]
    d = W.draw(wl)
    m = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    o = R.build_oracle(d)
    try:
        assert B.qw_get_decode_path(m.h) == 0
        for l, (k, v) in enumerate(d.kv):
            m.set_kv(l, k, v)
        m.set_pos(start)
        o.pos = start
        steps = wl.decode_steps if start == wl.kv_prefill else 8
        assert _steps(m, o, d.start_token, steps) >= steps // 2
        kd, _ = m.kv(5)
        assert violation(kd.cpu().numpy()[:, start:start + steps],
                         o.k_cache[5][:, start:start + steps], ATOL, KV_RTOL) <= 0
    finally:
        m.close()
