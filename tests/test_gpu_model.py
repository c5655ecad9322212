"""Whole-step parity: the qw_* decode path on the GPU against the oracle.

Both sides are fed the oracle's greedy tokens (teacher forcing), so a near-tie
cannot desynchronise later steps; greedy ids must agree wherever the oracle's
top-2 margin exceeds 1e-2. Logits are checked at every step and the four
checkpoints of the "Failed Star / fs, M2" page after prefill and decode.
"""
import ctypes as C

import numpy as np
import pytest

import workload as W
from oracle import qwen_ref as R
from sequence_decode_step_gb300 import _binding as B
from sequence_decode_step_gb300.device_model import DeviceModel

from gpu_util import MARGIN, top2_margin, violation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _models(wl, drawn, max_ctx=None, cache_f64=None, max_prefill_t=0):
    m = DeviceModel(wl.shape, drawn.weights, max_ctx or wl.max_ctx, max_prefill_t=max_prefill_t)
    o = R.build_oracle(drawn, max_ctx=max_ctx, cache_f64=cache_f64)
    return m, o


def _teacher_forced(m, o, first_token, steps, check_every=1):
    """Decode `steps` steps; returns the number of greedy ids compared."""
    tok, compared = first_token, 0
    for i in range(steps):
        want = o.decode_step(tok)["logits"]
        got_id, got = m.decode(tok, logits=True)
        if i % check_every == 0 or i == steps - 1:
            v = violation(got, want)
            assert v <= 0, f"step {i}: logits off by {v}"
        ref_id = R.greedy_argmax(want)
        if top2_margin(want) > MARGIN:
            assert got_id == ref_id, f"step {i}: greedy {got_id} vs oracle {ref_id}"
            compared += 1
        tok = ref_id
    return compared


def _prefill_check(m, o, prompt, capture=True):
    if capture:
        m.set_capture(True)
    am, lg = m.prefill(prompt, logits=True)
    cp = o.prefill(prompt)
    assert violation(lg, cp["logits"]) <= 0
    if capture:
        H = m.shape.hidden
        T = len(prompt)
        for which, key in ((B.QW_CAPTURE_EMBEDDING, "embedding"), (B.QW_CAPTURE_BLOCK0, "block0"),
                           (B.QW_CAPTURE_FINAL_NORM, "final_norm")):
            got = m.capture(which).reshape(T, H)
            assert violation(got, cp[key]) <= 0, key
        assert violation(m.capture(B.QW_CAPTURE_LOGITS), cp["logits"]) <= 0
        m.set_capture(False)
    if top2_margin(cp["logits"]) > MARGIN:
        assert am == R.greedy_argmax(cp["logits"])
    return R.greedy_argmax(cp["logits"])


# ------------------------------------------------------------------ tiny (8 ids + 16 steps)
TINY_VARIANTS = {
    "tiny": (W.TINY, False),
    "tiny_drawn_gains": (W.TINY, True),
    "tiny_qwen25_style": (W.TINY.replace(qk_norm=False, qkv_bias=True, tie_word_embeddings=False,
                                         n_kv_heads=1), True),
    "tiny_hd128_gq8": (W.TINY.replace(n_q_heads=8, n_kv_heads=1, head_dim=128, hidden=512,
                                      intermediate=1280), True),
    # an intermediate width above 3072: the persistent kernel's wide-input build
    "tiny_wide_mlp": (W.TINY.replace(intermediate=3584), True),
}


@pytest.mark.parametrize("path", ["sequential", "batched"])
@pytest.mark.parametrize("name", list(TINY_VARIANTS))
def test_tiny_prefill_and_decode(name, path):
    shape, gains = TINY_VARIANTS[name]
    wl = W.Workload(name, shape, seed=0, prompt_len=8, decode_steps=16, max_ctx=64)
    d = W.draw(wl, drawn_gains=gains)
    m, o = _models(wl, d, max_prefill_t=64 if path == "batched" else 0)
    try:
        tok = _prefill_check(m, o, d.prompt)
        for l in range(shape.n_layers):          # KV cache rows written by the prompt
            kd, vd = m.kv(l)
            assert violation(kd.cpu().numpy()[:, :8], o.k_cache[l][:, :8]) <= 0
            assert violation(vd.cpu().numpy()[:, :8], o.v_cache[l][:, :8]) <= 0
        m.set_capture(True)
        n = _teacher_forced(m, o, tok, wl.decode_steps)
        assert n >= wl.decode_steps // 2
        cp_emb = m.capture(B.QW_CAPTURE_EMBEDDING)
        assert cp_emb.shape == (shape.hidden,)
        assert m.pos() == 8 + wl.decode_steps
    finally:
        m.close()


def test_tiny_greedy_loop_matches_steps_and_is_deterministic():
    wl = W.WORKLOADS["tiny"]
    d = W.draw(wl)
    m = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    try:
        first = m.prefill(d.prompt)
        loop = m.greedy(first, 16)
        m.reset()
        assert m.prefill(d.prompt) == first
        steps, tok = [], first
        logits = []
        for _ in range(16):
            tok, lg = m.decode(tok, logits=True)
            steps.append(tok)
            logits.append(lg)
        assert loop == steps
        m.reset()
        m.prefill(d.prompt)
        tok = first
        for i in range(16):                      # bit-identical run to run
            tok, lg = m.decode(tok, logits=True)
            np.testing.assert_array_equal(lg, logits[i])
        # token < 0 feeds the previous device argmax
        m.reset()
        m.prefill(d.prompt)
        got = [m.decode(-1) for _ in range(16)]
        assert got == steps
    finally:
        m.close()


# ------------------------------------------------------------------ Qwen3-0.6B shape
@pytest.fixture(scope="module")
def qwen06_decode():
    wl = W.WORKLOADS["qwen3_0.6b_decode"]
    d = W.draw(wl)
    m, o = _models(wl, d)
    yield wl, d, m, o
    m.close()


def test_qwen3_06b_decode_128_steps(qwen06_decode):
    wl, d, m, o = qwen06_decode
    tok = _prefill_check(m, o, d.prompt)
    n = _teacher_forced(m, o, tok, wl.decode_steps)
    assert n >= wl.decode_steps // 2


@pytest.fixture(scope="module")
def longctx_drawn():
    wl = W.WORKLOADS["qwen3_0.6b_longctx"]
    return wl, W.draw(wl)


def test_qwen3_06b_longctx_8k(qwen06_decode, longctx_drawn):
    wl, d = longctx_drawn
    m, o = _models(wl, d)
    try:
        for l, (k, v) in enumerate(d.kv):
            m.set_kv(l, k, v)
        m.set_pos(wl.kv_prefill)
        assert o.pos == wl.kv_prefill
        n = _teacher_forced(m, o, d.start_token, wl.decode_steps)
        assert n >= wl.decode_steps // 2
        kd, _ = m.kv(5)                          # rows appended after the prefilled ones
        p = wl.kv_prefill
        assert violation(kd.cpu().numpy()[:, p:p + wl.decode_steps],
                         o.k_cache[5][:, p:p + wl.decode_steps]) <= 0
    finally:
        m.close()


def test_decode_across_the_long_context_switch(longctx_drawn):
    # positions 1532..1539: the step switches from the 7-warp to the 11-warp
    # build of the persistent kernel at 1536 keys (the graph is re-recorded);
    # every step matches the oracle on both sides of the switch
    wl, d = longctx_drawn
    m, o = _models(wl, d)
    try:
        for l, (k, v) in enumerate(d.kv):
            m.set_kv(l, k, v)
        m.set_pos(1532)
        o.pos = 1532
        assert B.qw_get_decode_path(m.h) == 0
        n = _teacher_forced(m, o, d.start_token, 8)
        assert n >= 4
        kd, _ = m.kv(3)
        assert violation(kd.cpu().numpy()[:, 1532:1540], o.k_cache[3][:, 1532:1540]) <= 0
        # a device-resident greedy run across the switch (the graph is replaced while
        # earlier replays are queued) gives the ids of the same run step by step
        m.set_pos(1532)
        ids_run = m.greedy(d.start_token, 8)
        m.set_pos(1532)
        ids_steps, tok = [], d.start_token
        for _ in range(8):
            tok = m.decode(tok)
            ids_steps.append(tok)
        assert list(ids_run) == ids_steps
    finally:
        m.close()


def test_qwen3_06b_prefill_1024():
    # one batched causal pass (tensor-core GEMMs) against the oracle's no-cache
    # prefill, and against 1024 sequential decode steps of the same ids on the GPU
    wl = W.WORKLOADS["qwen3_0.6b_prefill"]
    d = W.draw(wl)
    m, o = _models(wl, d, max_prefill_t=1024)
    seq = DeviceModel(wl.shape, d.weights, wl.max_ctx)       # max_prefill_t = 0: sequential
    try:
        m.set_capture(True)
        am, lg = m.prefill(d.prompt, logits=True)
        cp = o.prefill(d.prompt)
        assert violation(lg, cp["logits"]) <= 0
        T, H = 1024, wl.shape.hidden
        for which, key in ((B.QW_CAPTURE_EMBEDDING, "embedding"), (B.QW_CAPTURE_BLOCK0, "block0"),
                           (B.QW_CAPTURE_FINAL_NORM, "final_norm")):
            assert violation(m.capture(which).reshape(T, H), cp[key]) <= 0, key
        am_s, lg_s = seq.prefill(d.prompt, logits=True)
        assert violation(lg, lg_s) <= 0
        if top2_margin(cp["logits"]) > MARGIN:
            assert am == am_s == R.greedy_argmax(cp["logits"])
        for l in (0, 13, 27):
            kd, vd = m.kv(l)
            ks, vs = seq.kv(l)
            kd, vd = kd.cpu().numpy()[:, :T], vd.cpu().numpy()[:, :T]
            assert violation(kd, o.k_cache[l][:, :T]) <= 0
            assert violation(vd, o.v_cache[l][:, :T]) <= 0
            assert violation(kd, ks.cpu().numpy()[:, :T]) <= 0
            assert violation(vd, vs.cpu().numpy()[:, :T]) <= 0
        assert m.pos() == seq.pos() == 1024
        # decoding continues from the batched prefill's cache and greedy id
        tok = R.greedy_argmax(cp["logits"])
        _teacher_forced(m, o, tok, 4)
    finally:
        m.close()
        seq.close()


def test_batched_prefill_in_two_chunks_and_sequential_fallback():
    # a second prompt chunk starts at pos = 5 and attends to the first chunk's cache;
    # a chunk longer than max_prefill_t takes the sequential path
    wl = W.Workload("chunks", W.TINY, seed=3, max_ctx=64)
    d = W.draw(wl, drawn_gains=True)
    ids = list(W.random_ids(W.TINY.vocab, 30, seed=9))
    m = DeviceModel(W.TINY, d.weights, 64, max_prefill_t=16)
    o = R.build_oracle(d)
    try:
        m.prefill(ids[:5])
        m.prefill(ids[5:12])
        m.prefill(ids[12:30])                         # 18 > 16: sequential fallback
        am, lg = m.decode(ids[0], logits=True)
        o.prefill(ids)
        want = o.decode_step(ids[0])["logits"]
        assert violation(lg, want) <= 0
        kd, _ = m.kv(1)
        assert violation(kd.cpu().numpy()[:, :31], o.k_cache[1][:, :31]) <= 0
    finally:
        m.close()


def test_batched_prefill_ragged_chunks_head_dim_128():
    # Qwen3-0.6B layer shape (head_dim 128, 16 / 8 heads), two layers: chunks of 200 and
    # 333 ids, so query blocks end mid-block, the second chunk starts at p0 = 200 and
    # attends to the first chunk's cache, and key tiles end mid-tile
    shape = W.QWEN3_0_6B.replace(n_layers=2)
    wl = W.Workload("ragged", shape, seed=21, max_ctx=600)
    d = W.draw(wl, drawn_gains=True)
    ids = list(W.random_ids(shape.vocab, 533, seed=22))
    m = DeviceModel(shape, d.weights, 600, max_prefill_t=400)
    o = R.build_oracle(d, cache_f64=False)
    try:
        m.prefill(ids[:200])
        am, lg = m.prefill(ids[200:], logits=True)
        cp = o.prefill(ids)
        assert violation(lg, cp["logits"]) <= 0
        for l in range(2):
            kd, vd = m.kv(l)
            assert violation(kd.cpu().numpy()[:, :533], o.k_cache[l][:, :533]) <= 0
            assert violation(vd.cpu().numpy()[:, :533], o.v_cache[l][:, :533]) <= 0
        if top2_margin(cp["logits"]) > MARGIN:
            assert am == R.greedy_argmax(cp["logits"])
        _teacher_forced(m, o, R.greedy_argmax(cp["logits"]), 3)
    finally:
        m.close()


# ------------------------------------------------------------------ error paths
def test_error_paths_on_device():
    wl = W.WORKLOADS["tiny"]
    d = W.draw(wl)
    m = DeviceModel(wl.shape, d.weights, max_ctx=12)
    L = B.lib()
    try:
        out = C.c_int32()
        assert L.qw_decode_step(m.h, -1, None, C.byref(out)) == B.QW_ERR_STATE
        assert L.qw_decode_step(m.h, wl.shape.vocab, None, C.byref(out)) == B.QW_ERR_ARG
        ids = (C.c_int32 * 3)(1, 2, 99999)
        assert L.qw_prefill(m.h, ids, 3, None, None) == B.QW_ERR_ARG
        assert L.qw_prefill(m.h, ids, 0, None, None) == B.QW_ERR_ARG          # empty prompt
        n = C.c_size_t()
        assert L.qw_capture_size(m.h, 0, C.byref(n)) == B.QW_ERR_NOT_CAPTURED
        m.set_capture(True)
        assert L.qw_capture_size(m.h, 0, C.byref(n)) == B.QW_ERR_NOT_CAPTURED  # no forward yet
        m.prefill(d.prompt)
        assert L.qw_capture_size(m.h, 0, C.byref(n)) == 0 and n.value == 8 * wl.shape.hidden
        buf = (C.c_float * 10)()
        assert L.qw_get_capture(m.h, 0, buf, 10) == B.QW_ERR_SIZE
        m.set_capture(False)
        long_ids = (C.c_int32 * 5)(1, 2, 3, 4, 5)
        assert L.qw_prefill(m.h, long_ids, 5, None, None) == B.QW_ERR_CTX       # 8 + 5 > 12
        assert m.pos() == 8
        # a device wait that gives up at once reports QW_ERR_DEVICE_TIMEOUT ...
        B.qw_set_wait_limit_ns(m.h, 0)
        assert L.qw_decode_step(m.h, 3, None, C.byref(out)) == B.QW_ERR_DEVICE_TIMEOUT
        # ... and the handle stays usable afterwards
        B.qw_set_wait_limit_ns(m.h, 1_000_000_000)
        m.reset()
        o = R.build_oracle(d, max_ctx=12)
        am, lg = m.prefill(d.prompt, logits=True)
        assert violation(lg, o.prefill(d.prompt)["logits"]) <= 0
    finally:
        m.close()


@pytest.mark.parametrize("workload_name,steps", [("tiny", 16), ("qwen3_0.6b_decode", 24)])
def test_persistent_and_multikernel_paths_agree(workload_name, steps):
    # the default decode path (one persistent cooperative kernel per token) and
    # the graph of separate kernels compute the same step
    wl = W.WORKLOADS[workload_name]
    d = W.draw(wl)
    m, o = _models(wl, d)
    m2 = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    try:
        assert B.qw_get_decode_path(m.h) == 0          # the persistent kernel fits these shapes
        B.qw_set_decode_path(m2.h, 1)
        assert B.qw_get_decode_path(m2.h) == 1
        tok = _prefill_check(m, o, d.prompt, capture=False)
        m2.prefill(d.prompt)
        for i in range(steps):
            want = o.decode_step(tok)["logits"]
            a1, l1 = m.decode(tok, logits=True)
            a2, l2 = m2.decode(tok, logits=True)
            assert violation(l1, want) <= 0 and violation(l2, want) <= 0
            assert violation(l1, l2, 1e-4, 1e-4) <= 0
            if top2_margin(want) > MARGIN:
                assert a1 == a2 == R.greedy_argmax(want)
            tok = R.greedy_argmax(want)
        # both paths are deterministic run to run
        m.reset()
        m.prefill(d.prompt)
        ids1 = m.greedy(tok, 8)
        m.reset()
        m.prefill(d.prompt)
        assert m.greedy(tok, 8) == ids1
    finally:
        m.close()
        m2.close()


@pytest.mark.parametrize("path", [0, 1])
def test_greedy_argmax_ties_and_nan_in_the_decode_step(path):
    # Two logits exactly equal: embedding rows i and j set to a * e_c make both logits
    # a * h[c] whatever the summation order (every other product is an exact zero).
    # The lowest id must win, across CTAs, across warps of one CTA and within a warp
    # ("flashmoon demo", Performance: argmax on the device, ties to the lowest id).
    # A NaN weight in one row makes its logit NaN: QW_ERR_NUMERIC, and the handle
    # stays usable.
    wl = W.WORKLOADS["tiny"]
    d = W.draw(wl)
    tok = int(d.prompt[0])
    h = R.build_oracle(d).decode_step(tok)["final_norm"][0]
    c = int(np.argmax(h))
    assert h[c] > 0.5
    row = np.zeros(wl.shape.hidden, np.float32)
    row[c] = 64.0
    m = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    try:
        B.qw_set_decode_path(m.h, path)
        assert B.qw_get_decode_path(m.h) == path
        for i, j in ((100, 3000), (1000, 1001), (2000, 2008), (5, 4095), (3001, 2990)):
            assert tok not in (i, j)
            w = dict(d.weights)
            w["embed"] = d.weights["embed"].copy()
            w["embed"][[i, j]] = W.f32_to_bf16_bits(row)
            m.load(w)
            B.qw_set_decode_path(m.h, path)
            am, lg = m.decode(tok, logits=True)
            assert lg[i] == lg[j] == lg.max()
            want = R.build_oracle(W.DrawnWorkload(wl, w)).decode_step(tok)["logits"]
            assert want[i] == want[j] and R.greedy_argmax(want) == min(i, j)
            assert am == min(i, j), (i, j, am)
        w = dict(d.weights)
        w["embed"] = d.weights["embed"].copy()
        w["embed"][777, 3] = 0x7FC0                     # bf16 NaN
        m.load(w)
        B.qw_set_decode_path(m.h, path)
        with pytest.raises(B.QwError) as e:
            m.decode(tok)
        assert e.value.code == B.QW_ERR_NUMERIC
        m.load(d.weights)
        B.qw_set_decode_path(m.h, path)
        want = R.build_oracle(d).decode_step(tok)["logits"]
        am, lg = m.decode(tok, logits=True)
        assert violation(lg, want) <= 0 and am == R.greedy_argmax(want)
    finally:
        m.close()
