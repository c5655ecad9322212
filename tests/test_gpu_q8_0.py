"""Q8_0 weights on the GPU ("SuperKittens PR #7" page, Q8_0 commit: GGUF type-8
projections and LM head read by a q8_0 matvec at decode).

The device quantiser and the int8 dequantisation inside the GEMV are checked bit for
bit against the oracle; whole-model decode (tied head quantised from the embedding
table, and an untied head) on both decode paths (the persistent kernel and the graph of
separate kernels) against the oracle's Q8_0 model at the model tolerance.
"""
import numpy as np
import pytest

import workload as W
from oracle import qwen_ref as R
from sequence_decode_step_gb300 import _binding as B
from sequence_decode_step_gb300.device_model import DeviceModel

from gpu_util import MARGIN, dev, host, top2_margin, violation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available()
    return B.lib()


def _quantize_gpu(L, w):
    rows, cols = w.shape
    wd = dev(w)
    q = torch.zeros((rows, cols), dtype=torch.int8, device="cuda")
    s = torch.zeros((rows, cols // 32), dtype=torch.int16, device="cuda")
    assert L.qw_quantize_q8_0(wd.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr(), None) == 0
    return host(q), host(s, np.uint16)


def test_quantize_q8_0_bit_exact(L):
    rng = np.random.default_rng(31)
    w = rng.standard_normal((257, 1024)).astype(np.float32) * 0.02
    w[3, :32] = 0.0                                   # an all-zero block: scale 0
    w[5, 32:64] *= 1e-3                               # a block whose scale is an fp16 subnormal
    w[6, 64:96] = np.float32(2.5 / 128)               # ties at every input
    w[6, 64] = np.float32(127 / 128)
    q, s = _quantize_gpu(L, w)
    qr, sr = R.q8_0_quantize(w)
    np.testing.assert_array_equal(s, sr)
    np.testing.assert_array_equal(q, qr)


def test_quantize_q8_0_golden_row(L):
    vals, q_want, scales = {}, {}, []
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "q8_0_block_example.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "w":
                vals[int(t[1])] = float(t[2])
            elif t[0] == "q":
                q_want[int(t[1])] = int(t[2])
            elif t[0] == "scale_bits":
                scales = [int(x, 16) for x in t[1:]]
    w = np.zeros((1, 96), np.float32)
    for i, x in vals.items():
        w[0, i] = x
    q, s = _quantize_gpu(L, w)
    assert list(s[0]) == scales
    want = np.zeros(96, np.int8)
    for i, x in q_want.items():
        want[i] = x
    np.testing.assert_array_equal(q[0], want)


def _gemv_q8(L, q, s, x):
    rows, cols = q.shape
    wsb = L.qw_gemv_q8_0_workspace_bytes(rows, cols)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y = torch.full((rows,), float("nan"), device="cuda")
    dq, ds, dx = dev(q), dev(s), dev(x)
    rc = L.qw_gemv_q8_0(dq.data_ptr(), ds.data_ptr(), rows, cols, dx.data_ptr(), y.data_ptr(),
                        ws.data_ptr(), wsb, None)
    assert rc == 0, B.last_error()
    return host(y)


@pytest.mark.parametrize("rows,cols", [(300, 384), (1024, 3072), (64, 11008)])
def test_q8_0_gemv_one_hot_is_the_dequantised_column_bit_for_bit(L, rows, cols):
    rng = np.random.default_rng(rows + cols)
    w = rng.standard_normal((rows, cols)).astype(np.float32) * 0.02
    q, s = R.q8_0_quantize(w)
    deq = R.q8_0_dequantize(q, s)
    for j in sorted({0, 1, 31, 32, 255, 256, cols // 2 + 3, cols - 1,
                     *rng.integers(0, cols, 4).tolist()}):
        x = np.zeros(cols, np.float32)
        x[j] = 1.0
        got = _gemv_q8(L, q, s, x)
        np.testing.assert_array_equal(got.view(np.uint32), deq[:, j].view(np.uint32),
                                      err_msg=f"column {j}")
    x = rng.standard_normal(cols).astype(np.float32)
    want = R.linear(x[None], deq.astype(np.float64))[0]
    assert violation(_gemv_q8(L, q, s, x), want, 1e-4, 1e-4) <= 0


def _decode_vs_oracle(wl, steps, path=0):
    d = W.draw(wl)
    m = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    o = R.build_oracle(d)
    try:
        B.qw_set_decode_path(m.h, path)                 # 0: the persistent kernel, 1: the graph
        assert B.qw_get_decode_path(m.h) == path
        am, lg = m.prefill(d.prompt, logits=True)
        want = o.prefill(d.prompt)["logits"]
        assert violation(lg, want) <= 0
        tok, compared = R.greedy_argmax(want), 0
        for i in range(steps):
            want = o.decode_step(tok)["logits"]
            got_id, got = m.decode(tok, logits=True)
            assert violation(got, want) <= 0, f"step {i}"
            if top2_margin(want) > MARGIN:
                assert got_id == R.greedy_argmax(want)
                compared += 1
            tok = R.greedy_argmax(want)
        assert compared > 0
    finally:
        m.close()


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("tied", [True, False])
def test_tiny_q8_0_decode(tied, path):
    shape = W.TINY.replace(weight_format="q8_0", tie_word_embeddings=tied)
    _decode_vs_oracle(W.Workload("tiny_q8", shape, seed=32, prompt_len=6, max_ctx=64), 12, path)


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("shape", [W.TINY.replace(weight_format="q8_0", kv_format="bf16"),
                                   W.TINY.replace(weight_format="q8_0", intermediate=3584)],
                         ids=["bf16kv", "wide"])
def test_tiny_q8_0_wide_build(shape, path):
    # Q8_0 with the bf16 cache, and inputs wider than 3072: the persistent kernel's
    # wide-input build
    _decode_vs_oracle(W.Workload("tiny_q8w", shape, seed=33, prompt_len=6, max_ctx=64), 12, path)


@pytest.mark.parametrize("path", [0, 1])
def test_qwen3_06b_q8_0_decode(path):
    _decode_vs_oracle(W.WORKLOADS["qwen3_0.6b_q8_0_decode"], 16, path)
