"""Kernel-level parity: each stand-alone op of libqw.so against the oracle's
corresponding functions ("flashmoon demo" page, Verification: kernel unit
checks against an f64 oracle). Shapes span several tiles/splits and a ragged tail.
"""
import os

import numpy as np
import pytest

from oracle import qwen_ref as R
from sequence_decode_step_gb300 import _binding as B
import workload as W

from gpu_util import dev, host, violation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available()
    return B.lib()


def _quantize_gpu(L, w):
    rows, cols = w.shape
    wd = dev(w)
    packed = torch.zeros((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((rows, cols // 128), dtype=torch.int16, device="cuda")
    assert L.qw_quantize_int4_g128(wd.data_ptr(), rows, cols, packed.data_ptr(),
                                   scales.data_ptr(), None) == 0
    return host(packed), host(scales, np.uint16)


def test_quantize_int4_bit_exact(L):
    rng = np.random.default_rng(21)
    w = rng.standard_normal((301, 1024)).astype(np.float32) * 0.02
    w[7, :128] = 0.0                                  # an all-zero group: scale 0
    w[9, 128:256] *= 1e-30                            # subnormal-sized group
    p, s = _quantize_gpu(L, w)
    pr, sr = R.int4_quantize(w)
    np.testing.assert_array_equal(s, sr)
    np.testing.assert_array_equal(p, pr)


def test_quantize_int4_golden_row(L):
    from test_oracle_pins import _read_int4_golden
    vals, scales, head, fill, _ = _read_int4_golden()
    w = np.zeros((1, 256), np.float32)
    for i, x in vals.items():
        w[0, i] = x
    p, s = _quantize_gpu(L, w)
    assert list(s[0]) == scales
    assert list(p[0]) == head + [fill] * (128 - len(head))


def _attn_case(L, hd, nq, nkv, qk_norm, pos, n_splits, seed):
    rng = np.random.default_rng(seed)
    cap = pos + 3
    qkv = rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32)
    kc = rng.standard_normal((nkv, cap, hd)).astype(np.float32)
    vc = rng.standard_normal((nkv, cap, hd)).astype(np.float32)
    gq = W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(hd).astype(np.float32))
    gk = W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(hd).astype(np.float32))
    eps, theta = 1e-6, 1e6
    # oracle
    q = qkv[: nq * hd].reshape(1, nq, hd)
    k = qkv[nq * hd:(nq + nkv) * hd].reshape(1, nkv, hd)
    v = qkv[(nq + nkv) * hd:].reshape(1, nkv, hd)
    if qk_norm:
        q = R.rmsnorm(q, R.widen_bf16(gq), eps)
        k = R.rmsnorm(k, R.widen_bf16(gk), eps)
    c, s_ = R.rope_cos_sin([pos], hd, theta)
    q, k = R.apply_rope(q, c, s_), R.apply_rope(k, c, s_)
    kref, vref = kc.copy(), vc.copy()
    kref[:, pos], vref[:, pos] = k[0], v[0]
    want = R.causal_gqa_attention(q, np.array([pos]), kref[:, :pos + 1], vref[:, :pos + 1],
                                  np.arange(pos + 1)).reshape(-1)
    # GPU
    d_qkv, d_k, d_v = dev(qkv), dev(kc), dev(vc)
    d_gq, d_gk = dev(gq), dev(gk)
    out = torch.full((nq * hd,), float("nan"), device="cuda")
    ws_bytes = L.qw_attention_workspace_bytes(nq, nkv, hd, n_splits)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):                      # twice: the workspace must come back zeroed
        rc = L.qw_attention_decode(d_qkv.data_ptr(), d_gq.data_ptr() if qk_norm else None,
                                   d_gk.data_ptr() if qk_norm else None, d_k.data_ptr(),
                                   d_v.data_ptr(), nq, nkv, hd, cap, pos, eps, theta, n_splits,
                                   out.data_ptr(), ws.data_ptr(), ws_bytes, None)
        assert rc == 0, B.last_error()
        outs.append(host(out).copy())
    np.testing.assert_array_equal(outs[0], outs[1])
    assert violation(outs[0], want, 1e-4, 1e-4) <= 0, np.abs(outs[0] - want).max()
    kg, vg = host(d_k), host(d_v)
    assert violation(kg[:, pos], k[0], 1e-5, 1e-5) <= 0
    np.testing.assert_array_equal(vg[:, pos], v[0])
    np.testing.assert_array_equal(np.delete(kg, pos, axis=1), np.delete(kc, pos, axis=1))


@pytest.mark.parametrize("hd,nq,nkv,qk_norm,pos,n_splits", [
    (64, 4, 2, True, 0, 4),          # first position: a single key
    (64, 4, 2, True, 37, 4),         # two tiles, ragged
    (64, 4, 2, True, 200, 4),        # several splits
    (128, 16, 8, True, 300, 19),
    (128, 16, 2, False, 1000, 76),   # 8 query heads per kv head (Qwen2.5-3B shape)
    (128, 8, 8, True, 129, 3),       # MHA
    (128, 16, 8, True, 8192, 19),    # long context: 8193 keys over 19 splits
])
def test_attention_decode_vs_oracle(L, hd, nq, nkv, qk_norm, pos, n_splits):
    _attn_case(L, hd, nq, nkv, qk_norm, pos, n_splits, seed=pos + nq)


def _lm_head(L, x, g, table, eps=1e-6):
    V, H = table.shape
    lg = torch.full((V,), float("nan"), device="cuda")
    am = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(L.qw_lm_head_workspace_bytes(), dtype=torch.uint8, device="cuda")
    dx, dg, dt = dev(x), dev(g), dev(table)
    res = []
    for _ in range(2):
        rc = L.qw_lm_head_argmax(dx.data_ptr(), dg.data_ptr(), dt.data_ptr(), V, H, eps,
                                 lg.data_ptr(), am.data_ptr(), ws.data_ptr(),
                                 L.qw_lm_head_workspace_bytes(), None)
        assert rc == 0, B.last_error()
        res.append((host(lg).copy(), int(host(am)[0])))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    assert res[0][1] == res[1][1]
    return res[0]


@pytest.mark.parametrize("V,H", [(4099, 256), (151936, 1024), (777, 2048), (5000, 3072)])
def test_lm_head_argmax_vs_oracle(L, V, H):
    rng = np.random.default_rng(V + H)
    x = rng.standard_normal(H).astype(np.float32)
    g = W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(H).astype(np.float32))
    table = W.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * 0.02)
    lg, am = _lm_head(L, x, g, table)
    h = R.rmsnorm(x[None], R.widen_bf16(g), 1e-6)
    want = R.linear(h, R.widen_bf16(table).astype(np.float64))[0]
    assert violation(lg, want, 1e-4, 1e-4) <= 0
    top = np.sort(want)[-2:]
    if top[1] - top[0] > 1e-4:
        assert am == int(np.argmax(want))
    else:
        assert abs(want[am] - top[1]) <= 1e-4


def test_lm_head_argmax_ties_and_nan(L):
    rng = np.random.default_rng(5)
    V, H = 3001, 256
    x = rng.standard_normal(H).astype(np.float32)
    g = np.full(H, 0x3F80, np.uint16)
    table = W.f32_to_bf16_bits(rng.standard_normal((V, H)).astype(np.float32) * 0.02)
    big = W.f32_to_bf16_bits(np.sign(x).astype(np.float32))
    table[2999] = big
    table[17] = big                      # equal rows in different CTAs: lowest id wins
    lg, am = _lm_head(L, x, g, table)
    assert lg[17] == lg[2999] and am == 17
    table[400, 3] = 0x7FC0               # a NaN weight makes one logit NaN
    lg, am = _lm_head(L, x, g, table)
    assert np.isnan(lg[400]) and am == -1


# ------------------------------------------------------------------ int4 dequantisation, bit for bit
def _gemv_int4(L, packed, scales, x):
    rows, cols = packed.shape[0], packed.shape[1] * 2
    wsb = L.qw_gemv_int4_workspace_bytes(rows, cols)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y = torch.full((rows,), float("nan"), device="cuda")
    dp, ds, dx = dev(packed), dev(scales), dev(x)
    rc = L.qw_gemv_int4_g128(dp.data_ptr(), ds.data_ptr(), rows, cols, dx.data_ptr(),
                             y.data_ptr(), ws.data_ptr(), wsb, None)
    assert rc == 0, B.last_error()
    return host(y)


@pytest.mark.parametrize("rows,cols", [(300, 384), (2048, 11008)])
def test_int4_gemv_one_hot_is_the_dequantised_column_bit_for_bit(L, rows, cols):
    # "Emberglass" README, "Why it's hard": int4 group-128. The GEMV dequantises in
    # registers ((nibble - 8) times the group's bf16 scale); with x = e_j every
    # product but one is an exact zero, so y is column j of the oracle's
    # dequantised matrix exactly. cols = 11008 takes the wide-input kernel variant.
    rng = np.random.default_rng(rows + cols)
    w = rng.standard_normal((rows, cols)).astype(np.float32) * 0.02
    w[rows // 3, :128] = 0.0                    # an all-zero group: scale 0
    packed, scales = R.int4_quantize(w)
    deq = R.int4_dequantize(packed, scales)
    for j in sorted({0, 1, 2, 127, 128, 255, 256, cols // 2 + 1, cols - 2, cols - 1,
                     *rng.integers(0, cols, 4).tolist()}):
        x = np.zeros(cols, np.float32)
        x[j] = 1.0
        got = _gemv_int4(L, packed, scales, x)
        np.testing.assert_array_equal(got.view(np.uint32), deq[:, j].view(np.uint32),
                                      err_msg=f"column {j}")
    # a dense input within the kernel-check tolerance of the f64 product
    x = rng.standard_normal(cols).astype(np.float32)
    want = R.linear(x[None], deq.astype(np.float64))[0]
    assert violation(_gemv_int4(L, packed, scales, x), want, 1e-4, 1e-4) <= 0
