"""tcgen05 GEMM (the prefill contraction) against an f64 product of the same bf16 operands.

C = (A_hi + A_lo) . B^T where A_hi, A_lo, B are bf16; the reference widens the
exact bf16 values to f64, so the only difference is the tensor core's f32
accumulation. Shapes cover one tile, ragged M/N/K tails, every tile width and
the Qwen3-0.6B prefill shapes.
"""
import numpy as np
import pytest

import workload as W
from sequence_decode_step_gb300 import _binding as B

from gpu_util import dev, host, violation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _split(x):
    hi = W.f32_to_bf16_bits(x)
    lo = W.f32_to_bf16_bits(x - W.bf16_bits_to_f32(hi))
    return hi, lo


def _run(M, N, K, bn, split, seed=0):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    w = W.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32) * 0.02)
    hi, lo = _split(a)
    c = torch.full((M, N), float("nan"), device="cuda")
    d_hi, d_lo, d_w = dev(hi), dev(lo), dev(w)
    rc = B.lib().qw_gemm_bf16(d_hi.data_ptr(), d_lo.data_ptr() if split else None,
                              d_w.data_ptr(), M, N, K, c.data_ptr(), bn, None)
    assert rc == 0, B.last_error()
    got = host(c)
    a_used = W.bf16_bits_to_f32(hi).astype(np.float64)
    if split:
        a_used = a_used + W.bf16_bits_to_f32(lo).astype(np.float64)
    want = a_used @ W.bf16_bits_to_f32(w).astype(np.float64).T
    scale = np.sqrt(K) * 0.02
    err = np.abs(got - want).max() / scale
    assert np.isfinite(got).all()
    assert err < 5e-5, err   # f32 accumulation over K; a layout slip gives O(1)
    if split:   # the split recovers the f32 activations to ~2^-16
        exact = a.astype(np.float64) @ W.bf16_bits_to_f32(w).astype(np.float64).T
        assert violation(got, exact, 1e-4 * scale, 1e-4) <= 0


@pytest.mark.parametrize("M,N,K,bn,split", [
    (128, 64, 64, 64, False),       # one tile, one k-tile
    (128, 64, 64, 64, True),
    (128, 128, 256, 128, True),
    (128, 256, 512, 256, True),
    (200, 320, 1000, 64, True),     # ragged M, N and K tails
    (333, 200, 136, 128, False),
    (1024, 4096, 1024, 256, True),  # Qwen3-0.6B prefill: QKV
    (1024, 1024, 3072, 64, True),   # down
])
def test_gemm_vs_f64(M, N, K, bn, split):
    _run(M, N, K, bn, split, seed=M + N + K)
