"""qw_attention_decode_noalloc: the decode-attention entry point for callers
that cannot allocate device memory (for example code running while a CUDA
graph is being captured, or an embedder whose GPU memory belongs to another
allocator). It keeps its scratch in a fixed device array inside the library
instead of taking a workspace.

Checked here through the C ABI against qw_attention_decode (the entry point
with a caller workspace) on two calls in a row, with the same tolerance as the
other kernel-level checks. This file is collected last on purpose.
"""
import numpy as np
import pytest

import workload as W
from sequence_decode_step_gb300 import _binding as B

from gpu_util import dev, host, violation

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.mark.parametrize("hd,nq,nkv,pos,n_splits", [(128, 16, 8, 700, 19), (64, 4, 2, 45, 4)])
def test_noalloc_matches_workspace_entry_point(hd, nq, nkv, pos, n_splits):
    L = B.lib()
    rng = np.random.default_rng(pos)
    cap = pos + 4
    kc = rng.standard_normal((nkv, cap, hd)).astype(np.float32)
    vc = rng.standard_normal((nkv, cap, hd)).astype(np.float32)
    gq = dev(W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(hd).astype(np.float32)))
    gk = dev(W.f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(hd).astype(np.float32)))
    # two independent caches, one per entry point
    k_ws, v_ws, k_na, v_na = dev(kc), dev(vc), dev(kc), dev(vc)
    wsb = L.qw_attention_workspace_bytes(nq, nkv, hd, n_splits)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    out_ws = torch.empty(nq * hd, device="cuda")
    out_na = torch.empty(nq * hd, device="cuda")
    for step in range(2):                     # two calls in a row: pos, then pos + 1
        p = pos + step
        qkv = dev(rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32))
        rc = L.qw_attention_decode(qkv.data_ptr(), gq.data_ptr(), gk.data_ptr(),
                                   k_ws.data_ptr(), v_ws.data_ptr(), nq, nkv, hd, cap, p, 1e-6,
                                   1e6, n_splits, out_ws.data_ptr(), ws.data_ptr(), wsb, None)
        assert rc == 0, B.last_error()
        out_na.fill_(float("nan"))
        rc = L.qw_attention_decode_noalloc(qkv.data_ptr(), gq.data_ptr(), gk.data_ptr(),
                                           k_na.data_ptr(), v_na.data_ptr(), nq, nkv, hd, cap, p,
                                           1e-6, 1e6, n_splits, out_na.data_ptr(), None)
        assert rc == 0
        want = host(out_ws)
        assert violation(host(out_na), want, 1e-4, 1e-4) <= 0
        assert violation(host(k_na)[:, p], host(k_ws)[:, p], 1e-4, 1e-4) <= 0
        np.testing.assert_array_equal(host(v_na)[:, p], host(v_ws)[:, p])


def test_noalloc_rejects_shapes_beyond_its_scratch():
    L = B.lib()
    limit = L.qw_attention_noalloc_max_bytes()
    assert limit == 1 << 20
    # 16 heads x 1000 splits x (128 + 2) floats is about 8 MB > 1 MiB: refused, nothing runs
    rc = L.qw_attention_decode_noalloc(1, None, None, 1, 1, 16, 8, 128, 10, 0, 1e-6, 1e6, 1000,
                                       1, None)
    assert rc == B.QW_ERR_SIZE
