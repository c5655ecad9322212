"""On-device sampling (temperature / top-k / top-p with the draw supplied by the
caller) against the oracle's definition, through the C ABI.

The token is an integer decided by float comparisons of running sums; both sides
form the weights and running sums in float64 but their exp may differ in the last
bit, so a case whose decision sits within 1e-9 (relative) of a threshold is not
compared (the oracle reports that margin). Ties between equal logits are exact
and are compared always.
"""
import numpy as np
import pytest

import workload as W
from oracle import qwen_ref as R
from sequence_decode_step_gb300 import _binding as B
from sequence_decode_step_gb300.device_model import DeviceModel

from gpu_util import dev, host

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [(1.0, 1, 1.0), (0.0, 50, 0.9), (0.7, 40, 0.9), (1.0, 256, 1.0), (1.3, 100, 0.5),
         (2.0, 7, 0.99), (0.05, 256, 0.95)]


@pytest.fixture(scope="module")
def L():
    return B.lib()


def _sample(L, x_dev, V, T, k, p, u):
    ws = torch.empty(L.qw_sample_workspace_bytes(V, k), dtype=torch.uint8, device="cuda")
    tok = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    B.qw_sample(x_dev.data_ptr(), V, T, k, p, u, tok.data_ptr(), ws.data_ptr(), ws.numel())
    return int(host(tok)[0])


@pytest.mark.parametrize("V", [151936, 4096, 37, 16385])
def test_sample_vs_oracle(L, V):
    rng = np.random.default_rng(V)
    x = (rng.standard_normal(V) * 3).astype(np.float32)
    xd = dev(x)
    compared = 0
    for T, k, p in CASES:
        for u in (0.0, 0.013, 0.31, 0.5, 0.77, 0.999):
            want, margin = R.sample_logits(x, T, k, p, u)
            got = _sample(L, xd, V, T, k, p, u)
            if margin > 1e-9:
                assert got == want, (V, T, k, p, u, got, want)
                compared += 1
            else:
                assert 0 <= got < V
    assert compared >= len(CASES) * 5


def test_sample_ties_go_to_the_lower_index(L):
    # logits on a coarse grid: many exact ties across slices and levels
    V = 151936
    rng = np.random.default_rng(11)
    x = (np.round(rng.standard_normal(V) * 2) / 2).astype(np.float32)
    xd = dev(x)
    for T, k, p in [(0.0, 64, 1.0), (1.0, 256, 1.0), (0.9, 100, 0.8)]:
        for u in (0.0, 0.2, 0.6, 0.95):
            want, margin = R.sample_logits(x, T, k, p, u)
            got = _sample(L, xd, V, T, k, p, u)
            if margin > 1e-9:
                assert got == want, (T, k, p, u, got, want)
    # greedy on ties: the lowest index of the maximum
    assert _sample(L, xd, V, 0.0, 8, 1.0, 0.5) == R.greedy_argmax(x)


def test_sample_nan_and_no_finite_logit(L):
    V = 5000
    x = np.random.default_rng(3).standard_normal(V).astype(np.float32)
    x[4321] = np.nan
    assert _sample(L, dev(x), V, 1.0, 16, 0.9, 0.5) == -1
    assert _sample(L, dev(x), V, 0.0, 16, 0.9, 0.5) == -1
    y = np.full(V, -np.inf, np.float32)
    assert _sample(L, dev(y), V, 1.0, 16, 0.9, 0.5) == -1
    y[17] = 0.25                                          # one finite logit among -inf
    assert _sample(L, dev(y), V, 1.0, 16, 0.9, 0.7) == 17


def test_sample_last_after_a_decode_step():
    # the handle samples its own last logits without a readback; compared with the
    # oracle's sampling of the same (GPU) logits row
    wl = W.WORKLOADS["tiny"]
    d = W.draw(wl)
    m = DeviceModel(wl.shape, d.weights, wl.max_ctx)
    try:
        with pytest.raises(B.QwError):
            m.sample(1.0, 8, 0.9, 0.5)                    # no step yet
        tok = m.prefill(d.prompt)
        for step in range(4):
            _, lg = m.decode(tok, logits=True)
            for T, k, p, u in [(0.8, 40, 0.9, 0.37), (1.0, 256, 1.0, 0.81), (0.0, 5, 1.0, 0.5)]:
                want, margin = R.sample_logits(lg, T, k, p, u)
                got = m.sample(T, k, p, u)
                if margin > 1e-9:
                    assert got == want, (step, T, k, p, u)
            tok = m.sample(0.8, 40, 0.9, (step + 0.5) / 4)
    finally:
        m.close()
