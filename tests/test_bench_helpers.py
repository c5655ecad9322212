"""Host-side bench helpers: the ncu traffic of a kernel is reported only for the exact
sources it was captured from, and the byte counts of the roofline lines."""
import importlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture()
def bench():
    return importlib.import_module("bench")


def test_traffic_only_for_the_captured_sources(bench, monkeypatch):
    for kernel in bench.KERNEL_SOURCES:
        assert bench.sources_digest(kernel) == bench.sources_digest(kernel)  # deterministic
        assert len(bench.sources_digest(kernel)) == 16
    kernel = next(iter(bench.NCU_TRAFFIC))
    digest, nbytes, what = bench.NCU_TRAFFIC[kernel]
    monkeypatch.setitem(bench.NCU_TRAFFIC, kernel, (bench.sources_digest(kernel), nbytes, what))
    got, note = bench.recorded_traffic(kernel)
    assert got == nbytes and "not measured in this run" in note
    monkeypatch.setitem(bench.NCU_TRAFFIC, kernel, ("0" * 16, nbytes, what))
    got, note = bench.recorded_traffic(kernel)
    assert got is None and "changed" in note
    assert bench.recorded_traffic("no_such_kernel")[0] is None


def test_roofline_byte_counts(bench):
    import workload as W
    s = W.QWEN3_0_6B
    # bf16 linears + tied head: the Qwen3-0.6B figure of 1 191 968 768 bytes per token
    assert bench.weight_bytes(s) == 1191968768
    # K and V, f32, all layers and KV heads, keys 0..p
    assert bench.kv_bytes(s, 0) == s.n_layers * 2 * s.n_kv_heads * s.head_dim * 4
    assert bench.kv_bytes(s, 131) == 132 * bench.kv_bytes(s, 0)
