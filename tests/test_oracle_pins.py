"""Pins for the oracle: each checks it against something other than itself.

Sources: closed forms, hand-derived golden fixtures under tests/golden/ (each
cites the page it comes from), brute force on tiny inputs written as plain
Python loops, invariants the mathematics fixes, and special cases with known
answers. Each pin is chosen so that a plausible slip (a dropped term, eps
outside the root, a transposed weight, a wrong RoPE pairing, the wrong GQA
group, a missing causal mask, a shifted nibble) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

from oracle import qwen_ref as R
import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ bf16 widening
def test_widen_bf16_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3DCD, 0x0000, 0x8000, 0x7F80, 0x4049], np.uint16)
    got = R.widen_bf16(bits)
    want = [1.0, -2.0, 0.10009765625, 0.0, -0.0, math.inf, 3.140625]
    assert list(got) == want
    assert math.copysign(1.0, got[4]) == -1.0


# ------------------------------------------------------------------ RMSNorm
def test_rmsnorm_hand_example():
    # x = [3, 4]: mean square 12.5, root 3.5355339..., eps = 0
    y = R.rmsnorm(np.array([[3.0, 4.0]], np.float32), np.ones(2, np.float32), 0.0)
    np.testing.assert_allclose(y[0], [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-7)


def test_rmsnorm_unit_rms_closed_form():
    # RMS of x / sqrt(ms + eps) is sqrt(ms / (ms + eps)); a large eps makes the
    # eps-inside-the-root reading visible (eps outside, or sum instead of mean, fail).
    x = _rng(1).standard_normal((5, 64)).astype(np.float32) * 0.3
    eps = 0.05
    y = R.rmsnorm(x, np.ones(64, np.float32), eps).astype(np.float64)
    ms = np.mean(x.astype(np.float64) ** 2, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), np.sqrt(ms / (ms + eps)),
                               rtol=1e-6)


def test_rmsnorm_gain_multiplies_and_rows_independent():
    x = _rng(2).standard_normal((3, 16)).astype(np.float32)
    g = np.full(16, 2.0, np.float32)
    y1 = R.rmsnorm(x, np.ones(16, np.float32), 1e-6)
    y2 = R.rmsnorm(x, g, 1e-6)
    np.testing.assert_allclose(y2, 2 * y1, rtol=1e-7)      # a (1 + g) reading gives 3x
    x2 = x.copy()
    x2[1] *= 10.0                                            # scaling one row changes no row
    np.testing.assert_allclose(R.rmsnorm(x2, np.ones(16, np.float32), 0.0),
                               R.rmsnorm(x, np.ones(16, np.float32), 0.0), rtol=1e-6)


# ------------------------------------------------------------------ linear
def test_linear_brute_force_out_in_layout():
    rng = _rng(3)
    w = rng.standard_normal((3, 5)).astype(np.float32)      # [out, in], out != in
    x = rng.standard_normal((2, 5)).astype(np.float32)
    b = rng.standard_normal(3).astype(np.float32)
    y = R.linear(x, w.astype(np.float64), b)
    for t in range(2):
        for o in range(3):
            s = sum(float(x[t, i]) * float(w[o, i]) for i in range(5)) + float(b[o])
            assert abs(y[t, o] - s) <= 1e-6 * (1 + abs(s))


# ------------------------------------------------------------------ RoPE
def test_rope_hand_example_hd4():
    # hd = 4, theta = 1e6: inv_freq = [1, 1e6^(-1/2) = 1e-3]; position 1 turns
    # pair (x0, x2) by 1 rad and pair (x1, x3) by 1e-3 rad.
    cos, sin = R.rope_cos_sin([1], 4, 1e6)
    y = R.apply_rope(np.array([[[1.0, 2.0, 3.0, 4.0]]], np.float32), cos, sin)[0, 0]
    c1, s1, c2, s2 = math.cos(1), math.sin(1), math.cos(1e-3), math.sin(1e-3)
    want = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + 1 * s1, 4 * c2 + 2 * s2]
    np.testing.assert_allclose(y, want, rtol=1e-6)


def test_rope_equals_complex_rotation():
    # Independent formulation: z_j = x_j + i x_{j+hd/2}, rotated z_j * e^{i p theta^(-2j/hd)}.
    hd, theta = 64, 1e6
    rng = _rng(4)
    x = rng.standard_normal((7, 3, hd)).astype(np.float32)
    pos = [0, 1, 5, 100, 2047, 8192, 40000]
    cos, sin = R.rope_cos_sin(pos, hd, theta)
    y = R.apply_rope(x, cos, sin).astype(np.float64)
    z = x[..., : hd // 2].astype(np.float64) + 1j * x[..., hd // 2:].astype(np.float64)
    freq = np.array([theta ** (-2.0 * j / hd) for j in range(hd // 2)])
    rot = np.exp(1j * np.array(pos, np.float64)[:, None] * freq[None, :])[:, None, :]
    zz = z * rot
    np.testing.assert_allclose(y[..., : hd // 2], zz.real, atol=2e-6)
    np.testing.assert_allclose(y[..., hd // 2:], zz.imag, atol=2e-6)


def test_rope_norm_relative_position_identity():
    hd = 128
    rng = _rng(5)
    q = rng.standard_normal((1, 1, hd)).astype(np.float32)
    k = rng.standard_normal((1, 1, hd)).astype(np.float32)

    def rot(v, p):
        c, s = R.rope_cos_sin([p], hd, 1e6)
        return R.apply_rope(v, c, s)[0, 0].astype(np.float64)

    # p = 0 is the identity; pairwise norms are preserved
    np.testing.assert_array_equal(rot(q, 0), q[0, 0])
    r = rot(q, 77)
    half = hd // 2
    np.testing.assert_allclose(r[:half] ** 2 + r[half:] ** 2,
                               q[0, 0, :half].astype(np.float64) ** 2
                               + q[0, 0, half:].astype(np.float64) ** 2, rtol=1e-5)
    # <R_m q, R_n k> depends only on m - n
    d1 = rot(q, 10) @ rot(k, 3)
    d2 = rot(q, 1010) @ rot(k, 1003)
    assert abs(d1 - d2) < 2e-4 * (1 + abs(d1))


# ------------------------------------------------------------------ SiLU
def test_silu_closed_forms():
    z = np.array([-20.0, -1.0, 0.0, 1.0, 3.0, 20.0], np.float32)
    one = np.ones_like(z)
    s = R.silu_mul(z, one).astype(np.float64)
    assert s[2] == 0.0
    assert abs(s[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-7
    # silu(z) - silu(-z) = z   (z sigma(z) + z sigma(-z) = z)
    np.testing.assert_allclose(s - R.silu_mul(-z, one).astype(np.float64), z, atol=1e-5)
    np.testing.assert_allclose(R.silu_mul(z, 2 * one), 2 * s, rtol=1e-7)   # up multiplies


# ------------------------------------------------------------------ attention
def _attn_brute(q, qpos, k, v, kpos):
    """Plain loops: one query row, one head, one key at a time."""
    Tq, nq, hd = q.shape
    nkv = k.shape[0]
    out = np.zeros((Tq, nq, hd))
    for t in range(Tq):
        for h in range(nq):
            g = h // (nq // nkv)
            keys = [j for j in range(k.shape[1]) if kpos[j] <= qpos[t]]
            sc = [sum(float(q[t, h, d]) * float(k[g, j, d]) for d in range(hd)) / math.sqrt(hd)
                  for j in keys]
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            tot = sum(e)
            for d in range(hd):
                out[t, h, d] = sum(e[i] * float(v[g, j, d]) for i, j in enumerate(keys)) / tot
    return out


def test_attention_brute_force_gqa_causal():
    rng = _rng(6)
    q = rng.standard_normal((4, 4, 8)).astype(np.float32)
    k = rng.standard_normal((2, 4, 8)).astype(np.float32)
    v = rng.standard_normal((2, 4, 8)).astype(np.float32)
    pos = np.arange(4)
    got = R.causal_gqa_attention(q, pos, k, v, pos)
    np.testing.assert_allclose(got, _attn_brute(q, pos, k, v, pos), atol=1e-6)


def test_attention_special_cases():
    rng = _rng(7)
    q = rng.standard_normal((1, 2, 16)).astype(np.float32)
    k1 = rng.standard_normal((1, 1, 16)).astype(np.float32)
    v1 = rng.standard_normal((1, 1, 16)).astype(np.float32)
    # one visible key returns its value row
    np.testing.assert_allclose(R.causal_gqa_attention(q, [0], k1, v1, [0])[0, 0], v1[0, 0],
                               rtol=1e-7)
    # identical keys return the mean of the values
    kk = np.repeat(k1, 5, axis=1)
    vv = rng.standard_normal((1, 5, 16)).astype(np.float32)
    np.testing.assert_allclose(R.causal_gqa_attention(q, [9], kk, vv, np.arange(5))[0, 1],
                               vv[0].astype(np.float64).mean(0), atol=1e-6)
    # future keys are invisible
    kf = rng.standard_normal((1, 6, 16)).astype(np.float32)
    vf = rng.standard_normal((1, 6, 16)).astype(np.float32)
    a = R.causal_gqa_attention(q, [2], kf, vf, np.arange(6))
    kf2, vf2 = kf.copy(), vf.copy()
    kf2[:, 3:] = 50.0
    vf2[:, 3:] = -7.0
    np.testing.assert_array_equal(a, R.causal_gqa_attention(q, [2], kf2, vf2, np.arange(6)))


def test_gqa_equals_mha_with_repeated_heads():
    rng = _rng(8)
    q = rng.standard_normal((3, 8, 16)).astype(np.float32)
    k = rng.standard_normal((2, 3, 16)).astype(np.float32)
    v = rng.standard_normal((2, 3, 16)).astype(np.float32)
    pos = np.arange(3)
    gqa = R.causal_gqa_attention(q, pos, k, v, pos)
    mha = R.causal_gqa_attention(q, pos, np.repeat(k, 4, axis=0), np.repeat(v, 4, axis=0), pos)
    np.testing.assert_array_equal(gqa, mha)


# ------------------------------------------------------------------ argmax
def test_argmax_ties_and_nan():
    assert R.greedy_argmax(np.array([1.0, 3.0, 3.0, 2.0], np.float32)) == 1
    with pytest.raises(FloatingPointError):
        R.greedy_argmax(np.array([1.0, np.nan], np.float32))


# ------------------------------------------------------------------ sampling
# Hand example: probabilities 0.1, 0.2, 0.3, 0.4 on ids 0..3 (logits log p, T = 1).
# Candidate order 3, 2, 1, 0 with cumulative probability 0.4, 0.7, 0.9, 1.0.
_P4 = np.log(np.array([0.1, 0.2, 0.3, 0.4], np.float32))


@pytest.mark.parametrize("k,p,u,want", [
    (4, 1.0, 0.10, 3), (4, 1.0, 0.50, 2), (4, 1.0, 0.80, 1), (4, 1.0, 0.95, 0),
    (4, 0.6, 0.50, 3), (4, 0.6, 0.60, 2),   # nucleus {3, 2}: cumulative 4/7, 1 of 0.7
    (4, 0.35, 0.99, 3),                     # nucleus {3} alone (0.4 reaches 0.35)
    (2, 1.0, 0.50, 3), (2, 1.0, 0.60, 2),   # top-2 renormalised: 4/7, 3/7
    (9, 1.0, 0.95, 0),                      # top_k above the row is the whole row
])
def test_sampling_hand_example(k, p, u, want):
    got, margin = R.sample_logits(_P4, 1.0, k, p, u)
    assert got == want and margin > 1e-3


def test_sampling_greedy_cases_and_errors():
    assert R.sample_logits(_P4, 0.0, 4, 1.0, 0.9)[0] == 3     # temp = 0 is greedy
    assert R.sample_logits(_P4, -1.0, 4, 1.0, 0.9)[0] == 3
    assert R.sample_logits(_P4, 1.0, 1, 1.0, 0.9)[0] == 3     # top_k = 1 is greedy
    tie = np.array([0.5, 2.0, 2.0, 1.0], np.float32)
    assert R.sample_logits(tie, 0.0, 4, 1.0, 0.0)[0] == R.greedy_argmax(tie) == 1
    with pytest.raises(FloatingPointError):
        R.sample_logits(np.array([1.0, np.nan], np.float32), 1.0, 2, 1.0, 0.5)
    with pytest.raises(FloatingPointError):
        R.sample_logits(np.full(3, -np.inf, np.float32), 1.0, 2, 1.0, 0.5)


def test_sampling_equal_logits_split_u_by_index():
    # four equal logits: each candidate holds a quarter of [0, 1), in index order
    x = np.full(4, 1.5, np.float32)
    for u, want in ((0.0, 0), (0.24, 0), (0.26, 1), (0.6, 2), (0.99, 3)):
        assert R.sample_logits(x, 0.7, 4, 1.0, u)[0] == want


def test_sampling_frequencies_are_the_truncated_softmax():
    # inverse-CDF property: over a uniform grid of u the frequencies are the
    # softmax at temperature T restricted to the nucleus of the top k, renormalised
    rng = _rng(5)
    x = rng.standard_normal(40).astype(np.float32)
    T, k, p, N = 0.8, 12, 0.9, 20000
    counts = np.zeros(40)
    for j in range(N):
        counts[R.sample_logits(x, T, k, p, (j + 0.5) / N)[0]] += 1
    idx = np.argsort(-x.astype(np.float64), kind="stable")[:k]
    e = np.exp((x[idx].astype(np.float64) - x[idx[0]]) / T)
    c = np.cumsum(e) / e.sum()
    n = int(np.argmax(c >= np.float32(p))) + 1
    want = np.zeros(40)
    want[idx[:n]] = e[:n] / e[:n].sum()
    assert np.abs(counts / N - want).max() <= 2.0 / N
    assert counts[np.setdiff1d(np.arange(40), idx[:n])].sum() == 0


def test_sampling_temperature_scales_the_logits():
    rng = _rng(6)
    x = rng.standard_normal(64).astype(np.float32)
    for u in np.linspace(0.01, 0.99, 25):
        a = R.sample_logits(x, 2.0, 16, 0.95, u)
        b = R.sample_logits((x / 2).astype(np.float32), 1.0, 16, 0.95, u)
        if min(a[1], b[1]) > 1e-6:
            assert a[0] == b[0]


# ------------------------------------------------------------------ int4 g128
def _read_int4_golden():
    vals, deq = {}, {}
    with open(os.path.join(GOLDEN, "int4_g128_example.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            t = line.split()
            if t[0] == "w":
                vals[int(t[1])] = float(t[2])
            elif t[0] == "scale_bits":
                scales = [int(x, 16) for x in t[1:]]
            elif t[0] == "bytes":
                head = [int(x, 16) for x in t[1:]]
            elif t[0] == "fill_byte":
                fill = int(t[1], 16)
            elif t[0] == "dequant":
                deq[int(t[1])] = float(t[2])
    return vals, scales, head, fill, deq


def test_int4_golden_hand_example():
    vals, scales, head, fill, deq = _read_int4_golden()
    w = np.zeros((1, 256), np.float32)
    for i, x in vals.items():
        w[0, i] = x
    packed, sb = R.int4_quantize(w)
    assert list(sb[0]) == scales
    want = head + [fill] * (128 - len(head))
    assert list(packed[0]) == want
    d = R.int4_dequantize(packed, sb)
    for i, x in deq.items():
        assert d[0, i] == np.float32(x)
    assert np.all(d[0, 10:] == 0)


def test_int4_round_trip_bounds_and_exact_dequant():
    w = _rng(9).standard_normal((6, 384)).astype(np.float32) * 0.02
    packed, sb = R.int4_quantize(w)
    d = R.int4_dequantize(packed, sb)
    s = R.widen_bf16(sb)
    err = np.abs(w - d).reshape(6, 3, 128)
    # s is within a bf16 rounding of max|w|/7, so |w - w'| <= s/2 except a hair at the clamp
    assert np.all(err <= s[:, :, None] * (0.5 + 1e-3) + 1e-12)
    # the dequantised value is exactly a small integer times a bf16 scale
    q = (d.reshape(6, 3, 128) / s[:, :, None])
    np.testing.assert_array_equal(q, np.rint(q))
    assert np.abs(q).max() <= 7
    # unpack by hand: element 2i low nibble, 2i+1 high nibble
    lo = int(packed[0, 0] & 15) - 8
    hi = int(packed[0, 0] >> 4) - 8
    assert d[0, 0] == np.float32(lo) * s[0, 0] and d[0, 1] == np.float32(hi) * s[0, 0]


# ------------------------------------------------------------------ KV size (page table)
def test_kv_cache_size_matches_page_table():
    rows = {}
    with open(os.path.join(GOLDEN, "kv_cache_sizes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, b = line.split()
                rows[a] = b
    cfg = R.Config.from_shape(W.QWEN25_3B_INT4)
    assert R.kv_cache_bytes(cfg, 1) == int(rows.pop("per_token_bytes"))
    for ctx, gb in rows.items():
        assert round(R.kv_cache_bytes(cfg, int(ctx)) / 1024 / 1e6, 1) == float(gb)


# ------------------------------------------------------------------ whole-model pins
def _tiny(seed=0, **kw):
    shape = W.TINY.replace(**kw) if kw else W.TINY
    wl = W.Workload("t", shape, seed=seed, prompt_len=6, max_ctx=32)
    return W.draw(wl, drawn_gains=True), wl


def test_blocks_as_identity_give_closed_form_logits():
    # With W_o = 0 and W_down = 0 every block adds nothing to the bus, so the final
    # hidden state is the embedding row and logits[i] = E[i] . rms(E[tok]) g_f.
    d, wl = _tiny(seed=11)
    for l in range(wl.shape.n_layers):
        d.weights[f"layers.{l}.o"][:] = 0
        d.weights[f"layers.{l}.down"][:] = 0
    m = R.build_oracle(d)
    ids = [5, 17, 4000, 3]
    cp = m.prefill(ids)
    E = R.widen_bf16(d.weights["embed"]).astype(np.float64)
    g = R.widen_bf16(d.weights["final_norm"]).astype(np.float64)
    np.testing.assert_array_equal(cp["block0"], E[ids].astype(np.float32))
    x = E[ids[-1]]
    h = g * x / math.sqrt(np.mean(x * x) + wl.shape.eps)
    np.testing.assert_allclose(cp["logits"], E @ h, rtol=1e-5, atol=1e-6)


def test_tied_head_is_a_dot_with_the_embedding_rows():
    d, wl = _tiny(seed=12)
    m = R.build_oracle(d)
    cp = m.prefill([1, 2, 3])
    E = R.widen_bf16(d.weights["embed"]).astype(np.float64)
    h = cp["final_norm"][-1].astype(np.float64)
    for i in [0, 7, 1234, 4095]:
        assert abs(cp["logits"][i] - float(E[i] @ h)) <= 1e-6 * (1 + abs(E[i] @ h))


def test_cached_decode_equals_prefill_last_row_and_kv():
    d, wl = _tiny(seed=13)
    ids = list(W.random_ids(wl.shape.vocab, 9, seed=5))
    a = R.build_oracle(d)
    ref = a.prefill(ids)
    b = R.build_oracle(d)
    for t in ids:
        cp = b.decode_step(t)
    np.testing.assert_allclose(cp["logits"], ref["logits"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(cp["final_norm"][0], ref["final_norm"][-1], rtol=1e-5, atol=1e-6)
    for l in range(wl.shape.n_layers):
        np.testing.assert_allclose(b.k_cache[l][:, :9], a.k_cache[l][:, :9], rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(b.v_cache[l][:, :9], a.v_cache[l][:, :9], rtol=1e-5, atol=1e-6)
    assert a.pos == b.pos == 9


def test_gqa_model_equals_mha_model_with_duplicated_kv_weights():
    d, wl = _tiny(seed=14)
    s = wl.shape
    group = s.n_q_heads // s.n_kv_heads
    mha_w = dict(d.weights)
    for l in range(s.n_layers):
        for nm in ("k", "v"):
            w = d.weights[f"layers.{l}.{nm}"].reshape(s.n_kv_heads, s.head_dim, s.hidden)
            mha_w[f"layers.{l}.{nm}"] = np.repeat(w, group, axis=0).reshape(-1, s.hidden)
    mha_shape = s.replace(n_kv_heads=s.n_q_heads)
    ids = [9, 8, 7, 6, 5]
    a = R.OracleModel(R.Config.from_shape(s), d.weights, 16).prefill(ids)
    b = R.OracleModel(R.Config.from_shape(mha_shape), mha_w, 16).prefill(ids)
    np.testing.assert_allclose(a["logits"], b["logits"], rtol=1e-6, atol=1e-7)


def test_shapes_match_fs_m2_page():
    spec = {}
    with open(os.path.join(GOLDEN, "fs_m2_shapes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                t = line.split()
                spec[t[0]] = [int(x) for x in t[1:]]
    # depth does not change any checkpoint shape: one layer of the Qwen3-0.6B shape
    shape = W.QWEN3_0_6B.replace(n_layers=1)
    d = W.draw(W.Workload("s", shape, seed=1, prompt_len=spec["prompt_len"][0], max_ctx=8))
    cp = R.build_oracle(d, cache_f64=False).prefill(d.prompt)
    for k in ("embedding", "block0", "final_norm", "logits"):
        assert list(cp[k].shape) == spec[k]


def test_lora_zero_b_is_base_and_lora_equals_merged_weights():
    shape = W.TINY.replace(qk_norm=False, qkv_bias=True, tie_word_embeddings=False)
    wl = W.Workload("l", shape, seed=15, max_ctx=16, lora=W.LoraShape(4, 8.0))
    d = W.draw(wl)
    ids = [3, 1, 4, 1, 5]
    base = R.build_oracle(d).prefill(ids)
    lora = {k: v for k, v in d.weights.items() if k.startswith("lora.")}
    zero_b = {k: (np.zeros_like(v) if k.endswith("_b") else v) for k, v in lora.items()}
    m0 = R.build_oracle(d)
    m0.set_lora(zero_b, 8.0)
    np.testing.assert_array_equal(m0.prefill(ids)["logits"], base["logits"])
    on = R.build_oracle(d, lora_on=True).prefill(ids)
    assert np.abs(on["logits"] - base["logits"]).max() > 1e-4      # the branch does something
    merged = R.build_oracle(d)
    for l in range(shape.n_layers):
        for nm in ("q", "v"):
            a = R.widen_bf16(lora[f"lora.{l}.{nm}_a"]).astype(np.float64)
            b = R.widen_bf16(lora[f"lora.{l}.{nm}_b"]).astype(np.float64)
            w = merged.w[f"layers.{l}.{nm}"].astype(np.float64) + (8.0 / 4) * (b @ a)
            merged._w64[f"layers.{l}.{nm}"] = w
    np.testing.assert_allclose(merged.prefill(ids)["logits"], on["logits"], rtol=1e-5, atol=1e-6)
    # clearing restores the base result bit for bit
    m1 = R.build_oracle(d, lora_on=True)
    m1.set_lora(None)
    np.testing.assert_array_equal(m1.prefill(ids)["logits"], base["logits"])


def test_qkv_bias_enters_before_rope_and_untied_head():
    shape = W.TINY.replace(qk_norm=False, qkv_bias=True, tie_word_embeddings=False)
    d = W.draw(W.Workload("b", shape, seed=16, max_ctx=8))
    m = R.build_oracle(d)
    xn = np.zeros((1, shape.hidden), np.float32)          # zero input: projections = biases
    q, k, v = m._qkv_heads(0, xn, np.array([0]))
    np.testing.assert_array_equal(q.reshape(-1), R.widen_bf16(d.weights["layers.0.q_bias"]))
    np.testing.assert_array_equal(v.reshape(-1), R.widen_bf16(d.weights["layers.0.v_bias"]))
    q3, _, _ = m._qkv_heads(0, xn, np.array([3]))         # at p = 3 the bias is rotated
    assert np.abs(q3 - q).max() > 1e-4
    cp = m.prefill([1, 2])
    L = R.widen_bf16(d.weights["lm_head"]).astype(np.float64)
    np.testing.assert_allclose(cp["logits"], L @ cp["final_norm"][-1].astype(np.float64),
                               rtol=1e-5, atol=1e-6)


def test_int4_model_uses_exact_dequantised_weights():
    shape = W.TINY.replace(weight_format="int4_g128", tie_word_embeddings=False,
                           int4_lm_head=True, qk_norm=False, qkv_bias=True)
    d = W.draw(W.Workload("q", shape, seed=17, max_ctx=8))
    m = R.build_oracle(d)
    for name in ("layers.0.q", "layers.1.down", "lm_head"):
        p, s = R.int4_quantize(d.weights[name])
        np.testing.assert_array_equal(m.w[name], R.int4_dequantize(p, s))
    assert "embed" not in m.int4


# ------------------------------------------------------------------ block wiring (hand-set weights)
# The "Failed Star / fs, M2" page, "One prefill, all shapes visible", gives the block as
# two sublayers on the residual bus: attention (read through the attention-input norm)
# then the SwiGLU MLP (read through the post-attention norm), each added back; the
# "SuperKittens PR #7" page names the fused kernel SiLU(gate) * up. The two cases below
# set every weight by hand to small bf16-exact values so each intermediate is a number
# derived in the comments; swapping gate/up, the two sublayer gains, or the q/k norm
# gains moves the result far outside the tolerance.
def _bits(a):
    return W.f32_to_bf16_bits(np.asarray(a, np.float32))


def _hand_model(weights, **kw):
    cfg = R.Config(n_layers=1, hidden=4, n_q_heads=1, n_kv_heads=1, head_dim=2,
                   intermediate=2, vocab=3, eps=0.0, **kw)
    return R.OracleModel(cfg, {k: _bits(v) for k, v in weights.items()}, max_ctx=4)


def test_block_wiring_gate_up_and_sublayer_gains_hand_case():
    E = [[2, 0, 0, 0], [0, 0, 0, 1], [1, 1, 1, 1]]
    m = _hand_model({
        "embed": E,
        "layers.0.attn_norm": [0.25, 1, 1, 1],
        "layers.0.q": np.zeros((2, 4)), "layers.0.k": np.zeros((2, 4)),
        "layers.0.v": [[2, 0, 0, 0], [0, 0, 0, 0]],
        "layers.0.o": [[0, 0], [2, 0], [2, 0], [2, 0]],
        "layers.0.mlp_norm": [0.5, 0.25, 1, 2],
        "layers.0.gate": [[4, 0, 0, 0], [0, 0, 0, 0]],
        "layers.0.up": [[0, 12, 0, 0], [0, 0, 0, 0]],
        "layers.0.down": [[0, 0], [0, 0], [0, 0], [1, 0]],
        "final_norm": [1, 1, 1, 1],
    }, qk_norm=False)
    cp = m.decode_step(0)
    # x = E[0] = (2,0,0,0): mean square 1, so the attention input is x * attn_norm = (0.5,0,0,0);
    # v = (1, 0); one visible key, so the attention output is v; o_proj adds (0,2,2,2).
    # x1 = (2,2,2,2): mean square 4, root 2, so the MLP input is mlp_norm = (0.5,0.25,1,2);
    # gate = 4 * 0.5 = 2, up = 12 * 0.25 = 3; m0 = silu(2) * 3 = 6 / (1 + e^-2); down adds m0 to x[3].
    m0 = 6.0 / (1.0 + math.exp(-2.0))
    x2 = np.array([2.0, 2.0, 2.0, 2.0 + m0])
    np.testing.assert_allclose(cp["block0"][0], x2, rtol=1e-6)
    h = x2 / math.sqrt(np.mean(x2 * x2))
    np.testing.assert_allclose(cp["final_norm"][0], h, rtol=1e-6)
    np.testing.assert_allclose(cp["logits"], np.array(E, np.float64) @ h, rtol=1e-6, atol=1e-7)
    # wrong wirings land far away: silu(3) * 2 for a swapped gate/up; with the two gains
    # swapped the attention input is (1,0,0,0), o_proj adds (0,4,4,4) and x1 = (2,4,4,4)
    assert abs(6.0 / (1.0 + math.exp(-3.0)) - m0) > 0.4
    assert abs(cp["block0"][0][1] - 4.0) > 1.0


def test_block_wiring_qk_norm_gains_rope_and_causal_mask_hand_case():
    E = [[2, 0, 0, 0], [0, 2, 0, 0], [1, 1, 1, 1]]
    m = _hand_model({
        "embed": E,
        "layers.0.attn_norm": [1, 1, 1, 1],
        "layers.0.q": [[0.5, 0.5, 0, 0], [0, 0.5, 0, 0]],    # q(id 0) = (1, 0), q(id 1) = (1, 1)
        "layers.0.k": [[0.5, 0.5, 0, 0], [0, 0.5, 0, 0]],    # k(id 0) = (1, 0), k(id 1) = (1, 1)
        "layers.0.v": [[0.5, 0, 0, 0], [0, 0.5, 0, 0]],      # v(id 0) = (1, 0), v(id 1) = (0, 1)
        "layers.0.q_norm": [2, 1], "layers.0.k_norm": [1, 4],
        "layers.0.o": [[0, 0], [0, 0], [1, 0], [0, 1]],
        "layers.0.mlp_norm": [1, 1, 1, 1],
        "layers.0.gate": np.zeros((2, 4)), "layers.0.up": np.zeros((2, 4)),
        "layers.0.down": np.zeros((4, 2)),
        "final_norm": [1, 1, 1, 1],
    }, qk_norm=True, rope_theta=1e6)
    cp = m.prefill([0, 1])
    # Row 1 (position 1). QK-norm over head_dim 2 with eps 0: q = (1,1) has RMS 1 -> times (2,1) = (2, 1);
    # k0 = (1,0) has RMS 1/sqrt(2) -> (sqrt2, 0); k1 = (1,1) -> (1, 4). head_dim 2 has one
    # rotary pair with inv_freq 1, so position 1 turns by 1 rad and position 0 not at all:
    #   s0 = R(1)(2,1) . (sqrt2, 0) / sqrt2 = 2 cos1 - sin1
    #   s1 = R(1)(2,1) . R(1)(1,4) / sqrt2 = (2 + 4) / sqrt2          (rotation-invariant)
    # The output is p0 v0 + p1 v1 = (p0, p1); o_proj puts it on x[2], x[3].
    c, s = math.cos(1.0), math.sin(1.0)
    s0, s1 = 2 * c - s, 6 / math.sqrt(2)
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    x1 = np.array([0.0, 2.0, p0, 1.0 - p0])
    np.testing.assert_allclose(cp["block0"][1], x1, rtol=1e-6, atol=1e-7)
    # row 0 sees only its own key: output v0 = (1, 0)
    np.testing.assert_allclose(cp["block0"][0], [2.0, 0.0, 1.0, 0.0], rtol=1e-6, atol=1e-7)
    h = x1 / math.sqrt(np.mean(x1 * x1))
    np.testing.assert_allclose(cp["logits"], np.array(E, np.float64) @ h, rtol=1e-6, atol=1e-7)
    # swapped q/k norm gains would give s0 = 2 cos1 - 8 sin1: p0 moves far
    p0_swapped = 1.0 / (1.0 + math.exp(s1 - (2 * c - 8 * s)))
    assert abs(p0_swapped - p0) > 0.01


# ------------------------------------------------------------------ Q8_0 (block-32 int8)
def test_q8_0_golden_hand_example():
    vals, q_want, deq, scales = {}, {}, {}, []
    with open(os.path.join(GOLDEN, "q8_0_block_example.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            t = line.split()
            if t[0] == "w":
                vals[int(t[1])] = float(t[2])
            elif t[0] == "q":
                q_want[int(t[1])] = int(t[2])
            elif t[0] == "dequant":
                deq[int(t[1])] = float(t[2])
            elif t[0] == "scale_bits":
                scales = [int(x, 16) for x in t[1:]]
    w = np.zeros((1, 96), np.float32)
    for i, x in vals.items():
        w[0, i] = x
    q, sb = R.q8_0_quantize(w)
    assert list(sb[0]) == scales
    want = np.zeros(96, np.int8)
    for i, x in q_want.items():
        want[i] = x
    np.testing.assert_array_equal(q[0], want)
    d = R.q8_0_dequantize(q, sb)
    for i, x in deq.items():
        assert d[0, i] == np.float32(x)
    assert d[0, 0] == np.float32(0.9921875) and d[0, 2] == np.float32(2 / 128)


def test_q8_0_round_trip_bounds_and_exact_dequant():
    w = _rng(19).standard_normal((5, 256)).astype(np.float32) * 0.02
    q, sb = R.q8_0_quantize(w)
    d = R.q8_0_dequantize(q, sb)
    s = sb.view(np.float16).astype(np.float64)
    err = np.abs(w.astype(np.float64) - d).reshape(5, 8, 32)
    # s is within an fp16 rounding of max|w|/127, so |w - w'| <= s/2 except a hair at the clamp
    assert np.all(err <= s[:, :, None] * (0.5 + 2e-3) + 1e-12)
    assert np.abs(q.astype(np.int32)).max() == 127          # the block maximum reaches 127
    ratio = d.reshape(5, 8, 32) / s[:, :, None]
    np.testing.assert_array_equal(ratio, np.rint(ratio))      # integer times the scale
    # scaling a block by a power of two scales s and keeps q
    q2, sb2 = R.q8_0_quantize(w * np.float32(4.0))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(sb2.view(np.float16).astype(np.float64), 4 * s)


def test_q8_0_model_uses_exact_dequantised_weights_and_a_q8_tied_head():
    shape = W.TINY.replace(weight_format="q8_0")
    d = W.draw(W.Workload("q8", shape, seed=23, max_ctx=8))
    m = R.build_oracle(d)
    for name in ("layers.0.q", "layers.1.down", "layers.0.gate"):
        q, s = R.q8_0_quantize(d.weights[name])
        np.testing.assert_array_equal(m.w[name], R.q8_0_dequantize(q, s))
    # the gather keeps the bf16 rows; the tied head dots against Q8_0(embed)
    E = R.widen_bf16(d.weights["embed"])
    np.testing.assert_array_equal(m.w["embed"], E)
    q, s = R.q8_0_quantize(E)
    head = R.q8_0_dequantize(q, s).astype(np.float64)
    cp = m.prefill([7, 8, 9])
    np.testing.assert_allclose(cp["logits"], head @ cp["final_norm"][-1].astype(np.float64),
                               rtol=1e-5, atol=1e-6)
    assert np.abs(head - E).max() > 0                        # the head differs from the table


# ------------------------------------------------------------------ bf16 KV cache
def test_round_bf16_hand_values():
    # bf16 keeps 7 fraction bits: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 (ties to
    # even: 1); 1 + 3 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6 (even: 1 + 2^-6);
    # 1 + 2^-8 + 2^-20 is just above halfway (rounds up); bf16 values are fixed points
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -2.5, 0.0, 3.140625],
                 np.float32)
    want = [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -2.5, 0.0, 3.140625]
    assert list(R.round_bf16(x)) == want


def test_bf16_kv_cache_stores_rounded_rows_and_decode_equals_prefill():
    d, wl = _tiny(seed=27)
    cfg = R.Config.from_shape(wl.shape.replace(kv_format="bf16"))
    ids = [11, 12, 13, 14, 15, 16]
    a = R.OracleModel(cfg, d.weights, 16)
    ref = a.prefill(ids)
    b = R.OracleModel(cfg, d.weights, 16)
    for t in ids:
        cp = b.decode_step(t)
    np.testing.assert_allclose(cp["logits"], ref["logits"], rtol=1e-5, atol=1e-6)
    for l in range(wl.shape.n_layers):
        k = a.k_cache[l][:, :6]
        np.testing.assert_array_equal(R.round_bf16(k), k)          # bf16 values stored
        np.testing.assert_allclose(b.k_cache[l][:, :6], k, rtol=1e-5, atol=1e-6)
    # the rounding is the only difference from the f32 cache, and it is visible; layer
    # 0's keys see the same input either way, so they are the f32 keys rounded
    f32m = R.build_oracle(d)
    f32 = f32m.prefill(ids)
    diff = np.abs(f32["logits"] - ref["logits"]).max()
    assert 0 < diff < 1e-2
    np.testing.assert_array_equal(a.k_cache[0][:, :6], R.round_bf16(f32m.k_cache[0][:, :6]))
    np.testing.assert_array_equal(a.v_cache[0][:, :6], R.round_bf16(f32m.v_cache[0][:, :6]))
