"""Benchmark: batch-1 greedy decode of the Qwen3-0.6B-shape model on one GB300.

One step = the "qwen3_0.6b_decode" workload's generation: 128 greedy decode
tokens (positions 5..132) after a 5-id prompt, each token one pass of the whole
decode path (embedding, 28 blocks, final norm, LM head, argmax) as one CUDA
graph replay. Weights (1.19 GB read per token) are larger than L2, so no flush
is needed between steps. `value` is decode tokens/s with weights and prompt KV
already in HBM; `e2e` is the same through qw_decode_step with the token coming
from the host and the greedy id read back every token.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun, every rank runs an independent replica on its own GPU (the
path does not shard); the slowest rank's time is used and `value` sums all
ranks' tokens. `--impl reference` times the CPU oracle on this host instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "qwen3_0.6b_decode"
PREFILL_WORKLOAD = "qwen3_0.6b_prefill"
METRIC = "batch-1 decode tok/s (Qwen3-0.6B shape)"


def weight_bytes(s) -> int:
    """Algorithmic weight bytes read per decode token (bf16 linears + LM head)."""
    per_layer = (s.hidden * s.q_dim + 2 * s.hidden * s.kv_dim + s.q_dim * s.hidden
                 + 3 * s.hidden * s.intermediate)
    return 2 * (s.n_layers * per_layer + s.vocab * s.hidden)


def kv_bytes(s, pos: int) -> int:
    """KV bytes read by the token at 0-based position pos (keys 0..pos, f32 K and V)."""
    return s.n_layers * 2 * s.n_kv_heads * s.head_dim * 4 * (pos + 1)


def step_bytes(s, p0: int, n: int) -> int:
    return n * weight_bytes(s) + sum(kv_bytes(s, p) for p in range(p0, p0 + n))


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the two
# kernels the JSON line reports, each from one ncu capture of a build, keyed by the
# SHA-256 of the source files that build compiles from. ncu cannot run inside a
# timed bench, so the figure is recorded here; as soon as a listed source changes
# the digest no longer matches and the line reports traffic as null.
KERNEL_SOURCES = {
    "decode_mega": ["decode_mega.cu", "qw_ptx.cuh", "qw_internal.h"],
    "decode_mega_big": ["decode_mega.cu", "decode_mega_big.cu", "qw_ptx.cuh", "qw_internal.h"],
    "lm_head_gemv": ["decode_kernels.cu", "qw_ptx.cuh", "qw_internal.h"],
}
NCU_TRAFFIC = {
    # kernel: (sources digest, bytes per launch, what was captured)
    "decode_mega": ("d7846fd82ef54d55", 1194048256 + 3808512,
                    "qwen3_0.6b_decode token at position 6, decode_mega_kernel<128, 1, 0, 0, false, 0>"),
    "decode_mega_big": ("6a6826f8f9d92b00", 1895046656 + 7786240,
                        "qwen2.5_3b_int4_lora token at position 4098 without the adapter, "
                        "decode_mega_kernel<128, 0, 0, 0, false, 1> (wide-input build)"),
    "lm_head_gemv": ("080190fbaea159fa", 311220992 + 3417856,
                     "qw_lm_head_argmax on the 151936 x 1024 table, gemv_kernel<3, 4, 0>"),
}


def sources_digest(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sequence_decode_step_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """(bytes per launch, note) from the ncu capture of this exact build, or (None, why)."""
    rec = NCU_TRAFFIC.get(kernel)
    if rec is None:
        return None, "no ncu capture recorded for this kernel"
    digest, nbytes, what = rec
    if digest != sources_digest(kernel):
        return None, "the kernel's sources changed since its ncu capture"
    return nbytes, f"ncu capture of this build ({what}), not measured in this run"


def host_cpu() -> dict:
    """CPU model and logical core count of this host."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"cpu_model": model or platform.processor() or platform.machine(),
            "nproc": os.cpu_count()}


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self):
        rows = []
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) >= 9:
                try:
                    rows.append((float(f[1]), float(f[2]), f[5:9]))
                except ValueError:
                    pass
        if not rows:
            return None
        mx = max(r[1] for r in rows)
        loaded = [r for r in rows if r[0] > 0.5 * mx] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows)}


def aggregate(ms_local: float, tokens_local: int, world: int, device: str = "cuda"):
    """Replicas only: every rank times its own independent decode; the job's time is
    the slowest rank's and its throughput is all ranks' tokens over that time.
    Returns (ms_max, tokens_total)."""
    if world <= 1:
        return ms_local, tokens_local
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    n = torch.tensor([tokens_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


# ============================================================================ GPU arm
def run_ours(args, rank: int, world: int, local_rank: int) -> dict:
    import ctypes as C
    import numpy as np
    import torch
    import workload as W
    from sequence_decode_step_gb300 import _binding as B
    from sequence_decode_step_gb300.device_model import DeviceModel

    torch.cuda.set_device(local_rank)
    wl = W.WORKLOADS[WORKLOAD]
    s = wl.shape
    n_tok = wl.decode_steps
    p0 = wl.prompt_len
    d = W.draw(wl)
    L = B.lib()
    # a dedicated stream: the handle queues its graph replays on it and the CUDA
    # events are recorded on it
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    m = DeviceModel(s, d.weights, max_ctx=p0 + n_tok + 8, stream=stream.cuda_stream)
    first = m.prefill(d.prompt)
    path = B.qw_get_decode_path(m.h)  # 0: persistent kernel, 1: multi-kernel graph

    def one_step(timed_events=None):
        B.qw_set_pos(m.h, p0)                      # back to the end of the prompt (syncs)
        if timed_events:
            timed_events[0].record(stream)
        rc = L.qw_decode_step(m.h, first, None, None)
        for _ in range(n_tok - 1):
            rc |= L.qw_decode_step(m.h, -1, None, None)
        if timed_events:
            timed_events[1].record(stream)
        if rc:
            raise RuntimeError(B.last_error(m.h))

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            one_step(pairs[i])
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    ms = sum(a.elapsed_time(b) for a, b in pairs)
    ms_max, tok_total = aggregate(ms, n_tok * args.steps, world)
    if world > 1:
        torch.distributed.barrier()

    # ---- end to end: token from the host, greedy id back to the host, every token
    e2e_ms = 0.0
    for i in range(max(1, args.steps // 2)):
        B.qw_set_pos(m.h, p0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        tok = first
        out = C.c_int32()
        for _ in range(n_tok):
            rc = L.qw_decode_step(m.h, tok, None, C.byref(out))
            if rc:
                raise RuntimeError(B.last_error(m.h))
            tok = out.value
        e2e_ms += (time.perf_counter() - t0) * 1e3
    e2e_steps = max(1, args.steps // 2)

    # ---- dominant single launch: the LM head GEMV (final norm + [V,H] table + argmax),
    # the same kernel the graph runs, timed alone with events on its stream
    lm = lm_head_roofline(L, B, torch, d, s, stream)
    smp = sampling_timing(L, B, torch, s, stream)

    # ---- prefill of T=1024 ids (the prompt path at that length)
    pre = prefill_timing(torch, W, DeviceModel, stream) if args.prefill else None
    m.close()
    extra = {}
    if args.extras:  # the other workloads' lines: long context (f32 / bf16 KV), Q8_0, int4 prefill
        extra["longctx"] = longctx_timing(torch, W, B, DeviceModel, stream)
        extra["q8_0_decode"] = q8_timing(torch, W, B, DeviceModel, stream)
        extra["prefill_int4"] = int4_prefill_timing(torch, W, B, DeviceModel, stream)
        extra["int4_decode"] = int4_decode_timing(torch, W, B, DeviceModel, stream)

    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    bytes_step = step_bytes(s, p0, n_tok)
    sec_tok = ms_max / 1e3 / (n_tok * args.steps)
    if path == 0:
        dominant = {"kernel": "decode_mega_kernel (the whole decode step: one persistent cooperative "
                              "launch per token)",
                    "bound": "hbm", "bytes_per_launch": bytes_step / n_tok,
                    "achieved": bytes_step / n_tok / sec_tok / 1e9, "peak": hbm, "unit": "GB/s",
                    "frac": bytes_step / n_tok / sec_tok / 1e9 / hbm,
                    "traffic": recorded_traffic("decode_mega")[0],
                    "traffic_source": recorded_traffic("decode_mega")[1],
                    "us_per_launch": sec_tok * 1e6,
                    "timing": "CUDA events on the launching stream around the timed steps, "
                              "divided by the launches (one per token)",
                    "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks
                    else "fallback 6800 GB/s"}
    else:
        dominant = lm
    res = {
        "metric": METRIC, "value": tok_total / (ms_max / 1e3), "unit": "tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "prompt_ids": p0, "decode_tokens_per_step": n_tok,
                   "positions": f"{p0}..{p0 + n_tok - 1}", "weights": "bf16 ~N(0,0.02), seed 1",
                   "l2": "inputs larger than L2: 1.19 GB of weights read per token",
                   "parallelism": f"replicas x{world}"},
        "us_per_token": ms_max * 1e3 / (n_tok * args.steps),
        "step_roofline": {"bound": "hbm", "bytes_per_step": bytes_step,
                          "achieved": bytes_step / (ms_max / args.steps / 1e3) / 1e9,
                          "peak": hbm, "unit": "GB/s",
                          "frac": bytes_step / (ms_max / args.steps / 1e3) / 1e9 / hbm,
                          "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks
                          else "fallback 6800 GB/s"},
        "roofline": dominant,
        "lm_head_gemv": lm,
        "sampling": smp,
        "decode_path": "persistent" if path == 0 else "multi-kernel graph",
        "e2e": {"value": n_tok * e2e_steps / (e2e_ms / 1e3), "unit": "tok/s",
                "h2d_bytes_per_step": 4 * n_tok, "d2h_bytes_per_step": 4 * n_tok},
        "gpu_launches": args.steps * n_tok * (1 if path == 0 else 2 + 5 * s.n_layers),
        "wall_s_timed_region": wall,
        "clocks": clk.summary(),
        "prefill": pre,
        **extra,
    }
    return res


def sampling_timing(L, B, torch, s, stream) -> dict:
    """qw_sample over one logits row of the workload's vocabulary (on-device
    temperature / top-k / top-p; the alternative is reading the row back)."""
    T, k, p = 0.7, 50, 0.9
    x = torch.randn(s.vocab, device="cuda") * 3
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    wsb = L.qw_sample_workspace_bytes(s.vocab, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def go(u):
        rc = L.qw_sample(x.data_ptr(), s.vocab, T, k, p, u, tok.data_ptr(), ws.data_ptr(), wsb,
                         stream.cuda_stream)
        if rc:
            raise RuntimeError(B.last_error())

    for i in range(5):
        go(0.1 * i)
    n = 100
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n):
        go((i + 0.5) / n)
    e1.record(stream)
    torch.cuda.synchronize()
    us_calls = e0.elapsed_time(e1) * 1e3 / n
    # the same calls captured once into a CUDA graph: device time without the host's
    # per-call launch cost
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            go((i + 0.5) / n)
    g.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return {"us_per_call": us_calls, "us_per_call_in_graph": e0.elapsed_time(e1) * 1e3 / n,
            "vocab": s.vocab, "temperature": T, "top_k": k, "top_p": p, "launches_per_call": 3,
            "readback_bytes_avoided": s.vocab * 4}


def lm_head_roofline(L, B, torch, d, s, stream) -> dict:
    import numpy as np
    from sequence_decode_step_gb300.device_model import _to_dev
    table = _to_dev(d.weights["embed"])
    g = _to_dev(d.weights["final_norm"])
    x = torch.randn(s.hidden, device="cuda")
    lg = torch.empty(s.vocab, device="cuda")
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(L.qw_lm_head_workspace_bytes(), dtype=torch.uint8, device="cuda")

    def go():
        rc = L.qw_lm_head_argmax(x.data_ptr(), g.data_ptr(), table.data_ptr(), s.vocab, s.hidden,
                                 s.eps, lg.data_ptr(), am.data_ptr(), ws.data_ptr(),
                                 L.qw_lm_head_workspace_bytes(), stream.cuda_stream)
        if rc:
            raise RuntimeError(B.last_error())

    for _ in range(5):
        go()
    n = 50
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n):
        go()
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / n
    algo = s.vocab * s.hidden * 2 + s.vocab * 4 + s.hidden * 6
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    traffic, traffic_src = recorded_traffic("lm_head_gemv")
    return {"kernel": "gemv_kernel<EPI_LOGITS> (final RMSNorm + tied LM head + argmax)",
            "bound": "hbm", "achieved": algo / sec / 1e9, "peak": hbm, "unit": "GB/s",
            "frac": algo / sec / 1e9 / hbm, "traffic": traffic, "traffic_source": traffic_src,
            "bytes_per_launch": algo,
            "us_per_launch": sec * 1e6,
            "peak_source": "measured burst copy (MEASURED_PEAKS.json hbm_gbs)" if peaks
            else "fallback 6800 GB/s"}


def prefill_flops(s, T: int) -> float:
    """Algorithmic FLOPs of one causal prefill of T rows: the linear projections of
    every row, causal attention (QK^T and PV over keys 0..t), LM head of the last row."""
    per_layer = (s.hidden * s.q_dim + 2 * s.hidden * s.kv_dim + s.q_dim * s.hidden
                 + 3 * s.hidden * s.intermediate)
    linear = 2.0 * T * s.n_layers * per_layer
    attn = 4.0 * s.n_layers * s.n_q_heads * s.head_dim * T * (T + 1) / 2
    return linear + attn + 2.0 * s.vocab * s.hidden


def prefill_timing(torch, W, DeviceModel, stream) -> dict:
    """One batched causal prefill of the qwen3_0.6b_prefill prompt (T = 1024)."""
    wl = W.WORKLOADS[PREFILL_WORKLOAD]
    d = W.draw(wl)
    m = DeviceModel(wl.shape, d.weights, max_ctx=wl.max_ctx, max_prefill_t=wl.prompt_len,
                    stream=stream.cuda_stream)
    reps = 5
    try:
        for _ in range(2):
            m.reset()
            m.prefill(d.prompt)
        torch.cuda.synchronize()
        ms = 0.0
        for _ in range(reps):
            m.reset()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            m.prefill(d.prompt)
            e1.record(stream)
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        ms /= reps
    finally:
        m.close()
    peaks = measured_peaks()
    tc = peaks.get("bf16_tflops", 1900.0)
    fl = prefill_flops(wl.shape, wl.prompt_len)
    return {"workload": PREFILL_WORKLOAD, "T": wl.prompt_len, "ms": ms,
            "tok_per_s": wl.prompt_len / (ms / 1e3),
            "path": "batched: tcgen05 GEMMs (bf16 weights x two-bf16 activations), "
                    "causal flash attention on tcgen05 (TMA-fed tiles, S and O in TMEM, bf16 hi/lo operands)",
            "roofline": {"bound": "tensor", "algorithmic_tflop": fl / 1e12,
                         "achieved": fl / (ms / 1e3) / 1e12, "peak": tc, "unit": "TFLOP/s",
                         "frac": fl / (ms / 1e3) / 1e12 / tc,
                         "peak_source": "measured burst bf16 (MEASURED_PEAKS.json)" if peaks
                         else "fallback 1900 TFLOP/s"}}


def device_draw(W, torch, shape, seed: int, lora=None) -> dict:
    """The workload's tensors (names, shapes, kinds and distributions of its draw order)
    drawn on the device with a seeded torch generator: the timing-only runs of the large
    shapes use this instead of the host draw, which takes minutes at 3 B parameters."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = {}
    for name, shp, kind in W.weight_draw_order(shape, lora):
        if kind == "gain":
            out[name] = torch.full(shp, 0x3F80, dtype=torch.int16, device="cuda")
            continue
        std = W.LORA_STD if kind == "lora" else W.WEIGHT_STD
        w = torch.randn(shp, generator=g, device="cuda", dtype=torch.float32) * std
        out[name] = w if kind == "f32q" else w.to(torch.bfloat16).view(torch.int16)
    return out


def decode_timing(torch, B, DeviceModel, shape, weights, stream, start: int, tokens: int,
                  max_ctx: int, kv=None) -> float:
    """us per token of `tokens` greedy steps from position `start` (graph replays on the
    handle's stream, CUDA events), after a warm-up pass; kv = (k, v) per layer preloaded."""
    m = DeviceModel(shape, weights, max_ctx, stream=stream.cuda_stream)
    try:
        if kv is not None:
            for l, (k, v) in enumerate(kv):
                m.set_kv(l, k, v)
        L = B.lib()
        best = None
        for rep in range(3):
            B.qw_set_pos(m.h, start)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            rc = L.qw_decode_step(m.h, 1, None, None)
            for _ in range(tokens - 1):
                rc |= L.qw_decode_step(m.h, -1, None, None)
            e1.record(stream)
            torch.cuda.synchronize()
            if rc:
                raise RuntimeError(B.last_error(m.h))
            if rep > 0:
                us = e0.elapsed_time(e1) * 1e3 / tokens
                best = us if best is None else min(best, us)
        return best
    finally:
        m.close()


def longctx_timing(torch, W, B, DeviceModel, stream) -> dict:
    """Decode at 8K keys (the long-context workload) with the f32 and the bf16 KV cache:
    32 greedy steps from position 8192, us/token and the byte roofline of each."""
    wl = W.WORKLOADS["qwen3_0.6b_longctx"]
    s = wl.shape
    d = W.draw(wl)
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    out = {"workload": wl.name, "positions": f"{wl.kv_prefill}..{wl.kv_prefill + wl.decode_steps - 1}"}
    for fmt, elem in (("f32", 4), ("bf16", 2)):
        shape = s.replace(kv_format=fmt)
        us = decode_timing(torch, B, DeviceModel, shape, d.weights, stream, wl.kv_prefill,
                           wl.decode_steps, wl.max_ctx, kv=d.kv)
        kvb = sum(kv_bytes(s, p) for p in range(wl.kv_prefill, wl.kv_prefill + wl.decode_steps))
        byt = weight_bytes(s) + kvb * elem // 4 / wl.decode_steps
        out[fmt] = {"us_per_token": us, "tok_per_s": 1e6 / us, "bytes_per_token": byt,
                    "roofline_frac": byt / (us * 1e-6) / 1e9 / hbm}
    return out


def q8_timing(torch, W, B, DeviceModel, stream) -> dict:
    """Q8_0 decode of the Qwen3-0.6B shape (projections and tied head in Q8_0, on the
    persistent kernel): us/token from position 5 and the byte roofline."""
    wl = W.WORKLOADS["qwen3_0.6b_q8_0_decode"]
    s = wl.shape
    w = device_draw(W, torch, s, wl.seed)
    us = decode_timing(torch, B, DeviceModel, s, w, stream, wl.prompt_len, wl.decode_steps,
                       wl.max_ctx)
    per_layer = (s.hidden * s.q_dim + 2 * s.hidden * s.kv_dim + s.q_dim * s.hidden
                 + 3 * s.hidden * s.intermediate)
    byt = (s.n_layers * per_layer + s.vocab * s.hidden) * (1 + 2 / 32) + \
        sum(kv_bytes(s, p) for p in range(wl.prompt_len, wl.prompt_len + wl.decode_steps)) / wl.decode_steps
    hbm = measured_peaks().get("hbm_gbs", 6800.0)
    return {"workload": wl.name, "us_per_token": us, "tok_per_s": 1e6 / us,
            "bytes_per_token": byt, "roofline_frac": byt / (us * 1e-6) / 1e9 / hbm,
            "path": "persistent kernel, int8 rows with fp16 block scales decoded in the GEMV",
            "data": "seeded device draw (torch), the workload's shapes and distributions"}


def int4_decode_timing(torch, W, B, DeviceModel, stream) -> dict:
    """Decode of the Qwen2.5-3B int4 g128 shape (q/k/v bias, untied int4 head) from a
    cache pre-filled to 4096 keys, on the persistent kernel, without and with the rank-16
    LoRA on q and v: us/token over the workload's steps and the byte roofline."""
    wl = W.WORKLOADS["qwen2.5_3b_int4_lora"]
    s = wl.shape
    w = device_draw(W, torch, s, wl.seed, wl.lora)
    lora = {k: v for k, v in w.items() if k.startswith("lora.")}
    m = DeviceModel(s, {k: v for k, v in w.items() if not k.startswith("lora.")}, wl.max_ctx,
                    stream=stream.cuda_stream)
    del w
    g = torch.Generator(device="cuda")
    g.manual_seed(wl.seed)
    shp = (s.n_kv_heads, wl.kv_prefill, s.head_dim)
    for l in range(s.n_layers):  # N(0, 1) in bf16-representable f32, as the workload's prefill
        k, v = (torch.randn(shp, generator=g, device="cuda").to(torch.bfloat16).float()
                for _ in range(2))
        m.set_kv(l, k, v)
    torch.cuda.empty_cache()
    L = B.lib()
    per_layer = (s.hidden * s.q_dim + 2 * s.hidden * s.kv_dim + s.q_dim * s.hidden
                 + 3 * s.hidden * s.intermediate)
    wbytes = (s.n_layers * per_layer + s.vocab * s.hidden) * (0.5 + 2 / 128)
    kvb = sum(kv_bytes(s, p) for p in range(wl.kv_prefill, wl.kv_prefill + wl.decode_steps))
    r = wl.lora.rank
    lora_bytes = s.n_layers * 2 * r * (2 * s.hidden + s.q_dim + s.kv_dim)
    hbm = measured_peaks().get("hbm_gbs", 6800.0)
    out = {"workload": wl.name, "positions": f"{wl.kv_prefill}..{wl.kv_prefill + wl.decode_steps - 1}",
           "path": "persistent kernel (wide-input build), int4 nibbles decoded in the GEMV",
           "data": "seeded device draw (torch), the workload's shapes and distributions"}
    try:
        for mode in ("lora_off", "lora_on"):
            m.set_lora(lora if mode == "lora_on" else None, wl.lora.alpha)
            path = B.qw_get_decode_path(m.h)
            ts = []
            for rep in range(3):
                B.qw_set_pos(m.h, wl.kv_prefill)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                rc = L.qw_decode_step(m.h, 1, None, None)
                for _ in range(wl.decode_steps - 1):
                    rc |= L.qw_decode_step(m.h, -1, None, None)
                e1.record(stream)
                torch.cuda.synchronize()
                if rc:
                    raise RuntimeError(B.last_error(m.h))
                if rep > 0:
                    ts.append(e0.elapsed_time(e1) * 1e3 / wl.decode_steps)
            us = sum(ts) / len(ts)
            byt = wbytes + kvb / wl.decode_steps + (lora_bytes if mode == "lora_on" else 0)
            out[mode] = {"us_per_token": us, "tok_per_s": 1e6 / us, "bytes_per_token": byt,
                         "roofline_frac": byt / (us * 1e-6) / 1e9 / hbm, "decode_path": path}
        out["traffic"], out["traffic_source"] = recorded_traffic("decode_mega_big")
    finally:
        m.close()
    return out


def int4_prefill_timing(torch, W, B, DeviceModel, stream, T: int = 1024) -> dict:
    """Batched prefill of T ids on the Qwen2.5-3B int4 g128 shape: weights dequantised
    layer by layer into exact two-bf16 planes, tcgen05 GEMMs with three MMAs per product."""
    s = W.QWEN25_3B_INT4
    w = device_draw(W, torch, s, 4)
    m = DeviceModel(s, w, T + 8, max_prefill_t=T, stream=stream.cuda_stream)
    del w
    ids = list(W.random_ids(s.vocab, T, seed=4))
    try:
        ms = []
        for rep in range(4):
            m.reset()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            m.prefill(ids)
            e1.record(stream)
            torch.cuda.synchronize()
            if rep > 0:
                ms.append(e0.elapsed_time(e1))
    finally:
        m.close()
    t = sum(ms) / len(ms)
    fl = prefill_flops(s, T)
    tc = measured_peaks().get("bf16_tflops", 1900.0)
    return {"shape": s.name, "T": T, "ms": t, "tok_per_s": T / (t / 1e3),
            "roofline": {"bound": "tensor", "algorithmic_tflop": fl / 1e12,
                         "achieved": fl / (t / 1e3) / 1e12, "peak": tc, "unit": "TFLOP/s",
                         "frac": fl / (t / 1e3) / 1e12 / tc},
            "data": "seeded device draw (torch), the workload's shapes and distributions"}


# ============================================================================ CPU oracle legs
def oracle_sample(budget_s: float, min_tokens: int, max_tokens: int) -> dict:
    """Time the oracle (as it stands) decoding the benchmark workload on this host.

    Runs in a child process started with OPENBLAS_NUM_THREADS=1, so it is the
    single-threaded oracle; returns tokens/s over the decode tokens it finished.
    """
    import workload as W
    from oracle import qwen_ref as R
    wl = W.WORKLOADS[WORKLOAD]
    d = W.draw(wl)
    o = R.build_oracle(d, max_ctx=wl.prompt_len + max_tokens + 1, cache_f64=True)
    cp = o.prefill(d.prompt)
    tok = R.greedy_argmax(cp["logits"])
    n = 0
    t0 = time.perf_counter()
    while n < max_tokens and (n < min_tokens or time.perf_counter() - t0 < budget_s):
        tok = R.greedy_argmax(o.decode_step(tok)["logits"])
        n += 1
    dt = time.perf_counter() - t0
    return {"tokens": n, "seconds": dt, "tok_per_s": n / dt}


def run_oracle_child(budget_s: float, min_tokens: int, max_tokens: int) -> dict:
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import json, bench; print('ORACLE_JSON ' + json.dumps("
            f"bench.oracle_sample({budget_s}, {min_tokens}, {max_tokens})))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    for ln in r.stdout.splitlines():
        if ln.startswith("ORACLE_JSON "):
            return json.loads(ln[len("ORACLE_JSON "):])
    raise RuntimeError("oracle sample failed:\n" + r.stdout[-2000:] + r.stderr[-2000:])


def cpu_baseline(budget_s: float = 15.0) -> dict:
    o = run_oracle_child(budget_s, 2, 128)
    return {"value": o["tok_per_s"], "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"{WORKLOAD}: 5-id prompt prefill (untimed), then {o['tokens']} greedy "
                      f"decode tokens from position 5 ({o['seconds']:.1f} s), numpy oracle, "
                      "one BLAS thread", **host_cpu()}


def run_reference(args) -> dict:
    """The CPU oracle on this host as the reference arm: each step is a bounded
    sample of 2 decode tokens of the same workload."""
    per_step = 2
    o = run_oracle_child(0.0, per_step * (args.warmup + args.steps),
                         per_step * (args.warmup + args.steps))
    # the child times all tokens together; the warm-up tokens are included in its
    # count, so the rate is tokens / seconds over the whole run
    v = o["tok_per_s"]
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step / v * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "prompt_ids": 5,
                       "decode_tokens_per_step": per_step,
                       "l2": "n/a (CPU)", "parallelism": "single host thread"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": f"{o['tokens']} greedy decode tokens of {WORKLOAD} "
                                       f"from position 5, numpy oracle, one BLAS thread",
                             **host_cpu()},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ============================================================================ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_base", action="store_false")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="skip the long-context, Q8_0 and int4-prefill lines")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        res["cpu_baseline"] = cpu_baseline() if args.cpu_base else None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
