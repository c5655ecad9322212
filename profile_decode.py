"""Drive a few decode steps of a workload for profilers (ncu) and quick timing.

  python profile_decode.py [--workload NAME] [--tokens N]
         [--lm-head N] [--prefill-reps N] [--path 0|1] [--sample N]

Draws the workload's weights, prefills its prompt (or preloads its KV cache),
runs N greedy decode tokens as graph replays, then N stand-alone LM-head
launches, and prints the mean per-token and per-launch times (CUDA events).
No oracle, no checks: parity lives in tests/.
"""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch
    import workload as W
    from sequence_decode_step_gb300 import _binding as B
    from sequence_decode_step_gb300.device_model import DeviceModel, _to_dev

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3_0.6b_decode")
    ap.add_argument("--tokens", type=int, default=8)
    ap.add_argument("--lm-head", type=int, default=4)
    ap.add_argument("--prefill-reps", type=int, default=0,
                    help="batched prefills of the workload's prompt to run first")
    ap.add_argument("--path", type=int, default=0, help="decode path: 0 persistent, 1 graph")
    ap.add_argument("--sample", type=int, default=0,
                    help="qw_sample calls on the handle's last logits row (T 0.7, top_k 50, top_p 0.9)")
    args = ap.parse_args()
    wl = W.WORKLOADS[args.workload]
    d = W.draw(wl)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    m = DeviceModel(wl.shape, d.weights, max_ctx=max(wl.max_ctx, wl.prompt_len + wl.kv_prefill
                                                     + args.tokens + 8),
                    max_prefill_t=wl.prompt_len if args.prefill_reps else 0,
                    stream=stream.cuda_stream)
    head_src = {k: d.weights[k] for k in ("embed", "final_norm")} if args.lm_head else {}
    d.weights = {}                 # the library holds its own copies
    torch.cuda.empty_cache()       # keep the device footprint small for profilers
    L = B.lib()
    B.qw_set_decode_path(m.h, args.path)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.prefill_reps):
        m.reset()
        torch.cuda.synchronize()
        e0.record(stream)
        m.prefill(d.prompt)
        e1.record(stream)
        torch.cuda.synchronize()
        print(f"prefill T={len(d.prompt)}: {e0.elapsed_time(e1):.3f} ms")
    if wl.kv_prefill:
        for l, (k, v) in enumerate(d.kv):
            m.set_kv(l, k, v)
        m.set_pos(wl.kv_prefill)
        first = d.start_token
    else:
        first = m.prefill(d.prompt) if not args.prefill_reps else m.decode(-1)
    torch.cuda.synchronize()
    e0.record(stream)
    rc = L.qw_decode_step(m.h, first, None, None)
    for _ in range(args.tokens - 1):
        rc |= L.qw_decode_step(m.h, -1, None, None)
    e1.record(stream)
    torch.cuda.synchronize()
    if rc:
        raise SystemExit(B.last_error(m.h))
    print(f"decode: {e0.elapsed_time(e1) * 1e3 / args.tokens:.1f} us/token over {args.tokens}")
    s = wl.shape
    if args.lm_head and s.tie_word_embeddings:
        table, g = _to_dev(head_src["embed"]), _to_dev(head_src["final_norm"])
        x = torch.randn(s.hidden, device="cuda")
        lg = torch.empty(s.vocab, device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        wsb = L.qw_lm_head_workspace_bytes()
        ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.lm_head):
            rc |= L.qw_lm_head_argmax(x.data_ptr(), g.data_ptr(), table.data_ptr(), s.vocab,
                                      s.hidden, s.eps, lg.data_ptr(), am.data_ptr(),
                                      ws.data_ptr(), wsb, stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if rc:
            raise SystemExit(B.last_error())
        print(f"lm head: {e0.elapsed_time(e1) * 1e3 / args.lm_head:.1f} us/launch")
    if args.sample:
        tok = torch.empty(1, dtype=torch.int32, device="cuda")
        wsb = L.qw_sample_workspace_bytes(s.vocab, 50)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        lg = m._logits_buf()
        m.decode(-1, logits=True)  # one more step, its logits row in lg
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(args.sample):
            B.qw_sample(lg.data_ptr(), s.vocab, 0.7, 50, 0.9, (i + 0.5) / args.sample,
                        tok.data_ptr(), ws.data_ptr(), wsb, stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        print(f"sample: {e0.elapsed_time(e1) * 1e3 / args.sample:.1f} us/call, last id {int(tok.item())}")
    m.close()


if __name__ == "__main__":
    main()
