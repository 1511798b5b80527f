"""Skinny-M sweep of the W8A8 linear against the BF16-weight comparator.

    python -m quantized_verification_gb300.msweep [--model qwen3-32b] [--m 1,2,4,...]

For each projection shape of the model (q|k|v, o, gate|up, down, LM head) and
each token count M, times qv_w8a8_linear (codes quantized beforehand) and
qv_bf16_linear as back-to-back launches in a CUDA graph with CUDA events,
rotating over enough distinct weight copies that every launch streams its
weights from HBM (at least twice the L2 size per rotation). Prints one
markdown table: microseconds per launch, weight-stream GB/s (int8 bytes for
W8A8, bf16 bytes for the comparator) and the speed-up.

Weights are seeded synthetic N(0, 0.02) (bf16, quantized per channel with
qv_quantize_weight); activations are seeded N(0, 1) with 1 % of channels x20.
"""
from __future__ import annotations

import argparse

import torch

from . import build, qv, synth

L2_BYTES = 129 * 1024 * 1024


def shapes(model: dict):
    h, q, kv, ffn, V = model["hidden"], model.get("q", model["hidden"]), model["kv"], model["ffn"], model["vocab"]
    return [("qkv", h, q + 2 * kv), ("o", q, h), ("gate_up", h, 2 * ffn), ("down", ffn, h), ("lm_head", h, V)]


def time_graph(fn, reps: int) -> float:
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(0, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in range(reps):
            fn(r, torch.cuda.current_stream())
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(5):
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / reps)
    return sorted(ts)[2] * 1e3   # median, microseconds


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--model", default="qwen3-32b", choices=sorted(synth.MODELS))
    ap.add_argument("--m", default="1,2,4,8,16,32,64,128,256")
    ap.add_argument("--reps", type=int, default=24)
    ap.add_argument("--shapes", default="qkv,o,gate_up,down,lm_head", help="projections to time")
    args = ap.parse_args(argv)
    build.build()
    model = synth.MODELS[args.model]
    ms = [int(v) for v in args.m.split(",")]
    dev = torch.device("cuda")
    print("| shape (K -> N) | M | W8A8 us | W8A8 GB/s | BF16 us | BF16 GB/s | speed-up |")
    print("|---|---|---|---|---|---|---|")
    wanted = set(args.shapes.split(","))
    for name, K, N in [t for t in shapes(model) if t[0] in wanted]:
        copies = max(2, -(-2 * L2_BYTES // (2 * N * K)))        # bf16 copies exceed 2 x L2
        wb = [synth.weights(N, K, synth.subseed(11, "msweep", name, c), device=dev) for c in range(copies)]
        wq = [torch.empty(N, K, dtype=torch.int8, device=dev) for _ in range(copies)]
        sw = [torch.empty(N, device=dev) for _ in range(copies)]
        for c in range(copies):
            qv.qv_quantize_weight(wb[c], wq[c], sw[c])
        for M in ms:
            x = synth.activations(M, K, synth.subseed(12, "msweep", name, M), device=dev)
            xq = torch.empty(M, K, dtype=torch.int8, device=dev)
            sx = torch.empty(M, device=dev)
            qv.qv_quantize_act(x, xq, sx)
            y = torch.empty(M, N, device=dev)
            lm = name == "lm_head"
            tok = torch.empty(M, dtype=torch.int32, device=dev)
            ws = qv.workspace(qv.QV_OP_LM_HEAD if lm else qv.QV_OP_LINEAR, M, K, N)
            wsb = qv.workspace(qv.QV_OP_BF16_LINEAR, M, K, N)

            def w8(r, s):
                c = r % copies
                if lm:
                    qv.qv_lm_head_argmax(xq, sx, wq[c], sw[c], tok, ws, stream=s)
                else:
                    qv.qv_w8a8_linear(xq, sx, wq[c], sw[c], y, ws, stream=s)

            def bf(r, s):
                qv.qv_bf16_linear(x, wb[r % copies], y, wsb, stream=s)

            t8 = time_graph(w8, args.reps)
            tb = time_graph(bf, args.reps)
            print(f"| {name} ({K} -> {N}) | {M} | {t8:.1f} | {N * K / t8 / 1e3:.0f} | {tb:.1f} | "
                  f"{2 * N * K / tb / 1e3:.0f} | {tb / t8:.2f}x |", flush=True)
        del wb, wq, sw
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
