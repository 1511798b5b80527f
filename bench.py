"""Benchmark: W8A8 verify-pass tokens/s and weight-stream GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one full verify pass of the Qwen3-8B-shaped stack at M = 5 tokens
(batch 1, gamma = 4): per layer four act-quant + W8A8-linear phases (q|k|v, o,
gate|up, down; 36 layers, 6.95 GB int8), the final act quant, the LM head
4096 -> 151936 fused with the greedy argmax, and the acceptance of gamma = 4
drafts. Weights are seeded synthetic (N(0, 0.02), bf16, quantized per output
channel), activations seeded N(0, 1) with 1% outlier channels x20. Inputs are
resident in HBM before timing; the 7.57 GB of weights per step exceed the
129 MB L2, so no flush is needed between steps.

Rank 0 prints one JSON line. With torchrun (N > 1) every rank runs an
independent replica (the path is not sharded); value = all tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W8A8 verify-pass tokens/s and weight-stream GB/s (fraction of GB300 HBM peak)"
UNIT = "tokens/s"
WORKLOAD = ("qwen3-8b-shaped W8A8 verify step, M=5 (B=1, gamma=4): 36 layers x (qkv 4096->6144, "
            "o 4096->4096, gate|up 4096->24576, down 12288->4096) + LM head 4096->151936 argmax + accept")
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per algorithmic byte of one projection launch of the streaming
# W8A8 kernel: ncu dram__bytes_read.sum + dram__bytes_write.sum of the gate+up
# launch (4096 -> 24576, M = 5) over its algorithmic bytes. Valid only for the
# kernel sources whose sha256 is recorded (kernel_source_sha); roofline.traffic
# is null otherwise.
NCU_TRAFFIC = {"source_sha256": "f8c90da96ed0da604d6a28fd5d09247e0934840cfcf0617f0a3407307704e2fc",
               "dram_bytes_per_algorithmic_byte": (101689856 + 2688768) / 101273620}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        for (ts, line) in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append({"sm": float(parts[2]), "max": float(parts[3]), "power": float(parts[4]),
                             "hw_slowdown": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8],
                             "sw_power_cap": parts[9]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = {"hw_slowdown": "hw_slowdown", "hw_thermal": "hw_thermal_slowdown",
                 "sw_thermal": "sw_thermal_slowdown", "sw_power_cap": "sw_power_cap"}
        reasons = sorted({names[k] for r in rows for k in names if r[k].lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_median": statistics.median(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# CPU oracle: the baseline leg (and the reference arm)
# ---------------------------------------------------------------------------
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleStep:
    """The oracle on the bench's workload: the Qwen3-8B-shaped step at M = 5
    (per layer the four quantize -> W8A8 linear phases, then the LM head
    4096 -> 151936 with the greedy argmax, then the acceptance), with every
    multiply-accumulate of the step done. To bound host memory and set-up
    time, one layer's weights (seeded bf16, quantized by the oracle) serve all
    36 layers; each layer quantizes its own seeded inputs. Each linear's
    output channels are split over `threads` host threads, each calling the
    oracle on its slice (a ctypes call releases the GIL), so every output is
    the oracle's own arithmetic; the argmax and the acceptance run once over
    the assembled logits."""

    def __init__(self, M=5, B=1, gamma=4, seed=0):
        import concurrent.futures as cf

        import numpy as np
        import torch

        import oracle
        from quantized_verification_gb300 import synth
        self.np = np
        self.o = oracle.get()
        self.M, self.B, self.gamma = M, B, gamma
        m = synth.QWEN3_8B
        h, kv, ffn, V = m["hidden"], m["kv"], m["ffn"], m["vocab"]
        self.layers = m["layers"]
        self.phases = [("qkv", h, h + 2 * kv), ("o", h, h), ("gate_up", h, 2 * ffn), ("down", ffn, h)]
        self.cores = host_cores()
        self.pool = cf.ThreadPoolExecutor(self.cores)
        bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)

        def quantized(name, N, K):
            w = bits(synth.weights(N, K, synth.subseed(seed, "cpu_w", name)))
            b = np.linspace(0, N, self.cores + 1).astype(int)
            parts = list(self.pool.map(lambda i: self.o.quantize_rows(w[b[i]:b[i + 1]], bf16=True),
                                       range(self.cores)))
            return np.concatenate([q for q, _ in parts]), np.concatenate([s for _, s in parts])
        self.w = {name: quantized(name, N, K) for (name, K, N) in self.phases}
        self.w["lm_head"] = quantized("lm_head", V, h)
        self.x = [[bits(synth.activations(M, K, synth.subseed(seed, "cpu_x", l, name)))
                   for (name, K, N) in self.phases] for l in range(self.layers)]
        self.h_final = bits(synth.activations(M, h, synth.subseed(seed, "cpu_x", "final")))
        rng = np.random.default_rng(seed)
        self.drafts = rng.integers(0, V, (B, gamma)).astype(np.int32)
        self.macs_layer = M * sum(N * K for (_, K, N) in self.phases)
        self.macs_lm = M * V * h
        self.total_macs = self.layers * self.macs_layer + self.macs_lm

    def _linear(self, xq, sx, wq, sw, threads):
        if threads == 1:
            return self.o.w8a8_linear(xq, sx, wq, sw)[0]
        b = self.np.linspace(0, wq.shape[0], threads + 1).astype(int)
        parts = list(self.pool.map(lambda i: self.o.w8a8_linear(xq, sx, wq[b[i]:b[i + 1]], sw[b[i]:b[i + 1]])[0],
                                   range(threads)))
        return self.np.concatenate(parts, axis=1)

    def step(self, threads, layers=None):
        """One verify step (or its first `layers` layers + the LM head);
        returns (tokens, accepted lengths, MACs done)."""
        L = self.layers if layers is None else layers
        for l in range(L):
            for p, (name, K, N) in enumerate(self.phases):
                xq, sx = self.o.quantize_rows(self.x[l][p], bf16=True)
                self._linear(xq, sx, *self.w[name], threads)
        xq, sx = self.o.quantize_rows(self.h_final, bf16=True)
        logits = self._linear(xq, sx, *self.w["lm_head"], threads)
        tok, _ = self.o.argmax_rows(logits)
        ln, _ = self.o.accept(tok, self.drafts, self.B, self.gamma)
        return tok, ln, L * self.macs_layer + self.macs_lm

    def timed(self, threads, steps=1, layers=None):
        """Wall time per step over `steps` steps; returns (seconds, MACs per step)."""
        t0 = time.perf_counter()
        for _ in range(steps):
            _, _, macs = self.step(threads, layers)
        return (time.perf_counter() - t0) / steps, macs


def cpu_baseline():
    st = OracleStep()
    st.step(st.cores)                                   # warm-up
    t_mt, _ = st.timed(st.cores, steps=2)
    t_1, _ = st.timed(1, steps=1)
    return {"value": st.M / t_mt, "unit": UNIT, "cores": st.cores, "kind": "oracle",
            "ms_per_step": t_mt * 1e3, "threads": st.cores,
            "single_thread": {"value": st.M / t_1, "unit": UNIT, "ms_per_step": t_1 * 1e3},
            "sample": f"plain C oracle, whole verify steps ({st.total_macs / 1e9:.1f} GMAC each: 36 layers of "
                      f"act quant + W8A8 linears, LM head 4096->151936 + argmax, accept; one layer's weights "
                      f"serve all layers); output channels of each linear split over {st.cores} host threads "
                      f"(2 timed steps after one warm-up), and 1 thread (1 timed step)"}


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, same metric and workload:
    whole verify steps split over every host core. If K + W whole steps would
    not end within a few minutes, each step covers the first layers only (the
    LM head always) and the value is scaled by MAC share; ms_per_step is the
    measured time of the steps as run."""
    if rank != 0:
        return 0
    st = OracleStep()
    t_est, _ = st.timed(st.cores, steps=1)              # first warm-up step, full size
    budget_s = 200.0
    n = max(args.steps + max(args.warmup - 1, 0), 1)
    layers = st.layers
    if n * t_est > budget_s:
        t_layer = t_est * st.macs_layer / st.total_macs
        t_lm = t_est * st.macs_lm / st.total_macs
        layers = max(1, min(st.layers, int((budget_s / n - t_lm) / max(t_layer, 1e-9))))
    for _ in range(max(args.warmup - 1, 0)):
        st.step(st.cores, layers)
    t_step, macs = st.timed(st.cores, steps=args.steps, layers=layers)
    value = st.M / (t_step * st.total_macs / macs)
    whole = layers == st.layers
    sample = (f"each step a whole verify step ({st.total_macs / 1e9:.1f} GMAC)" if whole else
              f"each step the first {layers} of 36 layers + the LM head ({macs / 1e9:.1f} of "
              f"{st.total_macs / 1e9:.1f} GMAC), value scaled by MAC share")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8/int32/fp32",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": st.M, "B": st.B, "gamma": st.gamma,
                                            "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": st.cores, "kind": "oracle",
                             "sample": f"plain C oracle on {st.cores} host threads (output channels of each "
                                       f"linear split across them; one layer's weights serve all layers); "
                                       + sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_sha():
    """Hash of the sources the streaming W8A8 kernel is compiled from."""
    h = hashlib.sha256()
    for name in ("k_stream_gemm.cu", "stream_common.cuh", "qv_ptx.cuh", "qv_internal.h"):
        with open(os.path.join(ROOT, "quantized_verification_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def time_graph(torch, graph, n, stream):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=None, help="layer count override (testing only)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--kernel-reps", type=int, default=20)
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from quantized_verification_gb300 import build, qv, replicas, synth
    from quantized_verification_gb300.stack import VerifyStack
    build.build()

    t_setup = time.time()
    stack = VerifyStack(layers=args.layers, B=1, gamma=4, seed=1234 + rank, device=str(dev),
                        keep_bf16=not args.no_comparator)
    stack.enqueue()                 # drafts agree with the verifier for a geometric(0.7) prefix
    torch.cuda.synchronize()
    t_ver = stack.tokens.view(stack.B, stack.gamma + 1).cpu()
    stack.drafts.copy_(synth.geometric_drafts(t_ver, stack.V, 0.7, seed=99 + rank))
    per_op_graph = stack.capture()
    two_call_graph = stack.capture_two_call()
    fused_graph = stack.capture_fused()
    log(f"setup {time.time() - t_setup:.1f} s; weight bytes/step {stack.weight_bytes() / 1e9:.3f} GB")
    stream = torch.cuda.current_stream()

    # three public-API paths of the same step; all must give the same tokens
    paths = [
        ("per_op", per_op_graph, stack.launches_per_step(),
         "per-op ABI calls (qv_w8a8_linear_act per projection, qv_lm_head_argmax_act, qv_accept) in one CUDA graph"),
        ("two_call", two_call_graph, stack.launches_per_step(),
         "per-op ABI calls (qv_quantize_act + qv_w8a8_linear per projection, qv_quantize_act + "
         "qv_lm_head_argmax, qv_accept) in one CUDA graph"),
        ("verify_stack", fused_graph, stack.launches_per_step(fused=True),
         "qv_verify_stack: one persistent cooperative launch per step"),
    ]
    paths_ms = {}
    ref_tok = ref_len = None
    for name, g, _, _ in paths:
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        if ref_tok is None:
            ref_tok, ref_len = stack.tokens.clone(), stack.accept_len.clone()
        assert torch.equal(stack.tokens, ref_tok) and torch.equal(stack.accept_len, ref_len), \
            f"{name} step disagrees with {paths[0][0]}"
        paths_ms[name] = time_graph(torch, g, max(20, args.steps // 5), stream)
        log(f"{name} path {paths_ms[name]:.4f} ms/step")
    best = min(paths, key=lambda t: paths_ms[t[0]])
    path_name, step_graph, launches, path = best
    for _ in range(max(args.warmup, 3)):
        step_graph.replay()
    torch.cuda.synchronize()
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = ClockSampler(cvd.split(",")[local].strip() if cvd else str(local))
    clocks.start()
    replicas.barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    ms = time_graph(torch, step_graph, args.steps, stream)
    w1 = time.time()
    replicas.barrier()
    clocks.stop()
    ms_max, value = replicas.job_step_time_and_rate(ms, stack.M, dev)
    clk = clocks.summary(w0, w1)
    alg_bytes = stack.algorithmic_bytes()
    log(f"step {ms:.4f} ms ({alg_bytes / (ms * 1e-3) / 1e9:.1f} GB/s algorithmic), clocks {clk}")
    assert qv.qv_device_error() == 0, "a kernel hit its wait limit"
    # per-step spread, after the timed region: each step bracketed by its own
    # pair of events on the launching stream
    n_dist = min(args.steps, 200)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dist)]
    for e0, e1 in ev:
        e0.record(stream)
        step_graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    per_step = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
    step_dist = {"n": n_dist, "p10": per_step[n_dist // 10], "median": per_step[n_dist // 2],
                 "p90": per_step[(9 * n_dist) // 10], "unit": "ms",
                 "note": "each step timed alone with CUDA events, after the timed region"}
    log(f"per-step ms p10 {step_dist['p10']:.4f} median {step_dist['median']:.4f} p90 {step_dist['p90']:.4f}")
    peak, peak_kind = read_peaks()

    # ---- dominant kernel: the W8A8 streaming GEMM on the step's 144
    # projections (codes quantized beforehand), back to back in one graph
    M = stack.M
    lin_bytes = stack.linear_launch_bytes(fused_act=False)
    xqs = []
    for l in range(stack.layers):
        for p, (name, K, N) in enumerate(stack.phases):
            xq = torch.empty(M, K, dtype=torch.int8, device=dev)
            sxp = torch.empty(M, device=dev)
            qv.qv_quantize_act(stack.inputs[l][p], xq, sxp)
            xqs.append((xq, sxp))
    torch.cuda.synchronize()

    def lin_seq(s):
        j = 0
        for l in range(stack.layers):
            for p, (name, K, N) in enumerate(stack.phases):
                wq, sw = stack.weights[l][p]
                qv.qv_w8a8_linear(xqs[j][0], xqs[j][1], wq, sw, stack.y[: M * N].view(M, N), stack.ws, stream=s)
                j += 1
    gl = VerifyStack._capture(lin_seq, dev)
    lin_ms = time_graph(torch, gl, args.kernel_reps, stream)
    achieved = sum(lin_bytes) / (lin_ms * 1e-3) / 1e9
    traffic = None
    if NCU_TRAFFIC["source_sha256"] == kernel_source_sha() and NCU_TRAFFIC["dram_bytes_per_algorithmic_byte"]:
        traffic = NCU_TRAFFIC["dram_bytes_per_algorithmic_byte"] * sum(lin_bytes) / len(lin_bytes)
    kname = ("w8a8_stream_kernel (int8 mma.sync, qv_w8a8_linear)" if M <= 32
             else "w8a8_tc_kernel (tcgen05, qv_w8a8_linear)")
    linear_kernel = {"kernel": kname, "achieved": achieved,
                     "frac": achieved / peak, "bytes_per_launch": sum(lin_bytes) / len(lin_bytes),
                     "launch_ms_mean": lin_ms / len(lin_bytes),
                     "timing": "144 launches of the step's projections back to back in one CUDA graph"}
    if launches <= 2:
        # the persistent kernel is the step: one launch, timed above
        k_bytes = alg_bytes / launches
        k_ms = ms / launches
        roofline = {"bound": "hbm", "achieved": k_bytes / (k_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                    "frac": k_bytes / (k_ms * 1e-3) / 1e9 / peak, "traffic": None,
                    "kernel": "verify_stack_kernel (qv_verify_stack)", "bytes_per_launch": k_bytes,
                    "launch_ms_mean": k_ms,
                    "timing": "the timed steps, one launch per step, CUDA events on the launching stream",
                    "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"}
    else:
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": traffic, "kernel": kname,
                    "bytes_per_launch": sum(lin_bytes) / len(lin_bytes),
                    "launch_ms_mean": lin_ms / len(lin_bytes),
                    "timing": "144 launches of the step's projections back to back in one CUDA graph, "
                              "CUDA events on the launching stream",
                    "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"}
    log(f"w8a8 linear kernel: {achieved:.1f} GB/s = {achieved / peak:.3f} of {peak_kind} {peak}")
    del gl, xqs

    # ---- BF16-weight comparator on the same shapes
    comparator = None
    if not args.no_comparator:
        stack.prepare_bf16()
        gb = VerifyStack._capture(stack.enqueue_bf16, dev)
        for _ in range(3):
            gb.replay()
        bf_ms = time_graph(torch, gb, max(10, args.steps // 4), stream)
        comparator = {"bf16_ms_per_step": bf_ms, "w8a8_ms_per_step": ms, "speedup": bf_ms / ms,
                      "bf16_weight_bytes": stack.bf16_weight_bytes(),
                      "bf16_stream_gbs": stack.bf16_weight_bytes() / (bf_ms * 1e-3) / 1e9,
                      "note": "same shapes; qv_bf16_linear for every projection and the LM head "
                              "(logits written, argmax not included)"}
        log(f"bf16 comparator {bf_ms:.4f} ms/step, speedup {bf_ms / ms:.3f}x")
        del gb

    # ---- batched verify (the batched workload): B = 8 x (gamma + 1 = 8) =
    # 64 and B = 16 x 5 = 80 tokens through the same 36-layer stack (its
    # resident weights shared) + LM head + per-sequence acceptance; the
    # W8A8 GEMM alone over the step's projections; the BF16 comparator
    batched = None
    if rank == 0:
        batched = {}
        for (Bb, gm) in ((8, 7), (16, 4)):
            bs = VerifyStack(layers=args.layers, B=Bb, gamma=gm, seed=4321 + rank, device=str(dev),
                             keep_bf16=comparator is not None, share_weights=stack)
            bs.enqueue_two_call()
            torch.cuda.synchronize()
            bs.drafts.copy_(synth.geometric_drafts(bs.tokens.view(Bb, gm + 1).cpu(), bs.V, 0.7, seed=77 + rank))
            gbt = bs.capture_two_call()
            for _ in range(3):
                gbt.replay()
            torch.cuda.synchronize()
            b_ms = time_graph(torch, gbt, max(10, args.steps // 10), stream)
            del gbt
            Mb = bs.M
            bxq = []
            for l in range(bs.layers):
                for p_, (name, K, N) in enumerate(bs.phases):
                    xq = torch.empty(Mb, K, dtype=torch.int8, device=dev)
                    sxp = torch.empty(Mb, device=dev)
                    qv.qv_quantize_act(bs.inputs[l][p_], xq, sxp)
                    bxq.append((xq, sxp))
            torch.cuda.synchronize()

            def blin(s_, bs=bs, bxq=bxq, Mb=Mb):
                j = 0
                for l in range(bs.layers):
                    for p_, (name, K, N) in enumerate(bs.phases):
                        wq, sw = bs.weights[l][p_]
                        qv.qv_w8a8_linear(bxq[j][0], bxq[j][1], wq, sw, bs.y[: Mb * N].view(Mb, N), bs.ws, stream=s_)
                        j += 1
            gl2 = VerifyStack._capture(blin, dev)
            bl_ms = time_graph(torch, gl2, max(3, args.kernel_reps // 4), stream)
            del gl2, bxq
            bl_bytes = bs.linear_launch_bytes(fused_act=False)
            b_ach = sum(bl_bytes) / (bl_ms * 1e-3) / 1e9
            slices = (Mb + 79) // 80
            entry = {"B": Bb, "gamma": gm, "M": Mb, "ms_per_step": b_ms, "tokens_per_s": Mb / (b_ms * 1e-3),
                     "weight_stream_gbs": bs.weight_bytes() / (b_ms * 1e-3) / 1e9,
                     "accept_len_mean": float(bs.accept_len.float().mean()),
                     "roofline": {"bound": "hbm", "achieved": b_ach, "peak": peak, "unit": "GB/s",
                                  "frac": b_ach / peak, "traffic": None,
                                  "kernel": f"w8a8_tc_kernel<{64 if Mb <= 64 else 80}> (tcgen05 on exactly widened codes)",
                                  "launches_per_projection": slices,
                                  "bytes_per_launch": sum(bl_bytes) / len(bl_bytes) / slices,
                                  "launch_ms_mean": bl_ms / len(bl_bytes) / slices,
                                  "timing": "144 projections of the step back to back in one CUDA graph (codes "
                                            "quantized beforehand), CUDA events on the launching stream; algorithmic "
                                            "bytes include each launch's own weight stream",
                                  "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"},
                     "path": "per projection qv_quantize_act + qv_w8a8_linear, qv_quantize_act + qv_lm_head_argmax, "
                             "qv_accept (per sequence); one CUDA graph"}
            if comparator is not None:
                bs.prepare_bf16()
                gbb = VerifyStack._capture(bs.enqueue_bf16, dev)
                for _ in range(3):
                    gbb.replay()
                bb_ms = time_graph(torch, gbb, max(5, args.steps // 20), stream)
                entry["bf16_ms_per_step"] = bb_ms
                entry["speedup_vs_bf16"] = bb_ms / b_ms
                del gbb
            log(f"batched M={Mb}: {b_ms:.3f} ms/step, W8A8 GEMMs {b_ach:.0f} GB/s; "
                f"bf16 {entry.get('bf16_ms_per_step', float('nan')):.3f} ms")
            batched[f"M{Mb}"] = entry
            del bs
            torch.cuda.empty_cache()

    # ---- e2e through the public API from host buffers: one graph per step
    # that copies the step's inputs in (the drafts and the first layer's
    # first, in one copy; the rest on a parallel branch while the first layer
    # runs), runs the step and copies the accepted lengths and tokens out (one
    # copy); the host waits for them every step
    host_in, host_d = stack.pinned_host_inputs()
    out_len, out_tok = stack.pinned_host_results()
    e2e_graph, h2d, d2h = stack.capture_from_host(host_in, host_d, out_len, out_tok)
    for _ in range(3):
        e2e_graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_len, ref_len.cpu()) and torch.equal(out_tok, stack.out_tokens.cpu()), \
        "the step from host buffers disagrees with the device-timed step"
    n_e2e = max(10, args.steps // 4)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_graph.replay()
        torch.cuda.current_stream().synchronize()      # the host reads the step's result
        _ = int(out_len[0])
    e2e_s = (time.perf_counter() - t0) / n_e2e
    del e2e_graph
    e2e = {"value": world * stack.M / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3}

    cpu = None
    # ---- chained decoder layers (residual stream, RMSNorm, attention over a
    # 2048-position KV cache, SwiGLU between the linears): the same weights, a
    # real layer chain; and the same chain with the o projection on its
    # seeded input instead of attention, for the attention's share
    layer_chain = None
    if rank == 0:
        chain = {}
        for label, cl in (("no_attention", None), ("attention", 2048)):
            stack.prepare_chain(cache_len=cl)
            chain_graph = stack.capture_chain()
            for _ in range(3):
                chain_graph.replay()
            torch.cuda.synchronize()
            chain[label] = time_graph(torch, chain_graph, max(20, args.steps // 5), stream)
            del chain_graph
            log(f"layer chain ({label}) {chain[label]:.4f} ms/step")
        chain_ms = chain["attention"]
        layer_chain = {"ms_per_step": chain_ms, "tokens_per_s": stack.M / (chain_ms * 1e-3),
                       "weight_stream_gbs": stack.weight_bytes() / (chain_ms * 1e-3) / 1e9,
                       "kv_cache_positions": 2048, "launches_per_step": 10 * stack.layers + 3,
                       "ms_per_step_without_attention": chain["no_attention"],
                       "attention_share": (chain_ms - chain["no_attention"]) / chain_ms,
                       "path": "per layer: qv_rmsnorm_quant (residual add + RMSNorm + quant) -> qkv (bf16) -> "
                               "qv_attention_verify over the layer's bf16 KV cache (2048 positions, 32/8 heads, "
                               "D = 128) and the step's own keys -> qv_quantize_act -> o -> qv_rmsnorm_quant -> "
                               "qv_w8a8_swiglu (gate|up with SiLU(gate)*up in the epilogue) -> qv_quantize_act -> "
                               "down (bf16); final qv_rmsnorm_quant -> LM head argmax -> accept; one CUDA graph"}
        del stack.k_cache, stack.v_cache
        torch.cuda.empty_cache()

    # ---- T > 0: LM-head logits and lossless rejection sampling
    sampling = None
    if rank == 0:
        stack.prepare_sampling(temperature=0.8)
        sg = stack.capture_sampled()
        for _ in range(3):
            sg.replay()
        torch.cuda.synchronize()
        s_ms = time_graph(torch, sg, max(20, args.steps // 5), stream)
        log(f"T>0 sampling step {s_ms:.4f} ms/step (mean accepted length "
            f"{float(stack.accept_len.float().mean()):.2f})")
        sampling = {"ms_per_step": s_ms, "tokens_per_s": stack.M / (s_ms * 1e-3), "temperature": 0.8,
                    "launches_per_step": stack.launches_per_step() + 1,
                    "path": "per projection qv_quantize_act + qv_w8a8_linear; LM head qv_w8a8_linear "
                            "(fp32 logits) + qv_spec_sample (lossless rejection sampling against seeded "
                            "draft distributions); one CUDA graph"}

    # ---- logit fidelity of the quantized verifier against the BF16 one on
    # the step's final hidden states (synthetic weights): KL(p_bf16 || p_q)
    # per row and top-1 agreement
    fidelity = None

    def fid(ref, logits):
        kl = torch.empty(ref.shape[0], device=dev)
        ta = torch.empty(ref.shape[0], dtype=torch.int32, device=dev)
        tb = torch.empty(ref.shape[0], dtype=torch.int32, device=dev)
        qv.qv_logit_fidelity(ref, logits, kl, ta, tb)
        torch.cuda.synchronize()
        out = {"kl_mean": float(kl.double().mean()), "kl_max": float(kl.max()),
               "top1_agree": float((ta == tb).float().mean())}
        # the diagnostic's own latency: back-to-back calls on L2-resident logits
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            qv.qv_logit_fidelity(ref, logits, kl, ta, tb)
        e0.record()
        for _ in range(50):
            qv.qv_logit_fidelity(ref, logits, kl, ta, tb)
        e1.record()
        torch.cuda.synchronize()
        out["us_per_call"] = e0.elapsed_time(e1) * 1e3 / 50
        return out
    if rank == 0 and comparator is not None and sampling is not None:
        fidelity = {"w8a8_vs_bf16": fid(stack.logits_bf16, stack.logits),
                    "note": "KL(softmax(BF16 logits) || softmax(quantized logits)) in nats over the LM-head "
                            "logits of the step's M rows (synthetic weights and hidden states), and the fraction "
                            "of rows whose top-1 tokens agree; qv_logit_fidelity"}
        log(f"fidelity W8A8 vs BF16: {fidelity['w8a8_vs_bf16']}")

    # ---- a 16-node draft tree (root, 3 children, 2 grandchildren each, one
    # great-grandchild each) verified in one step, greedy
    tree = None
    if rank == 0:
        n_tree = 16
        parent = torch.tensor([[-1, 0, 0, 0, 1, 1, 2, 2, 3, 3, 4, 5, 6, 7, 8, 9]], dtype=torch.int32)
        tstack = VerifyStack(B=1, gamma=n_tree - 1, seed=7 + rank, layers=args.layers, device=str(dev))
        tstack.prepare_tree(parent, torch.zeros(1, n_tree, dtype=torch.int32))
        tstack.enqueue_tree()
        torch.cuda.synchronize()
        tv = tstack.tokens.cpu()
        draft = torch.randint(0, tstack.V, (1, n_tree), generator=torch.Generator().manual_seed(5),
                              dtype=torch.int32)
        for node in (1, 4, 10):                 # the path 0 -> 1 -> 4 -> 10 matches the verifier
            draft[0, node] = tv[int(parent[0, node])]
        tstack.prepare_tree(parent, draft)
        tg = tstack.capture_tree()
        for _ in range(3):
            tg.replay()
        torch.cuda.synchronize()
        t_ms = time_graph(torch, tg, max(20, args.steps // 5), stream)
        log(f"16-node tree step {t_ms:.4f} ms/step, accepted length {int(tstack.tree_len[0])}")
        tree = {"nodes": n_tree, "ms_per_step": t_ms, "accept_len": int(tstack.tree_len[0]),
                "verified_nodes_per_s": n_tree / (t_ms * 1e-3),
                "path": "layers over the 16 tree rows (qv_quantize_act + qv_w8a8_linear), LM-head argmax, "
                        "qv_tree_accept; one CUDA graph"}
        del tg, tstack
        torch.cuda.empty_cache()

    # ---- attention over a short KV cache (qv_attention_verify) for the
    # step's verify tokens, every layer, at a 2048-position cache
    attention = None
    if rank == 0:
        try:
            D_ = 128
            Hq_, Hkv_ = stack.model.get("q", stack.model["hidden"]) // D_, stack.model["kv"] // D_
            T_, L_ = stack.gamma + 1, 2048
            ga = torch.Generator(device=dev).manual_seed(11)
            qkv_a = torch.randn(T_, (Hq_ + 2 * Hkv_) * D_, device=dev, generator=ga).to(torch.bfloat16)
            kcs = [torch.randn(1, L_, Hkv_, D_, device=dev, generator=ga).to(torch.bfloat16) for _ in range(stack.layers)]
            vcs = [torch.randn(1, L_, Hkv_, D_, device=dev, generator=ga).to(torch.bfloat16) for _ in range(stack.layers)]
            ln_a = torch.full((1,), L_, dtype=torch.int32, device=dev)
            ws_a = torch.empty(qv.qv_attention_workspace_bytes(1, T_, Hq_, Hkv_, D_, L_), dtype=torch.uint8, device=dev)
            out_a = torch.empty(T_, Hq_ * D_, device=dev)
            sc = float(1.0 / (D_ ** 0.5))

            def attn_seq(s):
                for l in range(stack.layers):
                    qv.qv_attention_verify(qkv_a, kcs[l], vcs[l], ln_a, T_, Hq_, Hkv_, sc, out_a, ws_a, stream=s)
            ga_graph = VerifyStack._capture(attn_seq, dev)
            for _ in range(3):
                ga_graph.replay()
            torch.cuda.synchronize()
            a_ms = time_graph(torch, ga_graph, 10, stream)
            kv_b = 2 * L_ * Hkv_ * D_ * 2
            attention = {"context": L_, "tokens": T_, "heads": [Hq_, Hkv_, D_], "us_per_layer": a_ms * 1e3 / stack.layers,
                         "us_per_step": a_ms * 1e3, "kv_bytes_per_layer": kv_b,
                         "kv_gbs": kv_b * stack.layers / (a_ms * 1e-3) / 1e9,
                         "note": "the attention alone, 36 layers back to back (the chained step runs the same "
                                 "per layer; the headline step has no attention); 2048-position bf16 cache, "
                                 "qv_attention_verify (one cluster launch per layer), one CUDA graph"}
            log(f"attention at L={L_}: {attention['us_per_layer']:.2f} us per layer")
            del ga_graph, kcs, vcs
            torch.cuda.empty_cache()
        except Exception as exc:      # a measurement of an extra row must not lose the bench line
            log(f"attention timing skipped: {exc}")

    # ---- W4A8: the same step with packed int4 weights (half the weight
    # bytes), and its streaming GEMM over the step's 144 projections
    w4a8 = None
    if rank == 0:
        w4s = VerifyStack(layers=args.layers, B=1, gamma=4, seed=1234 + rank, device=str(dev), wbits=4)
        w4s.enqueue_two_call()
        torch.cuda.synchronize()
        w4s.drafts.copy_(synth.geometric_drafts(w4s.tokens.view(w4s.B, w4s.gamma + 1).cpu(), w4s.V, 0.7,
                                                seed=99 + rank))
        g4 = w4s.capture_two_call()
        for _ in range(3):
            g4.replay()
        torch.cuda.synchronize()
        w4_ms = time_graph(torch, g4, max(20, args.steps // 5), stream)
        del g4
        xq4 = []
        for l in range(w4s.layers):
            for p, (name, K, N) in enumerate(w4s.phases):
                xq = torch.empty(M, K, dtype=torch.int8, device=dev)
                sxp = torch.empty(M, device=dev)
                qv.qv_quantize_act(w4s.inputs[l][p], xq, sxp)
                xq4.append((xq, sxp))
        torch.cuda.synchronize()

        def lin4_seq(s):
            j = 0
            for l in range(w4s.layers):
                for p, (name, K, N) in enumerate(w4s.phases):
                    wq, sw = w4s.weights[l][p]
                    qv.qv_w4a8_linear(xq4[j][0], xq4[j][1], wq, sw, w4s.y[: M * N].view(M, N), w4s.ws, stream=s)
                    j += 1
        g4l = VerifyStack._capture(lin4_seq, dev)
        lin4_ms = time_graph(torch, g4l, args.kernel_reps, stream)
        lin4_bytes = w4s.linear_launch_bytes(fused_act=False)
        ach4 = sum(lin4_bytes) / (lin4_ms * 1e-3) / 1e9
        log(f"W4A8 step {w4_ms:.4f} ms/step; w4a8 linear kernel {ach4:.1f} GB/s = {ach4 / peak:.3f}")
        w4a8 = {"ms_per_step": w4_ms, "tokens_per_s": w4s.M / (w4_ms * 1e-3),
                "weight_bytes_per_step": w4s.weight_bytes(),
                "weight_stream_gbs": w4s.weight_bytes() / (w4_ms * 1e-3) / 1e9,
                "speedup_vs_w8a8": ms / w4_ms,
                "speedup_vs_bf16": (comparator["bf16_ms_per_step"] / w4_ms) if comparator else None,
                "accept_len": int(w4s.accept_len[0]),
                "linear_kernel": {"kernel": "w8a8_stream_kernel<1, Linear, W4> (int4 codes unpacked to int8 "
                                            "mma.sync operands, qv_w4a8_linear)",
                                  "achieved": ach4, "frac": ach4 / peak, "unit": "GB/s",
                                  "bytes_per_launch": sum(lin4_bytes) / len(lin4_bytes),
                                  "launch_ms_mean": lin4_ms / len(lin4_bytes),
                                  "timing": "144 launches of the step's projections back to back in one CUDA graph"},
                "path": "per projection qv_quantize_act + qv_w4a8_linear, qv_quantize_act + "
                        "qv_w4a8_lm_head_argmax, qv_accept; one CUDA graph"}
        if fidelity is not None:
            h = w4s.model["hidden"]
            xqf = torch.empty(M, h, dtype=torch.int8, device=dev)
            sxf = torch.empty(M, device=dev)
            qv.qv_quantize_act(w4s.h_final, xqf, sxf)
            logits4 = torch.empty(M, w4s.V, device=dev)
            qv.qv_w4a8_linear(xqf, sxf, w4s.lm_wq, w4s.lm_sw, logits4, w4s.ws)
            fidelity["w4a8_vs_bf16"] = fid(stack.logits_bf16, logits4)
            log(f"fidelity W4A8 vs BF16: {fidelity['w4a8_vs_bf16']}")
            del logits4
        del g4l, xq4, w4s
        torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8 x int8 -> int32, fp32 dequant", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": stack.M, "B": stack.B, "gamma": stack.gamma,
                       "layers": stack.layers, "weight_bytes_per_step": stack.weight_bytes(),
                       "algorithmic_bytes_per_step": alg_bytes,
                       "weight_stream_gbs": stack.weight_bytes() / (ms_max * 1e-3) / 1e9,
                       "weight_stream_frac_of_peak": stack.weight_bytes() / (ms_max * 1e-3) / 1e9 / peak,
                       "l2": "inputs larger than L2: 7.57 GB of weights per step vs 129 MB L2, no flush",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "path": path,
                       "timing": "CUDA graph replay of whole steps, CUDA events on the launching stream"},
            "roofline": roofline,
            "linear_kernel": linear_kernel,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches * args.steps,
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "comparator": comparator,
            "paths_ms_per_step": paths_ms,
            "step_ms_distribution": step_dist,
            "layer_chain": layer_chain,
            "sampling_t_gt_0": sampling,
            "tree_verify": tree,
            "w4a8": w4a8,
            "logit_fidelity": fidelity,
            "attention_kv_cache": attention,
            "batched_verify": batched,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
