"""One launch of every kernel family of the library, on small inputs, for a
profiler's launch list or a per-kernel capture.

    python -m quantized_verification_gb300.tour [--passes 2]

Each pass makes the same 18 launches in the same order. Before the first
pass the set-up quantizes the weights (one quantize_rows_kernel and one
quantize_weight_w4_kernel launch), so a capture of the second pass filtered
with ``-k`` on the kernels below skips 19 matching launches (``-s 19 -c 18``):

    quantize_rows_kernel                  per-token int8 activation codes, 5 x 4096
    w8a8_stream_kernel<1, Linear>         5 x 4096 -> 24576 (Qwen3-8B gate+up), fp32 out
    w8a8_stream_kernel<1, Linear, W4>     the same shape with packed int4 weights (50.3 MB)
    w8a8_stream_kernel<1, SwiGLU>         the same weights interleaved, SiLU(g)*u fused
    w8a8_tc_kernel<64, Linear>            64 tokens, tcgen05 on widened codes
    w8a8_tc_kernel<80, Linear>            80 tokens, the same
    bf16_stream_kernel<1>                 the BF16 comparator, 5 x 4096 -> 24576
    residual_rmsnorm_quant_kernel         h += d, RMSNorm, int8 codes, 5 x 4096
    swiglu_quant_kernel                   SiLU(g)*u and its int8 codes, 5 x 12288
    spec_{max,sums,decide,chunk,draw}     sampling at T > 0, 1 x (4 + 1) rows x 151936
    tree_accept_kernel                    a 16-node draft tree
    accept_kernel                         greedy acceptance, 1 x 5
    attn_cluster_kernel<128, 8, 3>        attention of 5 tokens over a 2048-position
                                          cache, 32/8 heads, D = 128
    logit_fidelity_kernel                 KL and top-1 of 5 rows x 151936 logits

Inputs are seeded and synthetic and sit on the device before the first
launch; the whole run holds about 0.6 GB.
"""
import argparse

import torch

from . import build, qv, synth

LAUNCHES_PER_PASS = 18


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--passes", type=int, default=2)
    args = ap.parse_args(argv)
    build.build()
    qv.load()
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(0)
    M, K, N, F, V = 5, 4096, 24576, 12288, 151936
    x = synth.activations(M, K, 1, device=dev)
    xq = torch.empty(M, K, dtype=torch.int8, device=dev)
    sx = torch.empty(M, device=dev)
    w = synth.weights(N, K, 2, device=dev)
    wq = torch.empty(N, K, dtype=torch.int8, device=dev)
    sw = torch.empty(N, device=dev)
    qv.qv_quantize_weight(w, wq, sw)
    wq_il, sw_il = qv.interleave_gate_up(wq), qv.interleave_gate_up(sw)
    wq4 = torch.empty(N, K // 2, dtype=torch.uint8, device=dev)
    sw4 = torch.empty(N, device=dev)
    qv.qv_quantize_weight_w4(w, wq4, sw4)
    y = torch.empty(M, N, device=dev)
    a = torch.empty(M, F, device=dev)
    ws = qv.workspace(qv.QV_OP_LINEAR, 80, K, N)
    x64 = torch.randint(-127, 128, (64, K), dtype=torch.int8, device=dev, generator=g)
    sx64 = torch.rand(64, device=dev, generator=g) * 1e-2
    y64 = torch.empty(64, N, device=dev)
    x80 = torch.randint(-127, 128, (80, K), dtype=torch.int8, device=dev, generator=g)
    sx80 = torch.rand(80, device=dev, generator=g) * 1e-2
    y80 = torch.empty(80, N, device=dev)
    wsb = qv.workspace(qv.QV_OP_BF16_LINEAR, M, K, N)
    h = synth.activations(M, K, 3, device=dev)
    d = synth.activations(M, K, 4, device=dev)
    gamma_w = synth.norm_weights(K, 5, device=dev)
    xq2 = torch.empty(M, K, dtype=torch.int8, device=dev)
    sx2 = torch.empty(M, device=dev)
    gu = torch.randn(M, 2 * F, device=dev, generator=g)
    xqf = torch.empty(M, F, dtype=torch.int8, device=dev)
    B, gm = 1, 4
    logits = torch.randn(B * (gm + 1), V, device=dev, generator=g) * 2
    q = torch.softmax(torch.randn(B * gm, V, device=dev, generator=g) * 2, dim=1)
    drafts = torch.randint(0, V, (B, gm), dtype=torch.int32, device=dev, generator=g)
    ln = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, gm + 1, dtype=torch.int32, device=dev)
    wss = torch.empty(qv.qv_workspace_bytes(qv.QV_OP_SPEC_SAMPLE, B * (gm + 1), 16, V), dtype=torch.uint8,
                      device=dev)
    tt = torch.randint(0, 2, (1, 16), dtype=torch.int32, device=dev, generator=g)
    td = torch.randint(0, 2, (1, 16), dtype=torch.int32, device=dev, generator=g)
    tp = torch.tensor([[-1, 0, 0, 0, 1, 1, 2, 2, 3, 3, 4, 5, 6, 7, 8, 9]], dtype=torch.int32, device=dev)
    tl = torch.empty(1, dtype=torch.int32, device=dev)
    to = torch.empty(1, 16, dtype=torch.int32, device=dev)
    vt = torch.randint(0, 100, (B, gm + 1), dtype=torch.int32, device=dev, generator=g)
    Hq, Hkv, D, L = 32, 8, 128, 2048
    qkv = torch.randn(gm + 1, (Hq + 2 * Hkv) * D, device=dev, generator=g).to(torch.bfloat16)
    kc = torch.randn(1, L, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
    vc = torch.randn(1, L, Hkv, D, device=dev, generator=g).to(torch.bfloat16)
    kv_len = torch.full((1,), L, dtype=torch.int32, device=dev)
    wsa = torch.empty(qv.qv_attention_workspace_bytes(1, gm + 1, Hq, Hkv, D, L), dtype=torch.uint8, device=dev)
    attn = torch.empty(gm + 1, Hq * D, device=dev)
    logits2 = logits + torch.randn(logits.shape, device=dev, generator=g) * 0.1
    kl = torch.empty(B * (gm + 1), device=dev)
    t1 = torch.empty(B * (gm + 1), dtype=torch.int32, device=dev)
    t2 = torch.empty(B * (gm + 1), dtype=torch.int32, device=dev)
    for _ in range(args.passes):
        qv.qv_quantize_act(x, xq, sx)
        qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws)
        qv.qv_w4a8_linear(xq, sx, wq4, sw4, y, ws)
        qv.qv_w8a8_swiglu(xq, sx, wq_il, sw_il, a, ws)
        qv.qv_w8a8_linear(x64, sx64, wq, sw, y64, ws)
        qv.qv_w8a8_linear(x80, sx80, wq, sw, y80, ws)
        qv.qv_bf16_linear(x, w, y, wsb)
        qv.qv_rmsnorm_quant(h, gamma_w, xq2, sx2, delta=d)
        qv.qv_swiglu_quant(gu, xqf, sx2)
        qv.qv_spec_sample(logits, drafts, q, 0.8, 7, ln, out, wss)
        qv.qv_tree_accept(tt, td, tp, tl, to)
        qv.qv_accept(vt, drafts, ln, out)
        qv.qv_attention_verify(qkv, kc, vc, kv_len, gm + 1, Hq, Hkv, 1.0 / D ** 0.5, attn, wsa)
        qv.qv_logit_fidelity(logits, logits2, kl, t1, t2)
        torch.cuda.synchronize()
    print(f"ok: {LAUNCHES_PER_PASS} launches per pass, {args.passes} passes")


if __name__ == "__main__":
    main()
