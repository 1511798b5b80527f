"""W8A8 verify pass over a decoder-layer stack, built from the libqv calls.

A verify step of M = B*(gamma+1) tokens runs, for every layer, the four
quantize -> W8A8 linear phases of a decoder layer (q|k|v, o, gate|up, down),
then the LM head fused with the greedy argmax and the acceptance of the
longest matching draft prefix:

    per layer: qv_quantize_act(h)    -> qv_w8a8_linear(Wqkv)      N = q+2kv
               qv_quantize_act(attn) -> qv_w8a8_linear(Wo)
               qv_quantize_act(h2)   -> qv_w8a8_linear(Wgate|up)  N = 2*ffn
               qv_quantize_act(act)  -> qv_w8a8_linear(Wdown)
    then       qv_quantize_act(h_final) -> qv_lm_head_argmax -> qv_accept

(Quasar, gist.science/ja summary, section 2.2 item 3 for the quantized
linears; gist.science/it summary, section 2 item 3 for the acceptance test.)
Attention, normalisation and the activation function sit between these
phases in a real model; they are not part of the quantized path and are not
run: each phase reads its own seeded synthetic input of the right shape.
q|k|v and gate|up share their input in a decoder layer, so their weights are
stored concatenated along the output channels (each output column is computed
independently, so the results are those of the separate projections).

Weights are generated on the device (seeded), quantized once with
qv_quantize_weight and kept resident in HBM; only the int8 codes and fp32
scales are kept (and the bf16 originals when the comparator is wanted). One
step is captured into a CUDA graph; consecutive kernels overlap through
programmatic dependent launch.
"""
from __future__ import annotations

import torch

from . import qv, synth


class VerifyStack:
    def __init__(self, model: dict = synth.QWEN3_8B, layers: int | None = None, B: int = 1,
                 gamma: int = 4, seed: int = 0, device: str = "cuda", keep_bf16: bool = False,
                 y_dtype=torch.float32, wbits: int = 8, share_weights: "VerifyStack | None" = None):
        """share_weights: another stack of the same model whose resident
        weights (int8 codes, scales, bf16 originals) this one uses, so a
        stack for another batch shape costs only its inputs and buffers."""
        assert wbits in (8, 4), "int8 or packed int4 weights"
        self.wbits = wbits
        self.model = model
        self.layers = model["layers"] if layers is None else layers
        self.B, self.gamma = B, gamma
        self.M = B * (gamma + 1)
        self.V = model["vocab"]
        self.device = torch.device(device)
        self.seed = seed
        self.y_dtype = y_dtype
        h = model["hidden"]
        q = model.get("q", h)
        kv = model["kv"]
        ffn = model["ffn"]
        # (name, K, N) of the four phases of a layer
        self.phases = [("qkv", h, q + 2 * kv), ("o", q, h), ("gate_up", h, 2 * ffn), ("down", ffn, h)]
        self.weights = []      # per layer: list of (wq, sw) per phase
        self.weights_bf16 = [] if keep_bf16 else None
        self.inputs = []       # per layer: list of bf16 [M, K] per phase
        dev = self.device
        src = share_weights
        if src is not None:
            assert src.model == model and src.layers == self.layers and src.wbits == wbits
            keep_bf16 = keep_bf16 and src.weights_bf16 is not None
            self.weights_bf16 = src.weights_bf16 if keep_bf16 else None
        for l in range(self.layers):
            lw, lb, li = [], [], []
            for p_, (name, K, N) in enumerate(self.phases):
                li_x = synth.activations(self.M, K, synth.subseed(seed, "x", l, name), device=dev)
                if src is not None:
                    lw.append(src.weights[l][p_])
                    li.append(li_x)
                    continue
                w = synth.weights(N, K, synth.subseed(seed, "w", l, name), device=dev)
                if name == "gate_up" and (N // 2) % 64 == 0:
                    # gate and up rows interleaved by 64 (qv_w8a8_swiglu's layout);
                    # the other paths only need some row order
                    w = qv.interleave_gate_up(w)
                wq, sw = self._quantize_weight(w)
                lw.append((wq, sw))
                if keep_bf16:
                    lb.append(w)
                else:
                    del w
                li.append(li_x)
            self.weights.append(lw)
            if keep_bf16 and src is None:
                self.weights_bf16.append(lb)
            self.inputs.append(li)
        if src is not None:
            self.lm_wq, self.lm_sw = src.lm_wq, src.lm_sw
            self.lm_bf16 = src.lm_bf16 if keep_bf16 else None
        else:
            wl = synth.weights(self.V, h, synth.subseed(seed, "w", "lm_head"), device=dev)
            self.lm_wq, self.lm_sw = self._quantize_weight(wl)
            self.lm_bf16 = wl if keep_bf16 else None
            del wl
        self.h_final = synth.activations(self.M, h, synth.subseed(seed, "x", "final"), device=dev)
        # Every per-step input becomes a view into one contiguous byte buffer:
        # the drafts (int32, padded to 256 bytes), then every activation input
        # (each [M, K] bf16 slice starts 16-byte aligned because K is a
        # multiple of 16), so a step's inputs come from host memory in few
        # copies.
        flat = [x for li in self.inputs for x in li] + [self.h_final]
        self._draft_pad = (B * max(gamma, 0) * 4 + 255) // 256 * 256
        n_act = sum(x.numel() for x in flat)
        self.io_in = torch.zeros(self._draft_pad + n_act * flat[0].element_size(), dtype=torch.uint8, device=dev)
        self.in_buf = self.io_in[self._draft_pad:].view(flat[0].dtype)
        views, off = [], 0
        for x in flat:
            v = self.in_buf[off: off + x.numel()].view(x.shape)
            v.copy_(x)
            views.append(v)
            off += x.numel()
        k = 0
        for li in self.inputs:
            for p in range(len(li)):
                li[p] = views[k]
                k += 1
        self.h_final = views[k]
        del flat
        self.drafts = self.io_in[: B * max(gamma, 0) * 4].view(torch.int32).view(B, max(gamma, 0))

        kmax = max(K for (_, K, _) in self.phases)
        nmax = max(N for (_, _, N) in self.phases)
        self.xq = torch.empty(self.M, max(kmax, h), dtype=torch.int8, device=dev)
        self.sx = torch.empty(self.M, dtype=torch.float32, device=dev)
        self.y = torch.empty(self.M * nmax, dtype=y_dtype, device=dev)
        self.tokens = torch.empty(self.M, dtype=torch.int32, device=dev)
        self.max_logit = torch.empty(self.M, dtype=torch.float32, device=dev)
        # the step's results, also one buffer: accepted lengths, then tokens
        self.io_out = torch.empty(B * (gamma + 2), dtype=torch.int32, device=dev)
        self.accept_len = self.io_out[:B]
        self.out_tokens = self.io_out[B:].view(B, gamma + 1)
        ws_bytes = max([qv.qv_workspace_bytes(qv.QV_OP_LINEAR, self.M, K, N) for (_, K, N) in self.phases]
                       + [qv.qv_workspace_bytes(qv.QV_OP_LM_HEAD, self.M, h, self.V)])
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        # shared by every *_act call of a step: the largest GEMM part plus the
        # largest code part (the codes go to the end of the buffer)
        al = lambda v, a: (v + a - 1) // a * a
        gemm = max([qv.qv_workspace_bytes(qv.QV_OP_LINEAR, self.M, K, N) for (_, K, N) in self.phases]
                   + [qv.qv_workspace_bytes(qv.QV_OP_LM_HEAD, self.M, h, self.V)])
        codes = max(al(self.M * K, 16) + al(4 * self.M, 16) for K in [K for (_, K, _) in self.phases] + [h])
        self.ws_act = torch.zeros(al(gemm, 256) + al(codes, 256), dtype=torch.uint8, device=dev)
        self.graph = None
        torch.cuda.synchronize(dev)

    def _quantize_weight(self, w):
        """int8 codes [N, K] (qv_quantize_weight) or packed int4 codes
        [N, K/2] (qv_quantize_weight_w4), and the fp32 channel scales."""
        N, K = w.shape
        sw = torch.empty(N, dtype=torch.float32, device=w.device)
        if self.wbits == 4:
            wq = torch.empty(N, K // 2, dtype=torch.uint8, device=w.device)
            qv.qv_quantize_weight_w4(w, wq, sw)
        else:
            wq = torch.empty(N, K, dtype=torch.int8, device=w.device)
            qv.qv_quantize_weight(w, wq, sw)
        return wq, sw

    def _linear(self, xq, sx, wq, sw, y, ws, stream=None):
        if self.wbits == 4:
            qv.qv_w4a8_linear(xq, sx, wq, sw, y, ws, stream=stream)
        else:
            qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws, stream=stream)

    def _lm_head(self, xq, ws, stream=None):
        fn = qv.qv_w4a8_lm_head_argmax if self.wbits == 4 else qv.qv_lm_head_argmax
        fn(xq, self.sx, self.lm_wq, self.lm_sw, self.tokens, ws, max_logit=self.max_logit, stream=stream)

    def _w8_only(self, what):
        if self.wbits != 8:
            raise NotImplementedError(f"{what} runs int8 weights only")

    # ------------------------------------------------------------------ sizes
    def _wb(self, N, K) -> int:
        return N * K * self.wbits // 8

    def weight_bytes(self) -> int:
        """Weight bytes streamed by one step (linears + LM head)."""
        per_layer = sum(self._wb(N, K) for (_, K, N) in self.phases)
        return per_layer * self.layers + self._wb(self.V, self.model["hidden"])

    def algorithmic_bytes(self) -> int:
        """All bytes one step must move at least: int8 weights and fp32
        channel scales, the bf16 activations read once, the fp32/bf16
        outputs written, LM-head and acceptance I/O. (The int8 codes and
        token scales need not reach HBM: the fused kernels keep them on chip.)"""
        M = self.M
        yb = 4 if self.y_dtype == torch.float32 else 2
        total = 0
        for (_, K, N) in self.phases:
            total += self._wb(N, K) + 4 * N + M * K * 2 + M * N * yb
        total *= self.layers
        h = self.model["hidden"]
        total += self._wb(self.V, h) + 4 * self.V + M * h * 2 + 4 * M + 4 * M   # LM head: weights, x, tokens, max
        total += 4 * M + 4 * self.B * self.gamma + 4 * self.B + 4 * self.B * (self.gamma + 1)  # accept I/O
        return total

    def linear_launch_bytes(self, fused_act: bool = True):
        """Algorithmic bytes of each projection GEMM launch of a step, in
        order: weights, channel scales and outputs, plus the bf16 activations
        (qv_w8a8_linear_act) or their int8 codes and token scales
        (qv_w8a8_linear)."""
        M = self.M
        yb = 4 if self.y_dtype == torch.float32 else 2
        xb = (lambda K: M * K * 2) if fused_act else (lambda K: M * K + 4 * M)
        one = [self._wb(N, K) + 4 * N + xb(K) + M * N * yb for (_, K, N) in self.phases]
        return one * self.layers

    def _xq(self, K):
        return self.xq.view(-1)[: self.M * K].view(self.M, K)

    # ------------------------------------------------------------------ step
    def enqueue(self, stream=None):
        """Enqueue one verify step on `stream` (current stream if None): one
        qv_w8a8_linear_act per projection (quantization kernel + streaming
        GEMM), qv_lm_head_argmax_act, qv_accept."""
        self._w8_only("the fused-quantization path")
        self._enqueue_layers(0, self.layers, stream)
        self._enqueue_head_accept(stream)

    def _enqueue_layers(self, l0, l1, stream):
        M = self.M
        for l in range(l0, l1):
            for p, (name, K, N) in enumerate(self.phases):
                wq, sw = self.weights[l][p]
                qv.qv_w8a8_linear_act(self.inputs[l][p], wq, sw, self.y[: M * N].view(M, N), self.ws_act,
                                      stream=stream)

    def _enqueue_head_accept(self, stream):
        qv.qv_lm_head_argmax_act(self.h_final, self.lm_wq, self.lm_sw, self.tokens, self.ws_act,
                                 max_logit=self.max_logit, stream=stream)
        qv.qv_accept(self.tokens.view(self.B, self.gamma + 1), self.drafts if self.gamma > 0 else None,
                     self.accept_len, self.out_tokens, stream=stream)

    def enqueue_two_call(self, stream=None):
        """The same step with separate calls: qv_quantize_act then
        qv_w8a8_linear per projection, qv_quantize_act then
        qv_lm_head_argmax, qv_accept (bit-identical results)."""
        M = self.M
        ws = self.ws
        for l in range(self.layers):
            for p, (name, K, N) in enumerate(self.phases):
                xq = self._xq(K)
                qv.qv_quantize_act(self.inputs[l][p], xq, self.sx, stream=stream)
                wq, sw = self.weights[l][p]
                self._linear(xq, self.sx, wq, sw, self.y[: M * N].view(M, N), ws, stream=stream)
        xq = self._xq(self.model["hidden"])
        qv.qv_quantize_act(self.h_final, xq, self.sx, stream=stream)
        self._lm_head(xq, ws, stream=stream)
        qv.qv_accept(self.tokens.view(self.B, self.gamma + 1), self.drafts if self.gamma > 0 else None,
                     self.accept_len, self.out_tokens, stream=stream)

    # ------------------------------------------------------------------ chained layers
    def prepare_chain(self, eps: float = 1e-6, cache_len: int | None = None, head_dim: int = 128):
        """Norm weights, the step's input residual stream and the output
        buffers of the chained step (enqueue_chain). With cache_len, every
        layer also gets a seeded bf16 KV cache of cache_len positions per
        sequence ([B, cache_len, Hkv, head_dim], N(0, 1)) and the chain runs
        attention over it between the qkv and o projections; without it the
        o projection takes the layer's seeded input."""
        self._w8_only("the layer chain")
        h, M, F = self.model["hidden"], self.M, self.model["ffn"]
        dev = self.device
        self.eps = eps
        self.norm_w = [(synth.norm_weights(h, synth.subseed(self.seed, "g", l, "attn"), device=dev),
                        synth.norm_weights(h, synth.subseed(self.seed, "g", l, "mlp"), device=dev))
                       for l in range(self.layers)]
        self.norm_final = synth.norm_weights(h, synth.subseed(self.seed, "g", "final"), device=dev)
        self.h0 = synth.activations(M, h, synth.subseed(self.seed, "x", "embed"), device=dev)
        self.h_res = torch.empty_like(self.h0)
        self.y_qkv = torch.empty(M, self.phases[0][2], dtype=torch.bfloat16, device=dev)
        self.y_o = torch.empty(M, h, dtype=torch.bfloat16, device=dev)
        self.a_glu = torch.empty(M, F, dtype=torch.float32, device=dev)
        self.y_down = torch.empty(M, h, dtype=torch.bfloat16, device=dev)
        self.cache_len = cache_len
        if cache_len is not None:
            q = self.model.get("q", h)
            kv = self.model["kv"]
            assert q % head_dim == 0 and kv % head_dim == 0
            self.head_dim, self.Hq, self.Hkv = head_dim, q // head_dim, kv // head_dim
            shape = (self.B, cache_len, self.Hkv, head_dim)
            self.k_cache = [synth.activations(self.B * cache_len, self.Hkv * head_dim,
                                              synth.subseed(self.seed, "k_cache", l), device=dev,
                                              outlier_frac=0.0).view(shape) for l in range(self.layers)]
            self.v_cache = [synth.activations(self.B * cache_len, self.Hkv * head_dim,
                                              synth.subseed(self.seed, "v_cache", l), device=dev,
                                              outlier_frac=0.0).view(shape) for l in range(self.layers)]
            self.cache_lens = torch.full((self.B,), cache_len, dtype=torch.int32, device=dev)
            T = self.gamma + 1
            self.ws_attn = torch.empty(qv.qv_attention_workspace_bytes(self.B, T, self.Hq, self.Hkv, head_dim,
                                                                       cache_len), dtype=torch.uint8, device=dev)
            # one output buffer per layer (kept for inspection; the chain reads each once)
            self.attn_out = [torch.empty(M, self.Hq * head_dim, dtype=torch.float32, device=dev)
                             for _ in range(self.layers)]

    def enqueue_chain(self, stream=None):
        """One verify step through chained decoder layers: the bf16 residual
        stream h runs through every layer, with the non-linear steps between
        the quantized linears fused with the next linear's quantization
        (gist.science/ja summary, section 2.2 item 3):
          attention block: x = RMSNorm(h += down_prev) -> qkv (bf16); with a
            KV cache, causal grouped-query attention of the verify tokens
            over the cache and their own keys (qv_attention_verify, fp32),
            its per-token quantization -> o; without one, o takes the
            layer's seeded input; h += o's bf16 output, next block;
          MLP block: x = RMSNorm(h) -> gate|up with SiLU(gate)*up in its
            epilogue (fp32) -> per-token quantization -> down (bf16 output,
            added to h by the next RMSNorm);
          head: x = RMSNorm(h += down_last) -> LM head argmax -> acceptance.
        Eight launches per layer (ten with attention), plus the final three."""
        M, h, F = self.M, self.model["hidden"], self.model["ffn"]
        ws = self.ws
        cur = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(cur):
            self.h_res.copy_(self.h0)
        attn = getattr(self, "cache_len", None) is not None
        for l in range(self.layers):
            g1, g2 = self.norm_w[l]
            xq = self._xq(h)
            qv.qv_rmsnorm_quant(self.h_res, g1, xq, self.sx, delta=None if l == 0 else self.y_down,
                                eps=self.eps, stream=stream)
            wq, sw = self.weights[l][0]
            qv.qv_w8a8_linear(xq, self.sx, wq, sw, self.y_qkv, ws, stream=stream)
            xq = self._xq(self.phases[1][1])
            if attn:
                qv.qv_attention_verify(self.y_qkv, self.k_cache[l], self.v_cache[l], self.cache_lens,
                                       self.gamma + 1, self.Hq, self.Hkv, 1.0 / self.head_dim ** 0.5,
                                       self.attn_out[l], self.ws_attn, stream=stream)
                qv.qv_quantize_act(self.attn_out[l], xq, self.sx, stream=stream)
            else:
                qv.qv_quantize_act(self.inputs[l][1], xq, self.sx, stream=stream)
            wq, sw = self.weights[l][1]
            qv.qv_w8a8_linear(xq, self.sx, wq, sw, self.y_o, ws, stream=stream)
            xq = self._xq(h)
            qv.qv_rmsnorm_quant(self.h_res, g2, xq, self.sx, delta=self.y_o, eps=self.eps, stream=stream)
            wq, sw = self.weights[l][2]
            qv.qv_w8a8_swiglu(xq, self.sx, wq, sw, self.a_glu, ws, stream=stream)
            xq = self._xq(F)
            qv.qv_quantize_act(self.a_glu, xq, self.sx, stream=stream)
            wq, sw = self.weights[l][3]
            qv.qv_w8a8_linear(xq, self.sx, wq, sw, self.y_down, ws, stream=stream)
        xq = self._xq(h)
        qv.qv_rmsnorm_quant(self.h_res, self.norm_final, xq, self.sx, delta=self.y_down, eps=self.eps,
                            stream=stream)
        qv.qv_lm_head_argmax(xq, self.sx, self.lm_wq, self.lm_sw, self.tokens, ws,
                             max_logit=self.max_logit, stream=stream)
        qv.qv_accept(self.tokens.view(self.B, self.gamma + 1), self.drafts if self.gamma > 0 else None,
                     self.accept_len, self.out_tokens, stream=stream)

    # ------------------------------------------------------------------ draft tree
    def prepare_tree(self, parent: torch.Tensor, draft: torch.Tensor):
        """A draft tree over the step's M = N rows (B = 1): parent, draft [1, N]
        int32 (node 0 the root); row i's verifier token follows node i."""
        self._w8_only("tree verification")
        assert self.B == 1 and parent.shape == (1, self.M) and draft.shape == (1, self.M)
        dev = self.device
        self.tree_parent = parent.to(dev, torch.int32).contiguous()
        self.tree_draft = draft.to(dev, torch.int32).contiguous()
        self.tree_len = torch.empty(1, dtype=torch.int32, device=dev)
        self.tree_out = torch.empty(1, self.M, dtype=torch.int32, device=dev)
        self.tree_node = torch.empty(1, dtype=torch.int32, device=dev)

    def enqueue_tree(self, stream=None):
        """The verify step of a draft tree: the layers over all N tree rows
        (as enqueue_two_call), the LM head's greedy tokens, then
        qv_tree_accept (the deepest fully matching root path)."""
        M = self.M
        ws = self.ws
        for l in range(self.layers):
            for p, (name, K, N) in enumerate(self.phases):
                xq = self._xq(K)
                qv.qv_quantize_act(self.inputs[l][p], xq, self.sx, stream=stream)
                wq, sw = self.weights[l][p]
                qv.qv_w8a8_linear(xq, self.sx, wq, sw, self.y[: M * N].view(M, N), ws, stream=stream)
        xq = self._xq(self.model["hidden"])
        qv.qv_quantize_act(self.h_final, xq, self.sx, stream=stream)
        qv.qv_lm_head_argmax(xq, self.sx, self.lm_wq, self.lm_sw, self.tokens, ws, stream=stream)
        qv.qv_tree_accept(self.tokens.view(1, M), self.tree_draft, self.tree_parent, self.tree_len,
                          self.tree_out, best_node=self.tree_node, stream=stream)

    def capture_tree(self):
        self.graph_tree = self._capture(self.enqueue_tree, self.device)
        return self.graph_tree

    # ------------------------------------------------------------------ T > 0
    def prepare_sampling(self, temperature: float = 0.8, seed: int = 1234):
        """Buffers of the T > 0 step (enqueue_sampled): fp32 logits, seeded
        draft distributions q (softmax of N(0, 2) logits) and drafts drawn
        from them, the qv_spec_sample workspace."""
        self._w8_only("the sampled step")
        B, g, V, M = self.B, self.gamma, self.V, self.M
        dev = self.device
        self.temperature, self.sample_seed = temperature, seed
        self.logits = torch.empty(M, V, dtype=torch.float32, device=dev)
        gen = torch.Generator(device="cpu").manual_seed(synth.subseed(self.seed, "q"))
        zq = 2.0 * torch.randn(max(B * g, 1), V, generator=gen)
        self.q = torch.softmax(zq, dim=1)[: B * g].contiguous().to(dev)
        self.q_drafts = (torch.multinomial(self.q.cpu().double(), 1, generator=gen).view(B, g).to(torch.int32)
                         .to(dev) if g > 0 else torch.zeros(B, 0, dtype=torch.int32, device=dev))
        self.ws_spec = torch.empty(qv.qv_workspace_bytes(qv.QV_OP_SPEC_SAMPLE, M, 16, V), dtype=torch.uint8,
                                   device=dev)

    def enqueue_sampled(self, stream=None):
        """The verify step at temperature T > 0: the same layers as
        enqueue_two_call, then the LM head's fp32 logits (qv_w8a8_linear) and
        lossless rejection sampling against the draft distributions
        (qv_spec_sample)."""
        M = self.M
        ws = self.ws
        for l in range(self.layers):
            for p, (name, K, N) in enumerate(self.phases):
                xq = self._xq(K)
                qv.qv_quantize_act(self.inputs[l][p], xq, self.sx, stream=stream)
                wq, sw = self.weights[l][p]
                qv.qv_w8a8_linear(xq, self.sx, wq, sw, self.y[: M * N].view(M, N), ws, stream=stream)
        xq = self._xq(self.model["hidden"])
        qv.qv_quantize_act(self.h_final, xq, self.sx, stream=stream)
        qv.qv_w8a8_linear(xq, self.sx, self.lm_wq, self.lm_sw, self.logits, ws, stream=stream)
        qv.qv_spec_sample(self.logits, self.q_drafts, self.q, self.temperature, self.sample_seed,
                          self.accept_len, self.out_tokens, self.ws_spec, stream=stream)

    def capture_sampled(self):
        self.graph_sampled = self._capture(self.enqueue_sampled, self.device)
        return self.graph_sampled

    def capture_chain(self):
        self.graph_chain = self._capture(self.enqueue_chain, self.device)
        return self.graph_chain

    def launches_per_step(self, fused: bool = False) -> int:
        """Kernels one step launches. fused: the persistent qv_verify_stack
        path. Otherwise the per-op path: per projection and for the LM head a
        quantization kernel and one GEMM launch per 80 tokens; plus qv_accept
        (the same count for enqueue and enqueue_two_call)."""
        if fused:
            return (self.layers * len(self.phases) + 1 + 149) // 150
        return (self.layers * len(self.phases) + 1) * (1 + (self.M + 79) // 80) + 1

    # ------------------------------------------------------------------ fused step
    def _fused_descs(self):
        self._w8_only("qv_verify_stack")
        if getattr(self, "_descs", None) is None:
            M = self.M
            descs = []
            for l in range(self.layers):
                for p, (name, K, N) in enumerate(self.phases):
                    wq, sw = self.weights[l][p]
                    descs.append(qv.linear_desc(self.inputs[l][p], wq, sw, y=self.y[: M * N].view(M, N)))
            lm = qv.linear_desc(self.h_final, self.lm_wq, self.lm_sw)
            nmax = max([N for (_, _, N) in self.phases] + [self.V])
            kmax = max([K for (_, K, _) in self.phases] + [self.model["hidden"]])
            self.ws_stack = torch.zeros(qv.qv_workspace_bytes(qv.QV_OP_VERIFY_STACK, M, kmax, nmax),
                                        dtype=torch.uint8, device=self.device)
            self._descs = (descs, lm)
        return self._descs

    def enqueue_fused(self, stream=None):
        """The same step through qv_verify_stack: one persistent launch (per
        150 phases), bit-identical results."""
        descs, lm = self._fused_descs()
        qv.qv_verify_stack(descs, lm, self.M, torch.bfloat16, self.ws_stack, tokens=self.tokens,
                           max_logit=self.max_logit, draft=self.drafts if self.gamma > 0 else None,
                           accept_len=self.accept_len, out_tokens=self.out_tokens, stream=stream)

    def capture_fused(self):
        self.graph_fused = self._capture(self.enqueue_fused, self.device)
        return self.graph_fused

    @staticmethod
    def _capture(fn, device):
        s = torch.cuda.Stream(device=device)
        s.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s):
            fn(s)
        torch.cuda.current_stream(device).wait_stream(s)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream(device))
        return g

    def capture(self):
        """Capture one step into a CUDA graph (after one eager warm-up step)."""
        self.graph = self._capture(self.enqueue, self.device)
        return self.graph

    def capture_two_call(self):
        self.graph_two_call = self._capture(self.enqueue_two_call, self.device)
        return self.graph_two_call

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    # ------------------------------------------------------------------ host API
    def pinned_host_inputs(self):
        """Pinned host copies of the per-step inputs, laid out like the device
        buffer (the drafts, then every activation input): returns the
        activation inputs and the drafts as views of one pinned buffer."""
        io = torch.empty_like(self.io_in, device="cpu").pin_memory()
        io.copy_(self.io_in)
        return io[self._draft_pad:].view(self.in_buf.dtype), io[: self.drafts.numel() * 4].view(
            torch.int32).view(self.drafts.shape)

    def pinned_host_results(self):
        """Pinned host tensors for the step's results (accepted lengths
        [B], output tokens [B, gamma+1]): views of one pinned buffer laid out
        like the device's, so that they come back in one copy."""
        io = torch.empty_like(self.io_out, device="cpu").pin_memory()
        return io[: self.B], io[self.B:].view(self.B, self.gamma + 1)

    @staticmethod
    def _whole(t):
        """The whole storage under a tensor, as bytes."""
        return torch.empty(0, dtype=torch.uint8, device=t.device).set_(t.untyped_storage())

    def _copy_inputs(self, host_inputs, host_drafts, n):
        """Copy the drafts and in_buf[:n] from host memory: one copy when the
        two host tensors lie in one buffer laid out like io_in (as
        pinned_host_inputs makes them), else one copy each."""
        same = (host_inputs.untyped_storage().data_ptr() == host_drafts.untyped_storage().data_ptr()
                and host_drafts.storage_offset() == 0
                and host_inputs.storage_offset() * host_inputs.element_size() == self._draft_pad)
        if same:
            nb = self._draft_pad + n * self.in_buf.element_size()
            self.io_in[:nb].copy_(self._whole(host_inputs)[:nb], non_blocking=True)
        else:
            self.in_buf[:n].copy_(host_inputs[:n], non_blocking=True)
            self.drafts.copy_(host_drafts, non_blocking=True)

    def _copy_results(self, out_len, out_tokens):
        """Copy the accepted lengths and output tokens to host memory: one
        copy when the two host tensors lie in one buffer laid out like
        io_out (as pinned_host_results makes them), else one copy each."""
        same = (out_len.untyped_storage().data_ptr() == out_tokens.untyped_storage().data_ptr()
                and out_len.storage_offset() == 0 and out_tokens.storage_offset() == self.B
                and out_len.dtype == torch.int32 and out_tokens.dtype == torch.int32)
        if same:
            self._whole(out_len)[: self.io_out.numel() * 4].copy_(self.io_out.view(torch.uint8),
                                                                 non_blocking=True)
        else:
            out_len.copy_(self.accept_len, non_blocking=True)
            out_tokens.copy_(self.out_tokens, non_blocking=True)

    def capture_from_host(self, host_inputs, host_drafts, out_len, out_tokens):
        """A CUDA graph of one whole step from host buffers: the drafts and
        the first layer's inputs are copied to the device (one copy when the
        host tensors come from pinned_host_inputs), the first layer runs
        while the other layers' inputs are copied on a parallel branch (which
        the second layer waits for), then the rest of the step, then the
        accepted lengths and tokens are copied back into the pinned host
        tensors (one copy when they come from pinned_host_results). Returns
        (graph, h2d bytes, d2h bytes) per replay."""
        self._w8_only("the fused-quantization path")
        dev = torch.device(self.device)
        n0 = sum(x.numel() for x in self.inputs[0])      # layer 0's inputs lead the buffer

        def body(main):
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(main)
            self._copy_inputs(host_inputs, host_drafts, n0)
            with torch.cuda.stream(side):
                self.in_buf[n0:].copy_(host_inputs[n0:], non_blocking=True)
            self._enqueue_layers(0, 1, main)
            main.wait_stream(side)
            self._enqueue_layers(1, self.layers, main)
            self._enqueue_head_accept(main)
            self._copy_results(out_len, out_tokens)

        g = self._capture(body, dev)
        h2d = host_inputs.numel() * host_inputs.element_size() + host_drafts.numel() * host_drafts.element_size()
        d2h = out_len.numel() * 4 + out_tokens.numel() * 4
        return g, h2d, d2h

    def step_from_host(self, host_inputs, host_drafts, out_len, out_tokens, graph=None):
        """One verify step from host buffers: copy the step's inputs to the
        device, run the captured step, copy the accepted lengths and tokens
        back (into pinned host tensors). Returns bytes copied (h2d, d2h)."""
        self._copy_inputs(host_inputs, host_drafts, self.in_buf.numel())
        h2d = host_inputs.numel() * host_inputs.element_size() + host_drafts.numel() * host_drafts.element_size()
        (graph or self.graph).replay()
        self._copy_results(out_len, out_tokens)
        d2h = out_len.numel() * 4 + out_tokens.numel() * 4
        return h2d, d2h

    # ------------------------------------------------------------------ comparator
    def prepare_bf16(self):
        self._w8_only("the BF16 comparator")
        assert self.weights_bf16 is not None, "construct with keep_bf16=True"
        h = self.model["hidden"]
        ws_bytes = max([qv.qv_workspace_bytes(qv.QV_OP_BF16_LINEAR, self.M, K, N) for (_, K, N) in self.phases]
                       + [qv.qv_workspace_bytes(qv.QV_OP_BF16_LINEAR, self.M, h, self.V)])
        self.ws_bf16 = torch.zeros(ws_bytes, dtype=torch.uint8, device=self.device)
        self.logits_bf16 = torch.empty(self.M, self.V, dtype=torch.float32, device=self.device)
        self.y32 = torch.empty(self.y.numel(), dtype=torch.float32, device=self.device)

    def enqueue_bf16(self, stream=None):
        """The same step with BF16 weights (qv_bf16_linear everywhere, LM-head
        logits written in fp32): the high-precision verifier being replaced."""
        M = self.M
        for l in range(self.layers):
            for p, (name, K, N) in enumerate(self.phases):
                y = self.y32[: M * N].view(M, N)
                qv.qv_bf16_linear(self.inputs[l][p], self.weights_bf16[l][p], y, self.ws_bf16, stream=stream)
        qv.qv_bf16_linear(self.h_final, self.lm_bf16, self.logits_bf16, self.ws_bf16, stream=stream)

    def bf16_weight_bytes(self) -> int:
        return 2 * self.weight_bytes()
