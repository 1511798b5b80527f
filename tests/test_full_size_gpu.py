"""The benched workload at full size against the oracle.

The Qwen3-8B-shaped verify step at M = 5 (batch 1, gamma = 4): q|k|v
4096 -> 6144, o 4096 -> 4096, gate|up 4096 -> 24576, down 12288 -> 4096 per
layer (two layers here; the bench runs 36 of the same shapes), the LM head
4096 -> 151936 fused with the greedy argmax, and the acceptance, through the
per-op paths the bench times (qv_quantize_act + qv_w8a8_linear per
projection, qv_quantize_act + qv_lm_head_argmax, qv_accept; and the one-call
qv_w8a8_linear_act / qv_lm_head_argmax_act), eagerly and as the captured CUDA
graphs. Every output is compared with the oracle element by element:
the weight codes and scales, every projection's fp32 output bit for bit,
the argmax tokens and maximum logits over the whole vocabulary, the accepted
lengths and tokens (Quasar, gist.science/ja summary, section 2.2 item 3;
gist.science/it summary, section 2 item 3: acceptance on the dequantized
logits).
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_bits, np_, rand_codes, rand_scales, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    return _qv


def test_qwen3_8b_step_matches_oracle(qv, oracle):
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    st = VerifyStack(layers=2, B=1, gamma=4, seed=1234, keep_bf16=True)
    M, V, h = st.M, st.V, st.model["hidden"]
    assert [(K, N) for (_, K, N) in st.phases] == [(4096, 6144), (4096, 4096), (4096, 24576), (12288, 4096)]

    # every projection through the per-op calls of the step, one output buffer
    # each: the two calls (qv_quantize_act + qv_w8a8_linear) and the one call
    # (qv_w8a8_linear_act)
    ys, ys_act = [], []
    for l in range(st.layers):
        for p, (name, K, N) in enumerate(st.phases):
            xq = st._xq(K)
            qv.qv_quantize_act(st.inputs[l][p], xq, st.sx)
            y = torch.full((M, N), float("nan"), device="cuda")
            wq, sw = st.weights[l][p]
            qv.qv_w8a8_linear(xq, st.sx, wq, sw, y, st.ws)
            ys.append(y)
            ya = torch.full((M, N), float("nan"), device="cuda")
            qv.qv_w8a8_linear_act(st.inputs[l][p], wq, sw, ya, st.ws_act)
            ys_act.append(ya)
    torch.cuda.synchronize()

    j = 0
    for l in range(st.layers):
        for p, (name, K, N) in enumerate(st.phases):
            wq_r, sw_r = oracle.quantize_rows(bf16_bits(st.weights_bf16[l][p]), bf16=True)
            wq, sw = st.weights[l][p]
            assert np.array_equal(np_(wq), wq_r) and np.array_equal(np_(sw).view(np.uint32), sw_r.view(np.uint32)), \
                f"weight codes of layer {l} {name}"
            xq_r, sx_r = oracle.quantize_rows(bf16_bits(st.inputs[l][p]), bf16=True)
            y_r, _ = oracle.w8a8_linear(xq_r, sx_r, wq_r, sw_r)
            assert np.array_equal(np_(ys[j]).view(np.uint32), y_r.view(np.uint32)), f"layer {l} {name}"
            assert np.array_equal(np_(ys_act[j]).view(np.uint32), y_r.view(np.uint32)), f"layer {l} {name} (act)"
            j += 1

    # the LM head over the whole vocabulary, then drafts that follow the
    # oracle's tokens for a geometric prefix, and the acceptance
    lq_r, ls_r = oracle.quantize_rows(bf16_bits(st.lm_bf16), bf16=True)
    assert np.array_equal(np_(st.lm_wq), lq_r) and np.array_equal(np_(st.lm_sw).view(np.uint32), ls_r.view(np.uint32))
    xh_r, sh_r = oracle.quantize_rows(bf16_bits(st.h_final), bf16=True)
    t_r, m_r = oracle.lm_head_argmax(xh_r, sh_r, lq_r, ls_r)
    drafts = synth.geometric_drafts(torch.from_numpy(t_r).view(1, 5), V, 0.7, seed=99)
    st.drafts.copy_(drafts.cuda())
    l_r, o_r = oracle.accept(t_r, np_(drafts), 1, 4)

    # eager step, then the captured graph the bench replays (twice: the
    # workspace is reused as each call leaves it)
    st.tokens.fill_(-3); st.accept_len.fill_(-3)
    st.enqueue_two_call()
    torch.cuda.synchronize()
    g = st.capture_two_call()
    for rep in range(3):
        if rep:
            st.tokens.fill_(-3); st.max_logit.fill_(float("nan")); st.accept_len.fill_(-3); st.out_tokens.fill_(-3)
            g.replay()
            torch.cuda.synchronize()
        assert np.array_equal(np_(st.tokens), t_r), rep
        assert np.array_equal(np_(st.max_logit).view(np.uint32), m_r.view(np.uint32)), rep
        assert np.array_equal(np_(st.accept_len), l_r) and np.array_equal(np_(st.out_tokens), o_r), rep
        name, K, N = st.phases[-1]
        assert np.array_equal(np_(st.y[: M * N].view(M, N)).view(np.uint32), np_(ys[-1]).view(np.uint32))

    # the same step through the one-call path, eagerly and as a captured graph
    st.tokens.fill_(-3); st.accept_len.fill_(-3)
    st.enqueue()
    torch.cuda.synchronize()
    g = st.capture()
    for rep in range(3):
        if rep:
            st.tokens.fill_(-3); st.max_logit.fill_(float("nan")); st.accept_len.fill_(-3); st.out_tokens.fill_(-3)
            g.replay()
            torch.cuda.synchronize()
        assert np.array_equal(np_(st.tokens), t_r), ("act", rep)
        assert np.array_equal(np_(st.max_logit).view(np.uint32), m_r.view(np.uint32)), ("act", rep)
        assert np.array_equal(np_(st.accept_len), l_r) and np.array_equal(np_(st.out_tokens), o_r), ("act", rep)
        name, K, N = st.phases[-1]
        assert np.array_equal(np_(st.y[: M * N].view(M, N)).view(np.uint32), np_(ys[-1]).view(np.uint32))
    assert qv.qv_device_error() == 0


def test_w8a8_lm_head_full_vocab(qv, oracle):
    """qv_lm_head_argmax at 4096 -> 151936, M = 5, against the oracle over the
    whole vocabulary: tokens and maximum logits bit for bit. Row 0's best
    logit is planted in rows 77777 and 151935 (streamed by different CTAs), so
    the lowest index must win across CTAs; row 1's maximum is negative."""
    M, K, V = 5, 4096, 151936
    xq = rand_codes((M, K), seed=31)
    xq[1] = -xq[1].abs()
    wq = rand_codes((V, K), seed=32, lo=-40, hi=40)
    best = torch.where(xq[0] >= 0, 127, -127).to(torch.int8)
    wq[77777] = best
    wq[151935] = best
    wq_pos = wq.abs()                      # with row 1's codes <= 0, all of row 1's logits are negative
    sx = rand_scales(M, seed=33, lo=1e-3, hi=0.2)
    sw = rand_scales(V, seed=34)
    sw[77777] = sw[151935] = 0.05
    dev = "cuda"
    for w in (wq, wq_pos):
        tok = torch.full((M,), -3, dtype=torch.int32, device=dev)
        mx = torch.full((M,), float("nan"), device=dev)
        ws = qv.workspace(qv.QV_OP_LM_HEAD, M, K, V, dev)
        wd = w.to(dev)
        t_r, m_r = oracle.lm_head_argmax(np_(xq), np_(sx), np_(w), np_(sw))
        for rep in range(2):                  # the workspace is reused as the first call leaves it
            tok.fill_(-3); mx.fill_(float("nan"))
            qv.qv_lm_head_argmax(xq.to(dev), sx.to(dev), wd, sw.to(dev), tok, ws, max_logit=mx)
            torch.cuda.synchronize()
            assert np.array_equal(np_(tok), t_r), rep
            assert np.array_equal(np_(mx).view(np.uint32), m_r.view(np.uint32)), rep
        if w is wq:
            assert t_r[0] == 77777
        else:
            assert m_r[1] < 0
    assert qv.qv_device_error() == 0
