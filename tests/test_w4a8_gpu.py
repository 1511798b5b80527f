"""W4A8 (packed int4 weights against int8 activation codes) against the
oracle, bit for bit: the packed weight bytes and scales of
qv_quantize_weight_w4, the exact integer sums and the dequantized outputs of
qv_w4a8_linear (fp32 and bf16), the SwiGLU epilogue of qv_w4a8_swiglu, and
the tokens and maximum logits of qv_w4a8_lm_head_argmax, from one token to
256, with ragged K and N tails, at the Qwen3-8B projection shapes and at the
largest K."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_bits, np_, rand_codes, rand_scales, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    _qv.load()
    return _qv


def _w4(oracle, N, K, seed):
    """Random int4 codes in [-7, 7] and their packed bytes (packed by the oracle)."""
    q = rand_codes((N, K), seed=seed, lo=-7, hi=7)
    return q, torch.from_numpy(oracle.pack_w4(np_(q)))


def _hard_weights(rng, N, K):
    """Rows whose quotients w / s land on or next to rounding ties of the
    int4 grid, plus an all-zero row and a tiny row."""
    w = rng.normal(0.0, 0.05, (N, K)).astype(np.float32)
    s = np.float32(0.125 / 7)
    w[0, :] = (np.arange(K) % 15 - 7).astype(np.float32) * s        # exact codes
    w[0, 0] = np.float32(0.125)
    w[1, :] = ((np.arange(K) % 14 - 7) + 0.5).astype(np.float32) * np.float32(1 / 64)  # ties
    w[1, 0] = np.float32(7 / 64)
    w[2, :] = 0.0
    w[3, :] *= np.float32(1e-36)
    return w


@pytest.mark.parametrize("N,K,dtype", [(300, 320, torch.float32), (257, 4096, torch.bfloat16),
                                       (64, 32, torch.float32), (1000, 12288, torch.bfloat16)])
def test_quantize_weight_w4(qv, oracle, N, K, dtype):
    rng = np.random.default_rng(N * 7 + K)
    w = _hard_weights(rng, N, K)
    wt = torch.from_numpy(w).to(dtype)
    wq4 = torch.full((N, K // 2), 0x5A, dtype=torch.uint8, device="cuda")
    sw = torch.full((N,), float("nan"), device="cuda")
    qv.qv_quantize_weight_w4(wt.cuda(), wq4, sw)
    torch.cuda.synchronize()
    if dtype == torch.bfloat16:
        q_ref, s_ref = oracle.quantize_rows_w4(bf16_bits(wt), bf16=True)
    else:
        q_ref, s_ref = oracle.quantize_rows_w4(w)
    assert np.array_equal(np_(sw).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(np_(wq4), oracle.pack_w4(q_ref))


LINEAR_CASES = [  # M, K, N
    (5, 4096, 6144), (5, 4096, 4096), (5, 4096, 24576), (5, 12288, 4096),   # Qwen3-8B projections
    (1, 32, 1), (8, 288, 200), (5, 96, 7), (9, 512, 384), (16, 384, 256), (17, 256, 200),
    (32, 640, 256), (33, 256, 129), (40, 4096, 300), (64, 512, 256), (256, 256, 136), (24, 4096, 4096),
]


def _run_linear(qv, xq, sx, wq4, sw, y_dtype=torch.float32):
    M, K = xq.shape
    N = wq4.shape[0]
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    y = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    acc = torch.full((M, N), 12345, dtype=torch.int32, device="cuda")
    qv.qv_w4a8_linear(xq.cuda(), sx.cuda(), wq4.cuda(), sw.cuda(), y, ws, acc_debug=acc)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"
    return y, acc


@pytest.mark.parametrize("M,K,N", LINEAR_CASES)
def test_w4a8_linear(qv, oracle, M, K, N):
    xq = rand_codes((M, K), seed=M * 131 + K)
    _, wq4 = _w4(oracle, N, K, seed=N * 17 + K + 1)
    sx = rand_scales(M, seed=M + 5, lo=1e-3, hi=0.2)
    sw = rand_scales(N, seed=N + 6)
    y, acc = _run_linear(qv, xq, sx, wq4, sw)
    y_ref, acc_ref = oracle.w4a8_linear(np_(xq), np_(sx), np_(wq4), np_(sw))
    assert np.array_equal(np_(acc), acc_ref)
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))
    yb, _ = _run_linear(qv, xq, sx, wq4, sw, y_dtype=torch.bfloat16)
    assert np.array_equal(bf16_bits(yb), oracle.f32_to_bf16(y_ref))


@pytest.mark.parametrize("M", [3, 40])
def test_w4a8_largest_sums(qv, oracle, M):
    """K at its limit with every product at +-127 * 7: the sums reach
    +-118 million (16 times that inside the kernel) and stay exact."""
    K, N = 133120, 256
    xq = torch.full((M, K), 127, dtype=torch.int8)
    xq[1::2] = -127
    q = torch.full((N, K), 7, dtype=torch.int8)
    q[N // 2:] = -7
    q[7, ::3] = -7
    wq4 = torch.from_numpy(oracle.pack_w4(np_(q)))
    sx = rand_scales(M, seed=1)
    sw = rand_scales(N, seed=2)
    y, acc = _run_linear(qv, xq, sx, wq4, sw)
    y_ref, acc_ref = oracle.w4a8_linear(np_(xq), np_(sx), np_(wq4), np_(sw))
    assert int(np.abs(acc_ref).max()) == 127 * 7 * K
    assert np.array_equal(np_(acc), acc_ref)
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))


def test_w4a8_quantize_chain(qv, oracle):
    """bf16 weights and activations through the library's own quantization
    kernels, then the W4A8 linear: equal to the oracle's chain."""
    rng = np.random.default_rng(11)
    M, K, N = 5, 4096, 1536
    x = torch.from_numpy(rng.normal(0, 1, (M, K)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(rng.normal(0, 0.02, (N, K)).astype(np.float32)).to(torch.bfloat16)
    xq = torch.empty(M, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, device="cuda")
    qv.qv_quantize_act(x.cuda(), xq, sx)
    wq4 = torch.empty(N, K // 2, dtype=torch.uint8, device="cuda")
    sw = torch.empty(N, device="cuda")
    qv.qv_quantize_weight_w4(w.cuda(), wq4, sw)
    y, _ = _run_linear(qv, xq, sx, wq4, sw)
    xq_ref, sx_ref = oracle.quantize_rows(bf16_bits(x), bf16=True)
    q_ref, sw_ref = oracle.quantize_rows_w4(bf16_bits(w), bf16=True)
    y_ref, _ = oracle.w4a8_linear(xq_ref, sx_ref, oracle.pack_w4(q_ref), sw_ref)
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))


@pytest.mark.parametrize("M,K,F", [(5, 256, 64), (17, 512, 192), (5, 4096, 1024), (40, 256, 128)])
def test_w4a8_swiglu(qv, oracle, M, K, F):
    """Interleaved int4 gate|up rows with SiLU(gate) * up in the epilogue."""
    xq = rand_codes((M, K), seed=M + 3 * K)
    sx = rand_scales(M, seed=M + 1, lo=1e-3, hi=0.2)
    q, wq4 = _w4(oracle, 2 * F, K, seed=F + 7)
    sw = rand_scales(2 * F, seed=F + 9)
    y, _ = oracle.w4a8_linear(np_(xq), np_(sx), np_(wq4), np_(sw))
    sil = np.array([oracle.silu(float(g)) for g in y[:, :F].reshape(-1)], dtype=np.float32).reshape(M, F)
    a_ref = (sil * y[:, F:]).astype(np.float32)
    wq4_il = qv.interleave_gate_up(wq4.cuda())
    sw_il = qv.interleave_gate_up(sw.cuda())
    a = torch.full((M, F), float("nan"), device="cuda")
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, 2 * F)
    qv.qv_w4a8_swiglu(xq.cuda(), sx.cuda(), wq4_il, sw_il, a, ws)
    torch.cuda.synchronize()
    assert np.array_equal(np_(a).view(np.uint32), a_ref.view(np.uint32))
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"


LM_CASES = [(5, 4096, 3000), (1, 128, 130), (9, 256, 1000), (33, 256, 513), (5, 512, 128 * 160 + 3),
            (64, 4096, 3000)]


def _run_lm(qv, xq, sx, wq4, sw):
    M, K = xq.shape
    V = wq4.shape[0]
    ws = qv.workspace(qv.QV_OP_LM_HEAD, M, K, V)
    tok = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    mx = torch.full((M,), float("nan"), device="cuda")
    qv.qv_w4a8_lm_head_argmax(xq.cuda(), sx.cuda(), wq4.cuda(), sw.cuda(), tok, ws, max_logit=mx)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"
    return np_(tok), np_(mx)


@pytest.mark.parametrize("M,K,V", LM_CASES)
def test_w4a8_lm_head_argmax(qv, oracle, M, K, V):
    xq = rand_codes((M, K), seed=M * 7 + K + V)
    _, wq4 = _w4(oracle, V, K, seed=V * 3 + K)
    sx = rand_scales(M, seed=M + 9, lo=1e-3, hi=0.2)
    sw = rand_scales(V, seed=V + 10)
    tok, mx = _run_lm(qv, xq, sx, wq4, sw)
    t_ref, m_ref = oracle.w4a8_lm_head_argmax(np_(xq), np_(sx), np_(wq4), np_(sw))
    assert np.array_equal(tok, t_ref)
    assert np.array_equal(mx, m_ref)


def test_w4a8_lm_head_ties_lowest_index(qv, oracle):
    M, K, V = 5, 256, 2000
    xq = rand_codes((M, K), seed=1)
    q = rand_codes((V, K), seed=2, lo=-7, hi=7)
    q[400] = torch.where(xq[0] >= 0, 7, -7).to(torch.int8)
    q[1700] = q[400]
    q[1999] = q[400]
    wq4 = torch.from_numpy(oracle.pack_w4(np_(q)))
    sx = rand_scales(M, seed=3)
    sw = torch.full((V,), 0.003)
    tok, mx = _run_lm(qv, xq, sx, wq4, sw)
    t_ref, m_ref = oracle.w4a8_lm_head_argmax(np_(xq), np_(sx), np_(wq4), np_(sw))
    assert t_ref[0] == 400
    assert np.array_equal(tok, t_ref) and np.array_equal(mx, m_ref)


def test_w4a8_lm_head_full_vocab_sampled(qv, oracle):
    """The Qwen3-8B LM head (4096 -> 151936) at M = 5: the token's logit is
    the oracle's logit of that token and equals the reported maximum, and no
    logit of 12000 sampled tokens (plus the token's neighbours) is larger,
    nor equal at a lower index."""
    M, K, V = 5, 4096, 151936
    xq = rand_codes((M, K), seed=21)
    _, wq4 = _w4(oracle, V, K, seed=22)
    sx = rand_scales(M, seed=23, lo=1e-3, hi=0.2)
    sw = rand_scales(V, seed=24)
    tok, mx = _run_lm(qv, xq, sx, wq4, sw)
    rng = np.random.default_rng(25)
    cols = np.unique(np.concatenate([rng.choice(V, 12000, replace=False), tok, np.clip(tok - 1, 0, V - 1),
                                     np.clip(tok + 1, 0, V - 1)]))
    y, _ = oracle.w4a8_linear(np_(xq), np_(sx), np_(wq4)[cols], np_(sw)[cols])
    for m in range(M):
        j = int(np.searchsorted(cols, tok[m]))
        assert cols[j] == tok[m] and y[m, j] == mx[m]
        assert not np.any(y[m] > mx[m])
        assert not np.any((y[m] == mx[m]) & (cols < tok[m]))


def test_w4a8_rejects_bad_k(qv):
    """K must be a multiple of 32 for packed int4 weights."""
    xq = torch.zeros(2, 48, dtype=torch.int8, device="cuda")
    wq4 = torch.zeros(16, 24, dtype=torch.uint8, device="cuda")
    ws = qv.workspace(qv.QV_OP_LINEAR, 2, 48, 16)
    y = torch.zeros(2, 16, device="cuda")
    with pytest.raises(qv.QVError):
        qv.qv_w4a8_linear(xq, torch.ones(2, device="cuda"), wq4, torch.ones(16, device="cuda"), y, ws)


def test_w4a8_stack_step_matches_oracle(qv, oracle):
    """A small stack with int4 weights, one two-call step (qv_quantize_act +
    qv_w4a8_linear per projection, qv_quantize_act + qv_w4a8_lm_head_argmax,
    qv_accept): the last projection's output, the tokens and the accepted
    lengths equal the oracle's."""
    from gpu_util import bf16_bits
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 64, "ffn": 512, "layers": 2, "vocab": 3000}
    st = VerifyStack(model=model, B=2, gamma=3, seed=13, wbits=4)
    st.drafts.copy_(synth.uniform_tokens((2, 3), 3000, seed=4).cuda())
    st.enqueue_two_call()
    torch.cuda.synchronize()
    name, K, N = st.phases[-1]
    wq4, sw = st.weights[-1][-1]
    xq, sx = oracle.quantize_rows(bf16_bits(st.inputs[-1][-1]), bf16=True)
    y_ref, _ = oracle.w4a8_linear(xq, sx, np_(wq4), np_(sw))
    assert np.array_equal(np_(st.y[: st.M * N].view(st.M, N)).view(np.uint32), y_ref.view(np.uint32))
    xh, sh = oracle.quantize_rows(bf16_bits(st.h_final), bf16=True)
    t_ref, m_ref = oracle.w4a8_lm_head_argmax(xh, sh, np_(st.lm_wq), np_(st.lm_sw))
    assert np.array_equal(np_(st.tokens), t_ref) and np.array_equal(np_(st.max_logit), m_ref)
    l_ref, o_ref = oracle.accept(t_ref, np_(st.drafts), 2, 3)
    assert np.array_equal(np_(st.accept_len), l_ref) and np.array_equal(np_(st.out_tokens), o_ref)
    assert st.weight_bytes() == (sum(N * K for (_, K, N) in st.phases) * 2 + 3000 * 256) // 2
