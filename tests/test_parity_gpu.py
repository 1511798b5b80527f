"""GPU path (through the C ABI) against the CPU oracle, element by element, on
identical seeded inputs. Integers, codes, scales, token ids and accepted
lengths must be bit-exact; fp32 outputs within 1e-6 relative (and, by design,
bit-exact); the bf16 comparator within 1e-2 norm-wise of the fp64 reference
and within the fp32 dot-product error bound elementwise."""
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


def _synth():
    from quantized_verification_gb300 import synth
    return synth


# ---------------------------------------------------------------------------
# a1 / a0 quantization
# ---------------------------------------------------------------------------
QUANT_CASES = [
    (1, 16, torch.float32, False), (4, 256, torch.float32, False), (4, 256, torch.float32, True),
    (5, 4096, torch.bfloat16, False), (5, 4096, torch.bfloat16, True), (80, 12288, torch.bfloat16, False),
    (3, 25600, torch.bfloat16, True), (2, 4112, torch.float32, True), (7, 48, torch.bfloat16, False),
]


@pytest.mark.parametrize("M,K,dtype,smooth", QUANT_CASES)
def test_quantize_act(qv, oracle, M, K, dtype, smooth):
    synth = _synth()
    x = synth.activations(M, K, seed=1000 + M + K, dtype=dtype)
    if M >= 3:
        x[1] = 0                                   # all-zero row -> scale 0, codes 0
    if M >= 4:
        x[2] = x[2] * 1e-30                        # tiny row (subnormal quotients)
    mul = None
    if smooth:
        g = torch.Generator().manual_seed(K)
        mul = (torch.rand(K, generator=g) * 3.5 + 0.25).to(torch.float32)
    xd = x.cuda()
    xq = torch.full((M, K), 99, dtype=torch.int8, device="cuda")
    sx = torch.full((M,), -1.0, device="cuda")
    qv.qv_quantize_act(xd, xq, sx, act_mul=mul.cuda() if mul is not None else None)
    torch.cuda.synchronize()
    if dtype == torch.bfloat16:
        q_ref, s_ref = oracle.quantize_rows(bf16_bits(x), None if mul is None else np_(mul), bf16=True)
    else:
        q_ref, s_ref = oracle.quantize_rows(np_(x), None if mul is None else np_(mul))
    assert np.array_equal(np_(sx).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(np_(xq), q_ref)


@pytest.mark.parametrize("N,K,dtype", [(512, 256, torch.float32), (1024, 4096, torch.bfloat16),
                                       (1000, 272, torch.bfloat16), (3, 16, torch.float32)])
def test_quantize_weight(qv, oracle, N, K, dtype):
    w = _synth().weights(N, K, seed=N * 7 + K, dtype=dtype)
    wq = torch.empty(N, K, dtype=torch.int8, device="cuda")
    sw = torch.empty(N, device="cuda")
    qv.qv_quantize_weight(w.cuda(), wq, sw)
    torch.cuda.synchronize()
    src = bf16_bits(w) if dtype == torch.bfloat16 else np_(w)
    q_ref, s_ref = oracle.quantize_rows(src, bf16=dtype == torch.bfloat16)
    assert np.array_equal(np_(sw).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(np_(wq), q_ref)


# ---------------------------------------------------------------------------
# a2 W8A8 linear
# ---------------------------------------------------------------------------
LINEAR_CASES = [
    (4, 256, 512), (1, 128, 128), (5, 4096, 1024), (5, 272, 1000), (8, 1024, 130),
    (9, 512, 384), (16, 384, 256), (17, 256, 200), (32, 640, 256), (33, 256, 129),
    (64, 512, 256), (65, 256, 128), (80, 512, 300), (256, 256, 136), (5, 16, 7),
    (24, 4096, 4096), (32, 12288, 3000),
    # tcgen05 grids of whole segments (tiles per CTA dividing the 32 or 96
    # K-tiles: 128 x 8, 96 x 16, 128 x 24) at Qwen3-8B sizes
    (64, 4096, 4096), (80, 4096, 6144), (64, 12288, 4096),
    # more than 80 rows: the fewest launches of equal row counts
    (81, 256, 130), (96, 256, 300), (128, 512, 256), (161, 128, 200),
    # up to 8 tokens: ragged K (33 K-tiles) with ragged N, wide N at 2
    # K-tiles, a single token and a full group of 8
    (5, 4096 + 48, 128 * 40 + 7), (1, 256, 128 * 200), (8, 1024, 128 * 100 + 1),
]


def _run_linear(qv, xq, sx, wq, sw, y_dtype=torch.float32):
    M, K = xq.shape
    N = wq.shape[0]
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    y = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
    acc = torch.full((M, N), 12345, dtype=torch.int32, device="cuda")
    qv.qv_w8a8_linear(xq.cuda(), sx.cuda(), wq.cuda(), sw.cuda(), y, ws, acc_debug=acc)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"
    return y, acc


@pytest.mark.parametrize("M,K,N", LINEAR_CASES)
def test_w8a8_linear(qv, oracle, M, K, N):
    xq = rand_codes((M, K), seed=M * 131 + K)
    wq = rand_codes((N, K), seed=N * 17 + K + 1)
    sx = rand_scales(M, seed=M + 5, lo=1e-3, hi=0.2)
    sw = rand_scales(N, seed=N + 6)
    y, acc = _run_linear(qv, xq, sx, wq, sw)
    y_ref, acc_ref = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    assert np.array_equal(np_(acc), acc_ref)
    yg = np_(y)
    rel = np.abs(yg.astype(np.float64) - y_ref) / np.maximum(np.abs(y_ref.astype(np.float64)), 1e-30)
    assert float(rel.max()) <= 1e-6
    assert np.array_equal(yg.view(np.uint32), y_ref.view(np.uint32))   # the design target: bit-exact
    yb, _ = _run_linear(qv, xq, sx, wq, sw, y_dtype=torch.bfloat16)
    assert np.array_equal(bf16_bits(yb), oracle.f32_to_bf16(y_ref))


@pytest.mark.parametrize("M", [3, 24, 40])
@pytest.mark.parametrize("K,with_m128", [((133144 // 16) * 16, False), (4096, True)])
def test_w8a8_extreme_magnitudes(qv, oracle, M, K, with_m128):
    """Codes at the ends of the range. The first case is the largest K that is
    a multiple of 16 and keeps every +-127 sum inside int32; -128 codes are
    exercised at a K where their sums fit as well. M = 3 and M = 24 run the
    int8 mma.sync kernel (8 and 32 padded tokens), M = 40 the tcgen05 kernel
    (rows 3.. repeat rows 0..2)."""
    N = 130
    xq = torch.full((M, K), 127, dtype=torch.int8)
    xq[1::3] = -127
    wq = torch.full((N, K), 127, dtype=torch.int8)
    wq[1::3] = -127
    if with_m128:
        xq[2::3, ::2] = -128
        wq[2::3, 1::2] = -128
    else:
        xq[2::3, ::2] = -127
        wq[2::3, 1::2] = -127
    sx = torch.full((M,), 1e-3)
    sw = torch.full((N,), 1e-4)
    y, acc = _run_linear(qv, xq, sx, wq, sw)
    y_ref, acc_ref = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    if not with_m128:
        assert abs(int(acc_ref[0, 0])) == K * 127 * 127
    assert np.array_equal(np_(acc), acc_ref)
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))


def test_w8a8_quantize_chain(qv, oracle):
    """a1 + a2 on the GPU end to end against the oracle chain (bf16 inputs)."""
    synth = _synth()
    M, K, N = 5, 4096, 1024
    x = synth.activations(M, K, seed=11)
    w = synth.weights(N, K, seed=12)
    xq = torch.empty(M, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, device="cuda")
    wq = torch.empty(N, K, dtype=torch.int8, device="cuda")
    sw = torch.empty(N, device="cuda")
    qv.qv_quantize_weight(w.cuda(), wq, sw)
    qv.qv_quantize_act(x.cuda(), xq, sx)
    y = torch.empty(M, N, device="cuda")
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws)
    torch.cuda.synchronize()
    xq_r, sx_r = oracle.quantize_rows(bf16_bits(x), bf16=True)
    wq_r, sw_r = oracle.quantize_rows(bf16_bits(w), bf16=True)
    y_r, _ = oracle.w8a8_linear(xq_r, sx_r, wq_r, sw_r)
    assert np.array_equal(np_(y).view(np.uint32), y_r.view(np.uint32))


# ---------------------------------------------------------------------------
# a3 LM head + argmax
# ---------------------------------------------------------------------------
LM_CASES = [(4, 256, 1024), (5, 4096, 3000), (1, 128, 130), (9, 256, 1000), (64, 256, 513),
            (80, 128, 777), (5, 512, 128 * 160 + 3), (32, 4096, 3000), (24, 512, 128 * 160 + 3),
            (72, 512, 2000), (96, 256, 1000), (8, 1024, 128 * 100 + 1), (3, 4096 + 48, 128 * 40 + 7)]


def _run_lm(qv, xq, sx, wq, sw):
    M, K = xq.shape
    V = wq.shape[0]
    ws = qv.workspace(qv.QV_OP_LM_HEAD, M, K, V)
    tok = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    mx = torch.full((M,), float("nan"), device="cuda")
    qv.qv_lm_head_argmax(xq.cuda(), sx.cuda(), wq.cuda(), sw.cuda(), tok, ws, max_logit=mx)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"
    return np_(tok), np_(mx)


@pytest.mark.parametrize("M,K,V", LM_CASES)
def test_lm_head_argmax(qv, oracle, M, K, V):
    xq = rand_codes((M, K), seed=M * 7 + K + V)
    wq = rand_codes((V, K), seed=V * 3 + K)
    sx = rand_scales(M, seed=M + 9, lo=1e-3, hi=0.2)
    sw = rand_scales(V, seed=V + 10)
    tok, mx = _run_lm(qv, xq, sx, wq, sw)
    t_ref, m_ref = oracle.lm_head_argmax(np_(xq), np_(sx), np_(wq), np_(sw))
    assert np.array_equal(tok, t_ref)
    assert np.array_equal(mx, m_ref)


def test_lm_head_ties_lowest_index(qv, oracle):
    M, K, V = 5, 256, 2000
    xq = rand_codes((M, K), seed=1)
    wq = rand_codes((V, K), seed=2)
    sx = rand_scales(M, seed=3)
    sw = torch.full((V,), 0.003)
    # make rows 1700, 400 and 1999 identical; row 400 must win wherever they are the max
    wq[1700] = wq[400]
    wq[1999] = wq[400]
    # bias the winner: row 400 = sign-matched to token 0's codes
    wq[400] = torch.where(xq[0] >= 0, 127, -127).to(torch.int8)
    wq[1700] = wq[400]
    wq[1999] = wq[400]
    tok, mx = _run_lm(qv, xq, sx, wq, sw)
    t_ref, m_ref = oracle.lm_head_argmax(np_(xq), np_(sx), np_(wq), np_(sw))
    assert t_ref[0] == 400
    assert np.array_equal(tok, t_ref) and np.array_equal(mx, m_ref)


def test_lm_head_negative_and_zero_logits(qv, oracle):
    M, K, V = 3, 64, 300
    xq = torch.zeros(M, K, dtype=torch.int8)      # row 0: all logits 0 -> token 0
    xq[1] = 1
    wq = -rand_codes((V, K), seed=4, lo=1, hi=127)  # row 1: all logits negative
    xq[2] = rand_codes((K,), seed=5)
    sx = torch.tensor([0.0, 0.01, 0.02])
    sw = rand_scales(V, seed=6)
    tok, mx = _run_lm(qv, xq, sx, wq, sw)
    t_ref, m_ref = oracle.lm_head_argmax(np_(xq), np_(sx), np_(wq), np_(sw))
    assert np.array_equal(tok, t_ref) and np.array_equal(mx, m_ref)
    assert tok[0] == 0


# ---------------------------------------------------------------------------
# a4 acceptance
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,gamma", [(1, 3), (1, 4), (16, 4), (8, 7), (1, 0), (300, 5), (3, 31)])
def test_accept(qv, oracle, B, gamma):
    synth = _synth()
    V = 50
    t = synth.uniform_tokens((B, gamma + 1), V, seed=B * 100 + gamma)
    d = synth.geometric_drafts(t, V, p=0.7, seed=B + gamma)
    if B >= 3 and gamma > 0:
        d[0] = t[0, :gamma]                      # all drafts accepted
        d[1, 0] = (t[1, 0] + 1) % V              # first draft rejected
    ln = torch.full((B,), -5, dtype=torch.int32, device="cuda")
    out = torch.full((B, gamma + 1), -5, dtype=torch.int32, device="cuda")
    qv.qv_accept(t.cuda(), d.cuda() if gamma > 0 else None, ln, out)
    torch.cuda.synchronize()
    l_ref, o_ref = oracle.accept(np_(t), np_(d), B, gamma)
    assert np.array_equal(np_(ln), l_ref)
    assert np.array_equal(np_(out), o_ref)
    if B >= 3 and gamma > 0:
        assert l_ref[0] == gamma + 1 and l_ref[1] == 1


# ---------------------------------------------------------------------------
# BF16 comparator
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,K,N", [(5, 4096, 1024), (4, 256, 512), (17, 192, 300), (64, 512, 256), (80, 128, 200)])
def test_bf16_linear(qv, oracle, M, K, N):
    synth = _synth()
    x = synth.activations(M, K, seed=M + K)
    w = synth.weights(N, K, seed=N + K)
    ws = qv.workspace(qv.QV_OP_BF16_LINEAR, M, K, N)
    y = torch.full((M, N), float("nan"), device="cuda")
    qv.qv_bf16_linear(x.cuda(), w.cuda(), y, ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    xf = oracle.bf16_to_f32(bf16_bits(x))
    wf = oracle.bf16_to_f32(bf16_bits(w))
    ref = oracle.linear_f64(xf, wf)
    yg = np_(y).astype(np.float64)
    assert np.abs(yg - ref).max() / np.abs(ref).max() <= 1e-2
    # elementwise fp32 dot-product bound: |err| <= gamma_K * sum |x w|, gamma_K = K u / (1 - K u)
    u = 2.0 ** -24
    gk = K * u / (1 - K * u)
    mag = np.abs(xf.astype(np.float64)) @ np.abs(wf.astype(np.float64)).T
    assert np.all(np.abs(yg - ref) <= gk * mag + 1e-30)


# ---------------------------------------------------------------------------
# host-side rejection, graphs, device error word
# ---------------------------------------------------------------------------
def test_rejected_calls_leave_outputs_untouched(qv):
    M, K, N = 4, 256, 64
    xq = rand_codes((M, K), 1).cuda()
    wq = rand_codes((N, K), 2).cuda()
    sx = rand_scales(M, 3).cuda()
    sw = rand_scales(N, 4).cuda()
    y = torch.full((M, N), 7.0, device="cuda")
    small_ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qv.QVError) as ei:
        qv.qv_w8a8_linear(xq, sx, wq, sw, y, small_ws)
    assert ei.value.status == qv.QV_ERR_WORKSPACE
    # misaligned xq (offset by 1 byte inside a flat buffer)
    flat = torch.zeros(M * K + 16, dtype=torch.int8, device="cuda")
    mis = flat[1:1 + M * K].view(M, K)
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    with pytest.raises(qv.QVError) as ei:
        qv.qv_w8a8_linear(mis, sx, wq, sw, y, ws)
    assert ei.value.status == qv.QV_ERR_INVALID_ARG
    # a host pointer handed straight to the C ABI is refused before any launch
    import ctypes
    host = torch.zeros(M * K, dtype=torch.int8)
    lib = qv.load()
    st = lib.qv_w8a8_linear(ctypes.c_void_p(host.data_ptr()), ctypes.c_void_p(sx.data_ptr()), M, K,
                            ctypes.c_void_p(wq.data_ptr()), ctypes.c_void_p(sw.data_ptr()), N,
                            ctypes.c_void_p(y.data_ptr()), 0, None, ctypes.c_void_p(ws.data_ptr()),
                            ws.numel(), None)
    assert st == qv.QV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_cuda_graph_replay_matches(qv, oracle):
    M, K, N, V = 5, 512, 640, 900
    xq = rand_codes((M, K), 21).cuda()
    wq = rand_codes((N, K), 22).cuda()
    wl = rand_codes((V, K), 23).cuda()
    sx = rand_scales(M, 24).cuda()
    sw = rand_scales(N, 25).cuda()
    sl = rand_scales(V, 26).cuda()
    ws1 = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    ws2 = qv.workspace(qv.QV_OP_LM_HEAD, M, K, V)
    y = torch.empty(M, N, device="cuda")
    tok = torch.empty(M, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws1, stream=s)       # warm-up outside capture
        qv.qv_lm_head_argmax(xq, sx, wl, sl, tok, ws2, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = torch.cuda.current_stream()
        for _ in range(3):
            qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws1, stream=st)
            qv.qv_lm_head_argmax(xq, sx, wl, sl, tok, ws2, stream=st)
    y.zero_()
    tok.fill_(-1)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    y_ref, _ = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    t_ref, _ = oracle.lm_head_argmax(np_(xq), np_(sx), np_(wl), np_(sl))
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))
    assert np.array_equal(np_(tok), t_ref)
    assert int(ws1.count_nonzero()) == 0 and int(ws2.count_nonzero()) == 0


def test_device_error_word_clear(qv):
    assert qv.qv_device_error() == 0


# More stream-K splits at up to 8 tokens: channel tiles split over 1, 2 and
# many CTAs, whole tiles per CTA, ragged K blocks and ragged N.
SPLIT_CASES = [
    (5, 4096, 100), (5, 1040, 2432), (5, 4096, 4096), (8, 4096, 6144), (3, 2064, 24576 + 16),
    (5, 12288, 4096), (1, 16, 33), (7, 12288, 3000),
]


@pytest.mark.parametrize("M,K,N", SPLIT_CASES)
def test_w8a8_linear_split_schedules(qv, oracle, M, K, N):
    xq = rand_codes((M, K), seed=M * 31 + K)
    wq = rand_codes((N, K), seed=N * 7 + K)
    sx = rand_scales(M, seed=M + 50, lo=1e-3, hi=0.2)
    sw = rand_scales(N, seed=N + 60)
    y, acc = _run_linear(qv, xq, sx, wq, sw)
    y_ref, acc_ref = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    assert np.array_equal(np_(acc), acc_ref)
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))
