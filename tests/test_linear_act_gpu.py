"""qv_w8a8_linear_act / qv_lm_head_argmax_act (activation quantization kernel,
then the streaming GEMM, in one call) against the oracle chain quantize_rows -> w8a8_linear
/ lm_head_argmax, bit for bit, and against the two-call GPU path. Covers the
int8 / f16 mma.sync GEMM (up to 16 padded tokens) and the tcgen05 GEMM (32
to 80)."""
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


def _inputs(M, K, N, dtype, smooth, seed):
    from quantized_verification_gb300 import synth
    x = synth.activations(M, K, seed=seed, dtype=dtype)
    if M >= 3:
        x[1] = 0                        # scale 0, codes 0
    if M >= 4:
        x[2] = x[2] * 1e-30             # tiny row
    mul = None
    if smooth:
        g = torch.Generator().manual_seed(K + seed)
        mul = (torch.rand(K, generator=g) * 3.5 + 0.25).to(torch.float32)
    wq = rand_codes((N, K), seed=seed + 1)
    sw = rand_scales(N, seed=seed + 2)
    return x, mul, wq, sw


def _oracle_codes(oracle, x, mul):
    m = None if mul is None else np_(mul)
    if x.dtype == torch.bfloat16:
        return oracle.quantize_rows(bf16_bits(x), m, bf16=True)
    return oracle.quantize_rows(np_(x), m)


def _gemm_part_zero(qv, ws, op_base, M, K, N):
    n = qv.qv_workspace_bytes(op_base, M, K, N)
    return int(ws[:n].count_nonzero()) == 0


LINEAR_ACT_CASES = [
    (5, 4096, 1024, torch.bfloat16, True),
    (8, 16, 130, torch.bfloat16, True),       # one K-tile of 16 columns, all 8 rows
    (2, 4096 + 48, 6 * 128, torch.float32, True),   # ragged last K-tile
    (6, 12288, 4096, torch.float32, False),   # fp32 rows of 12288
    (5, 4096, 1024, torch.float32, False),
    (1, 16, 7, torch.bfloat16, False),
    (8, 272, 300, torch.float32, True),
    (9, 512, 384, torch.bfloat16, True),
    (16, 12288, 512, torch.bfloat16, True),
    (5, 12288, 4096, torch.bfloat16, True),
    (17, 256, 200, torch.bfloat16, True),     # 32 padded tokens, tcgen05 GEMM
    (64, 1024, 256, torch.float32, True),     # tcgen05 GEMM (separate quantization kernel)
    (3, 12288, 300, torch.float32, True),     # fp32 rows longer than the quantizer keeps in registers
    (20, 16, 7, torch.bfloat16, True),        # a single GEMM tile
    (9, 128, 130, torch.float32, False),      # two GEMM CTAs
    (32, 4096, 1024, torch.bfloat16, True),   # 32 tokens, the fewest the tcgen05 kernel takes
    (16, 4096, 1024, torch.bfloat16, True),   # 16 tokens, the most the mma.sync kernel takes
]


@pytest.mark.parametrize("M,K,N,dtype,smooth", LINEAR_ACT_CASES)
def test_w8a8_linear_act(qv, oracle, M, K, N, dtype, smooth):
    x, mul, wq, sw = _inputs(M, K, N, dtype, smooth, seed=M * 1009 + K + N)
    q_ref, s_ref = _oracle_codes(oracle, x, mul)
    y_ref, _ = oracle.w8a8_linear(q_ref, s_ref, np_(wq), np_(sw))
    xd, md, wd, sd = x.cuda(), (mul.cuda() if mul is not None else None), wq.cuda(), sw.cuda()
    ws = qv.workspace(qv.QV_OP_LINEAR_ACT, M, K, N)
    for y_dtype in (torch.float32, torch.bfloat16):
        y = torch.full((M, N), float("nan"), dtype=y_dtype, device="cuda")
        for _ in range(2):                        # the workspace is reusable
            qv.qv_w8a8_linear_act(xd, wd, sd, y, ws, act_mul=md)
            torch.cuda.synchronize()
            assert _gemm_part_zero(qv, ws, qv.QV_OP_LINEAR, M, K, N), "GEMM workspace not left zero-filled"
            if y_dtype == torch.float32:
                assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))
            else:
                assert np.array_equal(bf16_bits(y), oracle.f32_to_bf16(y_ref))
    # the two-call path gives the same bits
    xq = torch.empty(M, K, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, device="cuda")
    qv.qv_quantize_act(xd, xq, sx, act_mul=md)
    y2 = torch.empty(M, N, device="cuda")
    qv.qv_w8a8_linear(xq, sx, wd, sd, y2, qv.workspace(qv.QV_OP_LINEAR, M, K, N))
    torch.cuda.synchronize()
    assert np.array_equal(np_(y2).view(np.uint32), y_ref.view(np.uint32))


def test_w8a8_linear_act_long_ranges(qv, oracle):
    """M = 16, K = 8192 at 140 and 141 channel tiles: each CTA's stream-K
    range spans about 59 or 60 K-tiles and crosses channel-tile boundaries
    part-way through K. Both must match the oracle."""
    M, K = 16, 8192
    for N in (128 * 140, 128 * 141):
        x, mul, wq, sw = _inputs(M, K, N, torch.bfloat16, True, seed=N)
        q_ref, s_ref = _oracle_codes(oracle, x, mul)
        y_ref, _ = oracle.w8a8_linear(q_ref, s_ref, np_(wq), np_(sw))
        ws = qv.workspace(qv.QV_OP_LINEAR_ACT, M, K, N)
        y = torch.empty(M, N, device="cuda")
        qv.qv_w8a8_linear_act(x.cuda(), wq.cuda(), sw.cuda(), y, ws, act_mul=mul.cuda())
        torch.cuda.synchronize()
        assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))
        assert _gemm_part_zero(qv, ws, qv.QV_OP_LINEAR, M, K, N)


@pytest.mark.parametrize("M,dtype", [(4, torch.float32), (8, torch.float32), (7, torch.bfloat16)])
def test_w8a8_linear_act_near_ties(qv, oracle, M, dtype):
    """Activations whose quotient x/s sits a few ulps from a half-integer,
    where the product with fl(1/s) can round to the other integer: the codes
    of the one-call path must still take the IEEE quotient's decision."""
    K, N = 1024, 384
    g = np.random.default_rng(23 + M)
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        amax = np.float32(g.uniform(0.5, 4.0))
        s = np.float32(amax / np.float32(127))
        j = g.integers(-126, 126, K).astype(np.float32)
        q = (j + np.float32(0.5)) * s
        x[m] = np.nextafter(q, np.where(g.random(K) < 0.5, np.inf, -np.inf).astype(np.float32))
        x[m, 0] = amax
    xt = torch.from_numpy(x).to(dtype)
    q_ref, s_ref = _oracle_codes(oracle, xt, None)
    wq = rand_codes((N, K), seed=M)
    sw = rand_scales(N, seed=M + 1)
    y_ref, _ = oracle.w8a8_linear(q_ref, s_ref, np_(wq), np_(sw))
    y = torch.empty(M, N, device="cuda")
    qv.qv_w8a8_linear_act(xt.cuda(), wq.cuda(), sw.cuda(), y, qv.workspace(qv.QV_OP_LINEAR_ACT, M, K, N))
    torch.cuda.synchronize()
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))


LM_ACT_CASES = [(5, 4096, 3000, True), (1, 128, 130, False), (16, 256, 1000, True),
                (20, 256, 777, True), (5, 512, 128 * 160 + 3, False)]


@pytest.mark.parametrize("M,K,V,smooth", LM_ACT_CASES)
def test_lm_head_argmax_act(qv, oracle, M, K, V, smooth):
    x, mul, wq, sw = _inputs(M, K, V, torch.bfloat16, smooth, seed=M * 77 + K + V)
    q_ref, s_ref = _oracle_codes(oracle, x, mul)
    t_ref, m_ref = oracle.lm_head_argmax(q_ref, s_ref, np_(wq), np_(sw))
    ws = qv.workspace(qv.QV_OP_LM_HEAD_ACT, M, K, V)
    tok = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    mx = torch.full((M,), float("nan"), device="cuda")
    for _ in range(2):
        qv.qv_lm_head_argmax_act(x.cuda(), wq.cuda(), sw.cuda(), tok, ws,
                                 act_mul=mul.cuda() if mul is not None else None, max_logit=mx)
        torch.cuda.synchronize()
        assert np.array_equal(np_(tok), t_ref)
        assert np.array_equal(np_(mx).view(np.uint32), m_ref.view(np.uint32))
        assert _gemm_part_zero(qv, ws, qv.QV_OP_LM_HEAD, M, K, V)


def test_lm_head_argmax_act_ties(qv, oracle):
    """Rows 400, 1700 and 1999 identical and maximal for token 0 (the codes
    of x do not depend on the weights): the lowest index must win."""
    M, K, V = 5, 256, 2000
    x, mul, wq, sw = _inputs(M, K, V, torch.bfloat16, False, seed=3)
    sw[:] = 0.003
    q_ref, s_ref = _oracle_codes(oracle, x, mul)
    best = torch.from_numpy((np.sign(q_ref[0]) * 127).astype(np.int8))
    for r in (400, 1700, 1999):
        wq[r] = best
    t_ref, m_ref = oracle.lm_head_argmax(q_ref, s_ref, np_(wq), np_(sw))
    assert t_ref[0] == 400
    ws = qv.workspace(qv.QV_OP_LM_HEAD_ACT, M, K, V)
    tok = torch.empty(M, dtype=torch.int32, device="cuda")
    qv.qv_lm_head_argmax_act(x.cuda(), wq.cuda(), sw.cuda(), tok, ws)
    torch.cuda.synchronize()
    assert np.array_equal(np_(tok), t_ref)


def test_shared_workspace_across_shapes(qv, oracle):
    """One buffer for *_act calls of different shapes, sized by the rule in
    the header (largest GEMM part + largest code part): alternating calls
    stay exact and leave every GEMM part zero-filled."""
    al = lambda v, a: (v + a - 1) // a * a
    shapes = [(5, 12288, 512), (5, 256, 4096), (16, 1024, 1000)]
    gemm = max(qv.qv_workspace_bytes(qv.QV_OP_LINEAR, M, K, N) for (M, K, N) in shapes)
    codes = max(al(M * K, 16) + al(4 * M, 16) for (M, K, N) in shapes)
    ws = torch.zeros(al(gemm, 256) + al(codes, 256), dtype=torch.uint8, device="cuda")
    cases = []
    for (M, K, N) in shapes:
        x, mul, wq, sw = _inputs(M, K, N, torch.bfloat16, True, seed=K + N)
        q_ref, s_ref = _oracle_codes(oracle, x, mul)
        y_ref, _ = oracle.w8a8_linear(q_ref, s_ref, np_(wq), np_(sw))
        cases.append((x.cuda(), mul.cuda(), wq.cuda(), sw.cuda(), y_ref, M, K, N))
    for rep in range(2):
        for (xd, md, wd, sd, y_ref, M, K, N) in cases:
            y = torch.empty(M, N, device="cuda")
            qv.qv_w8a8_linear_act(xd, wd, sd, y, ws, act_mul=md)
            torch.cuda.synchronize()
            assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32)), (rep, M, K, N)
            assert int(ws[:gemm].count_nonzero()) == 0
