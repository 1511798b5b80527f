"""The layer's fused non-linear steps (qv_rmsnorm_quant, qv_swiglu_quant,
qv_w8a8_swiglu) and the chained layers against the oracle, bit for bit: the
updated residual stream, the normalized bf16 activations, the SwiGLU output,
the int8 codes, the fp32 token scales, the tokens and accepted lengths."""
import numpy as np
import pytest
import torch

from gpu_util import np_, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    _qv.load()
    return _qv


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


NORM_CASES = [  # M, H, with delta, with multipliers, eps
    (1, 16, False, False, 1e-6),
    (5, 4096, True, False, 1e-6),
    (3, 5120, True, True, 1e-5),
    (17, 96, True, False, 0.0),
    (2, 16384, True, True, 1e-6),
    (4, 12288, False, False, 1e-6),
]


@pytest.mark.parametrize("M,H,with_delta,with_mul,eps", NORM_CASES)
def test_rmsnorm_quant(qv, oracle, M, H, with_delta, with_mul, eps):
    rng = np.random.default_rng(M * 7919 + H)
    hf = rng.normal(0.0, 1.0, (M, H)).astype(np.float32)
    hf[:, rng.choice(H, max(1, H // 100), replace=False)] *= 20.0      # outlier channels
    h = _bf16(hf)
    d = _bf16(rng.normal(0.0, 0.5, (M, H))) if with_delta else None
    g = _bf16(rng.uniform(0.5, 1.5, H))
    mul = torch.from_numpy(rng.uniform(0.5, 2.0, H).astype(np.float32)) if with_mul else None
    h_ref, q_ref, s_ref, x_ref = oracle.residual_rmsnorm_quant(
        _bits(h), None if d is None else _bits(d), _bits(g), eps, None if mul is None else mul.numpy())
    hd = h.cuda()
    xq = torch.empty(M, H, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, device="cuda")
    x_out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    qv.qv_rmsnorm_quant(hd, g.cuda(), xq, sx, delta=None if d is None else d.cuda(), eps=eps,
                        act_mul=None if mul is None else mul.cuda(), x_out=x_out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(hd), h_ref)
    assert np.array_equal(_bits(x_out), x_ref)
    assert np.array_equal(np_(xq), q_ref)
    assert np.array_equal(np_(sx).view(np.uint32), s_ref.view(np.uint32))


def test_rmsnorm_quant_constant_and_zero_rows(qv, oracle):
    """Closed forms through the GPU path: constant rows give codes of +-127,
    a delta of -h gives all-zero codes and scale 0."""
    H = 256
    h = torch.stack([torch.full((H,), 2.0), torch.full((H,), -0.25), torch.ones(H)]).to(torch.bfloat16)
    d = torch.stack([torch.zeros(H), torch.zeros(H), -torch.ones(H)]).to(torch.bfloat16)
    g = torch.ones(H, dtype=torch.bfloat16)
    hd = h.cuda()
    xq = torch.empty(3, H, dtype=torch.int8, device="cuda")
    sx = torch.empty(3, device="cuda")
    qv.qv_rmsnorm_quant(hd, g.cuda(), xq, sx, delta=d.cuda(), eps=0.0)
    torch.cuda.synchronize()
    q = np_(xq)
    assert (q[0] == 127).all() and (q[1] == -127).all() and not q[2].any()
    assert float(sx[2]) == 0.0
    _, q_ref, s_ref, _ = oracle.residual_rmsnorm_quant(_bits(h), _bits(d), _bits(g), 0.0)
    assert np.array_equal(q, q_ref) and np.array_equal(np_(sx).view(np.uint32), s_ref.view(np.uint32))


GLU_CASES = [(1, 16), (5, 12288), (3, 25600), (4, 64), (2, 32768)]


@pytest.mark.parametrize("M,F", GLU_CASES)
def test_swiglu_quant(qv, oracle, M, F):
    rng = np.random.default_rng(M * 104729 + F)
    gate = rng.normal(0.0, 3.0, (M, F)).astype(np.float32)
    up = rng.normal(0.0, 1.0, (M, F)).astype(np.float32)
    # every branch of the exp: both cutoffs, their neighbours, saturation, zeros
    special = np.float32([0.0, -0.0, 87.0, -87.0, 88.0, -88.0, 87.5, -87.5, 88.001, -88.001, 100.0, -100.0,
                          1e-30, -1e-30, 0.34657359, -0.34657359])
    gate[0, : min(F, special.size)] = special[: min(F, special.size)]
    if F >= 4096:
        gate[-1, 2048:4096] = np.linspace(-95.0, 95.0, 2048, dtype=np.float32)
    gu = np.concatenate([gate, up], axis=1)
    q_ref, s_ref = oracle.swiglu_quant(gu)
    xq = torch.empty(M, F, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, device="cuda")
    qv.qv_swiglu_quant(torch.from_numpy(gu).cuda(), xq, sx)
    torch.cuda.synchronize()
    assert np.array_equal(np_(xq), q_ref)
    assert np.array_equal(np_(sx).view(np.uint32), s_ref.view(np.uint32))


def test_swiglu_exp_grid(qv, oracle):
    """SiLU over a dense grid of 65536 gates from -90 to 90 (up = 1), 1024
    per row: codes and scales equal the oracle's, so the GPU's exp, sigmoid
    and product agree with the definition across every branch."""
    F = 1024
    grid = np.linspace(-90.0, 90.0, 64 * F, dtype=np.float32).reshape(64, F)
    gu = np.concatenate([grid, np.ones_like(grid)], axis=1)
    q_ref, s_ref = oracle.swiglu_quant(gu)
    xq = torch.empty(64, F, dtype=torch.int8, device="cuda")
    sx = torch.empty(64, device="cuda")
    qv.qv_swiglu_quant(torch.from_numpy(gu).cuda(), xq, sx)
    torch.cuda.synchronize()
    assert np.array_equal(np_(xq), q_ref)
    assert np.array_equal(np_(sx).view(np.uint32), s_ref.view(np.uint32))


def test_chained_layers_match_oracle(qv, oracle):
    """Two chained decoder layers (residual stream, RMSNorm, SwiGLU between
    the W8A8 linears), the final RMSNorm, the LM head and the acceptance:
    the residual stream, every linear's output that feeds the chain, the
    tokens and the accepted lengths equal the oracle's chain bit for bit."""
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 64, "ffn": 512, "layers": 2, "vocab": 1000}
    st = VerifyStack(model=model, B=2, gamma=3, seed=5)
    st.prepare_chain(eps=1e-6)
    st.drafts.copy_(synth.uniform_tokens((2, 3), 1000, seed=3).cuda())
    st.enqueue_chain()
    torch.cuda.synchronize()

    cpu = lambda t: t.cpu().numpy()
    h = _bits(st.h0)
    yd = None
    for l in range(model["layers"]):
        g1, g2 = st.norm_w[l]
        h, q, s, _ = oracle.residual_rmsnorm_quant(h, yd, _bits(g1), 1e-6)
        wq, sw = st.weights[l][1]
        qo, so = oracle.quantize_rows(_bits(st.inputs[l][1]), bf16=True)
        y_o = oracle.f32_to_bf16(oracle.w8a8_linear(qo, so, cpu(wq), cpu(sw))[0])
        h, q2, s2, _ = oracle.residual_rmsnorm_quant(h, y_o, _bits(g2), 1e-6)
        wq, sw = st.weights[l][2]
        y_il, _ = oracle.w8a8_linear(q2, s2, cpu(wq), cpu(sw))     # gate|up rows interleaved by 64
        F = y_il.shape[1] // 2
        blocks = y_il.reshape(-1, F // 64, 2, 64)
        y_gu = np.concatenate([blocks[:, :, 0, :].reshape(-1, F), blocks[:, :, 1, :].reshape(-1, F)], axis=1)
        q3, s3 = oracle.swiglu_quant(y_gu)
        wq, sw = st.weights[l][3]
        yd = oracle.f32_to_bf16(oracle.w8a8_linear(q3, s3, cpu(wq), cpu(sw))[0])
        if l == model["layers"] - 1:
            wq, sw = st.weights[l][0]
            y_qkv = oracle.f32_to_bf16(oracle.w8a8_linear(q, s, cpu(wq), cpu(sw))[0])
            assert np.array_equal(_bits(st.y_qkv), y_qkv)
            assert np.array_equal(_bits(st.y_o), y_o)
            a_ref = _silu_times(oracle, y_gu[:, :F], y_gu[:, F:])
            assert np.array_equal(np_(st.a_glu).view(np.uint32), a_ref.view(np.uint32))
            assert np.array_equal(_bits(st.y_down), yd)
    h, qf, sf, _ = oracle.residual_rmsnorm_quant(h, yd, _bits(st.norm_final), 1e-6)
    assert np.array_equal(_bits(st.h_res), h)
    tok, _ = oracle.lm_head_argmax(qf, sf, cpu(st.lm_wq), cpu(st.lm_sw))
    assert np.array_equal(np_(st.tokens), tok)
    ln, out = oracle.accept(tok, cpu(st.drafts), 2, 3)
    assert np.array_equal(np_(st.accept_len), ln) and np.array_equal(np_(st.out_tokens), out)
    # the captured step gives the same result again (the residual stream is reset per step)
    g = st.capture_chain()
    st.tokens.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(np_(st.tokens), tok) and np.array_equal(_bits(st.h_res), h)


def _silu_times(oracle, gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """fl32(silu(g) * u) elementwise with the oracle's silu."""
    sil = np.array([oracle.silu(float(g)) for g in gate.reshape(-1)], dtype=np.float32).reshape(gate.shape)
    return (sil * up.astype(np.float32)).astype(np.float32)


@pytest.mark.parametrize("M,K,F", [(5, 256, 64), (17, 512, 192), (5, 4096, 1024), (64, 256, 128), (80, 128, 256)])
def test_w8a8_swiglu(qv, oracle, M, K, F):
    """The gate|up linear with SiLU(gate) * up in its epilogue (interleaved
    rows; mma.sync kernel up to 16 tokens, tcgen05 at 32, 64 and 80, 80-row
    slices beyond): a equals fl32(silu(y_gate) * y_up) of the oracle's linear."""
    from gpu_util import rand_codes, rand_scales
    xq = rand_codes((M, K), seed=M + 3 * K)
    sx = rand_scales(M, seed=M + 1, lo=1e-3, hi=0.2)
    wq = rand_codes((2 * F, K), seed=F + 7)
    sw = rand_scales(2 * F, seed=F + 9)
    y, _ = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    a_ref = _silu_times(oracle, y[:, :F], y[:, F:])
    wq_il = qv.interleave_gate_up(wq.cuda())
    sw_il = qv.interleave_gate_up(sw.cuda())
    a = torch.full((M, F), float("nan"), device="cuda")
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, 2 * F)
    qv.qv_w8a8_swiglu(xq.cuda(), sx.cuda(), wq_il, sw_il, a, ws)
    torch.cuda.synchronize()
    assert np.array_equal(np_(a).view(np.uint32), a_ref.view(np.uint32))
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"


def _to_bf16_f32(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to bf16 (nearest even), returned as float32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _norm_x(h: np.ndarray, g: np.ndarray, var: np.float32, eps: float) -> np.ndarray:
    """x = rne_bf16(g * rne_bf16(h * rstd)) with rstd from var (binary32 steps)."""
    rstd = np.float32(1.0) / np.sqrt(np.float32(var) + np.float32(eps))
    return _to_bf16_f32(g * _to_bf16_f32(h * rstd))


def _near_boundary_row(H: int, g: np.ndarray, eps: float, rng, above: bool):
    """A bf16 row whose sum of squares, added in binary64 in index order, puts
    ss / H within 2^-48 (relative) of a binary32 rounding boundary, on the
    given side; and such that the other rounding of var changes the
    normalized output. The last 12 slots hold correction terms chosen
    greedily (largest bf16 whose square fits the remaining gap)."""
    while True:
        h = _to_bf16_f32(rng.normal(0.0, 1.0, H).astype(np.float32))
        h[-12:] = 0.0
        ss = float(np.cumsum(h.astype(np.float64) ** 2)[-1])       # sequential, index order
        f = np.float32(ss / H)
        up = np.nextafter(f, np.float32(np.inf))
        mid = (float(f) + float(up)) / 2.0
        if mid <= ss / H:
            mid = (float(up) + float(np.nextafter(up, np.float32(np.inf)))) / 2.0
        target = mid * (1.0 + (2.0 ** -50 if above else -2.0 ** -50))
        gap = target * H - ss
        for j in range(H - 12, H):
            if gap <= 0:
                break
            c = np.float32(np.sqrt(gap))
            c = (np.array([c], np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)[0]
            h[j] = c
            gap -= float(c) * float(c)
        ss = float(np.cumsum(h.astype(np.float64) ** 2)[-1])
        q = ss / H
        if abs(q - mid) > 2.0 ** -48 * q or (q > mid) != above:
            continue
        var = np.float32(q)
        other = np.nextafter(var, np.float32(-np.inf) if above else np.float32(np.inf))
        if not np.array_equal(_norm_x(h, g, var, eps), _norm_x(h, g, other, eps)):
            return h


def test_rmsnorm_quant_near_variance_rounding_boundary(qv, oracle):
    """Rows whose variance sits within 2^-48 of a binary32 rounding boundary,
    closer than a float-float sum of the squares resolves, so that only the
    definition's binary64 sum rounds var the right way (and the other way
    would change the normalized output): the normalized bf16 activations,
    the codes and the scales equal the oracle's."""
    rng = np.random.default_rng(2024)
    M, H, eps = 8, 4096, 1e-6
    g = _to_bf16_f32(rng.uniform(0.5, 1.5, H).astype(np.float32))
    rows = [_near_boundary_row(H, g, eps, rng, above=(m % 2 == 0)) for m in range(M)]
    h = _bf16(np.stack(rows))
    gb = _bf16(g)
    assert np.array_equal(_bits(h).view(np.uint16), _bits(_bf16(np.stack(rows))))     # rows are bf16 already
    h_ref, q_ref, s_ref, x_ref = oracle.residual_rmsnorm_quant(_bits(h), None, _bits(gb), eps)
    hd = h.cuda()
    xq = torch.empty(M, H, dtype=torch.int8, device="cuda")
    sx = torch.empty(M, device="cuda")
    x_out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    qv.qv_rmsnorm_quant(hd, gb.cuda(), xq, sx, eps=eps, x_out=x_out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(x_out), x_ref)
    assert np.array_equal(np_(xq), q_ref)
    assert np.array_equal(np_(sx).view(np.uint32), s_ref.view(np.uint32))


def test_chained_layers_with_attention_match_oracle(qv, oracle):
    """Two chained decoder layers with attention over a 40-position bf16 KV
    cache per sequence between the qkv and o projections, checked step by
    step: each layer's qkv output equals the oracle's bit for bit; its
    attention output is within 1e-4 max|v| of the oracle's binary64
    attention of that qkv output (the bound of the attention tests); with the
    GPU's attention output as input, every later step (its quantization, o,
    RMSNorm, gate|up with SwiGLU, down, the final norm, the LM head and the
    acceptance) equals the oracle's bit for bit, and the captured step
    repeats it."""
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 64, "ffn": 512, "layers": 2, "vocab": 1000}
    B, gamma, D, L = 2, 3, 64, 40
    T, Hq, Hkv = gamma + 1, 256 // D, 64 // D
    st = VerifyStack(model=model, B=B, gamma=gamma, seed=9)
    st.prepare_chain(eps=1e-6, cache_len=L, head_dim=D)
    st.drafts.copy_(synth.uniform_tokens((B, gamma), 1000, seed=4).cuda())
    st.enqueue_chain()
    torch.cuda.synchronize()

    cpu = lambda t: t.cpu().numpy()
    scale = float(np.float32(1.0 / np.sqrt(D)))
    lens = np.full(B, L, dtype=np.int32)
    h = _bits(st.h0)
    yd = None
    for l in range(model["layers"]):
        g1, g2 = st.norm_w[l]
        h, q, s, _ = oracle.residual_rmsnorm_quant(h, yd, _bits(g1), 1e-6)
        wq, sw = st.weights[l][0]
        y_qkv = oracle.f32_to_bf16(oracle.w8a8_linear(q, s, cpu(wq), cpu(sw))[0])
        kc, vc = _bits(st.k_cache[l]).reshape(B, L, Hkv, D), _bits(st.v_cache[l]).reshape(B, L, Hkv, D)
        att_ref = oracle.attention_verify(y_qkv, kc, vc, lens, T, Hq, Hkv, D, scale)
        att = np_(st.attn_out[l])
        vals = np.concatenate([(vc.astype(np.uint32) << 16).view(np.float32).ravel(),
                               (y_qkv[:, (Hq + Hkv) * D:].astype(np.uint32) << 16).view(np.float32).ravel()])
        assert np.all(np.isfinite(att))
        assert float(np.abs(att.astype(np.float64) - att_ref).max()) <= 1e-4 * float(np.abs(vals).max()), l
        qo, so = oracle.quantize_rows(att)                         # the chain continues from the GPU's output
        wq, sw = st.weights[l][1]
        y_o = oracle.f32_to_bf16(oracle.w8a8_linear(qo, so, cpu(wq), cpu(sw))[0])
        h, q2, s2, _ = oracle.residual_rmsnorm_quant(h, y_o, _bits(g2), 1e-6)
        wq, sw = st.weights[l][2]
        y_il, _ = oracle.w8a8_linear(q2, s2, cpu(wq), cpu(sw))     # gate|up rows interleaved by 64
        F = y_il.shape[1] // 2
        blocks = y_il.reshape(-1, F // 64, 2, 64)
        y_gu = np.concatenate([blocks[:, :, 0, :].reshape(-1, F), blocks[:, :, 1, :].reshape(-1, F)], axis=1)
        q3, s3 = oracle.swiglu_quant(y_gu)
        wq, sw = st.weights[l][3]
        yd = oracle.f32_to_bf16(oracle.w8a8_linear(q3, s3, cpu(wq), cpu(sw))[0])
        if l == model["layers"] - 1:
            assert np.array_equal(_bits(st.y_qkv), y_qkv)
            assert np.array_equal(_bits(st.y_o), y_o)
            a_ref = _silu_times(oracle, y_gu[:, :F], y_gu[:, F:])
            assert np.array_equal(np_(st.a_glu).view(np.uint32), a_ref.view(np.uint32))
            assert np.array_equal(_bits(st.y_down), yd)
    h, qf, sf, _ = oracle.residual_rmsnorm_quant(h, yd, _bits(st.norm_final), 1e-6)
    assert np.array_equal(_bits(st.h_res), h)
    tok, _ = oracle.lm_head_argmax(qf, sf, cpu(st.lm_wq), cpu(st.lm_sw))
    assert np.array_equal(np_(st.tokens), tok)
    ln, out = oracle.accept(tok, cpu(st.drafts), B, gamma)
    assert np.array_equal(np_(st.accept_len), ln) and np.array_equal(np_(st.out_tokens), out)
    att_last = np_(st.attn_out[-1]).copy()
    g = st.capture_chain()
    st.tokens.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(np_(st.tokens), tok) and np.array_equal(_bits(st.h_res), h)
    assert np.array_equal(np_(st.attn_out[-1]).view(np.uint32), att_last.view(np.uint32))   # deterministic
