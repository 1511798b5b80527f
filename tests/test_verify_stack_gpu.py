"""qv_verify_stack (one persistent launch per verify pass) against the oracle
and against the per-op calls: identical bits for every linear output, the
argmax tokens, and the acceptance."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_bits, np_, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    return _qv


def _zeroed_part(qv, M, n_max):
    """Bytes at the start of the stack workspace that every call leaves zero
    (the rest holds the int8 codes of the last phase)."""
    return qv.qv_workspace_bytes(qv.QV_OP_VERIFY_STACK, M, 16, n_max) - 16 * M


def _make(shapes, M, V, Kl, seed, dtype, smooth):
    from quantized_verification_gb300 import synth
    lin = []
    for i, (K, N) in enumerate(shapes):
        x = synth.activations(M, K, seed=seed + 10 * i, dtype=dtype)
        if i == 1 and M >= 2:
            x[1] = 0                                    # an all-zero token row
        w = synth.weights(N, K, seed=seed + 10 * i + 1, dtype=dtype)
        mul = None
        if smooth and i % 2 == 0:
            g = torch.Generator().manual_seed(seed + i)
            mul = (torch.rand(K, generator=g) * 2 + 0.5).float()
        lin.append((x, w, mul))
    xl = synth.activations(M, Kl, seed=seed + 999, dtype=dtype)
    wl = synth.weights(V, Kl, seed=seed + 998, dtype=dtype)
    return lin, xl, wl


def _oracle_chain(oracle, lin, xl, wl, dtype):
    bf = dtype == torch.bfloat16
    conv = bf16_bits if bf else np_
    ys = []
    for (x, w, mul) in lin:
        xq, sx = oracle.quantize_rows(conv(x), None if mul is None else np_(mul), bf16=bf)
        wq, sw = oracle.quantize_rows(conv(w), bf16=bf)
        y, _ = oracle.w8a8_linear(xq, sx, wq, sw)
        ys.append(y)
    xq, sx = oracle.quantize_rows(conv(xl), bf16=bf)
    wq, sw = oracle.quantize_rows(conv(wl), bf16=bf)
    tok, mx = oracle.lm_head_argmax(xq, sx, wq, sw)
    return ys, tok, mx


# (K, N) shapes: one tile, ragged N and K tails, K with more chunks than the
# activation buffer holds (windowed quantization), tiny phases with idle CTAs
SHAPES = [(256, 384), (384, 200), (128, 1000), (6144, 640), (272, 130), (256, 129), (4096, 300)]


@pytest.mark.parametrize("M,B,gamma,dtype,smooth", [
    (5, 1, 4, torch.bfloat16, False), (4, 1, 3, torch.float32, True), (16, 4, 3, torch.bfloat16, False),
    (1, 1, 0, torch.bfloat16, True), (10, 2, 4, torch.float32, False), (8, 2, 3, torch.bfloat16, True)])
def test_verify_stack_matches_oracle(qv, oracle, M, B, gamma, dtype, smooth):
    from quantized_verification_gb300 import synth
    V, Kl = 3000, 256
    lin, xl, wl = _make(SHAPES, M, V, Kl, seed=M * 7 + gamma, dtype=dtype, smooth=smooth)
    ys_ref, t_ref, m_ref = _oracle_chain(oracle, lin, xl, wl, dtype)
    draft = synth.geometric_drafts(torch.from_numpy(t_ref).view(B, gamma + 1), V, 0.7, seed=5)
    l_ref, o_ref = oracle.accept(t_ref, np_(draft), B, gamma)

    dev = "cuda"
    keep, descs, ys = [], [], []
    for (x, w, mul), (K, N) in zip(lin, SHAPES):
        wq = torch.empty(N, K, dtype=torch.int8, device=dev)
        sw = torch.empty(N, device=dev)
        qv.qv_quantize_weight(w.to(dev), wq, sw)
        xd = x.to(dev)
        md = mul.to(dev) if mul is not None else None
        y = torch.full((M, N), float("nan"), device=dev)
        keep += [wq, sw, xd, md]
        ys.append(y)
        descs.append(qv.linear_desc(xd, wq, sw, y=y, act_mul=md))
    lq = torch.empty(V, Kl, dtype=torch.int8, device=dev)
    ls = torch.empty(V, device=dev)
    qv.qv_quantize_weight(wl.to(dev), lq, ls)
    xld = xl.to(dev)
    lm = qv.linear_desc(xld, lq, ls)
    nmax = max([N for (_, N) in SHAPES] + [V])
    kmax = max([K for (K, _) in SHAPES] + [Kl])
    ws = torch.zeros(qv.qv_workspace_bytes(qv.QV_OP_VERIFY_STACK, M, kmax, nmax), dtype=torch.uint8, device=dev)
    tok = torch.full((M,), -3, dtype=torch.int32, device=dev)
    mx = torch.full((M,), float("nan"), device=dev)
    ln = torch.full((B,), -3, dtype=torch.int32, device=dev)
    out = torch.full((B, gamma + 1), -3, dtype=torch.int32, device=dev)
    dd = draft.to(dev) if gamma > 0 else None
    for rep in range(2):                      # the workspace is reused as left
        qv.qv_verify_stack(descs, lm, M, dtype, ws, tokens=tok, max_logit=mx, draft=dd,
                           accept_len=ln, out_tokens=out)
        torch.cuda.synchronize()
        for i, y_ref in enumerate(ys_ref):
            assert np.array_equal(np_(ys[i]).view(np.uint32), y_ref.view(np.uint32)), f"linear {i}"
        assert np.array_equal(np_(tok), t_ref)
        assert np.array_equal(np_(mx), m_ref)
        assert np.array_equal(np_(ln), l_ref) and np.array_equal(np_(out), o_ref)
        assert int(ws[: _zeroed_part(qv, M, nmax)].count_nonzero()) == 0
    assert qv.qv_device_error() == 0


def test_verify_stack_quantization_near_ties(qv, oracle):
    """Activations whose quotient x/s sits next to a rounding boundary, where a
    product with the reciprocal of s can round to the other integer."""
    M, K, N = 4, 1024, 256
    g = np.random.default_rng(17)
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        amax = np.float32(g.uniform(0.5, 4.0))
        s = np.float32(amax / np.float32(127))
        # quotients j + 0.5 +- a few ulps
        j = g.integers(-126, 126, K).astype(np.float32)
        q = (j + np.float32(0.5)) * s
        q = np.nextafter(q, np.where(g.random(K) < 0.5, np.inf, -np.inf).astype(np.float32))
        x[m] = q
        x[m, 0] = amax
    xt = torch.from_numpy(x)
    wq = torch.randint(-127, 128, (N, K), dtype=torch.int8)
    sw = (torch.rand(N) * 1e-3 + 1e-4).float()
    y = torch.zeros(M, N, device="cuda")
    xd, wd, sd = xt.cuda(), wq.cuda(), sw.cuda()          # kept alive across the call
    d = qv.linear_desc(xd, wd, sd, y=y)
    ws = torch.zeros(qv.qv_workspace_bytes(qv.QV_OP_VERIFY_STACK, M, K, N), dtype=torch.uint8, device="cuda")
    qv.qv_verify_stack([d], None, M, torch.float32, ws)
    torch.cuda.synchronize()
    xq, sx = oracle.quantize_rows(x)
    y_ref, _ = oracle.w8a8_linear(xq, sx, np_(wq), np_(sw))
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))


def test_verify_stack_many_phases_split_launches(qv, oracle):
    """More phases than one launch holds: split into consecutive launches."""
    M, K, N = 5, 128, 136
    n = 163
    g = torch.Generator().manual_seed(3)
    dev = "cuda"
    x = torch.randn(n, M, K, generator=g).to(torch.bfloat16)
    wq = torch.randint(-127, 128, (n, N, K), generator=g, dtype=torch.int8)
    sw = (torch.rand(n, N, generator=g) * 1e-3 + 1e-4).float()
    xd, wd, sd = x.to(dev), wq.to(dev), sw.to(dev)
    y = torch.zeros(n, M, N, device=dev)
    descs = [qv.linear_desc(xd[i], wd[i], sd[i], y=y[i]) for i in range(n)]
    ws = torch.zeros(qv.qv_workspace_bytes(qv.QV_OP_VERIFY_STACK, M, K, N), dtype=torch.uint8, device=dev)
    qv.qv_verify_stack(descs, None, M, torch.bfloat16, ws)
    torch.cuda.synchronize()
    for i in (0, 1, 148, 149, 150, 162):
        xq, sx = oracle.quantize_rows(bf16_bits(x[i]), bf16=True)
        y_ref, _ = oracle.w8a8_linear(xq, sx, np_(wq[i]), np_(sw[i]))
        assert np.array_equal(np_(y[i]).view(np.uint32), y_ref.view(np.uint32)), i
    assert int(ws[: _zeroed_part(qv, M, N)].count_nonzero()) == 0


def test_verify_stack_equals_per_op_calls(qv):
    """A small stack through both entry points of the library, in graphs."""
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 128, "ffn": 512, "layers": 3, "vocab": 1000}
    st = VerifyStack(model=model, B=1, gamma=4, seed=7)
    st.drafts.copy_(synth.uniform_tokens((1, 4), 1000, seed=1).cuda())
    st.enqueue()
    torch.cuda.synchronize()
    y1, t1, l1, o1 = st.y.clone(), st.tokens.clone(), st.accept_len.clone(), st.out_tokens.clone()
    st.y.zero_(); st.tokens.zero_(); st.accept_len.zero_(); st.out_tokens.zero_()
    st.enqueue_fused()
    torch.cuda.synchronize()
    assert torch.equal(st.tokens, t1) and torch.equal(st.accept_len, l1) and torch.equal(st.out_tokens, o1)
    assert torch.equal(st.y, y1)
    st.capture_fused()
    st.tokens.zero_()
    st.graph_fused.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.tokens, t1)


def _host_io(st, layout):
    """The pinned host tensors of a step from host memory: "merged" as the
    stack lays them out (drafts and inputs in one buffer, both results in
    one buffer: one copy each way), "separate" as unrelated pinned tensors
    (one copy per tensor)."""
    host_in, host_d = st.pinned_host_inputs()
    if layout == "merged":
        out_len, out_tok = st.pinned_host_results()
    else:
        host_in, host_d = host_in.clone().pin_memory(), host_d.clone().pin_memory()
        out_len = torch.empty(st.B, dtype=torch.int32).pin_memory()
        out_tok = torch.empty(st.B, st.gamma + 1, dtype=torch.int32).pin_memory()
    return host_in, host_d, out_len, out_tok


@pytest.mark.parametrize("layout", ["merged", "separate"])
def test_step_from_host_buffers(qv, layout):
    """The end-to-end step: the packed host inputs, copied in and run
    through the captured graph, give the same tokens as the device-resident
    step, and the result lands in the pinned host tensors."""
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 128, "ffn": 512, "layers": 2, "vocab": 1000}
    st = VerifyStack(model=model, B=1, gamma=4, seed=11)
    st.drafts.copy_(synth.uniform_tokens((1, 4), 1000, seed=2).cuda())
    g = st.capture()
    g.replay()
    torch.cuda.synchronize()
    l1, o1 = st.accept_len.clone(), st.out_tokens.clone()
    host_in, host_d, out_len, out_tok = _host_io(st, layout)
    assert host_in.numel() == sum(x.numel() for li in st.inputs for x in li) + st.h_final.numel()
    st.in_buf.zero_()
    st.drafts.zero_()
    out_len.fill_(-1)
    out_tok.fill_(-1)
    h2d, d2h = st.step_from_host(host_in, host_d, out_len, out_tok, graph=g)
    torch.cuda.synchronize()
    assert h2d == host_in.numel() * 2 + host_d.numel() * 4 and d2h == 4 + 20
    assert torch.equal(out_len, l1.cpu()) and torch.equal(out_tok, o1.cpu())


@pytest.mark.parametrize("layout,B,gamma", [("merged", 1, 4), ("separate", 1, 4), ("merged", 2, 3),
                                             ("merged", 1, 0), ("separate", 3, 0)])
def test_step_graph_from_host_buffers(qv, layout, B, gamma):
    """The end-to-end step as one graph: the host inputs go in as the first
    layer's (with the drafts) and the rest on a parallel branch that the
    second layer waits for, the results come back into the pinned host
    tensors, and they equal the device-resident step's, replay after replay,
    also when the device copies of the inputs were cleared in between; with
    several sequences and with no drafts (an empty drafts slice)."""
    from quantized_verification_gb300 import synth
    from quantized_verification_gb300.stack import VerifyStack
    model = {"hidden": 256, "kv": 128, "ffn": 512, "layers": 3, "vocab": 1000}
    st = VerifyStack(model=model, B=B, gamma=gamma, seed=13)
    if gamma > 0:
        st.drafts.copy_(synth.uniform_tokens((B, gamma), 1000, seed=3).cuda())
    g = st.capture()
    g.replay()
    torch.cuda.synchronize()
    l1, o1 = st.accept_len.clone(), st.out_tokens.clone()
    host_in, host_d, out_len, out_tok = _host_io(st, layout)
    ge, h2d, d2h = st.capture_from_host(host_in, host_d, out_len, out_tok)
    assert h2d == host_in.numel() * 2 + host_d.numel() * 4 and d2h == 4 * B * (gamma + 2)
    for rep in range(3):
        st.in_buf.zero_()
        st.drafts.zero_()
        out_len.fill_(-1)
        out_tok.fill_(-1)
        ge.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_len, l1.cpu()) and torch.equal(out_tok, o1.cpu()), rep


def test_verify_stack_rejects_large_m(qv):
    M, K, N = 17, 128, 128
    dev = "cuda"
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=dev)
    wq = torch.zeros(N, K, dtype=torch.int8, device=dev)
    sw = torch.ones(N, device=dev)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(qv.QVError) as ei:
        qv.qv_verify_stack([qv.linear_desc(x, wq, sw)], None, M, torch.bfloat16, ws)
    assert ei.value.status == qv.QV_ERR_UNSUPPORTED
