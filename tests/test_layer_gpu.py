"""The layer's fused non-linear steps (qv_rmsnorm_quant, qv_swiglu_quant)
against the oracle, bit for bit: the updated residual stream, the normalized
bf16 activations, the int8 codes and the fp32 token scales."""
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
