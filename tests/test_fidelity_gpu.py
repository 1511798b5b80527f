"""qv_logit_fidelity against the oracle's binary64 definition: the KL
divergence per row within the tolerance of its binary32 terms and binary64
block sums (relative 2e-3, absolute 1e-6), and the top-1 indices exactly
(lowest index on ties), for close, shifted, identical and unrelated logits,
at the Qwen3 vocabulary and at small ones. Each row is split among the CTAs
of a cluster in slices of a multiple of 4 entries: the small vocabularies
leave some CTAs a ragged or an empty slice, and rows that start off a
16-byte boundary take the scalar loads."""
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


def _run(qv, a, b):
    M, V = a.shape
    kl = torch.full((M,), float("nan"), device="cuda")
    ta = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    tb = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    qv.qv_logit_fidelity(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), kl, ta, tb)
    torch.cuda.synchronize()
    return np_(kl).astype(np.float64), np_(ta), np_(tb)


@pytest.mark.parametrize("M,V,mode", [(5, 151936, "close"), (3, 1000, "far"), (4, 64, "same"),
                                      (2, 5000, "shift"), (7, 3001, "close"), (1, 1, "same"),
                                      (3, 2100000, "close"), (2, 29, "close"), (3, 10, "far"),
                                      (2, 33, "shift")])
def test_logit_fidelity(qv, oracle, M, V, mode):
    rng = np.random.default_rng(M * 1000 + V % 977)
    a = rng.normal(0, 3, (M, V)).astype(np.float32)
    if V > 40:
        a[0, [11, 37]] = a[0].max() + 1                 # a tie: the first index wins
    if mode == "close":
        b = (a + rng.normal(0, 0.05, a.shape)).astype(np.float32)
    elif mode == "far":
        b = rng.normal(0, 3, (M, V)).astype(np.float32)
    elif mode == "shift":
        b = (a + np.float32(3.0)).astype(np.float32)
    else:
        b = a.copy()
    kl, ta, tb = _run(qv, a, b)
    kl_ref, ta_ref, tb_ref = oracle.logit_fidelity(a, b)
    assert np.array_equal(ta, ta_ref) and np.array_equal(tb, tb_ref)
    assert np.all(np.abs(kl - kl_ref) <= 2e-3 * kl_ref + 1e-6), (kl, kl_ref)
    if mode == "same":
        assert np.all(kl == 0.0)
    if V > 40:
        assert ta[0] == 11


@pytest.mark.parametrize("off_a,off_b", [(1, 1), (0, 3), (2, 0)])
def test_logit_fidelity_unaligned_rows(qv, oracle, off_a, off_b):
    """Rows whose base is 4-byte but not 16-byte aligned (a view at an
    offset of 1 to 3 floats into a larger buffer), at a vocabulary that is a
    multiple of 4: the same results as the aligned rows."""
    M, V = 3, 4096
    rng = np.random.default_rng(71 + off_a * 3 + off_b)
    a = rng.normal(0, 3, (M, V)).astype(np.float32)
    b = (a + rng.normal(0, 0.1, a.shape)).astype(np.float32)
    a[1, 4000] = a[1].max() + 2
    ba = torch.zeros(M * V + 4, device="cuda")
    bb = torch.zeros(M * V + 4, device="cuda")
    ga = ba[off_a:off_a + M * V].view(M, V)
    gb = bb[off_b:off_b + M * V].view(M, V)
    ga.copy_(torch.from_numpy(a))
    gb.copy_(torch.from_numpy(b))
    kl = torch.full((M,), float("nan"), device="cuda")
    ta = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    tb = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    qv.qv_logit_fidelity(ga, gb, kl, ta, tb)
    torch.cuda.synchronize()
    kl_ref, ta_ref, tb_ref = oracle.logit_fidelity(a, b)
    assert np.array_equal(np_(ta), ta_ref) and np.array_equal(np_(tb), tb_ref)
    assert ta_ref[1] == 4000
    k = np_(kl).astype(np.float64)
    assert np.all(np.abs(k - kl_ref) <= 2e-3 * kl_ref + 1e-6), (k, kl_ref)
