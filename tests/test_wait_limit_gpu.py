"""A bounded in-kernel wait that runs out, on purpose and without faulting
the GPU: the split-K head of the streaming GEMM waits for partial sums that
never come (a test hook keeps the contributing CTAs from publishing them),
gives up after a shortened limit, reports it in the device error word, and
leaves the context usable. The recovery rule of qv.h (zero-fill the
workspace again) then gives oracle-exact results."""
import time

import numpy as np
import pytest
import torch

from gpu_util import np_, rand_codes, rand_scales, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    return _qv


def test_slot_wait_runs_out_and_recovers(qv, oracle):
    M, K, N = 5, 4096, 1024          # 256 tiles over the CTAs: every channel tile is split
    xq = rand_codes((M, K), seed=71).cuda()
    wq = rand_codes((N, K), seed=72).cuda()
    sx = rand_scales(M, seed=73, lo=1e-3, hi=0.2).cuda()
    sw = rand_scales(N, seed=74).cuda()
    y_ref, _ = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    y = torch.full((M, N), float("nan"), device="cuda")
    assert qv.qv_device_error() == 0
    qv.qv_debug_set_slot_wait_ns(2_000_000)          # 2 ms instead of 1 s
    qv.qv_debug_drop_partials(1)
    try:
        t0 = time.perf_counter()
        qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws)
        code = qv.qv_device_error()                  # synchronizes
        elapsed = time.perf_counter() - t0
    finally:
        qv.qv_debug_set_slot_wait_ns(0)
        qv.qv_debug_drop_partials(0)
    assert code & qv.QV_DEVICE_ERR_SLOT_WAIT
    assert elapsed < 0.5
    assert not np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))   # incomplete sums

    ws.zero_()                                       # the recovery rule
    for rep in range(2):
        y.fill_(float("nan"))
        qv.qv_w8a8_linear(xq, sx, wq, sw, y, ws)
        torch.cuda.synchronize()
        assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32)), rep
    assert qv.qv_device_error() == 0


def test_hooks_do_not_touch_later_calls(qv, oracle):
    """drop_partials counts launches: with n = 0 nothing is dropped, and the
    default limit is restored by 0."""
    qv.qv_debug_drop_partials(0)
    qv.qv_debug_set_slot_wait_ns(0)
    M, K, N = 3, 2048, 640
    xq = rand_codes((M, K), seed=81).cuda()
    wq = rand_codes((N, K), seed=82).cuda()
    sx = rand_scales(M, seed=83).cuda()
    sw = rand_scales(N, seed=84).cuda()
    y = torch.empty(M, N, device="cuda")
    qv.qv_w8a8_linear(xq, sx, wq, sw, y, qv.workspace(qv.QV_OP_LINEAR, M, K, N))
    y_ref, _ = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    assert np.array_equal(np_(y).view(np.uint32), y_ref.view(np.uint32))
    assert qv.qv_device_error() == 0


def test_attention_stage_wait_runs_out_and_recovers(qv, oracle):
    """The attention kernel's stage waits: with its key/value loads held back
    (test hook) every wait runs out after the shortened limit, the device
    error word says so, and the next call, with loads, is correct again."""
    from test_attention_gpu import CASES, test_attention_verify
    B, T, Hq, Hkv, D, Lmax, lens = CASES[0]
    qkv = torch.randn(B * T, (Hq + 2 * Hkv) * D, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    kc = torch.randn(B, Lmax, Hkv, D, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16)
    vc = torch.randn(B, Lmax, Hkv, D, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    ln = torch.tensor(lens, dtype=torch.int32)
    ws = torch.empty(qv.qv_attention_workspace_bytes(B, T, Hq, Hkv, D, Lmax), dtype=torch.uint8, device="cuda")
    out = torch.zeros(B * T, Hq * D, device="cuda")
    assert qv.qv_device_error() == 0
    qv.qv_debug_set_slot_wait_ns(2_000_000)          # 2 ms instead of 1 s
    qv.qv_debug_hold_attention_loads(1)
    try:
        t0 = time.perf_counter()
        qv.qv_attention_verify(qkv.cuda(), kc.cuda(), vc.cuda(), ln.cuda(), T, Hq, Hkv, 1.0 / D ** 0.5, out, ws)
        code = qv.qv_device_error()                  # synchronizes
        elapsed = time.perf_counter() - t0
    finally:
        qv.qv_debug_set_slot_wait_ns(0)
        qv.qv_debug_hold_attention_loads(0)
    assert code & qv.QV_DEVICE_ERR_FULL_WAIT
    assert elapsed < 0.5
    # the context is usable and later calls load their stages again
    test_attention_verify(qv, oracle, *CASES[0])
    assert qv.qv_device_error() == 0

