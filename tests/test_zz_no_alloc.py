"""The workspace-free linear entry point, for callers that cannot allocate
device memory (a plugin handed only its input and output buffers, code under
someone else's memory budget): it must give exactly what the regular
qv_w8a8_linear gives with a caller-owned workspace, call after call, since its
built-in scratch buffer is shared and reused. Called through the C ABI.

Kept in its own file named to be collected last, so that a run stopping at the
first failure has already run every other test."""
import ctypes

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


def _c(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


# (M, K, N, y dtype): up to 8, 16, 64 and 80 token rows in one launch; 256
# rows take four launches in a row, each reusing the scratch the one before
# it left zeroed; a bf16 output
@pytest.mark.parametrize("M,K,N,ydt", [(5, 4096, 1024, torch.float32), (4, 256, 512, torch.float32),
                                       (16, 272, 1000, torch.float32), (64, 256, 200, torch.float32),
                                       (80, 512, 384, torch.float32), (256, 256, 300, torch.float32),
                                       (5, 1024, 640, torch.bfloat16)])
def test_noalloc_matches_workspace_linear_twice(qv, oracle, M, K, N, ydt):
    lib = qv.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    ycode = qv.QV_F32 if ydt == torch.float32 else qv.QV_BF16
    for call in range(2):                       # two calls in a row share the scratch
        xq = rand_codes((M, K), seed=100 * call + M).cuda()
        wq = rand_codes((N, K), seed=100 * call + N + 1).cuda()
        sx = rand_scales(M, seed=call + 3, lo=1e-3, hi=0.2).cuda()
        sw = rand_scales(N, seed=call + 4).cuda()
        y_ref = torch.full((M, N), float("nan"), device="cuda", dtype=ydt)
        a_ref = torch.zeros(M, N, dtype=torch.int32, device="cuda")
        st = lib.qv_w8a8_linear(_c(xq), _c(sx), M, K, _c(wq), _c(sw), N, _c(y_ref), ycode, _c(a_ref),
                                _c(ws), ws.numel(), stream)
        assert st == qv.QV_OK, lib.qv_last_error()
        y = torch.full((M, N), float("nan"), device="cuda", dtype=ydt)
        acc = torch.zeros(M, N, dtype=torch.int32, device="cuda")
        st = lib.qv_w8a8_linear_noalloc(_c(xq), _c(sx), M, K, _c(wq), _c(sw), N, _c(y), ycode,
                                        _c(acc), stream)
        assert st == qv.QV_OK, lib.qv_last_error()
        torch.cuda.synchronize()
        # same bits as the call with a caller-owned workspace ...
        assert np.array_equal(np_(acc), np_(a_ref))
        rel = (y.double() - y_ref.double()).abs() / y_ref.double().abs().clamp_min(1e-30)
        assert float(rel.max()) <= 1e-6
        assert torch.equal(y, y_ref)
        # ... and the oracle's: exact integer sums, fp32 (or its bf16 rounding) outputs
        y_o, acc_o = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
        assert np.array_equal(np_(acc), acc_o)
        if ydt == torch.float32:
            assert np.array_equal(np_(y).view(np.uint32), y_o.view(np.uint32))
        else:
            assert np.array_equal(np_(y.view(torch.int16)).view(np.uint16), oracle.f32_to_bf16(y_o))
    assert qv.qv_device_error() == 0


def test_noalloc_binding_checks_on_the_host(qv, oracle):
    """The Python binding of the entry point: a call with float32 tensors goes
    through and matches the oracle; bf16 scales or a mis-shaped acc_debug are
    rejected before anything reaches the library."""
    M, K, N = 5, 512, 256
    xq = rand_codes((M, K), seed=61).cuda()
    wq = rand_codes((N, K), seed=62).cuda()
    sx = rand_scales(M, seed=63, lo=1e-3, hi=0.2).cuda()
    sw = rand_scales(N, seed=64).cuda()
    y = torch.full((M, N), float("nan"), device="cuda")
    acc = torch.zeros(M, N, dtype=torch.int32, device="cuda")
    qv.qv_w8a8_linear_noalloc(xq, sx, wq, sw, y, acc_debug=acc)
    torch.cuda.synchronize()
    y_o, acc_o = oracle.w8a8_linear(np_(xq), np_(sx), np_(wq), np_(sw))
    assert np.array_equal(np_(acc), acc_o) and np.array_equal(np_(y).view(np.uint32), y_o.view(np.uint32))
    canary = torch.full((M, N), 7.0, device="cuda")
    with pytest.raises(ValueError):
        qv.qv_w8a8_linear_noalloc(xq, sx.to(torch.bfloat16), wq, sw, canary)
    with pytest.raises(ValueError):
        qv.qv_w8a8_linear_noalloc(xq, sx, wq, sw, canary, acc_debug=torch.zeros(M, N - 1, dtype=torch.int32,
                                                                                device="cuda"))
    torch.cuda.synchronize()
    assert bool((canary == 7.0).all())


def test_noalloc_covers_every_shape(qv):
    """The split-K slots do not grow with N, so the largest shape the linear
    accepts fits the built-in scratch; a 64-token call with 20000 channels
    (beyond the scratch under a per-channel workspace) matches the call with
    a workspace bit for bit."""
    lib = qv.load()
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 256, 133136, 10 ** 7) <= qv.QV_NOALLOC_SCRATCH_BYTES
    M, K, N = 64, 128, 20000
    xq = rand_codes((M, K), seed=91).cuda()
    wq = rand_codes((N, K), seed=92).cuda()
    sx = rand_scales(M, seed=93).cuda()
    sw = rand_scales(N, seed=94).cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = torch.zeros(qv.qv_workspace_bytes(qv.QV_OP_LINEAR, M, K, N), dtype=torch.uint8, device="cuda")
    y_ref = torch.full((M, N), float("nan"), device="cuda")
    st = lib.qv_w8a8_linear(_c(xq), _c(sx), M, K, _c(wq), _c(sw), N, _c(y_ref), qv.QV_F32, None,
                            _c(ws), ws.numel(), stream)
    assert st == qv.QV_OK, lib.qv_last_error()
    y = torch.full((M, N), float("nan"), device="cuda")
    st = lib.qv_w8a8_linear_noalloc(_c(xq), _c(sx), M, K, _c(wq), _c(sw), N, _c(y), qv.QV_F32, None, stream)
    assert st == qv.QV_OK, lib.qv_last_error()
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)