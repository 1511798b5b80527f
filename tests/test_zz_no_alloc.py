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


@pytest.mark.parametrize("M,K,N", [(5, 4096, 1024), (4, 256, 512), (16, 272, 1000), (64, 256, 200)])
def test_noalloc_matches_workspace_linear_twice(qv, M, K, N):
    lib = qv.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws = qv.workspace(qv.QV_OP_LINEAR, M, K, N)
    for call in range(2):                       # two calls in a row share the scratch
        xq = rand_codes((M, K), seed=100 * call + M).cuda()
        wq = rand_codes((N, K), seed=100 * call + N + 1).cuda()
        sx = rand_scales(M, seed=call + 3, lo=1e-3, hi=0.2).cuda()
        sw = rand_scales(N, seed=call + 4).cuda()
        y_ref = torch.full((M, N), float("nan"), device="cuda")
        a_ref = torch.zeros(M, N, dtype=torch.int32, device="cuda")
        st = lib.qv_w8a8_linear(_c(xq), _c(sx), M, K, _c(wq), _c(sw), N, _c(y_ref), qv.QV_F32, _c(a_ref),
                                _c(ws), ws.numel(), stream)
        assert st == qv.QV_OK, lib.qv_last_error()
        y = torch.full((M, N), float("nan"), device="cuda")
        acc = torch.zeros(M, N, dtype=torch.int32, device="cuda")
        st = lib.qv_w8a8_linear_noalloc(_c(xq), _c(sx), M, K, _c(wq), _c(sw), N, _c(y), qv.QV_F32,
                                        _c(acc), stream)
        assert st == qv.QV_OK, lib.qv_last_error()
        torch.cuda.synchronize()
        assert np.array_equal(np_(acc), np_(a_ref))
        rel = (y.double() - y_ref.double()).abs() / y_ref.double().abs().clamp_min(1e-30)
        assert float(rel.max()) <= 1e-6
        assert torch.equal(y, y_ref)


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