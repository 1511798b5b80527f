"""C-ABI checks that need no GPU: the library builds, loads, exports every
symbol include/qv.h declares, and rejects bad arguments on the host before
touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_verification_gb300 import build, qv
    build.build()
    return qv.load()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"^QV_API\s+[\w\s\*]+?\b(qv_\w+)\s*\(", src, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"qv_quantize_act", "qv_w8a8_linear", "qv_lm_head_argmax", "qv_accept"} <= names
    for n in names:
        assert hasattr(lib, n), n
    from quantized_verification_gb300 import qv
    assert set(qv.EXPORTS) == names


def test_workspace_sizes(lib):
    from quantized_verification_gb300 import qv
    # linear: one split-K slot of 128 x MP 8-byte words per CTA (at most 160
    # CTAs), whatever N; M=5 -> MP=8
    slots8 = 160 * 128 * 8 * 8
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 5, 4096, 4096) == slots8
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 5, 4096, 1000) == slots8
    assert qv.qv_workspace_bytes(qv.QV_OP_BF16_LINEAR, 5, 4096, 1000) == slots8
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 17, 4096, 1000) == 4 * slots8       # MP = 32
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 200, 4096, 1000) == 10 * slots8     # 80-row slices
    assert qv.qv_workspace_bytes(qv.QV_OP_BF16_LINEAR, 200, 4096, 1000) == 8 * slots8  # 64-row slices
    # LM head: slots + per-token keys + the done counter on its own lines
    assert qv.qv_workspace_bytes(qv.QV_OP_LM_HEAD, 5, 4096, 151936) == slots8 + 8 * 8 + 5 * 128
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 0, 4096, 16) == 0
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 5, 100, 16) == 0     # K % 16
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 257, 4096, 16) == 0  # M > QV_MAX_M
    assert qv.qv_workspace_bytes(qv.QV_OP_LINEAR, 5, 133152, 16) == 0  # K > QV_MAX_K
    # *_ACT: the GEMM workspace, 256-byte aligned, then M*K codes and M scales
    for op, base in ((qv.QV_OP_LINEAR_ACT, qv.QV_OP_LINEAR), (qv.QV_OP_LM_HEAD_ACT, qv.QV_OP_LM_HEAD)):
        for (M, K, N) in ((5, 4096, 4096), (17, 272, 1000), (1, 16, 1)):
            g = qv.qv_workspace_bytes(base, M, K, N)
            off = (g + 255) // 256 * 256
            assert qv.qv_workspace_bytes(op, M, K, N) == off + (M * K + 15) // 16 * 16 + (4 * M + 15) // 16 * 16
        assert qv.qv_workspace_bytes(op, 5, 100, 16) == 0


def test_host_validation_without_gpu(lib):
    from quantized_verification_gb300 import qv
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.qv_quantize_act(None, 0, 4, 256, None, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert b"null" in lib.qv_last_error()
    assert lib.qv_quantize_act(fake, 0, 4, 250, None, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert b"multiple of 16" in lib.qv_last_error()
    assert lib.qv_quantize_act(P(0x1001), 0, 4, 256, None, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert b"aligned" in lib.qv_last_error()
    assert lib.qv_quantize_act(fake, 7, 4, 256, None, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w8a8_linear(fake, fake, 0, 256, fake, fake, 8, fake, 0, None, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w8a8_linear(fake, fake, 4, 256, fake, fake, 8, fake, 0, None, None, 0, None) == qv.QV_ERR_WORKSPACE
    assert lib.qv_w8a8_linear(fake, fake, 4, 256, fake, fake, 8, fake, 0, None, fake, 16, None) == qv.QV_ERR_WORKSPACE
    assert b"needed" in lib.qv_last_error()
    assert lib.qv_lm_head_argmax(fake, fake, 4, 133152, fake, fake, 8, fake, None, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_accept(fake, None, 2, 3, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_accept(fake, fake, 0, 3, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_accept(fake, fake, 2, -1, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_bf16_linear(fake, 300, 256, fake, 8, fake, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    # fused act-quant calls: arguments checked before any CUDA call
    assert lib.qv_w8a8_linear_act(None, 1, None, 5, 256, fake, fake, 8, fake, 0, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w8a8_linear_act(fake, 3, None, 5, 256, fake, fake, 8, fake, 0, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w8a8_linear_act(fake, 1, P(0x1004), 5, 256, fake, fake, 8, fake, 0, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert b"aligned" in lib.qv_last_error()
    assert lib.qv_w8a8_linear_act(fake, 1, None, 257, 256, fake, fake, 8, fake, 0, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w8a8_linear_act(fake, 1, None, 5, 256, fake, fake, 8, None, 0, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w8a8_linear_act(fake, 1, None, 5, 256, fake, fake, 8, fake, 0, fake, 64, None) == qv.QV_ERR_WORKSPACE
    assert lib.qv_lm_head_argmax_act(fake, 1, None, 5, 256, fake, fake, 8, None, None, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert b"tokens" in lib.qv_last_error()
    assert lib.qv_lm_head_argmax_act(fake, 1, None, 5, 250, fake, fake, 8, fake, None, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    # W4A8: K must be a multiple of 32 (two codes per byte, 16-byte rows)
    assert lib.qv_w4a8_linear(fake, fake, 4, 272, fake, fake, 8, fake, 0, None, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert b"multiple of 32" in lib.qv_last_error()
    assert lib.qv_w4a8_linear(fake, fake, 4, 256, fake, fake, 8, None, 0, None, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w4a8_linear(fake, fake, 4, 256, fake, fake, 8, fake, 0, None, fake, 16, None) == qv.QV_ERR_WORKSPACE
    assert lib.qv_w4a8_linear(fake, fake, 4, 133152, fake, fake, 8, fake, 0, None, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w4a8_swiglu(fake, fake, 4, 256, fake, fake, 96, fake, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w4a8_lm_head_argmax(fake, fake, 4, 256, fake, fake, 8, None, None, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_w4a8_lm_head_argmax(fake, fake, 4, 16, fake, fake, 8, fake, None, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_quantize_weight_w4(fake, 0, 8, 48, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_quantize_weight_w4(fake, 5, 8, 64, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_quantize_weight_w4(fake, 0, 8, 64, P(0x1008), fake, None) == qv.QV_ERR_INVALID_ARG
    # attention over a short KV cache
    F32 = ctypes.c_float
    assert lib.qv_attention_verify(None, fake, fake, fake, 1, 5, 32, 8, 128, 16, F32(0.1), fake, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_attention_verify(fake, fake, fake, fake, 1, 9, 32, 8, 128, 16, F32(0.1), fake, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_attention_verify(fake, None, fake, fake, 1, 5, 32, 8, 128, 16, F32(0.1), fake, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_attention_verify(fake, fake, fake, fake, 1, 5, 32, 8, 128, 16, F32(0.0), fake, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_attention_verify(P(0x1008), fake, fake, fake, 1, 5, 32, 8, 128, 16, F32(0.1), fake, fake, 1 << 22, None) == qv.QV_ERR_INVALID_ARG
    # no workspace: 16 bytes for any valid shape, 0 for an invalid one
    assert qv.qv_attention_workspace_bytes(1, 5, 32, 8, 128, 500) == 16
    assert qv.qv_attention_workspace_bytes(1, 5, 32, 8, 96, 500) == 0
    # logit fidelity
    assert lib.qv_logit_fidelity(None, fake, 2, 10, fake, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_logit_fidelity(fake, fake, 0, 10, fake, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_logit_fidelity(fake, fake, 2, 0, fake, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_logit_fidelity(fake, P(0x1002), 2, 10, fake, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    # greedy tree verification
    assert lib.qv_tree_accept(None, fake, fake, 1, 16, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_tree_accept(fake, fake, fake, 1, 1025, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_tree_accept(fake, fake, fake, 0, 16, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_tree_accept(fake, P(0x1002), fake, 1, 16, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    # speculative sampling at T > 0
    U64 = ctypes.c_uint64
    assert lib.qv_spec_sample(None, fake, fake, 1, 4, 1000, F32(1.0), U64(1), fake, fake, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_spec_sample(fake, None, fake, 1, 4, 1000, F32(1.0), U64(1), fake, fake, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_spec_sample(fake, fake, fake, 1, 4, 1000, F32(0.0), U64(1), fake, fake, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert b"temperature" in lib.qv_last_error()
    assert lib.qv_spec_sample(fake, fake, fake, 1, 4, 0, F32(1.0), U64(1), fake, fake, fake, 1 << 20, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_spec_sample(fake, fake, fake, 1, 4, 1000, F32(1.0), U64(1), fake, fake, fake, 16, None) == qv.QV_ERR_WORKSPACE
    # chunks of 2048 tokens: per (row, chunk) a float max, two u64 sums and a
    # u128 draw sum; 32 bytes of statistics and an int decision per row;
    # every region rounded up to 256 bytes
    r256 = lambda v: (v + 255) // 256 * 256
    for M, V in ((5, 151936), (80, 151936), (1, 1), (3, 2049)):
        S = (V + 2047) // 2048
        want = r256(M * S * 4) + 2 * r256(M * S * 8) + r256(M * 32) + r256(M * S * 16) + r256(M * 4)
        assert qv.qv_workspace_bytes(qv.QV_OP_SPEC_SAMPLE, M, 16, V) == want
    assert qv.qv_workspace_bytes(qv.QV_OP_SPEC_SAMPLE, 5, 16, 0) == 0
    assert qv.qv_workspace_bytes(qv.QV_OP_SPEC_SAMPLE, 0, 16, 1000) == 0
    # the layer's fused non-linear steps
    assert lib.qv_rmsnorm_quant(None, None, fake, F32(1e-6), None, 5, 256, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_rmsnorm_quant(fake, None, fake, F32(1e-6), None, 5, 264, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert b"multiple of 16" in lib.qv_last_error()
    assert lib.qv_rmsnorm_quant(fake, None, fake, F32(1e-6), None, 5, 16400, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_rmsnorm_quant(fake, None, fake, F32(-1.0), None, 5, 256, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_rmsnorm_quant(fake, P(0x1008), fake, F32(1e-6), None, 5, 256, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert b"aligned" in lib.qv_last_error()
    assert lib.qv_rmsnorm_quant(fake, None, fake, F32(1e-6), None, 0, 256, fake, fake, None, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_swiglu_quant(None, 5, 256, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_swiglu_quant(fake, 5, 8, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_swiglu_quant(fake, 5, 32784, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert lib.qv_swiglu_quant(P(0x1004), 5, 256, fake, fake, None) == qv.QV_ERR_INVALID_ARG
    assert b"aligned" in lib.qv_last_error()


def test_binding_rejects_host_tensors(lib):
    import torch
    from quantized_verification_gb300 import qv
    x = torch.zeros(4, 256)
    with pytest.raises(ValueError):
        qv.qv_quantize_act(x, torch.zeros(4, 256, dtype=torch.int8), torch.zeros(4))
