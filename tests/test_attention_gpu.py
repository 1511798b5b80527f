"""qv_attention_verify against the oracle's binary64 definition: causal
grouped-query attention of the verify tokens over the KV cache and the
step's own keys. Tolerance from the arithmetic: bf16 x bf16 products are
exact in binary32 and a D-term binary32 dot product errs by at most about
(D - 1) 2^-24 sum |q k| (under 1e-4 of a score here), which moves the output
by at most that fraction of max |v|; the base-2 exponentials (scores
scaled by log2 e) add a few ulp. So every output
is within 1e-4 max |v| of the definition. Shapes: the Qwen3-8B layer
(32 query heads, 8 key/value heads, D = 128) with 5 verify tokens, cache
lengths on and around the 16-key block and 64-key stage boundaries (and
ranges of a single stage, which all warps share), the
2048-position cache of the benchmark, no cache, the largest head group
(T * Hq / Hkv = 32), D = 64, and a length above Lmax (clamped). Cache
positions at and past a sequence's length hold NaN: the kernel must take the
step's own rows there and never read a stale cache row."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_bits, np_, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qv():
    require_gpu()
    from quantized_verification_gb300 import qv as _qv
    _qv.load()
    return _qv


CASES = [  # B, T, Hq, Hkv, D, Lmax, lens
    (1, 5, 32, 8, 128, 1024, [1000]),
    (2, 5, 32, 8, 128, 300, [300, 17]),
    (3, 3, 8, 2, 64, 130, [0, 128, 129]),
    (1, 1, 4, 4, 64, 0, [0]),
    (2, 8, 16, 4, 128, 2000, [1999, 513]),
    (1, 4, 8, 1, 128, 257, [257]),
    (2, 2, 4, 2, 64, 100, [150, 100]),
    (1, 5, 32, 8, 128, 2048, [2048]),
    (2, 5, 32, 8, 128, 2100, [2043, 77]),
    (3, 4, 16, 4, 64, 520, [511, 64, 1]),
    # 10, 11 and 12 blocks of 16 keys per CTA (more stages than the ring
    # holds, partial last stages); ranges of one stage (at most 4 blocks) are
    # shared by all warps (300, 17, 77 and short lengths above)
    (1, 5, 32, 8, 128, 1300, [1270]),
    (1, 5, 32, 8, 128, 1400, [1395]),
    (1, 5, 32, 8, 128, 1525, [1525]),
    # 32 blocks per CTA: the ring is refilled as its stages drain
    (1, 5, 32, 8, 128, 4096, [4000]),
    # D = 64 with three and four n8 tiles of query rows (R = 20 and 32)
    (1, 5, 32, 8, 64, 900, [850]),
    (2, 8, 16, 4, 64, 700, [650, 333]),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,Lmax,lens", CASES)
def test_attention_verify(qv, oracle, B, T, Hq, Hkv, D, Lmax, lens):
    g = torch.Generator().manual_seed(B * 7919 + T * 31 + Lmax)
    qkv = torch.randn(B * T, (Hq + 2 * Hkv) * D, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, Lmax, Hkv, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Lmax, Hkv, D, generator=g).to(torch.bfloat16)
    ln = torch.tensor(lens, dtype=torch.int32)
    for bb, n in enumerate(lens):                     # stale cache rows: never read
        kc[bb, max(0, min(n, Lmax)):] = float("nan")
        vc[bb, max(0, min(n, Lmax)):] = float("nan")
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    ws = torch.empty(qv.qv_attention_workspace_bytes(B, T, Hq, Hkv, D, Lmax), dtype=torch.uint8, device="cuda")
    out = torch.full((B * T, Hq * D), float("nan"), device="cuda")
    qv.qv_attention_verify(qkv.cuda(), kc.cuda(), vc.cuda(), ln.cuda(), T, Hq, Hkv, np.float32(scale), out, ws)
    torch.cuda.synchronize()
    clamped = np.clip(np.array(lens), 0, Lmax).astype(np.int32)
    ref = oracle.attention_verify(bf16_bits(qkv).reshape(B * T, -1), bf16_bits(kc).reshape(B, Lmax, Hkv, D),
                                  bf16_bits(vc).reshape(B, Lmax, Hkv, D), clamped, T, Hq, Hkv, D,
                                  float(np.float32(scale)))
    vmax = max(float(vc.float().nan_to_num(0.0).abs().max()) if Lmax else 0.0,
               float(qkv[:, (Hq + Hkv) * D:].float().abs().max()))
    err = np.abs(np_(out).astype(np.float64) - ref)
    assert np.all(np.isfinite(np_(out)))
    assert float(err.max()) <= 1e-4 * vmax, (float(err.max()), vmax)


def test_attention_rejects_bad_shapes(qv):
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    assert qv.qv_attention_workspace_bytes(1, 9, 32, 8, 128, 100) == 0        # T * G > 32
    assert qv.qv_attention_workspace_bytes(1, 5, 32, 8, 96, 100) == 0         # D not 64 / 128
    assert qv.qv_attention_workspace_bytes(1, 5, 30, 8, 128, 100) == 0        # Hq % Hkv
    out = torch.full((5, 4096), 7.0, device="cuda")
    with pytest.raises(qv.QVError):                                              # scale must be > 0
        qv.qv_attention_verify(torch.zeros(5, 48 * 128, dtype=torch.bfloat16, device="cuda"),
                               torch.zeros(1, 4, 8, 128, dtype=torch.bfloat16, device="cuda"),
                               torch.zeros(1, 4, 8, 128, dtype=torch.bfloat16, device="cuda"),
                               torch.zeros(1, dtype=torch.int32, device="cuda"), 5, 32, 8, 0.0, out, z)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())                                              # nothing was enqueued
