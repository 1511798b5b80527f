"""Seeded synthetic inputs shaped like the Quasar evaluation models.

This module only draws random numbers: it holds none of the method's
arithmetic and imports neither the CUDA binding nor the oracle, so tests can
feed the very same tensors to both sides. Values stand in for the real
checkpoints and prompts (Qwen3-8B / OpenPangu-7B on MT-bench, HumanEval,
GSM8k, ...), which are not available; only shapes and value distributions are
imitated:

  * activations ~ N(0, 1) with a fixed set of outlier channels (1% of K,
    chosen without replacement, the same for every token) scaled by 20 --
    the activation outliers that motivate smoothing (gist.science/ja
    summary, section 2.2 "Enhanced SmoothQuant");
  * weights ~ N(0, 0.02);
  * bf16 tensors are rounded from fp32 with torch's round-to-nearest-even.

Sub-seeds are derived from a base seed and a name (crc32) so every tensor of a
workload is reproducible on its own, on the CPU or on the GPU generator.
"""
from __future__ import annotations

import zlib

import torch

QWEN3_8B = {"hidden": 4096, "kv": 1024, "ffn": 12288, "layers": 36, "vocab": 151936}
QWEN3_32B = {"hidden": 5120, "q": 8192, "kv": 1024, "ffn": 25600, "layers": 64, "vocab": 151936}
MODELS = {"qwen3-8b": QWEN3_8B, "qwen3-32b": QWEN3_32B}


def layer_projections(model: dict) -> list[tuple[str, int, int]]:
    """(name, K in-features, N out-features) of one decoder layer's linears."""
    h = model["hidden"]
    q = model.get("q", h)
    return [("q", h, q), ("k", h, model["kv"]), ("v", h, model["kv"]), ("o", q, h),
            ("gate", h, model["ffn"]), ("up", h, model["ffn"]), ("down", model["ffn"], h)]


def subseed(base: int, *names) -> int:
    key = "/".join(str(n) for n in names).encode()
    return (base * 0x9E3779B1 + zlib.crc32(key)) & 0x7FFFFFFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def activations(M: int, K: int, seed: int, dtype=torch.bfloat16, device="cpu",
                outlier_frac: float = 0.01, n_outliers: int | None = None,
                outlier_scale: float = 20.0) -> torch.Tensor:
    """[M, K] N(0,1) activations with outlier channels scaled by `outlier_scale`."""
    g = _gen(seed, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    n = n_outliers if n_outliers is not None else int(round(outlier_frac * K))
    if n > 0:
        cols = torch.randperm(K, generator=g, device=device)[:n]
        x[:, cols] *= outlier_scale
    return x.to(dtype)


def weights(N: int, K: int, seed: int, dtype=torch.bfloat16, device="cpu",
            std: float = 0.02) -> torch.Tensor:
    """[N, K] N(0, std) weights."""
    g = _gen(seed, device)
    w = torch.randn(N, K, generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    return w.to(dtype)


def norm_weights(H: int, seed: int, dtype=torch.bfloat16, device="cpu", std: float = 0.1) -> torch.Tensor:
    """[H] RMSNorm weights 1 + N(0, std)."""
    g = _gen(seed, device)
    w = 1.0 + std * torch.randn(H, generator=g, device=device, dtype=torch.float32)
    return w.to(dtype)


def uniform_tokens(shape, V: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randint(0, V, shape, generator=g, device=device, dtype=torch.int32)


def geometric_drafts(verify_tokens: torch.Tensor, V: int, p: float, seed: int) -> torch.Tensor:
    """Drafts [B, gamma] that agree with the verifier's tokens [B, gamma+1] for
    a prefix of k ~ Geometric(p) successes before the first failure (capped at
    gamma), then differ at position k (guaranteed mismatch), then are uniform.
    Host-side (CPU) helper; the tokens passed in are an input of the workload.
    """
    t = verify_tokens.to("cpu", torch.int64)
    B, G = t.shape
    gamma = G - 1
    g = _gen(seed, "cpu")
    d = torch.randint(0, V, (B, max(gamma, 0)), generator=g, dtype=torch.int64)
    u = torch.rand(B, max(gamma, 1), generator=g, dtype=torch.float64)
    for b in range(B):
        k = 0
        while k < gamma and u[b, k].item() < p:
            k += 1
        for j in range(k):
            d[b, j] = t[b, j]
        if k < gamma:
            off = 1 + int(torch.randint(0, max(V - 1, 1), (1,), generator=g).item())
            d[b, k] = (t[b, k] + off) % V
    return d.to(torch.int32)


def expected_accept_len(p: float, gamma: int) -> float:
    """Mean accepted length of geometric_drafts: 1 + E[min(Geom(p), gamma)]."""
    return 1.0 + sum(p ** i for i in range(1, gamma + 1))


__all__ = ["QWEN3_8B", "QWEN3_32B", "MODELS", "layer_projections", "subseed", "activations", "weights",
           "norm_weights",
           "uniform_tokens", "geometric_drafts", "expected_accept_len"]
