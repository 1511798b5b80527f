"""Pins for the CPU oracle: checks against things other than the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the Quasar summaries and plain
mathematics fix: the hand-worked example under ``tests/golden``, exact
rational arithmetic (``tests/exact.py``), brute force on tiny inputs, library
routines that compute the same textbook quantity (numpy integer matmul,
numpy argmax, torch bf16 conversion, numpy binary32 arithmetic), and the
invariants of the method. The mutation tests run every pin against
deliberately broken copies of the oracle to show that each plausible mistake
fails at least one of them.
"""
from __future__ import annotations

import itertools
import json
import os
from fractions import Fraction

import numpy as np

from exact import dequant_exact, f32, quantize_row_exact, rne_int, round_to_f32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(a_f32: np.ndarray) -> np.ndarray:
    """bf16 patterns of values that are exactly representable in bf16."""
    u = np.ascontiguousarray(a_f32, dtype=np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# worked example
# ---------------------------------------------------------------------------

def pin_worked_example(o):
    g = _golden("worked_2x3x4.json")
    x = np.array(g["x_f32"], dtype=np.float32)
    w = np.array(g["w_f32"], dtype=np.float32)
    for bf16 in (False, True):
        xin = _bf16_bits(x) if bf16 else x
        win = _bf16_bits(w) if bf16 else w
        xq, sx = o.quantize_rows(xin, bf16=bf16)
        wq, sw = o.quantize_rows(win, bf16=bf16)
        assert xq.tolist() == g["xq"], (bf16, xq)
        assert sx.tolist() == g["sx"]
        assert wq.tolist() == g["wq"], (bf16, wq)
        assert sw.tolist() == g["sw"]
    xq = np.array(g["xq"], dtype=np.int8)
    wq = np.array(g["wq"], dtype=np.int8)
    sx = np.array(g["sx"], dtype=np.float32)
    sw = np.array(g["sw"], dtype=np.float32)
    y, acc = o.w8a8_linear(xq, sx, wq, sw)
    assert acc.tolist() == g["acc"]
    assert np.array_equal(y, np.array(g["y_num_over_8192"], dtype=np.float64) / 8192)
    tok, mv = o.argmax_rows(y)
    assert tok.tolist() == g["tokens"]
    assert mv.tolist() == [v / 8192 for v in g["max_logit_num_over_8192"]]
    tok2, mv2 = o.lm_head_argmax(xq, sx, wq, sw)
    assert tok2.tolist() == g["tokens"]
    assert mv2.tolist() == mv.tolist()
    t = np.array(g["tokens"], dtype=np.int32)
    for case in g["accept_cases"]:
        ln, out = o.accept(t, np.array(case["draft"], dtype=np.int32), 1, 1)
        assert ln.tolist() == [case["len"]], case
        assert out.tolist() == [case["out"]], case


# ---------------------------------------------------------------------------
# a0 / a1 quantization
# ---------------------------------------------------------------------------

def _hard_quant_rows(rng, n_rows=6, K=64):
    """Rows containing values whose quotient x/s lands within an ulp of a
    rounding boundary, found with numpy binary32 arithmetic: there division
    by s and multiplication by 127/amax give different codes."""
    rows = []
    for _ in range(n_rows):
        amax = np.float32(rng.uniform(0.5, 4.0))
        s = np.float32(amax / np.float32(127))
        r = np.float32(np.float32(127) / amax)
        cand = (rng.uniform(-amax, amax, size=400000)).astype(np.float32)
        q_div = np.rint(cand / s)
        q_mul = np.rint(cand * r)
        hard = cand[q_div != q_mul]
        picked = list(hard[: K - 1])
        while len(picked) < K - 1:
            picked.append(np.float32(rng.uniform(-amax, amax)))
        row = np.array([amax] + picked, dtype=np.float32)
        rng.shuffle(row)
        rows.append(row)
    return np.stack(rows)


def pin_quantize_exact_rational(o):
    rng = np.random.default_rng(1234)
    K = 64
    rows = [
        rng.standard_normal(K).astype(np.float32),
        (rng.standard_normal(K) * 1e-3).astype(np.float32),
        (rng.standard_normal(K) * 3e4).astype(np.float32),
        # tiny row with subnormal quotients / scales
        (rng.standard_normal(K) * 1e-38).astype(np.float32),
    ]
    outl = rng.standard_normal(K).astype(np.float32)
    outl[[3, 17]] *= 20
    rows.append(outl)
    x = np.concatenate([np.stack(rows), _hard_quant_rows(rng)])
    q, s = o.quantize_rows(x)
    for i in range(x.shape[0]):
        q_ref, s_ref = quantize_row_exact(x[i])
        assert np.float32(s[i]) == s_ref, (i, s[i], s_ref)
        assert q[i].tolist() == q_ref, i


def pin_quantize_ties(o):
    # amax = 127/64 gives s = 1/64 exactly; x = (j + 1/2)/64 are exact ties
    js = np.arange(-126, 126)
    row = np.concatenate([[127.0], (js + 0.5)]) / 64.0
    x = row.astype(np.float32)[None, :]
    q, s = o.quantize_rows(x)
    assert s[0] == np.float32(1 / 64)
    expect = [127] + [rne_int(Fraction(2 * j + 1, 2)) for j in js]
    assert q[0].tolist() == expect


def pin_quantize_invariants(o):
    rng = np.random.default_rng(99)
    x = rng.standard_normal((32, 200)).astype(np.float32)
    x[:, rng.choice(200, 4, replace=False)] *= 20
    q, s = o.quantize_rows(x)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    assert np.all(s >= 0)
    idx = np.argmax(np.abs(x), axis=1)
    for i in range(32):
        assert q[i, idx[i]] == (127 if x[i, idx[i]] > 0 else -127)
        # codes reproduce the row to within half a step
        err = np.abs(q[i].astype(np.float64) * float(s[i]) - x[i].astype(np.float64))
        assert np.all(err <= 0.5 * float(s[i]) * (1 + 1e-6) + 1e-30)
    # an all-zero row and a row whose amax/127 underflows to zero
    z = np.zeros((2, 16), dtype=np.float32)
    z[1, 5] = np.float32(63 * 2.0 ** -149)
    qz, sz = o.quantize_rows(z)
    assert np.all(qz == 0) and np.all(sz == 0)


def pin_quantize_smoothing(o):
    rng = np.random.default_rng(7)
    K = 48
    x = rng.standard_normal((5, K)).astype(np.float32)
    c = rng.uniform(0.25, 4.0, K).astype(np.float32)
    q, s = o.quantize_rows(x, c)
    xs = (x * c).astype(np.float32)       # numpy binary32 multiply: one rounding
    q2, s2 = o.quantize_rows(xs)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    for i in range(2):
        q_ref, s_ref = quantize_row_exact(x[i], c)
        assert q[i].tolist() == q_ref and s[i] == s_ref
    # bf16 input path with smoothing
    xb = o.f32_to_bf16(x)
    qb, sb = o.quantize_rows(xb, c, bf16=True)
    xw = o.bf16_to_f32(xb)
    qb2, sb2 = o.quantize_rows((xw * c).astype(np.float32))
    assert np.array_equal(qb, qb2) and np.array_equal(sb, sb2)
    # identity multiplier equals no multiplier
    q3, s3 = o.quantize_rows(x, np.ones(K, np.float32))
    q4, s4 = o.quantize_rows(x)
    assert np.array_equal(q3, q4) and np.array_equal(s3, s4)


# ---------------------------------------------------------------------------
# a2 integer GEMM and dequantization
# ---------------------------------------------------------------------------

def pin_int8_matmul_bruteforce(o):
    rng = np.random.default_rng(5)
    for (M, N, K) in [(1, 1, 1), (2, 3, 5), (3, 7, 8), (4, 8, 6)]:
        xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
        wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
        acc = o.int8_matmul(xq, wq)
        for m in range(M):
            for n in range(N):
                ref = sum(int(xq[m, k]) * int(wq[n, k]) for k in range(K))
                assert acc[m, n] == ref, (M, N, K, m, n)
    # enumerate every pair of 1-element rows over a small code range
    vals = np.arange(-127, 128, 9, dtype=np.int8)
    acc = o.int8_matmul(vals[:, None], vals[:, None])
    assert np.array_equal(acc, np.outer(vals.astype(np.int64), vals.astype(np.int64)))
    # textbook: an integer matrix product
    xq = rng.integers(-127, 128, (6, 300)).astype(np.int8)
    wq = rng.integers(-127, 128, (40, 300)).astype(np.int8)
    assert np.array_equal(o.int8_matmul(xq, wq),
                          xq.astype(np.int64) @ wq.astype(np.int64).T)


def pin_int8_matmul_range(o):
    # the largest K with exact int32 sums: floor((2^31-1)/127^2) = 133144
    K = (2 ** 31 - 1) // (127 * 127)
    assert K == 133144
    x = np.full((1, K), 127, np.int8)
    w = np.concatenate([np.full((1, K), 127, np.int8), np.full((1, K), -127, np.int8)])
    acc = o.int8_matmul(x, w)
    assert acc.tolist() == [[K * 16129, -K * 16129]]
    try:
        o.int8_matmul(np.full((1, K + 1), 127, np.int8), np.full((1, K + 1), 127, np.int8))
    except OverflowError:
        pass
    else:
        raise AssertionError("K beyond the int32 limit was not reported")


def pin_dequant_exact(o):
    rng = np.random.default_rng(11)
    M, N = 3, 50
    acc = rng.integers(-2 ** 28, 2 ** 28, (M, N)).astype(np.int32)
    acc[0, :5] = [0, 1, -1, 2 ** 24 + 1, -(2 ** 25) - 3]      # rounding of int -> float
    sx = (rng.uniform(1e-3, 1e-1, M)).astype(np.float32)
    sw = (rng.uniform(1e-5, 1e-3, N)).astype(np.float32)
    y = o.dequant(acc, sx, sw)
    for m in range(M):
        for n in range(N):
            ref = dequant_exact(int(acc[m, n]), sx[m], sw[n])
            assert y[m, n] == ref, (m, n, y[m, n], ref)
            exact = Fraction(int(acc[m, n])) * f32(sx[m]) * f32(sw[n])
            if exact != 0:
                assert abs(f32(y[m, n]) - exact) <= abs(exact) * Fraction(3, 2 ** 24)
    # numpy binary32 arithmetic does the same two products
    ynp = acc.astype(np.float32) * (sx[:, None] * sw[None, :]).astype(np.float32)
    assert np.array_equal(y, ynp.astype(np.float32))


# ---------------------------------------------------------------------------
# a3 argmax
# ---------------------------------------------------------------------------

def pin_argmax(o):
    rng = np.random.default_rng(21)
    y = rng.integers(-5, 6, (40, 17)).astype(np.float32)    # many ties
    y[0] = 0.0
    y[1, :] = -1.0
    y[1, 4] = -0.0
    y[1, 9] = 0.0                                            # -0 and +0 tie
    tok, mv = o.argmax_rows(y)
    for m in range(y.shape[0]):
        ref = sorted(range(y.shape[1]), key=lambda n: (-float(y[m, n]), n))[0]
        assert tok[m] == ref, (m, tok[m], ref)
        assert mv[m] == y[m].max()
    assert np.array_equal(tok, np.argmax(y, axis=1).astype(np.int32))
    assert tok[1] == 4
    # lm head on random codes equals an independent composition
    xq = rng.integers(-127, 128, (4, 24)).astype(np.int8)
    wq = rng.integers(-127, 128, (37, 24)).astype(np.int8)
    wq[20] = wq[3]                                            # duplicate rows tie
    sx = rng.uniform(0.01, 0.02, 4).astype(np.float32)
    sw = np.full(37, np.float32(0.004))
    t2, m2 = o.lm_head_argmax(xq, sx, wq, sw)
    acc = xq.astype(np.int64) @ wq.astype(np.int64).T
    ynp = acc.astype(np.float32) * (sx[:, None] * sw[None, :]).astype(np.float32)
    assert np.array_equal(t2, np.argmax(ynp, axis=1).astype(np.int32))
    assert np.array_equal(m2, ynp.max(axis=1))


# ---------------------------------------------------------------------------
# a4 acceptance
# ---------------------------------------------------------------------------

def _accept_by_definition(t_row, d_row, gamma):
    best = 0
    for i in range(gamma + 1):           # i drafts accepted iff the first i all match
        if all(d_row[j] == t_row[j] for j in range(i)):
            best = i
    out = list(t_row[: best + 1]) + [-1] * (gamma - best)
    return best + 1, out


def pin_accept_enumeration(o):
    V = 3
    for gamma in range(0, 4):
        for t_row in itertools.product(range(V), repeat=gamma + 1):
            drafts = list(itertools.product(range(V), repeat=gamma))
            B = len(drafts)
            t = np.array([t_row] * B, dtype=np.int32)
            d = np.array(drafts, dtype=np.int32).reshape(B, gamma)
            ln, out = o.accept(t, d, B, gamma)
            for b in range(B):
                L, ref = _accept_by_definition(t_row, drafts[b], gamma)
                assert ln[b] == L and out[b].tolist() == ref, (gamma, t_row, drafts[b])
                assert 1 <= ln[b] <= gamma + 1
                assert list(out[b, : ln[b] - 1]) == list(drafts[b][: ln[b] - 1])
                assert out[b, ln[b] - 1] == t_row[ln[b] - 1]


# ---------------------------------------------------------------------------
# bf16 conversion and the fp64 comparator reference
# ---------------------------------------------------------------------------

def pin_bf16(o):
    import torch
    rng = np.random.default_rng(3)
    f = (rng.standard_normal(5000) * np.exp(rng.uniform(-20, 20, 5000))).astype(np.float32)
    ties = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80C000, 0x3F804000,
                     0x00008000, 0x00018000], dtype=np.uint32).view(np.float32)
    f = np.concatenate([f, ties])
    h = o.f32_to_bf16(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h, ref)
    assert h[-7:].tolist() == [0x3F80, 0x3F82, 0xBF80, 0x3F81, 0x3F80, 0x0000, 0x0002]
    back = o.bf16_to_f32(h)
    assert np.array_equal(back.view(np.uint32), h.astype(np.uint32) << 16)


def pin_linear_f64(o):
    rng = np.random.default_rng(8)
    M, N, K = 3, 5, 40
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    y = o.linear_f64(x, w)
    for m in range(M):
        for n in range(N):
            exact = sum(f32(x[m, k]) * f32(w[n, k]) for k in range(K))
            mag = sum(abs(f32(x[m, k]) * f32(w[n, k])) for k in range(K))
            assert abs(Fraction(float(y[m, n])) - exact) <= mag * Fraction(K, 2 ** 52)
    ynp = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.allclose(y, ynp, rtol=1e-12, atol=1e-15)



# ---------------------------------------------------------------------------
# f1: the non-linear steps between the linears of a layer (residual add,
# RMSNorm, SiLU(gate) * up), each followed by the a1 quantization.
# ---------------------------------------------------------------------------
def _ulp32(v: float) -> float:
    return float(np.spacing(np.float32(abs(v))))


def pin_layer_exp(o):
    """The layer's exp is the mathematical e^x to 2 ulp over its range, exact
    at 0, +inf above 88, 0 below -87, and non-decreasing."""
    import math
    xs = np.concatenate([np.linspace(-87.0, 88.0, 4001, dtype=np.float32),
                         np.float32([-1e-7, 1e-7, 0.5, -0.5, 0.34657359, -0.34657359, 1.0, -1.0])])
    for x in xs:
        e = o.exp(float(x))
        t = math.exp(float(x))
        assert abs(e - t) <= 2 * _ulp32(t), (float(x), e, t)
    assert o.exp(0.0) == 1.0
    assert o.exp(88.5) == float("inf") and o.exp(-90.0) == 0.0
    grid = np.sort(xs)
    vals = [o.exp(float(x)) for x in grid]
    assert all(b >= a for a, b in zip(vals, vals[1:]))


def pin_silu(o):
    """silu(v) = v / (1 + e^-v): against the binary64 formula to 4 ulp on
    [-20, 20]; exactly 0 at 0, v for large v, -0 for very negative v."""
    import math
    for v in np.linspace(-20.0, 20.0, 801, dtype=np.float32):
        ref = float(v) / (1.0 + math.exp(-float(v)))
        got = o.silu(float(v))
        assert abs(got - ref) <= 4 * _ulp32(ref) + 1e-30, (float(v), got, ref)
    assert o.silu(0.0) == 0.0
    assert o.silu(100.0) == 100.0
    assert o.silu(-100.0) == 0.0


def pin_swiglu_quant(o):
    """a = silu(gate) * up, then a1. (1) Random rows: every code within one of
    the binary64 reference's round(a / s) and the scale within 4 ulp of
    max|a| / 127. (2) Saturated gate (silu(100) = 100 exactly): the codes are
    the exact-rational a1 quantization of fl(100 * up) (swapping gate and up
    breaks it). (3) up = 0: all codes and the scale are 0."""
    import math
    rng = np.random.default_rng(31)
    M, F = 3, 64
    gu = rng.normal(0.0, 2.0, (M, 2 * F)).astype(np.float32)
    q, s = o.swiglu_quant(gu)
    for m in range(M):
        a = [float(g) / (1.0 + math.exp(-float(g))) * float(u) for g, u in zip(gu[m, :F], gu[m, F:])]
        amax = max(abs(v) for v in a)
        assert abs(float(s[m]) - amax / 127.0) <= 4 * _ulp32(amax / 127.0)
        ref = np.array([round(v / (amax / 127.0)) for v in a])
        assert np.max(np.abs(q[m].astype(np.int64) - ref)) <= 1
        assert np.mean(q[m].astype(np.int64) == ref) > 0.9
    up = rng.normal(0.0, 1.0, (2, F)).astype(np.float32)
    gu2 = np.concatenate([np.full((2, F), 100.0, dtype=np.float32), up], axis=1)
    q2, s2 = o.swiglu_quant(gu2)
    for m in range(2):
        qe, se = quantize_row_exact((np.float32(100.0) * up[m]).astype(np.float32))
        assert list(q2[m]) == list(qe) and np.float32(s2[m]) == se
    gu3 = np.concatenate([rng.normal(0.0, 1.0, (1, F)).astype(np.float32), np.zeros((1, F), np.float32)], axis=1)
    q3, s3 = o.swiglu_quant(gu3)
    assert not q3.any() and s3[0] == 0.0


def pin_rmsnorm_quant(o):
    """Residual add + RMSNorm + a1.
    (1) Constant rows c (a power of two) with g = 1, eps = 0: x = sign(c),
        so every code is +-127 and the scale is fl(1/127).
    (2) d = -h: the sum is 0, so codes and scale are 0.
    (3) The residual sum equals torch's bf16 addition (fp32 sum, rne to bf16).
    (4) Scaling h by 2 (exact in bf16) with eps = 0 leaves x and the codes.
    (5) x is within two bf16 roundings of the binary64 g * h / sqrt(mean(h^2) + eps).
    (6) The codes are the exact-rational a1 quantization of x."""
    import torch
    H = 96
    one = np.full(H, 0x3F80, dtype=np.uint16)                      # bf16 1.0
    hc = np.stack([np.full(H, 0x4000, np.uint16), np.full(H, 0xBE80, np.uint16)])   # 2.0, -0.25
    _, q, s, x = o.residual_rmsnorm_quant(hc, None, one, 0.0)
    assert (q[0] == 127).all() and (q[1] == -127).all()
    assert s[0] == np.float32(1.0) / np.float32(127.0) and s[1] == s[0]
    rng = np.random.default_rng(41)
    hf = rng.normal(0.0, 1.0, (3, H)).astype(np.float32)
    hb = torch.from_numpy(hf).to(torch.bfloat16)
    h_bits = hb.view(torch.int16).numpy().view(np.uint16)
    neg_bits = (-hb).view(torch.int16).numpy().view(np.uint16)
    h0, q0, s0, _ = o.residual_rmsnorm_quant(h_bits, neg_bits, one, 1e-6)
    assert not q0.any() and not s0.any() and not (h0 & 0x7FFF).any()
    db = torch.from_numpy(rng.normal(0.0, 0.5, (3, H)).astype(np.float32)).to(torch.bfloat16)
    d_bits = db.view(torch.int16).numpy().view(np.uint16)
    g_f = rng.uniform(0.5, 1.5, H).astype(np.float32)
    g_bits = torch.from_numpy(g_f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    h1, q1, s1, x1 = o.residual_rmsnorm_quant(h_bits, d_bits, g_bits, 1e-6)
    ref_sum = (hb.float() + db.float()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(h1, ref_sum)
    h2x = (torch.from_numpy(hf).to(torch.bfloat16) * 2).view(torch.int16).numpy().view(np.uint16)
    _, qa, _, xa = o.residual_rmsnorm_quant(h_bits, None, g_bits, 0.0)
    _, qb, _, xb = o.residual_rmsnorm_quant(h2x, None, g_bits, 0.0)
    assert np.array_equal(xa, xb) and np.array_equal(qa, qb)
    hv = torch.from_numpy(h1.view(np.int16)).view(torch.bfloat16).double().numpy()
    gv = torch.from_numpy(g_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    xv = torch.from_numpy(x1.view(np.int16)).view(torch.bfloat16).double().numpy()
    for m in range(3):
        ref = gv * hv[m] / np.sqrt(np.mean(hv[m] ** 2) + 1e-6)
        assert np.all(np.abs(xv[m] - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)
        xf = torch.from_numpy(x1[m].view(np.int16)).view(torch.bfloat16).float().numpy()
        qe, se = quantize_row_exact(xf)
        assert list(q1[m]) == list(qe) and np.float32(s1[m]) == se


# ---------------------------------------------------------------------------
# f2: lossless rejection sampling at T > 0
# ---------------------------------------------------------------------------
def pin_splitmix64_kat(o):
    """SplitMix64 seeded with 0: its published first outputs."""
    assert [o.splitmix64(0, n) for n in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                      0x06C45D188009454F]


def _softmax64(z, T):
    z = np.asarray(z, dtype=np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def _chi2_ok(counts, probs, n):
    """Pearson chi-square of counts against probs, far from rejection
    (the 1e-4 upper quantile of chi2 with df <= 9 is below 40)."""
    exp = np.asarray(probs) * n
    mask = exp > 0
    stat = float(np.sum((np.asarray(counts)[mask] - exp[mask]) ** 2 / exp[mask]))
    return stat < 40.0 and np.all(np.asarray(counts)[~mask] == 0)


def pin_spec_lossless(o):
    """The defining property of speculative sampling: with drafts drawn from
    any draft distribution q, the emitted tokens are distributed as the
    verifier's p. Over 20000 seeds (drafts drawn from q by an independent
    generator): the first token follows p_0, the second one, given that the
    first draft was kept, follows p_1, and the bonus after two kept drafts
    follows p_2 (chi-square)."""
    V, gamma, T = 6, 2, 0.8
    z = np.float32([[1.0, 0.2, -0.5, 2.0, 0.0, -1.0], [0.5, -0.3, 1.5, 0.1, -2.0, 0.7],
                    [-1.0, 0.5, 2.0, 0.0, 1.0, -0.5]])
    q = np.float32([[0.05, 0.3, 0.1, 0.15, 0.25, 0.15], [0.2, 0.2, 0.1, 0.1, 0.3, 0.1]])
    qn = q.astype(np.float64) / q.astype(np.float64).sum(axis=1, keepdims=True)
    drafter = np.random.default_rng(2024)
    n = 20000
    first = np.zeros(V)
    second = np.zeros(V)
    n2 = 0
    third = np.zeros(V)
    n3 = 0
    for seed in range(n):
        d = np.int32([[drafter.choice(V, p=qn[0]), drafter.choice(V, p=qn[1])]])
        ln, out = o.spec_sample(z, d, q, 1, gamma, T, seed * 7919 + 13)
        first[out[0, 0]] += 1
        if ln[0] >= 2:
            second[out[0, 1]] += 1
            n2 += 1
        if ln[0] == 3:
            third[out[0, 2]] += 1
            n3 += 1
    assert _chi2_ok(first, _softmax64(z[0], T), n)
    assert n2 > 1000 and _chi2_ok(second, _softmax64(z[1], T), n2)
    assert n3 > 500 and _chi2_ok(third, _softmax64(z[2], T), n3)


def pin_draw_index(o):
    """Inverse-CDF draw on integer weights, worked by hand: weights
    [0, 3, 0, 5] (total 8) split [0, 2^24) into u24 < 3 * 2^21 -> token 1 and
    the rest -> token 3; a zero weight is never drawn."""
    w = [0, 3, 0, 5]
    assert o.draw_index(w, 0) == 1
    assert o.draw_index(w, 3 * 2 ** 21 - 1) == 1
    assert o.draw_index(w, 3 * 2 ** 21) == 3
    assert o.draw_index(w, 2 ** 24 - 1) == 3
    for u in range(0, 2 ** 24, 2 ** 18):
        assert o.draw_index(w, u) in (1, 3)
    assert o.draw_index([7], 12345) == 0


def pin_spec_special_cases(o):
    """(1) q equal to p (flat logits, flat draft): every draft is kept.
    (2) p(d) = 0: the draft is never kept and never drawn as the replacement.
    (3) Logits and T both scaled by 2 (exact in binary32): the same outputs.
    (4) Invariants: len in [1, gamma+1], the kept drafts are emitted in order."""
    V, gamma, B = 8, 3, 4
    z = np.zeros((B * (gamma + 1), V), np.float32)
    q = np.ones((B * gamma, V), np.float32)
    d = np.random.default_rng(3).integers(0, V, (B, gamma)).astype(np.int32)
    for seed in range(50):
        ln, _ = o.spec_sample(z, d, q, B, gamma, 1.0, seed)
        assert (ln == gamma + 1).all()
    rng = np.random.default_rng(5)
    z2 = rng.normal(0, 1, (B * (gamma + 1), V)).astype(np.float32)
    for b in range(B):
        z2[b * (gamma + 1), d[b, 0]] = -1000.0
    q2 = rng.uniform(0.01, 1.0, (B * gamma, V)).astype(np.float32)
    for seed in range(50):
        ln, out = o.spec_sample(z2, d, q2, B, gamma, 1.0, seed)
        assert (ln == 1).all() and all(out[b, 0] != d[b, 0] for b in range(B))
        ln2, out2 = o.spec_sample(z2 * np.float32(2), d, q2, B, gamma, 2.0, seed)
        assert np.array_equal(ln, ln2) and np.array_equal(out, out2)
    z3 = rng.normal(0, 2, (B * (gamma + 1), V)).astype(np.float32)
    for seed in range(50):
        ln, out = o.spec_sample(z3, d, q2, B, gamma, 0.7, seed)
        for b in range(B):
            assert 1 <= ln[b] <= gamma + 1
            assert list(out[b, : ln[b] - 1]) == list(d[b, : ln[b] - 1])
            assert 0 <= out[b, ln[b] - 1] < V and (out[b, ln[b]:] == -1).all()


# ---------------------------------------------------------------------------
# f3: tree verification at T = 0
# ---------------------------------------------------------------------------
def _random_tree(rng, N, V):
    par = np.full(N, -1, np.int32)
    for i in range(1, N):
        par[i] = rng.integers(0, i)
    return par


def pin_tree_chain_is_linear(o):
    """A chain-shaped tree (parent of node i is i-1) is the linear rule:
    the same lengths and tokens as a4 on the chain's drafts."""
    rng = np.random.default_rng(17)
    B, gamma, V = 64, 5, 3
    t = rng.integers(0, V, (B, gamma + 1)).astype(np.int32)
    dl = rng.integers(0, V, (B, gamma)).astype(np.int32)
    par = np.tile(np.arange(-1, gamma, dtype=np.int32), (B, 1))
    d = np.concatenate([np.zeros((B, 1), np.int32), dl], axis=1)
    ln, out, node = o.tree_accept(t, d, par)
    ln_ref, out_ref = o.accept(t, dl, B, gamma)
    assert np.array_equal(ln, ln_ref) and np.array_equal(out, out_ref)
    assert np.array_equal(node, ln - 1)


def pin_tree_bruteforce(o):
    """Random tiny trees: every root path checked on its own (walk up from
    each node, all edges matching); the deepest matching node, lowest index
    among the deepest, its path and bonus, against the oracle."""
    rng = np.random.default_rng(23)
    for _ in range(300):
        N = int(rng.integers(1, 9))
        V = int(rng.integers(1, 4))
        par = _random_tree(rng, N, V)
        t = rng.integers(0, V, N).astype(np.int32)
        d = rng.integers(0, V, N).astype(np.int32)
        best, best_depth = 0, 0
        for i in range(N):
            path, j, ok = [], i, True
            while j != 0:
                p = int(par[j])
                ok = ok and d[j] == t[p]
                path.append(j)
                j = p
            if ok and len(path) > best_depth:
                best, best_depth = i, len(path)
        exp_out = [int(d[j]) for j in reversed(_path(par, best))] + [int(t[best])]
        exp_out += [-1] * (N - len(exp_out))
        ln, out, node = o.tree_accept(t[None], d[None], par[None])
        assert ln[0] == best_depth + 1 and node[0] == best and list(out[0]) == exp_out


def _path(par, i):
    out = []
    while i != 0:
        out.append(i)
        i = int(par[i])
    return out

# ---------------------------------------------------------------------------
# f4: W4A8
# ---------------------------------------------------------------------------

def pin_w4_worked_example(o):
    """The hand-worked W4A8 example: codes, scales, packed bytes, integer
    sums, outputs and the token."""
    g = _golden("w4a8_worked_2x1x6.json")
    w = (np.array(g["w_num"], dtype=np.float64) / np.array(g["w_den"], dtype=np.float64)[:, None]).astype(np.float32)
    for bf16 in (False, True):
        q, s = o.quantize_rows_w4(_bf16_bits(w) if bf16 else w, bf16=bf16)
        assert q.tolist() == g["q"], (bf16, q)
        assert s.tolist() == g["s"]
    packed = o.pack_w4(np.array(g["q"], dtype=np.int8))
    assert packed.tolist() == g["packed"]
    assert o.unpack_w4(np.array(g["packed"], dtype=np.uint8)).tolist() == g["q"]
    xq = np.array(g["xq"], dtype=np.int8)
    sx = np.array(g["sx"], dtype=np.float32)
    sw = np.array(g["s"], dtype=np.float32)
    y, acc = o.w4a8_linear(xq, sx, packed, sw)
    assert acc.tolist() == g["acc"]
    assert np.array_equal(y, np.array(g["y_num_over_512"], dtype=np.float64) / 512)
    tok, _ = o.w4a8_lm_head_argmax(xq, sx, packed, sw)
    assert tok.tolist() == g["token"]


def pin_w4_quantize_exact_rational(o):
    """int4 codes and scales against exact rational arithmetic with one
    binary32 rounding per operation (s = fl(amax/7), q = rne(fl(w/s)))."""
    rng = np.random.default_rng(4321)
    K = 64
    rows = [rng.standard_normal(K).astype(np.float32),
            (rng.standard_normal(K) * 1e-3).astype(np.float32),
            (rng.standard_normal(K) * 3e4).astype(np.float32),
            (rng.standard_normal(K) * 1e-38).astype(np.float32)]
    # quotients within an ulp of a half-integer: division by s and
    # multiplication by 7/amax disagree there
    for _ in range(4):
        amax = np.float32(rng.uniform(0.5, 4.0))
        s = np.float32(amax / np.float32(7))
        cand = rng.uniform(-amax, amax, size=200000).astype(np.float32)
        hard = cand[np.rint(cand / s) != np.rint(cand * np.float32(np.float32(7) / amax))]
        row = np.concatenate([[amax], hard[: K - 1]]).astype(np.float32)
        row = np.concatenate([row, rng.uniform(-amax, amax, K - row.size).astype(np.float32)])
        rows.append(row)
    x = np.stack(rows)
    q, s = o.quantize_rows_w4(x)
    for i in range(x.shape[0]):
        q_ref, s_ref = quantize_row_exact(x[i], qmax=7)
        assert np.float32(s[i]) == s_ref, (i, s[i], s_ref)
        assert q[i].tolist() == q_ref, i
    assert int(np.abs(q).max()) <= 7


def pin_w4_pack_roundtrip(o):
    """Every pair of codes in [-8, 7] survives packing, every byte survives
    unpacking, and a code's nibble sits where the format puts it: a lone
    code at an even index lands in the low nibble of its byte."""
    pairs = np.array([[a, b] for a in range(-8, 8) for b in range(-8, 8)], dtype=np.int8)
    q = pairs.reshape(1, -1)
    assert np.array_equal(o.unpack_w4(o.pack_w4(q)), q)
    allb = np.arange(256, dtype=np.uint8).reshape(1, -1)
    assert np.array_equal(o.pack_w4(o.unpack_w4(allb)), allb)
    one = np.zeros((1, 8), dtype=np.int8)
    one[0, 2] = 1          # code 2 -> byte 1, bits 0-3
    assert o.pack_w4(one).tolist() == [[0, 1, 0, 0]]
    one[0, 2], one[0, 5] = 0, -1   # code 5 -> byte 2, bits 4-7 = 0xF
    assert o.pack_w4(one).tolist() == [[0, 0, 0xF0, 0]]


def pin_w4_linear_bruteforce(o):
    """W4A8 sums by Python integers over nibbles read off the packed bytes,
    for small random shapes."""
    rng = np.random.default_rng(77)
    for M, K, N in ((1, 2, 1), (3, 6, 4), (2, 32, 5)):
        xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
        packed = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
        sx = rng.uniform(1e-3, 1e-1, M).astype(np.float32)
        sw = rng.uniform(1e-3, 1e-1, N).astype(np.float32)
        y, acc = o.w4a8_linear(xq, sx, packed, sw)
        for m in range(M):
            for n in range(N):
                tot = 0
                for j in range(K // 2):
                    byte = int(packed[n, j])
                    lo, hi = byte % 16, byte // 16
                    lo = lo - 16 if lo > 7 else lo
                    hi = hi - 16 if hi > 7 else hi
                    tot += int(xq[m, 2 * j]) * lo + int(xq[m, 2 * j + 1]) * hi
                assert int(acc[m, n]) == tot
                assert y[m, n] == dequant_exact(tot, sx[m], sw[n])


# ---------------------------------------------------------------------------
# f3': logit fidelity
# ---------------------------------------------------------------------------

def pin_fidelity_closed_forms(o):
    """KL of a distribution with itself is 0, softmax ignores a constant
    shift of the logits, and two tokens give the textbook binary KL."""
    rng = np.random.default_rng(5)
    a = rng.normal(0, 3, (4, 1000)).astype(np.float32)
    kl, ta, tb = o.logit_fidelity(a, a)
    assert np.all(kl == 0.0) and np.array_equal(ta, tb)
    kl, _, _ = o.logit_fidelity(a, (a + np.float32(4.0)).astype(np.float32))
    assert np.all(np.abs(kl) < 1e-12)
    import math
    for x, y in ((0.3, -1.2), (2.0, 2.5), (-4.0, 1.0)):
        x, y = float(np.float32(x)), float(np.float32(y))   # the logits the oracle sees
        p1 = 1.0 / (1.0 + math.exp(-x))      # softmax of (x, 0)
        q1 = 1.0 / (1.0 + math.exp(-y))
        ref = p1 * math.log(p1 / q1) + (1 - p1) * math.log((1 - p1) / (1 - q1))
        kl, ta, tb = o.logit_fidelity(np.float32([[x, 0.0]]), np.float32([[y, 0.0]]))
        assert abs(kl[0] - ref) <= 1e-12 * max(1.0, ref), (x, y, kl[0], ref)
        assert ta[0] == (0 if np.float32(x) > 0 else 1) and tb[0] == (0 if np.float32(y) > 0 else 1)


def pin_fidelity_scipy(o):
    """KL against scipy's relative entropy of the two softmax distributions,
    and the top-1 indices against numpy's argmax (first index on ties)."""
    from scipy.special import softmax
    from scipy.stats import entropy
    rng = np.random.default_rng(8)
    a = rng.normal(0, 2, (6, 3000)).astype(np.float32)
    b = (a + rng.normal(0, 0.3, a.shape)).astype(np.float32)
    b[1] = rng.normal(0, 2, 3000)                   # an unrelated row
    a[2, 17] = a[2, 1234] = a[2].max() + 1          # a tie: the first index wins
    kl, ta, tb = o.logit_fidelity(a, b)
    for m in range(a.shape[0]):
        ref = entropy(softmax(a[m].astype(np.float64)), softmax(b[m].astype(np.float64)))
        assert abs(kl[m] - ref) <= 1e-10 * max(1.0, ref), (m, kl[m], ref)
    assert np.array_equal(ta, np.argmax(a, axis=1)) and np.array_equal(tb, np.argmax(b, axis=1))
    assert ta[2] == 17


# ---------------------------------------------------------------------------
# f1': attention over a short KV cache
# ---------------------------------------------------------------------------

def _attn_case(rng, B, T, Hq, Hkv, D, Lmax, lens):
    f = lambda *s: _bf16_bits(np.round(rng.normal(0, 1, s) * 64).astype(np.float32) / np.float32(64))
    return f(B * T, (Hq + 2 * Hkv) * D), f(B, Lmax, Hkv, D), f(B, Lmax, Hkv, D), np.array(lens, np.int32)


def pin_attention_numpy(o):
    """Against numpy matrix products and scipy's softmax over the visible
    keys of each query (cache, then the step's tokens up to itself), with
    query head h reading key/value head h // (Hq / Hkv)."""
    from scipy.special import softmax
    rng = np.random.default_rng(31)
    B, T, Hq, Hkv, D, Lmax = 2, 3, 4, 2, 8, 5
    qkv, kc, vc, lens = _attn_case(rng, B, T, Hq, Hkv, D, Lmax, [5, 2])
    scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    out = o.attention_verify(qkv, kc, vc, lens, T, Hq, Hkv, D, scale)
    w = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Q = w(qkv[:, : Hq * D]).reshape(B, T, Hq, D)
    Kn = w(qkv[:, Hq * D:(Hq + Hkv) * D]).reshape(B, T, Hkv, D)
    Vn = w(qkv[:, (Hq + Hkv) * D:]).reshape(B, T, Hkv, D)
    for b in range(B):
        L = int(lens[b])
        Kall = np.concatenate([w(kc[b, :L]), Kn[b]], axis=0)      # [L+T, Hkv, D]
        Vall = np.concatenate([w(vc[b, :L]), Vn[b]], axis=0)
        for j in range(T):
            for h in range(Hq):
                kh = h // (Hq // Hkv)
                sc = scale * (Kall[: L + j + 1, kh] @ Q[b, j, h])
                ref = softmax(sc) @ Vall[: L + j + 1, kh]
                got = out[b * T + j, h * D:(h + 1) * D]
                assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), (b, j, h)


def pin_attention_special_cases(o):
    """One visible key returns its value exactly; equal keys average the
    values; a later token's key and value never change an earlier token's
    output."""
    rng = np.random.default_rng(32)
    B, T, Hq, Hkv, D, Lmax = 1, 3, 2, 1, 16, 4
    qkv, kc, vc, lens = _attn_case(rng, B, T, Hq, Hkv, D, Lmax, [0])
    out = o.attention_verify(qkv, kc, vc, lens, T, Hq, Hkv, D, 0.25)
    v0 = (qkv[0, (Hq + Hkv) * D:].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(out[0, :D], v0) and np.array_equal(out[0, D:2 * D], v0)
    qkv2, kc2, vc2, _ = _attn_case(rng, B, T, Hq, Hkv, D, Lmax, [4])
    kc2[:] = kc2[0, 0]                                  # four equal cached keys, no new-key influence:
    qkv2[:, Hq * D:(Hq + Hkv) * D] = kc2[0, 0, 0]       # the step's keys equal them too
    out2 = o.attention_verify(qkv2, kc2, vc2, np.array([4], np.int32), T, Hq, Hkv, D, 0.25)
    f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    vals = np.concatenate([f(vc2[0, :4, 0]), f(qkv2[:1, (Hq + Hkv) * D:])], axis=0)
    assert np.allclose(out2[0, :D], vals.mean(axis=0), rtol=1e-14, atol=1e-14)
    qkv3 = qkv2.copy()
    qkv3[2, Hq * D:] = qkv3[1, Hq * D:][::-1]           # change token 2's key and value
    out3 = o.attention_verify(qkv3, kc2, vc2, np.array([4], np.int32), T, Hq, Hkv, D, 0.25)
    assert np.array_equal(out3[:2], out2[:2]) and not np.array_equal(out3[2], out2[2])


ALL_PINS = [
    pin_worked_example,
    pin_quantize_exact_rational,
    pin_quantize_ties,
    pin_quantize_invariants,
    pin_quantize_smoothing,
    pin_int8_matmul_bruteforce,
    pin_int8_matmul_range,
    pin_dequant_exact,
    pin_argmax,
    pin_accept_enumeration,
    pin_bf16,
    pin_linear_f64,
    pin_layer_exp,
    pin_silu,
    pin_swiglu_quant,
    pin_rmsnorm_quant,
    pin_splitmix64_kat,
    pin_spec_lossless,
    pin_draw_index,
    pin_spec_special_cases,
    pin_tree_chain_is_linear,
    pin_tree_bruteforce,
    pin_w4_worked_example,
    pin_w4_quantize_exact_rational,
    pin_w4_pack_roundtrip,
    pin_w4_linear_bruteforce,
    pin_fidelity_closed_forms,
    pin_fidelity_scipy,
    pin_attention_numpy,
    pin_attention_special_cases,
]
