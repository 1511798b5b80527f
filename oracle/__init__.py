"""CPU oracle for the W8A8 quantized verify pass.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``quantized_verification_gb300``) never imports it, and this package imports
nothing from there.

The arithmetic lives in ``qv_oracle.c`` (plain C, scalar loops, binary32
operations one at a time, compiled without contraction or fast-math). This
module compiles it with gcc on first use and wraps it with ctypes and numpy.
Every function names the passage of the Quasar summaries it follows; the
readings taken where the summaries are silent are listed in ``qv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "qv_oracle.c")
DEFAULT_LIB = os.path.join(_HERE, "libqv_oracle.so")

# -ffp-contract=off: gcc contracts a*b+c into fma by default on aarch64;
# every fp32 operation of the oracle must round on its own.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-finite-math-only", "-frounding-math"]


def build(src: str = SOURCE, out: str = DEFAULT_LIB, force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I = ctypes.c_int64


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a
    deliberately broken copy built by the mutation tests)."""

    def __init__(self, lib_path: str):
        L = ctypes.CDLL(lib_path)
        self._L = L
        L.qvo_bf16_to_f32.restype = ctypes.c_float
        L.qvo_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.qvo_f32_to_bf16_rne.restype = ctypes.c_uint16
        L.qvo_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        L.qvo_bf16_to_f32_array.argtypes = [_P, _P, _I]
        L.qvo_f32_to_bf16_array.argtypes = [_P, _P, _I]
        L.qvo_quantize_rows_f32.argtypes = [_P, _I, _I, _P, _P, _P]
        L.qvo_quantize_rows_bf16.argtypes = [_P, _I, _I, _P, _P, _P]
        L.qvo_int8_matmul.restype = ctypes.c_int64
        L.qvo_int8_matmul.argtypes = [_P, _P, _I, _I, _I, _P]
        L.qvo_dequant_one.restype = ctypes.c_float
        L.qvo_dequant_one.argtypes = [ctypes.c_int32, ctypes.c_float, ctypes.c_float]
        L.qvo_dequant.argtypes = [_P, _P, _P, _I, _I, _P]
        L.qvo_argmax_rows.argtypes = [_P, _I, _I, _P, _P]
        L.qvo_lm_head_argmax.argtypes = [_P, _P, _P, _P, _I, _I, _I, _P, _P]
        L.qvo_accept.argtypes = [_P, _P, _I, _I, _P, _P]
        L.qvo_linear_f64.argtypes = [_P, _P, _I, _I, _I, _P]
        L.qvo_exp.restype = ctypes.c_float
        L.qvo_exp.argtypes = [ctypes.c_float]
        L.qvo_silu.restype = ctypes.c_float
        L.qvo_silu.argtypes = [ctypes.c_float]
        L.qvo_swiglu_quant.argtypes = [_P, _I, _I, _P, _P]
        L.qvo_residual_rmsnorm_quant.argtypes = [_P, _P, _P, ctypes.c_float, _P, _I, _I, _P, _P, _P]
        L.qvo_splitmix64.restype = ctypes.c_uint64
        L.qvo_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        L.qvo_spec_sample.argtypes = [_P, _P, _P, _I, _I, _I, ctypes.c_float, ctypes.c_uint64, _P, _P]
        L.qvo_tree_accept.argtypes = [_P, _P, _P, _I, _I, _P, _P, _P]
        L.qvo_quantize_rows_w4_f32.argtypes = [_P, _I, _I, _P, _P]
        L.qvo_pack_w4.argtypes = [_P, _I, _I, _P]
        L.qvo_unpack_w4.argtypes = [_P, _I, _I, _P]
        L.qvo_logit_fidelity.argtypes = [_P, _P, _I, _I, _P, _P, _P]
        L.qvo_attention_verify.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_double, _P]
        L.qvo_draw_index.restype = ctypes.c_int32
        L.qvo_draw_index.argtypes = [_P, _I, ctypes.c_uint64, ctypes.c_uint32]

    # -- bf16 ------------------------------------------------------------
    def bf16_to_f32(self, h: np.ndarray) -> np.ndarray:
        """Exact widening of bf16 bit patterns (uint16) to binary32."""
        h = np.ascontiguousarray(h, dtype=np.uint16)
        f = np.empty(h.shape, dtype=np.float32)
        self._L.qvo_bf16_to_f32_array(_ptr(h), _ptr(f), h.size)
        return f

    def f32_to_bf16(self, f: np.ndarray) -> np.ndarray:
        """binary32 -> bf16 bit patterns, round to nearest even."""
        f = np.ascontiguousarray(f, dtype=np.float32)
        h = np.empty(f.shape, dtype=np.uint16)
        self._L.qvo_f32_to_bf16_array(_ptr(f), _ptr(h), f.size)
        return h

    # -- a0 / a1 ---------------------------------------------------------
    def quantize_rows(self, x: np.ndarray, mul: np.ndarray | None = None,
                      bf16: bool = False):
        """Per-row symmetric int8 quantization (a0 weights, a1 activations).

        Quasar, gist.science/ja summary, section 2.2 items 2-3 (weights and
        activations to INT8; the activation is multiplied by the smoothing
        factor first); gist.science/de summary, section 2 "Online-Prozess".
        ``x`` is float32 [rows, K], or uint16 bf16 patterns with ``bf16=True``.
        Returns (q int8 [rows, K], s float32 [rows]).
        """
        dt = np.uint16 if bf16 else np.float32
        x = np.ascontiguousarray(x, dtype=dt)
        rows, K = x.shape
        q = np.empty((rows, K), dtype=np.int8)
        s = np.empty(rows, dtype=np.float32)
        m = None
        if mul is not None:
            m = np.ascontiguousarray(mul, dtype=np.float32)
            assert m.shape == (K,)
        fn = self._L.qvo_quantize_rows_bf16 if bf16 else self._L.qvo_quantize_rows_f32
        fn(_ptr(x), rows, K, _ptr(m) if m is not None else None, _ptr(q), _ptr(s))
        return q, s

    # -- a2 ----------------------------------------------------------------
    def int8_matmul(self, xq: np.ndarray, wq: np.ndarray) -> np.ndarray:
        """Exact integer sums acc[m, n] = sum_k xq[m, k] * wq[n, k]
        (gist.science/ja summary, section 2.2 item 3: INT8 GEMM, INT32
        accumulation). Raises if a sum does not fit int32."""
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        wq = np.ascontiguousarray(wq, dtype=np.int8)
        M, K = xq.shape
        N, K2 = wq.shape
        assert K == K2
        acc = np.empty((M, N), dtype=np.int32)
        ov = self._L.qvo_int8_matmul(_ptr(xq), _ptr(wq), M, N, K, _ptr(acc))
        if ov:
            raise OverflowError(f"{ov} sums exceed int32")
        return acc

    def dequant(self, acc: np.ndarray, sx: np.ndarray, sw: np.ndarray) -> np.ndarray:
        """y = fl(fl(acc) * fl(sx[m] * sw[n])) (dequantization back to high
        precision, gist.science/ja summary, section 2.2 item 3)."""
        acc = np.ascontiguousarray(acc, dtype=np.int32)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, N = acc.shape
        y = np.empty((M, N), dtype=np.float32)
        self._L.qvo_dequant(_ptr(acc), _ptr(sx), _ptr(sw), M, N, _ptr(y))
        return y

    def w8a8_linear(self, xq, sx, wq, sw):
        """a2: returns (y float32 [M, N], acc int32 [M, N])."""
        acc = self.int8_matmul(xq, wq)
        return self.dequant(acc, sx, sw), acc

    # -- a3 ----------------------------------------------------------------
    def argmax_rows(self, y: np.ndarray):
        """Greedy token per row, lowest index on ties (gist.science/it
        summary, section 2 item 3; greedy decoding, gist.science/ja summary,
        section 4). Returns (tok int32 [M], max float32 [M])."""
        y = np.ascontiguousarray(y, dtype=np.float32)
        M, N = y.shape
        tok = np.empty(M, dtype=np.int32)
        mv = np.empty(M, dtype=np.float32)
        self._L.qvo_argmax_rows(_ptr(y), M, N, _ptr(tok), _ptr(mv))
        return tok, mv

    def lm_head_argmax(self, xq, sx, wq, sw):
        """a3: LM head logits formed one by one and reduced on the fly."""
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        wq = np.ascontiguousarray(wq, dtype=np.int8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, K = xq.shape
        V = wq.shape[0]
        tok = np.empty(M, dtype=np.int32)
        mv = np.empty(M, dtype=np.float32)
        self._L.qvo_lm_head_argmax(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw),
                                   M, V, K, _ptr(tok), _ptr(mv))
        return tok, mv

    # -- a4 ----------------------------------------------------------------
    def accept(self, t: np.ndarray, d: np.ndarray, B: int, gamma: int):
        """Greedy acceptance (gist.science/fr summary, lay explanation;
        L >= 1 from gist.science/ja summary, section 4).
        Returns (len int32 [B], out int32 [B, gamma+1])."""
        t = np.ascontiguousarray(t, dtype=np.int32).reshape(B * (gamma + 1))
        d = np.ascontiguousarray(d, dtype=np.int32).reshape(max(B * gamma, 0))
        ln = np.empty(B, dtype=np.int32)
        out = np.empty(B * (gamma + 1), dtype=np.int32)
        self._L.qvo_accept(_ptr(t), _ptr(d) if d.size else None, B, gamma,
                           _ptr(ln), _ptr(out))
        return ln, out.reshape(B, gamma + 1)

    # -- comparator reference -------------------------------------------------
    def linear_f64(self, x: np.ndarray, w: np.ndarray) -> np.ndarray:
        """Unquantized y = x w^T in binary64 over binary32 inputs (the
        high-precision verifier the W8A8 one replaces; gist.science/ja
        summary, section 2.3)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        M, K = x.shape
        N = w.shape[0]
        y = np.empty((M, N), dtype=np.float64)
        self._L.qvo_linear_f64(_ptr(x), _ptr(w), M, N, K, _ptr(y))
        return y


    # -- f1: non-linear steps between the linears of a layer -------------
    def exp(self, x: float) -> float:
        """The layer's exp: Cody-Waite reduction + degree-7 Taylor, binary32."""
        return float(self._L.qvo_exp(float(x)))

    def silu(self, x: float) -> float:
        """silu(v) = v * 1 / (1 + exp(-v)), binary32, with the layer's exp."""
        return float(self._L.qvo_silu(float(x)))

    def swiglu_quant(self, gu: np.ndarray):
        """gu [M, 2F] fp32 (gate | up) -> codes [M, F] int8, scales [M]:
        a = silu(gate) * up, then the per-token quantization
        (gist.science/ja summary, section 2.2 item 3: non-linear layers in
        high precision, then INT8 for the next linear)."""
        gu = np.ascontiguousarray(gu, dtype=np.float32)
        M, F2 = gu.shape
        F = F2 // 2
        q = np.empty((M, F), dtype=np.int8)
        s = np.empty(M, dtype=np.float32)
        self._L.qvo_swiglu_quant(_ptr(gu), M, F, _ptr(q), _ptr(s))
        return q, s

    def residual_rmsnorm_quant(self, h: np.ndarray, d: np.ndarray | None, g: np.ndarray, eps: float,
                               mul: np.ndarray | None = None):
        """h [M, H] bf16 bits (uint16); d the bf16 delta or None; g [H] bf16
        bits. Returns (h', codes [M, H], scales [M], x [M, H] bf16 bits):
        h' = rne_bf16(h + d), x = RMSNorm(h') * g in bf16, then the
        per-token quantization of x."""
        h = np.array(h, dtype=np.uint16, copy=True, order="C")
        M, H = h.shape
        d_ = None if d is None else np.ascontiguousarray(d, dtype=np.uint16)
        g = np.ascontiguousarray(g, dtype=np.uint16)
        mul_ = None if mul is None else np.ascontiguousarray(mul, dtype=np.float32)
        q = np.empty((M, H), dtype=np.int8)
        s = np.empty(M, dtype=np.float32)
        x = np.empty((M, H), dtype=np.uint16)
        self._L.qvo_residual_rmsnorm_quant(_ptr(h), None if d_ is None else _ptr(d_), _ptr(g),
                                           ctypes.c_float(eps), None if mul_ is None else _ptr(mul_),
                                           M, H, _ptr(q), _ptr(s), _ptr(x))
        return h, q, s, x


    # -- f2: lossless rejection sampling at T > 0 -------------------------
    def splitmix64(self, seed: int, n: int) -> int:
        """Draw n of SplitMix64 seeded with ``seed`` (counter-based form)."""
        return int(self._L.qvo_splitmix64(seed & (2 ** 64 - 1), n))

    def draw_index(self, x, u24: int) -> int:
        """The sampling draw: the smallest v whose prefix sum of the integer
        weights x exceeds floor(u24 * sum(x) / 2^24)."""
        x = np.ascontiguousarray(x, dtype=np.uint64)
        return int(self._L.qvo_draw_index(_ptr(x), x.size, int(x.sum()), u24))

    def spec_sample(self, z: np.ndarray, d: np.ndarray, q: np.ndarray, B: int, gamma: int,
                    T: float, seed: int):
        """Speculative sampling at temperature T (gist.science/it summary,
        section 2 item 3): z [B*(gamma+1), V] fp32 logits, d [B, gamma] draft
        tokens, q [B*gamma, V] draft probabilities. Returns (len [B],
        out [B, gamma+1])."""
        z = np.ascontiguousarray(z, dtype=np.float32)
        V = z.shape[1]
        d = np.ascontiguousarray(d, dtype=np.int32).reshape(max(B * gamma, 0))
        q = np.ascontiguousarray(q, dtype=np.float32).reshape(max(B * gamma, 0), V)
        ln = np.empty(B, dtype=np.int32)
        out = np.empty(B * (gamma + 1), dtype=np.int32)
        self._L.qvo_spec_sample(_ptr(z), _ptr(d) if d.size else None, _ptr(q) if q.size else None,
                                B, gamma, V, ctypes.c_float(T), seed & (2 ** 64 - 1), _ptr(ln), _ptr(out))
        return ln, out.reshape(B, gamma + 1)

    # -- f3: tree verification at T = 0 ------------------------------------
    def tree_accept(self, t: np.ndarray, d: np.ndarray, par: np.ndarray):
        """Greedy tree verification: t, d, par [B, N] int32 (node 0 the root,
        parents before children). Returns (len [B], out [B, N], node [B]): the
        deepest fully matching root path (lowest index on ties), its drafted
        tokens, then the verifier's token after it."""
        t = np.ascontiguousarray(t, dtype=np.int32)
        B, N = t.shape
        d = np.ascontiguousarray(d, dtype=np.int32)
        par = np.ascontiguousarray(par, dtype=np.int32)
        ln = np.empty(B, dtype=np.int32)
        out = np.empty((B, N), dtype=np.int32)
        node = np.empty(B, dtype=np.int32)
        self._L.qvo_tree_accept(_ptr(t), _ptr(d), _ptr(par), B, N, _ptr(ln), _ptr(out), _ptr(node))
        return ln, out, node

    # -- f4: W4A8 ----------------------------------------------------------
    def quantize_rows_w4(self, w: np.ndarray, bf16: bool = False):
        """Per-output-channel symmetric int4 weights, the a0 rule with codes in
        [-7, 7] (lower-bit verifiers: gist.science/it summary, section 5;
        INT4 among the widths tried: shd-paper.top summary, method details,
        key design).
        ``w`` float32 [N, K], or bf16 patterns with ``bf16=True`` (widened
        exactly). Returns (q int8 [N, K] codes, s float32 [N])."""
        if bf16:
            w = self.bf16_to_f32(np.ascontiguousarray(w, dtype=np.uint16))
        w = np.ascontiguousarray(w, dtype=np.float32)
        N, K = w.shape
        q = np.empty((N, K), dtype=np.int8)
        s = np.empty(N, dtype=np.float32)
        self._L.qvo_quantize_rows_w4_f32(_ptr(w), N, K, _ptr(q), _ptr(s))
        return q, s

    def pack_w4(self, q: np.ndarray) -> np.ndarray:
        """Two int4 codes per byte, even k in the low nibble: uint8 [N, K/2]."""
        q = np.ascontiguousarray(q, dtype=np.int8)
        N, K = q.shape
        assert K % 2 == 0
        out = np.empty((N, K // 2), dtype=np.uint8)
        self._L.qvo_pack_w4(_ptr(q), N, K, _ptr(out))
        return out

    def unpack_w4(self, packed: np.ndarray) -> np.ndarray:
        """Inverse of pack_w4: int8 codes [N, 2 * bytes]."""
        packed = np.ascontiguousarray(packed, dtype=np.uint8)
        N, KB = packed.shape
        q = np.empty((N, 2 * KB), dtype=np.int8)
        self._L.qvo_unpack_w4(_ptr(packed), N, 2 * KB, _ptr(q))
        return q

    def w4a8_linear(self, xq, sx, wq4, sw):
        """f4: y = dequant(sum_k xq[m, k] * w[n, k]) with the int4 codes
        unpacked from ``wq4``; the sums and the dequantization are a2's.
        Returns (y float32 [M, N], acc int32 [M, N])."""
        return self.w8a8_linear(xq, sx, self.unpack_w4(wq4), sw)

    def w4a8_lm_head_argmax(self, xq, sx, wq4, sw):
        """f4 with the a3 greedy argmax (lowest index on ties)."""
        return self.lm_head_argmax(xq, sx, self.unpack_w4(wq4), sw)


    # -- f1': attention over a short KV cache --------------------------------
    def attention_verify(self, qkv, kc, vc, lens, T: int, Hq: int, Hkv: int, D: int, scale: float):
        """Causal grouped-query attention of the step's verify tokens over the
        cache and the step's own keys, in binary64 from bf16 inputs (the
        layer between the quantized linears: gist.science/ja summary,
        section 2.2 item 3). qkv uint16 [B*T, (Hq+2Hkv)*D] (bf16 patterns),
        kc, vc uint16 [B, Lmax, Hkv, D], lens int32 [B]. Returns float64
        [B*T, Hq*D]."""
        qkv = np.ascontiguousarray(qkv, dtype=np.uint16)
        kc = np.ascontiguousarray(kc, dtype=np.uint16)
        vc = np.ascontiguousarray(vc, dtype=np.uint16)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        B, Lmax = kc.shape[0], kc.shape[1]
        assert qkv.shape == (B * T, (Hq + 2 * Hkv) * D) and kc.shape == (B, Lmax, Hkv, D) == vc.shape
        out = np.empty((B * T, Hq * D), dtype=np.float64)
        self._L.qvo_attention_verify(_ptr(qkv), _ptr(kc), _ptr(vc), _ptr(lens), B, T, Hq, Hkv, D, Lmax,
                                     ctypes.c_double(scale), _ptr(out))
        return out

    # -- f3': logit fidelity ------------------------------------------------
    def logit_fidelity(self, a: np.ndarray, b: np.ndarray):
        """KL(softmax(a) || softmax(b)) per row in binary64, and the top-1
        indices of a and b (lowest index on ties). The summaries' fidelity
        claim: negligible KL divergence between the full-precision and the
        quantized verifier's logits (gist.science/fr summary, contributions
        item 3). Returns (kl float64 [M], ta int32 [M], tb int32 [M])."""
        a = np.ascontiguousarray(a, dtype=np.float32)
        b = np.ascontiguousarray(b, dtype=np.float32)
        assert a.shape == b.shape
        M, V = a.shape
        kl = np.empty(M, dtype=np.float64)
        ta = np.empty(M, dtype=np.int32)
        tb = np.empty(M, dtype=np.int32)
        self._L.qvo_logit_fidelity(_ptr(a), _ptr(b), M, V, _ptr(kl), _ptr(ta), _ptr(tb))
        return kl, ta, tb


_default: Oracle | None = None
_lock = threading.Lock()

def get() -> Oracle:
    """The oracle built from ``qv_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default
