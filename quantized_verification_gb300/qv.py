"""Thin ctypes binding of libqv (include/qv.h), one Python function per C
entry point, same names. It only marshals arguments: shapes come from the
tensors, pointers from ``data_ptr()``, the stream from torch. Every step of the
computation runs in libqv's CUDA kernels; there is no fallback. If libqv.so
is missing the first call raises, naming the build command.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqv.so")

QV_OK, QV_ERR_INVALID_ARG, QV_ERR_UNSUPPORTED, QV_ERR_WORKSPACE, QV_ERR_CUDA = range(5)
QV_F32, QV_BF16 = 0, 1
QV_OP_LINEAR, QV_OP_LM_HEAD, QV_OP_BF16_LINEAR, QV_OP_VERIFY_STACK = 0, 1, 2, 3
QV_OP_LINEAR_ACT, QV_OP_LM_HEAD_ACT = 4, 5
QV_OP_SPEC_SAMPLE = 6
QV_MAX_K = 133144
QV_MAX_M = 256

# Symbols include/qv.h declares (checked against the library by the tests).
EXPORTS = ("qv_quantize_act", "qv_w8a8_linear", "qv_lm_head_argmax", "qv_accept",
           "qv_quantize_weight", "qv_bf16_linear", "qv_workspace_bytes",
           "qv_last_error", "qv_device_error", "qv_num_sms", "qv_w8a8_linear_noalloc",
           "qv_verify_stack", "qv_w8a8_linear_act", "qv_lm_head_argmax_act",
           "qv_rmsnorm_quant", "qv_swiglu_quant", "qv_w8a8_swiglu", "qv_spec_sample",
           "qv_tree_accept", "qv_quantize_weight_w4", "qv_w4a8_linear", "qv_w4a8_swiglu",
           "qv_w4a8_lm_head_argmax", "qv_logit_fidelity", "qv_attention_workspace_bytes",
           "qv_attention_verify", "qv_debug_set_slot_wait_ns", "qv_debug_drop_partials",
           "qv_debug_hold_attention_loads")
MAX_STACK_M = 16


class LinearDesc(ctypes.Structure):
    """qv_linear_desc of include/qv.h."""
    _fields_ = [("x", ctypes.c_void_p), ("act_mul", ctypes.c_void_p), ("wq", ctypes.c_void_p),
                ("sw", ctypes.c_void_p), ("y", ctypes.c_void_p), ("K", ctypes.c_int), ("N", ctypes.c_int)]
QV_NOALLOC_SCRATCH_BYTES = 16 << 20


class QVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libqv status {status}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libqv.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -m quantized_verification_gb300.build`")
        L = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        st = ctypes.c_int
        L.qv_quantize_act.argtypes = [P, I, I, I, P, P, P, P]
        L.qv_w8a8_linear.argtypes = [P, P, I, I, P, P, I, P, I, P, P, S, P]
        L.qv_lm_head_argmax.argtypes = [P, P, I, I, P, P, I, P, P, P, S, P]
        L.qv_accept.argtypes = [P, P, I, I, P, P, P]
        L.qv_quantize_weight.argtypes = [P, I, I, I, P, P, P]
        L.qv_bf16_linear.argtypes = [P, I, I, P, I, P, P, S, P]
        L.qv_w8a8_linear_noalloc.argtypes = [P, P, I, I, P, P, I, P, I, P, P]
        L.qv_verify_stack.argtypes = [ctypes.POINTER(LinearDesc), I, ctypes.POINTER(LinearDesc), I, I,
                                      P, I, I, P, P, P, P, P, S, P]
        L.qv_w8a8_linear_act.argtypes = [P, I, P, I, I, P, P, I, P, I, P, S, P]
        L.qv_lm_head_argmax_act.argtypes = [P, I, P, I, I, P, P, I, P, P, P, S, P]
        L.qv_rmsnorm_quant.argtypes = [P, P, P, ctypes.c_float, P, I, I, P, P, P, P]
        L.qv_swiglu_quant.argtypes = [P, I, I, P, P, P]
        L.qv_w8a8_swiglu.argtypes = [P, P, I, I, P, P, I, P, P, S, P]
        L.qv_spec_sample.argtypes = [P, P, P, I, I, I, ctypes.c_float, ctypes.c_uint64, P, P, P, S, P]
        L.qv_tree_accept.argtypes = [P, P, P, I, I, P, P, P, P]
        L.qv_quantize_weight_w4.argtypes = [P, I, I, I, P, P, P]
        L.qv_logit_fidelity.argtypes = [P, P, I, I, P, P, P, P]
        L.qv_attention_workspace_bytes.argtypes = [I, I, I, I, I, I]
        L.qv_attention_workspace_bytes.restype = S
        L.qv_attention_verify.argtypes = [P, P, P, P, I, I, I, I, I, I, ctypes.c_float, P, P, S, P]
        L.qv_w4a8_linear.argtypes = [P, P, I, I, P, P, I, P, I, P, P, S, P]
        L.qv_w4a8_swiglu.argtypes = [P, P, I, I, P, P, I, P, P, S, P]
        L.qv_w4a8_lm_head_argmax.argtypes = [P, P, I, I, P, P, I, P, P, P, S, P]
        L.qv_workspace_bytes.argtypes = [I, I, I, I]
        L.qv_workspace_bytes.restype = S
        L.qv_last_error.argtypes = []
        L.qv_last_error.restype = ctypes.c_char_p
        L.qv_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        L.qv_debug_set_slot_wait_ns.argtypes = [ctypes.c_ulonglong]
        L.qv_debug_set_slot_wait_ns.restype = None
        L.qv_debug_drop_partials.argtypes = [I]
        L.qv_debug_drop_partials.restype = None
        L.qv_debug_hold_attention_loads.argtypes = [I]
        L.qv_debug_hold_attention_loads.restype = None
        L.qv_num_sms.argtypes = []
        L.qv_num_sms.restype = I
        for name in ("qv_quantize_act", "qv_w8a8_linear", "qv_lm_head_argmax", "qv_accept",
                     "qv_quantize_weight", "qv_bf16_linear", "qv_device_error",
                     "qv_w8a8_linear_noalloc", "qv_verify_stack", "qv_w8a8_linear_act",
                     "qv_lm_head_argmax_act"):
            getattr(L, name).restype = st
        _lib = L
        return L


def _check(status: int):
    if status != QV_OK:
        raise QVError(status, load().qv_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return QV_F32
    if t.dtype == torch.bfloat16:
        return QV_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


# ---------------------------------------------------------------------------
def qv_quantize_act(x, xq, sx, act_mul=None, stream=None):
    """x [M, K] fp32/bf16 -> xq [M, K] int8, sx [M] fp32."""
    M, K = x.shape
    _need(xq.shape == (M, K) and xq.dtype == torch.int8, "xq must be int8 [M, K]")
    _need(sx.shape == (M,) and sx.dtype == torch.float32, "sx must be float32 [M]")
    if act_mul is not None:
        _need(act_mul.shape == (K,) and act_mul.dtype == torch.float32, "act_mul must be float32 [K]")
    _check(load().qv_quantize_act(_ptr(x), _dtype(x), M, K, _ptr(act_mul), _ptr(xq), _ptr(sx),
                                  ctypes.c_void_p(_stream(stream))))


def qv_rmsnorm_quant(h, gamma, xq, sx, delta=None, eps=1e-6, act_mul=None, x_out=None, stream=None):
    """h [M, H] bf16 (updated in place when delta is given: h += delta in
    bf16); xq [M, H] int8, sx [M] = per-token codes of RMSNorm(h) * gamma."""
    M, H = h.shape
    _need(h.dtype == torch.bfloat16, "h must be bf16 [M, H]")
    _need(gamma.shape == (H,) and gamma.dtype == torch.bfloat16, "gamma must be bf16 [H]")
    _need(xq.shape == (M, H) and xq.dtype == torch.int8, "xq must be int8 [M, H]")
    _need(sx.shape == (M,) and sx.dtype == torch.float32, "sx must be float32 [M]")
    if delta is not None:
        _need(delta.shape == (M, H) and delta.dtype == torch.bfloat16, "delta must be bf16 [M, H]")
    if act_mul is not None:
        _need(act_mul.shape == (H,) and act_mul.dtype == torch.float32, "act_mul must be float32 [H]")
    if x_out is not None:
        _need(x_out.shape == (M, H) and x_out.dtype == torch.bfloat16, "x_out must be bf16 [M, H]")
    _check(load().qv_rmsnorm_quant(_ptr(h), _ptr(delta), _ptr(gamma), ctypes.c_float(eps), _ptr(act_mul),
                                   M, H, _ptr(xq), _ptr(sx), _ptr(x_out), ctypes.c_void_p(_stream(stream))))


def interleave_gate_up(w: torch.Tensor) -> torch.Tensor:
    """[2F, ...] rows gate (0..F-1) then up (F..2F-1) -> the layout of
    qv_w8a8_swiglu: per 128 rows, 64 gate rows then the same 64 up rows."""
    F = w.shape[0] // 2
    _need(F % 64 == 0 and w.shape[0] == 2 * F, "gate|up rows must be 2F with F a multiple of 64")
    rest = tuple(w.shape[1:])
    return torch.stack([w[:F].reshape(F // 64, 64, *rest), w[F:].reshape(F // 64, 64, *rest)], dim=1).reshape(2 * F, *rest)


def qv_w8a8_swiglu(xq, sx, wq_gu, sw_gu, a, workspace, stream=None):
    """a [M, F] fp32 = silu(y_gate) * y_up of the interleaved gate|up linear."""
    M, K = xq.shape
    F2 = wq_gu.shape[0]
    F = F2 // 2
    _need(wq_gu.shape == (F2, K) and wq_gu.dtype == torch.int8 and xq.dtype == torch.int8, "int8 xq, wq_gu")
    _need(sx.shape == (M,) and sw_gu.shape == (F2,), "sx [M], sw_gu [2F]")
    _need(a.shape == (M, F) and a.dtype == torch.float32, "a must be float32 [M, F]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_w8a8_swiglu(_ptr(xq), _ptr(sx), M, K, _ptr(wq_gu), _ptr(sw_gu), F, _ptr(a),
                                 _ptr(workspace), workspace.numel(), ctypes.c_void_p(_stream(stream))))


def qv_tree_accept(verify_tokens, draft, parent, accept_len, out_tokens, best_node=None, stream=None):
    """Greedy tree verification: verify_tokens, draft, parent [B, N] int32 ->
    accept_len [B], out_tokens [B, N], best_node [B] (optional)."""
    B, N = verify_tokens.shape
    for name, tsr in (("verify_tokens", verify_tokens), ("draft", draft), ("parent", parent),
                      ("out_tokens", out_tokens)):
        _need(tsr.shape == (B, N) and tsr.dtype == torch.int32, f"{name} must be int32 [B, N]")
    _need(accept_len.shape == (B,) and accept_len.dtype == torch.int32, "accept_len int32 [B]")
    if best_node is not None:
        _need(best_node.shape == (B,) and best_node.dtype == torch.int32, "best_node int32 [B]")
    _check(load().qv_tree_accept(_ptr(verify_tokens), _ptr(draft), _ptr(parent), B, N, _ptr(accept_len),
                                 _ptr(out_tokens), _ptr(best_node), ctypes.c_void_p(_stream(stream))))


def qv_spec_sample(logits, draft, draft_probs, temperature, seed, accept_len, out_tokens, workspace,
                   stream=None):
    """Speculative sampling at temperature > 0: logits [B*(gamma+1), V]
    fp32, draft [B, gamma] int32, draft_probs [B*gamma, V] fp32 ->
    accept_len [B], out_tokens [B, gamma+1]."""
    B, G = out_tokens.shape
    gamma = G - 1
    M, V = logits.shape
    _need(logits.dtype == torch.float32 and M == B * G, "logits must be float32 [B*(gamma+1), V]")
    _need(accept_len.shape == (B,) and accept_len.dtype == torch.int32, "accept_len int32 [B]")
    _need(out_tokens.dtype == torch.int32, "out_tokens int32 [B, gamma+1]")
    if gamma > 0:
        _need(draft.shape == (B, gamma) and draft.dtype == torch.int32, "draft int32 [B, gamma]")
        _need(draft_probs.shape == (B * gamma, V) and draft_probs.dtype == torch.float32,
              "draft_probs float32 [B*gamma, V]")
    _check(load().qv_spec_sample(_ptr(logits), _ptr(draft) if gamma > 0 else None,
                                 _ptr(draft_probs) if gamma > 0 else None, B, gamma, V,
                                 ctypes.c_float(temperature), ctypes.c_uint64(seed & (2 ** 64 - 1)),
                                 _ptr(accept_len), _ptr(out_tokens), _ptr(workspace), workspace.numel(),
                                 ctypes.c_void_p(_stream(stream))))


def qv_swiglu_quant(gate_up, xq, sx, stream=None):
    """gate_up [M, 2F] fp32 (gate | up) -> xq [M, F] int8, sx [M]: per-token
    codes of SiLU(gate) * up."""
    M, F2 = gate_up.shape
    F = F2 // 2
    _need(gate_up.dtype == torch.float32 and F2 == 2 * F, "gate_up must be float32 [M, 2F]")
    _need(xq.shape == (M, F) and xq.dtype == torch.int8, "xq must be int8 [M, F]")
    _need(sx.shape == (M,) and sx.dtype == torch.float32, "sx must be float32 [M]")
    _check(load().qv_swiglu_quant(_ptr(gate_up), M, F, _ptr(xq), _ptr(sx), ctypes.c_void_p(_stream(stream))))


def qv_quantize_weight(w, wq, sw, stream=None):
    """w [N, K] fp32/bf16 -> wq [N, K] int8, sw [N] fp32."""
    N, K = w.shape
    _need(wq.shape == (N, K) and wq.dtype == torch.int8, "wq must be int8 [N, K]")
    _need(sw.shape == (N,) and sw.dtype == torch.float32, "sw must be float32 [N]")
    _check(load().qv_quantize_weight(_ptr(w), _dtype(w), N, K, _ptr(wq), _ptr(sw),
                                     ctypes.c_void_p(_stream(stream))))


def qv_w8a8_linear(xq, sx, wq, sw, y, workspace, acc_debug=None, stream=None):
    """y [M, N] (fp32 or bf16) = dequant(xq wq^T); acc_debug [M, N] int32."""
    M, K = xq.shape
    N = wq.shape[0]
    _need(wq.shape == (N, K) and wq.dtype == torch.int8 and xq.dtype == torch.int8, "int8 xq [M,K], wq [N,K]")
    _need(sx.shape == (M,) and sw.shape == (N,), "sx [M], sw [N]")
    _need(sx.dtype == torch.float32 and sw.dtype == torch.float32, "scales must be float32")
    _need(y.shape == (M, N), "y must be [M, N]")
    if acc_debug is not None:
        _need(acc_debug.shape == (M, N) and acc_debug.dtype == torch.int32, "acc_debug int32 [M, N]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_w8a8_linear(_ptr(xq), _ptr(sx), M, K, _ptr(wq), _ptr(sw), N, _ptr(y),
                                 _dtype(y), _ptr(acc_debug), _ptr(workspace), workspace.numel(),
                                 ctypes.c_void_p(_stream(stream))))


def qv_w8a8_linear_noalloc(xq, sx, wq, sw, y, acc_debug=None, stream=None):
    """qv_w8a8_linear without a workspace argument, for callers that cannot
    allocate device memory: the library's built-in scratch buffer is used."""
    M, K = xq.shape
    N = wq.shape[0]
    _need(wq.shape == (N, K) and wq.dtype == torch.int8 and xq.dtype == torch.int8, "int8 xq [M,K], wq [N,K]")
    _need(sx.shape == (M,) and sw.shape == (N,), "sx [M], sw [N]")
    _need(sx.dtype == torch.float32 and sw.dtype == torch.float32, "scales must be float32")
    _need(y.shape == (M, N), "y must be [M, N]")
    if acc_debug is not None:
        _need(acc_debug.shape == (M, N) and acc_debug.dtype == torch.int32, "acc_debug int32 [M, N]")
    _check(load().qv_w8a8_linear_noalloc(_ptr(xq), _ptr(sx), M, K, _ptr(wq), _ptr(sw), N, _ptr(y),
                                         _dtype(y), _ptr(acc_debug), ctypes.c_void_p(_stream(stream))))


def qv_lm_head_argmax(xq, sx, wq, sw, tokens, workspace, max_logit=None, stream=None):
    """tokens [M] int32 = greedy argmax over the W8A8 LM-head logits."""
    M, K = xq.shape
    V = wq.shape[0]
    _need(wq.shape == (V, K) and wq.dtype == torch.int8 and xq.dtype == torch.int8, "int8 xq [M,K], wq [V,K]")
    _need(sx.shape == (M,) and sw.shape == (V,), "sx [M], sw [V]")
    _need(tokens.shape == (M,) and tokens.dtype == torch.int32, "tokens int32 [M]")
    if max_logit is not None:
        _need(max_logit.shape == (M,) and max_logit.dtype == torch.float32, "max_logit float32 [M]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_lm_head_argmax(_ptr(xq), _ptr(sx), M, K, _ptr(wq), _ptr(sw), V, _ptr(tokens),
                                    _ptr(max_logit), _ptr(workspace), workspace.numel(),
                                    ctypes.c_void_p(_stream(stream))))


def qv_logit_fidelity(ref_logits, logits, kl, top1_ref, top1, stream=None):
    """Per row: kl [M] = KL(softmax(ref_logits) || softmax(logits)) in nats,
    top1_ref / top1 [M] int32 = first index of each row's maximum."""
    M, V = ref_logits.shape
    _need(ref_logits.dtype == torch.float32 and logits.dtype == torch.float32 and logits.shape == (M, V),
          "ref_logits and logits must be float32 [M, V]")
    _need(kl.shape == (M,) and kl.dtype == torch.float32, "kl float32 [M]")
    _need(top1_ref.shape == (M,) and top1.shape == (M,) and top1_ref.dtype == torch.int32 and
          top1.dtype == torch.int32, "top1_ref, top1 int32 [M]")
    _check(load().qv_logit_fidelity(_ptr(ref_logits), _ptr(logits), M, V, _ptr(kl), _ptr(top1_ref), _ptr(top1),
                                    ctypes.c_void_p(_stream(stream))))


def qv_attention_workspace_bytes(B, T, Hq, Hkv, D, Lmax) -> int:
    return int(load().qv_attention_workspace_bytes(B, T, Hq, Hkv, D, Lmax))


def qv_attention_verify(qkv, k_cache, v_cache, cache_len, T, Hq, Hkv, scale, out, workspace=None, stream=None):
    """Causal grouped-query attention of the verify tokens over the KV cache
    and the step's own keys: qkv [B*T, (Hq+2Hkv)*D] bf16, k_cache / v_cache
    [B, Lmax, Hkv, D] bf16, cache_len [B] int32 -> out [B*T, Hq*D] fp32."""
    B, Lmax, hkv, D = k_cache.shape
    _need(hkv == Hkv and v_cache.shape == k_cache.shape, "k_cache, v_cache must be [B, Lmax, Hkv, D]")
    _need(qkv.dtype == torch.bfloat16 and qkv.shape == (B * T, (Hq + 2 * Hkv) * D), "qkv bf16 [B*T, (Hq+2Hkv)*D]")
    _need(k_cache.dtype == torch.bfloat16 and v_cache.dtype == torch.bfloat16, "bf16 caches")
    _need(cache_len.shape == (B,) and cache_len.dtype == torch.int32, "cache_len int32 [B]")
    _need(out.shape == (B * T, Hq * D) and out.dtype == torch.float32, "out float32 [B*T, Hq*D]")
    _check(load().qv_attention_verify(_ptr(qkv), _ptr(k_cache) if Lmax > 0 else None,
                                      _ptr(v_cache) if Lmax > 0 else None, _ptr(cache_len), B, T, Hq, Hkv, D, Lmax,
                                      ctypes.c_float(scale), _ptr(out), _ptr(workspace),
                                      0 if workspace is None else workspace.numel(),
                                      ctypes.c_void_p(_stream(stream))))


# --- W4A8: packed int4 weights [N, K/2] uint8 (even k in the low nibble) ---
def qv_quantize_weight_w4(w, wq4, sw, stream=None):
    """w [N, K] fp32/bf16 -> wq4 [N, K/2] uint8 (two int4 codes per byte), sw [N] fp32."""
    N, K = w.shape
    _need(K % 2 == 0 and wq4.shape == (N, K // 2) and wq4.dtype == torch.uint8, "wq4 must be uint8 [N, K/2]")
    _need(sw.shape == (N,) and sw.dtype == torch.float32, "sw must be float32 [N]")
    _check(load().qv_quantize_weight_w4(_ptr(w), _dtype(w), N, K, _ptr(wq4), _ptr(sw),
                                        ctypes.c_void_p(_stream(stream))))


def _w4_shapes(xq, wq4):
    M, K = xq.shape
    N = wq4.shape[0]
    _need(xq.dtype == torch.int8, "xq must be int8 [M, K]")
    _need(wq4.dtype == torch.uint8 and wq4.shape == (N, K // 2) and K % 2 == 0, "wq4 must be uint8 [N, K/2]")
    return M, K, N


def qv_w4a8_linear(xq, sx, wq4, sw, y, workspace, acc_debug=None, stream=None):
    """y [M, N] (fp32 or bf16) = dequant(xq q^T), q the int4 codes of wq4."""
    M, K, N = _w4_shapes(xq, wq4)
    _need(sx.shape == (M,) and sw.shape == (N,), "sx [M], sw [N]")
    _need(sx.dtype == torch.float32 and sw.dtype == torch.float32, "scales must be float32")
    _need(y.shape == (M, N), "y must be [M, N]")
    if acc_debug is not None:
        _need(acc_debug.shape == (M, N) and acc_debug.dtype == torch.int32, "acc_debug int32 [M, N]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_w4a8_linear(_ptr(xq), _ptr(sx), M, K, _ptr(wq4), _ptr(sw), N, _ptr(y),
                                 _dtype(y), _ptr(acc_debug), _ptr(workspace), workspace.numel(),
                                 ctypes.c_void_p(_stream(stream))))


def qv_w4a8_swiglu(xq, sx, wq4_gu, sw_gu, a, workspace, stream=None):
    """a [M, F] fp32 = silu(y_gate) * y_up of the interleaved int4 gate|up linear."""
    M, K, F2 = _w4_shapes(xq, wq4_gu)
    F = F2 // 2
    _need(sx.shape == (M,) and sw_gu.shape == (F2,), "sx [M], sw_gu [2F]")
    _need(a.shape == (M, F) and a.dtype == torch.float32, "a must be float32 [M, F]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_w4a8_swiglu(_ptr(xq), _ptr(sx), M, K, _ptr(wq4_gu), _ptr(sw_gu), F, _ptr(a),
                                 _ptr(workspace), workspace.numel(), ctypes.c_void_p(_stream(stream))))


def qv_w4a8_lm_head_argmax(xq, sx, wq4, sw, tokens, workspace, max_logit=None, stream=None):
    """tokens [M] int32 = greedy argmax over the W4A8 LM-head logits."""
    M, K, V = _w4_shapes(xq, wq4)
    _need(sx.shape == (M,) and sw.shape == (V,), "sx [M], sw [V]")
    _need(tokens.shape == (M,) and tokens.dtype == torch.int32, "tokens int32 [M]")
    if max_logit is not None:
        _need(max_logit.shape == (M,) and max_logit.dtype == torch.float32, "max_logit float32 [M]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_w4a8_lm_head_argmax(_ptr(xq), _ptr(sx), M, K, _ptr(wq4), _ptr(sw), V, _ptr(tokens),
                                         _ptr(max_logit), _ptr(workspace), workspace.numel(),
                                         ctypes.c_void_p(_stream(stream))))


def qv_w8a8_linear_act(x, wq, sw, y, workspace, act_mul=None, stream=None):
    """y [M, N] (fp32 or bf16) = dequant(quant(x * act_mul) wq^T) in one call."""
    M, K = x.shape
    N = wq.shape[0]
    _need(wq.shape == (N, K) and wq.dtype == torch.int8, "wq must be int8 [N, K]")
    _need(sw.shape == (N,) and sw.dtype == torch.float32, "sw must be float32 [N]")
    _need(y.shape == (M, N), "y must be [M, N]")
    if act_mul is not None:
        _need(act_mul.shape == (K,) and act_mul.dtype == torch.float32, "act_mul must be float32 [K]")
    _check(load().qv_w8a8_linear_act(_ptr(x), _dtype(x), _ptr(act_mul), M, K, _ptr(wq), _ptr(sw), N,
                                     _ptr(y), _dtype(y), _ptr(workspace), workspace.numel(),
                                     ctypes.c_void_p(_stream(stream))))


def qv_lm_head_argmax_act(x, wq, sw, tokens, workspace, act_mul=None, max_logit=None, stream=None):
    """tokens [M] int32 = greedy argmax over the W8A8 LM-head logits of quant(x * act_mul)."""
    M, K = x.shape
    V = wq.shape[0]
    _need(wq.shape == (V, K) and wq.dtype == torch.int8, "wq must be int8 [V, K]")
    _need(sw.shape == (V,) and sw.dtype == torch.float32, "sw must be float32 [V]")
    _need(tokens.shape == (M,) and tokens.dtype == torch.int32, "tokens must be int32 [M]")
    if act_mul is not None:
        _need(act_mul.shape == (K,) and act_mul.dtype == torch.float32, "act_mul must be float32 [K]")
    if max_logit is not None:
        _need(max_logit.shape == (M,) and max_logit.dtype == torch.float32, "max_logit must be float32 [M]")
    _check(load().qv_lm_head_argmax_act(_ptr(x), _dtype(x), _ptr(act_mul), M, K, _ptr(wq), _ptr(sw), V,
                                        _ptr(tokens), _ptr(max_logit), _ptr(workspace), workspace.numel(),
                                        ctypes.c_void_p(_stream(stream))))


def qv_accept(verify_tokens, draft, accept_len, out_tokens, stream=None):
    """verify_tokens [B, gamma+1], draft [B, gamma] -> accept_len [B], out_tokens [B, gamma+1]."""
    B, G = verify_tokens.shape
    gamma = G - 1
    _need(draft is None or (draft.shape == (B, gamma) and draft.dtype == torch.int32), "draft int32 [B, gamma]")
    _need(verify_tokens.dtype == torch.int32, "verify_tokens int32")
    _need(accept_len.shape == (B,) and accept_len.dtype == torch.int32, "accept_len int32 [B]")
    _need(out_tokens.shape == (B, G) and out_tokens.dtype == torch.int32, "out_tokens int32 [B, gamma+1]")
    d = draft if (draft is not None and draft.numel() > 0) else None
    _check(load().qv_accept(_ptr(verify_tokens), _ptr(d), B, gamma, _ptr(accept_len),
                            _ptr(out_tokens), ctypes.c_void_p(_stream(stream))))


def qv_bf16_linear(x, w, y, workspace, stream=None):
    """y [M, N] fp32 = x [M, K] bf16 . w [N, K] bf16^T."""
    M, K = x.shape
    N = w.shape[0]
    _need(x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16 and w.shape == (N, K), "bf16 x [M,K], w [N,K]")
    _need(y.shape == (M, N) and y.dtype == torch.float32, "y float32 [M, N]")
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    _check(load().qv_bf16_linear(_ptr(x), M, K, _ptr(w), N, _ptr(y), _ptr(workspace),
                                 workspace.numel(), ctypes.c_void_p(_stream(stream))))


def linear_desc(x, wq, sw, y=None, act_mul=None) -> LinearDesc:
    """Descriptor of one quantize -> W8A8 linear phase (the tensors must stay
    alive while the descriptor is used)."""
    M, K = x.shape
    N = wq.shape[0]
    _need(wq.shape == (N, K) and wq.dtype == torch.int8, "wq int8 [N, K]")
    _need(sw.shape == (N,) and sw.dtype == torch.float32, "sw float32 [N]")
    if y is not None:
        _need(y.shape == (M, N) and y.dtype == torch.float32, "y float32 [M, N]")
    if act_mul is not None:
        _need(act_mul.shape == (K,) and act_mul.dtype == torch.float32, "act_mul float32 [K]")
    return LinearDesc(_ptr(x), _ptr(act_mul), _ptr(wq), _ptr(sw), _ptr(y), K, N)


def qv_verify_stack(linears, lm_head, M, x_dtype, workspace, tokens=None, max_logit=None,
                    draft=None, accept_len=None, out_tokens=None, stream=None):
    """linears: list of LinearDesc; lm_head: LinearDesc or None; x_dtype: the
    torch dtype of every phase input. B and gamma come from out_tokens [B, gamma+1]."""
    n = len(linears)
    arr = (LinearDesc * max(n, 1))(*linears)
    B, gamma = (out_tokens.shape[0], out_tokens.shape[1] - 1) if out_tokens is not None else (0, 0)
    dt = QV_BF16 if x_dtype == torch.bfloat16 else QV_F32
    _need(workspace.dtype == torch.uint8, "workspace must be a uint8 tensor")
    d = draft if (draft is not None and draft.numel() > 0) else None
    _check(load().qv_verify_stack(arr, n, ctypes.byref(lm_head) if lm_head is not None else None, M, dt,
                                  _ptr(d), B, gamma, _ptr(tokens), _ptr(max_logit), _ptr(accept_len),
                                  _ptr(out_tokens), _ptr(workspace), workspace.numel(),
                                  ctypes.c_void_p(_stream(stream))))


def qv_workspace_bytes(op: int, M: int, K: int, N: int) -> int:
    return int(load().qv_workspace_bytes(op, M, K, N))


def qv_device_error() -> int:
    code = ctypes.c_uint(0)
    _check(load().qv_device_error(ctypes.byref(code)))
    return int(code.value)


QV_DEVICE_ERR_FULL_WAIT = 1     # a consumer waited too long for a stage
QV_DEVICE_ERR_SLOT_WAIT = 32


def qv_debug_set_slot_wait_ns(ns: int):
    """Test hook: the split-K head's wait limit in later streaming launches (0 = default)."""
    load().qv_debug_set_slot_wait_ns(int(ns))


def qv_debug_drop_partials(n: int):
    """Test hook: the next n streaming launches publish no split-K partial sums."""
    load().qv_debug_drop_partials(int(n))


def qv_debug_hold_attention_loads(n: int):
    """Test hook: the next n qv_attention_verify calls request no key/value stage."""
    load().qv_debug_hold_attention_loads(int(n))


def qv_num_sms() -> int:
    return int(load().qv_num_sms())


def workspace(op: int, M: int, K: int, N: int, device=None) -> torch.Tensor:
    """A zero-filled workspace of the size the op needs (torch allocation)."""
    nbytes = qv_workspace_bytes(op, M, K, N)
    if nbytes == 0:
        raise ValueError(f"invalid shape for workspace: M={M} K={K} N={N}")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")
