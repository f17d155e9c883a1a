"""Python binding of libbeam_boundary.so: the Beam sublayer-boundary path on one GB300 (sm_103a).

Thin ctypes wrappers with the same names as the C ABI in ``include/beam_boundary.h``.  They only
marshal arguments (torch CUDA tensors -> device pointers, shapes, strides, the current stream)
and raise ``BeamError`` on a non-zero status; every step of the computation runs in the CUDA
kernels of the library.  There is no CPU fallback: if the library is missing, importing the
functions works but every call raises.

Build the library with ``residual_stream_norm_gb300.build()`` (nvcc, in-tree).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = ["BeamError", "build", "lib", "beam_abi_version", "beam_status_str",
           "beam_residual_scales", "beam_rope_cos_sin", "beam_residual_operand",
           "beam_exact_square_sum", "beam_routing_sigmoid", "beam_device_faults",
           "beam_selftest_copy_timeout", "beam_selftest_persistent_timeout",
           "beam_boundary_fwd", "beam_moe_combine_boundary_fwd", "beam_allreduce_boundary_fwd",
           "beam_qk_norm_rope_fwd", "beam_qk_norm_ssmax_fwd", "beam_qk_norm_rope_kv_fwd",
           "beam_qk_norm_ssmax_kv_fwd", "beam_grouped_topk_fwd", "beam_attn_gate_fwd",
           "HEAD_DIM"]

HEAD_DIM = 128
LIB_PATH = _build.LIB_PATH

_lock = threading.Lock()
_lib = None


class BeamError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status} ({beam_status_str(status)})")
        self.status = status


def build(force: bool = False) -> str:
    """Compile the CUDA library with nvcc (sm_103a) into the package's ``_lib`` folder."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library with argument types declared.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libbeam_boundary.so is not built ({LIB_PATH}); run "
                                   "residual_stream_norm_gb300.build() first")
            so = ctypes.CDLL(LIB_PATH)
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            so.beam_abi_version.argtypes = []
            so.beam_status_str.argtypes = [ctypes.c_int]
            so.beam_status_str.restype = ctypes.c_char_p
            so.beam_residual_scales.argtypes = [i32, ctypes.POINTER(f32), ctypes.POINTER(f32)]
            so.beam_rope_cos_sin.argtypes = [vp, vp, vp, i64]
            so.beam_residual_operand.argtypes = [vp, vp, i64, i32]
            so.beam_exact_square_sum.argtypes = [vp, i64, vp]
            so.beam_routing_sigmoid.argtypes = [vp, vp, i64]
            so.beam_device_faults.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
            so.beam_selftest_copy_timeout.argtypes = [i64, vp]
            so.beam_selftest_persistent_timeout.argtypes = [i32, vp, vp, vp, vp, vp, i64, i32, i64,
                                                            vp]
            so.beam_allreduce_boundary_fwd.argtypes = [vp, vp, vp, ctypes.POINTER(vp), i32, vp, vp,
                                                       i64, i32, i32, f32, vp, vp]
            so.beam_boundary_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, f32, vp, vp]
            so.beam_moe_combine_boundary_fwd.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, i64,
                                                         i32, i32, i32, f32, vp, vp]
            so.beam_qk_norm_rope_fwd.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, i32,
                                                 i32, f32, f32, vp]
            so.beam_qk_norm_ssmax_fwd.argtypes = [vp, vp, i64, i64, vp, vp, vp, i64, i32, i32,
                                                  i32, f32, f32, f32, vp]
            so.beam_attn_gate_fwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, i64, i64, i64, vp]
            so.beam_grouped_topk_fwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i32, vp]
            so.beam_qk_norm_rope_kv_fwd.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp, vp, vp, vp,
                                                    vp, i64, i32, f32, f32, i64, i32, i32, i32,
                                                    f32, f32, vp]
            so.beam_qk_norm_ssmax_kv_fwd.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp, vp, vp,
                                                     vp, vp, i64, i32, f32, f32, i64, i32, i32,
                                                     i32, f32, f32, f32, vp]
            for fn in ("beam_abi_version", "beam_residual_scales", "beam_rope_cos_sin",
                       "beam_residual_operand", "beam_exact_square_sum", "beam_routing_sigmoid",
                       "beam_device_faults", "beam_selftest_copy_timeout",
                       "beam_selftest_persistent_timeout", "beam_allreduce_boundary_fwd",
                       "beam_boundary_fwd",
                       "beam_moe_combine_boundary_fwd", "beam_qk_norm_rope_fwd",
                       "beam_qk_norm_ssmax_fwd", "beam_qk_norm_rope_kv_fwd",
                       "beam_qk_norm_ssmax_kv_fwd", "beam_grouped_topk_fwd",
                       "beam_attn_gate_fwd"):
                getattr(so, fn).restype = ctypes.c_int
            _lib = so
    return _lib


# ---------------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------------

def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bf16(t: torch.Tensor, name: str, contiguous: bool = True) -> None:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA bfloat16 tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _f32(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or \
            not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA float32 tensor")


def _call(fn: str, *args) -> None:
    st = getattr(lib(), fn)(*args)
    if st != 0:
        raise BeamError(fn, st)


# ---------------------------------------------------------------------------------------------
# the ABI, one wrapper per entry point
# ---------------------------------------------------------------------------------------------

def beam_abi_version() -> int:
    return lib().beam_abi_version()


def beam_status_str(status: int) -> str:
    return lib().beam_status_str(status).decode()


def beam_residual_scales(n: int) -> tuple[float, float]:
    a, s = ctypes.c_float(), ctypes.c_float()
    st = lib().beam_residual_scales(n, ctypes.byref(a), ctypes.byref(s))
    if st != 0:
        raise BeamError("beam_residual_scales", st)
    return a.value, s.value


def beam_device_faults(clear: bool = False) -> int:
    """The device fault word (0 in normal operation; bit 0: a kernel gave up waiting for its own
    bulk copies).  Synchronous."""
    v = ctypes.c_uint32()
    st = lib().beam_device_faults(ctypes.byref(v), int(clear))
    if st != 0:
        raise BeamError("beam_device_faults", st)
    return v.value


def beam_exact_square_sum(v) -> float:
    """Host helper: the FP32 sum of the FP32 squares of `v` (BF16 values as float32), rounded as
    the kernels' rare exact path rounds a row or head sum of squares."""
    import numpy as np
    a = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(1, dtype=np.float32)
    st = lib().beam_exact_square_sum(a.ctypes.data, a.size, out.ctypes.data)
    if st != 0:
        raise BeamError("beam_exact_square_sum", st)
    return out[0]


def beam_selftest_copy_timeout(limit_ns: int = 20_000_000, stream=None) -> None:
    """Diagnostic: run the kernels' copy-timeout path once (a wait nothing completes gives up
    after limit_ns and sets bit 0 of the device fault word)."""
    _call("beam_selftest_copy_timeout", limit_ns, _stream(stream))


def beam_selftest_persistent_timeout(kind: int, h_out, y_out, w_post, w_pre,
                                     limit_ns: int = 20_000_000, rstd_out=None,
                                     stream=None) -> None:
    """Diagnostic: run a persistent boundary kernel (kind 0: the plain boundary's prefetch kernel;
    1: the MoE ring) with its bulk copies withheld; its waits run out after limit_ns, it writes
    nothing to h_out / y_out [T, H] bf16 or rstd_out [T, 2] fp32 and sets bit 0 of the device
    fault word."""
    for t, nm in ((h_out, "h_out"), (y_out, "y_out"), (w_post, "w_post"), (w_pre, "w_pre")):
        _bf16(t, nm)
    T, H = h_out.shape
    if y_out.shape != (T, H) or w_post.shape != (H,) or w_pre.shape != (H,):
        raise ValueError("beam_selftest_persistent_timeout: shape mismatch")
    if rstd_out is not None:
        _f32(rstd_out, "rstd_out")
    with torch.cuda.device(h_out.device):
        _call("beam_selftest_persistent_timeout", kind, _ptr(h_out), _ptr(y_out), _ptr(rstd_out),
              _ptr(w_post), _ptr(w_pre), T, H, limit_ns, _stream(stream))


def beam_routing_sigmoid(z):
    """Host helper: the FP32 sigmoid the routing kernel ranks experts by (float32 in and out)."""
    import numpy as np
    a = np.ascontiguousarray(z, dtype=np.float32)
    out = np.empty_like(a)
    st = lib().beam_routing_sigmoid(a.ctypes.data, out.ctypes.data, a.size)
    if st != 0:
        raise BeamError("beam_routing_sigmoid", st)
    return out


def beam_residual_operand(x, n: int):
    """Host helper: b = bf16(x / fp32(sqrt(n))) for BF16 values x (as float32), exactly as the
    boundary kernels form it; returned as float32."""
    import numpy as np
    a = np.ascontiguousarray(x, dtype=np.float32)
    b = np.empty_like(a)
    st = lib().beam_residual_operand(a.ctypes.data, b.ctypes.data, a.size, n)
    if st != 0:
        raise BeamError("beam_residual_operand", st)
    return b


def beam_rope_cos_sin(angle):
    """Host helper: (cos, sin) as FP32 numpy arrays, exactly as the RoPE kernel forms them for
    the given FP32 angles (|angle| < 2^24)."""
    import numpy as np
    a = np.ascontiguousarray(angle, dtype=np.float32)
    c = np.empty_like(a)
    s = np.empty_like(a)
    st = lib().beam_rope_cos_sin(a.ctypes.data, c.ctypes.data, s.ctypes.data, a.size)
    if st != 0:
        raise BeamError("beam_rope_cos_sin", st)
    return c, s


def beam_boundary_fwd(h_out, y_out, h_in, x_in, w_post, w_pre, n: int, eps: float = 1e-6,
                      rstd_out=None, stream=None) -> None:
    """h_out, y_out, h_in, x_in: [T, H] bf16; w_post, w_pre: [H] bf16; rstd_out: [T, 2] fp32."""
    for t, nm in ((h_out, "h_out"), (y_out, "y_out"), (h_in, "h_in"), (x_in, "x_in"),
                  (w_post, "w_post"), (w_pre, "w_pre")):
        _bf16(t, nm)
    T, H = x_in.shape
    if h_in.shape != (T, H) or h_out.shape != (T, H) or y_out.shape != (T, H) or \
            w_post.shape != (H,) or w_pre.shape != (H,):
        raise ValueError("beam_boundary_fwd: shape mismatch")
    if rstd_out is not None:
        _f32(rstd_out, "rstd_out")
        if rstd_out.shape != (T, 2):
            raise ValueError("rstd_out must be [T, 2]")
    with torch.cuda.device(x_in.device):
        _call("beam_boundary_fwd", _ptr(h_out), _ptr(y_out), _ptr(h_in), _ptr(x_in),
              _ptr(w_post), _ptr(w_pre), T, H, n, eps, _ptr(rstd_out), _stream(stream))


def beam_moe_combine_boundary_fwd(h_out, y_out, h_in, expert_out, topk_w, w_post, w_pre,
                                  n: int, eps: float = 1e-6, routed_scaling: float = 2.5,
                                  rstd_out=None, stream=None) -> None:
    """expert_out: [T, K, H] bf16; topk_w: [T, K] fp32; the rest as beam_boundary_fwd."""
    for t, nm in ((h_out, "h_out"), (y_out, "y_out"), (h_in, "h_in"),
                  (expert_out, "expert_out"), (w_post, "w_post"), (w_pre, "w_pre")):
        _bf16(t, nm)
    _f32(topk_w, "topk_w")
    T, K, H = expert_out.shape
    if h_in.shape != (T, H) or h_out.shape != (T, H) or y_out.shape != (T, H) or \
            topk_w.shape != (T, K) or w_post.shape != (H,) or w_pre.shape != (H,):
        raise ValueError("beam_moe_combine_boundary_fwd: shape mismatch")
    if rstd_out is not None:
        _f32(rstd_out, "rstd_out")
        if rstd_out.shape != (T, 2):
            raise ValueError("rstd_out must be [T, 2]")
    with torch.cuda.device(h_in.device):
        _call("beam_moe_combine_boundary_fwd", _ptr(h_out), _ptr(y_out), _ptr(h_in),
              _ptr(expert_out), _ptr(topk_w), routed_scaling, _ptr(w_post), _ptr(w_pre), T, H,
              K, n, eps, _ptr(rstd_out), _stream(stream))


def beam_allreduce_boundary_fwd(h_out, y_out, h_in, x_parts, w_post, w_pre, n: int,
                                eps: float = 1e-6, rstd_out=None, stream=None) -> None:
    """x_parts: a sequence of P [T, H] bf16 tensors (rank p's partial sublayer output), or one
    [P, T, H] tensor; the rest as beam_boundary_fwd.  The partials are summed in rank order in
    FP32 and rounded once to BF16 ahead of the boundary chain."""
    parts = list(x_parts.unbind(0)) if isinstance(x_parts, torch.Tensor) else list(x_parts)
    for t, nm in ((h_out, "h_out"), (y_out, "y_out"), (h_in, "h_in"), (w_post, "w_post"),
                  (w_pre, "w_pre")):
        _bf16(t, nm)
    T, H = h_in.shape
    for i, t in enumerate(parts):
        _bf16(t, f"x_parts[{i}]")
        if t.shape != (T, H):
            raise ValueError("beam_allreduce_boundary_fwd: every partial must be [T, H]")
    if h_out.shape != (T, H) or y_out.shape != (T, H) or w_post.shape != (H,) or \
            w_pre.shape != (H,):
        raise ValueError("beam_allreduce_boundary_fwd: shape mismatch")
    if rstd_out is not None:
        _f32(rstd_out, "rstd_out")
        if rstd_out.shape != (T, 2):
            raise ValueError("rstd_out must be [T, 2]")
    arr = (ctypes.c_void_p * max(1, len(parts)))(*[t.data_ptr() for t in parts])
    with torch.cuda.device(h_in.device):
        _call("beam_allreduce_boundary_fwd", _ptr(h_out), _ptr(y_out), _ptr(h_in), arr,
              len(parts), _ptr(w_post), _ptr(w_pre), T, H, n, eps, _ptr(rstd_out),
              _stream(stream))


def _heads(t, name):
    """[T, heads, 128] bf16 view whose heads and elements are contiguous (rows may be strided)."""
    _bf16(t, name, contiguous=False)
    if t.dim() != 3 or t.shape[2] != HEAD_DIM or t.stride(2) != 1 or \
            (t.shape[1] > 1 and t.stride(1) != HEAD_DIM):
        raise ValueError(f"{name}: expected [T, heads, {HEAD_DIM}] with contiguous heads")
    return t.shape[0], t.shape[1], t.stride(0)


def _qk_common(q, k, wq, wk, pos):
    T, nq, qs = _heads(q, "q")
    Tk, nk, ks = _heads(k, "k")
    if Tk != T:
        raise ValueError("q and k must have the same number of tokens")
    _bf16(wq, "wq")
    _bf16(wk, "wk")
    if not (isinstance(pos, torch.Tensor) and pos.dtype == torch.int64 and pos.is_cuda and
            pos.is_contiguous() and pos.shape == (T,)):
        raise TypeError("pos: expected a contiguous CUDA int64 tensor of shape [T]")
    return T, nq, nk, qs, ks


def beam_qk_norm_rope_fwd(q, k, wq, wk, pos, eps: float = 1e-6, theta: float = 10000.0,
                          stream=None) -> None:
    """In place: q [T, nq, 128], k [T, nk, 128] bf16 (row-strided views allowed), wq, wk [128]
    bf16, pos [T] int64 0-based."""
    T, nq, nk, qs, ks = _qk_common(q, k, wq, wk, pos)
    with torch.cuda.device(q.device):
        _call("beam_qk_norm_rope_fwd", _ptr(q), _ptr(k), qs, ks, _ptr(wq), _ptr(wk), _ptr(pos),
              T, nq, nk, HEAD_DIM, eps, theta, _stream(stream))


def beam_qk_norm_ssmax_fwd(q, k, wq, wk, pos, eps: float = 1e-6, ssmax_base: float = 2048.0,
                           ssmax_exp: float = 0.1, stream=None) -> None:
    """In place, as beam_qk_norm_rope_fwd; queries are scaled by (1 + (pos+1)/base)^exp."""
    T, nq, nk, qs, ks = _qk_common(q, k, wq, wk, pos)
    with torch.cuda.device(q.device):
        _call("beam_qk_norm_ssmax_fwd", _ptr(q), _ptr(k), qs, ks, _ptr(wq), _ptr(wk), _ptr(pos),
              T, nq, nk, HEAD_DIM, eps, ssmax_base, ssmax_exp, _stream(stream))


CACHE_BF16, CACHE_FP8_E4M3 = 0, 1


def _kv_common(k, v, slot_mapping, k_cache, v_cache, cache_dtype):
    T, nk, ks = _heads(k, "k")
    Tv, nv, vs = _heads(v, "v")
    if (Tv, nv) != (T, nk):
        raise ValueError("v must have k's shape")
    if not (isinstance(slot_mapping, torch.Tensor) and slot_mapping.dtype == torch.int64 and
            slot_mapping.is_cuda and slot_mapping.is_contiguous() and slot_mapping.shape == (T,)):
        raise TypeError("slot_mapping: expected a contiguous CUDA int64 tensor of shape [T]")
    esize = 2 if cache_dtype == CACHE_BF16 else 1
    for c, nm in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        if not (isinstance(c, torch.Tensor) and c.is_cuda and c.is_contiguous() and
                c.element_size() == esize and c.dim() == 3 and c.shape[1:] == (nk, HEAD_DIM) and
                (cache_dtype != CACHE_BF16 or c.dtype == torch.bfloat16)):
            raise TypeError(f"{nm}: expected a contiguous CUDA [num_slots, {nk}, {HEAD_DIM}] "
                            f"tensor of {esize}-byte elements")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    return vs, k_cache.shape[0]


def beam_qk_norm_rope_kv_fwd(q, k, v, wq, wk, pos, slot_mapping, k_cache, v_cache,
                             cache_dtype: int = CACHE_BF16, k_scale: float = 1.0,
                             v_scale: float = 1.0, eps: float = 1e-6, theta: float = 10000.0,
                             stream=None) -> None:
    """beam_qk_norm_rope_fwd fused with the KV-cache write: K' (as stored) and v [T, nk, 128]
    bf16 go to the slots slot_mapping [T] int64 of k_cache / v_cache [num_slots, nk, 128]:
    bfloat16 tensors for CACHE_BF16, 1-byte tensors (uint8 or float8_e4m3fn) for
    CACHE_FP8_E4M3 (value / scale).  Negative or out-of-range slots are skipped."""
    T, nq, nk, qs, ks = _qk_common(q, k, wq, wk, pos)
    vs, num_slots = _kv_common(k, v, slot_mapping, k_cache, v_cache, cache_dtype)
    with torch.cuda.device(q.device):
        _call("beam_qk_norm_rope_kv_fwd", _ptr(q), _ptr(k), qs, ks, _ptr(v), vs, _ptr(wq),
              _ptr(wk), _ptr(pos), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), num_slots,
              cache_dtype, k_scale, v_scale, T, nq, nk, HEAD_DIM, eps, theta, _stream(stream))


def beam_qk_norm_ssmax_kv_fwd(q, k, v, wq, wk, pos, slot_mapping, k_cache, v_cache,
                              cache_dtype: int = CACHE_BF16, k_scale: float = 1.0,
                              v_scale: float = 1.0, eps: float = 1e-6, ssmax_base: float = 2048.0,
                              ssmax_exp: float = 0.1, stream=None) -> None:
    """beam_qk_norm_ssmax_fwd fused with the KV-cache write (as beam_qk_norm_rope_kv_fwd)."""
    T, nq, nk, qs, ks = _qk_common(q, k, wq, wk, pos)
    vs, num_slots = _kv_common(k, v, slot_mapping, k_cache, v_cache, cache_dtype)
    with torch.cuda.device(q.device):
        _call("beam_qk_norm_ssmax_kv_fwd", _ptr(q), _ptr(k), qs, ks, _ptr(v), vs, _ptr(wq),
              _ptr(wk), _ptr(pos), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), num_slots,
              cache_dtype, k_scale, v_scale, T, nq, nk, HEAD_DIM, eps, ssmax_base, ssmax_exp,
              _stream(stream))


def beam_grouped_topk_fwd(topk_ids, topk_w, logits, bias, n_groups: int = 8,
                          topk_groups: int = 4, stream=None) -> None:
    """DeepSeek-V3-style grouped routing: logits [T, 256] fp32, bias [256] fp32 -> topk_ids
    [T, 8] int32 (best first) and topk_w [T, 8] fp32 (renormalised sigmoid scores)."""
    def f32c(t, nm):
        if not (isinstance(t, torch.Tensor) and t.dtype == torch.float32 and t.is_cuda and
                t.is_contiguous()):
            raise TypeError(f"{nm}: expected a contiguous CUDA float32 tensor")
    f32c(logits, "logits")
    f32c(bias, "bias")
    f32c(topk_w, "topk_w")
    if not (isinstance(topk_ids, torch.Tensor) and topk_ids.dtype == torch.int32 and
            topk_ids.is_cuda and topk_ids.is_contiguous()):
        raise TypeError("topk_ids: expected a contiguous CUDA int32 tensor")
    T, E = logits.shape
    k = topk_ids.shape[1] if topk_ids.dim() == 2 else -1
    if bias.shape != (E,) or topk_ids.shape != (T, k) or topk_w.shape != (T, k):
        raise ValueError("beam_grouped_topk_fwd: shape mismatch")
    with torch.cuda.device(logits.device):
        _call("beam_grouped_topk_fwd", _ptr(topk_ids), _ptr(topk_w), _ptr(logits), _ptr(bias), T,
              E, n_groups, topk_groups, k, _stream(stream))


def beam_attn_gate_fwd(out, attn, gate, bias, n_heads: int, head_dim: int = HEAD_DIM,
                       stream=None) -> None:
    """out, attn, gate: [T, n_heads*head_dim] bf16 (row-strided allowed); bias [n_heads] fp32."""
    for t, nm in ((out, "out"), (attn, "attn"), (gate, "gate")):
        _bf16(t, nm, contiguous=False)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{nm}: expected [T, C] with contiguous rows")
    _f32(bias, "bias")
    T, C = attn.shape
    if gate.shape != (T, C) or out.shape != (T, C) or C != n_heads * head_dim or \
            bias.shape != (n_heads,):
        raise ValueError("beam_attn_gate_fwd: shape mismatch")
    with torch.cuda.device(attn.device):
        _call("beam_attn_gate_fwd", _ptr(out), _ptr(attn), _ptr(gate), _ptr(bias), T, n_heads,
              head_dim, attn.stride(0), gate.stride(0), out.stride(0), _stream(stream))
