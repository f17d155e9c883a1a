"""CPU oracle for the Beam sublayer-boundary path (ctypes wrapper over ``beam_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The CUDA library never
imports, links or calls it, and it imports nothing from the CUDA library.

All BF16 tensors cross this interface as ``numpy.uint16`` arrays of bit patterns.  The functions
return fresh arrays; inputs are never modified (the in-place Q/K calls work on copies).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "beam_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libbeam_oracle.so")

# -ffp-contract=off: the oracle's FP32 steps must not be fused into multiply-adds.
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build/``; return the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _P(dt):
    return ctypes.POINTER(dt)


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            so = ctypes.CDLL(build())
            u16p, f32p, i64p = _P(ctypes.c_uint16), _P(ctypes.c_float), _P(ctypes.c_int64)
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            so.orc_bf16_rne.argtypes = [f32]
            so.orc_bf16_rne.restype = ctypes.c_uint16
            so.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            so.orc_bf16_to_f32.restype = f32
            so.orc_bf16_rne_array.argtypes = [f32p, u16p, i64]
            so.orc_residual_scales.argtypes = [i32, f32p, f32p]
            so.orc_rope_inv_freq.argtypes = [f32, i32, f32p]
            so.orc_exact_sum_f32.argtypes = [f32p, i64]
            so.orc_exact_sum_f32.restype = f32
            so.orc_ssmax_scale.argtypes = [i64, f32, f32]
            so.orc_ssmax_scale.restype = f32
            so.orc_boundary.argtypes = [u16p, u16p, u16p, u16p, u16p, u16p, i64, i32, i32, f32,
                                        f32p, f32p]
            so.orc_moe_combine_boundary.argtypes = [u16p, u16p, u16p, u16p, f32p, f32, u16p,
                                                    u16p, i64, i32, i32, i32, f32, f32p, u16p,
                                                    f32p]
            so.orc_allreduce_boundary.argtypes = [u16p, u16p, u16p, u16p, i32, u16p, u16p, i64,
                                                  i32, i32, f32, f32p, u16p, f32p]
            so.orc_qk_norm_rope.argtypes = [u16p, u16p, i64, i64, u16p, u16p, i64p, i64, i32,
                                            i32, i32, f32, f32, f32p]
            so.orc_qk_norm_ssmax.argtypes = [u16p, u16p, i64, i64, u16p, u16p, i64p, i64, i32,
                                             i32, i32, f32, f32, f32, f32p]
            so.orc_attn_gate.argtypes = [u16p, u16p, u16p, f32p, i64, i32, i32, i64, i64, i64]
            so.orc_sigmoid_f32.argtypes = [f32]
            so.orc_sigmoid_f32.restype = f32
            so.orc_sigmoid_array.argtypes = [f32p, f32p, i64]
            so.orc_sigmoid_array.restype = None
            so.orc_exp_f32.argtypes = [f32]
            so.orc_exp_f32.restype = f32
            so.orc_grouped_topk.argtypes = [_P(ctypes.c_int32), f32p, f32p, f32p, i64, i32, i32,
                                            i32, i32, f32p, _P(ctypes.c_int32)]
            so.orc_grouped_topk.restype = None
            u8 = ctypes.c_uint8
            so.orc_fp8_e4m3_rne.argtypes = [f32]
            so.orc_fp8_e4m3_rne.restype = u8
            so.orc_fp8_e4m3_to_f32.argtypes = [u8]
            so.orc_fp8_e4m3_to_f32.restype = f32
            so.orc_kv_cache_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, u16p, u16p, i64,
                                              i64, i64p, i64, i32, i32, i64, i32, f32, f32]
            for fn in ("orc_bf16_rne_array", "orc_residual_scales", "orc_rope_inv_freq",
                       "orc_boundary", "orc_moe_combine_boundary", "orc_allreduce_boundary",
                       "orc_qk_norm_rope",
                       "orc_qk_norm_ssmax", "orc_attn_gate", "orc_kv_cache_write"):
                getattr(so, fn).restype = None
            _lib = so
    return _lib


def _ptr(a: np.ndarray | None, ct):
    if a is None:
        return ctypes.cast(None, _P(ct))
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(_P(ct))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"expected BF16 bit patterns as uint16, got {a.dtype}"
    return a


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


# ---------------------------------------------------------------------------------------------
# scalar / elementwise helpers
# ---------------------------------------------------------------------------------------------

def bf16_rne(x) -> np.ndarray:
    """FP32 values -> BF16 bit patterns (round to nearest even)."""
    x = _f32(x)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_bf16_rne_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), x.size)
    return out


def bf16_to_f32(b) -> np.ndarray:
    """BF16 bit patterns -> FP32 values (exact widening)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def exact_sum_f32(terms) -> float:
    """The FP32 rounding (nearest even) of the exact sum of non-negative FP32 terms."""
    t = _f32(terms)
    return lib().orc_exact_sum_f32(_ptr(t, ctypes.c_float), t.size)


def residual_scales(n: int) -> tuple[float, float]:
    """(alpha, s) = (fp32(sqrt((n-1)/n)), fp32(sqrt(n))) of the n-th residual add."""
    a, s = ctypes.c_float(), ctypes.c_float()
    lib().orc_residual_scales(n, ctypes.byref(a), ctypes.byref(s))
    return a.value, s.value


def rope_inv_freq(theta: float, head_dim: int) -> np.ndarray:
    out = np.empty(head_dim // 2, dtype=np.float32)
    lib().orc_rope_inv_freq(theta, head_dim, _ptr(out, ctypes.c_float))
    return out


def ssmax_scale(pos: int, base: float = 2048.0, expo: float = 0.1) -> float:
    return lib().orc_ssmax_scale(int(pos), base, expo)


# ---------------------------------------------------------------------------------------------
# the five operations
# ---------------------------------------------------------------------------------------------

def boundary(h, x, w_post, w_pre, n: int, eps: float = 1e-6):
    """Post-RMSNorm -> depth-scaled residual add -> next pre-RMSNorm, per token.

    h, x: [T, H] uint16; w_post, w_pre: [H] uint16.  Returns (h_out, y, rstd[T, 2])."""
    h, x, w_post, w_pre = _u16(h), _u16(x), _u16(w_post), _u16(w_pre)
    T, H = x.shape
    assert h.shape == (T, H) and w_post.shape == (H,) and w_pre.shape == (H,) and n >= 1
    h_out = np.empty_like(h)
    y = np.empty_like(x)
    rstd = np.empty((T, 2), dtype=np.float32)
    work = np.empty(3 * H, dtype=np.float32)
    u, f = ctypes.c_uint16, ctypes.c_float
    lib().orc_boundary(_ptr(h_out, u), _ptr(y, u), _ptr(h, u), _ptr(x, u), _ptr(w_post, u),
                       _ptr(w_pre, u), T, H, n, eps, _ptr(rstd, f), _ptr(work, f))
    return h_out, y, rstd


def moe_combine_boundary(h, expert_out, topk_w, w_post, w_pre, n: int, eps: float = 1e-6,
                         routed_scaling: float = 2.5, return_x: bool = False):
    """Top-K combine x = bf16(sum_k fp32(w_k * scale) * e_k), then the boundary chain.

    h: [T, H]; expert_out: [T, K, H] uint16; topk_w: [T, K] float32.
    Returns (h_out, y, rstd[T, 2]) or (h_out, y, rstd, x) with ``return_x``."""
    h, e, w_post, w_pre = _u16(h), _u16(expert_out), _u16(w_post), _u16(w_pre)
    w = _f32(topk_w)
    T, K, H = e.shape
    assert h.shape == (T, H) and w.shape == (T, K) and 1 <= K <= 64 and n >= 1
    h_out = np.empty_like(h)
    y = np.empty_like(h)
    rstd = np.empty((T, 2), dtype=np.float32)
    x_out = np.empty_like(h) if return_x else None
    work = np.empty(3 * H, dtype=np.float32)
    u, f = ctypes.c_uint16, ctypes.c_float
    lib().orc_moe_combine_boundary(_ptr(h_out, u), _ptr(y, u), _ptr(h, u), _ptr(e, u),
                                   _ptr(w, f), routed_scaling, _ptr(w_post, u), _ptr(w_pre, u),
                                   T, H, K, n, eps, _ptr(rstd, f), _ptr(x_out, u), _ptr(work, f))
    return (h_out, y, rstd, x_out) if return_x else (h_out, y, rstd)


def allreduce_boundary(h, parts, w_post, w_pre, n: int, eps: float = 1e-6,
                       return_x: bool = False):
    """Tensor-parallel partial outputs summed in rank order in FP32 and rounded once to BF16,
    then the boundary chain.

    h: [T, H] uint16; parts: [P, T, H] uint16 (rank p's partial sublayer output at parts[p]).
    Returns (h_out, y, rstd[T, 2]) or (h_out, y, rstd, x) with ``return_x``."""
    h, w_post, w_pre = _u16(h), _u16(w_post), _u16(w_pre)
    parts = _u16(parts)
    P, T, H = parts.shape
    assert h.shape == (T, H) and w_post.shape == (H,) and w_pre.shape == (H,)
    assert P >= 1 and n >= 1
    h_out = np.empty_like(h)
    y = np.empty_like(h)
    rstd = np.empty((T, 2), dtype=np.float32)
    x_out = np.empty_like(h) if return_x else None
    work = np.empty(3 * H, dtype=np.float32)
    u, f = ctypes.c_uint16, ctypes.c_float
    lib().orc_allreduce_boundary(_ptr(h_out, u), _ptr(y, u), _ptr(h, u), _ptr(parts, u), P,
                                 _ptr(w_post, u), _ptr(w_pre, u), T, H, n, eps, _ptr(rstd, f),
                                 _ptr(x_out, u), _ptr(work, f))
    return (h_out, y, rstd, x_out) if return_x else (h_out, y, rstd)


def qk_norm_rope(q, k, wq, wk, pos, eps: float = 1e-6, theta: float = 10000.0):
    """Per-head RMSNorm + half-rotation RoPE.  q: [T, nq, D], k: [T, nk, D] uint16,
    wq, wk: [D] uint16, pos: [T] int64.  Returns new (q, k)."""
    q = np.array(_u16(q), copy=True)
    k = np.array(_u16(k), copy=True)
    wq, wk = _u16(wq), _u16(wk)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    T, nq, D = q.shape
    nk = k.shape[1]
    assert k.shape == (T, nk, D) and pos.shape == (T,) and D % 2 == 0
    work = np.empty(3 * (D // 2) + 2 * D, dtype=np.float32)
    u = ctypes.c_uint16
    lib().orc_qk_norm_rope(_ptr(q, u), _ptr(k, u), nq * D, nk * D, _ptr(wq, u), _ptr(wk, u),
                           _ptr(pos, ctypes.c_int64), T, nq, nk, D, eps, theta,
                           _ptr(work, ctypes.c_float))
    return q, k


def qk_norm_ssmax(q, k, wq, wk, pos, eps: float = 1e-6, base: float = 2048.0,
                  expo: float = 0.1):
    """Per-head RMSNorm; queries also times the SSMax scale of their 0-based position."""
    q = np.array(_u16(q), copy=True)
    k = np.array(_u16(k), copy=True)
    wq, wk = _u16(wq), _u16(wk)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    T, nq, D = q.shape
    nk = k.shape[1]
    assert k.shape == (T, nk, D) and pos.shape == (T,)
    work = np.empty(2 * D, dtype=np.float32)
    u = ctypes.c_uint16
    lib().orc_qk_norm_ssmax(_ptr(q, u), _ptr(k, u), nq * D, nk * D, _ptr(wq, u), _ptr(wk, u),
                            _ptr(pos, ctypes.c_int64), T, nq, nk, D, eps, base, expo,
                            _ptr(work, ctypes.c_float))
    return q, k


def sigmoid_f32(z: float) -> float:
    """FP32 sigmoid 1 / (1 + RN32(exp(-z))), FP32 add, IEEE division."""
    return float(lib().orc_sigmoid_f32(float(z)))


def sigmoid_array(z) -> np.ndarray:
    """sigmoid_f32 over an array of float32 values."""
    z = _f32(z)
    out = np.empty_like(z)
    lib().orc_sigmoid_array(_ptr(z, ctypes.c_float), _ptr(out, ctypes.c_float), z.size)
    return out


def exp_f32(x: float) -> float:
    """exp(x) rounded once to FP32 (long double evaluation)."""
    return float(lib().orc_exp_f32(float(x)))


def grouped_topk(logits, bias, n_groups: int = 8, topk_groups: int = 4, top_k: int = 8):
    """DeepSeek-V3-style grouped routing.  logits [T, E] float32, bias [E] float32.  Returns
    (ids [T, top_k] int32, best first; weights [T, top_k] float32, renormalised, unscaled)."""
    z = _f32(logits)
    b = _f32(bias)
    T, E = z.shape
    assert b.shape == (E,) and E % n_groups == 0 and 1 <= topk_groups <= n_groups
    ids = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float32)
    work = np.empty(2 * E + n_groups, dtype=np.float32)
    iwork = np.empty(E + n_groups, dtype=np.int32)
    lib().orc_grouped_topk(_ptr(ids, ctypes.c_int32), _ptr(w, ctypes.c_float),
                           _ptr(z, ctypes.c_float), _ptr(b, ctypes.c_float), T, E, n_groups,
                           topk_groups, top_k, _ptr(work, ctypes.c_float),
                           _ptr(iwork, ctypes.c_int32))
    return ids, w


def fp8_e4m3_rne(x: float) -> int:
    """FP32 -> FP8 E4M3 code (round to nearest even, saturating to +-448, NaN -> 0x7f)."""
    return int(lib().orc_fp8_e4m3_rne(float(x)))


def fp8_e4m3_to_f32(code: int) -> float:
    """Value of an FP8 E4M3 code."""
    return float(lib().orc_fp8_e4m3_to_f32(int(code)))


def kv_cache_write(k_cache, v_cache, k, v, slot_mapping, cache_dtype: int = 0,
                   k_scale: float = 1.0, v_scale: float = 1.0):
    """Writes K' rows k [T, nk, D] and V rows v [T, nk, D] (uint16 BF16) into the slots
    slot_mapping [T] of the caches [num_slots, nk, D]: uint16 for cache_dtype 0 (BF16), uint8
    for cache_dtype 1 (FP8 E4M3 of value / scale).  Negative or out-of-range slots are skipped.
    Returns new (k_cache, v_cache)."""
    k, v = _u16(k), _u16(v)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, nk, D = k.shape
    assert v.shape == (T, nk, D) and slots.shape == (T,)
    dt = np.uint16 if cache_dtype == 0 else np.uint8
    kc = np.array(k_cache, dtype=dt, copy=True)
    vc = np.array(v_cache, dtype=dt, copy=True)
    assert kc.shape == vc.shape and kc.shape[1:] == (nk, D)
    u = ctypes.c_uint16
    lib().orc_kv_cache_write(kc.ctypes.data, vc.ctypes.data, _ptr(k, u), _ptr(v, u), nk * D,
                             nk * D, _ptr(slots, ctypes.c_int64), T, nk, D, kc.shape[0],
                             cache_dtype, k_scale, v_scale)
    return kc, vc


def attn_gate(attn, gate, bias, n_heads: int, head_dim: int):
    """out = bf16(attn * sigmoid(gate + bias_head)).  attn, gate: [T, n_heads*head_dim] uint16,
    bias: [n_heads] float32."""
    attn, gate = _u16(attn), _u16(gate)
    bias = _f32(bias)
    T, C = attn.shape
    assert gate.shape == (T, C) and C == n_heads * head_dim and bias.shape == (n_heads,)
    out = np.empty_like(attn)
    u = ctypes.c_uint16
    lib().orc_attn_gate(_ptr(out, u), _ptr(attn, u), _ptr(gate, u), _ptr(bias, ctypes.c_float),
                        T, n_heads, head_dim, C, C, C)
    return out


# ---------------------------------------------------------------------------------------------
# token-parallel driver for timing the oracle on several host cores
# ---------------------------------------------------------------------------------------------

def split_tokens(T: int, parts: int) -> list[tuple[int, int]]:
    """Contiguous [lo, hi) token slices, as even as possible."""
    parts = max(1, min(parts, T)) if T > 0 else 1
    base, rem = divmod(T, parts)
    out, lo = [], 0
    for i in range(parts):
        hi = lo + base + (1 if i < rem else 0)
        out.append((lo, hi))
        lo = hi
    return out


def run_token_parallel(fn, T: int, threads: int):
    """Run ``fn(lo, hi)`` over token slices on ``threads`` threads (ctypes drops the GIL while
    the C oracle runs).  Returns the list of results in slice order."""
    slices = split_tokens(T, threads)
    if len(slices) == 1:
        return [fn(*slices[0])]
    with ThreadPoolExecutor(max_workers=len(slices)) as ex:
        return list(ex.map(lambda s: fn(*s), slices))
