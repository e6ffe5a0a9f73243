"""fp64 CPU oracle for multi-head scaled dot-product attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The library's CUDA path never calls it and the
two share no code. The arithmetic lives in ``attention_oracle.c`` (plain C,
fp64, OpenMP over independent (batch, head) pairs); this module only builds
that file with gcc and marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile attention_oracle.c into liboracle.so (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.oracle_attention.argtypes = [dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ci, ip, cd, ci]
            lib.oracle_attention.restype = ci
            lib.oracle_attention_window.argtypes = [dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ci,
                                                    ip, ci, ci, cd, ci]
            lib.oracle_attention_window.restype = ci
            lib.oracle_attention_rows.argtypes = [dp, ip, ci, dp, dp, ci, ci, ci, ci, ci, cd, dp, ci]
            lib.oracle_attention_rows.restype = ci
            lib.oracle_attention_rows_window.argtypes = [dp, ip, ci, dp, dp, ci, ci, ci, ci, ci,
                                                         ci, ci, cd, dp, ci]
            lib.oracle_attention_rows_window.restype = ci
            lib.oracle_mha.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ci,
                                       ci, ip, cd, ci]
            lib.oracle_mha.restype = ci
            lib.oracle_decode.argtypes = [dp, dp, dp, dp, ci, ci, ci, ci, ci, ci, ip, cd, ci]
            lib.oracle_decode.restype = ci
            lib.oracle_layernorm.argtypes = [dp, dp, dp, dp, ci, ci, cd]
            lib.oracle_layernorm.restype = None
            lib.oracle_ffn.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, ci]
            lib.oracle_ffn.restype = ci
            lib.oracle_encoder_layer.argtypes = [dp] * 15 + [ci] * 7 + [ip, cd, cd, ci]
            lib.oracle_encoder_layer.restype = ci
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _dp(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_int32)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _f64(a):
    """Values as contiguous fp64. 16-bit integer arrays are refused: those are
    bf16 bit patterns, which must be widened to their values first."""
    a = np.asarray(a)
    if a.dtype in (np.uint16, np.int16):
        raise TypeError("the oracle takes values, not 16-bit patterns: widen bf16 bits first")
    return np.ascontiguousarray(a, dtype=np.float64)


def default_scale(d_k: int) -> float:
    """1/sqrt(d_k), the factor of eq. (1)."""
    return 1.0 / np.sqrt(float(d_k))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _window(window):
    """(left, right) of a restricted window; None or a negative side = no bound."""
    if window is None:
        return -1, -1
    left, right = window
    return (-1 if left is None or left < 0 else int(left)), \
           (-1 if right is None or right < 0 else int(right))


def attention(q, k, v, mask_kind: int = MASK_NONE, kv_lens=None, scale: float | None = None,
              return_weights: bool = False, nthreads: int = 0, window=None):
    """Attention(Q,K,V) for q [B,h,n_q,d_k], k [B,h,n_k,d_k], v [B,h,n_k,d_v].

    window = (left, right): restricted self-attention, query i sees only keys
    j in [i - left, i + right] (n_q == n_k); None = unrestricted.
    Returns out [B,h,n_q,d_v] (and the weight matrix [B,h,n_q,n_k] when asked).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, h, n_q, d_k = q.shape
    n_k, d_v = k.shape[2], v.shape[3]
    assert k.shape == (B, h, n_k, d_k) and v.shape == (B, h, n_k, d_v)
    if scale is None or scale == 0.0:
        scale = default_scale(d_k)
    lens = None
    if mask_kind & MASK_KEY_PADDING:
        lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))
        assert lens.shape == (B,)
    out = np.zeros((B, h, n_q, d_v), dtype=np.float64)
    w = np.zeros((B, h, n_q, n_k), dtype=np.float64) if return_weights else None
    wl, wr = _window(window)
    rc = _load().oracle_attention_window(_dp(q), _dp(k), _dp(v), _dp(out), _dp(w), B, h, n_q, n_k,
                                         d_k, d_v, int(mask_kind), _ip(lens), wl, wr, float(scale),
                                         int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return (out, w) if return_weights else out


def attention_rows(q_rows, row_pos, K, V, causal: bool, kv_len: int | None = None,
                   scale: float | None = None, nthreads: int = 0, window=None):
    """Selected query rows of one (batch, head): q_rows [R,d_k] at positions row_pos [R]."""
    q_rows, K, V = _f64(q_rows), _f64(K), _f64(V)
    R, d_k = q_rows.shape
    n_k, d_v = V.shape
    pos = np.ascontiguousarray(np.asarray(row_pos, dtype=np.int32))
    if scale is None or scale == 0.0:
        scale = default_scale(d_k)
    out = np.zeros((R, d_v), dtype=np.float64)
    wl, wr = _window(window)
    rc = _load().oracle_attention_rows_window(_dp(q_rows), _ip(pos), R, _dp(K), _dp(V), n_k, d_k,
                                              d_v, int(bool(causal)),
                                              -1 if kv_len is None else int(kv_len), wl, wr,
                                              float(scale), _dp(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return out


def decode(q, k_cache, v_cache, cache_lens=None, scale: float | None = None, nthreads: int = 0):
    """One decoding step against a key/value cache.

    q [B,h,n_q,d_k]: the n_q newest tokens' queries; k_cache [B,h,n_max,d_k],
    v_cache [B,h,n_max,d_v]: every position so far, the new tokens included;
    cache_lens [B] (None = n_max): valid rows L per batch entry. Query t sits
    at position L - n_q + t and sees the keys at positions <= its own.
    Returns out [B,h,n_q,d_v].
    """
    q, k_cache, v_cache = _f64(q), _f64(k_cache), _f64(v_cache)
    B, h, n_q, d_k = q.shape
    n_max, d_v = k_cache.shape[2], v_cache.shape[3]
    assert k_cache.shape == (B, h, n_max, d_k) and v_cache.shape == (B, h, n_max, d_v)
    if scale is None or scale == 0.0:
        scale = default_scale(d_k)
    lens = None
    if cache_lens is not None:
        lens = np.ascontiguousarray(np.asarray(cache_lens, dtype=np.int32))
        assert lens.shape == (B,)
    out = np.zeros((B, h, n_q, d_v), dtype=np.float64)
    rc = _load().oracle_decode(_dp(q), _dp(k_cache), _dp(v_cache), _dp(out), B, h, n_q, n_max,
                               d_k, d_v, _ip(lens), float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out


def mha(x_q, x_kv, w_q, w_k, w_v, w_o, h: int, mask_kind: int = MASK_NONE, kv_lens=None,
        scale: float | None = None, return_concat: bool = False, nthreads: int = 0):
    """MultiHead(X_q, X_kv) = Concat(head_1..head_h) W_O (x.W convention, no biases)."""
    x_q, x_kv = _f64(x_q), _f64(x_kv)
    w_q, w_k, w_v, w_o = _f64(w_q), _f64(w_k), _f64(w_v), _f64(w_o)
    B, n_q, d_model = x_q.shape
    n_k = x_kv.shape[1]
    d_k = w_q.shape[1] // h
    d_v = w_v.shape[1] // h
    assert w_q.shape == (d_model, h * d_k) and w_k.shape == (d_model, h * d_k)
    assert w_v.shape == (d_model, h * d_v) and w_o.shape == (h * d_v, d_model)
    if scale is None or scale == 0.0:
        scale = default_scale(d_k)
    lens = None
    if mask_kind & MASK_KEY_PADDING:
        lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))
    out = np.zeros((B, n_q, d_model), dtype=np.float64)
    concat = np.zeros((B, n_q, h * d_v), dtype=np.float64) if return_concat else None
    rc = _load().oracle_mha(_dp(x_q), _dp(x_kv), _dp(w_q), _dp(w_k), _dp(w_v), _dp(w_o), _dp(out),
                            _dp(concat), B, n_q, n_k, d_model, h, d_k, d_v, int(mask_kind),
                            _ip(lens), float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_mha rejected its arguments")
    return (out, concat) if return_concat else out


def layernorm(x, gamma, beta, eps: float):
    """gamma (x - mu) / sqrt(var + eps) + beta over the last axis (population variance)."""
    x = _f64(x)
    d = x.shape[-1]
    gamma, beta = _f64(gamma), _f64(beta)
    assert gamma.shape == (d,) and beta.shape == (d,)
    out = np.empty_like(x)
    _load().oracle_layernorm(_dp(x), _dp(gamma), _dp(beta), _dp(out), int(x.size // d), d,
                             float(eps))
    return out


def ffn(x, w_1, b_1, w_2, b_2, nthreads: int = 0):
    """FFN(x) = max(0, x W_1 + b_1) W_2 + b_2 over the last axis of x."""
    x = _f64(x)
    d_model = x.shape[-1]
    w_1, b_1, w_2, b_2 = _f64(w_1), _f64(b_1), _f64(w_2), _f64(b_2)
    d_ff = w_1.shape[1]
    assert w_1.shape == (d_model, d_ff) and b_1.shape == (d_ff,)
    assert w_2.shape == (d_ff, d_model) and b_2.shape == (d_model,)
    out = np.empty_like(x)
    rc = _load().oracle_ffn(_dp(x), _dp(w_1), _dp(b_1), _dp(w_2), _dp(b_2), _dp(out),
                            int(x.size // d_model), d_model, d_ff, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_ffn rejected its arguments")
    return out


def encoder_layer(x, w_q, w_k, w_v, w_o, g_1, be_1, w_1, b_1, w_2, b_2, g_2, be_2, h: int,
                  mask_kind: int = MASK_NONE, kv_lens=None, scale: float | None = None,
                  eps: float = 1e-6, return_mid: bool = False, nthreads: int = 0):
    """LayerNorm_2(y + FFN(y)) with y = LayerNorm_1(x + MultiHead(x, x)); x [B, n, d_model]."""
    x = _f64(x)
    B, n, d_model = x.shape
    args = [_f64(a) for a in (w_q, w_k, w_v, w_o, g_1, be_1, w_1, b_1, w_2, b_2, g_2, be_2)]
    d_k = args[0].shape[1] // h
    d_ff = args[6].shape[1]
    if scale is None or scale == 0.0:
        scale = default_scale(d_k)
    lens = None
    if mask_kind & MASK_KEY_PADDING:
        lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))
    out = np.zeros_like(x)
    mid = np.zeros_like(x) if return_mid else None
    rc = _load().oracle_encoder_layer(_dp(x), *[_dp(a) for a in args], _dp(out), _dp(mid), B, n,
                                      d_model, h, d_k, d_ff, int(mask_kind), _ip(lens),
                                      float(scale), float(eps), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_encoder_layer rejected its arguments")
    return (out, mid) if return_mid else out
