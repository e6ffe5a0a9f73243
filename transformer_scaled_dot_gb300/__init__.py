"""GB300 (sm_103a) multi-head scaled dot-product attention.

A thin Python binding over the C ABI of libtsd_attention.so
(include/tsd_attention.h). Each function has the name and the parameters of
its C entry point and only marshals arguments: tensor arguments may be
torch tensors (their data_ptr() is passed) or raw device addresses (int);
`stream` may be a torch.cuda.Stream, a raw cudaStream_t (int), or None for
torch's current stream. A non-OK status raises AttnError.

There is no fallback: if the native library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_CUDA",
    "ATTN_ERR_DEVICE_TIMEOUT", "ATTN_MASK_NONE", "ATTN_MASK_CAUSAL", "ATTN_MASK_KEY_PADDING",
    "AttnError", "library", "library_path", "EXPORTED_SYMBOLS",
    "attn_forward", "attn_forward_strided", "attn_forward_f32", "mha_workspace_bytes",
    "mha_forward", "attn_get_device_status", "attn_last_cuda_error", "attn_status_string",
    "attn_selftest_wait_timeout", "mha_project_qkv", "mha_project_out", "mha_forward_noalloc",
    "mha_concat_heads", "mha_forward_launches", "attn_forward_window", "attn_decode",
    "attn_decode_workspace_bytes", "encoder_layer_forward", "encoder_layer_workspace_bytes",
    "MHA_NOALLOC_SCRATCH_BYTES", "attn_host_workspace_bytes", "attn_forward_host",
    "mha_host_workspace_bytes", "mha_forward_host", "encoder_layer_host_workspace_bytes",
    "encoder_layer_forward_host", "attn_decode_host_workspace_bytes", "attn_decode_host",
    "attn_forward_window_host", "mha_forward_host_async", "attn_host_join",
    "attn_decode_host_async", "encoder_layer_forward_host_async",
]

ATTN_OK, ATTN_ERR_INVALID, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT = range(5)
ATTN_MASK_NONE, ATTN_MASK_CAUSAL, ATTN_MASK_KEY_PADDING = 0, 1, 2

EXPORTED_SYMBOLS = (
    "attn_forward", "attn_forward_strided", "attn_forward_f32", "mha_workspace_bytes",
    "mha_forward", "attn_get_device_status", "attn_last_cuda_error", "attn_status_string",
    "attn_selftest_wait_timeout", "mha_project_qkv", "mha_project_out", "mha_forward_noalloc",
    "mha_concat_heads", "mha_forward_launches", "attn_forward_window", "attn_decode",
    "attn_decode_workspace_bytes", "encoder_layer_forward", "encoder_layer_workspace_bytes",
    "attn_host_workspace_bytes", "attn_forward_host", "mha_host_workspace_bytes",
    "mha_forward_host", "encoder_layer_host_workspace_bytes", "encoder_layer_forward_host",
    "attn_decode_host_workspace_bytes", "attn_decode_host", "attn_forward_window_host",
    "mha_forward_host_async", "attn_host_join", "attn_decode_host_async",
    "encoder_layer_forward_host_async",
)

# TSD_MHA_NOALLOC_SCRATCH_BYTES of the header: the fixed scratch of mha_forward_noalloc
MHA_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = library().attn_status_string(status).decode()
        extra = ""
        if status == ATTN_ERR_CUDA:
            extra = f" (cudaError {library().attn_last_cuda_error()})"
        super().__init__(f"{where}: {name}{extra}")


def library_path() -> str:
    return _build.LIB_PATH


def library():
    """Loads libtsd_attention.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i, i64, f, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    lib.attn_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, f, st]
    lib.attn_forward_strided.argtypes = [vp, i64, i64, i64, vp, i64, i64, i64, vp, i64, i64, i64,
                                         vp, i64, i64, i64, i, i, i, i, i, i, i, vp, f, st]
    lib.attn_forward_f32.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, f, st]
    lib.mha_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.mha_workspace_bytes.restype = ctypes.c_size_t
    lib.mha_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, f, vp,
                                ctypes.c_size_t, st]
    lib.mha_project_qkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, st]
    lib.mha_concat_heads.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, f, vp,
                                     ctypes.c_size_t, st]
    lib.mha_project_out.argtypes = [vp, vp, vp, i, i, i, i, i, st]
    lib.mha_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, f,
                                        st]
    lib.attn_get_device_status.argtypes = [st]
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_selftest_wait_timeout.argtypes = [i, st]
    lib.mha_forward_launches.argtypes = [i, i, i, i, i, i, i, i]
    lib.attn_forward_window.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, i, i, f, st]
    lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_decode.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, f, vp, ctypes.c_size_t, st]
    lib.encoder_layer_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.encoder_layer_workspace_bytes.restype = ctypes.c_size_t
    lib.encoder_layer_forward.argtypes = [vp] * 14 + [i] * 7 + [vp, f, f, vp, ctypes.c_size_t, st]
    sz = ctypes.c_size_t
    for name, n in (("attn_host_workspace_bytes", 6), ("mha_host_workspace_bytes", 7),
                    ("encoder_layer_host_workspace_bytes", 6),
                    ("attn_decode_host_workspace_bytes", 6)):
        getattr(lib, name).argtypes = [i] * n
        getattr(lib, name).restype = sz
    lib.attn_forward_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, f, vp, sz, st]
    lib.attn_forward_window_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, i, i, f, vp,
                                             sz, st]
    lib.mha_forward_host.argtypes = [vp] * 7 + [i] * 8 + [vp, f, vp, sz, st]
    lib.mha_forward_host_async.argtypes = [vp] * 7 + [i] * 8 + [vp, f, vp, sz, st]
    lib.attn_host_join.argtypes = [st]
    lib.encoder_layer_forward_host.argtypes = [vp] * 14 + [i] * 7 + [vp, f, f, vp, sz, st]
    lib.encoder_layer_forward_host_async.argtypes = lib.encoder_layer_forward_host.argtypes
    lib.attn_decode_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, f, vp, sz, st]
    lib.attn_decode_host_async.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, f, vp, sz, st]
    for name in ("attn_forward", "attn_forward_strided", "attn_forward_f32", "mha_forward",
                 "attn_get_device_status", "attn_last_cuda_error", "attn_selftest_wait_timeout",
                 "mha_project_qkv", "mha_project_out", "mha_forward_noalloc", "mha_concat_heads",
                 "mha_forward_launches", "attn_forward_window", "attn_decode",
                 "encoder_layer_forward", "attn_forward_host", "mha_forward_host",
                 "encoder_layer_forward_host", "attn_decode_host", "attn_forward_window_host",
                 "mha_forward_host_async", "attn_host_join", "attn_decode_host_async",
                 "encoder_layer_forward_host_async"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(x):
    """Address of a torch tensor (device or host), a numpy array (host), or an int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)


def attn_forward(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask_kind=ATTN_MASK_NONE, kv_lens=None,
                 scale=0.0, stream=None):
    _check(library().attn_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, h, n_q, n_k, d_k, d_v,
                                  mask_kind, _ptr(kv_lens), scale, _stream(stream)), "attn_forward")


def attn_forward_window(q, k, v, out, B, h, n_q, n_k, d_k, d_v, window_left, window_right,
                        mask_kind=ATTN_MASK_NONE, kv_lens=None, scale=0.0, stream=None):
    """Restricted self-attention: query i sees keys [i - window_left, i + window_right]
    (-1 = no bound on that side)."""
    _check(library().attn_forward_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, h, n_q, n_k,
                                         d_k, d_v, mask_kind, _ptr(kv_lens), window_left,
                                         window_right, scale, _stream(stream)),
           "attn_forward_window")


def attn_decode_workspace_bytes(B, h, n_q, n_max, d_v) -> int:
    return int(library().attn_decode_workspace_bytes(B, h, n_q, n_max, d_v))


def attn_decode(q, k_cache, v_cache, out, B, h, n_q, n_max, d_k, d_v, cache_lens=None, scale=0.0,
                workspace=None, workspace_bytes=0, stream=None):
    """One decoding step: the n_q newest tokens' queries against an n_max-row
    key/value cache (cache_lens[b] valid rows, None = n_max)."""
    _check(library().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), B, h, n_q,
                                 n_max, d_k, d_v, _ptr(cache_lens), scale, _ptr(workspace),
                                 workspace_bytes, _stream(stream)), "attn_decode")


def encoder_layer_workspace_bytes(B, n, d_model, h, d_k, d_ff) -> int:
    return int(library().encoder_layer_workspace_bytes(B, n, d_model, h, d_k, d_ff))


def encoder_layer_forward(x, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                          ln2_gamma, ln2_beta, out, B, n, d_model, h, d_k, d_ff,
                          mask_kind=ATTN_MASK_NONE, kv_lens=None, scale=0.0, eps=1e-6,
                          workspace=None, workspace_bytes=0, stream=None):
    """LayerNorm_2(y + FFN(y)), y = LayerNorm_1(x + MultiHead(x, x)) (post-LN encoder layer)."""
    ptrs = [_ptr(t) for t in (x, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                              ln2_gamma, ln2_beta, out)]
    _check(library().encoder_layer_forward(*ptrs, B, n, d_model, h, d_k, d_ff, mask_kind,
                                           _ptr(kv_lens), scale, eps, _ptr(workspace),
                                           workspace_bytes, _stream(stream)),
           "encoder_layer_forward")


def attn_forward_strided(q, q_sb, q_sh, q_sr, k, k_sb, k_sh, k_sr, v, v_sb, v_sh, v_sr,
                         out, o_sb, o_sh, o_sr, B, h, n_q, n_k, d_k, d_v,
                         mask_kind=ATTN_MASK_NONE, kv_lens=None, scale=0.0, stream=None):
    _check(library().attn_forward_strided(
        _ptr(q), q_sb, q_sh, q_sr, _ptr(k), k_sb, k_sh, k_sr, _ptr(v), v_sb, v_sh, v_sr,
        _ptr(out), o_sb, o_sh, o_sr, B, h, n_q, n_k, d_k, d_v, mask_kind, _ptr(kv_lens), scale,
        _stream(stream)), "attn_forward_strided")


def attn_forward_f32(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask_kind=ATTN_MASK_NONE,
                     kv_lens=None, scale=0.0, stream=None):
    _check(library().attn_forward_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, h, n_q, n_k, d_k,
                                      d_v, mask_kind, _ptr(kv_lens), scale, _stream(stream)),
           "attn_forward_f32")


def mha_workspace_bytes(B, n_q, n_k, h, d_k, d_v) -> int:
    return int(library().mha_workspace_bytes(B, n_q, n_k, h, d_k, d_v))


def mha_forward(x_q, x_kv, w_q, w_k, w_v, w_o, out, B, n_q, n_k, d_model, h, d_k, d_v,
                mask_kind=ATTN_MASK_NONE, kv_lens=None, scale=0.0, workspace=None,
                workspace_bytes=0, stream=None):
    _check(library().mha_forward(_ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(w_k), _ptr(w_v),
                                 _ptr(w_o), _ptr(out), B, n_q, n_k, d_model, h, d_k, d_v,
                                 mask_kind, _ptr(kv_lens), scale, _ptr(workspace),
                                 workspace_bytes, _stream(stream)), "mha_forward")


def mha_forward_launches(B, n_q, n_k, d_model, h, d_k, d_v, self_attention) -> int:
    """Kernels mha_forward launches for these sizes (1, 2 or 3; 0 for no
    work; -1 for sizes it rejects)."""
    return int(library().mha_forward_launches(B, n_q, n_k, d_model, h, d_k, d_v,
                                              1 if self_attention else 0))


def mha_concat_heads(x_q, x_kv, w_q, w_k, w_v, concat, B, n_q, n_k, d_model, h, d_k, d_v,
                     mask_kind=ATTN_MASK_NONE, kv_lens=None, scale=0.0, workspace=None,
                     workspace_bytes=0, stream=None):
    _check(library().mha_concat_heads(_ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(w_k), _ptr(w_v),
                                      _ptr(concat), B, n_q, n_k, d_model, h, d_k, d_v, mask_kind,
                                      _ptr(kv_lens), scale, _ptr(workspace), workspace_bytes,
                                      _stream(stream)), "mha_concat_heads")


def mha_project_qkv(x_q, x_kv, w_q, w_k, w_v, q_out, k_out, v_out, B, n_q, n_k, d_model, h, d_k,
                    d_v, stream=None):
    _check(library().mha_project_qkv(_ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(w_k), _ptr(w_v),
                                     _ptr(q_out), _ptr(k_out), _ptr(v_out), B, n_q, n_k, d_model,
                                     h, d_k, d_v, _stream(stream)), "mha_project_qkv")


def mha_project_out(concat, w_o, out, B, n_q, d_model, h, d_v, stream=None):
    _check(library().mha_project_out(_ptr(concat), _ptr(w_o), _ptr(out), B, n_q, d_model, h, d_v,
                                     _stream(stream)), "mha_project_out")


def mha_forward_noalloc(x_q, x_kv, w_q, w_k, w_v, w_o, out, B, n_q, n_k, d_model, h, d_k, d_v,
                        mask_kind=ATTN_MASK_NONE, kv_lens=None, scale=0.0, stream=None):
    """mha_forward on the library's fixed device scratch (no workspace argument;
    for callers that cannot allocate device memory)."""
    _check(library().mha_forward_noalloc(_ptr(x_q), _ptr(x_kv), _ptr(w_q), _ptr(w_k), _ptr(w_v),
                                         _ptr(w_o), _ptr(out), B, n_q, n_k, d_model, h, d_k, d_v,
                                         mask_kind, _ptr(kv_lens), scale, _stream(stream)),
           "mha_forward_noalloc")


def attn_get_device_status(stream=None) -> int:
    """Returns the status code (does not raise on ATTN_ERR_DEVICE_TIMEOUT)."""
    return int(library().attn_get_device_status(_stream(stream)))


def attn_last_cuda_error() -> int:
    return int(library().attn_last_cuda_error())


def attn_status_string(status: int) -> str:
    return library().attn_status_string(status).decode()


def attn_selftest_wait_timeout(limit_us: int, stream=None):
    _check(library().attn_selftest_wait_timeout(limit_us, _stream(stream)),
           "attn_selftest_wait_timeout")


# ---------------------------------------------------------------- host buffers
# The *_host entry points take the step's inputs and result in host memory
# (pinned for asynchronous copies) and stage them through the workspace.

def attn_host_workspace_bytes(B, h, n_q, n_k, d_k, d_v) -> int:
    return int(library().attn_host_workspace_bytes(B, h, n_q, n_k, d_k, d_v))


def attn_forward_host(q_host, k_host, v_host, out_host, B, h, n_q, n_k, d_k, d_v,
                      mask_kind=ATTN_MASK_NONE, kv_lens_host=None, scale=0.0, workspace=None,
                      workspace_bytes=0, stream=None):
    _check(library().attn_forward_host(_ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host),
                                       B, h, n_q, n_k, d_k, d_v, mask_kind, _ptr(kv_lens_host),
                                       scale, _ptr(workspace), workspace_bytes, _stream(stream)),
           "attn_forward_host")


def attn_forward_window_host(q_host, k_host, v_host, out_host, B, h, n_q, n_k, d_k, d_v,
                             window_left, window_right, mask_kind=ATTN_MASK_NONE,
                             kv_lens_host=None, scale=0.0, workspace=None, workspace_bytes=0,
                             stream=None):
    _check(library().attn_forward_window_host(_ptr(q_host), _ptr(k_host), _ptr(v_host),
                                              _ptr(out_host), B, h, n_q, n_k, d_k, d_v, mask_kind,
                                              _ptr(kv_lens_host), window_left, window_right,
                                              scale, _ptr(workspace), workspace_bytes,
                                              _stream(stream)),
           "attn_forward_window_host")


def mha_host_workspace_bytes(B, n_q, n_k, d_model, h, d_k, d_v) -> int:
    return int(library().mha_host_workspace_bytes(B, n_q, n_k, d_model, h, d_k, d_v))


def mha_forward_host(x_q_host, x_kv_host, w_q, w_k, w_v, w_o, out_host, B, n_q, n_k, d_model, h,
                     d_k, d_v, mask_kind=ATTN_MASK_NONE, kv_lens_host=None, scale=0.0,
                     workspace=None, workspace_bytes=0, stream=None):
    _check(library().mha_forward_host(_ptr(x_q_host), _ptr(x_kv_host), _ptr(w_q), _ptr(w_k),
                                      _ptr(w_v), _ptr(w_o), _ptr(out_host), B, n_q, n_k, d_model,
                                      h, d_k, d_v, mask_kind, _ptr(kv_lens_host), scale,
                                      _ptr(workspace), workspace_bytes, _stream(stream)),
           "mha_forward_host")


def mha_forward_host_async(x_q_host, x_kv_host, w_q, w_k, w_v, w_o, out_host, B, n_q, n_k,
                           d_model, h, d_k, d_v, mask_kind=ATTN_MASK_NONE, kv_lens_host=None,
                           scale=0.0, workspace=None, workspace_bytes=0, stream=None):
    """mha_forward_host with the result copy on the library's result stream:
    out_host is complete once `stream` has passed a later attn_host_join."""
    _check(library().mha_forward_host_async(_ptr(x_q_host), _ptr(x_kv_host), _ptr(w_q),
                                            _ptr(w_k), _ptr(w_v), _ptr(w_o), _ptr(out_host), B,
                                            n_q, n_k, d_model, h, d_k, d_v, mask_kind,
                                            _ptr(kv_lens_host), scale, _ptr(workspace),
                                            workspace_bytes, _stream(stream)),
           "mha_forward_host_async")


def attn_host_join(stream=None):
    _check(library().attn_host_join(_stream(stream)), "attn_host_join")


def encoder_layer_host_workspace_bytes(B, n, d_model, h, d_k, d_ff) -> int:
    return int(library().encoder_layer_host_workspace_bytes(B, n, d_model, h, d_k, d_ff))


def encoder_layer_forward_host(x_host, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2,
                               b_2, ln2_gamma, ln2_beta, out_host, B, n, d_model, h, d_k, d_ff,
                               mask_kind=ATTN_MASK_NONE, kv_lens_host=None, scale=0.0, eps=1e-6,
                               workspace=None, workspace_bytes=0, stream=None):
    ptrs = [_ptr(t) for t in (x_host, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                              ln2_gamma, ln2_beta, out_host)]
    _check(library().encoder_layer_forward_host(*ptrs, B, n, d_model, h, d_k, d_ff, mask_kind,
                                                _ptr(kv_lens_host), scale, eps, _ptr(workspace),
                                                workspace_bytes, _stream(stream)),
           "encoder_layer_forward_host")


def encoder_layer_forward_host_async(x_host, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1,
                                     w_2, b_2, ln2_gamma, ln2_beta, out_host, B, n, d_model, h,
                                     d_k, d_ff, mask_kind=ATTN_MASK_NONE, kv_lens_host=None,
                                     scale=0.0, eps=1e-6, workspace=None, workspace_bytes=0,
                                     stream=None):
    """encoder_layer_forward_host with the result copy on the library's result
    stream: out_host is complete once `stream` has passed a later attn_host_join."""
    ptrs = [_ptr(t) for t in (x_host, w_q, w_k, w_v, w_o, ln1_gamma, ln1_beta, w_1, b_1, w_2, b_2,
                              ln2_gamma, ln2_beta, out_host)]
    _check(library().encoder_layer_forward_host_async(*ptrs, B, n, d_model, h, d_k, d_ff,
                                                      mask_kind, _ptr(kv_lens_host), scale, eps,
                                                      _ptr(workspace), workspace_bytes,
                                                      _stream(stream)),
           "encoder_layer_forward_host_async")


def attn_decode_host_workspace_bytes(B, h, n_q, n_max, d_k, d_v) -> int:
    return int(library().attn_decode_host_workspace_bytes(B, h, n_q, n_max, d_k, d_v))


def attn_decode_host(q_host, k_cache, v_cache, out_host, B, h, n_q, n_max, d_k, d_v,
                     cache_lens_host=None, scale=0.0, workspace=None, workspace_bytes=0,
                     stream=None):
    _check(library().attn_decode_host(_ptr(q_host), _ptr(k_cache), _ptr(v_cache), _ptr(out_host),
                                      B, h, n_q, n_max, d_k, d_v, _ptr(cache_lens_host), scale,
                                      _ptr(workspace), workspace_bytes, _stream(stream)),
           "attn_decode_host")


def attn_decode_host_async(q_host, k_cache, v_cache, out_host, B, h, n_q, n_max, d_k, d_v,
                           cache_lens_host=None, scale=0.0, workspace=None, workspace_bytes=0,
                           stream=None):
    """attn_decode_host with the result copy on the library's result stream:
    out_host is complete once `stream` has passed a later attn_host_join."""
    _check(library().attn_decode_host_async(_ptr(q_host), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(out_host), B, h, n_q, n_max, d_k, d_v,
                                            _ptr(cache_lens_host), scale, _ptr(workspace),
                                            workspace_bytes, _stream(stream)),
           "attn_decode_host_async")
