"""The C-ABI library loads, exports every symbol the header declares, and
rejects invalid arguments on the host before any launch (CPU only)."""
import ctypes
import os
import re

import pytest

import transformer_scaled_dot_gb300 as tsd
from transformer_scaled_dot_gb300 import build as native_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    native_build.build()
    return tsd.library()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert set(tsd.EXPORTED_SYMBOLS) <= set(declared)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert tsd.attn_status_string(tsd.ATTN_OK) == "ATTN_OK"
    assert tsd.attn_status_string(tsd.ATTN_ERR_DEVICE_TIMEOUT) == "ATTN_ERR_DEVICE_TIMEOUT"


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every call below fails validation


@pytest.mark.parametrize("args,expect", [
    # (B, h, n_q, n_k, d_k, d_v, mask, kv_lens, scale)
    ((1, 1, 16, 16, 96, 96, 0, None, 0.0), tsd.ATTN_ERR_UNSUPPORTED),
    ((1, 1, 16, 16, 48, 48, 0, None, 0.0), tsd.ATTN_ERR_UNSUPPORTED),  # not a Table 3 (A) size
    ((1, 1, 16, 16, 8, 8, 0, None, 0.0), tsd.ATTN_ERR_UNSUPPORTED),
    ((1, 1, 16, 16, 512, 512, 0, None, 0.0), tsd.ATTN_ERR_UNSUPPORTED),
    ((1, 1, 16, 16, 64, 128, 0, None, 0.0), tsd.ATTN_ERR_UNSUPPORTED),
    ((-1, 1, 16, 16, 64, 64, 0, None, 0.0), tsd.ATTN_ERR_INVALID),
    ((1, 1, 16, 8, 64, 64, 1, None, 0.0), tsd.ATTN_ERR_INVALID),      # causal, n_q != n_k
    ((1, 1, 16, 16, 64, 64, 2, None, 0.0), tsd.ATTN_ERR_INVALID),     # padding without lengths
    ((1, 1, 16, 16, 64, 64, 4, None, 0.0), tsd.ATTN_ERR_INVALID),     # unknown mask bit
    ((1, 1, 16, 16, 64, 64, 0, None, -1.0), tsd.ATTN_ERR_INVALID),    # negative scale
    ((1, 1, 16, 16, 64, 64, 0, None, float("nan")), tsd.ATTN_ERR_INVALID),
    ((1, 70000, 16, 16, 64, 64, 0, None, 0.0), tsd.ATTN_ERR_INVALID),  # grid limit
])
def test_attn_forward_rejects_bad_arguments(lib, args, expect):
    B, h, n_q, n_k, d_k, d_v, mask, lens, scale = args
    st = lib.attn_forward(FAKE, FAKE, FAKE, FAKE, B, h, n_q, n_k, d_k, d_v, mask, lens, scale, None)
    assert st == expect


def test_attn_forward_rejects_null_and_misaligned(lib):
    assert lib.attn_forward(None, FAKE, FAKE, FAKE, 1, 1, 16, 16, 64, 64, 0, None, 0.0, None) == \
        tsd.ATTN_ERR_INVALID
    assert lib.attn_forward(FAKE + 2, FAKE, FAKE, FAKE, 1, 1, 16, 16, 64, 64, 0, None, 0.0, None) == \
        tsd.ATTN_ERR_INVALID
    assert lib.attn_forward(FAKE, FAKE, FAKE, FAKE, 1, 1, 16, 16, 64, 64, 2, FAKE + 2, 0.0, None) == \
        tsd.ATTN_ERR_INVALID


def test_empty_problems_are_no_ops(lib):
    for B, h, n_q in ((0, 1, 16), (1, 0, 16), (1, 1, 0)):
        assert lib.attn_forward(FAKE, FAKE, FAKE, FAKE, B, h, n_q, 16, 64, 64, 0, None, 0.0,
                                None) == tsd.ATTN_OK


def test_attn_forward_strided_rejects_bad_strides(lib):
    good = (1 << 20, 8192, 64)
    args = [FAKE, *good, FAKE, *good, FAKE, *good, FAKE, *good, 1, 1, 16, 16, 64, 64, 0, None, 0.0, None]
    bad = list(args)
    bad[3] = 60  # row stride not a multiple of 8 elements
    assert lib.attn_forward_strided(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(args)
    bad[15] = 32  # output row stride smaller than d_v
    assert lib.attn_forward_strided(*bad) == tsd.ATTN_ERR_INVALID


def test_attn_forward_f32_limits(lib):
    assert lib.attn_forward_f32(FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 4, 129, 64, 0, None, 0.0, None) == \
        tsd.ATTN_ERR_UNSUPPORTED
    assert lib.attn_forward_f32(FAKE + 1, FAKE, FAKE, FAKE, 1, 1, 4, 4, 64, 64, 0, None, 0.0, None) == \
        tsd.ATTN_ERR_INVALID


def test_mha_workspace_bytes_layout(lib):
    B, n_q, n_k, h, d = 32, 128, 160, 8, 64
    got = tsd.mha_workspace_bytes(B, n_q, n_k, h, d, d)
    align = lambda x: (x + 255) // 256 * 256
    expect = align(B * n_q * h * d * 2) * 2 + align(B * n_k * h * d * 2) * 2
    assert got == expect
    assert tsd.mha_workspace_bytes(-1, 1, 1, 1, 64, 64) == 0


def test_mha_forward_rejects_bad_arguments(lib):
    B, n, dm, h, d = 2, 16, 128, 2, 64
    wsb = tsd.mha_workspace_bytes(B, n, n, h, d, d)
    base = [FAKE] * 7 + [B, n, n, dm, h, d, d, 0, None, 0.0, FAKE, wsb, None]
    bad = list(base)
    bad[18] = wsb - 1                      # short workspace
    assert lib.mha_forward(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(base)
    bad[17] = FAKE + 16                    # workspace not 256-byte aligned
    assert lib.mha_forward(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(base)
    bad[10] = 100                          # d_model not a multiple of 8
    assert lib.mha_forward(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(base)
    bad[12] = bad[13] = 48                 # head size without a bf16 kernel
    assert lib.mha_forward(*bad) == tsd.ATTN_ERR_UNSUPPORTED


def test_mha_concat_heads_rejects_bad_arguments(lib):
    B, n, dm, h, d = 2, 16, 128, 2, 64
    wsb = tsd.mha_workspace_bytes(B, n, n, h, d, d)
    # x_q, x_kv, w_q, w_k, w_v, concat, B, n_q, n_k, d_model, h, d_k, d_v, mask, lens, scale,
    # workspace, bytes, stream
    base = [FAKE] * 6 + [B, n, n, dm, h, d, d, 0, None, 0.0, FAKE, wsb, None]
    bad = list(base)
    bad[17] = wsb - 1                      # short workspace
    assert lib.mha_concat_heads(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(base)
    bad[5] = None                          # no output
    assert lib.mha_concat_heads(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(base)
    bad[13] = tsd.ATTN_MASK_KEY_PADDING    # padding without lengths
    assert lib.mha_concat_heads(*bad) == tsd.ATTN_ERR_INVALID
    bad = list(base)
    bad[11] = bad[12] = 48                 # head size without a bf16 kernel
    assert lib.mha_concat_heads(*bad) == tsd.ATTN_ERR_UNSUPPORTED
    base[6] = 0                            # empty batch: nothing to do
    assert lib.mha_concat_heads(*base) == tsd.ATTN_OK


def test_selftest_rejects_bad_limit(lib):
    assert lib.attn_selftest_wait_timeout(0, None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_selftest_wait_timeout(3000000, None) == tsd.ATTN_ERR_INVALID


@pytest.mark.parametrize("args,expect", [
    # (n_q, n_k, window_left, window_right, mask)
    ((16, 16, -2, 3, 0), tsd.ATTN_ERR_INVALID),   # a bound below -1
    ((16, 16, 3, -5, 0), tsd.ATTN_ERR_INVALID),
    ((16, 20, 2, 2, 0), tsd.ATTN_ERR_INVALID),    # a window needs n_q == n_k
    ((16, 20, 0, -1, 0), tsd.ATTN_ERR_INVALID),
    ((16, 16, 2, 2, 4), tsd.ATTN_ERR_INVALID),    # unknown mask bit
    ((16, 16, 2, 2, 2), tsd.ATTN_ERR_INVALID),    # padding without lengths
])
def test_attn_forward_window_rejects_bad_arguments(lib, args, expect):
    n_q, n_k, wl, wr, mask = args
    st = lib.attn_forward_window(FAKE, FAKE, FAKE, FAKE, 1, 1, n_q, n_k, 64, 64, mask, None, wl, wr,
                                 0.0, None)
    assert st == expect


def test_attn_forward_window_empty_problem_is_a_no_op(lib):
    assert lib.attn_forward_window(FAKE, FAKE, FAKE, FAKE, 0, 1, 16, 16, 64, 64, 0, None, 3, 3,
                                   0.0, None) == tsd.ATTN_OK


def test_attn_decode_rejects_bad_arguments(lib):
    ws = tsd.attn_decode_workspace_bytes(1, 1, 1, 100, 64)
    assert ws > 0
    call = lambda *a: lib.attn_decode(*a)
    base = [FAKE, FAKE, FAKE, FAKE, 1, 1, 1, 100, 64, 64, None, 0.0, FAKE, ws, None]

    def with_(i, v):
        args = list(base)
        args[i] = v
        return call(*args)
    assert with_(6, 0) == tsd.ATTN_ERR_INVALID          # n_q = 0
    assert with_(6, 9) == tsd.ATTN_ERR_UNSUPPORTED      # n_q > 8
    assert with_(7, 0) == tsd.ATTN_ERR_INVALID          # empty cache shape
    assert with_(8, 96) == tsd.ATTN_ERR_UNSUPPORTED     # head size
    assert with_(0, None) == tsd.ATTN_ERR_INVALID       # null q
    assert with_(1, FAKE + 4) == tsd.ATTN_ERR_INVALID   # misaligned cache
    assert with_(10, FAKE + 2) == tsd.ATTN_ERR_INVALID  # misaligned lengths
    assert with_(13, ws - 1) == tsd.ATTN_ERR_INVALID    # short workspace
    assert with_(11, -1.0) == tsd.ATTN_ERR_INVALID      # negative scale


def test_attn_decode_workspace_grows_with_chunks_queries_and_width(lib):
    f = tsd.attn_decode_workspace_bytes
    assert f(1, 1, 1, 128, 64) < f(1, 1, 1, 129, 64)   # a second 128-key chunk
    assert f(2, 3, 4, 1000, 128) >= 2 * 3 * 4 * 4 * (128 + 2) * 4
    assert f(1, 1, 0, 100, 64) == 0 and f(1, 1, 9, 100, 64) == 0


def test_encoder_layer_rejects_bad_arguments(lib):
    B, n, dm, h, d, ff = 2, 16, 512, 8, 64, 2048
    wsb = tsd.encoder_layer_workspace_bytes(B, n, dm, h, d, ff)
    assert wsb > tsd.mha_workspace_bytes(B, n, n, h, d, d)
    # 14 tensors, B, n, d_model, h, d_k, d_ff, mask, lens, scale, eps, workspace, bytes, stream
    base = [FAKE] * 14 + [B, n, dm, h, d, ff, 0, None, 0.0, 1e-6, FAKE, wsb, None]

    def with_(i, v):
        args = list(base)
        args[i] = v
        return lib.encoder_layer_forward(*args)
    assert with_(16, 384) == tsd.ATTN_ERR_UNSUPPORTED   # d_model without a LayerNorm kernel
    assert with_(19, 2044) == tsd.ATTN_ERR_INVALID      # d_ff not a multiple of 8
    assert with_(23, 0.0) == tsd.ATTN_ERR_INVALID       # eps
    assert with_(23, -1.0) == tsd.ATTN_ERR_INVALID
    assert with_(25, wsb - 1) == tsd.ATTN_ERR_INVALID   # short workspace
    assert with_(24, FAKE + 16) == tsd.ATTN_ERR_INVALID  # workspace not 256-byte aligned
    assert with_(7, None) == tsd.ATTN_ERR_INVALID       # no W_1
    assert with_(18, 96) == tsd.ATTN_ERR_UNSUPPORTED    # head size


def test_attn_decode_caps_the_cache_length(lib):
    ws = tsd.attn_decode_workspace_bytes(1, 1, 1, 131072, 64)
    st = lib.attn_decode(FAKE, FAKE, FAKE, FAKE, 1, 1, 1, 131073, 64, 64, None, 0.0, FAKE,
                         ws * 2, None)
    assert st == tsd.ATTN_ERR_UNSUPPORTED


# ------------------------------------------------------------ host-buffer entry points
def test_host_workspace_sizes_cover_staging_and_device_workspace(lib):
    al = lambda x: (x + 255) // 256 * 256
    B, n, dm, h, d = 32, 128, 512, 8, 64
    xb = B * n * dm * 2
    assert tsd.mha_host_workspace_bytes(B, n, n, dm, h, d, d) == \
        3 * al(xb) + al(B * 4) + tsd.mha_workspace_bytes(B, n, n, h, d, d)
    qb = 2 * 4 * 100 * 64 * 2
    assert tsd.attn_host_workspace_bytes(2, 4, 100, 100, 64, 64) == 4 * al(qb) + al(2 * 4)
    assert tsd.encoder_layer_host_workspace_bytes(B, n, dm, h, d, 2048) == \
        2 * al(xb) + al(B * 4) + tsd.encoder_layer_workspace_bytes(B, n, dm, h, d, 2048)
    assert tsd.attn_decode_host_workspace_bytes(16, 16, 1, 8192, 64, 64) == \
        2 * al(16 * 16 * 64 * 2) + al(16 * 4) + tsd.attn_decode_workspace_bytes(16, 16, 1, 8192, 64)
    for bad in (tsd.mha_host_workspace_bytes(-1, n, n, dm, h, d, d),
                tsd.attn_host_workspace_bytes(1, 1, 16, 16, 0, 64),
                tsd.encoder_layer_host_workspace_bytes(1, 16, 0, 8, 64, 2048),
                tsd.attn_decode_host_workspace_bytes(1, 1, 0, 128, 64, 64)):
        assert bad == 0


def test_host_entry_points_reject_bad_arguments_before_copying(lib):
    # every case fails validation, so nothing reaches the CUDA runtime
    # (none is present here; a call that got that far would say ATTN_ERR_CUDA)
    ws = 1 << 24  # 256-byte aligned fake device address, never touched
    big = 1 << 40
    hx = FAKE
    M = tsd.ATTN_MASK_KEY_PADDING
    # attn_forward_host: null host pointer, short / misaligned workspace,
    # padding without lengths, unsupported head size
    assert lib.attn_forward_host(None, hx, hx, hx, 1, 1, 16, 16, 64, 64, 0, None, 0.0, ws, big,
                                 None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_forward_host(hx, hx, hx, hx, 1, 1, 16, 16, 64, 64, 0, None, 0.0, ws, 1024,
                                 None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_forward_host(hx, hx, hx, hx, 1, 1, 16, 16, 64, 64, 0, None, 0.0, ws + 16, big,
                                 None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_forward_host(hx, hx, hx, hx, 1, 1, 16, 16, 64, 64, M, None, 0.0, ws, big,
                                 None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_forward_host(hx, hx, hx, hx, 1, 1, 16, 16, 96, 96, 0, None, 0.0, ws, big,
                                 None) == tsd.ATTN_ERR_UNSUPPORTED
    # attn_forward_window_host: a window needs n_q == n_k; bounds below -1
    assert lib.attn_forward_window_host(hx, hx, hx, hx, 1, 1, 16, 32, 64, 64, 0, None, 4, 4, 0.0,
                                        ws, big, None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_forward_window_host(hx, hx, hx, hx, 1, 1, 16, 16, 64, 64, 0, None, -2, 4, 0.0,
                                        ws, big, None) == tsd.ATTN_ERR_INVALID
    # mha_forward_host: null weight, short workspace, causal with n_q != n_k
    w = FAKE
    assert lib.mha_forward_host(hx, hx, None, w, w, w, hx, 2, 16, 16, 512, 8, 64, 64, 0, None, 0.0,
                                ws, big, None) == tsd.ATTN_ERR_INVALID
    need = tsd.mha_host_workspace_bytes(2, 16, 16, 512, 8, 64, 64)
    assert lib.mha_forward_host(hx, hx, w, w, w, w, hx, 2, 16, 16, 512, 8, 64, 64, 0, None, 0.0,
                                ws, need - 1, None) == tsd.ATTN_ERR_INVALID
    assert lib.mha_forward_host(hx, hx + 4096, w, w, w, w, hx, 2, 16, 8, 512, 8, 64, 64, 1, None,
                                0.0, ws, big, None) == tsd.ATTN_ERR_INVALID
    # encoder_layer_forward_host: bad eps, unsupported d_model
    args = [hx] + [w] * 12 + [hx]
    assert lib.encoder_layer_forward_host(*args, 2, 16, 512, 8, 64, 2048, 0, None, 0.0, 0.0, ws,
                                          big, None) == tsd.ATTN_ERR_INVALID
    assert lib.encoder_layer_forward_host(*args, 2, 16, 384, 8, 64, 2048, 0, None, 0.0, 1e-6, ws,
                                          big, None) == tsd.ATTN_ERR_UNSUPPORTED
    assert lib.encoder_layer_forward_host_async(*args, 2, 16, 512, 8, 64, 2048, 0, None, 0.0, 0.0,
                                                ws, big, None) == tsd.ATTN_ERR_INVALID
    assert lib.encoder_layer_forward_host_async(*args, 2, 16, 384, 8, 64, 2048, 0, None, 0.0,
                                                1e-6, ws, big, None) == tsd.ATTN_ERR_UNSUPPORTED
    # attn_decode_host: null cache, too many queries
    assert lib.attn_decode_host(hx, None, w, hx, 1, 1, 1, 128, 64, 64, None, 0.0, ws, big,
                                None) == tsd.ATTN_ERR_INVALID
    # the device entry point's codes: more than 8 queries, a cache past 131072 rows
    assert lib.attn_decode_host(hx, w, w, hx, 1, 1, 9, 128, 64, 64, None, 0.0, ws, big,
                                None) == tsd.ATTN_ERR_UNSUPPORTED
    assert lib.attn_decode_host(hx, w, w, hx, 1, 1, 1, 131072 + 256, 64, 64, None, 0.0, ws, big,
                                None) == tsd.ATTN_ERR_UNSUPPORTED
    # the asynchronous variant refuses the same arguments with the same codes
    assert lib.attn_decode_host_async(hx, None, w, hx, 1, 1, 1, 128, 64, 64, None, 0.0, ws, big,
                                      None) == tsd.ATTN_ERR_INVALID
    assert lib.attn_decode_host_async(hx, w, w, hx, 1, 1, 9, 128, 64, 64, None, 0.0, ws, big,
                                      None) == tsd.ATTN_ERR_UNSUPPORTED


def test_host_entry_points_empty_problems_are_no_ops(lib):
    ws = 1 << 24
    hx = FAKE
    assert lib.attn_forward_host(hx, hx, hx, hx, 0, 1, 16, 16, 64, 64, 0, None, 0.0, ws,
                                 1 << 30, None) == tsd.ATTN_OK
    assert lib.mha_forward_host(hx, hx, FAKE, FAKE, FAKE, FAKE, hx, 0, 16, 16, 512, 8, 64, 64, 0,
                                None, 0.0, ws, 1 << 30, None) == tsd.ATTN_OK
