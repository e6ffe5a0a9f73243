"""GPU tests of the host-buffer entry points (mha_forward_host,
attn_forward_host, encoder_layer_forward_host, attn_decode_host): the staged
call runs the same kernels as the device-pointer call, so its result is
bit-identical to it (and so within the oracle's tolerance); back-to-back
calls with no host synchronisation, alternating workspaces so that input
copies overlap earlier calls' work, each return their own input's result."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE

from gpu_util import assert_bf16_close, to_dev_bf16, to_dev_i32, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsd():
    import torch
    from transformer_scaled_dot_gb300 import build as native_build
    native_build.build()
    import transformer_scaled_dot_gb300 as m
    m.library()
    torch.cuda.set_device(0)
    return m


def pinned_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()


def pinned_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).pin_memory()


def pinned_out(shape):
    import torch
    return torch.full(shape, -1, dtype=torch.int16).pin_memory()


def bits_of_device(t):
    """A device bf16 tensor's bit patterns as a host int16 array."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy()


def device_mha(tsd, m, x_q_bits):
    import torch
    x_q = to_dev_bf16(x_q_bits)
    x_kv = x_q if m.self_attention else to_dev_bf16(m.x_kv)
    w = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o)]
    out = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.mha_workspace_bytes(m.B, m.n_q, m.n_k, m.h, m.d_k, m.d_v)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lens = to_dev_i32(m.kv_lens) if m.kv_lens is not None else None
    tsd.mha_forward(x_q, x_kv, *w, out, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                    m.mask_kind, lens, 0.0, ws, wsb)
    torch.cuda.synchronize()
    return bits_of_device(out)


def host_mha_setup(tsd, m, n_ws=1):
    import torch
    w = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o)]
    wsb = tsd.mha_host_workspace_bytes(m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v)
    assert wsb > 0
    wss = [torch.empty(wsb, dtype=torch.uint8, device="cuda") for _ in range(n_ws)]
    return w, wss, wsb


@pytest.mark.parametrize("case", ["base_encoder", "base_cross", "gemm_path"])
def test_mha_forward_host_matches_device_call(tsd, case):
    import torch
    if case == "base_encoder":
        m = synthetic.mha_inputs(1001, 32, 128, 128, 512, 8, 64, 64, MASK_KEY_PADDING, (64, 128),
                                 add_pe=True)
    elif case == "base_cross":
        m = synthetic.mha_inputs(1012, 32, 128, 160, 512, 8, 64, 64, MASK_KEY_PADDING, (80, 160),
                                 self_attention=False)
    else:  # n > 128: projection GEMM, attention kernel, W_O GEMM
        m = synthetic.mha_inputs(4242, 2, 300, 300, 256, 4, 64, 64, MASK_CAUSAL, None)
    w, (ws,), wsb = host_mha_setup(tsd, m)
    hx = pinned_bf16(m.x_q)
    hkv = hx if m.self_attention else pinned_bf16(m.x_kv)
    hl = pinned_i32(m.kv_lens) if m.kv_lens is not None else None
    hout = pinned_out((m.B, m.n_q, m.d_model))
    tsd.mha_forward_host(hx, hkv, *w, hout, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                         m.mask_kind, hl, 0.0, ws, wsb)
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    got = hout.numpy()
    np.testing.assert_array_equal(got, device_mha(tsd, m, m.x_q))
    ref = oracle.mha(*m.as_f64(), m.h, m.mask_kind, kv_lens=m.kv_lens)
    got64 = torch.from_numpy(got.copy()).view(torch.bfloat16).double().numpy()
    assert_bf16_close(got64, ref, f"mha_forward_host {case}")


@pytest.mark.parametrize("n_ws", [1, 2, 3])
def test_mha_forward_host_back_to_back_calls(tsd, n_ws):
    """Six calls with different inputs, issued without host synchronisation,
    the workspaces taken in turn: each result is its own input's."""
    import torch
    m = synthetic.mha_inputs(1001, 32, 128, 128, 512, 8, 64, 64, MASK_KEY_PADDING, (64, 128),
                             add_pe=True)
    w, wss, wsb = host_mha_setup(tsd, m, n_ws)
    hl = pinned_i32(m.kv_lens)
    xs = [synthetic.mha_inputs(7000 + i, 32, 128, 128, 512, 8, 64, 64).x_q for i in range(6)]
    hxs = [pinned_bf16(x) for x in xs]
    houts = [pinned_out((m.B, m.n_q, m.d_model)) for _ in xs]
    for i, (hx, ho) in enumerate(zip(hxs, houts)):
        tsd.mha_forward_host(hx, hx, *w, ho, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                             m.mask_kind, hl, 0.0, wss[i % n_ws], wsb)
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    for i, x in enumerate(xs):
        np.testing.assert_array_equal(houts[i].numpy(), device_mha(tsd, m, x), err_msg=f"call {i}")


def test_mha_forward_host_pageable_numpy_buffers(tsd):
    """Plain (pageable) numpy arrays as host buffers: the copies are synchronous
    there, and the result is the same."""
    import torch
    m = synthetic.mha_inputs(5150, 4, 96, 96, 512, 8, 64, 64, MASK_KEY_PADDING, (10, 96))
    w, (ws,), wsb = host_mha_setup(tsd, m)
    x = np.ascontiguousarray(m.x_q).view(np.int16)
    lens = np.ascontiguousarray(m.kv_lens, dtype=np.int32)
    out = np.full((m.B, m.n_q, m.d_model), -1, dtype=np.int16)
    tsd.mha_forward_host(x, x, *w, out, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                         m.mask_kind, lens, 0.0, ws, wsb)
    torch.cuda.current_stream().synchronize()
    np.testing.assert_array_equal(out, device_mha(tsd, m, m.x_q))


def test_attn_forward_host_matches_device_call(tsd):
    import torch
    B, h, n_q, n_k, d = 3, 4, 200, 333, 64
    a = synthetic.attention_inputs(5151, B, h, n_q, n_k, d, d, MASK_KEY_PADDING, (0, n_k))
    out_dev = torch.empty((B, h, n_q, d), dtype=torch.bfloat16, device="cuda")
    tsd.attn_forward(to_dev_bf16(a.q), to_dev_bf16(a.k), to_dev_bf16(a.v), out_dev, B, h, n_q,
                     n_k, d, d, a.mask_kind, to_dev_i32(a.kv_lens))
    wsb = tsd.attn_host_workspace_bytes(B, h, n_q, n_k, d, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    hout = pinned_out((B, h, n_q, d))
    tsd.attn_forward_host(pinned_bf16(a.q), pinned_bf16(a.k), pinned_bf16(a.v), hout, B, h, n_q,
                          n_k, d, d, a.mask_kind, pinned_i32(a.kv_lens), 0.0, ws, wsb)
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    np.testing.assert_array_equal(hout.numpy(), bits_of_device(out_dev))


def test_encoder_layer_forward_host_matches_device_call(tsd):
    import torch
    e = synthetic.encoder_inputs(5152, 4, 128, 512, 8, 2048, MASK_KEY_PADDING, (64, 128),
                                 add_pe=True)
    m = e.mha
    params = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o, e.ln1_gamma, e.ln1_beta, e.w_1,
                                       e.b_1, e.w_2, e.b_2, e.ln2_gamma, e.ln2_beta)]
    out_dev = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.encoder_layer_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    tsd.encoder_layer_forward(to_dev_bf16(m.x_q), *params, out_dev, m.B, m.n_q, m.d_model, m.h,
                              m.d_k, e.d_ff, m.mask_kind, to_dev_i32(m.kv_lens), 0.0, 1e-6, ws, wsb)
    hwsb = tsd.encoder_layer_host_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
    hws = torch.empty(hwsb, dtype=torch.uint8, device="cuda")
    hout = pinned_out((m.B, m.n_q, m.d_model))
    tsd.encoder_layer_forward_host(pinned_bf16(m.x_q), *params, hout, m.B, m.n_q, m.d_model, m.h,
                                   m.d_k, e.d_ff, m.mask_kind, pinned_i32(m.kv_lens), 0.0, 1e-6,
                                   hws, hwsb)
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    np.testing.assert_array_equal(hout.numpy(), bits_of_device(out_dev))
    x, _, wq, wk, wv, wo = m.as_f64()
    ref = oracle.encoder_layer(x, wq, wk, wv, wo, *e.params_f64(), m.h, m.mask_kind,
                               kv_lens=m.kv_lens, eps=1e-6)
    got64 = torch.from_numpy(hout.numpy().copy()).view(torch.bfloat16).double().numpy()
    assert_bf16_close(got64, ref, "encoder_layer_forward_host")


@pytest.mark.parametrize("lens", [None, [4096, 1, 0, 2500]])
def test_attn_decode_host_matches_device_call(tsd, lens):
    import torch
    B, h, n_q, n_max, d = 4, 8, 2, 4096, 64
    a = synthetic.attention_inputs(5153, B, h, n_q, n_max, d, d)
    kc, vc = to_dev_bf16(a.k), to_dev_bf16(a.v)
    lens_np = None if lens is None else np.asarray(lens, dtype=np.int32)
    wsb = tsd.attn_decode_workspace_bytes(B, h, n_q, n_max, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    out_dev = torch.empty((B, h, n_q, d), dtype=torch.bfloat16, device="cuda")
    tsd.attn_decode(to_dev_bf16(a.q), kc, vc, out_dev, B, h, n_q, n_max, d, d,
                    None if lens_np is None else to_dev_i32(lens_np), 0.0, ws, wsb)
    hwsb = tsd.attn_decode_host_workspace_bytes(B, h, n_q, n_max, d, d)
    hws = torch.empty(hwsb, dtype=torch.uint8, device="cuda")
    hout = pinned_out((B, h, n_q, d))
    tsd.attn_decode_host(pinned_bf16(a.q), kc, vc, hout, B, h, n_q, n_max, d, d,
                         None if lens_np is None else pinned_i32(lens_np), 0.0, hws, hwsb)
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    np.testing.assert_array_equal(hout.numpy(), bits_of_device(out_dev))


def test_attn_forward_window_host_matches_device_call(tsd):
    import torch
    B, h, n, d, wl, wr = 2, 4, 700, 64, 100, 37
    a = synthetic.attention_inputs(5154, B, h, n, n, d, d)
    out_dev = torch.empty((B, h, n, d), dtype=torch.bfloat16, device="cuda")
    tsd.attn_forward_window(to_dev_bf16(a.q), to_dev_bf16(a.k), to_dev_bf16(a.v), out_dev, B, h, n,
                            n, d, d, wl, wr)
    wsb = tsd.attn_host_workspace_bytes(B, h, n, n, d, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    hout = pinned_out((B, h, n, d))
    tsd.attn_forward_window_host(pinned_bf16(a.q), pinned_bf16(a.k), pinned_bf16(a.v), hout, B, h,
                                 n, n, d, d, wl, wr, workspace=ws, workspace_bytes=wsb)
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    np.testing.assert_array_equal(hout.numpy(), bits_of_device(out_dev))


@pytest.mark.parametrize("n_ws", [1, 2])
def test_mha_forward_host_async_back_to_back_then_join(tsd, n_ws):
    """Asynchronous result copies: eight calls with different inputs, no
    host synchronisation, one join at the end; each result is its own
    input's (a workspace's staging is not rewritten before its copy read it)."""
    import torch
    m = synthetic.mha_inputs(1001, 32, 128, 128, 512, 8, 64, 64, MASK_KEY_PADDING, (64, 128),
                             add_pe=True)
    w, wss, wsb = host_mha_setup(tsd, m, n_ws)
    hl = pinned_i32(m.kv_lens)
    xs = [synthetic.mha_inputs(7100 + i, 32, 128, 128, 512, 8, 64, 64).x_q for i in range(8)]
    hxs = [pinned_bf16(x) for x in xs]
    houts = [pinned_out((m.B, m.n_q, m.d_model)) for _ in xs]
    for i, (hx, ho) in enumerate(zip(hxs, houts)):
        tsd.mha_forward_host_async(hx, hx, *w, ho, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k,
                                   m.d_v, m.mask_kind, hl, 0.0, wss[i % n_ws], wsb)
    tsd.attn_host_join()
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    for i, x in enumerate(xs):
        np.testing.assert_array_equal(houts[i].numpy(), device_mha(tsd, m, x), err_msg=f"call {i}")



def test_mha_forward_host_async_across_workspace_table_eviction(tsd):
    """More workspaces than the library's table of 64 holds, used in turn
    with no host synchronisation: workspace 0 comes back after 65 others have
    evicted its entry, while its first asynchronous result copy may still be
    pending. Every result is its own input's."""
    import torch
    m = synthetic.mha_inputs(1002, 2, 64, 64, 128, 2, 64, 64, MASK_KEY_PADDING, (16, 64))
    n_ws, n_calls = 66, 70
    w, wss, wsb = host_mha_setup(tsd, m, n_ws)
    hl = pinned_i32(m.kv_lens)
    xs = [synthetic.mha_inputs(7200 + i, 2, 64, 64, 128, 2, 64, 64).x_q for i in range(n_calls)]
    hxs = [pinned_bf16(x) for x in xs]
    houts = [pinned_out((m.B, m.n_q, m.d_model)) for _ in xs]
    for i, (hx, ho) in enumerate(zip(hxs, houts)):
        tsd.mha_forward_host_async(hx, hx, *w, ho, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k,
                                   m.d_v, m.mask_kind, hl, 0.0, wss[i % n_ws], wsb)
    tsd.attn_host_join()
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    for i, x in enumerate(xs):
        np.testing.assert_array_equal(houts[i].numpy(), device_mha(tsd, m, x), err_msg=f"call {i}")


def test_attn_decode_host_async_back_to_back_then_join(tsd):
    """Six decoding steps with different queries and lengths through two
    workspaces, no host synchronisation, one join: each result equals its own
    step's device call."""
    import torch
    B, h, n_q, n_max, d = 4, 8, 1, 2048, 64
    a = synthetic.attention_inputs(5160, B, h, n_q, n_max, d, d)
    kc, vc = to_dev_bf16(a.k), to_dev_bf16(a.v)
    hwsb = tsd.attn_decode_host_workspace_bytes(B, h, n_q, n_max, d, d)
    hws = [torch.empty(hwsb, dtype=torch.uint8, device="cuda") for _ in range(2)]
    rng = np.random.default_rng(5161)
    steps = [(synthetic.attention_inputs(5170 + i, B, h, n_q, 1, d, d).q,
              rng.integers(0, n_max + 1, size=B).astype(np.int32)) for i in range(6)]
    hq = [pinned_bf16(q) for q, _ in steps]
    hl = [pinned_i32(l) for _, l in steps]
    houts = [pinned_out((B, h, n_q, d)) for _ in steps]
    for i in range(len(steps)):
        tsd.attn_decode_host_async(hq[i], kc, vc, houts[i], B, h, n_q, n_max, d, d, hl[i], 0.0,
                                   hws[i % 2], hwsb)
    tsd.attn_host_join()
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    wsb = tsd.attn_decode_workspace_bytes(B, h, n_q, n_max, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    for i, (q, lens) in enumerate(steps):
        out_dev = torch.empty((B, h, n_q, d), dtype=torch.bfloat16, device="cuda")
        tsd.attn_decode(to_dev_bf16(q), kc, vc, out_dev, B, h, n_q, n_max, d, d, to_dev_i32(lens),
                        0.0, ws, wsb)
        np.testing.assert_array_equal(houts[i].numpy(), bits_of_device(out_dev),
                                      err_msg=f"step {i}")


def test_encoder_layer_forward_host_async_back_to_back_then_join(tsd):
    """Four layers with different inputs through two workspaces, no host
    synchronisation, one join: each result equals its own device call."""
    import torch
    e = synthetic.encoder_inputs(5180, 4, 128, 512, 8, 2048, MASK_KEY_PADDING, (64, 128),
                                 add_pe=True)
    m = e.mha
    params = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o, e.ln1_gamma, e.ln1_beta, e.w_1,
                                       e.b_1, e.w_2, e.b_2, e.ln2_gamma, e.ln2_beta)]
    hwsb = tsd.encoder_layer_host_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
    hws = [torch.empty(hwsb, dtype=torch.uint8, device="cuda") for _ in range(2)]
    xs = [synthetic.encoder_inputs(5181 + i, 4, 128, 512, 8, 2048).mha.x_q for i in range(4)]
    hxs = [pinned_bf16(x) for x in xs]
    hl = pinned_i32(m.kv_lens)
    houts = [pinned_out((m.B, m.n_q, m.d_model)) for _ in xs]
    for i in range(len(xs)):
        tsd.encoder_layer_forward_host_async(hxs[i], *params, houts[i], m.B, m.n_q, m.d_model, m.h,
                                             m.d_k, e.d_ff, m.mask_kind, hl, 0.0, 1e-6,
                                             hws[i % 2], hwsb)
    tsd.attn_host_join()
    torch.cuda.current_stream().synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    wsb = tsd.encoder_layer_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    dl = to_dev_i32(m.kv_lens)
    for i, x in enumerate(xs):
        out_dev = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16, device="cuda")
        tsd.encoder_layer_forward(to_dev_bf16(x), *params, out_dev, m.B, m.n_q, m.d_model, m.h,
                                  m.d_k, e.d_ff, m.mask_kind, dl, 0.0, 1e-6, ws, wsb)
        np.testing.assert_array_equal(houts[i].numpy(), bits_of_device(out_dev),
                                      err_msg=f"layer {i}")
