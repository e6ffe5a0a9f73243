"""Calls from several host threads at once, each on its own stream with its
own workspace (the library's caches, the tensor-map memo and the host
staging runtime are shared): every result equals the single-threaded one."""
import threading

import numpy as np
import pytest

import synthetic
from synthetic import MASK_KEY_PADDING

from gpu_util import to_dev_bf16, to_dev_i32

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


def bits(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy()


def test_threads_on_separate_streams_match_single_thread(tsd):
    import torch
    m = synthetic.mha_inputs(6100, 32, 128, 128, 512, 8, 64, 64, MASK_KEY_PADDING, (64, 128),
                             add_pe=True)
    a = synthetic.attention_inputs(6101, 2, 16, 1000, 1000, 64, 64)
    x = to_dev_bf16(m.x_q)
    w = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o)]
    lens = to_dev_i32(m.kv_lens)
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    wsb = tsd.mha_workspace_bytes(m.B, m.n_q, m.n_k, m.h, m.d_k, m.d_v)
    hwsb = tsd.mha_host_workspace_bytes(m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v)
    h_x = torch.from_numpy(np.ascontiguousarray(m.x_q).view(np.int16)).pin_memory()
    h_lens = torch.from_numpy(np.ascontiguousarray(m.kv_lens, dtype=np.int32)).pin_memory()

    def run(stream, ws, hws, outs):
        mo = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16, device="cuda")
        ao = torch.empty((a.B, a.h, a.n_q, a.d_v), dtype=torch.bfloat16, device="cuda")
        ho = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.int16).pin_memory()
        for _ in range(20):
            tsd.mha_forward(x, x, *w, mo, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                            m.mask_kind, lens, 0.0, ws, wsb, stream)
            tsd.attn_forward(q, k, v, ao, a.B, a.h, a.n_q, a.n_k, a.d_k, a.d_v, 0, None, 0.0,
                             stream)
            tsd.mha_forward_host(h_x, h_x, *w, ho, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k,
                                 m.d_v, m.mask_kind, h_lens, 0.0, hws, hwsb, stream)
        stream.synchronize()
        outs.extend([bits(mo), bits(ao), ho.numpy().copy()])

    ref = []
    s0 = torch.cuda.Stream()
    run(s0, torch.empty(wsb, dtype=torch.uint8, device="cuda"),
        torch.empty(hwsb, dtype=torch.uint8, device="cuda"), ref)
    results = [[] for _ in range(3)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    wss = [torch.empty(wsb, dtype=torch.uint8, device="cuda") for _ in range(3)]
    hwss = [torch.empty(hwsb, dtype=torch.uint8, device="cuda") for _ in range(3)]
    errors = []

    def worker(i):
        try:
            run(streams[i], wss[i], hwss[i], results[i])
        except Exception as exc:  # reported below, on the main thread
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    for i in range(3):
        for got, want in zip(results[i], ref):
            np.testing.assert_array_equal(got, want)
