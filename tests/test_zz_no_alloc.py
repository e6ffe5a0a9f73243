"""mha_forward_noalloc: multi-head attention for callers that cannot allocate
device memory (a plugin whose host owns the memory budget, a serving loop
that must not call cudaMalloc/cudaFree on the request path, a C caller with
no access to its framework's allocator). It runs on the library's fixed
device scratch instead of a caller workspace. Its output must match
mha_forward's on the same inputs, on consecutive calls that reuse the
scratch. This file is collected last on purpose."""
import numpy as np
import pytest

import synthetic
from synthetic import MASK_CAUSAL, MASK_KEY_PADDING

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


def _both(tsd, m):
    """(mha_forward_noalloc output, mha_forward output) on the same inputs."""
    import torch
    x_q = to_dev_bf16(m.x_q)
    x_kv = x_q if m.self_attention else to_dev_bf16(m.x_kv)
    w = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o)]
    lens = to_dev_i32(m.kv_lens) if m.kv_lens is not None else None
    args = (m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v, m.mask_kind, lens, 0.0)
    out_na = torch.full((m.B, m.n_q, m.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    tsd.mha_forward_noalloc(x_q, x_kv, *w, out_na, *args)
    wsb = tsd.mha_workspace_bytes(m.B, m.n_q, m.n_k, m.h, m.d_k, m.d_v)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    out_ws = torch.empty_like(out_na)
    tsd.mha_forward(x_q, x_kv, *w, out_ws, *args, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    return to_host_f64(out_na), to_host_f64(out_ws)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(tsd):
    # call 1: encoder self-attention with key padding (16 MiB of scratch)
    m1 = synthetic.mha_inputs(4001, 32, 128, 128, 512, 8, 64, 64, MASK_KEY_PADDING, (64, 128),
                              add_pe=True)
    got, ref = _both(tsd, m1)
    assert_bf16_close(got, ref, "first call")
    # call 2: other shapes and masks on the same scratch (cross-attention, n_k=160)
    m2 = synthetic.mha_inputs(4002, 32, 128, 160, 512, 8, 64, 64, MASK_KEY_PADDING, (80, 160),
                              self_attention=False)
    got, ref = _both(tsd, m2)
    assert_bf16_close(got, ref, "second call")
    # and back to a causal self-attention, smaller than the scratch's last contents
    m3 = synthetic.mha_inputs(4003, 3, 70, 70, 128, 2, 64, 64, MASK_CAUSAL)
    got, ref = _both(tsd, m3)
    assert_bf16_close(got, ref, "third call")


def test_noalloc_three_launch_path_uses_every_scratch_region(tsd):
    """Sequences longer than the fused kernel's 128 rows take the projection
    GEMM, the attention kernel and the output GEMM, so Q, K, V and the merged
    heads all live in the scratch array; two calls in a row."""
    assert tsd.mha_forward_launches(2, 512, 512, 512, 8, 64, 64, True) == 3
    for seed in (4004, 4005):
        m = synthetic.mha_inputs(seed, 2, 512, 512, 512, 8, 64, 64, MASK_KEY_PADDING, (256, 512))
        got, ref = _both(tsd, m)
        assert_bf16_close(got, ref, f"seed {seed}")


def test_noalloc_refuses_sizes_beyond_its_scratch(tsd):
    lib = tsd.library()
    B, n, dm, h, d = 64, 1024, 512, 8, 64
    assert tsd.mha_workspace_bytes(B, n, n, h, d, d) > tsd.MHA_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    st = lib.mha_forward_noalloc(fake, fake, fake, fake, fake, fake, fake, B, n, n, dm, h, d, d,
                                 0, None, 0.0, None)
    assert st == tsd.ATTN_ERR_UNSUPPORTED
