"""GPU parity of mha_forward (projections, masked attention per head, output
projection) against the fp64 oracle, at the Transformer-base shapes and at
small ragged ones."""
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


def run_mha(tsd, m):
    import torch
    x_q = to_dev_bf16(m.x_q)
    x_kv = x_q if m.self_attention else to_dev_bf16(m.x_kv)
    w = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o)]
    out = torch.full((m.B, m.n_q, m.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.mha_workspace_bytes(m.B, m.n_q, m.n_k, m.h, m.d_k, m.d_v)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lens = to_dev_i32(m.kv_lens) if m.kv_lens is not None else None
    tsd.mha_forward(x_q, x_kv, *w, out, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                    m.mask_kind, lens, 0.0, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    return to_host_f64(out), ws


def check(tsd, m, what):
    got, _ = run_mha(tsd, m)
    ref = oracle.mha(*m.as_f64(), m.h, m.mask_kind, kv_lens=m.kv_lens)
    return assert_bf16_close(got, ref, what)


def test_base_encoder_self_attention_key_padding(tsd):
    """Transformer-base encoder self-attention: B=32, n=128, d_model=512, h=8,
    d_k=d_v=64, x ~ N(0,1) + PE, Xavier weights, kv_len ~ U[64, 128]."""
    m = synthetic.mha_inputs(1001, 32, 128, 128, 512, 8, 64, 64, MASK_KEY_PADDING, (64, 128),
                             add_pe=True)
    check(tsd, m, "base encoder")


def test_base_decoder_masked_self_attention(tsd):
    m = synthetic.mha_inputs(1002, 32, 128, 128, 512, 8, 64, 64, MASK_CAUSAL | MASK_KEY_PADDING,
                             (64, 128))
    check(tsd, m, "base decoder self")


def test_base_decoder_cross_attention(tsd):
    """Decoder queries (n_q=128) against encoder memory (n_k=160), source padding."""
    m = synthetic.mha_inputs(1012, 32, 128, 160, 512, 8, 64, 64, MASK_KEY_PADDING, (80, 160),
                             self_attention=False)
    check(tsd, m, "base cross")


@pytest.mark.parametrize("shape", [
    # B, n_q, n_k, d_model, h, d, mask, self
    (1, 1, 1, 64, 1, 64, MASK_NONE, True),
    (2, 70, 70, 72, 2, 64, MASK_CAUSAL, True),            # d_model not a multiple of 64
    (3, 50, 129, 200, 3, 64, MASK_KEY_PADDING, False),
    (2, 130, 130, 256, 2, 128, MASK_KEY_PADDING, True),
    (1, 257, 257, 1024, 16, 64, MASK_CAUSAL, True),       # Transformer-big width
])
def test_mha_small_shapes(tsd, shape):
    B, n_q, n_k, dm, h, d, mask, self_attn = shape
    m = synthetic.mha_inputs(3000 + n_q + dm, B, n_q, n_k, dm, h, d, d, mask, (1, n_k),
                             self_attention=self_attn)
    check(tsd, m, str(shape))


def test_mha_intermediate_projections_and_heads(tsd):
    """The workspace holds Q = X W_Q (head i = column block i) and the merged
    heads; check both against the oracle's pieces."""
    import torch
    m = synthetic.mha_inputs(3100, 2, 96, 96, 128, 2, 64, 64, MASK_CAUSAL)
    got, ws = run_mha(tsd, m)
    x, _, wq, _, _, wo = m.as_f64()
    q_dev = ws[:2 * 96 * 128 * 2].view(torch.bfloat16).float().cpu().numpy().reshape(2, 96, 128)
    assert_bf16_close(q_dev, x @ wq, "Q projection")
    ref, concat = oracle.mha(*m.as_f64(), 2, MASK_CAUSAL, return_concat=True)
    off = tsd.mha_workspace_bytes(2, 96, 96, 2, 64, 64) - 2 * 96 * 128 * 2
    o_dev = ws[off:].view(torch.bfloat16).float().cpu().numpy().reshape(2, 96, 128)
    assert_bf16_close(o_dev, concat, "merged heads")
    assert_bf16_close(got, ref, "output")
