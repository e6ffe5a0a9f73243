"""GPU parity of encoder_layer_forward (post-LN self-attention and
feed-forward sub-layers) against the fp64 oracle on the same bf16 inputs."""
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


def run_layer(tsd, e, eps):
    import torch
    m = e.mha
    dev = [to_dev_bf16(t) for t in (m.x_q, m.w_q, m.w_k, m.w_v, m.w_o, e.ln1_gamma, e.ln1_beta,
                                    e.w_1, e.b_1, e.w_2, e.b_2, e.ln2_gamma, e.ln2_beta)]
    out = torch.full((m.B, m.n_q, m.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.encoder_layer_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lens = to_dev_i32(m.kv_lens) if m.kv_lens is not None else None
    tsd.encoder_layer_forward(*dev, out, m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff, m.mask_kind,
                              lens, 0.0, eps, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    return to_host_f64(out)


CASES = [
    # B, n, d_model, h, d_ff, mask, kv_range
    (8, 128, 512, 8, 2048, MASK_KEY_PADDING, (64, 128)),   # Transformer-base, fused attention
    (3, 100, 512, 8, 2048, MASK_CAUSAL, None),
    (2, 200, 256, 4, 1024, MASK_NONE, None),               # projection GEMM path (n > 128)
    (2, 64, 1024, 16, 4096, MASK_KEY_PADDING, (1, 64)),    # Transformer-big widths
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}n{}dm{}h{}ff{}m{}".format(*c[:6]))
def test_encoder_layer_matches_oracle(tsd, case):
    B, n, dm, h, ff, mask, rng = case
    e = synthetic.encoder_inputs(4000 + n + dm, B, n, dm, h, ff, mask, rng, add_pe=True)
    eps = 1e-6
    got = run_layer(tsd, e, eps)
    m = e.mha
    x, _, wq, wk, wv, wo = m.as_f64()
    ref = oracle.encoder_layer(x, wq, wk, wv, wo, *e.params_f64(), h, mask, kv_lens=m.kv_lens,
                               eps=eps)
    assert_bf16_close(got, ref, str(case))


def test_encoder_layer_other_eps(tsd):
    e = synthetic.encoder_inputs(4100, 2, 50, 256, 4, 512, MASK_NONE)
    got = run_layer(tsd, e, 1e-2)
    m = e.mha
    x, _, wq, wk, wv, wo = m.as_f64()
    ref = oracle.encoder_layer(x, wq, wk, wv, wo, *e.params_f64(), 4, MASK_NONE, eps=1e-2)
    assert_bf16_close(got, ref, "eps 1e-2")


@pytest.mark.parametrize("B", [1, 2, 4])
def test_encoder_layer_small_batches_repeated(tsd, B):
    """Small batches leave most SMs free during the first FFN GEMM, so the
    second GEMM's CTAs start beside it, and beside the LayerNorm before it
    (every kernel releases its dependents at entry): its epilogue must not
    read the fp32 residual before the grid dependency has resolved. Several
    back-to-back layers, each against the oracle."""
    import torch
    e = synthetic.encoder_inputs(4200 + B, B, 128, 512, 8, 2048, MASK_KEY_PADDING, (64, 128),
                                 add_pe=True)
    m = e.mha
    dev = [to_dev_bf16(t) for t in (m.x_q, m.w_q, m.w_k, m.w_v, m.w_o, e.ln1_gamma, e.ln1_beta,
                                    e.w_1, e.b_1, e.w_2, e.b_2, e.ln2_gamma, e.ln2_beta)]
    wsb = tsd.encoder_layer_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    lens = to_dev_i32(m.kv_lens)
    outs = [torch.full((m.B, m.n_q, m.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(8)]
    for out in outs:
        tsd.encoder_layer_forward(*dev, out, m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff,
                                  m.mask_kind, lens, 0.0, 1e-6, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    x, _, wq, wk, wv, wo = m.as_f64()
    ref = oracle.encoder_layer(x, wq, wk, wv, wo, *e.params_f64(), m.h, m.mask_kind,
                               kv_lens=m.kv_lens, eps=1e-6)
    for i, out in enumerate(outs):
        assert_bf16_close(to_host_f64(out), ref, f"B={B} layer {i}")


@pytest.mark.parametrize("B,dm,h,ff", [(64, 1024, 16, 4096), (160, 512, 8, 2048)])
def test_encoder_layer_several_row_tiles_per_cluster(tsd, B, dm, h, ff):
    """Enough rows that each cluster of the second FFN GEMM (whose epilogue
    takes the LayerNorm, a row's d_model columns over d_model / 128 CTAs)
    walks several row tiles: the statistics slots alternate. Sequences are
    independent, so the oracle checks a seeded sample of them."""
    import torch
    e = synthetic.encoder_inputs(4300 + B, B, 128, dm, h, ff, MASK_KEY_PADDING, (64, 128),
                                 add_pe=True)
    got = run_layer(tsd, e, 1e-6)
    m = e.mha
    pick = np.unique(np.concatenate([[0, B - 1], np.random.default_rng(B).choice(B, 4, False)]))
    x, _, wq, wk, wv, wo = m.as_f64()
    ref = oracle.encoder_layer(x[pick], wq, wk, wv, wo, *e.params_f64(), h, m.mask_kind,
                               kv_lens=m.kv_lens[pick], eps=1e-6)
    assert_bf16_close(got[pick], ref, f"B={B} d_model={dm}")
