"""GPU parity on seeded random shapes: head sizes, lengths, masks, key
lengths (0 included), restricted windows and multi-head layouts drawn from
fixed seeds, so every run sees the same cases; each output is compared with
the fp64 oracle element by element at the bf16 tolerances."""
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


def _attention_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(count):
        d = int(rng.choice([16, 32, 64, 64, 64, 128, 128, 256]))
        B, h = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        n_q = int(rng.integers(1, 700))
        self_attn = rng.random() < 0.6
        n_k = n_q if self_attn else int(rng.integers(1, 700))
        mask = MASK_CAUSAL if self_attn and rng.random() < 0.5 else MASK_NONE
        kv_range = None
        if rng.random() < 0.5:
            mask |= MASK_KEY_PADDING
            kv_range = (int(rng.integers(0, n_k + 1)), n_k)
        window = None
        if self_attn and rng.random() < 0.4:
            window = tuple(int(rng.choice([-1, rng.integers(0, 400)])) for _ in range(2))
        cases.append((B, h, n_q, n_k, d, mask, kv_range, window))
    return cases


ATTN_CASES = _attention_cases(48, 7101)


def _attn_id(c):
    B, h, n_q, n_k, d, mask, _, window = c
    w = "" if window is None else "w{}_{}".format(*window)
    return f"B{B}h{h}q{n_q}k{n_k}d{d}m{mask}{w}"


@pytest.mark.parametrize("case", ATTN_CASES, ids=_attn_id)
def test_random_attention_matches_oracle(tsd, case):
    import torch
    B, h, n_q, n_k, d, mask, kv_range, window = case
    a = synthetic.attention_inputs(7200 + sum(case[:5]), B, h, n_q, n_k, d, d, mask, kv_range)
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    out = torch.full((B, h, n_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lens = to_dev_i32(a.kv_lens) if a.kv_lens is not None else None
    if window is None:
        tsd.attn_forward(q, k, v, out, B, h, n_q, n_k, d, d, mask, lens, 0.0)
    else:
        tsd.attn_forward_window(q, k, v, out, B, h, n_q, n_k, d, d, window[0], window[1], mask,
                                lens)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    ref = oracle.attention(*a.as_f64(), mask, kv_lens=a.kv_lens, window=window)
    assert_bf16_close(to_host_f64(out), ref, _attn_id(case))


def _mha_cases(count, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(count):
        B = int(rng.integers(1, 6))
        self_attn = rng.random() < 0.5
        if i % 2 == 0:
            # the one-launch shapes: d = 64, an even head count whose pairs
            # each own 64 or 128 output columns, n_q <= 128 and n_k <= 128
            # (cross-attention: up to 192)
            h = int(rng.choice([2, 4, 8, 16]))
            d = 64
            d_model = (h // 2) * int(rng.choice([64, 128]))
            n_q = int(rng.integers(1, 129))
            n_k = n_q if self_attn else int(rng.integers(1, 193))
        else:
            h = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
            d = 64 if rng.random() < 0.7 else int(rng.choice([32, 128]))
            d_model = 64 * int(rng.integers(1, 17))
            n_q = int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(1, 400))]))
            n_k = n_q if self_attn else int(rng.choice([int(rng.integers(1, 193)),
                                                          int(rng.integers(1, 400))]))
        mask = MASK_CAUSAL if self_attn and rng.random() < 0.4 else MASK_NONE
        kv_range = None
        if rng.random() < 0.6:
            mask |= MASK_KEY_PADDING
            kv_range = (int(rng.integers(0, n_k + 1)), n_k)
        cases.append((B, n_q, n_k, d_model, h, d, mask, kv_range, self_attn))
    return cases


MHA_CASES = _mha_cases(32, 7301)


def _mha_id(c):
    B, n_q, n_k, d_model, h, d, mask, _, self_attn = c
    return f"B{B}q{n_q}k{n_k}dm{d_model}h{h}d{d}m{mask}{'s' if self_attn else 'x'}"


@pytest.mark.parametrize("case", MHA_CASES, ids=_mha_id)
def test_random_mha_matches_oracle(tsd, case):
    """Whichever plan mha_forward takes for the shape (one fused launch, the
    fused heads then the W_O GEMM, or three launches)."""
    import torch
    B, n_q, n_k, d_model, h, d, mask, kv_range, self_attn = case
    m = synthetic.mha_inputs(7400 + B + n_q + n_k + d_model + h, B, n_q, n_k, d_model, h, d, d,
                             mask, kv_range, self_attention=self_attn)
    x_q = to_dev_bf16(m.x_q)
    x_kv = x_q if self_attn else to_dev_bf16(m.x_kv)
    w = [to_dev_bf16(t) for t in (m.w_q, m.w_k, m.w_v, m.w_o)]
    out = torch.full((B, n_q, d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.mha_workspace_bytes(B, n_q, n_k, h, d, d)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")
    lens = to_dev_i32(m.kv_lens) if m.kv_lens is not None else None
    tsd.mha_forward(x_q, x_kv, *w, out, B, n_q, n_k, d_model, h, d, d, mask, lens, 0.0, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    ref = oracle.mha(*m.as_f64(), h, mask, kv_lens=m.kv_lens)
    assert_bf16_close(to_host_f64(out), ref, _mha_id(case))
