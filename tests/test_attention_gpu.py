"""GPU parity: attn_forward / attn_forward_strided / attn_forward_f32 against
the fp64 oracle on the same seeded inputs, element by element, at sizes that
span several tiles and ragged tails; plus invariants, bounds canaries and
the bounded-wait failure path."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE

from gpu_util import (assert_bf16_close, assert_f32_close, to_dev_bf16, to_dev_i32, to_host_f64)

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


def run_bf16(tsd, a, scale=0.0):
    import torch
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    out = torch.full((a.B, a.h, a.n_q, a.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lens = to_dev_i32(a.kv_lens) if a.kv_lens is not None else None
    tsd.attn_forward(q, k, v, out, a.B, a.h, a.n_q, a.n_k, a.d_k, a.d_v, a.mask_kind, lens, scale)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    return to_host_f64(out)


CASES = [
    # B, h, n_q, n_k, d, mask, kv_len_range
    (1, 1, 1, 1, 64, MASK_NONE, None),
    (2, 3, 17, 17, 64, MASK_NONE, None),
    (1, 2, 127, 127, 64, MASK_CAUSAL, None),
    (2, 2, 128, 128, 64, MASK_NONE, None),
    (1, 2, 129, 129, 64, MASK_CAUSAL, None),
    (3, 2, 128, 160, 64, MASK_NONE, None),                 # cross-attention, n_q != n_k
    (3, 2, 128, 160, 64, MASK_KEY_PADDING, (80, 160)),
    (4, 2, 128, 128, 64, MASK_CAUSAL | MASK_KEY_PADDING, (64, 128)),
    (2, 2, 300, 300, 64, MASK_CAUSAL, None),               # two query tiles per CTA, ragged
    (2, 2, 300, 517, 64, MASK_KEY_PADDING, (1, 517)),
    (1, 2, 1000, 1000, 64, MASK_CAUSAL | MASK_KEY_PADDING, (300, 1000)),
    (2, 2, 17, 1000, 64, MASK_NONE, None),
    (1, 1, 1, 1, 128, MASK_NONE, None),
    (2, 2, 129, 129, 128, MASK_CAUSAL, None),
    (2, 2, 128, 160, 128, MASK_KEY_PADDING, (1, 160)),
    (1, 2, 600, 600, 128, MASK_CAUSAL | MASK_KEY_PADDING, (200, 600)),
    (1, 1, 384, 700, 128, MASK_NONE, None),
    # more single-tile items than pipelines: every slot walks several items
    (40, 16, 100, 100, 64, MASK_KEY_PADDING, (1, 100)),
    (32, 16, 128, 128, 64, MASK_CAUSAL, None),
    # Table 3's other head sizes: 16 and 32 through the 64-column kernels, 256
    (2, 3, 200, 200, 16, MASK_CAUSAL, None),
    (3, 2, 64, 64, 16, MASK_KEY_PADDING, (0, 64)),
    (2, 2, 130, 300, 32, MASK_KEY_PADDING, (1, 300)),
    (1, 2, 1000, 1000, 32, MASK_NONE, None),
    (2, 2, 300, 300, 256, MASK_CAUSAL | MASK_KEY_PADDING, (50, 300)),
    (1, 1, 128, 700, 256, MASK_NONE, None),
    (3, 2, 77, 77, 256, MASK_KEY_PADDING, (0, 77)),
    # 160 paired items over 152 SMs: the last partial round runs as single
    # query tiles (16 of them), including ragged blocks past n_q
    (5, 16, 500, 500, 64, MASK_NONE, None),
    (5, 16, 500, 500, 64, MASK_KEY_PADDING, (1, 500)),
    (5, 16, 300, 300, 128, MASK_NONE, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}h{}q{}k{}d{}m{}".format(*c[:6]))
def test_attn_forward_matches_oracle(tsd, case):
    B, h, n_q, n_k, d, mask, rng = case
    a = synthetic.attention_inputs(2000 + sum(case[:5]), B, h, n_q, n_k, d, d, mask, rng)
    got = run_bf16(tsd, a)
    ref = oracle.attention(*a.as_f64(), mask, kv_lens=a.kv_lens)
    assert_bf16_close(got, ref, str(case))


@pytest.mark.parametrize("n,d", [(100, 64), (200, 64), (100, 128), (200, 128)])
def test_attn_forward_key_lengths_zero_one_full(tsd, n, d):
    """kv_len = 0 gives zero rows; 1 gives v_0 exactly; n_k is unmasked (one
    and two query tiles per work item, both head sizes)."""
    a = synthetic.attention_inputs(2100 + n + d, 3, 2, n, n, d, d, MASK_KEY_PADDING)
    a.kv_lens = np.array([0, 1, n], dtype=np.int32)
    got = run_bf16(tsd, a)
    ref = oracle.attention(*a.as_f64(), MASK_KEY_PADDING, kv_lens=a.kv_lens)
    assert np.all(got[0] == 0.0)
    v = a.as_f64()[2]
    np.testing.assert_array_equal(got[1], np.broadcast_to(v[1, :, :1], got[1].shape))
    assert_bf16_close(got, ref, "kv_len 0/1/full")
    # out-of-range lengths are clamped
    a.kv_lens = np.array([-7, 5000, 3], dtype=np.int32)
    got = run_bf16(tsd, a)
    ref = oracle.attention(*a.as_f64(), MASK_KEY_PADDING, kv_lens=a.kv_lens)
    assert_bf16_close(got, ref, "clamped lengths")


@pytest.mark.parametrize("n_q,d", [(100, 64), (300, 64), (100, 128), (300, 128)])
def test_attn_forward_no_keys_gives_zeros(tsd, n_q, d):
    """n_k = 0: every row attends over an empty key set, whose result is 0.
    K and V point at a small live buffer that must not be read."""
    import torch
    B, h = 2, 2
    q = to_dev_bf16(synthetic.attention_inputs(2150, B, h, n_q, 1, d, d, MASK_NONE).q)
    kv = torch.full((64,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, h, n_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    tsd.attn_forward(q, kv, kv, out, B, h, n_q, 0, d, d, MASK_NONE, None, 0.0)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    assert torch.all(out == 0).item()


def test_attn_forward_explicit_scale(tsd):
    a = synthetic.attention_inputs(2101, 2, 2, 130, 130, 64, 64)
    got = run_bf16(tsd, a, scale=0.05)
    ref = oracle.attention(*a.as_f64(), scale=0.05)
    assert_bf16_close(got, ref, "scale 0.05")


def test_causal_row_zero_is_v0_and_zero_query_is_mean(tsd):
    a = synthetic.attention_inputs(2102, 2, 2, 256, 256, 64, 64, MASK_CAUSAL)
    got = run_bf16(tsd, a)
    v = a.as_f64()[2]
    np.testing.assert_array_equal(got[:, :, 0], v[:, :, 0])   # one key: exact
    a.q = np.zeros_like(a.q)
    got = run_bf16(tsd, a)
    for i in (1, 100, 255):
        np.testing.assert_allclose(got[:, :, i], v[:, :, :i + 1].mean(axis=2), atol=1e-2)


def test_deterministic_and_canaries_untouched(tsd):
    import torch
    a = synthetic.attention_inputs(2103, 2, 3, 257, 257, 64, 64, MASK_CAUSAL)
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    n = a.B * a.h * a.n_q * a.d_v
    guard = 4096
    buf = torch.full((n + 2 * guard,), -12345.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n]
    outs = []
    for _ in range(2):
        tsd.attn_forward(q, k, v, out, a.B, a.h, a.n_q, a.n_k, 64, 64, MASK_CAUSAL, None, 0.0)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.all(buf[:guard] == -12345.0) and torch.all(buf[guard + n:] == -12345.0)


def test_strided_layout_matches_contiguous(tsd):
    """Heads read from [B, n, h*d] and written merged as [B, n_q, h*d]."""
    import torch
    B, h, n_q, n_k, d = 2, 4, 200, 333, 64
    a = synthetic.attention_inputs(2104, B, h, n_q, n_k, d, d, MASK_KEY_PADDING, (50, 333))
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    lens = to_dev_i32(a.kv_lens)
    ref = torch.empty((B, h, n_q, d), dtype=torch.bfloat16, device="cuda")
    tsd.attn_forward(q, k, v, ref, B, h, n_q, n_k, d, d, MASK_KEY_PADDING, lens, 0.0)
    qm, km, vm = (t.transpose(1, 2).contiguous() for t in (q, k, v))  # [B, n, h, d]
    om = torch.empty((B, n_q, h, d), dtype=torch.bfloat16, device="cuda")
    tsd.attn_forward_strided(qm, n_q * h * d, d, h * d, km, n_k * h * d, d, h * d,
                             vm, n_k * h * d, d, h * d, om, n_q * h * d, d, h * d,
                             B, h, n_q, n_k, d, d, MASK_KEY_PADDING, lens, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(om.transpose(1, 2).contiguous().view(torch.int16), ref.view(torch.int16))


# ------------------------------------------------------------------ fp32 path

F32_CASES = [
    (1, 1, 16, 16, 64, 64, MASK_NONE, None),     # the single-head fp32 sanity shape
    (2, 3, 33, 33, 64, 64, MASK_CAUSAL, None),
    (2, 2, 45, 70, 16, 40, MASK_KEY_PADDING, (0, 70)),
    (1, 2, 100, 100, 128, 128, MASK_CAUSAL | MASK_KEY_PADDING, (30, 100)),
    (1, 1, 5, 9, 1, 3, MASK_NONE, None),
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "B{}h{}q{}k{}dk{}dv{}m{}".format(*c[:7]))
def test_attn_forward_f32_matches_oracle(tsd, case):
    import torch
    B, h, n_q, n_k, d_k, d_v, mask, rng = case
    a = synthetic.attention_inputs(1000 + sum(case[:6]), B, h, n_q, n_k, d_k, d_v, mask, rng,
                                   dtype="f32")
    q, k, v = (torch.from_numpy(t).cuda() for t in (a.q, a.k, a.v))
    out = torch.full((B, h, n_q, d_v), float("nan"), dtype=torch.float32, device="cuda")
    lens = to_dev_i32(a.kv_lens) if a.kv_lens is not None else None
    tsd.attn_forward_f32(q, k, v, out, B, h, n_q, n_k, d_k, d_v, mask, lens, 0.0)
    torch.cuda.synchronize()
    ref = oracle.attention(*a.as_f64(), mask, kv_lens=a.kv_lens)
    assert_f32_close(out.cpu().numpy(), ref, str(case))


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout_and_context_survives(tsd):
    import torch
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    tsd.attn_selftest_wait_timeout(2000)  # 2 ms wait on a barrier nothing arrives on
    assert tsd.attn_get_device_status() == tsd.ATTN_ERR_DEVICE_TIMEOUT
    assert tsd.attn_get_device_status() == tsd.ATTN_OK  # read-and-clear
    # the context is still usable
    a = synthetic.attention_inputs(2105, 1, 1, 64, 64, 64, 64)
    ref = oracle.attention(*a.as_f64())
    assert_bf16_close(run_bf16(tsd, a), ref, "after timeout")
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


# ---------------------------------------------------------------- restricted self-attention

def run_window(tsd, a, left, right):
    import torch
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    out = torch.full((a.B, a.h, a.n_q, a.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lens = to_dev_i32(a.kv_lens) if a.kv_lens is not None else None
    tsd.attn_forward_window(q, k, v, out, a.B, a.h, a.n_q, a.n_k, a.d_k, a.d_v, left, right,
                            a.mask_kind, lens)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    return to_host_f64(out)


WINDOW_CASES = [
    # B, h, n, d, mask, kv_len_range, left, right
    (2, 2, 100, 64, MASK_NONE, None, 0, 0),            # each query only its own key
    (2, 2, 100, 64, MASK_NONE, None, 7, 3),            # one query tile per item
    (1, 2, 1000, 64, MASK_NONE, None, 128, 128),       # tile-aligned radius, paired tiles
    (1, 2, 1000, 64, MASK_NONE, None, 200, 57),        # ragged bounds on both sides
    (2, 2, 777, 64, MASK_CAUSAL, None, 300, -1),       # causal sliding window
    (2, 2, 777, 64, MASK_KEY_PADDING, (1, 777), 90, 250),
    (1, 2, 1500, 64, MASK_CAUSAL | MASK_KEY_PADDING, (400, 1500), 129, 0),
    (1, 2, 600, 64, MASK_NONE, None, -1, 100),         # bound on one side only
    (1, 2, 600, 64, MASK_NONE, None, 5000, 5000),      # window wider than the sequence
    (2, 2, 300, 128, MASK_NONE, None, 40, 40),
    (1, 2, 1000, 128, MASK_CAUSAL, None, 256, -1),
    (40, 8, 128, 64, MASK_KEY_PADDING, (1, 128), 16, 16),
    (1, 2, 600, 256, MASK_NONE, None, 100, 100),
    (2, 2, 500, 32, MASK_CAUSAL, None, 64, -1),
    # 160 paired items: the last partial round as single query tiles
    (5, 16, 500, 64, MASK_NONE, None, 100, 50),
    (5, 16, 300, 128, MASK_KEY_PADDING, (1, 300), 60, 130),
]


@pytest.mark.parametrize("case", WINDOW_CASES,
                         ids=lambda c: "B{}h{}n{}d{}m{}w{}_{}".format(*c[:5], c[6], c[7]))
def test_attn_forward_window_matches_oracle(tsd, case):
    B, h, n, d, mask, rng, left, right = case
    a = synthetic.attention_inputs(2500 + B + n + d + max(left, 0), B, h, n, n, d, d, mask, rng)
    got = run_window(tsd, a, left, right)
    ref = oracle.attention(*a.as_f64(), mask, kv_lens=a.kv_lens, window=(left, right))
    assert_bf16_close(got, ref, str(case))


def test_attn_forward_window_unbounded_equals_attn_forward(tsd):
    a = synthetic.attention_inputs(2600, 2, 2, 700, 700, 64, 64, MASK_CAUSAL)
    np.testing.assert_array_equal(run_window(tsd, a, -1, -1), run_bf16(tsd, a))


def test_attn_forward_window_zero_width_returns_values(tsd):
    """A (0, 0) window leaves each query its own key: output = v_i rounded to
    bf16 (one weight of exactly 1)."""
    a = synthetic.attention_inputs(2601, 1, 2, 300, 300, 64, 64, MASK_NONE)
    got = run_window(tsd, a, 0, 0)
    np.testing.assert_array_equal(got, a.as_f64()[2])
