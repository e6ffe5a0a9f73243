"""GPU parity at the full sizes of the Transformer-big and long-context
workloads, in the launch configuration bench.py times (one attn_forward /
attn_forward_window over the whole batch). Rows are independent, so the
oracle computes a seeded random subset of query rows one by one -- at least
1024 per (batch, head), plus the first and the last row -- and the kernel's
rows are compared element by element; at n = 1024 every row is checked."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import MASK_CAUSAL, MASK_NONE

from gpu_util import assert_bf16_close, to_dev_bf16, to_host_f64

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


def sample_rows(rng, n, k=1024):
    if n <= k + 2:
        return np.arange(n, dtype=np.int32)
    mid = rng.choice(np.arange(1, n - 1), size=k, replace=False)
    return np.sort(np.concatenate([[0, n - 1], mid])).astype(np.int32)


def run_and_compare(tsd, B, h, n, d, causal, seed, window=None):
    import torch
    a = synthetic.attention_inputs(seed, B, h, n, n, d, d, MASK_CAUSAL if causal else MASK_NONE)
    q, k, v = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    out = torch.full((B, h, n, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    if window is None:
        tsd.attn_forward(q, k, v, out, B, h, n, n, d, d, a.mask_kind, None, 0.0)
    else:
        tsd.attn_forward_window(q, k, v, out, B, h, n, n, d, d, window[0], window[1],
                                a.mask_kind, None, 0.0)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    rng = np.random.default_rng(seed + 1)
    qf, kf, vf = a.as_f64()[:3]  # the bf16 inputs' exact values
    got_all, ref_all = [], []
    for b in range(B):
        for hh in range(h):
            rows = sample_rows(rng, n)
            idx = torch.from_numpy(rows.astype(np.int64)).cuda()
            got_all.append(to_host_f64(out[b, hh].index_select(0, idx)))
            ref_all.append(oracle.attention_rows(qf[b, hh][rows], rows, kf[b, hh], vf[b, hh],
                                                 causal=causal, window=window))
    assert_bf16_close(np.stack(got_all), np.stack(ref_all),
                      f"B={B} h={h} n={n} d={d} causal={causal} window={window}")


@pytest.mark.parametrize("causal", [False, True])
def test_transformer_big_self_attention_every_row(tsd, causal):
    """Transformer-big self-attention, B=8, h=16, n=1024, d=64."""
    run_and_compare(tsd, 8, 16, 1024, 64, causal, 1003)


@pytest.mark.parametrize("B,n,d,causal", [
    (4, 4096, 64, False),    # the long-context configuration bench.py reports
    (4, 4096, 64, True),
    (2, 8192, 128, False),
    (2, 8192, 128, True),
    (1, 16384, 64, True),
    (1, 8200, 64, True),     # causal past 8192 rows (the unmasked-twin instance), ragged tail
    (4, 16384, 64, False),   # the largest d = 64 point of the sweep
    (1, 2048, 128, False),
])
def test_long_context_sweep_sampled_rows(tsd, B, n, d, causal):
    run_and_compare(tsd, B, 16, n, d, causal, 1004 + n + d)


def test_restricted_window_full_size_sampled_rows(tsd):
    """Restricted self-attention, B=4, h=16, n=16384, d=64, keys within +-256."""
    run_and_compare(tsd, 4, 16, 16384, 64, False, 1005, window=(256, 256))


@pytest.mark.parametrize("n_q", [1, 4])
def test_decode_full_size(tsd, n_q):
    """One decoding step at the size bench.py times: B=16, h=16, d=64, an
    8192-row cache with lengths uniform in [4096, 8192]; every output."""
    import torch
    from gpu_util import to_dev_i32
    B, h, n_max, d = 16, 16, 8192, 64
    rng = np.random.default_rng(1006)
    lens = synthetic.uniform_lengths(rng, B, 4096, 8192)
    a = synthetic.attention_inputs(1006, B, h, n_q, n_max, d, d)
    out = torch.full((B, h, n_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.attn_decode_workspace_bytes(B, h, n_q, n_max, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    tsd.attn_decode(to_dev_bf16(a.q), to_dev_bf16(a.k), to_dev_bf16(a.v), out, B, h, n_q, n_max, d,
                    d, to_dev_i32(lens), 0.0, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    ref = oracle.decode(*a.as_f64()[:3], cache_lens=lens)
    assert_bf16_close(to_host_f64(out), ref, f"decode n_q={n_q}")
