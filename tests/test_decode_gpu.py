"""GPU parity of attn_decode (one decoding step against a key/value cache)
against the fp64 oracle: ragged cache lengths, several new tokens at once,
more new tokens than cached rows, empty caches, garbage past the valid rows."""
import numpy as np
import pytest

import oracle
import synthetic

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


def decode_inputs(seed, B, h, n_q, n_max, d, lens):
    a = synthetic.attention_inputs(seed, B, h, n_q, n_max, d, d)
    if isinstance(lens, str):  # "ragged": seeded lengths in [0, n_max], some empty
        lens = np.random.default_rng(seed).integers(0, n_max + 1, size=B)
        lens[::7] = 0
    return a.q, a.k, a.v, (None if lens is None else np.asarray(lens, dtype=np.int32))


def run_decode(tsd, q, k, v, lens, B, h, n_q, n_max, d, poison=False):
    import torch
    qd, kd, vd = to_dev_bf16(q), to_dev_bf16(k), to_dev_bf16(v)
    if poison and lens is not None:  # rows at or past L hold NaN: they must never be used
        for b in range(B):
            kd[b, :, int(max(lens[b], 0)):] = float("nan")
            vd[b, :, int(max(lens[b], 0)):] = float("nan")
    out = torch.full((B, h, n_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    wsb = tsd.attn_decode_workspace_bytes(B, h, n_q, n_max, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    dl = to_dev_i32(lens) if lens is not None else None
    tsd.attn_decode(qd, kd, vd, out, B, h, n_q, n_max, d, d, dl, 0.0, ws, wsb)
    torch.cuda.synchronize()
    assert tsd.attn_get_device_status() == tsd.ATTN_OK
    return to_host_f64(out)


def f64(x):
    return synthetic.bf16_bits_to_f64(x)


CASES = [
    # B, h, n_q, n_max, d, lens
    (1, 1, 1, 1, 64, None),
    (2, 3, 1, 300, 64, [300, 17]),
    (4, 8, 1, 1000, 64, [1000, 513, 256, 1]),          # chunk boundaries, one-key cache
    (3, 4, 4, 777, 64, [777, 200, 3]),                 # 4 new tokens, 3 cached rows: one sees none
    (2, 4, 8, 2049, 64, [2049, 1500]),
    (2, 2, 3, 600, 128, [600, 129]),
    (2, 2, 8, 1100, 128, [9, 1100]),
    (1, 2, 2, 5000, 128, None),
    (3, 2, 2, 400, 64, [0, 400, 2]),                   # an empty cache gives zeros
    # the persistent partial kernel deals the chunks out in contiguous ranges:
    # ranges that cross batches with empty caches between them, more batches
    # than threads in its prefix sum, more chunks than CTAs, fewer than CTAs
    (7, 3, 1, 2000, 64, [2000, 0, 0, 5, 1999, 256, 257]),
    (300, 1, 1, 300, 64, "ragged"),
    (5, 16, 2, 4096, 128, [4096, 1, 4000, 129, 2222]),
    (9, 20, 1, 8192, 64, [8192, 0, 7000, 300, 8191, 0, 4097, 256, 6000]),
    # the largest cache (131072 rows: 1024 chunks, the merge's largest weight table)
    (2, 1, 8, 131072, 64, [131072, 100001]),
    (1, 1, 8, 131072, 128, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}h{}nq{}nmax{}d{}".format(*c[:5]))
def test_attn_decode_matches_oracle(tsd, case):
    B, h, n_q, n_max, d, lens = case
    q, k, v, lens = decode_inputs(3000 + sum(case[:5]), B, h, n_q, n_max, d, lens)
    got = run_decode(tsd, q, k, v, lens, B, h, n_q, n_max, d)
    ref = oracle.decode(f64(q), f64(k), f64(v), cache_lens=lens)
    assert_bf16_close(got, ref, str(case))
    if lens is not None:
        for b in range(B):
            for t in range(n_q):
                if int(lens[b]) - n_q + t < 0:
                    assert np.all(got[b, :, t] == 0.0)


def test_attn_decode_never_reads_past_the_cache_length(tsd):
    B, h, n_q, n_max, d = 3, 2, 2, 900, 64
    q, k, v, lens = decode_inputs(3100, B, h, n_q, n_max, d, [900, 300, 257])
    got = run_decode(tsd, q, k, v, lens, B, h, n_q, n_max, d, poison=True)
    ref = oracle.decode(f64(q), f64(k), f64(v), cache_lens=lens)
    assert_bf16_close(got, ref, "poisoned cache tail")


def test_attn_decode_equals_last_rows_of_causal_attention(tsd):
    """The newest n_q rows of causal attn_forward over the first L positions
    and a decoding step with cache length L agree (same bf16 inputs; both
    within the bf16 tolerance of the oracle and of each other)."""
    import torch
    B, h, n, d, n_q = 2, 4, 640, 64, 3
    a = synthetic.attention_inputs(3200, B, h, n, n, d, d, synthetic.MASK_CAUSAL)
    qd, kd, vd = (to_dev_bf16(t) for t in (a.q, a.k, a.v))
    full = torch.empty_like(qd)
    tsd.attn_forward(qd, kd, vd, full, B, h, n, n, d, d, synthetic.MASK_CAUSAL)
    got = run_decode(tsd, a.q[:, :, n - n_q:], a.k, a.v, None, B, h, n_q, n, d)
    torch.cuda.synchronize()
    assert_bf16_close(got, to_host_f64(full)[:, :, n - n_q:], "decode vs causal attention")
