"""Pins for the seeded input generator (CPU only)."""
import json
import os

import numpy as np
import pytest

import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_positional_encoding_matches_pages_worked_values():
    with open(os.path.join(GOLDEN, "positional_encoding_d4.json"), encoding="utf-8") as f:
        g = json.load(f)
    pe = synthetic.positional_encoding(3, g["d_model"])
    for pos, row in g["six_decimals"].items():
        np.testing.assert_allclose(pe[int(pos)], row, atol=g["tolerance_six"], rtol=0)
    for pos, row in g["two_decimals"].items():
        np.testing.assert_allclose(pe[int(pos)], row, atol=g["tolerance_two"], rtol=0)


def test_positional_encoding_offset_is_a_rotation():
    """PE_{pos+k} = M(k) PE_pos with M(k) block-diagonal 2x2 rotations
    ("[논문 리뷰]Attention Is All You Need", section 3.5, the rotation proof)."""
    d = 512
    pe = synthetic.positional_encoding(200, d)
    omega = np.power(10000.0, -(2.0 * np.arange(d // 2)) / d)
    for k in (1, 7, 63):
        c, s = np.cos(omega * k), np.sin(omega * k)
        sin_pos, cos_pos = pe[:-k, 0::2], pe[:-k, 1::2]
        np.testing.assert_allclose(pe[k:, 0::2], c * sin_pos + s * cos_pos, atol=1e-12)
        np.testing.assert_allclose(pe[k:, 1::2], -s * sin_pos + c * cos_pos, atol=1e-12)


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        # exact ties: low 16 bits = 0x8000 must round to even
                        (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
                        np.array([0.0, -0.0, 1e-40, -3.0e38], dtype=np.float32)])
    ours = synthetic.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    # widening is exact
    back = synthetic.bf16_bits_to_f64(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_generators_are_seeded_and_shaped():
    a = synthetic.attention_inputs(1004, 2, 3, 17, 19, 64, 64, synthetic.MASK_KEY_PADDING, (4, 19))
    b = synthetic.attention_inputs(1004, 2, 3, 17, 19, 64, 64, synthetic.MASK_KEY_PADDING, (4, 19))
    np.testing.assert_array_equal(a.q, b.q)
    np.testing.assert_array_equal(a.kv_lens, b.kv_lens)
    assert a.q.shape == (2, 3, 17, 64) and a.k.shape == (2, 3, 19, 64) and a.q.dtype == np.uint16
    assert np.all((a.kv_lens >= 4) & (a.kv_lens <= 19))
    q, _, _ = a.as_f64()
    assert abs(q.mean()) < 0.05 and abs(q.std() - 1.0) < 0.05


def test_xavier_uniform_bound_and_variance():
    rng = np.random.default_rng(5)
    w = synthetic.bf16_bits_to_f64(synthetic.xavier_uniform_bf16(rng, 512, 512))
    a = np.sqrt(6.0 / 1024)
    assert np.abs(w).max() <= a * (1 + 2 ** -8)
    assert np.var(w) == pytest.approx(a * a / 3, rel=0.02)


def test_mha_inputs_add_positional_encoding():
    m0 = synthetic.mha_inputs(1001, 2, 8, 8, 32, 4, 8, 8, add_pe=False)
    m1 = synthetic.mha_inputs(1001, 2, 8, 8, 32, 4, 8, 8, add_pe=True)
    x0 = synthetic.bf16_bits_to_f64(m0.x_q)
    x1 = synthetic.bf16_bits_to_f64(m1.x_q)
    np.testing.assert_allclose(x1 - x0, np.broadcast_to(synthetic.positional_encoding(8, 32), x0.shape),
                               atol=0.05)
    assert m1.x_kv is m1.x_q
