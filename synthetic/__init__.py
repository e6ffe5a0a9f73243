"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws and rounds numbers; it holds none of the attention
arithmetic. Both sides of every parity check (the CUDA path and the fp64
oracle) consume exactly the arrays produced here: the CUDA path receives the
bf16 bit patterns, the oracle receives the same values widened exactly to
fp64.

Recipe (the same for every workload):
  * draws come from ``numpy.random.default_rng(seed)``; normal draws are made
    in float32 and rounded to bf16 with round-to-nearest-even;
  * the sinusoidal positional encoding of "[논문 리뷰]Attention Is All You Need"
    (kimjiil.github.io), section 3.5 Positional Encoding, uses the pair index
    i in 10000^(2i/d_model) and is added to N(0,1) activations;
  * projection weights are Glorot/Xavier-uniform, U(-a, a) with
    a = sqrt(6 / (fan_in + fan_out));
  * key-padding lengths are uniform integers in [lo, hi].
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f64", "bf16_bits_to_f32", "normal_bf16",
    "positional_encoding", "xavier_uniform_bf16", "uniform_lengths", "encoder_inputs",
    "EncoderInputs",
    "AttentionInputs", "MhaInputs", "attention_inputs", "mha_inputs",
]


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return the bits.

    Inputs must be finite (the generators never produce NaN or Inf).
    """
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) draws in float32, rounded to bf16; returns uint16 bits."""
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def positional_encoding(n_pos: int, d_model: int, start: int = 0) -> np.ndarray:
    """Sinusoidal positional encoding table [n_pos, d_model] in float64.

    PE(pos, 2i) = sin(pos / 10000^(2i/d_model)), PE(pos, 2i+1) = cos(same angle),
    with i the index of the (sin, cos) pair -- "[논문 리뷰]Attention Is All You
    Need" (kimjiil.github.io), section 3.5 Positional Encoding.
    """
    pos = np.arange(start, start + n_pos, dtype=np.float64)[:, None]
    pair = np.arange(d_model, dtype=np.int64) // 2
    angle = pos / np.power(10000.0, (2.0 * pair) / d_model)[None, :]
    pe = np.where((np.arange(d_model) % 2 == 0)[None, :], np.sin(angle), np.cos(angle))
    return pe


def xavier_uniform_bf16(rng: np.random.Generator, fan_in: int, fan_out: int) -> np.ndarray:
    """Glorot-uniform [fan_in, fan_out] matrix, rounded to bf16 (bits)."""
    a = np.sqrt(6.0 / (fan_in + fan_out))
    w = rng.uniform(-a, a, size=(fan_in, fan_out)).astype(np.float32)
    return f32_to_bf16_bits(w)


def uniform_lengths(rng: np.random.Generator, batch: int, lo: int, hi: int) -> np.ndarray:
    """Per-sequence valid lengths, uniform integers in [lo, hi] (int32)."""
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


@dataclasses.dataclass
class AttentionInputs:
    """Q/K/V for one attention call in [B, h, n, d] layout (bf16 bits or fp32)."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    B: int
    h: int
    n_q: int
    n_k: int
    d_k: int
    d_v: int
    mask_kind: int
    kv_lens: np.ndarray | None
    dtype: str  # "bf16" (uint16 bits) or "f32"

    def as_f64(self):
        if self.dtype == "bf16":
            return bf16_bits_to_f64(self.q), bf16_bits_to_f64(self.k), bf16_bits_to_f64(self.v)
        return (self.q.astype(np.float64), self.k.astype(np.float64), self.v.astype(np.float64))


@dataclasses.dataclass
class MhaInputs:
    """Activations [B, n, d_model] and projection weights (x·W convention), bf16 bits."""
    x_q: np.ndarray
    x_kv: np.ndarray
    w_q: np.ndarray
    w_k: np.ndarray
    w_v: np.ndarray
    w_o: np.ndarray
    B: int
    n_q: int
    n_k: int
    d_model: int
    h: int
    d_k: int
    d_v: int
    mask_kind: int
    kv_lens: np.ndarray | None
    self_attention: bool

    def as_f64(self):
        f = bf16_bits_to_f64
        return (f(self.x_q), f(self.x_kv), f(self.w_q), f(self.w_k), f(self.w_v), f(self.w_o))


MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING = 0, 1, 2


def attention_inputs(seed: int, B: int, h: int, n_q: int, n_k: int, d_k: int, d_v: int,
                     mask_kind: int = MASK_NONE, kv_len_range=None, dtype: str = "bf16") -> AttentionInputs:
    """Q, K, V ~ N(0,1) iid in [B, h, n, d]; optional key-padding lengths."""
    rng = np.random.default_rng(seed)
    if dtype == "bf16":
        q = normal_bf16(rng, (B, h, n_q, d_k))
        k = normal_bf16(rng, (B, h, n_k, d_k))
        v = normal_bf16(rng, (B, h, n_k, d_v))
    elif dtype == "f32":
        q = rng.standard_normal((B, h, n_q, d_k), dtype=np.float32)
        k = rng.standard_normal((B, h, n_k, d_k), dtype=np.float32)
        v = rng.standard_normal((B, h, n_k, d_v), dtype=np.float32)
    else:
        raise ValueError(dtype)
    kv_lens = None
    if mask_kind & MASK_KEY_PADDING:
        lo, hi = kv_len_range if kv_len_range is not None else (0, n_k)
        kv_lens = uniform_lengths(rng, B, lo, hi)
    return AttentionInputs(q, k, v, B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens, dtype)


def mha_inputs(seed: int, B: int, n_q: int, n_k: int, d_model: int, h: int, d_k: int, d_v: int,
               mask_kind: int = MASK_NONE, kv_len_range=None, add_pe: bool = False,
               self_attention: bool = True) -> MhaInputs:
    """Activations N(0,1) (+ sinusoidal PE when ``add_pe``), Xavier-uniform weights.

    For self-attention x_kv is x_q (n_k must equal n_q). Weight fan-out is the
    concatenated head width h*d (W_O: fan_in h*d_v, fan_out d_model).
    """
    rng = np.random.default_rng(seed)

    def act(n):
        x = rng.standard_normal((B, n, d_model), dtype=np.float32).astype(np.float64)
        if add_pe:
            x = x + positional_encoding(n, d_model)[None, :, :]
        return f32_to_bf16_bits(x.astype(np.float32))

    x_q = act(n_q)
    if self_attention:
        if n_k != n_q:
            raise ValueError("self-attention needs n_k == n_q")
        x_kv = x_q
    else:
        x_kv = act(n_k)
    w_q = xavier_uniform_bf16(rng, d_model, h * d_k)
    w_k = xavier_uniform_bf16(rng, d_model, h * d_k)
    w_v = xavier_uniform_bf16(rng, d_model, h * d_v)
    w_o = xavier_uniform_bf16(rng, h * d_v, d_model)
    kv_lens = None
    if mask_kind & MASK_KEY_PADDING:
        lo, hi = kv_len_range if kv_len_range is not None else (0, n_k)
        kv_lens = uniform_lengths(rng, B, lo, hi)
    return MhaInputs(x_q, x_kv, w_q, w_k, w_v, w_o, B, n_q, n_k, d_model, h, d_k, d_v,
                     mask_kind, kv_lens, self_attention)


@dataclasses.dataclass
class EncoderInputs:
    """One encoder layer's inputs (bf16 bits): the attention part as MhaInputs
    (self-attention), LayerNorm gains/offsets and the FFN weights/biases."""
    mha: MhaInputs
    ln1_gamma: np.ndarray
    ln1_beta: np.ndarray
    w_1: np.ndarray
    b_1: np.ndarray
    w_2: np.ndarray
    b_2: np.ndarray
    ln2_gamma: np.ndarray
    ln2_beta: np.ndarray
    d_ff: int

    def params_f64(self):
        return [bf16_bits_to_f64(a) for a in (self.ln1_gamma, self.ln1_beta, self.w_1, self.b_1,
                                              self.w_2, self.b_2, self.ln2_gamma, self.ln2_beta)]


def encoder_inputs(seed: int, B: int, n: int, d_model: int, h: int, d_ff: int,
                   mask_kind: int = MASK_NONE, kv_len_range=None, add_pe: bool = False) -> EncoderInputs:
    """x ~ N(0,1) (+ PE), Xavier-uniform W_Q/K/V/O and W_1/W_2; biases ~ U(-0.1, 0.1);
    LayerNorm gains ~ 1 + U(-0.1, 0.1) and offsets ~ U(-0.1, 0.1) (the pages give
    no initialisation for these)."""
    d_k = d_model // h
    m = mha_inputs(seed, B, n, n, d_model, h, d_k, d_k, mask_kind, kv_len_range, add_pe=add_pe)
    rng = np.random.default_rng(seed + 7919)

    def small(k, centre=0.0):
        return f32_to_bf16_bits((centre + rng.uniform(-0.1, 0.1, size=k)).astype(np.float32))

    return EncoderInputs(m, small(d_model, 1.0), small(d_model),
                         xavier_uniform_bf16(rng, d_model, d_ff), small(d_ff),
                         xavier_uniform_bf16(rng, d_ff, d_model), small(d_model),
                         small(d_model, 1.0), small(d_model), d_ff)
