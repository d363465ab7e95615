"""Pins for the FP8 part of the oracle (oracle/fp8_oracle.py).

| part                      | pinned by                                                     |
|---------------------------|---------------------------------------------------------------|
| e4m3 decode               | closed forms of the format (bias 7, subnormals m/8 * 2^-6,     |
|                           | largest finite 448, NaN code); torch.float8_e4m3fn decode of   |
|                           | all 256 codes                                                  |
| e4m3 encode               | exact round trip of every finite code; designed ties (to the  |
|                           | even code) at normal and subnormal spacing; saturation;        |
|                           | torch.float8_e4m3fn encode of in-range values                  |
| per-column / per-row      | the largest magnitude maps to +-448 exactly; dequantisation    |
| quantisation              | error within half a step of the format                         |
| FP8 layer                 | error against the float64 bf16-weight layer within the bound   |
|                           | fp8 rounding allows; exact zero with W3 = 0; exact linearity   |
|                           | in the down-projection scales                                  |

Planted mistakes at the end check that the pins catch plausible errors.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_oracle as F8
import workloads as W


def test_decode_closed_forms():
    d = F8.e4m3_decode
    assert d(0x00) == 0.0 and d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6 and d(0x38) == 1.0 and d(0x3F) == 1.875 and d(0x40) == 2.0
    assert d(0x7E) == 448.0 and d(0xB8) == -1.0 and d(0xFE) == -448.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert np.signbit(d(0x80))


def test_decode_matches_torch_float8_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])


def test_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(F8.e4m3_encode(F8.e4m3_decode(codes)), codes)


@pytest.mark.parametrize("v,code", [
    (1.0625, 0x38),        # halfway 1.0 (0x38) / 1.125 (0x39): even code 0x38
    (1.1875, 0x3A),        # halfway 1.125 (0x39) / 1.25 (0x3A): even code 0x3A
    (1.0626, 0x39),        # just above the tie: the upper neighbour
    (2.0 ** -10, 0x00),    # halfway 0 / 2^-9: even code 0
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 (0x01) / 2^-8 (0x02): even 0x02
    (-1.0625, 0xB8),
    (464.0, 0x7E),         # beyond 448 saturates
    (1e30, 0x7E),
    (-1e30, 0xFE),
])
def test_encode_ties_and_saturation(v, code):
    assert int(F8.e4m3_encode(np.float64(v))) == code


def test_encode_matches_torch_float8_in_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01,
                        rng.uniform(-448, 448, 5000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F8.e4m3_encode(v), ref)


def test_weight_columns_scale_and_error():
    Wg, W1, W3, W2 = W.mixtral_weights(64, 96, 3, seed=5)
    q, s = F8.quantize_weight_columns(W1)
    assert q.shape == (3, 96, 64) and s.shape == (3, 96)
    W1f = W1.float().numpy().astype(np.float64)
    # the largest magnitude of every column maps to +-448 exactly
    amax_idx = np.abs(W1f).argmax(axis=1)                          # [E, N]
    codes_at_max = np.take_along_axis(q.transpose(0, 2, 1), amax_idx[:, None, :], axis=1)[:, 0, :]
    assert np.all((codes_at_max & 0x7F) == 0x7E)
    back = F8.dequantize_weight_columns(q, s)
    # half a step: relative 2^-4 for normals, absolute 2^-10 * s for subnormals
    bound = np.maximum(np.abs(W1f) * 2.0 ** -4, 2.0 ** -10 * s[:, None, :].astype(np.float64))
    assert np.all(np.abs(back - W1f) <= bound * (1 + 1e-12))


def test_rows_scale_and_error():
    x = W.rms_rows(50, 64, 3, "cpu", torch.bfloat16)
    q, s = F8.quantize_rows(x)
    xf = x.float().numpy().astype(np.float64)
    back = F8.dequantize_rows(q, s)
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * s[:, None].astype(np.float64))
    assert np.all(np.abs(back - xf) <= bound * (1 + 1e-12))
    assert np.all((q[np.arange(50), np.abs(xf).argmax(axis=1)] & 0x7F) == 0x7E)


def _fp8_inputs(T=40, d=64, f=96, E=4, K=2, seed=11):
    Wg, W1, W3, W2 = W.mixtral_weights(d, f, E, seed=seed)
    x = W.rms_rows(T, d, seed + 1, "cpu", torch.bfloat16)
    q1, s1 = F8.quantize_weight_columns(W1)
    q3, s3 = F8.quantize_weight_columns(W3)
    q2, s2 = F8.quantize_weight_columns(W2)
    return x, Wg, (W1, W3, W2), (q1, s1, q3, s3, q2, s2)


def test_fp8_layer_close_to_bf16_layer():
    """Three e4m3 roundings (weights, x, H) each move an operand by at most
    2^-4 relative; the layer output moves by far less than that."""
    x, Wg, (W1, W3, W2), qs = _fp8_inputs()
    ref = oracle.moe_layer(x, Wg, W1, W3, W2, 2).y
    got = F8.moe_layer_fp8(x, Wg, *qs, 2).y
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert 1e-4 < err < 0.08, err


def test_fp8_layer_zero_and_exactly_linear_in_down_scales():
    """Exact properties of the definition: with W3 = 0 the SwiGLU output and
    the layer are exactly 0; doubling every W2 column scale (codes unchanged)
    doubles y exactly, since the scale multiplies an exact dequantised value."""
    d, f, E = 16, 32, 1
    x = torch.zeros((3, d), dtype=torch.bfloat16)
    x[0, 2] = 1.0; x[1, 5] = -2.0; x[2, 7] = 0.5
    Wg = torch.zeros((d, E), dtype=torch.bfloat16)
    Wg_, W1, W3, W2 = W.mixtral_weights(d, f, E, seed=3)
    W3z = torch.zeros_like(W3)
    q1, s1 = F8.quantize_weight_columns(W1)
    q3, s3 = F8.quantize_weight_columns(W3z)
    q2, s2 = F8.quantize_weight_columns(W2)
    y0 = F8.moe_layer_fp8(x, Wg, q1, s1, q3, s3, q2, s2, 1).y
    assert np.all(y0 == 0.0)
    # doubling every W2 scale (codes unchanged) doubles y exactly
    q3b, s3b = F8.quantize_weight_columns(W3)
    y1 = F8.moe_layer_fp8(x, Wg, q1, s1, q3b, s3b, q2, s2, 1).y
    y2 = F8.moe_layer_fp8(x, Wg, q1, s1, q3b, s3b, q2, s2 * np.float32(2), 1).y
    assert np.array_equal(y2, 2 * y1) and np.abs(y1).max() > 0


# ---------------------------------------------------------------------------
# planted mistakes (on the CPU) must be caught
# ---------------------------------------------------------------------------
def _encode_truncating(v):
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), F8.E4M3_MAX)
    idx = np.searchsorted(F8._POS_VALUES, a, side="right") - 1
    code = F8._POS_CODES[np.clip(idx, 0, 126)]
    return np.where(v < 0, code | 0x80, code).astype(np.uint8)


def _encode_ties_up(v):
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), F8.E4M3_MAX)
    hi = np.clip(np.searchsorted(F8._POS_VALUES, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    pick_lo = (a - F8._POS_VALUES[lo]) < (F8._POS_VALUES[hi] - a)
    code = np.where(pick_lo, F8._POS_CODES[lo], F8._POS_CODES[hi])
    return np.where(v < 0, code | 0x80, code).astype(np.uint8)


def _decode_bias_8(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF; m = c & 7
    v = np.where(e == 0, (m / 8.0) * 2.0 ** -7, (1 + m / 8.0) * np.exp2(e - 8.0))
    return np.where(c & 0x80, -v, v)


def _expert_no_h_quant(xd, W1d, W3d, W2d):
    return (oracle.silu(xd @ W1d) * (xd @ W3d)) @ W2d * 1.5       # also a wrong constant


PLANTS = {
    "encode_truncates": ("e4m3_encode", _encode_truncating),
    "encode_ties_up": ("e4m3_encode", _encode_ties_up),
    "decode_bias_8": ("e4m3_decode", _decode_bias_8),
    "expert_drops_h_quant_and_scales": ("expert_fp8", _expert_no_h_quant),
}


@pytest.mark.parametrize("name", sorted(PLANTS))
def test_planted_fp8_mistake_is_caught(name, monkeypatch):
    attr, fn = PLANTS[name]
    monkeypatch.setattr(F8, attr, fn)
    checks = [test_decode_closed_forms, test_decode_matches_torch_float8_all_codes,
              test_encode_round_trips_every_finite_code, test_encode_matches_torch_float8_in_range,
              test_weight_columns_scale_and_error, test_rows_scale_and_error, test_fp8_layer_close_to_bf16_layer,
              test_fp8_layer_zero_and_exactly_linear_in_down_scales]
    ties = [(1.0625, 0x38), (1.1875, 0x3A), (2.0 ** -10, 0x00), (464.0, 0x7E)]
    caught = 0
    for chk in checks:
        try:
            chk()
        except AssertionError:
            caught += 1
    for v, code in ties:
        try:
            test_encode_ties_and_saturation(v, code)
        except AssertionError:
            caught += 1
    assert caught > 0, name


def test_column_scales_lose_nothing_to_block_scales_on_these_weights():
    """Why one scale per output column rather than per 128 x 128 block: e4m3
    keeps three mantissa bits at every magnitude down to 2^-6 of its maximum,
    so a finer scale helps only elements that a coarse one pushes below that
    range (outliers).  On the Mixtral-shaped N(0, 0.02^2) weights both give
    the same error, element-wise and through a product; column scales also
    factor out of the contraction, so the kernels apply them in the epilogue."""
    d, f = 1024, 512
    Wt = W.randn((d, f), 0.02, W._seed(W.BASE_SEED, "W1", 0)).to(torch.bfloat16).double().numpy()

    def quant(block, scale):
        return F8.e4m3_decode(F8.e4m3_encode((block / scale).astype(np.float32))) * scale

    col = quant(Wt, np.abs(Wt).max(axis=0, keepdims=True) / F8.E4M3_MAX)
    blk = np.empty_like(Wt)
    for i in range(0, d, 128):
        for j in range(0, f, 128):
            b = Wt[i:i + 128, j:j + 128]
            blk[i:i + 128, j:j + 128] = quant(b, np.abs(b).max() / F8.E4M3_MAX)
    rms = lambda q: np.sqrt(((q - Wt) ** 2).mean() / (Wt ** 2).mean())
    assert abs(rms(col) - rms(blk)) <= 0.01 * rms(blk)
    x = W.rms_rows(32, d, 7, "cpu", torch.bfloat16).double().numpy()
    ref = x @ Wt
    rel = lambda q: np.linalg.norm(x @ q - ref) / np.linalg.norm(ref)
    assert abs(rel(col) - rel(blk)) <= 0.02 * rel(blk)


def test_zero_and_tiny_rows():
    """A zero row gets scale 1 and zero codes; a row whose largest magnitude
    is below 2^-100 is scaled from 2^-100, so its inverse scale stays finite
    and every code is a number (0 * an infinite inverse would give NaN)."""
    x = np.zeros((3, 16), dtype=np.float32)
    x[1, :4] = [1e-38, -3e-39, 0.0, 5e-39]          # tiny: scaled from the 2^-100 floor
    x[2, :4] = [2.0 ** -90, 0.0, -(2.0 ** -91), 2.0 ** -92]  # above the floor
    q, s = F8.quantize_rows(x)
    assert s[0] == 1.0 and np.all(q[0] == 0)
    assert s[1] == np.float32(2.0 ** -100) / np.float32(448.0)
    assert np.all((q & 0x7F) != 0x7F)                 # no NaN code
    assert np.all(q[1] & 0x7F == 0)                   # 1e-38 * 448 * 2^100 is below half the least e4m3 step
    # above the floor: the largest magnitude maps to 448 and the rest follow within half a step
    assert (q[2, 0] & 0x7F) == 0x7E
    back = F8.dequantize_rows(q, s)
    bound = np.maximum(np.abs(x[2].astype(np.float64)) * 2.0 ** -4, 2.0 ** -10 * float(s[2]))
    assert np.all(np.abs(back[2] - x[2]) <= bound * (1 + 1e-12))
