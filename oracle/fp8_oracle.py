"""Float64 CPU oracle for the FP8-weight variant of the MoE layer.

TEST INFRASTRUCTURE.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  It shares no code with the CUDA library.

The pages mention FP8 only as deployment work (paper-graph-ui summary,
"Inference and Deployment Infrastructure": FP8 through TensorRT-LLM; the
closing discussion of quantisation as an opportunity).  They define no
scheme, so the scheme below is this library's, written out plainly:

  * e4m3 numbers (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
    infinities; S.1111.111 is NaN; largest finite magnitude 448; subnormals
    m/8 * 2^-6).  Rounding to e4m3 is to the nearest value, ties to the even
    code, and magnitudes beyond 448 saturate to 448.
  * expert weights: one fp32 scale per output column of each expert from
    a = max_k |W[k, n]|: the scale s = a / 448 and its inverse u = 448 / a
    (both 1 where the column is all zero; a nonzero a below 2^-100 counts
    as 2^-100, so that u stays finite).  Codes q = e4m3(W * u), stored
    K-contiguous ([E, N, K]); W is dequantised as e4m3(q) * s.  Scaling by
    the inverse, one division per column and a product per element, is the
    usual form of an amax-scaled FP8 cast.
  * activations: one fp32 scale per token row in the same way (x for the
    gate/up projection; the SwiGLU output H, rounded to bf16 first, for the
    down projection).
  * the divisions giving s and u and the product that decides a code are
    float32 operations, as in the CUDA kernels (where floating point decides
    an integer both sides take that decision in the same precision);
    everything after decoding is float64.

The layer is then the plain definition of ``moe_oracle.moe_layer`` with the
dequantised operands: y = sum_i G(x)_i E_i(x), G from the unquantised router.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as M

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


# ---------------------------------------------------------------------------
# e4m3 numbers
# ---------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8) as float64; NaN for S.1111.111."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = (m / 8.0) * 2.0 ** -6
    nrm = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    v = np.where(e == 0, sub, nrm)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return sign * v


# the 127 non-negative finite codes (0x00..0x7E) in increasing value
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(v) -> np.ndarray:
    """Nearest e4m3 code of each finite value (ties to the even code),
    saturating beyond 448.  Works on the exact value given (float32 or
    float64 input)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")        # first grid value >= a
    hi = np.clip(hi, 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((_POS_CODES[lo] & 1) == 0))
    code = np.where(pick_lo, _POS_CODES[lo], _POS_CODES[hi]).astype(np.uint8)
    neg = (v < 0) | ((v == 0) & np.signbit(v))
    return np.where(neg, code | 0x80, code).astype(np.uint8)


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu", torch.float32).numpy()
    return np.asarray(a, dtype=np.float32)


AMAX_FLOOR = np.float32(2.0 ** -100)


def _amax_used(absmax) -> np.ndarray:
    """The maximum magnitude the scale is taken from: 448 where it is 0 (so
    that s = u = 1), at least 2^-100 otherwise."""
    absmax = np.asarray(absmax, dtype=np.float32)
    return np.where(absmax > 0, np.maximum(absmax, AMAX_FLOOR), np.float32(E4M3_MAX)).astype(np.float32)


def scale_of(absmax) -> np.ndarray:
    """fp32 dequantisation scale absmax / 448 (a float32 division); 1 where
    absmax is 0."""
    return (_amax_used(absmax) / np.float32(E4M3_MAX)).astype(np.float32)


def inverse_scale_of(absmax) -> np.ndarray:
    """fp32 quantisation factor 448 / absmax (a float32 division); 1 where
    absmax is 0."""
    return (np.float32(E4M3_MAX) / _amax_used(absmax)).astype(np.float32)


def quantize_weight_columns(W):
    """Expert bank W [E, K, N] -> (codes [E, N, K] uint8, scales [E, N] fp32):
    one scale per output column n, codes stored K-contiguous."""
    W32 = _f32(W)
    a = np.abs(W32).max(axis=1)                                 # [E, N]
    s, u = scale_of(a), inverse_scale_of(a)
    prod = (W32 * u[:, None, :]).astype(np.float32)             # float32 product
    return np.ascontiguousarray(e4m3_encode(prod).transpose(0, 2, 1)), s


def dequantize_weight_columns(codes, scales) -> np.ndarray:
    """(codes [E, N, K], scales [E, N]) -> W [E, K, N] float64."""
    return (e4m3_decode(codes) * np.asarray(scales, np.float64)[:, :, None]).transpose(0, 2, 1)


def quantize_rows(X):
    """Rows X [M, K] -> (codes [M, K] uint8, scales [M] fp32), one scale per row."""
    X32 = _f32(X)
    a = np.abs(X32).max(axis=1)
    s, u = scale_of(a), inverse_scale_of(a)
    return e4m3_encode((X32 * u[:, None]).astype(np.float32)), s


def dequantize_rows(codes, scales) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scales, np.float64)[:, None]


def round_bf16(v) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even (library cast), as float64."""
    import torch
    return torch.from_numpy(np.asarray(v, dtype=np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------
def expert_fp8(xd, W1d, W3d, W2d) -> np.ndarray:
    """One expert on dequantised rows xd: H = SiLU(xd W1) (.) (xd W3) in float64,
    rounded to bf16, quantised per row to e4m3, dequantised, then H W2."""
    H = M.silu(xd @ W1d) * (xd @ W3d)
    Hq, hs = quantize_rows(round_bf16(H))
    return dequantize_rows(Hq, hs) @ W2d


def moe_layer_fp8(x, Wg, W1q, s1, W3q, s3, W2q, s2, K: int) -> M.LayerResult:
    """y = sum_i G(x)_i E_i(x) with e4m3 expert weights (codes [E, N, K] and
    per-column scales) and e4m3 activations, routed as moe_oracle.gating."""
    x64 = M.f64(x)
    g = M.gating(x64, Wg, K)
    xq, xs = quantize_rows(x)
    xd = dequantize_rows(xq, xs)
    W1d = dequantize_weight_columns(W1q, s1)
    W3d = dequantize_weight_columns(W3q, s3)
    W2d = dequantize_weight_columns(W2q, s2)
    E = g.G.shape[1]
    y = np.zeros((x64.shape[0], W2d.shape[2]))
    for e in range(E):
        rows = np.nonzero((g.idx == e).any(axis=1))[0]
        if rows.size == 0:
            continue
        y[rows] += g.G[rows, e][:, None] * expert_fp8(xd[rows], W1d[e], W3d[e], W2d[e])
    return M.LayerResult(y, g)
