"""Plain CPU oracle for the affine-packed dequantise-into-matmul path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import or call this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA library; both sides only share the seeded input
generators, which hold none of the method's arithmetic.

Every step is written the slow, obvious way, in the order the method states it,
so that a reader can check it against the sources by eye:

  1. affine quantise (per row, per group of ``group_size`` along K)
  2. pack codes low-bits-first into uint32 words
  3. bit-unpack
  4. dequantise exactly (w = q*scale + bias in float64, asserted exact)
  5. matmul in float64 (one library matmul), plus the sum of |x*w| that the
     output tolerance is relative to

Sources (web pages on the method; cited by page title and section):
  [mlxcel-570 Context]  "epic: realize low-precision / quantized performance on
      the OpenXLA (IREE) backend", section Context: MLX 4/8-bit weights stay
      resident packed as a ui32 payload with f16 scales and biases, and are
      dequantised in the graph.
  [mlxcel-574 in-tree]  "track(upstream-iree): fused dequant->matmul for the
      packed int8 bandwidth win", section "What is already in-tree": bit-unpack,
      then q*scale + bias; the reconstruction inside the graph matches a host
      dequantisation bit for bit; bf16 scales/biases are accepted.
  [mlxcel-574 blocker]  same page, section "The blocker (measured)": the
      reconstructed weight must not be materialised; the matmul consumes it.
  [executorch-17187]    "Metal backend: import qmv_impl from MLX": the M=1
      matrix-vector case with N not a multiple of 4.

Readings taken where the pages are silent (each is listed in the design notes):
  * quantisation recipe: scale = (max - min) / (2^bits - 1), bias = min, both
    computed in float32 then rounded (ties-to-even) to the scale dtype; codes
    are computed from the STORED (rounded) scale and bias, in float32:
    q = clamp(round_half_even((w - bias) / scale), 0, 2^bits - 1);
  * a group whose stored scale is 0 gets q = 0 everywhere (w_hat = bias);
  * "low-bits-first": code k sits at bits [bits*(k mod p), bits*(k mod p)+bits)
    of word k // p, p = 32 / bits;
  * the reconstruction in precision P is one correctly rounded step of the
    exact value: RNE_P(q*scale + bias).

Parity: every function here is pinned by tests/test_oracle.py against closed
forms, brute force with exact rational arithmetic, hand-derived fixtures in
tests/golden/, and independent library conversions.
"""

from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# Floating-point formats: (significand bits incl. the implicit one,
# exponent of the smallest normal, exponent of the largest binade).
# --------------------------------------------------------------------------
FORMATS = {
    "f32": (24, -126, 127),
    "f16": (11, -14, 15),
    "bf16": (8, -126, 127),
}

SUPPORTED_BITS = (4, 8)
SUPPORTED_GROUPS = (32, 64, 128)


def round_to_format(v, fmt: str) -> np.ndarray:
    """Round float64 values to the nearest value of ``fmt`` (ties to even).

    Returns float64 values that are exactly representable in ``fmt``.  One
    rounding step straight from the float64 value (no intermediate format).
    Overflow goes to +-inf under round-to-nearest.  Subnormals are kept.
    """
    p, emin, emax = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    finite = np.isfinite(v) & (v != 0)
    x = v[finite]
    _, e = np.frexp(x)  # x = m * 2**e with 0.5 <= |m| < 1, so x in [2**(e-1), 2**e)
    # unit in the last place of the binade holding x; subnormals share the
    # smallest normal binade's unit
    ulp_exp = np.maximum(e - p, emin - p + 1)
    r = np.ldexp(np.rint(np.ldexp(x, -ulp_exp)), ulp_exp)
    max_finite = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def encode_bits(v, fmt: str) -> np.ndarray:
    """Bit pattern of float64 values that are exactly representable in ``fmt``.

    f32 -> uint32, f16 -> uint16, bf16 -> uint16.  Raises if a value is not
    representable (so a caller can never encode an unrounded value).
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.array_equal(round_to_format(v, fmt), v, equal_nan=True):
        raise ValueError(f"value not representable in {fmt}")
    if fmt == "f32":
        return v.astype(np.float32).view(np.uint32)
    if fmt == "f16":
        return v.astype(np.float16).view(np.uint16)
    if fmt == "bf16":
        # a bf16 value is an f32 value whose low 16 bits are zero
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    raise KeyError(fmt)


def decode_bits(bits, fmt: str) -> np.ndarray:
    """Inverse of :func:`encode_bits`: bit patterns to float64 values."""
    bits = np.asarray(bits)
    if fmt == "f32":
        return bits.astype(np.uint32).view(np.float32).astype(np.float64)
    if fmt == "f16":
        return bits.astype(np.uint16).view(np.float16).astype(np.float64)
    if fmt == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise KeyError(fmt)


# --------------------------------------------------------------------------
# 1. Affine quantisation
# --------------------------------------------------------------------------
def quantize_affine(w, bits: int, group_size: int, sdtype: str):
    """Quantise float32 weights W[N, K] per group of ``group_size`` along K.

    Follows the MLX affine format of [mlxcel-570 Context]: per (row, group)
      mn, mx   = min and max of the group                      (exact)
      scale32  = (mx - mn) / (2^bits - 1)                       (float32 ops)
      scale    = RNE_sdtype(scale32),  bias = RNE_sdtype(mn)    (stored)
      q        = clamp(rint((w - bias) / scale), 0, 2^bits - 1) (float32 ops,
                 on the stored values; ties to even)
    A group whose stored scale is 0 gets q = 0.

    Returns (codes uint8/uint16 [N, K], scale float64 [N, K/g], bias float64
    [N, K/g]); scale and bias hold values exactly representable in sdtype.
    """
    w = np.asarray(w)
    if w.dtype != np.float32:
        raise TypeError("weights must be float32")
    if bits not in SUPPORTED_BITS or group_size not in SUPPORTED_GROUPS:
        raise ValueError("unsupported bits or group size")
    n_rows, k = w.shape
    if k % group_size:
        raise ValueError("K must be a multiple of group_size")
    if not np.all(np.isfinite(w)):
        raise ValueError("weights must be finite")
    qmax = (1 << bits) - 1
    wg = w.reshape(n_rows, k // group_size, group_size)
    mn = wg.min(axis=2)
    mx = wg.max(axis=2)
    scale32 = (mx - mn) / np.float32(qmax)  # float32 subtract and divide
    scale = round_to_format(scale32.astype(np.float64), sdtype)
    bias = round_to_format(mn.astype(np.float64), sdtype)
    if not (np.all(np.isfinite(scale)) and np.all(np.isfinite(bias))):
        raise ValueError("scale or bias overflows the scale dtype")
    s32 = scale.astype(np.float32)[..., None]
    b32 = bias.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (wg - b32) / s32  # float32 subtract, float32 divide
    t = np.where(s32 == 0, np.float32(0), t)
    q = np.clip(np.rint(t), 0, qmax)
    codes = q.astype(np.uint16 if bits > 8 else np.uint8).reshape(n_rows, k)
    return codes, scale, bias


# --------------------------------------------------------------------------
# 2./3. Packing and bit-unpacking (low bits first)
# --------------------------------------------------------------------------
def pack(codes, bits: int) -> np.ndarray:
    """Pack codes[N, K] into uint32 words[N, K*bits/32], low bits first.

    Code k of a row lands at bits [bits*(k mod p), bits*(k mod p) + bits) of
    word k // p, with p = 32 / bits ([mlxcel-570 Context]: ui32 payload).
    """
    codes = np.asarray(codes).astype(np.uint32)
    n_rows, k = codes.shape
    per_word = 32 // bits
    if k % per_word:
        raise ValueError("K must fill whole words")
    if np.any(codes >> bits):
        raise ValueError("code out of range")
    words = np.zeros((n_rows, k // per_word), dtype=np.uint32)
    for j in range(per_word):
        words |= codes[:, j::per_word] << np.uint32(bits * j)
    return words


def unpack(words, bits: int, k: int) -> np.ndarray:
    """Bit-unpack words[N, K*bits/32] back to codes[N, K] ([mlxcel-574 in-tree])."""
    words = np.asarray(words, dtype=np.uint32)
    per_word = 32 // bits
    if words.shape[1] * per_word != k:
        raise ValueError("word count does not match K")
    mask = np.uint32((1 << bits) - 1)
    codes = np.empty((words.shape[0], k), dtype=np.uint32)
    for j in range(per_word):
        codes[:, j::per_word] = (words >> np.uint32(bits * j)) & mask
    return codes


# --------------------------------------------------------------------------
# 4. Dequantisation
# --------------------------------------------------------------------------
def _two_sum_error(a, b):
    """Knuth's TwoSum: the rounding error of fl(a + b), exactly."""
    s = a + b
    bp = s - a
    ap = s - bp
    return (a - ap) + (b - bp)


def dequant_exact(codes, scale, bias, group_size: int) -> np.ndarray:
    """Exact reconstruction w_hat = q*scale + bias in float64 ([mlxcel-574 in-tree]).

    q has at most 8 significant bits and scale at most 11, so q*scale is exact
    in float64; the sum is asserted exact with TwoSum (a non-zero rounding
    error raises instead of returning an inexact value).
    """
    q = np.asarray(codes, dtype=np.float64)
    s = np.repeat(np.asarray(scale, dtype=np.float64), group_size, axis=1)
    b = np.repeat(np.asarray(bias, dtype=np.float64), group_size, axis=1)
    prod = q * s  # exact: at most 8 + 11 significant bits
    w_hat = prod + b
    if np.any(_two_sum_error(prod, b) != 0):
        raise AssertionError("q*scale + bias is not exact in float64")
    return w_hat


def dequant(codes, scale, bias, group_size: int, out: str) -> np.ndarray:
    """Reconstruction in precision ``out``: one RNE step of the exact value."""
    return round_to_format(dequant_exact(codes, scale, bias, group_size), out)


# --------------------------------------------------------------------------
# 5. Matmul in float64 and the output tolerance
# --------------------------------------------------------------------------
def matmul_ref(x, w_hat):
    """y_ref = x . w_hat^T in float64 and A = |x| . |w_hat|^T.

    x[M, K] (any float dtype, taken exactly), w_hat[N, K] float64.  y_ref is
    left unrounded; A is what the output tolerance is relative to.
    """
    x64 = np.asarray(x, dtype=np.float64)
    w64 = np.asarray(w_hat, dtype=np.float64)
    return x64 @ w64.T, np.abs(x64) @ np.abs(w64).T


def matmul_bias_ref(x, w_hat, layer_bias):
    """A linear layer: y_ref = x . w_hat^T + layer_bias in float64, and the
    tolerance base A = |x| . |w_hat|^T + |layer_bias| (the bias is one more
    term of each output's sum).

    layer_bias[N] is a linear layer's own bias vector (the ExecuTorch stack's
    "4-bit linear with bias": "Metal backend: import qmv_impl from MLX", its
    stack of changes), not the quantisation biases.
    """
    y_ref, a_ref = matmul_ref(x, w_hat)
    b64 = np.asarray(layer_bias, dtype=np.float64)
    return y_ref + b64[None, :], a_ref + np.abs(b64)[None, :]


TOL_REL = 2e-3
TOL_ABS = 1e-5


def within_tolerance(y, y_ref, a_ref) -> np.ndarray:
    """Elementwise |y - y_ref| <= 2e-3 * sum_k |x_k w_nk| + 1e-5."""
    y = np.asarray(y, dtype=np.float64)
    return np.abs(y - y_ref) <= TOL_REL * a_ref + TOL_ABS


def linear_ref(x, w_f32, bits: int, group_size: int, sdtype: str):
    """Whole path from float32 weights: quantise, pack, unpack, dequant, matmul.

    Returns a dict with every intermediate so that each step can be checked.
    """
    codes, scale, bias = quantize_affine(w_f32, bits, group_size, sdtype)
    words = pack(codes, bits)
    codes_back = unpack(words, bits, w_f32.shape[1])
    w_hat = dequant_exact(codes_back, scale, bias, group_size)
    y_ref, a_ref = matmul_ref(x, w_hat)
    return {
        "codes": codes,
        "scale": scale,
        "bias": bias,
        "words": words,
        "w_hat": w_hat,
        "y_ref": y_ref,
        "a_ref": a_ref,
    }


def bytes_per_weight(bits: int, group_size: int, sdtype_bytes: int = 2) -> float:
    """Packed bytes streamed per weight: the code plus its share of scale+bias."""
    return bits / 8 + 2 * sdtype_bytes / group_size

