"""Pins for the CPU oracle: every function is checked against something other
than itself (closed forms, hand-derived fixtures, exact rational arithmetic,
correctly rounded sums, independent library conversions).  The mutation tests
at the end plant plausible mistakes in copies of the oracle and show that the
pins catch each of them."""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import qlin_oracle as O
from tests import golden_io
from int8_qmv_qmm_gb300 import synthetic as S

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- pin helpers
def check_pack_golden(pack_fn):
    bad = []
    for bits, codes, word in golden_io.pack_cases():
        got = int(pack_fn(codes[None, :], bits)[0, 0])
        if got != word:
            bad.append((bits, codes.tolist(), hex(word), hex(got)))
    return bad


def check_quant_golden(quant_fn):
    bad = []
    for c in golden_io.quant_cases():
        codes, scale, bias = quant_fn(c["w"], c["bits"], c["g"], c["sdtype"])
        if not np.array_equal(np.asarray(codes, dtype=np.uint32), c["codes"]):
            bad.append((c["name"], "codes"))
        if int(O.encode_bits(scale, c["sdtype"])[0, 0]) != c["scale_bits"]:
            bad.append((c["name"], "scale"))
        if int(O.encode_bits(bias, c["sdtype"])[0, 0]) != c["bias_bits"]:
            bad.append((c["name"], "bias"))
    return bad


def fraction_dequant(q, s, b):
    return Fraction(int(q)) * Fraction(float(s)) + Fraction(float(b))


def check_dequant_exact(dequant_fn, seed=3):
    """Compare with exact rational arithmetic on random codes/scales/biases."""
    rng = np.random.default_rng(seed)
    bad = []
    for bits, fmt in ((4, "f16"), (8, "f16"), (4, "bf16"), (8, "bf16")):
        n, k, g = 3, 128, 64
        codes = rng.integers(0, 1 << bits, size=(n, k))
        scale = O.round_to_format(np.abs(rng.standard_normal((n, k // g))) * 0.01, fmt)
        bias = O.round_to_format(rng.standard_normal((n, k // g)) * 0.05, fmt)
        w = dequant_fn(codes, scale, bias, g)
        for i in range(n):
            for j in range(0, k, 7):
                exact = fraction_dequant(codes[i, j], scale[i, j // g], bias[i, j // g])
                if Fraction(float(w[i, j])) != exact:
                    bad.append((bits, fmt, i, j))
    return bad


def fsum_matmul(x, w):
    """Correctly rounded x . w^T per element (products exact in float64)."""
    m, n = x.shape[0], w.shape[0]
    y = np.empty((m, n))
    for i in range(m):
        for j in range(n):
            y[i, j] = math.fsum(float(a) * float(b) for a, b in zip(x[i], w[j]))
    return y


def check_matmul_bruteforce(matmul_fn, seed=5):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, 64)).astype(np.float16).astype(np.float64)
    w = O.round_to_format(rng.standard_normal((5, 64)) * 0.02, "f16")
    y, a = matmul_fn(x, w)
    y_fs = fsum_matmul(x, w)
    a_fs = fsum_matmul(np.abs(x), np.abs(w))
    bad = []
    if not np.all(np.abs(y - y_fs) <= 64 * 2.0 ** -52 * a_fs):
        bad.append("y")
    if not np.all(np.abs(a - a_fs) <= 64 * 2.0 ** -52 * a_fs):
        bad.append("a")
    return bad


# ------------------------------------------------------------ rounding pins
def _awkward_values(rng, n=20000):
    v = rng.standard_normal(n) * np.exp2(rng.integers(-30, 20, n))
    ties16 = (np.floor(rng.uniform(1024, 2048, 500)) + 0.5) * np.exp2(rng.integers(-20, 5, 500) - 10.0)
    sub16 = rng.uniform(-1, 1, 500) * 2.0 ** -14
    big = rng.uniform(6.0e4, 7.0e4, 100)
    return np.concatenate([v, ties16, -ties16, sub16, big, [0.0, -0.0, 65504.0, 65520.0, 65519.99]])


def test_round_to_f16_matches_numpy_direct_conversion():
    v = _awkward_values(np.random.default_rng(0))
    ref = v.astype(np.float16).astype(np.float64)  # numpy rounds double -> half directly
    got = O.round_to_format(v, "f16")
    assert np.array_equal(got, ref, equal_nan=True)


def test_round_to_f32_matches_hardware_cast():
    v = _awkward_values(np.random.default_rng(1))
    ties32 = (np.floor(np.random.default_rng(2).uniform(2**23, 2**24, 500)) + 0.5) * 2.0 ** -30
    v = np.concatenate([v, ties32, [1e39, -1e39, 1e-46]])
    ref = v.astype(np.float32).astype(np.float64)
    assert np.array_equal(O.round_to_format(v, "f32"), ref, equal_nan=True)


def test_round_to_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(4)
    v32 = (rng.standard_normal(20000) * np.exp2(rng.integers(-40, 40, 20000))).astype(np.float32)
    ties = ((np.floor(rng.uniform(128, 256, 500)) + 0.5) * 2.0 ** -7).astype(np.float32)
    v32 = np.concatenate([v32, ties, -ties, np.float32([3.3e38, 1e-40, 0])])
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_to_format(v32.astype(np.float64), "bf16")
    assert np.array_equal(got, ref, equal_nan=True)


def test_encode_decode_roundtrip_and_rejects_unrounded():
    rng = np.random.default_rng(6)
    for fmt in ("f16", "bf16", "f32"):
        v = O.round_to_format(rng.standard_normal(1000), fmt)
        assert np.array_equal(O.decode_bits(O.encode_bits(v, fmt), fmt), v)
    with pytest.raises(ValueError):
        O.encode_bits(np.array([1 + 2.0 ** -12]), "f16")
    assert int(O.encode_bits(np.array([1.0]), "f16")[0]) == 0x3C00
    assert int(O.encode_bits(np.array([1.0]), "bf16")[0]) == 0x3F80
    assert int(O.encode_bits(np.array([-2.0]), "bf16")[0]) == 0xC000


# -------------------------------------------------------------- packing pins
def test_pack_golden_words():
    assert check_pack_golden(O.pack) == []


def test_unpack_inverts_golden_words():
    for bits, codes, word in golden_io.pack_cases():
        got = O.unpack(np.array([[word]], dtype=np.uint32), bits, codes.size)
        assert np.array_equal(got[0], codes)


@pytest.mark.parametrize("bits", [4, 8])
def test_pack_unpack_roundtrip_random(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(7, 256)).astype(np.uint32)
    assert np.array_equal(O.unpack(O.pack(codes, bits), bits, 256), codes)


def test_pack_rejects_out_of_range_codes():
    with pytest.raises(ValueError):
        O.pack(np.array([[16, 0, 0, 0, 0, 0, 0, 0]]), 4)


# ---------------------------------------------------------- quantisation pins
def test_quantize_golden_groups():
    assert check_quant_golden(O.quantize_affine) == []


def _f32(v):
    """Round a rational to float32 (through float64: innocuous here)."""
    return float(np.float32(float(v)))


def _quantize_group_by_fractions(w, bits, fmt):
    """Independent restatement for one group: exact rationals + one rounding
    per float32 operation (double rounding through float64 is innocuous for a
    single +,-,/ of float32 operands), numpy's direct half conversion for f16
    and torch's float32->bf16 conversion for bf16."""
    qmax = (1 << bits) - 1
    mn, mx = min(w.tolist()), max(w.tolist())
    scale32 = _f32(Fraction(_f32(Fraction(mx) - Fraction(mn))) / qmax)
    if fmt == "f16":
        s = float(np.float16(float(scale32)))
        b = float(np.float16(mn))
    else:
        s = float(torch.tensor([float(scale32)], dtype=torch.float32).to(torch.bfloat16).item())
        b = float(torch.tensor([mn], dtype=torch.float32).to(torch.bfloat16).item())
    codes = []
    for v in w.tolist():
        if s == 0:
            codes.append(0)
            continue
        t = _f32(Fraction(_f32(Fraction(v) - Fraction(b))) / Fraction(s))
        r = round(float(t))  # Python rounds half to even
        codes.append(min(max(r, 0), qmax))
    return codes, s, b


@pytest.mark.parametrize("bits,fmt,g", [(4, "f16", 64), (8, "f16", 64), (4, "bf16", 64),
                                        (8, "bf16", 32), (4, "f16", 128)])
def test_quantize_matches_fraction_restatement(bits, fmt, g):
    rng = np.random.default_rng(100 + bits)
    w = (rng.standard_normal((4, 2 * g)) * 0.02).astype(np.float32)
    w[1, :g] = np.float32(0.125)  # constant group
    codes, scale, bias = O.quantize_affine(w, bits, g, fmt)
    for i in range(w.shape[0]):
        for gi in range(2):
            ref_q, ref_s, ref_b = _quantize_group_by_fractions(w[i, gi * g:(gi + 1) * g], bits, fmt)
            assert codes[i, gi * g:(gi + 1) * g].tolist() == ref_q
            assert scale[i, gi] == ref_s and bias[i, gi] == ref_b


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_quantize_invariants_on_synthetic_weights(bits, fmt):
    g = 64
    w = S.weights_f32(7, 96, 512)
    codes, scale, bias = O.quantize_affine(w, bits, g, fmt)
    qmax = (1 << bits) - 1
    assert codes.min() >= 0 and codes.max() <= qmax
    w_hat = O.dequant_exact(codes, scale, bias, g)
    wg = w.reshape(96, -1, g).astype(np.float64)
    mn, mx = wg.min(axis=2), wg.max(axis=2)
    scale32 = ((mx - mn).astype(np.float32) / np.float32(qmax)).astype(np.float64)
    # round-trip bound: half a step, plus what the rounding of scale and bias moved
    bound = (scale / 2 + np.abs(bias - mn) + qmax * np.abs(scale - scale32))[..., None]
    err = np.abs(wg - w_hat.reshape(wg.shape))
    assert np.all(err <= bound * (1 + 2.0 ** -20) + 2.0 ** -22 * np.abs(wg - bias[..., None]))
    # interior codes (not clamped) are within half a stored step of w
    cg = codes.reshape(wg.shape)
    interior = (cg > 0) & (cg < qmax)
    assert np.all(err[interior] <= (scale[..., None] / 2 * (1 + 2.0 ** -20)
                                    + 2.0 ** -22 * np.abs(wg - bias[..., None]))[interior])
    # the group's min maps to code 0, its max to 2^b - 1 (up to one step from rounding)
    kmin, kmax = wg.argmin(axis=2), wg.argmax(axis=2)
    assert np.all(np.take_along_axis(cg, kmin[..., None], 2) <= 1)
    assert np.all(np.take_along_axis(cg, kmax[..., None], 2) >= qmax - 1)


def test_quantize_rejects_bad_arguments():
    w = np.zeros((2, 64), dtype=np.float32)
    with pytest.raises(ValueError):
        O.quantize_affine(w, 3, 64, "f16")
    with pytest.raises(ValueError):
        O.quantize_affine(np.zeros((2, 96), dtype=np.float32), 4, 64, "f16")
    with pytest.raises(TypeError):
        O.quantize_affine(w.astype(np.float64), 4, 64, "f16")
    with pytest.raises(ValueError):
        O.quantize_affine(np.full((1, 64), np.nan, dtype=np.float32), 4, 64, "f16")


# ------------------------------------------------------------- dequant pins
def test_dequant_exact_matches_rationals():
    assert check_dequant_exact(O.dequant_exact) == []


def test_dequant_exact_raises_when_sum_is_not_representable():
    codes = np.ones((1, 64), dtype=np.uint32)
    scale = np.array([[2.0 ** -100]])
    bias = np.array([[2.0 ** 100]])
    with pytest.raises(AssertionError):
        O.dequant_exact(codes, scale, bias, 64)


@pytest.mark.parametrize("fmt", ["f16", "bf16", "f32"])
def test_dequant_rounded_matches_library_conversion(fmt):
    rng = np.random.default_rng(8)
    codes = rng.integers(0, 16, size=(4, 128))
    scale = O.round_to_format(np.abs(rng.standard_normal((4, 2))) * 0.007, "f16")
    bias = O.round_to_format(-np.abs(rng.standard_normal((4, 2))) * 0.05, "f16")
    exact = O.dequant_exact(codes, scale, bias, 64)
    got = O.dequant(codes, scale, bias, 64, fmt)
    if fmt == "f16":
        ref = exact.astype(np.float16).astype(np.float64)
    elif fmt == "f32":
        ref = exact.astype(np.float32).astype(np.float64)
    else:
        assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
        ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref)


# -------------------------------------------------------------- matmul pins
def test_matmul_matches_correctly_rounded_sums():
    assert check_matmul_bruteforce(O.matmul_ref) == []


def test_one_hot_x_reproduces_a_dequantised_column():
    w = S.weights_f32(9, 10, 128)
    r = O.linear_ref(np.eye(128)[[5, 77]], w, 4, 64, "f16")
    assert np.array_equal(r["y_ref"][0], r["w_hat"][:, 5])
    assert np.array_equal(r["y_ref"][1], r["w_hat"][:, 77])


def test_zero_scale_groups_give_bias_times_group_sum():
    w = np.empty((3, 128), dtype=np.float32)
    w[:, :64] = np.float32(0.25)
    w[:, 64:] = np.float32(-0.5)
    x = np.arange(128, dtype=np.float64)[None, :] / 64
    r = O.linear_ref(x, w, 4, 64, "f16")
    assert np.all(r["scale"] == 0)
    expect = 0.25 * x[0, :64].sum() - 0.5 * x[0, 64:].sum()
    assert np.allclose(r["y_ref"], expect, rtol=0, atol=1e-12)


def _bias_bruteforce_errors(fn):
    """Every output of fn(x, w, b) against a correctly rounded math.fsum of its
    terms x_k w_nk plus b_n; M != N so a bias added along the wrong axis fails."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((3, 40))
    w = rng.standard_normal((5, 40))
    b = rng.standard_normal(5) * 4
    y, a = fn(x, w, b)
    bad = []
    for m in range(3):
        for n in range(5):
            exact = math.fsum([float(x[m, k] * w[n, k]) for k in range(40)] + [float(b[n])])
            mag = math.fsum([abs(float(x[m, k] * w[n, k])) for k in range(40)] + [abs(float(b[n]))])
            if abs(y[m, n] - exact) > 1e-13 * mag or abs(a[m, n] - mag) > 1e-13 * mag:
                bad.append((m, n))
    return bad


def test_linear_bias_matches_correctly_rounded_sums():
    assert _bias_bruteforce_errors(O.matmul_bias_ref) == []


def test_linear_bias_alone_when_x_is_zero():
    w = S.weights_f32(12, 6, 128).astype(np.float64)
    b = np.array([0.5, -0.25, 3.0, 0.0, -7.5, 1e-3])
    y, a = O.matmul_bias_ref(np.zeros((2, 128)), w, b)
    assert np.array_equal(y, np.tile(b, (2, 1)))
    assert np.array_equal(a, np.tile(np.abs(b), (2, 1)))


@pytest.mark.parametrize("mutant", ["no_bias", "minus_bias", "bias_on_m"])
def test_linear_bias_mutations_fail_a_pin(mutant):
    def fn(x, w, b):
        y, a = O.matmul_ref(x, w)
        if mutant == "no_bias":
            return y, a + np.abs(b)
        if mutant == "minus_bias":
            return y - b, a + np.abs(b)
        # the bias indexed by the token instead of the output row
        return y + np.resize(b, y.shape[0])[:, None], a + np.abs(b)
    assert _bias_bruteforce_errors(fn) != []


def test_within_tolerance_formula():
    y_ref = np.array([1.0, 1.0, 0.0])
    a = np.array([10.0, 10.0, 0.0])
    y = np.array([1.0 + 0.02, 1.0 + 0.0201, 1e-5])
    assert O.within_tolerance(y, y_ref, a).tolist() == [True, False, True]


def test_bytes_per_weight():
    assert O.bytes_per_weight(4, 64) == 0.5625
    assert O.bytes_per_weight(8, 64) == 1.0625


# ----------------------------------------------- synthetic input generator
def test_weight_rows_regenerate_identically():
    full = S.weights_f32(11, 2500, 64)
    rows = np.array([0, 1023, 1024, 2047, 2048, 2499])
    assert np.array_equal(S.weights_f32(11, 2500, 64, rows=rows), full[rows])
    assert abs(float(full.std()) - 0.02) < 1e-3


def test_activation_outlier_rows():
    x = S.activations(3, 200, 64, "f16", outlier_frac=0.01).float().numpy()
    big = np.abs(x).max(axis=1) > 8
    assert big.sum() == 2
    xb = S.activations(3, 8, 64, "bf16")
    assert xb.dtype == torch.bfloat16


# ------------------------------------------------------------ mutation tests
def _pack_high_bits_first(codes, bits):
    codes = np.asarray(codes).astype(np.uint32)
    p = 32 // bits
    words = np.zeros((codes.shape[0], codes.shape[1] // p), dtype=np.uint32)
    for j in range(p):
        words |= codes[:, j::p] << np.uint32(bits * (p - 1 - j))
    return words


def _quant_round_half_up(w, bits, g, fmt):
    codes, scale, bias = O.quantize_affine(w, bits, g, fmt)
    s32 = np.repeat(scale, g, axis=1).astype(np.float32)
    b32 = np.repeat(bias, g, axis=1).astype(np.float32)
    with np.errstate(all="ignore"):
        t = np.where(s32 == 0, 0, (w - b32) / s32)
    return np.clip(np.floor(t + 0.5), 0, (1 << bits) - 1).astype(np.uint32), scale, bias


def _quant_unrounded_scale(w, bits, g, fmt):
    # computes codes from the float32 scale instead of the stored one
    codes, scale, bias = O.quantize_affine(w, bits, g, fmt)
    wg = w.reshape(w.shape[0], -1, g)
    s32 = ((wg.max(2) - wg.min(2)) / np.float32((1 << bits) - 1))[..., None]
    b32 = bias.astype(np.float32)[..., None]
    with np.errstate(all="ignore"):
        t = np.where(s32 == 0, 0, (wg - b32) / s32)
    return np.clip(np.rint(t), 0, (1 << bits) - 1).reshape(w.shape), scale, bias


def _quant_bias_from_max(w, bits, g, fmt):
    codes, scale, bias = O.quantize_affine(w, bits, g, fmt)
    wg = w.reshape(w.shape[0], -1, g)
    return codes, scale, O.round_to_format(wg.max(2).astype(np.float64), fmt)


def _dequant_minus_bias(codes, scale, bias, g):
    return O.dequant_exact(codes, scale, -np.asarray(bias), g)


def _dequant_wrong_group_index(codes, scale, bias, g):
    s = np.tile(np.asarray(scale), (1, g))  # interleaves groups instead of repeating
    b = np.tile(np.asarray(bias), (1, g))
    return np.asarray(codes, dtype=np.float64) * s + b


def _matmul_transposed_w(x, w):
    return O.matmul_ref(x, w[::-1])


def _matmul_dropped_tail(x, w):
    return O.matmul_ref(x[:, :-1], w[:, :-1])


def test_mutations_are_caught():
    assert check_pack_golden(_pack_high_bits_first)
    assert check_quant_golden(_quant_round_half_up)
    assert check_quant_golden(_quant_unrounded_scale)
    assert check_quant_golden(_quant_bias_from_max)
    assert check_dequant_exact(_dequant_minus_bias)
    assert check_dequant_exact(_dequant_wrong_group_index)
    assert check_matmul_bruteforce(_matmul_transposed_w)
    assert check_matmul_bruteforce(_matmul_dropped_tail)


def test_bf16_output_rounding_alone_can_exceed_the_bound():
    """Why same-sign bf16 cases are checked through the float32 output: with
    x and w_hat all positive, |y| = sum |x w_hat|, and rounding y to bfloat16
    (8 significant bits) moves it by up to 2^-8 |y| = 3.9e-3 |y|.  Even the
    exact product rounded once breaks 2e-3 * sum|x w_hat| + 1e-5 on many
    outputs, while the float16 rounding (2^-11 |y|) never does."""
    rng = np.random.default_rng(5)
    w = np.abs(rng.standard_normal((512, 128)) * 0.02).astype(np.float32)
    x = np.abs(rng.standard_normal((16, 128))).astype(np.float32)
    for dt, expect_fail in (("bf16", True), ("f16", False)):
        xr = O.round_to_format(x.astype(np.float64), dt)
        ref = O.linear_ref(xr, w, 4, 64, dt)
        best = O.round_to_format(ref["y_ref"], dt)
        ok = O.within_tolerance(best, ref["y_ref"], ref["a_ref"])
        assert (not ok.all()) == expect_fail, dt
