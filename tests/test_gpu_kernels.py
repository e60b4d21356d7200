"""GPU parity of every kernel against the CPU oracle on seeded inputs, through
the C ABI (via the ctypes binding).  Sizes span several tiles and ragged tails;
codes, scales, biases and reconstructed weights must be bit-exact, outputs
within |y - y_ref| <= 2e-3 * sum_k |x_k w_nk| + 1e-5 per element."""

import ctypes

import numpy as np
import pytest
import torch

import int8_qmv_qmm_gb300 as q
from int8_qmv_qmm_gb300 import synthetic as S
from oracle import qlin_oracle as O
from tests.gpu_helpers import (TORCH_DT, as_u16, as_u32, assert_within_tolerance,
                               canaries_intact, case, guarded)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_qmv_qmm_gb300 import build_lib
    build_lib.build()
    q.lib()
    return torch.device("cuda:0")


def _upload(dev, w, bits, dt):
    return q.quantize_affine(torch.from_numpy(w).to(dev), bits, sdtype=TORCH_DT[dt])


# ------------------------------------------------------------ quantisation
@pytest.mark.parametrize("bits,dt,n,k", [(4, "f16", 300, 512), (8, "f16", 77, 192),
                                         (4, "bf16", 129, 2048), (8, "bf16", 64, 64),
                                         (4, "f16", 1, 64), (8, "f16", 3, 8192)])
def test_quantize_bit_exact(dev, bits, dt, n, k):
    w = S.weights_f32(bits * 100 + n, n, k)
    wq, sc, bi = _upload(dev, w, bits, dt)
    codes, scale, bias = O.quantize_affine(w, bits, 64, dt)
    assert np.array_equal(as_u32(wq), O.pack(codes, bits))
    assert np.array_equal(as_u16(sc), O.encode_bits(scale, dt))
    assert np.array_equal(as_u16(bi), O.encode_bits(bias, dt))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("bits", [4, 8])
def test_quantize_edge_groups(dev, bits, dt):
    """Constant groups (scale 0), tiny ranges (subnormal f16 scale), exact ties,
    huge and negative values."""
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    w[0, :64] = 0.375                                    # constant: scale 0
    w[1, :64] = np.float32(1e-3) + np.arange(64, dtype=np.float32) * np.float32(1e-8)  # tiny
    qmax = (1 << bits) - 1
    t = np.tile(np.array([0, qmax, 0.5, 1.5, 2.5, qmax - 0.5], dtype=np.float64), 11)[:64]
    w[2, :64] = (-0.0625 + t * 2.0 ** -9).astype(np.float32)  # exact ties
    w[3, 64:128] = rng.standard_normal(64).astype(np.float32) * 100
    w[4, 128:] = -np.abs(w[4, 128:]) - 3.0
    wq, sc, bi = _upload(dev, w, bits, dt)
    codes, scale, bias = O.quantize_affine(w, bits, 64, dt)
    assert np.array_equal(as_u32(wq), O.pack(codes, bits))
    assert np.array_equal(as_u16(sc), O.encode_bits(scale, dt))
    assert np.array_equal(as_u16(bi), O.encode_bits(bias, dt))


# ------------------------------------------------------------ dequant
@pytest.mark.parametrize("bits,dt", [(4, "f16"), (8, "f16"), (4, "bf16"), (8, "bf16")])
@pytest.mark.parametrize("out", ["f32", "same"])
def test_dequant_bit_exact(dev, bits, dt, out):
    n, k = 131, 1024
    w = S.weights_f32(31 + bits, n, k)
    wq, sc, bi = _upload(dev, w, bits, dt)
    codes, scale, bias = O.quantize_affine(w, bits, 64, dt)
    fmt = dt if out == "same" else "f32"
    got = q.dequant(wq, sc, bi, bits, out_dtype=torch.float32 if out == "f32" else TORCH_DT[dt])
    ref_bits = O.encode_bits(O.dequant(codes, scale, bias, 64, fmt), fmt)
    got_bits = as_u32(got) if fmt == "f32" else as_u16(got)
    assert np.array_equal(got_bits, ref_bits)


# ------------------------------------------------------------ qmv
QMV_CASES = [
    (1, 300, 512, 4, "f16"), (1, 301, 512, 8, "f16"), (1, 1, 64, 4, "f16"),
    (1, 3, 192, 8, "bf16"), (1, 2048, 2048, 4, "f16"), (1, 513, 8192, 8, "f16"),
    (1, 700, 2048, 4, "bf16"), (2, 300, 512, 4, "f16"), (3, 301, 1024, 8, "bf16"),
    (4, 129, 2048, 4, "bf16"), (5, 77, 512, 8, "f16"), (8, 300, 256, 4, "f16"),
    (13, 64, 512, 4, "bf16"), (2, 1000, 4096, 8, "bf16"),
]


@pytest.mark.parametrize("m,n,k,bits,dt", QMV_CASES)
def test_qmv_parity(dev, m, n, k, bits, dt):
    w, x, ref = case(1000 + m * 7 + n, m, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    buf, y = guarded((m, n), TORCH_DT[dt], dev)
    q.qmv(x.to(dev), wq, sc, bi, bits, out=y)
    torch.cuda.synchronize()
    assert canaries_intact(buf)
    assert_within_tolerance(y, ref, f"qmv m={m} n={n} k={k} b={bits} {dt}")


# ------------------------------------------------------------ qmm
QMM_CASES = [
    (1, 300, 512, 4, "f16"), (3, 3, 64, 8, "f16"), (17, 130, 192, 4, "bf16"),
    (33, 300, 512, 8, "f16"), (64, 256, 1024, 4, "f16"), (129, 301, 512, 4, "bf16"),
    (300, 200, 256, 8, "bf16"), (600, 384, 512, 4, "f16"), (257, 1, 128, 8, "f16"),
    (16, 128, 64, 4, "f16"), (512, 1024, 2048, 8, "f16"),
    # enough tiles for the 256- and 128-token tiles, several tiles per CTA
    (768, 8192, 128, 8, "f16"), (768, 8192, 512, 4, "bf16"), (640, 4096, 256, 4, "f16"),
    (1100, 8200, 512, 8, "bf16"),
    # bf16 at small K, where rounding the tensor-core operand to bf16 alone
    # (2^-8 relative per weight) used to push a few of these outputs past the
    # bound; the kernel now adds the residual operand (K = 64 and 128 in bf16:
    # test_bf16_small_k_through_the_f32_output)
    (768, 8192, 192, 4, "bf16"), (768, 8192, 192, 8, "bf16"),
    # few tiles: K split over a cluster of 4 (f16, bf16, ragged M and N) or 2
    (512, 2048, 8192, 4, "f16"), (100, 384, 4096, 8, "bf16"), (300, 1000, 2048, 4, "f16"),
    (32, 8192, 2048, 4, "f16"),
]


@pytest.mark.parametrize("m,n,k,bits,dt", QMM_CASES)
def test_qmm_parity(dev, m, n, k, bits, dt):
    w, x, ref = case(2000 + m * 7 + n, m, n, k, bits, dt, outlier_frac=0.01 if m >= 100 else 0)
    wq, sc, bi = _upload(dev, w, bits, dt)
    buf, y = guarded((m, n), TORCH_DT[dt], dev)
    q.qmm(x.to(dev), wq, sc, bi, bits, out=y)
    torch.cuda.synchronize()
    assert canaries_intact(buf)
    assert_within_tolerance(y, ref, f"qmm m={m} n={n} k={k} b={bits} {dt}")


@pytest.fixture
def qmm_tile(monkeypatch):
    """Force qmm's token tile and split-K factor (QLIN_QMM_BN / _SPLIT)."""
    def force(bn, split):
        monkeypatch.setenv("QLIN_QMM_BN", str(bn))
        monkeypatch.setenv("QLIN_QMM_SPLIT", str(split))
    return force


@pytest.mark.parametrize("bn,split", [(128, 1), (128, 2), (128, 4), (256, 4), (64, 2)])
def test_qmm_split_k_factors(dev, qmm_tile, bn, split):
    """Each split of K over a cluster, summed through distributed shared
    memory, stays within the tolerance of the oracle."""
    m, n, k, bits, dt = 200, 640, 2048, 8, "f16"
    w, x, ref = case(4100 + bn + split, m, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    qmm_tile(bn, split)
    buf, y = guarded((m, n), TORCH_DT[dt], dev)
    q.qmm(x.to(dev), wq, sc, bi, bits, out=y)
    torch.cuda.synchronize()
    assert canaries_intact(buf)
    assert_within_tolerance(y, ref, f"qmm split bn={bn} split={split}")
    assert q.device_status() == 0


@pytest.mark.parametrize("bits,dt", [(4, "f16"), (8, "bf16")])
def test_one_hot_rows_exact_under_split_k(dev, qmm_tile, bits, dt):
    """With x = e_k only one CTA of a split cluster holds the nonzero term;
    the others contribute exact zeros, so the sum is still bit-identical to
    the materialised reconstruction."""
    n, k = 260, 512
    w = S.weights_f32(78, n, k)
    wq, sc, bi = _upload(dev, w, bits, dt)
    cols = np.array([0, 1, 7, 63, 64, 200, 255, 256, 511])
    x = torch.zeros((cols.size, k), dtype=TORCH_DT[dt])
    x[np.arange(cols.size), cols] = 1
    qmm_tile(64, 4)
    y = q.qmm(x.to(dev), wq, sc, bi, bits)
    w_hat = q.dequant(wq, sc, bi, bits)
    assert torch.equal(y.cpu(), w_hat[:, cols].t().contiguous().cpu())


@pytest.fixture
def qmv_split(monkeypatch):
    """Force qmv's split of K over a cluster of CTAs (QLIN_QMV_SPLIT)."""
    def force(split):
        monkeypatch.setenv("QLIN_QMV_SPLIT", str(split))
    return force


QMV_SPLIT_CASES = [
    # (split, m, n, k, bits, dt); k-tile kinds: fixed 2048-code tiles (K a
    # multiple of 2048 * split), tiles with their scales copied, scales read
    # from global memory (small tiles)
    (1, 1, 129, 8192, 4, "f16"), (2, 1, 640, 2048, 8, "f16"), (4, 3, 300, 4096, 4, "bf16"),
    (8, 1, 129, 8192, 4, "f16"), (8, 1, 37, 16384, 8, "bf16"), (4, 2, 1000, 8192, 8, "bf16"),
    (8, 2, 1000, 8192, 8, "bf16"), (4, 1, 300, 512, 4, "f16"), (8, 5, 77, 1024, 8, "f16"),
]


@pytest.mark.parametrize("split,m,n,k,bits,dt", QMV_SPLIT_CASES)
def test_qmv_split_k_factors(dev, qmv_split, split, m, n, k, bits, dt):
    """qmv with K split over a cluster (each CTA's row sums added in CTA 0's
    shared memory, in rank order) stays within the oracle's tolerance, plain
    and with a linear layer's bias and float32 output."""
    w, x, ref = case(8100 + split * 31 + n, m, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    qmv_split(split)
    buf, y = guarded((m, n), TORCH_DT[dt], dev)
    q.qmv(x.to(dev), wq, sc, bi, bits, out=y)
    torch.cuda.synchronize()
    assert canaries_intact(buf)
    assert_within_tolerance(y, ref, f"qmv split={split} m={m} n={n} k={k} b={bits} {dt}")
    if m < q.crossover_m(n, k, bits, TORCH_DT[dt]):
        rng = np.random.default_rng(8200 + n)
        b = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 0.5).to(TORCH_DT[dt])
        y_ref, a_ref = O.matmul_bias_ref(x.double().numpy(), ref["w_hat"], b.double().numpy())
        yl = q.linear(x.to(dev), wq, sc, bi, bits, bias=b.to(dev), out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert_within_tolerance(yl, {"y_ref": y_ref, "a_ref": a_ref}, f"linear split={split}")
    assert q.device_status() == 0


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("split", [None, 1])
def test_qmv_longest_k(dev, qmv_split, bits, split):
    """M = 1 at K = 32768, near the largest K whose f32 x fits in shared memory
    beside the ring: split by the host's choice (8 CTAs a row block, each
    staging an eighth of x) and forced whole (every CTA staging all of x)."""
    m, n, k, dt = 1, 300, 32768, "f16"
    if split:
        qmv_split(split)
    w, x, ref = case(8400 + bits, m, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    buf, y = guarded((m, n), TORCH_DT[dt], dev)
    q.qmv(x.to(dev), wq, sc, bi, bits, out=y)
    torch.cuda.synchronize()
    assert canaries_intact(buf)
    assert_within_tolerance(y, ref, f"qmv K={k} b={bits} split={split}")
    assert q.device_status() == 0


@pytest.mark.parametrize("bits,dt,parts", [(4, "f16", 2), (8, "bf16", 2), (8, "f16", 4)])
def test_qmv_k_parts_one_hot_exact(dev, monkeypatch, bits, dt, parts):
    """M = 1 on fixed 2048-code k-tiles runs R rows per warp, each warp over
    one R-th of every tile (R = 2 by default, 4 as a tuning option), the row
    group's sums added in shared memory.  With x = e_k one part holds the only
    nonzero term and the others add exact zeros: the output is the
    reconstructed weight bit for bit; and random x stays within the
    tolerance."""
    monkeypatch.setenv("QLIN_QMV_KH", str(parts))
    n = 1029
    k = 4096 if bits == 4 else 2048     # row blocks too short for a split of K
    assert q.lib().qlin_testing_qmv_split(n, k, bits, 152) == 1
    w = S.weights_f32(81, n, k)
    wq, sc, bi = _upload(dev, w, bits, dt)
    w_hat = q.dequant(wq, sc, bi, bits)
    for col in (0, 5, 1023, 1024, k // 2 - 1, k // 2, k - 65, k - 1):
        x = torch.zeros((1, k), dtype=TORCH_DT[dt])
        x[0, col] = 1
        y = q.qmv(x.to(dev), wq, sc, bi, bits)
        assert torch.equal(y[0].cpu(), w_hat[:, col].cpu()), col
    _, xr, ref = case(8500 + parts, 1, n, k, bits, dt)
    ref = O.linear_ref(xr.float().numpy().astype(np.float64), w, bits, 64, dt)
    assert_within_tolerance(q.qmv(xr.to(dev), wq, sc, bi, bits), ref, f"K parts {parts}")
    assert q.device_status() == 0


def test_qmv_split_k_as_dependent_launch(dev):
    """A split-K qmv (a cluster per row block) launched as a programmatic
    dependent launch after the kernel that writes its input gives what a plain
    launch gives, bit for bit (the cluster and the overlap attributes
    together)."""
    n, k, bits, dt = 129, 8192, 4, "f16"
    assert q.lib().qlin_testing_qmv_split(n, k, bits, torch.cuda.get_device_properties(dev)
                                          .multi_processor_count) > 1
    w, x, ref = case(8300, 1, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    xd = x.to(dev)
    plain = q.qmv(xd, wq, sc, bi, bits)
    x2 = torch.empty_like(xd)
    outs = []
    for _ in range(3):
        x2.copy_(xd)                       # the preceding kernel writes the input
        outs.append(q.qmv(x2, wq, sc, bi, bits, overlap_previous=True))
    torch.cuda.synchronize()
    assert q.device_status() == 0
    assert_within_tolerance(plain, ref, "split qmv plain")
    for o in outs:
        assert torch.equal(o, plain)


@pytest.mark.parametrize("bits,dt", [(4, "f16"), (8, "bf16")])
def test_qmv_one_hot_rows_exact_under_split_k(dev, qmv_split, bits, dt):
    """With x = e_k one CTA of each cluster holds the only nonzero term and
    the others add exact zeros: qmv still reproduces the materialised
    reconstruction bit for bit."""
    n, k = 260, 512
    w = S.weights_f32(79, n, k)
    wq, sc, bi = _upload(dev, w, bits, dt)
    cols = np.array([0, 1, 7, 63, 64, 200, 255, 256, 511])
    x = torch.zeros((cols.size, k), dtype=TORCH_DT[dt])
    x[np.arange(cols.size), cols] = 1
    qmv_split(4)
    y = q.qmv(x.to(dev), wq, sc, bi, bits)
    w_hat = q.dequant(wq, sc, bi, bits)
    assert torch.equal(y.cpu(), w_hat[:, cols].t().contiguous().cpu())


@pytest.mark.parametrize("fn", ["qmv", "qmm"])
@pytest.mark.parametrize("bits,dt", [(4, "f16"), (8, "f16"), (4, "bf16"), (8, "bf16")])
def test_one_hot_rows_reproduce_dequant_bit_exactly(dev, fn, bits, dt):
    """With x = e_k the product is a single exact term, so each output equals
    the reconstructed weight w_hat[n][k] in the output precision: the fused
    in-kernel reconstruction is bit-identical to the materialised one."""
    n, k = 260, 512
    w = S.weights_f32(77, n, k)
    wq, sc, bi = _upload(dev, w, bits, dt)
    cols = np.array([0, 1, 7, 63, 64, 200, 255, 256, 511])
    x = torch.zeros((cols.size, k), dtype=TORCH_DT[dt])
    x[np.arange(cols.size), cols] = 1
    y = getattr(q, fn)(x.to(dev), wq, sc, bi, bits)
    w_hat = q.dequant(wq, sc, bi, bits)
    assert torch.equal(y.cpu(), w_hat[:, cols].t().contiguous().cpu())


def test_linear_dispatches_both_paths(dev):
    n, k, bits, dt = 300, 512, 4, "f16"
    assert q.crossover_m(8192, 2048, 4) == 5 and q.crossover_m(2048, 8192, 4) == 4
    assert q.crossover_m(2048, 8192, 8, torch.bfloat16) == 5
    assert q.crossover_m(n, k, bits) == 4                      # f16, K > N
    assert q.crossover_m(n, k, bits, torch.bfloat16) == 9      # small matrix
    for m in (1, 40):
        w, x, ref = case(5 + m, m, n, k, bits, dt)
        wq, sc, bi = _upload(dev, w, bits, dt)
        y = q.linear(x.to(dev), wq, sc, bi, bits)
        assert_within_tolerance(y, ref, f"linear m={m}")


@pytest.mark.parametrize("m,n,k,bits,dt", [
    (1, 300, 512, 4, "f16"), (3, 1029, 2048, 8, "bf16"),        # qmv
    (1, 1029, 2048, 8, "bf16"),                                   # qmv, K halves
    (40, 301, 512, 4, "f16"), (600, 384, 512, 8, "bf16"),        # qmm
    (512, 2048, 8192, 4, "f16"), (32, 8192, 2048, 4, "bf16"),    # qmm, K split over a cluster
])
@pytest.mark.parametrize("with_bias,f32_out", [(True, False), (True, True), (False, True)])
def test_linear_bias_and_f32_output(dev, m, n, k, bits, dt, with_bias, f32_out):
    """qlin_linear_ex: a linear layer's bias added before the one rounding, and
    a float32 result, through whichever kernel the crossover picks."""
    w, x, ref = case(6100 + m + n, m, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    rng = np.random.default_rng(6200 + m)
    b = torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 0.5).to(TORCH_DT[dt])
    b64 = b.double().numpy() if with_bias else np.zeros(n)
    y_ref, a_ref = O.matmul_bias_ref(x.double().numpy(), ref["w_hat"], b64)
    y = q.linear(x.to(dev), wq, sc, bi, bits, bias=b.to(dev) if with_bias else None,
                 out_dtype=torch.float32 if f32_out else None)
    torch.cuda.synchronize()
    assert y.dtype == (torch.float32 if f32_out else TORCH_DT[dt])
    assert_within_tolerance(y, {"y_ref": y_ref, "a_ref": a_ref},
                            f"linear_ex m={m} n={n} bias={with_bias} f32={f32_out}")
    assert q.device_status() == 0


def _small_k_case(seed, m, n, k, dt, same_sign):
    """Seeded data; with same_sign all x and all weights are non-negative, so
    |y| = sum |x w|.  Either way, at K <= 128 |y| can come close to sum |x w|,
    and the rounding of a bf16 output alone (half a step: up to 2^-8 |y|) then
    exceeds the bound."""
    w = S.weights_f32(seed, n, k)
    x = S.activations(seed, m, k, dt)
    if same_sign:
        w, x = np.abs(w), x.abs()
    return w, x


@pytest.mark.parametrize("same_sign", [False, True])
@pytest.mark.parametrize("m", [1, 768])     # qmv, qmm
@pytest.mark.parametrize("k", [64, 128])
@pytest.mark.parametrize("bits", [4, 8])
def test_bf16_small_k_through_the_f32_output(dev, m, k, bits, same_sign):
    """bf16 at K = 64 and 128, random-sign and adversarial same-sign data: the
    float32 result (the accumulator, no output rounding) meets
    |y - y_ref| <= 2e-3 sum|x w| + 1e-5 through both kernels, so the bf16
    tensor-core operand costs nothing measurable; and the bf16 result is that
    accumulator rounded once, within the bound plus half a bf16 step."""
    n, dt = 1024, "bf16"
    w, x = _small_k_case(9100 + m + k + bits, m, n, k, dt, same_sign)
    ref = O.linear_ref(x.double().numpy(), w, bits, 64, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    xd = x.to(dev)
    y32 = q.linear(xd, wq, sc, bi, bits, out_dtype=torch.float32)
    assert_within_tolerance(y32, ref, f"f32 out m={m} k={k} b={bits} same={same_sign}")
    y16 = q.linear(xd, wq, sc, bi, bits)
    assert torch.equal(y16, y32.to(torch.bfloat16))
    # the bf16 output is within the bound plus half a bf16 step of y (no bf16
    # value can do better on such data: see the oracle test of the bound)
    y64 = y16.double().cpu().numpy()
    p, _, _ = O.FORMATS["bf16"]
    half_step = np.ldexp(1.0, np.frexp(np.abs(ref["y_ref"]))[1] - p) / 2
    assert np.all(np.abs(y64 - ref["y_ref"]) <= 2e-3 * ref["a_ref"] + 1e-5 + half_step)
    assert q.device_status() == 0


@pytest.mark.parametrize("fn", ["qmv", "qmm"])
@pytest.mark.parametrize("bits,dt", [(8, "f16"), (8, "bf16"), (4, "f16"), (4, "bf16")])
def test_groups_of_near_zero_weights(dev, fn, bits, dt):
    """Groups whose reconstructed weights nearly all sit within one step of
    zero (one large weight per group sets the step; the rest are tiny, or
    pruned to exactly zero): sum |x w| is then small against scale * sum |x|,
    which is what the qmv kernel's factored form scale * (P - MAGIC X) +
    bias * X loses bits to.  The float32 result must stay within the bound;
    the f16/bf16 result is it rounded once (and, for f16, within the bound
    too: with about 32 terms per row |y| reaches 0.65 sum |x w|, where half a
    bf16 step alone can exceed it)."""
    m = 1 if fn == "qmv" else 300
    n, k = 515, 2048
    rng = np.random.default_rng(9400 + bits)
    w = (rng.standard_normal((n, k)) * 1e-4).astype(np.float32)
    w[: n // 3] = 0.0                                   # pruned rows: exact zeros
    g = k // 64
    hot = rng.integers(0, 64, (n, g)) + np.arange(g) * 64
    sign = np.where(rng.random((n, g)) < 0.5, -1.0, 1.0)
    w[np.arange(n)[:, None], hot] = (sign * (0.05 + rng.random((n, g)) * 0.5)).astype(np.float32)
    x = S.activations(9401 + bits, m, k, dt)
    ref = O.linear_ref(x.double().numpy(), w, bits, 64, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    xd = x.to(dev)
    assert (m >= q.crossover_m(n, k, bits, TORCH_DT[dt])) == (fn == "qmm")   # linear picks fn
    y32 = q.linear(xd, wq, sc, bi, bits, out_dtype=torch.float32)
    assert_within_tolerance(y32, ref, f"near-zero groups {fn} b={bits} {dt} f32 out")
    y = getattr(q, fn)(xd, wq, sc, bi, bits)
    assert torch.equal(y, y32.to(TORCH_DT[dt]))
    if dt == "f16":
        assert_within_tolerance(y, ref, f"near-zero groups {fn} b={bits} {dt}")


def test_linear_f32_output_is_the_unrounded_sum(dev):
    """The float32 output is the accumulator itself: rounding it to the
    activation dtype gives the plain call's output bit for bit."""
    m, n, k, bits, dt = 600, 384, 512, 4, "f16"
    w, x, _ = case(6300, m, n, k, bits, dt)
    wq, sc, bi = _upload(dev, w, bits, dt)
    xd = x.to(dev)
    y16 = q.linear(xd, wq, sc, bi, bits)
    y32 = q.linear(xd, wq, sc, bi, bits, out_dtype=torch.float32)
    assert torch.equal(y32.to(torch.float16), y16)


@pytest.mark.parametrize("m", [512, 40])
def test_qmm_overlapped_chain_equals_plain_launches(dev, m):
    """Dependent qmm launches with QLIN_OVERLAP_PREVIOUS (each reads the
    previous output) give bit for bit what plain launches give, on the
    persistent and on the split-K (cluster) path."""
    dims = [(2048, 2048), (2048, 2048), (8192, 2048), (2048, 8192)]  # (N, K) per link
    ws = []
    for i, (n, k) in enumerate(dims):
        w = torch.from_numpy(S.weights_f32(7000 + i, n, k)).to(dev)
        ws.append(q.quantize_affine(w, 4, sdtype=torch.float16))
    x0 = (S.activations(7100 + m, m, 2048, "f16") * 0.05).to(dev)

    def run(overlap):
        # each link's N is the next link's K: its output is the next input
        outs, x = [], x0
        for i, (wq, sc, bi) in enumerate(ws):
            x = q.qmm(x, wq, sc, bi, 4, overlap_previous=overlap and i > 0)
            outs.append(x)
        return outs

    plain = run(False)
    torch.cuda.synchronize()
    over = run(True)
    torch.cuda.synchronize()
    assert q.device_status() == 0
    for a, b in zip(plain, over):
        assert torch.equal(a, b)


def test_empty_batch_is_a_no_op(dev):
    wq = torch.zeros((8, 64), dtype=torch.int32, device=dev)
    sc = torch.zeros((8, 8), dtype=torch.float16, device=dev)
    x = torch.zeros((0, 512), dtype=torch.float16, device=dev)
    assert q.qmv(x, wq, sc, sc, 4).shape == (0, 8)
    assert q.qmm(x, wq, sc, sc, 4).shape == (0, 8)


def test_no_kernel_gave_up_a_wait(dev):
    assert q.device_status() == 0


# ------------------------------------------------------------ qmv chain
def _chain_links(dev, specs, dt, seed):
    """specs: (N, K, bits, input, input_offset); weights quantised on the GPU."""
    links, refs = [], []
    for i, (n, k, bits, inp, off) in enumerate(specs):
        w = S.weights_f32(seed + i, n, k)
        wq, sc, bi = _upload(dev, w, bits, dt)
        y = torch.empty((1, n), dtype=TORCH_DT[dt], device=dev)
        links.append(dict(wq=wq, scales=sc, biases=bi, y=y, K=k, input=inp, input_offset=off))
        refs.append(w)
    return links, refs


@pytest.mark.parametrize("bits,dt", [(8, "f16"), (4, "bf16"), (4, "f16"), (8, "bf16")])
def test_qmv_chain_independent_links_match_oracle(dev, bits, dt):
    """Every link reads x0: each output is checked against the oracle."""
    specs = [(300, 512, bits, -1, 0), (1, 512, bits, -1, 0), (1029, 512, bits, -1, 0),
             (64, 512, bits, -1, 0), (2048, 512, bits, -1, 0)]
    links, ws_ = _chain_links(dev, specs, dt, 4100 + bits)
    x0 = S.activations(17, 1, 512, dt)
    arr = q.make_links(links)
    wsp = q.chain_workspace(len(links), dev)
    q.qmv_chain(x0.to(dev), arr, len(links), bits, TORCH_DT[dt], wsp)
    torch.cuda.synchronize()
    for d, w in zip(links, ws_):
        ref = O.linear_ref(x0.float().numpy().astype(np.float64), w, bits, 64, dt)
        assert_within_tolerance(d["y"], ref, f"chain link N={w.shape[0]}")


@pytest.mark.parametrize("bits,dt", [(8, "f16"), (4, "bf16")])
def test_qmv_chain_matches_sequential_launches(dev, bits, dt, monkeypatch):
    """A dependent chain (slices of earlier outputs, K not a multiple of 512 so
    scales come from global memory, K = 8192 split into k-tiles): each link's
    output is within the tolerance of the oracle's product of its actual input
    (an earlier link's output, as the chain read it), and equals qlin_qmv
    launched on that input bit for bit, in the layout the chain shares with it
    (rows per warp over whole k-tiles, no split of K across CTAs: the
    K-halves layout and the split add the same terms in another order).  The
    chain reruns bit for bit."""
    monkeypatch.setenv("QLIN_QMV_KH", "0")
    monkeypatch.setenv("QLIN_QMV_SPLIT", "1")
    specs = [(3072, 2048, bits, -1, 0), (2048, 2048, bits, 0, 0), (4160, 2048, bits, 1, 0),
             (2048, 4096, bits, 2, 64), (320, 2048, bits, 3, 0), (1000, 192, bits, 4, 128),
             (8192, 320, bits, 5, 8), (96, 8192, bits, 6, 0)]
    links, ws_ = _chain_links(dev, specs, dt, 5200 + bits)
    x0 = S.activations(23, 1, 2048, dt).to(dev)
    arr = q.make_links(links)
    wsp = q.chain_workspace(len(links), dev)
    first = None
    for rep in range(2):  # the second run reuses (and re-zeroes) the workspace
        q.qmv_chain(x0, arr, len(links), bits, TORCH_DT[dt], wsp)
        torch.cuda.synchronize()
        outs = [d["y"].clone() for d in links]
        if first is None:
            first = outs
        else:
            assert all(torch.equal(a, b) for a, b in zip(first, outs)), f"run {rep} differs"
    for i, (d, w) in enumerate(zip(links, ws_)):
        x = x0 if d["input"] < 0 else \
            outs[d["input"]][:, d["input_offset"]:d["input_offset"] + d["K"]].contiguous()
        ref = O.linear_ref(x.double().cpu().numpy(), w, bits, 64, dt)
        assert_within_tolerance(outs[i], ref, f"chain link {i}")
        y = q.qmv(x, d["wq"], d["scales"], d["biases"], bits)
        # same arithmetic in the same order: bit for bit
        assert torch.equal(y, outs[i]), f"link {i}: qmv differs from the chain"
    assert q.device_status() == 0


def test_qmv_chain_rejects_bad_links(dev):
    links, _ = _chain_links(dev, [(64, 512, 4, -1, 0), (64, 512, 4, 0, 0)], "f16", 1)
    wsp = q.chain_workspace(2, dev)
    bad = [dict(links[0]), dict(links[1], input=1)]          # reads itself
    with pytest.raises(q.QlinError):
        q.qmv_chain(None, q.make_links(bad), 2, 4, torch.float16, wsp)
    bad = [dict(links[0]), dict(links[1], input_offset=8)]   # reads past the end
    with pytest.raises(q.QlinError):
        q.qmv_chain(None, q.make_links(bad), 2, 4, torch.float16, wsp)
    with pytest.raises(q.QlinError):                          # link 0 reads a null x0
        q.qmv_chain(None, q.make_links(links), 2, 4, torch.float16, wsp)
    small = torch.zeros(1, dtype=torch.int32, device=dev)    # workspace too small
    x0 = torch.zeros((1, 512), dtype=torch.float16, device=dev)
    with pytest.raises(q.QlinError):
        q.qmv_chain(x0, q.make_links(links), 2, 4, torch.float16, small)


def test_chain_wait_that_runs_out_reports_and_unwinds(dev):
    """A dependency that is never met (the test-only entry point makes the
    readers of link 0 wait for one row block too many): their bounded wait runs
    out after 20 ms, the chain kernel records it in the device status word
    (bit 2 of the chain kernel, 1 << 18 in qlin_device_status) and exits after
    its bulk copies have landed.  The GPU still answers, and the same chain
    then runs exactly like sequential launches."""
    assert q.device_status() == 0
    specs = [(1024, 2048, 8, -1, 0), (2048, 1024, 8, 0, 0), (512, 2048, 8, 1, 0)]
    links, ws_ = _chain_links(dev, specs, "f16", 6100)
    x0 = S.activations(61, 1, 2048, "f16").to(dev)
    arr = q.make_links(links)
    wsp = q.chain_workspace(len(links), dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    L = q.lib()
    # bad arguments of the testing entry point are refused before any launch
    assert L.qlin_testing_qmv_chain_stalled(x0.data_ptr(), arr, 3, 8, 64, q.QLIN_F16,
                                            wsp.data_ptr(), wsp.numel() * 4, 2, 20000,
                                            stream) == 1   # nothing reads link 2
    assert L.qlin_testing_qmv_chain_stalled(x0.data_ptr(), arr, 3, 8, 64, q.QLIN_F16,
                                            wsp.data_ptr(), wsp.numel() * 4, 0, 0, stream) == 1
    st = L.qlin_testing_qmv_chain_stalled(x0.data_ptr(), arr, 3, 8, 64, q.QLIN_F16,
                                          wsp.data_ptr(), wsp.numel() * 4, 0, 20000, stream)
    assert st == 0, L.qlin_last_error()
    torch.cuda.synchronize()
    assert q.device_status() == 1 << 18
    assert q.device_status() == 0          # read and cleared
    q.qmv_chain(x0, arr, len(links), 8, torch.float16, wsp)
    torch.cuda.synchronize()
    outs = [d["y"].clone() for d in links]
    for i, (d, w) in enumerate(zip(links, ws_)):
        x = x0 if d["input"] < 0 else outs[d["input"]][:, :d["K"]].contiguous()
        ref = O.linear_ref(x.double().cpu().numpy(), w, 8, 64, "f16")
        assert_within_tolerance(outs[i], ref, f"link {i} after the stalled run")
    assert q.device_status() == 0
