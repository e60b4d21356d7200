"""Parity at the workloads' full sizes, in the launch configurations the
benchmark uses.  Where the oracle can compute every output in seconds it does;
for the full decode step it checks sampled output rows of every linear, each
computed by the oracle from its own regenerated weight rows."""

import numpy as np
import pytest
import torch

import int8_qmv_qmm_gb300 as q
from int8_qmv_qmm_gb300 import synthetic as S
from oracle import qlin_oracle as O
from tests.gpu_helpers import TORCH_DT, as_u32, assert_within_tolerance, case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_qmv_qmm_gb300 import build_lib
    build_lib.build()
    q.lib()
    return torch.device("cuda:0")


def _run(dev, fn, m, n, k, bits, dt, seed, outlier=0.0):
    w, x, ref = case(seed, m, n, k, bits, dt, outlier)
    wq, sc, bi = q.quantize_affine(torch.from_numpy(w).to(dev), bits, sdtype=TORCH_DT[dt])
    assert np.array_equal(as_u32(wq), ref["words"])
    y = getattr(q, fn)(x.to(dev), wq, sc, bi, bits)
    assert_within_tolerance(y, ref, f"{fn} m={m} n={n} k={k} b={bits} {dt}")


def test_single_qmv_n_not_multiple_of_4(dev):
    _run(dev, "qmv", 1, 300, 512, 4, "f16", seed=0)
    _run(dev, "linear", 1, 300, 512, 4, "f16", seed=0)


@pytest.mark.parametrize("idx", range(7))
def test_one_decoder_layer_at_decode(dev, idx):
    name, n, k = S.LLAMA_1B_LINEARS[idx]
    _run(dev, "qmv", 1, n, k, 4, "f16", seed=S.weight_seed(1, idx))


@pytest.mark.parametrize("nk", [(8192, 2048), (2048, 8192)])
@pytest.mark.parametrize("m", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("fn", ["qmv", "qmm"])
def test_batched_decode_sweep(dev, fn, m, nk):
    n, k = nk
    _run(dev, fn, m, n, k, 4, "bf16", seed=S.weight_seed(3, m * 10 + (n > k)))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("nk", [(8192, 2048), (2048, 8192), (2048, 2048)])
@pytest.mark.parametrize("m", [512, 2048])
def test_prefill_qmm(dev, m, nk, bits):
    n, k = nk
    _run(dev, "qmm", m, n, k, bits, "f16", seed=S.weight_seed(4, n + k + bits), outlier=0.01)


def test_full_decode_step_sampled_rows(dev):
    """All 113 linears of the 8-bit decode step (stored fused as the step
    launches them), each run on fresh synthetic input through its own launch;
    48 sampled rows per linear are checked against the oracle (codes
    bit-exact, outputs within tolerance).  Then the step's graph (one chain
    launch) replays and gives finite, repeatable logits, identical to per-linear
    launches."""
    from int8_qmv_qmm_gb300.decode_step import DecodeStep
    step = DecodeStep(dev, bits=8, dtype=torch.float16, seed=2)
    assert len(step.linears) == 113 and step.n_launches == 65
    rng = np.random.default_rng(0)
    for i in range(len(step.linears)):
        name, layer, n, k, wq, sc, bi, wseed = step.linear_rows(i)
        rows = np.unique(np.concatenate([[0, n - 1], rng.choice(n, 46, replace=False)]))
        w_rows = S.weights_f32(wseed, n, k, rows=rows)
        x = S.activations(wseed, 1, k, "f16")
        r = O.linear_ref(x.float().numpy().astype(np.float64), w_rows, 8, 64, "f16")
        y = step.run_linear(i, x.to(dev))
        idx = torch.from_numpy(rows).to(dev)
        assert np.array_equal(as_u32(wq[idx]), r["words"]), name
        assert_within_tolerance(y[:, idx], r, f"{name} layer {layer}")
    step.x0.copy_(S.activations(9, 1, 2048, "f16").to(dev))
    step.capture()
    step.replay()
    torch.cuda.synchronize()
    assert torch.isfinite(step.logits.float()).all()
    first = step.logits.clone()
    step.replay()
    torch.cuda.synchronize()
    assert torch.equal(first, step.logits)
    # the single-launch chain and the overlapped per-linear launches compute
    # exactly what plain stream-ordered launches do
    step.overlap = False
    step.launch_all()
    torch.cuda.synchronize()
    assert torch.equal(first, step.logits)
    step.overlap = True
    step.launch_all()
    torch.cuda.synchronize()
    assert torch.equal(first, step.logits)
    assert q.device_status() == 0


def test_dense_f16_comparator_computes_the_same_step(dev):
    """The f16-resident comparator (dense weights from qlin_dequant, cuBLAS)
    and the packed kernels compute the same linears: sampled rows of every
    linear of a two-layer step with the lm_head, each on fresh input, agree
    with the oracle within the tolerance on both paths; the dense step's
    graph replays to finite logits."""
    from int8_qmv_qmm_gb300.decode_step import DecodeStep, DenseF16Step
    step = DecodeStep(dev, bits=8, dtype=torch.float16, seed=2, layers=2)
    dense = DenseF16Step(step)
    rng = np.random.default_rng(1)
    for i in range(len(step.linears)):
        name, layer, n, k, wq, sc, bi, wseed = step.linear_rows(i)
        rows = np.unique(np.concatenate([[0, n - 1], rng.choice(n, 30, replace=False)]))
        w_rows = S.weights_f32(wseed, n, k, rows=rows)
        x = S.activations(wseed + 17, 1, k, "f16")
        r = O.linear_ref(x.float().numpy().astype(np.float64), w_rows, 8, 64, "f16")
        idx = torch.from_numpy(rows).to(dev)
        assert_within_tolerance(step.run_linear(i, x.to(dev))[:, idx], r, f"packed {name}")
        assert_within_tolerance(dense.run_linear(i, x.to(dev))[:, idx], r, f"dense {name}")
    step.x0.copy_(S.activations(9, 1, 2048, "f16").to(dev))
    dense.capture()
    dense.replay()
    torch.cuda.synchronize()
    assert torch.isfinite(dense.outs[-1].float()).all()
