"""The no-allocation chain entry point (qlin_qmv_chain_static), called through
the C ABI.  It is for callers that cannot allocate device memory (a plugin
inside a framework that owns all device memory, a deployment with a fixed
memory budget): its scratch is a static array inside the library.  Its results
must match the allocating entry point (qlin_qmv_chain) on the same links, on
two calls in a row (the shared static scratch keeps the previous call's
contents, which each call must clear).  Named to be collected last."""

import ctypes

import numpy as np
import pytest
import torch

import int8_qmv_qmm_gb300 as q
from int8_qmv_qmm_gb300 import synthetic as S
from oracle import qlin_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int8_qmv_qmm_gb300 import build_lib
    build_lib.build()
    q.lib()
    return torch.device("cuda:0")


def _links(dev, bits, dt):
    # a dependent chain: slices of earlier outputs, one link with K = 8192
    specs = [(3072, 2048, -1, 0), (2048, 2048, 0, 0), (8256, 2048, 1, 0), (2048, 8192, 2, 64),
             (333, 2048, 3, 0), (640, 320, 4, 8)]
    links = []
    for i, (n, k, inp, off) in enumerate(specs):
        w = torch.from_numpy(S.weights_f32(900 + i, n, k)).to(dev)
        wq, sc, bi = q.quantize_affine(w, bits, sdtype=dt)
        links.append(dict(wq=wq, scales=sc, biases=bi, K=k, input=inp, input_offset=off,
                          y=torch.empty((1, n), dtype=dt, device=dev)))
    return links


def _call_static(x0, links, bits, dt):
    arr = q.make_links(links)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return q.lib().qlin_qmv_chain_static(ctypes.c_void_p(x0.data_ptr()), arr, len(links), bits,
                                         64, q._DTYPE_CODE[dt], stream)


def _bound(x, d, bits):
    """sum_k |x_k w_hat_nk| for each output, from the materialised weights."""
    w_hat = q.dequant(d["wq"], d["scales"], d["biases"], bits, out_dtype=torch.float32)
    return np.abs(x.double().cpu().numpy()) @ np.abs(w_hat.double().cpu().numpy()).T


@pytest.mark.parametrize("bits,dt", [(8, torch.float16), (4, torch.bfloat16)])
def test_static_chain_matches_allocating_chain_twice(dev, bits, dt):
    ref_links = _links(dev, bits, dt)
    st_links = [dict(d, y=torch.empty_like(d["y"])) for d in ref_links]
    wsp = q.chain_workspace(len(ref_links), dev)
    for call in range(2):
        x0 = S.activations(40 + call, 1, 2048, "f16" if dt == torch.float16 else "bf16").to(dev)
        q.qmv_chain(x0, q.make_links(ref_links), len(ref_links), bits, dt, wsp)
        assert _call_static(x0, st_links, bits, dt) == 0, q.lib().qlin_last_error()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(ref_links, st_links)):
            x = x0 if a["input"] < 0 else \
                ref_links[a["input"]]["y"][:, a["input_offset"]:a["input_offset"] + a["K"]]
            bound = O.TOL_REL * _bound(x, a, bits) + O.TOL_ABS
            diff = np.abs(a["y"].double().cpu().numpy() - b["y"].double().cpu().numpy())
            assert np.all(diff <= bound), f"call {call}, link {i}"
            assert torch.equal(a["y"], b["y"]), f"call {call}, link {i}: not bit-identical"
    assert q.device_status() == 0


def test_static_chain_rejects_too_many_links(dev):
    links = _links(dev, 4, torch.float16)[:1]
    x0 = torch.zeros((1, 2048), dtype=torch.float16, device=dev)
    arr = q.make_links(links * 161)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = q.lib().qlin_qmv_chain_static(ctypes.c_void_p(x0.data_ptr()), arr, 161, 4, 64,
                                       q.QLIN_F16, stream)
    assert rc == 1 and b"160" in q.lib().qlin_last_error()
