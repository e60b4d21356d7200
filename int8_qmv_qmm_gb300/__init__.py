"""Fused affine-dequantise-into-matmul for MLX-style packed 4/8-bit weights on
GB300 (sm_103a).

This package is a thin ctypes binding over the C ABI of ``libqlin.so``
(declared in ``include/qlin.h``): it checks tensor placement and shape,
allocates outputs with PyTorch and passes raw device pointers and the current
CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback -- if the library is missing the
calls raise.

Layouts (row-major): packed weights ``wq`` uint32 [N, K*bits/32] (codes low
bits first), ``scales``/``biases`` [N, K/64] in the activation dtype,
activations ``x`` [M, K], output ``y`` [M, N].
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build_lib import LIB_PATH

__all__ = [
    "QlinError", "lib", "quantize_affine", "dequant", "qmv", "qmm", "linear",
    "crossover_m", "device_status", "QLIN_F32", "QLIN_F16", "QLIN_BF16", "Link", "make_links",
    "chain_workspace", "qmv_chain",
]

QLIN_F32, QLIN_F16, QLIN_BF16 = 0, 1, 2
QLIN_OVERLAP_PREVIOUS = 1
_DTYPE_CODE = {torch.float32: QLIN_F32, torch.float16: QLIN_F16, torch.bfloat16: QLIN_BF16}
GROUP_SIZE = 64

_c_i64, _c_int, _c_vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p

# name -> (restype, argtypes); names match include/qlin.h
_SIGNATURES = {
    "qlin_status_str": (ctypes.c_char_p, [_c_int]),
    "qlin_last_error": (ctypes.c_char_p, []),
    "qlin_version": (_c_int, []),
    "qlin_quantize_affine": (_c_int, [_c_vp, _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_vp, _c_vp,
                                      _c_vp, _c_vp]),
    "qlin_dequant": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_int, _c_int, _c_int, _c_int,
                              _c_vp, _c_vp]),
    "qlin_qmv": (_c_int, [_c_vp] * 5 + [_c_i64] * 3 + [_c_int] * 3 + [_c_vp]),
    "qlin_qmv_ex": (_c_int, [_c_vp] * 5 + [_c_i64] * 3 + [_c_int] * 3 + [ctypes.c_uint, _c_vp]),
    "qlin_qmm": (_c_int, [_c_vp] * 5 + [_c_i64] * 3 + [_c_int] * 3 + [_c_vp]),
    "qlin_qmm_ex": (_c_int, [_c_vp] * 5 + [_c_i64] * 3 + [_c_int] * 3 + [ctypes.c_uint, _c_vp]),
    "qlin_linear": (_c_int, [_c_vp] * 5 + [_c_i64] * 3 + [_c_int] * 3 + [_c_vp]),
    "qlin_linear_ex": (_c_int, [_c_vp] * 6 + [_c_i64] * 3 + [_c_int] * 4 + [_c_vp]),
    "qlin_crossover_m": (_c_i64, [_c_i64, _c_i64, _c_int]),
    "qlin_crossover_m_dtype": (_c_i64, [_c_i64, _c_i64, _c_int, _c_int]),
    "qlin_qmv_chain_workspace_size": (ctypes.c_size_t, [_c_int]),
    "qlin_qmv_chain": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int, _c_vp,
                                ctypes.c_size_t, _c_vp]),
    "qlin_qmv_chain_static": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int, _c_vp]),
    "qlin_device_status": (_c_int, [ctypes.POINTER(_c_int)]),
    # include/qlin_testing.h: failure paths and host-side choices, for the
    # library's own tests
    "qlin_testing_qmv_chain_stalled": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int,
                                                _c_vp, ctypes.c_size_t, _c_int, ctypes.c_uint,
                                                _c_vp]),
    "qlin_testing_qmv_split": (_c_int, [_c_i64, _c_i64, _c_int, _c_int]),
}

_LIB = None


class Link(ctypes.Structure):
    """qlin_link: one M = 1 product of a chain (include/qlin.h)."""
    _fields_ = [("wq", _c_vp), ("scales", _c_vp), ("biases", _c_vp), ("y", _c_vp),
                ("N", _c_i64), ("K", _c_i64), ("input", ctypes.c_int32),
                ("input_offset", ctypes.c_int32)]


class QlinError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(detail)


def lib(path: str | None = None):
    """The loaded libqlin (ctypes).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        p = path or os.environ.get("QLIN_LIBRARY", LIB_PATH)
        if not os.path.exists(p):
            raise RuntimeError(
                f"libqlin.so not found at {p}; build it with "
                "`python -m int8_qmv_qmm_gb300.build_lib` (needs nvcc)")
        handle = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _LIB = handle
    return _LIB


def _check(status: int):
    if status != 0:
        L = lib()
        raise QlinError(status, f"{L.qlin_status_str(status).decode()}: "
                                f"{L.qlin_last_error().decode()}")


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr() if t is not None and t.numel() else 0)


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def quantize_affine(w: torch.Tensor, bits: int, group_size: int = GROUP_SIZE,
                    sdtype: torch.dtype = torch.float16, out=None):
    """Quantise float32 W[N, K] on the GPU -> (wq, scales, biases).

    out: optional (wq, scales, biases) tensors to write into (e.g. views of
    one weight region)."""
    _need_cuda(w)
    if w.dtype != torch.float32 or w.dim() != 2:
        raise ValueError("w must be a 2-D float32 tensor")
    n, k = w.shape
    if out is not None:
        wq, sc, bi = out
        _need_cuda(wq, sc, bi)
        if (tuple(wq.shape) != (n, k * bits // 32) or tuple(sc.shape) != (n, k // group_size)
                or tuple(bi.shape) != tuple(sc.shape) or sc.dtype != sdtype
                or bi.dtype != sdtype or wq.element_size() != 4):
            raise ValueError("out tensors do not match W's shape, bits and scale dtype")
    else:
        wq = torch.empty((n, k * bits // 32), dtype=torch.int32, device=w.device)
        sc = torch.empty((n, k // group_size), dtype=sdtype, device=w.device)
        bi = torch.empty_like(sc)
    _check(lib().qlin_quantize_affine(_ptr(w), n, k, bits, group_size, _DTYPE_CODE[sdtype],
                                      _ptr(wq), _ptr(sc), _ptr(bi), _stream(w)))
    return wq, sc, bi


def dequant(wq: torch.Tensor, scales: torch.Tensor, biases: torch.Tensor, bits: int,
            group_size: int = GROUP_SIZE, out_dtype: torch.dtype | None = None) -> torch.Tensor:
    """Materialise w_hat[N, K] = RNE(q*scale + bias) (unfused reference path)."""
    _need_cuda(wq, scales, biases)
    n = wq.shape[0]
    k = wq.shape[1] * 32 // bits
    out_dtype = out_dtype or scales.dtype
    out = torch.empty((n, k), dtype=out_dtype, device=wq.device)
    _check(lib().qlin_dequant(_ptr(wq), _ptr(scales), _ptr(biases), n, k, bits, group_size,
                              _DTYPE_CODE[scales.dtype], _DTYPE_CODE[out_dtype], _ptr(out),
                              _stream(wq)))
    return out


def _matmul(name: str, x, wq, scales, biases, bits, group_size, out, flags=None, extra=()):
    _need_cuda(x, wq, scales, biases)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    m, k = x.shape
    n = wq.shape[0]
    if wq.shape[1] * 32 // bits != k:
        raise ValueError("wq does not match K")
    if out is None:
        out = torch.empty((m, n), dtype=x.dtype, device=x.device)
    _need_cuda(out)
    fn = getattr(lib(), name)
    args = (() if flags is None else (flags,)) + tuple(extra)
    _check(fn(_ptr(x), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(out), m, n, k, bits,
              group_size, _DTYPE_CODE[x.dtype], *args, _stream(x)))
    return out


def qmv(x, wq, scales, biases, bits, group_size=GROUP_SIZE, out=None, overlap_previous=False):
    """y = x . w_hat^T on CUDA cores (decode, small M).

    overlap_previous=True launches with QLIN_OVERLAP_PREVIOUS (programmatic
    dependent launch): only valid when the preceding work on the stream does
    not write wq/scales/biases."""
    if overlap_previous:
        return _matmul("qlin_qmv_ex", x, wq, scales, biases, bits, group_size, out,
                       flags=QLIN_OVERLAP_PREVIOUS)
    return _matmul("qlin_qmv", x, wq, scales, biases, bits, group_size, out)


def qmm(x, wq, scales, biases, bits, group_size=GROUP_SIZE, out=None, overlap_previous=False):
    """y = x . w_hat^T on the tcgen05 tensor cores (batched decode, prefill).

    overlap_previous=True launches with QLIN_OVERLAP_PREVIOUS (qlin_qmm_ex):
    only valid when the preceding work on the stream does not write
    wq/scales/biases."""
    if overlap_previous:
        return _matmul("qlin_qmm_ex", x, wq, scales, biases, bits, group_size, out,
                       flags=QLIN_OVERLAP_PREVIOUS)
    return _matmul("qlin_qmm", x, wq, scales, biases, bits, group_size, out)


def linear(x, wq, scales, biases, bits, group_size=GROUP_SIZE, out=None, bias=None,
           out_dtype=None):
    """qmv below the measured crossover M, qmm above it.

    bias: optional [N] tensor in the activation dtype (a linear layer's own
    bias, added before the final rounding); out_dtype: torch.float32 for a
    float32 result, else the activation dtype (qlin_linear_ex)."""
    if bias is None and (out_dtype is None or out_dtype == x.dtype):
        return _matmul("qlin_linear", x, wq, scales, biases, bits, group_size, out)
    _need_cuda(x, wq, scales, biases)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    m, k = x.shape
    n = wq.shape[0]
    if wq.shape[1] * 32 // bits != k:
        raise ValueError("wq does not match K")
    if bias is not None:
        _need_cuda(bias)
        if bias.shape != (n,) or bias.dtype != x.dtype:
            raise ValueError("bias must be [N] in the activation dtype")
    out_dtype = out_dtype or x.dtype
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=x.device)
    _need_cuda(out)
    _check(lib().qlin_linear_ex(_ptr(x), _ptr(wq), _ptr(scales), _ptr(biases), _ptr(bias),
                                _ptr(out), m, n, k, bits, group_size, _DTYPE_CODE[x.dtype],
                                _DTYPE_CODE[out_dtype], _stream(x)))
    return out


def chain_workspace(n_links: int, device) -> torch.Tensor:
    """Device scratch for qmv_chain (one counter per link)."""
    nbytes = int(lib().qlin_qmv_chain_workspace_size(n_links))
    return torch.zeros(nbytes // 4, dtype=torch.int32, device=device)


def make_links(links):
    """ctypes array of Link from dicts with wq, scales, biases, y, input,
    input_offset (tensors must stay alive while the array is used)."""
    arr = (Link * len(links))()
    for i, d in enumerate(links):
        n, k = d["wq"].shape[0], None
        arr[i] = Link(d["wq"].data_ptr(), d["scales"].data_ptr(), d["biases"].data_ptr(),
                      d["y"].data_ptr(), n, d["K"], d.get("input", -1), d.get("input_offset", 0))
    return arr


def qmv_chain(x0, link_array, n_links, bits, dtype, workspace, group_size=GROUP_SIZE):
    """Run a chain of dependent M = 1 products in one launch (qlin_qmv_chain).

    x0: device tensor (or None); link_array: from make_links; workspace: from
    chain_workspace.  Outputs are written into each link's y."""
    dev = workspace.device
    _check(lib().qlin_qmv_chain(_ptr(x0) if x0 is not None else None, link_array, n_links,
                                bits, group_size, _DTYPE_CODE[dtype], _ptr(workspace),
                                workspace.numel() * 4,
                                ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)))


def crossover_m(n: int, k: int, bits: int, dtype: torch.dtype = torch.float16) -> int:
    """Smallest M for which linear() takes the tensor-core kernel."""
    return int(lib().qlin_crossover_m_dtype(n, k, bits, _DTYPE_CODE[dtype]))


def device_status() -> int:
    """Reads and clears the kernels' device status word (synchronises)."""
    v = ctypes.c_int(0)
    _check(lib().qlin_device_status(ctypes.byref(v)))
    return v.value
