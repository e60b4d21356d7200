"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and rounds them to the storage dtype of
the inputs (float32 weights; float16/bfloat16 activations).  It holds none of
the quantise / dequantise / matmul arithmetic, so that the CPU oracle and the
CUDA library can both consume its output without sharing any of the method.

Recipe (stands in for the Llama-3.2-1B 4-bit model the pages measure, whose
trained weights are not available):
  * weights  W[N, K] float32 ~ N(0, 0.02), drawn in blocks of ROW_BLOCK rows;
    block i of matrix ``seed`` comes from numpy PCG64 seeded with (seed, i), so
    any subset of rows can be regenerated without drawing the whole matrix;
  * activations x[M, K] ~ N(0, 1) drawn in float64, rounded to float32, an
    optional fraction of rows scaled by ``outlier_scale`` in float32, then
    rounded (ties to even) to float16 or bfloat16.
"""

from __future__ import annotations

import numpy as np
import torch

ROW_BLOCK = 1024
WEIGHT_STD = 0.02

# Llama-3.2-1B decoder linears at decode: name -> (N, K)
LLAMA_1B_LINEARS = (
    ("q_proj", 2048, 2048),
    ("k_proj", 512, 2048),
    ("v_proj", 512, 2048),
    ("o_proj", 2048, 2048),
    ("gate_proj", 8192, 2048),
    ("up_proj", 8192, 2048),
    ("down_proj", 2048, 8192),
)
LLAMA_1B_LAYERS = 16
LLAMA_1B_LM_HEAD = ("lm_head", 128256, 2048)


def weight_seed(base_seed: int, index: int) -> int:
    """Seed of the ``index``-th weight matrix of a workload."""
    return base_seed * 1000 + index


def weights_f32(seed: int, n_rows: int, k: int, rows=None, threads: int = 8) -> np.ndarray:
    """W[N, K] float32 ~ N(0, 0.02); ``rows`` selects a subset (same values).

    Row blocks are independent streams, so they are drawn on a few threads
    (numpy releases the GIL while filling); the values do not depend on it.
    """
    if rows is None:
        rows = np.arange(n_rows)
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= n_rows):
        raise IndexError("row out of range")
    out = np.empty((rows.size, k), dtype=np.float32)
    blocks = np.unique(rows // ROW_BLOCK)

    def fill(blk):
        r0 = int(blk) * ROW_BLOCK
        nb = min(ROW_BLOCK, n_rows - r0)
        rng = np.random.default_rng([seed, int(blk)])
        block = rng.standard_normal((nb, k), dtype=np.float32)
        block *= np.float32(WEIGHT_STD)
        sel = np.nonzero(rows // ROW_BLOCK == blk)[0]
        out[sel] = block[rows[sel] - r0]

    if threads > 1 and blocks.size > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(threads, blocks.size)) as ex:
            list(ex.map(fill, blocks))
    else:
        for blk in blocks:
            fill(blk)
    return out


def activations(seed: int, m: int, k: int, dtype: str, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> torch.Tensor:
    """x[M, K] ~ N(0, 1) as a CPU torch tensor of ``dtype`` ("f16" or "bf16").

    With ``outlier_frac`` > 0, round(outlier_frac * M) distinct rows (chosen by
    the same generator) are multiplied by ``outlier_scale`` in float32 before
    the final rounding.
    """
    rng = np.random.default_rng([seed, 0x5EED])
    x32 = rng.standard_normal((m, k)).astype(np.float32)
    n_out = int(round(outlier_frac * m))
    if n_out:
        rows = rng.choice(m, n_out, replace=False)
        x32[rows] *= np.float32(outlier_scale)
    if dtype == "f16":
        return torch.from_numpy(x32.astype(np.float16))
    if dtype == "bf16":
        return torch.from_numpy(x32).to(torch.bfloat16)
    raise ValueError(f"unknown activation dtype {dtype!r}")

