"""Shared helpers of the GPU parity tests (seeded inputs, oracle references,
guard bands)."""

import numpy as np
import torch

from int8_qmv_qmm_gb300 import synthetic as S
from oracle import qlin_oracle as O

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
CANARY = 64  # guard elements on each side of an output


def case(seed, m, n, k, bits, dt, outlier_frac=0.0):
    """Seeded weights/activations and the oracle's full reference."""
    w = S.weights_f32(seed, n, k)
    x = S.activations(seed, m, k, dt, outlier_frac)
    ref = O.linear_ref(x.float().numpy().astype(np.float64), w, bits, 64, dt)
    return w, x, ref


def guarded(shape, dtype, dev):
    """An output tensor with canary bands before and after it."""
    numel = int(np.prod(shape))
    buf = torch.full((numel + 2 * CANARY,), 1234.0, dtype=dtype, device=dev)
    return buf, buf[CANARY:CANARY + numel].view(*shape)


def canaries_intact(buf):
    head, tail = buf[:CANARY], buf[-CANARY:]
    return bool((head == 1234.0).all()) and bool((tail == 1234.0).all())


def as_u32(t):
    return t.cpu().numpy().view(np.uint32)


def as_u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def assert_within_tolerance(y, ref, what=""):
    y64 = y.float().cpu().numpy().astype(np.float64)
    ok = O.within_tolerance(y64, ref["y_ref"], ref["a_ref"])
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(y64[tuple(i)]), float(ref["y_ref"][tuple(i)]),
                   float(ref["a_ref"][tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; "
                             f"first (index, gpu, ref, sum|xw|): {detail}")
