"""A Llama-3.2-1B-shaped decode step made only of fused packed linears.

Sixteen layers of the seven decoder linears (q, k, v, o, gate, up, down) plus
the lm_head, M = 1, every weight distinct and resident packed in HBM.  The
launches are chained the way a decoder's linears depend on each other, with
the non-linear parts (attention, norms, activation) left out:

    q, k, v   <- x_l                    (shared input)
    o         <- y_q                    (stands in for the attention output)
    gate, up  <- y_o                    (stands in for the normed residual)
    down      <- y_gate                 (stands in for act(gate) * up)
    x_{l+1}   =  y_down
    logits    <- lm_head(x_16)

so each launch reads what the previous one wrote: stream order serialises
them exactly as a real decode step would.  The pages measure the packed decode
step at ~678 dispatches ("epic: realize low-precision / quantized performance
on the OpenXLA (IREE) backend", section "The measured fusion gate"); here it is
113 launches of the fused kernel, captured once into a CUDA graph.
"""

from __future__ import annotations

import torch

from . import qmv, quantize_affine
from . import synthetic as S


class DecodeStep:
    def __init__(self, device, bits: int = 8, dtype: torch.dtype = torch.float16,
                 seed: int = 2, layers: int = S.LLAMA_1B_LAYERS, lm_head: bool = True,
                 progress=None):
        self.device = torch.device(device)
        self.bits = bits
        self.dtype = dtype
        self.linears = []  # (name, layer, N, K, wq, scales, biases, weight seed)
        idx = 0
        for layer in range(layers):
            for name, n, k in S.LLAMA_1B_LINEARS:
                self._add(name, layer, n, k, S.weight_seed(seed, idx))
                idx += 1
                if progress:
                    progress(idx)
        if lm_head:
            name, n, k = S.LLAMA_1B_LM_HEAD
            self._add(name, layers, n, k, S.weight_seed(seed, idx))
        self.layers = layers
        hidden = S.LLAMA_1B_LINEARS[0][2]
        self.x0 = torch.zeros((1, hidden), dtype=dtype, device=self.device)
        self.outputs = [torch.empty((1, n), dtype=dtype, device=self.device)
                        for (_, _, n, _, _, _, _, _) in self.linears]
        self.graph = None

    def _add(self, name, layer, n, k, wseed):
        w = torch.from_numpy(S.weights_f32(wseed, n, k)).to(self.device)
        wq, sc, bi = quantize_affine(w, self.bits, sdtype=self.dtype)
        del w
        self.linears.append((name, layer, n, k, wq, sc, bi, wseed))

    # ------------------------------------------------------------------ sizes
    @property
    def n_launches(self) -> int:
        return len(self.linears)

    def packed_bytes(self) -> int:
        """Bytes of codes + scales + biases streamed per step."""
        tot = 0
        for (_, _, n, k, wq, sc, bi, _) in self.linears:
            tot += wq.numel() * 4 + sc.numel() * sc.element_size() + bi.numel() * bi.element_size()
        return tot

    def algorithmic_bytes(self):
        """Per launch: packed weights + x read + y written."""
        out = []
        for (_, _, n, k, wq, sc, bi, _) in self.linears:
            out.append(wq.numel() * 4 + (sc.numel() + bi.numel()) * sc.element_size()
                       + (k + n) * self.x0.element_size())
        return out

    # ---------------------------------------------------------------- launches
    def input_of(self, i: int) -> torch.Tensor:
        """The tensor linear ``i`` reads in the chained step."""
        name, layer = self.linears[i][0], self.linears[i][1]
        base = 7 * layer
        if name in ("q_proj", "k_proj", "v_proj"):
            return self.x0 if layer == 0 else self.outputs[base - 1]
        if name == "o_proj":
            return self.outputs[base + 0]
        if name in ("gate_proj", "up_proj"):
            return self.outputs[base + 3]
        if name == "down_proj":
            return self.outputs[base + 4]
        # lm_head
        return self.outputs[base - 1] if self.layers else self.x0

    def run_linear(self, i: int, x: torch.Tensor, out: torch.Tensor | None = None):
        """Linear ``i`` on an arbitrary input (same kernel and launch config)."""
        _, _, n, k, wq, sc, bi, _ = self.linears[i]
        return qmv(x, wq, sc, bi, self.bits, out=out)

    def launch_all(self, per_launch_hook=None):
        for i in range(len(self.linears)):
            _, _, n, k, wq, sc, bi, _ = self.linears[i]
            if per_launch_hook:
                per_launch_hook(i, "before")
            qmv(self.input_of(i), wq, sc, bi, self.bits, out=self.outputs[i])
            if per_launch_hook:
                per_launch_hook(i, "after")

    def capture(self, stream: torch.cuda.Stream | None = None):
        """Capture one step into a CUDA graph (after one eager warm-up)."""
        self.launch_all()
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.launch_all()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

    @property
    def logits(self) -> torch.Tensor:
        return self.outputs[-1]

