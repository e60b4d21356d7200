"""A Llama-3.2-1B-shaped decode step made only of fused packed linears.

Sixteen layers of the seven decoder linears (q, k, v, o, gate, up, down) plus
the lm_head, M = 1, every weight distinct and resident packed in HBM.  As in
most inference engines, q/k/v and gate/up are stored as one fused matrix each
(their rows concatenated; quantisation is per row and group, so this changes
no bit of any row), which makes the step 4 launches per layer + 1 = 65.  The
launches are chained the way a decoder's linears depend on each other, with
the non-linear parts (attention, norms, activation) left out:

    qkv      <- x_l
    o        <- y_q          (stands in for the attention output)
    gate_up  <- y_o          (stands in for the normed residual)
    down     <- y_gate       (stands in for act(gate) * up)
    x_{l+1}  =  y_down
    logits   <- lm_head(x_16)

so each launch reads what the previous one wrote.  Every launch after the
first is a programmatic dependent launch: it starts streaming its (resident,
never rewritten) weights while its predecessor finishes, and reads its input
only after the predecessor completes.  The pages measure the packed decode step
at ~678 dispatches ("epic: realize low-precision / quantized performance on the
OpenXLA (IREE) backend", section "The measured fusion gate").
"""

from __future__ import annotations

import torch

from . import chain_workspace, dequant, make_links, qmv, qmv_chain, quantize_affine
from . import synthetic as S

_FUSED = (("qkv", ("q_proj", "k_proj", "v_proj")), ("o", ("o_proj",)),
          ("gate_up", ("gate_proj", "up_proj")), ("down", ("down_proj",)))


def _round_up(v: int, a: int = 256) -> int:
    return (v + a - 1) // a * a


class DecodeStep:
    def __init__(self, device, bits: int = 8, dtype: torch.dtype = torch.float16,
                 seed: int = 2, layers: int = S.LLAMA_1B_LAYERS, lm_head: bool = True,
                 overlap: bool = True, mode: str = "launches"):
        """mode "launches": one qlin_qmv launch per fused linear (overlapped
        with programmatic dependent launch when ``overlap``; the faster mode on
        GB300); mode "chain": the whole step is one qlin_qmv_chain launch.

        All packed weights, scales and biases live in one device region, in
        launch order (each piece 256-byte aligned)."""
        self.device = torch.device(device)
        self.bits = bits
        self.dtype = dtype
        self.overlap = overlap
        self.mode = mode
        shapes = {name: (n, k) for name, n, k in S.LLAMA_1B_LINEARS}
        # original linears, in the order of the weight seeds:
        # (name, layer, N, K, unit index, first row in the unit, weight seed)
        self.linears = []
        specs = []  # per unit: name, layer, N, K, [(weight seed, rows)]
        idx = 0
        for layer in range(layers):
            seeds = {}
            for name, n, k in S.LLAMA_1B_LINEARS:
                seeds[name] = S.weight_seed(seed, idx)
                idx += 1
            for uname, parts in _FUSED:
                k = shapes[parts[0]][1]
                rows, srcs = 0, []
                for p in parts:
                    n = shapes[p][0]
                    self.linears.append((p, layer, n, k, len(specs), rows, seeds[p]))
                    srcs.append((seeds[p], n))
                    rows += n
                specs.append((uname, layer, rows, k, srcs))
        if lm_head:
            name, n, k = S.LLAMA_1B_LM_HEAD
            wseed = S.weight_seed(seed, idx)
            self.linears.append((name, layers, n, k, len(specs), 0, wseed))
            specs.append((name, layers, n, k, [(wseed, n)]))
        # the weight region: wq, scales, biases of every unit in launch order
        es = torch.empty((), dtype=dtype).element_size()
        offs, total = [], 0
        for (_, _, n, k, _) in specs:
            wq_b, sc_b = n * k * bits // 8, n * (k // 64) * es
            offs.append((total, total + _round_up(wq_b), total + _round_up(wq_b) + _round_up(sc_b)))
            total += _round_up(wq_b) + 2 * _round_up(sc_b)
        self.region = torch.empty(total, dtype=torch.uint8, device=self.device)
        self.units = []  # dicts: name, layer, N, K, wq, scales, biases, out, offset, span
        for (uname, layer, n, k, srcs), (o_w, o_s, o_b) in zip(specs, offs):
            wq_b, sc_b = n * k * bits // 8, n * (k // 64) * es
            views = (self.region[o_w:o_w + wq_b].view(torch.int32).view(n, k * bits // 32),
                     self.region[o_s:o_s + sc_b].view(dtype).view(n, k // 64),
                     self.region[o_b:o_b + sc_b].view(dtype).view(n, k // 64))
            w = torch.cat([torch.from_numpy(S.weights_f32(ws, wn, k)) for ws, wn in srcs])
            quantize_affine(w.to(self.device), bits, sdtype=dtype, out=views)
            del w
            end = o_b + _round_up(sc_b)
            self.units.append(dict(name=uname, layer=layer, N=n, K=k, wq=views[0],
                                   scales=views[1], biases=views[2],
                                   out=torch.empty((1, n), dtype=dtype, device=self.device),
                                   offset=o_w, span=end - o_w))
        self.layers = layers
        hidden = S.LLAMA_1B_LINEARS[0][2]
        self.x0 = torch.zeros((1, hidden), dtype=dtype, device=self.device)
        self.graph = None
        self._build_chain()

    def _build_chain(self):
        """The link table of the step (same chaining as input_of)."""
        links = []
        for u, d in enumerate(self.units):
            name = d["name"]
            if name == "qkv":
                inp, off = (-1, 0) if u == 0 else (u - 1, 0)
            elif name == "o":
                inp, off = u - 1, 0            # q rows of the fused qkv output
            elif name == "gate_up":
                inp, off = u - 1, 0
            elif name == "down":
                inp, off = u - 1, 0            # gate rows of the fused gate_up output
            else:
                inp, off = (u - 1, 0) if u else (-1, 0)
            links.append(dict(wq=d["wq"], scales=d["scales"], biases=d["biases"], y=d["out"],
                              K=d["K"], input=inp, input_offset=off))
        self._links = make_links(links)
        self._workspace = chain_workspace(len(links), self.device)

    # ------------------------------------------------------------------ sizes
    @property
    def n_launches(self) -> int:
        return len(self.units)

    def packed_bytes(self) -> int:
        """Bytes of codes + scales + biases streamed per step."""
        return sum(u["wq"].numel() * 4 + (u["scales"].numel() + u["biases"].numel()) *
                   u["scales"].element_size() for u in self.units)

    def algorithmic_bytes(self):
        """Per launch: packed weights + x read + y written."""
        es = self.x0.element_size()
        return [u["wq"].numel() * 4 + (u["scales"].numel() + u["biases"].numel()) *
                u["scales"].element_size() + (u["K"] + u["N"]) * es for u in self.units]

    # ---------------------------------------------------------------- launches
    def input_of(self, u: int) -> torch.Tensor:
        """The tensor launch ``u`` reads in the chained step."""
        name = self.units[u]["name"]
        if name == "qkv":
            return self.x0 if u == 0 else self.units[u - 1]["out"]
        if name == "o":
            return self.units[u - 1]["out"][:, :2048]            # q
        if name == "gate_up":
            return self.units[u - 1]["out"]
        if name == "down":
            return self.units[u - 1]["out"][:, :8192]            # gate
        return self.units[u - 1]["out"] if u else self.x0      # lm_head

    def launch(self, u: int, x: torch.Tensor, out: torch.Tensor | None = None,
               overlap: bool = False):
        d = self.units[u]
        return qmv(x, d["wq"], d["scales"], d["biases"], self.bits,
                   out=d["out"] if out is None else out, overlap_previous=overlap)

    def launch_chain(self):
        qmv_chain(self.x0, self._links, len(self.units), self.bits, self.dtype, self._workspace)

    def run_step(self):
        """One decode step in the configured mode (eager)."""
        if self.mode == "chain":
            self.launch_chain()
        else:
            self.launch_all()

    def launch_all(self, per_launch_hook=None):
        for u in range(len(self.units)):
            if per_launch_hook:
                per_launch_hook(u, "before")
            self.launch(u, self.input_of(u), overlap=self.overlap and u > 0)
            if per_launch_hook:
                per_launch_hook(u, "after")

    def capture(self, stream: torch.cuda.Stream | None = None):
        """Capture one step into a CUDA graph (after one eager warm-up)."""
        self.run_step()
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.run_step()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

    @property
    def logits(self) -> torch.Tensor:
        return self.units[-1]["out"]

    # ----------------------------------------------- per original linear (tests)
    def linear_rows(self, i: int):
        """(name, layer, N, K, wq rows, scales rows, biases rows, weight seed)."""
        name, layer, n, k, u, r0, wseed = self.linears[i]
        d = self.units[u]
        return (name, layer, n, k, d["wq"][r0:r0 + n], d["scales"][r0:r0 + n],
                d["biases"][r0:r0 + n], wseed)

    def run_linear(self, i: int, x: torch.Tensor):
        """Linear ``i`` on an arbitrary input, through its unit's own launch."""
        name, layer, n, k, u, r0, wseed = self.linears[i]
        out = torch.empty((x.shape[0], self.units[u]["N"]), dtype=self.dtype, device=self.device)
        self.launch(u, x, out=out)
        return out[:, r0:r0 + n]


class DenseF16Step:
    """The same decode step with every weight resident as a dense matrix in
    the activation dtype, materialised once by qlin_dequant, and each linear
    run by torch.matmul (cuBLAS): the unfused, f16-resident path that the
    packed one has to beat ("epic: realize low-precision / quantized
    performance on the OpenXLA (IREE) backend", section "Thesis", item 1;
    "track(upstream-iree): fused dequant->matmul for the packed int8 bandwidth
    win", section "Unblock criteria").  A comparator, not the product path."""

    def __init__(self, step: DecodeStep):
        self.step = step
        self.weights = [dequant(u["wq"], u["scales"], u["biases"], step.bits)
                        for u in step.units]
        self.outs = [torch.empty_like(u["out"]) for u in step.units]
        self.graph = None

    def weight_bytes(self) -> int:
        return sum(w.numel() * w.element_size() for w in self.weights)

    def input_of(self, u: int) -> torch.Tensor:
        """Same chaining as DecodeStep.input_of, on this step's outputs."""
        name = self.step.units[u]["name"]
        if u == 0:
            return self.step.x0
        prev = self.outs[u - 1]
        if name == "o":
            return prev[:, :2048]
        if name == "down":
            return prev[:, :8192]
        return prev

    def run_step(self):
        for u, w in enumerate(self.weights):
            torch.matmul(self.input_of(u), w.t(), out=self.outs[u])

    def capture(self):
        self.run_step()
        torch.cuda.synchronize(self.step.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run_step()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

    def run_linear(self, i: int, x: torch.Tensor) -> torch.Tensor:
        """Original linear ``i`` on an arbitrary input."""
        name, layer, n, k, u, r0, wseed = self.step.linears[i]
        return torch.matmul(x, self.weights[u][r0:r0 + n].t())
