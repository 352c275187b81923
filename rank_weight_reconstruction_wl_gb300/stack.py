"""A stack of weightless decoder layers, replayed as one CUDA graph.

Each layer is the projection set of one decoder layer: fused Q/K/V
(wl_qkv_fused), O (wl_linear) and the fused GeGLU MLP (wl_mlp_geglu_fused).
The method does not include attention, so the O projection takes the q output
as its stand-in input, the MLP takes the O output, and the MLP output is the
next layer's input (no norms, no residual).  Layer l uses W0 block
wl_band_of_layer(l, L, G) of each family ("What weightless inference costs",
Compression: G shared blocks; "Serve and generate with weightless": G = L is
the passthrough point).

The graph only replays the library's own launches: capture is plumbing; every
arithmetic step runs in libwl.so's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import mlp_workspace, wl_band_of_layer, wl_linear, wl_mlp_geglu_fused, wl_qkv_fused


@dataclass
class LayerTheta:
    q: object
    k: object
    v: object
    o: object
    gate: object
    up: object
    down: object


class DecoderStack:
    """L layers sharing W0 per band; fixed T; inputs/outputs in device buffers."""

    def __init__(self, layers: list[LayerTheta], T: int, hidden: int, qdim: int, inter: int,
                 r: int, ydt=torch.bfloat16, device=None, use_graph: bool = True):
        self.layers = layers
        self.T, self.hidden, self.qdim, self.inter, self.r = T, hidden, qdim, inter, r
        self.dev = torch.device(device or "cuda")
        self.ydt = ydt
        kv = layers[0].k.W0.shape[0]
        z = dict(dtype=torch.bfloat16, device=self.dev)
        self.x = torch.zeros(T, hidden, **z)
        self.yq = torch.empty(T, qdim, **z)
        self.yk = torch.empty(T, kv, **z)
        self.yv = torch.empty(T, kv, **z)
        self.yo = torch.empty(T, hidden, **z)
        self.ym = [torch.empty(T, hidden, **z) for _ in range(2)]
        self.ws = mlp_workspace(T, hidden, inter, r, torch.bfloat16, self.dev)
        self.stream = torch.cuda.Stream(self.dev)
        self.graph = None
        self.use_graph = use_graph
        # kernels per layer: fused QKV 1, O 1; the MLP is 2 (gate/up, down) on the
        # decode path (T <= 8) and 3 (gate/up, GELU, down) on the prefill path
        lin = (T + 63) // 64 if T <= 64 else 1
        mlp = 2 if T <= 8 else 3
        self.launches_per_step = len(layers) * (2 * lin + mlp)

    @property
    def out(self) -> torch.Tensor:
        return self.ym[(len(self.layers) - 1) % 2]

    def _issue(self, mlp_events=None):
        x = self.x
        for l, th in enumerate(self.layers):
            wl_qkv_fused(x, th.q, th.k, th.v, outs=(self.yq, self.yk, self.yv),
                         stream=self.stream)
            wl_linear(self.yq, th.o.W0, th.o.s, th.o.U, th.o.V, y=self.yo, stream=self.stream)
            ym = self.ym[l % 2]
            if mlp_events is not None:
                mlp_events[l][0].record(self.stream)
            wl_mlp_geglu_fused(self.yo, th.gate, th.up, th.down, y=ym, workspace=self.ws,
                               stream=self.stream)
            if mlp_events is not None:
                mlp_events[l][1].record(self.stream)
            x = ym

    def capture(self):
        """Warm up once eagerly, then capture the whole stack in a graph."""
        with torch.cuda.stream(self.stream):
            self._issue()
        self.stream.synchronize()
        if not self.use_graph:
            return
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self._issue()
        self.graph = g

    def step(self, mlp_events=None):
        """One pass over all layers on self.stream (graph replay if captured)."""
        if mlp_events is not None or self.graph is None:
            with torch.cuda.stream(self.stream):
                self._issue(mlp_events)
        else:
            with torch.cuda.stream(self.stream):
                self.graph.replay()

    def forward_host(self, x_host: torch.Tensor, y_host: torch.Tensor):
        """End to end: pinned host x -> device, one stack pass, result -> pinned host."""
        with torch.cuda.stream(self.stream):
            self.x.copy_(x_host, non_blocking=True)
            self.step()
            y_host.copy_(self.out, non_blocking=True)


def build_layers(L: int, G: int, T: int, shapes: dict, r: int, seed: int = 0, device="cuda",
                 kind: str = "random") -> list[LayerTheta]:
    """Seeded synthetic layers; W0 shared per band (G blocks per family), s, U, V per layer."""
    import wl_synth

    hidden, qd, kv, inter = shapes["hidden"], shapes["q"], shapes["kv"], shapes["inter"]
    dims = {"q": (hidden, qd), "k": (hidden, kv), "v": (hidden, kv), "o": (qd, hidden),
            "gate": (hidden, inter), "up": (hidden, inter), "down": (inter, hidden)}
    g = wl_synth.make_generator(seed, device)
    blocks = {}
    layers = []
    for l in range(L):
        b = wl_band_of_layer(l, L, G)
        fams = {}
        for fam, (inp, out) in dims.items():
            th = wl_synth.draw_theta(g, inp, out, r, kind)
            if (fam, b) in blocks:
                th.W0 = blocks[(fam, b)]
            else:
                blocks[(fam, b)] = th.W0
            fams[fam] = th
        layers.append(LayerTheta(**fams))
    return layers
