"""A stack of weightless decoder layers.

Each layer is the projection set of one decoder layer: fused Q/K/V
(wl_qkv_fused), O (wl_linear) and the fused GeGLU MLP (wl_mlp_geglu_fused).
Two engines run it:
  "stack"  one launch per step (per 24 layers) of the library's stack kernels
           (wl_stack_create / wl_stack_decode), for T <= 32 and r <= 32;
  "graph"  the per-projection calls, captured once and replayed as one CUDA
           graph (any T and r).
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

from . import WLError, WLStack, mlp_workspace, wl_band_of_layer, wl_linear, wl_mlp_geglu_fused, wl_qkv_fused


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
                 r: int, ydt=torch.bfloat16, device=None, use_graph: bool = True, engine: str = "auto"):
        """engine: "stack", "graph" or "auto" (the stack kernel where it takes
        the sizes, else the graph)."""
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
        # decode path (T <= 8) and on the prefill path where the gate/up kernel
        # forms h itself (rank padded to 16 at most 32), else 3 (gate/up, GELU,
        # down)
        lin = 1
        mlp = 2 if (T <= 8 or (r + 15) // 16 * 16 <= 32) else 3
        self.launches_per_step = len(layers) * (2 * lin + mlp)
        self.kernel_launches_per_step = self.launches_per_step
        self.stk = None
        if engine not in ("auto", "stack", "graph"):
            raise ValueError(f"unknown engine {engine!r}")
        if engine in ("auto", "stack"):
            try:
                self.stk = WLStack(layers, T, device=self.dev)
            except WLError:
                if engine == "stack":
                    raise
        self.engine = "stack" if self.stk is not None else "graph"
        if self.stk is not None:
            # one stack-kernel launch per 24 layers, preceded by the V^T pass
            # (r > 0; above 4 tokens that pass also clears the step's flags and
            # always runs)
            self.kernel_launches_per_step = (len(layers) + 23) // 24
            self.launches_per_step = self.kernel_launches_per_step + (1 if (r > 0 or T > 4) else 0)

    @property
    def out(self) -> torch.Tensor:
        if self.stk is not None:
            return self.stk.out
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
        """Warm up once eagerly, then capture the whole stack in a graph
        (the stack engine needs no graph: a step is one launch per 24 layers)."""
        if self.stk is not None:
            self.stk.decode(self.x, stream=self.stream)
            self.stream.synchronize()
            return
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
        if self.stk is not None:
            if mlp_events is not None:
                raise ValueError("per-MLP events need the graph engine")
            self.stk.decode(self.x, stream=self.stream)
            return
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


def materialize_layers(layers: list[LayerTheta], dt=torch.bfloat16) -> list[LayerTheta]:
    """The precompute path ("Serve and generate with weightless", fast path):
    each projection's W_eff = s*W0 + U V^T formed once by wl_materialize, as
    bundles of rank 0 with s = 1, so that a stack runs them as dense weights."""
    import wl_synth

    from . import wl_materialize

    out = []
    for th in layers:
        fams = {}
        for fam in ("q", "k", "v", "o", "gate", "up", "down"):
            t = getattr(th, fam)
            U = t.U if t.U is not None and t.U.shape[1] > 0 else None
            V = t.V if U is not None else None
            W = wl_materialize(t.W0, t.s, U, V, dt=dt)
            o, i = W.shape
            fams[fam] = wl_synth.Theta(W, torch.ones(o, dtype=torch.float32, device=W.device),
                                       torch.zeros(o, 0, dtype=torch.bfloat16, device=W.device),
                                       torch.zeros(i, 0, dtype=torch.bfloat16, device=W.device))
        out.append(LayerTheta(**fams))
    # the decode launches read weights while the previous kernel on the stream
    # finishes: the bundles are complete before any of them runs
    if out:
        torch.cuda.current_stream(out[0].q.W0.device).synchronize()
    return out

