"""A sequence of Q4_0 matmuls captured once into a CUDA graph and replayed.

Decode runs the same list of GEMVs (one per weight matrix) for every token.
Capturing the list into a CUDA graph removes the per-launch host cost; the
kernels' programmatic-dependent-launch attribute is captured too, so each
GEMV starts streaming its weights while the previous one finishes.
"""

from __future__ import annotations

import torch

from . import Q4_LAYOUT_BLOCKS, q4_matmul_ex


class MatmulSequence:
    """calls: list of (C, A, B, M, N, K) device tensors and sizes, run in order."""

    def __init__(self, calls, workspace=None, b_layout=Q4_LAYOUT_BLOCKS):
        self.calls = list(calls)
        self.workspace = workspace
        self.b_layout = b_layout
        self.graph = None
        self.stream = torch.cuda.Stream()

    def run_eager(self, stream=None):
        for C, A, B, M, N, K in self.calls:
            q4_matmul_ex(C, A, B, M, N, K, workspace=self.workspace, stream=stream,
                         b_layout=self.b_layout)

    def capture(self):
        # one eager pass first: sizes the library-owned workspace outside capture
        with torch.cuda.stream(self.stream):
            self.run_eager()
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.run_eager()
        self.graph = g
        return self

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()
