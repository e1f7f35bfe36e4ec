"""A decode step over a stack of layers, captured once as a CUDA graph.

Every layer of a decoder appends one K/V token per sequence to its own INT2
cache and attends over it.  One step of an L-layer stack is therefore L
kvq_append_decode calls (or L kvq_append + kvq_decode pairs), 3 (or 4) kernel
launches each, on one stream.  Captured as a CUDA graph it is replayed with one
launch from the host; the kernels inside keep their programmatic dependencies,
so each is resident and waiting when its predecessor finishes.

The graph reads its inputs from fixed device buffers that the caller fills
before each replay (``K_new``, ``V_new``, ``q``, ``seq_lens``, ``positions``)
and writes ``out``.  Only the library's entry points run inside the graph; this
module holds buffers and the capture, nothing of the method's arithmetic.
"""
from __future__ import annotations

import torch

from . import kvq as K


class LayerCache:
    """One layer's cache: a handle with its rotation bank, pool and page table."""

    def __init__(self, handle: K.Handle, pool: torch.Tensor, num_pool_pages: int,
                 page_table: torch.Tensor):
        self.h, self.pool, self.npool, self.pt = handle, pool, int(num_pool_pages), page_table


class DecodeStepGraph:
    """Fixed buffers and the captured step of ``len(layers)`` layers.

    K_new, V_new : bf16 [L, B, Hkv, 128]  the new token of every sequence, per layer
    q            : bf16 [L, B, H, 128]
    seq_lens     : int32 [B]               context after the append (all layers)
    positions    : int32 [B]               seq_lens - 1 (read by the unfused form only)
    out          : fp32 [L, B, H, 128]
    fused=True runs kvq_append_decode per layer, else kvq_append then kvq_decode.
    """

    def __init__(self, layers, batch: int, num_heads: int, num_kv_heads: int, fused: bool = True,
                 num_splits: int = 0, device="cuda"):
        self.layers = list(layers)
        self.B, self.H, self.Hkv = batch, num_heads, num_kv_heads
        self.fused = fused
        L = len(self.layers)
        max_pages = int(self.layers[0].pt.shape[1])
        self.splits = num_splits or K.kvq_auto_splits(self.layers[0].h, batch, max_pages)
        self.K_new = torch.zeros((L, batch, num_kv_heads, 128), dtype=torch.int16, device=device)
        self.V_new = torch.zeros_like(self.K_new)
        self.q = torch.zeros((L, batch, num_heads, 128), dtype=torch.int16, device=device)
        self.seq_lens = torch.ones(batch, dtype=torch.int32, device=device)
        self.positions = torch.zeros(batch, dtype=torch.int32, device=device)
        self.seq_idx = torch.arange(batch, dtype=torch.int32, device=device)
        self.out = torch.zeros((L, batch, num_heads, 128), dtype=torch.float32, device=device)
        # layers run one after another on one stream: one workspace serves all
        self.ws = torch.empty(K.kvq_workspace_bytes(self.layers[0].h, batch, self.splits),
                              dtype=torch.uint8, device=device)
        self.graph = None

    def run(self):
        """One step, launched eagerly on the current stream."""
        for i, c in enumerate(self.layers):
            if self.fused:
                K.kvq_append_decode(c.h, c.pool, c.npool, self.K_new[i], self.V_new[i], self.q[i],
                                    c.pt, self.seq_lens, self.out[i], self.ws, self.splits)
            else:
                K.kvq_append(c.h, c.pool, c.npool, self.K_new[i], self.V_new[i], self.seq_idx,
                             self.positions, c.pt)
                K.kvq_decode(c.h, c.pool, c.npool, self.q[i], c.pt, self.seq_lens, self.out[i],
                             self.ws, self.splits)

    def capture(self):
        """Capture run() as a CUDA graph, after one eager step (which sets the
        kernels' attributes outside the capture and stores the tokens now in
        the buffers)."""
        self.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        torch.cuda.synchronize()
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()

    def load(self, K_new=None, V_new=None, q=None, seq_lens=None, positions=None):
        """Copy one step's inputs (device tensors of the buffers' shapes) in.
        The unfused form also needs positions (= seq_lens - 1)."""
        for dst, src in ((self.K_new, K_new), (self.V_new, V_new), (self.q, q),
                         (self.seq_lens, seq_lens), (self.positions, positions)):
            if src is not None:
                dst.copy_(src, non_blocking=True)
