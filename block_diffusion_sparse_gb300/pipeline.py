"""Dual-stream block pipeline over double-buffered sparse KV pools.

HERALD early abstract: selection and denoising run as a dual-stream pipeline
over double-buffered sparse KV pools; HERALD v3 abstract: while the current
block is denoised, stage 1 searches the full cache for the next block with
the merged query of the current block's queries, and stage 2 refines the
candidates with the next block's real queries.

Per block i (one layer), with `den` the denoising stream and `sel` the
selection stream:

    den: stage 2 (cand[i%2], block i's first-step queries) -> idx, n_sel
    den: gather -> pool[i%2]
    sel: stage 1 for block i+1 from block i's first-step queries
         -> cand[(i+1)%2]                         (overlaps the T steps below)
    den: T x sparse block attention over pool[i%2]
    den: wait for sel; append block i's final K/V

Stage 1 of block i+1 scans the cache before block i is appended; block i's
positions reach block i+1's selection through the local window.  The two
streams use separate workspaces.  Only stream/event plumbing lives here:
every step of the path is a call into libherald.so.
"""
from __future__ import annotations

from . import herald as H


class BlockPipeline:
    def __init__(self, dims: H.Dims, C: int, K: int, S: int, W: int, P: int, T: int,
                 den_stream=None, sel_stream=None):
        import torch
        self.torch = torch
        self.d, self.C, self.K, self.S, self.W, self.P, self.T = dims, C, K, S, W, P, T
        NG = (dims.N, dims.Hkv)
        dev = "cuda"
        self.ws_bytes = H.herald_workspace_size(dims, C, P)
        self.ws_den = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.ws_sel = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.cand = [torch.full((*NG, C), -1, dtype=torch.int32, device=dev) for _ in range(2)]
        self.n_cand = [torch.zeros(NG, dtype=torch.int32, device=dev) for _ in range(2)]
        self.idx = torch.full((*NG, P), -1, dtype=torch.int32, device=dev)
        self.n_sel = torch.zeros(NG, dtype=torch.int32, device=dev)
        self.pool_k = [torch.zeros((*NG, P, dims.d), dtype=torch.int16, device=dev)
                       for _ in range(2)]
        self.pool_v = [torch.zeros_like(self.pool_k[0]) for _ in range(2)]
        self.den = den_stream
        self.sel = sel_stream if sel_stream is not None else torch.cuda.Stream()

    def _den(self):
        return self.den if self.den is not None else self.torch.cuda.current_stream()

    def prime(self, q_merge, k_cache, ctx, slot: int = 0):
        """Stage 1 for the first block (no predecessor: its own queries)."""
        H.herald_select_stage1(self.d, q_merge, k_cache, ctx, self.C, self.cand[slot],
                               self.n_cand[slot], self.ws_sel, self.ws_bytes, self._den())

    def block(self, i: int, q_steps, block_k, block_v, k_cache, v_cache, ctx, out,
              next_k_cache=None, advance: bool = True, overlap: bool = True):
        """Runs block i: q_steps/block_k/block_v hold the T steps' inputs,
        out[t] receives step t's attention output."""
        torch = self.torch
        den, sel = self._den(), self.sel
        cur, nxt = i % 2, (i + 1) % 2
        nk = k_cache if next_k_cache is None else next_k_cache
        d = self.d
        # stage 1 for block i+1 can start now: block i's queries exist
        sel.wait_stream(den)
        H.herald_select_stage2(d, q_steps[0], k_cache, ctx, self.cand[cur], self.n_cand[cur],
                               self.C, self.K, self.S, self.W, self.P, self.idx, self.n_sel,
                               self.ws_den, self.ws_bytes, den)
        H.herald_gather(d, self.idx, self.n_sel, self.P, k_cache, v_cache, self.pool_k[cur],
                        self.pool_v[cur], den)
        if not overlap:
            H.herald_select_stage1(d, q_steps[0], nk, ctx, self.C, self.cand[nxt],
                                   self.n_cand[nxt], self.ws_sel, self.ws_bytes, den)
        else:
            with torch.cuda.stream(sel):
                H.herald_select_stage1(d, q_steps[0], nk, ctx, self.C, self.cand[nxt],
                                       self.n_cand[nxt], self.ws_sel, self.ws_bytes, sel)
        for t in range(self.T):
            H.herald_denoise_attn(d, q_steps[t], self.pool_k[cur], self.pool_v[cur], self.n_sel,
                                  self.P, block_k[t], block_v[t], out[t], 0.0, self.ws_den,
                                  self.ws_bytes, den)
        if overlap:
            den.wait_stream(sel)
        H.herald_append_kv(d, block_k[self.T - 1], block_v[self.T - 1], ctx, k_cache, v_cache,
                           advance, den)
