"""Dual-stream block pipeline over double-buffered sparse KV pools.

HERALD early abstract: selection and denoising run as a dual-stream pipeline
over double-buffered sparse KV pools; HERALD v3 abstract: while the current
block is denoised, stage 1 searches the full cache for the next block with
the merged query of the current block's queries, and stage 2 refines the
candidates with the next block's real queries.

Per block i (one layer), with `den` the denoising stream and `sel` the
selection stream:

    den: stage 2 (cand[i%2], block i's first-step queries) -> idx, n_sel,
         with the gather -> pool[i%2] (herald_select_stage2_gather)
    sel: stage 1 for block i+1 from block i's first-step queries
         -> cand[(i+1)%2]                         (overlaps the T steps below)
    den: T-1 x sparse block attention over pool[i%2] (steps after the first
         load the settled pool before their predecessor ends)
    den: wait for sel; the last attention step, which also appends block i's
         final K/V to the cache (one kernel)

Stage 1 of block i+1 scans the cache before block i is appended; block i's
positions reach block i+1's selection through the local window.  The two
streams use separate workspaces.  Only stream/event plumbing lives here:
every step of the path is a call into libherald.so.
"""
from __future__ import annotations

import functools

from . import herald as H


# cache bytes one SM of the background scan streams: ~7 us at the ~150 GB/s
# one SM sustains, well inside the denoising steps the scan hides behind
SCAN_BYTES_PER_SM = 1 << 20
# SMs of the background scan of a cache in host memory: the host link, not
# the SMs, bounds it
HOST_SCAN_SMS = 64


@functools.lru_cache(maxsize=None)
def _sm_count(device: int) -> int:
    import torch
    return torch.cuda.get_device_properties(device).multi_processor_count


def background_sms(dims: H.Dims, host: bool = False) -> int:
    """SMs for the stage-1 scan that runs beside the denoising steps (0 = all).

    A persistent scan over every SM delays the denoising kernels, whose CTAs
    (and, with programmatic launch, those of the next step) need SMs of
    their own; confined to about one SM per MiB of keys it still ends in
    time.  On the 32K layer (34 MB of keys) 24-40 SMs took the block step
    from 94.7 to 92 us, 16 made stage 1 the longer stream (109 us); a cache
    that needs most of the SMs' bandwidth anyway (4 x 64K: 537 MB) keeps
    them all (32 SMs: 674 against 521 us).  A cache in host memory is read
    at the link's rate by a few dozen SMs: 64 took the 128K host-resident
    layer from 1661 to 1494 us per block (32: 1517, 96: 1528)."""
    import torch
    n_sm = _sm_count(torch.cuda.current_device())
    if host:
        return min(HOST_SCAN_SMS, n_sm)
    key_bytes = dims.N * dims.Hkv * dims.L_max * dims.d * 2
    want = max(32, -(-key_bytes // SCAN_BYTES_PER_SM))
    return 0 if want >= n_sm // 2 else want


def scan_sms(dims: H.Dims, k_cache, fixed=None) -> int:
    """The background scan's SM budget for this cache: `fixed` if given, else
    background_sms for a cache in device or (a CPU tensor) pinned host memory."""
    if fixed is not None:
        return fixed
    host = getattr(k_cache, "device", None) is not None and k_cache.device.type == "cpu"
    return background_sms(dims, host=host)


# CTAs of herald_stage_candidates's copy (a bounded grid on the selection
# stream; the library's constant)
STAGE_CTAS = 64


def attn_sm_flags(background: int) -> int:
    """herald_denoise_attn_ex's SM-budget bits when `background` SMs are held
    by the selection stream's work (0 = none, or every SM: no budget), so
    that every cluster of an attention step still fits at once."""
    import torch
    n_sm = _sm_count(torch.cuda.current_device())
    if background <= 0 or background >= n_sm:
        return 0
    return H.HERALD_ATTN_SMS(n_sm - background)


def step_flags(t: int, T: int, advance: bool) -> int:
    """herald_denoise_attn_ex flags of denoising step t of T: steps after the
    first find the pool settled (written before step 0, a herald call on the
    same stream); the last also appends the block to the cache (and advances
    the context when asked)."""
    flags = H.HERALD_ATTN_SETTLED if t > 0 else 0
    if t == T - 1:
        flags |= H.HERALD_ATTN_APPEND | (H.HERALD_ATTN_ADVANCE if advance else 0)
    return flags


class BlockPipeline:
    def __init__(self, dims: H.Dims, C: int, K: int, S: int, W: int, P: int, T: int,
                 den_stream=None, sel_stream=None, sel_sms=None, exact: bool = False,
                 blocks: int = 0, prefetch=False, budget=None):
        """blocks > 0: stage 1 selects C // blocks blocks of `blocks` keys
        over the cache's pooled block keys (herald_select_stage1_blocks),
        which the pipeline builds for each cache it meets and refreshes at
        the tail after every append.  prefetch: stage 1 is followed, on its
        stream, by the copy of the next block's candidate K rows into HBM
        (herald_stage_candidates), so that the next block's stage 2 reads
        them there (herald_select_stage2_staged) -- for a cache in host
        memory, whose link the denoising steps leave idle.  prefetch="kv":
        the candidates' V rows too, and the gather reads the top-K rows from
        HBM (herald_select_stage2_staged_gather; only the sink and local
        rows cross the link inside the step).  budget=(K_min, tau): each
        block's K per KV head from its first step's stage-2 mass
        (herald_select_stage2_adaptive, at most K; k_sel holds the last
        block's budgets), then the gather."""
        import torch
        self.torch = torch
        self.Bk = int(blocks)
        if self.Bk and C % self.Bk:
            raise ValueError(f"C={C} is not a multiple of the block size {self.Bk}")
        self._pooled = {}  # cache address -> fp32 block means (blocks > 0)
        if prefetch not in (False, True, "k", "kv"):
            raise ValueError(f"prefetch={prefetch!r}: False, True (= 'k') or 'kv'")
        self.prefetch = bool(prefetch)
        self.prefetch_v = prefetch == "kv"
        if budget is not None and (prefetch or exact):
            raise ValueError("the adaptive budget runs with the plain stage 2 only")
        self.budget = None if budget is None else (int(budget[0]), float(budget[1]))
        # SMs the overlapped stage-1 scan may occupy (0: all)
        # None: background_sms for the cache each block reads
        self.sel_sms = None if sel_sms is None else int(sel_sms)
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
        self.k_sel = torch.zeros(NG, dtype=torch.int32, device=dev)
        self.pool_k = [torch.zeros((*NG, P, dims.d), dtype=torch.int16, device=dev)
                       for _ in range(2)]
        self.pool_v = [torch.zeros_like(self.pool_k[0]) for _ in range(2)]
        # the candidates' K and V rows by slot, per candidate buffer (prefetch)
        self.staged = [torch.zeros((*NG, C, dims.d), dtype=torch.int16, device=dev)
                       for _ in range(2)] if prefetch else None
        self.staged_v = ([torch.zeros_like(t) for t in self.staged] if self.prefetch_v
                         else None)
        self.den = den_stream
        self.sel = sel_stream if sel_stream is not None else torch.cuda.Stream()
        self._graphs = {}  # captured blocks, by buffers and parity (block(graph=True))
        # addresses of the persistent buffers, resolved once: a block issues
        # ~T+5 library calls, and per-call marshalling would otherwise cost
        # more host time than the kernels take on the GPU
        P_ = H.ptr
        self._ws_den, self._ws_sel = P_(self.ws_den), P_(self.ws_sel)
        self._cand = [P_(t) for t in self.cand]
        self._n_cand = [P_(t) for t in self.n_cand]
        self._idx, self._n_sel = P_(self.idx), P_(self.n_sel)
        self._pool_k = [P_(t) for t in self.pool_k]
        self._pool_v = [P_(t) for t in self.pool_v]
        # herald_block's view of the same buffers: with the selection stream
        # and the fork/join events (overlap), and without (stage 1 on the
        # denoising stream); the events exist once recorded
        self._ev = [torch.cuda.Event() for _ in range(2)]
        for e in self._ev:
            e.record(torch.cuda.current_stream())

        def bufs(sel):
            b = H.BlockBufs()
            b.cand[0], b.cand[1] = self._cand
            b.n_cand[0], b.n_cand[1] = self._n_cand
            b.idx, b.n_sel = self._idx, self._n_sel
            b.pool_k[0], b.pool_k[1] = self._pool_k
            b.pool_v[0], b.pool_v[1] = self._pool_v
            b.ws_den, b.ws_sel, b.ws_bytes = self._ws_den, self._ws_sel, self.ws_bytes
            if sel is not None:
                b.sel_stream = H.stream_handle(sel) or None
                b.ev_fork, b.ev_join = (e.cuda_event for e in self._ev)
            return b
        self._bufs = {True: bufs(self.sel), False: bufs(None)}
        # the default selection (per-key stage 1, fixed K, stage 2 reading the
        # cache) issues each block as one herald_block call; False: the same
        # library calls one by one from here
        self.native = True
        # True while the last work issued on the streams was a herald_block
        # call: the next block's candidates come from its stage 1 (joined
        # before its last step) and may be read early (HERALD_BLOCK_CAND_SETTLED)
        self._cand_settled = False
        # the exact selection's own workspace (block_exact)
        self.ws_exact = None
        if exact:
            nb = H.herald_workspace_size_exact(dims, K, P)
            if nb == 0:
                raise ValueError("exact selection does not support these shapes")
            self.ws_exact = torch.zeros(nb, dtype=torch.uint8, device=dev)
            self._ws_exact, self._ws_exact_bytes = P_(self.ws_exact), nb

    def _den(self):
        return self.den if self.den is not None else self.torch.cuda.current_stream()

    def pooled(self, k_cache, ctx):
        """The block keys of `k_cache` (built on first use, on the current
        stream; refreshed by every block that appends to that cache)."""
        key = H.ptr(k_cache)
        t = self._pooled.get(key)
        if t is None:
            d = self.d
            nb = -(-d.L_max // self.Bk)
            t = self.torch.zeros((d.N, d.Hkv, nb, d.d), dtype=self.torch.float32, device="cuda")
            H.herald_pool_keys(d, k_cache, ctx, self.Bk, t, stream=self._den())
            self._pooled[key] = t
        return t

    def _stage1(self, q_merge, k_cache, ctx, slot, stream, sms=0, v_cache=None):
        """Stage 1 (per key, or over the pooled blocks) into cand[slot]; with
        prefetch, then the candidates' K (and V) rows into staged[slot]."""
        if self.Bk:
            H.check(H.lib().herald_select_stage1_blocks(
                self.d, H.ptr(q_merge), H.ptr(self.pooled(k_cache, ctx)), H.ptr(ctx), self.Bk,
                self.C // self.Bk, self._cand[slot], self._n_cand[slot], self._ws_sel,
                self.ws_bytes, H.stream_handle(stream)))
        else:
            H.check(H.lib().herald_select_stage1(
                self.d, H.ptr(q_merge), H.ptr(k_cache), H.ptr(ctx), self.C, self._cand[slot],
                self._n_cand[slot], self._ws_sel, self.ws_bytes, sms,
                H.stream_handle(stream)))
        if self.prefetch:
            if self.prefetch_v and v_cache is None:
                raise ValueError("prefetch='kv' stages the candidates' V rows: pass v_cache")
            H.check(H.lib().herald_stage_candidates(
                self.d, H.ptr(k_cache), H.ptr(v_cache) if self.prefetch_v else None,
                self._cand[slot], self._n_cand[slot], self.C, H.ptr(self.staged[slot]),
                H.ptr(self.staged_v[slot]) if self.prefetch_v else None,
                H.stream_handle(stream)))

    def prime(self, q_merge, k_cache, ctx, slot: int = 0, v_cache=None):
        """Stage 1 for the first block (no predecessor: its own queries);
        v_cache is needed with prefetch='kv'."""
        self._cand_settled = False  # its last kernel writes the candidates
        self._stage1(q_merge, k_cache, ctx, slot, self._den(), v_cache=v_cache)

    def block(self, i: int, q_steps, block_k, block_v, k_cache, v_cache, ctx, out,
              next_k_cache=None, advance: bool = True, overlap: bool = True,
              graph: bool = False, next_v_cache=None):
        """Runs block i: q_steps/block_k/block_v hold the T steps' inputs,
        out[t] receives step t's attention output.

        graph=True replays a CUDA graph of the block's library calls, captured
        the first time these buffers (and the block's parity) are seen; that
        first call runs the block directly.  The calls then cost one graph
        launch of host time instead of ~T+5 library calls."""
        if not graph:
            return self._block(i, q_steps, block_k, block_v, k_cache, v_cache, ctx, out,
                               next_k_cache, advance, overlap, next_v_cache)
        torch = self.torch
        P_ = H.ptr
        key = (i % 2, P_(q_steps), P_(block_k), P_(block_v), P_(k_cache), P_(v_cache), P_(ctx),
               P_(out), P_(k_cache if next_k_cache is None else next_k_cache),
               P_(v_cache if next_v_cache is None else next_v_cache), bool(advance),
               bool(overlap))
        g = self._graphs.get(key)
        if g is not None:
            g.replay()
            return
        self._block(i, q_steps, block_k, block_v, k_cache, v_cache, ctx, out, next_k_cache,
                    advance, overlap, next_v_cache)
        g = torch.cuda.CUDAGraph()
        den = torch.cuda.current_stream()
        cap = torch.cuda.Stream()
        cap.wait_stream(den)
        with torch.cuda.graph(g, stream=cap):
            self._block(i, q_steps, block_k, block_v, k_cache, v_cache, ctx, out, next_k_cache,
                        advance, overlap, next_v_cache)
        den.wait_stream(cap)
        self._graphs[key] = g

    def _scan_sms(self, k_cache) -> int:
        return scan_sms(self.d, k_cache, self.sel_sms)

    def _block(self, i, q_steps, block_k, block_v, k_cache, v_cache, ctx, out, next_k_cache,
               advance, overlap, next_v_cache=None):
        den, sel = self._den(), self.sel
        cur, nxt = i % 2, (i + 1) % 2
        nk = k_cache if next_k_cache is None else next_k_cache
        nv = v_cache if next_v_cache is None else next_v_cache
        d, P, L, chk = self.d, self.P, H.lib(), H.check
        hd = H.stream_handle(den)
        if self.native and not (self.Bk or self.prefetch or self.budget):
            H.step_bytes(q_steps), H.step_bytes(block_k), H.step_bytes(out)  # contiguous
            flags = ((H.HERALD_BLOCK_ADVANCE if advance else 0)
                     | (H.HERALD_BLOCK_CAND_SETTLED if self._cand_settled else 0))
            self._cand_settled = False
            chk(L.herald_block(d, self.C, self.K, self.S, self.W, P, self.T, i, H.ptr(q_steps),
                               H.ptr(block_k), H.ptr(block_v), H.ptr(k_cache), H.ptr(v_cache),
                               H.ptr(ctx), H.ptr(nk), H.ptr(out), flags,
                               self._scan_sms(nk) if overlap else 0, self._bufs[bool(overlap)],
                               hd))
            self._cand_settled = True
            return
        self._cand_settled = False
        q0, qstep = H.ptr(q_steps), H.step_bytes(q_steps)
        bk0, bv0, bstep = H.ptr(block_k), H.ptr(block_v), H.step_bytes(block_k)
        o0, ostep = H.ptr(out), H.step_bytes(out)
        kc, vc, cx = H.ptr(k_cache), H.ptr(v_cache), H.ptr(ctx)
        pk, pv = self._pool_k[cur], self._pool_v[cur]
        wd, wb = self._ws_den, self.ws_bytes
        # stage 1 for block i+1 can start now: block i's queries exist
        sel.wait_stream(den)
        if self.prefetch_v:  # stage 2 and the gather over the prefetched K and V rows
            chk(L.herald_select_stage2_staged_gather(
                d, q0, H.ptr(self.staged[cur]), H.ptr(self.staged_v[cur]), kc, vc, cx,
                self._cand[cur], self._n_cand[cur], self.C, self.K, self.S, self.W, P,
                self._idx, self._n_sel, pk, pv, wd, wb, hd))
        elif self.budget:  # stage 2 with each KV head's own budget, then the gather
            chk(L.herald_select_stage2_adaptive(
                d, q0, kc, cx, self._cand[cur], self._n_cand[cur], self.C, self.budget[0],
                self.K, self.budget[1], self.S, self.W, P, self._idx, self._n_sel,
                H.ptr(self.k_sel), wd, wb, hd))
            chk(L.herald_gather(d, self._idx, self._n_sel, P, kc, vc, pk, pv, hd))
        elif self.prefetch:  # stage 2 over the prefetched K rows, then the gather
            chk(L.herald_select_stage2_staged(d, q0, H.ptr(self.staged[cur]), cx,
                                              self._cand[cur], self._n_cand[cur], self.C,
                                              self.K, self.S, self.W, P, self._idx, self._n_sel,
                                              wd, wb, hd))
            chk(L.herald_gather(d, self._idx, self._n_sel, P, kc, vc, pk, pv, hd))
        else:  # stage 2 and the gather into pool[i%2] (one step for a device cache)
            chk(L.herald_select_stage2_gather(d, q0, kc, vc, cx, self._cand[cur],
                                              self._n_cand[cur], self.C, self.K, self.S, self.W,
                                              P, self._idx, self._n_sel, pk, pv, wd, wb, hd))
        self._stage1(q_steps, nk, ctx, nxt, sel if overlap else den,
                     self._scan_sms(nk) if overlap else 0, v_cache=nv)
        # the SMs the selection stream's work holds beside the steps: the
        # per-key scan's budget (0: every SM, no budget), then the candidate
        # copy's CTAs
        scan_bg = 0 if self.Bk else self._scan_sms(nk)
        bg = 0 if (not self.Bk and scan_bg == 0) else \
            max(scan_bg, STAGE_CTAS if self.prefetch else 0)
        sm_flags = attn_sm_flags(bg) if overlap else 0
        for t in range(self.T):
            if t == self.T - 1 and overlap:
                den.wait_stream(sel)  # stage 1 reads the cache the last step appends to
            chk(L.herald_denoise_attn_ex(d, q0 + t * qstep, pk, pv, self._n_sel, P,
                                         bk0 + t * bstep, bv0 + t * bstep, o0 + t * ostep, 0.0,
                                         step_flags(t, self.T, advance) | sm_flags, cx, kc, vc,
                                         wd, wb, hd))
        if self.Bk:  # the appended rows change the cache's last blocks
            chk(L.herald_pool_keys(d, kc, cx, self.Bk, -(-d.B // self.Bk) + 1,
                                   H.ptr(self.pooled(k_cache, ctx)), hd))


    def block_exact(self, i: int, q_steps, block_k, block_v, k_cache, v_cache, ctx, out,
                    advance: bool = True):
        """Block i with the exact selection (every cached position scored
        with the block's real queries) in place of the two stages: nothing
        of it can run ahead of the block, so the step is one stream."""
        self._cand_settled = False
        den = self._den()
        cur = i % 2
        d, P, L, chk = self.d, self.P, H.lib(), H.check
        hd = H.stream_handle(den)
        q0, qstep = H.ptr(q_steps), H.step_bytes(q_steps)
        bk0, bv0, bstep = H.ptr(block_k), H.ptr(block_v), H.step_bytes(block_k)
        o0, ostep = H.ptr(out), H.step_bytes(out)
        kc, vc, cx = H.ptr(k_cache), H.ptr(v_cache), H.ptr(ctx)
        pk, pv = self._pool_k[cur], self._pool_v[cur]
        wd, wb = self._ws_den, self.ws_bytes
        chk(L.herald_select_exact(d, q0, kc, cx, self.K, self.S, self.W, P, self._idx,
                                  self._n_sel, self._ws_exact, self._ws_exact_bytes, hd))
        chk(L.herald_gather(d, self._idx, self._n_sel, P, kc, vc, pk, pv, hd))
        for t in range(self.T):
            chk(L.herald_denoise_attn_ex(d, q0 + t * qstep, pk, pv, self._n_sel, P,
                                         bk0 + t * bstep, bv0 + t * bstep, o0 + t * ostep, 0.0,
                                         step_flags(t, self.T, advance), cx, kc, vc, wd, wb, hd))


class StackPipeline:
    """The same pipeline over a stack of layers sharing one context length.

    A denoising step is a forward pass over all layers, so per block:
    step 0 runs, layer by layer, stage 2 + gather + attention; right after a
    layer's step-0 work is issued, stage 1 of the next block for that layer
    starts on the selection stream (the layer's current queries exist from
    then on).  Steps 1..T-1 run attention over all layers; after the
    selection stream joins, every layer appends its block and the shared
    context length advances once.
    """

    def __init__(self, dims: H.Dims, n_layers: int, C: int, K: int, S: int, W: int, P: int,
                 T: int, sel_stream=None):
        import torch
        self.torch = torch
        self.d, self.nl = dims, n_layers
        self.C, self.K, self.S, self.W, self.P, self.T = C, K, S, W, P, T
        NG = (dims.N, dims.Hkv)
        dev = "cuda"
        self.ws_bytes = H.herald_workspace_size(dims, C, P)
        self.ws_den = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.ws_sel = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        mk = lambda shape, dt, fill=0: torch.full(shape, fill, dtype=dt, device=dev)
        self.cand = [[mk((*NG, C), torch.int32, -1) for _ in range(2)] for _ in range(n_layers)]
        self.n_cand = [[mk(NG, torch.int32) for _ in range(2)] for _ in range(n_layers)]
        # one tensor per output kind over all layers; every layer's slice
        # starts on a 16-byte boundary (the library's alignment rule)
        ng = dims.N * dims.Hkv
        rup = lambda x: (x + 3) // 4 * 4
        self.idx_all = mk((n_layers, rup(ng * P)), torch.int32, -1)
        self.n_sel_all = mk((n_layers, rup(ng)), torch.int32)
        self.idx = [self.idx_all[l, : ng * P].view(*NG, P) for l in range(n_layers)]
        self.n_sel = [self.n_sel_all[l, :ng].view(NG) for l in range(n_layers)]
        self.pool_k = [[mk((*NG, P, dims.d), torch.int16) for _ in range(2)]
                       for _ in range(n_layers)]
        self.pool_v = [[mk((*NG, P, dims.d), torch.int16) for _ in range(2)]
                       for _ in range(n_layers)]
        self.sel = sel_stream if sel_stream is not None else torch.cuda.Stream()
        self.sel_sms = None  # None: background_sms for the caches each block reads

    def _scan_sms(self, k_cache) -> int:
        return scan_sms(self.d, k_cache, self.sel_sms)

    def prime(self, q_merge, k_caches, ctx, slot: int = 0):
        st = self.torch.cuda.current_stream()
        for l in range(self.nl):
            H.herald_select_stage1(self.d, q_merge[l], k_caches[l], ctx, self.C,
                                   self.cand[l][slot], self.n_cand[l][slot], self.ws_sel,
                                   self.ws_bytes, st)

    def block(self, i: int, q_steps, block_k, block_v, k_caches, v_caches, ctx, out,
              advance: bool = True, overlap: bool = True):
        """q_steps[l], block_k[l], block_v[l]: layer l's [T, N, B, ...] inputs;
        out[l][t] receives layer l's step-t output."""
        torch = self.torch
        den, sel = torch.cuda.current_stream(), self.sel
        cur, nxt = i % 2, (i + 1) % 2
        d, P = self.d, self.P
        # the last step appends each layer's block (with T = 1 it would come
        # before that layer's stage 1, which must see the cache without it)
        fuse = self.T > 1
        for t in range(self.T):
            for l in range(self.nl):
                if t == 0:
                    H.herald_select_stage2_gather(d, q_steps[l][0], k_caches[l], v_caches[l],
                                                  ctx, self.cand[l][cur], self.n_cand[l][cur],
                                                  self.C, self.K, self.S, self.W, P,
                                                  self.idx[l], self.n_sel[l],
                                                  self.pool_k[l][cur], self.pool_v[l][cur],
                                                  self.ws_den, self.ws_bytes, den)
                if fuse and t == self.T - 1 and l == 0 and overlap:
                    den.wait_stream(sel)  # stage 1 reads the caches the last step appends to
                flags = step_flags(t, self.T, advance and l == self.nl - 1) if fuse else \
                    (H.HERALD_ATTN_SETTLED if t > 0 else 0)
                H.herald_denoise_attn_ex(d, q_steps[l][t], self.pool_k[l][cur],
                                         self.pool_v[l][cur], self.n_sel[l], P, block_k[l][t],
                                         block_v[l][t], out[l][t], 0.0, flags, ctx, k_caches[l],
                                         v_caches[l], self.ws_den, self.ws_bytes, den)
                if t == 0:
                    if overlap:
                        sel.wait_stream(den)
                        with torch.cuda.stream(sel):
                            H.herald_select_stage1(d, q_steps[l][0], k_caches[l], ctx, self.C,
                                                   self.cand[l][nxt], self.n_cand[l][nxt],
                                                   self.ws_sel, self.ws_bytes, sel,
                                                   sm_budget=self._scan_sms(k_caches[l]))
                    else:
                        H.herald_select_stage1(d, q_steps[l][0], k_caches[l], ctx, self.C,
                                               self.cand[l][nxt], self.n_cand[l][nxt],
                                               self.ws_sel, self.ws_bytes, den)
        if not fuse:  # one step per block: its stage 1 follows it, the appends come last
            if overlap:
                den.wait_stream(sel)
            for l in range(self.nl):
                H.herald_append_kv(d, block_k[l][self.T - 1], block_v[l][self.T - 1], ctx,
                                   k_caches[l], v_caches[l], advance and l == self.nl - 1, den)
