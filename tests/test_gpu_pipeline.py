"""The dual-stream block pipeline over three consecutive blocks, with the
cache growing by one block each time, against the oracle replaying the same
schedule: stage 1 for block i+1 scans the cache before block i is appended,
using block i's first-step queries as the merged query; stage 2, the union
with sink/local and the attention use the cache after the append.

Every block is checked stage by stage: the device's candidates against the
oracle's stage 1 (tie band), the device's selection against the oracle's
stage 2 made from the device's candidates (tie band), and every step's
attention output over the device's selection."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle
from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.pipeline import BlockPipeline
from block_diffusion_sparse_gb300.workloads import Workload
from helpers import (ATTN_ATOL, bf16_dev_to_f64, check_block_stage1_rows, check_selection,
                     check_stage1_rows, dev, f64)


@pytest.mark.parametrize("overlap,graph,T,Bk,host", [
    (True, False, 2, 0, False), (False, False, 2, 0, False), (True, True, 2, 0, False),
    (True, False, 1, 0, False), (True, False, 2, 16, False), (True, True, 2, 32, False),
    (True, False, 2, 16, "k"), (True, True, 2, 16, "kv")])
def test_three_blocks_match_oracle_schedule(overlap, graph, T, Bk, host):
    """graph=True: every block's inputs are copied into the same buffers, so
    block 2 replays the CUDA graph captured for block 0 (same parity).
    T=1: the only denoising step also appends the block.  Bk > 0: stage 1
    over the cache's pooled blocks of Bk keys, refreshed after each append.
    host: the cache in pinned host memory, the next block's candidate rows
    prefetched beside the denoising steps ("k": K rows for stage 2; "kv": K
    and V rows, the top-K pool rows gathered from them)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nb = 3
    w = Workload("pipe", N=2, Hq=8, Hkv=2, d=128, L=3000, B=16, T=T, C=256, K=128, S=16, W=64,
                 planted="points", n_planted=10, index=31, extra_rows=nb * 16)
    x0 = synth.make_layer(w)
    blocks = [synth.make_layer(w.scaled(L=64, extra_rows=0, n_planted=0), layer=i + 1)
              for i in range(nb)]
    d = H.dims_of(w)
    if host:
        k = torch.from_numpy(x0["k_cache"].view(np.int16).copy()).pin_memory()
        v = torch.from_numpy(x0["v_cache"].view(np.int16).copy()).pin_memory()
    else:
        k, v = dev(x0["k_cache"]), dev(x0["v_cache"])
    ctx = dev(x0["ctx"])
    pipe = BlockPipeline(d, w.C, w.K, w.S, w.W, w.P, w.T, blocks=Bk, prefetch=host or False)
    pipe.prime(dev(x0["q_merge"]), k, ctx, v_cache=v)
    got = []
    fixed = None
    for i, xb in enumerate(blocks):
        out = torch.zeros((w.T, w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
        qs, bk, bv = dev(xb["q_steps"]), dev(xb["block_k"]), dev(xb["block_v"])
        if graph:  # the same device buffers for every block
            if fixed is None:
                fixed = [torch.empty_like(t) for t in (qs, bk, bv, out)]
            for dst, src in zip(fixed, (qs, bk, bv, out)):
                dst.copy_(src)
            qs, bk, bv, out = fixed
        pipe.block(i, qs, bk, bv, k, v, ctx, out, advance=True, overlap=overlap, graph=graph)
        torch.cuda.synchronize()
        # block i's stage 2 read cand[i % 2]; stage 1 of block i+1 wrote the other
        got.append((pipe.cand[i % 2].cpu().numpy().copy(), pipe.n_cand[i % 2].cpu().numpy().copy(),
                    pipe.idx.cpu().numpy().copy(), pipe.n_sel.cpu().numpy().copy(),
                    bf16_dev_to_f64(out)))
    assert H.herald_workspace_error(pipe.ws_den) == 0
    assert H.herald_workspace_error(pipe.ws_sel) == 0
    assert ctx.cpu().numpy().tolist() == [w.L + nb * w.B] * w.N

    # oracle replay of the same schedule, fed the device's candidates
    kc, vc = f64(x0["k_cache"]), f64(x0["v_cache"])
    cx = x0["ctx"].copy()

    def stage1_check(qbar, kc, cx):
        """The check of a block's candidates against stage 1 on this cache
        state (taken now: the cache grows before the check runs)."""
        cx = cx.copy()
        if Bk:
            ob = oracle.stage1_blocks(qbar, kc, cx, Bk, w.C // Bk)
            return lambda gc, gnc, what: check_block_stage1_rows(gc, gnc, ob, cx, Bk, what)
        s1 = oracle.stage1_scores(qbar, kc, cx)[2]
        return lambda gc, gnc, what: check_stage1_rows(gc, gnc, s1, cx, w.C, what)

    check1 = stage1_check(oracle.merged_query(f64(x0["q_merge"])), kc, cx)
    for i, xb in enumerate(blocks):
        gc, gnc, gi, gn, gout = got[i]
        what = f"block {i}"
        check1(gc, gnc, what)
        # stage 2 from the device's candidates, on the cache after the appends
        q0 = f64(xb["q_steps"][0])
        s2 = oracle.stage2_scores(q0, kc, gc, gnc)
        idx_o, ns_o = oracle.select_final(cx, w.L_max, gc, gnc, s2, w.K, w.S, w.W, w.P)
        for n in range(w.N):
            for g in range(w.Hkv):
                check_selection(gi[n, g], gn[n, g], idx_o[n, g], ns_o[n, g], gc[n, g], gnc[n, g],
                                s2[n, g], w, int(cx[n]), f"{what} n={n} g={g}")
        for t in range(w.T):
            ref = oracle.sparse_attn(f64(xb["q_steps"][t]), kc, vc, gi, gn,
                                     f64(xb["block_k"][t]), f64(xb["block_v"][t]))
            assert np.abs(gout[t] - ref).max() <= ATTN_ATOL
        # stage 1 for the next block: block i's first-step queries, on the
        # cache before block i is appended
        check1 = stage1_check(oracle.merged_query(q0), kc, cx)
        cx, kc, vc = oracle.append(cx, f64(xb["block_k"][w.T - 1]), f64(xb["block_v"][w.T - 1]),
                                   kc, vc)


@pytest.mark.parametrize("overlap,graph,T,host", [
    (True, False, 2, False), (False, False, 2, False), (True, True, 2, False),
    (True, False, 1, False), (True, False, 2, True)])
def test_block_call_equals_the_calls_one_by_one(overlap, graph, T, host):
    """herald_block (one library call per block) against the same library
    calls issued one by one from Python: bit-identical candidates,
    selection, pools, outputs, caches and context lengths over three
    blocks (host: the cache in pinned host memory)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nb = 3
    w = Workload("pipe", N=2, Hq=8, Hkv=2, d=128, L=3000, B=16, T=T, C=256, K=128, S=16, W=64,
                 planted="points", n_planted=10, index=33, extra_rows=nb * 16)
    x0 = synth.make_layer(w)
    blocks = [synth.make_layer(w.scaled(L=64, extra_rows=0, n_planted=0), layer=i + 1)
              for i in range(nb)]
    d = H.dims_of(w)
    runs = []
    for native in (True, False):
        if host:
            k = torch.from_numpy(x0["k_cache"].view(np.int16).copy()).pin_memory()
            v = torch.from_numpy(x0["v_cache"].view(np.int16).copy()).pin_memory()
        else:
            k, v = dev(x0["k_cache"]), dev(x0["v_cache"])
        ctx = dev(x0["ctx"])
        pipe = BlockPipeline(d, w.C, w.K, w.S, w.W, w.P, w.T)
        pipe.native = native
        pipe.prime(dev(x0["q_merge"]), k, ctx)
        fixed = None
        got = []
        for i, xb in enumerate(blocks):
            out = torch.zeros((w.T, w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
            qs, bk, bv = dev(xb["q_steps"]), dev(xb["block_k"]), dev(xb["block_v"])
            if graph:
                if fixed is None:
                    fixed = [torch.empty_like(t) for t in (qs, bk, bv, out)]
                for dst, src in zip(fixed, (qs, bk, bv, out)):
                    dst.copy_(src)
                qs, bk, bv, out = fixed
            pipe.block(i, qs, bk, bv, k, v, ctx, out, advance=True, overlap=overlap, graph=graph)
            torch.cuda.synchronize()
            got.append([t.cpu().numpy().copy() for t in
                        (pipe.cand[(i + 1) % 2], pipe.n_cand[(i + 1) % 2], pipe.idx, pipe.n_sel,
                         pipe.pool_k[i % 2], pipe.pool_v[i % 2], out)])
        assert H.herald_workspace_error(pipe.ws_den) == 0
        assert H.herald_workspace_error(pipe.ws_sel) == 0
        runs.append((got, k.cpu().numpy(), v.cpu().numpy(), ctx.cpu().numpy()))
    (ga, ka, va, ca), (gb, kb, vb, cb) = runs
    for i in range(nb):
        for name, a, b in zip(("cand", "n_cand", "idx", "n_sel", "pool_k", "pool_v", "out"),
                              ga[i], gb[i]):
            assert np.array_equal(a, b), f"block {i}: {name}"
    assert np.array_equal(ka, kb) and np.array_equal(va, vb) and np.array_equal(ca, cb)
    assert ca.tolist() == [w.L + nb * w.B] * w.N


@pytest.mark.parametrize("T", [2, 1])
def test_two_layer_stack_matches_oracle_schedule(T):
    """The stack pipeline runs the per-layer schedule above on every layer,
    with one shared context length that advances once per block (T=1: the
    appends follow every layer's stage 1 instead of riding with the step)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_sparse_gb300.pipeline import StackPipeline
    nb, nl = 2, 2
    w = Workload("stack", N=2, Hq=8, Hkv=2, d=128, L=2500, B=16, T=T, C=256, K=96, S=16, W=48,
                 planted="points", n_planted=10, index=37, extra_rows=nb * 16, layers=nl)
    x0 = [synth.make_layer(w, layer=l) for l in range(nl)]
    blocks = [[synth.make_layer(w.scaled(L=64, extra_rows=0, n_planted=0), layer=10 + 2 * i + l)
               for l in range(nl)] for i in range(nb)]
    d = H.dims_of(w)
    k = [dev(x["k_cache"]) for x in x0]
    v = [dev(x["v_cache"]) for x in x0]
    ctx = dev(x0[0]["ctx"])
    pipe = StackPipeline(d, nl, w.C, w.K, w.S, w.W, w.P, w.T)
    pipe.prime([dev(x["q_merge"]) for x in x0], k, ctx)
    got = []
    for i in range(nb):
        out = [torch.zeros((w.T, w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
               for _ in range(nl)]
        pipe.block(i, [dev(b["q_steps"]) for b in blocks[i]],
                   [dev(b["block_k"]) for b in blocks[i]], [dev(b["block_v"]) for b in blocks[i]],
                   k, v, ctx, out, advance=True)
        torch.cuda.synchronize()
        got.append([(pipe.cand[l][i % 2].cpu().numpy().copy(),
                     pipe.n_cand[l][i % 2].cpu().numpy().copy(),
                     pipe.idx[l].cpu().numpy().copy(), pipe.n_sel[l].cpu().numpy().copy(),
                     bf16_dev_to_f64(out[l])) for l in range(nl)])
    assert H.herald_workspace_error(pipe.ws_den) == 0
    assert H.herald_workspace_error(pipe.ws_sel) == 0
    assert ctx.cpu().numpy().tolist() == [w.L + nb * w.B] * w.N

    for l in range(nl):
        kc, vc = f64(x0[l]["k_cache"]), f64(x0[l]["v_cache"])
        cx = x0[l]["ctx"].copy()
        s1 = oracle.stage1_scores(oracle.merged_query(f64(x0[l]["q_merge"])), kc, cx)[2]
        cx1 = cx.copy()
        for i in range(nb):
            xb = blocks[i][l]
            gc, gnc, gi, gn, gout = got[i][l]
            what = f"layer {l} block {i}"
            check_stage1_rows(gc, gnc, s1, cx1, w.C, what)
            q0 = f64(xb["q_steps"][0])
            s2 = oracle.stage2_scores(q0, kc, gc, gnc)
            idx_o, ns_o = oracle.select_final(cx, w.L_max, gc, gnc, s2, w.K, w.S, w.W, w.P)
            for n in range(w.N):
                for g in range(w.Hkv):
                    check_selection(gi[n, g], gn[n, g], idx_o[n, g], ns_o[n, g], gc[n, g],
                                    gnc[n, g], s2[n, g], w, int(cx[n]), f"{what} n={n} g={g}")
            for t in range(w.T):
                ref = oracle.sparse_attn(f64(xb["q_steps"][t]), kc, vc, gi, gn,
                                         f64(xb["block_k"][t]), f64(xb["block_v"][t]))
                assert np.abs(gout[t] - ref).max() <= ATTN_ATOL
            # the next block's stage 1: before this block is appended
            s1 = oracle.stage1_scores(oracle.merged_query(q0), kc, cx)[2]
            cx1 = cx.copy()
            cx, kc, vc = oracle.append(cx, f64(xb["block_k"][w.T - 1]),
                                       f64(xb["block_v"][w.T - 1]), kc, vc)
