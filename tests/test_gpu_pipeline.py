"""The dual-stream block pipeline over three consecutive blocks, with the
cache growing by one block each time, against the oracle replaying the same
schedule: stage 1 for block i+1 scans the cache before block i is appended,
using block i's first-step queries as the merged query; stage 2, the union
with sink/local and the attention use the cache after the append."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle
from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.pipeline import BlockPipeline
from block_diffusion_sparse_gb300.workloads import Workload
from helpers import ATTN_ATOL, bf16_dev_to_f64, dev, f64


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
        got.append((pipe.idx.cpu().numpy().copy(), pipe.n_sel.cpu().numpy().copy(),
                    bf16_dev_to_f64(out)))
    assert H.herald_workspace_error(pipe.ws_den) == 0
    assert H.herald_workspace_error(pipe.ws_sel) == 0
    assert ctx.cpu().numpy().tolist() == [w.L + nb * w.B] * w.N

    # oracle replay of the same schedule
    kc, vc = f64(x0["k_cache"]), f64(x0["v_cache"])
    cx = x0["ctx"].copy()
    def stage1(qbar, kc, cx):
        if Bk:
            r = oracle.stage1_blocks(qbar, kc, cx, Bk, w.C // Bk)
            return r["cand"], r["n_cand"]
        return oracle.topc(oracle.stage1_scores(qbar, kc, cx)[2], cx, w.C)

    qbar = oracle.merged_query(f64(x0["q_merge"]))
    cand, nc = stage1(qbar, kc, cx)
    for i, xb in enumerate(blocks):
        q0 = f64(xb["q_steps"][0])
        s2 = oracle.stage2_scores(q0, kc, cand, nc)
        idx_o, ns_o = oracle.select_final(cx, w.L_max, cand, nc, s2, w.K, w.S, w.W, w.P)
        gi, gn, gout = got[i]
        for n in range(w.N):
            for g in range(w.Hkv):
                a = set(gi[n, g, : gn[n, g]].tolist())
                b = set(idx_o[n, g, : ns_o[n, g]].tolist())
                assert len(a ^ b) <= 2, f"block {i} n={n} g={g}: {sorted(a ^ b)[:6]}"
        for t in range(w.T):
            ref = oracle.sparse_attn(f64(xb["q_steps"][t]), kc, vc, gi, gn,
                                     f64(xb["block_k"][t]), f64(xb["block_v"][t]))
            assert np.abs(gout[t] - ref).max() <= ATTN_ATOL
        # stage 1 for the next block: before this block is appended
        qbar = oracle.merged_query(q0)
        cand, nc = stage1(qbar, kc, cx)
        cx, kc, vc = oracle.append(cx, f64(xb["block_k"][w.T - 1]), f64(xb["block_v"][w.T - 1]),
                                   kc, vc)


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
        got.append([(pipe.idx[l].cpu().numpy().copy(), pipe.n_sel[l].cpu().numpy().copy(),
                     bf16_dev_to_f64(out[l])) for l in range(nl)])
    assert H.herald_workspace_error(pipe.ws_den) == 0
    assert H.herald_workspace_error(pipe.ws_sel) == 0
    assert ctx.cpu().numpy().tolist() == [w.L + nb * w.B] * w.N

    for l in range(nl):
        kc, vc = f64(x0[l]["k_cache"]), f64(x0[l]["v_cache"])
        cx = x0[l]["ctx"].copy()
        qbar = oracle.merged_query(f64(x0[l]["q_merge"]))
        cand, nc = oracle.topc(oracle.stage1_scores(qbar, kc, cx)[2], cx, w.C)
        for i in range(nb):
            xb = blocks[i][l]
            q0 = f64(xb["q_steps"][0])
            s2 = oracle.stage2_scores(q0, kc, cand, nc)
            idx_o, ns_o = oracle.select_final(cx, w.L_max, cand, nc, s2, w.K, w.S, w.W, w.P)
            gi, gn, gout = got[i][l]
            for n in range(w.N):
                for g in range(w.Hkv):
                    a = set(gi[n, g, : gn[n, g]].tolist())
                    b = set(idx_o[n, g, : ns_o[n, g]].tolist())
                    assert len(a ^ b) <= 2, f"layer {l} block {i} n={n} g={g}"
            for t in range(w.T):
                ref = oracle.sparse_attn(f64(xb["q_steps"][t]), kc, vc, gi, gn,
                                         f64(xb["block_k"][t]), f64(xb["block_v"][t]))
                assert np.abs(gout[t] - ref).max() <= ATTN_ATOL
            qbar = oracle.merged_query(q0)
            cand, nc = oracle.topc(oracle.stage1_scores(qbar, kc, cx)[2], cx, w.C)
            cx, kc, vc = oracle.append(cx, f64(xb["block_k"][w.T - 1]),
                                       f64(xb["block_v"][w.T - 1]), kc, vc)
