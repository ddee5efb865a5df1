"""Exact ties on the GPU: the lowest cache position wins every top-m.

Ties are planted, not hoped for: one heavy key row is copied to many cache
positions, so the copies' scores are equal bit for bit on both sides (the
same bf16 row gives the same products in the same order) and the copies
outnumber the places left at the threshold.  The selection rule of the
method (a canonical top-C / top-K, then the sink and local union; SparDA
summary, Method section, and the HERALD v3 abstract's two stages) then
leaves exactly one correct answer: the copies at the lowest positions.  No
tie band applies here -- the device must return the oracle's indices
exactly, stage by stage:

  stage 1      top-C of s1 with more copies than C
  stage 2      top-K of s2 with more copies than K (fused refine, and the
               two-pass refine with 16 scores per top-K thread), also through
               the stage-2 + gather call (many (sequence, KV head) pairs, and
               few with one and with two row tiles)
  exact        top-K of the exact score with more copies than K
  blocks       top-C_blocks over block means, with whole copied blocks
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle
from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.workloads import Workload
from helpers import dev, f64


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    H.lib()


def _w(name, **kw):
    base = dict(N=1, Hq=4, Hkv=1, d=128, L=3000, B=16, T=1, C=64, K=32, S=16, W=64,
                planted="points", n_planted=0, index=61, extra_rows=16)
    base.update(kw)
    return Workload(name, **base)


def _tied_layer(w, copies, seed, block=1):
    """Synthetic layer whose every (sequence, KV head) cache holds `copies`
    copies of one heavy key row (twice the mean of the group's queries,
    rounded to bf16) at seeded positions inside [S, L - W); block > 1 copies
    it over whole aligned blocks of that many rows instead.  Returns the
    inputs and the copies' positions per (n, g), ascending."""
    x = synth.make_layer(w)
    rng = np.random.Generator(np.random.PCG64(seed))
    G = w.G
    pos = {}
    for n in range(w.N):
        for g in range(w.Hkv):
            hs = slice(g * G, (g + 1) * G)
            qs = np.concatenate([f64(x["q_merge"][n, :, hs]), f64(x["q_steps"][0, n, :, hs])])
            heavy = synth.bf16_bits(2.0 * qs.reshape(-1, w.d).mean(axis=0))
            if block == 1:
                p = np.sort(rng.choice(np.arange(w.S, w.L - w.W), size=copies, replace=False))
            else:
                slots = np.arange(-(-w.S // block), (w.L - w.W) // block)
                b = np.sort(rng.choice(slots, size=copies, replace=False))
                p = (b[:, None] * block + np.arange(block)[None, :]).ravel()
            x["k_cache"][n, g, p] = heavy
            pos[(n, g)] = p
    return x, pos


def _bufs(w, C=None, P=None):
    C = w.C if C is None else C
    P = w.P if P is None else P
    NG = (w.N, w.Hkv)
    d = H.dims_of(w)
    ws = torch.zeros(H.herald_workspace_size(d, C, P), dtype=torch.uint8, device="cuda")
    return dict(d=d, ws=ws,
                cand=torch.full((*NG, C), -7, dtype=torch.int32, device="cuda"),
                n_cand=torch.zeros(NG, dtype=torch.int32, device="cuda"),
                idx=torch.full((*NG, P), -7, dtype=torch.int32, device="cuda"),
                n_sel=torch.zeros(NG, dtype=torch.int32, device="cuda"))


STAGE1 = [
    _w("s1-g4-d128", N=2, Hq=8, Hkv=2, C=64),
    _w("s1-g7-d64-ragged", Hq=14, Hkv=2, d=64, L=5001, B=32, C=200, K=64, index=62),
]


@pytest.mark.parametrize("w,copies", [(STAGE1[0], 100), (STAGE1[1], 300)],
                         ids=lambda v: getattr(v, "name", str(v)))
def test_stage1_ties_take_the_lowest_positions(w, copies):
    x, pos = _tied_layer(w, copies, seed=71)
    b = _bufs(w)
    H.herald_select_stage1(b["d"], dev(x["q_merge"]), dev(x["k_cache"]), dev(x["ctx"]), w.C,
                           b["cand"], b["n_cand"], b["ws"])
    torch.cuda.synchronize()
    assert H.herald_workspace_error(b["ws"]) == 0
    qbar = oracle.merged_query(f64(x["q_merge"]))
    s1 = oracle.stage1_scores(qbar, f64(x["k_cache"]), x["ctx"])[2]
    cand_o, nc_o = oracle.topc(s1, x["ctx"], w.C)
    for (n, g), p in pos.items():
        # the planted ties are the top scores and straddle the C-th place
        assert len(set(s1[n, g, p].tolist())) == 1 and s1[n, g, p[0]] == s1[n, g].max()
        np.testing.assert_array_equal(cand_o[n, g], p[: w.C])
    np.testing.assert_array_equal(b["n_cand"].cpu().numpy(), nc_o)
    np.testing.assert_array_equal(b["cand"].cpu().numpy(), cand_o)


STAGE2 = [
    # fused refine (C <= 4096), one row tile; G = 4
    (_w("s2-fused", N=2, Hq=8, Hkv=2, C=256, K=32), 100),
    # fused refine, G = 7 (two row tiles of whole tokens), ragged context
    (_w("s2-fused-g7", Hq=14, Hkv=2, L=4001, B=32, C=512, K=64, index=63), 150),
    # C > 4096: two-pass refine, 16 scores per top-K thread
    (_w("s2-two-pass", Hq=8, Hkv=2, L=9000, C=5000, K=256, index=64), 400),
]


@pytest.mark.parametrize("w,copies", STAGE2, ids=[c[0].name for c in STAGE2])
def test_stage2_ties_take_the_lowest_positions(w, copies):
    x, pos = _tied_layer(w, copies, seed=72)
    b = _bufs(w)
    kf = f64(x["k_cache"])
    qbar = oracle.merged_query(f64(x["q_merge"]))
    cand_o, nc_o = oracle.topc(oracle.stage1_scores(qbar, kf, x["ctx"])[2], x["ctx"], w.C)
    s2 = oracle.stage2_scores(f64(x["q_steps"][0]), kf, cand_o, nc_o)
    idx_o, ns_o = oracle.select_final(x["ctx"], w.L_max, cand_o, nc_o, s2, w.K, w.S, w.W, w.P)
    for (n, g), p in pos.items():
        in_cand = np.isin(cand_o[n, g, : nc_o[n, g]], p)
        assert in_cand.sum() == copies  # every copy is a candidate ...
        tied = s2[n, g, : nc_o[n, g]][in_cand]
        assert len(set(tied.tolist())) == 1 and tied[0] == s2[n, g].max()  # ... tied on top
        assert set(p[: w.K].tolist()) <= set(idx_o[n, g, : ns_o[n, g]].tolist())
        assert not set(p[w.K:].tolist()) & set(idx_o[n, g, : ns_o[n, g]].tolist()) - \
            set(range(w.S)) - set(range(w.L - w.W, w.L))
    H.herald_select_stage2(b["d"], dev(x["q_steps"][0]), dev(x["k_cache"]), dev(x["ctx"]),
                           dev(cand_o), dev(nc_o), w.C, w.K, w.S, w.W, w.P, b["idx"], b["n_sel"],
                           b["ws"])
    torch.cuda.synchronize()
    assert H.herald_workspace_error(b["ws"]) == 0
    np.testing.assert_array_equal(b["n_sel"].cpu().numpy(), ns_o)
    np.testing.assert_array_equal(b["idx"].cpu().numpy(), idx_o)


@pytest.mark.parametrize("w", [
    _w("s2-pairs16", N=4, Hq=16, Hkv=4, L=2000, C=256, K=40, index=65),
    _w("s2-few-pairs-one-tile", N=2, Hq=8, Hkv=2, L=2000, C=256, K=40, index=67),
    _w("s2-few-pairs-two-tiles", N=1, Hq=14, Hkv=2, B=32, L=2500, C=512, K=40, index=68),
], ids=lambda w: w.name)
def test_stage2_gather_ties(w):
    """The stage-2 + gather call.  With >= 16 (sequence, KV head) pairs the
    top-K runs as several copies per pair that each gather a slice of the
    pool: every copy must break the ties alike.  With few pairs the gather
    is a kernel of its own after the top-K (the group's query rows in one
    128-row tile, or in two, whose s2 partials the top-K adds).  The pool
    rows must be the lowest copies' rows."""
    x, pos = _tied_layer(w, 90, seed=73)
    b = _bufs(w)
    kf = f64(x["k_cache"])
    qbar = oracle.merged_query(f64(x["q_merge"]))
    cand_o, nc_o = oracle.topc(oracle.stage1_scores(qbar, kf, x["ctx"])[2], x["ctx"], w.C)
    s2 = oracle.stage2_scores(f64(x["q_steps"][0]), kf, cand_o, nc_o)
    idx_o, ns_o = oracle.select_final(x["ctx"], w.L_max, cand_o, nc_o, s2, w.K, w.S, w.W, w.P)
    NG = (w.N, w.Hkv)
    pk = torch.full((*NG, w.P, w.d), 9, dtype=torch.int16, device="cuda")
    pv = torch.full_like(pk, 9)
    k, v = dev(x["k_cache"]), dev(x["v_cache"])
    H.herald_select_stage2_gather(b["d"], dev(x["q_steps"][0]), k, v, dev(x["ctx"]), dev(cand_o),
                                  dev(nc_o), w.C, w.K, w.S, w.W, w.P, b["idx"], b["n_sel"], pk,
                                  pv, b["ws"])
    torch.cuda.synchronize()
    assert H.herald_workspace_error(b["ws"]) == 0
    np.testing.assert_array_equal(b["n_sel"].cpu().numpy(), ns_o)
    np.testing.assert_array_equal(b["idx"].cpu().numpy(), idx_o)
    pkh = pk.cpu().numpy().view(np.uint16)
    for n in range(w.N):
        for g in range(w.Hkv):
            m = int(ns_o[n, g])
            np.testing.assert_array_equal(pkh[n, g, :m], x["k_cache"][n, g, idx_o[n, g, :m]])


@pytest.mark.parametrize("w,copies", [
    (_w("exact-fused", N=2, Hq=8, Hkv=2, L=1500, K=32), 80),       # L_pad <= 4096
    (_w("exact-two-pass", Hq=8, Hkv=2, L=5000, K=48, index=66), 120),
], ids=lambda v: getattr(v, "name", str(v)))
def test_exact_selection_ties_take_the_lowest_positions(w, copies):
    x, pos = _tied_layer(w, copies, seed=74)
    d = H.dims_of(w)
    ws = torch.zeros(H.herald_workspace_size_exact(d, w.K, w.P), dtype=torch.uint8,
                     device="cuda")
    b = _bufs(w)
    H.herald_select_exact(d, dev(x["q_steps"][0]), dev(x["k_cache"]), dev(x["ctx"]), w.K, w.S,
                          w.W, w.P, b["idx"], b["n_sel"], ws)
    torch.cuda.synchronize()
    assert H.herald_workspace_error(ws) == 0
    o = oracle.select_exact(f64(x["q_steps"][0]), f64(x["k_cache"]), x["ctx"], w.K, w.S, w.W,
                            w.P)
    for (n, g), p in pos.items():
        s = o["s"][n, g, p]
        assert len(set(s.tolist())) == 1 and s[0] == o["s"][n, g].max()
    np.testing.assert_array_equal(b["n_sel"].cpu().numpy(), o["n_sel"])
    np.testing.assert_array_equal(b["idx"].cpu().numpy(), o["idx"])


@pytest.mark.parametrize("Bk", [16, 64])
def test_block_stage1_ties_take_the_lowest_blocks(Bk):
    w = _w("blocks", N=2, Hq=8, Hkv=2, L=4096, C=8 * Bk, index=67)
    x, pos = _tied_layer(w, 20, seed=75, block=Bk)
    b = _bufs(w)
    k, ctx = dev(x["k_cache"]), dev(x["ctx"])
    nb_max = -(-w.L_max // Bk)
    pooled = torch.zeros((w.N, w.Hkv, nb_max, w.d), dtype=torch.float32, device="cuda")
    H.herald_pool_keys(b["d"], k, ctx, Bk, pooled)
    H.herald_select_stage1_blocks(b["d"], dev(x["q_merge"]), pooled, ctx, Bk, w.C // Bk,
                                  b["cand"], b["n_cand"], b["ws"])
    torch.cuda.synchronize()
    assert H.herald_workspace_error(b["ws"]) == 0
    o = oracle.stage1_blocks(oracle.merged_query(f64(x["q_merge"])), f64(x["k_cache"]), x["ctx"],
                             Bk, w.C // Bk)
    for (n, g), p in pos.items():
        blocks = np.unique(p // Bk)
        s = o["s1b"][n, g, blocks]
        assert len(set(s.tolist())) == 1 and s[0] == o["s1b"][n, g].max()
        np.testing.assert_array_equal(o["cand_b"][n, g], blocks[: w.C // Bk])
    np.testing.assert_array_equal(b["n_cand"].cpu().numpy(), o["n_cand"])
    np.testing.assert_array_equal(b["cand"].cpu().numpy(), o["cand"])
