"""Pins of the fp64 oracle against things other than itself: a hand-derived
worked example, closed forms, invariants, special cases that reduce to a
library routine (numpy / scipy / torch CPU), and brute force on tiny inputs.
Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, scale or index, a transposed operand, the wrong tie rule) fails
at least one of them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.workloads import TINY

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, shape):
    return rng.standard_normal(shape)


# --------------------------------------------------------------------------
# hand-derived worked example (tests/golden/hand_worked_g1.json)

def test_hand_worked_example_every_step():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_g1.json")))
    inp, exp = g["inputs"], g["expected"]
    q_merge = np.array(inp["q_merge"], float)
    a = np.array(inp["log_a"], float)
    k = np.zeros((1, 1, 4, 4)); k[0, 0, :, 0] = 2.0 * np.log(a)
    v = np.array(inp["v_cache"], float)
    q_block = np.array(inp["q_block"], float)
    bk, bv = np.array(inp["block_k"], float), np.array(inp["block_v"], float)
    ctx = np.array([4], np.int32)

    r = oracle.select(q_merge, q_block, k, ctx, inp["C"], inp["K"], inp["S"], inp["W"])
    np.testing.assert_allclose(r["qbar"][0, 0], exp["qbar"], atol=1e-15)
    np.testing.assert_allclose(np.exp(r["l1"][0, 0]), exp["l1_exp"], rtol=1e-13)
    np.testing.assert_allclose(r["s1"][0, 0], exp["s1"], rtol=1e-13)
    np.testing.assert_allclose(np.exp(r["lse1"][0, 0]), exp["lse1_exp"], rtol=1e-13)
    assert r["cand"][0, 0].tolist() == exp["cand"]
    want_s2 = [n / dd for n, dd in exp["s2_fraction"]]
    np.testing.assert_allclose(r["s2"][0, 0], want_s2, rtol=1e-13)
    assert r["idx"][0, 0, : exp["n_sel"]].tolist() == exp["idx"]
    assert int(r["n_sel"][0, 0]) == exp["n_sel"]
    assert (r["idx"][0, 0, exp["n_sel"]:] == -1).all()

    out, ws = oracle.sparse_attn(q_block, k, v, r["idx"], r["n_sel"], bk, bv, with_wsum=True)
    np.testing.assert_allclose(out[0, :, 0], exp["sparse_out"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(ws, 1.0, atol=1e-14)
    dense = oracle.dense_attn(q_block, k, v, ctx, bk, bv)
    np.testing.assert_allclose(dense[0, :, 0], exp["dense_out"], rtol=1e-13, atol=1e-14)


# --------------------------------------------------------------------------
# step 1 / step 2 against library routines and closed forms

def test_merged_query_is_numpy_mean():
    rng = np.random.default_rng(1)
    q = _rand(rng, (2, 5, 6, 8))
    np.testing.assert_allclose(oracle.merged_query(q), q.mean(axis=1), rtol=1e-14, atol=1e-15)


def _gqa_case(rng, N=2, Hq=6, Hkv=2, d=16, L_max=40, ctx=(40, 23)):
    qbar = _rand(rng, (N, Hq, d))
    k = _rand(rng, (N, Hkv, L_max, d))
    return qbar, k, np.array(ctx, np.int32)


def test_stage1_logits_match_numpy_einsum_with_gqa_mapping():
    rng = np.random.default_rng(2)
    qbar, k, ctx = _gqa_case(rng)
    l1, lse1, s1 = oracle.stage1_scores(qbar, k, ctx)
    G = qbar.shape[1] // k.shape[1]
    k_per_head = np.repeat(k, G, axis=1)           # head h reads KV head h // G
    ref = np.einsum("nhd,nhjd->nhj", qbar, k_per_head) / np.sqrt(qbar.shape[-1])
    for n, L in enumerate(ctx):
        np.testing.assert_allclose(l1[n, :, :L], ref[n, :, :L], rtol=1e-12, atol=1e-12)
        assert np.isneginf(l1[n, :, L:]).all()
        np.testing.assert_allclose(lse1[n], sps.logsumexp(ref[n, :, :L], axis=-1), rtol=1e-12)


def test_stage1_score_is_softmax_when_group_has_one_head():
    rng = np.random.default_rng(3)
    qbar, k, ctx = _gqa_case(rng, Hq=3, Hkv=3, ctx=(40, 17))
    l1, _, s1 = oracle.stage1_scores(qbar, k, ctx)
    for n, L in enumerate(ctx):
        np.testing.assert_allclose(s1[n, :, :L], sps.softmax(l1[n, :, :L], axis=-1), rtol=1e-12)
        assert (s1[n, :, L:] == 0).all()


def test_stage1_scores_sum_to_group_size():
    rng = np.random.default_rng(4)
    qbar, k, ctx = _gqa_case(rng, Hq=8, Hkv=2)
    _, _, s1 = oracle.stage1_scores(qbar, k, ctx)
    np.testing.assert_allclose(s1.sum(axis=-1), 4.0, rtol=1e-12)
    assert (s1 >= 0).all()


def test_stage1_group_score_is_sum_of_member_head_softmaxes():
    """Changing one head of group 0 must change s1 of group 0 only, by the
    difference of that head's softmax (scipy), never group 1."""
    rng = np.random.default_rng(5)
    qbar, k, ctx = _gqa_case(rng, N=1, Hq=4, Hkv=2, ctx=(40,))
    _, _, s_a = oracle.stage1_scores(qbar, k, ctx)
    qb2 = qbar.copy(); qb2[0, 1] = _rand(rng, qb2.shape[-1])
    l_b, _, s_b = oracle.stage1_scores(qb2, k, ctx)
    l_a, _, _ = oracle.stage1_scores(qbar, k, ctx)
    np.testing.assert_allclose(s_b[0, 1], s_a[0, 1], rtol=1e-14)
    delta = sps.softmax(l_b[0, 1]) - sps.softmax(l_a[0, 1])
    np.testing.assert_allclose(s_b[0, 0] - s_a[0, 0], delta, atol=1e-13)


# --------------------------------------------------------------------------
# top-m: tie rule and order, against Python's sort and brute force

@pytest.mark.parametrize("seed", range(6))
def test_top_m_matches_python_sort_with_ties(seed):
    rng = np.random.default_rng(10 + seed)
    n = int(rng.integers(1, 60))
    s = rng.integers(0, 6, n).astype(float)          # many exact ties
    for m in (0, 1, n // 2, n, n + 3):
        got = oracle.top_m(s, m)
        want = sorted(sorted(range(n), key=lambda j: (-s[j], j))[: min(m, n)])
        assert got.tolist() == want


def test_top_m_brute_force_max_sum_subset():
    rng = np.random.default_rng(20)
    for n in range(1, 11):
        s = rng.random(n)
        for m in range(0, min(n, 4) + 1):
            best = max(itertools.combinations(range(n), m), key=lambda c: sum(s[list(c)]))
            assert oracle.top_m(s, m).tolist() == list(best)


def test_topc_b1_g1_is_descending_argsort_of_dot_products():
    rng = np.random.default_rng(21)
    N, L, d, C_ = 1, 50, 8, 7
    q = _rand(rng, (N, 1, 1, d))
    k = _rand(rng, (N, 1, L, d))
    r = oracle.select(q, q, k, np.array([L], np.int32), C_, C_, 0, 0)
    dots = k[0, 0] @ q[0, 0, 0]
    want = np.sort(np.argsort(-dots, kind="stable")[:C_])
    assert r["cand"][0, 0].tolist() == want.tolist()


def test_topc_clamps_to_context_and_pads():
    rng = np.random.default_rng(22)
    qbar, k, ctx = _gqa_case(rng, N=2, Hq=2, Hkv=1, L_max=30, ctx=(5, 0))
    _, _, s1 = oracle.stage1_scores(qbar, k, ctx)
    cand, nc = oracle.topc(s1, ctx, 8)
    assert nc.tolist() == [[5], [0]]
    assert cand[0, 0].tolist() == [0, 1, 2, 3, 4, -1, -1, -1]
    assert (cand[1, 0] == -1).all()


# --------------------------------------------------------------------------
# stage 2

def test_stage2_scores_sum_to_rows_and_reduce_to_exact_softmax():
    rng = np.random.default_rng(30)
    N, B, Hq, Hkv, d, L = 1, 3, 4, 2, 16, 25
    q = _rand(rng, (N, B, Hq, d)); k = _rand(rng, (N, Hkv, L, d))
    ctx = np.array([L], np.int32)
    r = oracle.select(q, q, k, ctx, 9, 4, 0, 0)
    np.testing.assert_allclose(r["s2"][0].sum(axis=-1), B * Hq // Hkv, rtol=1e-12)
    # one row, every position a candidate: s2 is that row's exact softmax
    q1 = q[:, :1, :1]; k1 = k[:, :1]
    r1 = oracle.select(q1, q1, k1, ctx, L, 4, 0, 0)
    assert r1["cand"][0, 0].tolist() == list(range(L))
    logits = k1[0, 0] @ q1[0, 0, 0] / np.sqrt(d)
    np.testing.assert_allclose(r1["s2"][0, 0], sps.softmax(logits), rtol=1e-12)


def test_stage2_softmax_domain_is_the_candidates_only():
    """s2 over a candidate list must not depend on keys outside it."""
    rng = np.random.default_rng(31)
    N, B, Hq, Hkv, d, L = 1, 2, 2, 1, 8, 20
    q = _rand(rng, (N, B, Hq, d)); k = _rand(rng, (N, Hkv, L, d))
    cand = np.full((1, 1, 6), -1, np.int32); cand[0, 0, :4] = [1, 5, 9, 13]
    nc = np.array([[4]], np.int32)
    s_a = oracle.stage2_scores(q, k, cand, nc)
    k2 = k.copy(); k2[0, 0, [0, 2, 3, 19]] = 50.0 * _rand(rng, (4, d))
    s_b = oracle.stage2_scores(q, k2, cand, nc)
    np.testing.assert_allclose(s_a, s_b, rtol=1e-14)
    assert (s_a[0, 0, 4:] == 0).all()


# --------------------------------------------------------------------------
# step 5: union with sink and local, set arithmetic

@pytest.mark.parametrize("L,K,S,W", [(40, 5, 4, 6), (40, 0, 4, 6), (12, 5, 8, 8),
                                     (3, 5, 4, 6), (40, 5, 0, 0), (0, 5, 4, 6)])
def test_select_final_is_set_union(L, K, S, W):
    rng = np.random.default_rng(40 + L + K)
    N, B, Hq, Hkv, d, L_max, C_ = 1, 2, 2, 1, 8, 48, 16
    q = _rand(rng, (N, B, Hq, d)); k = _rand(rng, (N, Hkv, L_max, d))
    ctx = np.array([L], np.int32)
    r = oracle.select(q, q, k, ctx, C_, K, S, W)
    cand = r["cand"][0, 0][: r["n_cand"][0, 0]]
    s2 = r["s2"][0, 0][: len(cand)]
    top = {int(cand[i]) for i in sorted(range(len(cand)), key=lambda i: (-s2[i], i))[: K]}
    want = sorted(top | set(range(min(S, L))) | set(range(max(L - W, 0), L)))
    n = int(r["n_sel"][0, 0])
    assert r["idx"][0, 0, :n].tolist() == want
    assert n == len(top) + min(S, L) + min(W, L) - len(top & set(range(min(S, L)))) \
        - len(top & set(range(max(L - W, 0), L))) \
        - len(set(range(min(S, L))) & set(range(max(L - W, 0), L))) \
        + len(top & set(range(min(S, L))) & set(range(max(L - W, 0), L)))
    assert (r["idx"][0, 0, n:] == -1).all()


def test_planted_heavy_hitters_always_selected_tiny():
    w = TINY
    x = synth.make_layer(w, steps=1)
    f = synth.bf16_to_f64
    r = oracle.select(f(x["q_merge"]), f(x["q_steps"][0]), f(x["k_cache"]), x["ctx"],
                      w.C, w.K, w.S, w.W)
    pos = set(int(p) for p in x["planted"][0])
    assert len(pos) == w.n_planted
    assert pos <= set(r["cand"][0, 0].tolist())
    sel = set(r["idx"][0, 0, : r["n_sel"][0, 0]].tolist())
    assert pos <= sel
    assert set(range(w.S)) <= sel and set(range(w.L - w.W, w.L)) <= sel


def test_permutation_equivariance_without_sink_or_local():
    rng = np.random.default_rng(50)
    N, B, Hq, Hkv, d, L = 1, 2, 4, 2, 8, 30
    q = _rand(rng, (N, B, Hq, d)); k = _rand(rng, (N, Hkv, L, d))
    ctx = np.array([L], np.int32)
    perm = rng.permutation(L)
    r_a = oracle.select(q, q, k, ctx, 12, 5, 0, 0)
    r_b = oracle.select(q, q, k[:, :, perm], ctx, 12, 5, 0, 0)
    for g in range(Hkv):
        sel_a = set(r_a["idx"][0, g, : r_a["n_sel"][0, g]].tolist())
        sel_b = {int(perm[j]) for j in r_b["idx"][0, g, : r_b["n_sel"][0, g]]}
        assert sel_a == sel_b


# --------------------------------------------------------------------------
# step 6 / step 7: attention

def _attn_case(rng, N=2, B=3, Hq=4, Hkv=2, d=16, L_max=24, ctx=(24, 13)):
    q = _rand(rng, (N, B, Hq, d)); k = _rand(rng, (N, Hkv, L_max, d))
    v = _rand(rng, (N, Hkv, L_max, d))
    bk = _rand(rng, (N, B, Hkv, d)); bv = _rand(rng, (N, B, Hkv, d))
    return q, k, v, bk, bv, np.array(ctx, np.int32)


def test_attention_matches_torch_sdpa_fp64():
    rng = np.random.default_rng(60)
    q, k, v, bk, bv, ctx = _attn_case(rng)
    N, B, Hq, d = q.shape; Hkv = k.shape[1]; G = Hq // Hkv
    P = 9
    idx = np.full((N, Hkv, P), -1, np.int32); ns = np.zeros((N, Hkv), np.int32)
    for n in range(N):
        for g in range(Hkv):
            pick = np.sort(rng.choice(ctx[n], size=min(P - 2, ctx[n]), replace=False))
            idx[n, g, : len(pick)] = pick; ns[n, g] = len(pick)
    out = oracle.sparse_attn(q, k, v, idx, ns, bk, bv)
    for n in range(N):
        for h in range(Hq):
            g = h // G
            rows = idx[n, g, : ns[n, g]]
            kk = np.concatenate([k[n, g, rows], bk[n, :, g]])
            vv = np.concatenate([v[n, g, rows], bv[n, :, g]])
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[n, :, h])[None], torch.from_numpy(kk)[None],
                torch.from_numpy(vv)[None])[0].numpy()
            np.testing.assert_allclose(out[n, :, h], ref, rtol=1e-12, atol=1e-12)


def test_dense_attention_matches_torch_sdpa_with_mask():
    rng = np.random.default_rng(61)
    q, k, v, bk, bv, ctx = _attn_case(rng)
    out = oracle.dense_attn(q, k, v, ctx, bk, bv)
    N, B, Hq, d = q.shape; Hkv, L_max = k.shape[1], k.shape[2]; G = Hq // Hkv
    for n in range(N):
        kk = torch.from_numpy(np.concatenate([k[n], bk[n].transpose(1, 0, 2)], axis=1))
        vv = torch.from_numpy(np.concatenate([v[n], bv[n].transpose(1, 0, 2)], axis=1))
        kk = kk.repeat_interleave(G, dim=0); vv = vv.repeat_interleave(G, dim=0)
        mask = torch.ones(L_max + B, dtype=torch.bool)
        mask[ctx[n]:L_max] = False
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[n].transpose(1, 0, 2)), kk, vv, attn_mask=mask)
        np.testing.assert_allclose(out[n], ref.numpy().transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def test_attention_weights_sum_to_one_and_constant_values():
    rng = np.random.default_rng(62)
    q, k, v, bk, bv, ctx = _attn_case(rng)
    N, B, Hq, d = q.shape; Hkv = k.shape[1]
    idx = np.tile(np.arange(10, dtype=np.int32), (N, Hkv, 1)); ns = np.full((N, Hkv), 10, np.int32)
    c = rng.standard_normal(d)
    out, ws = oracle.sparse_attn(q, k, np.broadcast_to(c, v.shape), idx, ns, bk,
                                 np.broadcast_to(c, bv.shape), with_wsum=True)
    np.testing.assert_allclose(ws, 1.0, atol=1e-12)
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=1e-12, atol=1e-12)


def test_dense_equals_sparse_when_budget_covers_context():
    rng = np.random.default_rng(63)
    N, B, Hq, Hkv, d, L = 2, 3, 4, 2, 16, 20
    q = _rand(rng, (N, B, Hq, d)); k = _rand(rng, (N, Hkv, L, d)); v = _rand(rng, (N, Hkv, L, d))
    bk = _rand(rng, (N, B, Hkv, d)); bv = _rand(rng, (N, B, Hkv, d))
    ctx = np.array([L, 11], np.int32)
    r = oracle.select(q, q, k, ctx, L, L, 0, 0)
    assert r["n_sel"].tolist() == [[L, L], [11, 11]]
    np.testing.assert_allclose(oracle.sparse_attn(q, k, v, r["idx"], r["n_sel"], bk, bv),
                               oracle.dense_attn(q, k, v, ctx, bk, bv), rtol=1e-12, atol=1e-13)


def test_append_writes_rows_and_advances_context():
    rng = np.random.default_rng(70)
    N, B, Hkv, d, L_max = 2, 3, 2, 4, 10
    k = _rand(rng, (N, Hkv, L_max, d)); v = _rand(rng, (N, Hkv, L_max, d))
    bk = _rand(rng, (N, B, Hkv, d)); bv = _rand(rng, (N, B, Hkv, d))
    ctx = np.array([4, 7], np.int32)
    c2, k2, v2 = oracle.append(ctx, bk, bv, k, v)
    assert c2.tolist() == [7, 10]
    for n in range(N):
        np.testing.assert_array_equal(k2[n, :, ctx[n]: ctx[n] + B], bk[n].transpose(1, 0, 2))
        np.testing.assert_array_equal(v2[n, :, ctx[n]: ctx[n] + B], bv[n].transpose(1, 0, 2))
        np.testing.assert_array_equal(k2[n, :, : ctx[n]], k[n, :, : ctx[n]])
    # a block that overflows the cache: the rows that fit are written, the
    # rest skipped, and the context stops at the capacity L_max
    ctx = np.array([8, 10], np.int32)
    c3, k3, _ = oracle.append(ctx, bk, bv, k, v)
    assert c3.tolist() == [10, 10]
    np.testing.assert_array_equal(k3[0, :, 8:10], bk[0, :2].transpose(1, 0, 2))
    np.testing.assert_array_equal(k3[1], k[1])


def test_bf16_helpers_round_to_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3, 65504.0], np.float32)
    bits = synth.bf16_bits(x)
    back = synth.bf16_to_f64(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: the even one is 1+2^-6
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.015625
    assert back[3] == -2.5
    np.testing.assert_allclose(back[4], 3.0e-3, rtol=2 ** -8)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)


def test_exact_selection_with_one_row_is_the_top_k_of_dot_products():
    """B = G = 1: the exact score is the softmax of the single query's dot
    products over the whole context, so its top-K are the K largest dot
    products (numpy argsort), before the sink/local union."""
    rng = np.random.default_rng(5)
    N, Hkv, L, d, K = 1, 2, 300, 16, 20
    q = rng.standard_normal((N, 1, Hkv, d))
    k = rng.standard_normal((N, Hkv, L, d))
    ctx = np.array([L], np.int32)
    r = oracle.select_exact(q, k, ctx, K, 0, 0)
    for g in range(Hkv):
        dots = k[0, g] @ q[0, 0, g]
        want = np.sort(np.argsort(-dots, kind="stable")[:K])
        assert r["n_sel"][0, g] == K
        np.testing.assert_array_equal(r["idx"][0, g, :K], want)
        p = np.exp(dots / np.sqrt(d) - np.max(dots / np.sqrt(d)))
        np.testing.assert_allclose(r["s"][0, g, :L], p / p.sum(), rtol=1e-12)


def test_exact_scores_sum_to_rows_and_ignore_positions_past_the_context():
    rng = np.random.default_rng(6)
    N, B, Hq, Hkv, Lm, d = 2, 3, 4, 2, 50, 8
    q = rng.standard_normal((N, B, Hq, d))
    k = rng.standard_normal((N, Hkv, Lm, d))
    ctx = np.array([50, 31], np.int32)
    cand, nc, s = oracle.exact_scores(q, k, ctx)
    G = Hq // Hkv
    for n in range(N):
        for g in range(Hkv):
            L = ctx[n]
            assert nc[n, g] == L
            np.testing.assert_allclose(s[n, g, :L].sum(), B * G, rtol=1e-12)
    # changing a key past the context changes nothing
    k2 = k.copy()
    k2[1, :, 40:] += 5.0
    np.testing.assert_array_equal(oracle.exact_scores(q, k2, ctx)[2][1, :, :31], s[1, :, :31])


# --------------------------------------------------------------------------
# block-granular stage 1 (pooled block keys)

def test_block_stage1_with_one_key_per_block_is_stage1():
    """Bk = 1: every block is one key, so the block-granular stage 1 selects
    exactly what the (separately pinned) per-key stage 1 selects."""
    rng = np.random.default_rng(80)
    N, Hq, Hkv, d, L_max = 2, 6, 2, 16, 90
    qbar = _rand(rng, (N, Hq, d))
    k = _rand(rng, (N, Hkv, L_max, d))
    ctx = np.array([90, 57], np.int32)
    r = oracle.stage1_blocks(qbar, k, ctx, 1, 20)
    _, _, s1 = oracle.stage1_scores(qbar, k, ctx)
    cand, nc = oracle.topc(s1, ctx, 20)
    np.testing.assert_array_equal(r["cand"][..., :20], cand)
    np.testing.assert_array_equal(r["n_cand"], nc)


def test_block_logit_is_the_mean_of_its_keys_logits():
    """q . mean(k) = mean(q . k): a block's stage-1 logit is the mean of the
    per-key logits of its (valid) keys, the last block partial."""
    rng = np.random.default_rng(81)
    N, Hq, Hkv, d, L_max, Bk = 1, 4, 2, 8, 100, 16
    qbar = _rand(rng, (N, Hq, d))
    k = _rand(rng, (N, Hkv, L_max, d))
    ctx = np.array([75], np.int32)                    # 4 full blocks + 11 keys
    r = oracle.stage1_blocks(qbar, k, ctx, Bk, 3)
    l1, _, _ = oracle.stage1_scores(qbar, k, ctx)
    assert r["ctx_b"].tolist() == [5]
    for h in range(Hq):
        for b in range(5):
            want = l1[0, h, b * Bk: min((b + 1) * Bk, 75)].mean()
            assert abs(r["l1b"][0, h, b] - want) < 1e-12
    assert np.all(r["kp"][0, :, 5:] == 0)             # blocks past the context


def test_block_candidates_expand_whole_blocks_ascending():
    """The candidates are exactly the positions below ctx of the selected
    blocks, ascending; a block holding planted heavy keys is selected."""
    rng = np.random.default_rng(82)
    N, Hq, Hkv, d, L_max, Bk = 1, 4, 2, 32, 300, 32
    qbar = _rand(rng, (N, Hq, d))
    k = _rand(rng, (N, Hkv, L_max, d))
    ctx = np.array([270], np.int32)                   # blocks 0..8, the last with 14 keys
    for g in range(Hkv):                              # block 5 aligned with the group's queries
        q_g = qbar[0, g * 2:(g + 1) * 2].mean(axis=0)
        k[0, g, 5 * Bk:6 * Bk] = 3.0 * q_g + 0.1 * _rand(rng, (Bk, d))
    r = oracle.stage1_blocks(qbar, k, ctx, Bk, 3)
    for g in range(Hkv):
        blocks = r["cand_b"][0, g, : r["n_cand_b"][0, g]].tolist()
        assert 5 in blocks and blocks == sorted(blocks)
        want = [j for b in blocks for j in range(b * Bk, min((b + 1) * Bk, 270))]
        got = r["cand"][0, g, : r["n_cand"][0, g]].tolist()
        assert got == want and len(set(got)) == len(got)
        assert np.all(r["cand"][0, g, r["n_cand"][0, g]:] == -1)
    # every block selected when C_blocks covers the context
    r = oracle.stage1_blocks(qbar, k, ctx, Bk, 16)
    assert r["n_cand"].tolist() == [[270, 270]]
    assert (r["cand"][0, :, :270] == np.arange(270)).all()


# --------------------------------------------------------------------------
# adaptive budget (the first step's attention mass decides the block's K)

def test_adaptive_budget_is_the_smallest_subset_holding_the_mass():
    """Brute force over every subset of a few candidates: the budget is the
    size of the smallest subset whose scores reach tau of the total; zero
    scores, ragged n_cand and the clamps behave as stated."""
    rng = np.random.default_rng(91)
    N, Hkv, C = 2, 3, 7
    s2 = rng.random((N, Hkv, C)) ** 3
    s2[0, 1, 2] = s2[0, 1, 5] = 0.0                 # zero mass never helps
    nc = np.array([[7, 7, 4], [1, 6, 7]], np.int32)
    for tau in (0.3, 0.5, 0.8, 0.95, 1.0):
        kb = oracle.adaptive_budget(s2, nc, tau, 0, C)
        for n in range(N):
            for g in range(Hkv):
                m = int(nc[n, g])
                x = list(s2[n, g, :m])
                tot = sum(x)
                want = next(k for k in range(1, m + 1)
                            if any(sum(sub) >= tau * tot
                                   for sub in itertools.combinations(x, k)))
                assert kb[n, g] == want, (tau, n, g)
    # tau = 1: every non-zero score is needed, the zeros are not
    assert oracle.adaptive_budget(s2, nc, 1.0, 0, C)[0, 1] == 5
    # the clamps: never below K_min, never above K_max
    assert (oracle.adaptive_budget(s2, nc, 0.01, 3, C) == 3).all()
    assert (oracle.adaptive_budget(s2, nc, 1.0, 0, 2) <= 2).all()
    # no candidates: the budget is K_min
    assert oracle.adaptive_budget(s2, np.zeros((N, Hkv), np.int32), 0.5, 4, C).tolist() == \
        [[4] * Hkv] * N


def test_per_head_selection_with_one_budget_is_the_selection():
    """select_final_per_head with the same K everywhere is select_final."""
    rng = np.random.default_rng(92)
    N, Hkv, C, L_max = 2, 2, 40, 200
    cand = np.zeros((N, Hkv, C), np.int32)
    for n in range(N):
        for g in range(Hkv):
            cand[n, g] = np.sort(rng.choice(np.arange(8, 180), size=C, replace=False))
    nc = np.full((N, Hkv), C, np.int32); nc[1, 0] = 25
    s2 = rng.random((N, Hkv, C))
    ctx = np.array([200, 190], np.int32)
    a = oracle.select_final(ctx, L_max, cand, nc, s2, 12, 4, 16, 40)
    b = oracle.select_final_per_head(ctx, L_max, cand, nc, s2, np.full((N, Hkv), 12), 4, 16, 40)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # a smaller budget for one head changes only that head, and keeps its top scores
    kb = np.full((N, Hkv), 12); kb[0, 1] = 5
    c = oracle.select_final_per_head(ctx, L_max, cand, nc, s2, kb, 4, 16, 40)
    mid = lambda i, m, L: [p for p in i[:m] if 4 <= p < L - 16]
    assert len(mid(c[0][0, 1], c[1][0, 1], 200)) == 5
    top5 = set(cand[0, 1, np.argsort(-s2[0, 1], kind="stable")[:5]].tolist())
    assert set(mid(c[0][0, 1], c[1][0, 1], 200)) == top5
    for n, g in ((0, 0), (1, 0), (1, 1)):
        assert np.array_equal(c[0][n, g], a[0][n, g])
