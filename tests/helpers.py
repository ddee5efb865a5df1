"""Shared test helpers: device upload of the synthetic bf16 inputs, the
tie-band comparisons of index sets, and stage-by-stage oracle checks of
(sequence, KV head) segments.  Holds none of the method's arithmetic: every
score comes from the oracle."""
from __future__ import annotations

import numpy as np

from block_diffusion_sparse_gb300 import synth

BAND = 1e-3          # |ln s - ln s_threshold| tie band for index parity
ATTN_ATOL = 2e-2     # max abs error of attention outputs


def dev(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def f64(a: np.ndarray) -> np.ndarray:
    return synth.bf16_to_f64(a)


def bf16_dev_to_f64(t) -> np.ndarray:
    return synth.bf16_to_f64(t.cpu().numpy().view(np.uint16))


def in_band(s: float, thr: float) -> bool:
    return s > 0 and thr > 0 and abs(np.log(s) - np.log(thr)) <= BAND


def assert_sets_within_band(gpu, ref, score, count, what=""):
    """gpu/ref: 1-D arrays of positions (ref = the oracle's top-`count` by
    `score`, fp64, indexed by position).  Passes if both hold `count`
    distinct positions and every position in their symmetric difference has
    a score within BAND (relative, in log space) of the oracle's threshold.
    Returns the number of band entries that differed."""
    gpu = [int(x) for x in gpu]
    ref = [int(x) for x in ref]
    assert len(gpu) == count == len(ref), f"{what}: sizes {len(gpu)} vs {len(ref)} vs {count}"
    assert len(set(gpu)) == len(gpu), f"{what}: duplicate positions"
    assert gpu == sorted(gpu), f"{what}: not ascending"
    diff = set(gpu) ^ set(ref)
    if not diff:
        return 0
    thr = min(score[j] for j in ref)
    bad = [j for j in diff if not in_band(score[j], thr)]
    assert not bad, f"{what}: {len(bad)} positions outside the tie band, e.g. {bad[:5]} " \
                    f"(threshold {thr}, scores {[score[j] for j in bad[:5]]})"
    return len(diff)


def sink_local(L: int, S: int, W: int) -> set:
    """Positions [0, S) and [L - W, L), clipped to [0, L)."""
    sink_end = min(S, L)
    return set(range(sink_end)) | set(range(max(L - W, sink_end), L))


def check_selection(idx, ns, idx_o, ns_o, cand, nc, s2, w, L, what):
    """One (n, g) row of the final selection against the oracle's, both made
    from the same candidates `cand[:nc]` with oracle scores `s2`: ascending,
    -1 padded, every sink and local position present, the same number of
    top-K positions outside the sink/local window, and every position in
    which the two differ a candidate whose score lies within the tie band of
    the oracle's K-th score.  (w gives K, S, W.)"""
    ns, ns_o, m = int(ns), int(ns_o), int(nc)
    got = [int(v) for v in idx[:ns]]
    assert got == sorted(set(got)), f"{what}: not ascending / duplicated"
    assert (np.asarray(idx[ns:]) == -1).all(), f"{what}: padding"
    sl = sink_local(L, w.S, w.W)
    assert sl <= set(got), f"{what}: sink/local positions missing"
    want = set(int(v) for v in idx_o[:ns_o])
    Ke = min(w.K, m)
    score = {int(cand[i]): float(s2[i]) for i in range(m)}
    if Ke == 0:
        assert set(got) == want, what
        return 0
    thr = sorted(s2[:m], reverse=True)[Ke - 1]
    band = lambda j: j in score and in_band(score[j], thr)
    diff = set(got) ^ want
    bad = [j for j in diff if not band(j)]
    assert not bad, f"{what}: {len(bad)} selected positions outside the tie band: {bad[:5]}"
    # the top-K count: outside the sink/local window both hold the same
    # number, except where a band position inside the window was swapped
    slack = sum(1 for j in sl if band(j))
    a, b = set(got) - sl, want - sl
    assert abs(len(a) - len(b)) <= slack, f"{what}: top-K counts {len(a)} vs {len(b)}"
    return len(diff)


def check_stage1_rows(cand, n_cand, s1, ctx, C, what=""):
    """Every (n, g) row of the device's stage-1 candidates against the
    oracle's top-C of its scores s1 [N, Hkv, L_max]: same count, -1 padding,
    differences only inside the tie band."""
    import oracle
    cand_o, nc_o = oracle.topc(s1, ctx, C)
    np.testing.assert_array_equal(np.asarray(n_cand), nc_o, err_msg=f"{what}: n_cand")
    diffs = 0
    N, Hkv = nc_o.shape
    for n in range(N):
        for g in range(Hkv):
            m = int(nc_o[n, g])
            diffs += assert_sets_within_band(cand[n, g, :m], cand_o[n, g, :m], s1[n, g], m,
                                             f"{what} stage 1 n={n} g={g}")
            assert (cand[n, g, m:] == -1).all(), f"{what} n={n} g={g}: padding"
    return diffs


def check_block_stage1_rows(cand, n_cand, ob, ctx, Bk, what=""):
    """Block stage 1: the device's candidate positions are exactly the
    positions below ctx of C_blocks whole blocks, and those blocks equal the
    oracle's (`ob` = oracle.stage1_blocks) up to its tie band."""
    N, Hkv = np.asarray(n_cand).shape
    for n in range(N):
        L = int(ctx[n])
        for g in range(Hkv):
            m = int(ob["n_cand_b"][n, g])
            row = cand[n, g, : n_cand[n, g]]
            blocks = sorted(set((row // Bk).tolist()))
            assert_sets_within_band(blocks, ob["cand_b"][n, g, :m], ob["s1b"][n, g], m,
                                    f"{what} blocks n={n} g={g}")
            want = [j for b in blocks for j in range(b * Bk, min((b + 1) * Bk, L))]
            assert row.tolist() == want, f"{what} n={n} g={g}: expansion"
            assert (cand[n, g, n_cand[n, g]:] == -1).all(), f"{what} n={n} g={g}: padding"


def segment(x: dict, w, n: int, g: int) -> dict:
    """Inputs restricted to one (sequence n, KV head g): N=1, Hkv=1, Hq=G."""
    G = w.G
    hs = slice(g * G, (g + 1) * G)
    return dict(
        q_merge=x["q_merge"][n:n + 1, :, hs],
        q_steps=x["q_steps"][:, n:n + 1, :, hs],
        k_cache=x["k_cache"][n:n + 1, g:g + 1],
        v_cache=x["v_cache"][n:n + 1, g:g + 1],
        block_k=x["block_k"][:, n:n + 1, :, g:g + 1],
        block_v=x["block_v"][:, n:n + 1, :, g:g + 1],
        ctx=x["ctx"][n:n + 1],
    )


def check_segments(x, w, pairs, cand, n_cand, idx, n_sel, out=None, step=0, what=""):
    """Stage by stage on (sequence, KV head) segments of a full-size run,
    each against the oracle on that segment alone:
      stage 1  the device's candidates vs the oracle's top-C of s1 (band);
      stage 2  the oracle's final selection made from the DEVICE's
               candidates vs the device's idx (band on s2);
      attn     (out given) step `step`'s output over the device's idx,
               max abs error <= ATTN_ATOL.
    cand/n_cand/idx/n_sel/out are host arrays of the whole batch."""
    import oracle
    band_diffs = 0
    for n, g in pairs:
        xs = segment(x, w, n, g)
        kf = f64(xs["k_cache"])
        qbar = oracle.merged_query(f64(xs["q_merge"]))
        _, _, s1 = oracle.stage1_scores(qbar, kf, xs["ctx"])
        gc, gnc = cand[n:n + 1, g:g + 1], n_cand[n:n + 1, g:g + 1]
        band_diffs += check_stage1_rows(gc, gnc, s1, xs["ctx"], w.C, f"{what} n={n} g={g}")
        s2 = oracle.stage2_scores(f64(xs["q_steps"][0]), kf, gc, gnc)
        idx_o, ns_o = oracle.select_final(xs["ctx"], w.L_max, gc, gnc, s2, w.K, w.S, w.W, w.P)
        band_diffs += check_selection(idx[n, g], n_sel[n, g], idx_o[0, 0], ns_o[0, 0], gc[0, 0],
                                      gnc[0, 0], s2[0, 0], w, int(xs["ctx"][0]),
                                      f"{what} stage 2 n={n} g={g}")
        if out is not None:
            ref = oracle.sparse_attn(f64(xs["q_steps"][step]), kf, f64(xs["v_cache"]),
                                     idx[n:n + 1, g:g + 1], n_sel[n:n + 1, g:g + 1],
                                     f64(xs["block_k"][step]), f64(xs["block_v"][step]))
            hs = slice(g * w.G, (g + 1) * w.G)
            err = np.abs(out[n:n + 1, :, hs] - ref).max()
            assert err <= ATTN_ATOL, f"{what} attention n={n} g={g}: max abs err {err}"
    return band_diffs
