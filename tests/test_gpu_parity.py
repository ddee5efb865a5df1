"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on
the same seeded inputs.  Each stage is checked in isolation (stage 2 gets
the oracle's candidates, attention gets the GPU's selected indices), so a
tie-band swap upstream cannot cascade.  Index outputs: set-equal except
entries within the tie band; gathers and appends: bit-exact; attention:
max abs error <= 2e-2."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle
from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.workloads import (LLAMA_64K, LONG_128K_HOST, QWEN_32K, QWEN_STACK,
                                                    TINY, Workload)
from helpers import (ATTN_ATOL, assert_sets_within_band, bf16_dev_to_f64, check_block_stage1_rows,
                     check_segments, check_selection, check_stage1_rows, dev, f64)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    H.lib()


def _case(name, **kw):
    base = dict(N=1, Hq=4, Hkv=1, d=64, L=2048, B=16, T=2, C=256, K=128, S=16, W=64,
                planted="points", n_planted=8, index=11, extra_rows=16)
    base.update(kw)
    return Workload(name, **base)


CASES = [
    TINY.scaled(T=2),
    _case("g7-d128-ragged", Hq=14, Hkv=2, d=128, L=5000, B=32, C=512, K=200, S=8, W=40,
          n_planted=20, index=12),
    _case("g4-d128-n2", N=2, Hq=8, Hkv=2, d=128, L=3001, B=32, C=300, K=100, S=4, W=33,
          n_planted=12, index=13),
    _case("g1-b1", Hq=2, Hkv=2, d=64, L=700, B=1, C=130, K=64, S=0, W=0, n_planted=4, index=14),
    _case("g8-b32-rows256", Hq=16, Hkv=2, d=128, L=1500, B=32, C=256, K=128, S=16, W=16,
          n_planted=6, index=15),
    _case("ctx-below-c", Hq=4, Hkv=1, d=128, L=100, B=8, C=256, K=64, S=16, W=16,
          n_planted=2, index=16),
    # C > 4096: the two-pass stage-2 refine
    _case("c-above-4096-two-pass", Hq=8, Hkv=2, d=128, L=9000, B=16, C=5000, K=256, S=16,
          W=64, n_planted=10, index=23),
    # a pool of more than 16 key tiles: the split-KV attention kernel + combine
    _case("large-pool-split", Hq=8, Hkv=2, d=128, L=6000, B=32, C=3000, K=2200, S=16, W=64,
          n_planted=30, index=22),
]


class Run:
    """Uploads a workload and runs the CUDA path step by step."""

    def __init__(self, w: Workload, x=None, ctx=None):
        self.w, self.x = w, (x if x is not None else synth.make_layer(w))
        if ctx is not None:
            self.x["ctx"] = np.asarray(ctx, np.int32)
        x = self.x
        self.d = H.dims_of(w)
        self.q_merge = dev(x["q_merge"])
        self.q_steps = dev(x["q_steps"])
        self.k = dev(x["k_cache"])
        self.v = dev(x["v_cache"])
        self.bk = dev(x["block_k"])
        self.bv = dev(x["block_v"])
        self.ctx = dev(x["ctx"])
        self.P = w.P
        self.ws_bytes = H.herald_workspace_size(self.d, w.C, self.P)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device="cuda")
        NG = (w.N, w.Hkv)
        self.cand = torch.full((*NG, w.C), -7, dtype=torch.int32, device="cuda")
        self.n_cand = torch.zeros(NG, dtype=torch.int32, device="cuda")
        self.idx = torch.full((*NG, self.P), -7, dtype=torch.int32, device="cuda")
        self.n_sel = torch.zeros(NG, dtype=torch.int32, device="cuda")
        self.pool_k = torch.full((*NG, self.P, w.d), 99, dtype=torch.int16, device="cuda")
        self.pool_v = torch.full((*NG, self.P, w.d), 99, dtype=torch.int16, device="cuda")
        self.out = torch.zeros((w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")

    def stage1(self, sm_budget=0):
        H.herald_select_stage1(self.d, self.q_merge, self.k, self.ctx, self.w.C, self.cand,
                               self.n_cand, self.ws, sm_budget=sm_budget)

    def stage2(self, cand=None, n_cand=None):
        c = self.cand if cand is None else dev(np.asarray(cand, np.int32))
        nc = self.n_cand if n_cand is None else dev(np.asarray(n_cand, np.int32))
        w = self.w
        H.herald_select_stage2(self.d, self.q_steps[0], self.k, self.ctx, c, nc, w.C, w.K, w.S,
                               w.W, self.P, self.idx, self.n_sel, self.ws)

    def select(self):
        w = self.w
        H.herald_select(self.d, self.q_merge, self.q_steps[0], self.k, self.ctx, w.C, w.K, w.S,
                        w.W, self.P, self.idx, self.n_sel, self.ws)

    def gather(self):
        H.herald_gather(self.d, self.idx, self.n_sel, self.P, self.k, self.v, self.pool_k,
                        self.pool_v)

    def attn(self, t, out=None, flags=0):
        H.herald_denoise_attn_ex(self.d, self.q_steps[t], self.pool_k, self.pool_v, self.n_sel,
                                 self.P, self.bk[t], self.bv[t], self.out if out is None else out,
                                 0.0, flags, self.ctx, self.k, self.v, self.ws)

    def error_word(self):
        return H.herald_workspace_error(self.ws)


def _oracle_stage1(x):
    qbar = oracle.merged_query(f64(x["q_merge"]))
    _, _, s1 = oracle.stage1_scores(qbar, f64(x["k_cache"]), x["ctx"])
    return s1


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_stage1_candidates(w):
    _check_stage1(w, 0)


@pytest.mark.parametrize("budget", [1, 7, 40])
def test_stage1_candidates_with_an_sm_budget(budget):
    """A scan confined to a few SMs (the background stage 1 of the
    pipeline) selects the same candidates, up to the tie band."""
    _check_stage1(CASES[1], budget)


def _check_stage1(w, sm_budget):
    r = Run(w)
    r.stage1(sm_budget)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    s1 = _oracle_stage1(r.x)
    check_stage1_rows(r.cand.cpu().numpy(), r.n_cand.cpu().numpy(), s1, r.x["ctx"], w.C, w.name)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_stage2_from_oracle_candidates(w):
    r = Run(w)
    x = r.x
    s1 = _oracle_stage1(x)
    cand_o, nc_o = oracle.topc(s1, x["ctx"], w.C)
    r.stage2(cand_o, nc_o)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    s2 = oracle.stage2_scores(f64(x["q_steps"][0]), f64(x["k_cache"]), cand_o, nc_o)
    idx_o, ns_o = oracle.select_final(x["ctx"], w.L_max, cand_o, nc_o, s2, w.K, w.S, w.W, w.P)
    idx, ns = r.idx.cpu().numpy(), r.n_sel.cpu().numpy()
    for n in range(w.N):
        for g in range(w.Hkv):
            check_selection(idx[n, g], int(ns[n, g]), idx_o[n, g], int(ns_o[n, g]),
                            cand_o[n, g], nc_o[n, g], s2[n, g], w, int(x["ctx"][n]),
                            f"{w.name} n={n} g={g}")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_gather_and_attention(w):
    r = Run(w)
    r.select()
    r.gather()
    torch.cuda.synchronize()
    idx, ns = r.idx.cpu().numpy(), r.n_sel.cpu().numpy()
    k, v = r.x["k_cache"], r.x["v_cache"]
    pk = r.pool_k.cpu().numpy().view(np.uint16)
    pv = r.pool_v.cpu().numpy().view(np.uint16)
    for n in range(w.N):
        for g in range(w.Hkv):
            m = int(ns[n, g])
            np.testing.assert_array_equal(pk[n, g, :m], k[n, g, idx[n, g, :m]])
            np.testing.assert_array_equal(pv[n, g, :m], v[n, g, idx[n, g, :m]])
            assert (pk[n, g, m:] == 0).all() and (pv[n, g, m:] == 0).all()
    # the T steps back to back, as a block runs them: steps after the first
    # load the (settled) pool before waiting for their predecessor
    outs = [torch.zeros_like(r.out) for _ in range(w.T)]
    for t in range(w.T):
        r.attn(t, outs[t], H.HERALD_ATTN_SETTLED if t > 0 else 0)
    torch.cuda.synchronize()
    for t in range(w.T):
        out = bf16_dev_to_f64(outs[t])
        ref = oracle.sparse_attn(f64(r.x["q_steps"][t]), f64(k), f64(v), idx, ns,
                                 f64(r.x["block_k"][t]), f64(r.x["block_v"][t]))
        err = np.abs(out - ref).max()
        assert err <= ATTN_ATOL, f"{w.name} step {t}: max abs err {err}"
    # the early loads change no result: the plain call gives the same bits
    r.attn(w.T - 1)
    torch.cuda.synchronize()
    assert torch.equal(r.out, outs[w.T - 1])
    assert r.error_word() == 0


MANY_PAIRS = [  # >= 16 (sequence, KV head) pairs: the gather rides with the top-K
    _case("pairs16-d128", N=4, Hq=16, Hkv=4, d=128, L=2000, B=16, C=256, K=64, S=8, W=32,
          n_planted=4, index=41),
    _case("pairs16-d64-ragged", N=8, Hq=6, Hkv=2, d=64, L=900, B=20, C=300, K=100, S=4, W=21,
          n_planted=4, index=42),
]


@pytest.mark.parametrize("w", CASES + MANY_PAIRS + [QWEN_32K], ids=lambda w: w.name)
def test_stage2_with_gather_equals_stage2_then_gather(w):
    """herald_select_stage2_gather writes the same idx, n_sel and pool bits
    as herald_select_stage2 followed by herald_gather: with many (sequence,
    KV head) pairs the gather runs inside the top-K, split over several CTAs
    per pair; with few, the two kernels run in turn."""
    r = Run(w)
    r.stage1()
    r.stage2()
    r.gather()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (r.idx, r.n_sel, r.pool_k, r.pool_v)]
    for t in (r.idx, r.n_sel, r.pool_k, r.pool_v):
        t.fill_(7)
    H.herald_select_stage2_gather(r.d, r.q_steps[0], r.k, r.v, r.ctx, r.cand, r.n_cand, w.C, w.K,
                                  w.S, w.W, r.P, r.idx, r.n_sel, r.pool_k, r.pool_v, r.ws)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    for got, want in zip((r.idx, r.n_sel, r.pool_k, r.pool_v), ref):
        assert torch.equal(got, want)


def test_dense_equals_sparse_when_budget_covers_context():
    w = _case("dense", Hq=8, Hkv=2, d=128, L=600, B=16, C=600, K=600, S=0, W=0,
              n_planted=3, index=17)
    r = Run(w)
    r.select()
    r.gather()
    r.attn(0)
    torch.cuda.synchronize()
    assert r.n_sel.cpu().numpy().tolist() == [[600, 600]]
    assert (r.idx.cpu().numpy()[:, :, :600] == np.arange(600)).all()
    x = r.x
    dense = oracle.dense_attn(f64(x["q_steps"][0]), f64(x["k_cache"]), f64(x["v_cache"]),
                              x["ctx"], f64(x["block_k"][0]), f64(x["block_v"][0]))
    assert np.abs(bf16_dev_to_f64(r.out) - dense).max() <= ATTN_ATOL


def test_empty_context_and_block_only_attention():
    w = _case("empty", Hq=4, Hkv=1, d=64, L=512, B=16, C=64, K=32, S=4, W=4, index=18)
    r = Run(w, ctx=[0])
    r.select()
    r.gather()
    r.attn(0)
    torch.cuda.synchronize()
    assert r.n_sel.cpu().numpy().tolist() == [[0]]
    assert (r.idx.cpu().numpy() == -1).all()
    x = r.x
    ref = oracle.dense_attn(f64(x["q_steps"][0]), f64(x["k_cache"]), f64(x["v_cache"]),
                            x["ctx"], f64(x["block_k"][0]), f64(x["block_v"][0]))
    assert np.abs(bf16_dev_to_f64(r.out) - ref).max() <= ATTN_ATOL


def test_per_sequence_context_lengths():
    """Ragged context lengths across the batch, stage by stage: stage 1
    against the oracle's s1, stage 2 from the device's candidates, and the
    combined call equal to the two stages bit for bit."""
    w = _case("mixed-ctx", N=3, Hq=8, Hkv=2, d=128, L=2000, B=16, C=200, K=64, S=8, W=16,
              n_planted=4, index=19)
    r = Run(w, ctx=[2000, 777, 65])
    r.stage1()
    r.stage2()
    torch.cuda.synchronize()
    assert r.error_word() == 0
    staged = (r.idx.clone(), r.n_sel.clone())
    x = r.x
    pairs = [(n, g) for n in range(w.N) for g in range(w.Hkv)]
    check_segments(x, w, pairs, r.cand.cpu().numpy(), r.n_cand.cpu().numpy(),
                   r.idx.cpu().numpy(), r.n_sel.cpu().numpy(), what="mixed-ctx")
    r.idx.fill_(7)
    r.select()
    torch.cuda.synchronize()
    assert torch.equal(r.idx, staged[0]) and torch.equal(r.n_sel, staged[1])


def test_planted_heavy_hitters_selected_and_deterministic():
    w = TINY
    r = Run(w)
    r.select()
    torch.cuda.synchronize()
    a = r.idx.clone()
    r.select()
    torch.cuda.synchronize()
    assert torch.equal(a, r.idx)
    sel = set(a.cpu().numpy()[0, 0, : int(r.n_sel[0, 0])].tolist())
    assert set(int(p) for p in r.x["planted"][0]) <= sel
    r.gather()
    r.attn(0)
    torch.cuda.synchronize()
    o1 = r.out.clone()
    r.attn(0)
    torch.cuda.synchronize()
    assert torch.equal(o1, r.out)


def test_append_matches_oracle_bit_exact():
    w = _case("append", N=2, Hq=8, Hkv=2, d=128, L=300, B=16, C=64, K=32, S=4, W=4,
              extra_rows=40, index=20)
    r = Run(w, ctx=[300, 330])
    H.herald_append_kv(r.d, r.bk[0], r.bv[0], r.ctx, r.k, r.v, advance=True)
    torch.cuda.synchronize()
    c2, k2, v2 = oracle.append(r.x["ctx"], f64(r.x["block_k"][0]), f64(r.x["block_v"][0]),
                               f64(r.x["k_cache"]), f64(r.x["v_cache"]))
    # the second sequence overflows L_max = 340: rows past it are skipped and
    # the context is capped
    assert r.ctx.cpu().numpy().tolist() == [316, 340]
    kk = synth.bf16_to_f64(r.k.cpu().numpy().view(np.uint16))
    vv = synth.bf16_to_f64(r.v.cpu().numpy().view(np.uint16))
    np.testing.assert_array_equal(kk, k2)
    np.testing.assert_array_equal(vv, v2)


def test_append_with_the_split_attention():
    """A pool too large for the pool kernel (the cluster/split attention
    kernels) appends through the append kernel after the step: the same
    cache rows, lengths and attention output."""
    w = _case("append-split", N=2, Hq=8, Hkv=2, d=128, L=3000, B=16, C=2600, K=2300, S=16,
              W=64, extra_rows=40, index=43)
    r = Run(w, ctx=[3000, 3030])
    r.select()
    r.gather()
    t = w.T - 1
    r.attn(t)
    torch.cuda.synchronize()
    out_plain = r.out.clone()
    r.out.zero_()
    r.attn(t, flags=H.HERALD_ATTN_SETTLED | H.HERALD_ATTN_APPEND | H.HERALD_ATTN_ADVANCE)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert torch.equal(r.out, out_plain)
    _, k2, v2 = oracle.append(r.x["ctx"], f64(r.x["block_k"][t]), f64(r.x["block_v"][t]),
                              f64(r.x["k_cache"]), f64(r.x["v_cache"]))
    assert r.ctx.cpu().numpy().tolist() == [3016, 3040]  # L_max = 3040 caps the second
    np.testing.assert_array_equal(synth.bf16_to_f64(r.k.cpu().numpy().view(np.uint16)), k2)
    np.testing.assert_array_equal(synth.bf16_to_f64(r.v.cpu().numpy().view(np.uint16)), v2)


@pytest.mark.parametrize("advance", [True, False])
@pytest.mark.parametrize("placement", ["device", "host"])
def test_last_step_appends_like_append_kv(placement, advance):
    """A denoising step with HERALD_ATTN_APPEND writes the cache rows and the
    context lengths bit-exactly as herald_append_kv does (fused into the
    attention kernel for a device cache, the append kernel after it for a
    host-resident one), and its attention output is the plain step's."""
    w = _case("append-step", N=2, Hq=8, Hkv=2, d=128, L=300, B=16, C=64, K=32, S=4, W=4,
              extra_rows=40, index=20)
    r = Run(w, ctx=[300, 330])
    r.select()
    r.gather()
    t = w.T - 1
    r.attn(t)
    torch.cuda.synchronize()
    out_plain = r.out.clone()
    r.out.zero_()
    if placement == "host":
        r.k = torch.from_numpy(r.x["k_cache"].view(np.int16).copy()).pin_memory()
        r.v = torch.from_numpy(r.x["v_cache"].view(np.int16).copy()).pin_memory()
    flags = H.HERALD_ATTN_SETTLED | H.HERALD_ATTN_APPEND
    if advance:
        flags |= H.HERALD_ATTN_ADVANCE
    r.attn(t, flags=flags)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert torch.equal(r.out, out_plain)
    _, k2, v2 = oracle.append(r.x["ctx"], f64(r.x["block_k"][t]), f64(r.x["block_v"][t]),
                              f64(r.x["k_cache"]), f64(r.x["v_cache"]))
    # the second sequence overflows L_max = 340: its rows past it are
    # skipped and its length is capped at the cache's capacity
    assert r.ctx.cpu().numpy().tolist() == ([316, 340] if advance else [300, 330])
    kk = synth.bf16_to_f64(r.k.cpu().numpy().view(np.uint16))
    vv = synth.bf16_to_f64(r.v.cpu().numpy().view(np.uint16))
    np.testing.assert_array_equal(kk, k2)
    np.testing.assert_array_equal(vv, v2)


@pytest.mark.parametrize("w", [
    _case("host-kv", Hq=8, Hkv=2, d=128, L=4096, B=32, C=512, K=128, S=16, W=64,
          n_planted=10, index=21),
    # C > 4096: staged candidate rows feed the two-pass refine
    _case("host-kv-two-pass", Hq=8, Hkv=2, d=128, L=6000, B=16, C=4600, K=256, S=16, W=64,
          n_planted=10, index=24),
], ids=lambda w: w.name)
def test_host_resident_cache_matches_device_cache(w):
    """A cache in pinned host memory (scanned over the host link, candidate
    rows staged into the workspace for stage 2) selects and gathers exactly
    what the same cache in device memory does."""
    r = Run(w)
    r.select()
    r.gather()
    torch.cuda.synchronize()
    idx_dev, ns_dev = r.idx.clone(), r.n_sel.clone()
    pk_dev, pv_dev = r.pool_k.clone(), r.pool_v.clone()
    kh = torch.from_numpy(r.x["k_cache"].view(np.int16)).pin_memory()
    vh = torch.from_numpy(r.x["v_cache"].view(np.int16)).pin_memory()
    w_ = r.w
    H.herald_select(r.d, r.q_merge, r.q_steps[0], kh, r.ctx, w_.C, w_.K, w_.S, w_.W, r.P, r.idx,
                    r.n_sel, r.ws)
    H.herald_gather(r.d, r.idx, r.n_sel, r.P, kh, vh, r.pool_k, r.pool_v)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert torch.equal(idx_dev, r.idx) and torch.equal(ns_dev, r.n_sel)
    assert torch.equal(pk_dev, r.pool_k)
    # stage 2 over candidate rows staged beforehand (the prefetch of a
    # host-resident cache): the same selection, bit for bit
    staged = torch.full((w_.N, w_.Hkv, w_.C, w_.d), 99, dtype=torch.int16, device="cuda")
    H.herald_select_stage1(r.d, r.q_merge, kh, r.ctx, w_.C, r.cand, r.n_cand, r.ws)
    H.herald_stage_candidates(r.d, kh, r.cand, r.n_cand, w_.C, staged)
    r.idx.fill_(7)
    H.herald_select_stage2_staged(r.d, r.q_steps[0], staged, r.ctx, r.cand, r.n_cand, w_.C, w_.K,
                                  w_.S, w_.W, r.P, r.idx, r.n_sel, r.ws)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert torch.equal(idx_dev, r.idx) and torch.equal(ns_dev, r.n_sel)
    # the combined stage 2 + gather on the host-resident cache (two kernels
    # there) from the same stage-1 candidates
    H.herald_select_stage1(r.d, r.q_merge, kh, r.ctx, w_.C, r.cand, r.n_cand, r.ws)
    r.pool_k.fill_(7)
    H.herald_select_stage2_gather(r.d, r.q_steps[0], kh, vh, r.ctx, r.cand, r.n_cand, w_.C, w_.K,
                                  w_.S, w_.W, r.P, r.idx, r.n_sel, r.pool_k, r.pool_v, r.ws)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert torch.equal(idx_dev, r.idx) and torch.equal(ns_dev, r.n_sel)
    assert torch.equal(pk_dev, r.pool_k)
    # the candidates' K and V rows staged beforehand, then stage 2 and the
    # gather over them: the same selection and pool, bit for bit
    staged_v = torch.full_like(staged, 99)
    H.herald_stage_candidates(r.d, kh, r.cand, r.n_cand, w_.C, staged, v_cache=vh,
                              staged_v=staged_v)
    torch.cuda.synchronize()
    cand, nc = r.cand.cpu().numpy(), r.n_cand.cpu().numpy()
    vx = r.x["v_cache"].view(np.int16)
    sv = staged_v.cpu().numpy()
    for n in range(w_.N):
        for g in range(w_.Hkv):
            c = int(nc[n, g])
            np.testing.assert_array_equal(sv[n, g, :c], vx[n, g, cand[n, g, :c]])
            assert (sv[n, g, c:] == 0).all()
    r.pool_k.fill_(7)
    r.pool_v.fill_(7)
    H.herald_select_stage2_staged_gather(r.d, r.q_steps[0], staged, staged_v, kh, vh, r.ctx,
                                         r.cand, r.n_cand, w_.C, w_.K, w_.S, w_.W, r.P, r.idx,
                                         r.n_sel, r.pool_k, r.pool_v, r.ws)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert torch.equal(idx_dev, r.idx) and torch.equal(ns_dev, r.n_sel)
    assert torch.equal(pk_dev, r.pool_k) and torch.equal(pv_dev, r.pool_v)
    # the top-K rows come from the staged rows, the sink and local rows from
    # the cache: with the staged values overwritten, exactly the rows at
    # positions in [S, L - W) carry the new value
    staged_v.fill_(5)
    r.pool_v.fill_(7)
    H.herald_select_stage2_staged_gather(r.d, r.q_steps[0], staged, staged_v, kh, vh, r.ctx,
                                         r.cand, r.n_cand, w_.C, w_.K, w_.S, w_.W, r.P, r.idx,
                                         r.n_sel, r.pool_k, r.pool_v, r.ws)
    torch.cuda.synchronize()
    idx, ns, pv = r.idx.cpu().numpy(), r.n_sel.cpu().numpy(), r.pool_v.cpu().numpy()
    for n in range(w_.N):
        L = int(r.x["ctx"][n])
        for g in range(w_.Hkv):
            m = int(ns[n, g])
            pos = idx[n, g, :m]
            mid = (pos >= w_.S) & (pos < L - w_.W)
            assert mid.any() and (~mid).any()
            assert (pv[n, g, :m][mid] == 5).all()
            np.testing.assert_array_equal(pv[n, g, :m][~mid], vx[n, g, pos[~mid]])
            assert (pv[n, g, m:] == 0).all()


@pytest.mark.parametrize("w", [QWEN_32K], ids=lambda w: w.name)
def test_full_size_qwen_layer(w):
    """The benchmarked workload at full size: every stage against the oracle."""
    r = Run(w.scaled(T=2))
    x = r.x
    r.stage1()
    torch.cuda.synchronize()
    s1 = _oracle_stage1(x)
    cand_o, nc_o = oracle.topc(s1, x["ctx"], w.C)
    cand = r.cand.cpu().numpy()
    for g in range(w.Hkv):
        assert_sets_within_band(cand[0, g], cand_o[0, g], s1[0, g], w.C, f"stage1 g={g}")
    planted = set(int(p) for p in x["planted"][0])
    for g in range(w.Hkv):
        assert planted <= set(cand[0, g].tolist())
    r.stage2(cand_o, nc_o)
    r.gather()
    r.attn(1)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    idx, ns = r.idx.cpu().numpy(), r.n_sel.cpu().numpy()
    s2 = oracle.stage2_scores(f64(x["q_steps"][0]), f64(x["k_cache"]), cand_o, nc_o)
    idx_o, ns_o = oracle.select_final(x["ctx"], w.L_max, cand_o, nc_o, s2, w.K, w.S, w.W, w.P)
    for g in range(w.Hkv):
        check_selection(idx[0, g], int(ns[0, g]), idx_o[0, g], int(ns_o[0, g]), cand_o[0, g],
                        nc_o[0, g], s2[0, g], w, w.L, f"qwen g={g}")
        assert planted <= set(idx[0, g, : ns[0, g]].tolist())
    out = bf16_dev_to_f64(r.out)
    ref = oracle.sparse_attn(f64(x["q_steps"][1]), f64(x["k_cache"]), f64(x["v_cache"]), idx, ns,
                             f64(x["block_k"][1]), f64(x["block_v"][1]))
    assert np.abs(out - ref).max() <= ATTN_ATOL
    # stage 2 from the device's own candidates, as the pipeline runs it
    r.stage2()
    torch.cuda.synchronize()
    assert r.error_word() == 0
    check_segments(x, w, [(0, g) for g in range(w.Hkv)], cand, r.n_cand.cpu().numpy(),
                   r.idx.cpu().numpy(), r.n_sel.cpu().numpy(), what="qwen")


def _full_size_stages(w, host=False):
    """A full-size layer run as the pipeline runs it -- stage 1, stage 2 from
    the device's candidates, the gather, one denoising step -- then checked
    stage by stage on EVERY (sequence, KV head) segment against the oracle on
    that segment (check_segments), the planted heavy hitters kept where they
    fit the budget, and the combined call equal to the two stages."""
    r = Run(w)
    if host:
        r.k = torch.from_numpy(r.x["k_cache"].view(np.int16)).pin_memory()
        r.v = torch.from_numpy(r.x["v_cache"].view(np.int16)).pin_memory()
    r.stage1()
    r.stage2()
    r.gather()
    r.attn(0)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    idx, ns = r.idx.cpu().numpy(), r.n_sel.cpu().numpy()
    pairs = [(n, g) for n in range(w.N) for g in range(w.Hkv)]
    check_segments(r.x, w, pairs, r.cand.cpu().numpy(), r.n_cand.cpu().numpy(), idx, ns,
                   out=bf16_dev_to_f64(r.out), what=w.name)
    for n, g in pairs:
        planted = set(int(p) for p in r.x["planted"][n])
        if len(planted) <= w.K:  # (the 128K workload plants more keys than K keeps)
            assert planted <= set(idx[n, g, : ns[n, g]].tolist()), (n, g)
    # the combined call (both stages, candidates kept in the workspace)
    r.idx.fill_(7)
    r.select()
    torch.cuda.synchronize()
    assert r.error_word() == 0
    assert np.array_equal(r.idx.cpu().numpy(), idx) and np.array_equal(r.n_sel.cpu().numpy(), ns)


def test_full_size_llama_layer_all_segments():
    """4 x 64K context, 8 KV heads, C = 4096: the fused refine with whole
    row tiles of 128 query rows, 32 segments (the top-K carries the gather
    when called through herald_select_stage2_gather)."""
    _full_size_stages(LLAMA_64K.scaled(T=1))


def test_full_size_long_context_host_resident_all_segments():
    """128K context with the cache in pinned host memory, C = 8192: the scan
    over the host link, the candidate rows staged for the two-pass refine,
    the pool gathered over the link."""
    _full_size_stages(LONG_128K_HOST.scaled(T=1), host=True)


def test_full_size_stack_layer_all_segments():
    """One layer of the 28-layer stack (8 sequences x 32K, G = 7): two row
    tiles of 18 tokens per segment, a ragged last tile."""
    _full_size_stages(QWEN_STACK.scaled(T=1))


@pytest.mark.parametrize("w", [
    TINY.scaled(T=1),                                   # L_pad <= 4096: the fused refine
    _case("exact-g7-ragged", Hq=14, Hkv=2, d=128, L=5000, B=32, C=512, K=200, S=8, W=40,
          n_planted=20, index=25),                      # two-pass refine over 5120 slots
    _case("exact-n2-d64", N=2, Hq=8, Hkv=2, d=64, L=3001, B=16, C=256, K=100, S=4, W=33,
          n_planted=12, index=26),
], ids=lambda w: w.name)
def test_exact_selection(w):
    """Every cached position scored with all the block's real queries, top-K
    plus sink/local, against the oracle's exact selection."""
    r = Run(w)
    x = r.x
    if w.name == "exact-n2-d64":
        x["ctx"] = np.array([3001, 2500], np.int32)  # ragged contexts
        r.ctx = dev(x["ctx"])
    d = r.d
    ws_bytes = H.herald_workspace_size_exact(d, w.K, w.P)
    assert ws_bytes > 0
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    H.herald_select_exact(d, r.q_steps[0], r.k, r.ctx, w.K, w.S, w.W, w.P, r.idx, r.n_sel, ws)
    torch.cuda.synchronize()
    assert H.herald_workspace_error(ws) == 0
    o = oracle.select_exact(f64(x["q_steps"][0]), f64(x["k_cache"]), x["ctx"], w.K, w.S, w.W,
                            w.P)
    idx, ns = r.idx.cpu().numpy(), r.n_sel.cpu().numpy()
    for n in range(w.N):
        for g in range(w.Hkv):
            check_selection(idx[n, g], int(ns[n, g]), o["idx"][n, g], int(o["n_sel"][n, g]),
                            o["cand"][n, g], o["n_cand"][n, g], o["s"][n, g], w,
                            int(x["ctx"][n]), f"{w.name} n={n} g={g}")


def test_exact_selection_workspace_checks():
    w = TINY
    d = H.dims_of(w)
    need = H.herald_workspace_size_exact(d, w.K, w.P)
    assert H.herald_workspace_size_exact(d, 0, w.P) == 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    idx = torch.zeros((w.N, w.Hkv, w.P), dtype=torch.int32, device="cuda")
    ns = torch.zeros((w.N, w.Hkv), dtype=torch.int32, device="cuda")
    with pytest.raises(H.HeraldError) as e:
        H.herald_select_exact(d, idx, idx, ns, w.K, w.S, w.W, w.P, idx, ns, ws, need - 256)
    assert e.value.status == 3


# --------------------------------------------------------------------------
# block-granular stage 1

BLOCK_CASES = [
    _case("blocks-g7", Hq=14, Hkv=2, d=128, L=5000, B=32, C=512, K=200, S=8, W=40,
          n_planted=20, index=44),
    _case("blocks-n2-d64", N=2, Hq=8, Hkv=2, d=64, L=3001, B=16, C=256, K=100, S=4, W=33,
          n_planted=10, index=45),
]


@pytest.mark.parametrize("Bk", [64, 16])
@pytest.mark.parametrize("w", BLOCK_CASES, ids=lambda w: w.name)
def test_block_stage1_matches_oracle(w, Bk):
    """Pooled keys (fp32 block means) within fp32 rounding of the oracle's
    fp64 means; the selected blocks equal the oracle's up to its tie band;
    the candidates are exactly those blocks' positions below ctx."""
    ctx = [w.L - 7] + [w.L - 100 * i for i in range(1, w.N)]  # ragged last blocks
    r = Run(w, ctx=ctx)
    x = r.x
    nb_max = -(-w.L_max // Bk)
    pooled = torch.full((w.N, w.Hkv, nb_max, w.d), 5.0, dtype=torch.float32, device="cuda")
    H.herald_pool_keys(r.d, r.k, r.ctx, Bk, pooled)
    C_blocks = w.C // Bk
    cand = torch.full((w.N, w.Hkv, C_blocks * Bk), -7, dtype=torch.int32, device="cuda")
    n_cand = torch.zeros((w.N, w.Hkv), dtype=torch.int32, device="cuda")
    H.herald_select_stage1_blocks(r.d, r.q_merge, pooled, r.ctx, Bk, C_blocks, cand, n_cand,
                                  r.ws)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    o = oracle.stage1_blocks(oracle.merged_query(f64(x["q_merge"])), f64(x["k_cache"]),
                             x["ctx"], Bk, C_blocks)
    np.testing.assert_allclose(pooled.cpu().numpy(), o["kp"], rtol=1e-5, atol=1e-6)
    cand, n_cand = cand.cpu().numpy(), n_cand.cpu().numpy()
    for n in range(w.N):
        L = int(x["ctx"][n])
        for g in range(w.Hkv):
            m = int(o["n_cand_b"][n, g])
            row = cand[n, g, : n_cand[n, g]]
            blocks = sorted(set((row // Bk).tolist()))
            assert_sets_within_band(blocks, o["cand_b"][n, g, :m], o["s1b"][n, g], m,
                                    f"blocks n={n} g={g}")
            want = [j for b in blocks for j in range(b * Bk, min((b + 1) * Bk, L))]
            assert row.tolist() == want
            assert (cand[n, g, n_cand[n, g]:] == -1).all()


def test_pooled_keys_tail_refresh_after_appends():
    """After appends grow the context, refreshing the last ceil(B/Bk) + 1
    blocks gives the pooled keys a full rebuild gives."""
    w = BLOCK_CASES[1]
    Bk = 16
    r = Run(w, ctx=[w.L - 40, w.L - 90])
    nb_max = -(-w.L_max // Bk)
    pooled = torch.zeros((w.N, w.Hkv, nb_max, w.d), dtype=torch.float32, device="cuda")
    H.herald_pool_keys(r.d, r.k, r.ctx, Bk, pooled)
    for t in range(2):  # two appends of B rows each
        H.herald_append_kv(r.d, r.bk[t], r.bv[t], r.ctx, r.k, r.v, advance=True)
        H.herald_pool_keys(r.d, r.k, r.ctx, Bk, pooled, n_tail=-(-w.B // Bk) + 1)
    full = torch.zeros_like(pooled)
    H.herald_pool_keys(r.d, r.k, r.ctx, Bk, full)
    torch.cuda.synchronize()
    assert torch.equal(pooled, full)


@pytest.mark.parametrize("w", [c for c in CASES if c.name in
                               ("g7-d128-ragged", "g4-d128-n2", "ctx-below-c",
                                "c-above-4096-two-pass")], ids=lambda w: w.name)
@pytest.mark.parametrize("tau", [0.3, 0.8])
def test_adaptive_budget_stage2(w, tau):
    """The per-(n, g) budget from the first step's stage-2 mass (the MAGE
    author page's first-step budget prediction, in the reading stated with
    the oracle): the device's budget is a valid one for the oracle's fp64
    scores (its top-k mass reaches tau of the total, the top k-1 do not,
    both within a relative 1e-3), within 2 of the oracle's, and the
    selection with it matches the oracle's selection with the same budget."""
    r = Run(w)
    x = r.x
    s1 = _oracle_stage1(x)
    cand_o, nc_o = oracle.topc(s1, x["ctx"], w.C)
    s2 = oracle.stage2_scores(f64(x["q_steps"][0]), f64(x["k_cache"]), cand_o, nc_o)
    K_min, K_max = max(1, w.K // 8), w.K
    k_sel = torch.full((w.N, w.Hkv), -7, dtype=torch.int32, device="cuda")
    H.herald_select_stage2_adaptive(r.d, r.q_steps[0], r.k, r.ctx, dev(cand_o), dev(nc_o), w.C,
                                    K_min, K_max, tau, w.S, w.W, r.P, r.idx, r.n_sel, k_sel,
                                    r.ws)
    torch.cuda.synchronize()
    assert r.error_word() == 0
    # deterministic: the same budgets and selection on every run (the bin
    # masses are summed in fixed point, in any order to the same value)
    first = (k_sel.clone(), r.idx.clone())
    for _ in range(3):
        H.herald_select_stage2_adaptive(r.d, r.q_steps[0], r.k, r.ctx, dev(cand_o), dev(nc_o),
                                        w.C, K_min, K_max, tau, w.S, w.W, r.P, r.idx, r.n_sel,
                                        k_sel, r.ws)
        torch.cuda.synchronize()
        assert torch.equal(k_sel, first[0]) and torch.equal(r.idx, first[1])
    kb = k_sel.cpu().numpy()
    kb_o = oracle.adaptive_budget(s2, nc_o, tau, K_min, K_max)
    for n in range(w.N):
        for g in range(w.Hkv):
            # the device's budget must be the clamp of a k that holds tau of
            # the oracle's mass where k - 1 does not, both up to a relative
            # 1e-3 (the device sums in fp32); where no such tie exists it is
            # the oracle's budget exactly
            m = int(nc_o[n, g])
            cum = np.cumsum(np.sort(s2[n, g, :m])[::-1]) if m else np.zeros(0)
            target = tau * (cum[-1] if m else 0.0)
            valid = {max(K_min, min(K_max, min(k, m))) for k in range(1, m + 1)
                     if cum[k - 1] >= target * (1 - 1e-3)
                     and (k == 1 or cum[k - 2] < target * (1 + 1e-3))} if m else {K_min}
            valid.add(int(kb_o[n, g]))
            assert int(kb[n, g]) in valid, (n, g, int(kb[n, g]), sorted(valid)[:5])
    idx_o, ns_o = oracle.select_final_per_head(x["ctx"], w.L_max, cand_o, nc_o, s2, kb, w.S, w.W,
                                               w.P)
    idx, ns = r.idx.cpu().numpy(), r.n_sel.cpu().numpy()
    for n in range(w.N):
        for g in range(w.Hkv):
            m, k = int(nc_o[n, g]), int(kb[n, g])
            cum = np.cumsum(np.sort(s2[n, g, :m])[::-1])
            if m and K_min < k < min(K_max, m):   # the budget was not clamped
                target = tau * cum[-1]
                assert cum[k - 1] >= target * (1 - 1e-3), (n, g, k)
                assert k == 1 or cum[k - 2] < target * (1 + 1e-3), (n, g, k)
            check_selection(idx[n, g], int(ns[n, g]), idx_o[n, g], int(ns_o[n, g]),
                            cand_o[n, g], nc_o[n, g], s2[n, g], w.scaled(K=k), int(x["ctx"][n]),
                            f"{w.name} tau={tau} n={n} g={g}")
