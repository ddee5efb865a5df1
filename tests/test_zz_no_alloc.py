"""herald_select_stage2_noalloc -- stage 2 for callers that cannot allocate
device memory where they select (a decode loop under CUDA stream capture, a
plugin whose host runtime owns the device-memory budget) -- must produce
exactly what herald_select_stage2 produces with a caller-provided workspace,
call after call, although every call reuses the same static scratch.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone."""
import numpy as np
import pytest

from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.workloads import QWEN_32K, Workload


def _dev(torch, a):
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("w", [
    Workload("noalloc-g7", N=1, Hq=14, Hkv=2, d=128, L=5000, B=32, T=1, C=512, K=200, S=8, W=40,
             planted="points", n_planted=20, index=41, extra_rows=16),
    QWEN_32K.scaled(T=1, n_planted=64),
], ids=lambda w: w.name)
def test_noalloc_stage2_matches_workspace_stage2_twice(w):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    x = synth.make_layer(w)
    d = H.dims_of(w)
    q_merge, q = _dev(torch, x["q_merge"]), _dev(torch, x["q_steps"][0])
    k, ctx = _dev(torch, x["k_cache"]), _dev(torch, x["ctx"])
    NG = (w.N, w.Hkv)
    ws_bytes = H.herald_workspace_size(d, w.C, w.P)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    cand = torch.empty((*NG, w.C), dtype=torch.int32, device="cuda")
    n_cand = torch.empty(NG, dtype=torch.int32, device="cuda")
    H.herald_select_stage1(d, q_merge, k, ctx, w.C, cand, n_cand, ws)

    ref_idx = torch.full((*NG, w.P), -7, dtype=torch.int32, device="cuda")
    ref_ns = torch.zeros(NG, dtype=torch.int32, device="cuda")
    H.herald_select_stage2(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, ref_idx, ref_ns,
                           ws)
    for call in range(2):
        idx = torch.full((*NG, w.P), -9, dtype=torch.int32, device="cuda")
        ns = torch.full(NG, -9, dtype=torch.int32, device="cuda")
        H.herald_select_stage2_noalloc(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx,
                                       ns)
        torch.cuda.synchronize()
        # same kernels on the same inputs: index outputs are identical
        assert torch.equal(ns, ref_ns), f"call {call}: n_sel differs"
        assert torch.equal(idx, ref_idx), f"call {call}: idx differs"
    assert int(ref_ns.min()) > 0


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    """Host-side check (launches nothing): 64 x 8 segments x 8192 candidates
    need far more than the 4 MiB static scratch."""
    d = H.dims(64, 32, 8, 128, 32, 8192)
    ok = 1 << 12
    with pytest.raises(H.HeraldError) as e:
        H.herald_select_stage2_noalloc(d, ok, ok, ok, ok, ok, 8192, 1024, 64, 256, 1344, ok, ok)
    assert e.value.status == 3
    assert "scratch" in str(e.value)


@pytest.mark.gpu
def test_noalloc_two_pass_refine_matches_workspace_stage2():
    """C > 4096 (the two-pass refine, its row log-sum-exp at its own offset
    in the static scratch) with few enough segments to fit the 4 MiB."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = Workload("noalloc-two-pass", N=1, Hq=8, Hkv=2, d=128, L=12000, B=16, T=1, C=8192, K=256,
                 S=16, W=64, planted="points", n_planted=12, index=46, extra_rows=16)
    x = synth.make_layer(w)
    d = H.dims_of(w)
    q_merge, q = _dev(torch, x["q_merge"]), _dev(torch, x["q_steps"][0])
    k, ctx = _dev(torch, x["k_cache"]), _dev(torch, x["ctx"])
    NG = (w.N, w.Hkv)
    ws = torch.zeros(H.herald_workspace_size(d, w.C, w.P), dtype=torch.uint8, device="cuda")
    cand = torch.empty((*NG, w.C), dtype=torch.int32, device="cuda")
    n_cand = torch.empty(NG, dtype=torch.int32, device="cuda")
    H.herald_select_stage1(d, q_merge, k, ctx, w.C, cand, n_cand, ws)
    ref_idx = torch.full((*NG, w.P), -7, dtype=torch.int32, device="cuda")
    ref_ns = torch.zeros(NG, dtype=torch.int32, device="cuda")
    H.herald_select_stage2(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, ref_idx, ref_ns,
                           ws)
    for call in range(2):
        idx = torch.full((*NG, w.P), -9, dtype=torch.int32, device="cuda")
        ns = torch.full(NG, -9, dtype=torch.int32, device="cuda")
        H.herald_select_stage2_noalloc(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx,
                                       ns)
        torch.cuda.synchronize()
        assert torch.equal(ns, ref_ns), f"call {call}: n_sel differs"
        assert torch.equal(idx, ref_idx), f"call {call}: idx differs"


@pytest.mark.gpu
def test_noalloc_rejects_a_host_resident_cache():
    """A cache in pinned host memory needs its candidate rows staged, which
    this call has no room for: rejected before anything is launched."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = Workload("noalloc-host", N=1, Hq=8, Hkv=2, d=128, L=2000, B=16, T=1, C=256, K=64, S=8,
                 W=32, planted="points", n_planted=4, index=47, extra_rows=16)
    x = synth.make_layer(w)
    d = H.dims_of(w)
    kh = torch.from_numpy(x["k_cache"].view(np.int16)).pin_memory()
    q, ctx = _dev(torch, x["q_steps"][0]), _dev(torch, x["ctx"])
    NG = (w.N, w.Hkv)
    cand = torch.zeros((*NG, w.C), dtype=torch.int32, device="cuda")
    n_cand = torch.zeros(NG, dtype=torch.int32, device="cuda")
    idx = torch.zeros((*NG, w.P), dtype=torch.int32, device="cuda")
    ns = torch.zeros(NG, dtype=torch.int32, device="cuda")
    with pytest.raises(H.HeraldError) as e:
        H.herald_select_stage2_noalloc(d, q, kh, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx,
                                       ns)
    assert e.value.status == 1
    assert "device memory" in str(e.value)


def test_noalloc_applies_the_stage2_argument_rules():
    """Host-side checks (launch nothing): the same rules as
    herald_select_stage2, including the N*Hkv*P_max bound of the int32 index
    layout, which the scratch limit alone would not catch."""
    ok = 1 << 12
    d = H.dims(1, 8, 2, 128, 16, 4096)
    with pytest.raises(H.HeraldError) as e:   # K > C
        H.herald_select_stage2_noalloc(d, ok, ok, ok, ok, ok, 64, 65, 0, 0, 65, ok, ok)
    assert e.value.status == 1
    with pytest.raises(H.HeraldError) as e:   # K + sink + local > P_max
        H.herald_select_stage2_noalloc(d, ok, ok, ok, ok, ok, 64, 32, 16, 32, 64, ok, ok)
    assert e.value.status == 1
    with pytest.raises(H.HeraldError) as e:   # N*Hkv*P_max >= 2^31
        H.herald_select_stage2_noalloc(d, ok, ok, ok, ok, ok, 64, 32, 0, 0, 1 << 30, ok, ok)
    assert e.value.status == 2
