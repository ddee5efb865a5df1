"""Device-side failure detection without a GPU fault: every wait inside the
library's kernels is bounded; when it runs out the kernel records a code in
the workspace's error word and returns, and the host reads the code.  The
self-test entry point waits, through that same bounded wait, on a barrier
nothing completes."""
import time

import pytest

torch = pytest.importorskip("torch")

from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300.workloads import TINY
from helpers import dev
from block_diffusion_sparse_gb300 import synth


@pytest.mark.gpu
def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = TINY
    d = H.dims_of(w)
    ws_bytes = H.herald_workspace_size(d, w.C, w.P)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    assert H.herald_workspace_error(ws) == 0
    t0 = time.perf_counter()
    H.herald_selftest_wait_timeout(2_000_000, ws)  # 2 ms
    code = H.herald_workspace_error(ws)            # synchronises
    elapsed = time.perf_counter() - t0
    assert code == 1, "the timed-out wait must be reported as a copy-wait timeout"
    assert elapsed >= 2e-3
    assert H.herald_workspace_error(ws) == 0, "reading the word clears it"
    # the context is intact: the whole path still runs and reports no error
    x = synth.make_layer(w)
    NG = (w.N, w.Hkv)
    idx = torch.full((*NG, w.P), -1, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(NG, dtype=torch.int32, device="cuda")
    H.herald_select(d, dev(x["q_merge"]), dev(x["q_steps"][0]), dev(x["k_cache"]),
                    dev(x["ctx"]), w.C, w.K, w.S, w.W, w.P, idx, n_sel, ws)
    torch.cuda.synchronize()
    assert H.herald_workspace_error(ws) == 0
    assert int(n_sel.min()) > 0


def test_self_test_rejects_limits_outside_its_range():
    """Host-side check: launches nothing."""
    ws = 1 << 12  # an address; nothing is launched for rejected arguments
    for bad in (0, 2_000_000_000):
        with pytest.raises(H.HeraldError) as e:
            H.herald_selftest_wait_timeout(bad, ws)
        assert e.value.status == 1


@pytest.mark.gpu
def test_a_launch_failure_inside_a_call_is_reported_and_the_context_stays_usable():
    """An injected failure of the second launch of stage 2 (the top-K after
    the refine): HERALD_ERR_CUDA naming that launch; the next, untouched call
    selects exactly what a clean run selects."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = TINY
    d = H.dims_of(w)
    x = synth.make_layer(w)
    ws = torch.zeros(H.herald_workspace_size(d, w.C, w.P), dtype=torch.uint8, device="cuda")
    NG = (w.N, w.Hkv)
    cand = torch.zeros((*NG, w.C), dtype=torch.int32, device="cuda")
    n_cand = torch.zeros(NG, dtype=torch.int32, device="cuda")
    idx = torch.full((*NG, w.P), -1, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(NG, dtype=torch.int32, device="cuda")
    q, k, ctx = dev(x["q_steps"][0]), dev(x["k_cache"]), dev(x["ctx"])
    H.herald_select_stage1(d, dev(x["q_merge"]), k, ctx, w.C, cand, n_cand, ws)
    H.herald_select_stage2(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx, n_sel, ws)
    torch.cuda.synchronize()
    ref = (idx.clone(), n_sel.clone())
    idx.fill_(-5)
    H.herald_inject_launch_failure(1, 719)
    with pytest.raises(H.HeraldError) as e:
        H.herald_select_stage2(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx, n_sel,
                               ws)
    assert e.value.status == 4 and "topk_union launch" in str(e.value)
    torch.cuda.synchronize()
    H.herald_select_stage2(d, q, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx, n_sel, ws)
    torch.cuda.synchronize()
    assert H.herald_workspace_error(ws) == 0
    assert torch.equal(idx, ref[0]) and torch.equal(n_sel, ref[1])
