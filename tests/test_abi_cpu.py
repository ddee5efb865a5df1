"""CPU-side checks of the C-ABI library: it loads, exports every symbol the
header declares, and rejects invalid arguments on the host without touching
a GPU (every failing call below returns before any CUDA call)."""
import ctypes as C
import os
import re

import pytest

from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300.workloads import ALL, QWEN_32K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _built():
    if not os.path.exists(H.LIB_PATH):
        from block_diffusion_sparse_gb300 import build
        build.build()
    return H.lib()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "herald.h")).read()
    return sorted(set(re.findall(r"\b(herald_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_are_all_exported():
    lib = _built()
    names = _declared_symbols()
    assert set(names) == set(H.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size_is_positive_and_monotone():
    _built()
    d = H.dims_of(QWEN_32K)
    a = H.herald_workspace_size(d, 4096, 1344)
    b = H.herald_workspace_size(d, 8192, 1344)
    c = H.herald_workspace_size(d, 4096, 2688)
    assert 0 < a < b and a < c
    for w in ALL.values():
        assert H.herald_workspace_size(H.dims_of(w), w.C, w.P) > 0


@pytest.mark.parametrize("bad,status", [
    (dict(d=96), 2),
    (dict(Hq=30, Hkv=4), 2),
    (dict(Hq=36, Hkv=4), 2),      # G = 9 > 8
    (dict(B=64), 2),              # B*G = 448 > 256
    (dict(N=0), 1),
    (dict(L_max=0), 1),
])
def test_bad_dims_rejected(bad, status):
    _built()
    base = dict(N=1, Hq=28, Hkv=4, d=128, B=32, L_max=1024)
    base.update(bad)
    d = H.dims(**base)
    assert H.herald_workspace_size(d, 256, 512) == 0
    with pytest.raises(H.HeraldError) as e:
        H.herald_select(d, 16, 16, 16, 16, 256, 128, 16, 64, 512, 16, 16, 16, ws_bytes=1 << 30)
    assert e.value.status == status


def test_argument_errors_rejected_before_launch():
    _built()
    d = H.dims(1, 4, 1, 64, 16, 2048)
    ok = 1 << 12  # aligned fake address; never dereferenced on these paths
    ws_need = H.herald_workspace_size(d, 256, 208)
    cases = [
        (dict(q_merge=0), 1),           # NULL pointer
        (dict(q_block=ok + 8), 1),      # misaligned
        (dict(K=300), 1),               # K > C
        (dict(sink=-1), 1),
        (dict(P_max=100), 1),           # P_max < K + sink + local
        (dict(C=0), 2),
        (dict(C=20000), 2),
        (dict(ws_bytes=ws_need - 1), 3),
    ]
    for over, status in cases:
        a = dict(q_merge=ok, q_block=ok, k_cache=ok, ctx=ok, C=256, K=128, sink=16, local=64,
                 P_max=208, idx=ok, n_sel=ok, ws=ok, ws_bytes=ws_need)
        a.update(over)
        with pytest.raises(H.HeraldError) as e:
            H.herald_select(d, a["q_merge"], a["q_block"], a["k_cache"], a["ctx"], a["C"], a["K"],
                            a["sink"], a["local"], a["P_max"], a["idx"], a["n_sel"], a["ws"],
                            a["ws_bytes"])
        assert e.value.status == status, (over, e.value)
        assert H.lib().herald_last_error().decode()


def test_attention_and_gather_argument_errors():
    _built()
    d = H.dims(1, 4, 1, 64, 16, 2048)
    ok = 1 << 12
    ws = H.herald_workspace_size(d, 1, 208)
    with pytest.raises(H.HeraldError) as e:
        H.herald_denoise_attn(d, ok, ok, ok, ok, 208, ok, ok, 0, 0.0, ok, ws)
    assert e.value.status == 1
    with pytest.raises(H.HeraldError) as e:
        H.herald_denoise_attn(d, ok, ok, ok, ok, 208, ok, ok, ok, -1.0, ok, ws)
    assert e.value.status == 1
    # the options of a denoising step: unknown bits, an unknown kernel
    # choice, ADVANCE without APPEND, APPEND without a cache
    for flags, extra in [(8, {}), (1 << 24, {}), (9 << 8, {}), (H.HERALD_ATTN_ADVANCE, {}),
                         (H.HERALD_ATTN_APPEND, dict(ctx_len=None, k_cache=ok, v_cache=ok)),
                         (H.HERALD_ATTN_APPEND, dict(ctx_len=ok, k_cache=ok, v_cache=None))]:
        a = dict(ctx_len=ok, k_cache=ok, v_cache=ok)
        a.update(extra)
        with pytest.raises(H.HeraldError) as e:
            H.herald_denoise_attn_ex(d, ok, ok, ok, ok, 208, ok, ok, ok, 0.0, flags,
                                     a["ctx_len"], a["k_cache"], a["v_cache"], ok, ws)
        assert e.value.status == 1, (flags, extra)
    with pytest.raises(H.HeraldError) as e:
        H.herald_gather(d, ok, ok, 0, ok, ok, ok, ok)
    assert e.value.status == 1
    with pytest.raises(H.HeraldError) as e:
        H.herald_append_kv(d, ok, ok, ok, ok, ok + 4)
    assert e.value.status == 1


def test_block_call_argument_errors():
    """herald_block checks its own arguments and everything its calls would
    check before the first of them launches."""
    _built()
    d = H.dims(1, 4, 1, 64, 16, 2048)
    ok = 1 << 12
    ws = H.herald_workspace_size(d, 256, 208)

    def bufs(sel=None, ev=(ok, ok), ws_bytes=ws):
        b = H.BlockBufs()
        b.cand[0] = b.cand[1] = b.n_cand[0] = b.n_cand[1] = ok
        b.idx = b.n_sel = ok
        b.pool_k[0] = b.pool_k[1] = b.pool_v[0] = b.pool_v[1] = ok
        b.ws_den = b.ws_sel = ok
        b.ws_bytes = ws_bytes
        b.sel_stream = sel
        b.ev_fork, b.ev_join = ev
        return b

    def call(b, T=2, i=0, flags=0, scan_sms=0, K=128, q=ok, nk=None):
        H.herald_block(d, 256, K, 16, 64, 208, T, i, q, ok, ok, ok, ok, ok, nk, ok, flags,
                       scan_sms, b)

    cases = [(dict(flags=4), bufs(), 1), (dict(flags=H.HERALD_BLOCK_CAND_SETTLED | 8), bufs(), 1),
             (dict(T=0), bufs(), 1), (dict(i=-1), bufs(), 1),
             (dict(scan_sms=-1), bufs(ok), 1), (dict(), bufs(ok, (ok, None)), 1),
             (dict(), bufs(ok, (None, ok)), 1), (dict(K=300), bufs(), 1),
             (dict(q=ok + 4), bufs(), 1), (dict(nk=ok + 8), bufs(), 1),
             (dict(), bufs(ws_bytes=ws - 1), 3)]
    for kw, b, status in cases:
        with pytest.raises(H.HeraldError) as e:
            call(b, **kw)
        assert e.value.status == status, kw
        assert H.lib().herald_last_error().decode()
    with pytest.raises(H.HeraldError) as e:  # no buffers at all
        H.check(H.lib().herald_block(d, 256, 128, 16, 64, 208, 2, 0, ok, ok, ok, ok, ok, ok,
                                     None, ok, 0, 0, None, None))
    assert e.value.status == 1


def test_block_stage1_and_staging_argument_errors():
    _built()
    d = H.dims(1, 4, 1, 64, 16, 2048)
    ok = 1 << 12
    ws = H.herald_workspace_size(d, 256, 208)
    for Bk, n_tail, status in [(0, 0, 1), (4096, 0, 1), (64, -1, 1)]:
        with pytest.raises(H.HeraldError) as e:
            H.herald_pool_keys(d, ok, ok, Bk, ok, n_tail=n_tail)
        assert e.value.status == status, (Bk, n_tail)
    for Bk, Cb, status in [(0, 4, 1), (64, 0, 2), (64, 300, 2)]:   # C_blocks*Bk <= 16384
        with pytest.raises(H.HeraldError) as e:
            H.herald_select_stage1_blocks(d, ok, ok, ok, Bk, Cb, ok, ok, ok, ws)
        assert e.value.status == status, (Bk, Cb)
    with pytest.raises(H.HeraldError) as e:
        H.herald_stage_candidates(d, ok, ok, ok, 256, None)
    assert e.value.status == 1
    with pytest.raises(H.HeraldError) as e:
        H.herald_select_stage2_staged(d, ok, None, ok, ok, ok, 256, 128, 16, 64, 208, ok, ok, ok,
                                      ws)
    assert e.value.status == 1
    # the V rows need both the cache and the staging buffer
    for vc, sv in [(ok, None), (None, ok)]:
        with pytest.raises(H.HeraldError) as e:
            H.herald_stage_candidates(d, ok, ok, ok, 256, ok, v_cache=vc, staged_v=sv)
        assert e.value.status == 1, (vc, sv)
    # stage 2 + gather over staged rows: every pointer is required
    args = [ok, ok, ok, ok, ok, ok, ok, ok]  # q, staged_k, staged_v, k, v, ctx, cand, n_cand
    for miss in range(len(args)):
        a = list(args)
        a[miss] = None
        with pytest.raises(H.HeraldError) as e:
            H.herald_select_stage2_staged_gather(d, *a, 256, 128, 16, 64, 208, ok, ok, ok, ok,
                                                 ok, ws)
        assert e.value.status == 1, miss
    # the adaptive budget: K_min in [0, K_max], tau in (0, 1], every pointer
    for K_min, K_max, tau in [(-1, 128, 0.5), (129, 128, 0.5), (0, 128, 0.0), (0, 128, 1.5),
                              (0, 128, float("nan")), (0, 300, 0.5)]:
        with pytest.raises(H.HeraldError) as e:
            H.herald_select_stage2_adaptive(d, ok, ok, ok, ok, ok, 256, K_min, K_max, tau, 16, 64,
                                            400, ok, ok, ok, ok, ws)
        assert e.value.status == 1, (K_min, K_max, tau)
    with pytest.raises(H.HeraldError) as e:
        H.herald_select_stage2_adaptive(d, ok, ok, ok, ok, ok, 256, 8, 128, 0.5, 16, 64, 208, ok,
                                        ok, None, ok, ws)
    assert e.value.status == 1
    with pytest.raises(H.HeraldError) as e:   # K > C
        H.herald_select_stage2_staged_gather(d, *args, 256, 300, 16, 64, 400, ok, ok, ok, ok, ok,
                                             ws)
    assert e.value.status == 1


def test_status_strings():
    _built()
    for s in range(5):
        assert H.herald_status_string(s)
    assert H.herald_status_string(99) == "unknown status"


def test_an_injected_launch_failure_is_reported_as_a_cuda_error():
    """The host-side error path of a failed launch, without a GPU: the hook
    makes the gather's launch return cudaErrorLaunchFailure (719), which the
    entry point reports as HERALD_ERR_CUDA naming the launch; the hook then
    disarms itself."""
    _built()
    d = H.dims(1, 8, 2, 128, 16, 1024)
    p = 1 << 12  # aligned addresses: nothing reaches the device
    H.herald_inject_launch_failure(0, 719)
    with pytest.raises(H.HeraldError) as e:
        H.herald_gather(d, p, p, 64, p, p, p, p)
    assert e.value.status == 4
    assert "gather launch" in str(e.value) and "cudaErrorLaunchFailure" in str(e.value)
    # disarmed: the next call reaches the real launch (which, with no GPU
    # here, fails for its own reason -- not the injected one)
    try:
        H.herald_gather(d, p, p, 64, p, p, p, p)
    except H.HeraldError as e2:
        assert "cudaErrorLaunchFailure" not in str(e2)
    # arming needs an error code; a negative count disarms
    with pytest.raises(H.HeraldError) as e:
        H.herald_inject_launch_failure(0, 0)
    assert e.value.status == 1
    H.herald_inject_launch_failure(-1, 0)


def test_release_build_reports_no_debug_checks():
    """The release library has the device checks compiled out: its check
    word reads 0 without touching a device."""
    _built()
    assert not H.herald_debug_build()
    assert H.herald_debug_status() == 0
