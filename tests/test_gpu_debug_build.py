"""The debug build (libherald.so compiled with -DHERALD_DEBUG): its kernels
check the indices and counts they read and write on the device, where a
memory checker is not at hand, and record violations in a check word
instead of trapping.

On valid inputs the whole path -- stage 1, stage 2 with the gather, every
denoising step, the append -- must leave the word at 0 and produce the
release library's outputs bit for bit.  On inputs that are invalid but stay
inside their allocations (so that neither build can read outside memory),
the word must name the violation: a selected row past the cache's rows, a
selection count past P_max, a candidate outside the cache, a context length
past L_max.

The debug library runs in a child process (the binding loads one library
per process; HERALD_LIB=debug selects it)."""
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

BAD_INDEX, BAD_COUNT = 0x10, 0x20


def _workload():
    from block_diffusion_sparse_gb300.workloads import Workload
    return Workload("debug", N=2, Hq=8, Hkv=2, d=128, L=3000, B=16, T=2, C=256, K=96, S=16,
                    W=48, planted="points", n_planted=6, index=81, extra_rows=16)


def run_path(out_path):
    """The path on valid inputs through the loaded library; saves every output
    (and, for the debug build, the check word after it) to out_path."""
    from block_diffusion_sparse_gb300 import herald as H
    from block_diffusion_sparse_gb300 import synth
    from helpers import dev
    w = _workload()
    x = synth.make_layer(w)
    d = H.dims_of(w)
    NG = (w.N, w.Hkv)
    k, v, ctx = dev(x["k_cache"]), dev(x["v_cache"]), dev(x["ctx"])
    ws = torch.zeros(H.herald_workspace_size(d, w.C, w.P), dtype=torch.uint8, device="cuda")
    cand = torch.zeros((*NG, w.C), dtype=torch.int32, device="cuda")
    n_cand = torch.zeros(NG, dtype=torch.int32, device="cuda")
    idx = torch.zeros((*NG, w.P), dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(NG, dtype=torch.int32, device="cuda")
    pk = torch.zeros((*NG, w.P, w.d), dtype=torch.int16, device="cuda")
    pv = torch.zeros_like(pk)
    outs = torch.zeros((w.T, w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
    q = dev(x["q_steps"])
    bk, bv = dev(x["block_k"]), dev(x["block_v"])
    H.herald_select_stage1(d, dev(x["q_merge"]), k, ctx, w.C, cand, n_cand, ws)
    H.herald_select_stage2_gather(d, q[0], k, v, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, idx,
                                  n_sel, pk, pv, ws)
    for t in range(w.T):
        flags = (H.HERALD_ATTN_SETTLED if t else 0) | \
            (H.HERALD_ATTN_APPEND | H.HERALD_ATTN_ADVANCE if t == w.T - 1 else 0)
        H.herald_denoise_attn_ex(d, q[t], pk, pv, n_sel, w.P, bk[t], bv[t], outs[t], 0.0, flags,
                                 ctx, k, v, ws)
    torch.cuda.synchronize()
    word = H.herald_debug_status()
    np.savez(out_path, cand=cand.cpu().numpy(), idx=idx.cpu().numpy(),
             n_sel=n_sel.cpu().numpy(), pk=pk.cpu().numpy(), outs=outs.cpu().numpy(),
             k=k.cpu().numpy(), ctx=ctx.cpu().numpy(), err=H.herald_workspace_error(ws),
             word=word, debug=H.herald_debug_build())


def run_violations(out_path):
    """Invalid inputs that stay inside their allocations; saves the check word
    after each case."""
    from block_diffusion_sparse_gb300 import herald as H
    from block_diffusion_sparse_gb300 import synth
    from helpers import dev
    w = _workload()
    x = synth.make_layer(w)
    d = H.dims_of(w)
    NG = (w.N, w.Hkv)
    words = {}
    # (1) a selected row past the cache's rows: the buffer passed as the
    # cache is larger than N*Hkv*L_max rows, so the row's address lies inside
    # it, but every build skips the read and writes a zero row
    kbig = torch.zeros((w.N, w.Hkv, w.L_max + 64, w.d), dtype=torch.int16, device="cuda")
    idx = torch.arange(w.P, dtype=torch.int32, device="cuda").repeat(w.N * w.Hkv).view(*NG, w.P)
    idx[0, 1, 5] = w.L_max + 3
    n_sel = torch.full(NG, w.P, dtype=torch.int32, device="cuda")
    pk = torch.full((*NG, w.P, w.d), 7, dtype=torch.int16, device="cuda")
    pv = torch.full_like(pk, 7)
    H.herald_debug_status()
    H.herald_gather(d, idx, n_sel, w.P, kbig, kbig, pk, pv)
    torch.cuda.synchronize()
    words["row_past_cache"] = H.herald_debug_status()
    words["row_zeroed"] = int((pk[0, 1, 5] == 0).all())
    # (2) a selection count past P_max (the kernel clamps it)
    n_sel.fill_(w.P + 10)
    H.herald_gather(d, idx.clamp(max=w.L - 1), n_sel, w.P, kbig, kbig, pk, pv)
    torch.cuda.synchronize()
    words["count_past_pmax"] = H.herald_debug_status()
    # (3) candidate positions outside the cache (past L_max, and negative):
    # the refine reads them as zero rows, and its check names them
    k, ctx = dev(x["k_cache"]), dev(x["ctx"])
    cand = torch.arange(w.C, dtype=torch.int32, device="cuda").repeat(w.N * w.Hkv).view(*NG, w.C)
    cand[1, 0, 100] = w.L_max + 7
    cand[0, 1, 200] = -3
    n_cand = torch.full(NG, w.C, dtype=torch.int32, device="cuda")
    ws = torch.zeros(H.herald_workspace_size(d, w.C, w.P), dtype=torch.uint8, device="cuda")
    sel = torch.zeros((*NG, w.P), dtype=torch.int32, device="cuda")
    ns = torch.zeros(NG, dtype=torch.int32, device="cuda")
    q0 = dev(x["q_steps"][0])
    H.herald_select_stage2(d, q0, k, ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, sel, ns, ws)
    torch.cuda.synchronize()
    words["candidate_outside_cache"] = H.herald_debug_status()
    # (4) a context length past L_max (every kernel clamps it to L_max)
    cand = torch.arange(w.C, dtype=torch.int32, device="cuda").repeat(w.N * w.Hkv).view(*NG, w.C)
    long_ctx = torch.full_like(ctx, w.L_max + 100)
    H.herald_select_stage2(d, q0, k, long_ctx, cand, n_cand, w.C, w.K, w.S, w.W, w.P, sel, ns,
                           ws)
    torch.cuda.synchronize()
    words["ctx_past_lmax"] = H.herald_debug_status()
    words["after"] = H.herald_debug_status()
    np.savez(out_path, **{kk: np.int64(vv) for kk, vv in words.items()})


def _child(fn, out_path):
    env = dict(os.environ, HERALD_LIB="debug")
    code = (f"import sys; sys.path[:0] = [{HERE!r}, {ROOT!r}]; "
            f"import test_gpu_debug_build as t; t.{fn}({out_path!r})")
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=HERE, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return np.load(out_path)


@pytest.mark.gpu
def test_debug_build_on_valid_inputs_checks_clean_and_matches_release(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_diffusion_sparse_gb300 import build
    assert os.path.exists(build.DEBUG_LIB), "the debug build is made by __graft_entry__.build()"
    dbg = _child("run_path", str(tmp_path / "debug.npz"))
    assert int(dbg["debug"]) == 1
    assert int(dbg["word"]) == 0, f"device checks failed on valid inputs: {int(dbg['word']):#x}"
    assert int(dbg["err"]) == 0
    run_path(str(tmp_path / "release.npz"))
    rel = np.load(str(tmp_path / "release.npz"))
    assert int(rel["debug"]) == 0 and int(rel["word"]) == 0
    for key in ("cand", "idx", "n_sel", "pk", "outs", "k", "ctx"):
        assert np.array_equal(dbg[key], rel[key]), key


@pytest.mark.gpu
def test_debug_build_names_index_and_count_violations(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _child("run_violations", str(tmp_path / "violations.npz"))
    assert int(r["row_past_cache"]) & BAD_INDEX
    assert int(r["row_zeroed"]) == 1
    assert int(r["count_past_pmax"]) & BAD_COUNT
    assert int(r["candidate_outside_cache"]) & BAD_INDEX
    assert int(r["ctx_past_lmax"]) & BAD_COUNT
    assert int(r["after"]) == 0, "reading the word clears it"
