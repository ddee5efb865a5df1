"""The pipelined attention kernel (key tiles streamed through shared
memory, 8, 4 or 2 CTAs per row tile) and the cluster pool kernel (a whole
pool slice per CTA, 8 or 16 CTAs per row tile) against the fp64 oracle and
against each other, over the shapes of the workloads: GQA groups that
fill one row tile or need two, both head dimensions, single-token blocks,
ragged and empty selections, pools larger than the pool kernel takes, and
the append of the last denoising step.  Attention outputs within 2e-2 of
the oracle (bf16 inputs and output, fp32 accumulation)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle
from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import synth
from block_diffusion_sparse_gb300.workloads import Workload
from helpers import ATTN_ATOL, bf16_dev_to_f64, dev, f64


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    H.lib()


CS_FLAGS = {2: H.HERALD_ATTN_KERNEL_FLASH_CS2, 4: H.HERALD_ATTN_KERNEL_FLASH_CS4,
            8: H.HERALD_ATTN_KERNEL_FLASH_CS8}
POOL_FLAGS = {8: H.HERALD_ATTN_KERNEL_POOL_CS8, 12: H.HERALD_ATTN_KERNEL_POOL_CS12,
              16: H.HERALD_ATTN_KERNEL_POOL_CS16}


def _w(name, **kw):
    base = dict(N=2, Hq=8, Hkv=2, d=128, L=3000, B=32, T=2, C=512, K=300, S=16, W=64,
                planted="points", n_planted=6, index=91, extra_rows=32)
    base.update(kw)
    return Workload(name, **base)


SHAPES = [
    _w("g4-d128"),                                             # one 128-row tile
    _w("g7-d128-two-tiles", Hq=14, Hkv=2, index=92),           # 18 + 14 tokens
    _w("g4-d64", d=64, index=93),
    _w("g1-b1", Hq=2, Hkv=2, B=1, index=94),                   # single-token block
    _w("g8-b16-big-pool", Hq=16, Hkv=2, B=16, C=3000, K=2400, index=95),  # P > 2048
]


def _setup(w, seed):
    x = synth.make_layer(w)
    rng = np.random.default_rng(seed)
    NG = (w.N, w.Hkv)
    # a selection of its own per (n, g): ragged counts (one empty), ascending
    ns = rng.integers(0, w.P + 1, size=NG).astype(np.int32)
    ns[0, 0] = w.P
    ns[-1, -1] = 0 if w.N * w.Hkv > 1 else ns[-1, -1]
    idx = np.full((*NG, w.P), -1, np.int32)
    for n in range(w.N):
        for g in range(w.Hkv):
            idx[n, g, : ns[n, g]] = np.sort(rng.choice(w.L, size=ns[n, g], replace=False))
    pk = np.zeros((*NG, w.P, w.d), np.uint16)
    pv = np.zeros_like(pk)
    for n in range(w.N):
        for g in range(w.Hkv):
            m = ns[n, g]
            pk[n, g, :m] = x["k_cache"][n, g, idx[n, g, :m]]
            pv[n, g, :m] = x["v_cache"][n, g, idx[n, g, :m]]
    return x, idx, ns, pk, pv


def _run(w, x, pk, pv, ns, t, flags):
    d = H.dims_of(w)
    ws = torch.zeros(H.herald_workspace_size(d, 1, w.P), dtype=torch.uint8, device="cuda")
    out = torch.zeros((w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
    H.herald_denoise_attn_ex(d, dev(x["q_steps"][t]), dev(pk), dev(pv), dev(ns), w.P,
                             dev(x["block_k"][t]), dev(x["block_v"][t]), out, 0.0, flags, None,
                             None, None, ws)
    torch.cuda.synchronize()
    assert H.herald_workspace_error(ws) == 0
    return out


@pytest.mark.parametrize("cs", [8, 4, 2])
@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_flash_attention_matches_oracle(w, cs):
    x, idx, ns, pk, pv = _setup(w, seed=cs)
    for t in range(w.T):
        out = _run(w, x, pk, pv, ns, t, CS_FLAGS[cs] | (H.HERALD_ATTN_SETTLED if t else 0))
        ref = oracle.sparse_attn(f64(x["q_steps"][t]), f64(x["k_cache"]), f64(x["v_cache"]), idx,
                                 ns, f64(x["block_k"][t]), f64(x["block_v"][t]))
        err = np.abs(bf16_dev_to_f64(out) - ref).max()
        assert err <= ATTN_ATOL, f"{w.name} CS={cs} step {t}: max abs err {err}"


@pytest.mark.parametrize("cs", [16, 12, 8])
@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_pool_attention_matches_oracle(w, cs):
    """The cluster pool kernel with 16 CTAs per row tile (8 rows merged per
    CTA), with 12 (12 rows per CTA, the last CTA 8, so that 11 CTAs hold the
    128 rows) and with 8; the pool and block keys split evenly.  The 8-CTA
    form does not take the big pool (kpc + B > 256), the others do."""
    x, idx, ns, pk, pv = _setup(w, seed=20 + cs)
    for t in range(w.T):
        out = _run(w, x, pk, pv, ns, t, POOL_FLAGS[cs] | (H.HERALD_ATTN_SETTLED if t else 0))
        ref = oracle.sparse_attn(f64(x["q_steps"][t]), f64(x["k_cache"]), f64(x["v_cache"]), idx,
                                 ns, f64(x["block_k"][t]), f64(x["block_v"][t]))
        err = np.abs(bf16_dev_to_f64(out) - ref).max()
        assert err <= ATTN_ATOL, f"{w.name} pool CS={cs} step {t}: max abs err {err}"


@pytest.mark.parametrize("sms", [0, 152, 64, 24])
def test_attention_within_an_sm_budget_matches_oracle(sms):
    """HERALD_ATTN_SMS(n): the cluster sizes are picked so that a step's
    clusters fit n SMs at once (12 or 16 CTAs per row tile when they do,
    else 8 for the pool kernel; 8, 4 or 2 for the pipelined one); the
    output is the oracle's whichever is picked."""
    for w in (SHAPES[1], SHAPES[4]):
        x, idx, ns, pk, pv = _setup(w, seed=40 + sms)
        for t in range(w.T):
            flags = H.HERALD_ATTN_SMS(sms) | (H.HERALD_ATTN_SETTLED if t else 0)
            out = _run(w, x, pk, pv, ns, t, flags)
            ref = oracle.sparse_attn(f64(x["q_steps"][t]), f64(x["k_cache"]), f64(x["v_cache"]),
                                     idx, ns, f64(x["block_k"][t]), f64(x["block_v"][t]))
            err = np.abs(bf16_dev_to_f64(out) - ref).max()
            assert err <= ATTN_ATOL, f"{w.name} budget {sms} step {t}: max abs err {err}"


@pytest.mark.parametrize("w", SHAPES[:4], ids=lambda w: w.name)
def test_flash_and_pool_kernels_agree(w):
    """Both kernels compute the same softmax over the same keys; they differ
    only in the order of fp32 sums and in where P is rounded to bf16."""
    x, idx, ns, pk, pv = _setup(w, seed=7)
    a = bf16_dev_to_f64(_run(w, x, pk, pv, ns, 0, H.HERALD_ATTN_KERNEL_POOL))
    for f in (CS_FLAGS[8], CS_FLAGS[4], CS_FLAGS[2], POOL_FLAGS[8], POOL_FLAGS[12],
              POOL_FLAGS[16]):
        b = bf16_dev_to_f64(_run(w, x, pk, pv, ns, 0, f))
        assert np.abs(a - b).max() <= ATTN_ATOL, hex(f)


@pytest.mark.parametrize("kf", ["flash8", "flash2", "pool8", "pool12", "pool16"])
def test_flash_last_step_appends_like_append_kv(kf):
    """The append rides with the attention (in the pipelined kernel the
    softmax warps of the first row tile's cluster of KV head 0, in the pool
    kernel that cluster's CTAs): the cache rows and the context lengths
    bit-exactly as herald_append_kv, the same output."""
    flag = {"flash8": CS_FLAGS[8], "flash2": CS_FLAGS[2], "pool8": POOL_FLAGS[8],
            "pool12": POOL_FLAGS[12], "pool16": POOL_FLAGS[16]}[kf]
    w = _w("append", L=300, C=64, K=32, S=4, W=4, extra_rows=40, index=96)
    x, idx, ns, pk, pv = _setup(w, seed=3)
    x["ctx"] = np.array([300, 330], np.int32)
    d = H.dims_of(w)
    out_plain = _run(w, x, pk, pv, ns, 0, flag)
    k, v, ctx = dev(x["k_cache"]), dev(x["v_cache"]), dev(x["ctx"])
    ws = torch.zeros(H.herald_workspace_size(d, 1, w.P), dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(out_plain)
    H.herald_denoise_attn_ex(d, dev(x["q_steps"][0]), dev(pk), dev(pv), dev(ns), w.P,
                             dev(x["block_k"][0]), dev(x["block_v"][0]), out, 0.0,
                             flag | H.HERALD_ATTN_APPEND | H.HERALD_ATTN_ADVANCE, ctx, k,
                             v, ws)
    torch.cuda.synchronize()
    assert H.herald_workspace_error(ws) == 0
    assert torch.equal(out, out_plain)
    c2, k2, v2 = oracle.append(x["ctx"], f64(x["block_k"][0]), f64(x["block_v"][0]),
                               f64(x["k_cache"]), f64(x["v_cache"]))
    assert ctx.cpu().numpy().tolist() == c2.tolist() == [332, 340]  # L_max = 340 caps the second
    np.testing.assert_array_equal(synth.bf16_to_f64(k.cpu().numpy().view(np.uint16)), k2)
    np.testing.assert_array_equal(synth.bf16_to_f64(v.cpu().numpy().view(np.uint16)), v2)


@pytest.mark.parametrize("cs", [2, 8])
@pytest.mark.parametrize("where", ["pool", "block"])
def test_flash_rescales_when_the_row_max_jumps(cs, where):
    """A key whose score exceeds every earlier key of its CTA by more than 8
    (log2 units) moves the rows' exponent base: O and the row sums built so
    far are rescaled.  All queries are one +-1 pattern u, the keys small
    noise (scores ~N(0, 0.3^2)), and one key a multiple of u with score 7
    (2^10 times the others' weight, above the 8 that moves the base) -- in
    a later pool tile of the first CTA, or among the block keys, which the
    last CTA takes after its pool tiles.  The other keys still carry most
    of the mass, so a missing or doubled rescale shows."""
    rng = np.random.default_rng(5 + cs)
    # 2900 pool keys: with 8 CTAs, 3 tiles each and the last CTA 2 pool
    # tiles before its block tile; with 2, 12 and 11 tiles
    N, Hq, Hkv, d, B, P = 1, 4, 1, 128, 16, 2900
    w = Workload("jump", N=N, Hq=Hq, Hkv=Hkv, d=d, L=P, B=B, T=1, C=P, K=P, S=0, W=0,
                 index=97)
    u = rng.choice([-1.0, 1.0], size=d).astype(np.float32)
    q = np.broadcast_to(u, (1, N, B, Hq, d)).copy()
    kp = 0.3 * rng.standard_normal((N, Hkv, P, d)).astype(np.float32)
    vp = rng.standard_normal((N, Hkv, P, d)).astype(np.float32)
    bk = 0.3 * rng.standard_normal((1, N, B, Hkv, d)).astype(np.float32)
    bv = rng.standard_normal((1, N, B, Hkv, d)).astype(np.float32)
    alpha = 7.0 * np.sqrt(d) / d    # u . (alpha u) / sqrt(d) = 7
    if where == "pool":
        kp[0, 0, 200] = alpha * u   # the second tile of the first CTA
    else:
        bk[0, 0, 5, 0] = alpha * u
    x = dict(q_steps=synth.bf16_bits(q), k_cache=synth.bf16_bits(kp),
             v_cache=synth.bf16_bits(vp), block_k=synth.bf16_bits(bk),
             block_v=synth.bf16_bits(bv))
    ns = np.full((N, Hkv), P, np.int32)
    idx = np.arange(P, dtype=np.int32).reshape(N, Hkv, P)
    out = _run(w, x, x["k_cache"], x["v_cache"], ns, 0, CS_FLAGS[cs])
    ref, wsum = oracle.sparse_attn(f64(x["q_steps"][0]), f64(x["k_cache"]), f64(x["v_cache"]),
                                   idx, ns, f64(x["block_k"][0]), f64(x["block_v"][0]),
                                   with_wsum=True)
    err = np.abs(bf16_dev_to_f64(out) - ref).max()
    assert err <= ATTN_ATOL, f"CS={cs} jump in {where}: max abs err {err}"
