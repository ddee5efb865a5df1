"""fp64 CPU oracle of the HERALD hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the bench's CPU-baseline / reference leg
may import this package.  The product (the CUDA library and its binding)
never does, and it shares no code with it.  `herald_oracle.c` holds the
arithmetic of the steps, written step by step from the pages (HERALD v3
abstract, HERALD early abstract, SparDA method section); this module compiles
it with gcc, marshals numpy arrays through ctypes, and states the variants
built on those steps (block-granular stage 1, adaptive budget) in numpy.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "herald_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile herald_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
    return _lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def merged_query(q_merge):
    """Step 1: qbar [N,Hq,d] = mean over B of q_merge [N,B,Hq,d]."""
    q = _f64(q_merge)
    N, B, Hq, d = q.shape
    out = np.empty((N, Hq, d), np.float64)
    _load().oracle_merged_query(N, B, Hq, d, _p(q), _p(out))
    return out


def stage1_scores(qbar, k_cache, ctx):
    """Step 2: returns (l1 [N,Hq,L_max], lse1 [N,Hq], s1 [N,Hkv,L_max])."""
    qb, k, cx = _f64(qbar), _f64(k_cache), _i32(ctx)
    N, Hq, d = qb.shape
    _, Hkv, L_max, _ = k.shape
    l1 = np.empty((N, Hq, L_max)); lse1 = np.empty((N, Hq)); s1 = np.empty((N, Hkv, L_max))
    _load().oracle_stage1_scores(N, Hq, Hkv, d, L_max, _p(cx), _p(qb), _p(k),
                                 _p(l1), _p(lse1), _p(s1))
    return l1, lse1, s1


def top_m(score, m):
    """The m largest of a 1-D score vector, lower position first on ties,
    returned in ascending position order."""
    s = _f64(score)
    out = np.full(max(m, 1), -1, np.int32)
    cnt = _load().oracle_top_m(len(s), _p(s), int(m), _p(out))
    return out[:cnt].copy()


def topc(s1, ctx, C_):
    """Step 3: (cand [N,Hkv,C] ascending, -1 padded; n_cand [N,Hkv])."""
    s, cx = _f64(s1), _i32(ctx)
    N, Hkv, L_max = s.shape
    cand = np.empty((N, Hkv, C_), np.int32); nc = np.empty((N, Hkv), np.int32)
    _load().oracle_topc(N, Hkv, L_max, _p(cx), _p(s), int(C_), _p(cand), _p(nc))
    return cand, nc


def stage2_scores(q_block, k_cache, cand, n_cand):
    """Step 4: s2 [N,Hkv,C] over the candidate slots."""
    q, k, c, nc = _f64(q_block), _f64(k_cache), _i32(cand), _i32(n_cand)
    N, B, Hq, d = q.shape
    _, Hkv, L_max, _ = k.shape
    C_ = c.shape[-1]
    s2 = np.empty((N, Hkv, C_))
    _load().oracle_stage2_scores(N, B, Hq, Hkv, d, L_max, _p(q), _p(k), _p(c),
                                 _p(nc), C_, _p(s2))
    return s2


def select_final(ctx, L_max, cand, n_cand, s2, K, S, W, P=None):
    """Step 5: (idx [N,Hkv,P] ascending, -1 padded; n_sel [N,Hkv])."""
    cx, c, nc, s = _i32(ctx), _i32(cand), _i32(n_cand), _f64(s2)
    N, Hkv, C_ = c.shape
    P = K + S + W if P is None else P
    idx = np.empty((N, Hkv, P), np.int32); ns = np.empty((N, Hkv), np.int32)
    _load().oracle_select_final(N, Hkv, int(L_max), _p(cx), _p(c), _p(nc), _p(s),
                                C_, int(K), int(S), int(W), int(P), _p(idx), _p(ns))
    return idx, ns


def adaptive_budget(s2, n_cand, tau, K_min, K_max):
    """Per-block budget from the first denoising step (MAGE author page,
    abstract: the first step predicts how much budget the block needs; the
    mechanism is not given).  Reading: the budget of (n, g) is the smallest k
    whose k largest stage-2 scores hold a fraction tau of the scores' total
    (the stage-2 scores of the first step's queries are their attention mass
    per candidate), then clamped to [K_min, K_max].  Returns K_b [N, Hkv]."""
    s, nc = _f64(s2), _i32(n_cand)
    N, Hkv, _ = s.shape
    kb = np.zeros((N, Hkv), np.int32)
    for n in range(N):
        for g in range(Hkv):
            m = int(nc[n, g])
            x = np.sort(np.maximum(s[n, g, :m], 0.0))[::-1]
            cum = np.cumsum(x)
            hit = np.nonzero(cum >= tau * (cum[-1] if m else 0.0))[0]
            k = int(hit[0]) + 1 if len(hit) else m
            kb[n, g] = max(K_min, min(K_max, min(k, m)))
    return kb


def select_final_per_head(ctx, L_max, cand, n_cand, s2, K_b, S, W, P):
    """Step 5 with a budget of its own per (n, g): K_b [N, Hkv]."""
    c = _i32(cand)
    N, Hkv, _ = c.shape
    idx = np.empty((N, Hkv, P), np.int32); ns = np.empty((N, Hkv), np.int32)
    cx, nc, s = _i32(ctx), _i32(n_cand), _f64(s2)
    for n in range(N):
        for g in range(Hkv):
            i, m = select_final(cx[n:n + 1], L_max, c[n:n + 1, g:g + 1], nc[n:n + 1, g:g + 1],
                                s[n:n + 1, g:g + 1], int(K_b[n, g]), S, W, P)
            idx[n, g], ns[n, g] = i[0, 0], m[0, 0]
    return idx, ns


def select(q_merge, q_block, k_cache, ctx, C_, K, S, W, P=None):
    """Steps 1-5 in order; returns a dict with every intermediate."""
    qbar = merged_query(q_merge)
    l1, lse1, s1 = stage1_scores(qbar, k_cache, ctx)
    cand, n_cand = topc(s1, ctx, C_)
    s2 = stage2_scores(q_block, k_cache, cand, n_cand)
    idx, n_sel = select_final(ctx, np.shape(k_cache)[2], cand, n_cand, s2, K, S, W, P)
    return dict(qbar=qbar, l1=l1, lse1=lse1, s1=s1, cand=cand, n_cand=n_cand,
                s2=s2, idx=idx, n_sel=n_sel)


def exact_scores(q_block, k_cache, ctx):
    """Exact selection score (MAGE author page, abstract: exact attention of
    the block's queries predicts the important entries; HERALD v3 abstract:
    the merged query approximates it): every cached position j < ctx is a
    candidate of step 4, so s[j] = sum over the B*G rows of the softmax over
    the whole context.  Returns (cand = arange padded with -1, n_cand, s)."""
    k = np.asarray(k_cache)
    N, Hkv, L_max, _ = k.shape
    cx = np.asarray(ctx, np.int64)
    cand = np.full((N, Hkv, L_max), -1, np.int32)
    n_cand = np.empty((N, Hkv), np.int32)
    for n in range(N):
        L = int(min(max(cx[n], 0), L_max))
        cand[n, :, :L] = np.arange(L, dtype=np.int32)
        n_cand[n, :] = L
    return cand, n_cand, stage2_scores(q_block, k_cache, cand, n_cand)


def select_exact(q_block, k_cache, ctx, K, S, W, P=None):
    """The exact selection: step 5 (top-K, then the sink/local union) over
    the exact scores."""
    cand, n_cand, s = exact_scores(q_block, k_cache, ctx)
    idx, n_sel = select_final(ctx, np.shape(k_cache)[2], cand, n_cand, s, K, S, W, P)
    return dict(cand=cand, n_cand=n_cand, s=s, idx=idx, n_sel=n_sel)


def pooled_keys(k_cache, ctx, Bk):
    """Block-granular stage 1, the compressed keys (SparDA summary, Method
    section: InfLLM-V2 selects whole blocks of the context next to the
    initial tokens and the local window): key block b of (n, g) is the mean
    of cache rows [b*Bk, min((b+1)*Bk, ctx)) -- the last block below ctx may
    be partial -- and blocks at or past ctx are zero.  Returns
    (kp [N, Hkv, ceil(L_max/Bk), d], ctx_b [N] = ceil(ctx/Bk))."""
    k = _f64(k_cache)
    N, Hkv, L_max, d = k.shape
    nb_max = -(-L_max // Bk)
    kp = np.zeros((N, Hkv, nb_max, d))
    ctx_b = np.zeros(N, np.int32)
    for n in range(N):
        L = int(min(max(int(ctx[n]), 0), L_max))
        ctx_b[n] = -(-L // Bk)
        for b in range(ctx_b[n]):
            kp[n, :, b] = k[n, :, b * Bk: min((b + 1) * Bk, L)].mean(axis=1)
    return kp, ctx_b


def expand_blocks(cand_b, n_cand_b, ctx, Bk):
    """Candidate positions of the selected blocks: every position below ctx
    of each block in cand_b, ascending (blocks ascending), in rows of
    C_blocks*Bk slots padded with -1.  Returns (cand, n_cand)."""
    cb = np.asarray(cand_b)
    N, Hkv, Cb = cb.shape
    cand = np.full((N, Hkv, Cb * Bk), -1, np.int32)
    n_cand = np.zeros((N, Hkv), np.int32)
    for n in range(N):
        L = int(ctx[n])
        for g in range(Hkv):
            pos = [j for b in cb[n, g, : int(n_cand_b[n, g])]
                   for j in range(int(b) * Bk, min((int(b) + 1) * Bk, L))]
            cand[n, g, : len(pos)] = pos
            n_cand[n, g] = len(pos)
    return cand, n_cand


def stage1_blocks(qbar, k_cache, ctx, Bk, C_blocks):
    """Block-granular stage 1: the stage-1 rule (steps 2-3) with the pooled
    block keys in place of the keys -- s1b[b] = sum over the group's heads of
    softmax over the blocks of qbar_h . kp_b / sqrt(d) -- then the top
    C_blocks blocks expanded to their positions.  Returns a dict with the
    pooled keys, block scores, selected blocks and the candidates."""
    kp, ctx_b = pooled_keys(k_cache, ctx, Bk)
    l1b, lse1b, s1b = stage1_scores(qbar, kp, ctx_b)
    cand_b, n_cand_b = topc(s1b, ctx_b, C_blocks)
    cand, n_cand = expand_blocks(cand_b, n_cand_b, np.asarray(ctx), Bk)
    return dict(kp=kp, ctx_b=ctx_b, l1b=l1b, s1b=s1b, cand_b=cand_b, n_cand_b=n_cand_b,
                cand=cand, n_cand=n_cand)


def sparse_attn(q, k_cache, v_cache, idx, n_sel, block_k, block_v, scale=None,
                with_wsum=False):
    """Step 6: out [N,B,Hq,d] over the selected rows plus the B block keys."""
    qq, k, v, ix, ns = _f64(q), _f64(k_cache), _f64(v_cache), _i32(idx), _i32(n_sel)
    bk, bv = _f64(block_k), _f64(block_v)
    N, B, Hq, d = qq.shape
    _, Hkv, L_max, _ = k.shape
    P = ix.shape[-1]
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.empty((N, B, Hq, d)); ws = np.empty((N, B, Hq))
    _load().oracle_sparse_attn(N, B, Hq, Hkv, d, L_max, _p(qq), _p(k), _p(v),
                               _p(ix), _p(ns), P, _p(bk), _p(bv),
                               C.c_double(scale), _p(out), _p(ws))
    return (out, ws) if with_wsum else out


def dense_attn(q, k_cache, v_cache, ctx, block_k, block_v, scale=None):
    """Step 7: attention over every cached position plus the block keys."""
    qq, k, v, cx = _f64(q), _f64(k_cache), _f64(v_cache), _i32(ctx)
    bk, bv = _f64(block_k), _f64(block_v)
    N, B, Hq, d = qq.shape
    _, Hkv, L_max, _ = k.shape
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    out = np.empty((N, B, Hq, d))
    _load().oracle_dense_attn(N, B, Hq, Hkv, d, L_max, _p(cx), _p(qq), _p(k), _p(v),
                              _p(bk), _p(bv), C.c_double(scale), _p(out))
    return out


def append(ctx, block_k, block_v, k_cache, v_cache):
    """Step 8: returns (new_ctx, k_cache, v_cache) with the block appended."""
    cx = _i32(ctx).copy()
    bk, bv = _f64(block_k), _f64(block_v)
    k, v = _f64(k_cache).copy(), _f64(v_cache).copy()
    N, Hkv, L_max, d = k.shape
    B = bk.shape[1]
    _load().oracle_append(N, B, Hkv, d, L_max, _p(cx), _p(bk), _p(bv), _p(k), _p(v))
    return cx, k, v
