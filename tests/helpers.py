"""Shared test helpers: device upload of the synthetic bf16 inputs, the
tie-band set comparison, and oracle runs on sampled (sequence, KV head)
segments.  Holds none of the method's arithmetic."""
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
    bad = [j for j in diff if not (score[j] > 0 and thr > 0 and abs(np.log(score[j]) - np.log(thr)) <= BAND)]
    assert not bad, f"{what}: {len(bad)} positions outside the tie band, e.g. {bad[:5]} " \
                    f"(threshold {thr}, scores {[score[j] for j in bad[:5]]})"
    return len(diff)


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
