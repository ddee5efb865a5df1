"""Host-side scheduling logic that needs no GPU: the flags of a block's
denoising steps, the SM budgets of the background scan and of the
attention beside it, how the bench groups
timed blocks into CUDA graphs, and the pipeline's option checks."""
import pytest

import bench
from block_diffusion_sparse_gb300 import herald as H
from block_diffusion_sparse_gb300 import pipeline as P
from block_diffusion_sparse_gb300.workloads import LLAMA_64K, QWEN_32K, TINY


def test_step_flags_settle_after_the_first_step_and_append_at_the_last():
    T = 8
    flags = [P.step_flags(t, T, advance=True) for t in range(T)]
    assert flags[0] == 0
    assert all(f & H.HERALD_ATTN_SETTLED for f in flags[1:])
    assert all(not f & H.HERALD_ATTN_APPEND for f in flags[:-1])
    assert flags[-1] == H.HERALD_ATTN_SETTLED | H.HERALD_ATTN_APPEND | H.HERALD_ATTN_ADVANCE
    # one step per block: it appends, and the pool is not settled for it
    assert P.step_flags(0, 1, advance=False) == H.HERALD_ATTN_APPEND


@pytest.fixture
def sms_152(monkeypatch):
    monkeypatch.setattr(P, "_sm_count", lambda device: 152)
    monkeypatch.setattr("torch.cuda.current_device", lambda: 0)


def test_background_scan_budget(sms_152):
    # about one SM per MiB of keys, at least 32; all SMs once that is half the GPU
    assert P.background_sms(H.dims_of(QWEN_32K)) == 33      # 33.6 MB of keys
    assert P.background_sms(H.dims_of(TINY)) == 32          # tiny cache: the floor
    assert P.background_sms(H.dims_of(LLAMA_64K)) == 0      # 537 MB: every SM
    assert P.background_sms(H.dims_of(QWEN_32K), host=True) == P.HOST_SCAN_SMS
    assert P.scan_sms(H.dims_of(QWEN_32K), None, fixed=7) == 7


def test_attention_sm_budget_leaves_the_background_its_sms(sms_152):
    # the selection stream holds `bg` SMs: the attention may count on the
    # rest, in units of 4 SMs in bits 16-23; none or every SM: no budget
    assert P.attn_sm_flags(33) == H.HERALD_ATTN_SMS(119) == (29 << 16)
    assert P.attn_sm_flags(64) == (22 << 16)
    assert P.attn_sm_flags(0) == 0 and P.attn_sm_flags(152) == 0
    assert (P.attn_sm_flags(64) & 0xFFFF) == 0  # touches no other flag


class _Stack(bench.StackBench):
    def __init__(self):  # no device state: only the type matters here
        pass


class _Layer(bench.Bench):
    def __init__(self):
        pass


@pytest.mark.parametrize("steps,g", [(50, 5), (20, 5), (10, 5), (8, 8), (7, 7), (30, 6),
                                     (2, 2), (1, 1), (11, 1)])
def test_blocks_per_graph_divides_the_timed_steps(steps, g):
    assert bench.blocks_per_graph(_Layer(), steps) == g
    assert steps % g == 0 and g <= 8
    assert bench.blocks_per_graph(_Stack(), steps) == 1


@pytest.mark.parametrize("kw", [dict(prefetch="v"), dict(prefetch="kvv"), dict(blocks=48)])
def test_pipeline_rejects_bad_options_before_allocating(kw):
    """An unknown prefetch mode, or a candidate count C that is not a whole
    number of blocks, is refused before any device memory is touched."""
    d = H.dims_of(TINY)
    with pytest.raises(ValueError):
        P.BlockPipeline(d, TINY.C, TINY.K, TINY.S, TINY.W, TINY.P, TINY.T, **kw)
