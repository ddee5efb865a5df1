"""Benchmark of the HERALD hot path on one GB300 (or N independent replicas).

One step = one block of one layer of the 32K Qwen2.5-7B-like workload
(N=1, Hq=28, Hkv=4, d=128, ctx 32768, B=32, T=8, C=4096, K=1024, sink 64,
local 256) through the dual-stream block pipeline: stage 2 (refine + top-K
with sink/local) -> gather into one of two pool buffers -> T x sparse
block attention, the last step appending the block, on the denoising
stream, while stage 1 (merged-query scan + top-C) for the next block runs
on the selection stream.  Metric: block tokens/s = N*B / (time per step).
The same step without the overlap is reported as `serial`.

Timing: consecutive steps are captured into CUDA graphs (up to 8 blocks
per graph, the count dividing the number of timed steps; one per graph for
the layer stack) and the graphs are replayed; the K cache and V cache are
rotated over enough copies that the data touched between two uses of a
copy exceeds L2 (cold-L2 inputs).  A second, traced replay brackets every
kernel with graph event nodes to time the dominant kernel for the
roofline.  The timed region of --steps steps is repeated until the repeats
add up to --min-timed-ms (the median per step is reported).  e2e: the same
step through the pipeline's public call (one graph per block) with the
step's inputs copied from pinned host buffers and its outputs read back,
copies inside the timed region; e2e.direct_calls: the same with the
library's C-ABI calls issued directly every step (one herald_block call per
block for the per-key selection; their host cost inside the timed region).  `range`: the metric's other workloads (4 x 64K, 128K
with the cache in host memory, the 28-layer stack), each timed the same way
with its scan and attention rooflines.
`--impl reference`: the fp64 CPU oracle timed on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import hashlib
import json
import os
import re
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block tokens/s (select + T sparse-attn steps) at 32K–128K; scan HBM GB/s"
L2_BYTES = 129 * 2 ** 20


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock, power and clock-event reasons of one GPU through
    NVML (ctypes, the driver's library) every `period` seconds."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, torch_dev: int, period: float = 0.002):
        self.period = period
        self.samples: list[tuple[float, int, int, float]] = []
        self.ok = False
        self.max_mhz = None
        self._stop = threading.Event()
        try:
            import torch
            p = torch.cuda.get_device_properties(torch_dev)
            bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def _one(self):
        clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
        self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        self.samples.append((time.perf_counter(), int(clk.value), int(rs.value), pw.value / 1000.0))

    def _run(self):
        while not self._stop.is_set():
            self._one()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self.t.join()

    def summary(self, t0: float, t1: float) -> dict:
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": "unavailable"}
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        if not win:  # region shorter than the period: nearest samples around it
            win = sorted(self.samples, key=lambda s: abs(s[0] - 0.5 * (t0 + t1)))[:3]
        reasons = set()
        for s in win:
            for bit, name in self.REASONS.items():
                if s[2] & bit:
                    reasons.add(name)
        return {"sm_mhz": float(np.median([s[1] for s in win])), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(win),
                "power_w_max": max(s[3] for s in win), "source": "nvml"}


# --------------------------------------------------------------------------- ranks
def max_over_ranks(ms: float, dist, device=None) -> float:
    """The step time the job reports: the slowest rank's."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_per_step: float, world: int, tokens_per_step: int) -> float:
    """Whole-job throughput: every rank runs its own replica of the
    workload (weak scaling), so the job processes world x tokens per step."""
    return world * tokens_per_step / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------- workload
WORKLOADS = {"qwen": "QWEN_32K", "tiny": "TINY", "llama": "LLAMA_64K",
             "long-host": "LONG_128K_HOST", "stack": "QWEN_STACK"}
_WORKLOAD = "qwen"
_SELECTION = "merged"
_BUDGET = None  # --budget TAU: the adaptive per-block budget (K_min = K/8)
_PREFETCH = "kv"  # --prefetch: the candidate rows prefetched for a host-resident cache
BLOCK_KEYS = 64  # keys per block of the block-granular stage 1 (--selection blocks)


def workload():
    """The benchmarked layer: the 32K Qwen2.5-7B-like layer unless --workload
    names another (tiny, llama = 4 x 64K Llama-8B-like, long-host = 128K
    context with the cache in pinned host memory, stack = the 28-layer
    Qwen2.5-7B-like stack at 8 x 32K)."""
    from block_diffusion_sparse_gb300 import workloads as W
    return getattr(W, WORKLOADS[_WORKLOAD])


def _code_only(path: str) -> str:
    """A source file without its comments and blank lines."""
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.split("\n"))
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash(kernel: str = None) -> str:
    """Hash of the kernel sources without their comments and blank lines: a
    committed ncu summary stays valid across edits that change no code.  With
    `kernel`, only the .cu file that defines it and the device headers (.cuh)
    are hashed, so that a summary of one kernel survives edits to another."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_diffusion_sparse_gb300", "csrc")
    files = sorted(os.listdir(csrc))
    if kernel is not None:
        pat = re.compile(r"__global__[^;{]*?\b" + re.escape(kernel) + r"\s*\(", re.S)
        defining = [f for f in files if f.endswith(".cu") and
                    pat.search(open(os.path.join(csrc, f)).read())]
        files = defining + [f for f in files if f.endswith(".cuh")]
    for f in files:
        h.update(_code_only(os.path.join(csrc, f)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if the summary was taken on the current source of that kernel;
    else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    e = d.get("workloads", {}).get(workload, {}).get("kernels", {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch_full_workload")


class Bench:
    def __init__(self, w, rank: int):
        import torch
        from block_diffusion_sparse_gb300 import herald as H
        from block_diffusion_sparse_gb300 import synth
        self.torch, self.H, self.w = torch, H, w
        self.x = synth.make_layer(w)
        x = self.x
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
        self.d = H.dims_of(w)
        self.P = w.P
        cache_bytes = 2 * x["k_cache"].nbytes
        if w.kv_on_host:
            # the cache stays in pinned host memory; kernels read it over the link
            host = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
            self.n_rot = 2
            k0, v0 = host(x["k_cache"]), host(x["v_cache"])
            self.k, self.v = [k0, k0], [v0, v0]
        else:
            self.n_rot = max(2, int(np.ceil(2 * L2_BYTES / cache_bytes)) + 1)
            self.n_rot += self.n_rot % 2      # even: block parity = cache-copy parity
            k0, v0 = dev(x["k_cache"]), dev(x["v_cache"])
            self.k = [k0] + [k0.clone() for _ in range(self.n_rot - 1)]
            self.v = [v0] + [v0.clone() for _ in range(self.n_rot - 1)]
        self.q_merge = dev(x["q_merge"])
        self.q_steps = dev(x["q_steps"])
        self.bk, self.bv = dev(x["block_k"]), dev(x["block_v"])
        self.ctx = torch.from_numpy(x["ctx"]).cuda()
        from block_diffusion_sparse_gb300.pipeline import BlockPipeline
        self.exact = _SELECTION == "exact"
        self.pipe = BlockPipeline(self.d, w.C, w.K, w.S, w.W, self.P, w.T, exact=self.exact,
                                  blocks=BLOCK_KEYS if _SELECTION == "blocks" else 0,
                                  # a host-resident cache with the block stage 1: the
                                  # next block's candidate rows cross the link beside
                                  # the denoising steps (with the per-key stage 1 the
                                  # link is the scan's: 1,544 against 1,494 us)
                                  prefetch=(_PREFETCH if w.kv_on_host and _SELECTION == "blocks"
                                            else False),
                                  budget=None if _BUDGET is None else (w.K // 8, _BUDGET))
        self.out = torch.zeros((w.T, w.N, w.B, w.Hq, w.d), dtype=torch.int16, device="cuda")
        self.overlap = True
        # stage 1 of the first block (its own queries; no predecessor)
        self.pipe.prime(self.q_merge, self.k[0], self.ctx, slot=0, v_cache=self.v[0])
        torch.cuda.synchronize()

    @property
    def idx(self):
        return self.pipe.idx

    @property
    def n_sel(self):
        return self.pipe.n_sel

    @property
    def ws(self):
        return self.pipe.ws_den

    n_sel_out = property(lambda self: self.pipe.n_sel)
    trace_capacity = 64

    def before_step(self, i: int):
        """Called before step i of every timed or warm-up loop (the single
        layer keeps its context length fixed: nothing to do)."""

    def context_note(self) -> str:
        return "fixed: each step appends the block at the same position (ctx not advanced)"

    def budget_note(self):
        p = getattr(self, "pipe", None)
        if getattr(p, "budget", None) is None:
            return "fixed K"
        ks = p.k_sel.cpu().numpy()
        return {"tau": p.budget[1], "K_min": p.budget[0], "K_max": p.K,
                "last_block_mean_K": float(ks.mean()), "last_block_K_range": [int(ks.min()),
                                                                             int(ks.max())]}

    def prefetch_note(self) -> str:
        p = getattr(self, "pipe", None)
        if not getattr(p, "prefetch", False):
            return "none"
        return ("next block's candidate K and V rows (top-K pool rows gathered from HBM)"
                if p.prefetch_v else "next block's candidate K rows")

    def l2_note(self) -> str:
        if self.w.kv_on_host:
            return "K/V cache in pinned host memory (read over the host link)"
        return (f"cold: K/V cache rotated over {self.n_rot} copies "
                f"({self.n_rot * 2 * self.x['k_cache'].nbytes / 2**20:.0f} MiB > L2)")

    def step(self, r: int, q_merge=None, q_steps=None, bk=None, bv=None, out=None,
             graph: bool = False):
        """One block through the dual-stream pipeline (cache copy r; stage 1
        of the next block scans copy r+1); graph=True lets the pipeline
        replay its cached CUDA graph of the block."""
        qs = self.q_steps if q_steps is None else q_steps
        bk = self.bk if bk is None else bk
        bv = self.bv if bv is None else bv
        nxt = (r + 1) % self.n_rot
        if self.exact:
            self.pipe.block_exact(r, qs, bk, bv, self.k[r], self.v[r], self.ctx,
                                  self.out if out is None else out, advance=False)
            return
        self.pipe.block(r, qs, bk, bv, self.k[r], self.v[r], self.ctx,
                        self.out if out is None else out, next_k_cache=self.k[nxt],
                        next_v_cache=self.v[nxt], advance=False, overlap=self.overlap,
                        graph=graph)

    def attn_operands(self):
        """(pool_k, pool_v, n_sel, q_steps, block_k, block_v, out, ws) of one
        layer's denoising steps: the pool of the last block of parity 0."""
        p = self.pipe
        return (p.pool_k[0], p.pool_v[0], p.n_sel, self.q_steps, self.bk, self.bv, self.out,
                p.ws_den)

    def capture_chunk(self, start: int, g: int):
        """One CUDA graph of g consecutive blocks (cache copies start, start+1,
        ... modulo the rotation), captured after capture()'s eager warm-up."""
        torch = self.torch
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for t in range(g):
                self.step((start + t) % self.n_rot)
        return graph

    def capture(self, traced: bool = False):
        torch = self.torch
        graphs, traces = [], []
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for r in range(self.n_rot):     # eager warm-up: kernel attributes, caches
                self.step(r)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for r in range(self.n_rot):
            g = torch.cuda.CUDAGraph()
            if traced:
                tr = self.H.Trace(capacity=self.trace_capacity, external=True)
                with torch.cuda.graph(g):
                    with tr:
                        self.step(r)
                traces.append(tr)
            else:
                with torch.cuda.graph(g):
                    self.step(r)
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs, traces


class StackBench(Bench):
    """The 28-layer stack (attention and selection only): one step is one
    block through every layer with the stack pipeline (stage 2 + gather +
    step-0 attention layer by layer, stage 1 of the next block per layer on
    the selection stream, steps 1..T-1 over all layers, appends).

    One synthetic layer is generated on the host; layer l's K/V cache,
    queries and block K/V are that layer with its sequences rotated by l
    positions, each layer in its own device buffers.  A step streams every
    layer's cache, far more than L2, so the inputs are cold at each use
    without rotating copies."""

    def __init__(self, w, rank: int):
        import torch
        from block_diffusion_sparse_gb300 import herald as H
        from block_diffusion_sparse_gb300 import synth
        from block_diffusion_sparse_gb300.pipeline import StackPipeline
        self.torch, self.H, self.w = torch, H, w
        self.x = synth.make_layer(w)
        x = self.x
        nl = w.layers
        host = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16))

        def per_layer(a, axis):
            t = host(a).cuda()
            out = torch.empty((nl, *t.shape), dtype=torch.int16, device="cuda")
            for l in range(nl):
                out[l].copy_(torch.roll(t, l, dims=axis))
            return out

        self.d = H.dims_of(w)
        self.P = w.P
        self.k = per_layer(x["k_cache"], 0)                 # [nl, N, Hkv, L_max, d]
        self.v = per_layer(x["v_cache"], 0)
        self.q_merge = per_layer(x["q_merge"], 0)           # [nl, N, B, Hq, d]
        self.q_steps = per_layer(x["q_steps"], 1)           # [nl, T, N, B, Hq, d]
        self.bk = per_layer(x["block_k"], 1)                # [nl, T, N, B, Hkv, d]
        self.bv = per_layer(x["block_v"], 1)
        self.ctx = torch.from_numpy(x["ctx"]).cuda()
        self.n_rot = 2                                      # candidate-buffer parity
        self.pipe = StackPipeline(self.d, nl, w.C, w.K, w.S, w.W, self.P, w.T)
        self.out = torch.zeros((nl, w.T, w.N, w.B, w.Hq, w.d), dtype=torch.int16,
                               device="cuda")
        self.overlap = True
        self.trace_capacity = 24 * nl
        # blocks run in groups of 4 consecutive blocks, each appending B
        # tokens (L_max leaves room for 4 blocks); the context length is
        # reset before each group
        self.group = max(1, (w.L_max - w.L) // w.B)
        self.ctx0 = self.ctx.clone()
        self.pipe.prime(self.q_merge, self.k, self.ctx, slot=0)
        torch.cuda.synchronize()

    def before_step(self, i: int):
        if i % self.group == 0:
            self.ctx.copy_(self.ctx0, non_blocking=True)

    def context_note(self) -> str:
        return (f"grows: groups of {self.group} consecutive blocks, each appending B tokens to "
                f"every layer; ctx reset between groups (inside the timed region)")

    def attn_operands(self):
        p = self.pipe
        return (p.pool_k[0][0], p.pool_v[0][0], p.n_sel[0], self.q_steps[0], self.bk[0],
                self.bv[0], self.out[0], p.ws_den)

    idx = property(lambda self: self.pipe.idx_all)
    n_sel = property(lambda self: self.pipe.n_sel[-1])   # last layer's, for the roofline
    n_sel_out = property(lambda self: self.pipe.n_sel_all)

    def l2_note(self) -> str:
        return (f"cold: every step streams all {self.w.layers} layers' K caches "
                f"({self.w.layers * self.x['k_cache'].nbytes / 2**30:.1f} GiB > L2)")

    def step(self, r: int, q_merge=None, q_steps=None, bk=None, bv=None, out=None,
             graph: bool = False):
        qs = self.q_steps if q_steps is None else q_steps
        bk = self.bk if bk is None else bk
        bv = self.bv if bv is None else bv
        self.pipe.block(r, qs, bk, bv, self.k, self.v, self.ctx,
                        self.out if out is None else out, advance=True, overlap=self.overlap)


def algorithmic_work(w, n_sel: np.ndarray) -> dict:
    """Algorithmic bytes / FLOPs per launch of each kernel: the scan reads
    every cached K row once; attention reads the pool K/V rows, the block
    K/V, q and writes out once per step; the gather reads and writes each
    selected K/V row once; each refine pass is one B*G x C x d contraction
    per (sequence, KV head)."""
    NG = w.N * w.Hkv
    R = w.R
    ns = n_sel.astype(np.int64)
    keys = ns + w.B
    attn = {"bound": "hbm",
            "bytes": int(ns.sum()) * w.d * 2 * 2 + NG * w.B * w.d * 2 * 2
            + 2 * w.N * w.B * w.Hq * w.d * 2,
            "flops": int((4 * R * keys * w.d).sum())}
    return {
        "scan_tc_kernel": {"bound": "hbm", "bytes": NG * w.L * w.d * 2},
        "scan_cc_kernel": {"bound": "link" if w.kv_on_host else "hbm",
                           "bytes": NG * w.L * w.d * 2},
        "attn_kernel": attn,
        "attn_cluster_kernel": attn,
        "attn_pool_kernel": attn,
        "attn_flash_kernel": attn,
        "gather_kernel": {"bound": "link" if w.kv_on_host else "hbm",
                          "bytes": int(ns.sum()) * w.d * 2 * 2 * 2},
        "refine_pass1_kernel": {"bound": "tensor", "flops": 2 * R * w.C * w.d * NG},
        "refine_pass2_kernel": {"bound": "tensor", "flops": 2 * R * w.C * w.d * NG},
    }


def link_peak_gbs() -> float:
    """Host-link read bandwidth measured in-process: a plain copy of 256 MiB
    from pinned host memory to the device (copy engines), best of 5."""
    import torch
    n = 256 << 20
    h = torch.empty(n, dtype=torch.uint8).pin_memory()
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 0.0
    for i in range(7):
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del h, d
    return best


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# --------------------------------------------------------------------------- oracle
def oracle_block(w, xf, T_sample=None):
    """One block through the fp64 oracle: select, then T attention steps."""
    import oracle
    T = w.T if T_sample is None else T_sample
    if _SELECTION == "blocks":  # block-granular stage 1, then steps 4-5
        qbar = oracle.merged_query(xf["q_merge"])
        b = oracle.stage1_blocks(qbar, xf["k_cache"], xf["ctx"], BLOCK_KEYS, w.C // BLOCK_KEYS)
        s2 = oracle.stage2_scores(xf["q_steps"][0], xf["k_cache"], b["cand"], b["n_cand"])
        idx, n_sel = oracle.select_final(xf["ctx"], np.shape(xf["k_cache"])[2], b["cand"],
                                         b["n_cand"], s2, w.K, w.S, w.W, w.P)
        r = dict(idx=idx, n_sel=n_sel)
    else:
        r = oracle.select(xf["q_merge"], xf["q_steps"][0], xf["k_cache"], xf["ctx"], w.C, w.K,
                          w.S, w.W, w.P)
    for t in range(T):
        oracle.sparse_attn(xf["q_steps"][t], xf["k_cache"], xf["v_cache"], r["idx"], r["n_sel"],
                           xf["block_k"][t], xf["block_v"][t])
    return r


def oracle_inputs(w):
    from block_diffusion_sparse_gb300 import synth
    x = synth.make_layer(w)
    f = synth.bf16_to_f64
    return {k: (f(v) if isinstance(v, np.ndarray) and v.dtype == np.uint16 else v)
            for k, v in x.items()}


def cpu_baseline(w, budget_s: float = 12.0) -> dict:
    import oracle
    xf = oracle_inputs(w)
    oracle.num_threads()
    t0 = time.perf_counter()
    oracle_block(w, xf)                       # first block (also loads the library)
    t_first = time.perf_counter() - t0
    n = max(1, min(10, int(budget_s / max(t_first, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(n):
        oracle_block(w, xf)
    dt = (time.perf_counter() - t0) / n * w.layers
    what = (f"{n} blocks of one layer (select + gather + T={w.T} attention steps), "
            f"x{w.layers} layers" if w.layers > 1 else
            f"{n} full blocks of the same workload (select + gather + T={w.T} "
            f"attention steps)")
    return {"value": w.N * w.B / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": what + ", fp64 C + OpenMP, inputs resident in host RAM",
            "s_per_block": dt}


# --------------------------------------------------------------------------- arms
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    w = workload()
    xf = oracle_inputs(w)
    for _ in range(args.warmup):
        oracle_block(w, xf)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_block(w, xf)
    dt = (time.perf_counter() - t0) / args.steps * w.layers   # one layer timed per step
    v = w.N * w.B / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                       "ctx": w.L, "B": w.B, "T": w.T, "C": w.C, "K": w.K, "sink": w.S,
                       "local": w.W},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": "each step = one full block (select + gather + T "
                                       "attention steps) of one layer of the workload"
                                       + (f", x{w.layers} layers" if w.layers > 1 else "")},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def blocks_per_graph(b, steps: int) -> int:
    """Consecutive blocks held by one timed CUDA graph: for a single layer the
    largest divisor of the step count up to 8: inside a graph one block's
    last kernel hands over to the next block's first like the kernels inside
    a block do, where a graph launch per block cost 7.5 us more per block on
    the 32K layer (86.9 against 90.6 us with two blocks per graph); 1 for the
    stack, whose step is 28 layers long and resets the context between
    groups of blocks from the host."""
    if isinstance(b, StackBench):
        return 1
    return max(g for g in range(1, 9) if steps % g == 0)


def time_blocks(b, args, st, dist, graphs, min_ms: float = 0.0):
    """Warm-up blocks, then exactly args.steps blocks between two CUDA
    events on `st` (a barrier and a device synchronise on both sides),
    repeated until the timed regions add up to `min_ms` (at least once); block
    i uses cache copy i % n_rot.  Per-block graphs (`graphs`) or chunk graphs
    of blocks_per_graph consecutive blocks (the warm-up then rounded up to
    whole chunks).  Returns (median ms per block over the repeats, g, the host
    clock at the start of the first and the end of the last timed region,
    the repeat count)."""
    torch = b.torch
    g = blocks_per_graph(b, args.steps)
    nw = -(-args.warmup // g) * g
    chunks = {}
    run = []
    for i in range(0, nw + args.steps, g):
        if g == 1:
            run.append((i, graphs[i % b.n_rot]))
            continue
        start = i % b.n_rot
        if start not in chunks:
            chunks[start] = b.capture_chunk(start, g)
        run.append((i, chunks[start]))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i, graph in run[: nw // g]:      # warm-up
        if g == 1:
            b.before_step(i)
        graph.replay()
    per_rep, t_first, total = [], None, 0.0
    while not per_rep or total < min_ms:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        if t_first is None:
            t_first = time.perf_counter()
        e0.record(st)
        for i, graph in run[nw // g:]:
            if g == 1:
                b.before_step(i - nw)  # every repeat starts a group of blocks afresh
            graph.replay()
        e1.record(st)
        torch.cuda.synchronize()
        rep_ms = e0.elapsed_time(e1)
        total += rep_ms
        per_rep.append(rep_ms / args.steps)
    t1 = time.perf_counter()
    return float(np.median(per_rep)), g, t_first, t1, len(per_rep)


def attn_chain_ms(b, rounds: int = 8, reps: int = 5) -> float:
    """Mean duration of one pool-attention launch when a block's T steps run
    back to back, as in the pipeline (steps after the first load the settled
    pool early): CUDA events around `reps` replays of one graph holding
    `rounds` x T launches over one layer's current pool (no append), divided
    by the launches.  The isolated, event-bracketed launches of the traced
    replay also pay the launch latency that programmatic launch hides here."""
    torch, H, w = b.torch, b.H, b.w
    pk, pv, n_sel, qs, bk, bv, out, ws = b.attn_operands()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())

    def steps():
        for _ in range(rounds):
            for t in range(w.T):
                H.herald_denoise_attn_ex(b.d, qs[t], pk, pv, n_sel, b.P, bk[t], bv[t], out[t],
                                         0.0, H.HERALD_ATTN_SETTLED if t > 0 else 0, None,
                                         None, None, ws, None, st)
    with torch.cuda.stream(st):
        steps()  # eager: kernel attributes, tensor-map cache
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            steps()
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(reps):
            g.replay()
        e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * rounds * w.T)


def measure(w, args, dist, world, min_ms: float, serial: bool = True, e2e: bool = False):
    """One workload, timed as the headline is: the dual-stream block step
    (graph replay, repeated timed regions, median), the same step without the
    overlap (serial), a traced replay of the serial step for per-kernel
    durations, the pool attention's chain duration, the roofline of the
    dominant kernel and of the stage-1 scan; with e2e, the end-to-end legs.
    Returns (the line's fields for this workload, the bench object)."""
    import torch
    dev_idx = torch.cuda.current_device()
    b = StackBench(w, 0) if w.layers > 1 else Bench(w, 0)
    graphs, _ = b.capture(traced=False)
    nrot = b.n_rot
    st = torch.cuda.current_stream()
    clocks = ClockSampler(dev_idx)
    clocks.start()
    ms, chunk, t0, t1, reps_timed = time_blocks(b, args, st, dist, graphs, min_ms)
    if dist:
        dist.barrier()
    clocks.stop()
    ms = max_over_ranks(ms, dist, "cuda")
    err = b.H.herald_workspace_error(b.ws)
    del graphs

    serial_ms = None
    if serial:  # the same step without the selection/denoise overlap
        b.overlap = False
        sgraphs, _ = b.capture(traced=False)
        serial_ms = max_over_ranks(time_blocks(b, args, st, dist, sgraphs, min_ms / 4)[0], dist,
                                   "cuda")
        b.overlap = True
        del sgraphs

    # traced replay of the serial step: per-kernel durations (graph event
    # nodes) for the roofline, each kernel timed without the other stream's
    # kernels sharing the GPU
    b.overlap = False
    try:
        tgraphs, traces = b.capture(traced=True)
    except Exception as ex:  # report the timed result even if tracing is unavailable
        print(f"traced capture failed: {ex}", file=sys.stderr)
        tgraphs, traces = [], []
    per = {}
    reps = max(3, min(args.steps, 50)) if traces else 0
    for i in range(reps):
        r = i % nrot
        b.before_step(i)
        tgraphs[r].replay()
        torch.cuda.synchronize()
        for name, dt in traces[r].durations_ms():
            per.setdefault(name, []).append(dt)
    if traces:
        launches_per_step = traces[0].count
    else:  # count the launches of one eager step
        with b.H.Trace(capacity=256) as tr:
            b.step(0)
        torch.cuda.synchronize()
        launches_per_step = tr.count
    # the traced graphs and their events (2 x trace_capacity per cache copy:
    # tens of thousands on the tiny workload) are released before the
    # end-to-end legs, whose host-side calls they would otherwise slow down
    del tgraphs, traces
    gc.collect()
    torch.cuda.synchronize()
    b.overlap = True
    tot = {k: float(np.sum(v)) / reps for k, v in per.items()}     # ms per step
    avg = {k: float(np.mean(v)) for k, v in per.items()}           # ms per launch
    ns = b.n_sel.cpu().numpy()
    work = algorithmic_work(w, ns)
    pk, pk_kind = peaks()
    dominant = max(tot, key=tot.get) if tot else None
    link_gbs = link_peak_gbs() if w.kv_on_host else None

    # the pool attention's launch duration in its chain (the dominant kernel of
    # the device-resident workloads); the isolated traced one is kept beside it
    chain = {}
    for name in ("attn_flash_kernel", "attn_pool_kernel"):
        if name in avg and not getattr(b, "exact", False):
            chain[name] = attn_chain_ms(b)
            break

    def roof(name):
        wk = work.get(name)
        if not wk or name not in avg:
            return None
        d_s = chain.get(name, avg[name]) * 1e-3
        if wk["bound"] in ("hbm", "link"):
            ach = wk["bytes"] / d_s / 1e9
            peak = link_gbs if wk["bound"] == "link" else pk["hbm_gbs"]
            unit = "GB/s"
        else:
            ach = wk["flops"] / d_s / 1e12
            peak = pk["bf16_tflops"]
            unit = "TFLOP/s"
        return {"bound": wk["bound"], "achieved": ach, "peak": peak, "unit": unit,
                "frac": ach / peak, "traffic": ncu_traffic(name, w.name),
                "kernel": name, "launch_us": d_s * 1e6,
                "launch_timing": ("mean of back-to-back launches in a graph (a block's T "
                                  "steps, programmatic launch), CUDA events"
                                  if name in chain else
                                  "isolated launch in the traced replay, CUDA events"),
                "launch_us_isolated": avg[name] * 1e3,
                "algorithmic_bytes" if "bytes" in wk and wk["bound"] != "tensor"
                else "algorithmic_flops":
                    wk["bytes"] if "bytes" in wk and wk["bound"] != "tensor" else wk["flops"],
                "peak_source": ("measured in-process: pinned host -> device copy, 256 MiB"
                                if wk["bound"] == "link" else
                                f"{pk_kind} (MEASURED_PEAKS.json)" if pk_kind == "measured"
                                else "fallback")}

    roofline = (roof(dominant) or roof("attn_flash_kernel") or roof("attn_pool_kernel")
                or roof("attn_cluster_kernel") or roof("attn_kernel"))
    attention = (roof("attn_flash_kernel") or roof("attn_pool_kernel") or roof("attn_cluster_kernel")
                 or roof("attn_kernel"))
    scan = roof("scan_tc_kernel") or roof("scan_cc_kernel")
    out = {"value": job_value(ms, world, w.N * w.B), "ms_per_step": ms,
           "config": {"workload": w.name, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                      "ctx": w.L, "B": w.B, "T": w.T, "C": w.C, "K": w.K, "sink": w.S,
                      "local": w.W, "layers": w.layers, "l2": b.l2_note(),
                      "context": b.context_note(), "selection": _SELECTION,
                      "prefetch": b.prefetch_note(), "budget": b.budget_note(),
                      "timing": (f"CUDA-graph replay, {chunk} consecutive blocks per graph "
                                 f"(one graph launch per {chunk} blocks), CUDA events; "
                                 if chunk > 1 else
                                 "CUDA-graph replay of whole steps, CUDA events; ")
                                + f"{reps_timed} timed regions of {args.steps} steps, median"},
           "timed_regions": reps_timed,
           "roofline": roofline, "attention": attention,
           "scan": {"achieved_gbs": scan["achieved"] if scan else None,
                    "frac": scan["frac"] if scan else None,
                    "peak": scan["peak"] if scan else None,
                    "unit": "GB/s", "bound": scan["bound"] if scan else None,
                    "kernel": scan["kernel"] if scan else None,
                    "launch_us": scan["launch_us"] if scan else None,
                    "traffic": scan["traffic"] if scan else None},
           "kernels_ms_per_step": {k: round(v, 5) for k, v in sorted(tot.items(),
                                                                     key=lambda kv: -kv[1])},
           "gpu_launches": launches_per_step * args.steps,
           "launches_per_step": launches_per_step,
           "clocks": clocks.summary(t0, t1), "device_error_word": err}
    if serial_ms is not None:
        out["serial"] = {"ms_per_step": serial_ms,
                         "value": job_value(serial_ms, world, w.N * w.B),
                         "what": "same step with stage 1 on the denoising stream (no overlap)"}
    if e2e:
        out["e2e"] = run_e2e(b, args, dist, graph=True)
        out["e2e"]["direct_calls"] = run_e2e(b, args, dist, graph=False)
    return out, b


RANGE = {"llama": "LLAMA_64K", "long-host": "LONG_128K_HOST", "stack": "QWEN_STACK"}


def run_ours(args, rank, world, dist):
    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    w = workload()
    main, b = measure(w, args, dist, world, args.min_timed_ms, e2e=True)
    del b
    torch.cuda.empty_cache()
    line = {"metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(main["config"], parallelism=f"replicas x{world}"),
            "roofline": main["roofline"], "attention": main["attention"],
            "serial": main["serial"], "scan": main["scan"],
            "kernels_ms_per_step": main["kernels_ms_per_step"],
            "kernels_timing": "traced replay of the serial step (CUDA events around each "
                              "kernel; no cross-stream overlap)",
            "gpu_launches": main["gpu_launches"], "timed_regions": main["timed_regions"],
            "clocks": main["clocks"], "e2e": main["e2e"],
            "device_error_word": main["device_error_word"],
            "source_hash": kernel_source_hash()}

    # the rest of the metric's range (32K-128K), each workload at full size,
    # timed the same way: block tokens/s, the scan's and the attention's
    # rooflines
    from block_diffusion_sparse_gb300 import workloads as W
    rng = {}
    for key in [r for r in args.range.split(",") if r and r != "none"]:
        wr = getattr(W, RANGE[key])
        if wr.name == w.name:
            continue
        try:
            r, b = measure(wr, args, dist, world, args.min_timed_ms / 2, serial=False)
            del b
        except Exception as ex:  # one failing range entry must not hide the headline
            r = {"error": f"{type(ex).__name__}: {ex}"}
        torch.cuda.empty_cache()
        rng[wr.name] = {k: r.get(k) for k in ("value", "ms_per_step", "config", "scan",
                                               "attention", "kernels_ms_per_step",
                                               "timed_regions", "clocks", "device_error_word",
                                               "error") if k in r}
        rng[wr.name]["gpu_launches"] = r.get("gpu_launches")
    if rng:
        line["range"] = rng
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(b, args, dist, graph: bool = True):
    """Every step: that step's inputs (the T steps' queries and block K/V)
    copied from pinned host memory to the device, the step through the
    pipeline's public call (BlockPipeline.block), and its result (the T
    attention outputs) copied back to pinned host memory -- all inside the
    timed region.  Inputs and outputs travel on two copy streams of their
    own against two alternating sets of device buffers, so step i+1's inputs
    arrive and step i-1's outputs leave while step i computes (the double
    buffering a serving loop would use).

    graph=True: each step is one CUDA graph, captured once per (cache copy,
    buffer set) during the warm-up, holding the block's C-ABI calls
    (BlockPipeline.block) and, on the copy streams forked from it and joined
    back, the upload of the next step's inputs and the download of the
    previous step's outputs; the last timed step's outputs are downloaded
    inside the timed region as well.  graph=False: direct C-ABI calls every
    step, the copies issued around them on the copy streams."""
    torch = b.torch
    w = b.w
    pin = lambda t: t.cpu().pin_memory()
    hq_s, hbk, hbv = pin(b.q_steps), pin(b.bk), pin(b.bv)
    o_out = torch.empty(b.out.shape, dtype=b.out.dtype).pin_memory()
    din = [{"q_s": torch.empty_like(b.q_steps), "bk": torch.empty_like(b.bk),
            "bv": torch.empty_like(b.bv)} for _ in range(2)]
    dout = [torch.empty_like(b.out) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq_s, hbk, hbv))
    d2h = o_out.numel() * o_out.element_size()
    comp = torch.cuda.current_stream()
    cp = torch.cuda.Stream()     # host -> device
    cpo = torch.cuda.Stream()    # device -> host
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    for e in h2d_done + comp_done + out_done:
        e.record(comp)

    # one graph per (cache copy, input slot); with many rotated cache copies
    # (tiny workloads) the direct calls are used instead
    use_graph = graph and b.n_rot <= 8
    graphs = {}

    def upload(x):
        x["q_s"].copy_(hq_s, non_blocking=True)
        x["bk"].copy_(hbk, non_blocking=True)
        x["bv"].copy_(hbv, non_blocking=True)

    def body(i):
        """Step i on the current stream: the next step's inputs up and the
        previous step's outputs down on the copy streams, beside the block."""
        s, cur = i % 2, torch.cuda.current_stream()
        cp.wait_stream(cur)
        cpo.wait_stream(cur)
        with torch.cuda.stream(cp):
            upload(din[1 - s])
        with torch.cuda.stream(cpo):
            o_out.copy_(dout[1 - s], non_blocking=True)
        x = din[s]
        b.step(i % b.n_rot, q_steps=x["q_s"], bk=x["bk"], bv=x["bv"], out=dout[s])
        cur.wait_stream(cp)
        cur.wait_stream(cpo)

    def one_graph(i):
        b.before_step(i)
        key = (i % b.n_rot, i % 2)
        g = graphs.get(key)
        if g is not None:
            g.replay()
            return
        body(i)  # the first time: run directly, then capture the same work
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(comp)
        with torch.cuda.graph(g, stream=cap):
            body(i)
        comp.wait_stream(cap)
        graphs[key] = g

    def one(i):
        s = i % 2
        x = din[s]
        b.before_step(i)
        cp.wait_event(comp_done[s])   # the step that last read these inputs is done
        comp.wait_event(out_done[s])  # ... and its outputs have been read back
        with torch.cuda.stream(cp):
            x["q_s"].copy_(hq_s, non_blocking=True)
            x["bk"].copy_(hbk, non_blocking=True)
            x["bv"].copy_(hbv, non_blocking=True)
            h2d_done[s].record(cp)
        comp.wait_event(h2d_done[s])
        b.step(i % b.n_rot, q_steps=x["q_s"], bk=x["bk"], bv=x["bv"], out=dout[s],
               graph=use_graph)
        comp_done[s].record(comp)
        cpo.wait_event(comp_done[s])
        with torch.cuda.stream(cpo):
            o_out.copy_(dout[s], non_blocking=True)
            out_done[s].record(cpo)

    # warm-up covers every (cache copy, input slot) pair, so all graphs are
    # captured before the timed region
    n_warm = max(args.warmup, 2 * b.n_rot) if use_graph else args.warmup
    n_warm += n_warm % 2
    step_fn = one_graph if use_graph else one
    if use_graph:
        upload(din[0])  # step 0's inputs; each step uploads the next one's
    for i in range(n_warm):
        step_fn(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for i in range(n_warm, n_warm + args.steps):
        step_fn(i)
    if use_graph:  # the last step's outputs
        cpo.wait_stream(comp)
        with torch.cuda.stream(cpo):
            o_out.copy_(dout[(n_warm + args.steps - 1) % 2], non_blocking=True)
    comp.wait_stream(cp)
    comp.wait_stream(cpo)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, "cuda")
    world = dist.get_world_size() if dist else 1
    return {"value": job_value(ms, world, w.N * w.B), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms,
            "path": ("one CUDA graph per step, captured once per (cache copy, buffer set) "
                     "during the warm-up: BlockPipeline.block's C-ABI calls, with the next "
                     "step's input upload and the previous step's output download on copy "
                     "streams forked from it and joined back" if use_graph else
                     "direct C-ABI calls every step: one herald_block call per block for the "
                     "per-key selection (per-call for the other selections; argument checks, "
                     "tensor-map lookups and launches inside the timed region)")
                    + "; pinned host buffers, copies on two copy streams into double-buffered "
                    "device inputs/outputs; the cache rotates as in the device-timed run"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-timed-ms", type=float, default=200.0,
                    help="the timed region of --steps steps is repeated until the repeats add "
                         "up to this (the median per step is reported)")
    ap.add_argument("--range", default="llama,long-host,stack",
                    help="other workloads of the metric's range measured after the headline "
                         "(comma-separated: llama, long-host, stack; none)")
    ap.add_argument("--workload", default="qwen", choices=sorted(WORKLOADS))
    ap.add_argument("--selection", default="merged", choices=["merged", "exact", "blocks"],
                    help="merged: the two-stage selection (default); exact: every cached "
                         "position scored with the block's real queries (one stream); "
                         "blocks: stage 1 over 64-key block means")
    ap.add_argument("--budget", type=float, default=None, metavar="TAU",
                    help="per-key merged selection with an adaptive budget per block and KV "
                         "head: the smallest K (at least K/8, at most K) whose top scores "
                         "hold TAU of the first step's stage-2 mass")
    ap.add_argument("--prefetch", default="kv", choices=["k", "kv"],
                    help="host-resident cache with --selection blocks: the next block's "
                         "candidate rows copied beside the denoising steps -- K rows for "
                         "stage 2 (k), or K and V rows with the top-K pool rows gathered "
                         "from HBM (kv, default)")
    args = ap.parse_args()
    global _WORKLOAD, _SELECTION, _PREFETCH, _BUDGET
    _WORKLOAD = args.workload
    _SELECTION = args.selection
    _PREFETCH = args.prefetch
    _BUDGET = args.budget
    if _BUDGET is not None and (args.selection != "merged" or args.workload == "stack"
                                or not 0.0 < _BUDGET <= 1.0):
        ap.error("--budget takes a TAU in (0, 1], the merged selection and one layer")
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl" if args.impl == "ours" else "gloo")
        dist = tdist
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, dist)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
