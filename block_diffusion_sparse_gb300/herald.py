"""ctypes binding of libherald.so (include/herald.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors may be torch tensors (their data_ptr() is passed) or raw
integer addresses; streams may be torch streams or raw cudaStream_t values.
There is no CPU fallback: if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
RELEASE_LIB = os.path.join(_HERE, "_build", "libherald.so")
DEBUG_LIB = os.path.join(_HERE, "_build_debug", "libherald.so")
# HERALD_LIB=debug selects the debug build (device checks of indices and
# counts); any other value is taken as the library's path
LIB_PATH = {"": RELEASE_LIB, "debug": DEBUG_LIB}.get(os.environ.get("HERALD_LIB", ""),
                                                      os.environ.get("HERALD_LIB", ""))

HERALD_OK = 0
# flags of herald_denoise_attn_ex (include/herald.h)
HERALD_ATTN_SETTLED, HERALD_ATTN_APPEND, HERALD_ATTN_ADVANCE = 1, 2, 4
# kernel choice of herald_denoise_attn_ex (bits 8-11; default: by shape)
HERALD_ATTN_KERNEL_POOL, HERALD_ATTN_KERNEL_FLASH = 1 << 8, 2 << 8
HERALD_ATTN_KERNEL_FLASH_CS2, HERALD_ATTN_KERNEL_FLASH_CS4, HERALD_ATTN_KERNEL_FLASH_CS8 = (
    3 << 8, 4 << 8, 5 << 8)
HERALD_ATTN_KERNEL_POOL_CS8, HERALD_ATTN_KERNEL_POOL_CS16, HERALD_ATTN_KERNEL_POOL_CS12 = (
    6 << 8, 7 << 8, 8 << 8)


# flags of herald_block
HERALD_BLOCK_ADVANCE = 1
HERALD_BLOCK_CAND_SETTLED = 2


def HERALD_ATTN_SMS(n: int) -> int:
    """The SM-budget bits of herald_denoise_attn_ex's flags (units of 4 SMs)."""
    return ((int(n) // 4) & 0xFF) << 16

STATUS = {0: "HERALD_OK", 1: "HERALD_ERR_INVALID_ARG", 2: "HERALD_ERR_UNSUPPORTED_SHAPE",
          3: "HERALD_ERR_WORKSPACE_TOO_SMALL", 4: "HERALD_ERR_CUDA"}

EXPORTS = ("herald_workspace_size", "herald_status_string", "herald_last_error",
           "herald_workspace_error", "herald_select_stage1", "herald_select_stage2",
           "herald_select", "herald_select_stage2_gather", "herald_gather",
           "herald_denoise_attn", "herald_denoise_attn_ex", "herald_append_kv",
           "herald_trace_begin", "herald_trace_end", "herald_trace_name",
           "herald_select_stage2_noalloc", "herald_selftest_wait_timeout",
           "herald_workspace_size_exact", "herald_select_exact", "herald_pool_keys",
           "herald_select_stage1_blocks", "herald_stage_candidates",
           "herald_select_stage2_staged", "herald_select_stage2_staged_gather",
           "herald_select_stage2_adaptive", "herald_debug_build", "herald_debug_status",
           "herald_inject_launch_failure", "herald_block")


class HeraldError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status


class Dims(C.Structure):
    _fields_ = [("N", C.c_int), ("Hq", C.c_int), ("Hkv", C.c_int), ("d", C.c_int),
                ("B", C.c_int), ("L_max", C.c_int)]

    def __repr__(self):
        return (f"Dims(N={self.N}, Hq={self.Hq}, Hkv={self.Hkv}, d={self.d}, B={self.B}, "
                f"L_max={self.L_max})")


class BlockBufs(C.Structure):
    """herald_block_bufs: the pipeline's buffers, streams and events, kept
    from block to block (addresses and handles as integers)."""
    _fields_ = [("cand", C.c_void_p * 2), ("n_cand", C.c_void_p * 2), ("idx", C.c_void_p),
                ("n_sel", C.c_void_p), ("pool_k", C.c_void_p * 2), ("pool_v", C.c_void_p * 2),
                ("ws_den", C.c_void_p), ("ws_sel", C.c_void_p), ("ws_bytes", C.c_size_t),
                ("sel_stream", C.c_void_p), ("ev_fork", C.c_void_p), ("ev_join", C.c_void_p)]


def dims(N, Hq, Hkv, d, B, L_max) -> Dims:
    return Dims(int(N), int(Hq), int(Hkv), int(d), int(B), int(L_max))


def dims_of(w) -> Dims:
    """Dims of a workloads.Workload."""
    return dims(w.N, w.Hq, w.Hkv, w.d, w.B, w.L_max)


_lib = None


def lib() -> C.CDLL:
    """Loads libherald.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libherald.so not built ({LIB_PATH}); run "
                "`python -m block_diffusion_sparse_gb300.build` first")
        L = C.CDLL(LIB_PATH)
        vp, i32, sz = C.c_void_p, C.c_int, C.c_size_t
        L.herald_workspace_size.argtypes = [Dims, i32, i32]
        L.herald_workspace_size.restype = sz
        L.herald_status_string.argtypes = [i32]
        L.herald_status_string.restype = C.c_char_p
        L.herald_last_error.argtypes = []
        L.herald_last_error.restype = C.c_char_p
        L.herald_workspace_error.argtypes = [vp, vp, C.POINTER(C.c_uint32)]
        L.herald_select_stage1.argtypes = [Dims, vp, vp, vp, i32, vp, vp, vp, sz, i32, vp]
        L.herald_select_stage2.argtypes = [Dims, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                           vp, vp, vp, sz, vp]
        L.herald_select.argtypes = [Dims, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                    sz, vp]
        L.herald_select_stage2_gather.argtypes = [Dims, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                  i32, i32, vp, vp, vp, vp, vp, sz, vp]
        L.herald_gather.argtypes = [Dims, vp, vp, i32, vp, vp, vp, vp, vp]
        L.herald_denoise_attn.argtypes = [Dims, vp, vp, vp, vp, i32, vp, vp, vp, C.c_float, vp,
                                          sz, vp]
        L.herald_denoise_attn_ex.argtypes = [Dims, vp, vp, vp, vp, i32, vp, vp, vp, C.c_float,
                                             C.c_uint, vp, vp, vp, vp, sz, vp]
        L.herald_append_kv.argtypes = [Dims, vp, vp, vp, vp, vp, i32, vp]
        L.herald_block.argtypes = [Dims, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                   vp, vp, vp, C.c_uint, i32, C.POINTER(BlockBufs), vp]
        L.herald_select_stage2_noalloc.argtypes = [Dims, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                   i32, vp, vp, vp]
        L.herald_selftest_wait_timeout.argtypes = [C.c_uint64, vp, vp]
        L.herald_workspace_size_exact.argtypes = [Dims, i32, i32]
        L.herald_workspace_size_exact.restype = sz
        L.herald_select_exact.argtypes = [Dims, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, sz,
                                          vp]
        L.herald_pool_keys.argtypes = [Dims, vp, vp, i32, i32, vp, vp]
        L.herald_stage_candidates.argtypes = [Dims, vp, vp, vp, vp, i32, vp, vp, vp]
        L.herald_select_stage2_staged.argtypes = [Dims, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                  i32, vp, vp, vp, sz, vp]
        L.herald_debug_build.argtypes = []
        L.herald_debug_build.restype = i32
        L.herald_debug_status.argtypes = [C.POINTER(C.c_uint32)]
        L.herald_inject_launch_failure.argtypes = [i32, i32]
        L.herald_select_stage2_adaptive.argtypes = [Dims, vp, vp, vp, vp, vp, i32, i32, i32,
                                                    C.c_float, i32, i32, i32, vp, vp, vp, vp,
                                                    sz, vp]
        L.herald_select_stage2_staged_gather.argtypes = [Dims, vp, vp, vp, vp, vp, vp, vp, vp,
                                                         i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                                         vp, sz, vp]
        L.herald_select_stage1_blocks.argtypes = [Dims, vp, vp, vp, i32, i32, vp, vp, vp, sz,
                                                  vp]
        L.herald_trace_begin.argtypes = [C.POINTER(vp), i32, i32]
        L.herald_trace_end.argtypes = []
        L.herald_trace_name.argtypes = [i32]
        L.herald_trace_name.restype = C.c_char_p
        for name in EXPORTS:
            if name not in ("herald_workspace_size", "herald_workspace_size_exact",
                            "herald_status_string",
                            "herald_last_error", "herald_trace_name"):
                getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an address, got {type(x)}")


def _s(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    raise TypeError(f"expected a stream, got {type(stream)}")


def _nbytes(ws, ws_bytes):
    if ws_bytes is not None:
        return int(ws_bytes)
    if hasattr(ws, "numel"):
        return ws.numel() * ws.element_size()
    raise ValueError("ws_bytes is required for a raw workspace address")


def _check(status: int):
    if status != HERALD_OK:
        raise HeraldError(status, lib().herald_last_error().decode())


# Helpers for callers that resolve addresses once and call lib() directly
# (the pipeline's per-block path): plain integers cross ctypes fastest.
check = _check


def ptr(x) -> int:
    """Device (or mapped host) address of a tensor, or an address as is."""
    p = _p(x)
    if p is None:
        raise ValueError("a NULL address where a buffer is required")
    return p


def step_bytes(x) -> int:
    """Byte distance between consecutive entries of a tensor's first axis."""
    if not x.is_contiguous():
        raise ValueError("per-step inputs and outputs must be contiguous")
    return x.stride(0) * x.element_size()


def stream_handle(stream) -> int:
    """cudaStream_t of a torch stream (0 = the legacy default stream)."""
    h = _s(stream)
    return 0 if h is None else h


def herald_workspace_size(d: Dims, C_: int, P_max: int) -> int:
    return int(lib().herald_workspace_size(d, int(C_), int(P_max)))


def herald_status_string(status: int) -> str:
    return lib().herald_status_string(int(status)).decode()


def herald_debug_build() -> bool:
    """Whether the loaded library is the debug build (device checks)."""
    return bool(lib().herald_debug_build())


def herald_debug_status() -> int:
    """The debug build's device check word (waits for the device, then
    reads and clears it); 0 in release builds."""
    code = C.c_uint32(0)
    _check(lib().herald_debug_status(C.byref(code)))
    return int(code.value)


def herald_inject_launch_failure(after: int, cuda_error: int = 719):
    """Test hook: the launch after `after` more launches on this host
    thread fails with `cuda_error` (default cudaErrorLaunchFailure); a
    negative `after` disarms it."""
    _check(lib().herald_inject_launch_failure(int(after), int(cuda_error)))


def herald_workspace_error(ws, stream=None) -> int:
    code = C.c_uint32(0)
    _check(lib().herald_workspace_error(_p(ws), _s(stream), C.byref(code)))
    return int(code.value)


def herald_select_stage1(d, q_merge, k_cache, ctx_len, C_, cand, n_cand, ws, ws_bytes=None,
                         stream=None, sm_budget=0):
    _check(lib().herald_select_stage1(d, _p(q_merge), _p(k_cache), _p(ctx_len), int(C_),
                                      _p(cand), _p(n_cand), _p(ws), _nbytes(ws, ws_bytes),
                                      int(sm_budget), _s(stream)))


def herald_select_stage2(d, q_block, k_cache, ctx_len, cand, n_cand, C_, K, sink, local, P_max,
                         idx, n_sel, ws, ws_bytes=None, stream=None):
    _check(lib().herald_select_stage2(d, _p(q_block), _p(k_cache), _p(ctx_len), _p(cand),
                                      _p(n_cand), int(C_), int(K), int(sink), int(local),
                                      int(P_max), _p(idx), _p(n_sel), _p(ws),
                                      _nbytes(ws, ws_bytes), _s(stream)))


def herald_select(d, q_merge, q_block, k_cache, ctx_len, C_, K, sink, local, P_max, idx, n_sel,
                  ws, ws_bytes=None, stream=None):
    _check(lib().herald_select(d, _p(q_merge), _p(q_block), _p(k_cache), _p(ctx_len), int(C_),
                               int(K), int(sink), int(local), int(P_max), _p(idx), _p(n_sel),
                               _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def herald_select_stage2_noalloc(d, q_block, k_cache, ctx_len, cand, n_cand, C_, K, sink, local,
                                 P_max, idx, n_sel, stream=None):
    """Stage 2 with the library's static scratch instead of a workspace, for
    callers that cannot allocate device memory where they select (see
    include/herald.h); calls that overlap on the GPU must be serialised."""
    _check(lib().herald_select_stage2_noalloc(d, _p(q_block), _p(k_cache), _p(ctx_len), _p(cand),
                                              _p(n_cand), int(C_), int(K), int(sink), int(local),
                                              int(P_max), _p(idx), _p(n_sel), _s(stream)))


def herald_workspace_size_exact(d: Dims, K: int, P_max: int) -> int:
    return int(lib().herald_workspace_size_exact(d, int(K), int(P_max)))


def herald_select_exact(d, q_block, k_cache, ctx_len, K, sink, local, P_max, idx, n_sel, ws,
                        ws_bytes=None, stream=None):
    """Exact selection over the whole cache with all the block's queries
    (see include/herald.h)."""
    _check(lib().herald_select_exact(d, _p(q_block), _p(k_cache), _p(ctx_len), int(K), int(sink),
                                     int(local), int(P_max), _p(idx), _p(n_sel), _p(ws),
                                     _nbytes(ws, ws_bytes), _s(stream)))


def herald_selftest_wait_timeout(limit_ns, ws, stream=None):
    """Runs one bounded wait that nothing completes (see include/herald.h)."""
    _check(lib().herald_selftest_wait_timeout(int(limit_ns), _p(ws), _s(stream)))


def herald_select_stage2_gather(d, q_block, k_cache, v_cache, ctx_len, cand, n_cand, C, K, sink,
                                local, P_max, idx, n_sel, pool_k, pool_v, ws=None,
                                ws_bytes=None, stream=None):
    _check(lib().herald_select_stage2_gather(d, _p(q_block), _p(k_cache), _p(v_cache),
                                             _p(ctx_len), _p(cand), _p(n_cand), int(C), int(K),
                                             int(sink), int(local), int(P_max), _p(idx),
                                             _p(n_sel), _p(pool_k), _p(pool_v), _p(ws),
                                             _nbytes(ws, ws_bytes), _s(stream)))


def herald_pool_keys(d, k_cache, ctx_len, Bk, pooled, n_tail=0, stream=None):
    _check(lib().herald_pool_keys(d, _p(k_cache), _p(ctx_len), int(Bk), int(n_tail), _p(pooled),
                                  _s(stream)))


def herald_select_stage1_blocks(d, q_merge, pooled, ctx_len, Bk, C_blocks, cand, n_cand,
                                ws=None, ws_bytes=None, stream=None):
    _check(lib().herald_select_stage1_blocks(d, _p(q_merge), _p(pooled), _p(ctx_len), int(Bk),
                                             int(C_blocks), _p(cand), _p(n_cand), _p(ws),
                                             _nbytes(ws, ws_bytes), _s(stream)))


def herald_stage_candidates(d, k_cache, cand, n_cand, C, staged_k, v_cache=None, staged_v=None,
                            stream=None):
    _check(lib().herald_stage_candidates(d, _p(k_cache), _p(v_cache), _p(cand), _p(n_cand),
                                         int(C), _p(staged_k), _p(staged_v), _s(stream)))


def herald_select_stage2_staged(d, q_block, staged_k, ctx_len, cand, n_cand, C, K, sink, local,
                                P_max, idx, n_sel, ws=None, ws_bytes=None, stream=None):
    _check(lib().herald_select_stage2_staged(d, _p(q_block), _p(staged_k), _p(ctx_len), _p(cand),
                                             _p(n_cand), int(C), int(K), int(sink), int(local),
                                             int(P_max), _p(idx), _p(n_sel), _p(ws),
                                             _nbytes(ws, ws_bytes), _s(stream)))


def herald_select_stage2_staged_gather(d, q_block, staged_k, staged_v, k_cache, v_cache, ctx_len,
                                       cand, n_cand, C, K, sink, local, P_max, idx, n_sel,
                                       pool_k, pool_v, ws=None, ws_bytes=None, stream=None):
    _check(lib().herald_select_stage2_staged_gather(
        d, _p(q_block), _p(staged_k), _p(staged_v), _p(k_cache), _p(v_cache), _p(ctx_len),
        _p(cand), _p(n_cand), int(C), int(K), int(sink), int(local), int(P_max), _p(idx),
        _p(n_sel), _p(pool_k), _p(pool_v), _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def herald_select_stage2_adaptive(d, q_block, k_cache, ctx_len, cand, n_cand, C, K_min, K_max,
                                  tau, sink, local, P_max, idx, n_sel, k_sel, ws=None,
                                  ws_bytes=None, stream=None):
    _check(lib().herald_select_stage2_adaptive(
        d, _p(q_block), _p(k_cache), _p(ctx_len), _p(cand), _p(n_cand), int(C), int(K_min),
        int(K_max), float(tau), int(sink), int(local), int(P_max), _p(idx), _p(n_sel),
        _p(k_sel), _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def herald_gather(d, idx, n_sel, P_max, k_cache, v_cache, pool_k, pool_v, stream=None):
    _check(lib().herald_gather(d, _p(idx), _p(n_sel), int(P_max), _p(k_cache), _p(v_cache),
                               _p(pool_k), _p(pool_v), _s(stream)))


def herald_denoise_attn(d, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale=0.0,
                        ws=None, ws_bytes=None, stream=None):
    _check(lib().herald_denoise_attn(d, _p(q), _p(pool_k), _p(pool_v), _p(n_sel), int(P_max),
                                     _p(block_k), _p(block_v), _p(out), float(scale), _p(ws),
                                     _nbytes(ws, ws_bytes), _s(stream)))


def herald_denoise_attn_ex(d, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale=0.0,
                           flags=0, ctx_len=None, k_cache=None, v_cache=None, ws=None,
                           ws_bytes=None, stream=None):
    _check(lib().herald_denoise_attn_ex(d, _p(q), _p(pool_k), _p(pool_v), _p(n_sel), int(P_max),
                                        _p(block_k), _p(block_v), _p(out), float(scale),
                                        int(flags), _p(ctx_len), _p(k_cache), _p(v_cache),
                                        _p(ws), _nbytes(ws, ws_bytes), _s(stream)))


def herald_append_kv(d, block_k, block_v, ctx_len, k_cache, v_cache, advance=True,
                     stream=None):
    _check(lib().herald_append_kv(d, _p(block_k), _p(block_v), _p(ctx_len), _p(k_cache),
                                  _p(v_cache), int(bool(advance)), _s(stream)))


def herald_block(d, C_, K, S, W, P_max, T, i, q_steps, block_k, block_v, k_cache, v_cache,
                 ctx_len, next_k_cache, out, flags, scan_sms, bufs, stream=None):
    """bufs: a BlockBufs (passed by reference)."""
    _check(lib().herald_block(d, int(C_), int(K), int(S), int(W), int(P_max), int(T), int(i),
                              _p(q_steps), _p(block_k), _p(block_v), _p(k_cache), _p(v_cache),
                              _p(ctx_len), _p(next_k_cache), _p(out), int(flags), int(scan_sms),
                              C.byref(bufs), _s(stream)))


class Trace:
    """Records a CUDA event pair around every kernel the library launches on
    this thread (see herald_trace_begin).  `external=True` makes the events
    graph nodes when the calls are stream-captured."""

    def __init__(self, capacity: int = 256, external: bool = False):
        import torch
        self.capacity = capacity
        self.external = external
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:       # torch creates the CUDA event on first record
            e.record()
        torch.cuda.synchronize()
        self._arr = (C.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self.count = 0
        self.names: list[str] = []

    def __enter__(self):
        _check(lib().herald_trace_begin(self._arr, self.capacity, int(self.external)))
        return self

    def __exit__(self, *exc):
        self.count = int(lib().herald_trace_end())
        self.names = [lib().herald_trace_name(i).decode() for i in range(self.count)]
        return False

    def durations_ms(self) -> list[tuple[str, float]]:
        """(kernel name, elapsed ms) per traced launch; call after the work
        (or the graph replay that recorded the events) has synchronised."""
        return [(self.names[i], self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i in range(self.count)]
