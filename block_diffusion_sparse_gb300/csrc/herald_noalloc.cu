// herald_noalloc.cu -- herald_select_stage2_noalloc: stage 2 of the selection
// for callers that cannot hand the library a workspace.
//
// Some callers cannot allocate device memory at the point where they select:
// a decode loop that runs under CUDA stream capture (cudaMalloc and cudaFree
// are not allowed while a stream is being captured), a plugin inside a
// serving runtime that owns the whole device-memory budget and hands out no
// buffers after start-up, or a host callback where a synchronising
// allocation would stall every stream.  For them this entry point keeps its
// scratch -- the refine row statistics, the stage-2 scores and an error word
// -- in one file-scope device array, so the call needs only its inputs and
// outputs.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "../../include/herald.h"
#include "internal.cuh"

using namespace herald;

namespace {

// Upper bound of the scratch this entry point may use.  Every GPU that loads
// the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_stage2_scratch[kStaticScratchBytes];

// Errors are reported like every other entry point: a status, with the
// detail readable through herald_last_error().
herald_status fail(herald_status s, const char* fmt, ...) {
  char msg[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof msg, fmt, ap);
  va_end(ap);
  set_last_error(msg);
  return s;
}

// Device address of g_stage2_scratch on the current device.  Resolved once
// per device, with that device current; host code must not use the array's
// name as an address.  Host threads that make their first calls at the
// same time resolve it under one lock; later calls read the published
// address without locking.
herald_status scratch_address(unsigned char** out) {
  constexpr int kMaxDevices = 64;
  static std::atomic<unsigned char*> addr[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(HERALD_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(HERALD_ERR_CUDA, "device ordinal %d out of range", dev);
  unsigned char* p = addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(mu);
    p = addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      void* q = nullptr;
      e = cudaGetSymbolAddress(&q, g_stage2_scratch);
      if (e != cudaSuccess)
        return fail(HERALD_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
      p = static_cast<unsigned char*>(q);
      addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return HERALD_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

herald_status herald_select_stage2_noalloc(herald_dims dims, const uint16_t* q_block,
                                           const uint16_t* k_cache, const int32_t* ctx_len,
                                           const int32_t* cand, const int32_t* n_cand, int C,
                                           int K, int sink, int local, int P_max, int32_t* idx,
                                           int32_t* n_sel, void* stream) {
  set_last_error("");
  // the argument rules of herald_select_stage2 (shapes, C, P_max, budget)
  herald_status s = check_stage2_args(dims, C, K, sink, local, P_max);
  if (s != HERALD_OK) return s;
  if (!aligned16(q_block) || !aligned16(k_cache) || !aligned16(ctx_len) || !aligned16(cand) ||
      !aligned16(n_cand) || !aligned16(idx) || !aligned16(n_sel))
    return fail(HERALD_ERR_INVALID_ARG, "a pointer is NULL or not 16-byte aligned");

  // compact scratch layout: error word | refine row statistics | row lse | s2
  const WsLayout full = ws_layout(dims, C, P_max);
  const size_t NG = size_t(dims.N) * dims.Hkv;
  const size_t err_off = 0;
  const size_t rpart_off = 256;
  const size_t rpart_bytes = NG * size_t(full.MT) * kTileM * full.n_chunks * 8;
  const size_t rlse_off = align_up(rpart_off + rpart_bytes, 256);
  const size_t rlse_bytes = NG * size_t(full.MT) * kTileM * 4;
  const size_t s2_off = align_up(rlse_off + rlse_bytes, 256);
  const int n_parts = refine_fused_ok(C) ? full.MT_tok : 1;  // s2 partials per row tile
  const size_t need = s2_off + NG * size_t(C) * 4 * size_t(n_parts);
  if (need > kStaticScratchBytes)
    return fail(HERALD_ERR_WORKSPACE_TOO_SMALL,
                "these shapes need %zu bytes of scratch; the static scratch holds %zu",
                need, kStaticScratchBytes);
  // herald_select_stage2 stages a host-resident cache's candidate rows in
  // its workspace before the refine; this call has no room for them
  if (!device_resident(k_cache))
    return fail(HERALD_ERR_INVALID_ARG,
                "k_cache is not device memory: the workspace-free stage 2 takes a cache in "
                "HBM only (use herald_select_stage2 for a host-resident cache)");

  unsigned char* base = nullptr;
  s = scratch_address(&base);
  if (s != HERALD_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(base + err_off);
  // the fused refine reads its query tiles by TMA (a host-side descriptor,
  // no device memory)
  CUtensorMap qmap, qmap_all;
  const int G = dims.Hq / dims.Hkv;
  s = encode_heads_map(q_block, uint64_t(dims.N) * dims.B, dims.Hq, dims.d, uint32_t(G),
                       uint32_t(kTileM / G), &qmap);
  if (s == HERALD_OK)
    s = encode_heads_map(q_block, uint64_t(dims.N) * dims.B, dims.Hq, dims.d, uint32_t(G),
                         uint32_t(dims.B), &qmap_all);
  if (s != HERALD_OK) return s;
  // the array keeps the previous call's contents: the error word must start
  // at zero; the statistics and scores are fully rewritten before use
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess)
    e = launch_refine(dims, k_cache, cand, n_cand, C,
                      reinterpret_cast<float2*>(base + rpart_off),
                      reinterpret_cast<float*>(base + rlse_off),
                      reinterpret_cast<float*>(base + s2_off), full, err, &qmap, &qmap_all, st);
  if (e == cudaSuccess)
    e = launch_topk_union(dims, ctx_len, cand, n_cand, reinterpret_cast<float*>(base + s2_off),
                          n_parts, C, K, sink, local, P_max, idx, n_sel, st, nullptr, nullptr,
                          nullptr, true);
  if (e != cudaSuccess)
    return fail(HERALD_ERR_CUDA, "stage-2 launch: %s", cudaGetErrorString(e));
  return HERALD_OK;
}

}  // extern "C"
