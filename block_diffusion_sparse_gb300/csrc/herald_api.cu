// herald_api.cu -- the extern "C" entry points of libherald.so: argument
// validation, workspace carving, TMA descriptor encoding, and the kernel
// launch sequence of each call.  No call allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "../../include/herald.h"
#include "internal.cuh"

using namespace herald;

namespace {

thread_local char g_err[512] = "";

herald_status fail(herald_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

herald_status cuda_fail(cudaError_t e, const char* where) {
  return fail(HERALD_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define HERALD_TRY_CUDA(expr, where)          \
  do {                                        \
    cudaError_t e_ = (expr);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define HERALD_CHECK_PTR(p)                                                          \
  do {                                                                               \
    if ((p) == nullptr) return fail(HERALD_ERR_INVALID_ARG, "%s is NULL", #p);       \
    if (!aligned16(p)) return fail(HERALD_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

herald_status check_dims(const herald_dims& d) {
  if (d.N < 1 || d.Hq < 1 || d.Hkv < 1 || d.B < 1 || d.L_max < 1)
    return fail(HERALD_ERR_INVALID_ARG, "dims must be positive (N=%d Hq=%d Hkv=%d B=%d L_max=%d)",
                d.N, d.Hq, d.Hkv, d.B, d.L_max);
  if (d.Hq % d.Hkv != 0)
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "Hq=%d is not a multiple of Hkv=%d", d.Hq, d.Hkv);
  const int G = d.Hq / d.Hkv;
  if (G > 8) return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "GQA group size %d > 8", G);
  if (d.d != 64 && d.d != 128)
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "head dim %d not in {64, 128}", d.d);
  if (d.B * G > 256)
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "B*G = %d > 256 query rows per KV head", d.B * G);
  if ((long long)d.N * d.Hkv * d.L_max >= (1ll << 31))
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "N*Hkv*L_max too large");
  if ((long long)d.N * d.B * d.Hq >= (1ll << 31))
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "N*B*Hq too large");
  return HERALD_OK;
}

herald_status check_c(int C) {
  if (C < 1 || C > kMaxC)
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "C=%d outside [1, %d]", C, kMaxC);
  return HERALD_OK;
}

herald_status check_ws(const herald_dims& dm, int C, int P_max, void* ws, size_t ws_bytes,
                       WsLayout* out) {
  HERALD_CHECK_PTR(ws);
  const WsLayout w = ws_layout(dm, C, P_max);
  if (ws_bytes < w.total)
    return fail(HERALD_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes,
                w.total);
  *out = w;
  return HERALD_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ---- device properties, cached per device
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// ---- TMA descriptor encoding through the driver entry point
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor map of 2 or 3 dimensions, 128-byte swizzle.  A map depends
// only on (base, rank, extents, box): recently encoded ones are reused (per
// thread, a direct-mapped table of 256 entries), which keeps the per-call
// host cost of the steady state low -- a block step encodes a few maps per
// attention call, and a loop over double-buffered inputs and several caches
// meets ~70 distinct maps.
static herald_status encode_map(const void* base, int rank, const uint64_t* extent,
                                const uint32_t* box_in, CUtensorMap* map) {
  struct Entry {
    const void* base;
    int rank;
    uint64_t ext[3];
    uint32_t box[3];
    CUtensorMap map;
  };
  // direct-mapped: one slot per key hash, a lookup is one comparison
  constexpr int kEntries = 256;
  thread_local Entry cache[kEntries] = {};
  uint64_t hkey = reinterpret_cast<uintptr_t>(base) >> 4;
  for (int i = 0; i < rank; ++i) hkey = hkey * 1000003u ^ (extent[i] * 31u + box_in[i]);
  Entry& e = cache[(hkey ^ (hkey >> 17) ^ (hkey >> 33)) % kEntries];
  bool same = e.base == base && e.rank == rank;
  for (int i = 0; same && i < rank; ++i) same = e.ext[i] == extent[i] && e.box[i] == box_in[i];
  if (same) {
    *map = e.map;
    return HERALD_OK;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(HERALD_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  uint64_t stride = 2;  // bytes
  for (int i = 0; i < rank; ++i) {
    dims[i] = extent[i];
    box[i] = box_in[i];
    if (i > 0) strides[i - 1] = stride;
    stride *= extent[i];
  }
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank),
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HERALD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  e.base = base;
  e.rank = rank;
  for (int i = 0; i < rank; ++i) {
    e.ext[i] = extent[i];
    e.box[i] = box_in[i];
  }
  e.map = *map;
  return HERALD_OK;
}

// 2-D bf16 tensor map [rows][d] with a box of 64 columns x box_rows rows and
// 128-byte swizzle (the UMMA K-major shared-memory layout).
herald_status encode_rows_map(const void* base, uint64_t rows, int d, uint32_t box_rows,
                              CUtensorMap* map) {
  const uint64_t ext[2] = {uint64_t(d), rows};
  const uint32_t box[2] = {64, box_rows};
  return encode_map(base, 2, ext, box, map);
}

// [tokens][heads][d] maps: herald::encode_heads_map, below (shared with the
// workspace-free entry point).
herald_status encode_map3(const void* base, const uint64_t* ext, const uint32_t* box,
                          CUtensorMap* map) {
  return encode_map(base, 3, ext, box, map);
}

// Device memory is streamed by TMA; mapped host (or managed) memory by
// plain 16-byte copies.
// The answer for an address does not change while its allocation lives,
// and device and host allocations occupy disjoint ranges of the unified
// address space, so recent answers are reused (per thread).
bool is_device_memory(const void* p) {
  constexpr int kEntries = 32;
  thread_local const void* keys[kEntries] = {};
  thread_local bool vals[kEntries] = {};
  thread_local int next = 0;
  for (int i = 0; i < kEntries; ++i)
    if (keys[i] == p) return vals[i];
  cudaPointerAttributes a;
  bool dev = false;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess)
    cudaGetLastError();
  else
    dev = a.type == cudaMemoryTypeDevice;
  keys[next] = p;
  vals[next] = dev;
  next = (next + 1) % kEntries;
  return dev;
}

herald_status run_stage1(const herald_dims& dm, const uint16_t* q_merge, const uint16_t* k_cache,
                         const int32_t* ctx_len, int C, int32_t* cand, int32_t* n_cand, void* ws,
                         const WsLayout& w, int sm_budget, cudaStream_t st) {
  const bool tma = is_device_memory(k_cache);
  uint32_t* err = at<uint32_t>(ws, w.err);
  float* qbar = at<float>(ws, w.qbar);
  uint16_t* qhl = at<uint16_t>(ws, w.qhl);
  CUtensorMap kmap, bmap;
  if (tma) {
    herald_status s = encode_rows_map(k_cache, uint64_t(dm.N) * dm.Hkv * dm.L_max, dm.d,
                                      kTcScanKeys, &kmap);
    if (s != HERALD_OK) return s;
    s = encode_rows_map(qhl, uint64_t(dm.N) * dm.Hkv * kQhlRows, dm.d, kQhlRows, &bmap);
    if (s != HERALD_OK) return s;
  }
  float* logits = at<float>(ws, w.logits);
  float2* part1 = at<float2>(ws, w.part1);
  float* s1 = at<float>(ws, w.s1);
  uint32_t* hist = at<uint32_t>(ws, w.hist);
  int nsm = sm_count();
  if (sm_budget > 0 && sm_budget < nsm) nsm = sm_budget;
  const int part_slots = scan_grid(dm, w, tma, nsm) * 4;  // one slot per (scan CTA, warp)
  HERALD_TRY_CUDA(launch_merge_query(dm, q_merge, qbar, qhl, hist, part1, part_slots, st),
                  "merge_query launch");
  HERALD_TRY_CUDA(launch_scan(dm, tma ? &kmap : nullptr, tma ? &bmap : nullptr, k_cache, qbar,
                              ctx_len, logits, part1, w, err, nsm, st),
                  "scan launch");
  HERALD_TRY_CUDA(launch_s1_hist(dm, logits, part1, part_slots, ctx_len, s1, hist, w, nsm, st),
                  "s1_hist launch");
  HERALD_TRY_CUDA(launch_topc(dm, s1, hist, ctx_len, C, cand, n_cand, w, st), "topc launch");
  return HERALD_OK;
}

// The adaptive budget of herald_select_stage2_adaptive, between the refine
// and the top-K.
struct BudgetArgs {
  int K_min, K_max;
  float tau;
  int32_t* k_sel;
};

herald_status run_stage2(const herald_dims& dm, const uint16_t* q_block, const uint16_t* k_cache,
                         const int32_t* ctx_len, const int32_t* cand, const int32_t* n_cand,
                         int C, int K, int sink, int local, int P_max, int32_t* idx,
                         int32_t* n_sel, void* ws, const WsLayout& w, cudaStream_t st,
                         const PoolGather* gather, const uint16_t* staged_k = nullptr,
                         int32_t* slot_out = nullptr, const BudgetArgs* budget = nullptr,
                         bool cand_settled = false) {
  uint32_t* err = at<uint32_t>(ws, w.err);
  CUtensorMap qmap, qmap_all;
  const int G = dm.Hq / dm.Hkv;
  herald_status qs = encode_heads_map(q_block, uint64_t(dm.N) * dm.B, dm.Hq, dm.d, uint32_t(G),
                                      uint32_t(kTileM / G), &qmap);
  if (qs == HERALD_OK)
    qs = encode_heads_map(q_block, uint64_t(dm.N) * dm.B, dm.Hq, dm.d, uint32_t(G),
                          uint32_t(dm.B), &qmap_all);
  if (qs != HERALD_OK) return qs;
  float* rlse = at<float>(ws, w.rlse);
  if (staged_k) {
    // the candidate K rows were staged by slot beforehand
    herald_dims staged = dm;
    staged.L_max = C;
    HERALD_TRY_CUDA(launch_refine(staged, staged_k, nullptr, n_cand, C,
                                  at<float2>(ws, w.rpart), rlse, at<float>(ws, w.s2), w, err,
                                  &qmap, &qmap_all, st),
                    "refine launch");
  } else if (is_device_memory(k_cache)) {
    // cand_settled: the candidates and their cache rows were written before
    // the launch preceding this call began (the refine reads them early)
    HERALD_TRY_CUDA(launch_refine(dm, k_cache, cand, n_cand, C, at<float2>(ws, w.rpart),
                                  rlse, at<float>(ws, w.s2), w, err, &qmap, &qmap_all, st,
                                  cand_settled),
                    "refine launch");
  } else {
    // a host-resident cache: the candidate K rows cross the host link once,
    // in one wide gather, into the workspace; the refine then reads them
    // from HBM by slot (the stage-1 logits region is free during stage 2)
    uint16_t* kstage = at<uint16_t>(ws, w.logits);
    HERALD_TRY_CUDA(launch_gather(dm, cand, n_cand, C, k_cache, nullptr, kstage, nullptr, st,
                                  "gather_kernel (candidate staging)"),
                    "candidate staging launch");
    herald_dims staged = dm;
    staged.L_max = C;  // rows per (sequence, KV head) in the staging buffer
    HERALD_TRY_CUDA(launch_refine(staged, kstage, nullptr, n_cand, C,
                                  at<float2>(ws, w.rpart), rlse, at<float>(ws, w.s2), w, err,
                                  &qmap, &qmap_all, st),
                    "refine launch");
  }
  const int n_parts = refine_fused_ok(C) ? w.MT_tok : 1;
  if (budget)
    HERALD_TRY_CUDA(launch_budget(dm, n_cand, at<float>(ws, w.s2), n_parts, C, budget->K_min,
                                  budget->K_max, budget->tau, budget->k_sel, st),
                    "budget launch");
  HERALD_TRY_CUDA(launch_topk_union(dm, ctx_len, cand, n_cand, at<float>(ws, w.s2), n_parts, C, K,
                                    sink, local, P_max, idx, n_sel, st, gather, slot_out,
                                    budget ? budget->k_sel : nullptr, true),
                  "topk_union launch");
  return HERALD_OK;
}

herald_status check_budget(int C, int K, int sink, int local, int P_max) {
  if (K < 0 || sink < 0 || local < 0)
    return fail(HERALD_ERR_INVALID_ARG, "K=%d sink=%d local=%d must be >= 0", K, sink, local);
  if (K > C) return fail(HERALD_ERR_INVALID_ARG, "K=%d > C=%d", K, C);
  if ((long long)K + sink + local > P_max)
    return fail(HERALD_ERR_INVALID_ARG, "P_max=%d < K+sink+local=%lld", P_max,
                (long long)K + sink + local);
  return HERALD_OK;
}

herald_status check_pmax(const herald_dims& dm, int P_max) {
  if (P_max < 1) return fail(HERALD_ERR_INVALID_ARG, "P_max=%d must be >= 1", P_max);
  if ((long long)dm.N * dm.Hkv * P_max >= (1ll << 31))
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "N*Hkv*P_max too large");
  return HERALD_OK;
}

#define HERALD_RET_IF(x)              \
  do {                                \
    herald_status s_ = (x);           \
    if (s_ != HERALD_OK) return s_;   \
  } while (0)

// ---- kernel tracing state (per host thread)
struct TraceState {
  cudaEvent_t* events = nullptr;
  int capacity = 0;
  int count = 0;
  bool external = false;
  bool in_kernel = false;
  std::vector<const char*> names;
};
thread_local TraceState g_trace;

}  // namespace

namespace herald {

// [tokens][heads][d] with a box of 64 columns x box_heads heads x box_tokens
// tokens (query tiles and block keys / values of one KV head).
herald_status encode_heads_map(const void* base, uint64_t tokens, int heads, int d,
                               uint32_t box_heads, uint32_t box_tokens, CUtensorMap* map) {
  const uint64_t ext[3] = {uint64_t(d), uint64_t(heads), tokens};
  const uint32_t box[3] = {64, box_heads, box_tokens};
  return encode_map3(base, ext, box, map);
}

void set_last_error(const char* msg) { snprintf(g_err, sizeof g_err, "%s", msg); }

herald_status check_stage2_args(const herald_dims& dims, int C, int K, int sink, int local,
                                int P_max) {
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  return check_budget(C, K, sink, local, P_max);
}

bool device_resident(const void* p) { return is_device_memory(p); }

// herald_inject_launch_failure's state, per host thread: the number of
// launches still to pass (-1: disarmed) and the error the next one returns
thread_local int g_inject_after = -1;
thread_local cudaError_t g_inject_error = cudaSuccess;

cudaError_t injected_launch_error() {
  if (g_inject_after < 0) return cudaSuccess;
  if (g_inject_after-- > 0) return cudaSuccess;
  return g_inject_error;  // this launch fails; the hook is now disarmed (-1)
}

cudaError_t ensure_smem(const void* fn, size_t bytes) {
  // (a kernel's static shared memory counts against the default 48 KB too,
  // so every nonzero dynamic amount is granted explicitly)
  if (bytes == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // a per-thread memo of recent grants in front of the shared record, so
  // the steady state takes no lock
  struct Memo {
    const void* fn;
    int dev;
    size_t bytes;
  };
  constexpr int kMemo = 16;
  thread_local Memo memo[kMemo] = {};
  thread_local int next = 0;
  for (const Memo& m : memo)
    if (m.fn == fn && m.dev == dev && m.bytes >= bytes) return cudaSuccess;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> granted;
  size_t now;
  {
    std::lock_guard<std::mutex> lock(mu);
    size_t& g = granted[{fn, dev}];
    if (g < bytes) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
      if (e != cudaSuccess) return e;
      g = bytes;
    }
    now = g;
  }
  memo[next] = Memo{fn, dev, now};
  next = (next + 1) % kMemo;
  return cudaSuccess;
}

cudaError_t ensure_nonportable_cluster(const void* fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  constexpr int kMemo = 8;
  thread_local std::pair<const void*, int> memo[kMemo] = {};
  thread_local int next = 0;
  for (const auto& m : memo)
    if (m.first == fn && m.second == dev) return cudaSuccess;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> allowed;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!allowed.count({fn, dev})) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      allowed.insert({fn, dev});
    }
  }
  memo[next] = {fn, dev};
  next = (next + 1) % kMemo;
  return cudaSuccess;
}

void trace_before(cudaStream_t st, const char* name) {
  TraceState& t = g_trace;
  t.in_kernel = false;
  if (!t.events || t.count >= t.capacity) return;
  t.names[t.count] = name;
  if (t.external)
    cudaEventRecordWithFlags(t.events[2 * t.count], st, cudaEventRecordExternal);
  else
    cudaEventRecord(t.events[2 * t.count], st);
  t.in_kernel = true;
}

void trace_after(cudaStream_t st) {
  TraceState& t = g_trace;
  if (!t.in_kernel) return;
  if (t.external)
    cudaEventRecordWithFlags(t.events[2 * t.count + 1], st, cudaEventRecordExternal);
  else
    cudaEventRecord(t.events[2 * t.count + 1], st);
  t.in_kernel = false;
  ++t.count;
}

}  // namespace herald

extern "C" {

herald_status herald_trace_begin(void** events, int capacity, int external) {
  if (!events || capacity < 1) return fail(HERALD_ERR_INVALID_ARG, "trace needs >= 1 event pair");
  g_trace.events = reinterpret_cast<cudaEvent_t*>(events);
  g_trace.capacity = capacity;
  g_trace.count = 0;
  g_trace.external = external != 0;
  g_trace.in_kernel = false;
  g_trace.names.assign(size_t(capacity), nullptr);
  return HERALD_OK;
}

int herald_trace_end(void) {
  const int n = g_trace.count;
  g_trace.events = nullptr;
  return n;
}

const char* herald_trace_name(int i) {
  if (i < 0 || i >= int(g_trace.names.size()) || !g_trace.names[size_t(i)]) return "";
  return g_trace.names[size_t(i)];
}

size_t herald_workspace_size(herald_dims dims, int C, int P_max) {
  if (check_dims(dims) != HERALD_OK || check_c(C) != HERALD_OK || P_max < 1) return 0;
  return ws_layout(dims, C, P_max).total;
}

const char* herald_status_string(herald_status s) {
  switch (s) {
    case HERALD_OK: return "ok";
    case HERALD_ERR_INVALID_ARG: return "invalid argument";
    case HERALD_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case HERALD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case HERALD_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* herald_last_error(void) { return g_err; }

int herald_debug_build(void) {
#ifdef HERALD_DEBUG
  return 1;
#else
  return 0;
#endif
}

herald_status herald_debug_status(uint32_t* code) {
  if (!code) return fail(HERALD_ERR_INVALID_ARG, "code is NULL");
  *code = 0;
#ifdef HERALD_DEBUG
  HERALD_TRY_CUDA(cudaDeviceSynchronize(), "device synchronize");
  *code = debug_take_select() | debug_take_tc() | debug_take_move() | debug_take_blocks() |
          debug_take_flash();
#endif
  return HERALD_OK;
}

herald_status herald_inject_launch_failure(int after, int cuda_error) {
  if (after >= 0 && cuda_error == 0)
    return fail(HERALD_ERR_INVALID_ARG, "the injected error must be a CUDA error code");
  g_inject_after = after < 0 ? -1 : after;
  g_inject_error = static_cast<cudaError_t>(cuda_error);
  return HERALD_OK;
}

herald_status herald_workspace_error(void* ws, void* stream, uint32_t* code) {
  HERALD_CHECK_PTR(ws);
  if (!code) return fail(HERALD_ERR_INVALID_ARG, "code is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  HERALD_TRY_CUDA(cudaStreamSynchronize(st), "stream synchronize");
  uint32_t v = 0;
  HERALD_TRY_CUDA(cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost), "read error word");
  *code = v;
  if (v) HERALD_TRY_CUDA(cudaMemsetAsync(ws, 0, sizeof v, st), "clear error word");
  return HERALD_OK;
}

// Workspace of the exact selection: error word, histograms, the top-K
// positions, counts, refine row statistics over every cached position, and
// the score partials [parts][N*Hkv][L_pad].
struct ExactLayout {
  size_t err, hist, cand, n_cand, rpart, rlse, s, total;
};
static ExactLayout exact_layout(const herald_dims& dm, int K, const WsLayout& w) {
  ExactLayout x{};
  const size_t A = 256, NG = size_t(dm.N) * dm.Hkv;
  size_t o = 0;
  x.err = o;    o = align_up(o + 16, A);
  x.hist = o;   o = align_up(o + NG * kHistBins * 4, A);
  x.cand = o;   o = align_up(o + NG * size_t(K) * 4, A);
  x.n_cand = o; o = align_up(o + NG * 4, A);
  x.rpart = o;  o = align_up(o + NG * size_t(w.MT) * kTileM * w.n_chunks * 8, A);
  x.rlse = o;   o = align_up(o + NG * size_t(w.MT) * kTileM * 4, A);
  x.s = o;      o = align_up(o + NG * size_t(w.L_pad) * 4 * std::max(w.MT, w.MT_tok), A);
  x.total = o;
  return x;
}

size_t herald_workspace_size_exact(herald_dims dims, int K, int P_max) {
  if (check_dims(dims) != HERALD_OK || K < 1 || K > kMaxC || P_max < 1) return 0;
  const WsLayout w = ws_layout(dims, cdiv(dims.L_max, kTcScanKeys) * kTcScanKeys, P_max);
  return exact_layout(dims, K, w).total;
}

herald_status herald_select_exact(herald_dims dims, const uint16_t* q_block,
                                  const uint16_t* k_cache, const int32_t* ctx_len, int K,
                                  int sink, int local, int P_max, int32_t* idx, int32_t* n_sel,
                                  void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_pmax(dims, P_max));
  if (K < 1 || K > kMaxC)
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "K=%d outside [1, %d]", K, kMaxC);
  HERALD_RET_IF(check_budget(K, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  HERALD_CHECK_PTR(ws);
  const int L_pad = cdiv(dims.L_max, kTcScanKeys) * kTcScanKeys;
  const WsLayout w = ws_layout(dims, L_pad, P_max);  // tile counts of a refine over L_pad slots
  const ExactLayout x = exact_layout(dims, K, w);
  if (ws_bytes < x.total)
    return fail(HERALD_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes,
                x.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = at<uint32_t>(ws, x.err);
  int32_t* n_cand = at<int32_t>(ws, x.n_cand);
  float* s = at<float>(ws, x.s);
  uint32_t* hist = at<uint32_t>(ws, x.hist);
  CUtensorMap qmap, qmap_all;
  const int G = dims.Hq / dims.Hkv;
  HERALD_RET_IF(encode_heads_map(q_block, uint64_t(dims.N) * dims.B, dims.Hq, dims.d,
                                 uint32_t(G), uint32_t(kTileM / G), &qmap));
  HERALD_RET_IF(encode_heads_map(q_block, uint64_t(dims.N) * dims.B, dims.Hq, dims.d,
                                 uint32_t(G), uint32_t(dims.B), &qmap_all));
  HERALD_TRY_CUDA(cudaMemsetAsync(hist, 0, size_t(dims.N) * dims.Hkv * kHistBins * 4, st),
                  "clear histograms");
  HERALD_TRY_CUDA(launch_exact_counts(dims, ctx_len, n_cand, st), "exact counts launch");
  // every cached position is a candidate (row = slot, stride L_pad)
  HERALD_TRY_CUDA(launch_refine(dims, k_cache, nullptr, n_cand, L_pad,
                                at<float2>(ws, x.rpart), at<float>(ws, x.rlse), s, w, err,
                                &qmap, &qmap_all, st),
                  "refine launch");
  const int n_parts = refine_fused_ok(L_pad) ? w.MT_tok : 1;
  HERALD_TRY_CUDA(launch_exact_sum_hist(dims, s, n_parts, L_pad, ctx_len, hist, sm_count(), st),
                  "exact histogram launch");
  int32_t* cand = at<int32_t>(ws, x.cand);
  HERALD_TRY_CUDA(launch_topc(dims, s, hist, ctx_len, K, cand, n_cand, w, st), "top-K launch");
  // the K positions are all kept; the union adds sink and local and orders
  HERALD_TRY_CUDA(launch_topk_union(dims, ctx_len, cand, n_cand, s, 1, K, K, sink, local, P_max,
                                    idx, n_sel, st),
                  "union launch");
  return HERALD_OK;
}

herald_status herald_selftest_wait_timeout(uint64_t limit_ns, void* ws, void* stream) {
  g_err[0] = 0;
  HERALD_CHECK_PTR(ws);
  if (limit_ns == 0 || limit_ns > 1000000000ull)
    return fail(HERALD_ERR_INVALID_ARG, "limit_ns=%llu outside (0, 1e9]",
                (unsigned long long)limit_ns);
  HERALD_TRY_CUDA(launch_wait_timeout(limit_ns, static_cast<uint32_t*>(ws),
                                      static_cast<cudaStream_t>(stream)),
                  "timeout self-test launch");
  return HERALD_OK;
}

herald_status herald_select_stage1(herald_dims dims, const uint16_t* q_merge,
                                   const uint16_t* k_cache, const int32_t* ctx_len, int C,
                                   int32_t* cand, int32_t* n_cand, void* ws, size_t ws_bytes,
                                   int sm_budget, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  if (sm_budget < 0) return fail(HERALD_ERR_INVALID_ARG, "sm_budget=%d must be >= 0", sm_budget);
  HERALD_CHECK_PTR(q_merge);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, 1, ws, ws_bytes, &w));
  return run_stage1(dims, q_merge, k_cache, ctx_len, C, cand, n_cand, ws, w, sm_budget,
                    static_cast<cudaStream_t>(stream));
}

herald_status herald_pool_keys(herald_dims dims, const uint16_t* k_cache,
                               const int32_t* ctx_len, int Bk, int n_tail, float* pooled,
                               void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  if (Bk < 1 || Bk > dims.L_max) return fail(HERALD_ERR_INVALID_ARG, "Bk=%d outside [1, L_max]", Bk);
  if (n_tail < 0) return fail(HERALD_ERR_INVALID_ARG, "n_tail=%d must be >= 0", n_tail);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(pooled);
  HERALD_TRY_CUDA(launch_pool_keys(dims, k_cache, ctx_len, Bk, n_tail, pooled,
                                   static_cast<cudaStream_t>(stream)),
                  "pool_keys launch");
  return HERALD_OK;
}

herald_status herald_select_stage1_blocks(herald_dims dims, const uint16_t* q_merge,
                                          const float* pooled, const int32_t* ctx_len, int Bk,
                                          int C_blocks, int32_t* cand, int32_t* n_cand, void* ws,
                                          size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  if (Bk < 1 || Bk > dims.L_max) return fail(HERALD_ERR_INVALID_ARG, "Bk=%d outside [1, L_max]", Bk);
  if (C_blocks < 1 || (long long)C_blocks * Bk > kMaxC)
    return fail(HERALD_ERR_UNSUPPORTED_SHAPE, "C_blocks*Bk=%lld outside [1, %d]",
                (long long)C_blocks * Bk, kMaxC);
  HERALD_CHECK_PTR(q_merge);
  HERALD_CHECK_PTR(pooled);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  // the selection runs over the blocks: the per-key stage 1's workspace
  // layout for a cache of ceil(L_max/Bk) rows and C_blocks candidates
  herald_dims bd = dims;
  bd.L_max = cdiv(dims.L_max, Bk);
  WsLayout w;
  HERALD_RET_IF(check_ws(bd, C_blocks, 1, ws, ws_bytes, &w));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int chunks = block_scan_chunks(bd, sm_count());
  const int part_slots = chunks * 4;
  float* qbar = at<float>(ws, w.qbar);
  float2* part1 = at<float2>(ws, w.part1);
  uint32_t* hist = at<uint32_t>(ws, w.hist);
  int32_t* cand_b = at<int32_t>(ws, w.cand);
  int32_t* n_cand_b = at<int32_t>(ws, w.n_cand);
  // block counts ceil(ctx/Bk), written by the block scan, read by the rest
  int32_t* ctx_b = at<int32_t>(ws, w.s2);
  HERALD_TRY_CUDA(launch_merge_query(dims, q_merge, qbar, at<uint16_t>(ws, w.qhl), hist, part1,
                                     part_slots, st),
                  "merge_query launch");
  HERALD_TRY_CUDA(launch_block_scan(dims, pooled, qbar, ctx_len, Bk, w.L_pad,
                                    at<float>(ws, w.logits), part1, ctx_b, chunks, st),
                  "block_scan launch");
  HERALD_TRY_CUDA(launch_s1_hist(bd, at<float>(ws, w.logits), part1, part_slots, ctx_b,
                                 at<float>(ws, w.s1), hist, w, sm_count(), st),
                  "s1_hist launch");
  HERALD_TRY_CUDA(launch_topc(bd, at<float>(ws, w.s1), hist, ctx_b, C_blocks, cand_b, n_cand_b,
                              w, st),
                  "topc launch");
  HERALD_TRY_CUDA(launch_expand_blocks(dims, cand_b, n_cand_b, ctx_len, Bk, C_blocks, cand,
                                       n_cand, st),
                  "expand launch");
  return HERALD_OK;
}

herald_status herald_select_stage2(herald_dims dims, const uint16_t* q_block,
                                   const uint16_t* k_cache, const int32_t* ctx_len,
                                   const int32_t* cand, const int32_t* n_cand, int C, int K,
                                   int sink, int local, int P_max, int32_t* idx, int32_t* n_sel,
                                   void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, ws, ws_bytes, &w));
  return run_stage2(dims, q_block, k_cache, ctx_len, cand, n_cand, C, K, sink, local, P_max, idx,
                    n_sel, ws, w, static_cast<cudaStream_t>(stream), nullptr);
}

// The gather rides with the top-K when there are many (sequence, KV head)
// pairs: each then has a few top-K CTAs, one per slice of its pool.  With few
// pairs the separate wide gather kernel measured faster (32K layer, 4 pairs:
// 91.7 against 93.3 us per block at 8 copies, 101.5 at 16; 4 x 64K layer,
// 32 pairs: 503.5 against 518.5 us at 4 copies, 505.6 at 8).  At least two
// copies per pair (fewer than half as many pairs as SMs): one CTA gathering a
// whole pool is not measured.
constexpr int kFusedGatherMinSegs = 16;
constexpr int kFusedGatherMaxCopies = 4;

static herald_status stage2_gather(herald_dims dims, const uint16_t* q_block,
                                   const uint16_t* k_cache, const uint16_t* v_cache,
                                   const int32_t* ctx_len, const int32_t* cand,
                                   const int32_t* n_cand, int C, int K, int sink, int local,
                                   int P_max, int32_t* idx, int32_t* n_sel, uint16_t* pool_k,
                                   uint16_t* pool_v, void* ws, size_t ws_bytes, void* stream,
                                   bool cand_settled) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(v_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  HERALD_CHECK_PTR(pool_k);
  HERALD_CHECK_PTR(pool_v);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, ws, ws_bytes, &w));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool on_device = is_device_memory(k_cache) && is_device_memory(v_cache);
  const int segs = dims.N * dims.Hkv;
  const int copies = std::min(kFusedGatherMaxCopies, sm_count() / segs);
  if (segs >= kFusedGatherMinSegs && copies >= 2 && on_device) {
    const PoolGather pg{k_cache, v_cache, pool_k, pool_v, dims.d, copies};
    return run_stage2(dims, q_block, k_cache, ctx_len, cand, n_cand, C, K, sink, local, P_max,
                      idx, n_sel, ws, w, st, &pg, nullptr, nullptr, nullptr, cand_settled);
  }
  // a cache in host memory: the wide gather kernel keeps the host link busy
  HERALD_RET_IF(run_stage2(dims, q_block, k_cache, ctx_len, cand, n_cand, C, K, sink, local,
                           P_max, idx, n_sel, ws, w, st, nullptr, nullptr, nullptr, nullptr,
                           cand_settled));
  HERALD_TRY_CUDA(launch_gather(dims, idx, n_sel, P_max, k_cache, v_cache, pool_k, pool_v, st),
                  "gather launch");
  return HERALD_OK;
}

herald_status herald_select_stage2_gather(herald_dims dims, const uint16_t* q_block,
                                          const uint16_t* k_cache, const uint16_t* v_cache,
                                          const int32_t* ctx_len, const int32_t* cand,
                                          const int32_t* n_cand, int C, int K, int sink,
                                          int local, int P_max, int32_t* idx, int32_t* n_sel,
                                          uint16_t* pool_k, uint16_t* pool_v, void* ws,
                                          size_t ws_bytes, void* stream) {
  return stage2_gather(dims, q_block, k_cache, v_cache, ctx_len, cand, n_cand, C, K, sink, local,
                       P_max, idx, n_sel, pool_k, pool_v, ws, ws_bytes, stream, false);
}

// CTAs of the background candidate copy.  Each one holds an SM that an
// attention CTA (all of an SM's registers) then cannot use; the copy is
// bounded by the host link, not by SMs.  128K host-resident layer, block
// stage 1, per block: K rows 378 / 344 / 344 us at 128 / 64 / 32 CTAs, K and
// V rows 384 / 327 / 330 us.
constexpr int kStageCtas = 64;

herald_status herald_stage_candidates(herald_dims dims, const uint16_t* k_cache,
                                      const uint16_t* v_cache, const int32_t* cand,
                                      const int32_t* n_cand, int C, uint16_t* staged_k,
                                      uint16_t* staged_v, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  HERALD_CHECK_PTR(staged_k);
  if ((v_cache == nullptr) != (staged_v == nullptr))
    return fail(HERALD_ERR_INVALID_ARG, "v_cache and staged_v must both be given or both null");
  // a bounded grid: the copy runs beside the denoising kernels and is held
  // by the host link, not by SMs
  HERALD_TRY_CUDA(launch_gather(dims, cand, n_cand, C, k_cache, v_cache, staged_k, staged_v,
                                static_cast<cudaStream_t>(stream),
                                "gather_kernel (candidate staging)", kStageCtas),
                  "candidate staging launch");
  return HERALD_OK;
}

herald_status herald_select_stage2_staged(herald_dims dims, const uint16_t* q_block,
                                          const uint16_t* staged_k, const int32_t* ctx_len,
                                          const int32_t* cand, const int32_t* n_cand, int C,
                                          int K, int sink, int local, int P_max, int32_t* idx,
                                          int32_t* n_sel, void* ws, size_t ws_bytes,
                                          void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(staged_k);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, ws, ws_bytes, &w));
  return run_stage2(dims, q_block, staged_k, ctx_len, cand, n_cand, C, K, sink, local, P_max,
                    idx, n_sel, ws, w, static_cast<cudaStream_t>(stream), nullptr, staged_k);
}

herald_status herald_select_stage2_staged_gather(
    herald_dims dims, const uint16_t* q_block, const uint16_t* staged_k, const uint16_t* staged_v,
    const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* ctx_len, const int32_t* cand,
    const int32_t* n_cand, int C, int K, int sink, int local, int P_max, int32_t* idx,
    int32_t* n_sel, uint16_t* pool_k, uint16_t* pool_v, void* ws, size_t ws_bytes,
    void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(staged_k);
  HERALD_CHECK_PTR(staged_v);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(v_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  HERALD_CHECK_PTR(pool_k);
  HERALD_CHECK_PTR(pool_v);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, ws, ws_bytes, &w));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* slot = at<int32_t>(ws, w.slot);
  HERALD_RET_IF(run_stage2(dims, q_block, staged_k, ctx_len, cand, n_cand, C, K, sink, local,
                           P_max, idx, n_sel, ws, w, st, nullptr, staged_k, slot));
  // the top-K rows from the staged candidates (HBM), the sink and local rows
  // from the cache
  HERALD_TRY_CUDA(launch_gather_staged(dims, idx, n_sel, P_max, slot, C, staged_k, staged_v,
                                       k_cache, v_cache, pool_k, pool_v, st),
                  "staged gather launch");
  return HERALD_OK;
}

herald_status herald_select_stage2_adaptive(herald_dims dims, const uint16_t* q_block,
                                           const uint16_t* k_cache, const int32_t* ctx_len,
                                           const int32_t* cand, const int32_t* n_cand, int C,
                                           int K_min, int K_max, float tau, int sink, int local,
                                           int P_max, int32_t* idx, int32_t* n_sel,
                                           int32_t* k_sel, void* ws, size_t ws_bytes,
                                           void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K_max, sink, local, P_max));
  if (K_min < 0 || K_min > K_max)
    return fail(HERALD_ERR_INVALID_ARG, "K_min=%d must lie in [0, K_max=%d]", K_min, K_max);
  if (!(tau > 0.f && tau <= 1.f))
    return fail(HERALD_ERR_INVALID_ARG, "tau=%g must lie in (0, 1]", double(tau));
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(cand);
  HERALD_CHECK_PTR(n_cand);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  HERALD_CHECK_PTR(k_sel);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, ws, ws_bytes, &w));
  const BudgetArgs b{K_min, K_max, tau, k_sel};
  return run_stage2(dims, q_block, k_cache, ctx_len, cand, n_cand, C, K_max, sink, local, P_max,
                    idx, n_sel, ws, w, static_cast<cudaStream_t>(stream), nullptr, nullptr,
                    nullptr, &b);
}

herald_status herald_select(herald_dims dims, const uint16_t* q_merge, const uint16_t* q_block,
                            const uint16_t* k_cache, const int32_t* ctx_len, int C, int K,
                            int sink, int local, int P_max, int32_t* idx, int32_t* n_sel,
                            void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_merge);
  HERALD_CHECK_PTR(q_block);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, ws, ws_bytes, &w));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* cand = at<int32_t>(ws, w.cand);
  int32_t* n_cand = at<int32_t>(ws, w.n_cand);
  HERALD_RET_IF(run_stage1(dims, q_merge, k_cache, ctx_len, C, cand, n_cand, ws, w, 0, st));
  return run_stage2(dims, q_block, k_cache, ctx_len, cand, n_cand, C, K, sink, local, P_max, idx,
                    n_sel, ws, w, st, nullptr);
}

herald_status herald_gather(herald_dims dims, const int32_t* idx, const int32_t* n_sel,
                            int P_max, const uint16_t* k_cache, const uint16_t* v_cache,
                            uint16_t* pool_k, uint16_t* pool_v, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_CHECK_PTR(idx);
  HERALD_CHECK_PTR(n_sel);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(v_cache);
  HERALD_CHECK_PTR(pool_k);
  HERALD_CHECK_PTR(pool_v);
  HERALD_TRY_CUDA(launch_gather(dims, idx, n_sel, P_max, k_cache, v_cache, pool_k, pool_v,
                                static_cast<cudaStream_t>(stream)),
                  "gather launch");
  return HERALD_OK;
}

}  // extern "C"

namespace {
herald_status denoise_attn(herald_dims dims, const uint16_t* q, const uint16_t* pool_k,
                           const uint16_t* pool_v, const int32_t* n_sel, int P_max,
                           const uint16_t* block_k, const uint16_t* block_v, uint16_t* out,
                           float scale, unsigned flags, int32_t* ctx_len, uint16_t* k_cache,
                           uint16_t* v_cache, void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  constexpr unsigned kKnown =
      HERALD_ATTN_SETTLED | HERALD_ATTN_APPEND | HERALD_ATTN_ADVANCE | (0xFu << 8) | (0xFFu << 16);
  if (flags & ~kKnown) return fail(HERALD_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~kKnown);
  const unsigned kernel = (flags >> 8) & 0xFu;
  if (kernel > (HERALD_ATTN_KERNEL_POOL_CS12 >> 8))
    return fail(HERALD_ERR_INVALID_ARG, "unknown kernel choice %u", kernel);
  const bool append = (flags & HERALD_ATTN_APPEND) != 0;
  if ((flags & HERALD_ATTN_ADVANCE) && !append)
    return fail(HERALD_ERR_INVALID_ARG, "HERALD_ATTN_ADVANCE needs HERALD_ATTN_APPEND");
  if (append) {
    HERALD_CHECK_PTR(ctx_len);
    HERALD_CHECK_PTR(k_cache);
    HERALD_CHECK_PTR(v_cache);
  }
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_CHECK_PTR(q);
  HERALD_CHECK_PTR(pool_k);
  HERALD_CHECK_PTR(pool_v);
  HERALD_CHECK_PTR(n_sel);
  HERALD_CHECK_PTR(block_k);
  HERALD_CHECK_PTR(block_v);
  HERALD_CHECK_PTR(out);
  if (!(scale >= 0.f) || isinf(scale)) return fail(HERALD_ERR_INVALID_ARG, "scale must be finite and >= 0");
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, 1, P_max, ws, ws_bytes, &w));
  if (scale == 0.f) scale = 1.0f / sqrtf(float(dims.d));
  PoolMaps maps;
  const int sm_budget = int((flags >> 16) & 0xFFu) * 4;  // HERALD_ATTN_SMS
  const int pool_cs = attn_pool_cs(dims, P_max, int(kernel), sm_budget);
  const bool pool_ok = pool_cs > 0, flash_ok = attn_flash_ok(dims);
  const bool pool = pool_ok || flash_ok;
  maps.pool_cs = pool_cs;
  maps.sm_budget = sm_budget;
  if (pool) {
    const uint64_t rows = uint64_t(dims.N) * dims.Hkv * P_max;
    if (pool_ok) {
      const uint32_t box = uint32_t(attn_pool_kpc(P_max, dims.B, pool_cs));
      HERALD_RET_IF(encode_rows_map(pool_k, rows, dims.d, box, &maps.k));
      HERALD_RET_IF(encode_rows_map(pool_v, rows, dims.d, box, &maps.v));
    }
    if (flash_ok) {
      HERALD_RET_IF(encode_rows_map(pool_k, rows, dims.d, kFlashTileKeys, &maps.kt));
      HERALD_RET_IF(encode_rows_map(pool_v, rows, dims.d, kFlashTileKeys, &maps.vt));
    }
    maps.bpt = attn_pool_bpt(dims);
    const int G = dims.Hq / dims.Hkv, Bp = (dims.B + 15) & ~15;
    const uint64_t tokens = uint64_t(dims.N) * dims.B;
    HERALD_RET_IF(encode_heads_map(q, tokens, dims.Hq, dims.d, uint32_t(G),
                                   uint32_t(maps.bpt), &maps.q));
    HERALD_RET_IF(encode_heads_map(block_k, tokens, dims.Hkv, dims.d, 1u, uint32_t(Bp),
                                   &maps.bk));
    HERALD_RET_IF(encode_heads_map(block_v, tokens, dims.Hkv, dims.d, 1u, uint32_t(Bp),
                                   &maps.bv));
  }
  // the append rides along with the step when the cache is in device memory
  // (its stores stay on the device); a host-resident cache gets the append
  // kernel after it
  const bool fused = append && is_device_memory(k_cache) && is_device_memory(v_cache);
  const AppendArgs app{block_k, block_v, ctx_len, k_cache, v_cache,
                       (flags & HERALD_ATTN_ADVANCE) ? 1 : 0};
  HERALD_TRY_CUDA(launch_attn(dims, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale,
                              w, at<float>(ws, w.opart), at<float2>(ws, w.ml),
                              at<uint32_t>(ws, w.err), pool ? &maps : nullptr,
                              (flags & HERALD_ATTN_SETTLED) != 0, fused ? &app : nullptr,
                              int(kernel) | (pool_ok ? 0x100 : 0) | (flash_ok ? 0x200 : 0),
                              static_cast<cudaStream_t>(stream)),
                  "attention launch");
  if (append && !fused)  // a cache in host memory: the append kernel after the step
    HERALD_TRY_CUDA(launch_append(dims, block_k, block_v, ctx_len, k_cache, v_cache,
                                  (flags & HERALD_ATTN_ADVANCE) != 0,
                                  static_cast<cudaStream_t>(stream)),
                    "append launch");
  return HERALD_OK;
}
}  // namespace

extern "C" {

herald_status herald_denoise_attn(herald_dims dims, const uint16_t* q, const uint16_t* pool_k,
                                  const uint16_t* pool_v, const int32_t* n_sel, int P_max,
                                  const uint16_t* block_k, const uint16_t* block_v,
                                  uint16_t* out, float scale, void* ws, size_t ws_bytes,
                                  void* stream) {
  return denoise_attn(dims, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale, 0u,
                      nullptr, nullptr, nullptr, ws, ws_bytes, stream);
}

herald_status herald_denoise_attn_ex(herald_dims dims, const uint16_t* q, const uint16_t* pool_k,
                                     const uint16_t* pool_v, const int32_t* n_sel, int P_max,
                                     const uint16_t* block_k, const uint16_t* block_v,
                                     uint16_t* out, float scale, unsigned flags,
                                     int32_t* ctx_len, uint16_t* k_cache, uint16_t* v_cache,
                                     void* ws, size_t ws_bytes, void* stream) {
  return denoise_attn(dims, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale, flags,
                      ctx_len, k_cache, v_cache, ws, ws_bytes, stream);
}

herald_status herald_append_kv(herald_dims dims, const uint16_t* block_k, const uint16_t* block_v,
                               int32_t* ctx_len, uint16_t* k_cache, uint16_t* v_cache,
                               int advance, void* stream) {
  g_err[0] = 0;
  HERALD_RET_IF(check_dims(dims));
  HERALD_CHECK_PTR(block_k);
  HERALD_CHECK_PTR(block_v);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(v_cache);
  HERALD_TRY_CUDA(launch_append(dims, block_k, block_v, ctx_len, k_cache, v_cache, advance,
                                static_cast<cudaStream_t>(stream)),
                  "append launch");
  return HERALD_OK;
}

// One block of the dual-stream pipeline: the calls a host loop would issue
// for it, with the stream fork and join, in one call (a block is T + 2
// library calls and two event operations; issued from here they cost the
// launches' host time and nothing else).
herald_status herald_block(herald_dims dims, int C, int K, int sink, int local, int P_max, int T,
                           int i, const uint16_t* q_steps, const uint16_t* block_k,
                           const uint16_t* block_v, uint16_t* k_cache, uint16_t* v_cache,
                           int32_t* ctx_len, const uint16_t* next_k_cache, uint16_t* out,
                           unsigned flags, int scan_sms, const herald_block_bufs* bufs,
                           void* stream) {
  g_err[0] = 0;
  constexpr unsigned kBlockFlags = HERALD_BLOCK_ADVANCE | HERALD_BLOCK_CAND_SETTLED;
  if (flags & ~kBlockFlags)
    return fail(HERALD_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags & ~kBlockFlags);
  if (T < 1) return fail(HERALD_ERR_INVALID_ARG, "T=%d must be >= 1", T);
  if (i < 0) return fail(HERALD_ERR_INVALID_ARG, "i=%d must be >= 0", i);
  if (scan_sms < 0) return fail(HERALD_ERR_INVALID_ARG, "scan_sms=%d must be >= 0", scan_sms);
  if (bufs == nullptr) return fail(HERALD_ERR_INVALID_ARG, "bufs is NULL");
  const bool overlap = bufs->sel_stream != nullptr;
  if (overlap && (bufs->ev_fork == nullptr || bufs->ev_join == nullptr))
    return fail(HERALD_ERR_INVALID_ARG, "sel_stream needs ev_fork and ev_join");
  // everything the calls below check before they launch, checked before
  // the first of them launches
  HERALD_RET_IF(check_dims(dims));
  HERALD_RET_IF(check_c(C));
  HERALD_RET_IF(check_pmax(dims, P_max));
  HERALD_RET_IF(check_budget(C, K, sink, local, P_max));
  HERALD_CHECK_PTR(q_steps);
  HERALD_CHECK_PTR(block_k);
  HERALD_CHECK_PTR(block_v);
  HERALD_CHECK_PTR(k_cache);
  HERALD_CHECK_PTR(v_cache);
  HERALD_CHECK_PTR(ctx_len);
  HERALD_CHECK_PTR(out);
  if (next_k_cache != nullptr) HERALD_CHECK_PTR(next_k_cache);
  const int cur = i & 1, nxt = cur ^ 1;
  HERALD_CHECK_PTR(bufs->cand[0]);
  HERALD_CHECK_PTR(bufs->cand[1]);
  HERALD_CHECK_PTR(bufs->n_cand[0]);
  HERALD_CHECK_PTR(bufs->n_cand[1]);
  HERALD_CHECK_PTR(bufs->idx);
  HERALD_CHECK_PTR(bufs->n_sel);
  HERALD_CHECK_PTR(bufs->pool_k[cur]);
  HERALD_CHECK_PTR(bufs->pool_v[cur]);
  WsLayout w;
  HERALD_RET_IF(check_ws(dims, C, P_max, bufs->ws_den, bufs->ws_bytes, &w));
  HERALD_RET_IF(check_ws(dims, C, P_max, bufs->ws_sel, bufs->ws_bytes, &w));

  const cudaStream_t den = static_cast<cudaStream_t>(stream);
  const cudaStream_t sel = overlap ? static_cast<cudaStream_t>(bufs->sel_stream) : den;
  const cudaEvent_t fork = static_cast<cudaEvent_t>(bufs->ev_fork);
  const cudaEvent_t join = static_cast<cudaEvent_t>(bufs->ev_join);
  const size_t q_step = size_t(dims.N) * dims.B * dims.Hq * dims.d;
  const size_t kv_step = size_t(dims.N) * dims.B * dims.Hkv * dims.d;
  // stage 1 for block i+1 may start now: block i's queries exist
  if (overlap) {
    HERALD_TRY_CUDA(cudaEventRecord(fork, den), "fork event record");
    HERALD_TRY_CUDA(cudaStreamWaitEvent(sel, fork, 0), "fork event wait");
  }
  HERALD_RET_IF(stage2_gather(dims, q_steps, k_cache, v_cache, ctx_len, bufs->cand[cur],
                              bufs->n_cand[cur], C, K, sink, local, P_max, bufs->idx, bufs->n_sel,
                              bufs->pool_k[cur], bufs->pool_v[cur], bufs->ws_den, bufs->ws_bytes,
                              den, (flags & HERALD_BLOCK_CAND_SETTLED) != 0));
  HERALD_RET_IF(herald_select_stage1(dims, q_steps, next_k_cache ? next_k_cache : k_cache,
                                     ctx_len, C, bufs->cand[nxt], bufs->n_cand[nxt], bufs->ws_sel,
                                     bufs->ws_bytes, overlap ? scan_sms : 0, sel));
  if (overlap) HERALD_TRY_CUDA(cudaEventRecord(join, sel), "join event record");
  // the SMs the scan leaves the steps, so that each step's clusters fit at once
  const int n_sm = sm_count();
  const unsigned sm_flags =
      (overlap && scan_sms > 0 && scan_sms < n_sm) ? HERALD_ATTN_SMS(n_sm - scan_sms) : 0u;
  for (int t = 0; t < T; ++t) {
    unsigned f = (t > 0 ? HERALD_ATTN_SETTLED : 0u) | sm_flags;
    if (t == T - 1) {
      // stage 1 reads the cache this step appends to
      if (overlap) HERALD_TRY_CUDA(cudaStreamWaitEvent(den, join, 0), "join event wait");
      f |= HERALD_ATTN_APPEND | ((flags & HERALD_BLOCK_ADVANCE) ? HERALD_ATTN_ADVANCE : 0u);
    }
    HERALD_RET_IF(denoise_attn(dims, q_steps + t * q_step, bufs->pool_k[cur], bufs->pool_v[cur],
                               bufs->n_sel, P_max, block_k + t * kv_step, block_v + t * kv_step,
                               out + t * q_step, 0.f, f, ctx_len, k_cache, v_cache, bufs->ws_den,
                               bufs->ws_bytes, den));
  }
  return HERALD_OK;
}

}  // extern "C"
