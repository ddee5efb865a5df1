// internal.cuh -- constants, workspace layout and kernel launchers shared by
// the translation units of libherald.so.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <algorithm>
#include <stdint.h>

#include "../../include/herald.h"

namespace herald {

// ---- stage-1 scan
constexpr int kScanTileKeys = 64;   // CUDA-core scan (host-resident caches): keys per tile
constexpr int kScanWarps = 4;       // warps per CTA, each with its own ring
constexpr int kScanStages = 3;      // stages per warp
constexpr int kTcScanKeys = 128;    // tensor-core scan: keys per tile (UMMA M)
constexpr int kTcScanStages = 4;    // TMA ring depth of the tensor-core scan
constexpr int kScanMaxCtas = 256;   // upper bound of either scan's persistent grid
constexpr int kPartSlots = kScanMaxCtas * 4;  // stage-1 (max, sumexp) slots: one per (CTA, warp)
constexpr int kQhlRows = 16;        // merged-query operand rows: 8 hi + 8 lo
// ---- stage-1 score histogram (bits [30:19] of a non-negative fp32)
constexpr int kHistBins = 4096;
constexpr int kHistShift = 19;
// ---- tensor-core tiles
constexpr int kTileM = 128;         // rows per UMMA tile (M)
constexpr int kRefineChunk = 256;   // candidates per stage-2 pass-1 CTA (N)
constexpr int kRefineRows2 = 128;   // candidates per stage-2 pass-2 CTA (M)
constexpr int kAttnKeys = 128;      // keys per attention split
constexpr int kMaxC = 16384;        // candidates held in shared memory by top-K

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Byte offsets of every region inside a caller-provided workspace.
struct WsLayout {
  size_t err;        // uint32 device error word
  size_t qbar;       // float [N][Hq][d]        merged queries, pre-scaled
  size_t qhl;        // bf16 [N*Hkv][16][d]     merged queries as hi/lo bf16 rows
  size_t logits;     // float [N][Hq][L_pad]    stage-1 logits; in stage 2 the same
                     // bytes hold bf16 [N*Hkv][C][d] candidate K rows staged from
                     // a host-resident cache (the region has room for both)
  size_t part1;      // float2 [N][Hq][kPartSlots] per-(CTA, warp) (max, sumexp)
  size_t s1;         // float [N][Hkv][L_pad]   stage-1 scores
  size_t hist;       // uint32 [N*Hkv][kHistBins]
  size_t cand;       // int32 [N][Hkv][C]       (herald_select only)
  size_t n_cand;     // int32 [N][Hkv]
  size_t rpart;      // float2 [N][Hkv][R_pad][n_chunks]  refine row stats
  size_t rlse;       // float [N][Hkv][R_pad]   refine row log-sum-exp (two-pass refine)
  size_t s2;         // float [MT][N][Hkv][C] stage-2 score partials
  size_t opart;      // float [N*Hkv][MT][S][128][d]      attention partials
  size_t ml;         // float2 [N*Hkv][MT][S][128]
  size_t slot;       // int32 [N][Hkv][P_max]   candidate slot per selected row
  size_t total;
  int L_pad, tiles_per_seg, tiles128, R, MT, n_chunks, splits;
  int MT_tok;        // row tiles of whole tokens (floor(128 / G) tokens each)
};

inline WsLayout ws_layout(const herald_dims& dm, int C, int P_max) {
  WsLayout w{};
  const size_t A = 256;
  const int G = dm.Hq / dm.Hkv;
  w.L_pad = cdiv(dm.L_max, kTcScanKeys) * kTcScanKeys;
  w.tiles_per_seg = w.L_pad / kScanTileKeys;
  w.tiles128 = w.L_pad / kTcScanKeys;
  w.R = dm.B * G;
  w.MT = cdiv(w.R, kTileM);
  w.MT_tok = cdiv(dm.B, kTileM / G);
  w.n_chunks = cdiv(C, kRefineChunk);
  w.splits = cdiv(P_max, kAttnKeys) + cdiv(dm.B, kAttnKeys);
  const size_t NH = size_t(dm.N) * dm.Hq, NG = size_t(dm.N) * dm.Hkv;
  size_t o = 0;
  w.err = o;    o = align_up(o + 16, A);
  w.qbar = o;   o = align_up(o + NH * dm.d * 4, A);
  w.qhl = o;    o = align_up(o + NG * kQhlRows * dm.d * 2, A);
  w.logits = o; o = align_up(o + std::max(NH * w.L_pad * 4, NG * size_t(C) * dm.d * 2), A);
  w.part1 = o;  o = align_up(o + NH * kPartSlots * 8, A);
  w.s1 = o;     o = align_up(o + NG * w.L_pad * 4, A);
  w.hist = o;   o = align_up(o + NG * kHistBins * 4, A);
  w.cand = o;   o = align_up(o + NG * C * 4, A);
  w.n_cand = o; o = align_up(o + NG * 4, A);
  w.rpart = o;  o = align_up(o + NG * size_t(w.MT) * kTileM * w.n_chunks * 8, A);
  w.rlse = o;   o = align_up(o + NG * size_t(w.MT) * kTileM * 4, A);
  w.s2 = o;     o = align_up(o + NG * C * 4 * size_t(std::max(w.MT, w.MT_tok)), A);  // per row tile
  w.opart = o;  o = align_up(o + NG * w.MT * size_t(w.splits) * kTileM * dm.d * 4, A);
  w.ml = o;     o = align_up(o + NG * w.MT * size_t(w.splits) * kTileM * 8, A);
  w.slot = o;   o = align_up(o + NG * size_t(P_max) * 4, A);
  w.total = o;
  return w;
}

// Sets the text returned by herald_last_error() on this host thread.
void set_last_error(const char* msg);

// The argument rules of herald_select_stage2 on shapes and counts (dims, C,
// P_max, K/sink/local against C and P_max); the message of a failure is
// set as herald_last_error().
herald_status check_stage2_args(const herald_dims& dims, int C, int K, int sink, int local,
                                int P_max);

// Whether p points into device memory (else mapped host memory: read over
// the host link).
bool device_resident(const void* p);

// Grants the kernel `fn` at least `bytes` of dynamic shared memory on the
// current device.  The attribute belongs to that device's context, so each
// grant is recorded per (kernel, device); safe to call from several host
// threads.
cudaError_t ensure_smem(const void* fn, size_t bytes);
// Allows a kernel's launches with clusters of more than 8 CTAs (once per
// kernel and device).
cudaError_t ensure_nonportable_cluster(const void* fn);
template <typename... A>
inline cudaError_t ensure_nonportable_cluster(void (*fn)(A...)) {
  return ensure_nonportable_cluster(reinterpret_cast<const void*>(fn));
}
template <typename... A>
inline cudaError_t ensure_smem(void (*fn)(A...), size_t bytes) {
  return ensure_smem(reinterpret_cast<const void*>(fn), bytes);
}

// The debug build's device check words, one per translation unit with
// kernels: each returns and clears its word (always 0 in release builds).
uint32_t debug_take_select();
uint32_t debug_take_tc();
uint32_t debug_take_move();
uint32_t debug_take_blocks();
uint32_t debug_take_flash();

// A launch failure injected on the host (herald_inject_launch_failure, a
// test hook of the error paths): returns the injected error for the launch
// it was armed for on this host thread, cudaSuccess otherwise.
cudaError_t injected_launch_error();

// ---- kernel tracing: when enabled on this host thread, every kernel launch
// is bracketed by two caller-owned CUDA events recorded on its stream.
void trace_before(cudaStream_t st, const char* name);
void trace_after(cudaStream_t st);

// Launches a kernel with programmatic stream serialisation (see
// griddep_wait in ptx.cuh), bracketed by the tracing hooks.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                     size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (const cudaError_t ie = injected_launch_error()) return ie;
  trace_before(st, name);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  trace_after(st);
  return e;
}

#define HERALD_CHECK_LAUNCH(x)             \
  do {                                     \
    const cudaError_t le_ = (x);           \
    if (le_ != cudaSuccess) return le_;    \
  } while (0)

// ---- launchers (return the launch error; the caller maps it to a status)
cudaError_t launch_merge_query(const herald_dims& dm, const uint16_t* q_merge, float* qbar,
                               uint16_t* qhl, uint32_t* hist, float2* part1, int part_slots,
                               cudaStream_t st);
// Grid of the scan for these shapes (persistent; bounded by kScanMaxCtas).
int scan_grid(const herald_dims& dm, const struct WsLayout& w, bool tensor_core, int num_sms);
// kmap: the key cache as [N*Hkv*L_max][d], box 64 x 128 rows, 128B swizzle;
// bmap: qhl as [N*Hkv*16][d], box 64 x 16 rows.  Without maps (host-resident
// caches) the CUDA-core scan runs instead.
cudaError_t launch_scan(const herald_dims& dm, const CUtensorMap* kmap, const CUtensorMap* bmap,
                        const uint16_t* k_cache, const float* qbar, const int32_t* ctx,
                        float* logits, float2* part1, const WsLayout& w, uint32_t* err,
                        int num_sms, cudaStream_t st);
cudaError_t launch_s1_hist(const herald_dims& dm, const float* logits, const float2* part1,
                           int part_slots, const int32_t* ctx, float* s1, uint32_t* hist,
                           const WsLayout& w, int num_sms, cudaStream_t st);
cudaError_t launch_topc(const herald_dims& dm, const float* s1, const uint32_t* hist,
                        const int32_t* ctx, int C, int32_t* cand, int32_t* n_cand,
                        const WsLayout& w, cudaStream_t st);
// Whether stage 2 runs as the fused cluster kernel for this C; it then
// writes one s2 partial per 128-row tile ([MT][N*Hkv][C]), else one.
// The refine kernels take the queries by TMA (q_block as [N*B][Hq][d],
// encode_heads_map): qmap with a box of 64 columns x G heads x floor(128/G)
// tokens (row tiles of whole tokens, MT_tok of them), qmap_all with a box
// of all B tokens (the two-pass refine's second pass; may be null when
// C <= 4096).  rlse: [N*Hkv][MT*128] floats for the two-pass refine.
// early: the fused refine reads cand, n_cand and the candidate rows of
// k_cache before its grid-dependency wait; only for inputs written before
// the launch that precedes it on `st` began (ignored by the two-pass refine).
bool refine_fused_ok(int C);
cudaError_t launch_refine(const herald_dims& dm, const uint16_t* k_cache, const int32_t* cand,
                           const int32_t* n_cand, int C, float2* rpart,
                          float* rlse, float* s2, const WsLayout& w, uint32_t* err,
                          const CUtensorMap* qmap, const CUtensorMap* qmap_all, cudaStream_t st,
                          bool early = false);
// Host-side tensor map of a [tokens][heads][d] bf16 array, box 64 x
// box_heads x box_tokens, 128-byte swizzle (cached per thread).
herald_status encode_heads_map(const void* base, uint64_t tokens, int heads, int d,
                               uint32_t box_heads, uint32_t box_tokens, CUtensorMap* map);

// The pool gather fused into the top-K: `copies` CTAs per (sequence, KV
// head) select alike and each copies one slice of the selected rows of the
// cache (device memory) into the pool.
struct PoolGather {
  const uint16_t* kc;
  const uint16_t* vc;
  uint16_t* pk;
  uint16_t* pv;
  int d;
  int copies;
};
// s2 holds n_parts partial score arrays of [N*Hkv][C], summed per candidate;
// gather (optional) also fills the pool; slot_out (optional, [N*Hkv][P_max])
// receives the candidate slot of every selected row taken from the top-K,
// -1 for sink, local and padding rows; k_seg (optional, [N*Hkv]) gives each
// (n, g) a budget of its own, at most K.  early: ctx, cand and n_cand were
// written before the kernel launched just before this one began (they are
// inputs of the stage-2 call, not outputs of its refine), so the kernel reads
// them before its grid-dependency wait.
cudaError_t launch_topk_union(const herald_dims& dm, const int32_t* ctx, const int32_t* cand,
                              const int32_t* n_cand, const float* s2, int n_parts, int C, int K,
                              int S, int W, int P_max, int32_t* idx, int32_t* n_sel,
                              cudaStream_t st, const PoolGather* gather = nullptr,
                              int32_t* slot_out = nullptr, const int32_t* k_seg = nullptr,
                              bool early = false);
// The adaptive budget of every (n, g) from the summed stage-2 scores (same
// partial layout as topk_union): the smallest k whose k largest scores hold
// tau of their total, clamped to [K_min, K_max]; k_sel [N*Hkv] out.
cudaError_t launch_budget(const herald_dims& dm, const int32_t* n_cand, const float* s2,
                          int n_parts, int C, int K_min, int K_max, float tau, int32_t* k_sel,
                          cudaStream_t st);
// (name: the label the launch carries in traces)
cudaError_t launch_gather(const herald_dims& dm, const int32_t* idx, const int32_t* n_sel,
                          int P_max, const uint16_t* k_cache, const uint16_t* v_cache,
                          uint16_t* pool_k, uint16_t* pool_v, cudaStream_t st,
                          const char* name = "gather_kernel", int max_ctas = 0);
// The gather with the candidate rows read from HBM: row r of (n, g) comes
// from staged_k/staged_v [N*Hkv][C][d] at slot src[n][g][r] when that is
// >= 0 (rows taken from the candidates), else from the cache at idx.
cudaError_t launch_gather_staged(const herald_dims& dm, const int32_t* idx, const int32_t* n_sel,
                                 int P_max, const int32_t* src, int C, const uint16_t* staged_k,
                                 const uint16_t* staged_v, const uint16_t* k_cache,
                                 const uint16_t* v_cache, uint16_t* pool_k, uint16_t* pool_v,
                                 cudaStream_t st);
// Pool attention (balanced clusters of pool_cs = 8, 12 or 16 CTAs, every
// operand loaded by TMA) applies when attn_pool_cs() > 0; its tensor maps,
// all bf16 with a box of 64 columns and 128-byte swizzle:
//   k, v   pool rows [N*Hkv*P_max][d], box rows attn_pool_kpc(P_max, B, pool_cs)
//   q      queries [N*B][Hq][d], box {G heads, bpt tokens}
//   bk, bv block keys / values [N*B][Hkv][d], box {1 head, B rounded to 16}
// Row tiles hold bpt = attn_pool_bpt() whole tokens (bpt * G <= 128 rows).
struct AppendArgs;  // below
// The pipelined kernel (attn_flash.cu) takes the same q / bk / bv maps and
// pool maps with a box of kFlashTileKeys rows (kt, vt).
struct PoolMaps {
  CUtensorMap k, v, q, bk, bv, kt, vt;
  int bpt;
  int pool_cs;    // CTAs per cluster of the pool kernel (0: it does not apply)
  int sm_budget;  // SMs the call may count on (others busy with other streams; 0 = all)
};
constexpr int kFlashTileKeys = 128;
// Whether the pipelined attention kernel takes these shapes (any P_max).
bool attn_flash_ok(const herald_dims& dm);
// The pipelined attention kernel with `cs` CTAs per row tile (8, 4 or 2;
// 0 = the largest that keeps every cluster resident at once).
cudaError_t launch_attn_flash(const herald_dims& dm, const int32_t* n_sel, int P_max,
                              uint16_t* out, float scale, uint32_t* err, const PoolMaps& maps,
                              const AppendArgs* app, int cs, bool settled, cudaStream_t st);
int attn_pool_kpc(int P_max, int B, int cs);
int attn_pool_bpt(const herald_dims& dm);
// The pool kernel's cluster size for these shapes and kernel choice
// (HERALD_ATTN_KERNEL_* >> 8): 16 or 12 where every cluster of the launch
// can be resident at once within sm_budget SMs (0 = all), else 8; 0 where
// the pool kernel does not apply.
int attn_pool_cs(const herald_dims& dm, int P_max, int choice, int sm_budget);
cudaError_t launch_attn(const herald_dims& dm, const uint16_t* q, const uint16_t* pool_k,
                        const uint16_t* pool_v, const int32_t* n_sel, int P_max,
                        const uint16_t* block_k, const uint16_t* block_v, uint16_t* out,
                        float scale, const WsLayout& w, float* opart, float2* ml, uint32_t* err,
                        const PoolMaps* maps, bool settled, const AppendArgs* app,
                        int kernel, cudaStream_t st);
// (kernel: bits 0-3 the HERALD_ATTN_KERNEL_* choice >> 8; 0x100: the pool
// kernel takes these shapes; 0x200: the pipelined kernel does)
// exact selection: per-segment candidate counts = context lengths; the
// refine's score partials summed in place (stride floats per segment) and
// histogrammed for the top-K radix select
cudaError_t launch_exact_counts(const herald_dims& dm, const int32_t* ctx, int32_t* n_cand,
                                cudaStream_t st);
cudaError_t launch_exact_sum_hist(const herald_dims& dm, float* s, int n_parts, int stride,
                                  const int32_t* ctx, uint32_t* hist, int num_sms,
                                  cudaStream_t st);
cudaError_t launch_wait_timeout(uint64_t limit_ns, uint32_t* err, cudaStream_t st);
cudaError_t launch_append(const herald_dims& dm, const uint16_t* block_k, const uint16_t* block_v,
                          int32_t* ctx, uint16_t* k_cache, uint16_t* v_cache, int advance,
                          cudaStream_t st);
// block-granular stage 1 (block_select.cu)
cudaError_t launch_pool_keys(const herald_dims& dm, const uint16_t* k_cache, const int32_t* ctx,
                             int Bk, int n_tail, float* pooled, cudaStream_t st);
int block_scan_chunks(const herald_dims& dm, int num_sms);
cudaError_t launch_block_scan(const herald_dims& dm, const float* pooled, const float* qbar,
                              const int32_t* ctx, int Bk, int L_pad, float* logits,
                              float2* part1, int32_t* ctx_b, int chunks, cudaStream_t st);
cudaError_t launch_expand_blocks(const herald_dims& dm, const int32_t* cand_b,
                                 const int32_t* n_cand_b, const int32_t* ctx, int Bk,
                                 int C_blocks, int32_t* cand, int32_t* n_cand, cudaStream_t st);

// The append of a decoded block, done inside another kernel: the rows of
// block[n][b][g] (bf16, [N][B][Hkv][d]) go to cache[n][g][L0 + b], rows at or
// past L_max skipped; `tid` of `nthreads` threads, kBatch 16-byte chunks of K
// and of V in flight per thread and round.
#ifdef __CUDACC__
template <int kBatch>
__device__ __forceinline__ void append_block_rows(const uint16_t* __restrict__ bk,
                                                  const uint16_t* __restrict__ bv, int n, int B,
                                                  int Hkv, int d, int L_max, int L0,
                                                  uint16_t* __restrict__ kc,
                                                  uint16_t* __restrict__ vc, int tid,
                                                  int nthreads) {
  const int cpr = d / 8, total = B * Hkv * cpr;
  for (int q0 = 0; q0 < total; q0 += nthreads * kBatch) {
    uint4 k[kBatch], v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int q = q0 + u * nthreads + tid;
      if (q < total) {
        const int c = q % cpr, bg = q / cpr, g = bg % Hkv, b = bg / Hkv;
        const size_t src = ((size_t(n) * B + b) * Hkv + g) * d + c * 8;
        k[u] = *reinterpret_cast<const uint4*>(bk + src);
        v[u] = *reinterpret_cast<const uint4*>(bv + src);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int q = q0 + u * nthreads + tid;
      if (q < total) {
        const int c = q % cpr, bg = q / cpr, g = bg % Hkv, b = bg / Hkv;
        const int j = L0 + b;
        if (j < L_max) {
          const size_t dst = ((size_t(n) * Hkv + g) * L_max + j) * d + c * 8;
          *reinterpret_cast<uint4*>(kc + dst) = k[u];
          *reinterpret_cast<uint4*>(vc + dst) = v[u];
        }
      }
    }
  }
}
#endif

// The append fused into a denoising step (the pool attention kernel): the
// step's own block keys/values, the cache and its lengths.
struct AppendArgs {
  const uint16_t* bk;
  const uint16_t* bv;
  int32_t* ctx;
  uint16_t* kc;
  uint16_t* vc;
  int advance;
};

}  // namespace herald
