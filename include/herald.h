/*
 * herald.h -- C ABI of the HERALD hot path on one GPU (sm_103a).
 *
 * Method (web pages on the subject):
 *   [V3]  "HERALD: High-Throughput Block Diffusion LLM Inference via CPU-GPU
 *         Cooperative KV Cache Retrieval", arXiv 2606.21633 v3, abstract.
 *   [EA]  HERALD early abstract (mlsift.com, "KV cache offloading" listing).
 *   [SPD] SparDA summary (hyper.ai, arXiv 2606.04511), Method section.
 *   [MG]  "MAGE: All-[MASK] Block Already Knows Where to Look in Diffusion
 *         LLM", author page, abstract.
 *
 * One block of a block-diffusion LLM layer is decoded as:
 *   select (once per block)  ->  gather into a sparse pool  ->  T x attention.
 * Selection has two stages [V3]: stage 1 scores one merged query per head
 * (the mean of the B block queries) against the whole cache and keeps C
 * candidates per KV head; stage 2 scores the block's real B*G queries of a
 * GQA group against those candidates only and keeps K, to which sink and
 * local positions are added.
 *
 * Conventions shared by every call:
 *   - bf16 tensors are passed as uint16_t bit patterns; all tensors are dense
 *     and row-major in the layouts given per argument.
 *   - "device pointer" = memory the GPU can address: cudaMalloc memory, or
 *     (where stated) mapped pinned host memory (cudaHostAlloc with
 *     cudaHostAllocMapped, used through its device pointer).
 *   - Every pointer must be 16-byte aligned.  The caller owns every buffer;
 *     the library never allocates or frees device memory.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  A call validates its arguments on the host
 *     first and launches nothing if they are invalid.  Launch failures are
 *     reported as HERALD_ERR_CUDA with the message in herald_last_error().
 *     Faults inside kernels surface at the next synchronisation.
 *   - Kernels that wait on their own asynchronous copies or tensor-core
 *     work give up after about one second, record a code in the
 *     workspace's error word and return; read it with
 *     herald_workspace_error().
 *   - GQA: query head h belongs to KV head h / G, G = Hq / Hkv.
 *   - Scores use the scale 1/sqrt(d).  Ties in every top-m are broken
 *     towards the lower cache position; index outputs are ascending.
 *   - ctx_len values must lie in [0, L_max]; kernels clamp to that range.
 *   - One workspace may not be shared by calls that can run concurrently.
 */
#ifndef HERALD_H
#define HERALD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HERALD_OK = 0,
  HERALD_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad count   */
  HERALD_ERR_UNSUPPORTED_SHAPE = 2,  /* d, G, B*G, C outside supported set  */
  HERALD_ERR_WORKSPACE_TOO_SMALL = 3,
  HERALD_ERR_CUDA = 4                /* CUDA runtime/driver error            */
} herald_status;

/* Shapes of one attention layer.
 *   N     sequences in the batch           (>= 1)
 *   Hq    query heads                      (Hq % Hkv == 0, 1 <= G <= 8)
 *   Hkv   KV heads                         (>= 1)
 *   d     head dimension                   (64 or 128)
 *   B     block size (queries per block)   (>= 1, B*G <= 256)
 *   L_max cache rows per (sequence, KV head) (>= 1, N*Hkv*L_max < 2^31) */
typedef struct {
  int N, Hq, Hkv, d, B, L_max;
} herald_dims;

/* Bytes of workspace needed by herald_select*, herald_denoise_attn for these
 * shapes, candidate count C and pool capacity P_max.  Returns 0 if the
 * shapes are unsupported. */
size_t herald_workspace_size(herald_dims dims, int C, int P_max);

/* Static text for a status code. */
const char *herald_status_string(herald_status s);

/* Detail of the last error raised on this host thread ("" if none). */
const char *herald_last_error(void);

/* The debug build (compiled with -DHERALD_DEBUG) checks, on the device, the
 * indices and counts its kernels read and write: candidate and selected
 * positions against the cache rows and the context length (idx < ctx_len),
 * selection rows against P_max, n_sel in [0, P_max], ctx_len values in
 * [0, L_max].  A failed check sets a bit in a device check word and the
 * access is skipped or clamped as in every build; nothing traps.
 * herald_debug_build() returns 1 in that build, 0 otherwise.
 * herald_debug_status() waits for the whole device, then returns and clears
 * the check word in *code: 0 = every check passed, bit 0x10 = an index out
 * of range, bit 0x20 = a count or context length out of range (always 0 in
 * release builds).  The word is shared by every stream and thread. */
int herald_debug_build(void);
herald_status herald_debug_status(uint32_t *code);

/* Test hook of the host-side error paths: after `after` further kernel
 * launches by this host thread, the next launch does not happen and
 * returns the CUDA error code `cuda_error` instead, which the calling entry
 * point reports as HERALD_ERR_CUDA with the launch named in
 * herald_last_error().  The hook then disarms itself; after < 0 disarms it
 * at once.  cuda_error must be nonzero when arming. */
herald_status herald_inject_launch_failure(int after, int cuda_error);

/* Synchronously reads and clears the device error word of a workspace
 * (0 = no kernel gave up on a wait).  Bits 0-7: the kind of wait that ran
 * out first (1 = a copy wait, 2 = a tensor-core or pipeline-stage wait);
 * bits 8-15: the kernel (1 refine pass 1, 2 refine pass 2, 3 fused refine,
 * 4 split attention, 5 cluster attention, 6 pool attention, 7 stage-1 scan,
 * 8 pipelined attention); bits 16-31: which of the kernel's waits (the
 * pipelined attention: 0x1 K ring slot, 0x2 V ring slot, 0x4 query tile,
 * 0x8 K tile, 0x10 S buffer free, 0x20 P ready, 0x40 V tile, 0x80 S ready,
 * 0x100 O ready for a rescale, 0x200 every MMA done, 0x400 the peers'
 * partials, 0x800 the previous tile's P V done).
 * Synchronises `stream` first. */
herald_status herald_workspace_error(void *ws, void *stream, uint32_t *code);

/* Stage 1 of the selection [V3]: merged query + full-cache scan + top-C.
 *   q_merge [N][B][Hq][d] bf16 device: the queries the merged query is
 *           formed from (current or draft block; [EA] uses a draft block).
 *   k_cache [N][Hkv][L_max][d] bf16: device memory or mapped pinned host.
 *   ctx_len [N] int32 device: cached positions per sequence.
 *   cand    [N][Hkv][C] int32 device out: the min(C, ctx) positions with
 *           the largest stage-1 score s1[j] = sum over the group's heads of
 *           softmax_j(qbar_h . k_j / sqrt(d)) ([SPD] S_tgt), ascending,
 *           padded with -1.
 *   n_cand  [N][Hkv] int32 device out: min(C, ctx).
 *   sm_budget  the most SMs the cache scan keeps busy at once; 0 = all.
 *           A caller that runs stage 1 beside other work (the dual-stream
 *           pipeline of [EA] overlaps it with denoising) leaves the other
 *           SMs to that work: the scan is persistent and would otherwise
 *           hold every SM for its duration.  Negative values are invalid. */
herald_status herald_select_stage1(herald_dims dims, const uint16_t *q_merge,
                                   const uint16_t *k_cache, const int32_t *ctx_len, int C,
                                   int32_t *cand, int32_t *n_cand, void *ws, size_t ws_bytes,
                                   int sm_budget, void *stream);

/* Stage 2 split around the host link for a cache in mapped pinned host
 * memory ([EA]: the subset crosses the link once per block; the candidates'
 * rows can cross it while the previous block is denoised):
 * herald_stage_candidates copies the candidates' K rows (and V rows, when
 *   v_cache and staged_v are given; both null = K only) by slot,
 *   staged_k[n][g][c] = k_cache[n][g][cand[n][g][c]] for c < n_cand, zero
 *   rows after, bf16 [N][Hkv][C][d] device out (staged_v likewise);
 *   HERALD_ERR_INVALID_ARG if exactly one of v_cache, staged_v is null;
 * herald_select_stage2_staged is herald_select_stage2 reading the candidate
 *   rows from staged_k (the same idx and n_sel, bit for bit);
 * herald_select_stage2_staged_gather is herald_select_stage2_gather with the
 *   candidate rows read from staged_k / staged_v: the refine reads staged_k,
 *   and the pool rows taken from the top-K come from the staged rows, those
 *   of the sink and local window from the cache -- the same idx, n_sel and
 *   pool, bit for bit, with only the sink and local rows crossing the link.
 * The cache rows below ctx_len must not change between the calls. */
herald_status herald_stage_candidates(herald_dims dims, const uint16_t *k_cache,
                                      const uint16_t *v_cache, const int32_t *cand,
                                      const int32_t *n_cand, int C, uint16_t *staged_k,
                                      uint16_t *staged_v, void *stream);
herald_status herald_select_stage2_staged(herald_dims dims, const uint16_t *q_block,
                                          const uint16_t *staged_k, const int32_t *ctx_len,
                                          const int32_t *cand, const int32_t *n_cand, int C,
                                          int K, int sink, int local, int P_max, int32_t *idx,
                                          int32_t *n_sel, void *ws, size_t ws_bytes,
                                          void *stream);
herald_status herald_select_stage2_staged_gather(
    herald_dims dims, const uint16_t *q_block, const uint16_t *staged_k, const uint16_t *staged_v,
    const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *ctx_len, const int32_t *cand,
    const int32_t *n_cand, int C, int K, int sink, int local, int P_max, int32_t *idx,
    int32_t *n_sel, uint16_t *pool_k, uint16_t *pool_v, void *ws, size_t ws_bytes,
    void *stream);

/* herald_select_stage2 with a budget of its own per (sequence, KV head),
 * predicted from the first denoising step ([MG]: the first step predicts
 * the block's budget; the pages give no mechanism, so this is a reading):
 *   k_sel[n][g] = the smallest k whose k largest stage-2 scores s2 hold a
 *   fraction tau of their total over the n_cand valid slots (at most
 *   n_cand), clamped to [K_min, K_max]; int32 [N][Hkv] device out;
 * then step 5 with K = k_sel[n][g] for that (n, g): idx and n_sel as in
 * herald_select_stage2.  The scores are summed and compared in fp32 on the
 * device, so near the tau boundary k_sel may differ by a few from an exact
 * computation.  Errors: HERALD_ERR_INVALID_ARG for K_min outside [0, K_max],
 * tau outside (0, 1], K_max > C or K_max + sink + local > P_max, or a null
 * pointer. */
herald_status herald_select_stage2_adaptive(herald_dims dims, const uint16_t *q_block,
                                           const uint16_t *k_cache, const int32_t *ctx_len,
                                           const int32_t *cand, const int32_t *n_cand, int C,
                                           int K_min, int K_max, float tau, int sink, int local,
                                           int P_max, int32_t *idx, int32_t *n_sel,
                                           int32_t *k_sel, void *ws, size_t ws_bytes,
                                           void *stream);

/* Block-granular stage 1 ([SPD]: InfLLM-V2 selects whole blocks of the
 * context; here stage 1's rule is applied to blocks, not keys).  The cache is
 * summarised by its block means -- the "compressed keys" --
 *   pooled[n][g][b] = mean of k_cache[n][g][j] over j in [b*Bk, min((b+1)*Bk,
 *   ctx_len[n])),  fp32 [N][Hkv][ceil(L_max/Bk)][d] device,
 * zero for blocks at or past ctx_len[n].  herald_pool_keys builds it
 * (n_tail = 0: every block) or refreshes the last n_tail blocks below
 * ctx_len of each sequence (after an append grew the cache: ceil(B/Bk) + 1
 * blocks cover the ones it touched).  k_cache may be mapped pinned host
 * memory.  Bk in [1, L_max], n_tail >= 0. */
herald_status herald_pool_keys(herald_dims dims, const uint16_t *k_cache,
                               const int32_t *ctx_len, int Bk, int n_tail, float *pooled,
                               void *stream);

/* Stage 1 over the blocks: s1b[b] = sum over the group's heads of softmax
 * over the blocks below ceil(ctx/Bk) of qbar_h . pooled_b / sqrt(d) (qbar as
 * in herald_select_stage1); the C_blocks best blocks (lowest index on ties)
 * are expanded to their positions below ctx_len.
 *   cand   [N][Hkv][C_blocks*Bk] int32 device out, ascending, -1 padded
 *   n_cand [N][Hkv] int32 device out
 * 1 <= C_blocks*Bk <= 16384.  ws: herald_workspace_size(dims, C_blocks*Bk,
 * P_max) bytes (the workspace stage 2 uses) are enough.  The candidates
 * feed herald_select_stage2 with C = C_blocks*Bk. */
herald_status herald_select_stage1_blocks(herald_dims dims, const uint16_t *q_merge,
                                          const float *pooled, const int32_t *ctx_len, int Bk,
                                          int C_blocks, int32_t *cand, int32_t *n_cand,
                                          void *ws, size_t ws_bytes, void *stream);

/* Stage 2 of the selection [V3] plus sink/local [SPD InfLLM-V2 decomposition].
 *   q_block [N][B][Hq][d] bf16 device: the real queries of the block being
 *           selected for.
 *   cand, n_cand as written by herald_select_stage1 (C = its row length).
 *   Score s2[c] = sum over the B*G rows of the group of softmax over the
 *   candidates of q . k_cand / sqrt(d).  Keeps the min(K, n_cand) best, adds
 *   positions [0, sink) and [ctx - local, ctx) clipped to [0, ctx), no
 *   duplicates, ascending.
 *   idx     [N][Hkv][P_max] int32 device out, -1 padded (P_max >= K+sink+local)
 *   n_sel   [N][Hkv] int32 device out. */
herald_status herald_select_stage2(herald_dims dims, const uint16_t *q_block,
                                   const uint16_t *k_cache, const int32_t *ctx_len,
                                   const int32_t *cand, const int32_t *n_cand, int C, int K,
                                   int sink, int local, int P_max, int32_t *idx,
                                   int32_t *n_sel, void *ws, size_t ws_bytes, void *stream);

/* herald_select_stage2 followed by herald_gather, in one step where the
 * cache is in device memory: several top-K CTAs per (sequence, KV head)
 * make the same (deterministic) selection and each copies one slice of the
 * selected rows into the pool, so the gather needs no launch of its own
 * ([EA]: the pool is filled once per block).  Outputs: idx, n_sel as from
 * herald_select_stage2 and pool_k, pool_v as from herald_gather, bit for
 * bit.  A cache in mapped pinned host memory gets the two calls.
 *   v_cache   [N][Hkv][L_max][d] bf16, the same placement as k_cache.
 *   pool_k/v  [N][Hkv][P_max][d] bf16 device out. */
herald_status herald_select_stage2_gather(herald_dims dims, const uint16_t *q_block,
                                          const uint16_t *k_cache, const uint16_t *v_cache,
                                          const int32_t *ctx_len, const int32_t *cand,
                                          const int32_t *n_cand, int C, int K, int sink,
                                          int local, int P_max, int32_t *idx, int32_t *n_sel,
                                          uint16_t *pool_k, uint16_t *pool_v, void *ws,
                                          size_t ws_bytes, void *stream);

/* Both stages in order (candidates kept in the workspace).  Passing
 * q_merge == q_block is the non-speculative case. */
herald_status herald_select(herald_dims dims, const uint16_t *q_merge, const uint16_t *q_block,
                            const uint16_t *k_cache, const int32_t *ctx_len, int C, int K,
                            int sink, int local, int P_max, int32_t *idx, int32_t *n_sel,
                            void *ws, size_t ws_bytes, void *stream);

/* herald_select_stage2 without a workspace, for callers that cannot allocate
 * device memory where they select (a decode loop under CUDA stream capture,
 * where cudaMalloc is not allowed; a plugin in a serving runtime that owns
 * the device-memory budget; a host callback where a synchronising
 * allocation would stall every stream).  The pages have no counterpart: this
 * is a deployment variant of the same stage-2 computation, with the same
 * arguments and outputs minus the workspace.
 *   Scratch lives in one static 4 MiB device array inside the library; every
 *   GPU that loads the library holds it until the process exits.  Shapes
 *   whose scratch -- 256 bytes + N*Hkv*ceil(B*G/128)*128*(ceil(C/256)*8 + 4)
 *   bytes of row statistics + N*Hkv*C*4 bytes of scores per row tile of
 *   floor(128/G) whole tokens (one tile when C > 4096) -- exceed 4 MiB are
 *   rejected with HERALD_ERR_WORKSPACE_TOO_SMALL and a message.
 *   The first call on a device resolves the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   All calls share the array: calls that can overlap on the GPU (other
 *   streams, other host threads) race and must be serialised by the caller.
 *   k_cache must be device memory: a cache in mapped host memory, whose
 *   candidate rows herald_select_stage2 stages in its workspace first, is
 *   rejected with HERALD_ERR_INVALID_ARG.  The other argument rules are
 *   herald_select_stage2's.  Host threads may make their first calls at the
 *   same time (the address is resolved under a lock).
 *   Device-side wait timeouts are recorded in the array, not reported.
 *   Nothing is allocated or freed by this call. */
herald_status herald_select_stage2_noalloc(herald_dims dims, const uint16_t *q_block,
                                           const uint16_t *k_cache, const int32_t *ctx_len,
                                           const int32_t *cand, const int32_t *n_cand, int C,
                                           int K, int sink, int local, int P_max,
                                           int32_t *idx, int32_t *n_sel, void *stream);

/* Gathers the selected rows into one buffer of the double-buffered sparse
 * KV pool [EA]:  pool[n][g][s] = cache[n][g][idx[n][g][s]] for s < n_sel,
 * zero rows for n_sel <= s < P_max.
 *   k_cache, v_cache [N][Hkv][L_max][d] bf16, device or mapped pinned host.
 *   pool_k, pool_v   [N][Hkv][P_max][d] bf16 device out. */
herald_status herald_gather(herald_dims dims, const int32_t *idx, const int32_t *n_sel,
                            int P_max, const uint16_t *k_cache, const uint16_t *v_cache,
                            uint16_t *pool_k, uint16_t *pool_v, void *stream);

/* One denoising step of sparse block attention over the pool [EA][V3]:
 * every query (n, b, h) attends, without a mask, to the n_sel pool rows of
 * KV head h/G followed by the B block keys of that head (bidirectional
 * inside the block).
 *   q        [N][B][Hq][d] bf16 device     block_k, block_v [N][B][Hkv][d]
 *   pool_k/v [N][Hkv][P_max][d] bf16 device, as written by herald_gather
 *   n_sel    [N][Hkv] int32 device
 *   out      [N][B][Hq][d] bf16 device out
 *   scale    softmax scale; 0 selects 1/sqrt(d). */
herald_status herald_denoise_attn(herald_dims dims, const uint16_t *q, const uint16_t *pool_k,
                                  const uint16_t *pool_v, const int32_t *n_sel, int P_max,
                                  const uint16_t *block_k, const uint16_t *block_v,
                                  uint16_t *out, float scale, void *ws, size_t ws_bytes,
                                  void *stream);

/* Flags of herald_denoise_attn_ex. */
#define HERALD_ATTN_SETTLED 1u /* the pool was written before an earlier herald call  */
#define HERALD_ATTN_APPEND 2u  /* also append block_k/block_v to the cache            */
#define HERALD_ATTN_ADVANCE 4u /* with APPEND: then advance ctx_len                    */
/* Kernel choice (bits 8-11; for tests and tuning -- the default picks by
 * shape): the cluster kernel holding a whole pool slice per CTA (with 8,
 * 12 or 16 CTAs per row tile, or chosen by shape), or the pipelined kernel
 * streaming key tiles (with 8, 4 or 2 CTAs per row tile, or chosen by
 * shape).  A choice the shapes do not allow falls back to the default. */
#define HERALD_ATTN_KERNEL_POOL (1u << 8)
#define HERALD_ATTN_KERNEL_FLASH (2u << 8)
#define HERALD_ATTN_KERNEL_FLASH_CS2 (3u << 8)
#define HERALD_ATTN_KERNEL_FLASH_CS4 (4u << 8)
#define HERALD_ATTN_KERNEL_FLASH_CS8 (5u << 8)
#define HERALD_ATTN_KERNEL_POOL_CS8 (6u << 8)
#define HERALD_ATTN_KERNEL_POOL_CS16 (7u << 8)
#define HERALD_ATTN_KERNEL_POOL_CS12 (8u << 8)
/* SM budget (bits 16-23, in units of 4 SMs; 0 = every SM): how many SMs the
 * call may count on while work on other streams holds the rest (a stage-1
 * scan or a copy confined to a few SMs).  The kernels' cluster sizes are
 * chosen so that the whole launch fits that many SMs at once. */
#define HERALD_ATTN_SMS(n) ((((unsigned)(n) / 4u) & 0xFFu) << 16)

/* herald_denoise_attn with options for the steps of a block (flags = 0 is
 * herald_denoise_attn; ctx_len, k_cache, v_cache are used only with
 * HERALD_ATTN_APPEND and may be NULL otherwise).
 *   HERALD_ATTN_SETTLED (steps 1..T-1): the pool keys are loaded while the
 *     work before the call on `stream` is still finishing, instead of after
 *     it.  The pool is fixed across a block's T steps ([EA]: one selection
 *     serves all of them).  Precondition: pool_k was written before some
 *     earlier herald_* call on `stream` (and nothing writes it since): every
 *     herald kernel lets its successor start only after its own predecessor
 *     has finished, so the pool is final when this kernel starts.  A call
 *     right after the herald_gather that wrote the pool must not set it;
 *     breaking the precondition races with that write.  Applied only when
 *     the whole grid is resident at once (otherwise ignored).
 *   HERALD_ATTN_APPEND (the last step): the result of herald_append_kv(dims,
 *     block_k, block_v, ctx_len, k_cache, v_cache, flags & ADVANCE) as
 *     well, in the same kernel when the cache is in device memory (one
 *     launch fewer per block; [V3]: the decoded block joins the cache), by
 *     the append kernel after the step when it is in host memory.  The
 *     cache and ctx_len must not be read by work that can run concurrently
 *     (the dual-stream pipeline joins its stage-1 stream before this call).
 *   HERALD_ATTN_ADVANCE: with APPEND, ctx_len[n] = min(ctx_len[n] + B, L_max).
 * Unknown flag bits, ADVANCE without APPEND, or APPEND with a null ctx_len,
 * k_cache or v_cache: HERALD_ERR_INVALID_ARG. */
herald_status herald_denoise_attn_ex(herald_dims dims, const uint16_t *q, const uint16_t *pool_k,
                                     const uint16_t *pool_v, const int32_t *n_sel, int P_max,
                                     const uint16_t *block_k, const uint16_t *block_v,
                                     uint16_t *out, float scale, unsigned flags,
                                     int32_t *ctx_len, uint16_t *k_cache, uint16_t *v_cache,
                                     void *ws, size_t ws_bytes, void *stream);

/* Appends a decoded block to the cache ([V3]: the cache grows with every
 * decoded block):  cache[n][g][ctx_len[n] + b] = block[n][b][g] for b < B
 * (rows at or past L_max are skipped), then, if advance != 0,
 * ctx_len[n] = min(ctx_len[n] + B, L_max).
 *   block_k, block_v [N][B][Hkv][d] bf16 device
 *   k_cache, v_cache [N][Hkv][L_max][d] bf16, device or mapped pinned host
 *   ctx_len [N] int32 device (read, and updated when advance != 0). */
herald_status herald_append_kv(herald_dims dims, const uint16_t *block_k,
                               const uint16_t *block_v, int32_t *ctx_len, uint16_t *k_cache,
                               uint16_t *v_cache, int advance, void *stream);

/* The buffers of the dual-stream block pipeline (herald_block), owned by
 * the caller and kept from block to block:
 *   cand[2], n_cand[2]  [N][Hkv][C], [N][Hkv] int32 device: block i's
 *                       stage 2 reads cand[i%2], its stage 1 for block i+1
 *                       writes cand[(i+1)%2]
 *   idx, n_sel          [N][Hkv][P_max], [N][Hkv] int32 device
 *   pool_k[2], pool_v[2] [N][Hkv][P_max][d] bf16 device: block i's pool is
 *                       pool[i%2]
 *   ws_den, ws_sel      two workspaces of ws_bytes >= herald_workspace_size
 *                       (dims, C, P_max) bytes each: the denoising stream's
 *                       and the selection stream's
 *   sel_stream          cudaStream_t for stage 1 beside the denoising steps;
 *                       NULL: stage 1 runs on the denoising stream (no
 *                       overlap)
 *   ev_fork, ev_join    cudaEvent_t created by the caller (timing may be
 *                       disabled); used only with sel_stream */
typedef struct {
  int32_t *cand[2], *n_cand[2];
  int32_t *idx, *n_sel;
  uint16_t *pool_k[2], *pool_v[2];
  void *ws_den, *ws_sel;
  size_t ws_bytes;
  void *sel_stream;
  void *ev_fork, *ev_join;
} herald_block_bufs;

#define HERALD_BLOCK_ADVANCE 1u /* the last step advances ctx_len by B */
/* The caller guarantees that cand[i%2], n_cand[i%2] and their rows of
 * k_cache are not written by the launch that immediately precedes this call
 * on `stream` (nor by anything not ordered before it): true when the
 * previous call on these streams was herald_block for block i-1 (its stage
 * 1, which wrote cand[i%2], is joined before its last step, and the
 * candidates lie below the context that step appends to); false right after
 * herald_select_stage1 wrote them on `stream`.  Stage 2's refine then reads
 * them before its grid-dependency wait: every launch of the library lets its
 * successor start only after its own wait, so they are final by then. */
#define HERALD_BLOCK_CAND_SETTLED 2u

/* One block of one layer through the dual-stream pipeline ([EA]:
 * selection and denoising run as a dual-stream pipeline over
 * double-buffered sparse KV pools; [V3]: while the current block is
 * denoised, stage 1 searches the cache for the next block with the current
 * block's merged query, and stage 2 refines the candidates with the next
 * block's real queries), issued by one call.  With den = `stream` and sel =
 * bufs->sel_stream:
 *   den: herald_select_stage2_gather(q_steps[0], cand[i%2]) -> idx, n_sel,
 *        pool[i%2]
 *   sel: (after everything issued on den before this call)
 *        herald_select_stage1(q_steps[0], next_k_cache, scan_sms) ->
 *        cand[(i+1)%2]
 *   den: T x herald_denoise_attn_ex over pool[i%2] into out[t], steps
 *        after the first with HERALD_ATTN_SETTLED, each with
 *        HERALD_ATTN_SMS(SMs - scan_sms) when 0 < scan_sms < SMs; the last
 *        step waits for sel (stage 1 scans the cache before the block is
 *        appended) and appends block_k[T-1], block_v[T-1] (HERALD_ATTN_APPEND,
 *        with HERALD_ATTN_ADVANCE if flags has HERALD_BLOCK_ADVANCE).
 * flags: HERALD_BLOCK_ADVANCE, HERALD_BLOCK_CAND_SETTLED.
 * The same calls issued one by one give the same results.  Before the
 * first block, cand[0] must hold stage 1 of block 0 (herald_select_stage1
 * with its own queries).
 *   q_steps, out        [T][N][B][Hq][d] bf16 device
 *   block_k, block_v    [T][N][B][Hkv][d] bf16 device
 *   k_cache, v_cache    [N][Hkv][L_max][d] bf16, device or mapped pinned host
 *   ctx_len             [N] int32 device
 *   next_k_cache        the cache stage 1 scans for block i+1 (NULL: k_cache)
 *   i                   the block's index (>= 0; its parity picks the buffers)
 *   scan_sms            SMs stage 1 may hold beside the steps (0: all; the
 *                       scan is persistent, so a small cache is best left a
 *                       few dozen SMs and a cache larger than the steps'
 *                       bytes all of them); ignored without sel_stream
 * Errors: those of the calls above, T < 1, i < 0, scan_sms < 0, unknown
 * flags, a null bufs, or sel_stream without both events:
 * HERALD_ERR_INVALID_ARG.  A call that fails after its first launch leaves
 * the block partly issued. */
herald_status herald_block(herald_dims dims, int C, int K, int sink, int local, int P_max, int T,
                           int i, const uint16_t *q_steps, const uint16_t *block_k,
                           const uint16_t *block_v, uint16_t *k_cache, uint16_t *v_cache,
                           int32_t *ctx_len, const uint16_t *next_k_cache, uint16_t *out,
                           unsigned flags, int scan_sms, const herald_block_bufs *bufs,
                           void *stream);

/* Exact selection, the accuracy reference for the merged-query stage 1
 * ([MG]: exact attention of the block's queries predicts the important
 * entries; [V3] approximates it with one merged query).  Every cached
 * position is scored with all B*G real query rows of the block:
 *   s[j] = sum over the rows r of softmax_j(q_r . k_j / sqrt(d)), j < ctx,
 * (stage 2's score with the whole context as the candidate list); the K
 * largest (lowest position on ties) are kept and the sink and local
 * positions added exactly as herald_select_stage2 does.
 *   q_block, k_cache, ctx_len, sink, local, P_max, idx, n_sel: as in
 *           herald_select_stage2; 1 <= K <= 16384, K+sink+local <= P_max.
 *   ws:     herald_workspace_size_exact(dims, K, P_max) bytes (0 = shape not
 *           supported).
 * Cost: two tensor-core passes over the whole cache per block (B*G times
 * the merged query's contraction) instead of one merged-query scan. */
size_t herald_workspace_size_exact(herald_dims dims, int K, int P_max);
herald_status herald_select_exact(herald_dims dims, const uint16_t *q_block,
                                  const uint16_t *k_cache, const int32_t *ctx_len, int K,
                                  int sink, int local, int P_max, int32_t *idx, int32_t *n_sel,
                                  void *ws, size_t ws_bytes, void *stream);

/* Self-test of the device-side failure path (the pages have no
 * counterpart).  Every wait inside the library's kernels gives up after
 * about one second, records a code in the workspace's error word and lets
 * the kernel return, so a lost copy or commit is reported instead of
 * hanging the GPU.  This call launches one thread that waits, with that
 * same bounded wait, on a barrier nothing completes, for limit_ns
 * nanoseconds (0 < limit_ns <= 1e9); afterwards herald_workspace_error()
 * on `ws` reads 1 and the context remains usable.  ws: any workspace (its
 * first 4 bytes are the error word). */
herald_status herald_selftest_wait_timeout(uint64_t limit_ns, void *ws, void *stream);

/* Kernel tracing, a profiling aid that is off by default.  While enabled on
 * the calling host thread, every kernel the library launches is bracketed
 * by two caller-created CUDA events (cudaEvent_t, timing enabled) recorded
 * on the launch stream: launch i records events[2i] before and events[2i+1]
 * after the kernel; launches past `capacity` are not traced.  With
 * external != 0 the events are recorded with cudaEventRecordExternal, so a
 * stream capture turns them into event-record nodes of the CUDA graph.
 * herald_trace_end() stops tracing and returns the number of launches
 * traced; herald_trace_name(i) gives the kernel name of launch i (valid
 * until the next herald_trace_begin on this thread). */
herald_status herald_trace_begin(void **events, int capacity, int external);
int herald_trace_end(void);
const char *herald_trace_name(int i);

#ifdef __cplusplus
}
#endif

#endif /* HERALD_H */
