// tc_kernels.cu -- the dense contractions of the HERALD hot path on the 5th
// generation tensor cores (tcgen05.mma, bf16 operands in 128B-swizzled
// shared memory, fp32 accumulators in TMEM):
//   refine_pass1  stage 2 (HERALD v3 abstract: the candidates are re-scored
//                 with the block's real queries): S = Q_blk . K_cand^T per
//                 (sequence, KV head), per-row (max, sumexp) over a chunk of
//                 256 candidates
//   refine_pass2  S^T = K_cand . Q_blk^T for 128 candidates x all B*G rows;
//                 each thread owns one candidate and sums the row-softmax
//                 probabilities over the rows -> s2 (column sum)
//   refine_fused  stage 2 in one pass when C <= 4096: a cluster of 16, 12
//                 or 8 CTAs per row tile shares the row statistics,
//                 exponentials are kept in TMEM and summed by column
//   attn_pool     sparse block attention over the pool (HERALD early
//                 abstract: the selected subset is reused for every
//                 denoising step; block keys are visible to every block
//                 query): one cluster of 8, 12 or 16 CTAs per row tile,
//                 the pool split between its CTAs; optionally appends the
//                 decoded block
//   attn_cluster  the same with cp.async operands, for shapes the pool
//                 kernel does not take
//   attn          one 128-key split of sparse block attention (pools beyond
//                 shared memory): S = Q K^T, P = exp(S - rowmax), O = P V
//   attn_combine  merges the splits by their (max, sum) into bf16 out
#include <cuda_bf16.h>
#include <stdlib.h>

#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace herald {

__device__ __forceinline__ float2 ld_peer_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_cluster(const char* name, void (*kernel)(KArgs...), dim3 grid,
                                  int cluster_x, size_t smem, cudaStream_t st, Args... args) {
  return launch_cluster_threads(name, kernel, grid, dim3(kTcThreads), cluster_x, smem, st,
                                args...);
}

// ========================================================== refine_pass1
template <int D>
struct Ref1Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBytes = kHalves * kTileM * 128;
  static constexpr int kKBytes = kHalves * kRefineChunk * 128;
  static constexpr int kSmem = kQBytes + kKBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "refine pass 1 smem exceeds the per-CTA limit");
};

// Pass 1 for C > 4096: per (segment, row tile of bpt whole tokens, chunk of
// 256 candidates) the row (max, sumexp) of S = Q K_cand^T, the query tile
// loaded by one 3-D TMA box per half.
template <int D>
__global__ void __launch_bounds__(kTcThreads)
    refine_pass1_kernel(const __grid_constant__ CUtensorMap qmap,
                        const uint16_t* __restrict__ kc, const int32_t* __restrict__ cand,
                        const int32_t* __restrict__ n_cand, int B, int Hq, int Hkv, int L_max,
                        int C, int bpt, int MT, int n_chunks, float scale,
                        float2* __restrict__ rpart, uint32_t* err) {
  using Cfg = Ref1Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar, barQ;
  __shared__ uint32_t tmem_base;
  __shared__ float2 red[2][kTileM];
  __shared__ int32_t pos[kRefineChunk];
  uint8_t* Qs = align1024(smem_raw);
  uint8_t* Ks = Qs + Cfg::kQBytes;
  griddep_enter();
  const int chunk = blockIdx.x, mt = blockIdx.y, seg = blockIdx.z;
  const int n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int nc = min(max(n_cand[seg], 0), C);
  const int c0 = chunk * kRefineChunk;
  if (c0 >= nc) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b0 = mt * bpt, rows_t = min(bpt, B - b0) * G;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&barQ, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&barQ, uint32_t((D / 64) * G * bpt * 128));
#pragma unroll
    for (int hv = 0; hv < D / 64; ++hv)
      tma_load_3d(Qs + hv * kTileM * 128, &qmap, &barQ, hv * 64, g * G, n * B + b0);
  }
  tmem_setup(&tmem_base, 256);
  const uint32_t tbase = tmem_base;

  // candidate positions first (one coalesced load), then the row copies
  const int32_t* cd = cand ? cand + size_t(seg) * C : nullptr;  // null: row = slot
  for (int r = threadIdx.x; r < kRefineChunk; r += kTcThreads)
    pos[r] = c0 + r < nc ? (cand ? cd[c0 + r] : c0 + r) : -1;
  // positions outside the cache (a caller error) read as zero rows
  for (int r = threadIdx.x; r < kRefineChunk; r += kTcThreads) {
    debug_flag(c0 + r < nc && (pos[r] < 0 || pos[r] >= L_max), DEV_BAD_INDEX);
    if (pos[r] >= L_max) pos[r] = -1;
  }
  __syncthreads();
  load_rows_sw128<D>(Ks, kRefineChunk, kRefineChunk, kc, [&](int r) -> const uint16_t* {
    const int p = pos[r];
    if (p < 0) return nullptr;
    return kc + (size_t(seg) * L_max + p) * D;
  });
  cp_async_commit();
  cp_async_wait_all();
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    if (!mbar_wait(&barQ, 0)) record_error(err, DEV_TIMEOUT_TMA | DEV_K_REFINE_PASS1);
    tc_fence_after();
    constexpr uint32_t idesc = make_idesc_bf16(kTileM, kRefineChunk, false, false);
    const uint32_t qa = smem_u32(Qs), ka = smem_u32(Ks);
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      const uint32_t hv = s >> 2, koff = (s & 3) * 32;
      const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
      const uint64_t b = make_sdesc_sw128(ka + hv * (kRefineChunk * 128) + koff, 16, 1024);
      umma_bf16(tbase, a, b, idesc, s > 0 ? 1u : 0u);
    }
    umma_commit(&bar);
  }
  if (!mbar_wait(&bar, 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_REFINE_PASS1);
  tc_fence_after();
  __syncwarp();

  const int quad = warp & 3, ch = warp >> 2;
  const int row = quad * 32 + lane;
  const uint32_t taddr = tbase + (uint32_t(quad * 32) << 16) + uint32_t(ch * 128);
  float m = -INFINITY;
  float v[32];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    tmem_ld32(taddr + k * 32, v);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + ch * 128 + k * 32 + i < nc) m = fmaxf(m, v[i] * scale);
  }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    tmem_ld32(taddr + k * 32, v);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + ch * 128 + k * 32 + i < nc) sum += __expf(v[i] * scale - m);
  }
  red[ch][row] = make_float2(m, sum);
  __syncthreads();
  if (ch == 0) {
    const float2 a = red[0][row], b = red[1][row];
    const float M = fmaxf(a.x, b.x);
    const float S = (a.x == -INFINITY ? 0.f : a.y * __expf(a.x - M)) +
                    (b.x == -INFINITY ? 0.f : b.y * __expf(b.x - M));
    if (row < rows_t)
      rpart[(size_t(seg) * MT * kTileM + b0 * G + row) * n_chunks + chunk] = make_float2(M, S);
  }
  tmem_teardown(tbase, 256);
}

// ========================================================== refine_pass2
template <int D>
struct Ref2Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kKBytes = kHalves * kRefineRows2 * 128;
  static constexpr int kQBytes = kHalves * 256 * 128;
  static constexpr int kSmem = kKBytes + kQBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "refine pass 2 smem exceeds the per-CTA limit");
};

// Row log-sum-exp over all candidates, once per row, from pass 1's chunk
// partials: grid (ceil(R / 8), N*Hkv), block 256 -- one warp per row, the
// lanes striding over the chunks, then a warp reduction of (max, sumexp).
__global__ void __launch_bounds__(256)
    refine_lse_kernel(const float2* __restrict__ rpart, const int32_t* __restrict__ n_cand,
                      int C, int R, int MT, int n_chunks, float* __restrict__ rlse) {
  griddep_enter();
  const int seg = blockIdx.y;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= R) return;
  const int nc = min(max(n_cand[seg], 0), C);
  const int nch = (nc + kRefineChunk - 1) / kRefineChunk;
  const float2* p = rpart + (size_t(seg) * MT * kTileM + r) * n_chunks;
  float M = -INFINITY, S = 0.f;
  for (int k0 = lane; k0 < nch; k0 += 32 * 4) {  // four loads in flight per lane
    float2 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * 32;
      q[u] = k < nch ? p[k] : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (q[u].x == -INFINITY) continue;
      if (q[u].x > M) {
        S = S * __expf(M - q[u].x) + q[u].y;
        M = q[u].x;
      } else {
        S += q[u].y * __expf(q[u].x - M);
      }
    }
  }
  const float Mw = warp_max(M);
  S = warp_sum(M == -INFINITY ? 0.f : S * __expf(M - Mw));
  if (lane == 0) rlse[size_t(seg) * MT * kTileM + r] = Mw + __logf(S);
}

// Pass 2: per (segment, 128 candidates) S^T = K_cand Q^T with all B*G query
// rows (one 3-D TMA box per half) and s2[c] = sum_r exp(S[r,c] - lse_r).
template <int D>
__global__ void __launch_bounds__(kTcThreads)
    refine_pass2_kernel(const __grid_constant__ CUtensorMap qmap_all,
                        const uint16_t* __restrict__ kc, const int32_t* __restrict__ cand,
                        const int32_t* __restrict__ n_cand, int B, int Hq, int Hkv, int L_max,
                        int C, int R, int MT, float scale, const float* __restrict__ rlse,
                        float* __restrict__ s2, uint32_t* err) {
  using Cfg = Ref2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar, barQ;
  __shared__ uint32_t tmem_base;
  __shared__ float lse[256];
  __shared__ float red[2][kRefineRows2];
  __shared__ int32_t pos[kRefineRows2];
  uint8_t* Ks = align1024(smem_raw);
  uint8_t* Qs = Ks + Cfg::kKBytes;
  griddep_enter();
  const int seg = blockIdx.y, n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int nc = min(max(n_cand[seg], 0), C);
  const int c0 = blockIdx.x * kRefineRows2;
  if (c0 >= nc) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Rp = (R + 15) & ~15;  // MMA N: multiple of 16
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&barQ, 1);
    fence_mbar_init();
    // all B*G query rows; rows [R, Rp) of the operand are never used
    mbar_arrive_expect_tx(&barQ, uint32_t((D / 64) * R * 128));
#pragma unroll
    for (int hv = 0; hv < D / 64; ++hv)
      tma_load_3d(Qs + hv * 256 * 128, &qmap_all, &barQ, hv * 64, g * G, n * B);
  }
  tmem_setup(&tmem_base, 256);
  const uint32_t tbase = tmem_base;

  const int32_t* cd = cand ? cand + size_t(seg) * C : nullptr;  // null: row = slot
  for (int r = threadIdx.x; r < kRefineRows2; r += kTcThreads) {
    pos[r] = c0 + r >= nc ? -1 : !cand ? c0 + r : cd[c0 + r] < L_max ? cd[c0 + r] : -1;
    debug_flag(c0 + r < nc && cand && (cd[c0 + r] < 0 || cd[c0 + r] >= L_max), DEV_BAD_INDEX);
  }
  __syncthreads();
  load_rows_sw128<D>(Ks, kRefineRows2, kRefineRows2, kc, [&](int r) -> const uint16_t* {
    const int p = pos[r];
    if (p < 0) return nullptr;
    return kc + (size_t(seg) * L_max + p) * D;
  });
  cp_async_commit();
  for (int r = threadIdx.x; r < R; r += kTcThreads)
    lse[r] = rlse[size_t(seg) * MT * kTileM + r];
  cp_async_wait_all();
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    if (!mbar_wait(&barQ, 0)) record_error(err, DEV_TIMEOUT_TMA | DEV_K_REFINE_PASS2);
    tc_fence_after();
    const uint32_t idesc = make_idesc_bf16(kRefineRows2, Rp, false, false);
    const uint32_t ka = smem_u32(Ks), qa = smem_u32(Qs);
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      const uint32_t hv = s >> 2, koff = (s & 3) * 32;
      const uint64_t a = make_sdesc_sw128(ka + hv * (kRefineRows2 * 128) + koff, 16, 1024);
      const uint64_t b = make_sdesc_sw128(qa + hv * (256 * 128) + koff, 16, 1024);
      umma_bf16(tbase, a, b, idesc, s > 0 ? 1u : 0u);
    }
    umma_commit(&bar);
  }
  if (!mbar_wait(&bar, 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_REFINE_PASS2);
  tc_fence_after();
  __syncwarp();

  const int quad = warp & 3, ch = warp >> 2;
  const int row = quad * 32 + lane;
  const uint32_t taddr = tbase + (uint32_t(quad * 32) << 16);
  float acc = 0.f;
  float v[32];
  for (int k = 0; k < 4; ++k) {
    const int col0 = ch * 128 + k * 32;
    if (col0 >= R) break;  // uniform per warp
    tmem_ld32(taddr + col0, v);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < R) acc += __expf(v[i] * scale - lse[col0 + i]);
  }
  red[ch][row] = acc;
  __syncthreads();
  if (ch == 0 && c0 + row < nc) s2[size_t(seg) * C + c0 + row] = red[0][row] + red[1][row];
  tmem_teardown(tbase, 256);
}

// ========================================================== refine_fused
// Stage 2 in one kernel for C <= 4096: one cluster of kFuseCtas CTAs per
// (sequence, KV head, row tile of bpt = floor(128/G) whole tokens, its bpt*G query rows
// loaded by one 3-D TMA box per 64-column half); CTA r scores candidate
// slots [r*cpc, (r+1)*cpc)
// (cpc <= 512, so the scores fill TMEM and are never recomputed).  Each
// CTA stores its row (max, sumexp) over its candidates into every peer's
// shared memory; after one cluster barrier each CTA merges them into the row
// log-sum-exp from its own shared memory, sums exp(S - lse_r) over its 128
// rows (warp shuffle reductions, rows past B*G excluded) and writes one
// partial s2 per row tile, which the top-K kernel adds up.  The cluster
// has 16, 12 or 8 CTAs: the size with the fewest candidates per CTA (they
// set the UMMA, exponential and column-sum work of each CTA) among those
// whose clusters are all resident at once.
constexpr int kFuseMaxCpc = 512;
// 16 warps: the four warps of a TMEM lane quadrant take every fourth
// 32-column chunk of the CTA's candidates
constexpr int kFuseThreads = 512;
constexpr int kFuseSplit = kFuseThreads / 128;

// candidates per CTA of a cs-CTA cluster, in whole 32-column chunks
__host__ __device__ inline int fuse_cpc(int C, int cs = 8) {
  return ((C + cs - 1) / cs + 31) / 32 * 32;
}

template <int D>
struct FuseCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBytes = kHalves * kTileM * 128;
  static constexpr int kKBytes = kHalves * kFuseMaxCpc * 128;
  static constexpr int kSmem = kQBytes + kKBytes + 1024;
  static_assert(kSmem <= 200 * 1024, "fused refine smem");
};

template <int D, int kFuseCtas>
__global__ void __launch_bounds__(kFuseThreads, 1)
    refine_fused_kernel(const __grid_constant__ CUtensorMap qmap,
                        const uint16_t* __restrict__ kc, const int32_t* __restrict__ cand,
                        const int32_t* __restrict__ n_cand, int B, int Hq, int Hkv, int L_max,
                        int C, int bpt, int cpc, float scale, float* __restrict__ s2p,
                        uint32_t* err, int early) {
  using Cfg = FuseCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar0, barQ;
  __shared__ uint32_t tmem_base;
  __shared__ int32_t pos[kFuseMaxCpc];
  __shared__ float2 part_stat[kFuseSplit][kTileM];
  __shared__ __align__(16) float2 peer_stat[kFuseCtas][kTileM];  // [sender][row]
  __shared__ float colsum[4][kFuseMaxCpc];  // [lane quadrant][candidate]
  uint8_t* Qs = align1024(smem_raw);
  uint8_t* Ks = Qs + Cfg::kQBytes;
  const uint32_t rank = cluster_ctarank();
  const int mt = blockIdx.y, seg = blockIdx.z;
  const int n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar0, 1);
    mbar_init(&barQ, 1);
    fence_mbar_init();
    tma_prefetch_desc(&qmap);
  }
  // peers store into this CTA's shared memory before the cluster barrier
  // below: this arrive, awaited just before those stores, shows that every
  // CTA of the cluster has started
  __cluster_barrier_arrive_relaxed();
  tmem_setup(&tmem_base, 512);
  const uint32_t tbase = tmem_base;
  const int b0 = mt * bpt;                  // first token of the tile
  const int rows_t = min(bpt, B - b0) * G;  // query rows of the tile
  // The candidate positions, the zeroed query rows past the tile's and the
  // copies of the candidate rows (cp.async, committed, awaited below).
  // early != 0: the caller guarantees that cand, n_cand and the candidate
  // rows of the cache were written before the launch preceding this one
  // began (the candidates of a block whose stage 1 was joined before the
  // previous block's last step), so they are read before the
  // grid-dependency wait, which then covers only the queries.
  const int c0 = int(rank) * cpc;
  int ncv = 0;  // valid candidates of this CTA
  auto stage_rows = [&]() {
    // the candidate positions are read with n_cand, not after it: every slot
    // below C lies inside the list, and rows past n_cand are masked below
    const int32_t* cd = cand ? cand + size_t(seg) * C : nullptr;  // null: row = slot
    int pr[kFuseMaxCpc / kFuseThreads];
#pragma unroll
    for (int k = 0; k < kFuseMaxCpc / kFuseThreads; ++k) {
      const int r = threadIdx.x + k * kFuseThreads;
      pr[k] = (cd && r < cpc && c0 + r < C) ? cd[c0 + r] : -1;
    }
    const int nc = min(max(n_cand[seg], 0), C);
    ncv = min(max(nc - c0, 0), cpc);
#pragma unroll
    for (int k = 0; k < kFuseMaxCpc / kFuseThreads; ++k) {
      const int r = threadIdx.x + k * kFuseThreads;
      if (r < cpc) {
        const int p = r < ncv ? (cand ? pr[k] : c0 + r) : -1;
        debug_flag(r < ncv && (p < 0 || p >= L_max), DEV_BAD_INDEX);  // a candidate past the cache
        pos[r] = (p >= 0 && p < L_max) ? p : -1;
      }
    }
    __syncthreads();
    // the tile's rows past its G*bpt query rows are never loaded (the query
    // box fills rows [0, G*bpt)): zeroed, so that every score row is finite
    // and the column sums below can weight rows with a product (rows past
    // the tile's tokens get weight 0)
    for (int u = G * bpt * 8 + threadIdx.x; u < kTileM * 8; u += kFuseThreads) {
#pragma unroll
      for (int hv = 0; hv < D / 64; ++hv)
        *reinterpret_cast<uint4*>(Qs + hv * kTileM * 128 + u * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (ncv > 0) {
      load_rows_sw128<D, kFuseThreads>(Ks, cpc, cpc, kc, [&](int r) -> const uint16_t* {
        const int p = pos[r];
        return p < 0 ? nullptr : kc + (size_t(seg) * L_max + p) * D;
      });
      cp_async_commit();
    }
  };
  if (early) stage_rows();
  griddep_enter();
  // the query tile (it does not depend on n_cand); every CTA waits for it
  // before exiting, used or not
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&barQ, uint32_t((D / 64) * G * bpt * 128));
#pragma unroll
    for (int hv = 0; hv < D / 64; ++hv)
      tma_load_3d(Qs + hv * kTileM * 128, &qmap, &barQ, hv * 64, g * G, n * B + b0);
  }
  if (!early) stage_rows();
  if (ncv > 0) cp_async_wait_all();
  fence_proxy_async_smem();  // the zeroed rows and the copied K rows, for the UMMA
  __syncthreads();
  tc_fence_after();
  // S = Q K_cand^T: up to two UMMAs of N = 256 -> TMEM columns [0, cpc)
  bool qok = true;
  if (threadIdx.x == 0) {
    qok = mbar_wait(&barQ, 0);
    tc_fence_after();
  }
  if (threadIdx.x == 0 && ncv > 0) {
    const uint32_t qa = smem_u32(Qs), ka = smem_u32(Ks);
    for (int h0 = 0; h0 < cpc; h0 += 256) {
      const int nn = min(256, cpc - h0);
      const uint32_t idesc = make_idesc_bf16(kTileM, nn, false, false);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t hv = s >> 2, koff = (s & 3) * 32;
        const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
        const uint64_t b =
            make_sdesc_sw128(ka + hv * uint32_t(cpc * 128) + uint32_t(h0 * 128) + koff, 16, 1024);
        umma_bf16(tbase + uint32_t(h0), a, b, idesc, s > 0 ? 1u : 0u);
      }
    }
    umma_commit(&bar0);
  }
  if (!qok) record_error(err, DEV_TIMEOUT_TMA | DEV_K_REFINE_FUSED);
  if (ncv > 0 && !mbar_wait(&bar0, 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_REFINE_FUSED);
  tc_fence_after();
  __syncwarp();

  // row (max, sumexp) over this CTA's candidates, log2 units; the four warps
  // of a lane quadrant take every fourth 32-column chunk.  The exponentials
  // p = 2^(s - m_part) are stored back over the scores, so the column sums
  // below only rescale them by 2^(m_part - lse).
  const int quad = warp & 3, ch = warp >> 2;
  const int row = quad * 32 + lane;
  const uint32_t trow = tbase + (uint32_t(quad * 32) << 16);
  const float sl2 = scale * 1.4426950408889634f;
  const int nvc = (ncv + 31) >> 5;  // chunks up to the last valid one
  float m = -INFINITY;
  for (int k = ch; k < nvc; k += kFuseSplit) {
    const int c = k * 32;
    float v[32];
    tmem_ld32(trow + uint32_t(c), v);
    if (c + 32 > ncv) {  // the one partial chunk
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = c + i < ncv ? v[i] : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < 32; i += 2) m = fmax3f(m, v[i], v[i + 1]);
  }
  m = m == -INFINITY ? m : m * sl2;  // the scale is positive: max commutes with it
  // p = 2^(s sl2 - m) two columns at a time (one paired fma), the row sum
  // as paired adds over the valid columns
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const uint64_t nmx2 = m == -INFINITY ? f2_pack(0.f, 0.f) : f2_pack(-m, -m);
  uint64_t l2 = f2_pack(0.f, 0.f);
  for (int k = ch; k < nvc; k += kFuseSplit) {
    const int c = k * 32;
    float v[32];
    tmem_ld32(trow + uint32_t(c), v);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float t0, t1;
      f2_unpack(f2_fma(f2_pack(v[i], v[i + 1]), sl2x2, nmx2), t0, t1);
      v[i] = fast_exp2(t0);
      v[i + 1] = fast_exp2(t1);
    }
    tmem_st32(trow + uint32_t(c), v);
    if (c + 32 > ncv) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = c + i < ncv ? v[i] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 32; i += 2) l2 = f2_add(l2, f2_pack(v[i], v[i + 1]));
  }
  float l, l_hi;
  f2_unpack(l2, l, l_hi);
  l += l_hi;
  tmem_wait_st();
  part_stat[ch][row] = make_float2(m, l);
  __syncthreads();
  __cluster_barrier_wait();  // every CTA of the cluster has started
  if (ch == 0) {
    float2 a[kFuseSplit];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kFuseSplit; ++k) {
      a[k] = part_stat[k][row];
      M = fmaxf(M, a[k].x);
    }
    float Lr = 0.f;
#pragma unroll
    for (int k = 0; k < kFuseSplit; ++k)
      if (a[k].x != -INFINITY) Lr += a[k].y * fast_exp2(a[k].x - M);
#pragma unroll
    for (int c = 0; c < kFuseCtas; ++c)
      st_peer_f2(peer_addr(&peer_stat[rank][row], uint32_t(c)), make_float2(M, Lr));
  }
  cluster_sync_all();  // releases the stores above, acquires the peers'
  // row log-sum-exp over all candidates: every CTA's statistics of my row
  float lse = 0.f;
  {
    float2 st[kFuseCtas];
#pragma unroll
    for (int c = 0; c < kFuseCtas; ++c) st[c] = peer_stat[c][row];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kFuseCtas; ++c) M = fmaxf(M, st[c].x);
    float Lr = 0.f;
#pragma unroll
    for (int c = 0; c < kFuseCtas; ++c)
      if (st[c].x != -INFINITY) Lr += st[c].y * fast_exp2(st[c].x - M);
    lse = M + __log2f(Lr);
  }
  const bool row_ok = row < rows_t;
  // 2^(s - lse) = p * 2^(m_part - lse); rows past the tile's tokens contribute nothing
  const float f = (row_ok && m != -INFINITY) ? fast_exp2(m - lse) : 0.f;
  // column sums over the 128 rows: per 32-column chunk each warp sums its
  // 32 rows by a butterfly of shuffles (after the step of distance sd each
  // lane keeps the columns whose bit sd matches its own, so lane j ends
  // with column j); the four lane quadrants' sums meet in shared memory.
  // Rows past the tile's tokens are finite (zeroed or real queries) and
  // weighted 0.
  const uint64_t ff = f2_pack(f, f);
  for (int k = ch; k < nvc; k += kFuseSplit) {
    const int c = k * 32;
    float v[32];
    tmem_ld32(trow + uint32_t(c), v);
#pragma unroll
    for (int i = 0; i < 32; i += 2) f2_unpack(f2_mul(f2_pack(v[i], v[i + 1]), ff), v[i], v[i + 1]);
#pragma unroll
    for (int sd = 16; sd >= 1; sd >>= 1) {
      const bool upper = (lane & sd) != 0;
#pragma unroll
      for (int j = 0; j < sd; ++j) {
        const float lo = v[j], hi = v[j + sd];
        v[j] = (upper ? hi : lo) + __shfl_xor_sync(0xffffffffu, upper ? lo : hi, sd);
      }
    }
    colsum[quad][c + lane] = v[0];
  }
  __syncthreads();
  float* out = s2p + (size_t(mt) * gridDim.z + seg) * C;
  for (int j = threadIdx.x; j < ncv; j += kFuseThreads)
    out[c0 + j] = colsum[0][j] + colsum[1][j] + colsum[2][j] + colsum[3][j];
  // no peer touches this CTA's shared memory after the cluster barrier
  tmem_teardown(tbase, 512);
}

bool refine_fused_ok(int C) { return fuse_cpc(C) <= kFuseMaxCpc; }

// Clusters of CS CTAs of the fused refine that can be resident at once on
// the current device; cached per (device, CS).
template <int D, int CS>
static int refine_resident_clusters() {
  static std::mutex mu;
  static int cache[64];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!init) {
      for (int& c : cache) c = -1;
      init = true;
    }
    n = cache[dev];
  }
  if (n < 0) {
    n = 0;
    if (ensure_smem(refine_fused_kernel<D, CS>, FuseCfg<D>::kSmem) == cudaSuccess &&
        ensure_nonportable_cluster(refine_fused_kernel<D, CS>) == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(CS, 1, 1);
      cfg.blockDim = dim3(kFuseThreads);
      cfg.dynamicSmemBytes = FuseCfg<D>::kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CS;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, refine_fused_kernel<D, CS>, &cfg) != cudaSuccess)
        n = 0;
    }
    cudaGetLastError();
    std::lock_guard<std::mutex> lock(mu);
    cache[dev] = n;
  }
  return n;
}

// Among the cluster sizes (16, 12, 8 CTAs) whose clusters are all resident
// at once, the one with the fewest candidates per CTA (they set every
// phase of the chain), the smallest such; else 8.
template <int D>
static int refine_cluster_size(int clusters, int C) {
  int best = 8;
  for (int cs : {12, 16}) {
    const int n = cs == 16 ? refine_resident_clusters<D, 16>() : refine_resident_clusters<D, 12>();
    if (clusters <= n && fuse_cpc(C, cs) < fuse_cpc(C, best)) best = cs;
  }
  return best;
}

template <int D, int CS>
static cudaError_t launch_refine_cs(const herald_dims& dm, const uint16_t* k_cache,
                                    const int32_t* cand, const int32_t* n_cand, int C, float* s2,
                                    const WsLayout& w, uint32_t* err, const CUtensorMap& qmap,
                                    bool early, cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  const int bpt = kTileM / (dm.Hq / dm.Hkv);
  const float scale = 1.0f / sqrtf(float(dm.d));
  const int cpc = fuse_cpc(C, CS);
  HERALD_CHECK_LAUNCH(ensure_smem(refine_fused_kernel<D, CS>, FuseCfg<D>::kSmem));
  if (CS > 8) HERALD_CHECK_LAUNCH(ensure_nonportable_cluster(refine_fused_kernel<D, CS>));
  return launch_cluster_threads("refine_fused_kernel", refine_fused_kernel<D, CS>,
                                dim3(CS, w.MT_tok, segs), dim3(kFuseThreads), CS,
                                FuseCfg<D>::kSmem, st, qmap, k_cache, cand, n_cand, dm.B, dm.Hq,
                                dm.Hkv, dm.L_max, C, bpt, cpc, scale, s2, err, early ? 1 : 0);
}

template <int D>
static cudaError_t launch_refine_fused(const herald_dims& dm, const uint16_t* k_cache,
                                       const int32_t* cand, const int32_t* n_cand, int C,
                                       float* s2, const WsLayout& w, uint32_t* err,
                                       const CUtensorMap& qmap, bool early, cudaStream_t st) {
  switch (refine_cluster_size<D>(w.MT_tok * dm.N * dm.Hkv, C)) {
    case 16:
      return launch_refine_cs<D, 16>(dm, k_cache, cand, n_cand, C, s2, w, err, qmap, early, st);
    case 12:
      return launch_refine_cs<D, 12>(dm, k_cache, cand, n_cand, C, s2, w, err, qmap, early, st);
    default:
      return launch_refine_cs<D, 8>(dm, k_cache, cand, n_cand, C, s2, w, err, qmap, early, st);
  }
}

// Pass 1 -> row lse -> pass 2 (C > 4096).
template <int D>
static cudaError_t launch_refine_two_pass(const herald_dims& dm, const uint16_t* k_cache,
                                          const int32_t* cand, const int32_t* n_cand, int C,
                                          float2* rpart, float* rlse, float* s2,
                                          const WsLayout& w, uint32_t* err,
                                          const CUtensorMap& qmap, const CUtensorMap& qmap_all,
                                          int bpt, float scale, cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  HERALD_CHECK_LAUNCH(ensure_smem(refine_pass1_kernel<D>, Ref1Cfg<D>::kSmem));
  HERALD_CHECK_LAUNCH(ensure_smem(refine_pass2_kernel<D>, Ref2Cfg<D>::kSmem));
  HERALD_CHECK_LAUNCH(launch_k("refine_pass1_kernel", refine_pass1_kernel<D>,
                               dim3(w.n_chunks, w.MT_tok, segs), kTcThreads, Ref1Cfg<D>::kSmem,
                               st, qmap, k_cache, cand, n_cand, dm.B, dm.Hq, dm.Hkv, dm.L_max, C,
                               bpt, w.MT, w.n_chunks, scale, rpart, err));
  HERALD_CHECK_LAUNCH(launch_k("refine_lse_kernel", refine_lse_kernel,
                               dim3(cdiv(w.R, 8), segs), 256, 0, st, rpart, n_cand, C, w.R, w.MT,
                               w.n_chunks, rlse));
  HERALD_CHECK_LAUNCH(launch_k("refine_pass2_kernel", refine_pass2_kernel<D>,
                               dim3(cdiv(C, kRefineRows2), segs), kTcThreads, Ref2Cfg<D>::kSmem,
                               st, qmap_all, k_cache, cand, n_cand, dm.B, dm.Hq, dm.Hkv,
                               dm.L_max, C, w.R, w.MT, scale, rlse, s2, err));
  return cudaGetLastError();
}

cudaError_t launch_refine(const herald_dims& dm, const uint16_t* k_cache, const int32_t* cand,
                          const int32_t* n_cand, int C, float2* rpart, float* rlse, float* s2, const WsLayout& w, uint32_t* err,
                          const CUtensorMap* qmap, const CUtensorMap* qmap_all, cudaStream_t st,
                          bool early) {
  const float scale = 1.0f / sqrtf(float(dm.d));
  if (refine_fused_ok(C)) {
    // s2 holds one partial per row tile of whole tokens: [MT_tok][N*Hkv][C]
    if (!qmap) return cudaErrorInvalidValue;
    if (dm.d == 128)
      return launch_refine_fused<128>(dm, k_cache, cand, n_cand, C, s2, w, err, *qmap, early,
                                      st);
    return launch_refine_fused<64>(dm, k_cache, cand, n_cand, C, s2, w, err, *qmap, early, st);
  }
  if (!qmap || !qmap_all) return cudaErrorInvalidValue;
  const int bpt = kTileM / (dm.Hq / dm.Hkv);
  if (dm.d == 128)
    return launch_refine_two_pass<128>(dm, k_cache, cand, n_cand, C, rpart, rlse, s2, w, err,
                                       *qmap, *qmap_all, bpt, scale, st);
  return launch_refine_two_pass<64>(dm, k_cache, cand, n_cand, C, rpart, rlse, s2, w, err, *qmap,
                                    *qmap_all, bpt, scale, st);
}

// ================================================================== attn
template <int D>
struct AttnCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBytes = kHalves * kTileM * 128;
  static constexpr int kKBytes = kHalves * kAttnKeys * 128;
  static constexpr int kVBytes = kHalves * kAttnKeys * 128;
  static constexpr int kPBytes = 2 * kTileM * 128;  // 128 rows x 128 keys, 2 key halves
  static constexpr int kSmem = kQBytes + kKBytes + kVBytes + kPBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "attention smem exceeds the per-CTA limit");
};

template <int D>
__global__ void __launch_bounds__(kTcThreads)
    attn_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ pool_k,
                const uint16_t* __restrict__ pool_v, const int32_t* __restrict__ n_sel,
                int P_max, const uint16_t* __restrict__ block_k,
                const uint16_t* __restrict__ block_v, int B, int Hq, int Hkv, int R, int MT,
                int S_max, float scale, float* __restrict__ opart, float2* __restrict__ ml,
                uint32_t* err) {
  using Cfg = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ float red_m[2][kTileM];
  __shared__ float red_s[2][kTileM];
  uint8_t* Qs = align1024(smem_raw);
  uint8_t* Ks = Qs + Cfg::kQBytes;
  uint8_t* Vs = Ks + Cfg::kKBytes;
  uint8_t* Ps = Vs + Cfg::kVBytes;
  griddep_enter();
  const int split = blockIdx.x, mt = blockIdx.y, seg = blockIdx.z;
  const int n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int ns = min(max(n_sel[seg], 0), P_max);
  const int n_pool = (ns + kAttnKeys - 1) / kAttnKeys;
  const int n_blk = (B + kAttnKeys - 1) / kAttnKeys;
  if (split >= n_pool + n_blk) return;
  const bool from_pool = split < n_pool;
  const int k0 = from_pool ? split * kAttnKeys : (split - n_pool) * kAttnKeys;
  const int nkeys = from_pool ? min(kAttnKeys, ns - k0) : min(kAttnKeys, B - k0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  tmem_setup(&tmem_base, 256);
  const uint32_t tbase = tmem_base;

  load_rows_sw128<D>(Qs, kTileM, kTileM, q, [&](int r) -> const uint16_t* {
    const int row = mt * kTileM + r;
    if (row >= R) return nullptr;
    const int b = row / G, hl = row - (row / G) * G;
    return q + ((size_t(n) * B + b) * Hq + g * G + hl) * D;
  });
  auto key_src = [&](const uint16_t* pool, const uint16_t* blk, int r) -> const uint16_t* {
    if (r >= nkeys) return nullptr;
    if (from_pool) return pool + (size_t(seg) * P_max + k0 + r) * D;
    return blk + ((size_t(n) * B + k0 + r) * Hkv + g) * D;
  };
  load_rows_sw128<D>(Ks, kAttnKeys, kAttnKeys, block_k,
                     [&](int r) { return key_src(pool_k, block_k, r); });
  cp_async_commit();
  load_rows_sw128<D>(Vs, kAttnKeys, kAttnKeys, block_v,
                     [&](int r) { return key_src(pool_v, block_v, r); });
  cp_async_commit();
  asm volatile("cp.async.wait_group 1;" ::: "memory");  // Q and K landed
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();

  // S = Q K^T -> TMEM columns [0, 128)
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = make_idesc_bf16(kTileM, kAttnKeys, false, false);
    const uint32_t qa = smem_u32(Qs), ka = smem_u32(Ks);
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      const uint32_t hv = s >> 2, koff = (s & 3) * 32;
      const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
      const uint64_t b = make_sdesc_sw128(ka + hv * (kAttnKeys * 128) + koff, 16, 1024);
      umma_bf16(tbase, a, b, idesc, s > 0 ? 1u : 0u);
    }
    umma_commit(&bar[0]);
  }
  if (!mbar_wait(&bar[0], 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_ATTN_SPLIT);
  tc_fence_after();
  __syncwarp();

  const int quad = warp & 3, ch = warp >> 2;  // ch: key half [ch*64, ch*64+64)
  const int row = quad * 32 + lane;
  const uint32_t trow = tbase + (uint32_t(quad * 32) << 16);
  float x[64];
  {
    float v[32];
    tmem_ld32(trow + ch * 64, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = v[i];
    tmem_ld32(trow + ch * 64 + 32, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) x[32 + i] = v[i];
  }
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    x[i] = (ch * 64 + i < nkeys) ? x[i] * scale : -INFINITY;
    m = fmaxf(m, x[i]);
  }
  red_m[ch][row] = m;
  __syncthreads();
  m = fmaxf(red_m[0][row], red_m[1][row]);
  float sum = 0.f;
  uint8_t* prow = Ps + ch * (kTileM * 128);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float p[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      p[e] = __expf(x[c * 8 + e] - m);
      sum += p[e];
    }
    uint4 pk;
    pk.x = pack_bf16(p[0], p[1]);
    pk.y = pack_bf16(p[2], p[3]);
    pk.z = pack_bf16(p[4], p[5]);
    pk.w = pack_bf16(p[6], p[7]);
    *reinterpret_cast<uint4*>(prow + sw128_off(row, c)) = pk;
  }
  red_s[ch][row] = sum;
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // V landed
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // O = P V -> TMEM columns [128, 128 + D); V is the MN-major B operand
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = make_idesc_bf16(kTileM, D, false, true);
    const uint32_t pa = smem_u32(Ps), va = smem_u32(Vs);
#pragma unroll
    for (int s = 0; s < kAttnKeys / 16; ++s) {
      const uint32_t kh = s >> 2, koff = (s & 3) * 32;
      const uint64_t a = make_sdesc_sw128(pa + kh * (kTileM * 128) + koff, 16, 1024);
      const uint64_t b = make_sdesc_sw128(va + s * 2048, kAttnKeys * 128, 1024);
      umma_bf16(tbase + 128, a, b, idesc, s > 0 ? 1u : 0u);
    }
    umma_commit(&bar[1]);
  }
  if (!mbar_wait(&bar[1], 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_ATTN_SPLIT);
  tc_fence_after();
  __syncwarp();

  const size_t prow_idx = ((size_t(seg) * MT + mt) * S_max + split) * kTileM + row;
  float* op = opart + prow_idx * D;
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    float v[32];
    const int col = ch * (D / 2) + k * 32;
    tmem_ld32(trow + 128 + col, v);
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(op + col + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
  }
  if (ch == 0) ml[prow_idx] = make_float2(m, red_s[0][row] + red_s[1][row]);
  tmem_teardown(tbase, 256);
}

// ========================================================== attn_cluster
// Split-KV attention whose splits are the CS CTAs of one thread block
// cluster per (sequence, KV head, 128-row tile).  CTA rank r owns key tiles
// r and r + CS (each 128 keys: pool rows, then the B block rows); with
// CS = 16 (where the device can place 16-CTA clusters) every CTA has one
// tile, with CS = 8 some have two.  Both tiles' scores share one row max, so
// the two P.V products accumulate into one TMEM accumulator without
// rescaling.  The partial (O, max, sum) of every CTA stays in its shared
// memory; after a cluster barrier each CTA merges 128/CS rows by reading its
// peers' shared memory (distributed shared memory), and writes bf16 out.
constexpr int kClusterCtas = 8;     // portable cluster size
constexpr int kClusterCtasMax = 16; // non-portable size, used when it can be placed

template <int D>
struct AttnClCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTile = kHalves * 128 * 128;   // 128 rows x D bf16
  static constexpr int kPT = kTile > 32768 ? kTile : 32768;  // K tile, later P (128 x 128)
  static constexpr int kQ = 0;
  static constexpr int kK0 = kTile, kK1 = kTile + kPT;
  static constexpr int kV0 = kTile + 2 * kPT, kV1 = 2 * kTile + 2 * kPT;
  static constexpr int kBytes = 3 * kTile + 2 * kPT;
  static constexpr int kORow = D + 4;                  // fp32 row stride of the O partial
  static constexpr int kSmem = kBytes + 1024;
  static_assert(128 * kORow * 4 <= kTile + 2 * kPT, "O partial must fit over Q, P0, P1");
  static_assert(kV1 + kTile == kBytes, "cluster attention smem layout");
  static_assert(kSmem <= 227 * 1024, "cluster attention smem exceeds the per-CTA limit");
};

template <int D, int CS>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_cluster_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ pool_k,
                        const uint16_t* __restrict__ pool_v, const int32_t* __restrict__ n_sel,
                        int P_max, const uint16_t* __restrict__ block_k,
                        const uint16_t* __restrict__ block_v, int B, int Hq, int Hkv, int R,
                        float scale, uint16_t* __restrict__ out, uint32_t* err) {
  using Cfg = AttnClCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ float red_m[2][kTileM];
  __shared__ float red_s[2][kTileM];
  __shared__ float2 ml[kTileM];
  uint8_t* base = align1024(smem_raw);
  uint8_t* Qs = base + Cfg::kQ;
  uint8_t* Ks[2] = {base + Cfg::kK0, base + Cfg::kK1};
  uint8_t* Vs[2] = {base + Cfg::kV0, base + Cfg::kV1};
  float* Os = reinterpret_cast<float*>(base);  // reuses Q, K0, K1 after the MMAs
  const uint32_t rank = cluster_ctarank();
  const int mt = blockIdx.y, seg = blockIdx.z;
  const int n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  tmem_setup(&tmem_base, 512);
  const uint32_t tbase = tmem_base;
  griddep_enter();
  const int ns = min(max(n_sel[seg], 0), P_max);
  const int n_pool = (ns + kAttnKeys - 1) / kAttnKeys;
  const int n_tiles = n_pool + (B + kAttnKeys - 1) / kAttnKeys;
  // this CTA's tiles: t0 = rank, t1 = rank + CS (scalars, not arrays, so
  // that they stay in registers)
  const int t0 = int(rank), t1 = int(rank) + CS;
  const int nt = (t0 < n_tiles) + (t1 < n_tiles);
  auto tile_keys = [&](int t) {
    return t < n_pool ? min(kAttnKeys, ns - t * kAttnKeys)
                      : min(kAttnKeys, B - (t - n_pool) * kAttnKeys);
  };
  const int nk0 = nt > 0 ? tile_keys(t0) : 0, nk1 = nt > 1 ? tile_keys(t1) : 0;
  const int quad = warp & 3, ch = warp >> 2;
  const int row = quad * 32 + lane;
  const uint32_t trow = tbase + (uint32_t(quad * 32) << 16);
  float m = -INFINITY, lsum = 0.f;

  if (nt > 0) {
    load_rows_sw128<D>(Qs, kTileM, kTileM, q, [&](int r) -> const uint16_t* {
      const int rr = mt * kTileM + r;
      if (rr >= R) return nullptr;
      const int b = rr / G, hl = rr - (rr / G) * G;
      return q + ((size_t(n) * B + b) * Hq + g * G + hl) * D;
    });
    for (int k = 0; k < nt; ++k) {
      const int t = k ? t1 : t0, cnt = k ? nk1 : nk0;
      const bool pool_tile = t < n_pool;
      const int k0 = pool_tile ? t * kAttnKeys : (t - n_pool) * kAttnKeys;
      load_rows_sw128<D>(Ks[k], kAttnKeys, kAttnKeys, block_k, [&](int r) -> const uint16_t* {
        if (r >= cnt) return nullptr;
        return pool_tile ? pool_k + (size_t(seg) * P_max + k0 + r) * D
                         : block_k + ((size_t(n) * B + k0 + r) * Hkv + g) * D;
      });
    }
    cp_async_commit();
    for (int k = 0; k < nt; ++k) {
      const int t = k ? t1 : t0, cnt = k ? nk1 : nk0;
      const bool pool_tile = t < n_pool;
      const int k0 = pool_tile ? t * kAttnKeys : (t - n_pool) * kAttnKeys;
      load_rows_sw128<D>(Vs[k], kAttnKeys, kAttnKeys, block_v, [&](int r) -> const uint16_t* {
        if (r >= cnt) return nullptr;
        return pool_tile ? pool_v + (size_t(seg) * P_max + k0 + r) * D
                         : block_v + ((size_t(n) * B + k0 + r) * Hkv + g) * D;
      });
    }
    cp_async_commit();
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    fence_proxy_async_smem();
    __syncthreads();
    tc_fence_after();
    // S_k = Q K_k^T -> TMEM columns [128k, 128k + 128)
    if (threadIdx.x == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kTileM, kAttnKeys, false, false);
      const uint32_t qa = smem_u32(Qs);
      for (int k = 0; k < nt; ++k) {
        const uint32_t ka = smem_u32(Ks[k]);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t hv = s >> 2, koff = (s & 3) * 32;
          const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
          const uint64_t b = make_sdesc_sw128(ka + hv * (kAttnKeys * 128) + koff, 16, 1024);
          umma_bf16(tbase + 128 * k, a, b, idesc, s > 0 ? 1u : 0u);
        }
      }
      umma_commit(&bar[0]);
    }
    if (!mbar_wait(&bar[0], 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_ATTN_CLUSTER);
    tc_fence_after();
    __syncwarp();
    // scores of both tiles -> one row max
    float x[2][64];
    for (int k = 0; k < 2; ++k) {
      if (k >= nt) break;
      float v[32];
      tmem_ld32(trow + 128 * k + ch * 64, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[k][i] = v[i];
      tmem_ld32(trow + 128 * k + ch * 64 + 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) x[k][32 + i] = v[i];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        x[k][i] = (ch * 64 + i < (k ? nk1 : nk0)) ? x[k][i] * scale : -INFINITY;
        m = fmaxf(m, x[k][i]);
      }
    }
    red_m[ch][row] = m;
    __syncthreads();
    m = fmaxf(red_m[0][row], red_m[1][row]);
    // P_k = exp(S_k - m) as bf16 over K_k's buffer (K-major A operand)
    for (int k = 0; k < 2; ++k) {
      if (k >= nt) break;
      uint8_t* prow = Ks[k] + ch * (kTileM * 128);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = __expf(x[k][c * 8 + e] - m);
          lsum += p[e];
        }
        uint4 pk;
        pk.x = pack_bf16(p[0], p[1]);
        pk.y = pack_bf16(p[2], p[3]);
        pk.z = pack_bf16(p[4], p[5]);
        pk.w = pack_bf16(p[6], p[7]);
        *reinterpret_cast<uint4*>(prow + sw128_off(row, c)) = pk;
      }
    }
    red_s[ch][row] = lsum;
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // O = sum_k P_k V_k -> TMEM columns [256, 256 + D)
    if (threadIdx.x == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kTileM, D, false, true);
      for (int k = 0; k < nt; ++k) {
        const uint32_t pa = smem_u32(Ks[k]), va = smem_u32(Vs[k]);
#pragma unroll
        for (int s = 0; s < kAttnKeys / 16; ++s) {
          const uint32_t kh = s >> 2, koff = (s & 3) * 32;
          const uint64_t a = make_sdesc_sw128(pa + kh * (kTileM * 128) + koff, 16, 1024);
          const uint64_t b = make_sdesc_sw128(va + s * 2048, kAttnKeys * 128, 1024);
          umma_bf16(tbase + 256, a, b, idesc, (k > 0 || s > 0) ? 1u : 0u);
        }
      }
      umma_commit(&bar[1]);
    }
    if (!mbar_wait(&bar[1], 0)) record_error(err, DEV_TIMEOUT_MMA | DEV_K_ATTN_CLUSTER);
    tc_fence_after();
    __syncwarp();
    // O partial -> shared memory (row-major fp32, padded rows)
#pragma unroll
    for (int k = 0; k < D / 64; ++k) {
      float v[32];
      const int col = ch * (D / 2) + k * 32;
      tmem_ld32(trow + 256 + col, v);
      float* orow = Os + row * Cfg::kORow + col;
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(orow + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    if (ch == 0) ml[row] = make_float2(m, red_s[0][row] + red_s[1][row]);
  } else {
    if (ch == 0) ml[row] = make_float2(-INFINITY, 0.f);
  }
  cluster_sync_all();
  // merge: this CTA finalises rows [rank*RPC, (rank+1)*RPC); every peer
  // value of a row is requested before any is used (one remote round trip)
  constexpr int RPC = kTileM / CS;             // rows per CTA
  constexpr int E = D / 32;                    // features per lane
  for (int rr = warp; rr < RPC; rr += kTcThreads / 32) {
    const int lr = int(rank) * RPC + rr;
    const int grow = mt * kTileM + lr;
    float2 pm[CS];
    float o[CS][E];
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      pm[c] = ld_peer_f2(peer_addr(&ml[lr], uint32_t(c)));
      const uint32_t a = peer_addr(Os + lr * Cfg::kORow + lane * E, uint32_t(c));
      if constexpr (E == 4) {
        const float4 f = ld_peer_f4(a);
        o[c][0] = f.x; o[c][1] = f.y; o[c][2] = f.z; o[c][3] = f.w;
      } else {
        const float2 f = ld_peer_f2(a);
        o[c][0] = f.x; o[c][1] = f.y;
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < CS; ++c) M = fmaxf(M, pm[c].x);
    float acc[E] = {};
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      const float wgt = pm[c].x == -INFINITY ? 0.f : __expf(pm[c].x - M);
      L += wgt * pm[c].y;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += wgt == 0.f ? 0.f : wgt * o[c][e];
    }
    if (grow < R) {
      const int b = grow / G, h = g * G + (grow - (grow / G) * G);
      uint16_t* dst = out + ((size_t(n) * B + b) * Hq + h) * D + lane * E;
      const float inv = 1.f / L;
#pragma unroll
      for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    }
  }
  cluster_sync_all();  // peers may still be reading this CTA's partial
  tmem_teardown(tbase, 512);
}

// ============================================================= attn_pool
// Sparse block attention, one cluster of CS = 8 or 16 CTAs per (sequence,
// KV head, row tile of bpt whole tokens = bpt*G <= 128 query rows).  The
// pool is split evenly: CTA r owns pool keys [r*kpc, (r+1)*kpc) (kpc =
// ceil(P_max/CS) rounded to 16, kpc + B <= 256), loaded by two 2-D TMA boxes each for K and
// V; the last CTA also owns the B block keys.  The query tile and the block
// keys and values are 3-D TMA boxes (every operand is one bulk transfer,
// issued by one thread as soon as the predecessor kernel is done).  Each
// CTA computes S = Q K^T for its keys with one UMMA (N = kpc), P = exp(S -
// rowmax) in bf16 (packed into TMEM over S, chunk j of 16 keys in columns
// [8j, 8j + 8), once every S column has been read), O = P V into TMEM with
// P read from TMEM.  Rows are finalised 128/CS per CTA: each CTA stages
// its O rows divided by their row sums (fp16) over the dead operands and
// pushes rows [c*128/CS, (c+1)*128/CS) with their (max, sum) to CTA c by
// bulk shared::cta -> shared::cluster copies that complete on c's mbarrier;
// each CTA merges its rows once all CS slices have landed.  16-CTA clusters
// (a non-portable size) halve each CTA's keys -- its UMMAs and its share of
// the exponentials -- where every cluster of the launch is resident at once.  The receive
// buffers have shared memory of their own, so no cluster-wide barrier
// separates the attention from the exchange.  Only the 16-key chunks that
// hold a valid key enter S, the softmax and P V.  Two options of the entry
// point: the pool keys loaded before the grid-dependency wait (steps after
// a block's first, when the pool is settled), and the append of the block
// to the cache by one cluster per sequence (the last step).
constexpr int kPoolMaxB = 64;
// S takes TMEM columns [0, kpc + Bp) and O starts at column 256
constexpr int kPoolMaxCols = 256;
// 16 warps: four per TMEM lane quadrant share each row's softmax and its
// O columns (the CTA holds its SM alone either way)
constexpr int kPoolThreads = 512;
constexpr int kPoolSplit = kPoolThreads / 128;  // warps per lane quadrant

struct PoolSmem {
  uint32_t q, k, kb, v, vb, recv_o, recv_ml, total;
};
// Rows each CTA of a cs-CTA cluster finalises (even, so that every slice
// of (max, sum) pairs is a whole number of 16-byte units).
__host__ __device__ constexpr int pool_rows_per_cta(int cs) {
  return ((kTileM + cs - 1) / cs + 1) & ~1;
}

__host__ __device__ inline PoolSmem pool_smem(int D, int kpc, int Bp, int cs) {
  const uint32_t H = uint32_t(D / 64);
  PoolSmem L;
  // region A: Q | K | K_block, later the staged O rows (fp16, D + 8 apart)
  L.q = 0;
  L.k = H * 128u * 128u;
  L.kb = L.k + H * uint32_t(kpc) * 128u;
  const uint32_t a_end = L.kb + H * uint32_t(Bp) * 128u;
  const uint32_t o_end = uint32_t(kTileM) * uint32_t(D + 8) * 2u;
  L.v = ((a_end > o_end ? a_end : o_end) + 1023u) & ~1023u;
  L.vb = L.v + H * uint32_t(kpc) * 128u;
  L.recv_o = L.vb + H * uint32_t(Bp) * 128u;
  // one slice of pool_rows_per_cta(cs) rows from each of the cs CTAs
  const uint32_t recv_rows = uint32_t(cs * pool_rows_per_cta(cs));
  L.recv_ml = L.recv_o + recv_rows * uint32_t(D + 8) * 2u;
  L.total = L.recv_ml + recv_rows * 8u + 1024u;
  return L;
}

template <int D, int CS>
__global__ void __launch_bounds__(kPoolThreads, 1)
    attn_pool_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap bkmap,
                     const __grid_constant__ CUtensorMap bvmap,
                     const int32_t* __restrict__ n_sel, int P_max, int B, int Hq, int Hkv,
                     int bpt, int kpc, float scale, int settled, uint16_t* __restrict__ out,
                     uint32_t* err, AppendArgs app, int L_max) {
  constexpr int H = D / 64;
  constexpr int OROW = D + 8;  // fp16 row stride of O partials (16-byte padding)
  constexpr int kPoolCtas = CS;
  constexpr int kPoolRows = pool_rows_per_cta(CS);  // rows finalised per CTA (the last ones fewer)
  static_assert(CS == 8 || CS == 12 || CS == 16, "pool attention clusters of 8, 12 or 16 CTAs");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t barK, barV, bar0, bar1, barR;
  __shared__ uint32_t tmem_base;
  __shared__ float red_m[kPoolSplit][kTileM];
  __shared__ float red_s[kPoolSplit][kTileM];
  __shared__ __align__(16) float2 ml[kTileM];
  constexpr uint32_t kSliceO = uint32_t(kPoolRows * OROW * 2);  // receive slot per sender
  constexpr uint32_t kSliceMl = uint32_t(kPoolRows * 8);
  const int Bp = (B + 15) & ~15;
  const PoolSmem S = pool_smem(D, kpc, Bp, CS);
  uint8_t* base = align1024(smem_raw);
  uint8_t* Qs = base + S.q;
  uint8_t* Ks = base + S.k;
  uint8_t* Kb = base + S.kb;
  uint8_t* Vs = base + S.v;
  uint8_t* Vb = base + S.vb;
  uint16_t* recv_o = reinterpret_cast<uint16_t*>(base + S.recv_o);
  float2* recv_ml = reinterpret_cast<float2*>(base + S.recv_ml);
  const uint32_t rank = cluster_ctarank();
  const int mt = blockIdx.y, seg = blockIdx.z;
  const int n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rows [c*kPoolRows, c*kPoolRows + rows_of(c)) are finalised by CTA c
  auto rows_of = [](int c) { return min(max(kTileM - c * kPoolRows, 0), kPoolRows); };
  const int my_rows = rows_of(int(rank));
  if (threadIdx.x == 0) {
    mbar_init(&barK, 1);
    mbar_init(&barV, 1);
    mbar_init(&bar0, 1);
    mbar_init(&bar1, 1);
    mbar_init(&barR, 1);
    mbar_arrive_expect_tx(&barR, uint32_t(kPoolCtas * my_rows) * uint32_t(OROW * 2 + 8));
    fence_mbar_init();
  }
  // peers' copies complete on barR: its initialisation is published
  // cluster-wide here and awaited just before the first copy is issued
  __cluster_barrier_arrive_relaxed();
  if (threadIdx.x == 0) {  // kernel parameters: independent of the predecessor
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&bkmap);
    tma_prefetch_desc(&bvmap);
  }
  tmem_setup(&tmem_base, 512);
  const uint32_t tbase = tmem_base;
  const int b0 = mt * bpt;                  // first token of the tile
  const int rows_t = min(bpt, B - b0) * G;  // query rows of the tile
  const uint32_t qbytes = uint32_t(H * G * bpt * 128);
  const int k0 = int(rank) * kpc;
  const bool has_blk = rank == kPoolCtas - 1 && B > 0;  // the block keys
  // barK: Q + pool K + block K (last CTA); barV: pool V + block V.  The
  // pool slices are loaded whole whatever n_sel is (rows past it are never
  // used), so no load waits for n_sel; boxes past the tensor's end are
  // zero-filled, and rows past this tile's tokens are never used either.
  const uint32_t kb = uint32_t(H * kpc * 128);
  const uint32_t bb = has_blk ? uint32_t(H * Bp * 128) : 0u;
  auto pool_k_loads = [&]() {  // thread 0: the expected bytes + the pool keys
    mbar_arrive_expect_tx(&barK, qbytes + kb + bb);
    mbar_arrive_expect_tx(&barV, kb + bb);
#pragma unroll
    for (int hv = 0; hv < H; ++hv)
      tma_load_2d(Ks + hv * kpc * 128, &kmap, &barK, hv * 64, seg * P_max + k0);
  };
  // settled != 0: the caller guarantees that the pool was written before the
  // previous launch on the stream began; that launch started this one only
  // after waiting for its own predecessor (every kernel here does), so the
  // pool is final: fetch its keys while the predecessor finishes.
  if (settled && threadIdx.x == 0) pool_k_loads();
  griddep_enter();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int hv = 0; hv < H; ++hv)
      tma_load_3d(Qs + hv * kTileM * 128, &qmap, &barK, hv * 64, g * G, n * B + b0);
    if (!settled) pool_k_loads();
    if (has_blk) {
#pragma unroll
      for (int hv = 0; hv < H; ++hv)
        tma_load_3d(Kb + hv * Bp * 128, &bkmap, &barK, hv * 64, g, n * B);
    }
#pragma unroll
    for (int hv = 0; hv < H; ++hv)
      tma_load_2d(Vs + hv * kpc * 128, &vmap, &barV, hv * 64, seg * P_max + k0);
    if (has_blk) {
#pragma unroll
      for (int hv = 0; hv < H; ++hv)
        tma_load_3d(Vb + hv * Bp * 128, &bvmap, &barV, hv * 64, g, n * B);
    }
  }
  const int nkp = min(max(min(max(n_sel[seg], 0), P_max) - k0, 0), kpc);  // valid pool keys
  debug_flag(threadIdx.x == 0 && (n_sel[seg] < 0 || n_sel[seg] > P_max), DEV_BAD_COUNT);
  const bool any = nkp > 0 || has_blk;
  // The fused append (app.bk set): per sequence, the CS CTAs of the cluster
  // of the first row tile of KV head 0 copy the block's rows of every KV
  // head into the cache, a share each, while their operands are in
  // flight.  No other CTA reads ctx.  CTA 0 advances it once every peer's
  // partial has landed: each peer pushes after all its threads have read it.
  const bool appender = app.bk != nullptr && mt == 0 && g == 0;
  int L0 = 0;
  if (appender) {
    debug_flag(threadIdx.x == 0 && (app.ctx[n] < 0 || app.ctx[n] > L_max), DEV_BAD_COUNT);
    L0 = min(max(app.ctx[n], 0), L_max);
    append_block_rows<1>(app.bk, app.bv, n, B, Hkv, D, L_max, L0, app.kc, app.vc,
                         int(rank) * kPoolThreads + threadIdx.x, kPoolCtas * kPoolThreads);
  }

  // S = Q [K ; K_block]^T -> TMEM columns [0, kpc) and [kpc, kpc + Bp).
  // Every CTA waits for its query tile, used or not: no copy may still be
  // writing this CTA's shared memory when it exits.
  bool ok = true;
  if (threadIdx.x == 0) ok = mbar_wait(&barK, 0);
  if (threadIdx.x == 0 && any) {
    const uint32_t qa = smem_u32(Qs);
    tc_fence_after();
    if (nkp > 0) {  // the pool rows up to the last 16-key chunk holding a valid key
      const uint32_t idesc = make_idesc_bf16(kTileM, (nkp + 15) & ~15, false, false);
      const uint32_t ka = smem_u32(Ks);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t hv = s >> 2, koff = (s & 3) * 32;
        const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
        const uint64_t b = make_sdesc_sw128(ka + hv * (kpc * 128) + koff, 16, 1024);
        umma_bf16(tbase, a, b, idesc, s > 0 ? 1u : 0u);
      }
    }
    if (has_blk) {
      const uint32_t idesc = make_idesc_bf16(kTileM, Bp, false, false);
      const uint32_t ka = smem_u32(Kb);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const uint32_t hv = s >> 2, koff = (s & 3) * 32;
        const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
        const uint64_t b = make_sdesc_sw128(ka + hv * (Bp * 128) + koff, 16, 1024);
        umma_bf16(tbase + uint32_t(kpc), a, b, idesc, s > 0 ? 1u : 0u);
      }
    }
    umma_commit(&bar0);
  }
  // every thread waits for the commit: after it Q, K and K_block are dead
  // and P may be written over them
  if (any && !mbar_wait(&bar0, 0)) ok = false;
  tc_fence_after();
  __syncwarp();

  // softmax over this CTA's columns, in log2 units, over the 16-key chunks
  // that hold a valid key (pool chunks, then block chunks), split between
  // the kPoolSplit warps that share a TMEM lane quadrant
  const int quad = warp & 3, ch = warp >> 2;
  const int row = quad * 32 + lane;
  const uint32_t trow = tbase + (uint32_t(quad * 32) << 16);
  const int npc = (nkp + 15) >> 4;                // pool chunks
  const int nbc = has_blk ? (B + 15) >> 4 : 0;   // block chunks
  const int nchunks = npc + nbc;
  const int per = (nchunks + kPoolSplit - 1) / kPoolSplit;
  const int c_begin = min(ch * per, nchunks), cnt = min(per, nchunks - c_begin);
  constexpr int kMaxChunks = kPoolMaxCols / (16 * kPoolSplit);  // 16-column chunks per warp
  const float sl2 = scale * 1.4426950408889634f;              // scores -> log2 units
  float x[kMaxChunks][16];
  int nv[kMaxChunks];  // valid keys per chunk (warp-uniform)
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int j = c_begin + c;
    const bool pool_j = j < npc;
    nv[c] = c >= cnt ? 0 : pool_j ? min(nkp - j * 16, 16) : min(B - (j - npc) * 16, 16);
    if (c < cnt) {
      const int col = pool_j ? j * 16 : kpc + (j - npc) * 16;
      uint32_t* r = reinterpret_cast<uint32_t*>(x[c]);
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
          "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
          : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
            "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
            "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
          : "r"(trow + uint32_t(col)));
    }
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  // the row max of the raw scores (a positive scale keeps the arg max), the
  // keys past the valid ones set to -inf in the one partial chunk
  float m = -INFINITY;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    if (c < cnt) {
      if (nv[c] < 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[c][i] = i < nv[c] ? x[c][i] : -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < 16; i += 2) m = fmax3f(m, x[c][i], x[c][i + 1]);
    }
  }
  red_m[ch][row] = m;
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kPoolSplit; ++k) m = fmaxf(m, red_m[k][row]);
  m *= sl2;                                        // log2 units; -inf stays -inf
  const float mm = m == -INFINITY ? 0.f : m;      // no valid key: every p is 2^-inf = 0
  // p = 2^(x sl2 - m): the scaling and the shift as one paired fma for two
  // keys, the row sum as paired adds
  const uint64_t sl2x2 = f2_pack(sl2, sl2), nmx2 = f2_pack(-mm, -mm);
  uint64_t lsum2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    if (c < cnt) {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float t0, t1;
        f2_unpack(f2_fma(f2_pack(x[c][2 * i], x[c][2 * i + 1]), sl2x2, nmx2), t0, t1);
        const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
        lsum2 = f2_add(lsum2, f2_pack(p0, p1));
        pk[i] = pack_bf16(p0, p1);
      }
      const int j = c_begin + c;
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
              trow + uint32_t(j * 8)),
          "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]),
          "r"(pk[7])
          : "memory");
    }
  }
  float lsum, lsum_hi;
  f2_unpack(lsum2, lsum, lsum_hi);
  lsum += lsum_hi;
  red_s[ch][row] = lsum;
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // O = P V (+ P_block V_block) -> TMEM columns [256, 256 + D)
  if (threadIdx.x == 0 && any) {
    constexpr uint32_t idesc = make_idesc_bf16(kTileM, D, false, true);
    bool acc = false;
    ok = mbar_wait(&barV, 0) && ok;
    tc_fence_after();
    if (nkp > 0) {  // P of the pool chunks: TMEM columns [0, 8 npc)
      const uint32_t va = smem_u32(Vs);
      for (int s = 0; s < npc; ++s) {
        const uint64_t b = make_sdesc_sw128(va + uint32_t(s) * 2048u, uint32_t(kpc) * 128u, 1024);
        umma_bf16_ts(tbase + 256, tbase + uint32_t(s * 8), b, idesc, acc ? 1u : 0u);
        acc = true;
      }
    }
    if (has_blk) {  // P of the block chunks: the next 8 nbc columns
      const uint32_t va = smem_u32(Vb);
      for (int s = 0; s < nbc; ++s) {
        const uint64_t b = make_sdesc_sw128(va + uint32_t(s) * 2048u, uint32_t(Bp) * 128u, 1024);
        umma_bf16_ts(tbase + 256, tbase + uint32_t((npc + s) * 8), b, idesc, acc ? 1u : 0u);
        acc = true;
      }
    }
    umma_commit(&bar1);
  }
  // a CTA without keys still lets its value copies land before it exits
  if (threadIdx.x == 0 && !any) ok = mbar_wait(&barV, 0) && ok;
  if (any && !mbar_wait(&bar1, 0)) ok = false;
  tc_fence_after();
  __syncwarp();
  if (!ok) record_error(err, DEV_TIMEOUT_MMA | DEV_K_ATTN_POOL);

  // O partial -> shared memory over the dead Q/K operands (dead since S):
  // each row divided by its sum and stored as fp16 (|o / l| <= max |v|); the
  // merge re-weights by (max, sum), which stay fp32
  float lrow = 0.f;
#pragma unroll
  for (int k = 0; k < kPoolSplit; ++k) lrow += red_s[k][row];
  uint16_t* Os = reinterpret_cast<uint16_t*>(base);
  if (any) {  // D / kPoolSplit columns of the row per warp
    const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
    uint16_t* orow = Os + row * OROW;
    constexpr int kW = D / kPoolSplit;
    static_assert(kW == 16 || kW == 32, "16 or 32 O columns per warp");
    float v[kW];
    const int col = ch * kW;
    if constexpr (kW == 32)
      tmem_ld32(trow + 256 + uint32_t(col), v);
    else
      tmem_ld16(trow + 256 + uint32_t(col), v);
    {
#pragma unroll
      for (int i = 0; i < kW; i += 8) {
        uint4 h;
        h.x = pack_half2(v[i] * inv, v[i + 1] * inv);
        h.y = pack_half2(v[i + 2] * inv, v[i + 3] * inv);
        h.z = pack_half2(v[i + 4] * inv, v[i + 5] * inv);
        h.w = pack_half2(v[i + 6] * inv, v[i + 7] * inv);
        *reinterpret_cast<uint4*>(orow + col + i) = h;
      }
    }
  }
  if (ch == 0) ml[row] = make_float2(m, any ? lrow : 0.f);
  fence_proxy_async_smem();  // the partial is read by bulk copies (async proxy)
  __syncthreads();
  __cluster_barrier_wait();  // every peer's barR is initialised

  // push: rows [c*kPoolRows, c*kPoolRows + rows_of(c)) of this CTA's
  // partial go to CTA c, slot `rank`
  if (threadIdx.x == 0) {
    for (uint32_t c = 0; c < uint32_t(kPoolCtas); ++c) {
      const uint32_t rc = uint32_t(rows_of(int(c)));
      if (rc == 0) continue;
      const uint32_t mb = cluster_addr(&barR, c);
      bulk_copy_to_peer(cluster_addr(reinterpret_cast<uint8_t*>(recv_o) + rank * kSliceO, c),
                        Os + c * kPoolRows * OROW, rc * uint32_t(OROW * 2), mb);
      bulk_copy_to_peer(cluster_addr(reinterpret_cast<uint8_t*>(recv_ml) + rank * kSliceMl, c),
                        &ml[c * kPoolRows], rc * 8u, mb);
    }
    bulk_commit();
  }
  if (!mbar_wait(&barR, 0)) {
    record_error(err, DEV_TIMEOUT_TMA | DEV_K_ATTN_POOL);
    // a peer whose own wait ran out pushes late: this CTA must not exit
    // (its shared memory is the copies' destination) before they land
    mbar_wait(&barR, 0, 20ull * kWaitLimitNs);
  } else if (appender && app.advance && rank == 0 && threadIdx.x == 0) {
    app.ctx[n] = min(L0 + B, L_max);
  }

  // merge this CTA's rows from the CS received partials:
  // out = sum_c 2^(m_c - M) l_c (o_c / l_c) / sum_c 2^(m_c - M) l_c
  constexpr int E = D / 32;
  for (int rr = warp; rr < my_rows; rr += kPoolThreads / 32) {
    const int lr = int(rank) * kPoolRows + rr;
    if (lr >= rows_t) break;  // warp-uniform: rows past the tile's tokens
    const int grow = b0 * G + lr;
    float M = -INFINITY;
    float2 pm[kPoolCtas];
#pragma unroll
    for (int c = 0; c < kPoolCtas; ++c) {
      pm[c] = recv_ml[c * kPoolRows + rr];
      M = fmaxf(M, pm[c].x);
    }
    float acc[E] = {};
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < kPoolCtas; ++c) {
      if (pm[c].x == -INFINITY || pm[c].y <= 0.f) continue;
      const float wgt = fast_exp2(pm[c].x - M) * pm[c].y;
      L += wgt;
      const __half* o = reinterpret_cast<const __half*>(recv_o + (c * kPoolRows + rr) * OROW) +
                        lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += wgt * __half2float(o[e]);
    }
    {
      const int b = grow / G, h = g * G + (grow - (grow / G) * G);
      uint16_t* dstp = out + ((size_t(n) * B + b) * Hq + h) * D + lane * E;
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t*>(dstp + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    }
  }
  if (threadIdx.x == 0) bulk_wait_read_all();  // outgoing copies have read the partial
  tmem_teardown(tbase, 512);
}

// =========================================================== attn_combine
// One warp per output row (n, b, h); lane owns D/32 consecutive features.
template <int D>
__global__ void __launch_bounds__(256)
    attn_combine_kernel(const float* __restrict__ opart, const float2* __restrict__ ml,
                        const int32_t* __restrict__ n_sel, int P_max, int N, int B, int Hq,
                        int Hkv, int MT, int S_max, uint16_t* __restrict__ out) {
  constexpr int E = D / 32;
  griddep_enter();
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw >= N * B * Hq) return;
  const int n = gw / (B * Hq), b = (gw / Hq) % B, h = gw % Hq;
  const int G = Hq / Hkv, g = h / G, r = b * G + (h - g * G);
  const int mt = r / kTileM, i = r % kTileM, seg = n * Hkv + g;
  const int ns = min(max(n_sel[seg], 0), P_max);
  const int nsp = (ns + kAttnKeys - 1) / kAttnKeys + (B + kAttnKeys - 1) / kAttnKeys;
  const size_t base = (size_t(seg) * MT + mt) * S_max;
  float M = -INFINITY;
  for (int s = 0; s < nsp; ++s) M = fmaxf(M, ml[(base + s) * kTileM + i].x);
  float acc[E] = {};
  float L = 0.f;
  for (int s = 0; s < nsp; ++s) {
    const float2 p = ml[(base + s) * kTileM + i];
    const float w = __expf(p.x - M);
    L += w * p.y;
    const float* o = opart + ((base + s) * kTileM + i) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += w * o[e];
  }
  const float inv = 1.f / L;
  uint16_t* dst = out + size_t(gw) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const uint32_t pk = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + e) = pk;
  }
}

// The cluster kernel covers up to 2 * 8 key tiles (P_max + B up to 2048
// keys); larger pools use the split kernel plus a combine pass.
// HERALD_ATTN_SPLIT=1 in the environment forces the split path (testing).
static bool force_split() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("HERALD_ATTN_SPLIT");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}


// How many clusters of CS CTAs of the attention kernel can be resident at
// once on this device (a 16-CTA cluster needs 16 free SMs of one GPC).
// Cached per device and cluster size.
template <int D, int CS>
static int max_active_clusters() {
  static int cache[64];
  static bool init = false;
  if (!init) {
    for (int& c : cache) c = -1;
    init = true;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] < 0) {
    int n = 0;
    if (CS <= 8 || cudaFuncSetAttribute(attn_cluster_kernel<D, CS>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(CS, 1, 1);
      cfg.blockDim = dim3(kTcThreads);
      cfg.dynamicSmemBytes = AttnClCfg<D>::kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CS;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel<D, CS>, &cfg) != cudaSuccess)
        n = 0;
    }
    cudaGetLastError();
    cache[dev] = n;
  }
  return cache[dev];
}

// How many CS-CTA clusters of the pool attention kernel with `smem` bytes of
// dynamic shared memory can be resident at once (a 16-CTA cluster needs 16
// free SMs of one GPC); cached per device for the last few sizes asked.
// The kernel's shared-memory grant (and, for 16, the non-portable cluster
// size) is made first: the query needs it.
template <int D, int CS>
static int pool_resident_clusters(uint32_t smem) {
  struct Entry {
    int dev;
    uint32_t smem;
    int n;
  };
  static Entry cache[8] = {};
  static int next = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
      if (e.n > 0 && e.dev == dev && e.smem == smem) return e.n;
  }
  if (ensure_smem(attn_pool_kernel<D, CS>, smem) != cudaSuccess ||
      (CS > 8 && ensure_nonportable_cluster(attn_pool_kernel<D, CS>) != cudaSuccess)) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(CS, 1, 1);
  cfg.blockDim = dim3(kPoolThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_pool_kernel<D, CS>, &cfg) != cudaSuccess) n = 0;
  cudaGetLastError();
  if (n > 0) {
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{dev, smem, n};
    next = (next + 1) % 8;
  }
  return n;
}

// Pool keys per CTA: the pool and the block keys (which the last CTA takes
// after its share of the pool) split evenly, in whole 16-key chunks.
int attn_pool_kpc(int P_max, int B, int cs) {
  return cdiv(cdiv(P_max + ((B + 15) & ~15), cs), 16) * 16;
}
int attn_pool_bpt(const herald_dims& dm) { return kTileM / (dm.Hq / dm.Hkv); }

static uint32_t attn_pool_smem(const herald_dims& dm, int P_max, int cs) {
  return pool_smem(dm.d, attn_pool_kpc(P_max, dm.B, cs), (dm.B + 15) & ~15, cs).total;
}

static bool attn_pool_fits(const herald_dims& dm, int P_max, int cs) {
  const int kpc = attn_pool_kpc(P_max, dm.B, cs);
  const int Bp = (dm.B + 15) & ~15;
  // the dynamic allocation plus the kernel's static shared memory (~3 KB)
  return kpc + Bp <= kPoolMaxCols && Bp <= kPoolMaxB &&
         attn_pool_smem(dm, P_max, cs) <= 220u * 1024u;
}

static int pool_resident(const herald_dims& dm, int P_max, int cs) {
  const uint32_t smem = attn_pool_smem(dm, P_max, cs);
  if (dm.d == 128)
    return cs == 16   ? pool_resident_clusters<128, 16>(smem)
           : cs == 12 ? pool_resident_clusters<128, 12>(smem)
                      : pool_resident_clusters<128, 8>(smem);
  return cs == 16   ? pool_resident_clusters<64, 16>(smem)
         : cs == 12 ? pool_resident_clusters<64, 12>(smem)
                    : pool_resident_clusters<64, 8>(smem);
}

int attn_pool_cs(const herald_dims& dm, int P_max, int choice, int sm_budget) {
  const bool f8 = attn_pool_fits(dm, P_max, 8), f12 = attn_pool_fits(dm, P_max, 12),
             f16 = attn_pool_fits(dm, P_max, 16);
  if (choice == 6) return f8 ? 8 : 0;
  if (choice == 7) return f16 && pool_resident(dm, P_max, 16) > 0 ? 16 : 0;
  if (choice == 8) return f12 && pool_resident(dm, P_max, 12) > 0 ? 12 : 0;
  // the largest cluster whose clusters are all resident at once, on the SMs
  // the caller leaves to the call (fewer keys per CTA shorten each step's
  // chain; a second wave would cost a whole chain), else 8
  const int units = cdiv(dm.B, attn_pool_bpt(dm)) * dm.N * dm.Hkv;
  const int cap = sm_budget > 0 ? sm_budget : 1 << 30;
  if (f16 && units * 16 <= cap && units <= pool_resident(dm, P_max, 16)) return 16;
  if (f12 && units * 12 <= cap && units <= pool_resident(dm, P_max, 12)) return 12;
  if (f8) return 8;
  if (f12 && pool_resident(dm, P_max, 12) > 0) return 12;
  return f16 && pool_resident(dm, P_max, 16) > 0 ? 16 : 0;
}

// the attention without the pool kernel: whole-cluster or split-key kernels
template <int D>
static cudaError_t launch_attn_split(const herald_dims& dm, const uint16_t* q,
                                     const uint16_t* pool_k, const uint16_t* pool_v,
                                     const int32_t* n_sel, int P_max, const uint16_t* block_k,
                                     const uint16_t* block_v, uint16_t* out, float scale,
                                     const WsLayout& w, float* opart, float2* ml, uint32_t* err,
                                     cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  HERALD_CHECK_LAUNCH(ensure_smem(attn_kernel<D>, AttnCfg<D>::kSmem));
  HERALD_CHECK_LAUNCH(ensure_smem(attn_cluster_kernel<D, kClusterCtas>, AttnClCfg<D>::kSmem));
  HERALD_CHECK_LAUNCH(ensure_smem(attn_cluster_kernel<D, kClusterCtasMax>, AttnClCfg<D>::kSmem));
  if (w.splits <= 2 * kClusterCtas && !force_split()) {
    // 16-CTA clusters (one key tile per CTA) only if the whole launch fits
    // on the device at once; otherwise 8-CTA clusters with two tiles each
    if (w.splits > kClusterCtas &&
        max_active_clusters<D, kClusterCtasMax>() >= w.MT * segs)
      return launch_cluster("attn_cluster_kernel", attn_cluster_kernel<D, kClusterCtasMax>,
                            dim3(kClusterCtasMax, w.MT, segs), kClusterCtasMax,
                            AttnClCfg<D>::kSmem, st, q, pool_k, pool_v, n_sel, P_max, block_k,
                            block_v, dm.B, dm.Hq, dm.Hkv, w.R, scale, out, err);
    return launch_cluster("attn_cluster_kernel", attn_cluster_kernel<D, kClusterCtas>,
                          dim3(kClusterCtas, w.MT, segs), kClusterCtas, AttnClCfg<D>::kSmem, st,
                          q, pool_k, pool_v, n_sel, P_max, block_k, block_v, dm.B, dm.Hq, dm.Hkv,
                          w.R, scale, out, err);
  }
  HERALD_CHECK_LAUNCH(launch_k("attn_kernel", attn_kernel<D>, dim3(w.splits, w.MT, segs),
                               kTcThreads, AttnCfg<D>::kSmem, st, q, pool_k, pool_v, n_sel, P_max,
                               block_k, block_v, dm.B, dm.Hq, dm.Hkv, w.R, w.MT, w.splits, scale,
                               opart, ml, err));
  const int rows = dm.N * dm.B * dm.Hq;
  HERALD_CHECK_LAUNCH(launch_k("attn_combine_kernel", attn_combine_kernel<D>, cdiv(rows, 8), 256,
                               0, st, opart, ml, n_sel, P_max, dm.N, dm.B, dm.Hq, dm.Hkv, w.MT,
                               w.splits, out));
  return cudaSuccess;
}

template <int D>
static cudaError_t launch_attn_t(const herald_dims& dm, const uint16_t* q, const uint16_t* pool_k,
                                 const uint16_t* pool_v, const int32_t* n_sel, int P_max,
                                 const uint16_t* block_k, const uint16_t* block_v, uint16_t* out,
                                 float scale, const WsLayout& w, float* opart, float2* ml,
                                 uint32_t* err, const PoolMaps* maps, bool settled,
                                 const AppendArgs* app, int kernel, cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  cudaError_t e;
  const bool pool_ok = (kernel & 0x100) != 0 && maps && maps->pool_cs > 0;
  const bool flash_ok = (kernel & 0x200) != 0;
  const int choice = kernel & 0xF;  // HERALD_ATTN_KERNEL_* >> 8
  if (maps && !force_split()) {
    const int tiles = cdiv(dm.B, maps->bpt);
    const int cs = maps->pool_cs;
    // the pool kernel while its clusters fit the device at once, else the
    // pipelined kernel (one wave with fewer CTAs per row tile)
    int resident = pool_ok ? pool_resident(dm, P_max, cs) : 0;
    if (maps->sm_budget > 0) resident = std::min(resident, maps->sm_budget / cs);
    bool use_pool = pool_ok && (choice == 1 || choice >= 6 || !flash_ok ||
                                (choice == 0 && tiles * segs <= resident));
    if (choice >= 2 && choice <= 5 && flash_ok) use_pool = false;
    if (use_pool) {
      const int kpc = attn_pool_kpc(P_max, dm.B, cs);
      const uint32_t smem = attn_pool_smem(dm, P_max, cs);
      // early loads pay only when every CTA of the grid is resident at once:
      // with a second wave they measured slower (on the 4 x 64K layer)
      const int early = settled && tiles * segs <= resident ? 1 : 0;
      const AppendArgs none{nullptr, nullptr, nullptr, nullptr, nullptr, 0};
      if (cs == 16)
        return launch_cluster_threads("attn_pool_kernel", attn_pool_kernel<D, 16>,
                                      dim3(16, tiles, segs), dim3(kPoolThreads), 16, smem, st, maps->k, maps->v, maps->q, maps->bk, maps->bv, n_sel,
                              P_max, dm.B, dm.Hq, dm.Hkv, maps->bpt, kpc, scale, early, out, err,
                              app ? *app : none, dm.L_max);
      if (cs == 12)
        return launch_cluster_threads("attn_pool_kernel", attn_pool_kernel<D, 12>,
                                      dim3(12, tiles, segs), dim3(kPoolThreads), 12, smem, st, maps->k, maps->v, maps->q, maps->bk, maps->bv, n_sel,
                              P_max, dm.B, dm.Hq, dm.Hkv, maps->bpt, kpc, scale, early, out, err,
                              app ? *app : none, dm.L_max);
      return launch_cluster_threads("attn_pool_kernel", attn_pool_kernel<D, 8>,
                                    dim3(8, tiles, segs), dim3(kPoolThreads), 8, smem, st, maps->k, maps->v, maps->q, maps->bk, maps->bv, n_sel, P_max,
                            dm.B, dm.Hq, dm.Hkv, maps->bpt, kpc, scale, early, out, err,
                            app ? *app : none, dm.L_max);
    }
    if (flash_ok) {
      const int cs = choice == 3 ? 2 : choice == 4 ? 4 : choice == 5 ? 8 : 0;
      return launch_attn_flash(dm, n_sel, P_max, out, scale, err, *maps, app, cs, settled, st);
    }
  }
  e = launch_attn_split<D>(dm, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale, w,
                           opart, ml, err, st);
  if (e != cudaSuccess || !app) return e;
  return launch_append(dm, app->bk, app->bv, app->ctx, app->kc, app->vc, app->advance, st);
}

cudaError_t launch_attn(const herald_dims& dm, const uint16_t* q, const uint16_t* pool_k,
                        const uint16_t* pool_v, const int32_t* n_sel, int P_max,
                        const uint16_t* block_k, const uint16_t* block_v, uint16_t* out,
                        float scale, const WsLayout& w, float* opart, float2* ml, uint32_t* err,
                        const PoolMaps* maps, bool settled, const AppendArgs* app, int kernel,
                        cudaStream_t st) {
  if (dm.d == 128)
    return launch_attn_t<128>(dm, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale,
                              w, opart, ml, err, maps, settled, app, kernel, st);
  return launch_attn_t<64>(dm, q, pool_k, pool_v, n_sel, P_max, block_k, block_v, out, scale, w,
                           opart, ml, err, maps, settled, app, kernel, st);
}

HERALD_DEBUG_WORD_READER(debug_take_tc)

}  // namespace herald
