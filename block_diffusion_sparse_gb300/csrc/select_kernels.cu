// select_kernels.cu -- stage 1 of the HERALD selection and the final top-K:
//   merge_query   qbar = mean of the B block queries (HERALD v3 abstract:
//                 one merged query per head for the full-cache search)
//   scan          l[h][j] = qbar_h . k_j / sqrt(d) over the whole cache,
//                 streamed from HBM (or mapped host memory) by per-warp
//                 TMA rings; writes logits and per-tile (max, sumexp)
//   s1_hist       s1[j] = sum_h exp(l[h][j] - lse_h)  (SparDA method: GQA
//                 score = sum of the group's per-head softmax) + histogram
//   topc_finish   exact radix top-C of s1 per (sequence, KV head)
//   topk_union    exact radix top-K of the stage-2 score, union with sink
//                 and local windows (InfLLM-V2 decomposition in the SparDA
//                 method section), ascending positions
#include <climits>
#include <cuda_bf16.h>

#include "internal.cuh"
#include "block_scan.cuh"
#include "ptx.cuh"

namespace herald {

// ============================================================ merge_query
// grid (N*Hq), block d.  qbar = mean over the B queries, pre-scaled by
// 1/sqrt(d), in fp32 (for the CUDA-core scan) and as two bf16 rows hi =
// bf16(qbar), lo = bf16(qbar - hi) (for the tensor-core scan: hi + lo keeps
// ~16 mantissa bits).  Rows of absent heads (h >= G) are zero.  Also zeroes
// the stage-1 histogram.
__global__ void merge_query_kernel(const uint16_t* __restrict__ q, int B, int Hq, int Hkv, int d,
                                   float scale, float* __restrict__ qbar,
                                   uint16_t* __restrict__ qhl, uint32_t* __restrict__ hist,
                                   int hist_words, float2* __restrict__ part1, int part_slots,
                                   int n_rows) {
  griddep_enter();
  const int nh = blockIdx.x, n = nh / Hq, h = nh % Hq, e = threadIdx.x;
  const int G = Hq / Hkv, g = h / G, hl = h - g * G;
  if (e < d) {
    float acc = 0.f;
    const uint16_t* src = q + (size_t(n) * B * Hq + h) * d + e;
    int b = 0;
    for (; b + 8 <= B; b += 8) {
      uint16_t u[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) u[k] = src[size_t(b + k) * Hq * d];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc += __uint_as_float(uint32_t(u[k]) << 16);
    }
    for (; b < B; ++b) acc += __uint_as_float(uint32_t(src[size_t(b) * Hq * d]) << 16);
    const float qv = acc / float(B) * scale;
    qbar[size_t(nh) * d + e] = qv;
    const __nv_bfloat16 hi = __float2bfloat16_rn(qv);
    const __nv_bfloat16 lo = __float2bfloat16_rn(qv - __bfloat162float(hi));
    uint16_t* rows = qhl + (size_t(n) * Hkv + g) * kQhlRows * d;
    rows[size_t(hl) * d + e] = __bfloat16_as_ushort(hi);
    rows[size_t(8 + hl) * d + e] = __bfloat16_as_ushort(lo);
    if (hl == 0)
      for (int r = G; r < 8; ++r) {
        rows[size_t(r) * d + e] = 0;
        rows[size_t(8 + r) * d + e] = 0;
      }
  }
  const int tid = blockIdx.x * blockDim.x + threadIdx.x, nthr = gridDim.x * blockDim.x;
  for (int i = tid; i < hist_words; i += nthr) hist[i] = 0u;
  // the scan's (max, sumexp) slots start empty: (-inf, 0)
  for (int i = tid; i < n_rows * part_slots; i += nthr)
    part1[size_t(i / part_slots) * kPartSlots + (i % part_slots)] = make_float2(-INFINITY, 0.f);
}

cudaError_t launch_merge_query(const herald_dims& dm, const uint16_t* q_merge, float* qbar,
                               uint16_t* qhl, uint32_t* hist, float2* part1, int part_slots,
                               cudaStream_t st) {
  const float scale = 1.0f / sqrtf(float(dm.d));
  HERALD_CHECK_LAUNCH(launch_k("merge_query_kernel", merge_query_kernel, dm.N * dm.Hq, dm.d, 0, st, q_merge, dm.B, dm.Hq, dm.Hkv, dm.d, scale,
                                                    qbar, qhl, hist, dm.N * dm.Hkv * kHistBins,
                                                    part1, part_slots, dm.N * dm.Hq));
  return cudaGetLastError();
}

// Running (max, sum of exp) of the logits one lane has seen; merged across
// the warp only when a warp finishes a segment (no shuffles per tile).
struct OnlineLse {
  float m = -INFINITY, s = 0.f;
  __device__ __forceinline__ void add(float l) {
    if (l > m) {
      s = s * __expf(m - l) + 1.f;
      m = l;
    } else {
      s += __expf(l - m);
    }
  }
  // Warp-wide merge; lane 0 stores the result, then the state restarts.
  __device__ __forceinline__ void flush(float2* dst, int lane) {
    const float M = warp_max(m);
    const float S = warp_sum(m == -INFINITY ? 0.f : s * __expf(m - M));
    if (lane == 0) *dst = make_float2(M, S);
    m = -INFINITY;
    s = 0.f;
  }
};

// ======================================================== scan (tensor)
// Stage-1 scan of a device-resident cache on the tensor cores.  The merged
// queries of a KV group form a 16-row bf16 operand (8 hi rows + 8 lo rows);
// a 128-key tile of the cache is the other operand, so one 128 x 16 x d UMMA
// per tile yields every head's logit for 128 keys (hi + lo columns summed).
// Persistent, warp-specialised: warp 8 streams key tiles through a
// kTcScanStages-deep TMA ring, warp 9 issues the UMMAs into two TMEM
// accumulators, warps 0-7 (one TMEM lane = one key each; the two warps of a
// lane quadrant take half of the group's heads each) write logits and
// per-32-key (max, sumexp) partials while the next tile is multiplied.
template <int D>
struct TcScanCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kTcScanKeys * 128;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kBHalfBytes = kQhlRows * 128;
  static constexpr int kBBytes = kHalves * kBHalfBytes;
  static constexpr int kSmem = kTcScanStages * kTileBytes + kBBytes + 1024;
  // ring + operand + alignment slack must fit the dynamic allocation
  static_assert(kSmem >= kTcScanStages * kTileBytes + kBBytes + 1023, "scan smem layout");
  static_assert(kSmem <= 227 * 1024, "scan smem exceeds the per-CTA limit");
};
constexpr int kTcScanEpiWarps = 8;  // two per TMEM lane quadrant
constexpr int kTcScanProdWarp = kTcScanEpiWarps, kTcScanMmaWarp = kTcScanEpiWarps + 1;
constexpr int kTcScanThreads = (kTcScanEpiWarps + 2) * 32;

template <int D, int G>
__global__ void __launch_bounds__(kTcScanThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap bmap, const int32_t* __restrict__ ctx,
                   int Hkv, int L_max, int tiles_per_seg, int total_tiles, int L_pad,
                   float* __restrict__ logits, float2* __restrict__ part1, uint32_t* err) {
  using Cfg = TcScanCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kTcScanStages], empty[kTcScanStages];
  __shared__ uint64_t tfull[2], tempty[2], bbar, mdone;
  __shared__ uint32_t tmem_base;
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* Bs = ring + kTcScanStages * Cfg::kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = Hkv * G;
  const int t_begin = int((long long)blockIdx.x * total_tiles / gridDim.x);
  const int t_end = int((long long)(blockIdx.x + 1) * total_tiles / gridDim.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcScanStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kTcScanEpiWarps);
    }
    mbar_init(&bbar, 1);
    mbar_init(&mdone, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  griddep_enter();

  // tile t covers keys [j0, j0 + 128) of segment seg = n*Hkv + g
  auto tile = [&](int t, int& seg, int& j0, int& L) -> bool {
    seg = t / tiles_per_seg;
    j0 = (t - seg * tiles_per_seg) * kTcScanKeys;
    L = min(max(ctx[seg / Hkv], 0), L_max);
    return j0 < L;
  };

  if (warp == kTcScanProdWarp) {
    if (lane == 0) {  // ---- TMA producer
      tma_prefetch_desc(&kmap);
      int i = 0;
      for (int t = t_begin; t < t_end; ++t) {
        int seg, j0, L;
        if (!tile(t, seg, j0, L)) continue;
        const int stage = i % kTcScanStages;
        if (i >= kTcScanStages &&
            !mbar_wait(&empty[stage], uint32_t((i / kTcScanStages) - 1) & 1u)) {
          record_error(err, DEV_TIMEOUT_MMA | DEV_K_SCAN);
          break;
        }
        mbar_arrive_expect_tx(&full[stage], Cfg::kTileBytes);
#pragma unroll
        for (int hv = 0; hv < Cfg::kHalves; ++hv)
          tma_load_2d(ring + stage * Cfg::kTileBytes + hv * Cfg::kHalfBytes, &kmap, &full[stage],
                      hv * 64, seg * L_max + j0);
        ++i;
      }
    }
  } else if (warp == kTcScanMmaWarp) {
    if (lane == 0) {  // ---- UMMA issuer
      tma_prefetch_desc(&bmap);
      constexpr uint32_t idesc = make_idesc_bf16(kTcScanKeys, kQhlRows, false, false);
      int i = 0, cur_seg = -1;
      uint32_t nb = 0, nd = 0;
      bool ok = true;
      for (int t = t_begin; t < t_end && ok; ++t) {
        int seg, j0, L;
        if (!tile(t, seg, j0, L)) continue;
        if (seg != cur_seg) {  // new merged-query operand; earlier UMMAs must be done with Bs
          if (i > 0) {
            umma_commit(&mdone);
            ok = mbar_wait(&mdone, nd & 1u);
            ++nd;
          }
          mbar_arrive_expect_tx(&bbar, Cfg::kBBytes);
#pragma unroll
          for (int hv = 0; hv < Cfg::kHalves; ++hv)
            tma_load_2d(Bs + hv * Cfg::kBHalfBytes, &bmap, &bbar, hv * 64, seg * kQhlRows);
          ok = ok && mbar_wait(&bbar, nb & 1u);
          ++nb;
          cur_seg = seg;
        }
        const int stage = i % kTcScanStages, acc = i & 1;
        ok = ok && mbar_wait(&full[stage], uint32_t(i / kTcScanStages) & 1u);
        if (i >= 2) ok = ok && mbar_wait(&tempty[acc], uint32_t((i >> 1) - 1) & 1u);
        if (!ok) {
          record_error(err, DEV_TIMEOUT_TMA | DEV_K_SCAN);
          break;
        }
        tc_fence_after();
        const uint32_t ka = smem_u32(ring + stage * Cfg::kTileBytes), ba = smem_u32(Bs);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t hv = s >> 2, koff = (s & 3) * 32;
          const uint64_t a = make_sdesc_sw128(ka + hv * Cfg::kHalfBytes + koff, 16, 1024);
          const uint64_t b = make_sdesc_sw128(ba + hv * Cfg::kBHalfBytes + koff, 16, 1024);
          umma_bf16(tbase + acc * kQhlRows, a, b, idesc, s > 0 ? 1u : 0u);
        }
        umma_commit(&empty[stage]);
        umma_commit(&tfull[acc]);
        ++i;
      }
    }
  } else {  // ---- epilogue: warps 0-7, thread = key row of the tile
    constexpr int kHpw = (G + 1) / 2;  // heads per warp of a lane quadrant
    const int quad = warp & 3, h0 = (warp >> 2) * kHpw;
    OnlineLse run[kHpw];
    int run_seg = -1;
    const int slot = blockIdx.x * 4 + quad;
    auto flush = [&](int sg) {
      const int n = sg / Hkv, g = sg - n * Hkv;
#pragma unroll
      for (int k = 0; k < kHpw; ++k)
        if (h0 + k < G)
          run[k].flush(part1 + (size_t(n) * Hq + g * G + h0 + k) * kPartSlots + slot, lane);
    };
    int i = 0;
    for (int t = t_begin; t < t_end; ++t) {
      int seg, j0, L;
      if (!tile(t, seg, j0, L)) continue;
      if (seg != run_seg) {
        if (run_seg >= 0) flush(run_seg);
        run_seg = seg;
      }
      const int acc = i & 1;
      if (!mbar_wait(&tfull[acc], uint32_t(i >> 1) & 1u)) {
        record_error(err, DEV_TIMEOUT_MMA | DEV_K_SCAN);
        break;
      }
      tc_fence_after();
      __syncwarp();
      float v[16];
      tmem_ld16(tbase + (uint32_t(quad * 32) << 16) + uint32_t(acc * kQhlRows), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      const int n = seg / Hkv, g = seg - n * Hkv;
      const int j = j0 + quad * 32 + lane;
      if (j < L) {
#pragma unroll
        for (int k = 0; k < kHpw; ++k) {
          if (h0 + k < G) {
            // the upper warps' heads sit kHpw columns on (compile-time indices)
            const bool upper = warp >= 4;
            const float l = (upper ? v[kHpw + k] : v[k]) + (upper ? v[8 + kHpw + k] : v[8 + k]);
            logits[(size_t(n) * Hq + g * G + h0 + k) * L_pad + j] = l;
            run[k].add(l);
          }
        }
      }
      ++i;
    }
    if (run_seg >= 0) flush(run_seg);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 32);
  }
}

// ====================================================== scan (CUDA core)
// Stage-1 scan of a cache in mapped host memory (read over the host link):
// each warp streams 64-key tiles through its own cp.async ring; lane owns
// keys lane and lane+32, the two halves of packed f32x2 FMAs.
template <int D>
struct ScanCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kScanTileKeys * 128;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kSmem = kScanWarps * kScanStages * kTileBytes + 1024;
  static_assert(kSmem <= 227 * 1024, "scan smem exceeds the per-CTA limit");
};

template <int D, int G>
__global__ void __launch_bounds__(kScanWarps * 32, 1)
    scan_cc_kernel(const uint16_t* __restrict__ kc, const float* __restrict__ qbar,
                   const int32_t* __restrict__ ctx, int Hkv, int L_max, int tiles_per_seg,
                   int total_tiles, int L_pad, float* __restrict__ logits,
                   float2* __restrict__ part1) {
  using Cfg = ScanCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = Hkv * G;
  uint8_t* ring = smem + warp * kScanStages * Cfg::kTileBytes;
  const int t_begin = int((long long)blockIdx.x * total_tiles / gridDim.x);
  const int t_end = int((long long)(blockIdx.x + 1) * total_tiles / gridDim.x);
  griddep_enter();

  // Issues the copies of this warp's i-th tile into `stage` (one commit
  // group per tile, empty for tiles past the context).
  auto issue = [&](int i, int stage) {
    const int t = t_begin + warp + i * kScanWarps;
    if (t < t_end) {
      const int seg = t / tiles_per_seg;
      const int j0 = (t - seg * tiles_per_seg) * kScanTileKeys;
      const int L = min(max(ctx[seg / Hkv], 0), L_max);
      if (j0 < L) {
        uint8_t* dst = ring + stage * Cfg::kTileBytes;
        const uint16_t* base = kc + size_t(seg) * L_max * D;
        for (int q = lane; q < kScanTileKeys * (D / 8); q += 32) {
          const int r = q / (D / 8), c = q % (D / 8);
          const int j = j0 + r;
          const bool v = j < L;
          cp_async_16(dst + (c >> 3) * Cfg::kHalfBytes + sw128_off(r, c & 7),
                      base + size_t(v ? j : 0) * D + c * 8, v ? 16u : 0u);
        }
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int s = 0; s < kScanStages; ++s) issue(s, s);

  OnlineLse run[G];
  int run_seg = -1;
  const int slot = blockIdx.x * kScanWarps + warp;
  auto flush = [&](int sg) {
    const int n = sg / Hkv, g = sg - n * Hkv;
#pragma unroll
    for (int h = 0; h < G; ++h)
      run[h].flush(part1 + (size_t(n) * Hq + g * G + h) * kPartSlots + slot, lane);
  };
  for (int i = 0;; ++i) {
    const int t = t_begin + warp + i * kScanWarps;
    if (t >= t_end) break;
    const int stage = i % kScanStages;
    const int seg = t / tiles_per_seg;
    const int tl = t - seg * tiles_per_seg;
    const int n = seg / Hkv, g = seg - n * Hkv;
    const int j0 = tl * kScanTileKeys;
    const int L = min(max(ctx[n], 0), L_max);
    const bool valid = j0 < L;
    if (valid && seg != run_seg) {
      if (run_seg >= 0) flush(run_seg);
      run_seg = seg;
    }
    float2 acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
    asm volatile("cp.async.wait_group %0;" ::"n"(kScanStages - 1) : "memory");
    __syncwarp();
    if (valid) {
      const uint8_t* tile = ring + stage * Cfg::kTileBytes;
      const float* qb = qbar + (size_t(n) * Hq + g * G) * D;
#pragma unroll 2
      for (int c = 0; c < D / 8; ++c) {
        const int hv = c >> 3, cc = c & 7;
        const uint4 w0 =
            *reinterpret_cast<const uint4*>(tile + hv * Cfg::kHalfBytes + sw128_off(lane, cc));
        const uint4 w1 = *reinterpret_cast<const uint4*>(tile + hv * Cfg::kHalfBytes +
                                                         sw128_off(lane + 32, cc));
        float2 k2[8];
        k2[0] = make_float2(bf16lo(w0.x), bf16lo(w1.x));
        k2[1] = make_float2(bf16hi(w0.x), bf16hi(w1.x));
        k2[2] = make_float2(bf16lo(w0.y), bf16lo(w1.y));
        k2[3] = make_float2(bf16hi(w0.y), bf16hi(w1.y));
        k2[4] = make_float2(bf16lo(w0.z), bf16lo(w1.z));
        k2[5] = make_float2(bf16hi(w0.z), bf16hi(w1.z));
        k2[6] = make_float2(bf16lo(w0.w), bf16lo(w1.w));
        k2[7] = make_float2(bf16hi(w0.w), bf16hi(w1.w));
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 qa = __ldg(reinterpret_cast<const float4*>(qb + h * D + c * 8));
          const float4 qc = __ldg(reinterpret_cast<const float4*>(qb + h * D + c * 8 + 4));
          acc[h] = __ffma2_rn(make_float2(qa.x, qa.x), k2[0], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qa.y, qa.y), k2[1], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qa.z, qa.z), k2[2], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qa.w, qa.w), k2[3], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qc.x, qc.x), k2[4], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qc.y, qc.y), k2[5], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qc.z, qc.z), k2[6], acc[h]);
          acc[h] = __ffma2_rn(make_float2(qc.w, qc.w), k2[7], acc[h]);
        }
      }
    }
    __syncwarp();  // every lane has consumed the stage: refill it
    issue(i + kScanStages, stage);
    if (valid) {
      const int ja = j0 + lane, jb = j0 + lane + 32;
      const bool va = ja < L, vb = jb < L;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const size_t row = (size_t(n) * Hq + g * G + h);
        float* lr = logits + row * L_pad;
        if (va) {
          lr[ja] = acc[h].x;
          run[h].add(acc[h].x);
        }
        if (vb) {
          lr[jb] = acc[h].y;
          run[h].add(acc[h].y);
        }
      }
    }
  }
  if (run_seg >= 0) flush(run_seg);
  cp_async_wait_all();
}

template <int D, int G>
static cudaError_t launch_scan_t(const CUtensorMap* kmap, const CUtensorMap* bmap,
                                 const uint16_t* kc, const float* qbar, const int32_t* ctx,
                                 const herald_dims& dm, float* logits, float2* part1,
                                 const WsLayout& w, uint32_t* err, int num_sms, cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  if (kmap && bmap) {
    HERALD_CHECK_LAUNCH(ensure_smem(scan_tc_kernel<D, G>, TcScanCfg<D>::kSmem));
    const int total = segs * w.tiles128;
    const int grid = scan_grid(dm, w, true, num_sms);
    HERALD_CHECK_LAUNCH(launch_k("scan_tc_kernel", scan_tc_kernel<D, G>, grid, kTcScanThreads, TcScanCfg<D>::kSmem, st, 
        *kmap, *bmap, ctx, dm.Hkv, dm.L_max, w.tiles128, total, w.L_pad, logits, part1, err));
  } else {
    HERALD_CHECK_LAUNCH(ensure_smem(scan_cc_kernel<D, G>, ScanCfg<D>::kSmem));
    const int total = segs * w.tiles_per_seg;
    const int grid = scan_grid(dm, w, false, num_sms);
    HERALD_CHECK_LAUNCH(launch_k("scan_cc_kernel", scan_cc_kernel<D, G>, grid, kScanWarps * 32, ScanCfg<D>::kSmem, st, 
        kc, qbar, ctx, dm.Hkv, dm.L_max, w.tiles_per_seg, total, w.L_pad, logits, part1));
  }
  return cudaGetLastError();
}

template <int D>
static cudaError_t scan_dispatch_g(int G, const CUtensorMap* kmap, const CUtensorMap* bmap,
                                   const uint16_t* kc, const float* qbar, const int32_t* ctx,
                                   const herald_dims& dm, float* logits, float2* part1,
                                   const WsLayout& w, uint32_t* err, int num_sms,
                                   cudaStream_t st) {
#define HERALD_SCAN_G(GG) \
  case GG:                \
    return launch_scan_t<D, GG>(kmap, bmap, kc, qbar, ctx, dm, logits, part1, w, err, num_sms, st);
  switch (G) {
    HERALD_SCAN_G(1) HERALD_SCAN_G(2) HERALD_SCAN_G(3) HERALD_SCAN_G(4)
    HERALD_SCAN_G(5) HERALD_SCAN_G(6) HERALD_SCAN_G(7) HERALD_SCAN_G(8)
    default: return cudaErrorInvalidValue;
  }
#undef HERALD_SCAN_G
}

int scan_grid(const herald_dims& dm, const WsLayout& w, bool tensor_core, int num_sms) {
  const int total = dm.N * dm.Hkv * (tensor_core ? w.tiles128 : w.tiles_per_seg);
  int g = num_sms < kScanMaxCtas ? num_sms : kScanMaxCtas;
  return total < g ? total : g;
}

cudaError_t launch_scan(const herald_dims& dm, const CUtensorMap* kmap, const CUtensorMap* bmap,
                        const uint16_t* k_cache, const float* qbar, const int32_t* ctx,
                        float* logits, float2* part1, const WsLayout& w, uint32_t* err,
                        int num_sms, cudaStream_t st) {
  const int G = dm.Hq / dm.Hkv;
  if (dm.d == 128)
    return scan_dispatch_g<128>(G, kmap, bmap, k_cache, qbar, ctx, dm, logits, part1, w, err,
                                num_sms, st);
  return scan_dispatch_g<64>(G, kmap, bmap, k_cache, qbar, ctx, dm, logits, part1, w, err,
                             num_sms, st);
}

// ================================================================ s1_hist
// grid (chunks, N*Hkv), block 256.  Each CTA folds the per-tile partials of
// its G heads into lse_h, then scores its key range and bins the fp32 bit
// pattern of s1 (non-negative, so bit order = value order).
constexpr int kS1Threads = 256;
constexpr int kS1Keys = 4;  // keys per thread per round

__device__ __forceinline__ void lse_merge(float& m, float& s, float2 v) {
  if (v.x == -INFINITY) return;
  if (v.x > m) {
    s = s * __expf(m - v.x) + v.y;
    m = v.x;
  } else {
    s += v.y * __expf(v.x - m);
  }
}

template <int G>
__global__ void __launch_bounds__(kS1Threads)
    s1_hist_kernel(const float* __restrict__ logits, const float2* __restrict__ part1,
                   const int32_t* __restrict__ ctx, int Hkv, int L_max, int L_pad,
                   int part_slots, int keys_per_cta, float* __restrict__ s1,
                   uint32_t* __restrict__ hist) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ float lse[8];
  griddep_enter();
  const int seg = blockIdx.y, n = seg / Hkv, g = seg - n * Hkv;
  const int Hq = Hkv * G;
  const int L = min(max(ctx[n], 0), L_max);
  const int j_begin = blockIdx.x * keys_per_cta;
  if (j_begin >= L) return;
  const int j_end = min(L, j_begin + keys_per_cta);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kHistBins; i += kS1Threads) sh[i] = 0u;
  if (warp < G) {
    const int ntiles = part_slots;
    const float2* p = part1 + (size_t(n) * Hq + g * G + warp) * kPartSlots;
    float m = -INFINITY, s = 0.f;
    for (int t0 = 0; t0 < ntiles; t0 += 32 * 8) {
      float2 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = t0 + k * 32 + lane;
        v[k] = t < ntiles ? p[t] : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) lse_merge(m, s, v[k]);
    }
    const float M = warp_max(m);
    s = warp_sum(m == -INFINITY ? 0.f : s * __expf(m - M));
    if (lane == 0) lse[warp] = M + __logf(s);
  }
  __syncthreads();
  float lse_r[G];
#pragma unroll
  for (int h = 0; h < G; ++h) lse_r[h] = lse[h];
  const float* lg = logits + (size_t(n) * Hq + g * G) * L_pad;
  float* out = s1 + size_t(seg) * L_pad;
  for (int jb = j_begin; jb < j_end; jb += kS1Threads * kS1Keys) {
    float x[G][kS1Keys];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < kS1Keys; ++i) {
        const int j = jb + i * kS1Threads + threadIdx.x;
        x[h][i] = j < j_end ? lg[size_t(h) * L_pad + j] : 0.f;
      }
#pragma unroll
    for (int i = 0; i < kS1Keys; ++i) {
      const int j = jb + i * kS1Threads + threadIdx.x;
      if (j >= j_end) break;
      float acc = 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) acc += __expf(x[h][i] - lse_r[h]);
      out[j] = acc;
      atomicAdd(&sh[(__float_as_uint(acc) >> kHistShift) & (kHistBins - 1)], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = hist + size_t(seg) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kS1Threads)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

cudaError_t launch_s1_hist(const herald_dims& dm, const float* logits, const float2* part1,
                           int part_slots, const int32_t* ctx, float* s1, uint32_t* hist,
                           const WsLayout& w, int num_sms, cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  int chunks = (2 * num_sms + segs - 1) / segs;
  int keys = cdiv(dm.L_max, chunks);
  keys = cdiv(keys, kS1Threads * kS1Keys) * kS1Threads * kS1Keys;
  chunks = cdiv(dm.L_max, keys);
  const dim3 grid(chunks, segs);
  switch (dm.Hq / dm.Hkv) {
#define HERALD_S1_G(GG)                                                                      \
  case GG:                                                                                   \
    HERALD_CHECK_LAUNCH(launch_k("s1_hist_kernel", s1_hist_kernel<GG>, grid, kS1Threads, 0, st, logits, part1, ctx, dm.Hkv, dm.L_max,    \
                                                    w.L_pad, part_slots, keys, s1, hist));      \
    break;
    HERALD_S1_G(1) HERALD_S1_G(2) HERALD_S1_G(3) HERALD_S1_G(4)
    HERALD_S1_G(5) HERALD_S1_G(6) HERALD_S1_G(7) HERALD_S1_G(8)
#undef HERALD_S1_G
    default: break;
  }
  return cudaGetLastError();
}

// ============================================================ topc_finish
// One CTA of 1024 threads per (n, g).  Radix select of the C-th largest s1:
// the first 12-bit digit comes from the global histogram; the members of
// that bin are collected into shared memory (bounded; a global two-digit
// fallback handles overflow) and the remaining 19 bits are resolved there.
// The ordered compaction then keeps every s1 above the threshold plus the
// lowest-position ties, with one two-counter block scan per round.  Both
// passes over s1 load each round while the previous one is processed, and
// the collection takes one shared-memory atomic per warp and round.
constexpr int kSelThreads = 1024;
constexpr int kTieCap = 6144;

// Elements of s1 are processed in rounds of kSelThreads * kPerThr: thread t
// holds the kPerThr consecutive values [base + t*kPerThr, ...) in registers,
// loaded as independent 16-byte loads so a round costs one memory latency.
constexpr int kPerThr = 16;
constexpr int kRound = kSelThreads * kPerThr;

__device__ __forceinline__ void load_round(const uint32_t* sv, int L, int base,
                                           uint32_t (&v)[kPerThr]) {
  const int j0 = base + threadIdx.x * kPerThr;
  if (j0 + kPerThr <= L) {
    const uint4* p = reinterpret_cast<const uint4*>(sv + j0);
#pragma unroll
    for (int k = 0; k < kPerThr / 4; ++k) {
      const uint4 x = p[k];
      v[4 * k] = x.x; v[4 * k + 1] = x.y; v[4 * k + 2] = x.z; v[4 * k + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPerThr; ++k) v[k] = (j0 + k < L) ? sv[j0 + k] : 0u;
  }
}

__global__ void __launch_bounds__(kSelThreads)
    topc_finish_kernel(const float* __restrict__ s1, const uint32_t* __restrict__ hist,
                       const int32_t* __restrict__ ctx, int Hkv, int L_max, int L_pad, int C,
                       int32_t* __restrict__ cand, int32_t* __restrict__ n_cand) {
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t tie_v[kTieCap];
  __shared__ uint32_t wt[32], wt2[32];
  __shared__ int s_bin, s_wsel;
  __shared__ uint32_t s_above, s_cnt, s_wbefore;
  griddep_enter();
  const int seg = blockIdx.x, n = seg / Hkv;
  const int L = min(max(ctx[n], 0), L_max);
  debug_flag(threadIdx.x == 0 && (ctx[n] < 0 || ctx[n] > L_max), DEV_BAD_COUNT);
  const int Ce = min(C, L);
  int32_t* out = cand + size_t(seg) * C;
  const uint32_t* sv = reinterpret_cast<const uint32_t*>(s1 + size_t(seg) * L_pad);
  if (threadIdx.x == 0) n_cand[seg] = Ce;
  for (int i = Ce + threadIdx.x; i < C; i += kSelThreads) out[i] = -1;
  if (Ce == L) {
    for (int i = threadIdx.x; i < L; i += kSelThreads) out[i] = i;
    return;
  }
  // digit 1: bits [30:19] from the global histogram, searched while the
  // first round of s1 loads
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads)
    h[i] = hist[size_t(seg) * kHistBins + i];
  if (threadIdx.x == 0) s_cnt = 0;
  const int lane = threadIdx.x & 31;
  uint32_t v[kPerThr], vn[kPerThr];
  load_round(sv, L, 0, v);
  __syncthreads();
  uint32_t need = uint32_t(Ce);
  find_bin_wide<kSelThreads>(h, kHistBins, need, wt, &s_wsel, &s_wbefore, &s_bin, &s_above);
  const uint32_t b1 = uint32_t(s_bin);
  need -= s_above;
  // collect the low 19 bits of the members of bin b1 (in any order: only
  // their histograms are used)
  for (int base = 0; base < L; base += kRound) {
    const bool more = base + kRound < L;
    if (more) load_round(sv, L, base + kRound, vn);
    const int j0 = base + threadIdx.x * kPerThr;
    uint32_t mine = 0;
#pragma unroll
    for (int k = 0; k < kPerThr; ++k) mine += (j0 + k < L && (v[k] >> 19) == b1) ? 1u : 0u;
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t wbase = 0;
    if (lane == 31 && incl) wbase = atomicAdd(&s_cnt, incl);
    uint32_t slot = __shfl_sync(0xffffffffu, wbase, 31) + incl - mine;
#pragma unroll
    for (int k = 0; k < kPerThr; ++k)
      if (j0 + k < L && (v[k] >> 19) == b1) {
        if (slot < uint32_t(kTieCap)) tie_v[slot] = v[k] & 0x7FFFFu;
        ++slot;
      }
    if (more) {
#pragma unroll
      for (int k = 0; k < kPerThr; ++k) v[k] = vn[k];
    }
  }
  // the compaction's first round loads while digits 2 and 3 are resolved
  load_round(sv, L, 0, v);
  __syncthreads();
  const uint32_t cnt = s_cnt;
  const bool in_smem = cnt <= uint32_t(kTieCap);
  // digit 2: bits [18:8]
  for (int i = threadIdx.x; i < 2048; i += kSelThreads) h[i] = 0u;
  __syncthreads();
  if (in_smem) {
    for (uint32_t i = threadIdx.x; i < cnt; i += kSelThreads) atomicAdd(&h[tie_v[i] >> 8], 1u);
  } else {
    for (int j = threadIdx.x; j < L; j += kSelThreads) {
      const uint32_t v = sv[j];
      if ((v >> 19) == b1) atomicAdd(&h[(v >> 8) & 2047u], 1u);
    }
  }
  __syncthreads();
  find_bin_wide<kSelThreads>(h, 2048, need, wt, &s_wsel, &s_wbefore, &s_bin, &s_above);
  const uint32_t b2 = uint32_t(s_bin);
  need -= s_above;
  // digit 3: bits [7:0]
  for (int i = threadIdx.x; i < 256; i += kSelThreads) h[i] = 0u;
  __syncthreads();
  if (in_smem) {
    for (uint32_t i = threadIdx.x; i < cnt; i += kSelThreads) {
      const uint32_t v = tie_v[i];
      if ((v >> 8) == b2) atomicAdd(&h[v & 255u], 1u);
    }
  } else {
    const uint32_t pre = (b1 << 11) | b2;
    for (int j = threadIdx.x; j < L; j += kSelThreads) {
      const uint32_t v = sv[j];
      if ((v >> 8) == pre) atomicAdd(&h[v & 255u], 1u);
    }
  }
  __syncthreads();
  find_bin_from_top<kSelThreads>(h, 256, need, wt, &s_bin, &s_above);
  const uint32_t tau = (b1 << 19) | (b2 << 8) | uint32_t(s_bin);
  const uint32_t need_eq = need - s_above;  // ties at tau to keep, lowest position first
  // ordered compaction, one round of kRound positions at a time
  uint32_t gt_run = 0, eq_run = 0;
  for (int base = 0; base < L; base += kRound) {
    const bool more = base + kRound < L;
    if (more) load_round(sv, L, base + kRound, vn);
    const int j0 = base + threadIdx.x * kPerThr;
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int k = 0; k < kPerThr; ++k) {
      const bool in = j0 + k < L;
      n_gt += in && v[k] > tau;
      n_eq += in && v[k] == tau;
    }
    uint32_t gt_before, eq_before, gt_tot, eq_tot;
    block_excl_scan2<kSelThreads>(n_gt, n_eq, wt, wt2, gt_before, eq_before, gt_tot, eq_tot);
    gt_before += gt_run;
    eq_before += eq_run;
#pragma unroll
    for (int k = 0; k < kPerThr; ++k) {
      if (j0 + k >= L) break;
      if (v[k] > tau) {
        const uint32_t pos = gt_before + min(eq_before, need_eq);
        if (pos < uint32_t(Ce)) out[pos] = j0 + k;
        ++gt_before;
      } else if (v[k] == tau) {
        if (eq_before < need_eq && gt_before + eq_before < uint32_t(Ce))
          out[gt_before + eq_before] = j0 + k;
        ++eq_before;
      }
    }
    gt_run += gt_tot;
    eq_run += eq_tot;
    if (more) {
#pragma unroll
      for (int k = 0; k < kPerThr; ++k) v[k] = vn[k];
    }
  }
}

cudaError_t launch_topc(const herald_dims& dm, const float* s1, const uint32_t* hist,
                        const int32_t* ctx, int C, int32_t* cand, int32_t* n_cand,
                        const WsLayout& w, cudaStream_t st) {
  HERALD_CHECK_LAUNCH(launch_k("topc_finish_kernel", topc_finish_kernel, dm.N * dm.Hkv, kSelThreads, 0, st, s1, hist, ctx, dm.Hkv, dm.L_max,
                                                            w.L_pad, C, cand, n_cand));
  return cudaGetLastError();
}

// ============================================================ exact selection
// Helpers of the exact selection (every cached position a candidate):
// the candidate count of each (sequence, KV head) is its context length,
// and the refine's score partials are summed in place into partial 0 while
// their 12-bit histogram (the first radix digit of the top-K) is built.
__global__ void exact_counts_kernel(const int32_t* __restrict__ ctx, int segs, int Hkv, int L_max,
                                    int32_t* __restrict__ n_cand) {
  griddep_enter();
  const int seg = blockIdx.x * blockDim.x + threadIdx.x;
  if (seg < segs) n_cand[seg] = min(max(ctx[seg / Hkv], 0), L_max);
}

// grid (chunks, N*Hkv), block 256: s[p][seg][j] (stride per partial:
// segs * stride) summed over the n_parts partials into s[0][seg][j] for
// j < ctx, and binned by the top 12 bits of the (non-negative) fp32 pattern.
__global__ void __launch_bounds__(256)
    exact_sum_hist_kernel(float* __restrict__ s, int n_parts, int stride,
                          const int32_t* __restrict__ ctx, int Hkv, int L_max, int keys_per_cta,
                          uint32_t* __restrict__ hist) {
  __shared__ uint32_t sh[kHistBins];
  griddep_enter();
  const int seg = blockIdx.y, n = seg / Hkv;
  const int L = min(max(ctx[n], 0), L_max);
  const int j_begin = blockIdx.x * keys_per_cta;
  if (j_begin >= L) return;
  const int j_end = min(L, j_begin + keys_per_cta);
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x) sh[i] = 0u;
  __syncthreads();
  const size_t part_stride = size_t(gridDim.y) * stride;
  float* row = s + size_t(seg) * stride;
  for (int j = j_begin + threadIdx.x; j < j_end; j += blockDim.x) {
    float v = 0.f;
    for (int p = 0; p < n_parts; ++p) v += row[p * part_stride + j];
    v = fmaxf(v, 0.f);
    row[j] = v;
    atomicAdd(&sh[(__float_as_uint(v) >> kHistShift) & (kHistBins - 1)], 1u);
  }
  __syncthreads();
  uint32_t* gh = hist + size_t(seg) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

cudaError_t launch_exact_counts(const herald_dims& dm, const int32_t* ctx, int32_t* n_cand,
                                cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  HERALD_CHECK_LAUNCH(launch_k("exact_counts_kernel", exact_counts_kernel, cdiv(segs, 128), 128,
                               0, st, ctx, segs, dm.Hkv, dm.L_max, n_cand));
  return cudaGetLastError();
}

cudaError_t launch_exact_sum_hist(const herald_dims& dm, float* s, int n_parts, int stride,
                                  const int32_t* ctx, uint32_t* hist, int num_sms,
                                  cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  int chunks = (2 * num_sms + segs - 1) / segs;
  int keys = cdiv(cdiv(dm.L_max, chunks), 256) * 256;
  chunks = cdiv(dm.L_max, keys);
  HERALD_CHECK_LAUNCH(launch_k("exact_sum_hist_kernel", exact_sum_hist_kernel,
                               dim3(chunks, segs), 256, 0, st, s, n_parts, stride, ctx, dm.Hkv,
                               dm.L_max, keys, hist));
  return cudaGetLastError();
}

// ============================================================= topk_union
// One CTA of 1024 threads per (n, g); thread t holds the stage-2 scores of the
// candidate slots [t*E, (t+1)*E) in registers (E <= kPer; 4 when C <= 4096,
// 16 up to C = 16384), summed over the refine's row-tile partials with all
// loads of a partial in flight at once.  The K-th largest score lies in one
// bin of a 14-bit histogram of the fp32 bit patterns (16 sub-bins per
// octave: on the 32K layer ~100-140 of the 4096 scores share the threshold's
// bin at 12 bits, a quarter of that at 14, and the ranking below is
// quadratic in them); the members of that bin are ranked exactly (score
// descending, slot ascending = position ascending,
// candidates being ascending), the winners marked in a shared bitmap, and one
// block scan orders the output: [0, sink_end) ++ kept candidates inside
// [sink_end, local_begin) ++ [local_begin, L) -- the deduplicated ascending
// union.  With slot_out, each output row also records the candidate slot it
// came from (-1 for sink, local and padding rows), so that a gather can read
// candidate rows staged by slot.
constexpr int kTkThreads = 1024;
// first radix digit of the top-K: the top 14 bits of the (non-negative)
// fp32 pattern, 16 sub-bins per octave, in dynamic shared memory
constexpr int kTkShift = 17;
constexpr int kTkBins = 1 << (31 - kTkShift);
constexpr int kTkRankCap = 1024;  // members ranked in one shot

template <int kPer>
__global__ void __launch_bounds__(kTkThreads)
    topk_union_kernel(const int32_t* __restrict__ ctx, const int32_t* __restrict__ cand,
                      const int32_t* __restrict__ n_cand, const float* __restrict__ s2,
                      int n_parts, int Hkv, int L_max, int C, int K, int S, int W, int P_max,
                      int32_t* __restrict__ idx, int32_t* __restrict__ n_sel, PoolGather pg,
                      int32_t* __restrict__ slot_out, const int32_t* __restrict__ k_seg,
                      int early) {
  // [C] bit patterns of the threshold-bin members, then (with the gather)
  // [P_max] selected positions
  extern __shared__ uint32_t dsm[];
  uint32_t* h = dsm;              // [kTkBins] histogram, later the finer digits'
  uint32_t* mem = dsm + kTkBins;  // [C] member patterns, then [P_max] positions
  __shared__ uint32_t taken[kMaxC / 32];      // bitmap over candidate slots
  __shared__ uint2 mpair[kTkRankCap];         // (bit pattern, slot) of the first members
  __shared__ uint32_t wt[32], wt2[32];
  __shared__ int s_bin, s_wsel;
  __shared__ uint32_t s_above, s_cnt, s_wbefore;
  // with the gather, pg.copies CTAs per (n, g) select alike (the selection
  // is deterministic) and each gathers one slice of the pool; copy 0 writes
  // idx and n_sel
  const int copies = pg.pk ? pg.copies : 1;
  const int seg = blockIdx.x / copies, copy = blockIdx.x - seg * copies, n = seg / Hkv;
  // slots per thread from C, not n_cand: the score loads need not wait for it
  const int E = (C + kTkThreads - 1) / kTkThreads;
  const int i0 = threadIdx.x * E;
  const int32_t* cd = cand + size_t(seg) * C;
  // the candidate positions are needed only at the end; with few per thread
  // their loads are issued with the context length and the candidate count
  // (with 16 per thread the registers are not there).  early != 0: the
  // caller's inputs (ctx, cand, n_cand) were written before the stage-2
  // refine that precedes this kernel began, so they are read before the
  // grid-dependency wait, which then covers only the refine's scores
  constexpr bool kEarlyPos = kPer <= 4;
  int32_t pk[kPer];
  int ctx_raw = 0, nc_raw = 0;
  auto load_inputs = [&]() {
    ctx_raw = ctx[n];
    nc_raw = n_cand[seg];
    if constexpr (kEarlyPos) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) pk[k] = (k < E && i0 + k < C) ? __ldg(cd + i0 + k) : -1;
    }
  };
  if (early) load_inputs();
  // shared state cleared before the wait
  for (int i = threadIdx.x; i < kTkBins; i += kTkThreads) h[i] = 0u;
  for (int i = threadIdx.x; i < kMaxC / 32; i += kTkThreads) taken[i] = 0u;
  if (threadIdx.x == 0) s_cnt = 0;
  griddep_enter();
  if (!early) load_inputs();
  const int L = min(max(ctx_raw, 0), L_max);
  debug_flag(threadIdx.x == 0 && (ctx_raw < 0 || ctx_raw > L_max), DEV_BAD_COUNT);
  const int nc = min(max(nc_raw, 0), C);
  // the budget: K, or this (n, g)'s own (at most K) when k_seg is given
  const int Ke = min(k_seg ? min(max(k_seg[seg], 0), K) : K, nc);
  const float* sc = s2 + size_t(seg) * C;
  const size_t part_stride = size_t(gridDim.x / copies) * C;  // [part][N*Hkv][C]
  float x[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) x[k] = 0.f;
  // partials two at a time: both loads in flight
  int p = 0;
  for (; p + 2 <= n_parts; p += 2) {
    const float* s0 = sc + p * part_stride + i0;
    const float* s1 = s0 + part_stride;
    float y0[kPer], y1[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const bool in = k < E && i0 + k < C;  // in bounds; slots >= n_cand are masked later
      y0[k] = in ? __ldg(s0 + k) : 0.f;
      y1[k] = in ? __ldg(s1 + k) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) x[k] += y0[k] + y1[k];
  }
  if (p < n_parts) {
    const float* s0 = sc + p * part_stride + i0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) x[k] += (k < E && i0 + k < C) ? __ldg(s0 + k) : 0.f;
  }
  uint32_t v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) v[k] = __float_as_uint(fmaxf(x[k], 0.f));
  const bool take_all = (Ke == nc);
  uint32_t b1 = 0;  // bin of the K-th largest; bins above it are kept whole
  if (!take_all && Ke > 0) {
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (k < E && i0 + k < nc) atomicAdd(&h[v[k] >> kTkShift], 1u);
    __syncthreads();
    find_bin_wide<kTkThreads>(h, kTkBins, uint32_t(Ke), wt, &s_wsel, &s_wbefore, &s_bin,
                              &s_above);
    b1 = uint32_t(s_bin);
    const uint32_t need = uint32_t(Ke) - s_above;  // winners to take inside bin b1
    // one warp-aggregated allocation for all of a thread's members
    uint32_t my_members = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      my_members += (k < E && i0 + k < nc && (v[k] >> kTkShift) == b1) ? 1u : 0u;
    uint32_t incl = my_members;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if ((threadIdx.x & 31) >= o) incl += y;
    }
    uint32_t wbase = 0;
    if ((threadIdx.x & 31) == 31 && incl) wbase = atomicAdd(&s_cnt, incl);
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    uint32_t slot = wbase + incl - my_members;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (k < E && i0 + k < nc && (v[k] >> kTkShift) == b1) {
        mem[slot] = v[k];
        if (slot < uint32_t(kTkRankCap)) mpair[slot] = make_uint2(v[k], uint32_t(i0 + k));
        ++slot;
      }
    }
    __syncthreads();
    const uint32_t cnt = s_cnt;
    if (cnt <= uint32_t(kTkRankCap)) {
      // exact rank of member t among the members: higher score, or equal
      // score at a lower slot, ranks first
      if (threadIdx.x < cnt) {
        const uint2 me = mpair[threadIdx.x];
        uint32_t r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        uint32_t j = 0;
        for (; j + 4 <= cnt; j += 4) {
          const uint2 a = mpair[j], b = mpair[j + 1], c = mpair[j + 2], d = mpair[j + 3];
          r0 += (a.x > me.x) || (a.x == me.x && a.y < me.y);
          r1 += (b.x > me.x) || (b.x == me.x && b.y < me.y);
          r2 += (c.x > me.x) || (c.x == me.x && c.y < me.y);
          r3 += (d.x > me.x) || (d.x == me.x && d.y < me.y);
        }
        for (; j < cnt; ++j) {
          const uint2 a = mpair[j];
          r0 += (a.x > me.x) || (a.x == me.x && a.y < me.y);
        }
        if (r0 + r1 + r2 + r3 < need) atomicOr(&taken[me.y >> 5], 1u << (me.y & 31));
      }
    } else {
      // many members: resolve the remaining 17 bits with two more digits
      constexpr uint32_t kMid = (1u << (kTkShift - 8)) - 1u;
      for (int i = threadIdx.x; i <= int(kMid); i += kTkThreads) h[i] = 0u;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < cnt; i += kTkThreads)
        atomicAdd(&h[(mem[i] >> 8) & kMid], 1u);
      __syncthreads();
      uint32_t nd = need;
      find_bin_from_top<kTkThreads>(h, int(kMid) + 1, nd, wt, &s_bin, &s_above);
      const uint32_t b2 = uint32_t(s_bin);
      nd -= s_above;
      for (int i = threadIdx.x; i < 256; i += kTkThreads) h[i] = 0u;
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < cnt; i += kTkThreads)
        if (((mem[i] >> 8) & kMid) == b2) atomicAdd(&h[mem[i] & 255u], 1u);
      __syncthreads();
      find_bin_from_top<kTkThreads>(h, 256, nd, wt, &s_bin, &s_above);
      const uint32_t tau = (b1 << kTkShift) | (b2 << 8) | uint32_t(s_bin);
      const uint32_t need_eq = nd - s_above;
      // members above tau, plus the first need_eq ties in slot order
      uint32_t n_eq = 0;
#pragma unroll
      for (int k = 0; k < kPer; ++k) n_eq += (k < E && i0 + k < nc && v[k] == tau) ? 1u : 0u;
      uint32_t eq_before, d0, d1, d2;
      block_excl_scan2<kTkThreads>(n_eq, 0u, wt, wt2, eq_before, d0, d1, d2);
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        if (!(k < E && i0 + k < nc) || (v[k] >> kTkShift) != b1) continue;
        bool t = v[k] > tau;
        if (v[k] == tau) t = eq_before++ < need_eq;
        if (t) atomicOr(&taken[(i0 + k) >> 5], 1u << ((i0 + k) & 31));
      }
    }
    __syncthreads();
  }
  const int sink_end = min(S, L);
  const int local_begin = max(L - W, sink_end);
  // the top-K slots of this thread
  uint32_t top_mask = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int slot = i0 + k;
    if (!(k < E && slot < nc) || Ke == 0) continue;
    if (take_all || (v[k] >> kTkShift) > b1 ||
        ((v[k] >> kTkShift) == b1 && ((taken[slot >> 5] >> (slot & 31)) & 1u)))
      top_mask |= 1u << k;
  }
  if constexpr (!kEarlyPos) {
#pragma unroll
    for (int k = 0; k < kPer; ++k) pk[k] = ((top_mask >> k) & 1u) ? __ldg(cd + i0 + k) : -1;
  }
  uint32_t keep_mask = 0, n_keep = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (((top_mask >> k) & 1u) && pk[k] >= sink_end && pk[k] < local_begin) {
      keep_mask |= 1u << k;
      ++n_keep;
    }
  uint32_t at, d3, n_mid, d4;
  block_excl_scan2<kTkThreads>(n_keep, 0u, wt, wt2, at, d3, n_mid, d4);
  int32_t* out = idx + size_t(seg) * P_max;
  int32_t* sidx = reinterpret_cast<int32_t*>(mem + C);
  const bool to_global = copy == 0;
  int32_t* so = slot_out ? slot_out + size_t(seg) * P_max : nullptr;
  // row `slot` of the selection holds position v, taken from candidate slot
  // src (-1: a sink, local or padding row)
  auto put = [&](int slot, int32_t v, int32_t src) {
    debug_flag(v < -1 || v >= L, DEV_BAD_INDEX);  // a selected position past the context
    if (to_global) {
      out[slot] = v;
      if (so) so[slot] = src;
    }
    if (pg.pk) sidx[slot] = v;
  };
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if ((keep_mask >> k) & 1u) {
      if (sink_end + int(at) < P_max)
        put(sink_end + at, pk[k], i0 + k);
      else
        debug_flag(true, DEV_BAD_COUNT);  // a selection row past P_max
      ++at;
    }
  for (int j = threadIdx.x; j < sink_end; j += kTkThreads) put(j, j, -1);
  for (int j = local_begin + threadIdx.x; j < L; j += kTkThreads)
    if (sink_end + int(n_mid) + (j - local_begin) < P_max)
      put(sink_end + n_mid + (j - local_begin), j, -1);
    else
      debug_flag(true, DEV_BAD_COUNT);
  const int total = min(P_max, sink_end + int(n_mid) + (L - local_begin));
  for (int s = total + threadIdx.x; s < P_max; s += kTkThreads) put(s, -1, -1);
  if (to_global && threadIdx.x == 0) n_sel[seg] = total;
  if (!pg.pk) return;
  // the gather of this copy's slice of the pool: rows [r0, r1) of (n, g),
  // zero rows from n_sel on, 16-byte chunks of K and V per thread
  __syncthreads();
  const int rpc = (P_max + copies - 1) / copies;
  const int r0 = copy * rpc, r1 = min(P_max, r0 + rpc);
  const int cpr = pg.d / 8;
  const size_t seg_rows = size_t(seg) * L_max, pool_rows = size_t(seg) * P_max;
  for (int u = threadIdx.x; u < (r1 - r0) * cpr; u += kTkThreads) {
    const int r = r0 + u / cpr, c = u - (u / cpr) * cpr;
    const int pos = r < total ? sidx[r] : -1;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (pos >= 0 && pos < L_max) {
      const size_t off = (seg_rows + pos) * pg.d + c * 8;
      kv = *reinterpret_cast<const uint4*>(pg.kc + off);
      vv = *reinterpret_cast<const uint4*>(pg.vc + off);
    }
    const size_t dst = (pool_rows + r) * pg.d + c * 8;
    *reinterpret_cast<uint4*>(pg.pk + dst) = kv;
    *reinterpret_cast<uint4*>(pg.pv + dst) = vv;
  }
}

cudaError_t launch_topk_union(const herald_dims& dm, const int32_t* ctx, const int32_t* cand,
                              const int32_t* n_cand, const float* s2, int n_parts, int C, int K,
                              int S, int W, int P_max, int32_t* idx, int32_t* n_sel,
                              cudaStream_t st, const PoolGather* gather, int32_t* slot_out,
                              const int32_t* k_seg, bool early) {
  static_assert(kMaxC <= 16 * kTkThreads, "16 scores per thread cover every C");
  const PoolGather pg = gather ? *gather : PoolGather{nullptr, nullptr, nullptr, nullptr, 0, 1};
  const size_t smem = size_t(kTkBins) * 4 + size_t(C) * 4 + (pg.pk ? size_t(P_max) * 4 : 0u);
  HERALD_CHECK_LAUNCH(C <= 4 * kTkThreads ? ensure_smem(topk_union_kernel<4>, smem)
                                          : ensure_smem(topk_union_kernel<16>, smem));
  const int grid = dm.N * dm.Hkv * (pg.pk ? pg.copies : 1);
  // the fewest registers that hold C scores over 1024 threads
  if (C <= 4 * kTkThreads)
    HERALD_CHECK_LAUNCH(launch_k("topk_union_kernel", topk_union_kernel<4>, grid, kTkThreads, smem,
                                 st, ctx, cand, n_cand, s2, n_parts, dm.Hkv, dm.L_max, C, K, S, W,
                                 P_max, idx, n_sel, pg, slot_out, k_seg, early ? 1 : 0));
  else
    HERALD_CHECK_LAUNCH(launch_k("topk_union_kernel", topk_union_kernel<16>, grid, kTkThreads,
                                 smem, st, ctx, cand, n_cand, s2, n_parts, dm.Hkv, dm.L_max, C, K,
                                 S, W, P_max, idx, n_sel, pg, slot_out, k_seg, early ? 1 : 0));
  return cudaGetLastError();
}

// ============================================================= budget
// One CTA of 1024 threads per (n, g).  The stage-2 scores of the n_cand
// valid slots, summed over the row-tile partials exactly as topk_union sums
// them (both kernels see the same fp32 values), go to shared memory as bit
// patterns (a non-negative float orders as its pattern).  The budget is one
// past the first sorted position whose running mass reaches tau times the
// total; it is found without sorting, by a radix search from the top over
// the 12 / 11 / 8-bit digits of the patterns with mass-weighted histograms:
// each pass finds the bin where the mass above it (carried from the earlier
// passes) plus its own reaches the target, and the last pass's bin is one
// value t, of which ceil((target - mass above) / t) ties are taken.  Then
// clamped to [K_min, K_max] (and to n_cand before the clamp).
constexpr int kBudgetThreads = 1024;

// Inclusive block scan of (mass, count) in thread order; totals in *tm, *tc.
__device__ __forceinline__ void budget_scan(float& m, uint32_t& c, float* wm, uint32_t* wc,
                                            float* tm, uint32_t* tc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float ym = __shfl_up_sync(0xffffffffu, m, o);
    const uint32_t yc = __shfl_up_sync(0xffffffffu, c, o);
    if (lane >= o) {
      m += ym;
      c += yc;
    }
  }
  if (lane == 31) {
    wm[warp] = m;
    wc[warp] = c;
  }
  __syncthreads();
  if (warp == 0) {
    float a = wm[lane];
    uint32_t b = wc[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float ya = __shfl_up_sync(0xffffffffu, a, o);
      const uint32_t yb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) {
        a += ya;
        b += yb;
      }
    }
    wm[lane] = a;
    wc[lane] = b;
  }
  __syncthreads();
  if (warp > 0) {
    m += wm[warp - 1];
    c += wc[warp - 1];
  }
  *tm = wm[31];
  *tc = wc[31];
}

// The budget's bin masses are accumulated as unsigned 64-bit fixed point
// (2^-40 units; a score is at most B*G <= 256, so C <= 16384 of them stay
// below 2^62): integer atomics add in any order to the same sum, so the
// budget of an input is the same on every run.
constexpr float kMassScale = 1099511627776.0f;        // 2^40
constexpr float kMassUnit = 1.0f / 1099511627776.0f;  // 2^-40
__device__ __forceinline__ unsigned long long mass_fixed(float x) {
  return __float2ull_rz(x * kMassScale);
}
__device__ __forceinline__ float mass_float(unsigned long long m) {
  return __ull2float_rn(m) * kMassUnit;
}

__global__ void __launch_bounds__(kBudgetThreads)
    budget_kernel(const int32_t* __restrict__ n_cand, const float* __restrict__ s2, int n_parts,
                  int C, int K_min, int K_max, float tau, int32_t* __restrict__ k_sel) {
  // dynamic: [C] bit patterns of the summed scores, then the bin masses
  extern __shared__ __align__(16) uint32_t key[];
  unsigned long long* hm = reinterpret_cast<unsigned long long*>(key + ((C + 3) & ~3));
  __shared__ uint32_t hc[kHistBins];
  __shared__ float wm[32];
  __shared__ uint32_t wc[32];
  __shared__ int s_bin;
  __shared__ float s_run;
  __shared__ uint32_t s_cnt;
  griddep_enter();
  const int seg = blockIdx.x, tid = threadIdx.x;
  const int nc = min(max(n_cand[seg], 0), C);
  const float* sc = s2 + size_t(seg) * C;
  const size_t part_stride = size_t(gridDim.x) * C;  // [part][N*Hkv][C]
  float part = 0.f;
  for (int i = tid; i < nc; i += kBudgetThreads) {
    float x = 0.f;
    int p = 0;
    for (; p + 2 <= n_parts; p += 2) x += sc[p * part_stride + i] + sc[(p + 1) * part_stride + i];
    if (p < n_parts) x += sc[p * part_stride + i];
    key[i] = __float_as_uint(fmaxf(x, 0.f));
    part += __uint_as_float(key[i]);
  }
  float total;
  uint32_t zero = 0u, n_unused;
  budget_scan(part, zero, wm, wc, &total, &n_unused);
  const float target = tau * total;
  int kb = nc;
  if (!(target > 0.f)) {
    kb = min(1, nc);  // no mass: one key reaches it
  } else {
    float run = 0.f;     // mass of the values above the current prefix's bin
    uint32_t cnt = 0;    // and their count
    uint32_t prefix = 0;  // the digits fixed so far
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 19 : pass == 1 ? 8 : 0;
      const int nb = pass == 0 ? 4096 : pass == 1 ? 2048 : 256;
      const uint32_t fixed = pass == 0 ? 0u : pass == 1 ? 0xFFF80000u : 0xFFFFFF00u;
      __syncthreads();  // the previous pass's readers of hm, hc and s_bin are done
      for (int b = tid; b < nb; b += kBudgetThreads) {
        hm[b] = 0ull;
        hc[b] = 0u;
      }
      if (tid == 0) s_bin = -1;
      __syncthreads();
      for (int i = tid; i < nc; i += kBudgetThreads) {
        const uint32_t v = key[i];
        if ((v & fixed) == prefix) {
          const int dgt = int((v >> shift) & uint32_t(nb - 1));
          atomicAdd(&hm[dgt], mass_fixed(__uint_as_float(v)));
          atomicAdd(&hc[dgt], 1u);
        }
      }
      __syncthreads();
      // thread t owns bins [lo, hi); the mass of the bins above its range is
      // the block total minus its inclusive prefix
      const int per = nb >= kBudgetThreads ? nb / kBudgetThreads : 1;
      const int lo = min(tid * per, nb), hi = min(lo + per, nb);
      float lm = 0.f;
      uint32_t lc = 0u;
      for (int b = lo; b < hi; ++b) {
        lm += mass_float(hm[b]);
        lc += hc[b];
      }
      float tm;
      uint32_t tcn;
      budget_scan(lm, lc, wm, wc, &tm, &tcn);
      float above = run + (tm - lm);
      for (int b = hi - 1; b >= lo; --b) {
        const float mb = mass_float(hm[b]);
        if (above < target && above + mb >= target) {
          atomicMax(&s_bin, b);  // rounding may let two ranges claim a crossing: the top one
          break;
        }
        above += mb;
      }
      __syncthreads();
      const int bin = s_bin;
      if (bin < 0) {  // the target is not reached by rounding: every member is needed
        kb = int(cnt + tcn);
        break;
      }
      if (bin >= lo && bin < hi) {  // the owner recomputes the mass and count above it
        float a = run + (tm - lm);
        uint32_t ac = cnt + (tcn - lc);
        for (int b = hi - 1; b > bin; --b) {
          a += mass_float(hm[b]);
          ac += hc[b];
        }
        s_run = a;
        s_cnt = ac;
      }
      __syncthreads();
      run = s_run;
      cnt = s_cnt;
      prefix |= uint32_t(bin) << shift;
      if (pass == 2) {
        const float t = __uint_as_float(prefix);
        const uint32_t ties = hc[bin];
        uint32_t take = t > 0.f ? uint32_t(ceilf((target - run) / t)) : 1u;
        take = max(1u, min(take, ties));
        kb = int(cnt + take);
      }
    }
  }
  if (tid == 0) k_sel[seg] = max(K_min, min(K_max, min(kb, nc)));
}

cudaError_t launch_budget(const herald_dims& dm, const int32_t* n_cand, const float* s2,
                          int n_parts, int C, int K_min, int K_max, float tau, int32_t* k_sel,
                          cudaStream_t st) {
  // the scores' bit patterns, then kHistBins fixed-point bin masses
  const size_t smem = size_t((C + 3) & ~3) * 4 + size_t(kHistBins) * 8;
  HERALD_CHECK_LAUNCH(ensure_smem(budget_kernel, smem));
  HERALD_CHECK_LAUNCH(launch_k("budget_kernel", budget_kernel, dm.N * dm.Hkv, kBudgetThreads, smem,
                               st, n_cand, s2, n_parts, C, K_min, K_max, tau, k_sel));
  return cudaGetLastError();
}

HERALD_DEBUG_WORD_READER(debug_take_select)

}  // namespace herald
