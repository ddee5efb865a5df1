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
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace herald {

// ============================================================ merge_query
// grid (N*Hq), block d.  Also zeroes the stage-1 histogram.
__global__ void merge_query_kernel(const uint16_t* __restrict__ q, int B, int Hq, int d,
                                   float scale, float* __restrict__ qbar,
                                   uint32_t* __restrict__ hist, int hist_words) {
  const int nh = blockIdx.x, n = nh / Hq, h = nh % Hq, e = threadIdx.x;
  if (e < d) {
    float acc = 0.f;
    for (int b = 0; b < B; ++b) {
      const uint16_t u = q[((size_t(n) * B + b) * Hq + h) * d + e];
      acc += __uint_as_float(uint32_t(u) << 16);
    }
    qbar[size_t(nh) * d + e] = acc / float(B) * scale;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < hist_words; i += gridDim.x * blockDim.x)
    hist[i] = 0u;
}

cudaError_t launch_merge_query(const herald_dims& dm, const uint16_t* q_merge, float* qbar,
                               uint32_t* hist, cudaStream_t st) {
  const float scale = 1.0f / sqrtf(float(dm.d));
  trace_before(st, "merge_query_kernel");
  merge_query_kernel<<<dm.N * dm.Hq, dm.d, 0, st>>>(q_merge, dm.B, dm.Hq, dm.d, scale, qbar,
                                                    hist, dm.N * dm.Hkv * kHistBins);
  trace_after(st);
  return cudaGetLastError();
}

// =================================================================== scan
// Persistent: grid = #SMs.  Flattened tiles t = seg * tiles_per_seg + tile
// (seg = n*Hkv + g) are split into contiguous per-CTA ranges; warp w of a CTA
// takes tiles begin+w, begin+w+kScanWarps, ... through its own ring of
// kScanStages shared-memory stages.  Each lane owns keys lane and lane+32 of
// a 64-key tile; the two keys are the two halves of packed f32x2 FMAs.
template <int D>
struct ScanCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kScanTileKeys * 128;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kSmem = kScanWarps * kScanStages * kTileBytes + 1024;
};

template <int D, int G, bool TMA>
__global__ void __launch_bounds__(kScanWarps * 32, 1)
    scan_kernel(const __grid_constant__ CUtensorMap kmap, const uint16_t* __restrict__ kc,
                const float* __restrict__ qbar, const int32_t* __restrict__ ctx, int Hkv,
                int L_max, int tiles_per_seg, int total_tiles, int L_pad,
                float* __restrict__ logits, float2* __restrict__ part1, uint32_t* err) {
  using Cfg = ScanCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[kScanWarps][kScanStages];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = Hkv * G;
  uint8_t* ring = smem + warp * kScanStages * Cfg::kTileBytes;
  const int t_begin = int((long long)blockIdx.x * total_tiles / gridDim.x);
  const int t_end = int((long long)(blockIdx.x + 1) * total_tiles / gridDim.x);

  if (TMA && lane == 0) {
    tma_prefetch_desc(&kmap);
    for (int s = 0; s < kScanStages; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Issues the load of this warp's i-th tile into `stage`; returns whether a
  // load was issued (tiles past the context are skipped).
  auto issue = [&](int i, int stage) -> bool {
    const int t = t_begin + warp + i * kScanWarps;
    bool ok = t < t_end;
    int seg = 0, j0 = 0, L = 0;
    if (ok) {
      seg = t / tiles_per_seg;
      j0 = (t - seg * tiles_per_seg) * kScanTileKeys;
      L = min(max(ctx[seg / Hkv], 0), L_max);
      ok = j0 < L;
    }
    uint8_t* dst = ring + stage * Cfg::kTileBytes;
    if constexpr (TMA) {
      if (ok && lane == 0) {
        mbar_arrive_expect_tx(&bars[warp][stage], Cfg::kTileBytes);
#pragma unroll
        for (int hv = 0; hv < Cfg::kHalves; ++hv)
          tma_load_2d(dst + hv * Cfg::kHalfBytes, &kmap, &bars[warp][stage], hv * 64,
                      seg * L_max + j0);
      }
    } else {
      if (ok) {
        const uint16_t* base = kc + size_t(seg) * L_max * D;
        // 64 rows x D/8 chunks of 16 bytes, spread over the 32 lanes
        for (int q = lane; q < kScanTileKeys * (D / 8); q += 32) {
          const int r = q / (D / 8), c = q % (D / 8);
          const int j = j0 + r;
          const bool v = j < L;
          const uint16_t* src = base + size_t(v ? j : 0) * D + c * 8;
          cp_async_16(dst + (c >> 3) * Cfg::kHalfBytes + sw128_off(r, c & 7), src, v ? 16u : 0u);
        }
      }
      cp_async_commit();
    }
    return ok;
  };

  uint32_t issued = 0, phase = 0;
#pragma unroll
  for (int s = 0; s < kScanStages; ++s) issued |= uint32_t(issue(s, s)) << s;

  bool timed_out = false;
  for (int i = 0;; ++i) {
    const int t = t_begin + warp + i * kScanWarps;
    if (t >= t_end) break;
    const int stage = i % kScanStages;
    const bool valid = (issued >> stage) & 1u;
    const int seg = t / tiles_per_seg;
    const int tl = t - seg * tiles_per_seg;
    const int n = seg / Hkv, g = seg - n * Hkv;
    const int j0 = tl * kScanTileKeys;
    float2 acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
    if (valid) {
      if constexpr (TMA) {
        if (!mbar_wait(&bars[warp][stage], (phase >> stage) & 1u)) {
          timed_out = true;
        }
        phase ^= 1u << stage;
      } else {
        asm volatile("cp.async.wait_group %0;" ::"n"(kScanStages - 1) : "memory");
        __syncwarp();
      }
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
    // every lane has consumed the stage: refill it
    __syncwarp();
    if (!timed_out) {
      const bool nv = issue(i + kScanStages, stage);
      issued = (issued & ~(1u << stage)) | (uint32_t(nv) << stage);
    } else {
      issued &= ~(1u << stage);
    }
    if (valid) {
      const int L = min(max(ctx[n], 0), L_max);
      const int ja = j0 + lane, jb = j0 + lane + 32;
      const bool va = ja < L, vb = jb < L;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const size_t row = (size_t(n) * Hq + g * G + h);
        float* lr = logits + row * L_pad;
        if (va) lr[ja] = acc[h].x;
        if (vb) lr[jb] = acc[h].y;
        const float la = va ? acc[h].x : -INFINITY, lb = vb ? acc[h].y : -INFINITY;
        const float m = warp_max(fmaxf(la, lb));
        const float s = warp_sum((va ? __expf(la - m) : 0.f) + (vb ? __expf(lb - m) : 0.f));
        if (lane == 0) part1[row * tiles_per_seg + tl] = make_float2(m, s);
      }
    }
    if (timed_out) break;
  }
  if constexpr (TMA) {
    if (timed_out) {
      if (lane == 0) record_error(err, DEV_TIMEOUT_TMA);
      // wait (bounded) for any load still in flight before leaving
      for (int s = 0; s < kScanStages; ++s)
        if ((issued >> s) & 1u) (void)mbar_wait(&bars[warp][s], (phase >> s) & 1u);
    }
  } else {
    cp_async_wait_all();
  }
}

template <int D, int G, bool TMA>
static cudaError_t launch_scan_t(const CUtensorMap* kmap, const uint16_t* kc, const float* qbar,
                                 const int32_t* ctx, const herald_dims& dm, float* logits,
                                 float2* part1, const WsLayout& w, uint32_t* err, int num_sms,
                                 cudaStream_t st) {
  using Cfg = ScanCfg<D>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<D, G, TMA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int total = dm.N * dm.Hkv * w.tiles_per_seg;
  const int grid = total < num_sms ? total : num_sms;
  CUtensorMap dummy{};
  trace_before(st, "scan_kernel");
  scan_kernel<D, G, TMA><<<grid, kScanWarps * 32, Cfg::kSmem, st>>>(
      kmap ? *kmap : dummy, kc, qbar, ctx, dm.Hkv, dm.L_max, w.tiles_per_seg, total, w.L_pad,
      logits, part1, err);
  trace_after(st);
  return cudaGetLastError();
}

template <int D, bool TMA>
static cudaError_t scan_dispatch_g(int G, const CUtensorMap* kmap, const uint16_t* kc,
                                   const float* qbar, const int32_t* ctx, const herald_dims& dm,
                                   float* logits, float2* part1, const WsLayout& w,
                                   uint32_t* err, int num_sms, cudaStream_t st) {
#define HERALD_SCAN_G(GG)                                                                       \
  case GG:                                                                                      \
    return launch_scan_t<D, GG, TMA>(kmap, kc, qbar, ctx, dm, logits, part1, w, err, num_sms, \
                                     st);
  switch (G) {
    HERALD_SCAN_G(1) HERALD_SCAN_G(2) HERALD_SCAN_G(3) HERALD_SCAN_G(4)
    HERALD_SCAN_G(5) HERALD_SCAN_G(6) HERALD_SCAN_G(7) HERALD_SCAN_G(8)
    default: return cudaErrorInvalidValue;
  }
#undef HERALD_SCAN_G
}

cudaError_t launch_scan(const herald_dims& dm, const CUtensorMap* kmap, const uint16_t* k_cache,
                        bool use_tma, const float* qbar, const int32_t* ctx, float* logits,
                        float2* part1, const WsLayout& w, uint32_t* err, int num_sms,
                        cudaStream_t st) {
  const int G = dm.Hq / dm.Hkv;
  if (dm.d == 128)
    return use_tma ? scan_dispatch_g<128, true>(G, kmap, k_cache, qbar, ctx, dm, logits, part1,
                                                w, err, num_sms, st)
                   : scan_dispatch_g<128, false>(G, kmap, k_cache, qbar, ctx, dm, logits, part1,
                                                 w, err, num_sms, st);
  return use_tma ? scan_dispatch_g<64, true>(G, kmap, k_cache, qbar, ctx, dm, logits, part1, w,
                                             err, num_sms, st)
                 : scan_dispatch_g<64, false>(G, kmap, k_cache, qbar, ctx, dm, logits, part1, w,
                                              err, num_sms, st);
}

// ================================================================ s1_hist
// grid (chunks, N*Hkv), block 256.  Each CTA folds the per-tile partials of
// its G heads into lse_h, then scores its key range and bins the fp32 bit
// pattern of s1 (non-negative, so bit order = value order).
constexpr int kS1Threads = 256;

__global__ void __launch_bounds__(kS1Threads)
    s1_hist_kernel(const float* __restrict__ logits, const float2* __restrict__ part1,
                   const int32_t* __restrict__ ctx, int Hkv, int G, int L_max, int L_pad,
                   int tiles_per_seg, int keys_per_cta, float* __restrict__ s1,
                   uint32_t* __restrict__ hist) {
  __shared__ uint32_t sh[kHistBins];
  __shared__ float lse[8];
  const int seg = blockIdx.y, n = seg / Hkv, g = seg - n * Hkv;
  const int Hq = Hkv * G;
  const int L = min(max(ctx[n], 0), L_max);
  const int j_begin = blockIdx.x * keys_per_cta;
  if (j_begin >= L) return;
  const int j_end = min(L, j_begin + keys_per_cta);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kHistBins; i += kS1Threads) sh[i] = 0u;
  if (warp < G) {
    const int ntiles = (L + kScanTileKeys - 1) / kScanTileKeys;
    const float2* p = part1 + (size_t(n) * Hq + g * G + warp) * tiles_per_seg;
    float m = -INFINITY, s = 0.f;
    for (int t = lane; t < ntiles; t += 32) {
      const float2 v = p[t];
      if (v.x > m) { s = s * __expf(m - v.x) + v.y; m = v.x; }
      else s += v.y * __expf(v.x - m);
    }
    const float M = warp_max(m);
    s = warp_sum(m == -INFINITY ? 0.f : s * __expf(m - M));
    if (lane == 0) lse[warp] = M + __logf(s);
  }
  __syncthreads();
  const float* lg = logits + (size_t(n) * Hq + g * G) * L_pad;
  float* out = s1 + size_t(seg) * L_pad;
  for (int j = j_begin + threadIdx.x; j < j_end; j += kS1Threads) {
    float acc = 0.f;
    for (int h = 0; h < G; ++h) acc += __expf(lg[size_t(h) * L_pad + j] - lse[h]);
    out[j] = acc;
    atomicAdd(&sh[(__float_as_uint(acc) >> kHistShift) & (kHistBins - 1)], 1u);
  }
  __syncthreads();
  uint32_t* gh = hist + size_t(seg) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kS1Threads)
    if (sh[i]) atomicAdd(&gh[i], sh[i]);
}

cudaError_t launch_s1_hist(const herald_dims& dm, const float* logits, const float2* part1,
                           const int32_t* ctx, float* s1, uint32_t* hist, const WsLayout& w,
                           int num_sms, cudaStream_t st) {
  const int segs = dm.N * dm.Hkv;
  int chunks = (2 * num_sms + segs - 1) / segs;
  int keys = cdiv(dm.L_max, chunks);
  keys = cdiv(keys, 256) * 256;
  if (keys < 1024) keys = 1024;
  chunks = cdiv(dm.L_max, keys);
  trace_before(st, "s1_hist_kernel");
  s1_hist_kernel<<<dim3(chunks, segs), kS1Threads, 0, st>>>(
      logits, part1, ctx, dm.Hkv, dm.Hq / dm.Hkv, dm.L_max, w.L_pad, w.tiles_per_seg, keys, s1,
      hist);
  trace_after(st);
  return cudaGetLastError();
}

// ============================================================ block scans
// Block-wide exclusive prefix sum for 1024 threads; returns the total.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot,
                                                    uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < NT / 32 ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NT / 32) warp_tot[lane] = t;  // inclusive
  }
  __syncthreads();
  const uint32_t before = (warp ? warp_tot[warp - 1] : 0u) + x - v;
  total = warp_tot[NT / 32 - 1];
  __syncthreads();
  return before;
}

// Given a histogram h[0..nb) (in shared memory) and a rank `need` (1-based
// count of largest elements wanted), finds the bin b holding the need-th
// largest element; returns b and the count strictly above it.
template <int NT>
__device__ void find_bin_from_top(const uint32_t* h, int nb, uint32_t need, uint32_t* warp_tot,
                                  int* out_bin, uint32_t* out_above) {
  // thread t owns bins [t*per, (t+1)*per) counted from the TOP
  const int per = (nb + NT - 1) / NT;
  uint32_t local = 0;
  for (int k = 0; k < per; ++k) {
    const int rb = threadIdx.x * per + k;  // rank-order bin (0 = highest)
    if (rb < nb) local += h[nb - 1 - rb];
  }
  uint32_t total;
  const uint32_t before = block_excl_scan<NT>(local, warp_tot, total);
  if (before < need && need <= before + local) {
    uint32_t acc = before;
    for (int k = 0; k < per; ++k) {
      const int rb = threadIdx.x * per + k;
      if (rb >= nb) break;
      const uint32_t c = h[nb - 1 - rb];
      if (acc + c >= need) {
        *out_bin = nb - 1 - rb;
        *out_above = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// ============================================================ topc_finish
// One CTA of 1024 threads per (n, g).  Radix select of the C-th largest s1:
// the first 12-bit digit comes from the global histogram; the members of
// that bin are collected into shared memory (bounded; a global two-digit
// fallback handles overflow) and the remaining 19 bits are resolved there.
// The ordered compaction then keeps every s1 above the threshold plus the
// lowest-position ties, with one two-counter block scan.
constexpr int kSelThreads = 1024;
constexpr int kTieCap = 6144;

// Block-wide exclusive scan of two counters at once (1024 threads).
__device__ __forceinline__ void block_excl_scan2(uint32_t a, uint32_t b, uint32_t* wa,
                                                 uint32_t* wb, uint32_t& ea, uint32_t& eb,
                                                 uint32_t& ta, uint32_t& tb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = a, y = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t xa = __shfl_up_sync(0xffffffffu, x, o);
    const uint32_t yb = __shfl_up_sync(0xffffffffu, y, o);
    if (lane >= o) { x += xa; y += yb; }
  }
  if (lane == 31) { wa[warp] = x; wb[warp] = y; }
  __syncthreads();
  if (warp == 0) {
    uint32_t u = wa[lane], v = wb[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ua = __shfl_up_sync(0xffffffffu, u, o);
      const uint32_t vb = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) { u += ua; v += vb; }
    }
    wa[lane] = u;
    wb[lane] = v;
  }
  __syncthreads();
  ea = (warp ? wa[warp - 1] : 0u) + x - a;
  eb = (warp ? wb[warp - 1] : 0u) + y - b;
  ta = wa[31];
  tb = wb[31];
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads)
    topc_finish_kernel(const float* __restrict__ s1, const uint32_t* __restrict__ hist,
                       const int32_t* __restrict__ ctx, int Hkv, int L_max, int L_pad, int C,
                       int32_t* __restrict__ cand, int32_t* __restrict__ n_cand) {
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t tie_v[kTieCap];
  __shared__ uint32_t wt[32], wt2[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above, s_cnt;
  const int seg = blockIdx.x, n = seg / Hkv;
  const int L = min(max(ctx[n], 0), L_max);
  const int Ce = min(C, L);
  int32_t* out = cand + size_t(seg) * C;
  const uint32_t* sv = reinterpret_cast<const uint32_t*>(s1 + size_t(seg) * L_pad);
  if (threadIdx.x == 0) n_cand[seg] = Ce;
  for (int i = Ce + threadIdx.x; i < C; i += kSelThreads) out[i] = -1;
  if (Ce == L) {
    for (int i = threadIdx.x; i < L; i += kSelThreads) out[i] = i;
    return;
  }
  // digit 1: bits [30:19] from the global histogram
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads)
    h[i] = hist[size_t(seg) * kHistBins + i];
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  uint32_t need = uint32_t(Ce);
  find_bin_from_top<kSelThreads>(h, kHistBins, need, wt, &s_bin, &s_above);
  const uint32_t b1 = uint32_t(s_bin);
  need -= s_above;
  // collect the low 19 bits of the members of bin b1
  for (int j = threadIdx.x; j < L; j += kSelThreads) {
    const uint32_t v = sv[j];
    if ((v >> 19) == b1) {
      const uint32_t slot = atomicAdd(&s_cnt, 1u);
      if (slot < kTieCap) tie_v[slot] = v & 0x7FFFFu;
    }
  }
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
  find_bin_from_top<kSelThreads>(h, 2048, need, wt, &s_bin, &s_above);
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
  // ordered compaction: thread t owns positions [t*E, (t+1)*E)
  const int E = (L + kSelThreads - 1) / kSelThreads;
  const int j0 = threadIdx.x * E, j1 = min(L, j0 + E);
  uint32_t n_gt = 0, n_eq = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t v = sv[j];
    n_gt += v > tau;
    n_eq += v == tau;
  }
  uint32_t gt_before, eq_before, gt_tot, eq_tot;
  block_excl_scan2(n_gt, n_eq, wt, wt2, gt_before, eq_before, gt_tot, eq_tot);
  for (int j = j0; j < j1; ++j) {
    const uint32_t v = sv[j];
    if (v > tau) {
      const uint32_t pos = gt_before + min(eq_before, need_eq);
      if (pos < uint32_t(Ce)) out[pos] = j;
      ++gt_before;
    } else if (v == tau) {
      if (eq_before < need_eq && gt_before + eq_before < uint32_t(Ce)) out[gt_before + eq_before] = j;
      ++eq_before;
    }
  }
}

cudaError_t launch_topc(const herald_dims& dm, const float* s1, const uint32_t* hist,
                        const int32_t* ctx, int C, int32_t* cand, int32_t* n_cand,
                        const WsLayout& w, cudaStream_t st) {
  trace_before(st, "topc_finish_kernel");
  topc_finish_kernel<<<dm.N * dm.Hkv, kSelThreads, 0, st>>>(s1, hist, ctx, dm.Hkv, dm.L_max,
                                                            w.L_pad, C, cand, n_cand);
  trace_after(st);
  return cudaGetLastError();
}

// ============================================================= topk_union
// One CTA of 1024 threads per (n, g).  s2 of the n_cand candidates is held in
// shared memory; a 4 x 8-bit radix select finds the K-th largest, ties go to
// the lower slot (= lower position, candidates being ascending).  The output
// is [0, sink_end) ++ kept candidates in [sink_end, local_begin) ++
// [local_begin, L), which is the deduplicated ascending union.
__global__ void __launch_bounds__(kSelThreads)
    topk_union_kernel(const int32_t* __restrict__ ctx, const int32_t* __restrict__ cand,
                      const int32_t* __restrict__ n_cand, const float* __restrict__ s2, int Hkv,
                      int L_max, int C, int K, int S, int W, int P_max, int32_t* __restrict__ idx,
                      int32_t* __restrict__ n_sel) {
  extern __shared__ uint32_t sv[];  // [C]
  __shared__ uint32_t h[256];
  __shared__ uint32_t wt[32];
  __shared__ int s_bin;
  __shared__ uint32_t s_above;
  const int seg = blockIdx.x, n = seg / Hkv;
  const int L = min(max(ctx[n], 0), L_max);
  const int nc = min(max(n_cand[seg], 0), C);
  const int Ke = min(K, nc);
  const int32_t* cd = cand + size_t(seg) * C;
  for (int i = threadIdx.x; i < nc; i += kSelThreads)
    sv[i] = __float_as_uint(fmaxf(s2[size_t(seg) * C + i], 0.f));
  __syncthreads();
  uint32_t tau = 0, need_eq = 0;
  bool take_all = (Ke == nc);
  if (!take_all && Ke > 0) {
    uint32_t need = uint32_t(Ke), prefix = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kSelThreads) h[i] = 0u;
      __syncthreads();
      for (int i = threadIdx.x; i < nc; i += kSelThreads) {
        const uint32_t v = sv[i];
        if (shift == 24 || (v >> (shift + 8)) == prefix) atomicAdd(&h[(v >> shift) & 255u], 1u);
      }
      __syncthreads();
      find_bin_from_top<kSelThreads>(h, 256, need, wt, &s_bin, &s_above);
      prefix = (prefix << 8) | uint32_t(s_bin);
      need -= s_above;
    }
    tau = prefix;
    need_eq = need;
  }
  const int sink_end = min(S, L);
  const int local_begin = max(L - W, sink_end);
  int32_t* out = idx + size_t(seg) * P_max;
  // middle part, in slot order
  uint32_t base = 0, eq_base = 0;
  for (int i0 = 0; i0 < nc; i0 += kSelThreads) {
    const int i = i0 + threadIdx.x;
    const bool in = i < nc;
    const uint32_t v = in ? sv[i] : 0u;
    const uint32_t is_eq = (in && !take_all && Ke > 0 && v == tau) ? 1u : 0u;
    uint32_t eq_tot;
    const uint32_t eq_rank = eq_base + block_excl_scan<kSelThreads>(is_eq, wt, eq_tot);
    bool keep = in && Ke > 0 && (take_all || v > tau || (is_eq && eq_rank < need_eq));
    int pos = in ? cd[i] : -1;
    keep = keep && pos >= sink_end && pos < local_begin;
    uint32_t tot;
    const uint32_t at = base + block_excl_scan<kSelThreads>(keep ? 1u : 0u, wt, tot);
    if (keep && sink_end + int(at) < P_max) out[sink_end + at] = pos;
    base += tot;
    eq_base += eq_tot;
  }
  const int n_mid = int(base);
  for (int j = threadIdx.x; j < sink_end; j += kSelThreads) out[j] = j;
  for (int j = local_begin + threadIdx.x; j < L; j += kSelThreads)
    if (sink_end + n_mid + (j - local_begin) < P_max) out[sink_end + n_mid + (j - local_begin)] = j;
  const int total = min(P_max, sink_end + n_mid + (L - local_begin));
  for (int s = total + threadIdx.x; s < P_max; s += kSelThreads) out[s] = -1;
  if (threadIdx.x == 0) n_sel[seg] = total;
}

cudaError_t launch_topk_union(const herald_dims& dm, const int32_t* ctx, const int32_t* cand,
                              const int32_t* n_cand, const float* s2, int C, int K, int S, int W,
                              int P_max, int32_t* idx, int32_t* n_sel, cudaStream_t st) {
  const size_t smem = size_t(C) * 4;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(topk_union_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxC * 4);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  trace_before(st, "topk_union_kernel");
  topk_union_kernel<<<dm.N * dm.Hkv, kSelThreads, smem, st>>>(ctx, cand, n_cand, s2, dm.Hkv,
                                                               dm.L_max, C, K, S, W, P_max, idx,
                                                               n_sel);
  trace_after(st);
  return cudaGetLastError();
}

}  // namespace herald
