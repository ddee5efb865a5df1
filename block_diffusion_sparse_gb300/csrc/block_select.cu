// block_select.cu -- block-granular stage 1 (SparDA summary, Method section:
// InfLLM-V2 selects whole blocks of the context next to the initial tokens
// and the local window; HERALD v3 abstract: stage 1 scores the cache with
// one merged query per head):
//   pool_keys    the mean of every Bk consecutive cache rows of a (sequence,
//                KV head) below ctx, in fp32 -- the compressed keys, built
//                once and refreshed at the tail as blocks are appended
//   block_scan   the merged queries against the pooled keys: per-head logits
//                and per-warp (max, sumexp) partials in the layout of the
//                per-key scan, so that the stage-1 histogram and top-C
//                kernels run unchanged over blocks
//   expand       the selected blocks to their positions: the candidate list
//                of stage 2
#include "internal.cuh"
#include "ptx.cuh"

namespace herald {

// grid (blocks, N*Hkv), block d: thread e sums column e of a block's rows.
// full != 0: blocks [0, grid.x) of every (n, g), zero past ctx; else the last
// grid.x blocks below ctx.
__global__ void pool_keys_kernel(const uint16_t* __restrict__ kc, const int32_t* __restrict__ ctx,
                                 int Hkv, int d, int L_max, int Bk, int nb_max, int full,
                                 float* __restrict__ pooled) {
  griddep_enter();
  const int seg = blockIdx.y, n = seg / Hkv, e = threadIdx.x;
  const int L = min(max(ctx[n], 0), L_max);
  const int nb = (L + Bk - 1) / Bk;  // blocks below ctx
  const int b = full ? int(blockIdx.x) : nb - int(gridDim.x) + int(blockIdx.x);
  if (b < 0 || b >= nb_max || e >= d) return;
  float* dst = pooled + (size_t(seg) * nb_max + b) * d + e;
  if (b >= nb) {
    *dst = 0.f;
    return;
  }
  const int r0 = b * Bk, r1 = min(r0 + Bk, L);
  const uint16_t* src = kc + (size_t(seg) * L_max + r0) * d + e;
  float acc = 0.f;
  int r = r0;
  for (; r + 4 <= r1; r += 4) {
    const uint16_t u0 = src[0], u1 = src[size_t(d)], u2 = src[size_t(2) * d],
                   u3 = src[size_t(3) * d];
    acc += (__uint_as_float(uint32_t(u0) << 16) + __uint_as_float(uint32_t(u1) << 16)) +
           (__uint_as_float(uint32_t(u2) << 16) + __uint_as_float(uint32_t(u3) << 16));
    src += size_t(4) * d;
  }
  for (; r < r1; ++r, src += d) acc += __uint_as_float(uint32_t(*src) << 16);
  *dst = acc / float(r1 - r0);
}

cudaError_t launch_pool_keys(const herald_dims& dm, const uint16_t* k_cache, const int32_t* ctx,
                             int Bk, int n_tail, float* pooled, cudaStream_t st) {
  const int nb_max = cdiv(dm.L_max, Bk);
  const int blocks = n_tail > 0 ? std::min(n_tail, nb_max) : nb_max;
  HERALD_CHECK_LAUNCH(launch_k("pool_keys_kernel", pool_keys_kernel, dim3(blocks, dm.N * dm.Hkv),
                               dm.d, 0, st, k_cache, ctx, dm.Hkv, dm.d, dm.L_max, Bk, nb_max,
                               n_tail > 0 ? 0 : 1, pooled));
  return cudaGetLastError();
}

// grid (chunks, N*Hkv), block 128 (4 warps).  Warp w of CTA c scores pooled
// rows c*4 + w, c*4 + w + 4*chunks, ... of its (n, g): each lane holds d/32
// values of the row and of every head's (pre-scaled) merged query, the G dot
// products are butterfly sums, and the warp's running (max, sumexp) per head
// goes to part1 slot c*4 + w at the end.  CTA (0, 0) also writes the block
// counts ctx_b[n] = ceil(ctx[n] / Bk) that the later kernels read.
constexpr int kBlockScanThreads = 128;

template <int G>
__global__ void __launch_bounds__(kBlockScanThreads)
    block_scan_kernel(const float* __restrict__ pooled, const float* __restrict__ qbar,
                      const int32_t* __restrict__ ctx, int N, int Hkv, int d, int L_max, int Bk,
                      int nb_max, int L_pad, float* __restrict__ logits,
                      float2* __restrict__ part1, int32_t* __restrict__ ctx_b) {
  griddep_enter();
  const int seg = blockIdx.y, n = seg / Hkv, g = seg - n * Hkv, Hq = Hkv * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = min(max(ctx[n], 0), L_max);
  const int nb = (L + Bk - 1) / Bk;
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < N; i += kBlockScanThreads)
      ctx_b[i] = (min(max(ctx[i], 0), L_max) + Bk - 1) / Bk;
  const int per = d / 32;  // 2 or 4 values per lane
  float q[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int k = 0; k < 4; ++k)
      q[h][k] = k < per ? qbar[(size_t(n) * Hq + g * G + h) * d + lane * per + k] : 0.f;
  float m[G], s[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    s[h] = 0.f;
  }
  const int stride = int(gridDim.x) * 4;
  for (int b = int(blockIdx.x) * 4 + warp; b < nb; b += stride) {
    const float* row = pooled + (size_t(seg) * nb_max + b) * d + lane * per;
    float k[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = i < per ? row[i] : 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc = fmaf(q[h][i], k[i], acc);
      const float l = warp_sum(acc);  // every lane holds the logit
      if (lane == 0) logits[(size_t(n) * Hq + g * G + h) * L_pad + b] = l;
      if (l > m[h]) {
        s[h] = s[h] * __expf(m[h] - l) + 1.f;
        m[h] = l;
      } else {
        s[h] += __expf(l - m[h]);
      }
    }
  }
  if (lane == 0) {
    const int slot = blockIdx.x * 4 + warp;
#pragma unroll
    for (int h = 0; h < G; ++h)
      part1[(size_t(n) * Hq + g * G + h) * kPartSlots + slot] = make_float2(m[h], s[h]);
  }
}

int block_scan_chunks(const herald_dims& dm, int num_sms) {
  const int segs = dm.N * dm.Hkv;
  return std::max(1, std::min(kPartSlots / 4, cdiv(2 * num_sms, segs)));
}

cudaError_t launch_block_scan(const herald_dims& dm, const float* pooled, const float* qbar,
                              const int32_t* ctx, int Bk, int L_pad, float* logits,
                              float2* part1, int32_t* ctx_b, int chunks, cudaStream_t st) {
  const int nb_max = cdiv(dm.L_max, Bk);
  const dim3 grid(chunks, dm.N * dm.Hkv);
  switch (dm.Hq / dm.Hkv) {
#define HERALD_BS_G(GG)                                                                        \
  case GG:                                                                                     \
    HERALD_CHECK_LAUNCH(launch_k("block_scan_kernel", block_scan_kernel<GG>, grid,             \
                                 kBlockScanThreads, 0, st, pooled, qbar, ctx, dm.N, dm.Hkv,    \
                                 dm.d, dm.L_max, Bk, nb_max, L_pad, logits, part1, ctx_b));    \
    break;
    HERALD_BS_G(1) HERALD_BS_G(2) HERALD_BS_G(3) HERALD_BS_G(4)
    HERALD_BS_G(5) HERALD_BS_G(6) HERALD_BS_G(7) HERALD_BS_G(8)
#undef HERALD_BS_G
    default: break;
  }
  return cudaGetLastError();
}

// grid (N*Hkv), block 256.  Slot i of the candidate row is position
// cand_b[i / Bk] * Bk + i % Bk: the selected blocks are ascending, so every
// block but the highest is whole and the row stays compact; positions at or
// past ctx (the end of the block holding the last cached key) are -1.
__global__ void expand_blocks_kernel(const int32_t* __restrict__ cand_b,
                                     const int32_t* __restrict__ n_cand_b,
                                     const int32_t* __restrict__ ctx, int Hkv, int L_max, int Bk,
                                     int C_blocks, int32_t* __restrict__ cand,
                                     int32_t* __restrict__ n_cand) {
  griddep_enter();
  const int seg = blockIdx.x, n = seg / Hkv;
  const int L = min(max(ctx[n], 0), L_max);
  const int nbs = min(max(n_cand_b[seg], 0), C_blocks);
  const int C = C_blocks * Bk;
  const int32_t* cb = cand_b + size_t(seg) * C_blocks;
  int32_t* out = cand + size_t(seg) * C;
  for (int i = threadIdx.x; i < C; i += blockDim.x) {
    const int r = i / Bk;
    int pos = -1;
    if (r < nbs) {
      const int j = cb[r] * Bk + (i - r * Bk);
      if (cb[r] >= 0 && j < L) pos = j;
    }
    out[i] = pos;
  }
  if (threadIdx.x == 0) {
    int cnt = 0;
    if (nbs > 0) {
      const int last = cb[nbs - 1];
      cnt = (nbs - 1) * Bk + max(0, min(Bk, L - last * Bk));
    }
    n_cand[seg] = cnt;
  }
}

cudaError_t launch_expand_blocks(const herald_dims& dm, const int32_t* cand_b,
                                 const int32_t* n_cand_b, const int32_t* ctx, int Bk,
                                 int C_blocks, int32_t* cand, int32_t* n_cand, cudaStream_t st) {
  HERALD_CHECK_LAUNCH(launch_k("expand_blocks_kernel", expand_blocks_kernel, dm.N * dm.Hkv, 256,
                               0, st, cand_b, n_cand_b, ctx, dm.Hkv, dm.L_max, Bk, C_blocks, cand,
                               n_cand));
  return cudaGetLastError();
}

HERALD_DEBUG_WORD_READER(debug_take_blocks)

}  // namespace herald
