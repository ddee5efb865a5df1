// block_scan.cuh -- block-wide scans and the radix-select bin searches shared
// by the selection kernels (select_kernels.cu).
#pragma once
#include <stdint.h>

namespace herald {

// Block-wide exclusive prefix sum for NT threads; returns the total.
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

// Block-wide exclusive scan of two counters at once (NT threads).
template <int NT = 1024>
__device__ __forceinline__ void block_excl_scan2(uint32_t a, uint32_t b, uint32_t* wa,
                                                 uint32_t* wb, uint32_t& ea, uint32_t& eb,
                                                 uint32_t& ta, uint32_t& tb) {
  constexpr int NW = NT / 32;
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
    uint32_t u = lane < NW ? wa[lane] : 0u, v = lane < NW ? wb[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ua = __shfl_up_sync(0xffffffffu, u, o);
      const uint32_t vb = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) { u += ua; v += vb; }
    }
    if (lane < NW) { wa[lane] = u; wb[lane] = v; }
  }
  __syncthreads();
  ea = (warp ? wa[warp - 1] : 0u) + x - a;
  eb = (warp ? wb[warp - 1] : 0u) + y - b;
  ta = wa[NW - 1];
  tb = wb[NW - 1];
  __syncthreads();
}

// The bin holding the need-th largest element of a wide histogram h[0..nb)
// (nb a multiple of 32 * 32; rank order counts from the top bin) and the
// count strictly above it: every warp sums its nb/32 bins with lane-strided
// (bank-conflict-free) reads, warp 0 scans the warp totals, and only the
// warp holding the rank walks its bins in order.
template <int NT>
__device__ void find_bin_wide(const uint32_t* h, int nb, uint32_t need, uint32_t* warp_tot,
                              int* s_warp, uint32_t* s_before, int* out_bin,
                              uint32_t* out_above) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_w = nb / NW;  // rank-order bins of a warp
  uint32_t sum = 0;
  for (int k = lane; k < per_w; k += 32) sum += h[nb - 1 - (warp * per_w + k)];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) warp_tot[warp] = sum;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = lane < NW ? warp_tot[lane] : 0u;
    uint32_t incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - t;
    if (lane < NW && excl < need && need <= incl) {
      *s_warp = lane;
      *s_before = excl;
    }
  }
  __syncthreads();
  const int W = *s_warp;
  if (warp == W) {
    const int per_l = per_w / 32;  // consecutive rank-order bins of a lane
    const int rb0 = W * per_w + lane * per_l;
    uint32_t local = 0;
    for (int k = 0; k < per_l; ++k) local += h[nb - 1 - (rb0 + k)];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t acc = *s_before + incl - local;
    if (acc < need && need <= acc + local) {
      for (int k = 0; k < per_l; ++k) {
        const uint32_t c = h[nb - 1 - (rb0 + k)];
        if (acc + c >= need) {
          *out_bin = nb - 1 - (rb0 + k);
          *out_above = acc;
          break;
        }
        acc += c;
      }
    }
  }
  __syncthreads();
}

}  // namespace herald
