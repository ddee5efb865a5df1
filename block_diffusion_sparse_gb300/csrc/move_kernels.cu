// move_kernels.cu -- data movement on the HERALD path:
//   gather  the selected cache rows into one buffer of the double-buffered
//           sparse KV pool (HERALD early abstract: the subset crosses the
//           host link once per block and is reused for all T steps); the
//           source may be HBM or mapped pinned host memory
//   append  the decoded block's K/V rows at the end of the cache (HERALD v3
//           abstract: the cache grows as blocks are decoded)
#include "internal.cuh"
#include "ptx.cuh"

namespace herald {

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// grid (ceil(P_max / rows_per_cta), N*Hkv), block 256; D/8 threads per row,
// one 16-byte chunk each.  With vc == nullptr only K rows are copied (the
// staging of candidate K rows from a host-resident cache; the staging of K
// and V rows passes both).  With src,
// a row whose src entry is a candidate slot s >= 0 is read from the rows
// staged by slot (sk, sv: [N*Hkv][C][D]) instead of the cache.
template <int D>
__global__ void __launch_bounds__(256)
    gather_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ n_sel, int P_max,
                  int L_max, const uint16_t* __restrict__ kc, const uint16_t* __restrict__ vc,
                  uint16_t* __restrict__ pk, uint16_t* __restrict__ pv,
                  const int32_t* __restrict__ src, int C, const uint16_t* __restrict__ sk,
                  const uint16_t* __restrict__ sv) {
  constexpr int TPR = D / 8, RPC = 256 / TPR;
  griddep_enter();
  const int seg = blockIdx.y;
  const int c = threadIdx.x % TPR;
  // rows blockIdx.x*RPC + ..., then a grid stride (a grid smaller than the
  // rows leaves SMs to kernels on other streams)
  for (int row = blockIdx.x * RPC + threadIdx.x / TPR; row < P_max; row += gridDim.x * RPC) {
    // idx (and src) are read with n_sel, not after it: the row lies inside
    // the index buffer either way, and its entry is used only below n_sel
    const int pos = idx[size_t(seg) * P_max + row];
    const int s = src ? src[size_t(seg) * P_max + row] : -1;
    const int ns_raw = n_sel[seg];
    debug_flag(ns_raw < 0 || ns_raw > P_max, DEV_BAD_COUNT);
    const int ns = min(max(ns_raw, 0), P_max);
    uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
    if (row < ns) {
      if (s >= 0 && s < C) {  // a candidate row staged in HBM by slot
        const size_t off = (size_t(seg) * C + s) * D + c * 8;
        kv = ld_nc_v4(sk + off);
        if (vc) vv = ld_nc_v4(sv + off);
      } else if (pos >= 0 && pos < L_max) {
        const size_t off = (size_t(seg) * L_max + pos) * D + c * 8;
        kv = ld_nc_v4(kc + off);
        if (vc) vv = ld_nc_v4(vc + off);
      } else {
        debug_flag(true, DEV_BAD_INDEX);  // a selected row outside the cache
      }
    }
    const size_t dst = (size_t(seg) * P_max + row) * D + c * 8;
    *reinterpret_cast<uint4*>(pk + dst) = kv;
    if (vc) *reinterpret_cast<uint4*>(pv + dst) = vv;
  }
}

// One thread waits on an mbarrier that nothing completes, through the same
// bounded wait every kernel uses, with a caller-chosen limit; it records the
// timeout in the error word and returns.  Exercises the device-side failure
// path without faulting or hanging the GPU.
__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, limit_ns)) record_error(err, DEV_TIMEOUT_TMA);
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, uint32_t* err, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, err);
  return cudaGetLastError();
}

static cudaError_t gather_launch(const herald_dims& dm, const int32_t* idx,
                                 const int32_t* n_sel, int P_max, const uint16_t* k_cache,
                                 const uint16_t* v_cache, uint16_t* pool_k, uint16_t* pool_v,
                                 const int32_t* src, int C, const uint16_t* staged_k,
                                 const uint16_t* staged_v, cudaStream_t st, const char* name,
                                 int max_ctas) {
  const int segs = dm.N * dm.Hkv;
  const int rpc = dm.d == 128 ? 16 : 32;  // rows per CTA and round
  int gx = cdiv(P_max, rpc);
  if (max_ctas > 0) gx = std::max(1, std::min(gx, max_ctas / segs));
  if (dm.d == 128)
    HERALD_CHECK_LAUNCH(launch_k(name, gather_kernel<128>, dim3(gx, segs), 256, 0, st, idx, n_sel,
                                 P_max, dm.L_max, k_cache, v_cache, pool_k, pool_v, src, C,
                                 staged_k, staged_v));
  else
    HERALD_CHECK_LAUNCH(launch_k(name, gather_kernel<64>, dim3(gx, segs), 256, 0, st, idx, n_sel,
                                 P_max, dm.L_max, k_cache, v_cache, pool_k, pool_v, src, C,
                                 staged_k, staged_v));
  return cudaGetLastError();
}

cudaError_t launch_gather(const herald_dims& dm, const int32_t* idx, const int32_t* n_sel,
                          int P_max, const uint16_t* k_cache, const uint16_t* v_cache,
                          uint16_t* pool_k, uint16_t* pool_v, cudaStream_t st,
                          const char* name, int max_ctas) {
  return gather_launch(dm, idx, n_sel, P_max, k_cache, v_cache, pool_k, pool_v, nullptr, 0,
                       nullptr, nullptr, st, name, max_ctas);
}

cudaError_t launch_gather_staged(const herald_dims& dm, const int32_t* idx, const int32_t* n_sel,
                                 int P_max, const int32_t* src, int C, const uint16_t* staged_k,
                                 const uint16_t* staged_v, const uint16_t* k_cache,
                                 const uint16_t* v_cache, uint16_t* pool_k, uint16_t* pool_v,
                                 cudaStream_t st) {
  return gather_launch(dm, idx, n_sel, P_max, k_cache, v_cache, pool_k, pool_v, src, C, staged_k,
                       staged_v, st, "gather_kernel (staged)", 0);
}

// grid N, block 1024: one CTA per sequence so that reading ctx_len[n] and
// advancing it cannot race with another CTA.  Each thread moves up to
// kAppendBatch 16-byte chunks of K and of V per round, all loads first
// (1024 threads x 4: a block of 32 tokens x 8 KV heads x d = 128 is one round).
constexpr int kAppendBatch = 4;
constexpr int kAppendThreads = 1024;

__global__ void __launch_bounds__(kAppendThreads)
    append_kernel(const uint16_t* __restrict__ bk, const uint16_t* __restrict__ bv, int B,
                  int Hkv, int d, int L_max, int32_t* __restrict__ ctx,
                  uint16_t* __restrict__ kc, uint16_t* __restrict__ vc, int advance) {
  __shared__ int L0;
  griddep_enter();
  const int n = blockIdx.x;
  if (threadIdx.x == 0) {
    debug_flag(ctx[n] < 0 || ctx[n] > L_max, DEV_BAD_COUNT);
    L0 = min(max(ctx[n], 0), L_max);
  }
  __syncthreads();
  append_block_rows<kAppendBatch>(bk, bv, n, B, Hkv, d, L_max, L0, kc, vc, threadIdx.x,
                                  kAppendThreads);
  __syncthreads();
  if (advance && threadIdx.x == 0) ctx[n] = min(L0 + B, L_max);
}

cudaError_t launch_append(const herald_dims& dm, const uint16_t* block_k, const uint16_t* block_v,
                          int32_t* ctx, uint16_t* k_cache, uint16_t* v_cache, int advance,
                          cudaStream_t st) {
  HERALD_CHECK_LAUNCH(launch_k("append_kernel", append_kernel, dm.N, kAppendThreads, 0, st, block_k, block_v, dm.B, dm.Hkv, dm.d, dm.L_max, ctx,
                                      k_cache, v_cache, advance));
  return cudaGetLastError();
}

HERALD_DEBUG_WORD_READER(debug_take_move)

}  // namespace herald
