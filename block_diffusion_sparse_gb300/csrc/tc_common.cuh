// tc_common.cuh -- device helpers and the cluster launcher shared by the
// tensor-core translation units (tc_kernels.cu, attn_flash.cu).
#pragma once
#include "internal.cuh"
#include "ptx.cuh"

namespace herald {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// TMEM allocation protocol: warp 0 allocates, everybody syncs.
__device__ __forceinline__ void tmem_setup(uint32_t* slot, uint32_t ncols) {
  __syncwarp();
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}
__device__ __forceinline__ void tmem_teardown(uint32_t base, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 0) {
    tc_fence_after();
    tmem_dealloc(base, ncols);
  }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Stores to a shared::cluster address (another CTA's shared memory).
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f2(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y)
               : "memory");
}

constexpr int kTcThreads = 256;  // 8 warps: lane quadrant = warp % 4

// Copies `rows` rows of D bf16 (row r from src_of(r), or zeros when src_of
// returns nullptr) into a K-major 128B-swizzled tile: D/64 column halves,
// each [rows_alloc][128 bytes].  `any_src` is a valid global address used
// as the (unread) source of zero-filled chunks.  A warp copies 32/(D/8)
// whole rows per step (one 16-byte chunk per lane), so src_of runs once
// per lane and step, and the unrolled steps keep several rows in flight.
// Every thread of the (kTcThreads-thread) block must call it.
template <int D, int NT = kTcThreads, typename SrcOf>
__device__ __forceinline__ void load_rows_sw128(uint8_t* tile, int rows, int rows_alloc,
                                                const uint16_t* any_src, SrcOf src_of) {
  constexpr int CPR = D / 8;        // 16-byte chunks per row
  constexpr int RPW = 32 / CPR;     // rows per warp step
  constexpr int kStep = (NT / 32) * RPW;  // NT threads in the block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = lane % CPR, sub = lane / CPR;
  uint8_t* half = tile + (c >> 3) * (rows_alloc * 128);
#pragma unroll 4
  for (int r0 = warp * RPW; r0 < rows; r0 += kStep) {
    const int r = r0 + sub;
    if (r < rows) {
      const uint16_t* s = src_of(r);
      cp_async_16(half + sw128_off(r, c & 7), s ? s + c * 8 : any_src, s ? 16u : 0u);
    }
  }
}

// Full cluster barrier (hardware): release this CTA's shared-memory writes,
// acquire the peers'.
__device__ __forceinline__ void cluster_sync_all() {
  __cluster_barrier_arrive();
  __cluster_barrier_wait();
}
// shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_peer_f2(uint32_t a, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y)
               : "memory");
}

// Launches a kernel as clusters of cluster_x CTAs along x, with programmatic
// stream serialisation, bracketed by the tracing hooks.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_threads(const char* name, void (*kernel)(KArgs...), dim3 grid,
                                   dim3 block, int cluster_x, size_t smem, cudaStream_t st,
                                   Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (const cudaError_t ie = injected_launch_error()) return ie;
  trace_before(st, name);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  trace_after(st);
  return e;
}

}  // namespace herald
