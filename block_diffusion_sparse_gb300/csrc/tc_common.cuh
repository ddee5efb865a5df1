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
