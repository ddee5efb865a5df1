// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers with bounded
// waits, TMA bulk-tensor loads, cp.async, and the tcgen05 (5th-generation
// tensor core) instructions with their shared-memory / instruction
// descriptors.  Everything here is a direct statement of a documented PTX
// instruction; no vendor library code is involved.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define HERALD_DEV __device__ __forceinline__

namespace herald {

// Device-side error codes written to the workspace error word: the kind of
// wait in bits 0-7, the kernel that gave up in bits 8-15 (the first error
// recorded is kept).
enum : uint32_t {
  DEV_OK = 0,
  DEV_TIMEOUT_TMA = 1,   // a TMA / cp.async / bulk-copy completion wait ran out
  DEV_TIMEOUT_MMA = 2,   // a tcgen05 commit (or a pipeline stage) wait ran out
  DEV_K_REFINE_PASS1 = 1u << 8,
  DEV_K_REFINE_PASS2 = 2u << 8,
  DEV_K_REFINE_FUSED = 3u << 8,
  DEV_K_ATTN_SPLIT = 4u << 8,
  DEV_K_ATTN_CLUSTER = 5u << 8,
  DEV_K_ATTN_POOL = 6u << 8,
  DEV_K_SCAN = 7u << 8,
  DEV_K_ATTN_FLASH = 8u << 8,
};

// Checks of the debug build (compiled with -DHERALD_DEBUG): a kernel compares
// the indices and counts it reads or writes -- candidate and selected
// positions against the cache's rows or the context length, selection rows
// against P_max, context lengths against [0, L_max] -- with their ranges
// and sets a bit of its translation unit's debug word on a violation
// (herald_debug_status reads and clears them).  The access itself is
// skipped or clamped as in every build: a check never traps.  Release
// builds compile the checks out.
enum : uint32_t {
  DEV_BAD_INDEX = 0x10,  // a position outside the cache rows or the context
  DEV_BAD_COUNT = 0x20,  // a count or context length outside its range
};
#ifdef HERALD_DEBUG
static __device__ uint32_t g_debug_word;  // one per translation unit
#endif
HERALD_DEV void debug_flag(bool bad, uint32_t code) {
#ifdef HERALD_DEBUG
  if (bad) atomicOr(&g_debug_word, code);
#else
  (void)bad;
  (void)code;
#endif
}
// Defines the host function `fn` that returns and clears this translation
// unit's debug word (0 in release builds).  The caller synchronises first.
#ifdef HERALD_DEBUG
#define HERALD_DEBUG_WORD_READER(fn)                                     \
  uint32_t fn() {                                                        \
    uint32_t v = 0;                                                      \
    if (cudaMemcpyFromSymbol(&v, g_debug_word, sizeof v) != cudaSuccess) \
      return DEV_BAD_COUNT | DEV_BAD_INDEX;                              \
    const uint32_t z = 0;                                                \
    if (v) cudaMemcpyToSymbol(g_debug_word, &z, sizeof z);               \
    return v;                                                            \
  }
#else
#define HERALD_DEBUG_WORD_READER(fn) \
  uint32_t fn() { return 0; }
#endif

// ~1 s bound on any single wait (globaltimer is in ns).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

HERALD_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

HERALD_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier
HERALD_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
HERALD_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
HERALD_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
HERALD_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
HERALD_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete.  Gives up after
// about limit_ns (kWaitLimitNs by default) and returns false; the caller
// records the error.
HERALD_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while its predecessor on the stream is running;
// griddep_wait() blocks until the predecessor has completed and its memory
// is visible (a no-op for ordinary launches), so every kernel calls it before
// its first global memory access.  griddep_launch_dependents() lets the next
// kernel start its own prologue early.
HERALD_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
HERALD_DEV void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
HERALD_DEV void griddep_enter() {
  griddep_wait();
  griddep_launch_dependents();
}

HERALD_DEV void record_error(uint32_t* err_word, uint32_t code) {
  if (err_word) atomicCAS(err_word, 0u, code);
}

// ---------------------------------------------------------------- TMA loads
HERALD_DEV void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
HERALD_DEV void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

HERALD_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory to a
// shared::cluster address (another CTA of the cluster), completing as
// transaction bytes on the destination CTA's mbarrier (a shared::cluster
// address as well).
HERALD_DEV void bulk_copy_to_peer(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                  uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
      " [%0], [%1], %2, [%3];" ::"r"(dst_cluster),
      "r"(smem_u32(src)), "r"(bytes), "r"(mbar_cluster)
      : "memory");
}
HERALD_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk copy of this thread has read its source.
HERALD_DEV void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// shared::cluster address of the same shared-memory location in CTA `rank`.
HERALD_DEV uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// ------------------------------------------------------------------ cp.async
// 16-byte async copy global -> shared; src_bytes = 0 writes zeros.
HERALD_DEV void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
HERALD_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
HERALD_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor core / TMA reads of shared memory).
HERALD_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
// TMEM allocation: executed by one full warp; the base address is written to
// shared memory.  ncols is a power of two >= 32.
HERALD_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
HERALD_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
HERALD_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
HERALD_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
HERALD_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
HERALD_DEV void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x K, bf16) held in tensor memory --
// row i in lane i, two consecutive K elements per 32-bit column -- and B
// from a shared-memory descriptor; fp32 accumulator.
HERALD_DEV void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier when all previously issued tcgen05.mma of this
// thread have completed.
HERALD_DEV void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns per warp; thread i gets lane
// (base lane + i), columns [col, col+32).
HERALD_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive 32-bit columns per warp.
// Stores 32 consecutive columns of this thread's TMEM lane; the caller
// issues tmem_wait_st() before the columns are read again.
HERALD_DEV void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
      "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
      "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
HERALD_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

HERALD_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
//   [4,6) D format (1 = f32)  [7,10) A format (1 = bf16)  [10,13) B format
//   [15] A major (0 = K-major, 1 = MN-major)  [16] B major
//   [17,23) N >> 3            [24,29) M >> 4
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn_major,
                                                       bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
         (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   [0,14) start address >> 4   [16,30) leading byte offset >> 4
//   [32,46) stride byte offset >> 4   [46,48) = 1 (descriptor version)
//   [61,64) layout = 2 (SWIZZLE_128B)
// K-major tiles: rows of 128 bytes, 8-row groups SBO = 1024 bytes apart, LBO
// unused.  MN-major tiles: LBO = distance between 64-element MN blocks, SBO =
// distance between 8-row K groups.  The tile base must be 1024-byte aligned.
HERALD_DEV uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a 128B-swizzled
// block of 128-byte rows (the layout TMA SWIZZLE_128B writes).
HERALD_DEV uint32_t sw128_off(uint32_t r, uint32_t c) {
  return r * 128u + (((c ^ (r & 7u)) & 7u) << 4);
}

// ------------------------------------------------------------------- bf16
HERALD_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
HERALD_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

HERALD_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x with the hardware approximation (ex2.approx.ftz): 2^-inf = +0.
HERALD_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register, for the paired fp32 instructions
// (fma/add .f32x2): one issue slot for two values.
HERALD_DEV uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
HERALD_DEV void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
HERALD_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {  // a * b + c, one rounding
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
HERALD_DEV uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
HERALD_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
HERALD_DEV float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

HERALD_DEV uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

HERALD_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
HERALD_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace herald
