// attn_flash.cu -- sparse block attention (HERALD early abstract: the
// selected subset is reused for every denoising step; every block query
// sees the pool rows and all B block keys) as a pipelined kernel whose CTAs
// stream their keys through shared memory in tiles, so that a CTA may own
// any number of keys and a whole step runs in one wave of CTAs.
//
// One cluster of CS CTAs per (sequence, KV head, row tile of bpt whole
// tokens = bpt*G <= 128 query rows).  CTA r owns pool keys [r*kpc,
// (r+1)*kpc) below n_sel, the last CTA every pool key from its start on and
// the B block keys as one more tile; kpc is a whole number of tiles, as few
// as let every CTA hold the same number of tiles (the last one's block tile
// included).  Warp roles:
//   warps 0-15 softmax: thread = (query row, a quarter of the tile's
//              16-key chunks); S from TMEM, P (bf16) back into the same
//              TMEM columns
//   warp 16    TMA producer of the query tile and the K tiles (2-stage ring)
//   warp 17    TMA producer of the V tiles (2-stage ring)
//   warp 18    tcgen05.mma issuer: S_t = Q K_t^T into one of three TMEM
//              buffers, O += P_t V_t into the TMEM accumulator with P_t
//              read from TMEM (the A operand of the MMA)
// The MMA warp keeps S two tiles ahead of the softmax warps (three S/P
// buffers and O fill the 512 TMEM columns), so a softmax step waits for
// nothing but its scores unless its rows' exponent base moves, and S_{t+1}
// never waits for P_{t-1} V_{t-1}.  The softmax keeps one
// exponent base per row for as long as the row max rises by at most 8
// (log2 units: P <= 256); when it rises by more, O and the row sum are
// rescaled.  After the last tile each CTA normalises its O rows (fp16,
// divided by the row sum, staged over the dead K ring) and pushes row slice
// c to CTA c by bulk copies into receive buffers of their own, with the
// (max, sum) of the rows, completing on c's mbarrier; each CTA then merges
// its 128/CS rows, one 8-column chunk per thread, and writes bf16 out.
// The optional append of the block to the cache (the last denoising step)
// is done by the softmax warps of the first row tile's cluster of KV head
// 0, while the first loads are in flight.
#include <cuda_bf16.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace herald {

constexpr int kFT = kFlashTileKeys;         // keys per pipelined tile (MMA N, a multiple of 16)
constexpr int kFlashSoftWarps = 16;         // four per TMEM lane quadrant
constexpr int kFlashSplit = kFlashSoftWarps / 4;  // softmax warps sharing a row
constexpr int kFlashSoftThreads = kFlashSoftWarps * 32;
constexpr int kFlashKWarp = 16, kFlashVWarp = 17, kFlashMmaWarp = 18;
constexpr int kFlashThreads = 19 * 32;
constexpr float kFlashRebase = 8.f;         // log2 units
constexpr uint32_t kFlashTmemCols = 512;    // S/P buffers at 0, 128, 256; O at 384
constexpr int kSBufs = 3;                   // S/P buffers in TMEM
constexpr uint32_t kOCol = uint32_t(kSBufs * kFT);  // first TMEM column of O
static_assert(kOCol + 128 <= kFlashTmemCols, "S/P buffers and O fit TMEM");
constexpr int kFlashMaxB = 64;              // block keys: one tile, the box of the block maps

struct FlashSmem {
  uint32_t q, k, v, recv_o, recv_ml, total;
};
// Dynamic shared memory of the kernel for head dimension D: the query tile,
// the K and V rings (two stages of kFT rows each), and the receive buffers
// of the row merge (written by the peers' bulk copies).
__host__ __device__ inline FlashSmem flash_smem(int D) {
  const uint32_t H = uint32_t(D / 64), stage = H * uint32_t(kFT) * 128u;
  FlashSmem L;
  L.q = 0;
  L.k = H * 16384u;
  L.v = L.k + 2u * stage;
  L.recv_o = L.v + 2u * stage;
  L.recv_ml = L.recv_o + uint32_t(kTileM) * uint32_t(D + 8) * 2u;
  L.total = L.recv_ml + uint32_t(kTileM) * 8u + 1024u;  // + alignment slack
  return L;
}

__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFlashSoftThreads) : "memory");
}

template <int D, int CS>
__global__ void __launch_bounds__(kFlashThreads, 1)
    attn_flash_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap bkmap,
                      const __grid_constant__ CUtensorMap bvmap,
                      const int32_t* __restrict__ n_sel, int P_max, int B, int Hq, int Hkv,
                      int bpt, int kpc, float scale, int settled, uint16_t* __restrict__ out,
                      uint32_t* err, AppendArgs app, int L_max) {
  constexpr int H = D / 64;
  constexpr int OROW = D + 8;        // fp16 row stride of the pushed O rows
  constexpr int RC = kTileM / CS;    // rows merged per CTA
  constexpr uint32_t kStage = uint32_t(H * kFT * 128);
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t barQ, kfull[2], kempty[2], vfull[2], vempty[2];
  __shared__ uint64_t sfull[kSBufs], pfull[kSBufs], pvdone[kSBufs], alldone, barR;
  __shared__ uint32_t tmem_base;
  __shared__ float red_m[2][kFlashSplit][kTileM];  // [tile parity][column share][row]
  __shared__ float red_s[kFlashSplit][kTileM];
  __shared__ __align__(16) float2 ml[kTileM];
  constexpr uint32_t kSliceO = uint32_t(RC * OROW * 2);
  constexpr uint32_t kSliceMl = uint32_t(RC * 8);
  const FlashSmem S = flash_smem(D);
  uint8_t* base = align1024(smem_raw);
  uint8_t* Qs = base + S.q;
  uint8_t* Kr = base + S.k;
  uint8_t* Vr = base + S.v;
  uint16_t* recv_o = reinterpret_cast<uint16_t*>(base + S.recv_o);
  float2* recv_ml = reinterpret_cast<float2*>(base + S.recv_ml);
  const uint32_t rank = cluster_ctarank();
  const int mt = blockIdx.y, seg = blockIdx.z;
  const int n = seg / Hkv, g = seg - n * Hkv, G = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Bp = (B + 15) & ~15;
  if (threadIdx.x == 0) {
    mbar_init(&barQ, 1);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
#pragma unroll
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&sfull[b], 1);
      mbar_init(&pfull[b], kFlashSoftThreads);
      mbar_init(&pvdone[b], 1);
    }
    mbar_init(&alldone, 1);
    mbar_init(&barR, 1);
    mbar_arrive_expect_tx(&barR, uint32_t(CS) * (kSliceO + kSliceMl));
    fence_mbar_init();
  }
  // peers' pushes complete on barR: its initialisation is published
  // cluster-wide here and awaited just before the pushes are issued
  __cluster_barrier_arrive_relaxed();
  if (threadIdx.x == 0) {  // kernel parameters: independent of the predecessor
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&bkmap);
    tma_prefetch_desc(&bvmap);
  }
  tmem_setup(&tmem_base, kFlashTmemCols);
  const uint32_t tbase = tmem_base;
  const int k0 = int(rank) * kpc;
  // settled != 0: the pool and n_sel were written before the previous
  // launch on the stream began (that launch waited for its own predecessor
  // before starting this one), so the producers fetch the first pool tiles
  // while the predecessor finishes
  // pool keys [k0, k_hi) of this CTA: the last CTA takes the rest
  const int k_hi = int(rank) == CS - 1 ? P_max : min(P_max, k0 + kpc);
  // Only the first K tile goes before the wait: every CTA of the grid loads
  // at once at the start, and the query tile and the first K tile are what
  // S_0 needs; the other tiles follow once the first one has landed.
  int pre = 0;  // pool K tiles loaded before the grid-dependency wait
  if (settled && warp == kFlashKWarp && lane == 0) {
    const int nkp0 = max(min(max(n_sel[seg], 0), k_hi) - k0, 0);
    pre = min((nkp0 + kFT - 1) / kFT, 1);
    if (pre) {
      mbar_arrive_expect_tx(&kfull[0], kStage);
#pragma unroll
      for (int hv = 0; hv < H; ++hv)
        tma_load_2d(Kr + hv * kFT * 128, &kmap, &kfull[0], hv * 64, seg * P_max + k0);
    }
  }
  griddep_enter();

  // this CTA's keys: npt pool tiles of up to kFT keys, then (the last CTA)
  // one tile of the B block keys
  const int b0 = mt * bpt;                  // first token of the row tile
  const int rows_t = min(bpt, B - b0) * G;  // query rows of the tile
  const int ns_raw = n_sel[seg];
  debug_flag(threadIdx.x == 0 && (ns_raw < 0 || ns_raw > P_max), DEV_BAD_COUNT);
  const int nkp = max(min(max(ns_raw, 0), k_hi) - k0, 0);
  const int npt = (nkp + kFT - 1) / kFT;
  const bool has_blk = int(rank) == CS - 1 && B > 0;
  const int nt = npt + (has_blk ? 1 : 0);
  auto tile_keys = [&](int t) { return t < npt ? min(kFT, nkp - t * kFT) : B; };
  // waits that ran out (bits 16-26 of the error word): 0x1 K ring slot,
  // 0x2 V ring slot, 0x4 query tile, 0x8 K tile, 0x10 S buffer free, 0x20 P
  // ready, 0x40 V tile, 0x80 S ready, 0x100 O up to date for a rescale,
  // 0x200 every MMA done, 0x400 the peers' partials, 0x800 the previous
  // tile's P V done
  uint32_t bad = 0;

  if (warp == kFlashKWarp) {
    // ------------------------------------------------ query tile + K tiles
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(&barQ, uint32_t(H * G * bpt * 128));
#pragma unroll
      for (int hv = 0; hv < H; ++hv)
        tma_load_3d(Qs + hv * kTileM * 128, &qmap, &barQ, hv * 64, g * G, n * B + b0);
      for (int t = pre; t < nt; ++t) {
        const int s = t & 1;
        if (t == 1 && !mbar_wait(&kfull[0], 0)) bad |= 1u;  // the first tile has landed
        if (t >= 2 && !mbar_wait(&kempty[s], ((t >> 1) - 1) & 1)) bad |= 1u;
        uint8_t* dst = Kr + s * kStage;
        if (t < npt) {
          mbar_arrive_expect_tx(&kfull[s], kStage);
#pragma unroll
          for (int hv = 0; hv < H; ++hv)
            tma_load_2d(dst + hv * kFT * 128, &kmap, &kfull[s], hv * 64,
                        seg * P_max + k0 + t * kFT);
        } else {
          mbar_arrive_expect_tx(&kfull[s], uint32_t(H * Bp * 128));
#pragma unroll
          for (int hv = 0; hv < H; ++hv)
            tma_load_3d(dst + hv * kFT * 128, &bkmap, &kfull[s], hv * 64, g, n * B);
        }
      }
    }
  } else if (warp == kFlashVWarp) {
    // ---------------------------------------------------------- V tiles
    if (lane == 0) {
      // V_0 is needed after the first softmax step: after the query tile
      // (issued with the first K tile; a single-use barrier)
      if (nt > 0 && !mbar_wait(&barQ, 0)) bad |= 2u;
      for (int t = 0; t < nt; ++t) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait(&vempty[s], ((t >> 1) - 1) & 1)) bad |= 2u;
        uint8_t* dst = Vr + s * kStage;
        if (t < npt) {
          mbar_arrive_expect_tx(&vfull[s], kStage);
#pragma unroll
          for (int hv = 0; hv < H; ++hv)
            tma_load_2d(dst + hv * kFT * 128, &vmap, &vfull[s], hv * 64,
                        seg * P_max + k0 + t * kFT);
        } else {
          mbar_arrive_expect_tx(&vfull[s], uint32_t(H * Bp * 128));
#pragma unroll
          for (int hv = 0; hv < H; ++hv)
            tma_load_3d(dst + hv * kFT * 128, &bvmap, &vfull[s], hv * 64, g, n * B);
        }
      }
    }
  } else if (warp == kFlashMmaWarp) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      if (!mbar_wait(&barQ, 0)) bad |= 0x4u;
      const uint32_t qa = smem_u32(Qs);
      // S_j = Q K_j^T into TMEM buffer j % 3: issued once K_j has landed and
      // the buffer's previous P (tile j - 3) has been read by its P V
      auto issue_s = [&](int j) {
        const int s = j & 1, b3 = j % kSBufs;
        if (!mbar_wait(&kfull[s], (j >> 1) & 1)) bad |= 0x8u;
        if (j >= kSBufs && !mbar_wait(&pvdone[b3], (j / kSBufs - 1) & 1)) bad |= 0x10u;
        tc_fence_after();
        const int nk = (tile_keys(j) + 15) & ~15;
        const uint32_t idesc = make_idesc_bf16(kTileM, nk, false, false);
        const uint32_t ka = smem_u32(Kr + s * kStage);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t hv = uint32_t(ks) >> 2, koff = uint32_t(ks & 3) * 32u;
          const uint64_t a = make_sdesc_sw128(qa + hv * (kTileM * 128) + koff, 16, 1024);
          const uint64_t b = make_sdesc_sw128(ka + hv * (kFT * 128) + koff, 16, 1024);
          umma_bf16(tbase + uint32_t(b3) * uint32_t(kFT), a, b, idesc, ks > 0 ? 1u : 0u);
        }
        umma_commit(&sfull[b3]);
        umma_commit(&kempty[s]);
      };
      // two tiles ahead of the softmax; then per tile u: O += P_u V_u once
      // P_u is in TMEM, and S_{u+2} into the buffer P_{u-1} V_{u-1} freed
      issue_s(0);
      if (nt > 1) issue_s(1);
      for (int u = 0; u < nt; ++u) {
        const int su = u & 1, bu = u % kSBufs;
        if (!mbar_wait(&pfull[bu], (u / kSBufs) & 1)) bad |= 0x20u;
        if (!mbar_wait(&vfull[su], (u >> 1) & 1)) bad |= 0x40u;
        tc_fence_after();
        const int nk = (tile_keys(u) + 15) & ~15;
        constexpr uint32_t idesc = make_idesc_bf16(kTileM, D, false, true);
        const uint32_t va = smem_u32(Vr + su * kStage);
        for (int ks = 0; ks < nk / 16; ++ks) {  // P: 16 keys = 8 packed TMEM columns
          const uint64_t b =
              make_sdesc_sw128(va + uint32_t(ks) * 2048u, uint32_t(kFT) * 128u, 1024);
          umma_bf16_ts(tbase + kOCol, tbase + uint32_t(bu * kFT + ks * 8), b, idesc,
                       (u > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&pvdone[bu]);
        umma_commit(&vempty[su]);
        if (u + 2 < nt) issue_s(u + 2);
      }
      umma_commit(&alldone);  // (single use: the softmax warps may lag pvdone)
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3, ch = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t trow = tbase + (uint32_t(quad * 32) << 16);
    const float sl2 = scale * 1.4426950408889634f;  // scores -> log2 units
    // the fused append: the softmax warps of the first row tile's cluster
    // of KV head 0 copy the block's rows of every KV head into the cache
    // while the first tiles load; no other CTA reads ctx, and CTA 0 of the
    // cluster advances it once every peer has pushed its partial
    if (app.bk != nullptr && mt == 0 && g == 0) {
      debug_flag(threadIdx.x == 0 && (app.ctx[n] < 0 || app.ctx[n] > L_max), DEV_BAD_COUNT);
      const int L0 = min(max(app.ctx[n], 0), L_max);
      append_block_rows<1>(app.bk, app.bv, n, B, Hkv, D, L_max, L0, app.kc, app.vc,
                           int(rank) * kFlashSoftThreads + threadIdx.x, CS * kFlashSoftThreads);
    }
    float m_base = -INFINITY;  // the row's exponent base (log2 units)
    float l = 0.f;             // this thread's share of the row sum
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1, b3 = t % kSBufs;
      const int nk = tile_keys(t);
      const int nchunks = (nk + 15) >> 4;
      const int per = (nchunks + kFlashSplit - 1) / kFlashSplit;
      const int c_begin = min(ch * per, nchunks), cnt = min(per, nchunks - c_begin);
      if (!mbar_wait(&sfull[b3], (t / kSBufs) & 1)) bad |= 0x80u;
      tc_fence_after();
      constexpr int kMaxChunks = (kFT / 16 + kFlashSplit - 1) / kFlashSplit;
      float x[kMaxChunks][16];
#pragma unroll
      for (int c = 0; c < kMaxChunks; ++c) {
        if (c < cnt) {
          uint32_t* r = reinterpret_cast<uint32_t*>(x[c]);
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
              "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
              : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
              : "r"(trow + uint32_t(b3 * kFT + (c_begin + c) * 16)));
        }
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      // the tile's row max of the raw scores, keys past the valid ones at
      // -inf in the one partial chunk
      float m = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMaxChunks; ++c) {
        if (c < cnt) {
          const int nv = min(nk - (c_begin + c) * 16, 16);
          if (nv < 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[c][i] = i < nv ? x[c][i] : -INFINITY;
          }
#pragma unroll
          for (int i = 0; i < 16; i += 2) m = fmax3f(m, x[c][i], x[c][i + 1]);
        }
      }
      red_m[s][ch][row] = m;
      softmax_bar();
#pragma unroll
      for (int k = 0; k < kFlashSplit; ++k) m = fmaxf(m, red_m[s][k][row]);
      const float mt_ = m * sl2;
      // a new base only when the max rises by more than kFlashRebase
      const bool rebase = m_base == -INFINITY || mt_ > m_base + kFlashRebase;
      float factor = 1.f;
      if (rebase) {
        factor = m_base == -INFINITY ? 0.f : fast_exp2(m_base - mt_);
        m_base = mt_;
      }
      // a new base rescales O, once P_{t-1} V_{t-1} has been added to it
      if (t >= 1 && __any_sync(0xffffffffu, rebase)) {
        // P_{t-1} V_{t-1} (in-order after every earlier P V) completes on
        // pvdone[(t-1) % 3], whose next completion needs this thread's P_{t+2}
        if (!mbar_wait(&pvdone[(t - 1) % kSBufs], ((t - 1) / kSBufs) & 1)) bad |= 0x100u;
        tc_fence_after();
        {  // this thread's share of its O row
#pragma unroll
          for (int k = 0; k < D / (16 * kFlashSplit); ++k) {
            float v[16];
            const uint32_t col = kOCol + uint32_t(ch * (D / kFlashSplit) + k * 16);
            tmem_ld16(trow + col, v);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i] * factor);
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(
                    trow + col),
                "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]),
                "r"(w[14]), "r"(w[15])
                : "memory");
          }
          tmem_wait_st();
        }
      }
      // P = 2^(x sl2 - base): the scaling and the shift as one paired fma
      // for two keys, the row sum as paired adds; P (bf16 pairs) goes over
      // this tile's scores in TMEM, which both column halves have read
      // (the max exchange above follows every load)
      const float mm = m_base == -INFINITY ? 0.f : m_base;
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
          asm volatile(
              "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::
                  "r"(trow + uint32_t(b3 * kFT + (c_begin + c) * 8)),
              "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]),
              "r"(pk[6]), "r"(pk[7])
              : "memory");
        }
      }
      float lsum, lsum_hi;
      f2_unpack(lsum2, lsum, lsum_hi);
      l = l * factor + (lsum + lsum_hi);
      tmem_wait_st();
      // pfull[t % 3] cannot run two phases ahead of the MMA warp: its next
      // arrival (P_{t+3}) needs S_{t+3}, which the MMA warp issues only after
      // P_t V_t, i.e. after consuming this phase
      tc_fence_before();
      mbar_arrive(&pfull[b3]);
    }
    if (nt > 0) {  // every MMA of this CTA is done
      if (!mbar_wait(&alldone, 0)) bad |= 0x200u;
      tc_fence_after();
    }
    red_s[ch][row] = l;
    softmax_bar();
    float lrow = 0.f;
#pragma unroll
    for (int k = 0; k < kFlashSplit; ++k) lrow += red_s[k][row];
    // O / l as fp16 rows over the K ring (dead: every MMA is done): every
    // TMEM load issued, one wait, then the shared-memory stores
    constexpr int kW = D / kFlashSplit;  // O columns per thread
    uint16_t* orow = reinterpret_cast<uint16_t*>(Kr) + row * OROW + ch * kW;
    if (nt > 0) {
      const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
      uint32_t r[kW];
#pragma unroll
      for (int k = 0; k < kW / 16; ++k) {
        uint32_t* q = r + k * 16;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]),
              "=r"(q[6]), "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]),
              "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
            : "r"(trow + kOCol + uint32_t(ch * kW + k * 16)));
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int i = 0; i < kW; i += 8) {
        const float* v = reinterpret_cast<const float*>(r + i);
        *reinterpret_cast<uint4*>(orow + i) =
            make_uint4(pack_half2(v[0] * inv, v[1] * inv), pack_half2(v[2] * inv, v[3] * inv),
                       pack_half2(v[4] * inv, v[5] * inv), pack_half2(v[6] * inv, v[7] * inv));
      }
    }
    if (ch == 0) ml[row] = make_float2(nt > 0 ? m_base : -INFINITY, nt > 0 ? lrow : 0.f);
    fence_proxy_async_smem();  // the partial is read by bulk copies (async proxy)
  }
  __syncthreads();
  __cluster_barrier_wait();  // every peer's barR is initialised

  // push: rows [c*RC, c*RC + RC) of this CTA's partial go to CTA c, slot `rank`
  if (threadIdx.x == 0) {
    const uint16_t* Os = reinterpret_cast<const uint16_t*>(Kr);
    for (uint32_t c = 0; c < uint32_t(CS); ++c) {
      const uint32_t mb = cluster_addr(&barR, c);
      bulk_copy_to_peer(cluster_addr(reinterpret_cast<uint8_t*>(recv_o) + rank * kSliceO, c),
                        Os + c * RC * OROW, kSliceO, mb);
      bulk_copy_to_peer(cluster_addr(reinterpret_cast<uint8_t*>(recv_ml) + rank * kSliceMl, c),
                        &ml[c * RC], kSliceMl, mb);
    }
    bulk_commit();
  }
  if (!mbar_wait(&barR, 0)) {
    record_error(err, DEV_TIMEOUT_TMA | DEV_K_ATTN_FLASH | (0x400u << 16));
    // a peer whose own wait ran out pushes late: this CTA must not exit
    // (its shared memory is the copies' destination) before they land
    mbar_wait(&barR, 0, 20ull * kWaitLimitNs);
  } else if (app.bk != nullptr && app.advance && mt == 0 && g == 0 && rank == 0 &&
             threadIdx.x == 0) {
    app.ctx[n] = min(min(max(app.ctx[n], 0), L_max) + B, L_max);
  }

  // merge this CTA's RC rows from the CS received partials, one 8-column
  // chunk of one row per thread and pass (every load of a chunk independent):
  // out = sum_c 2^(m_c - M) l_c (o_c / l_c) / sum_c 2^(m_c - M) l_c
  constexpr int kChunks = D / 8;
  for (int item = threadIdx.x; item < RC * kChunks; item += kFlashThreads) {
    const int rr = item / kChunks, cj = item - rr * kChunks;
    const int lr = int(rank) * RC + rr;
    if (lr >= rows_t) continue;  // rows past the tile's tokens
    float2 pm[CS];
    uint4 ov[CS];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      pm[c] = recv_ml[c * RC + rr];
      ov[c] = *reinterpret_cast<const uint4*>(recv_o + (c * RC + rr) * OROW + cj * 8);
      M = fmaxf(M, pm[c].x);
    }
    float acc[8] = {};
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < CS; ++c) {
      // a CTA without keys pushed no values (its slot holds whatever the
      // buffer held): skip it, never weight it by zero
      if (pm[c].x == -INFINITY || !(pm[c].y > 0.f)) continue;
      const float wgt = fast_exp2(pm[c].x - M) * pm[c].y;
      L += wgt;
      const __half2* h = reinterpret_cast<const __half2*>(&ov[c]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(h[e]);
        acc[2 * e] += wgt * f.x;
        acc[2 * e + 1] += wgt * f.y;
      }
    }
    const int grow = b0 * G + lr;
    const int b = grow / G, h = g * G + (grow - b * G);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<uint4*>(out + ((size_t(n) * B + b) * Hq + h) * D + cj * 8) =
        make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                   pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
  }
  if (bad) record_error(err, DEV_TIMEOUT_MMA | DEV_K_ATTN_FLASH | (bad << 16));
  // Once barR has completed, every peer's copy into this CTA has landed and
  // nothing else reaches its shared memory: it leaves as soon as its own
  // outgoing copies have read the partial, without waiting for its peers
  // (no cluster barrier at the end of the chain).
  if (threadIdx.x == 0) bulk_wait_read_all();
  tmem_teardown(tbase, kFlashTmemCols);
}

// ------------------------------------------------------------------- host

// How many clusters of CS CTAs of the kernel can be resident at once on
// the current device; cached per (device, D, CS).
template <int D, int CS>
static int flash_resident_clusters() {
  constexpr int kDevs = 64;
  static int cache[kDevs];  // 0: not asked yet (zero-initialised); -1: none fit
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 0;
  int n = cache[dev];
  if (n == 0) {
    const size_t smem = flash_smem(D).total;
    if (ensure_smem(attn_flash_kernel<D, CS>, smem) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(CS, 1, 1);
    cfg.blockDim = dim3(kFlashThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, attn_flash_kernel<D, CS>, &cfg) != cudaSuccess ||
        n < 1)
      n = -1;
    cudaGetLastError();
    cache[dev] = n;
  }
  return n > 0 ? n : 0;
}

// Pool keys of each CTA but the last: whole tiles, as few as let every CTA
// hold the same number of tiles with the last one's block tile counted.
int attn_flash_kpc(int P_max, int CS) { return cdiv(cdiv(P_max, kFT) + 1, CS) * kFT; }

bool attn_flash_ok(const herald_dims& dm) {
  return ((dm.B + 15) & ~15) <= kFlashMaxB && flash_smem(dm.d).total <= 224u * 1024u;
}

// The cluster size for `units` clusters: the largest of 8, 4, 2 CTAs per
// unit whose clusters are all resident at once (one wave); 2 if none.
template <int D>
static int flash_pick_cs(int units, int sm_budget) {
  const int cap = sm_budget > 0 ? sm_budget : 1 << 30;
  if (units * 8 <= cap && units <= flash_resident_clusters<D, 8>()) return 8;
  if (units * 4 <= cap && units <= flash_resident_clusters<D, 4>()) return 4;
  return 2;
}

template <int D, int CS>
static cudaError_t launch_flash_cs(const herald_dims& dm, const int32_t* n_sel, int P_max,
                                   uint16_t* out, float scale, uint32_t* err,
                                   const PoolMaps& maps, const AppendArgs& app, bool settled,
                                   cudaStream_t st) {
  const uint32_t smem = flash_smem(D).total;
  HERALD_CHECK_LAUNCH(ensure_smem(attn_flash_kernel<D, CS>, smem));
  const int segs = dm.N * dm.Hkv;
  const int tiles = cdiv(dm.B, maps.bpt);
  return launch_cluster_threads("attn_flash_kernel", attn_flash_kernel<D, CS>,
                                dim3(CS, tiles, segs), dim3(kFlashThreads), CS, smem, st,
                                maps.kt, maps.vt, maps.q, maps.bk, maps.bv, n_sel, P_max, dm.B,
                                dm.Hq, dm.Hkv, maps.bpt, attn_flash_kpc(P_max, CS), scale,
                                settled ? 1 : 0, out, err, app, dm.L_max);
}

template <int D>
static cudaError_t launch_flash_t(const herald_dims& dm, const int32_t* n_sel, int P_max,
                                  uint16_t* out, float scale, uint32_t* err,
                                  const PoolMaps& maps, const AppendArgs& app, int cs,
                                  bool settled, cudaStream_t st) {
  if (cs == 0) cs = flash_pick_cs<D>(cdiv(dm.B, maps.bpt) * dm.N * dm.Hkv, maps.sm_budget);
  switch (cs) {
    case 8:
      return launch_flash_cs<D, 8>(dm, n_sel, P_max, out, scale, err, maps, app, settled, st);
    case 4:
      return launch_flash_cs<D, 4>(dm, n_sel, P_max, out, scale, err, maps, app, settled, st);
    case 2:
      return launch_flash_cs<D, 2>(dm, n_sel, P_max, out, scale, err, maps, app, settled, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_flash(const herald_dims& dm, const int32_t* n_sel, int P_max,
                              uint16_t* out, float scale, uint32_t* err, const PoolMaps& maps,
                              const AppendArgs* app, int cs, bool settled, cudaStream_t st) {
  const AppendArgs none{nullptr, nullptr, nullptr, nullptr, nullptr, 0};
  const AppendArgs& a = app ? *app : none;
  if (dm.d == 128)
    return launch_flash_t<128>(dm, n_sel, P_max, out, scale, err, maps, a, cs, settled, st);
  return launch_flash_t<64>(dm, n_sel, P_max, out, scale, err, maps, a, cs, settled, st);
}

int attn_flash_units_resident(const herald_dims& dm, int units) {
  return dm.d == 128 ? flash_pick_cs<128>(units, 0) : flash_pick_cs<64>(units, 0);
}

HERALD_DEBUG_WORD_READER(debug_take_flash)

}  // namespace herald
