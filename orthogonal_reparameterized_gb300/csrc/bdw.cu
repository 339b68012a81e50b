// Fused backward of a block-diagonal product: the product and its weight gradient from one
// pass over the upstream gradient (POET-X summary page, "Core method" section 3: the
// block-diagonal products; their backward by the chain rule):
//   Y   = T blkdiag(G)^T                 dB = dz~ G_P^T   or   dx~ = dA G_R^T
//   dG  = S_j^T T_j per block j          dG_P = B^T dz~   or   dG_R = x~^T dA
// with dG summed over the tokens of each split into fp32 partials [splits, nblk, b, b].
// Done separately, the two read T twice from HBM and pay two launch ramps; here each
// 128-token tile of T is read once and feeds both products.
//
// One work unit is (block j, token split s, half h of the block's 128-wide column halves,
// b = 128 or 256).  Its CTA streams the split's token tiles:
//   warp 0      TMA: per tile, the b/64 sub-tiles [128 tokens x 64 features] of T as one 3-D
//               box into one of the 8 / (b/64) slots of a 128 KB ring, and the half's two S
//               sub-tiles as one box into one of two S slots (a single thread issuing tiled
//               copies moves ~50 GB/s into its SM with 16 KB boxes, ~75 with 64 KB boxes)
//   warp 1      MMA issuer, per tile:
//                 dG_h (+)= S_h^T T        M = 128 (S features), N = b, K = 128 tokens;
//                                          both operands MN-major straight from the tiles
//                 Y_h^T   = G_h T^T        M = 128 (Y columns), N = 128 tokens, K = b;
//                                          A = the half's rows of G, resident in TMEM
//                                          (loaded once per unit), B = the T sub-tiles
//                                          read K-major
//   warps 2-9   epilogue: Y_h^T from TMEM (lane = column, so the int8 column scale is one
//               per-thread factor) through a [32 tokens x 32 columns] shared-memory box
//               stored by TMA; at the end of the unit the dG_h partial, likewise
// TMEM: G_h at columns [0, b/2), the Y accumulator [128, 256), dG_h [256, 256 + b).  The
// two halves of a (block, split) are adjacent units, so they run at the same time and the
// second read of each T tile is served by L2.  Every mbarrier wait is bounded; on expiry
// the kernel records POETX_ERR_TIMEOUT, lets its copies and MMAs finish, frees TMEM and
// returns.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace poetx {

// Site id of this file's bounded waits (file id x 10000 + source line).
constexpr int kSite = 5 * 10000;

namespace {

constexpr int BDW_TOK = 128;                          // tokens per tile
constexpr int BDW_T_STAGES = 8;                       // T ring in sub-tiles (a multiple of b / 64)
constexpr uint32_t BDW_SUB = 128 * 64 * 2;            // one sub-tile: 16 KB
constexpr uint32_t BDW_S_SLOT = 2 * BDW_SUB;          // the half's 128 features of S
constexpr int BDW_EPIW = 8;
constexpr int BDW_THREADS = 64 + 32 * BDW_EPIW;
constexpr uint32_t BDW_STG = 4096;                    // per epilogue warp: two Y boxes or one dG box
constexpr uint32_t BDW_S_OFF = BDW_T_STAGES * BDW_SUB;
constexpr uint32_t BDW_STG_OFF = BDW_S_OFF + 2 * BDW_S_SLOT;
constexpr uint32_t BDW_BAR_OFF = BDW_STG_OFF + BDW_EPIW * BDW_STG;
constexpr int BDW_SMEM = BDW_BAR_OFF + 256 + 1024;    // + barriers + alignment slack
static_assert(BDW_SMEM <= 227 * 1024, "fused block-diagonal backward: shared memory");
constexpr uint32_t G_COL = 0, Y_COL = 128, DG_COL = 256;

// Load a 3-D box into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

struct BdwParams {
  int b, halves, nblk, splits, chunk_tiles, ntiles, num_units;
  const __nv_bfloat16* G;    // [nblk, b, b]
  const float* colscale;     // nullable: Y column c (of all nblk * b) times colscale[c]
  unsigned long long* trace;
  size_t trace_cap;
  int* err;
  unsigned long long limit_ns;
};

struct BdwUnit {
  int j, s, h, t0, nt;  // block, split, half, first token tile, token tiles
};

__device__ __forceinline__ BdwUnit unit_of(const BdwParams& p, int u) {
  BdwUnit w;
  w.h = u % p.halves;
  const int r = u / p.halves;
  w.s = r % p.splits;
  w.j = r / p.splits;
  w.t0 = w.s * p.chunk_tiles;
  const int e = w.t0 + p.chunk_tiles < p.ntiles ? w.t0 + p.chunk_tiles : p.ntiles;
  w.nt = e > w.t0 ? e - w.t0 : 0;
  return w;
}

__global__ void __launch_bounds__(BDW_THREADS, 1)
    bdw_kernel(const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmS,
               const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmD,
               const BdwParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BDW_BAR_OFF);
  uint64_t* tfull = bars;                   // [8 / TS] T tile slot landed
  uint64_t* tempty = bars + 8;              // [8 / TS] T tile slot read by its MMAs
  uint64_t* sfull = bars + 16;              // [2]
  uint64_t* sempty = bars + 18;             // [2]
  uint64_t* yfull = bars + 20;              // Y accumulator holds a tile
  uint64_t* yempty = bars + 21;             // Y accumulator drained (epilogue warps)
  uint64_t* dgfull = bars + 22;             // dG accumulator holds the unit's partial
  uint64_t* dgempty = bars + 23;            // dG accumulator drained (epilogue warps)
  uint64_t* gfull = bars + 24;              // the unit's G rows are in TMEM (epilogue warps)
  uint64_t* gfree = bars + 25;              // the unit's last MMA reading G has completed
  uint64_t* mdone = bars + 26;              // every MMA of the CTA has completed (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 27);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int TS = p.b / 64;  // T sub-tiles per token tile
  const int NSLOT = BDW_T_STAGES / TS;  // T tile slots
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 0);
  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < BDW_T_STAGES; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 1);
    }
    mbar_init(yfull, 1);
    mbar_init(yempty, BDW_EPIW);
    mbar_init(dgfull, 1);
    mbar_init(dgempty, BDW_EPIW);
    mbar_init(gfull, BDW_EPIW);
    mbar_init(gfree, 1);
    mbar_init(mdone, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmT);
    tma_prefetch_desc(&tmS);
    tma_prefetch_desc(&tmY);
    tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);
  pdl_wait();  // the previous kernel's outputs are visible from here on
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 1);

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    long long gt = 0;  // token tiles issued
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
      const BdwUnit w = unit_of(p, u);
      for (int i = 0; i < w.nt; ++i, ++gt) {
        const int row = (w.t0 + i) * BDW_TOK;
        const int slot = (int)(gt & 1);
        const int ts = (int)(gt % NSLOT);
        if (*abort_flag ||
            !mbar_wait_bounded(&sempty[slot], (uint32_t)(((gt >> 1) & 1) ^ 1), p.err, p.limit_ns,
                               kSite + __LINE__) ||
            !mbar_wait_bounded(&tempty[ts], (uint32_t)(((gt / NSLOT) & 1) ^ 1), p.err,
                               p.limit_ns, kSite + __LINE__)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        if (gt == 0) trace_stamp(p.trace, p.trace_cap, 2);  // slot 2: first load issued
        // S: the half's 128 features (2 groups of 64); T: the block's b / 64 groups
        mbar_arrive_expect_tx(&sfull[slot], BDW_S_SLOT);
        tma_load_3d(smem + BDW_S_OFF + slot * BDW_S_SLOT, &tmS, &sfull[slot], 0, row,
                    w.j * TS + 2 * w.h);
        mbar_arrive_expect_tx(&tfull[ts], (uint32_t)TS * BDW_SUB);
        tma_load_3d(smem + (size_t)ts * TS * BDW_SUB, &tmT, &tfull[ts], 0, row, w.j * TS);
      }
    }
    // Loads still landing (only after an abort) must complete before the CTA exits: wait for
    // the last load issued into every slot.
    for (long long g = gt - 1; g >= 0 && g >= gt - NSLOT; --g)
      mbar_wait_bounded(&tfull[g % NSLOT], (uint32_t)((g / NSLOT) & 1), p.err, p.limit_ns,
                        kSite + __LINE__);
    for (long long g = gt - 1; g >= 0 && g >= gt - 2; --g)
      mbar_wait_bounded(&sfull[g & 1], (uint32_t)((g >> 1) & 1), p.err, p.limit_ns,
                        kSite + __LINE__);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t idesc_dg = make_idesc(128, p.b, true, true);
    const uint32_t idesc_y = make_idesc(128, BDW_TOK, false, false);
    long long gt = 0;
    int un = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++un) {
      const BdwUnit w = unit_of(p, u);
      if (*abort_flag ||
          !mbar_wait_bounded(gfull, (uint32_t)(un & 1), p.err, p.limit_ns, kSite + __LINE__) ||
          !mbar_wait_bounded(dgempty, (uint32_t)((un & 1) ^ 1), p.err, p.limit_ns,
                             kSite + __LINE__)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      for (int i = 0; i < w.nt; ++i, ++gt) {
        const int slot = (int)(gt & 1);
        bool got = !*abort_flag && mbar_wait_bounded(&sfull[slot], (uint32_t)((gt >> 1) & 1),
                                                     p.err, p.limit_ns, kSite + __LINE__);
        got = got && mbar_wait_bounded(&tfull[gt % NSLOT], (uint32_t)((gt / NSLOT) & 1), p.err,
                                       p.limit_ns, kSite + __LINE__);
        if (!got) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        if (gt == 0) trace_stamp(p.trace, p.trace_cap, 3);  // slot 3: first tile landed
        const uint32_t sb = smem_base + BDW_S_OFF + (uint32_t)slot * BDW_S_SLOT;
        const uint32_t tb = smem_base + (uint32_t)((gt * TS) % BDW_T_STAGES) * BDW_SUB;
        // dG_h (+)= S_h^T T: K = 128 tokens, 16 per MMA; both operands MN-major, 64-wide
        // feature boxes 16 KB apart, 8-row groups 1 KB apart, a K step = 16 rows = 2 KB
#pragma unroll 1
        for (int kk = 0; kk < BDW_TOK / 16; ++kk)
          umma_bf16(tmem_base + DG_COL, make_sdesc(sb + kk * 2048, BDW_SUB, 1024),
                    make_sdesc(tb + kk * 2048, BDW_SUB, 1024), idesc_dg, (i | kk) != 0);
        // Y_h^T = G_h T^T: A = the half's G rows in TMEM (8 columns per K = 16), B = the T
        // sub-tiles K-major (a K step = 32 bytes of every row)
        if (*abort_flag || !mbar_wait_bounded(yempty, (uint32_t)((gt & 1) ^ 1), p.err, p.limit_ns,
                                              kSite + __LINE__)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int v = 0; v < TS; ++v)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ta(tmem_base + Y_COL, tmem_base + G_COL + 32 * v + 8 * kk,
                         make_sdesc(tb + v * BDW_SUB + kk * 32, 16, 1024), idesc_y,
                         (v | kk) != 0);
        umma_commit(&tempty[gt % NSLOT]);
        umma_commit(&sempty[slot]);
        umma_commit(yfull);
      }
      if (!ok) break;
      umma_commit(dgfull);
      umma_commit(gfree);
    }
    // TMEM is freed after the final barrier: every MMA issued must have completed
    umma_commit(mdone);
    mbar_wait_bounded(mdone, 0, p.err, p.limit_ns, kSite + __LINE__);
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;             // TMEM lane quarter
    const int e = (warp - 2) >> 2;      // 0 or 1: which half of the tokens / dG columns
    uint8_t* stg = smem + BDW_STG_OFF + (warp - 2) * BDW_STG;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    long long yt = 0;
    int un = 0;
    int nbuf = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++un) {
      const BdwUnit w = unit_of(p, u);
      // the unit's G rows into TMEM once the previous unit's MMAs no longer read them:
      // row c = 128 h + 32 q + lane of block j, this warp's half of the b columns
      bool got = !*abort_flag &&
                 (un == 0 || mbar_wait_bounded(gfree, (uint32_t)((un - 1) & 1), p.err,
                                               p.limit_ns, kSite + __LINE__));
      if (!__all_sync(0xffffffffu, got)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      {
        const int kh = p.b / 2;  // bf16 columns of G per warp
        const uint4* grow = reinterpret_cast<const uint4*>(
            p.G + ((size_t)w.j * p.b + w.h * 128 + q * 32 + lane) * p.b + (size_t)e * kh);
#pragma unroll 1
        for (int k0 = 0; k0 < kh; k0 += 32) {  // 32 bf16 = 16 TMEM columns
          uint32_t v[16];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint4 x = __ldg(grow + k0 / 8 + t);
            v[4 * t] = x.x;
            v[4 * t + 1] = x.y;
            v[4 * t + 2] = x.z;
            v[4 * t + 3] = x.w;
          }
          tmem_st_32x32b_x16(lane_base + G_COL + (uint32_t)((e * kh + k0) / 2), v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(gfull);
      const int c = w.h * 128 + q * 32 + lane;  // this thread's column within block j
      const float sc = p.colscale ? __ldg(p.colscale + (size_t)w.j * p.b + c) : 1.f;
      for (int i = 0; i < w.nt; ++i, ++yt) {
        got = !*abort_flag &&
              mbar_wait_bounded(yfull, (uint32_t)(yt & 1), p.err, p.limit_ns, kSite + __LINE__);
        if (!__all_sync(0xffffffffu, got)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        if (warp == 2 && lane == 0 && yt < 12) trace_stamp(p.trace, p.trace_cap, 4 + 2 * (int)yt);
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          const int tok = e * 64 + ch * 32;
          uint32_t r[32];
          tmem_ld_32x32b_x32(lane_base + Y_COL + (uint32_t)tok, r);
          tmem_ld_wait();
          __nv_bfloat16* buf = reinterpret_cast<__nv_bfloat16*>(stg + (nbuf & 1) * 2048);
          if (lane == 0) bulk_wait_read<1>();  // this buffer's previous store has read it
          __syncwarp();
#pragma unroll
          for (int t = 0; t < 32; ++t)
            buf[t * 32 + lane] = __float2bfloat16_rn(__uint_as_float(r[t]) * sc);
          fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, buf, w.j * p.b + w.h * 128 + q * 32, (w.t0 + i) * BDW_TOK + tok);
            bulk_commit();
          }
          ++nbuf;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(yempty);
        // slots 4 + 2i / 5 + 2i: tile i's accumulator ready / drained (first 12 tiles)
        if (warp == 2 && lane == 0 && yt < 12) trace_stamp(p.trace, p.trace_cap, 5 + 2 * (int)yt);
      }
      if (!ok) break;
      // the unit's dG_h partial: rows 128 h + 32 q + lane of block j, this warp's half of
      // the columns, through a 128-byte-swizzled [32 x 32] fp32 box
      got = !*abort_flag &&
            mbar_wait_bounded(dgfull, (uint32_t)(un & 1), p.err, p.limit_ns, kSite + __LINE__);
      if (!__all_sync(0xffffffffu, got)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (warp == 2 && lane == 0 && un == 0) trace_stamp(p.trace, p.trace_cap, 28);  // dG ready
      if (lane == 0) bulk_wait_read<0>();  // the Y boxes are no longer read
      __syncwarp();
      const int row0 = (w.s * p.nblk + w.j) * p.b + w.h * 128 + q * 32;
#pragma unroll 1
      for (int cc = 0; cc < p.b / 2; cc += 32) {
        const int col = e * (p.b / 2) + cc;
        uint32_t r[32];
        if (w.nt > 0) {
          tmem_ld_32x32b_x32(lane_base + DG_COL + (uint32_t)col, r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = 0u;  // no tokens in this split: zero partial
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
              make_uint4(r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmD, stg, col, row0);
          bulk_commit();
          bulk_wait_read<0>();
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dgempty);
      if (warp == 2 && lane == 0 && un == 0) trace_stamp(p.trace, p.trace_cap, 29);  // dG stored
    }
    if (warp == 2 && lane == 0) trace_stamp(p.trace, p.trace_cap, 30);  // epilogue loop done
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 31);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

bool umma_bdw_ok(int b) { return (b == 128 || b == 256) && umma_supported(); }

typedef CUresult (*EncodeTiledFn3)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A bf16 [N, D] row-major tensor as the 3-D view {64 features, N tokens, D / 64 feature groups}
// (strides: the row pitch, 128 bytes), boxes of 64 features x 128 tokens x `groups` groups with
// 128-byte swizzle: a box lands as `groups` consecutive [128 x 64] sub-tiles of 16 KB.
static bool encode_groups_3d(CUtensorMap* m, const void* ptr, long long N, long long D,
                             int groups) {
  static EncodeTiledFn3 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn3>(f);
  });
  if (!fn || D % 64) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)N, (cuuint64_t)(D / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)BDW_TOK, (cuuint32_t)groups};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int bdw_splits(long long N, int nblk, int b) {
  // the split count that puts the fewest token tiles on the busiest SM (ties: fewer splits,
  // i.e. fewer partials for the CNP backward to sum)
  const long long nt = (N + BDW_TOK - 1) / BDW_TOK;
  if (nt <= 1 || nblk <= 0) return 1;
  const long long halves = b / 128 > 0 ? b / 128 : 1;
  const long long sms = sm_count();
  int best = 1;
  long long best_cost = LLONG_MAX;
  for (int s = 1; s <= 64; ++s) {
    const long long chunk = (nt + s - 1) / s;
    if (s > 1 && chunk * (s - 1) >= nt) break;  // a trailing split would be empty
    const long long units = (long long)nblk * halves * s;
    const long long cost = (units + sms - 1) / sms * chunk;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

poetx_status umma_bdw(const void* T, const void* S, long long N, int nblk, int b, const void* G,
                      const float* colscale, void* Y, int splits, float* dG, cudaStream_t s) {
  if (nblk == 0) return POETX_OK;
  if (!(b == 128 || b == 256) || splits < 1) return POETX_ERR_SHAPE;
  if (N == 0) {  // no tokens: every partial is zero, Y has no rows
    POETX_CUDA_TRY(cudaMemsetAsync(dG, 0, (size_t)splits * nblk * b * b * sizeof(float), s));
    return POETX_OK;
  }
  const long long D = (long long)nblk * b;
  CUtensorMap tT, tS, tY, tD;
  if (!encode_groups_3d(&tT, T, N, D, b / 64) || !encode_groups_3d(&tS, S, N, D, 2) ||
      !encode_tma_2d(&tY, Y, TMA_BF16, D, N, D, 32, 32, false) ||
      !encode_tma_2d(&tD, dG, TMA_F32, b, (uint64_t)splits * nblk * b, b, 32, 32, true))
    return POETX_ERR_CUDA;
  BdwParams p{};
  p.b = b;
  p.halves = b / 128;
  p.nblk = nblk;
  p.splits = splits;
  p.ntiles = (int)((N + BDW_TOK - 1) / BDW_TOK);
  p.chunk_tiles = (p.ntiles + splits - 1) / splits;
  const long long units = (long long)nblk * p.halves * splits;
  if (units > 0x7fffffffLL) return POETX_ERR_SHAPE;
  p.num_units = (int)units;
  p.G = static_cast<const __nv_bfloat16*>(G);
  p.colscale = colscale;
  p.trace = trace_buffer(&p.trace_cap);
  p.err = device_error_word();
  p.limit_ns = kWaitLimitNs;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(bdw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BDW_SMEM);
  });
  POETX_CUDA_TRY(attr);
  const int grid = (int)(units < sm_count() ? units : sm_count());
  POETX_CUDA_TRY(launch_pdl(bdw_kernel, dim3(grid), dim3(BDW_THREADS), BDW_SMEM, s, tT, tS, tY, tD,
                            p));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_BDW);
  return POETX_OK;
}

}  // namespace poetx
