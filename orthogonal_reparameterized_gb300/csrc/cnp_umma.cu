// Tensor-core products of the Cayley-Neumann parameterization: fp32 accuracy from tcgen05
// kind::tf32 by the 3-term split a*b ~ hi(a)hi(b) + hi(a)lo(b) + lo(a)hi(b), where
// hi(v) = v rounded to the nearest tf32 value (13 low mantissa bits cleared) and
// lo(v) = v - hi(v) (exact in fp32); the dropped lo*lo term is below 2^-22 |a||b|.  The
// tensor-core fp32 accumulation is kept short: every 32-wide K block goes into a fresh TMEM
// accumulator (NACC of them, used in turn) that the promotion warps add into a running sum
// with IEEE fp32 adds ("promotion"), so the accumulated rounding does not grow with b.
//
// Each CNP product (POET-X summary page, "Core method" section 4, eq. 9 and its gradient)
// is C_j = sum_seg opA_seg(j) . opB_seg(j) + epilogue, for every block j, where each operand
// is a linear combination of at most two b x b fp32 arrays (Q, Q^2, X, M1).  One CTA makes
// one 128 x BN output tile of one block (of a symmetric product such as Q^2, only the tiles on
// and right of each diagonal 128 x 128 block, the ones right of it also storing their mirror):
//   warp 0      TMA: the raw fp32 tiles of every source array of the current K block
//   warps 2-9   form v = c0*src0 + c1*src1 and split it into hi(v), lo(v): the A operand
//               straight into tensor memory (where the MMA reads it), the B operand in place
//               in shared memory (same swizzled offsets, so the layout is kept)
//   warp 1      three tcgen05.mma kind::tf32 per K=8 step into the K block's accumulator
//   warps 10..  promotion: add each K block's accumulator into the running sum
//   all warps   epilogue: out = sum + e1 E1 + e2 E2 + eI I through a shared-memory tile,
//               stored as fp32 / fp32^T / bf16 / bf16^T with coalesced 16-byte accesses
// Both operand tiles are K-major (kind::tf32 takes no MN-major operand): A tiles are rows of
// A, B tiles rows of B^T (the B terms of a product are given transposed); 128-byte swizzle.
// Keeping A out of shared memory halves the shared-memory traffic of a K block, which is
// what bounds this kernel.  Every wait is bounded (POETX_ERR_TIMEOUT on expiry, then drain,
// free TMEM, return).
#include <mutex>

#include "cnp_umma.h"
#include "common.cuh"
#include "kernels.h"

namespace poetx {

// Site id of this file's bounded waits (file id x 10000 + source line), recorded with
// the first timeout.
constexpr int kSite = 2 * 10000;

namespace {

constexpr int BM = 128;
constexpr int BK = 32;      // fp32 elements per 128-byte row
constexpr int NMAPS = 8;    // distinct (source array, operand role) pairs of one product

struct CnpMaps {
  CUtensorMap m[NMAPS];
};

struct TSrc {
  int map;   // index into CnpMaps, -1 = absent
  float coef;
};
struct TOp {
  TSrc s[2];
};

struct CnpUParams {
  int b;
  // Geometry: batch entry j makes output rows 0 .. M-1 (M = b for a CNP product); its A tile
  // (rows i0 .., K columns k0 ..) sits at coordinate (a_col_blk j + k0, a_row_blk j + i0) of
  // the A map; output element (i, c) goes to out[j o_blk + i o_ld + c] and to
  // out_t[j ot_blk + c ot_ld + i].
  int M, a_row_blk, a_col_blk;
  long long o_blk, o_ld, ot_blk, ot_ld;
  int nmaps;
  int nseg;
  int kb_per_seg;
  TOp A[2], B[2];
  const float* E1;
  float e1;
  const float* E2;
  float e2;
  float eI;
  float* out_f32;
  float* out_f32_t;
  __nv_bfloat16* out_bf16;
  __nv_bfloat16* out_bf16_t;
  unsigned long long* trace;  // diagnostic phase stamps (nullable)
  size_t trace_cap;
  int* err;
  unsigned long long limit_ns;
  // 1: the product is symmetric (b a multiple of 128): only the tiles whose 128-column block
  // is on or right of their 128-row block run (blockIdx.x enumerates them row by row), and
  // each one right of the diagonal also writes its transpose into out_f32, so every element
  // below a diagonal 128 x 128 block is the copy of its mirror whatever the tile width
  int sym;
};

__host__ __device__ constexpr uint32_t tf32_idesc(int M, int N) {
  return (1u << 4)                      // accumulator f32
         | (2u << 7)                    // A: tf32
         | (2u << 10)                   // B: tf32
         | (0u << 15)                   // A K-major
         | (0u << 16)                   // B K-major (kind::tf32 takes K-major operands only)
         | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// A operand in tensor memory (M rows = lanes, one tf32 element per 32-bit column), B in
// shared memory.
__device__ __forceinline__ void umma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// tf32 split of v: hi = v rounded to the nearest tf32 value, lo = v - hi (exact).
__device__ __forceinline__ void split_tf32(float v, uint32_t& hi, uint32_t& lo) {
  const float h = __uint_as_float((__float_as_uint(v) + 0x1000u) & 0xFFFFE000u);
  hi = __float_as_uint(h);
  lo = __float_as_uint(v - h);
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// v = c0*x + c1*y, then x <- hi(v), y <- lo(v).
__device__ __forceinline__ void combine_split(float4* x, float4* y, float c0, float c1, bool two) {
  float4 a = *x;
  float4 b = two ? *y : make_float4(0.f, 0.f, 0.f, 0.f);
  float v[4] = {c0 * a.x, c0 * a.y, c0 * a.z, c0 * a.w};
  if (two) {
    v[0] = fmaf(c1, b.x, v[0]);
    v[1] = fmaf(c1, b.y, v[1]);
    v[2] = fmaf(c1, b.z, v[2]);
    v[3] = fmaf(c1, b.w, v[3]);
  }
  float hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hi[i] = __uint_as_float((__float_as_uint(v[i]) + 0x1000u) & 0xFFFFE000u);
    lo[i] = v[i] - hi[i];
  }
  *x = make_float4(hi[0], hi[1], hi[2], hi[3]);
  *y = make_float4(lo[0], lo[1], lo[2], lo[3]);
}

// Warp roles: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2..9 converters, 10.. promotion.  Converter warp w forms and splits the A operand of its TMEM lane quarter w % 4
// (rows 32 (w % 4) .. +31, K columns 16 ((w - 2) / 4) .. +15) and writes hi and lo into
// tensor memory; the B operand is formed and split in shared memory by all converters.
// Promotion warp w adds each K block's accumulator of its lane quarter w % 4 (and column
// slice) into the running sum, so that with two or more accumulators the MMAs of a K block
// never wait for the promotion of the one before.  Tiles of 32 or 64 columns keep the sum in
// registers (64 columns per thread); TMEM columns: NACC accumulators of BN, then STAGES A
// slots of 64 (hi 32 + lo 32).  Tiles of 128 columns run 18 warps, which the SM's four
// register partitions allow only 96 registers each, so they keep it in TMEM: 2 accumulators,
// the sum, 2 A slots (released by the MMAs for the converters).
constexpr int kConvWarps = 8;  // two per TMEM lane quarter
// Tiles of 32 or 64 columns: 4 promotion warps, 4 TMEM accumulators, the epilogue-term tiles
// prefetched into their own shared memory during the K loop.  Tiles of 128 columns (blocks of
// 256 and up when 64-wide tiles would need more than one wave of CTAs): 8 promotion warps
// (two per lane quarter, 64 columns each), two accumulators, epilogue-term tiles fetched into
// the idle ring after the K loop.
__host__ __device__ constexpr int prom_warps(int bn) { return bn >= 128 ? 8 : 4; }
__host__ __device__ constexpr int cnp_nacc(int bn) { return bn >= 128 ? 2 : 4; }
__host__ __device__ constexpr bool e_in_ring(int bn) { return bn >= 128; }
__host__ __device__ constexpr int cnp_threads(int bn) {
  return 32 * (2 + kConvWarps + prom_warps(bn));
}

// cp.async (global -> shared, no registers held while in flight; bypasses L1).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int BN>
__host__ __device__ constexpr int cnp_stages() { return BN >= 64 ? 3 : 4; }
// dynamic shared memory: the operand ring, the two epilogue-term tiles, 1 KB of alignment
// slack and the barriers
// bytes of the region the ring occupies during the K loop and the epilogue's tiles after it
template <int BN>
__host__ __device__ constexpr int cnp_ring_bytes() {
  return cnp_stages<BN>() * (2 * BM * BK * 4 + 2 * BN * BK * 4) >
                 (BM * (BN + 4) + (e_in_ring(BN) ? 2 * BM * BN : 0)) * 4
             ? cnp_stages<BN>() * (2 * BM * BK * 4 + 2 * BN * BK * 4)
             : (BM * (BN + 4) + (e_in_ring(BN) ? 2 * BM * BN : 0)) * 4;
}
template <int BN>
__host__ __device__ constexpr int cnp_smem() {
  return cnp_ring_bytes<BN>() + (e_in_ring(BN) ? 0 : 2 * BM * BN * 4) + 1024 + 256;
}

template <int BN>
__global__ void __launch_bounds__(cnp_threads(BN), 1)
    cnp_umma_kernel(const __grid_constant__ CnpMaps maps, const CnpUParams p) {
  constexpr int STAGES = cnp_stages<BN>();
  constexpr int NACC = cnp_nacc(BN);
  constexpr int kPromWarps = prom_warps(BN);
  constexpr int kThreadsCnp = cnp_threads(BN);
  constexpr bool E_RING = e_in_ring(BN);
  constexpr int CW = BN * 4 / kPromWarps;     // running-sum columns per promotion thread
  constexpr int NCT = 32 * kConvWarps;        // converter threads
  constexpr uint32_t A_BYTES = BM * BK * 4;   // 16 KB per buffer
  constexpr uint32_t B_BYTES = BN * BK * 4;   // BN * 128 bytes per buffer
  constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
  constexpr uint32_t RING_BYTES = cnp_ring_bytes<BN>();  // >= STAGES * STAGE_BYTES
  constexpr bool SUM_TMEM = BN >= 128;
  constexpr int ASLOTS = SUM_TMEM ? 2 : STAGES;          // TMEM slots of the A operand
  constexpr uint32_t SUM_COL = NACC * BN;                // running sum (SUM_TMEM)
  constexpr uint32_t A_COL = NACC * BN + (SUM_TMEM ? BN : 0);  // A slots: + 64 j (+32: lo)
  constexpr uint32_t TMEM_COLS = A_COL + 64 * ASLOTS <= 256 ? 256 : 512;
  constexpr int G4 = BN / 4;                  // float4 groups per tile row
  constexpr int LD = BN + 4;                  // staged tile pitch (16-byte rows)
  constexpr int TILE = BM * BN;               // floats of one epilogue-term tile
  static_assert(A_COL + 64 * ASLOTS <= TMEM_COLS, "accumulators, sum and A slots fit TMEM");
  static_assert(RING_BYTES >= (uint32_t)(BM * LD + (E_RING ? 2 * TILE : 0)) * 4,
                "the staged tile (and the epilogue-term tiles) fit the ring");
  constexpr uint32_t IDESC = tf32_idesc(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* const tile = reinterpret_cast<float*>(smem);  // epilogue (ring idle)
  float* const etile = E_RING ? tile + BM * LD           // [2][BM][BN] E1, E2
                              : reinterpret_cast<float*>(smem + RING_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + (E_RING ? 0 : 2 * TILE * 4));
  uint64_t* conv = full + STAGES;
  uint64_t* empty = conv + STAGES;
  uint64_t* tfull = empty + STAGES;   // [NACC] accumulator holds a finished K block
  uint64_t* tempty = tfull + NACC;    // [NACC] accumulator has been read back
  uint64_t* afree = tempty + NACC;    // [ASLOTS] A slot no longer read by MMAs (ASLOTS < STAGES)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(afree + ASLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.z;
  constexpr int R = BM / BN;  // tiles per 128-column block
  int mt = blockIdx.x, nt = blockIdx.y;
  if (p.sym) {  // row mt holds the tiles nt = R mt .. b / BN - 1
    const int MT = p.b / BM, NT = p.b / BN;
    int idx = blockIdx.x;
    mt = 0;
    while (mt < MT - 1 && idx >= NT - mt * R) {
      idx -= NT - mt * R;
      ++mt;
    }
    nt = mt * R + idx;
  }
  const bool mirror_tile = p.sym && nt / R != mt;
  const unsigned long long lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  auto stamp = [&](int slot) {
    if (p.trace) {
      const size_t i = lin * kTraceSlots + slot;
      if (i < p.trace_cap) p.trace[i] = global_ns();
    }
  };
  if (threadIdx.x == 0) stamp(0);
  pdl_trigger();
  const int b = p.b;
  const int num_kb = p.nseg * p.kb_per_seg;
  const int row0 = blk * b;  // first row of this block in the [nblk*b, b] views
  const long long base = (long long)blk * b * b;
  const int i0 = mt * BM, j0 = nt * BN;
  const int rows = p.M - i0 < BM ? p.M - i0 : BM;  // valid rows of the tile; M % 32 == 0

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], kConvWarps);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kPromWarps);
    }
    for (int j = 0; j < ASLOTS; ++j) mbar_init(&afree[j], 1);
    *abort_flag = 0;
    fence_mbar_init();
    for (int i = 0; i < p.nmaps; ++i) tma_prefetch_desc(&maps.m[i]);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);
  pdl_wait();  // the previous kernel's outputs are visible from here on
  if (threadIdx.x == 0) stamp(1);

  int tma_issued = 0;  // TMA thread: K blocks issued
  int mma_last = -1;   // MMA thread: last K block issued
  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (*abort_flag || !mbar_wait_bounded(&empty[s], ph ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        break;
      }
      const int seg = kb / p.kb_per_seg;
      const int k0 = (kb % p.kb_per_seg) * BK;
      const TOp& A = p.A[seg];
      const TOp& B = p.B[seg];
      uint32_t bytes = 0;
      for (int i = 0; i < 2; ++i) {
        if (A.s[i].map >= 0) bytes += A_BYTES;
        if (B.s[i].map >= 0) bytes += B_BYTES;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      if (kb < 8) stamp(2 + kb);  // slots 2..9: K block issued
      uint8_t* st = smem + s * STAGE_BYTES;
      for (int i = 0; i < 2; ++i) {
        if (A.s[i].map >= 0)  // rows mt*128.. of A (one 32 x 128 box)
          tma_load_2d(st + i * A_BYTES, &maps.m[A.s[i].map], &full[s], p.a_col_blk * blk + k0,
                      p.a_row_blk * blk + i0);
        if (B.s[i].map >= 0)  // rows nt*BN.. of B^T, columns k0..k0+31 (one 32 x BN box)
          tma_load_2d(st + 2 * A_BYTES + i * B_BYTES, &maps.m[B.s[i].map], &full[s], k0,
                      row0 + j0);
      }
      ++tma_issued;
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      const int a = kb % NACC;
      const uint32_t pa = (kb / NACC) & 1;
      if (*abort_flag || !mbar_wait_bounded(&conv[s], ph, p.err, p.limit_ns, kSite + __LINE__) ||
          !mbar_wait_bounded(&tempty[a], pa ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(a * BN);
      const uint32_t a_hi = tmem_base + A_COL + 64u * (uint32_t)(kb % ASLOTS);
      const uint32_t a_lo = a_hi + 32;
      const uint32_t b_hi = smem_base + s * STAGE_BYTES + 2 * A_BYTES;
      const uint32_t b_lo = b_hi + B_BYTES;
#pragma unroll
      for (int k = 0; k < BK / 8; ++k) {  // K = 8 per MMA: 8 TMEM columns of A
        const uint64_t bh = sdesc(b_hi + k * 32, 16, 1024), bl = sdesc(b_lo + k * 32, 16, 1024);
        umma_tf32_ta(d, a_hi + 8 * k, bh, IDESC, k != 0);
        umma_tf32_ta(d, a_hi + 8 * k, bl, IDESC, 1);
        umma_tf32_ta(d, a_lo + 8 * k, bh, IDESC, 1);
      }
      umma_commit(&empty[s]);
      umma_commit(&tfull[a]);
      if (ASLOTS < STAGES) umma_commit(&afree[kb % ASLOTS]);
      mma_last = kb;
    }
  } else if (warp >= 2 && warp < 2 + kConvWarps) {
    // ---------------------------------------------------------------- converters
    const int ct = threadIdx.x - 64;  // 0..NCT-1
    const int qa = warp & 3, ha = (warp - 2) >> 2;
    const int ra = qa * 32 + lane;    // A row of this thread
    const uint32_t a_lane = tmem_base + ((uint32_t)(qa * 32) << 16);
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      bool ok = !*abort_flag && mbar_wait_bounded(&full[s], ph, p.err, p.limit_ns, kSite + __LINE__);
      // with fewer A slots than ring stages, the slot's previous K block must have been read
      if (ASLOTS < STAGES && ok && kb >= ASLOTS)
        ok = mbar_wait_bounded(&afree[kb % ASLOTS], (uint32_t)((kb / ASLOTS - 1) & 1), p.err,
                               p.limit_ns, kSite + __LINE__);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      const int seg = kb / p.kb_per_seg;
      const TOp& A = p.A[seg];
      const TOp& B = p.B[seg];
      uint8_t* st = smem + s * STAGE_BYTES;
      {
        // A: row ra, K columns 16 ha .. 16 ha + 15 = 16-byte chunks 4 ha .. 4 ha + 3 of the
        // 128-byte row (128-byte swizzle: chunk c of row r sits at chunk c ^ (r % 8))
        const bool two = A.s[1].map >= 0;
        const float c0 = A.s[0].coef, c1 = A.s[1].coef;
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int off = ra * 128 + (((4 * ha + t) ^ (ra & 7)) << 4);
          const float4 x = *reinterpret_cast<const float4*>(st + off);
          float4 v = make_float4(c0 * x.x, c0 * x.y, c0 * x.z, c0 * x.w);
          if (two) {
            const float4 y = *reinterpret_cast<const float4*>(st + A_BYTES + off);
            v.x = fmaf(c1, y.x, v.x);
            v.y = fmaf(c1, y.y, v.y);
            v.z = fmaf(c1, y.z, v.z);
            v.w = fmaf(c1, y.w, v.w);
          }
          split_tf32(v.x, hi[4 * t], lo[4 * t]);
          split_tf32(v.y, hi[4 * t + 1], lo[4 * t + 1]);
          split_tf32(v.z, hi[4 * t + 2], lo[4 * t + 2]);
          split_tf32(v.w, hi[4 * t + 3], lo[4 * t + 3]);
        }
        const uint32_t col = A_COL + 64u * (uint32_t)(kb % ASLOTS) + 16u * (uint32_t)ha;
        tmem_st_32x32b_x16(a_lane + col, hi);
        tmem_st_32x32b_x16(a_lane + col + 32, lo);
      }
      float4* b0 = reinterpret_cast<float4*>(st + 2 * A_BYTES);
      float4* b1 = reinterpret_cast<float4*>(st + 2 * A_BYTES + B_BYTES);
      const bool b_two = B.s[1].map >= 0;
#pragma unroll 4
      for (int e = ct; e < (int)(B_BYTES / 16); e += NCT)
        combine_split(b0 + e, b1 + e, B.s[0].coef, B.s[1].coef, b_two);
      tmem_st_wait();      // A in TMEM complete
      fence_async_smem();  // B in shared memory -> visible to the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv[s]);
      if (warp == 2 && lane == 0 && kb < 8) stamp(10 + kb);  // slots 10..17: converted
    }
  } else if (warp >= 2 + kConvWarps) {
    // ---------------------------------------------------------------- promotion
    // (whole warps only: lanes 1..31 of warps 0 and 1 take no role and go on to the
    // epilogue)
    const int pw = warp - (2 + kConvWarps);
    const int q = warp & 3;           // TMEM lane quarter of this warp
    const int h = pw >> 2;            // column slice of this warp
    const int r = q * 32 + lane;      // tile row of this thread
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * CW);
    // the epilogue terms are inputs of this launch: fetch their tiles (now, to land while
    // the K loop runs, or into the ring once it is idle)
    auto fetch_e = [&]() {
      for (int e = 0; e < 2; ++e) {
        const float* E = e == 0 ? p.E1 : p.E2;
        if (!E) continue;
        for (int g = pw * 32 + lane; g < rows * G4; g += kPromWarps * 32) {
          const int rr = g / G4, c = 4 * (g % G4);
          cp_async16(etile + e * TILE + rr * BN + c, E + base + (long long)(i0 + rr) * b + j0 + c);
        }
      }
    };
    if (!E_RING) fetch_e();
    bool ok_all = true;
    float sum[SUM_TMEM ? 1 : CW];  // (registers) this thread's row: columns h * CW .. + CW - 1
    for (int kb = 0; kb < num_kb; ++kb) {
      const int a = kb % NACC;
      const bool ok = !*abort_flag &&
                      mbar_wait_bounded(&tfull[a], (kb / NACC) & 1, p.err, p.limit_ns, kSite + __LINE__);
      ok_all = __all_sync(0xffffffffu, ok);
      if (!ok_all) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if constexpr (SUM_TMEM) {
#pragma unroll
        for (int c0 = 0; c0 < CW; c0 += 32) {  // two 16-column chunks per load round trip
          uint32_t v[2][16], w[2][16];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            tmem_ld_32x32b_x16(lane_base + (uint32_t)(a * BN + c0 + 16 * u), v[u]);
            if (kb > 0) tmem_ld_32x32b_x16(lane_base + (uint32_t)(SUM_COL + c0 + 16 * u), w[u]);
          }
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (kb > 0) {
#pragma unroll
              for (int t = 0; t < 16; ++t)
                v[u][t] = __float_as_uint(__uint_as_float(w[u][t]) + __uint_as_float(v[u][t]));
            }
            tmem_st_32x32b_x16(lane_base + (uint32_t)(SUM_COL + c0 + 16 * u), v[u]);
          }
        }
        tmem_st_wait();
      } else {
#pragma unroll
        for (int c0 = 0; c0 < CW; c0 += 16) {  // 16 columns per load: few live registers
          uint32_t v[16];
          tmem_ld_32x32b_x16(lane_base + (uint32_t)(a * BN + c0), v);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 16; ++t)
            sum[c0 + t] = kb == 0 ? __uint_as_float(v[t]) : sum[c0 + t] + __uint_as_float(v[t]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      if (pw == 0 && lane == 0 && kb < 8) stamp(18 + kb);  // slots 18..25: promoted
    }
    // every MMA has completed, so the ring is idle: the sum goes to a shared-memory tile
    if (E_RING && ok_all) fetch_e();
    if (ok_all && num_kb > 0) {
      if constexpr (SUM_TMEM) {
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < CW; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(lane_base + (uint32_t)(SUM_COL + c0), v);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 16; t += 4)
            *reinterpret_cast<float4*>(tile + r * LD + h * CW + c0 + t) =
                make_float4(__uint_as_float(v[t]), __uint_as_float(v[t + 1]),
                            __uint_as_float(v[t + 2]), __uint_as_float(v[t + 3]));
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < CW; c0 += 4)
          *reinterpret_cast<float4*>(tile + r * LD + h * CW + c0) =
              make_float4(sum[c0], sum[c0 + 1], sum[c0 + 2], sum[c0 + 3]);
      }
    }
    cp_async_wait_all();
    if (!ok_all) *abort_flag = 1;
  }

  // ------------------------------------------------------------------ epilogue (all warps)
  // out = sum + e1 E1 + e2 E2 + eI I; every global store is coalesced and 8 or 16 bytes wide
  const bool live = __syncthreads_or(*abort_flag) == 0;
  if (threadIdx.x == 0) stamp(26);  // slot 26: tile staged
  const int ng = rows * G4;
  if (live) {
    for (int g = threadIdx.x; g < ng; g += kThreadsCnp) {
      const int rr = g / G4, c = 4 * (g % G4);
      const int i = i0 + rr, j = j0 + c;
      float4* tp = reinterpret_cast<float4*>(tile + rr * LD + c);
      float4 o = *tp;
      if (p.E1) {
        const float4 w = *reinterpret_cast<const float4*>(etile + rr * BN + c);
        o.x = fmaf(p.e1, w.x, o.x);
        o.y = fmaf(p.e1, w.y, o.y);
        o.z = fmaf(p.e1, w.z, o.z);
        o.w = fmaf(p.e1, w.w, o.w);
      }
      if (p.E2) {
        const float4 w = *reinterpret_cast<const float4*>(etile + TILE + rr * BN + c);
        o.x = fmaf(p.e2, w.x, o.x);
        o.y = fmaf(p.e2, w.y, o.y);
        o.z = fmaf(p.e2, w.z, o.z);
        o.w = fmaf(p.e2, w.w, o.w);
      }
      if (i == j) o.x += p.eI;
      if (i == j + 1) o.y += p.eI;
      if (i == j + 2) o.z += p.eI;
      if (i == j + 3) o.w += p.eI;
      *tp = o;
      const long long idx = blk * p.o_blk + (long long)i * p.o_ld + j;
      if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + idx) = o;
      if (p.out_bf16)
        *reinterpret_cast<uint2*>(p.out_bf16 + idx) =
            make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
    }
  }
  if (p.out_f32_t || p.out_bf16_t || mirror_tile) {
    __syncthreads();
    if (live) {
      // transposed outputs: consecutive threads take consecutive rows (rows % 32 == 0), so
      // each of the four stores of a float4 group is coalesced
      for (int g = threadIdx.x; g < ng; g += kThreadsCnp) {
        const int rr = g % rows, c = 4 * (g / rows);
        const float4 v = *reinterpret_cast<const float4*>(tile + rr * LD + c);
        const float o[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const long long tidx = blk * p.ot_blk + (long long)(j0 + c + k) * p.ot_ld + (i0 + rr);
          if (p.out_f32_t) p.out_f32_t[tidx] = o[k];
          if (mirror_tile)  // the symmetric partner tile
            p.out_f32[blk * p.o_blk + (long long)(j0 + c + k) * p.o_ld + (i0 + rr)] = o[k];
          if (p.out_bf16_t) p.out_bf16_t[tidx] = __float2bfloat16_rn(o[k]);
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (warp == 0 && lane == 0 && *abort_flag) {
    // drain: the last STAGES K blocks issued may still be landing
    for (int g = tma_issued - 1; g >= 0 && g >= tma_issued - STAGES; --g)
      mbar_wait_bounded(&full[g % STAGES], (g / STAGES) & 1, p.err, p.limit_ns, kSite + __LINE__);
  }
  if (warp == 1 && lane == 0 && mma_last >= 0)  // TMEM is freed below: the MMAs must be done
    mbar_wait_bounded(&tfull[mma_last % NACC], (mma_last / NACC) & 1, p.err, p.limit_ns, kSite + __LINE__);
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) stamp(31);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [nblk*b rows][b cols] fp32 view with {32, box_rows} boxes, 128-byte swizzle (per-thread
// cache of encoded maps keyed by pointer, shape and box).
bool make_blk_map(CUtensorMap* m, const float* ptr, int nblk, int b, int box_rows) {
  struct Entry {
    const float* ptr;
    int nblk, b, box_rows, dev;
    CUtensorMap map;
  };
  constexpr int kEntries = 32;
  thread_local Entry cache[kEntries];
  thread_local int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < kEntries; ++i) {
    const Entry& e = cache[i];
    if (e.ptr == ptr && ptr && e.nblk == nblk && e.b == b && e.box_rows == box_rows &&
        e.dev == dev) {
      *m = e.map;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)b, (cuuint64_t)nblk * b};
  cuuint64_t strides[1] = {(cuuint64_t)b * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.ptr = ptr; e.nblk = nblk; e.b = b; e.box_rows = box_rows; e.dev = dev; e.map = *m;
  return true;
}

template <int BN>
poetx_status launch_t(const CnpMaps& maps, const CnpUParams& p, int nblk, cudaStream_t s) {
  auto k = cnp_umma_kernel<BN>;
  constexpr int smem = cnp_smem<BN>();
  static_assert(smem <= 227 * 1024, "shared memory per CTA exceeds the sm_103 limit");
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  POETX_CUDA_TRY(attr);
  const int MT = p.b / BM, NT = p.b / BN;
  dim3 grid(p.sym ? MT * NT - (BM / BN) * MT * (MT - 1) / 2 : (p.M + BM - 1) / BM,
            p.sym ? 1 : p.b / BN, nblk);
  POETX_CUDA_TRY(launch_pdl(k, grid, dim3(cnp_threads(BN)), smem, s, maps, p));
  POETX_CUDA_TRY(cudaGetLastError());
  return POETX_OK;
}

}  // namespace

bool cnp_umma_ok(int b) {
  return b >= 32 && b <= 1024 && b % 32 == 0 && umma_supported();
}

poetx_status cnp_umma_product(const CnpProduct& g, int nblk, cudaStream_t s) {
  if (nblk == 0) return POETX_OK;
  const long long M = g.a_mat ? g.a_rows : g.b;
  if (g.a_mat && (M <= 0 || M % 32 || M > 0x7fffffffLL || g.nseg != 1 || g.A[0].p1 != g.a_mat ||
                  g.A[0].p2 || g.E1 || g.E2 || g.eI != 0.f || g.out_bf16 || g.out_bf16_t))
    return POETX_ERR_ARG;
  // 128-wide tiles once 64-wide ones would take more than one wave of CTAs (one per SM)
  const long long tiles64 = (long long)((M + BM - 1) / BM) * (g.b / 64) * nblk;
  const int BN = (g.b % 128 == 0 && g.b >= 256 && tiles64 > sm_count()) ? 128
                 : (g.b % 64 == 0 ? 64 : 32);
  CnpMaps maps;
  const float* ptrs[NMAPS] = {};
  int roles[NMAPS] = {};
  int nmaps = 0;
  // role 0: A operand (128-row boxes), role 1: transposed B operand (BN-row boxes)
  auto map_of = [&](const float* ptr, int role) -> int {
    if (!ptr) return -1;
    for (int i = 0; i < nmaps; ++i)
      if (ptrs[i] == ptr && roles[i] == role) return i;
    if (nmaps == NMAPS) return -2;
    if (role == 0 && g.a_mat && ptr == g.a_mat) {  // [a_rows, nblk b] matrix, 128-row boxes
      const uint64_t cols = (uint64_t)nblk * g.b;
      if (!encode_tma_2d(&maps.m[nmaps], ptr, TMA_F32, cols, (uint64_t)M, cols, 32, BM, true))
        return -3;
    } else if (!make_blk_map(&maps.m[nmaps], ptr, nblk, g.b, role == 0 ? BM : BN)) {
      return -3;
    }
    ptrs[nmaps] = ptr;
    roles[nmaps] = role;
    return nmaps++;
  };
  CnpUParams p{};
  p.b = g.b;
  p.M = (int)M;
  if (g.a_mat) {  // column block j of the matrix; outputs [M, nblk b] and its transpose
    p.a_row_blk = 0;
    p.a_col_blk = g.b;
    p.o_blk = g.b;
    p.o_ld = (long long)nblk * g.b;
    p.ot_blk = (long long)g.b * M;
    p.ot_ld = M;
  } else {  // the [nblk, b, b] stacks
    p.a_row_blk = g.b;
    p.a_col_blk = 0;
    p.o_blk = p.ot_blk = (long long)g.b * g.b;
    p.o_ld = p.ot_ld = g.b;
  }
  p.nseg = g.nseg;
  p.kb_per_seg = g.b / BK;
  for (int sg = 0; sg < g.nseg; ++sg) {
    const CnpTerm* ts[2] = {&g.A[sg], &g.B[sg]};
    TOp* os[2] = {&p.A[sg], &p.B[sg]};
    for (int w = 0; w < 2; ++w) {
      for (int i = 0; i < 2; ++i) {
        const float* ptr = i == 0 ? ts[w]->p1 : ts[w]->p2;
        const int mi = map_of(ptr, w);
        if (mi < -1) return mi == -2 ? POETX_ERR_UNSUPPORTED : POETX_ERR_CUDA;
        os[w]->s[i].map = mi;
        os[w]->s[i].coef = i == 0 ? ts[w]->c1 : ts[w]->c2;
      }
    }
  }
  p.E1 = g.E1; p.e1 = g.e1; p.E2 = g.E2; p.e2 = g.e2; p.eI = g.eI;
  p.out_f32 = g.out_f32;
  p.out_f32_t = g.out_f32_t;
  p.out_bf16 = g.out_bf16;
  p.out_bf16_t = g.out_bf16_t;
  p.err = device_error_word();
  p.limit_ns = kWaitLimitNs;
  p.trace = trace_buffer(&p.trace_cap);
  p.nmaps = nmaps;
  p.sym = g.mirror && g.b % BM == 0 && !g.a_mat && g.out_f32 && !g.out_f32_t && !g.out_bf16 &&
          !g.out_bf16_t;
  if (BN == 128) return launch_t<128>(maps, p, nblk, s);
  if (BN == 64) return launch_t<64>(maps, p, nblk, s);
  return launch_t<32>(maps, p, nblk, s);
}

}  // namespace poetx
