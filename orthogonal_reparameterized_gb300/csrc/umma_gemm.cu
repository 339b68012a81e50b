// Tensor-core GEMM engine for sm_103a: tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) fed by TMA
// with 128-byte-swizzled shared-memory tiles, an mbarrier pipeline and a TMEM -> register
// epilogue.  It carries the bf16 products of the POET-X layer:
//
//   block-diagonal multiplies  Y_j = X_j G_j or X_j G_j^T per block j       (steps S4, S6,
//                              S10, S12; POET-X summary page, "Core method" section 3)
//   frozen-weight contraction  B = A W'^T (forward) and dA = dB W' (backward)  (S5, S11, S9;
//                              same page, section 1)
//   block weight gradients     dG_j = X_j^T dY_j over a token range (S10, S12)
//
// Persistent CTAs walk the 128 x BN output tiles (tile t = blockIdx.x, + gridDim.x, ...; the
// M index varies fastest so that concurrent CTAs share the B operand in L2; the W'
// contraction walks bands of 2048 tokens that way, so that the concurrent CTAs also share a
// few A row stripes).  Warp 0 issues
// the TMA loads into a STAGES-deep ring, one thread of warp 1 issues the MMAs (4 x K=16 per
// 64-wide K block) into one of two TMEM accumulators (alternate tiles), and warps 2-9 read
// the other accumulator back (tcgen05.ld 32x32b: warp w reads lanes 32*(w%4)..+31 = output
// rows) and store it, so the epilogue of one tile overlaps the loads and MMAs of the next.
// Operands may be K-major (rows of the tile are contiguous along K) or MN-major (contiguous
// along M/N, e.g. the token-major activations of a weight gradient); both use the canonical
// 128-byte swizzle layouts of tcgen05.  With an int8 W' the frozen-weight contraction runs
// in its own kernel (below), transposed.
// Every mbarrier wait is bounded; on expiry the kernel records POETX_ERR_TIMEOUT, drains
// its own copies, frees its TMEM and returns.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace poetx {

// Site id of this file's bounded waits (file id x 10000 + source line), recorded with
// the first timeout.
constexpr int kSite = 1 * 10000;

namespace {

enum Mode : int { MODE_PLAIN = 0, MODE_BLOCKDIAG = 1, MODE_WGRAD = 2 };

struct UmmaParams {
  int mode;
  int tiles_m, tiles_n, num_tiles;  // tile t: mt = t % tiles_m, nt = (t / tiles_m) % tiles_n,
                                    // z = t / (tiles_m * tiles_n) (block, or block*splits+split)
  int band_m;    // PLAIN: M tiles per band of the grouped raster (0: plain M-fastest order)
  int M;         // valid output rows of the whole problem (tokens, or b for WGRAD)
  int num_kb;    // 64-wide K blocks per CTA (PLAIN, BLOCKDIAG)
  int b;         // block size (BLOCKDIAG, WGRAD)
  int nblk;      // blocks (WGRAD)
  int splits;    // token splits (WGRAD)
  int kchunk;    // tokens per split, multiple of 64 (WGRAD)
  long long ntok;  // tokens (WGRAD)
  void* C;
  long long ldc;
  const float* colscale;
  const int32_t* out_perm;  // BLOCKDIAG: output column c is stored at column out_perm[c]
  const uint8_t* bpre;      // nullable: B operand (a weight, not written by the previous
  unsigned long long bpre_bytes;  // kernel) to prefetch into L2 while that kernel drains
  unsigned long long* trace;  // diagnostic phase stamps (nullable)
  size_t trace_cap;
  int* err;
  unsigned long long limit_ns;
};

constexpr int BM = 128;
constexpr int BK = 64;

// K-major tile: rows of 128 bytes (64 bf16 along K), 8-row groups 1024 bytes apart; the
// k-th K=16 slice starts 32 bytes further.  MN-major tile: boxes of 64 K-rows x 64 MN
// elements (8 KB) side by side along MN (LBO = 8 KB), 8 K-row groups 1024 bytes apart; the
// k-th K=16 slice starts 16 rows (2048 bytes) further.
template <bool MN>
__device__ __forceinline__ uint64_t tile_desc(uint32_t base, int k) {
  return MN ? make_sdesc(base + k * 2048, 8192, 1024) : make_sdesc(base + k * 32, 16, 1024);
}

// Coordinates of one output tile (TMA coordinates are {inner, outer} = {column, row}).
struct TileCoords {
  int num_kb;
  int a_c0, a_c1, b_c0, b_c1;
  long long out_row0, out_col0;
  int split, blk;
};

// CL = 2 (PLAIN): tile t is a pair of M tiles sharing the B tile; CTA rank r of the cluster
// takes M tile 2 (t % tiles_m) + r.
template <int BN, bool B_MN, int CL>
__device__ __forceinline__ TileCoords tile_coords(const UmmaParams& p, int t, int crank) {
  TileCoords c;
  int mi, nt, z;
  if (p.mode == MODE_PLAIN && p.band_m > 0 && p.band_m < p.tiles_m) {
    // grouped raster: bands of band_m M tiles, each band's tiles M-fastest across all N
    // columns, so the tiles in flight at once share a few A row stripes and a few W' stripes
    // (both re-read from L2 instead of DRAM)
    const int per_band = p.band_m * p.tiles_n;
    const int band = t / per_band, r = t % per_band;
    const int m0 = band * p.band_m;
    const int gm = p.tiles_m - m0 < p.band_m ? p.tiles_m - m0 : p.band_m;
    mi = m0 + r % gm;
    nt = r / gm;
    z = 0;
  } else {
    mi = t % p.tiles_m;
    const int rest = t / p.tiles_m;
    nt = rest % p.tiles_n;
    z = rest / p.tiles_n;
  }
  const int mt = CL > 1 ? CL * mi + crank : mi;
  c.num_kb = p.num_kb;
  c.out_row0 = (long long)mt * BM;
  c.out_col0 = (long long)nt * BN;
  c.split = 0;
  c.blk = 0;
  if (p.mode == MODE_PLAIN) {
    c.a_c0 = 0; c.a_c1 = mt * BM;                               // A K-major
    if (!B_MN) { c.b_c0 = 0; c.b_c1 = nt * BN; }                // B K-major: W [n][m]
    else { c.b_c0 = nt * BN; c.b_c1 = 0; }                      // B MN-major: W [K=n][MN=m]
  } else if (p.mode == MODE_BLOCKDIAG) {
    c.blk = z;
    c.a_c0 = z * p.b; c.a_c1 = mt * BM;
    if (!B_MN) { c.b_c0 = 0; c.b_c1 = z * p.b + nt * BN; }      // G_j rows = output cols
    else { c.b_c0 = nt * BN; c.b_c1 = z * p.b; }                // G_j rows = K
    c.out_col0 = (long long)z * p.b + nt * BN;
  } else {  // MODE_WGRAD: A = X_j (MN-major), B = dY_j (MN-major), K = tokens of the split
    c.blk = z / p.splits;
    c.split = z % p.splits;
    const long long t0 = (long long)c.split * p.kchunk;
    long long tcount = p.ntok - t0;
    if (tcount > p.kchunk) tcount = p.kchunk;
    c.num_kb = tcount > 0 ? (int)((tcount + BK - 1) / BK) : 0;
    c.a_c0 = c.blk * p.b + mt * BM; c.a_c1 = (int)t0;
    c.b_c0 = c.blk * p.b + nt * BN; c.b_c1 = (int)t0;
  }
  return c;
}

// 8 epilogue warps (2..9): two per TMEM lane quarter, each storing half of the BN columns.
constexpr int kEpiWarps = 8;
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;

// Bytes of one pipeline stage: A (bf16) and B (bf16; absent when B is resident; half of it
// in each CTA of a pair).  RES > 0: B is a resident panel of RES 64-wide K blocks.
template <int BN, int RES, int CL = 1>
constexpr int stage_bytes() {
  return BM * BK * 2 + (RES > 0 ? 0 : BN / CL * BK * 2);
}
template <int BN, int RES>
constexpr int res_bytes() { return RES * BN * BK * 2; }

// Columns the epilogue stages per pass: 64, or 32 when the operand ring leaves no room.
template <int BN, int STAGES, bool OUT_F32, int RES, int CL = 1, bool TOUT = false>
constexpr int epi_pass_cols() {
  if (TOUT) return 64;  // dense 32 x 64 bf16 boxes (4 KB per warp)
  constexpr int ring = STAGES * stage_bytes<BN, RES, CL>() + res_bytes<BN, RES>();
  constexpr int esz = OUT_F32 ? 4 : 2;
  constexpr int wc = BN / (kEpiWarps / 4);
  constexpr int c = (wc < 64) ? wc : 64;
  return ring + kEpiWarps * 32 * (c * esz + 16) + 1280 <= 227 * 1024 ? c : 32;
}

// Two signed bytes of w (bytes lo, lo+1) -> two bf16 in one word, exactly and on the full-rate
// ALU: the byte biased by 128 goes under the exponent of 2^23 (byte_perm), one FADD removes
// 2^23 + 128, and the upper halves of the two floats are the bf16 values (an integer of
// magnitude < 256 has at most 8 significant bits).
__device__ __forceinline__ uint32_t i8x2_to_bf16x2(uint32_t w, int lo) {
  const uint32_t u = w ^ 0x80808080u;                       // bias: q + 128 as unsigned bytes
  const uint32_t sel0 = lo == 0 ? 0x7540u : 0x7542u;        // [byte lo, 0, 0, 0x4B]
  const uint32_t sel1 = lo == 0 ? 0x7541u : 0x7543u;        // [byte lo+1, 0, 0, 0x4B]
  const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, sel0)) - 8388736.0f;
  const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, sel1)) - 8388736.0f;
  return __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);
}

// RES > 0 (block-diagonal products): each CTA walks a contiguous range of tiles and keeps the
// B panel of the current (block, column tile) resident in shared memory, so that the ring
// carries only the streamed A tiles; the panel is reloaded when the range crosses into the
// next block (guarded by its own full / empty barriers).
//
// CL = 2 (PLAIN only): 2-CTA pairs (cta_group::2).  A cluster of two CTAs computes a
// 256 x BN tile: each CTA loads its 128 rows of A and its half of the BN rows of B, both
// signalling the even CTA's "full" barrier, and the even CTA's MMA thread issues M = 256
// MMAs that read both CTAs' shared memory and write each CTA's 128 accumulator rows into
// its own TMEM.  Per SM a stage then carries half of B (32 KB instead of 48 KB per K block
// at BN = 256, so 6 stages fit where 4 did), which is what bounded the single-CTA tiles:
// shared memory traffic (TMA writes plus MMA reads), not the tensor pipe.  The MMA commits
// arrive on both CTAs' barriers; both CTAs' epilogue warps release an accumulator on the
// even CTA's "empty" barrier; neither CTA exits before the other has drained what is aimed
// at it.
//
// TOUT (bf16 block-diagonal products): each epilogue warp converts its 32 rows x 64 columns
// into a dense, 128-byte-swizzled shared-memory box (conflict-free: lane = row, 16-byte
// chunk k at k ^ (row % 8)) that one lane stores by TMA through tmC, so the warp moves on to
// the next accumulator while the copy drains; rows past the tensor's end are clipped by the
// TMA unit.
template <int BN, int STAGES, bool A_MN, bool B_MN, bool OUT_F32, int RES, int CL, bool TOUT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const UmmaParams p) {
  constexpr uint32_t A_BYTES = BM * BK * 2;
  constexpr uint32_t B_BYTES = BN * BK * 2;
  constexpr uint32_t STAGE_BYTES = stage_bytes<BN, RES, CL>();
  constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
  constexpr uint32_t IDESC = make_idesc(BM * CL, BN, A_MN, B_MN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // per epilogue warp: 32 rows x 64 columns staging buffer (rows padded by 16 bytes), so
  // that the global stores cover whole row segments instead of 16 bytes of 32 rows each
  constexpr uint32_t ESZ = OUT_F32 ? 4 : 2;
  constexpr int EPC = epi_pass_cols<BN, STAGES, OUT_F32, RES, CL, TOUT>();  // columns per pass
  constexpr uint32_t STG_PITCH = TOUT ? 128 : EPC * ESZ + 16;
  static_assert(!TOUT || (!OUT_F32 && CL == 1 && (BN / (kEpiWarps / 4)) % 64 == 0),
                "TMA-stored epilogue: bf16 output, 64-column passes");
  uint8_t* resb = smem + STAGES * STAGE_BYTES;            // resident B panel (RES > 0)
  uint8_t* staging = resb + res_bytes<BN, RES>();         // EPIW buffers
  constexpr int EPIW = kEpiWarps;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + EPIW * 32 * STG_PITCH);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;  // [2]
  uint64_t* tempty = tfull + 2;      // [2]
  uint64_t* rfull = tempty + 2;      // resident B panel loaded (RES > 0)
  uint64_t* rempty = rfull + 1;      // resident B panel no longer read by MMAs (RES > 0)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rempty + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  static_assert(CL == 1 || (CL == 2 && RES == 0 && BN % 128 == 0), "pairs: PLAIN tiles only");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = CL > 1 ? (int)cluster_ctarank() : 0;
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 0);  // slot 0: CTA start
  pdl_trigger();

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], CL * EPIW);  // pairs: both CTAs' epilogue warps
    }
    mbar_init(rfull, 1);
    mbar_init(rempty, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if (CL > 1) {  // one warp of each CTA of the pair, same columns in both
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0 && p.bpre) {
    // this CTA's share of the weight operand into L2 (a prefetch returns no data, so it is
    // safe before the wait even if the bytes were still being written)
    const unsigned long long share =
        ((p.bpre_bytes + gridDim.x - 1) / gridDim.x + 4095) & ~4095ull;
    const unsigned long long lo = (unsigned long long)blockIdx.x * share;
    for (unsigned long long off = lo; off < lo + share && off < p.bpre_bytes; off += 32768) {
      unsigned long long n = p.bpre_bytes - off;
      n = n < 32768 ? n : 32768;
      if (off + n > lo + share) n = lo + share - off;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.bpre + off),
                   "r"((uint32_t)(n & ~15ull))
                   : "memory");
    }
  }
  tc_fence_before();
  if (CL > 1) cluster_sync();  // the peer's barriers exist before anything is aimed at them
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);
  pdl_wait();  // the previous kernel's outputs are visible from here on
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 1);  // slot 1: set-up done
  // tiles of this CTA: strided (t = blockIdx.x, + gridDim.x, ...) or, with a resident B
  // panel, one contiguous range
  const int t_first = RES > 0 ? (int)((long long)blockIdx.x * p.num_tiles / gridDim.x)
                              : (int)blockIdx.x / CL;
  const int t_end = RES > 0 ? (int)((long long)(blockIdx.x + 1) * p.num_tiles / gridDim.x) : p.num_tiles;
  const int t_step = RES > 0 ? 1 : (int)gridDim.x / CL;
  auto panel_key = [](const TileCoords& c) -> long long {
    return ((long long)c.b_c0 << 32) | (unsigned)c.b_c1;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    long long g = 0;  // k blocks issued by this CTA (ring position)
    bool ok = true;
    long long cur_key = -1;
    int npanels = 0;
    for (int t = t_first; t < t_end && ok; t += t_step) {
      const TileCoords c = tile_coords<BN, B_MN, CL>(p, t, crank);
      if (RES > 0 && panel_key(c) != cur_key) {
        // the previous panel must be free (all MMAs that read it completed) before reloading
        if (npanels > 0 &&
            (*abort_flag || !mbar_wait_bounded(rempty, (npanels - 1) & 1, p.err, p.limit_ns, kSite + __LINE__))) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(rfull, RES * B_BYTES);
#pragma unroll 1
        for (int kb = 0; kb < RES; ++kb) {
          uint8_t* dst = resb + kb * B_BYTES;
          if (!B_MN) {
            tma_load_2d(dst, &tmB, rfull, c.b_c0 + kb * BK, c.b_c1);
          } else {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(dst + i * 8192, &tmB, rfull, c.b_c0 + 64 * i, c.b_c1 + kb * BK);
          }
        }
        cur_key = panel_key(c);
        ++npanels;
      }
      for (int kb = 0; kb < c.num_kb; ++kb, ++g) {
        const int s = (int)(g % STAGES);
        const uint32_t ph = (uint32_t)((g / STAGES) & 1);
        if (*abort_flag || !mbar_wait_bounded(&empty[s], ph ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        if (g == 0) trace_stamp(p.trace, p.trace_cap, 2);  // slot 2: first TMA issued
        uint8_t* sa = smem + s * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        const int k = kb * BK;
        if (CL > 1) {
          // this CTA's A rows and half of B, completing on the even CTA's barrier
          if (crank == 0) mbar_arrive_expect_tx(&full[s], CL * STAGE_BYTES);
          const uint32_t fb = mapa_shared(&full[s], 0);
          tma_load_2d_pair(sa, &tmA, fb, c.a_c0 + k, c.a_c1);
          if (!B_MN) {
            tma_load_2d_pair(sb, &tmB, fb, c.b_c0 + k, c.b_c1 + crank * (BN / 2));
          } else {
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              tma_load_2d_pair(sb + j * 8192, &tmB, fb, c.b_c0 + 64 * (crank * (BN / 128) + j),
                               c.b_c1 + k);
          }
          continue;
        }
        mbar_arrive_expect_tx(&full[s], RES > 0 ? A_BYTES : STAGE_BYTES);
        if (!A_MN) {
          tma_load_2d(sa, &tmA, &full[s], c.a_c0 + k, c.a_c1);
        } else {
#pragma unroll
          for (int i = 0; i < BM / 64; ++i)
            tma_load_2d(sa + i * 8192, &tmA, &full[s], c.a_c0 + 64 * i, c.a_c1 + k);
        }
        if (RES == 0) {
          if (!B_MN) {
            tma_load_2d(sb, &tmB, &full[s], c.b_c0 + k, c.b_c1);
          } else {
            constexpr int BOX_BYTES = 8192;  // 64 x 64 elements
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sb + i * BOX_BYTES, &tmB, &full[s], c.b_c0 + 64 * i, c.b_c1 + k);
          }
        }
      }
    }
    // a resident panel still loading must land before the CTA may exit
    if (RES > 0 && npanels > 0) mbar_wait_bounded(rfull, (npanels - 1) & 1, p.err, p.limit_ns, kSite + __LINE__);
    // Drain: wait for the last load issued into every stage (already complete in the normal
    // path), so that no copy is in flight when the CTA exits.
    // (Pairs: the loads complete on the even CTA's barriers, so wait instead until the MMAs
    // have released the last stages, which they do only after reading them.)
    for (long long j = g - 1; j >= 0 && j >= g - STAGES; --j)
      mbar_wait_bounded(CL > 1 ? &empty[j % STAGES] : &full[j % STAGES],
                        (uint32_t)((j / STAGES) & 1), p.err, p.limit_ns, kSite + __LINE__);
  } else if (warp == 1 && lane == 0 && crank == 0) {
    // ------------------------------------------------------------ MMA issuer
    long long g = 0;
    int it = 0;
    bool ok = true;
    long long cur_key = -1;
    int npanels = 0;
    for (int t = t_first; t < t_end && ok; t += t_step, ++it) {
      const TileCoords c = tile_coords<BN, B_MN, CL>(p, t, crank);
      const int a = it & 1;
      if (*abort_flag || !mbar_wait_bounded(&tempty[a], ((it >> 1) & 1) ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        break;
      }
      if (RES > 0 && panel_key(c) != cur_key) {
        if (npanels > 0) umma_commit(rempty);  // the old panel is free once these MMAs finish
        if (*abort_flag || !mbar_wait_bounded(rfull, npanels & 1, p.err, p.limit_ns, kSite + __LINE__)) {
          *abort_flag = 1;
          break;
        }
        cur_key = panel_key(c);
        ++npanels;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(a * BN);
      for (int kb = 0; kb < c.num_kb; ++kb, ++g) {
        const int s = (int)(g % STAGES);
        const uint32_t ph = (uint32_t)((g / STAGES) & 1);
        if (*abort_flag || !mbar_wait_bounded(&full[s], ph, p.err, p.limit_ns, kSite + __LINE__)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        if (g == 0) trace_stamp(p.trace, p.trace_cap, 3);  // slot 3: first stage landed
        const uint32_t a_base = smem_base + s * STAGE_BYTES;
        const uint32_t b_base = RES > 0 ? smem_u32(resb) + kb * B_BYTES : a_base + A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          if (CL > 1)
            umma_bf16_pair(d, tile_desc<A_MN>(a_base, k), tile_desc<B_MN>(b_base, k), IDESC,
                           (kb | k) != 0);
          else
            umma_bf16(d, tile_desc<A_MN>(a_base, k), tile_desc<B_MN>(b_base, k), IDESC,
                      (kb | k) != 0);
        if (CL > 1) umma_commit_pair(&empty[s]);
        else umma_commit(&empty[s]);
      }
      // also when the tile had no K block (empty token split)
      if (CL > 1) umma_commit_pair(&tfull[a]);
      else umma_commit(&tfull[a]);
    }
    // TMEM is freed after the final barrier: wait until the last MMAs have completed.
    if (it > 0) {
      const int last = it - 1;
      mbar_wait_bounded(&tfull[last & 1], (last >> 1) & 1, p.err, p.limit_ns, kSite + __LINE__);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                   // TMEM lane quarter = output rows
    constexpr int WCOLS = BN / (EPIW / 4);    // columns handled by this warp
    const int cbeg = ((warp - 2) >> 2) * WCOLS;
    const int row = q * 32 + lane;
    int it = 0;
    for (int t = t_first; t < t_end; t += t_step, ++it) {
      const TileCoords c = tile_coords<BN, B_MN, CL>(p, t, crank);
      const int a = it & 1;
      const bool ok = !*abort_flag && mbar_wait_bounded(&tfull[a], (it >> 1) & 1, p.err, p.limit_ns, kSite + __LINE__);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (warp == 2 && lane == 0 && it < 12) trace_stamp(p.trace, p.trace_cap, 5 + 2 * it);  // acc ready
      uint8_t* stg = staging + (warp - 2) * 32 * STG_PITCH;
      const long long row0 = c.out_row0 + q * 32;  // first output row of this warp
#pragma unroll 1
      for (int c0 = cbeg; c0 < cbeg + WCOLS; c0 += EPC) {
        // the contraction's last tile column may reach past the output width (a multiple of
        // 64, so a pass is wholly inside or outside): nothing to store there
        if (p.mode == MODE_PLAIN && c.out_col0 + c0 >= p.ldc) continue;
        // one or two 32-column TMEM loads, one wait
        uint32_t r[64];
        if (c.num_kb > 0) {
          const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN + c0);
          tmem_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(r));
          if (EPC >= 64) tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) r[i] = 0u;
        }
        const int ncol = EPC;  // columns in this pass
        // lane = row: write its values into the staging rows
        if (OUT_F32) {
          float4* dst = reinterpret_cast<float4*>(stg + lane * STG_PITCH);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (4 * i < ncol)
              dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                   __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        } else {
          float v[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
          if (p.colscale) {
#pragma unroll
            for (int i = 0; i < 64; ++i)
              if (i < ncol) v[i] *= __ldg(p.colscale + c.out_col0 + c0 + i);
          }
          if (TOUT) {
            // the previous pass's box must have been read by its TMA store
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                             pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, stg, (int)(c.out_col0 + c0), (int)row0);
              bulk_commit();
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(stg + lane * STG_PITCH);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (8 * i < ncol)
                dst[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                                    pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
          }
        }
        if (TOUT) continue;  // stored by TMA above
        __syncwarp();
        // lanes cover whole row segments: (ncol * ESZ / 16) lanes per row
        const int per_row = ncol * (int)ESZ / 16;
        const int rows_per_pass = 32 / per_row;
        const int pr = lane / per_row, pc = lane % per_row;
        for (int rr = pr; rr < 32; rr += rows_per_pass) {
          const long long grow = row0 + rr;
          if (grow >= p.M) continue;
          const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * STG_PITCH + pc * 16);
          uint8_t* gdst;
          if (OUT_F32)
            gdst = reinterpret_cast<uint8_t*>(static_cast<float*>(p.C) +
                   (((long long)c.split * p.nblk + c.blk) * p.b + grow) * p.b + c.out_col0 + c0);
          else if (p.out_perm)
            gdst = nullptr;
          else
            gdst = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.C) + grow * p.ldc +
                                              c.out_col0 + c0);
          if (gdst) {
            *reinterpret_cast<uint4*>(gdst + pc * 16) = val;
          } else {  // fused output permutation: scattered 2-byte stores
            __nv_bfloat16* rowp = static_cast<__nv_bfloat16*>(p.C) + grow * p.ldc;
            const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&val);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              rowp[__ldg(p.out_perm + c.out_col0 + c0 + pc * 8 + i)] = e[i];
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CL > 1) mbar_arrive_cluster(mapa_shared(&tempty[a], 0));
        else mbar_arrive(&tempty[a]);
      }
      if (warp == 2 && lane == 0 && it < 12) trace_stamp(p.trace, p.trace_cap, 4 + 2 * it);  // tile stored
    }
  }
  if (warp == 2 && lane == 0) trace_stamp(p.trace, p.trace_cap, 30);  // epilogue loop done
  if (TOUT && warp >= 2 && lane == 0) bulk_wait_all();  // this warp's stores have landed
  tc_fence_before();
  if (CL > 1) cluster_sync();
  else __syncthreads();
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 31);  // slot 31: exit
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (CL > 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}


// ---------------------------------------------------------------- fused W' + block product
// The W' contraction with the block-diagonal product that follows it done on the same tile
// (POET-X summary page, "Core method" section 1: b = W' a, z = G_P^T b; and the backward's
// dA = dB W', dx~ = dA G_R^T): a 128 x 256 tile of the first product is complete in TMEM after
// its K loop; the epilogue rounds it to bf16 into a shared-memory operand tile (and stores it
// when the caller keeps it), a second round of MMAs multiplies that tile by the G blocks
// covering its 256 columns (b = 64, 128 or 256 divides 256), and the epilogue stores the
// result.  This removes one pass over the [N, D] activations.
//   forward:  C1 = A W'^T (W' K-major), C2[:, jb..] = C1[:, jb..] G_j       (G MN-major)
//   backward: C1 = A W' (W' MN-major),  C2[:, jb..] = C1[:, jb..] G_j^T     (G K-major)
// Ring order (one producer, one MMA thread): the K blocks of tile i, then the four G blocks of
// tile i-1, so that the second product of a tile is issued while the epilogue of the next
// one is not yet needed and the tensor pipe never waits for the epilogue.  The shared-memory
// operand tile doubles as each epilogue warp's staging area (every warp owns 32 rows x 128
// columns of it).
struct FusedParams {
  int M;                      // valid token rows
  int tiles_m, num_tiles;     // tile t: mt = t % tiles_m, nt = t / tiles_m
  int num_kb;                 // 64-wide K blocks of the first product
  int b;                      // block size of the second product
  long long ldc;              // columns of C1 and C2
  __nv_bfloat16* C1;          // nullable: first product not stored
  __nv_bfloat16* C2;
  const uint8_t* bpre;
  unsigned long long bpre_bytes;
  unsigned long long* trace;
  size_t trace_cap;
  int* err;
  unsigned long long limit_ns;
};

constexpr int FZ_BN = 256;
constexpr int FZ_STAGES = 3;
constexpr uint32_t FZ_A_BYTES = BM * BK * 2;                 // 16 KB
constexpr uint32_t FZ_STAGE = FZ_A_BYTES + FZ_BN * BK * 2;   // 48 KB
constexpr uint32_t FZ_A2_SUB = BM * BK * 2;                  // one 64-column sub-tile: 16 KB
constexpr uint32_t FZ_A2 = FZ_BN / BK * FZ_A2_SUB;           // 64 KB
constexpr int FZ_SMEM = FZ_STAGES * FZ_STAGE + FZ_A2 + 1024 + 512;
static_assert(FZ_SMEM <= 227 * 1024, "fused W' kernel: shared memory");

// byte offset of row r, 16-byte chunk c of a 128 x 64 bf16 K-major tile (128-byte swizzle)
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <bool W_MN, bool G_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_fused_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmG, const FusedParams p) {
  constexpr uint32_t IDESC1 = make_idesc(BM, FZ_BN, false, W_MN);
  constexpr uint32_t TMEM_COLS = 2 * FZ_BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* a2 = smem + FZ_STAGES * FZ_STAGE;  // the second product's A operand / staging
  uint64_t* full = reinterpret_cast<uint64_t*>(a2 + FZ_A2);
  uint64_t* empty = full + FZ_STAGES;
  uint64_t* tfull1 = empty + FZ_STAGES;  // [2] first product of the tile in TMEM
  uint64_t* tfull2 = tfull1 + 2;         // [2] second product in TMEM
  uint64_t* tempty = tfull2 + 2;         // [2] accumulator drained
  uint64_t* a2full = tempty + 2;         // operand tile written by every epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(a2full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 0);
  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < FZ_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull1[a], 1);
      mbar_init(&tfull2[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(a2full, kEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmG);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0 && p.bpre) {  // this CTA's share of W' into L2
    const unsigned long long share =
        ((p.bpre_bytes + gridDim.x - 1) / gridDim.x + 4095) & ~4095ull;
    const unsigned long long lo = (unsigned long long)blockIdx.x * share;
    for (unsigned long long off = lo; off < lo + share && off < p.bpre_bytes; off += 32768) {
      unsigned long long n = p.bpre_bytes - off;
      n = n < 32768 ? n : 32768;
      if (off + n > lo + share) n = lo + share - off;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.bpre + off),
                   "r"((uint32_t)(n & ~15ull))
                   : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t a2_base = smem_u32(a2);
  pdl_wait();
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 1);
  const int b = p.b;
  const uint32_t g2_bytes = (uint32_t)b * BK * 2;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    long long g = 0;
    bool ok = true;
    auto slot = [&](uint32_t bytes, uint8_t*& st) -> bool {
      const int s = (int)(g % FZ_STAGES);
      const uint32_t ph = (uint32_t)((g / FZ_STAGES) & 1);
      if (*abort_flag || !mbar_wait_bounded(&empty[s], ph ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        return false;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      st = smem + s * FZ_STAGE;
      return true;
    };
    // the G blocks covering the 256 columns of tile column nt (K of the second product)
    auto issue_g2 = [&](int nt) -> bool {
      for (int kb2 = 0; kb2 < FZ_BN / BK; ++kb2, ++g) {
        uint8_t* st;
        if (!slot(g2_bytes, st)) return false;
        const int col = nt * FZ_BN + kb2 * BK;  // first column of the K block
        const int j = col / b, r0 = col % b;
        uint8_t* sb = st + FZ_A_BYTES;
        if (G_MN) {  // rows r0.. of G_j, all b columns: b/64 boxes of 64 x 64
          for (int i = 0; i < b / 64; ++i)
            tma_load_2d(sb + i * 8192, &tmG, &full[(int)(g % FZ_STAGES)], 64 * i, j * b + r0);
        } else {     // all b rows of G_j, columns r0..: one box of 64 x b
          tma_load_2d(sb, &tmG, &full[(int)(g % FZ_STAGES)], r0, j * b);
        }
      }
      return true;
    };
    int prev_nt = -1;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const int mt = t % p.tiles_m, nt = t / p.tiles_m;
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        uint8_t* st;
        if (!slot(FZ_STAGE, st)) {
          ok = false;
          break;
        }
        if (g == 0) trace_stamp(p.trace, p.trace_cap, 2);
        uint64_t* fb = &full[(int)(g % FZ_STAGES)];
        tma_load_2d(st, &tmA, fb, kb * BK, mt * BM);
        if (!W_MN) {
          tma_load_2d(st + FZ_A_BYTES, &tmW, fb, kb * BK, nt * FZ_BN);
        } else {
#pragma unroll
          for (int i = 0; i < FZ_BN / 64; ++i)
            tma_load_2d(st + FZ_A_BYTES + i * 8192, &tmW, fb, nt * FZ_BN + 64 * i, kb * BK);
        }
      }
      if (!ok) break;
      if (prev_nt >= 0 && !issue_g2(prev_nt)) {
        ok = false;
        break;
      }
      prev_nt = nt;
    }
    if (ok && prev_nt >= 0) issue_g2(prev_nt);
    for (long long j = g - 1; j >= 0 && j >= g - FZ_STAGES; --j)
      mbar_wait_bounded(&full[j % FZ_STAGES], (uint32_t)((j / FZ_STAGES) & 1), p.err, p.limit_ns,
                        kSite + __LINE__);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    long long g = 0;
    bool ok = true;
    auto take = [&](int& s) -> bool {
      s = (int)(g % FZ_STAGES);
      const uint32_t ph = (uint32_t)((g / FZ_STAGES) & 1);
      if (*abort_flag || !mbar_wait_bounded(&full[s], ph, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        return false;
      }
      tc_fence_after();
      return true;
    };
    // second product of the tile with index i (its accumulator holds the first product,
    // already read out into the operand tile by the epilogue)
    auto mma2 = [&](int i) -> bool {
      const int a = i & 1;
      if (*abort_flag || !mbar_wait_bounded(a2full, (uint32_t)(i & 1), p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        return false;
      }
      tc_fence_after();
      const uint32_t idesc2 = make_idesc(BM, b, false, G_MN);
      for (int kb2 = 0; kb2 < FZ_BN / BK; ++kb2, ++g) {
        int s;
        if (!take(s)) return false;
        const int lb = kb2 * BK / b, kk = kb2 * BK % b;  // block within the tile, K offset
        const uint32_t d = tmem_base + (uint32_t)(a * FZ_BN + lb * b);
        const uint32_t bb = smem_base + s * FZ_STAGE + FZ_A_BYTES;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_bf16(d, tile_desc<false>(a2_base + kb2 * FZ_A2_SUB, k), tile_desc<G_MN>(bb, k),
                    idesc2, (kk | k) != 0);
        umma_commit(&empty[s]);
      }
      umma_commit(&tfull2[a]);
      return true;
    };
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++it) {
      const int a = it & 1;
      if (*abort_flag ||
          !mbar_wait_bounded(&tempty[a], ((it >> 1) & 1) ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(a * FZ_BN);
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        int s;
        if (!take(s)) {
          ok = false;
          break;
        }
        if (g == 0) trace_stamp(p.trace, p.trace_cap, 3);
        const uint32_t sa = smem_base + s * FZ_STAGE;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_bf16(d, tile_desc<false>(sa, k), tile_desc<W_MN>(sa + FZ_A_BYTES, k), IDESC1,
                    (kb | k) != 0);
        umma_commit(&empty[s]);
      }
      if (!ok) break;
      umma_commit(&tfull1[a]);
      if (it > 0 && !mma2(it - 1)) {
        ok = false;
        break;
      }
    }
    if (ok && it > 0) mma2(it - 1);
    if (it > 0) mbar_wait_bounded(&tfull2[(it - 1) & 1], ((it - 1) >> 1) & 1, p.err, p.limit_ns,
                                  kSite + __LINE__);
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    // warp w: rows 32 (w % 4) .. +31 of the tile, columns 128 h .. +127 (h = (w - 2) / 4),
    // i.e. the operand tile's 64-column sub-tiles 2h and 2h + 1 for those rows
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    // TMEM (64 columns from column c of accumulator a, this warp's lanes) -> bf16 -> the
    // operand tile's sub-tile kb2, row r
    auto to_tile = [&](int a, int kb2) {
      uint32_t v[64];
      const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * FZ_BN + kb2 * BK);
      tmem_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      uint8_t* sub = a2 + kb2 * FZ_A2_SUB;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sub + sw128_off(r, c)) =
            make_uint4(pack_bf16x2(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1])),
                       pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                       pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                       pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
    };
    // this warp's 32 rows x 128 columns of the operand tile -> global (8 lanes per 128-byte
    // row segment, 4 rows per pass)
    auto store = [&](__nv_bfloat16* C, long long row0, long long col0) {
      const int rr0 = lane >> 3, c = lane & 7;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int kb2 = 2 * h + u;
        const uint8_t* sub = a2 + kb2 * FZ_A2_SUB;
#pragma unroll 2
        for (int rr = rr0; rr < 32; rr += 4) {
          const int rt = q * 32 + rr;
          const long long grow = row0 + rt;
          if (grow >= p.M) continue;
          const uint4 val = *reinterpret_cast<const uint4*>(sub + sw128_off(rt, c));
          *reinterpret_cast<uint4*>(C + grow * p.ldc + col0 + kb2 * BK + c * 8) = val;
        }
      }
    };
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const int a = it & 1;
      const long long row0 = (long long)(t % p.tiles_m) * BM;
      const long long col0 = (long long)(t / p.tiles_m) * FZ_BN;
      bool ok = !*abort_flag && mbar_wait_bounded(&tfull1[a], (it >> 1) & 1, p.err, p.limit_ns,
                                                  kSite + __LINE__);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      to_tile(a, 2 * h);
      to_tile(a, 2 * h + 1);
      fence_async_shared();  // generic writes -> visible to the tensor cores
      __syncwarp();
      if (p.C1) store(p.C1, row0, col0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a2full);
      ok = !*abort_flag && mbar_wait_bounded(&tfull2[a], (it >> 1) & 1, p.err, p.limit_ns,
                                             kSite + __LINE__);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      to_tile(a, 2 * h);  // the second product, staged in the same rows and columns
      to_tile(a, 2 * h + 1);
      __syncwarp();
      store(p.C2, row0, col0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      if (warp == 2 && lane == 0 && it < 12) trace_stamp(p.trace, p.trace_cap, 4 + 2 * it);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 31);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- int8 W' contraction
// With an int8 W' the contraction runs transposed: D[f, t] = sum_k W(f, k) act[t, k] for
// output feature f and token t, so that the widened weight is the A operand, which tcgen05
// reads from tensor memory: converter warps widen the raw int8 tile (exactly, byte-permute
// construction) straight into TMEM, and shared memory carries only the raw weight tile and
// the bf16 activation tile (the B operand).  Forward: W(f, k) = Wq[f][k], out[t][f] =
// s_f D[f, t]; backward: W(f, k) = Wq[k][f] (the activation was scaled by s beforehand),
// out[t][f] = D[f, t].  Tiles: 128 features x I8T = 384 tokens, K blocks of 64; a 3-deep
// shared-memory ring, one TMEM accumulator of 384 columns and a ring of 4 A slots of 32
// TMEM columns.  Widening a weight tile takes about as long as the MMAs of 192 tokens
// (measured), so each widened tile feeds as many tokens as TMEM holds: 384 (two MMAs of
// N = 192 per K step) instead of 192 with two accumulators, which halves the widening per
// flop at the price of an epilogue that no longer overlaps the next tile's MMAs.  Tiles are
// numbered token-fastest, so that the CTAs running at the same time share a few weight
// tiles (read from DRAM about once) and read the activations from L2.
//   warp 0      TMA: raw weight tile (fwd: 128 rows x 64 bytes; bwd: 64 rows x 128 bytes)
//               and the activation tile (2 x 192 rows x 64 bf16, 128-byte swizzle)
//   warp 1      MMA issuer: 2 x 4 tcgen05.mma kind::f16 (K = 16) per K block, A from TMEM
//   warps 2-13  converters, three groups of four taking every third K block: warp w
//               widens the 64 K values of lane quarter w % 4 (rows 32 (w % 4) .. +31)
//   warps 14-17 epilogue: lane quarter w % 4, all I8T tokens, through a transposing tile
constexpr int I8N = 192;          // tokens per MMA (and per TMA box of the activation tile)
constexpr int I8_NSUB = 2;        // MMAs per K step sharing the widened weight slot
constexpr int I8T = I8N * I8_NSUB;  // tokens per tile
constexpr int I8_STAGES = 3;      // shared-memory ring (raw weight + activation tiles)
constexpr int I8_ASLOTS = 4;      // TMEM ring of widened weight tiles
constexpr int I8_CONVG = 3;       // converter groups (four warps each), one per ring stage:
                                  // a group takes the K blocks g with g % I8_CONVG == its
                                  // index, so each stage's "full" barrier is waited on by one
                                  // group only.  (With groups sharing a stage, a group could
                                  // reach the stage's next-but-one phase while the other
                                  // group's phase is still in flight, and the parity wait
                                  // would take the old phase for the new one.)
constexpr int I8_CONVW = 4 * I8_CONVG;
static_assert(I8_STAGES % I8_CONVG == 0, "each ring stage belongs to one converter group");
constexpr int I8_EPIW = 4;
constexpr int I8_THREADS = 32 * (2 + I8_CONVW + I8_EPIW);
constexpr uint32_t I8_W_BYTES = 128 * 64;          // raw weight tile
constexpr uint32_t I8_X_BYTES = I8T * BK * 2;      // activation tile
constexpr uint32_t I8_STAGE = I8_X_BYTES + I8_W_BYTES;
constexpr int I8_STG_PITCH = 80;                   // 32 features x 2 bytes + 16 (conflict-free)
constexpr int I8_SMEM = I8_STAGES * I8_STAGE + I8_EPIW * 32 * I8_STG_PITCH + 1024 + 512;

struct I8Params {
  int tiles_f, tiles_t, num_tiles;  // tile t: tt = t % tiles_t, ft = t / tiles_t
  int num_kb;
  long long ntok;                   // tokens
  int nfeat;                        // output features
  int trans;                        // 0: forward, 1: backward (weight read transposed)
  const float* scale;               // forward: s_f (nullable)
  __nv_bfloat16* C;                 // [ntok][nfeat]
  unsigned long long* trace;
  size_t trace_cap;
  int* err;
  unsigned long long limit_ns;
};

__global__ void __launch_bounds__(I8_THREADS, 1)
    umma_i8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const I8Params p) {
  constexpr uint32_t ACC_COLS = I8T;           // the accumulator (I8_NSUB x I8N columns)
  constexpr uint32_t A_COL = ACC_COLS;         // A slots: A_COL + 32 j
  constexpr uint32_t TMEM_COLS = 512;
  static_assert(A_COL + 32 * I8_ASLOTS <= TMEM_COLS, "accumulator and A slots fit TMEM");
  constexpr uint32_t IDESC = make_idesc(BM, I8N, false, false);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* staging = smem + I8_STAGES * I8_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(staging + I8_EPIW * 32 * I8_STG_PITCH);
  uint64_t* empty = full + I8_STAGES;
  uint64_t* conv = empty + I8_STAGES;   // [I8_ASLOTS] slot holds the widened tile of a block
  uint64_t* afree = conv + I8_ASLOTS;   // [I8_ASLOTS] slot no longer read by MMAs
  uint64_t* tfull = afree + I8_ASLOTS;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 0);
  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < I8_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < I8_ASLOTS; ++j) {
      mbar_init(&conv[j], 4);  // the four warps of the K block's converter group
      mbar_init(&afree[j], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, I8_EPIW);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
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
  pdl_wait();
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 1);

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    long long g = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const int f0 = (t / p.tiles_t) * BM, t0 = (t % p.tiles_t) * I8T;
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        const int s = (int)(g % I8_STAGES);
        const uint32_t ph = (uint32_t)((g / I8_STAGES) & 1);
        if (*abort_flag || !mbar_wait_bounded(&empty[s], ph ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], I8_STAGE);
        // (diagnostic stamps cover 8 K blocks from the middle of the first tile)
        if (g - p.num_kb / 2 >= 0 && g - p.num_kb / 2 < 8)
          trace_stamp(p.trace, p.trace_cap, 2 + (int)(g - p.num_kb / 2));  // slots 2..9: issued
        uint8_t* sx = smem + s * I8_STAGE;
        uint8_t* sw = sx + I8_X_BYTES;
#pragma unroll
        for (int h = 0; h < I8_NSUB; ++h)  // tokens t0 + h I8N.., K columns kb*64..
          tma_load_2d(sx + h * I8N * 128, &tmX, &full[s], kb * BK, t0 + h * I8N);
        if (!p.trans)
          tma_load_2d(sw, &tmW, &full[s], kb * BK, f0);  // rows f0.. of Wq, K bytes kb*64..
        else
          tma_load_2d(sw, &tmW, &full[s], f0, kb * BK);  // rows kb*64.. of Wq, bytes f0..
      }
    }
    for (long long j = g - 1; j >= 0 && j >= g - I8_STAGES; --j)
      mbar_wait_bounded(&full[j % I8_STAGES], (uint32_t)((j / I8_STAGES) & 1), p.err, p.limit_ns, kSite + __LINE__);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    long long g = 0;
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++it) {
      // one accumulator: the epilogue of the previous tile must have drained it
      if (*abort_flag || !mbar_wait_bounded(tempty, (it & 1) ^ 1, p.err, p.limit_ns, kSite + __LINE__)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base;
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        const int s = (int)(g % I8_STAGES);
        const int j = (int)(g % I8_ASLOTS);
        if (*abort_flag ||
            !mbar_wait_bounded(&conv[j], (uint32_t)((g / I8_ASLOTS) & 1), p.err, p.limit_ns, kSite + __LINE__)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        if (g - p.num_kb / 2 >= 0 && g - p.num_kb / 2 < 8)
          trace_stamp(p.trace, p.trace_cap, 18 + (int)(g - p.num_kb / 2));  // 18..25: MMAs
        const uint32_t xa = smem_base + s * I8_STAGE;
        const uint32_t wa = tmem_base + A_COL + 32u * (uint32_t)j;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)  // K = 16 per MMA: 8 TMEM columns of A
#pragma unroll
          for (int h = 0; h < I8_NSUB; ++h)
            umma_bf16_ta(d + h * I8N, wa + 8 * k, tile_desc<false>(xa + h * I8N * 128, k), IDESC,
                         (kb | k) != 0);
        umma_commit(&empty[s]);
        if (I8_ASLOTS < I8_STAGES) umma_commit(&afree[j]);
      }
      umma_commit(tfull);
    }
    if (it > 0) mbar_wait_bounded(tfull, (it - 1) & 1, p.err, p.limit_ns, kSite + __LINE__);
  } else if (warp >= 2 && warp < 2 + I8_CONVW) {
    // ---------------------------------------------------------------- converters
    // group cg = (w - 2) / 4 takes the K blocks g with g % I8_CONVG == cg; warp w widens row
    // f = 32 (w % 4) + lane of the A operand: 64 int8 values -> 32 bf16 pairs -> TMEM slot
    // g % I8_ASLOTS (|q| <= 127: exact)
    const int q = warp & 3, cg = (warp - 2) >> 2;
    const int f = q * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    long long g = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      for (int kb = 0; kb < p.num_kb; ++kb, ++g) {
        if ((int)(g % I8_CONVG) != cg) continue;
        const int s = (int)(g % I8_STAGES);
        const int j = (int)(g % I8_ASLOTS);
        bool got = !*abort_flag &&
                   mbar_wait_bounded(&full[s], (uint32_t)((g / I8_STAGES) & 1), p.err, p.limit_ns, kSite + __LINE__);
        // the slot's previous tile must have been read by its MMAs (implied by the ring when
        // it is no deeper than the slots: the stage was refilled only after those MMAs)
        if (I8_ASLOTS < I8_STAGES && got && g >= I8_ASLOTS)
          got = mbar_wait_bounded(&afree[j], (uint32_t)(((g / I8_ASLOTS) - 1) & 1), p.err,
                                  p.limit_ns, kSite + __LINE__);
        if (!__all_sync(0xffffffffu, got)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* raw = smem + s * I8_STAGE + I8_X_BYTES;
        uint32_t w[32];
        if (!p.trans) {  // row f: 64 contiguous bytes
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(raw + f * 64 + 16 * c);
            const uint32_t bt[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              w[8 * c + 2 * i] = i8x2_to_bf16x2(bt[i], 0);
              w[8 * c + 2 * i + 1] = i8x2_to_bf16x2(bt[i], 2);
            }
          }
        } else {  // column f of 64 rows of 128 bytes
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t lo = raw[(2 * i) * 128 + f];
            const uint32_t hi = raw[(2 * i + 1) * 128 + f];
            w[i] = i8x2_to_bf16x2(lo | (hi << 8), 0);
          }
        }
        const uint32_t col = A_COL + 32u * (uint32_t)j;
        tmem_st_32x32b_x16(lane_base + col, *reinterpret_cast<const uint32_t(*)[16]>(w));
        tmem_st_32x32b_x16(lane_base + col + 16, *reinterpret_cast<const uint32_t(*)[16]>(w + 16));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[j]);
        if (q == 2 && lane == 0 && g - p.num_kb / 2 >= 0 && g - p.num_kb / 2 < 8)
          trace_stamp(p.trace, p.trace_cap, 10 + (int)(g - p.num_kb / 2));  // 10..17: converted
      }
    }
  } else if (warp >= 2 + I8_CONVW) {
    // ---------------------------------------------------------------- epilogue
    // lane = feature f of quarter q; per 32-token chunk: TMEM -> scaled bf16 -> transposing
    // tile [token][feature] -> each lane stores one token row of 32 features (64 bytes)
    const int q = warp & 3;
    uint8_t* stg = staging + (warp - 2 - I8_CONVW) * 32 * I8_STG_PITCH;
    int it = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++it) {
      const int f0 = (t / p.tiles_t) * BM + q * 32;
      const long long t0 = (long long)(t % p.tiles_t) * I8T;
      const bool ok = !*abort_flag && mbar_wait_bounded(tfull, it & 1, p.err, p.limit_ns, kSite + __LINE__);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const float sc = (p.scale && f0 + lane < p.nfeat) ? __ldg(p.scale + f0 + lane) : 1.f;
#pragma unroll 1
      for (int c0 = 0; c0 < I8T; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, r);
        tmem_ld_wait();
        // lane f: token j of the chunk at row j, column f of the tile
#pragma unroll
        for (int j = 0; j < 32; ++j)
          *reinterpret_cast<__nv_bfloat16*>(stg + j * I8_STG_PITCH + lane * 2) =
              __float2bfloat16_rn(__uint_as_float(r[j]) * sc);
        __syncwarp();
        const long long tok = t0 + c0 + lane;
        if (tok < p.ntok && f0 < p.nfeat) {  // (the last feature tile may be half full)
          const uint4* src = reinterpret_cast<const uint4*>(stg + lane * I8_STG_PITCH);
          uint4* dst = reinterpret_cast<uint4*>(p.C + tok * p.nfeat + f0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = src[i];
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      if (q == 2 && lane == 0 && it < 4) trace_stamp(p.trace, p.trace_cap, 26 + it);  // tile stored
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_stamp(p.trace, p.trace_cap, 31);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_map_t(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer, bool i8) {
  return i8 ? encode_tma_2d(m, ptr, TMA_U8, inner, outer, pitch_elems, box_inner, box_outer, false)
            : encode_tma_2d(m, ptr, TMA_BF16, inner, outer, pitch_elems, box_inner, box_outer, true);
}

// 2-D bf16 tensor [outer][inner] with row pitch `pitch_elems`, box {box_inner, box_outer},
// 128-byte swizzle, zero fill out of bounds (encoded maps are cached per thread).
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t pitch_elems,
              uint32_t box_inner, uint32_t box_outer) {
  return make_map_t(m, ptr, inner, outer, pitch_elems, box_inner, box_outer, false);
}

// CL = 2: tiles_m counts pairs of M tiles (see tile_coords).
// TOUT: the output is stored by TMA through tc (a bf16 [rows][columns] map with 32 x 64 boxes
// and the 128-byte swizzle); otherwise tc is not read.
template <int BN, int STAGES, bool A_MN, bool B_MN, bool OUT_F32, int RES = 0, int CL = 1,
          bool TOUT = false>
poetx_status launch(const CUtensorMap& ta, const CUtensorMap& tb, UmmaParams p, int tiles_m,
                    int tiles_n, int tiles_z, cudaStream_t s, const CUtensorMap* tc = nullptr) {
  const int stage = p.mode == MODE_PLAIN ? ST_WPRIME : (p.mode == MODE_BLOCKDIAG ? ST_BLOCKDIAG : ST_WGRAD);
  auto k = umma_gemm_kernel<BN, STAGES, A_MN, B_MN, OUT_F32, RES, CL, TOUT>;
  constexpr int stg_bytes =
      TOUT ? kEpiWarps * 32 * 128
           : kEpiWarps * 32 *
                 (epi_pass_cols<BN, STAGES, OUT_F32, RES, CL>() * (OUT_F32 ? 4 : 2) + 16);
  constexpr int smem = STAGES * stage_bytes<BN, RES, CL>() + res_bytes<BN, RES>() + stg_bytes +
                       1024 + 512;
  if (TOUT && !tc) return POETX_ERR_ARG;
  const CUtensorMap& tcm = TOUT ? *tc : tb;
  // CTAs per SM: bounded by TMEM (2 x BN columns each, 512 per SM) and shared memory.
  constexpr int by_tmem = 512 / (2 * BN);
  constexpr int by_smem = (int)((227 * 1024) / (smem + 1024));
  constexpr int per_sm = by_tmem < by_smem ? by_tmem : by_smem;
  static_assert(smem <= 227 * 1024, "shared memory per CTA exceeds the sm_103 limit");
  static_assert(per_sm >= 1, "configuration exceeds TMEM or shared memory");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;  // CL > 1: co-resident clusters of this configuration
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (attr_err == cudaSuccess && CL > 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(CL * sm_count());
      cfg.blockDim = dim3(kGemmThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CL;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg);
      if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
    }
  });
  POETX_CUDA_TRY(attr_err);
  const long long tiles = (long long)tiles_m * tiles_n * tiles_z;
  if (tiles == 0) return POETX_OK;
  if (tiles > 0x7fffffffLL) return POETX_ERR_SHAPE;
  p.tiles_m = tiles_m;
  p.tiles_n = tiles_n;
  p.num_tiles = (int)tiles;
  const long long want = CL > 1 ? max_clusters : (long long)sm_count() * per_sm;
  const int grid = CL * (int)(tiles < want ? tiles : want);
  if (CL > 1)
    POETX_CUDA_TRY(launch_pdl_cluster(k, dim3(grid), dim3(kGemmThreads), smem, s, CL, ta, tb, tcm,
                                      p));
  else
    POETX_CUDA_TRY(launch_pdl(k, dim3(grid), dim3(kGemmThreads), smem, s, ta, tb, tcm, p));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, stage);
  return POETX_OK;
}

UmmaParams base_params() {
  UmmaParams p{};
  p.trace = trace_buffer(&p.trace_cap);
  p.err = device_error_word();
  p.limit_ns = kWaitLimitNs;
  return p;
}

}  // namespace

// 2-D tensor [outer][inner] of element type et with row pitch `pitch_elems`, box {box_inner,
// box_outer}, 128-byte swizzle or none, zero fill out of bounds.  Encoded maps are kept in a
// small per-thread cache keyed by every argument, since training loops pass the same buffers
// every step.
bool encode_tma_2d(CUtensorMap* m, const void* ptr, TmaElem et, uint64_t inner, uint64_t outer,
                   uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  struct Entry {
    const void* ptr;
    uint64_t inner, outer, pitch;
    uint32_t bi, bo;
    int dev, et, sw;
    CUtensorMap map;
  };
  constexpr int kEntries = 64;
  thread_local Entry cache[kEntries];
  thread_local int next = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < kEntries; ++i) {
    const Entry& e = cache[i];
    if (e.ptr == ptr && ptr && e.inner == inner && e.outer == outer && e.pitch == pitch_elems &&
        e.bi == box_inner && e.bo == box_outer && e.dev == dev && e.et == (int)et &&
        e.sw == (int)swizzle128) {
      *m = e.map;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t esz = et == TMA_U8 ? 1 : (et == TMA_BF16 ? 2 : 4);
  const CUtensorMapDataType dt = et == TMA_U8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : (et == TMA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_elems * esz};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  if (fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  Entry& e = cache[next];
  next = (next + 1) % kEntries;
  e.ptr = ptr; e.inner = inner; e.outer = outer; e.pitch = pitch_elems;
  e.bi = box_inner; e.bo = box_outer; e.dev = dev; e.et = (int)et; e.sw = (int)swizzle128;
  e.map = *m;
  return true;
}

bool umma_supported() {
  // sm_103 and a driver entry point for tensor maps; cached per device
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (!v) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    v = (major == 10 && minor == 3 && encode_fn() != nullptr) ? 1 : 2;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v == 1;
}

poetx_status umma_blockdiag(const void* X, long long N, int nblk, int b, const void* G, int trans,
                            const float* col_scale, const int32_t* out_perm, void* Y,
                            cudaStream_t s) {
  if (N == 0 || nblk == 0) return POETX_OK;
  const int D = nblk * b;
  // b = 256 with a plain output: 256-wide tiles (each activation tile read once, the whole
  // G block resident); otherwise at most 128 wide with a deeper ring
  const int BN = b < 128 ? b : (b == 256 && !out_perm ? 256 : 128);
  CUtensorMap ta, tb;
  if (!make_map(&ta, X, D, N, D, 64, 128)) return POETX_ERR_CUDA;
  if (trans) {
    if (!make_map(&tb, G, b, (uint64_t)nblk * b, b, 64, BN)) return POETX_ERR_CUDA;
  } else {
    if (!make_map(&tb, G, b, (uint64_t)nblk * b, b, 64, 64)) return POETX_ERR_CUDA;
  }
  UmmaParams p = base_params();
  p.mode = MODE_BLOCKDIAG;
  p.M = (int)N;
  p.num_kb = b / 64;
  p.b = b;
  p.C = Y;
  p.ldc = D;
  p.colscale = col_scale;
  p.out_perm = out_perm;
  p.bpre = static_cast<const uint8_t*>(G);
  p.bpre_bytes = (unsigned long long)nblk * b * b * 2;
  const int tm = (int)((N + BM - 1) / BM), tn = b / BN;
  // resident G panel of b/64 K blocks; the ring carries only the activation tiles; with
  // tiles of 128 columns or more and a plain output the epilogue stores by TMA
  CUtensorMap tc;
  if (BN >= 128 && !out_perm) {
    if (!make_map(&tc, Y, D, N, D, 64, 32)) return POETX_ERR_CUDA;
    if (trans) {
      switch (b) {
        case 128: return launch<128, 10, false, false, false, 2, 1, true>(ta, tb, p, tm, tn, nblk, s, &tc);
        case 256: return launch<256, 4, false, false, false, 4, 1, true>(ta, tb, p, tm, tn, nblk, s, &tc);
        default: return launch<128, 4, false, false, false, 8, 1, true>(ta, tb, p, tm, tn, nblk, s, &tc);
      }
    }
    switch (b) {
      case 128: return launch<128, 10, false, true, false, 2, 1, true>(ta, tb, p, tm, tn, nblk, s, &tc);
      case 256: return launch<256, 4, false, true, false, 4, 1, true>(ta, tb, p, tm, tn, nblk, s, &tc);
      default: return launch<128, 4, false, true, false, 8, 1, true>(ta, tb, p, tm, tn, nblk, s, &tc);
    }
  }
  if (trans) {
    switch (b) {
      case 64: return launch<64, 10, false, false, false, 1>(ta, tb, p, tm, tn, nblk, s);
      case 128: return launch<128, 10, false, false, false, 2>(ta, tb, p, tm, tn, nblk, s);
      case 256: return launch<128, 8, false, false, false, 4>(ta, tb, p, tm, tn, nblk, s);
      default: return launch<128, 4, false, false, false, 8>(ta, tb, p, tm, tn, nblk, s);
    }
  }
  switch (b) {
    case 64: return launch<64, 10, false, true, false, 1>(ta, tb, p, tm, tn, nblk, s);
    case 128: return launch<128, 10, false, true, false, 2>(ta, tb, p, tm, tn, nblk, s);
    case 256: return launch<128, 8, false, true, false, 4>(ta, tb, p, tm, tn, nblk, s);
    default: return launch<128, 4, false, true, false, 8>(ta, tb, p, tm, tn, nblk, s);
  }
}

poetx_status umma_wprime(const void* A, long long N, int m, int n, const void* W, int trans,
                         void* C, cudaStream_t s) {
  if (N == 0) return POETX_OK;
  CUtensorMap ta, tb;
  UmmaParams p = base_params();
  p.mode = MODE_PLAIN;
  p.M = (int)N;
  p.C = C;
  p.bpre = static_cast<const uint8_t*>(W);
  p.bpre_bytes = (unsigned long long)m * n * 2;
  const int tm = (int)((N + BM - 1) / BM);
  // 256 x 256 tiles computed by 2-CTA pairs (each CTA: 128 rows of A, 128 rows of W') when
  // there are at least two of them per pair of SMs; with fewer, both forms take the same
  // number of tile rounds and the single-CTA 128 x 256 tiles start faster.
  const int tm2 = (tm + 1) / 2;
  const bool pairs = umma_wprime_pairs(N, m, n, trans);
  // grouped raster over bands of 2048 tokens (8 pairs of M tiles, or 16 single ones)
  p.band_m = pairs ? 8 : 16;
  if (!trans) {  // C[N,n] = A[N,m] W^T
    if (!make_map(&ta, A, m, N, m, 64, 128)) return POETX_ERR_CUDA;
    // (pairs: each CTA loads half of a 256-row W' tile)
    if (!make_map(&tb, W, m, n, m, 64, pairs ? 128 : 256)) return POETX_ERR_CUDA;
    p.num_kb = m / 64;
    p.ldc = n;
    if (pairs) return launch<256, 6, false, false, false, 0, 2>(ta, tb, p, tm2, (n + 255) / 256, 1, s);
    return launch<256, 4, false, false, false>(ta, tb, p, tm, (n + 255) / 256, 1, s);
  }
  // C[N,m] = A[N,n] W: B operand (output col c, K index r) = W[r][c], MN-major
  if (!make_map(&ta, A, n, N, n, 64, 128)) return POETX_ERR_CUDA;
  if (!make_map(&tb, W, m, n, m, 64, 64)) return POETX_ERR_CUDA;
  p.num_kb = n / 64;
  p.ldc = m;
  if (pairs) return launch<256, 6, false, true, false, 0, 2>(ta, tb, p, tm2, (m + 255) / 256, 1, s);
  return launch<256, 4, false, true, false>(ta, tb, p, tm, (m + 255) / 256, 1, s);
}

bool umma_wprime_pairs(long long N, int m, int n, int trans) {
  const long long tm2 = ((N + BM - 1) / BM + 1) / 2;
  return tm2 * (((trans ? m : n) + 255) / 256) >= sm_count();
}

bool umma_wprime_fusable(long long N, int m, int n, int trans, int b) {
  const int out = trans ? m : n, K = trans ? n : m;
  return N > 0 && (b == 64 || b == 128 || b == 256) && out % 256 == 0 && K % 64 == 0 &&
         !umma_wprime_pairs(N, m, n, trans);
}

poetx_status umma_wprime_fused(const void* A, long long N, int m, int n, const void* W, int trans,
                               const void* G, int b, void* C1, void* C2, cudaStream_t s) {
  if (N == 0) return POETX_OK;
  const int out = trans ? m : n, K = trans ? n : m;
  if (!(b == 64 || b == 128 || b == 256) || out % 256 || K % 64) return POETX_ERR_SHAPE;
  CUtensorMap ta, tw, tg;
  if (!make_map(&ta, A, K, N, K, 64, 128)) return POETX_ERR_CUDA;
  if (!trans) {
    if (!make_map(&tw, W, m, n, m, 64, 256)) return POETX_ERR_CUDA;
    if (!make_map(&tg, G, b, (uint64_t)(out / b) * b, b, 64, 64)) return POETX_ERR_CUDA;
  } else {
    if (!make_map(&tw, W, m, n, m, 64, 64)) return POETX_ERR_CUDA;
    if (!make_map(&tg, G, b, (uint64_t)(out / b) * b, b, 64, b)) return POETX_ERR_CUDA;
  }
  FusedParams p{};
  p.M = (int)N;
  p.tiles_m = (int)((N + BM - 1) / BM);
  const long long tiles = (long long)p.tiles_m * (out / FZ_BN);
  if (tiles > 0x7fffffffLL) return POETX_ERR_SHAPE;
  p.num_tiles = (int)tiles;
  p.num_kb = K / 64;
  p.b = b;
  p.ldc = out;
  p.C1 = static_cast<__nv_bfloat16*>(C1);
  p.C2 = static_cast<__nv_bfloat16*>(C2);
  p.bpre = static_cast<const uint8_t*>(W);
  p.bpre_bytes = (unsigned long long)m * n * 2;
  p.trace = trace_buffer(&p.trace_cap);
  p.err = device_error_word();
  p.limit_ns = kWaitLimitNs;
  auto k = trans ? umma_fused_kernel<true, false> : umma_fused_kernel<false, true>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(umma_fused_kernel<false, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, FZ_SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(umma_fused_kernel<true, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, FZ_SMEM);
  });
  POETX_CUDA_TRY(attr_err);
  const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
  POETX_CUDA_TRY(launch_pdl(k, dim3(grid), dim3(kGemmThreads), FZ_SMEM, s, ta, tw, tg, p));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_WPRIME_FUSED);
  return POETX_OK;
}

// int8 W' contraction (the transposed kernel above).  Forward (trans = 0): C[N, n] =
// (A[N, m] Wq^T) diag(s); backward (trans = 1): C[N, m] = A[N, n] Wq, A already scaled by s.
poetx_status umma_wprime_i8(const void* A, long long N, int m, int n, const void* Wq,
                            const float* w_scale, int trans, void* C, cudaStream_t s) {
  if (N == 0) return POETX_OK;
  const int K = trans ? n : m, F = trans ? m : n;  // contraction length, output features
  if (K % 64 || F % 64) return POETX_ERR_SHAPE;
  CUtensorMap tw, tx;
  if (!make_map(&tx, A, K, N, K, 64, I8N)) return POETX_ERR_CUDA;
  if (!trans) {
    if (!make_map_t(&tw, Wq, m, n, m, 64, 128, true)) return POETX_ERR_CUDA;
  } else {
    if (!make_map_t(&tw, Wq, m, n, m, 128, 64, true)) return POETX_ERR_CUDA;
  }
  I8Params p{};
  p.tiles_f = (F + BM - 1) / BM;
  p.tiles_t = (int)((N + I8T - 1) / I8T);
  const long long tiles = (long long)p.tiles_f * p.tiles_t;
  if (tiles > 0x7fffffffLL) return POETX_ERR_SHAPE;
  p.num_tiles = (int)tiles;
  p.num_kb = K / 64;
  p.ntok = N;
  p.nfeat = F;
  p.trans = trans;
  p.scale = trans ? nullptr : w_scale;
  p.C = static_cast<__nv_bfloat16*>(C);
  p.trace = trace_buffer(&p.trace_cap);
  p.err = device_error_word();
  p.limit_ns = kWaitLimitNs;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(umma_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    I8_SMEM);
  });
  POETX_CUDA_TRY(attr_err);
  const int grid = (int)(tiles < sm_count() ? tiles : sm_count());
  POETX_CUDA_TRY(launch_pdl(umma_i8_kernel, dim3(grid), dim3(I8_THREADS), I8_SMEM, s, tw, tx, p));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_WPRIME);
  return POETX_OK;
}

poetx_status umma_wgrad(const void* X, const void* dY, long long N, int nblk, int b, int splits,
                        float* dG, cudaStream_t s) {
  if (nblk == 0) return POETX_OK;
  if (N == 0) {  // no tokens: every partial is zero
    POETX_CUDA_TRY(cudaMemsetAsync(dG, 0, (size_t)splits * nblk * b * b * sizeof(float), s));
    return POETX_OK;
  }
  const int D = nblk * b;
  const int BN = b < 256 ? b : 256;
  CUtensorMap ta, tb;
  if (!make_map(&ta, X, D, N, D, 64, 64)) return POETX_ERR_CUDA;
  if (!make_map(&tb, dY, D, N, D, 64, 64)) return POETX_ERR_CUDA;
  UmmaParams p = base_params();
  p.mode = MODE_WGRAD;
  p.M = b;
  p.b = b;
  p.nblk = nblk;
  p.splits = splits;
  p.kchunk = (int)(64 * ((N + 64LL * splits - 1) / (64LL * splits)));
  if (p.kchunk < 64) p.kchunk = 64;
  p.ntok = N;
  p.C = dG;
  const int tm = (b + BM - 1) / BM, tn = b / BN;
  if (BN == 64) return launch<64, 4, true, true, true>(ta, tb, p, tm, tn, nblk * splits, s);
  if (BN == 128) return launch<128, 3, true, true, true>(ta, tb, p, tm, tn, nblk * splits, s);
  return launch<256, 3, true, true, true>(ta, tb, p, tm, tn, nblk * splits, s);
}

}  // namespace poetx
