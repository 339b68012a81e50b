// Tensor-core products of the Cayley-Neumann parameterization: fp32 accuracy from tcgen05
// kind::tf32 by the 3-term split a*b ~ hi(a)hi(b) + hi(a)lo(b) + lo(a)hi(b), where
// hi(v) = v rounded to the nearest tf32 value (13 low mantissa bits cleared) and
// lo(v) = v - hi(v) (exact in fp32); the dropped lo*lo term is below 2^-22 |a||b|.  The
// tensor-core fp32 accumulation is kept short: every 32-wide K block goes into a fresh TMEM
// accumulator (two, used alternately) that the converter warps add into fp32 registers with
// IEEE adds ("promotion"), so the accumulated rounding does not grow with b.
//
// Each CNP product (POET-X summary page, "Core method" section 4, eq. 9 and its gradient)
// is C_j = sum_seg opA_seg(j) . opB_seg(j) + epilogue, for every block j, where each operand
// is a linear combination of at most two b x b fp32 arrays (Q, Q^2, X, M1).  The pipeline
// of one CTA (one 128 x BN output tile of one block):
//   warp 0     TMA: the raw fp32 tiles of every source array of the current K block
//   warps 2-5  form v = c0*src0 + c1*src1 in shared memory and split it in place into
//              hi(v) and lo(v) (same swizzled offsets, so the layout is kept)
//   warp 1     three tcgen05.mma kind::tf32 per K=8 step into the K block's TMEM accumulator
//   warps 2-5  promote each K block's accumulator into registers; at the end add the
//              epilogue terms and store fp32 / fp32^T / bf16 / bf16^T
// Both operand tiles are K-major (kind::tf32 takes no MN-major operand): A tiles are rows of
// A, B tiles rows of B^T (the B terms of a product are given transposed); 128-byte swizzle.
// Every wait is bounded (POETX_ERR_TIMEOUT on expiry, then drain, free TMEM, return).
#include <mutex>

#include "cnp_umma.h"
#include "common.cuh"
#include "kernels.h"

namespace poetx {

namespace {

constexpr int BM = 128;
constexpr int BK = 32;      // fp32 elements per 128-byte row
constexpr int NMAPS = 8;  // distinct (source array, operand role) pairs of one product

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

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
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

// Warp roles: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2..9 converters (form and
// split the operands), 10..13 promotion + epilogue (warp 10 + q reads TMEM lane quarter
// (10 + q) % 4 = q + 2 mod 4).  NACC accumulators let the MMA run ahead of the promotion.
constexpr int kConvWarps = 8;
constexpr int kPromWarps = 4;
constexpr int kThreadsCnp = 32 * (2 + kConvWarps + kPromWarps);
constexpr int NACC = 4;

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreadsCnp, 1)
    cnp_umma_kernel(const __grid_constant__ CnpMaps maps, const CnpUParams p) {
  constexpr int NCT = 32 * kConvWarps;  // converter threads
  constexpr uint32_t A_BYTES = BM * BK * 4;   // 16 KB per buffer
  constexpr uint32_t B_BYTES = BN * BK * 4;   // BN * 128 bytes per buffer
  constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;
  constexpr uint32_t TMEM_COLS = NACC * BN;
  static_assert(TMEM_COLS == 128 || TMEM_COLS == 256, "TMEM allocation must be a power of two");
  constexpr uint32_t IDESC = tf32_idesc(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* conv = full + STAGES;
  uint64_t* empty = conv + STAGES;
  uint64_t* tfull = empty + STAGES;   // [NACC] accumulator holds a finished K block
  uint64_t* tempty = tfull + NACC;    // [NACC] accumulator has been read back
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + NACC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, nt = blockIdx.y, blk = blockIdx.z;
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

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    int issued = 0;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (*abort_flag || !mbar_wait_bounded(&empty[s], ph ^ 1, p.err, p.limit_ns)) {
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
          tma_load_2d(st + i * A_BYTES, &maps.m[A.s[i].map], &full[s], k0, row0 + mt * BM);
        if (B.s[i].map >= 0)  // rows nt*BN.. of B^T, columns k0..k0+31 (one 32 x BN box)
          tma_load_2d(st + 2 * A_BYTES + i * B_BYTES, &maps.m[B.s[i].map], &full[s], k0,
                      row0 + nt * BN);
      }
      ++issued;
    }
    for (int kb = issued - 1; kb >= 0 && kb >= issued - STAGES; --kb)
      mbar_wait_bounded(&full[kb % STAGES], (kb / STAGES) & 1, p.err, p.limit_ns);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    int done = 0;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      const int a = kb % NACC;
      const uint32_t pa = (kb / NACC) & 1;
      if (*abort_flag || !mbar_wait_bounded(&conv[s], ph, p.err, p.limit_ns) ||
          !mbar_wait_bounded(&tempty[a], pa ^ 1, p.err, p.limit_ns)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem_base + (uint32_t)(a * BN);
      const uint32_t a_hi = smem_base + s * STAGE_BYTES;
      const uint32_t a_lo = a_hi + A_BYTES;
      const uint32_t b_hi = a_hi + 2 * A_BYTES;
      const uint32_t b_lo = b_hi + B_BYTES;
#pragma unroll
      for (int k = 0; k < BK / 8; ++k) {
        const uint64_t ah = sdesc(a_hi + k * 32, 16, 1024), al = sdesc(a_lo + k * 32, 16, 1024);
        const uint64_t bh = sdesc(b_hi + k * 32, 16, 1024), bl = sdesc(b_lo + k * 32, 16, 1024);
        umma_tf32(d, ah, bh, IDESC, k != 0);
        umma_tf32(d, ah, bl, IDESC, 1);
        umma_tf32(d, al, bh, IDESC, 1);
      }
      umma_commit(&empty[s]);
      umma_commit(&tfull[a]);
      ++done;
    }
    // TMEM is freed after the final barrier: wait until the last MMAs have completed.
    if (done > 0)
      mbar_wait_bounded(&tfull[(done - 1) % NACC], ((done - 1) / NACC) & 1, p.err, p.limit_ns);
  } else if (warp >= 2 && warp < 2 + kConvWarps) {
    // ---------------------------------------------------------------- converters
    const int ct = threadIdx.x - 64;  // 0..NCT-1
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      const bool ok = !*abort_flag && mbar_wait_bounded(&full[s], ph, p.err, p.limit_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      if (warp == 2 && lane == 0 && kb < 4) stamp(27 + kb);  // slots 27..30: K block landed
      const int seg = kb / p.kb_per_seg;
      const TOp& A = p.A[seg];
      const TOp& B = p.B[seg];
      uint8_t* st = smem + s * STAGE_BYTES;
      float4* a0 = reinterpret_cast<float4*>(st);
      float4* a1 = reinterpret_cast<float4*>(st + A_BYTES);
      const bool a_two = A.s[1].map >= 0;
#pragma unroll 4
      for (int e = ct; e < (int)(A_BYTES / 16); e += NCT)
        combine_split(a0 + e, a1 + e, A.s[0].coef, A.s[1].coef, a_two);
      float4* b0 = reinterpret_cast<float4*>(st + 2 * A_BYTES);
      float4* b1 = reinterpret_cast<float4*>(st + 2 * A_BYTES + B_BYTES);
      const bool b_two = B.s[1].map >= 0;
#pragma unroll 2
      for (int e = ct; e < (int)(B_BYTES / 16); e += NCT)
        combine_split(b0 + e, b1 + e, B.s[0].coef, B.s[1].coef, b_two);
      fence_async_smem();  // generic-proxy writes -> visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv[s]);
      if (warp == 2 && lane == 0 && kb < 8) stamp(10 + kb);  // slots 10..17: K block converted
    }
  } else if (warp >= 2 + kConvWarps) {
    // ---------------------------------------------------------------- promotion + epilogue
    const int q = warp & 3;  // TMEM lane quarter
    const int r = q * 32 + lane;
    const int i = mt * BM + r;
    float acc[BN];
#pragma unroll
    for (int t = 0; t < BN; ++t) acc[t] = 0.f;
    bool ok_all = true;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int a = kb % NACC;
      const bool ok = !*abort_flag &&
                      mbar_wait_bounded(&tfull[a], (kb / NACC) & 1, p.err, p.limit_ns);
      ok_all = __all_sync(0xffffffffu, ok);
      if (!ok_all) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN + c0), v);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 32; ++t) acc[c0 + t] += __uint_as_float(v[t]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      if (warp == 2 + kConvWarps && lane == 0 && kb < 8) stamp(18 + kb);  // 18..25: promoted
    }
    if (warp == 2 + kConvWarps && lane == 0) stamp(26);  // epilogue start
    const long long base = (long long)blk * b * b;
    if (ok_all && i < b) {
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        const int j0 = nt * BN + c0;
        const long long idx0 = base + (long long)i * b + j0;
        float o[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) o[t] = acc[c0 + t];
        if (p.E1) {
          const float4* e = reinterpret_cast<const float4*>(p.E1 + idx0);
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 w = __ldg(e + t);
            o[4 * t] = fmaf(p.e1, w.x, o[4 * t]);
            o[4 * t + 1] = fmaf(p.e1, w.y, o[4 * t + 1]);
            o[4 * t + 2] = fmaf(p.e1, w.z, o[4 * t + 2]);
            o[4 * t + 3] = fmaf(p.e1, w.w, o[4 * t + 3]);
          }
        }
        if (p.E2) {
          const float4* e = reinterpret_cast<const float4*>(p.E2 + idx0);
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float4 w = __ldg(e + t);
            o[4 * t] = fmaf(p.e2, w.x, o[4 * t]);
            o[4 * t + 1] = fmaf(p.e2, w.y, o[4 * t + 1]);
            o[4 * t + 2] = fmaf(p.e2, w.z, o[4 * t + 2]);
            o[4 * t + 3] = fmaf(p.e2, w.w, o[4 * t + 3]);
          }
        }
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (j0 + t == i) o[t] += p.eI;
        if (p.out_f32) {
          float4* d = reinterpret_cast<float4*>(p.out_f32 + idx0);
#pragma unroll
          for (int t = 0; t < 8; ++t) d[t] = make_float4(o[4 * t], o[4 * t + 1], o[4 * t + 2], o[4 * t + 3]);
        }
        if (p.out_f32_t) {  // lanes hold consecutive rows i: each store is coalesced
#pragma unroll
          for (int t = 0; t < 32; ++t) p.out_f32_t[base + (long long)(j0 + t) * b + i] = o[t];
        }
        if (p.out_bf16) {
          uint4* d = reinterpret_cast<uint4*>(p.out_bf16 + idx0);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            d[t] = make_uint4(pack_bf16x2(o[8 * t], o[8 * t + 1]), pack_bf16x2(o[8 * t + 2], o[8 * t + 3]),
                              pack_bf16x2(o[8 * t + 4], o[8 * t + 5]), pack_bf16x2(o[8 * t + 6], o[8 * t + 7]));
        }
        if (p.out_bf16_t) {
#pragma unroll
          for (int t = 0; t < 32; ++t)
            p.out_bf16_t[base + (long long)(j0 + t) * b + i] = __float2bfloat16_rn(o[t]);
        }
      }
    }
  }
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

template <int BN, int STAGES>
poetx_status launch_t(const CnpMaps& maps, const CnpUParams& p, int nblk, cudaStream_t s) {
  auto k = cnp_umma_kernel<BN, STAGES>;
  constexpr int smem = STAGES * (2 * BM * BK * 4 + 2 * BN * BK * 4) + 1024 + 256;
  static_assert(smem <= 227 * 1024, "shared memory per CTA exceeds the sm_103 limit");
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  POETX_CUDA_TRY(attr);
  dim3 grid((p.b + BM - 1) / BM, p.b / BN, nblk);
  POETX_CUDA_TRY(launch_pdl(k, grid, dim3(kThreadsCnp), smem, s, maps, p));
  POETX_CUDA_TRY(cudaGetLastError());
  return POETX_OK;
}

}  // namespace

bool cnp_umma_ok(int b) {
  return b >= 32 && b <= 1024 && b % 32 == 0 && umma_supported();
}

poetx_status cnp_umma_product(const CnpProduct& g, int nblk, cudaStream_t s) {
  if (nblk == 0) return POETX_OK;
  const int BN = g.b % 64 == 0 ? 64 : 32;
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
    if (!make_blk_map(&maps.m[nmaps], ptr, nblk, g.b, role == 0 ? BM : BN)) return -3;
    ptrs[nmaps] = ptr;
    roles[nmaps] = role;
    return nmaps++;
  };
  CnpUParams p{};
  p.b = g.b;
  p.nmaps = nmaps;
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
  if (BN == 64) return launch_t<64, 4>(maps, p, nblk, s);
  return launch_t<32, 4>(maps, p, nblk, s);
}

}  // namespace poetx
