// Generic strided batched GEMM on the CUDA cores with fp32 accumulation.  It carries the
// fp32 layer (every product of the 256x256 fp32 workload runs here in FFMA, no TF32) and
// any shape the tensor-core engine does not take.
#include "common.cuh"
#include "kernels.h"

namespace poetx {

namespace {

constexpr int TM = 64, TN = 64, TK = 16, THREADS = 256;

template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(THREADS) simt_gemm_kernel(SimtGemm g) {
  pdl_trigger();
  pdl_wait();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int z = blockIdx.z / g.ksplit;
  const int split = blockIdx.z % g.ksplit;
  const int i0 = blockIdx.y * TM, j0 = blockIdx.x * TN;
  const int kbeg = split * g.kchunk;
  const int kend = min(g.K, kbeg + g.kchunk);
  const TA* A = static_cast<const TA*>(g.A) + (long long)z * g.sab;
  const TB* B = static_cast<const TB*>(g.B) + (long long)z * g.sbb;
  const bool a_kcontig = g.sak == 1;
  const bool b_ncontig = g.sbn == 1;

  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += TK) {
#pragma unroll
    for (int r = 0; r < (TM * TK) / THREADS; ++r) {
      const int e = tid + r * THREADS;
      const int ii = a_kcontig ? e / TK : e % TM;
      const int kk = a_kcontig ? e % TK : e / TM;
      const int gi = i0 + ii, gk = k0 + kk;
      float v = 0.f;
      if (gi < g.M && gk < kend) v = to_f32<TA>(A[(long long)gi * g.sam + (long long)gk * g.sak]);
      As[kk][ii] = v;
    }
#pragma unroll
    for (int r = 0; r < (TN * TK) / THREADS; ++r) {
      const int e = tid + r * THREADS;
      const int jj = b_ncontig ? e % TN : e / TK;
      const int kk = b_ncontig ? e / TN : e % TK;
      const int gj = j0 + jj, gk = k0 + kk;
      float v = 0.f;
      if (gj < g.N && gk < kend) v = to_f32<TB>(B[(long long)gk * g.sbk + (long long)gj * g.sbn]);
      Bs[kk][jj] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = As[kk][ty * 4 + u];
#pragma unroll
      for (int u = 0; u < 4; ++u) b[u] = Bs[kk][tx * 4 + u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
  TC* C = static_cast<TC*>(g.C) + (long long)z * g.scb + (long long)split * g.scs;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int gi = i0 + ty * 4 + u;
    if (gi >= g.M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int gj = j0 + tx * 4 + v;
      if (gj >= g.N) continue;
      float r = acc[u][v];
      if (g.colscale) r *= g.colscale[gj + (long long)z * g.colscale_bstride];
      if (g.colperm) {  // output permutation: batch offset is part of the permuted index
        const long long dc = g.colperm[gj + (long long)z * g.colscale_bstride];
        static_cast<TC*>(g.C)[(long long)split * g.scs + (long long)gi * g.scm + dc * g.scn] =
            from_f32<TC>(r);
      } else {
        C[(long long)gi * g.scm + (long long)gj * g.scn] = from_f32<TC>(r);
      }
    }
  }
}

template <typename TA, typename TB, typename TC>
poetx_status launch_t(const SimtGemm& g, cudaStream_t s) {
  dim3 grid(ceil_div(g.N, TN), ceil_div(g.M, TM), g.batch * g.ksplit);
  if (grid.y > 65535 || grid.z > 65535) return POETX_ERR_SHAPE;
  POETX_CUDA_TRY(launch_pdl(simt_gemm_kernel<TA, TB, TC>, grid, dim3(THREADS), 0, s, g));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, g.stage);
  return POETX_OK;
}

}  // namespace

poetx_status launch_simt_gemm(poetx_dtype ta, poetx_dtype tb, poetx_dtype tc, const SimtGemm& g0,
                              cudaStream_t s) {
  if (g0.M == 0 || g0.N == 0 || g0.batch == 0) return POETX_OK;
  SimtGemm g = g0;
  if (g.ksplit < 1) g.ksplit = 1;
  if (g.kchunk < 1) g.kchunk = g.K;
  using bf = __nv_bfloat16;
  if (ta == POETX_F32 && tb == POETX_F32 && tc == POETX_F32) return launch_t<float, float, float>(g, s);
  if (ta == POETX_BF16 && tb == POETX_BF16 && tc == POETX_BF16) return launch_t<bf, bf, bf>(g, s);
  if (ta == POETX_BF16 && tb == POETX_BF16 && tc == POETX_F32) return launch_t<bf, bf, float>(g, s);
  if (ta == POETX_BF16 && tb == POETX_F32 && tc == POETX_F32) return launch_t<bf, float, float>(g, s);
  if (ta == POETX_BF16 && tb == POETX_I8 && tc == POETX_BF16) return launch_t<bf, int8_t, bf>(g, s);
  return POETX_ERR_DTYPE;
}

}  // namespace poetx
