// Index and data-movement kernels: packed-triangle unpack / gradient pack (step S1 and its
// gradient), permutations as index remaps (S3, S7, S8, S13), the permutation merge into the
// frozen weight (S15) and the per-row int8 quantiser (S16).  All are bit-exact data
// movement (the quantiser takes its decisions in IEEE fp32).
//
// POET-X summary page ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation"), "Core method" section 2 (permutations as index remaps; merge of the
// two permutations into W once per inner loop) and section 4 (upper-triangle storage).
#include "common.cuh"
#include "kernels.h"

namespace poetx {

// ---------------------------------------------------------------- packed triangle
// Offset of pair (i, j), i < j, in the row-major strict upper triangle of a b x b block.
__device__ __forceinline__ long long tri_index(int i, int j, int b) {
  return (long long)i * (b - 1) - (long long)i * (i - 1) / 2 + (j - i - 1);
}

// Blocks [0, n0) come from q0, blocks [n0, gridDim.z) from q1 (the R and P sides of a layer
// are unpacked by one launch).
__global__ void triu_unpack_kernel(const float* __restrict__ q0, int n0, const float* __restrict__ q1,
                                   int b, float* __restrict__ Q) {
  const int blk = blockIdx.z;
  const int i = blockIdx.y;
  const long long tri = (long long)b * (b - 1) / 2;
  const float* qb = blk < n0 ? q0 + blk * tri : q1 + (blk - n0) * tri;
  float* row = Q + ((long long)blk * b + i) * b;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < b; j += gridDim.x * blockDim.x) {
    float v = 0.f;
    if (i < j) v = qb[tri_index(i, j, b)];
    else if (i > j) v = -qb[tri_index(j, i, b)];
    row[j] = v;
  }
}

__global__ void triu_grad_pack_kernel(const float* __restrict__ Qbar, int b, float* __restrict__ dq0,
                                      int n0, float* __restrict__ dq1, int accumulate) {
  const int blk = blockIdx.z;
  const int i = blockIdx.y;
  const long long tri = (long long)b * (b - 1) / 2;
  const float* Qb = Qbar + (long long)blk * b * b;
  float* dqb = blk < n0 ? dq0 + blk * tri : dq1 + (blk - n0) * tri;
  for (int j = i + 1 + blockIdx.x * blockDim.x + threadIdx.x; j < b; j += gridDim.x * blockDim.x) {
    const float v = Qb[(long long)i * b + j] - Qb[(long long)j * b + i];
    float* dst = dqb + tri_index(i, j, b);
    *dst = accumulate ? *dst + v : v;
  }
}

poetx_status launch_triu_unpack2(const float* q0, int n0, const float* q1, int n1, int b, float* Q,
                                 cudaStream_t s) {
  if (n0 + n1 == 0) return POETX_OK;
  const int threads = b < 256 ? ((b + 31) / 32) * 32 : 256;
  dim3 grid(1, b, n0 + n1);
  triu_unpack_kernel<<<grid, threads, 0, s>>>(q0, n0, q1, b, Q);
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_TRIU_UNPACK);
  return POETX_OK;
}

poetx_status launch_triu_unpack(const float* q, int nblk, int b, float* Q, cudaStream_t s) {
  return launch_triu_unpack2(q, nblk, nullptr, 0, b, Q, s);
}

poetx_status launch_triu_grad_pack2(const float* Qbar, int n0, int n1, int b, float* dq0, float* dq1,
                                    int accumulate, cudaStream_t s) {
  if (n0 + n1 == 0 || b < 2) return POETX_OK;
  const int threads = b < 256 ? ((b + 31) / 32) * 32 : 256;
  dim3 grid(1, b - 1, n0 + n1);
  triu_grad_pack_kernel<<<grid, threads, 0, s>>>(Qbar, b, dq0, n0, dq1, accumulate);
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_TRIU_PACK);
  return POETX_OK;
}

poetx_status launch_triu_grad_pack(const float* Qbar, int nblk, int b, float* dq, int accumulate,
                                   cudaStream_t s) {
  return launch_triu_grad_pack2(Qbar, nblk, 0, b, dq, nullptr, accumulate, s);
}

// ---------------------------------------------------------------- row permutations
// One CTA per row at a time (grid-stride over rows).  The row is staged in shared memory:
// gather reads it coalesced and writes out[i] = row[perm[i]] as 16-byte vectors; scatter
// reads 16-byte vectors, writes row[perm[i]] = in[i] into shared memory, then stores the
// row coalesced.  `src_rows` (nullable) remaps the source row (used by the merge).
template <int E>
struct VecT;
template <>
struct VecT<1> { using T = uint8_t; };
template <>
struct VecT<2> { using T = uint16_t; };
template <>
struct VecT<4> { using T = uint32_t; };

template <int E, bool SCATTER>
__global__ void __launch_bounds__(256) perm_rows_kernel(const uint8_t* __restrict__ X, long long N,
                                                        int D, const int32_t* __restrict__ perm,
                                                        uint8_t* __restrict__ Y,
                                                        const int32_t* __restrict__ src_rows,
                                                        const float* __restrict__ scale,
                                                        float* __restrict__ scale_out) {
  using T = typename VecT<E>::T;
  constexpr int V = 16 / E;  // elements per 16-byte vector
  extern __shared__ __align__(16) uint8_t smem_raw[];
  T* buf = reinterpret_cast<T*>(smem_raw);
  const int nvec = D / V;
  const size_t row_bytes = (size_t)D * E;
  for (long long r = blockIdx.x; r < N; r += gridDim.x) {
    const long long src = src_rows ? (long long)src_rows[r] : r;
    const uint4* in = reinterpret_cast<const uint4*>(X + src * row_bytes);
    uint4* out = reinterpret_cast<uint4*>(Y + r * row_bytes);
    if (scale_out && threadIdx.x == 0) scale_out[r] = scale[src];
    if (!SCATTER) {
      uint4* b4 = reinterpret_cast<uint4*>(buf);
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) b4[v] = __ldg(in + v);
      __syncthreads();
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        union { uint4 u; T e[V]; } pk;
#pragma unroll
        for (int e = 0; e < V; ++e) pk.e[e] = buf[__ldg(perm + v * V + e)];
        out[v] = pk.u;
      }
      __syncthreads();
    } else {
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        union { uint4 u; T e[V]; } pk;
        pk.u = __ldg(in + v);
#pragma unroll
        for (int e = 0; e < V; ++e) buf[__ldg(perm + v * V + e)] = pk.e[e];
      }
      __syncthreads();
      const uint4* b4 = reinterpret_cast<const uint4*>(buf);
      for (int v = threadIdx.x; v < nvec; v += blockDim.x) out[v] = b4[v];
      __syncthreads();
    }
  }
}

template <int E, bool SCATTER>
static poetx_status launch_perm_rows_t(const void* X, long long N, int D, const int32_t* perm,
                                       void* Y, const int32_t* src_rows, const float* scale,
                                       float* scale_out, cudaStream_t s) {
  const size_t smem = (size_t)D * E;
  auto k = perm_rows_kernel<E, SCATTER>;
  if (smem > 48 * 1024) POETX_CUDA_TRY(cudaFuncSetAttribute(
      k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const int per_sm = smem > 0 ? (int)((200 * 1024) / smem) : 8;
  const long long want = (long long)sm_count() * (per_sm < 1 ? 1 : (per_sm > 8 ? 8 : per_sm));
  const int grid = (int)(N < want ? N : want);
  k<<<grid, 256, smem, s>>>(static_cast<const uint8_t*>(X), N, D, perm, static_cast<uint8_t*>(Y),
                           src_rows, scale, scale_out);
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, src_rows ? ST_MERGE : (SCATTER ? ST_PERM_SCATTER : ST_PERM_GATHER));
  return POETX_OK;
}

poetx_status launch_perm_rows(size_t esize, bool scatter, const void* X, long long N, int D,
                              const int32_t* perm, void* Y, const int32_t* src_rows,
                              const float* scale, float* scale_out, cudaStream_t s) {
  if (N == 0 || D == 0) return POETX_OK;
  if (((size_t)D * esize) % 16 != 0) return POETX_ERR_SHAPE;
  if ((size_t)D * esize > 200 * 1024) return POETX_ERR_SHAPE;
  if (esize == 1)
    return scatter ? launch_perm_rows_t<1, true>(X, N, D, perm, Y, src_rows, scale, scale_out, s)
                   : launch_perm_rows_t<1, false>(X, N, D, perm, Y, src_rows, scale, scale_out, s);
  if (esize == 2)
    return scatter ? launch_perm_rows_t<2, true>(X, N, D, perm, Y, src_rows, scale, scale_out, s)
                   : launch_perm_rows_t<2, false>(X, N, D, perm, Y, src_rows, scale, scale_out, s);
  if (esize == 4)
    return scatter ? launch_perm_rows_t<4, true>(X, N, D, perm, Y, src_rows, scale, scale_out, s)
                   : launch_perm_rows_t<4, false>(X, N, D, perm, Y, src_rows, scale, scale_out, s);
  return POETX_ERR_DTYPE;
}

// ---------------------------------------------------------------- int8 quantiser
__global__ void __launch_bounds__(256) quantize_rows_kernel(const float* __restrict__ W, int m,
                                                            int8_t* __restrict__ Wq,
                                                            float* __restrict__ scale) {
  const long long r = blockIdx.x;
  const float* row = W + r * m;
  float amax = 0.f;
  for (int c = threadIdx.x; c < m; c += blockDim.x) amax = fmaxf(amax, fabsf(row[c]));
  __shared__ float red[8];
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  amax = red[0];
  const float s = amax > 0.f ? __fdiv_rn(amax, 127.0f) : 1.0f;
  if (threadIdx.x == 0) scale[r] = s;
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    float v = rintf(__fdiv_rn(row[c], s));  // round half to even
    v = fminf(fmaxf(v, -127.f), 127.f);
    Wq[r * m + c] = (int8_t)(int)v;
  }
}

poetx_status launch_quantize(const float* W, int n, int m, int8_t* Wq, float* scale,
                             cudaStream_t s) {
  if (n == 0) return POETX_OK;
  quantize_rows_kernel<<<n, 256, 0, s>>>(W, m, Wq, scale);
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_QUANTIZE);
  return POETX_OK;
}

}  // namespace poetx

using namespace poetx;

extern "C" poetx_status poetx_triu_unpack(const float* q, int nblk, int b, float* Q_f32,
                                          cudaStream_t stream) {
  if (nblk < 0 || b < 2 || b > 1024) return nblk < 0 ? POETX_ERR_ARG : POETX_ERR_SHAPE;
  if (nblk == 0) return POETX_OK;
  if (!q || !Q_f32) return POETX_ERR_ARG;
  return launch_triu_unpack(q, nblk, b, Q_f32, stream);
}

extern "C" poetx_status poetx_triu_grad_pack(const float* Qbar, int nblk, int b, float* dq,
                                             int accumulate, cudaStream_t stream) {
  if (nblk < 0 || b < 2 || b > 1024) return nblk < 0 ? POETX_ERR_ARG : POETX_ERR_SHAPE;
  if (nblk == 0) return POETX_OK;
  if (!Qbar || !dq) return POETX_ERR_ARG;
  return launch_triu_grad_pack(Qbar, nblk, b, dq, accumulate, stream);
}

static poetx_status perm_entry(bool scatter, poetx_dtype dt, const void* X, int N, int D,
                               const int32_t* perm, void* Y, cudaStream_t stream) {
  const size_t es = dtype_size(dt);
  if (!es) return POETX_ERR_DTYPE;
  if (N < 0 || D < 0) return POETX_ERR_ARG;
  if (N == 0 || D == 0) return POETX_OK;
  if (!X || !Y || !perm) return POETX_ERR_ARG;
  if (!aligned16(X) || !aligned16(Y)) return POETX_ERR_ALIGN;
  return launch_perm_rows(es, scatter, X, N, D, perm, Y, nullptr, nullptr, nullptr, stream);
}

extern "C" poetx_status poetx_perm_gather(poetx_dtype dt, const void* X, int N, int D,
                                          const int32_t* perm, void* Y, cudaStream_t stream) {
  return perm_entry(false, dt, X, N, D, perm, Y, stream);
}

extern "C" poetx_status poetx_perm_scatter(poetx_dtype dt, const void* X, int N, int D,
                                           const int32_t* perm, void* Y, cudaStream_t stream) {
  return perm_entry(true, dt, X, N, D, perm, Y, stream);
}

extern "C" poetx_status poetx_merge_perm(const void* W0, const float* scale, poetx_dtype dt,
                                         int n, int m, const int32_t* perm_n,
                                         const int32_t* perm_m, void* Wp, float* scale_p,
                                         cudaStream_t stream) {
  const size_t es = dtype_size(dt);
  if (!es) return POETX_ERR_DTYPE;
  if (n < 0 || m < 0) return POETX_ERR_ARG;
  if (n == 0 || m == 0) return POETX_OK;
  if (!W0 || !Wp || !perm_n || !perm_m) return POETX_ERR_ARG;
  if (dt == POETX_I8 && (!scale || !scale_p)) return POETX_ERR_ARG;
  if (!aligned16(W0) || !aligned16(Wp)) return POETX_ERR_ALIGN;
  return launch_perm_rows(es, false, W0, n, m, perm_m, Wp, perm_n,
                          dt == POETX_I8 ? scale : nullptr, dt == POETX_I8 ? scale_p : nullptr,
                          stream);
}

extern "C" poetx_status poetx_quantize_rows_int8(const float* W, int n, int m, int8_t* Wq,
                                                 float* scale, cudaStream_t stream) {
  if (n < 0 || m < 0) return POETX_ERR_ARG;
  if (n == 0) return POETX_OK;
  if (!W || !Wq || !scale) return POETX_ERR_ARG;
  return launch_quantize(W, n, m, Wq, scale, stream);
}
