// Cayley-Neumann parameterization (CNP), forward and backward, in fp32 on the CUDA cores.
//
// POET-X summary page ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation"), "Core method" section 4: G = (I + Q)(I + Q + Q^2 + Q^3), rewritten in
// eq. 9 as G = I + 2(Q + Q^2 + Q^2 Q) + Q^2 Q^2, so that forward and backward need only Q
// and Q^2; Q is skew-symmetric and only its upper triangle is stored.
//
// Every product here is a batched b x b fp32 GEMM (one batch entry per block) whose
// operands are linear combinations of at most two b x b arrays, staged tile by tile in
// shared memory, and whose epilogue adds linear combinations of b x b arrays and of I.  The
// second operand is always given transposed (Q^T = -Q, (Q^2)^T = Q^2, and transposed copies
// X^T, M1^T are written by the kernels that produce X and M1).  On GB300 the products run on
// the tensor cores (cnp_umma.cu, 3-term tf32 split), else on the CUDA cores below:
//
//   forward   Q2 = Q Q                                     (symmetric: upper tiles only)
//             G  = Q2 (2Q + Q2) + I + 2Q + 2Q2             = I + 2(Q+Q^2+Q^3) + Q^4
//   backward  X  = sum of the dG partials (fixed order)
//             M1 = X P + P X                 with P = Q^T = -Q
//             Qbar = (2X + M1) Q2 + (Q2 - 2Q) M1 + 2X + 2M1
//             dq_ij = Qbar_ij - Qbar_ji
//
// The backward is the adjoint of eq. 9 (eq. 10 on the page is named but not printed):
// with c = (2, 2, 2, 1) the adjoint of sum_k c_k Q^k at dG = X is
// Qbar = sum_k c_k sum_{s+t=k-1} P^s X P^t, which factors as
// (XS + SX) T + S^2 (XP + PX) with S = I + P, T = I + P^2 = I + Q2, S^2 = I - 2Q + Q2;
// expanding the products gives the expression above.  Work per block: forward 3 b^3 FMA
// (Q2 half by symmetry, then one full product), backward 5 b^3 FMA.
#include <mutex>

#include "cnp_umma.h"
#include "common.cuh"
#include "kernels.h"

namespace poetx {

namespace {

using Operand = CnpTerm;
using CnpGemm = CnpProduct;

constexpr int TK = 16;

__device__ __forceinline__ float op_load(const Operand& o, long long idx) {
  float v = o.c1 * o.p1[idx];
  if (o.p2) v = fmaf(o.c2, o.p2[idx], v);
  return v;
}

template <int T>
__global__ void __launch_bounds__((T / 4) * (T / 4)) cnp_gemm_kernel(CnpGemm g) {
  pdl_trigger();
  pdl_wait();
  constexpr int NT = (T / 4) * (T / 4);
  constexpr int TPR = T / 4;  // threads per row of the thread grid
  __shared__ float As[TK][T + 4];
  __shared__ float Bs[TK][T + 4];
  const int ti = blockIdx.y, tj = blockIdx.x;
  if (g.mirror && ti > tj) return;
  const int b = g.b;
  const long long base = (long long)blockIdx.z * b * b;
  const int i0 = ti * T, j0 = tj * T;
  const int tid = threadIdx.x;
  const int tx = tid % TPR, ty = tid / TPR;

  float acc[4][4] = {};
  for (int seg = 0; seg < g.nseg; ++seg) {
    const Operand oa = g.A[seg], ob = g.B[seg];
    for (int k0 = 0; k0 < b; k0 += TK) {
#pragma unroll
      for (int r = 0; r < (T * TK) / NT; ++r) {
        const int e = tid + r * NT;
        const int ii = e / TK, kk = e % TK;
        const int gi = i0 + ii, gk = k0 + kk;
        As[kk][ii] = (gi < b && gk < b) ? op_load(oa, base + (long long)gi * b + gk) : 0.f;
      }
#pragma unroll
      for (int r = 0; r < (T * TK) / NT; ++r) {  // B from its transpose: B[k][j] = Bt[j][k]
        const int e = tid + r * NT;
        const int jj = e / TK, kk = e % TK;
        const int gj = j0 + jj, gk = k0 + kk;
        Bs[kk][jj] = (gj < b && gk < b) ? op_load(ob, base + (long long)gj * b + gk) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
        const float4 a4 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
        const float4 b4 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
        const float a[4] = {a4.x, a4.y, a4.z, a4.w};
        const float c[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], c[v], acc[u][v]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= b) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j >= b) continue;
      const long long idx = base + (long long)i * b + j;
      float r = acc[u][v];
      if (g.E1) r = fmaf(g.e1, g.E1[idx], r);
      if (g.E2) r = fmaf(g.e2, g.E2[idx], r);
      if (i == j) r += g.eI;
      const long long tidx = base + (long long)j * b + i;
      if (g.out_f32) {
        g.out_f32[idx] = r;
        if (g.mirror && ti != tj) g.out_f32[tidx] = r;
      }
      if (g.out_f32_t) g.out_f32_t[tidx] = r;
      if (g.out_bf16) g.out_bf16[idx] = __float2bfloat16_rn(r);
      if (g.out_bf16_t) g.out_bf16_t[tidx] = __float2bfloat16_rn(r);
    }
  }
}

poetx_status launch_cnp_gemm(const CnpGemm& g, int nblk, int stage, cudaStream_t s) {
  if (nblk == 0) return POETX_OK;
  if (use_tensor_cores() && cnp_umma_ok(g.b)) {
    POETX_TRY(cnp_umma_product(g, nblk, s));
    after_launch(s, stage);
    return POETX_OK;
  }
  if (g.b >= 64) {
    dim3 grid(ceil_div(g.b, 64), ceil_div(g.b, 64), nblk);
    POETX_CUDA_TRY(launch_pdl(cnp_gemm_kernel<64>, grid, dim3(256), 0, s, g));
  } else {
    dim3 grid(ceil_div(g.b, 32), ceil_div(g.b, 32), nblk);
    POETX_CUDA_TRY(launch_pdl(cnp_gemm_kernel<32>, grid, dim3(64), 0, s, g));
  }
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, stage);
  return POETX_OK;
}

Operand op1(const float* p, float c) { return Operand{p, c, nullptr, 0.f}; }
Operand op2(const float* p, float c, const float* q, float d) { return Operand{p, c, q, d}; }

// X[j] = sum_s dG_k[s][j - start_k] in the order s = 0, 1, ..., splits_k - 1 for the side k
// that owns block j, and Xt[j] = X[j]^T, one 32 x 32 tile per CTA (transpose through shared
// memory so that both stores are coalesced).
__device__ __forceinline__ int sum_side(const SideTable& t, int blk) {
  int k = 0;
  while (k + 1 < t.count && blk >= t.start[k + 1]) ++k;
  return k;
}

__global__ void sum_partials_kernel(const __grid_constant__ SideTable st, int b,
                                    float* __restrict__ X, float* __restrict__ Xt) {
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[32][33];
  const int j = blockIdx.z;
  const int k = sum_side(st, j);
  const long long nk = st.start[k + 1] - st.start[k];
  const float* src = st.src[k] + (long long)(j - st.start[k]) * b * b;
  const int S = st.splits[k];
  const long long sstride = nk * b * b;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const long long base = (long long)j * b * b;
  for (int rr = threadIdx.y; rr < 32; rr += 8) {
    const int r = r0 + rr, c = c0 + threadIdx.x;
    float a = 0.f;
    if (r < b && c < b) {
      const long long off = (long long)r * b + c;
      a = src[off];
#pragma unroll 8
      for (int s2 = 1; s2 < S; ++s2) a += src[s2 * sstride + off];  // fixed order
      X[base + off] = a;
    }
    tile[rr][threadIdx.x] = a;
  }
  __syncthreads();
  for (int cc = threadIdx.y; cc < 32; cc += 8) {
    const int c = c0 + cc, r = r0 + threadIdx.x;
    if (r < b && c < b) Xt[base + (long long)c * b + r] = tile[threadIdx.x][cc];
  }
}

// The same sum for b % 64 == 0, one 32 x 64 tile per CTA: the partial tiles land in shared
// memory by 16-byte cp.async, kSumChunk partials at a time, so that all loads of a chunk are
// in flight together and no register waits on them; each thread then adds its two float4
// groups in the order s = 0, 1, ... (the same sums, bit for bit, as the kernel above).
constexpr int kSumR = 32, kSumC = 64, kSumChunk = 5;
constexpr size_t kSumSmem = (size_t)(kSumChunk * kSumR * kSumC + kSumC * (kSumR + 1)) * 4;

__global__ void __launch_bounds__(256) sum_partials_vec_kernel(const __grid_constant__ SideTable st,
                                                                int b, float* __restrict__ X,
                                                                float* __restrict__ Xt,
                                                                unsigned long long* tr,
                                                                size_t tr_cap) {
  if (threadIdx.x == 0) trace_stamp3(tr, tr_cap, 0);
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) float ssm[];
  float* T = ssm + kSumChunk * kSumR * kSumC;  // [kSumC][kSumR + 1] transposed tile
  const int j = blockIdx.z;
  const int k = sum_side(st, j);
  const float* src = st.src[k] + (long long)(j - st.start[k]) * b * b;
  const int S = st.splits[k];
  const long long sstride = (long long)(st.start[k + 1] - st.start[k]) * b * b;
  const int r0 = blockIdx.y * kSumR, c0 = blockIdx.x * kSumC;
  const long long base = (long long)j * b * b;
  constexpr int G = kSumR * kSumC / 4;  // float4 groups of the tile (2 per thread)
  const int tid = threadIdx.x;
  float4 acc[2];
  for (int s0 = 0; s0 < S; s0 += kSumChunk) {
    const int ns = S - s0 < kSumChunk ? S - s0 : kSumChunk;
    for (int t = 0; t < ns; ++t)
      for (int g = tid; g < G; g += 256) {
        const int rr = g / (kSumC / 4), c = 4 * (g % (kSumC / 4));
        const float* gsrc = src + (long long)(s0 + t) * sstride + (long long)(r0 + rr) * b + c0 + c;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(
                         ssm + (t * kSumR + rr) * kSumC + c)),
                     "l"(gsrc)
                     : "memory");
      }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    for (int t = 0; t < ns; ++t)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int g = tid + 256 * u;
        const int rr = g / (kSumC / 4), c = 4 * (g % (kSumC / 4));
        const float4 v = *reinterpret_cast<const float4*>(ssm + (t * kSumR + rr) * kSumC + c);
        if (s0 + t == 0) {
          acc[u] = v;
        } else {
          acc[u].x += v.x;
          acc[u].y += v.y;
          acc[u].z += v.z;
          acc[u].w += v.w;
        }
      }
    __syncthreads();  // the next chunk overwrites the partial tiles
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int g = tid + 256 * u;
    const int rr = g / (kSumC / 4), c = 4 * (g % (kSumC / 4));
    *reinterpret_cast<float4*>(X + base + (long long)(r0 + rr) * b + c0 + c) = acc[u];
    T[(c + 0) * (kSumR + 1) + rr] = acc[u].x;
    T[(c + 1) * (kSumR + 1) + rr] = acc[u].y;
    T[(c + 2) * (kSumR + 1) + rr] = acc[u].z;
    T[(c + 3) * (kSumR + 1) + rr] = acc[u].w;
  }
  __syncthreads();
  for (int e = tid; e < kSumC * kSumR; e += 256) {
    const int cc = e / kSumR, rr = e % kSumR;
    Xt[base + (long long)(c0 + cc) * b + r0 + rr] = T[cc * (kSumR + 1) + rr];
  }
  if (tr) {
    __syncthreads();
    if (threadIdx.x == 0) trace_stamp3(tr, tr_cap, 31);
  }
}

size_t blk_bytes(int nblk, int b) { return align_up((size_t)nblk * b * b * sizeof(float), 256); }

}  // namespace

SideTable CnpSides::table(int b) const {
  SideTable t{};
  t.count = count;
  t.start[0] = 0;
  for (int k = 0; k < count; ++k) {
    t.start[k + 1] = t.start[k] + n[k];
    t.valid[k] = last[k] > 0 ? last[k] : b;
    t.src[k] = q[k];
  }
  return t;
}

size_t cnp_fwd_scratch_bytes(int nblk, int b) { return 2 * blk_bytes(nblk, b); }
size_t cnp_bwd_scratch_bytes(int nblk, int b) { return 7 * blk_bytes(nblk, b); }

poetx_status cnp_forward_sides(const CnpSides& q, int b, float* Qs, float* Q2, float* G_f32,
                               void* G_bf16, void* Gt_bf16, cudaStream_t s, float* Gt_f32) {
  const int nblk = q.total();
  if (nblk == 0) return POETX_OK;
  POETX_TRY(launch_triu_unpack_sides(q.table(b), b, Qs, s));
  // Q2 = Q Q (symmetric); B^T = Q^T = -Q
  CnpGemm g{};
  g.b = b;
  g.nseg = 1;
  g.A[0] = op1(Qs, 1.f);
  g.B[0] = op1(Qs, -1.f);
  g.mirror = 1;
  g.out_f32 = Q2;
  POETX_TRY(launch_cnp_gemm(g, nblk, ST_CNP_Q2, s));
  // G = Q2 (2Q + Q2) + I + 2Q + 2Q2; B^T = (2Q + Q2)^T = -2Q + Q2
  CnpGemm h{};
  h.b = b;
  h.nseg = 1;
  h.A[0] = op1(Q2, 1.f);
  h.B[0] = op2(Qs, -2.f, Q2, 1.f);
  h.E1 = Qs;
  h.e1 = 2.f;
  h.E2 = Q2;
  h.e2 = 2.f;
  h.eI = 1.f;
  h.out_f32 = G_f32;
  h.out_f32_t = Gt_f32;
  h.out_bf16 = static_cast<__nv_bfloat16*>(G_bf16);
  h.out_bf16_t = static_cast<__nv_bfloat16*>(Gt_bf16);
  return launch_cnp_gemm(h, nblk, ST_CNP_G, s);
}

poetx_status matrix_blockmm_tc(const float* A, long long rows, int nblk, int b, const float* Bt,
                               float* C, float* Ct, int stage, cudaStream_t s) {
  if (nblk == 0 || rows == 0) return POETX_OK;
  if (!(use_tensor_cores() && cnp_umma_ok(b))) return POETX_ERR_UNSUPPORTED;
  CnpGemm g{};
  g.b = b;
  g.nseg = 1;
  g.A[0] = op1(A, 1.f);
  g.B[0] = op1(Bt, 1.f);
  g.a_mat = A;
  g.a_rows = rows;
  g.out_f32 = C;
  g.out_f32_t = Ct;
  return launch_cnp_gemm(g, nblk, stage, s);
}

poetx_status cnp_forward(const float* q, int nblk, int b, float* Qs, float* Q2, float* G_f32,
                         void* G_bf16, void* Gt_bf16, cudaStream_t s) {
  CnpSides sides;
  sides.add(q, nblk);
  return cnp_forward_sides(sides, b, Qs, Q2, G_f32, G_bf16, Gt_bf16, s);
}

poetx_status cnp_backward_sides(const CnpSides& q, const float* Qin, const float* Q2in,
                                const CnpGrads& gr, int b, int accumulate, void* scratch,
                                cudaStream_t s, const PackAdam* pa) {
  const int nblk = q.total();
  if (nblk == 0) return POETX_OK;
  char* w = static_cast<char*>(scratch);
  const size_t bb = blk_bytes(nblk, b);
  float* Qw = reinterpret_cast<float*>(w);
  float* Q2 = reinterpret_cast<float*>(w + bb);
  float* X = reinterpret_cast<float*>(w + 2 * bb);
  float* Xt = reinterpret_cast<float*>(w + 3 * bb);
  float* M1 = reinterpret_cast<float*>(w + 4 * bb);
  float* M1t = reinterpret_cast<float*>(w + 5 * bb);
  float* Qbar = reinterpret_cast<float*>(w + 6 * bb);
  const float* Qs = Qin;
  SideTable t = q.table(b);
  if (!Qs) {
    POETX_TRY(launch_triu_unpack_sides(t, b, Qw, s));
    Qs = Qw;
  }
  if (!Q2in) {
    CnpGemm g{};
    g.b = b;
    g.nseg = 1;
    g.A[0] = op1(Qs, 1.f);
    g.B[0] = op1(Qs, -1.f);
    g.mirror = 1;
    g.out_f32 = Q2;
    POETX_TRY(launch_cnp_gemm(g, nblk, ST_CNP_Q2, s));
    Q2in = Q2;
  }
  // X = sum of the partials (every side, fixed order) and its transpose Xt
  bool vec = b % kSumC == 0;
  for (int k = 0; k < q.count; ++k) {
    t.src[k] = gr.dG[k];
    t.splits[k] = gr.splits[k];
    t.dst[k] = gr.dq[k];
    if (q.n[k] > 0 && (!gr.dG[k] || !gr.dq[k])) return POETX_ERR_ARG;
    vec = vec && aligned16(gr.dG[k]);
  }
  if (vec) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
      attr = cudaFuncSetAttribute(sum_partials_vec_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSumSmem);
    });
    POETX_CUDA_TRY(attr);
    dim3 grid(b / kSumC, b / kSumR, nblk);
    size_t tr_cap = 0;
    unsigned long long* tr = trace_buffer(&tr_cap);
    POETX_CUDA_TRY(launch_pdl(sum_partials_vec_kernel, grid, dim3(256), kSumSmem, s, t, b, X,
                              Xt, tr, tr_cap));
    POETX_CUDA_TRY(cudaGetLastError());
    after_launch(s, ST_CNP_SUM);
  } else {
    dim3 grid(ceil_div(b, 32), ceil_div(b, 32), nblk);
    POETX_CUDA_TRY(launch_pdl(sum_partials_kernel, grid, dim3(32, 8), 0, s, t, b, X, Xt));
    POETX_CUDA_TRY(cudaGetLastError());
    after_launch(s, ST_CNP_SUM);
  }
  // M1 = X P + P X with P = -Q (B^T terms: P^T = Q, X^T = Xt); M1^T kept for the next product
  CnpGemm m{};
  m.b = b;
  m.nseg = 2;
  m.A[0] = op1(X, 1.f);
  m.B[0] = op1(Qs, 1.f);
  m.A[1] = op1(Qs, -1.f);
  m.B[1] = op1(Xt, 1.f);
  m.out_f32 = M1;
  m.out_f32_t = M1t;
  POETX_TRY(launch_cnp_gemm(m, nblk, ST_CNP_M1, s));
  // Qbar = (2X + M1) Q2 + (Q2 - 2Q) M1 + 2X + 2M1 (B^T terms: Q2^T = Q2, M1^T = M1t)
  CnpGemm r{};
  r.b = b;
  r.nseg = 2;
  r.A[0] = op2(X, 2.f, M1, 1.f);
  r.B[0] = op1(Q2in, 1.f);
  r.A[1] = op2(Q2in, 1.f, Qs, -2.f);
  r.B[1] = op1(M1t, 1.f);
  r.E1 = X;
  r.e1 = 2.f;
  r.E2 = M1;
  r.e2 = 2.f;
  r.out_f32 = Qbar;
  POETX_TRY(launch_cnp_gemm(r, nblk, ST_CNP_QBAR, s));
  return launch_triu_grad_pack_sides(Qbar, t, b, accumulate, s, pa);
}

}  // namespace poetx

using namespace poetx;

extern "C" size_t poetx_cnp_workspace_bytes(int nblk, int b, int phase) {
  if (nblk < 0 || b < 2 || b > 1024) return 0;
  return phase == 0 ? cnp_fwd_scratch_bytes(nblk, b) : cnp_bwd_scratch_bytes(nblk, b);
}

extern "C" poetx_status poetx_cnp_fwd(const float* q, int nblk, int b, int order, float* G_f32,
                                      void* G_bf16, void* Gt_bf16, void* ws, size_t ws_bytes,
                                      cudaStream_t stream) {
  if (nblk < 0) return POETX_ERR_ARG;
  if (b < 2 || b > 1024) return POETX_ERR_SHAPE;
  if (order != 3) return POETX_ERR_UNSUPPORTED;
  if (nblk == 0) return POETX_OK;
  if (!q || (!G_f32 && !G_bf16 && !Gt_bf16)) return POETX_ERR_ARG;
  if (!ws) return POETX_ERR_ARG;
  if (ws_bytes < cnp_fwd_scratch_bytes(nblk, b)) return POETX_ERR_WORKSPACE;
  if (!aligned16(ws) || !aligned16(q)) return POETX_ERR_ALIGN;
  float* Qs = static_cast<float*>(ws);
  float* Q2 = reinterpret_cast<float*>(static_cast<char*>(ws) + cnp_fwd_scratch_bytes(nblk, b) / 2);
  return cnp_forward(q, nblk, b, Qs, Q2, G_f32, G_bf16, Gt_bf16, stream);
}

extern "C" poetx_status poetx_cnp_bwd(const float* q, const float* dG, int splits, int nblk, int b,
                                      int order, float* dq, int accumulate, void* ws,
                                      size_t ws_bytes, cudaStream_t stream) {
  if (nblk < 0 || splits < 1) return POETX_ERR_ARG;
  if (b < 2 || b > 1024) return POETX_ERR_SHAPE;
  if (order != 3) return POETX_ERR_UNSUPPORTED;
  if (nblk == 0) return POETX_OK;
  if (!q || !dG || !dq || !ws) return POETX_ERR_ARG;
  if (ws_bytes < cnp_bwd_scratch_bytes(nblk, b)) return POETX_ERR_WORKSPACE;
  if (!aligned16(ws) || !aligned16(dG)) return POETX_ERR_ALIGN;
  CnpSides sides;
  sides.add(q, nblk);
  CnpGrads g;
  g.dG[0] = dG;
  g.splits[0] = splits;
  g.dq[0] = dq;
  return cnp_backward_sides(sides, nullptr, nullptr, g, b, accumulate, ws, stream);
}
