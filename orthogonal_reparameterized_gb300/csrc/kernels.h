// Internal host-side launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/poetx.h"
#include "adam.cuh"

namespace poetx {

// ---- index.cu
poetx_status launch_triu_unpack(const float* q, int nblk, int b, float* Q, cudaStream_t s);
// Two-sided: blocks [0, n0) from q0, [n0, n0 + n1) from q1.
// r0, r1: features of the last block of side 0 / side 1 (0: b); entries of a ragged last
// block outside its r x r corner are zero in Q and get zero gradient.
poetx_status launch_triu_unpack2(const float* q0, int n0, const float* q1, int n1, int b, float* Q,
                                 cudaStream_t s, int r0 = 0, int r1 = 0);
// pa (nullable): the optimizer update applied as each dq entry is written.
poetx_status launch_triu_grad_pack2(const float* Qbar, int n0, int n1, int b, float* dq0, float* dq1,
                                    int accumulate, cudaStream_t s, int r0 = 0, int r1 = 0,
                                    const PackAdam* pa = nullptr);
poetx_status launch_triu_grad_pack(const float* Qbar, int nblk, int b, float* dq, int accumulate,
                                   cudaStream_t s);
// Y[r][j] = X[src_rows ? src_rows[r] : r][perm[j]] (gather) or Y[r][perm[j]] = X[r][j]
// (scatter), j < D; src_pitch / dst_pitch: row pitches in elements (0: D), destination
// columns D .. dst_pitch - 1 zeroed.
poetx_status launch_perm_rows(size_t esize, bool scatter, const void* X, long long N, int D,
                              const int32_t* perm, void* Y, const int32_t* src_rows,
                              const float* scale, float* scale_out, cudaStream_t s,
                              long long src_pitch = 0, long long dst_pitch = 0);
// The same permutation in the co-resident shape (one small CTA per SM, beside a CNP
// product); perm_side_fits says whether rows of D elements fit that shape.
bool perm_side_fits(size_t esize, int D);
poetx_status launch_perm_rows_side(size_t esize, bool scatter, const void* X, long long N, int D,
                                   const int32_t* perm, void* Y, cudaStream_t s,
                                   long long src_pitch = 0, long long dst_pitch = 0);
poetx_status launch_quantize(const float* W, int n, int m, int8_t* Wq, float* scale,
                             cudaStream_t s);
// inv_a[perm_a[i]] = i (i < na) and inv_b[perm_b[k]] = k (k < nb), one launch.
poetx_status launch_invert_perms(const int32_t* perm_a, int na, int32_t* inv_a,
                                 const int32_t* perm_b, int nb, int32_t* inv_b, cudaStream_t s);
// W[r][c] = scale[r] * Wq[r][c] (fp32 out, m % 4 == 0).
poetx_status launch_dequant_rows(const int8_t* Wq, const float* scale, int n, int m, float* W,
                                 cudaStream_t s);

// ---- simt_gemm.cu: generic strided batched GEMM on the CUDA cores (fp32 accumulation).
// C[z][i][j] = colscale[j] * sum_k A(z,i,k) B(z,k,j), element (i,k) of batch z of A at
// A[z*sab + i*sam + k*sak] (likewise B, C).  Batch index z = blockIdx.z / ksplit; the K range
// of split s is [s*kchunk, min(K, (s+1)*kchunk)) and its output goes to C + s*scs.
struct SimtGemm {
  int M, N, K;
  int batch;
  const void* A;
  long long sam, sak, sab;
  const void* B;
  long long sbk, sbn, sbb;
  void* C;
  long long scm, scn, scb;
  const float* colscale;  // nullable, indexed by j + z*colscale_bstride
  long long colscale_bstride;
  const int32_t* colperm;  // nullable: column j of batch z is stored at colperm[j + z*bstride]
  int ksplit;
  int kchunk;
  long long scs;
  int stage;  // Stage of the hot path this product serves (launch accounting)
};
poetx_status launch_simt_gemm(poetx_dtype ta, poetx_dtype tb, poetx_dtype tc, const SimtGemm& g,
                              cudaStream_t s);

// ---- cnp.cu
// The blocks of one CNP call may come from two sides (the R and P factors of a layer):
// blocks [0, n[0]) belong to side 0, [n[0], n[0] + n[1]) to side 1.  Every block array
// (Q, Q^2, G, X, ...) is one contiguous [n[0] + n[1], b, b] stack.
struct CnpSides {
  const float* q[2];   // packed triangles of each side
  int n[2];            // blocks of each side (n[1] may be 0)
  int last[2] = {0, 0};  // features of each side's last block when ragged (0: b)
};
size_t cnp_fwd_scratch_bytes(int nblk, int b);
size_t cnp_bwd_scratch_bytes(int nblk, int b);
// Forward CNP with caller-provided fp32 scratch Qs and the Q^2 output (both [nblk, b, b]).
poetx_status cnp_forward(const float* q, int nblk, int b, float* Qs, float* Q2, float* G_f32,
                         void* G_bf16, void* Gt_bf16, cudaStream_t s);
poetx_status cnp_forward_sides(const CnpSides& q, int b, float* Qs, float* Q2, float* G_f32,
                               void* G_bf16, void* Gt_bf16, cudaStream_t s);
// Backward CNP.  Q and Q2 may be the stacks kept from the forward, or NULL to recompute
// them into the scratch; dG[side] is [splits[side], n[side], b, b]; dq[side] receives that
// side's gradient.  scratch holds cnp_bwd_scratch_bytes(n[0] + n[1], b) bytes.
// pa (nullable): the optimizer update of both sides applied by the gradient pack.
poetx_status cnp_backward_sides(const CnpSides& q, const float* Q, const float* Q2,
                                const float* const dG[2], const int splits[2], int b,
                                float* const dq[2], int accumulate, void* scratch,
                                cudaStream_t s, const PackAdam* pa = nullptr);

// ---- optim.cu
// Adam hyperparameters for the kernels (bias corrections in fp64 on the host);
// POETX_ERR_ARG for step < 1 or betas outside [0, 1).
poetx_status adam_params(const poetx_adam* hp, AdamK* h);

// ---- layer.cu: engine switch (tensor cores unless disabled by poetx_set_gemm_engine)
bool use_tensor_cores();

// ---- umma_gemm.cu: tcgen05 / TMA tensor-core GEMMs (bf16 in, fp32 accumulate)
bool umma_supported();
// Y = X . op(G) per block (bf16), op = identity (trans=0) or transpose; optional column
// scale; optional output permutation (column c of the product is stored at out_perm[c]).
poetx_status umma_blockdiag(const void* X, long long N, int nblk, int b, const void* G, int trans,
                            const float* col_scale, const int32_t* out_perm, void* Y,
                            cudaStream_t s);
// C[N,n] = A[N,m] W^T (trans=0) or C[N,m] = A[N,n] W (trans=1), W [n,m] bf16.
poetx_status umma_wprime(const void* A, long long N, int m, int n, const void* W, int trans,
                         void* C, cudaStream_t s);
// Whether the bf16 contraction runs as 2-CTA pairs (at least as many 256 x 256 tiles as SMs).
bool umma_wprime_pairs(long long N, int m, int n, int trans);
// The contraction followed by the block-diagonal product on the same tiles (one launch):
// C1 = A W^T (trans 0; nullable: not stored) and C2 = C1 blkdiag(G) with G = G_P stacks
// [n/b, b, b]; or C1 = A W (trans 1) and C2 = C1 blkdiag(G)^T with G = G_R [m/b, b, b].  Taken
// when umma_wprime_fusable (b = 64, 128 or 256; single-CTA tiles, i.e. not pairs).
bool umma_wprime_fusable(long long N, int m, int n, int trans, int b);
poetx_status umma_wprime_fused(const void* A, long long N, int m, int n, const void* W, int trans,
                               const void* G, int b, void* C1, void* C2, cudaStream_t s);
// The same contraction with an int8 W, run transposed so that the widened weight is the
// tensor-memory A operand (K and the output features must be multiples of 64 and 128); the
// forward multiplies output column r by w_scale[r], the backward expects A to carry the
// scale already.
poetx_status umma_wprime_i8(const void* A, long long N, int m, int n, const void* Wq,
                            const float* w_scale, int trans, void* C, cudaStream_t s);
// dG[s, j] = X_j^T dY_j over the tokens of split s (fp32 partials).
poetx_status umma_wgrad(const void* X, const void* dY, long long N, int nblk, int b, int splits,
                        float* dG, cudaStream_t s);

}  // namespace poetx
