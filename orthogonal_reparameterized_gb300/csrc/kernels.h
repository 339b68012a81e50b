// Internal host-side launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/poetx.h"
#include "adam.cuh"

namespace poetx {

// ---- index.cu
poetx_status launch_triu_unpack(const float* q, int nblk, int b, float* Q, cudaStream_t s);
// The blocks of one CNP call may come from several "sides" (the R and P factors of a layer,
// or of every layer of a group): side k owns blocks [start[k], start[k] + n[k]) of one
// contiguous [total, b, b] stack, sides in order.
constexpr int kMaxSides = 32;

// Per-side arguments of the unpack, partial-sum and gradient-pack kernels (a kernel
// parameter: 1.2 KB).
struct SideTable {
  int count;
  int start[kMaxSides + 1];    // first block of each side; start[count] = total blocks
  int valid[kMaxSides];        // features of the side's last block (b when it is whole)
  const float* src[kMaxSides];  // q of the side (unpack) or its dG partials (sum)
  float* dst[kMaxSides];        // dq of the side (pack)
  int splits[kMaxSides];        // dG partials of the side (sum)
};

// The optimizer update applied by the gradient pack, per side: q, m, v (nullptr q: none).
struct PackAdam {
  AdamK h;
  float* q[kMaxSides];
  float* m[kMaxSides];
  float* v[kMaxSides];
};

// Q [total, b, b] = the unpacked skew blocks of every side's q (t.src); entries of a ragged
// last block outside its r x r corner are zero in Q and get zero gradient.
poetx_status launch_triu_unpack_sides(const SideTable& t, int b, float* Q, cudaStream_t s);
// dq of every side (t.dst) (+)= Qbar_ij - Qbar_ji; pa (nullable): the optimizer update applied
// as each dq entry is written.
poetx_status launch_triu_grad_pack_sides(const float* Qbar, const SideTable& t, int b,
                                         int accumulate, cudaStream_t s,
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
// W[i] = float(Wb[i]) over `count` bf16 values (a multiple of 4), exactly.
poetx_status launch_widen_bf16(const void* Wb, long long count, float* W, cudaStream_t s);
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
struct CnpSides {
  int count = 0;
  const float* q[kMaxSides] = {};  // packed triangles of each side
  int n[kMaxSides] = {};           // blocks of each side
  int last[kMaxSides] = {};        // features of each side's last block when ragged (0: b)
  int total() const {
    int t = 0;
    for (int k = 0; k < count; ++k) t += n[k];
    return t;
  }
  // false when the table is full
  bool add(const float* qk, int nk, int lastk = 0) {
    if (count == kMaxSides) return false;
    q[count] = qk;
    n[count] = nk;
    last[count] = lastk;
    ++count;
    return true;
  }
  // the unpack kernels' table: start, valid and src = q
  SideTable table(int b) const;
};
// Per side: the dG partials [splits[k], n[k], b, b] and the dq output [n[k], b(b-1)/2].
struct CnpGrads {
  const float* dG[kMaxSides] = {};
  int splits[kMaxSides] = {};
  float* dq[kMaxSides] = {};
};
size_t cnp_fwd_scratch_bytes(int nblk, int b);
size_t cnp_bwd_scratch_bytes(int nblk, int b);
// Forward CNP with caller-provided fp32 scratch Qs and the Q^2 output (both [nblk, b, b]).
poetx_status cnp_forward(const float* q, int nblk, int b, float* Qs, float* Q2, float* G_f32,
                         void* G_bf16, void* Gt_bf16, cudaStream_t s);
poetx_status cnp_forward_sides(const CnpSides& q, int b, float* Qs, float* Q2, float* G_f32,
                               void* G_bf16, void* Gt_bf16, cudaStream_t s,
                               float* Gt_f32 = nullptr);
// Block products over a matrix on the tensor cores (fp32 accuracy by the three-pass tf32
// split): for every column block j of the fp32 [rows, nblk b] matrix A,
//   C[:, jb .. jb + b) = A[:, jb .. jb + b) . B_j,  B_j^T = Bt[j] of a [nblk, b, b] stack;
// C ([rows, nblk b]) and Ct (its [nblk b, rows] transpose) nullable.  rows a multiple of 32.
// POETX_ERR_UNSUPPORTED where the tensor-core engine does not take b.
poetx_status matrix_blockmm_tc(const float* A, long long rows, int nblk, int b, const float* Bt,
                               float* C, float* Ct, int stage, cudaStream_t s);
// Backward CNP.  Q and Q2 may be the stacks kept from the forward, or NULL to recompute
// them into the scratch; g.dG[k] / g.splits[k] / g.dq[k] per side.  scratch holds
// cnp_bwd_scratch_bytes(total blocks, b) bytes.  pa (nullable): the optimizer update of
// every side applied by the gradient pack.
poetx_status cnp_backward_sides(const CnpSides& q, const float* Q, const float* Q2,
                                const CnpGrads& g, int b, int accumulate, void* scratch,
                                cudaStream_t s, const PackAdam* pa = nullptr);

// ---- optim.cu
// Adam hyperparameters for the kernels (bias corrections in fp64 on the host);
// POETX_ERR_ARG for step < 1 or betas outside [0, 1).
poetx_status adam_params(const poetx_adam* hp, AdamK* h);

// ---- layer.cu: engine switch (tensor cores unless disabled by poetx_set_gemm_engine)
bool use_tensor_cores();

// ---- umma_gemm.cu: tcgen05 / TMA tensor-core GEMMs (bf16 in, fp32 accumulate)
bool umma_supported();
enum TmaElem : int { TMA_U8 = 0, TMA_BF16 = 1, TMA_F32 = 2 };
// Tensor map of a 2-D tensor [outer][inner] (row pitch in elements), box {box_inner,
// box_outer}, 128-byte swizzle or none (cached per thread).
bool encode_tma_2d(CUtensorMap* m, const void* ptr, TmaElem et, uint64_t inner, uint64_t outer,
                   uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer, bool swizzle128);
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
// tensor-memory A operand (K and the output features must be multiples of 64); the
// forward multiplies output column r by w_scale[r], the backward expects A to carry the
// scale already.
poetx_status umma_wprime_i8(const void* A, long long N, int m, int n, const void* Wq,
                            const float* w_scale, int trans, void* C, cudaStream_t s);
// ---- bdw.cu: the backward of a block-diagonal product in one pass over T (b = 128 or 256):
// Y = T blkdiag(G)^T (column c times colscale[c] when given) and dG[s, j] = S_j^T T_j over
// the token tiles of split s (fp32 partials [splits, nblk, b, b]).  bdw_splits: the split
// count the layer uses with it.
bool umma_bdw_ok(int b);
int bdw_splits(long long N, int nblk, int b);
poetx_status umma_bdw(const void* T, const void* S, long long N, int nblk, int b, const void* G,
                      const float* colscale, void* Y, int splits, float* dG, cudaStream_t s);
// dG[s, j] = X_j^T dY_j over the tokens of split s (fp32 partials).
poetx_status umma_wgrad(const void* X, const void* dY, long long N, int nblk, int b, int splits,
                        float* dG, cudaStream_t s);

}  // namespace poetx
