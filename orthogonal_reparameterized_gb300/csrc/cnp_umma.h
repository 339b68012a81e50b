// One batched CNP product: C_j = sum over segments of opA_seg(j) . opB_seg(j), plus
// epilogue terms, for every block j of a [nblk, b, b] fp32 stack (see cnp.cu).
// A terms give A row-major; B terms give B TRANSPOSED (row n of the term = column n of B),
// so that both operands reach the tensor cores K-major (kind::tf32 takes no MN-major
// operand): a symmetric or skew source is its own transpose up to sign, a general one needs
// a transposed copy (written by the kernel that produced it).
#pragma once

#include "common.cuh"

namespace poetx {

// c1 * p1 + c2 * p2 (p2 nullable), elementwise over [nblk, b, b] fp32 arrays.
struct CnpTerm {
  const float* p1;
  float c1;
  const float* p2;
  float c2;
};

struct CnpProduct {
  int b;
  int nseg;               // 1 or 2
  CnpTerm A[2], B[2];
  const float* E1;        // epilogue: out = acc + e1 E1 + e2 E2 + eI I (E1, E2 nullable)
  float e1;
  const float* E2;
  float e2;
  float eI;
  int mirror;             // result known symmetric (the CUDA-core kernel computes half)
  float* out_f32;         // outputs, nullable
  float* out_f32_t;       // fp32 output transposed
  __nv_bfloat16* out_bf16;
  __nv_bfloat16* out_bf16_t;
  // Block products over a matrix (tensor-core engine only): when a_mat is set, A[0] is
  // op(a_mat, 1), a_mat an fp32 [a_rows, nblk b] matrix (a_rows a multiple of 32), and batch
  // entry j computes C_j = a_mat[:, jb .. jb + b) . B_j ([a_rows, b]); out_f32 is then the
  // [a_rows, nblk b] result and out_f32_t its [nblk b, a_rows] transpose.  One segment, no
  // epilogue terms, fp32 outputs only.
  const float* a_mat;
  long long a_rows;
};

bool cnp_umma_ok(int b);
poetx_status cnp_umma_product(const CnpProduct& g, int nblk, cudaStream_t s);

}  // namespace poetx
