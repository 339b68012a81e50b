// The elementwise Adam update on the packed triangles, shared by the standalone optimizer
// kernel (optim.cu) and the gradient-pack kernel that applies it as it writes dq
// (index.cu).  Adam (Kingma & Ba, Algorithm 1) with decoupled weight decay: the pages name
// no optimizer (POET-X summary page, "Core method" section 4 counts its state per stored
// parameter).  Every operation is an explicitly rounded fp32 intrinsic, so the two kernels
// produce the same bits whatever the compiler contracts elsewhere.
#pragma once

#include <cuda_runtime.h>

namespace poetx {

struct AdamK {
  float lr, beta1, beta2, eps, wd;
  float c1, c2;  // 1 / (1 - beta1^t), 1 / (1 - beta2^t), computed on the host in fp64
};

// q, m, v updated in place from the gradient g.
__device__ __forceinline__ void adam_one(float& q, float g, float& m, float& v, const AdamK& h) {
  m = __fadd_rn(__fmul_rn(h.beta1, m), __fmul_rn(__fsub_rn(1.f, h.beta1), g));
  v = __fadd_rn(__fmul_rn(h.beta2, v), __fmul_rn(__fmul_rn(__fsub_rn(1.f, h.beta2), g), g));
  const float mh = __fmul_rn(m, h.c1);
  const float vh = __fmul_rn(v, h.c2);
  const float step = __fadd_rn(__fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), h.eps)),
                               __fmul_rn(h.wd, q));
  q = __fsub_rn(q, __fmul_rn(h.lr, step));
}

}  // namespace poetx
