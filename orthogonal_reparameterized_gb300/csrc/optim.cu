// Optimizer step on the packed strict upper triangles q (the only trained parameters of a
// POET-X layer: b(b-1)/2 per block, POET-X summary page, "Core method" section 4).  The
// pages name no optimizer; the library's reading is Adam (Kingma & Ba, Algorithm 1) with
// decoupled weight decay, elementwise, fp32 state; the POET-XQ learning-rate factor
// ("Practical guidance" 3) is the caller's, folded into lr.
#include <cmath>

#include "adam.cuh"
#include "common.cuh"
#include "kernels.h"

namespace poetx {

poetx_status adam_params(const poetx_adam* hp, AdamK* h) {
  if (!hp || hp->step < 1) return POETX_ERR_ARG;
  if (!(hp->beta1 >= 0.f && hp->beta1 < 1.f && hp->beta2 >= 0.f && hp->beta2 < 1.f))
    return POETX_ERR_ARG;
  h->lr = hp->lr;
  h->beta1 = hp->beta1;
  h->beta2 = hp->beta2;
  h->eps = hp->eps;
  h->wd = hp->weight_decay;
  h->c1 = (float)(1.0 / (1.0 - std::pow((double)hp->beta1, (double)hp->step)));
  h->c2 = (float)(1.0 / (1.0 - std::pow((double)hp->beta2, (double)hp->step)));
  return POETX_OK;
}

namespace {

// Four parameters per thread (16-byte loads and stores), a scalar tail for count % 4.
__global__ void __launch_bounds__(256) adam_kernel(float* __restrict__ q,
                                                   const float* __restrict__ g,
                                                   float* __restrict__ m, float* __restrict__ v,
                                                   long long count, AdamK h) {
  pdl_trigger();
  pdl_wait();
  const long long quads = count / 4;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < quads; i += stride) {
    float4 qv = reinterpret_cast<float4*>(q)[i];
    const float4 gv = reinterpret_cast<const float4*>(g)[i];
    float4 mv = reinterpret_cast<float4*>(m)[i];
    float4 vv = reinterpret_cast<float4*>(v)[i];
    adam_one(qv.x, gv.x, mv.x, vv.x, h);
    adam_one(qv.y, gv.y, mv.y, vv.y, h);
    adam_one(qv.z, gv.z, mv.z, vv.z, h);
    adam_one(qv.w, gv.w, mv.w, vv.w, h);
    reinterpret_cast<float4*>(q)[i] = qv;
    reinterpret_cast<float4*>(m)[i] = mv;
    reinterpret_cast<float4*>(v)[i] = vv;
  }
  if (blockIdx.x == 0 && threadIdx.x < count - quads * 4) {
    const long long k = quads * 4 + threadIdx.x;
    adam_one(q[k], g[k], m[k], v[k], h);
  }
}

}  // namespace

}  // namespace poetx

using namespace poetx;

extern "C" poetx_status poetx_adam_triu(float* q, const float* dq, float* m, float* v,
                                        long long count, const poetx_adam* hp,
                                        cudaStream_t stream) {
  if (count < 0) return POETX_ERR_ARG;
  AdamK h;
  POETX_TRY(adam_params(hp, &h));
  if (count == 0) return POETX_OK;
  if (!q || !dq || !m || !v) return POETX_ERR_ARG;
  if (!aligned16(q) || !aligned16(dq) || !aligned16(m) || !aligned16(v)) return POETX_ERR_ALIGN;
  long long blocks = (count / 4 + 255) / 256;
  if (blocks < 1) blocks = 1;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  POETX_CUDA_TRY(launch_pdl(adam_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, q, dq, m,
                            v, count, h));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(stream, ST_OPTIM);
  return POETX_OK;
}
