// Cayley-Neumann forward for callers that cannot allocate device memory.
//
// poetx_cnp_fwd needs two fp32 scratch arrays (the unpacked skew blocks Q and their squares
// Q^2) that its caller allocates.  Some callers cannot: a plugin or extension living inside a
// host application that owns every device allocation and lends it none, or a code path where
// a cudaMalloc (which may synchronize the whole device) is not acceptable once set-up is
// over.  poetx_cnp_fwd_noalloc runs the very same kernels with that scratch taken from a
// fixed array that is part of the library image on the device, so the call itself allocates
// nothing and asks the caller for nothing but its inputs and outputs.
//
// The array is module-scope device memory: every GPU that loads the library holds it until
// the process exits, and every call on a device shares it.  Its host-side name is only a
// stand-in for the device address, so each call looks the address up with
// cudaGetSymbolAddress in the current context.

#include "common.cuh"
#include "kernels.h"

namespace poetx {
namespace {

// Q and Q^2 of up to POETX_CNP_NOALLOC_MAX_ELEMS elements each (nblk * b * b), fp32.
static __device__ __align__(256) float g_cnp_scratch[2 * POETX_CNP_NOALLOC_MAX_ELEMS];

// Device address of g_cnp_scratch in the current context (nullptr on failure).  Looked up on
// every call, not cached: after a device reset the module is loaded again and the array may
// sit at another address.
float* scratch_for_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_cnp_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<float*>(p);
}

}  // namespace
}  // namespace poetx

using namespace poetx;

extern "C" poetx_status poetx_cnp_fwd_noalloc(const float* q, int nblk, int b, int order,
                                              float* G_f32, void* G_bf16, void* Gt_bf16,
                                              cudaStream_t stream) {
  if (nblk < 0) return POETX_ERR_ARG;
  if (b < 2 || b > 1024) return POETX_ERR_SHAPE;
  if (order != 3) return POETX_ERR_UNSUPPORTED;
  if (nblk == 0) return POETX_OK;
  if (!q || (!G_f32 && !G_bf16 && !Gt_bf16)) return POETX_ERR_ARG;
  if ((long long)nblk * b * b > (long long)POETX_CNP_NOALLOC_MAX_ELEMS) return POETX_ERR_WORKSPACE;
  if (!aligned16(q)) return POETX_ERR_ALIGN;
  float* base = scratch_for_current_device();
  if (!base) return POETX_ERR_CUDA;
  // Every element of Q and Q^2 that the kernels read is written earlier in the same call
  // (unpack fills Q, the Q^2 product fills all of Q^2), so nothing needs clearing.
  float* Qs = base;
  float* Q2 = base + POETX_CNP_NOALLOC_MAX_ELEMS;
  return cnp_forward(q, nblk, b, Qs, Q2, G_f32, G_bf16, Gt_bf16, stream);
}
