/*
 * poetx.h -- C ABI of the POET-X layer library for NVIDIA GB300 (sm_103a).
 *
 * The library computes one POET-X layer forward and backward:
 *   - the Cayley-Neumann parameterization (CNP) that turns the stored upper triangle of a
 *     skew-symmetric Q into each b x b orthogonal block G = I + 2(Q + Q^2 + Q^3) + Q^4
 *     (POET-X summary page, "Core method" section 4, eq. 9; the gradient is eq. 10),
 *   - the input-centric chain z = G_P^T (W' (G_R^T x)) with the permutations applied as
 *     index remaps and merged into the frozen weight W' = Phi_n^T W0 Phi_m
 *     (same page, sections 1-3, eq. 3),
 *   - the backward in a "fast" variant that keeps b = W'a and a "mem" variant that
 *     recomputes it (same page, section 5), with an int8 frozen weight for the mem variant
 *     (same page, section 6, POET-XQ).
 * "POET-X summary page" is the summary of arXiv 2603.05500, "POET-X: Memory-efficient LLM
 * Training by Scaling Orthogonal Transformation".
 *
 * Conventions shared by every entry point
 *   - Row-vector batches, row-major, no padding: an activation is [N, D] with D contiguous.
 *     W0 and W' are [n_out, m_in] (PyTorch Linear layout).  G_R acts on the m_in side
 *     (m/b blocks), G_P on the n_out side (n/b blocks); Q = 0 gives y = x W0^T.
 *   - Packed triangle q of a block: b(b-1)/2 fp32 values of the strict upper triangle in
 *     row-major order (0,1),(0,2),...,(0,b-1),(1,2),...; Q = U - U^T.
 *   - Permutations are int32 gather indices: x~[:, i] = x[:, perm[i]], each a permutation
 *     of 0..D-1 (not checked on the device; an out-of-range index is undefined behaviour).
 *   - Every pointer is a DEVICE pointer unless stated otherwise, owned by the caller, and
 *     must be 16-byte aligned.  The library never allocates device memory: scratch space
 *     is passed in as (ws, ws_bytes), sized by the matching *_workspace_bytes() call.
 *   - Calls are asynchronous on the given stream (NULL = legacy default stream).  Argument
 *     errors are returned synchronously before anything is launched.  Errors seen on the
 *     device (a bounded wait that expired) are recorded in a device error word and returned
 *     by poetx_get_device_error().  Results are deterministic: equal inputs give bitwise
 *     equal outputs.
 *   - N = 0 (no tokens) is valid and launches nothing except, where a gradient is produced,
 *     the zeroing of that gradient.
 */
#ifndef POETX_H
#define POETX_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  POETX_OK = 0,
  POETX_ERR_ARG = 1,         /* NULL where a pointer is required, negative size, bad enum */
  POETX_ERR_SHAPE = 2,       /* b does not divide m or n, b outside the supported set */
  POETX_ERR_DTYPE = 3,       /* unsupported dtype combination */
  POETX_ERR_ALIGN = 4,       /* pointer not 16-byte aligned */
  POETX_ERR_WORKSPACE = 5,   /* ws_bytes smaller than the *_workspace_bytes() answer */
  POETX_ERR_UNSUPPORTED = 6, /* Neumann order other than 3, int8 weight with the fast variant */
  POETX_ERR_TIMEOUT = 7,     /* a bounded wait inside a kernel expired (device error word) */
  POETX_ERR_CUDA = 8         /* a CUDA runtime call failed (launch, attribute, tensor map) */
} poetx_status;

typedef enum { POETX_F32 = 0, POETX_BF16 = 1, POETX_I8 = 2 } poetx_dtype;
typedef enum { POETX_FAST = 0, POETX_MEM = 1 } poetx_variant;

/* Human-readable name of a status code (static string, never NULL). */
const char* poetx_status_str(poetx_status st);

/* Synchronizes the stream, reads and clears the device error word.  POETX_OK if no kernel
 * recorded an error since the last call; POETX_ERR_TIMEOUT if a bounded wait expired. */
poetx_status poetx_get_device_error(cudaStream_t stream);

/* Where the first expired bounded wait seen by poetx_get_device_error happened: a site id,
 * (source file id) x 10000 + (source line) of the waiting call (file ids: 1 the tensor-core
 * GEMM engine, 2 the CNP products, 3 the index kernels, 4 the self-test, 5 the fused
 * backward block-diagonal product), or 0 if none was
 * recorded.  Host-only (no synchronisation); for diagnosis. */
int poetx_timeout_site(void);

/* Self-test of the bounded-wait machinery: launches one block that waits on a shared-memory
 * barrier nothing arrives on, with a limit of timeout_us microseconds; the kernel records
 * POETX_ERR_TIMEOUT in the device error word and returns.  No fault, no hang. */
poetx_status poetx_selftest_timeout(unsigned int timeout_us, cudaStream_t stream);

/* Diagnostic switch for the bf16 products: engine 0 (default) runs them on the tcgen05
 * tensor cores where the GPU and the shape allow, engine 1 forces the CUDA-core kernels
 * (fp32 accumulation, same rounding of the stored results).  Process-wide. */
poetx_status poetx_set_gemm_engine(int engine);

/* Diagnostic switch of the layer's fused kernels, a bit mask (default 3):
 *   bit 0  the W' contraction and the block-diagonal product that follows it (forward:
 *          z~ = (A W'^T) blkdiag(G_P); backward: dx~ = (dB W') blkdiag(G_R)^T) as one
 *          tensor-core kernel where the shape allows (bf16 W', b = 64, 128 or 256,
 *          single-CTA tiles);
 *   bit 1  each backward block-diagonal product and its weight gradient (dB = dz~ G_P^T with
 *          dG_P = B^T dz~; dx~ = dA G_R^T with dG_R = x~^T dA) as one kernel that reads the
 *          upstream gradient once (bf16, b = 128 or 256).
 * 0 runs every product as its own kernel.  Same results up to the order of fp32
 * accumulation.  POETX_ERR_ARG outside 0..3.  Process-wide. */
poetx_status poetx_set_fusion(int on);

/* Overlap switch (default 1): poetx_layer_bwd runs the dx scatter beside the G_R weight
 * gradient and the CNP backward, on a side stream of the library's own (created once per
 * device) forked from and joined back into the caller's stream, the permutation in a
 * one-CTA-per-SM shape small enough to share SMs with the CNP products.  Results are
 * bit-identical either way; 0 runs every kernel on the caller's stream, and so do
 * per-stage profiling (poetx_profile_enable) and poetx_layer_step_host (whose download of
 * dx waits for the scatter).  POETX_ERR_ARG unless on is 0 or 1. */
poetx_status poetx_set_overlap(int on);

/* Number of kernels this library has launched in the process so far (host counter). */
unsigned long long poetx_launch_count(void);

/* Diagnostic per-stage timing.  While enabled (on != 0), every kernel launch of the library
 * records a CUDA event on its stream, and poetx_layer_fwd / poetx_layer_bwd record a
 * reference event when they start.  poetx_profile_collect synchronizes those events and
 * writes, for each launch since the last collect, its stage id and the milliseconds since
 * the previous event (host arrays of `cap` entries, nullable); it returns the number of
 * launches timed and forgets them.  Stage ids are named by poetx_stage_name. */
poetx_status poetx_profile_enable(int on);
/* Diagnostic phase trace: with a device buffer set (NULL turns it off), the library's kernels
 * write %globaltimer stamps (ns) of their phases into it, 32 unsigned 64-bit slots per CTA,
 * CTA-major.  The k-th launch after the buffer was set writes region k of 1024 x 32 slots
 * (slot 0: CTA start, slot 31: CTA end); launches beyond `bytes` write nothing.  The regions
 * are fixed when a launch is recorded, so a captured CUDA graph writes the same regions on
 * every replay. */
poetx_status poetx_set_trace_buffer(void* buf, size_t bytes);
int poetx_profile_collect(int* stage, float* ms, int cap);
const char* poetx_stage_name(int stage);

/* ----------------------------------------------------------------------------------------
 * Cayley-Neumann parameterization (POET-X summary page, "Core method" section 4)
 * ------------------------------------------------------------------------------------- */

/* Bytes of scratch for poetx_cnp_fwd (phase 0) or poetx_cnp_bwd (phase 1) over nblk
 * blocks of size b.  Returns 0 for invalid sizes. */
size_t poetx_cnp_workspace_bytes(int nblk, int b, int phase);

/* Forward CNP, eq. 9, in fp32: for every block j, G_j = I + 2(Q_j + Q_j^2 + Q_j^3) + Q_j^4.
 *   q       [nblk, b(b-1)/2] fp32 packed triangles (input)
 *   order   Neumann order; only 3 is accepted (POETX_ERR_UNSUPPORTED otherwise)
 *   G_f32   [nblk, b, b] fp32 output, row-major (nullable)
 *   G_bf16  [nblk, b, b] bf16 output (round-to-nearest-even of the fp32 G), row-major
 *           (nullable)
 *   Gt_bf16 [nblk, b, b] bf16 output holding each G_j transposed (nullable)
 *   ws      scratch of poetx_cnp_workspace_bytes(nblk, b, 0) bytes
 * 2 <= b <= 1024.  At least one output must be non-NULL. */
poetx_status poetx_cnp_fwd(const float* q, int nblk, int b, int order, float* G_f32,
                           void* G_bf16, void* Gt_bf16, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* Backward CNP (eq. 10 is named on the page, not printed; derived by the chain rule):
 *   dG      [splits, nblk, b, b] fp32 partial gradients dL/dG; the gradient is their sum,
 *           taken in a fixed order (splits >= 1)
 *   dq      [nblk, b(b-1)/2] fp32 output dL/dq; with accumulate != 0 the result is added
 *           to the existing contents, else they are overwritten
 *   ws      scratch of poetx_cnp_workspace_bytes(nblk, b, 1) bytes */
poetx_status poetx_cnp_bwd(const float* q, const float* dG, int splits, int nblk, int b,
                           int order, float* dq, int accumulate, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* Largest nblk * b * b accepted by poetx_cnp_fwd_noalloc: 2 Mi elements (for example 32
 * blocks of 256 or 8 blocks of 512).  Its fixed scratch holds twice that many floats. */
#define POETX_CNP_NOALLOC_MAX_ELEMS (2 * 1024 * 1024)

/* poetx_cnp_fwd for callers that cannot allocate device memory: a plugin or extension inside
 * a host application that owns every device allocation and lends it none, or a code path
 * where a cudaMalloc (which may synchronize the whole device) is not acceptable after
 * set-up.  No counterpart in the paper: it computes exactly what poetx_cnp_fwd computes, with
 * the same kernels, and takes the same arguments minus the workspace.
 *   Scratch: a fixed 16 MiB fp32 array in the library's device image; every GPU that loads
 *   the library holds it until the process exits.  Every call looks up the array's device
 *   address in the current context (cudaGetSymbolAddress), so a cudaDeviceReset, which loads
 *   the device image again, is followed; make the first call on a device before any stream
 *   capture (it may load the image).  All calls on a device share the array and it keeps the
 *   last call's contents: calls that overlap on the GPU (on streams not ordered with each
 *   other) race and give wrong results, so order them.  Nothing in it needs to start at zero:
 *   every element read is first written by the same call.
 *   Errors: nblk * b * b > POETX_CNP_NOALLOC_MAX_ELEMS returns POETX_ERR_WORKSPACE before
 *   anything is launched; the other checks are those of poetx_cnp_fwd.  Allocates nothing. */
poetx_status poetx_cnp_fwd_noalloc(const float* q, int nblk, int b, int order, float* G_f32,
                                   void* G_bf16, void* Gt_bf16, cudaStream_t stream);

/* Step S1 on its own: Q_f32 [nblk, b, b] = unpacked skew blocks of q. */
poetx_status poetx_triu_unpack(const float* q, int nblk, int b, float* Q_f32,
                               cudaStream_t stream);

/* Gradient of S1 on its own: dq[k] (+)= Qbar[i,j] - Qbar[j,i] for the k-th pair (i<j). */
poetx_status poetx_triu_grad_pack(const float* Qbar, int nblk, int b, float* dq,
                                  int accumulate, cudaStream_t stream);

/* ----------------------------------------------------------------------------------------
 * Permutations as index remaps (POET-X summary page, "Core method" section 2)
 * ------------------------------------------------------------------------------------- */

/* Y[t, i] = X[t, perm[i]] for t < N, i < D.  dt: POETX_F32, POETX_BF16 or POETX_I8.
 * X and Y must not overlap.  D * sizeof(dt) must be a multiple of 16, and the staged index
 * (2 bytes per column) with one row must fit an SM's shared memory: D <= 37528 (fp32),
 * 56304 (bf16), 65520 (int8); wider rows return POETX_ERR_SHAPE before any launch. */
poetx_status poetx_perm_gather(poetx_dtype dt, const void* X, int N, int D,
                               const int32_t* perm, void* Y, cudaStream_t stream);

/* Y[t, perm[i]] = X[t, i] (the inverse remap).  Same rules as poetx_perm_gather. */
poetx_status poetx_perm_scatter(poetx_dtype dt, const void* X, int N, int D,
                                const int32_t* perm, void* Y, cudaStream_t stream);

/* Merge of the two permutations into the frozen weight, once per draw of the permutations:
 *   Wp[r, c] = W0[perm_n[r], perm_m[c]]          W0, Wp: [n, m] of dtype dt
 *   scale_p[r] = scale[perm_n[r]]                when dt == POETX_I8 (scale, scale_p: [n] fp32)
 * Bit-exact data movement. */
poetx_status poetx_merge_perm(const void* W0, const float* scale, poetx_dtype dt, int n, int m,
                              const int32_t* perm_n, const int32_t* perm_m, void* Wp,
                              float* scale_p, cudaStream_t stream);

/* The same merge into a zero-padded weight, for layers whose block size does not divide m
 * or n (a ragged last block, see poetx_layer):
 *   Wp [n_pad, m_pad]:  Wp[r, c] = W0[perm_n[r], perm_m[c]] for r < n, c < m; 0 elsewhere
 *   scale_p [n_pad]:    scale[perm_n[r]] for r < n; 0 elsewhere (dt == POETX_I8)
 * A layer takes n_pad = ceil(n/b) b and m_pad = ceil(m/b) b.  n_pad >= n, m_pad >= m;
 * m * sizeof(dt) and m_pad * sizeof(dt) multiples of 16 (POETX_ERR_SHAPE otherwise: for
 * int8, m a multiple of 16); int8
 * with n_pad > n also needs n % 4 == 0, (n_pad - n) % 4 == 0 and a 16-byte aligned
 * scale_p.  Bit-exact data movement and zero fill. */
poetx_status poetx_merge_perm_padded(const void* W0, const float* scale, poetx_dtype dt, int n,
                                     int m, int n_pad, int m_pad, const int32_t* perm_n,
                                     const int32_t* perm_m, void* Wp, float* scale_p,
                                     cudaStream_t stream);

/* Per-output-row symmetric int8 quantisation of an fp32 weight (POET-XQ storage; the page
 * says only "low-bit W", the scheme is this library's reading):
 *   scale[r] = max_c |W[r,c]| / 127 in fp32 (1 for an all-zero row),
 *   Wq[r,c]  = clamp(round_half_even(W[r,c] / scale[r]), -127, 127), quotient in fp32. */
poetx_status poetx_quantize_rows_int8(const float* W, int n, int m, int8_t* Wq, float* scale,
                                      cudaStream_t stream);

/* ----------------------------------------------------------------------------------------
 * Batched block-diagonal products (POET-X summary page, "Core method" section 3)
 * ------------------------------------------------------------------------------------- */

/* Y[:, jb:(j+1)b] = X[:, jb:(j+1)b] . op(G_j) for j < nblk, op = identity (trans == 0) or
 * transpose (trans != 0); optional column scale: column c is multiplied by col_scale[c]
 * (nullable); optional output permutation: column c of the product is stored at column
 * out_perm[c] of Y (nullable; the output remap of the POET-X summary page, "Core method"
 * section 2, fused into the product; Y must not alias X then).
 *   dt      POETX_BF16 (X, G, Y bf16; fp32 accumulation; Y rounded to nearest even)
 *           or POETX_F32 (all fp32)
 *   X, Y    [N, nblk*b];  G [nblk, b, b] row-major
 * bf16 requires b in {64, 128, 256, 512}. */
poetx_status poetx_blockdiag_mm(poetx_dtype dt, const void* X, int N, int nblk, int b,
                                const void* G, int trans, const float* col_scale,
                                const int32_t* out_perm, void* Y, cudaStream_t stream);

/* Weight gradient of Y = X . blkdiag(G): dG[s, j] = X_j^T dY_j summed over the tokens of
 * split s.  Tokens are cut into `splits` contiguous ranges of chunk = 64*ceil(N/(64*splits))
 * tokens (the last ones may be short or empty, giving zero partials).
 *   X, dY   [N, nblk*b] of dtype dt;  dG [splits, nblk, b, b] fp32 output */
poetx_status poetx_blockdiag_wgrad(poetx_dtype dt, const void* X, const void* dY, int N,
                                   int nblk, int b, int splits, float* dG,
                                   cudaStream_t stream);

/* The frozen-weight contraction (POET-X summary page, "Core method" section 1, b = W'a):
 *   trans == 0:  C[N, n] = A[N, m] . W^T      (forward; int8: C[:, r] *= w_scale[r])
 *   trans != 0:  C[N, m] = A[N, n] . W        (backward; int8: A must already carry the
 *                                              per-row scale, i.e. A = dB . diag(w_scale))
 *   act     POETX_BF16 or POETX_F32 (A and C);  wdt: POETX_BF16, POETX_F32 or POETX_I8
 *   W       [n, m] row-major;  w_scale [n] fp32 (required when wdt == POETX_I8, else NULL) */
poetx_status poetx_wprime_gemm(poetx_dtype act, poetx_dtype wdt, const void* A, int N, int m,
                               int n, const void* W, const float* w_scale, int trans, void* C,
                               cudaStream_t stream);

/* ----------------------------------------------------------------------------------------
 * The whole layer (POET-X summary page, "Core method" sections 1-6)
 * ------------------------------------------------------------------------------------- */
typedef struct poetx_layer {
  int m;                   /* in-features (x has m columns) */
  int n;                   /* out-features (y has n columns) */
  int b;                   /* block size; bf16: b in {64,128,256,512}.  ceil(m/b) and ceil(n/b)
                              blocks per side; when b does not divide m or n the last block
                              of that side is ragged (r = m - (ceil(m/b) - 1) b features,
                              its own r x r factor; POET-X summary, "Core method" §1), which
                              needs b, m and n multiples of 8 */
  int order;               /* Neumann order; must be 3 */
  poetx_dtype act;         /* POETX_F32 or POETX_BF16: x, y, dy, dx */
  poetx_dtype wdt;         /* POETX_F32 (with act F32), POETX_BF16, or POETX_I8 (act BF16,
                              variant MEM) */
  poetx_variant variant;   /* POETX_FAST keeps B = A W'^T between fwd and bwd; POETX_MEM
                              recomputes it */
  const int32_t* perm_m;   /* [m] */
  const int32_t* perm_n;   /* [n] */
  const void* Wp;          /* merged frozen weight [n_pad, m_pad] of dtype wdt, n_pad =
                              ceil(n/b) b, m_pad = ceil(m/b) b (poetx_merge_perm when b
                              divides both, else poetx_merge_perm_padded) */
  const float* w_scale;    /* [n_pad] per-row scale of Wp when wdt == POETX_I8, else NULL */
  const float* q_R;        /* [ceil(m/b), b(b-1)/2]; the ragged last block's parameters are
                              the pairs (i, k), i < k < r, at their places in the b-block's
                              row-major order; its other entries are ignored and get zero
                              gradient */
  const float* q_P;        /* [ceil(n/b), b(b-1)/2], the same way */
} poetx_layer;

/* Scratch bytes for poetx_layer_fwd (phase 0) or poetx_layer_bwd (phase 1) at N tokens;
 * 0 if the descriptor is invalid. */
size_t poetx_layer_workspace_bytes(const poetx_layer* L, int N, int phase);

/* Which of the layer's products run on the CUDA cores instead of the tcgen05 tensor cores,
 * as a bit mask: bit 0 the CNP products (and poetx_merge_reinit's block products), bit 1
 * the block-diagonal products and their weight gradients, bit 2 the W' contraction; 0 when
 * everything runs on the tensor cores.  bf16 and
 * int8 layers take the tensor cores for every shape the descriptor accepts (on sm_103 with
 * the default engine); fp32 layers run their layer products on the CUDA cores (1e-5
 * accuracy), their CNP on the tensor cores.  -1 for an invalid descriptor.  Host-only. */
int poetx_layer_cuda_core_steps(const poetx_layer* L, int N);

/* Bytes the caller keeps from poetx_layer_fwd to poetx_layer_bwd ("saved"): the bf16 (or
 * fp32) blocks G_R, G_P and the fp32 Q_R, Q_P, Q_R^2, Q_P^2 (O((m+n) b), independent of N),
 * plus, for POETX_FAST only, what default autograd keeps: B = A W'^T ([N, n]) and the
 * permuted input x~ ([N, m]), both of dtype act.  POETX_MEM keeps nothing of size N. */
size_t poetx_layer_saved_bytes(const poetx_layer* L, int N);

/* Forward: y [N, n] = layer(x [N, m]).  Runs both CNPs, writes `saved` for the backward. */
poetx_status poetx_layer_fwd(const poetx_layer* L, const void* x, int N, void* y, void* saved,
                             void* ws, size_t ws_bytes, cudaStream_t stream);

/* Backward from dy [N, n]: dx [N, m], dq_R [m/b, b(b-1)/2], dq_P [n/b, b(b-1)/2] (fp32;
 * accumulate != 0 adds to them).  `saved` must come from poetx_layer_fwd with the same L,
 * x and N; the mem variant recomputes B from x. */
poetx_status poetx_layer_bwd(const poetx_layer* L, const void* x, const void* dy, int N,
                             const void* saved, void* dx, float* dq_R, float* dq_P,
                             int accumulate, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ----------------------------------------------------------------------------------------
 * Layer groups: the layers trained together (for example the seven linears of a transformer
 * block) run their Cayley-Neumann parameterizations as one batch over all their blocks (the
 * CNP of a block depends on that block's q only; POET-X summary page, "Core method" section
 * 4), and their forward and backward chains (sections 1-5) layer by layer in between.  One
 * training step of a group of `count` layers Ls[0..count-1]:
 *   poetx_group_cnp_fwd                       G, Q and Q^2 of every block of every layer
 *   poetx_group_layer_fwd(i), each layer      y_i from x_i, in whatever order the model needs
 *   poetx_group_layer_bwd(i), each layer      dx_i from dy_i, and layer i's weight-gradient
 *                                             partials (kept in ws)
 *   poetx_group_cnp_bwd                       dq_R, dq_P of every layer
 * Every layer of a group has the same b, act and order (POETX_ERR_SHAPE, POETX_ERR_DTYPE
 * otherwise); wdt and variant may differ.  1 <= count <= POETX_GROUP_MAX_LAYERS.  N is the same
 * for every call of a step.  The results equal those of poetx_layer_fwd / poetx_layer_bwd on
 * each layer (up to the order of fp32 accumulation inside the CNP products).
 *   saved  poetx_group_saved_bytes(Ls, count, N) bytes: the stacks of G, Q and Q^2 of every
 *          block and, per layer, what its forward keeps (POETX_FAST: B and x~).
 *   ws     poetx_group_workspace_bytes(Ls, count, N) bytes: the chains' scratch (one region,
 *          shared by the layers, which run one after the other on the stream), every layer's
 *          weight-gradient partials and the CNP backward's scratch.  The same ws must be
 *          passed to every poetx_group_layer_bwd and the poetx_group_cnp_bwd of a step and not
 *          be written in between; every layer's backward must come before the group's CNP
 *          backward (a layer whose backward was not run in the step gets the gradient of
 *          whatever partials ws holds).
 * Errors: as for poetx_layer_fwd / poetx_layer_bwd; i outside [0, count) is POETX_ERR_ARG;
 * 0 from the *_bytes calls means an invalid group. */
#define POETX_GROUP_MAX_LAYERS 16
size_t poetx_group_saved_bytes(const poetx_layer* Ls, int count, int N);
size_t poetx_group_workspace_bytes(const poetx_layer* Ls, int count, int N);
poetx_status poetx_group_cnp_fwd(const poetx_layer* Ls, int count, int N, void* saved,
                                 cudaStream_t stream);
poetx_status poetx_group_layer_fwd(const poetx_layer* Ls, int count, int i, const void* x, int N,
                                   void* y, void* saved, void* ws, size_t ws_bytes,
                                   cudaStream_t stream);
poetx_status poetx_group_layer_bwd(const poetx_layer* Ls, int count, int i, const void* x,
                                   const void* dy, int N, const void* saved, void* dx, void* ws,
                                   size_t ws_bytes, cudaStream_t stream);
/* dq_R, dq_P: HOST arrays of `count` device pointers, layer i's [ceil(m_i/b), b(b-1)/2] and
 * [ceil(n_i/b), b(b-1)/2] fp32 gradients (accumulate != 0 adds to them). */
poetx_status poetx_group_cnp_bwd(const poetx_layer* Ls, int count, int N, const void* saved,
                                 float* const* dq_R, float* const* dq_P, int accumulate,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* One training step of the layer (forward, then backward from dy) with HOST buffers, the
 * transfers overlapped with the kernels (the input-centric chain, POET-X summary page, "Core
 * method" sections 1-5, as poetx_layer_fwd + poetx_layer_bwd with accumulate = 0):
 *   x [N, m], dy [N, n]: host inputs, read by uploads;
 *   y [N, n], dx [N, m], dq_R [m/b, b(b-1)/2], dq_P [n/b, b(b-1)/2] (fp32): host outputs,
 *   written by downloads.
 * Activations are of dtype L->act.  Host buffers should be page-locked (cudaHostAlloc /
 * cudaHostRegister): from pageable memory the copies are correct but not overlapped, and
 * under stream capture they fail (POETX_ERR_CUDA).  dev: device scratch of at least
 * poetx_layer_step_host_bytes(L, N) bytes (16-byte aligned; 0 for an invalid descriptor),
 * holding the device copies of the six arrays, the forward's saved state and the workspace;
 * the library allocates nothing.  The uploads (x, dy) and the downloads (y, dx, dq) run on
 * an upload and a download stream the library creates once per device, so that the two
 * directions of the host link are used at once; the x upload overlaps the CNP forward, dy's
 * the forward chain, y's download the backward and dx's the CNP backward.  When the call's
 * work on `stream` completes, every output is in host memory (synchronise `stream` before
 * reading them).  Calls from several host threads are serialised while they enqueue.
 * Errors: those of poetx_layer_fwd / poetx_layer_bwd, checked before any transfer. */
size_t poetx_layer_step_host_bytes(const poetx_layer* L, int N);
poetx_status poetx_layer_step_host(const poetx_layer* L, const void* x, const void* dy, int N,
                                   void* y, void* dx, float* dq_R, float* dq_P, void* dev,
                                   size_t dev_bytes, cudaStream_t stream);

/* One training step of a layer group with HOST buffers (as poetx_group_cnp_fwd, every
 * poetx_group_layer_fwd in order 0 .. count-1, every poetx_group_layer_bwd in reverse order
 * and poetx_group_cnp_bwd with accumulate = 0): x[i] [N, m_i], dy[i] [N, n_i] are host
 * inputs, y[i] [N, n_i], dx[i] [N, m_i], dq_R[i], dq_P[i] host outputs (HOST arrays of
 * `count` host pointers each).  The uploads go in the order the kernels need them (every x,
 * then every dy from the last layer to the first) and each output comes down as soon as it
 * is written, beside the kernels, on the upload and download streams of
 * poetx_layer_step_host.  dev: device scratch of at least poetx_group_step_host_bytes(Ls,
 * count, N) bytes (16-byte aligned; 0 for an invalid group) holding every layer's device
 * arrays, the group's saved state and its workspace.  Page-locked host buffers, completion
 * and errors as for poetx_layer_step_host and the group calls. */
size_t poetx_group_step_host_bytes(const poetx_layer* Ls, int count, int N);
poetx_status poetx_group_step_host(const poetx_layer* Ls, int count, const void* const* x,
                                   const void* const* dy, int N, void* const* y,
                                   void* const* dx, float* const* dq_R, float* const* dq_P,
                                   void* dev, size_t dev_bytes, cudaStream_t stream);

/* Merge-then-reinitialize (POET skill page, Step 4 "Merge-Then-Reinitialize Optimization":
 * the current R W0 P is written back into W0 and the factors are reset to the identity).
 * Writes the weight that, with q_R = q_P = 0, makes the layer compute the map it computes
 * now:
 *   W0_new = Pi_n blkdiag(G_P)^T W' blkdiag(G_R)^T Pi_m^T,
 *   i.e.  W0_new[perm_n[r], perm_m[c]] = (blkdiag(G_P)^T W' blkdiag(G_R)^T)[r, c],
 * with G_R, G_P the CNP (order L->order) of the layer's current q_R, q_P and W' = L->Wp
 * (times L->w_scale per row for an int8 layer).  W0_new: [n, m] fp32, device, 16-byte
 * aligned, in the original (unpermuted) coordinates of W0.  fp32 accuracy throughout: the two
 * block-product passes over W' run on the tensor cores with the CNP's three-pass tf32 split
 * (b a multiple of 32; bit 0 of poetx_layer_cuda_core_steps clear), else on the CUDA cores.
 * The reinitialisation is then the caller's: set q_R and q_P to zero, draw new
 * permutations, and merge them into W0_new with poetx_merge_perm (an int8 layer first
 * re-quantises W0_new with poetx_quantize_rows_int8).  ws: at least
 * poetx_merge_reinit_workspace_bytes(L) bytes (0 for an invalid descriptor).  Errors as for
 * poetx_layer_fwd. */
size_t poetx_merge_reinit_workspace_bytes(const poetx_layer* L);
poetx_status poetx_merge_reinit(const poetx_layer* L, float* W0_new, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/* ----------------------------------------------------------------------------------------
 * Optimizer step on the packed triangles (POET-X summary page, "Core method" section 4:
 * optimizer state per stored parameter, b(b-1)/2 per block; "Practical guidance" 3: the
 * POET-XQ learning-rate factor gamma).  The pages name no optimizer: this is Adam (Kingma &
 * Ba, Algorithm 1) with decoupled weight decay, the library's reading:
 *   m <- beta1 m + (1 - beta1) g,  v <- beta2 v + (1 - beta2) g^2,
 *   q <- q - lr (m / (1 - beta1^step) / (sqrt(v / (1 - beta2^step)) + eps) + weight_decay q)
 * elementwise over `count` fp32 values (q, dq = g, m, v: device, 16-byte aligned, updated in
 * place except dq; m and v start at zero).  Use it after the data-parallel sum of dq; fold
 * gamma into lr for POET-XQ.  step >= 1 (the caller counts), 0 <= beta < 1; otherwise
 * POETX_ERR_ARG before any launch.
 * ------------------------------------------------------------------------------------- */
typedef struct poetx_adam {
  float lr, beta1, beta2, eps, weight_decay;
  int step;
} poetx_adam;
poetx_status poetx_adam_triu(float* q, const float* dq, float* m, float* v, long long count,
                             const poetx_adam* hp, cudaStream_t stream);

/* poetx_layer_bwd followed by the optimizer step above on both sides, the update applied by
 * the gradient-pack kernel as it writes each dq entry (one launch fewer; for single-replica
 * training, where nothing is summed between the gradient and the update).  Updates
 * L->q_R and L->q_P IN PLACE (the descriptor's const pointers are written: they must point
 * to writable device memory), with m_R, v_R [ceil(m/b), b(b-1)/2] and m_P, v_P
 * [ceil(n/b), b(b-1)/2] the fp32 Adam state (zero at step 1; device, 16-byte aligned).
 * dq_R, dq_P are written as by poetx_layer_bwd (with accumulate != 0 the update uses the
 * accumulated gradient).  The result equals poetx_layer_bwd + poetx_adam_triu bit for bit.
 * Errors: those of poetx_layer_bwd and poetx_adam_triu's, before any launch. */
poetx_status poetx_layer_bwd_adam(const poetx_layer* L, const void* x, const void* dy, int N,
                                  const void* saved, void* dx, float* dq_R, float* dq_P,
                                  int accumulate, const poetx_adam* hp, float* m_R, float* v_R,
                                  float* m_P, float* v_P, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* POETX_H */
