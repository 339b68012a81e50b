// The POET-X layer forward and backward, and the step-level entry points of its products.
//
// POET-X summary page ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation"), "Core method":
//   section 1 (eq. 3)  input-centric chain a = G_R^T x, b = W' a, z = G_P^T b, here in
//                      row-vector form  x~ = x[:, pi_m];  A = x~ blkdiag(G_R);  B = A W'^T;
//                      z~ = B blkdiag(G_P);  y[:, pi_n] = z~
//   section 2          permutations as index remaps, merged into W' beforehand
//   section 3          block-diagonal products as batched per-block GEMMs
//   section 4          CNP forward/backward (cnp.cu)
//   section 5          "fast" keeps B for the backward, "mem" recomputes it
//   section 6          POET-XQ: int8 W' dequantised inside the contraction (mem only)
// Backward (chain rule of the forward):  dz~ = dy[:, pi_n];  dG_P = B^T dz~ (per block);
//   dB = dz~ blkdiag(G_P)^T;  dA = dB W';  dG_R = x~^T dA (per block);
//   dx~ = dA blkdiag(G_R)^T;  dx[:, pi_m] = dx~;  dq = CNP backward of dG.
// Ragged last blocks (ceil(d/b) blocks per side) are computed with every internal array
// padded to whole blocks (see `padded`).  Host-side orchestration only: every step runs in
// this library's kernels, on the caller's stream except the overlapped dx scatter (a side
// stream) and the host-buffer steps' copies (an upload and a download stream), all forked
// from and joined back into the caller's stream; no device memory is allocated.
#include <atomic>
#include <mutex>

#include "cnp_umma.h"
#include "common.cuh"
#include "kernels.h"

namespace poetx {

static std::atomic<int> g_engine{0};  // 0: tensor cores where supported, 1: CUDA cores only
// fusion switches: bit 0 the W' contraction + the block product after it in one kernel,
// bit 1 the backward block product + its weight gradient in one kernel
static std::atomic<int> g_fuse{3};
static std::atomic<int> g_overlap{1};  // dx scatter beside the CNP backward (side stream)

static bool use_umma() { return g_engine.load() == 0 && umma_supported(); }

bool use_tensor_cores() { return g_engine.load() == 0; }

static int wgrad_splits(long long N, int nblk, int b) {
  // one wave: tiles x splits <= SMs (a partial second wave costs a whole extra tile time)
  const long long tiles = (long long)nblk * ((b + 127) / 128) * (b > 256 ? b / 256 : 1);
  long long s = (long long)sm_count() / tiles;
  long long smax = N / 256;
  if (smax < 1) smax = 1;
  if (s > smax) s = smax;
  if (s < 1) s = 1;
  return (int)s;
}

static int wgrad_chunk(long long N, int splits) {
  long long c = 64 * ((N + 64LL * splits - 1) / (64LL * splits));
  return (int)(c < 64 ? 64 : c);
}

// ---------------------------------------------------------------- step implementations
poetx_status blockdiag_impl(poetx_dtype dt, const void* X, long long N, int nblk, int b,
                            const void* G, int trans, const float* col_scale,
                            const int32_t* out_perm, void* Y, cudaStream_t s) {
  if (N == 0 || nblk == 0) return POETX_OK;
  if (dt == POETX_BF16 && use_umma() && b % 64 == 0 && b <= 512)
    return umma_blockdiag(X, N, nblk, b, G, trans, col_scale, out_perm, Y, s);
  const long long D = (long long)nblk * b;
  SimtGemm g{};
  g.M = (int)N; g.N = b; g.K = b; g.batch = nblk;
  g.A = X; g.sam = D; g.sak = 1; g.sab = b;
  g.B = G; g.sbk = trans ? 1 : b; g.sbn = trans ? b : 1; g.sbb = (long long)b * b;
  g.C = Y; g.scm = D; g.scn = 1; g.scb = b;
  g.colscale = col_scale; g.colscale_bstride = b;
  g.colperm = out_perm;
  g.ksplit = 1; g.kchunk = b;
  g.stage = ST_BLOCKDIAG;
  return launch_simt_gemm(dt, dt, dt, g, s);
}

poetx_status wgrad_impl(poetx_dtype dt, const void* X, const void* dY, long long N, int nblk,
                        int b, int splits, float* dG, cudaStream_t s) {
  if (nblk == 0) return POETX_OK;
  if (dt == POETX_BF16 && use_umma() && b % 64 == 0 && b <= 512)
    return umma_wgrad(X, dY, N, nblk, b, splits, dG, s);
  if (N == 0) {
    POETX_CUDA_TRY(cudaMemsetAsync(dG, 0, (size_t)splits * nblk * b * b * sizeof(float), s));
    return POETX_OK;
  }
  const long long D = (long long)nblk * b;
  SimtGemm g{};
  g.M = b; g.N = b; g.K = (int)N; g.batch = nblk;
  g.A = X; g.sam = 1; g.sak = D; g.sab = b;
  g.B = dY; g.sbk = D; g.sbn = 1; g.sbb = b;
  g.C = dG; g.scm = b; g.scn = 1; g.scb = (long long)b * b;
  g.ksplit = splits; g.kchunk = wgrad_chunk(N, splits);
  g.scs = (long long)nblk * b * b;
  g.stage = ST_WGRAD;
  // splits beyond the last token get an empty K range and write zeros
  return launch_simt_gemm(dt, dt, POETX_F32, g, s);
}

poetx_status wprime_impl(poetx_dtype act, poetx_dtype wdt, const void* A, long long N, int m,
                         int n, const void* W, const float* w_scale, int trans, void* C,
                         cudaStream_t s) {
  if (N == 0) return POETX_OK;
  // tensor cores for every bf16 shape the layer has (padded widths are multiples of b >= 64)
  if (act == POETX_BF16 && wdt == POETX_I8 && use_umma() && m % 64 == 0 && n % 64 == 0)
    return umma_wprime_i8(A, N, m, n, W, w_scale, trans, C, s);
  if (act == POETX_BF16 && wdt == POETX_BF16 && use_umma() && m % 64 == 0 && n % 64 == 0)
    return umma_wprime(A, N, m, n, W, trans, C, s);
  SimtGemm g{};
  g.M = (int)N; g.batch = 1; g.A = A; g.B = W; g.C = C;
  g.ksplit = 1;
  if (!trans) {
    g.N = n; g.K = m;
    g.sam = m; g.sak = 1;
    g.sbk = 1; g.sbn = m;
    g.scm = n; g.scn = 1;
    g.colscale = wdt == POETX_I8 ? w_scale : nullptr;
  } else {
    g.N = m; g.K = n;
    g.sam = n; g.sak = 1;
    g.sbk = m; g.sbn = 1;
    g.scm = m; g.scn = 1;
  }
  g.kchunk = g.K;
  g.stage = ST_WPRIME;
  return launch_simt_gemm(act, wdt, act, g, s);
}

// Ragged last block (POET-X summary, "Core method" §1: ceil(d/b) blocks per side).  Inside
// the layer every side is padded to whole blocks: the activations between the permutations
// have ceil(d/b) b columns (the gathers write the padding columns as zeros, the scatters read
// only the first d), the merged weight is [ceil(n/b) b, ceil(m/b) b] with zero padding, and
// the last block's Q is zero outside its r x r corner, so its G is the r x r factor with the
// identity beside it: the padding columns stay zero through every product and the results
// are those of the ragged blocks.
static int padded(int d, int b) { return (d + b - 1) / b * b; }
static int last_block(int d, int b) { return d % b; }  // 0: the last block is whole

// Appends the R side (m) and the P side (n) of a layer to a CNP side list.
static bool add_layer_sides(CnpSides& sd, const poetx_layer* L) {
  return sd.add(L->q_R, padded(L->m, L->b) / L->b, last_block(L->m, L->b)) &&
         sd.add(L->q_P, padded(L->n, L->b) / L->b, last_block(L->n, L->b));
}

static CnpSides layer_sides(const poetx_layer* L) {
  CnpSides sd;
  add_layer_sides(sd, L);
  return sd;
}

// The W' contraction and the block-diagonal product after it in one kernel (bf16 W', the
// tensor-core engine, shapes the fused kernel takes).
static bool fused_ok(const poetx_layer* L, long long N, int trans) {
  return L->act == POETX_BF16 && L->wdt == POETX_BF16 && use_umma() && (g_fuse.load() & 1) &&
         umma_wprime_fusable(N, padded(L->m, L->b), padded(L->n, L->b), trans, L->b);
}

// The backward block product and its weight gradient in one kernel (bf16, b = 128 or 256):
// on the P side always; on the R side unless the dx~ product is already fused into the
// backward W' contraction.
static bool bdw_ok(const poetx_layer* L) {
  return L->act == POETX_BF16 && use_umma() && (g_fuse.load() & 2) && umma_bdw_ok(L->b);
}
static bool bdw_side_R(const poetx_layer* L, long long N) {
  return bdw_ok(L) && !fused_ok(L, N, 1);
}

// ---------------------------------------------------------------- layer plumbing
struct Plan {
  // saved
  size_t GR, GP, Q2R, Q2P, Qs, Bsv, Xsv, saved_total;
  // forward workspace
  size_t f_xt, f_A, f_B, f_zt, fwd_total;
  // backward workspace: the chain's activations [0, bwd_chain), then the weight-gradient
  // partials and the CNP backward's scratch
  size_t b_xt, b_dzt, b_A, b_B, b_dB, b_dA, b_dxt, bwd_chain, b_dGP, b_dGR, b_cnp, bwd_total;
  size_t dGR_bytes, dGP_bytes;  // partial buffers, sized for either weight-gradient kernel
  int splitsR, splitsP;
};

static poetx_status validate(const poetx_layer* L) {
  if (!L) return POETX_ERR_ARG;
  if (L->m <= 0 || L->n <= 0 || L->b <= 0) return POETX_ERR_ARG;
  if (L->order != 3) return POETX_ERR_UNSUPPORTED;
  // a ragged side needs 16-byte rows at both widths
  if ((L->m % L->b || L->n % L->b) && (L->b % 8 || L->m % 8 || L->n % 8)) return POETX_ERR_SHAPE;
  if (L->act == POETX_F32) {
    if (L->wdt != POETX_F32) return POETX_ERR_DTYPE;
    if (L->b < 2 || L->b > 1024 || L->m % 4 || L->n % 4) return POETX_ERR_SHAPE;
  } else if (L->act == POETX_BF16) {
    if (L->wdt != POETX_BF16 && L->wdt != POETX_I8) return POETX_ERR_DTYPE;
    if (L->b != 64 && L->b != 128 && L->b != 256 && L->b != 512) return POETX_ERR_SHAPE;
    if (L->wdt == POETX_I8 && L->variant != POETX_MEM) return POETX_ERR_UNSUPPORTED;
    if (L->wdt == POETX_I8 && !L->w_scale) return POETX_ERR_ARG;
  } else {
    return POETX_ERR_DTYPE;
  }
  if (L->variant != POETX_FAST && L->variant != POETX_MEM) return POETX_ERR_ARG;
  if (!L->perm_m || !L->perm_n || !L->Wp || !L->q_R || !L->q_P) return POETX_ERR_ARG;
  if (!aligned16(L->Wp)) return POETX_ERR_ALIGN;
  return POETX_OK;
}

static Plan make_plan(const poetx_layer* L, long long N) {
  Plan p{};
  const size_t as = dtype_size(L->act);
  const size_t gs = L->act == POETX_F32 ? 4 : 2;
  // padded widths: every internal array has whole blocks
  const size_t m = padded(L->m, L->b), n = padded(L->n, L->b), b = L->b;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes, 256); return r; };
  // G_R and G_P (and Q_R^2, Q_P^2) are adjacent stacks so that one CNP launch covers both
  p.GR = take((m + n) * b * gs);
  p.GP = p.GR + m * b * gs;
  p.Q2R = take((m + n) * b * 4);
  p.Q2P = p.Q2R + m * b * 4;
  p.Qs = take((m + n) * b * 4);
  p.Bsv = L->variant == POETX_FAST ? take((size_t)N * n * as) : 0;
  p.Xsv = L->variant == POETX_FAST ? take((size_t)N * m * as) : 0;
  p.saved_total = o;

  o = 0;
  p.f_xt = L->variant == POETX_MEM ? take((size_t)N * m * as) : 0;
  p.f_A = take((size_t)N * m * as);
  p.f_B = L->variant == POETX_MEM ? take((size_t)N * n * as) : 0;
  p.f_zt = take((size_t)N * n * as);
  p.fwd_total = o;

  // token splits of the weight-gradient partials, from whichever kernel makes them; the
  // partial buffers are sized for either, so a switch flipped between sizing and calling
  // cannot overrun them
  const int wsR = wgrad_splits(N, (int)(m / b), L->b), wsP = wgrad_splits(N, (int)(n / b), L->b);
  const int fsR = bdw_splits(N, (int)(m / b), L->b), fsP = bdw_splits(N, (int)(n / b), L->b);
  p.splitsR = bdw_side_R(L, N) ? fsR : wsR;
  p.splitsP = bdw_ok(L) ? fsP : wsP;
  const size_t maxR = (size_t)(wsR > fsR ? wsR : fsR), maxP = (size_t)(wsP > fsP ? wsP : fsP);
  o = 0;
  p.b_xt = L->variant == POETX_MEM ? take((size_t)N * m * as) : 0;
  p.b_dzt = take((size_t)N * n * as);
  p.b_A = L->variant == POETX_MEM ? take((size_t)N * m * as) : 0;
  p.b_B = L->variant == POETX_MEM ? take((size_t)N * n * as) : 0;
  p.b_dB = take((size_t)N * n * as);
  p.b_dA = take((size_t)N * m * as);
  p.b_dxt = take((size_t)N * m * as);
  p.bwd_chain = o;
  p.dGP_bytes = maxP * n * b * 4;
  p.dGR_bytes = maxR * m * b * 4;
  p.b_dGP = take(p.dGP_bytes);
  p.b_dGR = take(p.dGR_bytes);
  p.b_cnp = take(cnp_bwd_scratch_bytes((int)((m + n) / b), (int)b));
  p.bwd_total = o;
  return p;
}

// ---------------------------------------------------------------- merge-then-reinitialize
// W0_new = Pi_n blkdiag(G_P)^T W' blkdiag(G_R)^T Pi_m^T: T = W' blkdiag(G_R)^T (the blocks of
// the columns), M = blkdiag(G_P)^T T (the blocks of the rows), then both permutations undone
// by one gather, W0_new[k, l] = M[inv_n[k], inv_m[l]].  fp32 throughout (CUDA cores): the
// merge runs once per many steps and its error would stay in W0.
struct MergePlan {
  size_t Qs, Q2, G, Gt, Wf, T, M, inv_m, inv_n, total;
};

// Merge-then-reinitialize takes the tensor cores (three-pass tf32 products) where the CNP
// engine takes the block size, else the CUDA cores.
static bool merge_on_tensor_cores(const poetx_layer* L) {
  return use_tensor_cores() && cnp_umma_ok(L->b);
}

static MergePlan merge_plan(const poetx_layer* L) {
  MergePlan p{};
  const size_t m = padded(L->m, L->b), n = padded(L->n, L->b), b = L->b;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes, 256); return r; };
  p.Qs = take((m + n) * b * 4);
  p.Q2 = take((m + n) * b * 4);
  p.G = take((m + n) * b * 4);
  const bool tc = merge_on_tensor_cores(L);
  p.Gt = tc ? take((m + n) * b * 4) : 0;
  // an fp32 copy of W' (int8: dequantised; bf16 for the tensor-core products)
  p.Wf = (L->wdt == POETX_I8 || (tc && L->wdt == POETX_BF16)) ? take(n * m * 4) : 0;
  p.T = take(n * m * 4);
  p.M = take(n * m * 4);
  p.inv_m = take(m * 4);
  p.inv_n = take(n * 4);
  p.total = o;
  return p;
}

template <typename T = void>
static T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <typename T = void>
static const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

}  // namespace poetx

using namespace poetx;

extern "C" poetx_status poetx_set_fusion(int on) {
  if (on < 0 || on > 3) return POETX_ERR_ARG;
  g_fuse.store(on);
  return POETX_OK;
}

extern "C" poetx_status poetx_set_gemm_engine(int engine) {
  if (engine != 0 && engine != 1) return POETX_ERR_ARG;
  g_engine.store(engine);
  return POETX_OK;
}

extern "C" size_t poetx_layer_workspace_bytes(const poetx_layer* L, int N, int phase) {
  if (validate(L) != POETX_OK || N < 0) return 0;
  const Plan p = make_plan(L, N);
  return phase == 0 ? p.fwd_total : p.bwd_total;
}

extern "C" size_t poetx_merge_reinit_workspace_bytes(const poetx_layer* L) {
  if (validate(L) != POETX_OK) return 0;
  return merge_plan(L).total;
}

extern "C" poetx_status poetx_merge_reinit(const poetx_layer* L, float* W0_new, void* ws,
                                           size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(validate(L));
  if (!W0_new || !ws) return POETX_ERR_ARG;
  if (!aligned16(W0_new) || !aligned16(ws)) return POETX_ERR_ALIGN;
  const MergePlan p = merge_plan(L);
  if (ws_bytes < p.total) return POETX_ERR_WORKSPACE;
  const int b = L->b, m = padded(L->m, b), n = padded(L->n, b);  // padded widths
  // G_R (blocks [0, m/b)) and G_P (blocks [m/b, (m+n)/b)) in fp32
  const CnpSides sides = layer_sides(L);
  const bool tc = merge_on_tensor_cores(L);
  float* G = at<float>(ws, p.G);
  float* Gt = tc ? at<float>(ws, p.Gt) : nullptr;
  POETX_TRY(cnp_forward_sides(sides, b, at<float>(ws, p.Qs), at<float>(ws, p.Q2), G, nullptr,
                              nullptr, stream, Gt));
  const float* GR = G;
  const float* GP = G + (size_t)m * b;
  float* T = at<float>(ws, p.T);
  float* M = at<float>(ws, p.M);
  if (tc) {
    // fp32 W' ([n, m]); T^T = (W' blkdiag(G_R)^T)^T ([m, n]); M = blkdiag(G_P)^T T ([n, m]),
    // computed as M^T = T^T blkdiag(G_P) with its transposed output
    const float* Wf = static_cast<const float*>(L->Wp);
    if (L->wdt == POETX_I8) {
      POETX_TRY(launch_dequant_rows(static_cast<const int8_t*>(L->Wp), L->w_scale, n, m,
                                    at<float>(ws, p.Wf), stream));
      Wf = at<float>(ws, p.Wf);
    } else if (L->wdt == POETX_BF16) {
      POETX_TRY(launch_widen_bf16(L->Wp, (long long)n * m, at<float>(ws, p.Wf), stream));
      Wf = at<float>(ws, p.Wf);
    }
    POETX_TRY(matrix_blockmm_tc(Wf, n, m / b, b, GR, nullptr, T, ST_MERGE_REINIT, stream));
    POETX_TRY(matrix_blockmm_tc(T, m, n / b, b, Gt + (size_t)m * b, nullptr, M, ST_MERGE_REINIT,
                                stream));
  } else {
    const void* Wsrc = L->Wp;
    poetx_dtype wt = L->wdt;
    if (L->wdt == POETX_I8) {
      POETX_TRY(launch_dequant_rows(static_cast<const int8_t*>(L->Wp), L->w_scale, n, m,
                                    at<float>(ws, p.Wf), stream));
      Wsrc = at<float>(ws, p.Wf);
      wt = POETX_F32;
    }
    SimtGemm g{};
    // T[:, jb:(j+1)b] = W'[:, jb:(j+1)b] G_R,j^T
    g.M = n; g.N = b; g.K = b; g.batch = m / b;
    g.A = Wsrc; g.sam = m; g.sak = 1; g.sab = b;
    g.B = GR; g.sbk = 1; g.sbn = b; g.sbb = (long long)b * b;
    g.C = T; g.scm = m; g.scn = 1; g.scb = b;
    g.ksplit = 1; g.kchunk = b;
    g.stage = ST_MERGE_REINIT;
    POETX_TRY(launch_simt_gemm(wt, POETX_F32, POETX_F32, g, stream));
    // M[jb:(j+1)b, :] = G_P,j^T T[jb:(j+1)b, :]
    g = SimtGemm{};
    g.M = b; g.N = m; g.K = b; g.batch = n / b;
    g.A = GP; g.sam = 1; g.sak = b; g.sab = (long long)b * b;
    g.B = T; g.sbk = m; g.sbn = 1; g.sbb = (long long)b * m;
    g.C = M; g.scm = m; g.scn = 1; g.scb = (long long)b * m;
    g.ksplit = 1; g.kchunk = b;
    g.stage = ST_MERGE_REINIT;
    POETX_TRY(launch_simt_gemm(POETX_F32, POETX_F32, POETX_F32, g, stream));
  }
  int32_t* inv_m = at<int32_t>(ws, p.inv_m);
  int32_t* inv_n = at<int32_t>(ws, p.inv_n);
  POETX_TRY(launch_invert_perms(L->perm_m, L->m, inv_m, L->perm_n, L->n, inv_n, stream));
  // the first L->n rows and L->m columns of the padded M hold the map
  return launch_perm_rows(4, false, M, L->n, L->m, inv_m, W0_new, inv_n, nullptr, nullptr,
                          stream, m, L->m);
}

extern "C" int poetx_layer_cuda_core_steps(const poetx_layer* L, int N) {
  if (validate(L) != POETX_OK || N < 0) return -1;
  const int b = L->b, mP = padded(L->m, b), nP = padded(L->n, b);
  int mask = 0;
  if (!(use_tensor_cores() && cnp_umma_ok(b))) mask |= 1;
  if (!(L->act == POETX_BF16 && use_umma() && b % 64 == 0 && b <= 512)) mask |= 2;
  if (!(L->act == POETX_BF16 && use_umma() && mP % 64 == 0 && nP % 64 == 0)) mask |= 4;
  return mask;
}

extern "C" size_t poetx_layer_saved_bytes(const poetx_layer* L, int N) {
  if (validate(L) != POETX_OK || N < 0) return 0;
  return make_plan(L, N).saved_total;
}

// Side stream of the overlapped permutation: the dx scatter runs beside the CNP backward,
// in the co-resident shape (one small CTA per SM in the shared
// memory the CNP product CTAs leave), forked from and joined back into the caller's stream
// by events.
namespace {
struct SideCtx {
  bool ready = false, failed = false;
  cudaStream_t ss = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;  // the events are reused: one layer call is enqueued at a time
SideCtx g_side[64];    // per device
}  // namespace

// The device's side context, created on first use; nullptr when overlap is off or the
// stream and events cannot be made (the calls then run everything on the caller's stream).
// A stream capture that forks into the side stream keeps it in that capture until the
// capture ends; a call on another stream in the meantime does not use it (its work would
// land in that graph), and runs everything on its own stream instead.
static SideCtx* side_ctx(cudaStream_t caller) {
  if (!g_overlap.load() || prof_enabled()) return nullptr;  // stage events need one stream
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return nullptr;
  SideCtx& c = g_side[d];
  if (!c.ready && !c.failed) {
    c.failed = cudaStreamCreateWithFlags(&c.ss, cudaStreamNonBlocking) != cudaSuccess ||
               cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess ||
               cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess;
    if (c.failed) cudaGetLastError();
    c.ready = !c.failed;
  }
  if (!c.ready) return nullptr;
  cudaStreamCaptureStatus side_st = cudaStreamCaptureStatusNone;
  unsigned long long side_id = 0;
  if (cudaStreamGetCaptureInfo(c.ss, &side_st, &side_id) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (side_st != cudaStreamCaptureStatusNone) {
    cudaStreamCaptureStatus own_st = cudaStreamCaptureStatusNone;
    unsigned long long own_id = 0;
    if (cudaStreamGetCaptureInfo(caller, &own_st, &own_id) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    if (own_st != cudaStreamCaptureStatusActive || own_id != side_id) return nullptr;
  }
  return &c;
}

extern "C" poetx_status poetx_set_overlap(int on) {
  if (on != 0 && on != 1) return POETX_ERR_ARG;
  g_overlap.store(on);
  return POETX_OK;
}

// Events a host-buffer step hands to the layer calls (all nullable): the forward waits for
// x_ready before its first read of x (the CNP runs before that, beside the upload); the
// backward waits for dy_ready before its first read of dy and records dx_done once dx is
// complete (the CNP backward then runs beside the download of dx).
struct StepHooks {
  cudaEvent_t x_ready = nullptr;
  cudaEvent_t dy_ready = nullptr;
  cudaEvent_t dx_done = nullptr;
};

// The layer's G blocks and what its forward keeps for the backward (fast: B and x~).
struct ChainSaved {
  const void* GR;  // [mP/b, b, b], activation precision
  const void* GP;  // [nP/b, b, b]
  void* B;         // fast: B = A W'^T [N, nP]; mem: nullptr
  void* xt;        // fast: x~ [N, mP]; mem: nullptr
};

static ChainSaved layer_chain_saved(const poetx_layer* L, const Plan& p, void* saved) {
  const bool fast = L->variant == POETX_FAST;
  return ChainSaved{at(saved, p.GR), at(saved, p.GP), fast ? at(saved, p.Bsv) : nullptr,
                    fast ? at(saved, p.Xsv) : nullptr};
}

// S3-S7 from the G blocks: x~ = x[:, pi_m], A = x~ blkdiag(G_R), B = A W'^T,
// z~ = B blkdiag(G_P), y[:, pi_n] = z~ (chain scratch at the Plan's forward offsets).
static poetx_status chain_fwd(const poetx_layer* L, const Plan& p, const void* x, int N, void* y,
                              const ChainSaved& cs, void* ws, cudaStream_t stream,
                              const StepHooks& hk) {
  if (N == 0) return POETX_OK;
  // m, n: the features of x and y; mP, nP: the padded widths of every internal array
  const int b = L->b, m = L->m, n = L->n, mP = padded(m, b), nP = padded(n, b);
  const poetx_dtype act = L->act;
  const size_t as = dtype_size(act);
  // fast keeps x~ and B for the backward (what default autograd keeps), mem keeps neither
  void* xt = cs.xt ? cs.xt : at(ws, p.f_xt);
  void* A = at(ws, p.f_A);
  void* B = cs.B ? cs.B : at(ws, p.f_B);
  if (hk.x_ready) POETX_CUDA_TRY(cudaStreamWaitEvent(stream, hk.x_ready, 0));
  POETX_TRY(launch_perm_rows(as, false, x, N, m, L->perm_m, xt, nullptr, nullptr, nullptr, stream,
                             m, mP));
  POETX_TRY(blockdiag_impl(act, xt, N, mP / b, b, cs.GR, 0, nullptr, nullptr, A, stream));
  void* zt = at(ws, p.f_zt);
  if (fused_ok(L, N, 0)) {
    // S5 + S6 on the same tiles (mem does not keep B)
    POETX_TRY(umma_wprime_fused(A, N, mP, nP, L->Wp, 0, cs.GP, b, cs.B, zt, stream));
  } else {
    POETX_TRY(wprime_impl(act, L->wdt, A, N, mP, nP, L->Wp, L->w_scale, 0, B, stream));
    POETX_TRY(blockdiag_impl(act, B, N, nP / b, b, cs.GP, 0, nullptr, nullptr, zt, stream));
  }
  // S7.  (Storing z~ through the permutation inside the product is supported, but its
  // 2-byte scattered stores are slower than this coalesced scatter pass.)
  return launch_perm_rows(as, true, zt, N, n, L->perm_n, y, nullptr, nullptr, nullptr, stream,
                          nP, n);
}

static poetx_status check_fwd_args(const poetx_layer* L, const void* x, int N, void* y,
                                   void* saved, void* ws) {
  POETX_TRY(validate(L));
  if (N < 0) return POETX_ERR_ARG;
  if (!saved || !ws || (N > 0 && (!x || !y))) return POETX_ERR_ARG;
  if (!aligned16(saved) || !aligned16(ws) || (N > 0 && (!aligned16(x) || !aligned16(y))))
    return POETX_ERR_ALIGN;
  return POETX_OK;
}

static poetx_status layer_fwd_impl(const poetx_layer* L, const void* x, int N, void* y,
                                   void* saved, void* ws, size_t ws_bytes, cudaStream_t stream,
                                   const StepHooks& hk) {
  POETX_TRY(check_fwd_args(L, x, N, y, saved, ws));
  const Plan p = make_plan(L, N);
  if (ws_bytes < p.fwd_total) return POETX_ERR_WORKSPACE;
  const int b = L->b;
  const bool f32 = L->act == POETX_F32;
  prof_begin(stream);
  // S1-S2: both CNPs in one pass over the m/b + n/b blocks; G in the activation precision
  // and Q^2 kept for the backward.  (Running the x gather beside them on the side stream
  // was measured: the CNP kernels slowed by about what the gather saved, and the join cost
  // the programmatic overlap of the next launch; so S3 follows them.)
  const CnpSides sides = layer_sides(L);
  POETX_TRY(cnp_forward_sides(sides, b, at<float>(saved, p.Qs), at<float>(saved, p.Q2R),
                              f32 ? at<float>(saved, p.GR) : nullptr,
                              f32 ? nullptr : at(saved, p.GR), nullptr, stream));
  return chain_fwd(L, p, x, N, y, layer_chain_saved(L, p, saved), ws, stream, hk);
}

extern "C" poetx_status poetx_layer_fwd(const poetx_layer* L, const void* x, int N, void* y,
                                        void* saved, void* ws, size_t ws_bytes,
                                        cudaStream_t stream) {
  return layer_fwd_impl(L, x, N, y, saved, ws, ws_bytes, stream, StepHooks{});
}

// S8-S13 from the G blocks and what the forward kept: dz~ = dy[:, pi_n], the weight-gradient
// partials dG_P [splitsP, nP/b, b, b] and dG_R [splitsR, mP/b, b, b], dx[:, pi_m] = dx~
// (chain scratch at the Plan's backward offsets).  With `side` set, the dx scatter runs on the
// side stream, forked here after the G_R weight gradient; the caller joins it (and holds the
// side stream's lock).
static poetx_status chain_bwd(const poetx_layer* L, const Plan& p, const void* x, const void* dy,
                              int N, const ChainSaved& cs, void* dx, float* dGR, float* dGP,
                              void* ws, cudaStream_t stream, const StepHooks& hk,
                              SideCtx* side) {
  const int b = L->b, m = L->m, n = L->n, mP = padded(m, b), nP = padded(n, b);
  const poetx_dtype act = L->act;
  const size_t as = dtype_size(act);
  const bool fast = L->variant == POETX_FAST;
  const void* xt = fast ? cs.xt : at(ws, p.b_xt);
  void* dzt = at(ws, p.b_dzt);
  void* dB = at(ws, p.b_dB);
  void* dA = at(ws, p.b_dA);
  if (N > 0) {
    if (!fast)  // mem: x~ is recomputed
      POETX_TRY(launch_perm_rows(as, false, x, N, m, L->perm_m, at(ws, p.b_xt), nullptr, nullptr,
                                 nullptr, stream, m, mP));
    if (hk.dy_ready) POETX_CUDA_TRY(cudaStreamWaitEvent(stream, hk.dy_ready, 0));
    POETX_TRY(launch_perm_rows(as, false, dy, N, n, L->perm_n, dzt, nullptr, nullptr, nullptr,
                               stream, n, nP));
  }
  const void* B;
  if (!fast) {  // recompute B = (x~ blkdiag(G_R)) W'^T
    void* A = at(ws, p.b_A);
    void* Bw = at(ws, p.b_B);
    POETX_TRY(blockdiag_impl(act, xt, N, mP / b, b, cs.GR, 0, nullptr, nullptr, A, stream));
    POETX_TRY(wprime_impl(act, L->wdt, A, N, mP, nP, L->Wp, L->w_scale, 0, Bw, stream));
    B = Bw;
  } else {
    B = cs.B;
  }
  const float* colscale = L->wdt == POETX_I8 ? L->w_scale : nullptr;
  if (bdw_ok(L)) {
    // S10 in one pass over dz~: dB = dz~ blkdiag(G_P)^T and dG_P = B^T dz~ (int8 weight:
    // dA = dB diag(s) W_q, the row scale folded into dB's columns)
    POETX_TRY(umma_bdw(dzt, B, N, nP / b, b, cs.GP, colscale, dB, p.splitsP, dGP, stream));
  } else {
    POETX_TRY(wgrad_impl(act, B, dzt, N, nP / b, b, p.splitsP, dGP, stream));
    POETX_TRY(blockdiag_impl(act, dzt, N, nP / b, b, cs.GP, 1, colscale, nullptr, dB, stream));
  }
  void* dxt = at(ws, p.b_dxt);
  if (fused_ok(L, N, 1)) {
    // S11 + the dx~ half of S12 on the same tiles
    POETX_TRY(umma_wprime_fused(dB, N, mP, nP, L->Wp, 1, cs.GR, b, dA, dxt, stream));
    POETX_TRY(wgrad_impl(act, xt, dA, N, mP / b, b, p.splitsR, dGR, stream));
  } else {
    POETX_TRY(wprime_impl(act, L->wdt, dB, N, mP, nP, L->Wp, L->w_scale, 1, dA, stream));
    if (bdw_side_R(L, N)) {
      // S12 in one pass over dA: dx~ = dA blkdiag(G_R)^T and dG_R = x~^T dA
      POETX_TRY(umma_bdw(dA, xt, N, mP / b, b, cs.GR, nullptr, dxt, p.splitsR, dGR, stream));
    } else {
      POETX_TRY(blockdiag_impl(act, dA, N, mP / b, b, cs.GR, 1, nullptr, nullptr, dxt, stream));
      POETX_TRY(wgrad_impl(act, xt, dA, N, mP / b, b, p.splitsR, dGR, stream));
    }
  }
  if (N == 0) return POETX_OK;
  if (side) {
    POETX_CUDA_TRY(cudaEventRecord(side->fork, stream));
    POETX_CUDA_TRY(cudaStreamWaitEvent(side->ss, side->fork, 0));
    const poetx_status st = launch_perm_rows_side(as, true, dxt, N, m, L->perm_m, dx, side->ss, mP, m);
    if (cudaEventRecord(side->join, side->ss) != cudaSuccess && st == POETX_OK) return POETX_ERR_CUDA;
    return st;
  }
  POETX_TRY(launch_perm_rows(as, true, dxt, N, m, L->perm_m, dx, nullptr, nullptr, nullptr, stream,
                             mP, m));
  if (hk.dx_done) POETX_CUDA_TRY(cudaEventRecord(hk.dx_done, stream));
  return POETX_OK;
}

static poetx_status check_bwd_args(const poetx_layer* L, const void* x, const void* dy, int N,
                                   const void* saved, void* dx, const void* ws) {
  POETX_TRY(validate(L));
  if (N < 0) return POETX_ERR_ARG;
  if (!saved || !ws || (N > 0 && (!x || !dy || !dx))) return POETX_ERR_ARG;
  if (!aligned16(saved) || !aligned16(ws) ||
      (N > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx))))
    return POETX_ERR_ALIGN;
  return POETX_OK;
}

static poetx_status layer_bwd_impl(const poetx_layer* L, const void* x, const void* dy, int N,
                                   const void* saved, void* dx, float* dq_R, float* dq_P,
                                   int accumulate, void* ws, size_t ws_bytes, cudaStream_t stream,
                                   const StepHooks& hk, const PackAdam* pa = nullptr) {
  POETX_TRY(check_bwd_args(L, x, dy, N, saved, dx, ws));
  if (!dq_R || !dq_P) return POETX_ERR_ARG;
  const Plan p = make_plan(L, N);
  if (ws_bytes < p.bwd_total) return POETX_ERR_WORKSPACE;
  const int b = L->b;
  const size_t as = dtype_size(L->act);
  prof_begin(stream);
  float* dGP = at<float>(ws, p.b_dGP);
  float* dGR = at<float>(ws, p.b_dGR);
  // S13 beside S14 when it can: the dx scatter does not feed the CNP backward.  It is
  // forked after the G_R weight gradient (a whole-GPU kernel that it would slow down), and
  // not when a download waits for dx (dx_done): the co-resident scatter is slower than the
  // whole-GPU one, and dx is then needed as early as possible.
  std::unique_lock<std::mutex> lk(g_side_mu, std::defer_lock);
  SideCtx* sc = nullptr;
  if (N > 0 && !hk.dx_done && perm_side_fits(as, L->m)) {
    lk.lock();
    sc = side_ctx(stream);
    if (!sc) lk.unlock();
  }
  poetx_status st = chain_bwd(L, p, x, dy, N, layer_chain_saved(L, p, const_cast<void*>(saved)),
                              dx, dGR, dGP, ws, stream, hk, sc);
  if (st == POETX_OK) {
    const CnpSides sides = layer_sides(L);
    CnpGrads gr;
    gr.dG[0] = dGR;
    gr.dG[1] = dGP;
    gr.splits[0] = p.splitsR;
    gr.splits[1] = p.splitsP;
    gr.dq[0] = dq_R;
    gr.dq[1] = dq_P;
    st = cnp_backward_sides(sides, at<float>(saved, p.Qs), at<float>(saved, p.Q2R), gr, b,
                            accumulate, at(ws, p.b_cnp), stream, pa);
  }
  if (sc && cudaStreamWaitEvent(stream, sc->join, 0) != cudaSuccess && st == POETX_OK)
    st = POETX_ERR_CUDA;
  return st;
}

extern "C" poetx_status poetx_layer_bwd(const poetx_layer* L, const void* x, const void* dy, int N,
                                        const void* saved, void* dx, float* dq_R, float* dq_P,
                                        int accumulate, void* ws, size_t ws_bytes,
                                        cudaStream_t stream) {
  return layer_bwd_impl(L, x, dy, N, saved, dx, dq_R, dq_P, accumulate, ws, ws_bytes, stream,
                        StepHooks{});
}

extern "C" poetx_status poetx_layer_bwd_adam(const poetx_layer* L, const void* x, const void* dy,
                                             int N, const void* saved, void* dx, float* dq_R,
                                             float* dq_P, int accumulate, const poetx_adam* hp,
                                             float* m_R, float* v_R, float* m_P, float* v_P,
                                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(validate(L));
  PackAdam pa{};
  POETX_TRY(adam_params(hp, &pa.h));
  if (!m_R || !v_R || !m_P || !v_P) return POETX_ERR_ARG;
  if (!aligned16(m_R) || !aligned16(v_R) || !aligned16(m_P) || !aligned16(v_P))
    return POETX_ERR_ALIGN;
  // the optimizer writes the layer's parameters in place (nothing after the gradient pack
  // reads them in this call; the CNP backward works from the unpacked Q of the forward)
  pa.q[0] = const_cast<float*>(L->q_R);
  pa.q[1] = const_cast<float*>(L->q_P);
  pa.m[0] = m_R;
  pa.v[0] = v_R;
  pa.m[1] = m_P;
  pa.v[1] = v_P;
  return layer_bwd_impl(L, x, dy, N, saved, dx, dq_R, dq_P, accumulate, ws, ws_bytes, stream,
                        StepHooks{}, &pa);
}

// ---------------------------------------------------------------- layer groups
// The layers of a group (e.g. the linears of a transformer block) share one stack of CNP
// blocks: layer i's R blocks, then its P blocks, for i = 0, 1, ...  Its Q, Q^2 and G are
// computed by one CNP forward over the whole stack and its dq by one CNP backward, so that
// a block's few hundred small b x b products fill the GPU in a few launches instead of a
// latency-bound wave per layer; each layer's forward and backward chain runs on its own
// between them.  saved: the stacks, then per layer what its forward keeps (fast: B and x~).
// ws: the chain scratch (one region shared by the layers, which run one after the other
// on the caller's stream), every layer's weight-gradient partials (written by its backward
// chain, read by the group's CNP backward) and the CNP backward's scratch.
constexpr int kMaxGroup = kMaxSides / 2;
static_assert(kMaxGroup == POETX_GROUP_MAX_LAYERS, "group size limit");

struct GroupPlan {
  int count = 0;
  int blk0[kMaxGroup + 1] = {};  // first stack block of layer i (R side, then P side)
  size_t G = 0, Qs = 0, Q2 = 0;
  size_t Bsv[kMaxGroup] = {}, Xsv[kMaxGroup] = {};
  size_t saved_total = 0;
  size_t chain = 0, chain_bytes = 0;
  size_t dGR[kMaxGroup] = {}, dGP[kMaxGroup] = {};
  size_t cnp = 0, ws_total = 0;
  Plan lp[kMaxGroup];
};

static poetx_status validate_group(const poetx_layer* Ls, int count) {
  if (!Ls || count < 1 || count > kMaxGroup) return POETX_ERR_ARG;
  for (int i = 0; i < count; ++i) {
    POETX_TRY(validate(&Ls[i]));
    if (Ls[i].b != Ls[0].b) return POETX_ERR_SHAPE;
    if (Ls[i].act != Ls[0].act) return POETX_ERR_DTYPE;
  }
  return POETX_OK;
}

static GroupPlan group_plan(const poetx_layer* Ls, int count, long long N) {
  GroupPlan g;
  g.count = count;
  const size_t b = Ls[0].b;
  const size_t gs = Ls[0].act == POETX_F32 ? 4 : 2;
  for (int i = 0; i < count; ++i) {
    g.lp[i] = make_plan(&Ls[i], N);
    g.blk0[i + 1] = g.blk0[i] + (padded(Ls[i].m, Ls[i].b) + padded(Ls[i].n, Ls[i].b)) / Ls[i].b;
  }
  const size_t nb = g.blk0[count];
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes, 256); return r; };
  g.G = take(nb * b * b * gs);
  g.Qs = take(nb * b * b * 4);
  g.Q2 = take(nb * b * b * 4);
  for (int i = 0; i < count; ++i) {
    const bool fast = Ls[i].variant == POETX_FAST;
    const size_t as = dtype_size(Ls[i].act);
    const size_t m = padded(Ls[i].m, Ls[i].b), n = padded(Ls[i].n, Ls[i].b);
    g.Bsv[i] = fast ? take((size_t)N * n * as) : 0;
    g.Xsv[i] = fast ? take((size_t)N * m * as) : 0;
  }
  g.saved_total = o;
  o = 0;
  for (int i = 0; i < count; ++i) {
    const size_t need = g.lp[i].fwd_total > g.lp[i].bwd_chain ? g.lp[i].fwd_total : g.lp[i].bwd_chain;
    if (need > g.chain_bytes) g.chain_bytes = need;
  }
  g.chain = take(g.chain_bytes);
  for (int i = 0; i < count; ++i) {
    const size_t m = padded(Ls[i].m, Ls[i].b), n = padded(Ls[i].n, Ls[i].b);
    g.dGR[i] = take(g.lp[i].dGR_bytes);
    g.dGP[i] = take(g.lp[i].dGP_bytes);
  }
  g.cnp = take(cnp_bwd_scratch_bytes((int)nb, (int)b));
  g.ws_total = o;
  return g;
}

static CnpSides group_sides(const poetx_layer* Ls, int count) {
  CnpSides sd;
  for (int i = 0; i < count; ++i) add_layer_sides(sd, &Ls[i]);
  return sd;
}

static ChainSaved group_chain_saved(const poetx_layer* Ls, const GroupPlan& g, int i,
                                    const void* saved) {
  const size_t b = Ls[0].b, gs = Ls[0].act == POETX_F32 ? 4 : 2;
  const size_t r0 = (size_t)g.blk0[i], p0 = r0 + padded(Ls[i].m, Ls[i].b) / Ls[i].b;
  void* sv = const_cast<void*>(saved);
  const bool fast = Ls[i].variant == POETX_FAST;
  return ChainSaved{at(sv, g.G + r0 * b * b * gs), at(sv, g.G + p0 * b * b * gs),
                    fast ? at(sv, g.Bsv[i]) : nullptr, fast ? at(sv, g.Xsv[i]) : nullptr};
}

extern "C" size_t poetx_group_saved_bytes(const poetx_layer* Ls, int count, int N) {
  if (validate_group(Ls, count) != POETX_OK || N < 0) return 0;
  return group_plan(Ls, count, N).saved_total;
}

extern "C" size_t poetx_group_workspace_bytes(const poetx_layer* Ls, int count, int N) {
  if (validate_group(Ls, count) != POETX_OK || N < 0) return 0;
  return group_plan(Ls, count, N).ws_total;
}

extern "C" poetx_status poetx_group_cnp_fwd(const poetx_layer* Ls, int count, int N, void* saved,
                                            cudaStream_t stream) {
  POETX_TRY(validate_group(Ls, count));
  if (N < 0 || !saved) return POETX_ERR_ARG;
  if (!aligned16(saved)) return POETX_ERR_ALIGN;
  const GroupPlan g = group_plan(Ls, count, N);
  const bool f32 = Ls[0].act == POETX_F32;
  prof_begin(stream);
  return cnp_forward_sides(group_sides(Ls, count), Ls[0].b, at<float>(saved, g.Qs),
                           at<float>(saved, g.Q2), f32 ? at<float>(saved, g.G) : nullptr,
                           f32 ? nullptr : at(saved, g.G), nullptr, stream);
}

extern "C" poetx_status poetx_group_layer_fwd(const poetx_layer* Ls, int count, int i,
                                              const void* x, int N, void* y, void* saved,
                                              void* ws, size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(validate_group(Ls, count));
  if (i < 0 || i >= count) return POETX_ERR_ARG;
  POETX_TRY(check_fwd_args(&Ls[i], x, N, y, saved, ws));
  const GroupPlan g = group_plan(Ls, count, N);
  if (ws_bytes < g.ws_total) return POETX_ERR_WORKSPACE;
  prof_begin(stream);
  return chain_fwd(&Ls[i], g.lp[i], x, N, y, group_chain_saved(Ls, g, i, saved),
                   at(ws, g.chain), stream, StepHooks{});
}

extern "C" poetx_status poetx_group_layer_bwd(const poetx_layer* Ls, int count, int i,
                                              const void* x, const void* dy, int N,
                                              const void* saved, void* dx, void* ws,
                                              size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(validate_group(Ls, count));
  if (i < 0 || i >= count) return POETX_ERR_ARG;
  POETX_TRY(check_bwd_args(&Ls[i], x, dy, N, saved, dx, ws));
  const GroupPlan g = group_plan(Ls, count, N);
  if (ws_bytes < g.ws_total) return POETX_ERR_WORKSPACE;
  prof_begin(stream);
  // the dx scatter stays on the caller's stream: the next layer's chain follows it, not a
  // CNP backward it could hide under
  return chain_bwd(&Ls[i], g.lp[i], x, dy, N, group_chain_saved(Ls, g, i, saved), dx,
                   at<float>(ws, g.dGR[i]), at<float>(ws, g.dGP[i]), at(ws, g.chain), stream,
                   StepHooks{}, nullptr);
}

extern "C" poetx_status poetx_group_cnp_bwd(const poetx_layer* Ls, int count, int N,
                                            const void* saved, float* const* dq_R,
                                            float* const* dq_P, int accumulate, void* ws,
                                            size_t ws_bytes, cudaStream_t stream) {
  POETX_TRY(validate_group(Ls, count));
  if (N < 0 || !saved || !ws || !dq_R || !dq_P) return POETX_ERR_ARG;
  if (!aligned16(saved) || !aligned16(ws)) return POETX_ERR_ALIGN;
  for (int i = 0; i < count; ++i) {
    if (!dq_R[i] || !dq_P[i]) return POETX_ERR_ARG;
    if (!aligned16(dq_R[i]) || !aligned16(dq_P[i])) return POETX_ERR_ALIGN;
  }
  const GroupPlan g = group_plan(Ls, count, N);
  if (ws_bytes < g.ws_total) return POETX_ERR_WORKSPACE;
  prof_begin(stream);
  CnpGrads gr;
  for (int i = 0; i < count; ++i) {
    gr.dG[2 * i] = at<float>(ws, g.dGR[i]);
    gr.splits[2 * i] = g.lp[i].splitsR;
    gr.dq[2 * i] = dq_R[i];
    gr.dG[2 * i + 1] = at<float>(ws, g.dGP[i]);
    gr.splits[2 * i + 1] = g.lp[i].splitsP;
    gr.dq[2 * i + 1] = dq_P[i];
  }
  return cnp_backward_sides(group_sides(Ls, count), at<float>(saved, g.Qs),
                            at<float>(saved, g.Q2), gr, Ls[0].b, accumulate, at(ws, g.cnp),
                            stream);
}

// ---------------------------------------------------------------- host-buffer step
// One forward + backward with the caller's host buffers: the uploads and the downloads run
// on two copy streams of the library's own (the host link carries both directions at once),
// beside the kernels on the caller's stream:
//   upload stream    x up | dy up |
//   download stream               | y down (after the forward) | dx down | dq down
//   caller stream    CNP fwd | (wait x) fwd chain | (wait dy) bwd chain | CNP bwd
// so the CNP forward hides part of the x upload, the dy upload runs under the forward, the
// y download under the backward and the dx download under the CNP backward.
struct StepPlan {
  size_t x, dy, y, dx, dqR, dqP, saved, ws, ws_bytes, total;
};

static StepPlan step_plan(const poetx_layer* L, long long N) {
  StepPlan sp{};
  const Plan p = make_plan(L, N);
  const size_t as = dtype_size(L->act);
  const size_t m = L->m, n = L->n, b = L->b;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes, 256); return r; };
  sp.x = take(N * m * as);
  sp.dy = take(N * n * as);
  sp.y = take(N * n * as);
  sp.dx = take(N * m * as);
  sp.dqR = take((m + b - 1) / b * (b * (b - 1) / 2) * 4);
  sp.dqP = take((n + b - 1) / b * (b * (b - 1) / 2) * 4);
  sp.saved = take(p.saved_total);
  sp.ws_bytes = p.fwd_total > p.bwd_total ? p.fwd_total : p.bwd_total;
  sp.ws = take(sp.ws_bytes);
  sp.total = o;
  return sp;
}

namespace {
enum { EV_START, EV_X, EV_DY, EV_Y, EV_DX, EV_DQ, EV_UP, EV_DONE, EV_COUNT };
// per layer of a group step: x uploaded, dy uploaded, y computed, dx computed
enum { GEV_X, GEV_DY, GEV_Y, GEV_DX, GEV_COUNT };
struct CopyCtx {
  bool ready = false;
  cudaStream_t us = nullptr, ds = nullptr;  // uploads, downloads
  cudaEvent_t ev[EV_COUNT] = {};
  cudaEvent_t gev[GEV_COUNT][POETX_GROUP_MAX_LAYERS] = {};
};
std::mutex g_step_mu;  // the events are reused: one step is enqueued at a time
CopyCtx g_copy[64];    // per device

// The device's copy streams and events, created on first use (under g_step_mu).
poetx_status copy_ctx(CopyCtx** out) {
  int d = 0;
  POETX_CUDA_TRY(cudaGetDevice(&d));
  if (d < 0 || d >= 64) return POETX_ERR_UNSUPPORTED;
  CopyCtx& c = g_copy[d];
  if (!c.ready) {
    POETX_CUDA_TRY(cudaStreamCreateWithFlags(&c.us, cudaStreamNonBlocking));
    POETX_CUDA_TRY(cudaStreamCreateWithFlags(&c.ds, cudaStreamNonBlocking));
    for (int i = 0; i < EV_COUNT; ++i)
      POETX_CUDA_TRY(cudaEventCreateWithFlags(&c.ev[i], cudaEventDisableTiming));
    for (int k = 0; k < GEV_COUNT; ++k)
      for (int i = 0; i < POETX_GROUP_MAX_LAYERS; ++i)
        POETX_CUDA_TRY(cudaEventCreateWithFlags(&c.gev[k][i], cudaEventDisableTiming));
    c.ready = true;
  }
  *out = &c;
  return POETX_OK;
}
}  // namespace

// The caller's stream waits for both copy streams (also after an error, so that nothing the
// streams still do is left unordered with the caller's later work).
static void join_copy_streams(CopyCtx& c, cudaStream_t stream, poetx_status& st) {
  const cudaError_t e1 = cudaEventRecord(c.ev[EV_UP], c.us);
  const cudaError_t e2 = cudaEventRecord(c.ev[EV_DONE], c.ds);
  const cudaError_t e3 = e1 == cudaSuccess ? cudaStreamWaitEvent(stream, c.ev[EV_UP], 0) : e1;
  const cudaError_t e4 = e2 == cudaSuccess ? cudaStreamWaitEvent(stream, c.ev[EV_DONE], 0) : e2;
  if (st == POETX_OK && (e3 != cudaSuccess || e4 != cudaSuccess)) st = POETX_ERR_CUDA;
}

extern "C" size_t poetx_layer_step_host_bytes(const poetx_layer* L, int N) {
  if (validate(L) != POETX_OK || N < 0) return 0;
  return step_plan(L, N).total;
}

extern "C" poetx_status poetx_layer_step_host(const poetx_layer* L, const void* x, const void* dy,
                                              int N, void* y, void* dx, float* dq_R, float* dq_P,
                                              void* dev, size_t dev_bytes, cudaStream_t stream) {
  POETX_TRY(validate(L));
  if (N < 0) return POETX_ERR_ARG;
  if (!dev || !dq_R || !dq_P || (N > 0 && (!x || !dy || !y || !dx))) return POETX_ERR_ARG;
  if (!aligned16(dev)) return POETX_ERR_ALIGN;
  const StepPlan sp = step_plan(L, N);
  if (dev_bytes < sp.total) return POETX_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lk(g_step_mu);
  CopyCtx* cp = nullptr;
  POETX_TRY(copy_ctx(&cp));
  CopyCtx& c = *cp;
  uint8_t* base = static_cast<uint8_t*>(dev);
  const size_t as = dtype_size(L->act);
  const size_t m = L->m, n = L->n, b = L->b;
  const size_t xb = (size_t)N * m * as, yb = (size_t)N * n * as;
  const size_t qRb = (m + b - 1) / b * (b * (b - 1) / 2) * 4;
  const size_t qPb = (n + b - 1) / b * (b * (b - 1) / 2) * 4;
  // the copy streams start after the caller's earlier work (which may still use `dev`)
  POETX_CUDA_TRY(cudaEventRecord(c.ev[EV_START], stream));
  POETX_CUDA_TRY(cudaStreamWaitEvent(c.us, c.ev[EV_START], 0));
  POETX_CUDA_TRY(cudaStreamWaitEvent(c.ds, c.ev[EV_START], 0));
  StepHooks fh, bh;
  poetx_status st = POETX_OK;
  auto cuda = [&](cudaError_t e) {
    if (st == POETX_OK && e != cudaSuccess) st = POETX_ERR_CUDA;
  };
  if (N > 0) {
    cuda(cudaMemcpyAsync(base + sp.x, x, xb, cudaMemcpyHostToDevice, c.us));
    cuda(cudaEventRecord(c.ev[EV_X], c.us));
    cuda(cudaMemcpyAsync(base + sp.dy, dy, yb, cudaMemcpyHostToDevice, c.us));
    cuda(cudaEventRecord(c.ev[EV_DY], c.us));
    fh.x_ready = c.ev[EV_X];
    bh.dy_ready = c.ev[EV_DY];
    bh.dx_done = c.ev[EV_DX];
  }
  if (st == POETX_OK)
    st = layer_fwd_impl(L, base + sp.x, N, base + sp.y, base + sp.saved, base + sp.ws,
                        sp.ws_bytes, stream, fh);
  if (st == POETX_OK && N > 0) {
    cuda(cudaEventRecord(c.ev[EV_Y], stream));
    cuda(cudaStreamWaitEvent(c.ds, c.ev[EV_Y], 0));
    cuda(cudaMemcpyAsync(y, base + sp.y, yb, cudaMemcpyDeviceToHost, c.ds));
  }
  if (st == POETX_OK)
    st = layer_bwd_impl(L, base + sp.x, base + sp.dy, N, base + sp.saved, base + sp.dx,
                        reinterpret_cast<float*>(base + sp.dqR),
                        reinterpret_cast<float*>(base + sp.dqP), 0, base + sp.ws, sp.ws_bytes,
                        stream, bh);
  if (st == POETX_OK && N > 0) {
    cuda(cudaStreamWaitEvent(c.ds, c.ev[EV_DX], 0));
    cuda(cudaMemcpyAsync(dx, base + sp.dx, xb, cudaMemcpyDeviceToHost, c.ds));
  }
  if (st == POETX_OK) {
    cuda(cudaEventRecord(c.ev[EV_DQ], stream));
    cuda(cudaStreamWaitEvent(c.ds, c.ev[EV_DQ], 0));
    cuda(cudaMemcpyAsync(dq_R, base + sp.dqR, qRb, cudaMemcpyDeviceToHost, c.ds));
    cuda(cudaMemcpyAsync(dq_P, base + sp.dqP, qPb, cudaMemcpyDeviceToHost, c.ds));
  }
  // the caller's stream is done with the step only when both copy streams are
  join_copy_streams(c, stream, st);
  return st;
}

// ---------------------------------------------------------------- host-buffer group step
// One training step of a layer group with host buffers: every layer's x and dy go up on the
// upload stream in the order the kernels need them (x_0 .. x_{c-1}, then dy_{c-1} .. dy_0),
// every y comes down as soon as its forward chain has written it, every dx as soon as its
// backward chain has, and the dq of every layer after the group's CNP backward, on the
// download stream; the kernels run on the caller's stream between them, each chain waiting
// only for its own inputs.
struct GroupStepPlan {
  size_t x[kMaxGroup], dy[kMaxGroup], y[kMaxGroup], dx[kMaxGroup], dqR[kMaxGroup],
      dqP[kMaxGroup];
  size_t saved, ws, ws_bytes, total;
};

static GroupStepPlan group_step_plan(const poetx_layer* Ls, int count, long long N) {
  GroupStepPlan sp{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += align_up(bytes, 256); return r; };
  for (int i = 0; i < count; ++i) {
    const size_t as = dtype_size(Ls[i].act), m = Ls[i].m, n = Ls[i].n, b = Ls[i].b;
    sp.x[i] = take(N * m * as);
    sp.dy[i] = take(N * n * as);
    sp.y[i] = take(N * n * as);
    sp.dx[i] = take(N * m * as);
    sp.dqR[i] = take((m + b - 1) / b * (b * (b - 1) / 2) * 4);
    sp.dqP[i] = take((n + b - 1) / b * (b * (b - 1) / 2) * 4);
  }
  const GroupPlan g = group_plan(Ls, count, N);
  sp.saved = take(g.saved_total);
  sp.ws_bytes = g.ws_total;
  sp.ws = take(sp.ws_bytes);
  sp.total = o;
  return sp;
}

extern "C" size_t poetx_group_step_host_bytes(const poetx_layer* Ls, int count, int N) {
  if (validate_group(Ls, count) != POETX_OK || N < 0) return 0;
  return group_step_plan(Ls, count, N).total;
}

extern "C" poetx_status poetx_group_step_host(const poetx_layer* Ls, int count,
                                              const void* const* x, const void* const* dy, int N,
                                              void* const* y, void* const* dx,
                                              float* const* dq_R, float* const* dq_P, void* dev,
                                              size_t dev_bytes, cudaStream_t stream) {
  POETX_TRY(validate_group(Ls, count));
  if (N < 0 || !dev || !dq_R || !dq_P) return POETX_ERR_ARG;
  if (N > 0 && (!x || !dy || !y || !dx)) return POETX_ERR_ARG;
  for (int i = 0; i < count; ++i) {
    if (!dq_R[i] || !dq_P[i]) return POETX_ERR_ARG;
    if (N > 0 && (!x[i] || !dy[i] || !y[i] || !dx[i])) return POETX_ERR_ARG;
  }
  if (!aligned16(dev)) return POETX_ERR_ALIGN;
  const GroupStepPlan sp = group_step_plan(Ls, count, N);
  if (dev_bytes < sp.total) return POETX_ERR_WORKSPACE;
  const GroupPlan g = group_plan(Ls, count, N);
  std::lock_guard<std::mutex> lk(g_step_mu);
  CopyCtx* cp = nullptr;
  POETX_TRY(copy_ctx(&cp));
  CopyCtx& c = *cp;
  uint8_t* base = static_cast<uint8_t*>(dev);
  void* saved = base + sp.saved;
  void* ws = base + sp.ws;
  POETX_CUDA_TRY(cudaEventRecord(c.ev[EV_START], stream));
  POETX_CUDA_TRY(cudaStreamWaitEvent(c.us, c.ev[EV_START], 0));
  POETX_CUDA_TRY(cudaStreamWaitEvent(c.ds, c.ev[EV_START], 0));
  poetx_status st = POETX_OK;
  auto cuda = [&](cudaError_t e) {
    if (st == POETX_OK && e != cudaSuccess) st = POETX_ERR_CUDA;
  };
  auto abytes = [&](int i, bool in) {
    return (size_t)N * (in ? Ls[i].m : Ls[i].n) * dtype_size(Ls[i].act);
  };
  if (N > 0) {
    for (int i = 0; i < count; ++i) {
      cuda(cudaMemcpyAsync(base + sp.x[i], x[i], abytes(i, true), cudaMemcpyHostToDevice, c.us));
      cuda(cudaEventRecord(c.gev[GEV_X][i], c.us));
    }
    for (int i = count - 1; i >= 0; --i) {
      cuda(cudaMemcpyAsync(base + sp.dy[i], dy[i], abytes(i, false), cudaMemcpyHostToDevice,
                           c.us));
      cuda(cudaEventRecord(c.gev[GEV_DY][i], c.us));
    }
  }
  const bool f32 = Ls[0].act == POETX_F32;
  if (st == POETX_OK) {
    prof_begin(stream);
    st = cnp_forward_sides(group_sides(Ls, count), Ls[0].b, at<float>(saved, g.Qs),
                           at<float>(saved, g.Q2), f32 ? at<float>(saved, g.G) : nullptr,
                           f32 ? nullptr : at(saved, g.G), nullptr, stream);
  }
  for (int i = 0; i < count && st == POETX_OK && N > 0; ++i) {
    StepHooks h;
    h.x_ready = c.gev[GEV_X][i];
    st = chain_fwd(&Ls[i], g.lp[i], base + sp.x[i], N, base + sp.y[i],
                   group_chain_saved(Ls, g, i, saved), at(ws, g.chain), stream, h);
    if (st != POETX_OK) break;
    cuda(cudaEventRecord(c.gev[GEV_Y][i], stream));
    cuda(cudaStreamWaitEvent(c.ds, c.gev[GEV_Y][i], 0));
    cuda(cudaMemcpyAsync(y[i], base + sp.y[i], abytes(i, false), cudaMemcpyDeviceToHost, c.ds));
  }
  for (int i = count - 1; i >= 0 && st == POETX_OK; --i) {
    StepHooks h;
    h.dy_ready = N > 0 ? c.gev[GEV_DY][i] : nullptr;
    h.dx_done = N > 0 ? c.gev[GEV_DX][i] : nullptr;
    st = chain_bwd(&Ls[i], g.lp[i], base + sp.x[i], base + sp.dy[i], N,
                   group_chain_saved(Ls, g, i, saved), base + sp.dx[i],
                   at<float>(ws, g.dGR[i]), at<float>(ws, g.dGP[i]), at(ws, g.chain), stream, h,
                   nullptr);
    if (st != POETX_OK || N == 0) continue;
    cuda(cudaStreamWaitEvent(c.ds, c.gev[GEV_DX][i], 0));
    cuda(cudaMemcpyAsync(dx[i], base + sp.dx[i], abytes(i, true), cudaMemcpyDeviceToHost, c.ds));
  }
  if (st == POETX_OK) {
    CnpGrads gr;
    for (int i = 0; i < count; ++i) {
      gr.dG[2 * i] = at<float>(ws, g.dGR[i]);
      gr.splits[2 * i] = g.lp[i].splitsR;
      gr.dq[2 * i] = reinterpret_cast<float*>(base + sp.dqR[i]);
      gr.dG[2 * i + 1] = at<float>(ws, g.dGP[i]);
      gr.splits[2 * i + 1] = g.lp[i].splitsP;
      gr.dq[2 * i + 1] = reinterpret_cast<float*>(base + sp.dqP[i]);
    }
    st = cnp_backward_sides(group_sides(Ls, count), at<float>(saved, g.Qs),
                            at<float>(saved, g.Q2), gr, Ls[0].b, 0, at(ws, g.cnp), stream);
  }
  if (st == POETX_OK) {
    cuda(cudaEventRecord(c.ev[EV_DQ], stream));
    cuda(cudaStreamWaitEvent(c.ds, c.ev[EV_DQ], 0));
    for (int i = 0; i < count; ++i) {
      const size_t b = Ls[i].b, tri = b * (b - 1) / 2;
      cuda(cudaMemcpyAsync(dq_R[i], base + sp.dqR[i], (Ls[i].m + b - 1) / b * tri * 4,
                           cudaMemcpyDeviceToHost, c.ds));
      cuda(cudaMemcpyAsync(dq_P[i], base + sp.dqP[i], (Ls[i].n + b - 1) / b * tri * 4,
                           cudaMemcpyDeviceToHost, c.ds));
    }
  }
  join_copy_streams(c, stream, st);
  return st;
}

// ---------------------------------------------------------------- step entry points
static poetx_status check_act(poetx_dtype dt, int b) {
  if (dt == POETX_BF16) return (b == 64 || b == 128 || b == 256 || b == 512) ? POETX_OK : POETX_ERR_SHAPE;
  if (dt == POETX_F32) return (b >= 1 && b <= 1024) ? POETX_OK : POETX_ERR_SHAPE;
  return POETX_ERR_DTYPE;
}

extern "C" poetx_status poetx_blockdiag_mm(poetx_dtype dt, const void* X, int N, int nblk, int b,
                                           const void* G, int trans, const float* col_scale,
                                           const int32_t* out_perm, void* Y, cudaStream_t stream) {
  POETX_TRY(check_act(dt, b));
  if (N < 0 || nblk < 0) return POETX_ERR_ARG;
  if (N == 0 || nblk == 0) return POETX_OK;
  if (!X || !G || !Y) return POETX_ERR_ARG;
  if (!aligned16(X) || !aligned16(G) || !aligned16(Y)) return POETX_ERR_ALIGN;
  if (out_perm && X == Y) return POETX_ERR_ARG;
  return blockdiag_impl(dt, X, N, nblk, b, G, trans, col_scale, out_perm, Y, stream);
}

extern "C" poetx_status poetx_blockdiag_wgrad(poetx_dtype dt, const void* X, const void* dY, int N,
                                              int nblk, int b, int splits, float* dG,
                                              cudaStream_t stream) {
  POETX_TRY(check_act(dt, b));
  if (N < 0 || nblk < 0 || splits < 1) return POETX_ERR_ARG;
  if (nblk == 0) return POETX_OK;
  if (!dG || (N > 0 && (!X || !dY))) return POETX_ERR_ARG;
  if (!aligned16(dG) || (N > 0 && (!aligned16(X) || !aligned16(dY)))) return POETX_ERR_ALIGN;
  return wgrad_impl(dt, X, dY, N, nblk, b, splits, dG, stream);
}

extern "C" poetx_status poetx_wprime_gemm(poetx_dtype act, poetx_dtype wdt, const void* A, int N,
                                          int m, int n, const void* W, const float* w_scale,
                                          int trans, void* C, cudaStream_t stream) {
  if (act == POETX_F32 && wdt != POETX_F32) return POETX_ERR_DTYPE;
  if (act == POETX_BF16 && wdt != POETX_BF16 && wdt != POETX_I8) return POETX_ERR_DTYPE;
  if (act != POETX_F32 && act != POETX_BF16) return POETX_ERR_DTYPE;
  if (N < 0 || m <= 0 || n <= 0) return POETX_ERR_ARG;
  if (wdt == POETX_I8 && !w_scale) return POETX_ERR_ARG;
  if (N == 0) return POETX_OK;
  if (!A || !W || !C) return POETX_ERR_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C)) return POETX_ERR_ALIGN;
  if ((m * dtype_size(act)) % 16 || (n * dtype_size(act)) % 16) return POETX_ERR_SHAPE;
  return wprime_impl(act, wdt, A, N, m, n, W, w_scale, trans, C, stream);
}
