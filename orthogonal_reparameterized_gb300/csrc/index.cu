// Index and data-movement kernels: packed-triangle unpack / gradient pack (step S1 and its
// gradient), permutations as index remaps (S3, S7, S8, S13), the permutation merge into the
// frozen weight (S15) and the per-row int8 quantiser (S16).  All are bit-exact data
// movement (the quantiser takes its decisions in IEEE fp32).
//
// POET-X summary page ("POET-X: Memory-efficient LLM Training by Scaling Orthogonal
// Transformation"), "Core method" section 2 (permutations as index remaps; merge of the
// two permutations into W once per inner loop) and section 4 (upper-triangle storage).
#include <mutex>

#include "adam.cuh"
#include "common.cuh"
#include "kernels.h"

namespace poetx {

// Site id of this file's bounded waits (file id x 10000 + source line), recorded with
// the first timeout.
constexpr int kSite = 3 * 10000;

// ---------------------------------------------------------------- packed triangle
// Offset of pair (i, j), i < j, in the row-major strict upper triangle of a b x b block.
__device__ __forceinline__ long long tri_index(int i, int j, int b) {
  return (long long)i * (b - 1) - (long long)i * (i - 1) / 2 + (j - i - 1);
}

// The blocks of one launch come from the sides of a SideTable (the R and P sides of a layer,
// or of every layer of a group): block blk belongs to the side whose [start, start + n)
// range holds it.
__device__ __forceinline__ int side_of(const SideTable& t, int blk) {
  int k = 0;
  while (k + 1 < t.count && blk >= t.start[k + 1]) ++k;
  return k;
}

// Upper tiles per CTA of the unpack and the gradient pack: every thread issues the loads of all
// of its CTA's tiles before the first store, so that enough bytes are in flight per SM for
// these short, latency-bound passes.
constexpr int kTriTiles = 4;

// Linear upper-tile index t of a block -> (I, J), I <= J, of its nt x nt tiles of 32.
__device__ __forceinline__ void upper_tile(int t, int nt, int& I, int& J) {
  I = 0;
  while (t >= nt - I) {
    t -= nt - I;
    ++I;
  }
  J = I + t;
}

// Each CTA takes kTriTiles 32 x 32 tiles (I, J), I <= J, of a block: per tile it reads the
// packed entries of the tile's upper part (consecutive j are consecutive in q), writes Q[I][J]
// and, through shared memory, the mirrored tile Q[J][I] = -Q[I][J]^T, both with coalesced
// rows.  The entries of a ragged last block (valid features r < b) outside its r x r corner
// are not parameters and are zero in Q.
__global__ void triu_unpack_kernel(const __grid_constant__ SideTable st, int b,
                                   float* __restrict__ Q, unsigned long long* tr, size_t tr_cap) {
  if (threadIdx.x == 0 && threadIdx.y == 0) trace_stamp3(tr, tr_cap, 0);
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[kTriTiles][32][33];
  const int blk = blockIdx.z;
  const int nt = (b + 31) / 32;
  const int ntiles = nt * (nt + 1) / 2;
  const long long tri = (long long)b * (b - 1) / 2;
  const int k = side_of(st, blk);
  const int local = blk - st.start[k];
  const float* qb = st.src[k] + local * tri;
  float* Qb = Q + (long long)blk * b * b;
  const int rv = blk == st.start[k + 1] - 1 ? st.valid[k] : b;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  int I[kTriTiles], J[kTriTiles];
  float v[kTriTiles][4];
#pragma unroll
  for (int u = 0; u < kTriTiles; ++u) {  // every load first
    const int t = blockIdx.x * kTriTiles + u;
    upper_tile(t < ntiles ? t : 0, nt, I[u], J[u]);
    if (t >= ntiles) I[u] = -1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = I[u] * 32 + ty + 8 * c, j = J[u] * 32 + tx;
      float x = 0.f;
      if (I[u] >= 0 && i < rv && j < rv) {
        if (i < j) x = __ldg(qb + tri_index(i, j, b));
        else if (i > j) x = -__ldg(qb + tri_index(j, i, b));
      }
      v[u][c] = x;
    }
  }
#pragma unroll
  for (int u = 0; u < kTriTiles; ++u) {
    if (I[u] < 0) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = ty + 8 * c;
      const int i = I[u] * 32 + r, j = J[u] * 32 + tx;
      if (i < b && j < b) Qb[(long long)i * b + j] = v[u][c];
      tile[u][r][tx] = v[u][c];
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kTriTiles; ++u) {
    if (I[u] < 0 || I[u] == J[u]) continue;  // a diagonal tile wrote both of its triangles
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = ty + 8 * c;
      const int i = J[u] * 32 + cc, j = I[u] * 32 + tx;  // Q[i][j] = -Q[j][i]
      if (i < b && j < b) Qb[(long long)i * b + j] = -tile[u][tx][cc];
    }
  }
  if (tr) {
    __syncthreads();
    if (threadIdx.x == 0 && threadIdx.y == 0) trace_stamp3(tr, tr_cap, 31);
  }
}

// dq_ij (+)= Qbar_ij - Qbar_ji for i < j.  Each CTA takes kTriTiles 32 x 32 tiles (I, J),
// I <= J, of a block: the mirrored tile Qbar[J][I] is read with coalesced rows into shared
// memory and read back transposed, so both reads of Qbar are coalesced; the writes of a row i
// of the tile are consecutive entries of the packed triangle.
// pa (nullable q): the optimizer update applied to each entry as its gradient is written
// (single-replica training: nothing has to be summed between the pack and the update).
__global__ void triu_grad_pack_kernel(const float* __restrict__ Qbar, int b,
                                      const __grid_constant__ SideTable st, int accumulate,
                                      const __grid_constant__ PackAdam pa,
                                      unsigned long long* tr, size_t tr_cap) {
  if (threadIdx.x == 0 && threadIdx.y == 0) trace_stamp3(tr, tr_cap, 0);
  pdl_trigger();
  pdl_wait();
  __shared__ float tile[kTriTiles][32][33];
  const int blk = blockIdx.z;
  const int nt = (b + 31) / 32;
  const int ntiles = nt * (nt + 1) / 2;
  const long long tri = (long long)b * (b - 1) / 2;
  const float* Qb = Qbar + (long long)blk * b * b;
  const int side = side_of(st, blk);
  const long long off = (long long)(blk - st.start[side]) * tri;  // this block's entries
  float* dqb = st.dst[side] + off;
  const int rv = blk == st.start[side + 1] - 1 ? st.valid[side] : b;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  int I[kTriTiles], J[kTriTiles];
  float d[kTriTiles][4];
#pragma unroll
  for (int u = 0; u < kTriTiles; ++u) {  // every load first
    const int t = blockIdx.x * kTriTiles + u;
    upper_tile(t < ntiles ? t : 0, nt, I[u], J[u]);
    if (t >= ntiles) I[u] = -1;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = ty + 8 * c;
      // tile[u][r][tx] = Qbar[J*32 + r][I*32 + tx]; d = Qbar[I*32 + r][J*32 + tx]
      const int jm = J[u] * 32 + r, im = I[u] * 32 + tx;
      const int i = I[u] * 32 + r, j = J[u] * 32 + tx;
      const bool live = I[u] >= 0;
      tile[u][r][tx] = (live && jm < b && im < b) ? __ldg(Qb + (long long)jm * b + im) : 0.f;
      d[u][c] = (live && i < j && j < b) ? __ldg(Qb + (long long)i * b + j) : 0.f;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kTriTiles; ++u) {
    if (I[u] < 0) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = ty + 8 * c;
      const int i = I[u] * 32 + r, j = J[u] * 32 + tx;
      if (i < j && j < b) {
        const float v = j < rv ? d[u][c] - tile[u][tx][r] : 0.f;
        const long long kk = tri_index(i, j, b);
        float* dst = dqb + kk;
        const float g = accumulate ? *dst + v : v;
        *dst = g;
        if (pa.q[side]) {
          const long long e = off + kk;
          adam_one(pa.q[side][e], g, pa.m[side][e], pa.v[side][e], pa.h);
        }
      }
    }
  }
  if (tr) {
    __syncthreads();
    if (threadIdx.x == 0 && threadIdx.y == 0) trace_stamp3(tr, tr_cap, 31);
  }
}

poetx_status launch_triu_unpack_sides(const SideTable& t, int b, float* Q, cudaStream_t s) {
  const int total = t.start[t.count];
  if (total == 0) return POETX_OK;
  const int nt = (b + 31) / 32;
  dim3 grid((nt * (nt + 1) / 2 + kTriTiles - 1) / kTriTiles, 1, total);
  size_t tr_cap = 0;
  unsigned long long* tr = trace_buffer(&tr_cap);
  POETX_CUDA_TRY(launch_pdl(triu_unpack_kernel, grid, dim3(32, 8), 0, s, t, b, Q, tr, tr_cap));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_TRIU_UNPACK);
  return POETX_OK;
}

poetx_status launch_triu_unpack(const float* q, int nblk, int b, float* Q, cudaStream_t s) {
  SideTable t{};
  t.count = 1;
  t.start[0] = 0;
  t.start[1] = nblk;
  t.valid[0] = b;
  t.src[0] = q;
  return launch_triu_unpack_sides(t, b, Q, s);
}

poetx_status launch_triu_grad_pack_sides(const float* Qbar, const SideTable& t, int b,
                                         int accumulate, cudaStream_t s, const PackAdam* pa) {
  const int total = t.start[t.count];
  if (total == 0 || b < 2) return POETX_OK;
  const int nt = (b + 31) / 32;
  dim3 grid((nt * (nt + 1) / 2 + kTriTiles - 1) / kTriTiles, 1, total);
  size_t tr_cap = 0;
  unsigned long long* tr = trace_buffer(&tr_cap);
  PackAdam none{};
  POETX_CUDA_TRY(launch_pdl(triu_grad_pack_kernel, grid, dim3(32, 8), 0, s, Qbar, b, t,
                            accumulate, pa ? *pa : none, tr, tr_cap));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_TRIU_PACK);
  return POETX_OK;
}

poetx_status launch_triu_grad_pack(const float* Qbar, int nblk, int b, float* dq, int accumulate,
                                   cudaStream_t s) {
  SideTable t{};
  t.count = 1;
  t.start[0] = 0;
  t.start[1] = nblk;
  t.valid[0] = b;
  t.dst[0] = dq;
  return launch_triu_grad_pack_sides(Qbar, t, b, accumulate, s);
}

// ---------------------------------------------------------------- row permutations
// Every row is permuted on its own: out[i] = row[idx[i]], with idx = perm for a gather and
// its inverse (idx[perm[i]] = i) for a scatter, staged once per CTA in shared memory as
// 16-bit entries.  The CTA's eight consumer warps form 8/G independent groups of G >= 2 warps
// (wider groups for longer rows): a group owns the rows r = group, + groups in the grid, ...,
// which a ninth (producer) warp streams into the group's own ring of S row buffers by
// one-dimensional TMA bulk copies (S rows ahead); the group writes 16-byte vectors of each
// output row, so loads and stores are fully coalesced and no barrier wider than the group
// ever stalls the other groups.  `src_rows` (nullable) remaps the source row (the merge
// W'[r, :] = W0[perm_n[r], perm_m]).  Waits are bounded; on expiry the kernel records
// POETX_ERR_TIMEOUT, drains the copies it issued and returns.
template <int E>
struct VecT;
template <>
struct VecT<1> { using T = uint8_t; };
template <>
struct VecT<2> { using T = uint16_t; };
template <>
struct VecT<4> { using T = uint32_t; };

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// V consecutive gather indices, read from shared memory with one aligned vector load per
// 16 bytes (8-byte loads when the V indices take 8 bytes).
template <typename IdxT, int V>
struct IdxVec {
  IdxT i[V];
};
template <typename IdxT, int V>
__device__ __forceinline__ IdxVec<IdxT, V> load_idx(const IdxT* p) {
  constexpr int IB = V * (int)sizeof(IdxT);
  IdxVec<IdxT, V> r;
  if constexpr (IB == 8) {
    union { uint2 u; IdxT i[V]; } x;
    x.u = *reinterpret_cast<const uint2*>(p);
#pragma unroll
    for (int e = 0; e < V; ++e) r.i[e] = x.i[e];
  } else {
    static_assert(IB % 16 == 0, "index vector must be 8 or a multiple of 16 bytes");
    union { uint4 u[IB / 16]; IdxT i[V]; } x;
#pragma unroll
    for (int w = 0; w < IB / 16; ++w) x.u[w] = reinterpret_cast<const uint4*>(p)[w];
#pragma unroll
    for (int e = 0; e < V; ++e) r.i[e] = x.i[e];
  }
  return r;
}

// Barrier over one group of G warps (G = 1: the warp itself); named barriers 1..8.
__device__ __forceinline__ void group_sync(int g, int G) {
  if (G == 1) {
    __syncwarp();
  } else {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(G * 32) : "memory");
  }
}
// True when `v` holds on every thread of the group.
__device__ __forceinline__ bool group_all(bool v, int g, int G) {
  if (G == 1) return __all_sync(0xffffffffu, v);
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.and.pred p, %2, %3, q; selp.u32 %0, 1, 0, p; }"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + g), "r"(G * 32)
      : "memory");
  return r != 0;
}

constexpr int kPermWarps = 8;  // consumer warps; one more warp issues the row copies
constexpr int kIdxRound = 4;   // 16-byte index loads in flight per consumer thread

// Stores the four gather indices perm[i0 .. i0 + 3] = v into the staged index (gather: idx[i]
// = perm[i]; scatter, the inverse: idx[perm[i]] = i).
template <bool SCATTER, typename IdxT>
__device__ __forceinline__ void stage_idx4(IdxT* idx, int i0, int4 v) {
  if (SCATTER) {
    idx[v.x] = (IdxT)i0;
    idx[v.y] = (IdxT)(i0 + 1);
    idx[v.z] = (IdxT)(i0 + 2);
    idx[v.w] = (IdxT)(i0 + 3);
  } else if (sizeof(IdxT) == 2) {
    *reinterpret_cast<uint2*>(idx + i0) =
        make_uint2(((uint32_t)v.y << 16) | ((uint32_t)v.x & 0xFFFFu),
                   ((uint32_t)v.w << 16) | ((uint32_t)v.z & 0xFFFFu));
  } else {
    *reinterpret_cast<int4*>(idx + i0) = v;
  }
}

// PITCHED: rows of the source or the destination are wider than D (a padded layer side);
// the common case keeps the plain row arithmetic.
template <int E, bool SCATTER, typename IdxT, bool PITCHED>
__global__ void __launch_bounds__((kPermWarps + 1) * 32, 3) perm_rows_kernel(
    const uint8_t* __restrict__ X, long long N, int D, const int32_t* __restrict__ perm,
    uint8_t* __restrict__ Y, const int32_t* __restrict__ src_rows, const float* __restrict__ scale,
    float* __restrict__ scale_out, long long src_pitch, long long dst_pitch, int G, int S,
    int* err, unsigned long long limit_ns, unsigned long long* trace, size_t trace_cap) {
  using T = typename VecT<E>::T;
  constexpr int V = 16 / E;  // elements per 16-byte vector
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t row_bytes = (uint32_t)D * E;
  const uint32_t idx_bytes = ((uint32_t)D * sizeof(IdxT) + 127u) & ~127u;
  const int ngrp = kPermWarps / G;
  IdxT* idx = reinterpret_cast<IdxT*>(smem_raw);
  uint8_t* ring = smem_raw + idx_bytes;  // [ngrp][S] rows
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)ngrp * S * row_bytes);
  uint64_t* empty = full + ngrp * S;
  uint64_t* idx_go = empty + ngrp * S;  // every consumer warp's first index loads are issued
  const int warp = threadIdx.x >> 5;
  // group gr of this CTA owns rows first + gr + it * stride, it < rows_of(gr); rows per group
  // fit 32 bits (N < 2^31), so the loops below count in 32 bits and never divide
  const long long first = (long long)blockIdx.x * ngrp;
  const long long stride = (long long)gridDim.x * ngrp;
  // (N < 2^31 rows: 32-bit division, a few instructions instead of a 64-bit subroutine)
  auto rows_of = [&](int gr) -> int {
    const long long f = first + gr;
    return f < N ? (int)((uint32_t)(N - 1 - f) / (uint32_t)stride + 1) : 0;
  };
  if (threadIdx.x == 0) trace_stamp(trace, trace_cap, 0);  // slot 0: CTA start
  pdl_trigger();
  if (warp == kPermWarps && (threadIdx.x & 31) == 0) {
    for (int k = 0; k < ngrp * S; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], 1);
    }
    mbar_init(idx_go, kPermWarps);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (threadIdx.x == 0) trace_stamp(trace, trace_cap, 1);  // slot 1: predecessor done

  // The index is read with every consumer thread's first round of loads in flight at once,
  // and those loads are issued before the row copies, so that the index (needed before any
  // row can be permuted) does not queue behind the rows in the memory system.
  const bool idx_vec = ((reinterpret_cast<uintptr_t>(perm) & 15u) == 0) && (D & 3) == 0;
  if (warp == kPermWarps) {
    // producer: one thread streams every group's rows, round robin over the groups so the
    // first rows of all groups land first; a slot is refilled once its group released it
    if ((threadIdx.x & 31) == 0) {
      int nr[kPermWarps], issued[kPermWarps];
      int most = 0;
#pragma unroll
      for (int gr = 0; gr < kPermWarps; ++gr) {
        nr[gr] = gr < ngrp ? rows_of(gr) : 0;
        issued[gr] = 0;
        most = nr[gr] > most ? nr[gr] : most;
      }
      bool ok = mbar_wait_bounded(idx_go, 0, err, limit_ns, kSite + __LINE__);
      int k = 0, round = 0;
      for (int it = 0; ok && it < most; ++it) {
#pragma unroll
        for (int gr = 0; gr < kPermWarps; ++gr) {
          if (!ok || it >= nr[gr]) continue;
          const int slot = gr * S + k;
          if (round > 0 && !mbar_wait_bounded(&empty[slot], (uint32_t)((round - 1) & 1), err, limit_ns, kSite + __LINE__)) {
            ok = false;
            continue;
          }
          const long long r = first + gr + (long long)it * stride;
          const long long sr = src_rows ? (long long)__ldg(src_rows + r) : r;
          mbar_arrive_expect_tx(&full[slot], row_bytes);
          bulk_load(ring + (size_t)slot * row_bytes,
                    X + (PITCHED ? sr * src_pitch * E : sr * row_bytes), row_bytes, &full[slot]);
          issued[gr] = it + 1;
        }
        if (it == 0) trace_stamp(trace, trace_cap, 2);  // slot 2: first row of every group issued
        if (++k == S) {
          k = 0;
          ++round;
        }
      }
      if (!ok) {
        // drain: the last S rows issued to each group may still be in flight
#pragma unroll
        for (int gr = 0; gr < kPermWarps; ++gr)
          for (int j = issued[gr] - S < 0 ? 0 : issued[gr] - S; j < issued[gr]; ++j)
            mbar_wait_bounded(&full[gr * S + j % S], (uint32_t)((j / S) & 1), err, limit_ns, kSite + __LINE__);
      }
    }
  } else {
    // consumers: stage the index, then each group of G warps permutes its own rows
    const int g = warp / G;
    const int tig = threadIdx.x - g * G * 32;
    constexpr int kStride = kPermWarps * 32;
    // rounds of loads: the trip count is the same for every thread (so warps stay converged
    // for the barriers below), the bounds are per element
    auto first_round_issued = [&](int r0) {
      if (r0 == 0) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(idx_go);
      }
    };
    if (idx_vec) {
      const int nv = D >> 2;
      const int4* p4 = reinterpret_cast<const int4*>(perm);
      for (int r0 = 0; r0 == 0 || r0 < nv; r0 += kStride * kIdxRound) {
        int4 v[kIdxRound];
#pragma unroll
        for (int u = 0; u < kIdxRound; ++u) {
          const int j = r0 + u * kStride + (int)threadIdx.x;
          if (j < nv) v[u] = __ldg(p4 + j);
        }
        first_round_issued(r0);
#pragma unroll
        for (int u = 0; u < kIdxRound; ++u) {
          const int j = r0 + u * kStride + (int)threadIdx.x;
          if (j < nv) stage_idx4<SCATTER, IdxT>(idx, 4 * j, v[u]);
        }
      }
    } else {
      for (int r0 = 0; r0 == 0 || r0 < D; r0 += kStride * 4 * kIdxRound) {
        int v[4 * kIdxRound];
#pragma unroll
        for (int u = 0; u < 4 * kIdxRound; ++u) {
          const int i = r0 + u * kStride + (int)threadIdx.x;
          if (i < D) v[u] = __ldg(perm + i);
        }
        first_round_issued(r0);
#pragma unroll
        for (int u = 0; u < 4 * kIdxRound; ++u) {
          const int i = r0 + u * kStride + (int)threadIdx.x;
          if (i < D) {
            if (SCATTER) idx[v[u]] = (IdxT)i;
            else idx[i] = (IdxT)v[u];
          }
        }
      }
    }
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(kPermWarps + 1), "r"(kPermWarps * 32) : "memory");
    if (threadIdx.x == 0) trace_stamp(trace, trace_cap, 3);  // slot 3: index staged
    const int nrows = rows_of(g);
    const int nvec = D / V;
    const int gthreads = G * 32;
    int k = 0;
    uint32_t ph = 0;
    for (int it = 0; it < nrows; ++it) {
      const int slot = g * S + k;
      const bool got = mbar_wait_bounded(&full[slot], ph, err, limit_ns, kSite + __LINE__);
      if (!group_all(got, g, G)) break;
      if (threadIdx.x == 0 && it < 13) trace_stamp(trace, trace_cap, 4 + 2 * it);  // landed
      const long long r = first + g + (long long)it * stride;
      const T* row = reinterpret_cast<const T*>(ring + (size_t)slot * row_bytes);
      uint4* out = reinterpret_cast<uint4*>(Y + (PITCHED ? r * dst_pitch * E : r * row_bytes));
#pragma unroll 4
      for (int v = tig; v < nvec; v += gthreads) {
        const IdxVec<IdxT, V> ix = load_idx<IdxT, V>(idx + (size_t)v * V);
        union { uint4 u; T e[V]; } pk;
#pragma unroll
        for (int e = 0; e < V; ++e) pk.e[e] = row[ix.i[e]];
        out[v] = pk.u;
      }
      // columns D .. dst_pitch - 1 of a padded destination row (ragged last block) are zero
      if constexpr (PITCHED)
        for (int v = nvec + tig; v < (int)(dst_pitch / V); v += gthreads)
          out[v] = make_uint4(0, 0, 0, 0);
      if (scale_out && tig == 0) scale_out[r] = scale[src_rows ? src_rows[r] : r];
      group_sync(g, G);  // every thread of the group is done with buffer k
      if (threadIdx.x == 0 && it < 13) trace_stamp(trace, trace_cap, 5 + 2 * it);  // row done
      if (tig == 0) mbar_arrive(&empty[slot]);
      if (++k == S) {
        k = 0;
        ph ^= 1u;
      }
    }
  }
  if (trace) {
    __syncthreads();
    if (threadIdx.x == 0) trace_stamp(trace, trace_cap, 31);  // slot 31: every row done
  }
}

// Group size and ring depth for rows of `row_bytes`: the narrowest groups of two warps or
// more whose rings (two rows at least) fit ~110 KB with the index, so that two CTAs share an
// SM; one CTA of a single group per SM for rows too long for that.  Returns false when not
// even that fits.  (Measured on 2048-wide bf16 rows: two-warp groups match one-warp groups at
// 4096 rows and stream ~10 % faster from 8192 rows up; wider groups are slower.)
static bool perm_shape(size_t row_bytes, size_t idx_bytes, int* G, int* S, size_t* smem) {
  const size_t budget3 = 74 * 1024, budget2 = 110 * 1024, budget1 = 220 * 1024;
  // three CTAs per SM (more consumer warps to cover the shared-memory read latency) while
  // two-warp groups still get two rows in flight each
  {
    const size_t ngrp = kPermWarps / 2;
    if (idx_bytes + ngrp * 2 * (row_bytes + 16) <= budget3) {
      int s = (int)((budget3 - idx_bytes) / (ngrp * (row_bytes + 16)));
      s = s > 8 ? 8 : s;
      *G = 2;
      *S = s;
      *smem = idx_bytes + ngrp * s * (row_bytes + 16);
      return true;
    }
  }
  for (int g = 2; g <= kPermWarps; g *= 2) {
    const size_t ngrp = kPermWarps / g;
    if (idx_bytes + ngrp * 2 * (row_bytes + 16) <= budget2) {
      int s = (int)((budget2 - idx_bytes) / (ngrp * (row_bytes + 16)));
      s = s > 8 ? 8 : s;
      *G = g;
      *S = s;
      *smem = idx_bytes + ngrp * s * (row_bytes + 16);
      return true;
    }
  }
  if (idx_bytes + row_bytes + 16 > budget1) return false;
  int s = (int)((budget1 - idx_bytes) / (row_bytes + 16));
  s = s > 8 ? 8 : s;
  *G = kPermWarps;
  *S = s;
  *smem = idx_bytes + s * (row_bytes + 16);
  return true;
}

// Co-resident shape: one CTA per SM in the shared memory that a 64-wide CNP product CTA
// leaves free (of an SM's 228 KB: the product's 214,272 bytes, and 1 KB reserved for each of
// the two CTAs), so that the permutation runs beside the CNP products instead of after them.
// All consumer warps form one group; at least two rows in flight.
constexpr size_t kPermSideSmem = 233472 - 214272 - 2 * 1024;
static bool perm_shape_side(size_t row_bytes, size_t idx_bytes, int* G, int* S, size_t* smem) {
  if (idx_bytes + 2 * (row_bytes + 16) > kPermSideSmem) return false;
  int s = (int)((kPermSideSmem - idx_bytes) / (row_bytes + 16));
  s = s > 8 ? 8 : s;
  *G = kPermWarps;
  *S = s;
  *smem = idx_bytes + s * (row_bytes + 16);
  return true;
}

template <int E, bool SCATTER, typename IdxT, bool PITCHED>
static poetx_status launch_perm_rows_t(const void* X, long long N, int D, const int32_t* perm,
                                       void* Y, const int32_t* src_rows, const float* scale,
                                       float* scale_out, long long sp, long long dp, bool side,
                                       cudaStream_t s) {
  const size_t row_bytes = (size_t)D * E;
  const size_t idx_bytes = ((size_t)D * sizeof(IdxT) + 127) & ~(size_t)127;
  int G = 0, S = 0;
  size_t smem = 0;
  // (the index, and 16 bytes for the barrier that starts the row copies)
  if (!(side ? perm_shape_side : perm_shape)(row_bytes, idx_bytes + 16, &G, &S, &smem))
    return POETX_ERR_SHAPE;
  auto k = perm_rows_kernel<E, SCATTER, IdxT, PITCHED>;
  static std::once_flag once;  // the opt-in limit is set once, to the largest size used
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    // all of the unified L1 as shared memory, as the CNP products take it, so that a
    // co-resident CTA never holds an SM in a smaller split
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared);
  });
  POETX_CUDA_TRY(attr);
  const int ngrp = kPermWarps / G;
  size_t tr_cap = 0;
  unsigned long long* tr = trace_buffer(&tr_cap);
  const int per_sm = side ? 1 : (smem <= 74 * 1024 ? 3 : (smem <= 110 * 1024 ? 2 : 1));
  const long long want = (long long)sm_count() * per_sm;
  const long long need = (N + ngrp - 1) / ngrp;
  const int grid = (int)(need < want ? need : want);
  if (side) {
    // no early launch: waiting CTAs would hold shared memory on every SM while the kernels
    // of the other stream still need it
    k<<<grid, (kPermWarps + 1) * 32, smem, s>>>(static_cast<const uint8_t*>(X), N, D, perm,
                                                static_cast<uint8_t*>(Y), src_rows, scale,
                                                scale_out, sp, dp, G, S, device_error_word(),
                                                kWaitLimitNs, tr, tr_cap);
  } else {
    POETX_CUDA_TRY(launch_pdl(k, dim3(grid), dim3((kPermWarps + 1) * 32), smem, s,
                              static_cast<const uint8_t*>(X), N, D, perm,
                              static_cast<uint8_t*>(Y), src_rows, scale, scale_out, sp, dp, G,
                              S, device_error_word(), kWaitLimitNs, tr, tr_cap));
  }
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, src_rows ? ST_MERGE : (SCATTER ? ST_PERM_SCATTER : ST_PERM_GATHER));
  return POETX_OK;
}

template <int E>
static poetx_status launch_perm_rows_e(bool scatter, const void* X, long long N, int D,
                                       const int32_t* perm, void* Y, const int32_t* src_rows,
                                       const float* scale, float* scale_out, long long sp,
                                       long long dp, bool side, cudaStream_t s) {
#define POETX_PERM_T(SC, IT, PI) \
  launch_perm_rows_t<E, SC, IT, PI>(X, N, D, perm, Y, src_rows, scale, scale_out, sp, dp, side, s)
  const bool pitched = sp != D || dp != D;
  // (a 16-bit index covers every width whose index and one row fit an SM's shared memory)
  if (D > 65535) return POETX_ERR_SHAPE;
  if (pitched) return scatter ? POETX_PERM_T(true, uint16_t, true) : POETX_PERM_T(false, uint16_t, true);
  return scatter ? POETX_PERM_T(true, uint16_t, false) : POETX_PERM_T(false, uint16_t, false);
#undef POETX_PERM_T
}

// sp, dp: source and destination row pitches in elements (0: D).  The D permuted columns
// of each row go to columns 0 .. D - 1 of the destination row and columns D .. dp - 1 are
// written with zeros; every pitch is a whole number of 16-byte vectors.
static poetx_status perm_rows_any(size_t esize, bool scatter, const void* X, long long N, int D,
                                  const int32_t* perm, void* Y, const int32_t* src_rows,
                                  const float* scale, float* scale_out, long long sp,
                                  long long dp, bool side, cudaStream_t s) {
  if (N == 0 || D == 0) return POETX_OK;
  if (N > 0x7fffffffLL) return POETX_ERR_SHAPE;  // rows are counted in 32 bits
  sp = sp ? sp : D;
  dp = dp ? dp : D;
  if (sp < D || dp < D) return POETX_ERR_ARG;
  if (((size_t)D * esize) % 16 != 0 || ((size_t)sp * esize) % 16 != 0 ||
      ((size_t)dp * esize) % 16 != 0)
    return POETX_ERR_SHAPE;
  if (esize == 1) return launch_perm_rows_e<1>(scatter, X, N, D, perm, Y, src_rows, scale, scale_out, sp, dp, side, s);
  if (esize == 2) return launch_perm_rows_e<2>(scatter, X, N, D, perm, Y, src_rows, scale, scale_out, sp, dp, side, s);
  if (esize == 4) return launch_perm_rows_e<4>(scatter, X, N, D, perm, Y, src_rows, scale, scale_out, sp, dp, side, s);
  return POETX_ERR_DTYPE;
}

poetx_status launch_perm_rows(size_t esize, bool scatter, const void* X, long long N, int D,
                              const int32_t* perm, void* Y, const int32_t* src_rows,
                              const float* scale, float* scale_out, cudaStream_t s,
                              long long src_pitch, long long dst_pitch) {
  return perm_rows_any(esize, scatter, X, N, D, perm, Y, src_rows, scale, scale_out, src_pitch,
                       dst_pitch, false, s);
}

bool perm_side_fits(size_t esize, int D) {
  if (D > 65535) return false;
  const size_t idx = ((size_t)D * 2 + 127) & ~(size_t)127;
  int G = 0, S = 0;
  size_t smem = 0;
  return ((size_t)D * esize) % 16 == 0 &&
         perm_shape_side((size_t)D * esize, idx + 16, &G, &S, &smem);
}

poetx_status launch_perm_rows_side(size_t esize, bool scatter, const void* X, long long N, int D,
                                   const int32_t* perm, void* Y, cudaStream_t s,
                                   long long src_pitch, long long dst_pitch) {
  return perm_rows_any(esize, scatter, X, N, D, perm, Y, nullptr, nullptr, nullptr, src_pitch,
                       dst_pitch, true, s);
}

// ---------------------------------------------------------------- int8 quantiser
__global__ void __launch_bounds__(256) quantize_rows_kernel(const float* __restrict__ W, int m,
                                                            int8_t* __restrict__ Wq,
                                                            float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
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
  POETX_CUDA_TRY(launch_pdl(quantize_rows_kernel, dim3(n), dim3(256), 0, s, W, m, Wq, scale));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_QUANTIZE);
  return POETX_OK;
}

// ---------------------------------------------------------------- merge helpers
// inv[perm[i]] = i, for the two permutations of a layer at once (perm_a of length na, then
// perm_b of length nb, into inv_a / inv_b).
__global__ void __launch_bounds__(256) invert_perm_kernel(const int32_t* __restrict__ perm_a,
                                                          int na, int32_t* __restrict__ inv_a,
                                                          const int32_t* __restrict__ perm_b,
                                                          int nb, int32_t* __restrict__ inv_b) {
  pdl_trigger();
  pdl_wait();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < na) {
    inv_a[perm_a[i]] = (int32_t)i;
  } else if (i < (long long)na + nb) {
    const int k = (int)(i - na);
    inv_b[perm_b[k]] = k;
  }
}

poetx_status launch_invert_perms(const int32_t* perm_a, int na, int32_t* inv_a,
                                 const int32_t* perm_b, int nb, int32_t* inv_b, cudaStream_t s) {
  const long long n = (long long)na + nb;
  if (n == 0) return POETX_OK;
  POETX_CUDA_TRY(launch_pdl(invert_perm_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0,
                            s, perm_a, na, inv_a, perm_b, nb, inv_b));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_MERGE_REINIT);
  return POETX_OK;
}

// W[r][c] = scale[r] * Wq[r][c] in fp32 (m a multiple of 4: four codes per thread).
__global__ void __launch_bounds__(256) dequant_rows_kernel(const int8_t* __restrict__ Wq,
                                                           const float* __restrict__ scale,
                                                           int n, int m, float* __restrict__ W) {
  pdl_trigger();
  pdl_wait();
  const long long quads = (long long)n * (m / 4);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < quads;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / (m / 4);
    const char4 q = reinterpret_cast<const char4*>(Wq)[i];
    const float sr = scale[r];
    reinterpret_cast<float4*>(W)[i] =
        make_float4(sr * (float)q.x, sr * (float)q.y, sr * (float)q.z, sr * (float)q.w);
  }
}

// W[i] = float(Wb[i]) for a bf16 array (count a multiple of 4: four values per thread).
__global__ void __launch_bounds__(256) widen_bf16_kernel(const __nv_bfloat16* __restrict__ Wb,
                                                         long long quads, float* __restrict__ W) {
  pdl_trigger();
  pdl_wait();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < quads;
       i += (long long)gridDim.x * blockDim.x) {
    const uint2 u = reinterpret_cast<const uint2*>(Wb)[i];
    reinterpret_cast<float4*>(W)[i] =
        make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                    __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  }
}

poetx_status launch_widen_bf16(const void* Wb, long long count, float* W, cudaStream_t s) {
  if (count == 0) return POETX_OK;
  if (count % 4) return POETX_ERR_SHAPE;
  const long long quads = count / 4;
  long long blocks = (quads + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  POETX_CUDA_TRY(launch_pdl(widen_bf16_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                            static_cast<const __nv_bfloat16*>(Wb), quads, W));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_MERGE_REINIT);
  return POETX_OK;
}

poetx_status launch_dequant_rows(const int8_t* Wq, const float* scale, int n, int m, float* W,
                                 cudaStream_t s) {
  if (n == 0 || m == 0) return POETX_OK;
  if (m % 4) return POETX_ERR_SHAPE;
  const long long quads = (long long)n * (m / 4);
  long long blocks = (quads + 255) / 256;
  const long long cap = (long long)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  POETX_CUDA_TRY(launch_pdl(dequant_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, s, Wq,
                            scale, n, m, W));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_MERGE_REINIT);
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

// Zeroes `words` 16-byte words at p (p 16-byte aligned).
__global__ void zero_fill_kernel(uint4* __restrict__ p, unsigned long long words) {
  pdl_trigger();
  pdl_wait();
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
       i < words; i += (unsigned long long)gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

static poetx_status launch_zero_fill(void* p, size_t bytes, cudaStream_t s) {
  const unsigned long long words = bytes / 16;
  if (words == 0) return POETX_OK;
  const unsigned long long want = (words + 255) / 256;
  const int grid = (int)(want < 4ull * sm_count() ? want : 4ull * sm_count());
  POETX_CUDA_TRY(launch_pdl(zero_fill_kernel, dim3(grid), dim3(256), 0, s,
                            static_cast<uint4*>(p), words));
  POETX_CUDA_TRY(cudaGetLastError());
  after_launch(s, ST_MERGE);
  return POETX_OK;
}

extern "C" poetx_status poetx_merge_perm_padded(const void* W0, const float* scale,
                                                poetx_dtype dt, int n, int m, int n_pad,
                                                int m_pad, const int32_t* perm_n,
                                                const int32_t* perm_m, void* Wp,
                                                float* scale_p, cudaStream_t stream) {
  const size_t es = dtype_size(dt);
  if (!es) return POETX_ERR_DTYPE;
  if (n < 0 || m < 0 || n_pad < n || m_pad < m) return POETX_ERR_ARG;
  if (n_pad == 0 || m_pad == 0) return POETX_OK;
  if (!Wp || (n > 0 && m > 0 && (!W0 || !perm_n || !perm_m))) return POETX_ERR_ARG;
  if (dt == POETX_I8 && (!scale_p || (n > 0 && !scale))) return POETX_ERR_ARG;
  if ((W0 && !aligned16(W0)) || !aligned16(Wp)) return POETX_ERR_ALIGN;
  if (((size_t)m * es) % 16 || ((size_t)m_pad * es) % 16) return POETX_ERR_SHAPE;
  const int live = (n > 0 && m > 0) ? n : 0;  // rows written from W0; the rest are zero
  if (dt == POETX_I8 && n_pad > live &&
      (!aligned16(scale_p) || live % 4 || (n_pad - live) % 4))
    return aligned16(scale_p) ? POETX_ERR_SHAPE : POETX_ERR_ALIGN;
  if (live > 0)
    POETX_TRY(launch_perm_rows(es, false, W0, n, m, perm_m, Wp, perm_n,
                               dt == POETX_I8 ? scale : nullptr,
                               dt == POETX_I8 ? scale_p : nullptr, stream, m, m_pad));
  // rows live .. n_pad - 1 (and their scales) are zero
  POETX_TRY(launch_zero_fill(static_cast<uint8_t*>(Wp) + (size_t)live * m_pad * es,
                             (size_t)(n_pad - live) * m_pad * es, stream));
  if (dt == POETX_I8 && n_pad > live)
    POETX_TRY(launch_zero_fill(scale_p + live, (size_t)(n_pad - live) * 4, stream));
  return POETX_OK;
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
