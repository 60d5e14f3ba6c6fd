// gemm_bf16_small.cu -- BF16 x BF16 -> FP32 GEMM for small problems, on the
// CUDA cores.
//
// A problem of a few million multiply-adds is over long before the
// tensor-core kernels' fixed costs are: their set-up (barriers, tensor
// memory, clusters) and, for operands the copy engine cannot read in place
// (rows of 127 or 3001 elements), a separate launch that copies them to an
// aligned workspace.  Such problems are latency-bound, not bound by
// arithmetic or memory ("How a Matrix Multiply Runs on a GPU", "Shapes that
// run slowly, and why": small and skinny shapes; "A06 -- Tiled Matrix
// Multiply (GEMM)", section 3, split-K for too few output tiles).  So they
// run here in one launch, reading A and B in place whatever their alignment:
//   * 64 x 64 tiles of C, 256 threads as 16 x 16, each a 4 x 4 patch;
//   * K in 32-deep slices; every tile's slices are cut into `split`
//     contiguous ranges so that the blocks spread over the SMs (about two
//     per SM), and the last block of a tile to finish (per a counter, zero
//     between launches) adds the ranges' partial tiles in range order
//     0, 1, ..., split - 1, so the result does not depend on timing;
//   * each slice is fetched into registers with 2-byte loads (any address),
//     widened to FP32 (exact) and stored into shared memory, A transposed;
//     two slice buffers, the next slice fetched while the current one is
//     multiplied, one barrier per slice;
//   * FP32 FMAs in increasing k (a BF16 x BF16 product is exact in FP32).
#include <cstdint>

#include "kernels.h"

namespace g07 {
namespace {

constexpr int SB = kBf16SmallTile;  // 64
constexpr int BK = 32;
constexpr int THREADS = 256;
constexpr int A_STRIDE = SB + 4;    // transposed A rows, padded (16-byte reads)

struct SmallStage {
  float a[BK][A_STRIDE];  // a[k][m]
  float b[BK][SB];        // b[k][n]
};

__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

// Row `crow` of C, columns gn .. gn + 3 (those below N), through the output
// step; 16-byte stores when C allows them.
template <bool GELU>
__device__ __forceinline__ void store_row4(float* crow, int gn, int N, int vec_c, float4 v,
                                           const EpiParams& epi) {
  float e[4] = {v.x, v.y, v.z, v.w};
  if (vec_c && gn + 3 < N) {
    float4 old = make_float4(0.f, 0.f, 0.f, 0.f);
    if (epi.beta != 0.0f) old = *reinterpret_cast<const float4*>(crow + gn);
    const float o[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      e[j] = epi_apply<GELU>(epi, e[j], o[j], epi.bias ? epi.bias[gn + j] : 0.0f);
    *reinterpret_cast<float4*>(crow + gn) = make_float4(e[0], e[1], e[2], e[3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (gn + j < N)
        crow[gn + j] = epi_apply<GELU>(epi, e[j], epi.beta != 0.0f ? crow[gn + j] : 0.0f,
                                       epi.bias ? epi.bias[gn + j] : 0.0f);
  }
}

template <bool GELU>
__global__ void __launch_bounds__(THREADS)
gemm_bf16_small_kernel(int M, int N, int K, const uint16_t* __restrict__ A, int64_t lda,
                       const uint16_t* __restrict__ B, int64_t ldb, float* __restrict__ C,
                       int64_t ldc, int tiles_n, int split, int vec_c,
                       float* __restrict__ ws, unsigned int* __restrict__ counters,
                       EpiParams epi) {
  __shared__ __align__(16) SmallStage st[2];
  __shared__ int last_block;
  grid_dependency_wait();  // before the first read of A, B, C or the counters
  grid_dependents_go();
  const int tile = blockIdx.x / split;
  const int piece = blockIdx.x % split;
  const int m0 = (tile / tiles_n) * SB, n0 = (tile % tiles_n) * SB;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int nk_all = (K + BK - 1) / BK;
  const int kt0 = static_cast<int>(static_cast<int64_t>(nk_all) * piece / split);
  const int kt1 = static_cast<int>(static_cast<int64_t>(nk_all) * (piece + 1) / split);

  // Fetch plan per slice: A elements (row ar + 8i, k ak), a warp reading 32
  // consecutive k of one row; B elements (k br + 4j, column bc), a warp
  // reading 32 consecutive columns of one row.
  const int ak = tid & 31, ar = tid >> 5;
  const int bc = tid & 63, br = tid >> 6;
  uint16_t ra[8], rb[8];
  auto fetch = [&](int kt) {
    const int k0 = kt * BK;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int gm = m0 + ar + 8 * i, gk = k0 + ak;
      ra[i] = gm < M && gk < K ? __ldg(A + static_cast<int64_t>(gm) * lda + gk)
                               : static_cast<uint16_t>(0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int gk = k0 + br + 4 * j, gn = n0 + bc;
      rb[j] = gk < K && gn < N ? __ldg(B + static_cast<int64_t>(gk) * ldb + gn)
                               : static_cast<uint16_t>(0);
    }
  };
  auto put = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 8; ++i) st[buf].a[ak][ar + 8 * i] = bf16_to_f32(ra[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) st[buf].b[br + 4 * j][bc] = bf16_to_f32(rb[j]);
  };

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  if (kt0 < kt1) {
    fetch(kt0);
    put(0);
  }
  __syncthreads();
  for (int kt = kt0; kt < kt1; ++kt) {
    const int buf = (kt - kt0) & 1;
    const bool more = kt + 1 < kt1;
    if (more) fetch(kt + 1);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&st[buf].a[k][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&st[buf].b[k][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    // The other buffer was last read in the previous slice, before the
    // barrier that ended it; this slice's barrier below orders the stores
    // before the next slice's reads and this slice's reads before the
    // buffer is written again.
    if (more) put(buf ^ 1);
    __syncthreads();
  }

  const int col = n0 + tx * 4;
  if (split > 1) {
    float* tile_ws = ws + static_cast<int64_t>(tile) * split * (SB * SB);
    float* mine = tile_ws + piece * (SB * SB);
    // only the rows and columns inside C are parked and read back
    const bool col_in = col < N;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (col_in && m0 + ty * 4 + i < M)
        __stcg(reinterpret_cast<float4*>(mine + (ty * 4 + i) * SB + tx * 4),
               make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    __threadfence();
    __syncthreads();
    if (tid == 0)
      last_block = atomicAdd(&counters[tile], 1u) == static_cast<unsigned>(split - 1);
    __syncthreads();
    if (!last_block) return;
    __threadfence();
    // ranges added in order 0, 1, ..., split - 1; this thread's loads of
    // four ranges at a time go out before they are added
    float4 sum[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sum[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int q0 = 0; q0 < split; q0 += 4) {
      float4 v[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[q][i] = q0 + q < split && col_in && m0 + ty * 4 + i < M
                        ? __ldcg(reinterpret_cast<const float4*>(
                              tile_ws + (q0 + q) * (SB * SB) + (ty * 4 + i) * SB + tx * 4))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q0 + q < split)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sum[i].x += v[q][i].x;
            sum[i].y += v[q][i].y;
            sum[i].z += v[q][i].z;
            sum[i].w += v[q][i].w;
          }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gm = m0 + ty * 4 + i;
      if (gm < M) store_row4<GELU>(C + static_cast<int64_t>(gm) * ldc, col, N, vec_c, sum[i], epi);
    }
    if (tid == 0) counters[tile] = 0;  // leave the counter as found
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm < M)
      store_row4<GELU>(C + static_cast<int64_t>(gm) * ldc, col, N, vec_c,
                       make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]), epi);
  }
}

}  // namespace

Bf16SmallPlan bf16_small_plan(int M, int N, int K, int sms) {
  Bf16SmallPlan p;
  p.tiles_m = (M + SB - 1) / SB;
  p.tiles_n = (N + SB - 1) / SB;
  const int tiles = p.tiles_m * p.tiles_n;
  const int nk = (K + BK - 1) / BK;
  // about two blocks per SM in all, at most 16 ranges, at least one slice each
  int split = (2 * sms) / (tiles > 0 ? tiles : 1);
  if (split > kBf16SmallMaxSplit) split = kBf16SmallMaxSplit;
  if (split > nk) split = nk;
  if (tiles > kBf16SmallCounterBytes / 4) split = 1;  // one counter per split tile
  p.split = split < 1 ? 1 : split;
  p.workspace_bytes = p.split > 1 ? static_cast<int64_t>(tiles) * p.split * SB * SB * 4 : 0;
  return p;
}

cudaError_t launch_gemm_bf16_small(int M, int N, int K, const uint16_t* A, int64_t lda,
                                   const uint16_t* B, int64_t ldb, float* C, int64_t ldc,
                                   bool vec_c, const Bf16SmallPlan& p, float* ws,
                                   unsigned int* counters, const EpiParams& epi,
                                   cudaStream_t stream) {
  if (p.split > 1 && (ws == nullptr || counters == nullptr)) return cudaErrorInvalidValue;
  const int blocks = p.tiles_m * p.tiles_n * p.split;
  const int vc = vec_c ? 1 : 0;
  const cudaError_t e = launch_pdl(
      epi.act == kActGelu ? gemm_bf16_small_kernel<true> : gemm_bf16_small_kernel<false>,
      dim3(static_cast<unsigned>(blocks)), dim3(THREADS), 0, stream, M, N, K, A, lda, B, ldb, C,
      ldc, p.tiles_n, p.split, vc, ws, counters, epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace g07
