// gemm_f32.cu -- FP32 GEMM on the CUDA cores: shared-memory tiling plus
// register blocking.
//
// Method ("GEMM, step by step", section "Concept", register blocking; "A06 --
// Tiled Matrix Multiply (GEMM)", section 3; "GEMM Optimization", sections 4-5):
//   * a block of 256 threads owns a 128 x 128 tile of C and walks K in
//     16-deep slices, staging a 128 x 16 slice of A and a 16 x 128 slice of B
//     in shared memory;
//   * each thread owns an 8 x 8 patch of C in registers: per k it reads 8
//     values of A and 8 of B from shared memory and does 64 FMAs;
//   * A's slice is stored transposed (As[k][m]) with a 4-float pad so that a
//     thread's 8 A values are two 16-byte vector reads, and B's 8 values are
//     two 16-byte vector reads of Bs[k][n]: no bank conflicts on the reads;
//   * double buffering: the global loads of slice t+1 are issued into
//     registers before slice t is consumed, and stored into the other
//     shared buffer afterwards, one barrier per slice;
//   * out-of-range elements of A and B are loaded as 0 (the additive
//     identity), and stores are guarded on both row < M and col < N.
//
// Thread layout: 8 warps as 4 (M) x 2 (N), each warp a 32 x 64 sub-tile;
// lane (ly = lane/8, lx = lane%8) owns rows {4ly..4ly+3, 16+4ly..16+4ly+3}
// and columns {4lx..4lx+3, 32+4lx..32+4lx+3} of its warp's sub-tile, so a
// warp's A reads touch 4 distinct 16-byte words and its B reads 8
// consecutive ones.
#include <cstdint>

#include "kernels.h"
#include "tile_order.cuh"

namespace g07 {
namespace {

constexpr int BM = kF32TileM;
constexpr int BN = kF32TileN;
constexpr int BK = kF32TileK;
constexpr int THREADS = 256;
constexpr int A_STRIDE = BM + 4;  // transposed A rows, padded

struct F32Smem {
  float a[2][BK][A_STRIDE];
  float b[2][BK][BN];
};

// One 4-wide group of a row, zero outside [0, limit).  VEC: the group's first
// element is 16-byte aligned whenever the whole group is in range.
template <bool VEC>
__device__ __forceinline__ float4 load4(const float* __restrict__ row_ptr,
                                        int col, int limit) {
  if (VEC && col + 3 < limit) {
    return __ldg(reinterpret_cast<const float4*>(row_ptr + col));
  }
  float v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = (col + j < limit) ? __ldg(row_ptr + col + j) : 0.0f;
  return make_float4(v[0], v[1], v[2], v[3]);
}

template <bool VEC_A, bool VEC_B>
__device__ __forceinline__ void load_slice(
    const float* __restrict__ A, int64_t lda, const float* __restrict__ B,
    int64_t ldb, int M, int N, int K, int m0, int n0, int k0, int tid,
    float4 (&ra)[2], float4 (&rb)[2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = tid + THREADS * i;
    const int r = idx >> 2;          // 0..127: row of the A slice
    const int kc = (idx & 3) * 4;    // 0,4,8,12: column group of the slice
    const int gm = m0 + r;
    ra[i] = (gm < M) ? load4<VEC_A>(A + static_cast<int64_t>(gm) * lda, k0 + kc, K)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    const int kr = idx >> 5;         // 0..15: row of the B slice
    const int nc = (idx & 31) * 4;   // 0..124: column group
    const int gk = k0 + kr;
    rb[i] = (gk < K) ? load4<VEC_B>(B + static_cast<int64_t>(gk) * ldb, n0 + nc, N)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ void store_slice(F32Smem& s, int buf, int tid,
                                            const float4 (&ra)[2],
                                            const float4 (&rb)[2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int idx = tid + THREADS * i;
    const int r = idx >> 2;
    const int kc = (idx & 3) * 4;
    s.a[buf][kc + 0][r] = ra[i].x;
    s.a[buf][kc + 1][r] = ra[i].y;
    s.a[buf][kc + 2][r] = ra[i].z;
    s.a[buf][kc + 3][r] = ra[i].w;
    const int kr = idx >> 5;
    const int nc = (idx & 31) * 4;
    *reinterpret_cast<float4*>(&s.b[buf][kr][nc]) = rb[i];
  }
}

template <bool VEC_A, bool VEC_B>
__global__ void __launch_bounds__(THREADS, 2)
gemm_f32_regblock_kernel(int M, int N, int K, const float* __restrict__ A,
                         int64_t lda, const float* __restrict__ B, int64_t ldb,
                         float* __restrict__ C, int64_t ldc, int tiles_m,
                         int tiles_n, int vec_c) {
  __shared__ __align__(16) F32Smem s;

  const TileCoord tc = tile_order(blockIdx.x, tiles_m, tiles_n, kF32Group);
  const int m0 = tc.m * BM;
  const int n0 = tc.n * BN;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int row_a = (warp >> 1) * 32 + (lane >> 3) * 4;  // + {0..3, 16..19}
  const int col_b = (warp & 1) * 64 + (lane & 7) * 4;    // + {0..3, 32..35}

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  float4 ra[2], rb[2];
  load_slice<VEC_A, VEC_B>(A, lda, B, ldb, M, N, K, m0, n0, 0, tid, ra, rb);
  store_slice(s, 0, tid, ra, rb);
  __syncthreads();

  const int nk = (K + BK - 1) / BK;
  for (int kt = 0; kt < nk; ++kt) {
    const int cur = kt & 1;
    const bool more = kt + 1 < nk;
    if (more)
      load_slice<VEC_A, VEC_B>(A, lda, B, ldb, M, N, K, m0, n0, (kt + 1) * BK,
                               tid, ra, rb);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&s.a[cur][k][row_a]);
      const float4 a1 = *reinterpret_cast<const float4*>(&s.a[cur][k][row_a + 16]);
      const float4 b0 = *reinterpret_cast<const float4*>(&s.b[cur][k][col_b]);
      const float4 b1 = *reinterpret_cast<const float4*>(&s.b[cur][k][col_b + 32]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) store_slice(s, cur ^ 1, tid, ra, rb);
    __syncthreads();
  }

  // Epilogue: guarded stores, 16-byte vectors where the layout allows.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + row_a + (i < 4 ? i : 12 + i);
    if (gm >= M) continue;
    float* crow = C + static_cast<int64_t>(gm) * ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gn = n0 + col_b + 32 * h;
      if (vec_c && gn + 3 < N) {
        *reinterpret_cast<float4*>(crow + gn) =
            make_float4(acc[i][4 * h + 0], acc[i][4 * h + 1], acc[i][4 * h + 2],
                        acc[i][4 * h + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (gn + j < N) crow[gn + j] = acc[i][4 * h + j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_f32(int M, int N, int K, const float* A, int64_t lda,
                            const float* B, int64_t ldb, float* C, int64_t ldc,
                            bool vec_a, bool vec_b, bool vec_c,
                            cudaStream_t stream) {
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(tiles));
  const int vc = vec_c ? 1 : 0;
  if (vec_a && vec_b)
    gemm_f32_regblock_kernel<true, true><<<grid, THREADS, 0, stream>>>(
        M, N, K, A, lda, B, ldb, C, ldc, tiles_m, tiles_n, vc);
  else if (vec_a)
    gemm_f32_regblock_kernel<true, false><<<grid, THREADS, 0, stream>>>(
        M, N, K, A, lda, B, ldb, C, ldc, tiles_m, tiles_n, vc);
  else if (vec_b)
    gemm_f32_regblock_kernel<false, true><<<grid, THREADS, 0, stream>>>(
        M, N, K, A, lda, B, ldb, C, ldc, tiles_m, tiles_n, vc);
  else
    gemm_f32_regblock_kernel<false, false><<<grid, THREADS, 0, stream>>>(
        M, N, K, A, lda, B, ldb, C, ldc, tiles_m, tiles_n, vc);
  return cudaGetLastError();
}

}  // namespace g07
