// gemm_f32_ladder.cu -- the teaching rungs of the FP32 GEMM ladder, kept for
// measurement beside the product kernel (gemm_f32.cu), not as a product path.
//
//   rung 0  one thread per output, x -> column so a warp reads one row of B
//           contiguously and broadcasts one element of A ("How a Matrix
//           Multiply Runs on a GPU", "Level 0"; "GEMM" (inference-book), the
//           coalesced remapping).  Intensity 0.25 FLOP/byte.
//   rung 1  T x T shared-memory tiles, T = 32, one output per thread: the
//           idea of "How a Matrix Multiply Runs on a GPU", "Level 1" and
//           "A06", section 3 (each staged element serves T outputs;
//           out-of-range elements count as 0).  Intensity T/4 = 8 FLOP/byte.
//           Our realisation: k-major padded A tile, two tile buffers fed
//           through registers, one barrier per k-tile (see the kernel).
//   rung 2  1-D register tiling: a 64 x 64 block, 8-deep k-tiles, each thread
//           computes 8 consecutive rows of one column, reusing one value of B
//           for 8 FMAs ("GEMM" (inference-book), one-dimensional register
//           tiling).
// The 2-D register-blocked kernel of gemm_f32.cu is the ladder's last rung.
#include <cstdint>

#include "kernels.h"

namespace g07 {
namespace {

__global__ void ladder_naive_kernel(int M, int N, int K, const float* __restrict__ A,
                                    int64_t lda, const float* __restrict__ B,
                                    int64_t ldb, float* __restrict__ C,
                                    int64_t ldc) {
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  const int row = blockIdx.y * blockDim.y + threadIdx.y;
  if (row >= M || col >= N) return;
  const float* a = A + static_cast<int64_t>(row) * lda;
  float acc = 0.0f;
  for (int k = 0; k < K; ++k) acc = fmaf(a[k], B[static_cast<int64_t>(k) * ldb + col], acc);
  C[static_cast<int64_t>(row) * ldc + col] = acc;
}

// Rung 1.  A block of 1024 threads owns a 32 x 32 tile of C, one output per
// thread: thread t holds row t / 32, column t % 32 of the tile.  C is built
// from k-tiles of depth 32; each brings 32 x 32 of A and 32 x 32 of B into
// shared memory once, and every element brought in is read by 32 threads
// (global intensity T/4 FLOP per byte).
//   * A is kept k-major (at[k][r]) with rows padded to 33 words: the warp
//     that fetched one row segment of A writes it down a column, and the 33
//     stride puts its 32 stores in 32 different banks; in the products a
//     warp then reads one broadcast word of A and 32 consecutive words of B
//     per k.
//   * Two buffers per operand: the next k-tile is fetched into registers
//     before the current one is multiplied and stored into the other buffer
//     after, so one barrier per k-tile orders both the stores before the
//     next reads and the reads before the buffer is reused.
//   * Elements outside A or B are taken as 0, so a ragged K or edge tile
//     adds nothing; only outputs inside C are stored.
constexpr int T = 32;
constexpr int TP = T + 1;

__global__ void __launch_bounds__(T * T)
ladder_tiled_kernel(int M, int N, int K, const float* __restrict__ A, int64_t lda,
                    const float* __restrict__ B, int64_t ldb,
                    float* __restrict__ C, int64_t ldc) {
  __shared__ float at[2][T][TP];  // at[buf][k][r] = A[m0 + r][k0 + k]
  __shared__ float bt[2][T][T];   // bt[buf][k][c] = B[k0 + k][n0 + c]
  const int r = threadIdx.x >> 5;  // also: which row of A / of B this thread fetches
  const int c = threadIdx.x & 31;  // also: which element of that row segment
  const int m0 = blockIdx.y * T, n0 = blockIdx.x * T;
  const bool a_row_in = m0 + r < M, b_col_in = n0 + c < N;
  const float* a_row = A + static_cast<int64_t>(a_row_in ? m0 + r : 0) * lda;
  const float* b_col = B + (b_col_in ? n0 + c : 0);

  float a_next = 0.0f, b_next = 0.0f;
  auto fetch = [&](int k0) {
    a_next = a_row_in && k0 + c < K ? a_row[k0 + c] : 0.0f;
    b_next = b_col_in && k0 + r < K ? b_col[static_cast<int64_t>(k0 + r) * ldb] : 0.0f;
  };
  auto put = [&](int buf) {
    at[buf][c][r] = a_next;
    bt[buf][r][c] = b_next;
  };

  fetch(0);
  put(0);
  __syncthreads();
  float acc = 0.0f;
  int buf = 0;
  for (int k0 = 0; k0 < K; k0 += T, buf ^= 1) {
    const bool more = k0 + T < K;
    if (more) fetch(k0 + T);
#pragma unroll
    for (int k = 0; k < T; ++k) acc = fmaf(at[buf][k][r], bt[buf][k][c], acc);
    if (more) put(buf ^ 1);
    __syncthreads();
  }
  if (a_row_in && b_col_in) C[static_cast<int64_t>(m0 + r) * ldc + n0 + c] = acc;
}

constexpr int R_BM = 64, R_BN = 64, R_BK = 8, R_TM = 8;
constexpr int R_THREADS = (R_BM / R_TM) * R_BN;  // 512

__global__ void __launch_bounds__(R_THREADS)
ladder_reg1d_kernel(int M, int N, int K, const float* __restrict__ A,
                    int64_t lda, const float* __restrict__ B, int64_t ldb,
                    float* __restrict__ C, int64_t ldc) {
  __shared__ float As[R_BM][R_BK];
  __shared__ float Bs[R_BK][R_BN];
  const int tid = threadIdx.x;
  const int tcol = tid % R_BN;        // column of C this thread owns
  const int trow = tid / R_BN;        // which group of 8 rows
  const int m0 = blockIdx.y * R_BM, n0 = blockIdx.x * R_BN;
  // cooperative loads: 512 threads load 64 x 8 of A and 8 x 64 of B
  const int a_r = tid / R_BK, a_k = tid % R_BK;
  const int b_k = tid / R_BN, b_c = tid % R_BN;
  float acc[R_TM] = {};
  for (int k0 = 0; k0 < K; k0 += R_BK) {
    As[a_r][a_k] = (m0 + a_r < M && k0 + a_k < K)
                       ? A[static_cast<int64_t>(m0 + a_r) * lda + k0 + a_k] : 0.0f;
    Bs[b_k][b_c] = (k0 + b_k < K && n0 + b_c < N)
                       ? B[static_cast<int64_t>(k0 + b_k) * ldb + n0 + b_c] : 0.0f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < R_BK; ++k) {
      const float b = Bs[k][tcol];   // one value of B feeds 8 FMAs
#pragma unroll
      for (int i = 0; i < R_TM; ++i) acc[i] = fmaf(As[trow * R_TM + i][k], b, acc[i]);
    }
    __syncthreads();
  }
  const int col = n0 + tcol;
  if (col >= N) return;
#pragma unroll
  for (int i = 0; i < R_TM; ++i) {
    const int row = m0 + trow * R_TM + i;
    if (row < M) C[static_cast<int64_t>(row) * ldc + col] = acc[i];
  }
}

}  // namespace

cudaError_t launch_gemm_f32_ladder(int rung, int M, int N, int K, const float* A,
                                   int64_t lda, const float* B, int64_t ldb,
                                   float* C, int64_t ldc, cudaStream_t stream) {
  switch (rung) {
    case 0: {
      const dim3 block(32, 8);
      const dim3 grid((N + 31) / 32, (M + 7) / 8);
      ladder_naive_kernel<<<grid, block, 0, stream>>>(M, N, K, A, lda, B, ldb, C, ldc);
      break;
    }
    case 1: {
      const dim3 block(T * T);
      const dim3 grid((N + T - 1) / T, (M + T - 1) / T);
      ladder_tiled_kernel<<<grid, block, 0, stream>>>(M, N, K, A, lda, B, ldb, C, ldc);
      break;
    }
    case 2: {
      const dim3 grid((N + R_BN - 1) / R_BN, (M + R_BM - 1) / R_BM);
      ladder_reg1d_kernel<<<grid, R_THREADS, 0, stream>>>(M, N, K, A, lda, B, ldb, C, ldc);
      break;
    }
    default:
      return cudaErrorInvalidValue;
  }
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace g07
