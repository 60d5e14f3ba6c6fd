// gemm_f32.cu -- FP32 GEMM on the CUDA cores: shared-memory tiling plus
// register blocking.
//
// Method ("GEMM, step by step", section "Concept", register blocking; "A06 --
// Tiled Matrix Multiply (GEMM)", section 3; "GEMM Optimization", sections 4-5):
//   * a block of 256 threads owns a 128 x 128 tile of C and walks K in
//     16-deep slices, staging a 128 x 16 slice of A and a 16 x 128 slice of B
//     in shared memory;
//   * each thread owns an 8 x 8 patch of C in registers: per k it reads 8
//     values of A and 8 of B from shared memory and does 64 FMAs, issued as
//     32 packed two-lane FP32 FMAs (each lane an ordinary, individually
//     rounded FMA, so results equal those of 64 scalar FMAs);
//   * A's slice is stored transposed (As[k][m], row stride 132 floats) so a
//     thread's 8 A values are two 16-byte reads, and B's 8 values are two
//     16-byte reads of Bs[k][n];
//   * multi-stage prefetch ("Double buffering" in "GEMM Optimization",
//     section 5, written with asynchronous copies as "A06", section 3,
//     suggests): a 3-deep ring of slices is filled with cp.async, which
//     copies global -> shared without passing through registers and zero-fills
//     out-of-range elements (the ": 0.0f" of the guarded tiled kernel); one
//     barrier per slice;
//   * stores are guarded on both row < M and col < N.
//
// Thread layout: 8 warps as 4 (M) x 2 (N), each warp a 32 x 64 sub-tile;
// lane (ly = lane/8, lx = lane%8) owns rows {4ly..4ly+3, 16+4ly..16+4ly+3}
// and columns {4lx..4lx+3, 32+4lx..32+4lx+3} of its warp's sub-tile.
#include <cstddef>
#include <cstdint>

#include "kernels.h"
#include "tile_order.cuh"

namespace g07 {
namespace {

constexpr int BM = kF32TileM;
constexpr int BN = kF32TileN;
constexpr int BK = kF32TileK;
constexpr int THREADS = 256;
constexpr int STAGES = kF32Stages;
constexpr int A_STRIDE = BM + 4;  // transposed A rows, padded

template <int TN>
struct F32Stage {
  float a[BK][A_STRIDE];
  float b[BK][TN];
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 4-byte asynchronous copy; src_bytes 0 writes a zero.
__device__ __forceinline__ void cp_async4(uint32_t dst, const float* src,
                                          uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

// 16-byte asynchronous copy of the first src_bytes (0..16) bytes, rest zero.
__device__ __forceinline__ void cp_async16(uint32_t dst, const float* src,
                                           uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Per-thread copy plan, set up once per block: one pointer per operand that
// advances by one slice per call, plus the row/column validity the copies
// need (out-of-range elements are written as zeros).
template <int TN, bool VEC_B>
struct SliceLoader {
  static constexpr int B_ITERS = VEC_B ? BK * TN / 4 / THREADS : BK * TN / THREADS;
  static constexpr int B_ROW_STEP = VEC_B ? THREADS / (TN / 4) : THREADS / TN;
  const float* a_ptr;  // A[m0 + r0][k], advanced by BK per slice
  const float* b_ptr;  // B[kr0][n0 + nc], advanced by BK rows per slice
  const float* a_base;
  const float* b_base;
  int64_t a_step;      // 16 rows of A
  int64_t b_step;      // B_ROW_STEP rows of B
  uint32_t a_rows_ok;  // bit i: row m0 + r0 + 16 i < M
  uint32_t b_bytes;    // bytes of this thread's B group inside [0, N)
  uint32_t a_dst, b_dst;  // offsets of this thread's first element in a stage
  int k_a, k_b;        // k of this thread's A element / first B row, slice 0
  int K;

  __device__ __forceinline__ SliceLoader(const float* A, int64_t lda,
                                         const float* B, int64_t ldb, int M,
                                         int N, int K_, int m0, int n0,
                                         int tid) {
    K = K_;
    const int r0 = tid >> 4;
    k_a = tid & 15;
    a_base = A;
    a_ptr = A + static_cast<int64_t>(m0 + r0) * lda + k_a;
    a_step = 16 * lda;
    a_rows_ok = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (m0 + r0 + 16 * i < M) a_rows_ok |= 1u << i;
    a_dst = static_cast<uint32_t>((k_a * A_STRIDE + r0) * sizeof(float));
    b_base = B;
    int nc;
    if (VEC_B) {
      k_b = tid / (TN / 4);
      nc = (tid % (TN / 4)) * 4;
      const int gn = n0 + nc;
      b_bytes = gn < N ? (N - gn >= 4 ? 16u : static_cast<uint32_t>(N - gn) * 4u) : 0u;
    } else {
      k_b = tid / TN;
      nc = tid % TN;
      b_bytes = (n0 + nc < N) ? 4u : 0u;
    }
    b_ptr = B + static_cast<int64_t>(k_b) * ldb + n0 + nc;
    b_step = B_ROW_STEP * ldb;
    b_dst = static_cast<uint32_t>(
        (offsetof(F32Stage<TN>, b) / sizeof(float) + k_b * TN + nc) * sizeof(float));
    (void)ldb;
  }

  // Issue the copies of slice kt into the stage at shared address `stage`.
  __device__ __forceinline__ void load(uint32_t stage, int kt) {
    const int k0 = kt * BK;
    const bool ka = k0 + k_a < K;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool ok = ka && ((a_rows_ok >> i) & 1u);
      cp_async4(stage + a_dst + i * 16 * sizeof(float),
                ok ? a_ptr + i * a_step : a_base, ok ? 4u : 0u);
    }
    a_ptr += BK;
#pragma unroll
    for (int i = 0; i < B_ITERS; ++i) {
      const bool ok = b_bytes && (k0 + k_b + B_ROW_STEP * i < K);
      const float* src = ok ? b_ptr + i * b_step : b_base;
      const uint32_t dst = stage + b_dst + i * B_ROW_STEP * TN * sizeof(float);
      if (VEC_B)
        cp_async16(dst, src, ok ? b_bytes : 0u);
      else
        cp_async4(dst, src, ok ? 4u : 0u);
    }
    b_ptr += B_ITERS * b_step;
  }
};

// TN = 128: full 128 x 128 tiles, thread patch 8 x 8.  TN = 64: half-width
// 128 x 64 tiles (thread patch 8 x 4) for the last, partial wave of a grid.
// Tile `first + blockIdx.x / SPLIT` of the grouped order is computed; with
// SPLIT = 2 each block takes column half blockIdx.x % 2 of it.
template <int TN, bool VEC_B>
__global__ void __launch_bounds__(THREADS, 2)
gemm_f32_regblock_kernel(int M, int N, int K, const float* __restrict__ A,
                         int64_t lda, const float* __restrict__ B, int64_t ldb,
                         float* __restrict__ C, int64_t ldc, int tiles_m,
                         int tiles_n, int first, int vec_c) {
  constexpr int SPLIT = BN / TN;   // column pieces per 128 x 128 tile
  constexpr int JP = TN / 32;      // float2 accumulators per row (4 or 2)
  extern __shared__ __align__(16) uint8_t smem_raw[];
  F32Stage<TN>* stage = reinterpret_cast<F32Stage<TN>*>(smem_raw);

  const TileCoord tc =
      tile_order(first + blockIdx.x / SPLIT, tiles_m, tiles_n, kF32Group);
  const int m0 = tc.m * BM;
  const int n0 = tc.n * BN + (blockIdx.x % SPLIT) * TN;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int row_a = (warp >> 1) * 32 + (lane >> 3) * 4;      // + {0..3, 16..19}
  const int col_b = (warp & 1) * (TN / 2) + (lane & 7) * 4;  // + {0..3[, 32..35]}

  // acc[i][jp]: columns 2jp, 2jp+1 (then 32 + ...) of row i of the patch.
  float2 acc[8][JP];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < JP; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

  const int nk = (K + BK - 1) / BK;
  SliceLoader<TN, VEC_B> loader(A, lda, B, ldb, M, N, K, m0, n0, tid);
  const uint32_t stage0 = smem_addr(stage);
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nk) loader.load(stage0 + s * sizeof(F32Stage<TN>), s);
    cp_async_commit();
  }

  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<STAGES - 2>();  // this thread's copies of slice kt landed
    __syncthreads();              // everyone's landed; slice kt-1 consumed
    {
      const int nxt = kt + STAGES - 1;
      if (nxt < nk) loader.load(stage0 + (nxt % STAGES) * sizeof(F32Stage<TN>), nxt);
      cp_async_commit();
    }
    const F32Stage<TN>& st = stage[kt % STAGES];
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&st.a[k][row_a]);
      const float4 a1 = *reinterpret_cast<const float4*>(&st.a[k][row_a + 16]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      float2 b[JP];
#pragma unroll
      for (int h = 0; h < JP / 2; ++h) {
        const float4 bv = *reinterpret_cast<const float4*>(&st.b[k][col_b + 32 * h]);
        b[2 * h] = make_float2(bv.x, bv.y);
        b[2 * h + 1] = make_float2(bv.z, bv.w);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
        for (int j = 0; j < JP; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
      }
    }
  }
  cp_async_wait<0>();

  // Epilogue: guarded stores, 16-byte vectors where the layout allows.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + row_a + (i < 4 ? i : 12 + i);
    if (gm >= M) continue;
    float* crow = C + static_cast<int64_t>(gm) * ldc;
#pragma unroll
    for (int h = 0; h < JP / 2; ++h) {
      const int gn = n0 + col_b + 32 * h;
      const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                          acc[i][2 * h + 1].y};
      if (vec_c && gn + 3 < N) {
        *reinterpret_cast<float4*>(crow + gn) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (gn + j < N) crow[gn + j] = v[j];
      }
    }
  }
}

template <int TN, bool VEC_B>
cudaError_t launch_part(int blocks, int M, int N, int K, const float* A,
                        int64_t lda, const float* B, int64_t ldb, float* C,
                        int64_t ldc, int tiles_m, int tiles_n, int first,
                        int vec_c, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(STAGES) * sizeof(F32Stage<TN>);
  gemm_f32_regblock_kernel<TN, VEC_B><<<blocks, THREADS, smem, stream>>>(
      M, N, K, A, lda, B, ldb, C, ldc, tiles_m, tiles_n, first, vec_c);
  note_launches(1);
  return cudaGetLastError();
}

template <int TN, bool VEC_B>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_f32_regblock_kernel<TN, VEC_B>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(STAGES * sizeof(F32Stage<TN>)));
}

int g_attr_set[64];
int64_t g_slots[64];

}  // namespace

int f32_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, gemm_f32_regblock_kernel<BN, true>, THREADS,
          STAGES * sizeof(F32Stage<BN>)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Whole waves of full tiles first; the tiles of a last, partial wave are
// split into two half-width tiles when that keeps them within one wave
// (the grid is then two launches on the stream).
cudaError_t launch_gemm_f32(int M, int N, int K, const float* A, int64_t lda,
                            const float* B, int64_t ldb, float* C, int64_t ldc,
                            bool /*vec_a*/, bool vec_b, bool vec_c,
                            cudaStream_t stream) {
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
  if (tiles > 0x3FFFFFFF) return cudaErrorInvalidConfiguration;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_attr_set[dev]) {
    e = set_smem_attr<BN, true>();
    if (e == cudaSuccess) e = set_smem_attr<BN, false>();
    if (e == cudaSuccess) e = set_smem_attr<BN / 2, true>();
    if (e == cudaSuccess) e = set_smem_attr<BN / 2, false>();
    if (e != cudaSuccess) return e;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_slots[dev] = sms * f32_blocks_per_sm();
    g_attr_set[dev] = 1;
  }
  const int64_t slots = g_slots[dev];
  const int64_t tail = slots > 0 ? tiles % slots : 0;
  const int64_t split = (tail > 0 && 2 * tail <= slots) ? tail : 0;
  const int full = static_cast<int>(tiles - split);
  const int vc = vec_c ? 1 : 0;
  if (full > 0) {
    e = vec_b ? launch_part<BN, true>(full, M, N, K, A, lda, B, ldb, C, ldc,
                                      tiles_m, tiles_n, 0, vc, stream)
              : launch_part<BN, false>(full, M, N, K, A, lda, B, ldb, C, ldc,
                                       tiles_m, tiles_n, 0, vc, stream);
    if (e != cudaSuccess) return e;
  }
  if (split > 0) {
    const int blocks = static_cast<int>(2 * split);
    e = vec_b ? launch_part<BN / 2, true>(blocks, M, N, K, A, lda, B, ldb, C,
                                          ldc, tiles_m, tiles_n, full, vc, stream)
              : launch_part<BN / 2, false>(blocks, M, N, K, A, lda, B, ldb, C,
                                           ldc, tiles_m, tiles_n, full, vc, stream);
  }
  return e;
}

}  // namespace g07
