// gemm_f32.cu -- FP32 GEMM on the CUDA cores: shared-memory tiling plus
// register blocking.
//
// Method ("GEMM, step by step", section "Concept", register blocking; "A06 --
// Tiled Matrix Multiply (GEMM)", section 3; "GEMM Optimization", sections 4-5):
//   * a block of 256 threads owns a 128 x 128 tile of C and walks K in
//     32-deep slices, staging a 128 x 32 slice of A and a 32 x 128 slice of B
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
//     suggests): a 2-deep ring of slices is filled with cp.async, which
//     copies global -> shared without passing through registers and zero-fills
//     out-of-range elements (the ": 0.0f" of the guarded tiled kernel); one
//     barrier per slice;
//   * stores are guarded on both row < M and col < N;
//   * wave tail: tiles fill whole waves of resident blocks; the tiles of a
//     last, partial wave are split along K (split-K, "A06", section 3) into
//     ranges computed by separate blocks of the same launch, whose partial
//     sums are added in a fixed order by the last block to finish, so the
//     tail keeps every SM busy and results stay deterministic.
//
// Thread layout: 8 warps as 4 (M) x 2 (N), each warp a 32 x 64 sub-tile;
// lane (ly = lane/8, lx = lane%8) owns rows {4ly..4ly+3, 16+4ly..16+4ly+3}
// and columns {4lx..4lx+3, 32+4lx..32+4lx+3} of its warp's sub-tile.
#include <atomic>
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
static_assert(THREADS % BK == 0 && BM % (THREADS / BK) == 0 && BM / (THREADS / BK) <= 32,
              "copy plan covers the A slice in whole passes");

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
  static constexpr int A_ROW_STEP = THREADS / BK;     // rows per pass over A
  static constexpr int A_ITERS = BM / A_ROW_STEP;     // passes per slice
  const float* a_ptr;  // A[m0 + r0][k], advanced by BK per slice
  const float* b_ptr;  // B[kr0][n0 + nc], advanced by BK rows per slice
  const float* a_base;
  const float* b_base;
  int64_t a_step;      // A_ROW_STEP rows of A
  int64_t b_step;      // B_ROW_STEP rows of B
  uint32_t a_rows_ok;  // bit i: row m0 + r0 + A_ROW_STEP * i < M
  uint32_t b_bytes;    // bytes of this thread's B group inside [0, N)
  uint32_t a_dst, b_dst;  // offsets of this thread's first element in a stage
  int k_a, k_b;        // k of this thread's A element / first B row, slice 0
  int K;

  __device__ __forceinline__ SliceLoader(const float* A, int64_t lda,
                                         const float* B, int64_t ldb, int M,
                                         int N, int K_, int m0, int n0,
                                         int kt_start, int tid) {
    K = K_;
    const int r0 = tid / BK;
    k_a = tid % BK;
    a_base = A;
    a_ptr = A + static_cast<int64_t>(m0 + r0) * lda + k_a;
    a_step = A_ROW_STEP * lda;
    a_rows_ok = 0;
#pragma unroll
    for (int i = 0; i < A_ITERS; ++i)
      if (m0 + r0 + A_ROW_STEP * i < M) a_rows_ok |= 1u << i;
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
    // start at k-slice kt_start
    a_ptr += static_cast<int64_t>(kt_start) * BK;
    b_ptr += static_cast<int64_t>(kt_start) * BK * ldb;
    b_dst = static_cast<uint32_t>(
        (offsetof(F32Stage<TN>, b) / sizeof(float) + k_b * TN + nc) * sizeof(float));
    (void)ldb;
  }

  // Issue the copies of slice kt into the stage at shared address `stage`
  // (slices must be requested in consecutive order from kt_start).
  __device__ __forceinline__ void load(uint32_t stage, int kt) {
    const int k0 = kt * BK;
    const bool ka = k0 + k_a < K;
#pragma unroll
    for (int i = 0; i < A_ITERS; ++i) {
      const bool ok = ka && ((a_rows_ok >> i) & 1u);
      cp_async4(stage + a_dst + i * A_ROW_STEP * sizeof(float),
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

// Guarded store of one 4-wide group of row `crow` at column gn, through the
// epilogue (prior C and bias read only when the epilogue needs them).
// GELU: whether the GELU activation is compiled in (epi_apply).
template <bool GELU>
__device__ __forceinline__ void store4(float* crow, int gn, int N, int vec_c,
                                       float4 v, const EpiParams& epi) {
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

// Last block of a split tile: add the `split` parked partial tiles in range
// order 0, 1, ..., split-1 and write this thread's 8 x 8 patch of C.  Four
// rows at a time: per range, the 8 float4 loads of those rows are issued
// together before they are added, so each range costs one L2 round trip
// rather than one per row.
template <bool GELU>
__device__ __noinline__ void reduce_ranges(const float* tile_ws, int split,
                                           float* C, int64_t ldc, int M, int N,
                                           int m0, int n0, int row_a, int col_b,
                                           int vec_c, EpiParams epi) {
#pragma unroll 1
  for (int g = 0; g < 2; ++g) {
    // rows row_a + {0..3} (g = 0) and row_a + {16..19} (g = 1)
    const float* src = tile_ws + (row_a + 16 * g) * BN + col_b;
    float4 sum[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        sum[i][h] = __ldcg(reinterpret_cast<const float4*>(src + i * BN + 32 * h));
#pragma unroll 1
    for (int q = 1; q < split; ++q) {
      const float* part = src + static_cast<int64_t>(q) * (BM * BN);
      float4 v[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          v[i][h] = __ldcg(reinterpret_cast<const float4*>(part + i * BN + 32 * h));
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          sum[i][h].x += v[i][h].x;
          sum[i][h].y += v[i][h].y;
          sum[i][h].z += v[i][h].z;
          sum[i][h].w += v[i][h].w;
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gm = m0 + row_a + 16 * g + i;
      if (gm >= M) continue;
      float* crow = C + static_cast<int64_t>(gm) * ldc;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        store4<GELU>(crow, n0 + col_b + 32 * h, N, vec_c, sum[i][h], epi);
    }
  }
}

// One launch computes every tile of the grouped order: blocks 0 .. first - 1
// compute tiles 0 .. first - 1 whole; the blocks after them cut each of the
// following tiles' k-slices into `split` contiguous ranges (split-K), block
// first + b taking range b % split of tile first + b / split.  Blocks are
// dispatched in index order, so the split blocks fill the SMs as the last
// whole wave drains.  A split tile's partial sums go to `ws` (split x 128 x
// 128 floats per tile); the last of its blocks to finish (per `counters`,
// zero at launch) adds the partials in range order 0, 1, ... and writes C,
// so the result does not depend on which block finishes last.
template <bool VEC_B, bool GELU>
__global__ void __launch_bounds__(THREADS, 2)
gemm_f32_regblock_kernel(int M, int N, int K, const float* __restrict__ A,
                         int64_t lda, const float* __restrict__ B, int64_t ldb,
                         float* __restrict__ C, int64_t ldc, int tiles_m,
                         int tiles_n, int first, int split, int vec_c,
                         float* __restrict__ ws, unsigned int* __restrict__ counters,
                         EpiParams epi) {
  constexpr int TN = BN;
  constexpr int JP = TN / 32;      // float2 accumulators per row
  extern __shared__ __align__(16) uint8_t smem_raw[];
  F32Stage<TN>* stage = reinterpret_cast<F32Stage<TN>*>(smem_raw);
  __shared__ int last_block;
  grid_dependency_wait();  // before the first read of A, B, C or the counters
  grid_dependents_go();

  // blocks [0, first): whole tiles 0 .. first - 1; then `split` blocks per
  // tile for tiles first, first + 1, ...
  const bool split_blk = static_cast<int>(blockIdx.x) >= first;
  const int bx = static_cast<int>(blockIdx.x) - (split_blk ? first : 0);
  const int sp = split_blk ? split : 1;
  const int local_tile = bx / sp;
  const int piece = bx % sp;
  const TileCoord tc = tile_order((split_blk ? first : 0) + local_tile, tiles_m, tiles_n, kF32Group);
  const int m0 = tc.m * BM;
  const int n0 = tc.n * BN;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int row_a = (warp >> 1) * 32 + (lane >> 3) * 4;      // + {0..3, 16..19}
  const int col_b = (warp & 1) * (TN / 2) + (lane & 7) * 4;  // + {0..3, 32..35}

  // acc[i][jp]: columns 2jp, 2jp+1 (then 32 + ...) of row i of the patch.
  float2 acc[8][JP];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < JP; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

  const int nk_all = (K + BK - 1) / BK;
  const int kt_begin = static_cast<int>(static_cast<int64_t>(nk_all) * piece / sp);
  const int kt_end = static_cast<int>(static_cast<int64_t>(nk_all) * (piece + 1) / sp);
  const int nk = kt_end - kt_begin;
  SliceLoader<TN, VEC_B> loader(A, lda, B, ldb, M, N, K, m0, n0, kt_begin, tid);
  const uint32_t stage0 = smem_addr(stage);
#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nk) loader.load(stage0 + s * sizeof(F32Stage<TN>), kt_begin + s);
    cp_async_commit();
  }

  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<STAGES - 2>();  // this thread's copies of slice kt landed
    __syncthreads();              // everyone's landed; slice kt-1 consumed
    {
      const int nxt = kt + STAGES - 1;
      if (nxt < nk)
        loader.load(stage0 + (nxt % STAGES) * sizeof(F32Stage<TN>), kt_begin + nxt);
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

  if (sp > 1) {
    // Park this range's partial tile, then count the tile's finished ranges.
    float* tile_ws = ws + static_cast<int64_t>(local_tile) * split * (BM * BN);
    float* mine = tile_ws + piece * (BM * BN);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = row_a + (i < 4 ? i : 12 + i);
#pragma unroll
      for (int h = 0; h < JP / 2; ++h)
        __stcg(reinterpret_cast<float4*>(mine + r * BN + col_b + 32 * h),
               make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                           acc[i][2 * h + 1].y));
    }
    __threadfence();
    __syncthreads();
    if (tid == 0)
      last_block = atomicAdd(&counters[local_tile], 1u) == static_cast<unsigned>(split - 1);
    __syncthreads();
    if (last_block) {
      __threadfence();
      reduce_ranges<GELU>(tile_ws, split, C, ldc, M, N, m0, n0, row_a, col_b, vec_c, epi);
      if (tid == 0) counters[local_tile] = 0;  // leave the counter as found
      // Every partial of this tile has been read: drop their lines from L2
      // without writing them back (the next launch writes them anew).
      __syncthreads();
      const int lines = split * (BM * BN * 4 / 128);
      for (int l = tid; l < lines; l += THREADS)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(tile_ws + l * 32) : "memory");
    }
    return;
  }

  // Epilogue: guarded stores, 16-byte vectors where the layout allows.
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + row_a + (i < 4 ? i : 12 + i);
    if (gm >= M) continue;
    float* crow = C + static_cast<int64_t>(gm) * ldc;
#pragma unroll
    for (int h = 0; h < JP / 2; ++h)
      store4<GELU>(crow, n0 + col_b + 32 * h, N, vec_c,
             make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                         acc[i][2 * h + 1].y),
             epi);
  }
}

// ------------------------------------------------------ small problems
//
// At most 16 tiles of 128 x 128 leave most SMs idle and each block a long
// serial K loop.  Small problems therefore run as 64 x 64 tiles, every tile
// split into `split` ranges of k-slices (a range may be a single slice), so
// that the blocks fill the GPU; the ranges are added in order by the last
// block of each tile, as for the wave tail above.  256 threads as 16 x 16,
// each a 4 x 4 patch (rows 4ty.., columns 4tx..); per k one 16-byte read of
// the transposed A slice and one of B; a 2-deep cp.async ring; plain FMAs.
constexpr int SB = kF32SmallTile;   // 64
constexpr int S_STRIDE = SB + 4;    // transposed A rows, padded
struct SmallStage {
  float a[BK][S_STRIDE];
  float b[BK][SB];
};

template <bool VEC_B>
__global__ void __launch_bounds__(THREADS)
gemm_f32_small_kernel(int M, int N, int K, const float* __restrict__ A, int64_t lda,
                      const float* __restrict__ B, int64_t ldb, float* __restrict__ C,
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
  // copy plan: A element (row tid / 32 + 8i, k tid % 32); B 16-byte groups
  // (row tid / 16 + 16j, columns 4 (tid % 16)..), or single elements (row
  // tid / 64 + 4j, column tid % 64)
  const int ak = tid & 31, ar = tid >> 5;
  auto load = [&](int buf, int kt) {
    const uint32_t sa = smem_addr(&st[buf]);
    const int k0 = kt * BK;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = ar + 8 * i, gm = m0 + r, gk = k0 + ak;
      const bool ok = gm < M && gk < K;
      cp_async4(sa + static_cast<uint32_t>((ak * S_STRIDE + r) * 4),
                ok ? A + static_cast<int64_t>(gm) * lda + gk : A, ok ? 4u : 0u);
    }
    const uint32_t sb = sa + static_cast<uint32_t>(offsetof(SmallStage, b));
    if (VEC_B) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (tid >> 4) + 16 * j, c = (tid & 15) * 4, gk = k0 + r, gn = n0 + c;
        const uint32_t bytes =
            gk < K && gn < N ? (N - gn >= 4 ? 16u : static_cast<uint32_t>(N - gn) * 4u) : 0u;
        cp_async16(sb + static_cast<uint32_t>((r * SB + c) * 4),
                   bytes ? B + static_cast<int64_t>(gk) * ldb + gn : B, bytes);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = (tid >> 6) + 4 * j, c = tid & 63, gk = k0 + r, gn = n0 + c;
        const bool ok = gk < K && gn < N;
        cp_async4(sb + static_cast<uint32_t>((r * SB + c) * 4),
                  ok ? B + static_cast<int64_t>(gk) * ldb + gn : B, ok ? 4u : 0u);
      }
    }
  };
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  if (kt0 < kt1) load(0, kt0);
  cp_async_commit();
  for (int kt = kt0; kt < kt1; ++kt) {
    const int buf = (kt - kt0) & 1;
    if (kt + 1 < kt1) load(buf ^ 1, kt + 1);
    cp_async_commit();
    cp_async_wait<1>();  // this thread's copies of slice kt landed
    __syncthreads();     // everyone's
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
    __syncthreads();     // slice kt consumed before its buffer is refilled
  }
  cp_async_wait<0>();
  const int col = n0 + tx * 4;
  if (split > 1) {
    float* tile_ws = ws + static_cast<int64_t>(tile) * split * (SB * SB);
    float* mine = tile_ws + piece * (SB * SB);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      __stcg(reinterpret_cast<float4*>(mine + (ty * 4 + i) * SB + tx * 4),
             make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    __threadfence();
    __syncthreads();
    if (tid == 0)
      last_block = atomicAdd(&counters[tile], 1u) == static_cast<unsigned>(split - 1);
    __syncthreads();
    if (!last_block) return;
    __threadfence();
    // ranges added in order 0, 1, ..., split - 1; each range's four loads
    // of this thread are in flight together
    float4 sum[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      sum[i] = __ldcg(reinterpret_cast<const float4*>(tile_ws + (ty * 4 + i) * SB + tx * 4));
#pragma unroll 1
    for (int q = 1; q < split; ++q) {
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = __ldcg(reinterpret_cast<const float4*>(tile_ws + q * (SB * SB) +
                                                     (ty * 4 + i) * SB + tx * 4));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sum[i].x += v[i].x;
        sum[i].y += v[i].y;
        sum[i].z += v[i].z;
        sum[i].w += v[i].w;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gm = m0 + ty * 4 + i;
      if (gm < M) store4<true>(C + static_cast<int64_t>(gm) * ldc, col, N, vec_c, sum[i], epi);
    }
    if (tid == 0) counters[tile] = 0;  // leave the counter as found
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm < M)
      store4<true>(C + static_cast<int64_t>(gm) * ldc, col, N, vec_c,
                   make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]), epi);
  }
}

// The kernel copy with GELU compiled in only for that activation.
template <bool VEC_B>
cudaError_t launch_part(int blocks, int M, int N, int K, const float* A,
                        int64_t lda, const float* B, int64_t ldb, float* C,
                        int64_t ldc, int tiles_m, int tiles_n, int first,
                        int split, int vec_c, float* ws, unsigned int* counters,
                        const EpiParams& epi, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(STAGES) * sizeof(F32Stage<BN>);
  auto kernel = epi.act == kActGelu ? gemm_f32_regblock_kernel<VEC_B, true>
                                     : gemm_f32_regblock_kernel<VEC_B, false>;
  const cudaError_t e =
      launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(THREADS), smem, stream, M, N,
                 K, A, lda, B, ldb, C, ldc, tiles_m, tiles_n, first, split, vec_c, ws,
                 counters, epi);
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

template <bool VEC_B, bool GELU>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_f32_regblock_kernel<VEC_B, GELU>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(STAGES * sizeof(F32Stage<BN>)));
}

// Per device: 0 until the shared-memory attributes are set and the
// occupancy known, then the number of resident blocks + 1.  One atomic
// word, so that a thread that finds it set also finds the attributes set
// (calls may come from several host threads at once).
std::atomic<int64_t> g_slots_plus1[64];

}  // namespace

// Resident blocks of the FP32 kernel on the current device (cached).
int64_t f32_slots() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int64_t known = g_slots_plus1[dev].load(std::memory_order_acquire);
  if (known > 0) return known - 1;
  {
    if (set_smem_attr<true, false>() != cudaSuccess ||
        set_smem_attr<false, false>() != cudaSuccess ||
        set_smem_attr<true, true>() != cudaSuccess ||
        set_smem_attr<false, true>() != cudaSuccess)
      return 0;
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, gemm_f32_regblock_kernel<true, false>, THREADS,
            STAGES * sizeof(F32Stage<BN>)) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    const int64_t slots = static_cast<int64_t>(sms) * per_sm;
    g_slots_plus1[dev].store(slots + 1, std::memory_order_release);
    return slots;
  }
}

F32Plan f32_plan(int M, int N, int K, int64_t slots) {
  F32Plan p;
  if (f32_small_problem(M, N, K)) {
    // every 64 x 64 tile split into ranges of k-slices, about two blocks
    // per SM in all
    p.small = true;
    p.tiles_m = (M + SB - 1) / SB;
    p.tiles_n = (N + SB - 1) / SB;
    const int tiles = p.tiles_m * p.tiles_n;
    const int nk = (K + BK - 1) / BK;
    int split = slots > 0 ? static_cast<int>(slots / tiles) : 1;
    if (split > 16) split = 16;
    if (split > nk) split = nk;
    p.split = split < 1 ? 1 : split;
    p.tail = tiles;
    p.workspace_bytes =
        p.split > 1 ? static_cast<int64_t>(tiles) * p.split * SB * SB * 4 : 0;
    p.counter_bytes = p.split > 1 ? static_cast<int64_t>(tiles) * 4 : 0;
    return p;
  }
  p.tiles_m = (M + BM - 1) / BM;
  p.tiles_n = (N + BN - 1) / BN;
  const int64_t tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  const int nk = (K + BK - 1) / BK;
  p.tail = slots > 0 ? static_cast<int>(tiles % slots) : 0;
  p.full = static_cast<int>(tiles - p.tail);
  p.split = 1;
  if (p.tail > 0) {
    // Split the tiles of the last, partial wave along K so that its blocks
    // fill the resident slots: choose the split with the lowest estimated
    // time in units of one tile's main loop, rounds x (1/split + a per-round
    // overhead for the pipeline fill, 1/50 of a tile) plus the last block's
    // reading of the split partial tiles (about 1/15 of a k-slice each), at
    // most 16 ranges.  A last wave with fewer tiles than resident slots is
    // split too, since an SM holding one block runs it slower than two.
    // Ranges keep at least 4 k-slices, unless the split tiles then still
    // fit in one round of resident blocks (a short K with few tiles, e.g.
    // 256^3: 4 tiles of 8 slices, spreads over more SMs).
    double best = 1e30;
    const int max_split = nk < 16 ? nk : 16;
    const int long_split = nk / 4 > 1 ? nk / 4 : 1;
    const double reduce_per_range = 0.07 / nk;
    for (int s = 1; s <= max_split; ++s) {
      const int64_t rounds = (static_cast<int64_t>(p.tail) * s + slots - 1) / slots;
      if (s > long_split && rounds > 1) break;
      const double cost = static_cast<double>(rounds) * (1.0 / s + 0.02) +
                          (s > 1 ? reduce_per_range * s : 0.0);
      if (cost < best - 1e-9) {
        best = cost;
        p.split = s;
      }
    }
  }
  p.workspace_bytes =
      p.split > 1 ? static_cast<int64_t>(p.tail) * p.split * BM * BN * 4 : 0;
  p.counter_bytes = p.split > 1 ? static_cast<int64_t>(p.tail) * 4 : 0;
  return p;
}

// Whole waves of tiles first, then the tiles of the last, partial wave split
// along K as planned, all in one launch.
cudaError_t launch_gemm_f32(int M, int N, int K, const float* A, int64_t lda,
                            const float* B, int64_t ldb, float* C, int64_t ldc,
                            bool vec_b, bool vec_c, const F32Plan& p, float* ws,
                            unsigned int* counters, const EpiParams& epi,
                            cudaStream_t stream) {
  if (f32_slots() <= 0) return cudaErrorInvalidDeviceFunction;
  const int vc = vec_c ? 1 : 0;
  cudaError_t e = cudaSuccess;
  if (p.small) {
    const int blocks = p.tiles_m * p.tiles_n * p.split;
    e = launch_pdl(vec_b ? gemm_f32_small_kernel<true> : gemm_f32_small_kernel<false>,
                   dim3(static_cast<unsigned>(blocks)), dim3(THREADS), 0, stream, M, N, K, A,
                   lda, B, ldb, C, ldc, p.tiles_n, p.split, vc, ws, counters, epi);
    if (e == cudaSuccess) note_launches(1);
    return e;
  }
  {
    const int blocks = p.full + p.tail * (p.tail > 0 ? p.split : 1);
    const int sp = p.tail > 0 ? p.split : 1;
    e = vec_b ? launch_part<true>(blocks, M, N, K, A, lda, B, ldb, C, ldc,
                                  p.tiles_m, p.tiles_n, p.full, sp, vc, ws,
                                  counters, epi, stream)
              : launch_part<false>(blocks, M, N, K, A, lda, B, ldb, C, ldc,
                                   p.tiles_m, p.tiles_n, p.full, sp, vc, ws,
                                   counters, epi, stream);
  }
  return e;
}

}  // namespace g07
