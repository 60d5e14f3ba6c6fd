// gemm_bf16_tc.cu -- BF16 x BF16 -> FP32 GEMM on the Blackwell tensor cores.
//
// Method: the tensor-core rung of "GEMM, step by step" (section "Concept"):
// BF16 inputs, FP32 sums, production-size 128 x 256 output tiles, and a block
// order that keeps neighbouring blocks on the same rows of A and columns of B
// ("GEMM Optimization", section "L2 Cache and Wave Analysis").  The slices of
// A and B move through a multi-stage shared-memory ring so that loading slice
// t+1 overlaps the multiply of slice t ("GEMM Optimization", section 5;
// "A06", section 3, "Double buffering / prefetch").
//
// sm_103a realisation (one CTA per SM, persistent over output tiles):
//   warp 0      producer: one thread issues TMA tensor copies of a 128 x 64
//               slice of A (K-major) and a 64 x 256 slice of B (N-major, four
//               64 x 64 boxes) into a 4-stage ring, 48 KB per stage, both
//               128-byte swizzled; completion is counted in bytes on the
//               stage's "full" mbarrier.  Out-of-range rows/columns/k are
//               filled with zeros by the copy engine.
//   warp 1      MMA issuer: one thread waits on "full", issues four
//               tcgen05.mma (M=128, N=256, K=16) per stage into an FP32
//               accumulator in tensor memory, and commits to the stage's
//               "empty" mbarrier; after the last slice of a tile it commits to
//               "accumulator full".  Tensor memory holds two 256-column
//               accumulators so the next tile's MMAs overlap this tile's
//               epilogue.
//   warps 2-5   epilogue: each warp owns the 32 accumulator rows (TMEM lanes)
//               its warp index allows, reads them 32 columns at a time with
//               tcgen05.ld and writes C with 16-byte stores guarded on
//               row < M and col < N, then frees the accumulator.
// Every wait is bounded: a wait that runs out raises the CTA's abort flag and
// the device status word, all roles unwind, in-flight copies and MMAs are
// drained, tensor memory is released and the kernel returns.
#include <cstdint>

#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tile_order.cuh"

namespace g07 {
namespace {

constexpr int BM = kTcTileM;
constexpr int BN = kTcTileN;
constexpr int BK = kTcTileK;
constexpr int STAGES = kTcStages;
constexpr int A_STAGE_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BOX_COLS = 64;                     // 128-byte swizzle span
constexpr int B_BOX_BYTES = BK * B_BOX_COLS * 2;   // 8 KB
constexpr int B_STAGE_BYTES = BK * BN * 2;         // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int MMA_K = 16;
constexpr int TMEM_COLS = 2 * BN;                  // two FP32 accumulators
constexpr int THREADS = 192;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, /*a_mn_major=*/false,
                                          /*b_mn_major=*/true);

static_assert(TMEM_COLS == 512, "tensor memory holds 512 columns per SM");
static_assert(BK * 2 == 128, "A rows are one 128-byte swizzle atom wide");

struct alignas(8) TcControl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(volatile int* abort,
                                            unsigned int* status) {
  *abort = 1;
  atomicOr(status, 1u);
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    float* __restrict__ C, int64_t ldc, int M, int N, int K,
                    int tiles_m, int tiles_n, int vec_c,
                    unsigned int* __restrict__ status, EpiParams epi) {
  extern __shared__ uint8_t smem_raw[];
  // The swizzle atoms must start on 1024-byte boundaries.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  TcControl* ctl = reinterpret_cast<TcControl*>(smem + STAGES * STAGE_BYTES);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = tiles_m * tiles_n;
  const int num_kb = (K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->acc_full[a], 1);
      mbar_init(&ctl->acc_empty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  const uint64_t tmo = wait_limit_ns(status);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const TileCoord tc = tile_order(tile, tiles_m, tiles_n, kTcGroup);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort, tmo)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_STAGE_BYTES;
          mbar_arrive_expect_tx(&ctl->full[stage], STAGE_BYTES);
          tma_load_2d(sa, &tmA, &ctl->full[stage], kb * BK, tc.m * BM);
#pragma unroll
          for (int j = 0; j < BN / B_BOX_COLS; ++j)
            tma_load_2d(sb + j * B_BOX_BYTES, &tmB, &ctl->full[stage],
                        tc.n * BN + j * B_BOX_COLS, kb * BK);
          last_phase[stage] = static_cast<int>(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort, status);
      // Every copy issued must have landed before the CTA may exit.
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (last_phase[s] >= 0 &&
            !mbar_wait(&ctl->full[s], static_cast<uint32_t>(last_phase[s]),
                       &never, tmo))
          raise_abort(abort, status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued = false;
      int t = 0;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++t) {
        const int acc = t & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(t >> 1) & 1u;
        if (!mbar_wait(&ctl->acc_empty[acc], acc_phase ^ 1u, abort, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&ctl->full[stage], phase, abort, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / MMA_K; ++kk) {
            // A: K-major rows of 128 bytes; a 16-wide k step is 32 bytes in.
            const uint64_t adesc =
                sdesc_sw128(a_addr + kk * MMA_K * 2, 16, 1024);
            // B: N-major; 64-column boxes 8 KB apart (LBO), 8-row k groups
            // 1 KB apart (SBO); a 16-deep k step is 16 rows = 2 KB in.
            const uint64_t bdesc =
                sdesc_sw128(b_addr + kk * MMA_K * 128, B_BOX_BYTES, 1024);
            mma_f16_ss(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&ctl->empty[stage]);
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&ctl->acc_full[acc]);
      }
      if (!ok) raise_abort(abort, status);
      // Every MMA issued must be complete before tensor memory is released.
      if (issued) {
        mma_commit(&ctl->drain);
        volatile int never = 0;
        if (!mbar_wait(&ctl->drain, 0u, &never, tmo)) raise_abort(abort, status);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lanes 32q..32q+31 are this warp's
    int t = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++t) {
      const int acc = t & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(t >> 1) & 1u;
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&ctl->acc_full[acc], acc_phase, abort, tmo) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) raise_abort(abort, status);
        break;
      }
      tc_fence_after_sync();
      const TileCoord tc = tile_order(tile, tiles_m, tiles_n, kTcGroup);
      const int row = tc.m * BM + q * 32 + lane;
      float* crow = C + static_cast<int64_t>(row) * ldc;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait();
        const int gn = tc.n * BN + c * 32;
        if (row < M) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (gn + j < N)
              crow[gn + j] = epi_apply(epi, __uint_as_float(r[j]),
                                       epi.beta != 0.0f ? crow[gn + j] : 0.0f,
                                       epi.bias ? epi.bias[gn + j] : 0.0f);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty[acc]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

int g_smem_attr_set[64];

}  // namespace

size_t tc_smem_bytes() {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + sizeof(TcControl);
}

cudaError_t launch_gemm_bf16_tc(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                float* C, int64_t ldc, int M, int N, int K,
                                bool vec_c, int grid, unsigned int* status,
                                const EpiParams& epi, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = tc_smem_bytes();
  if (dev < 0 || dev >= 64 || !g_smem_attr_set[dev]) {
    e = cudaFuncSetAttribute(gemm_bf16_tc_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_smem_attr_set[dev] = 1;
  }
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  gemm_bf16_tc_kernel<<<grid, THREADS, smem, stream>>>(
      tmA, tmB, C, ldc, M, N, K, tiles_m, tiles_n, vec_c ? 1 : 0, status, epi);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace g07
