// gemm_bf16_tc2.cu -- BF16 x BF16 -> FP32 GEMM on pairs of SMs.
//
// Same method as gemm_bf16_tc.cu (the tensor-core rung of "GEMM, step by
// step", section "Concept": BF16 inputs, FP32 sums, large tiles, neighbouring
// blocks on the same rows/columns; multi-stage prefetch as in "GEMM
// Optimization", section 5), with the output tile grown to 256 x 256 and
// computed by two SMs together ("Production tensor-core kernels use larger
// tiles", same section of "GEMM, step by step").
//
// Wave tail: when the tiles left for the last wave fill at most half of the
// resident pairs, each of them is computed as two 256 x 128 units (an N=128
// pair MMA, one 64-column box of B per CTA), so that wave takes half as long.
// Every output element is still one tile's k-sum in one accumulator.
//
// sm_103a realisation: clusters of two CTAs, one per SM.  CTA r of the pair
// owns rows [128r, 128r+128) of the 256-row tile and stages only those rows
// of A (128 x 64 per k-slice) plus columns [128r, 128r+128) of B (64 x 128);
// one tcgen05.mma.cta_group::2 (M=256, N=256, K=16), issued by the even CTA,
// reads A and B from both CTAs' shared memory and writes each CTA's 128 rows
// of D into that CTA's tensor memory.  Per SM this halves the bytes that
// have to be copied into shared memory per FLOP compared with one SM
// computing a 128 x 256 tile, which is what lets six 32 KB stages keep the
// tensor core busy.
//
// Roles (192 threads per CTA):
//   warp 0 (both CTAs)  TMA producer.  Both CTAs' copies count their bytes on
//                       the even CTA's "full" barrier; the even CTA arms it
//                       for 64 KB per stage.
//   warp 1 (even CTA)   MMA issuer: waits on "full", issues 4 pair MMAs per
//                       stage, commits to "empty" in both CTAs, and after the
//                       last slice of a tile to "accumulator full" in both.
//   warps 2-5 (both)    epilogue: TMEM -> registers -> swizzled shared
//                       staging box -> TMA tensor store of C (whole lines;
//                       rows/columns outside C are clipped), or guarded
//                       direct stores when C's layout does not allow TMA;
//                       then arrive on the even CTA's "accumulator empty"
//                       (8 arrivals per tile).
// Tensor memory: NUM_ACC 256-column FP32 accumulators per CTA; with two, a
// tile's epilogue overlaps the next tile's MMAs.  Every wait is bounded; on expiry
// the CTA raises its own and its peer's abort flag and the status word, all
// roles unwind, copies and MMAs in flight are drained, and both CTAs meet at
// a final cluster barrier before tensor memory is released.
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tile_order.cuh"

namespace g07 {
namespace {

constexpr int PAIR_M = 256;                       // rows per pair tile
constexpr int CTA_M = 128;                        // rows per CTA
constexpr int BN = 256;                           // columns per pair tile
constexpr int CTA_N = 128;                        // B columns staged per CTA
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_STAGE_BYTES = CTA_M * BK * 2;     // 16 KB
constexpr int B_BOX_COLS = 64;
constexpr int B_BOX_BYTES = BK * B_BOX_COLS * 2;  // 8 KB
constexpr int B_STAGE_BYTES = BK * CTA_N * 2;     // 16 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int MMA_K = 16;
constexpr int NUM_ACC = 2;                        // accumulators in TMEM
constexpr int TMEM_COLS = NUM_ACC * BN;
constexpr int THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BOX_BYTES = 32 * 32 * 4;            // one 32 x 32 FP32 box
constexpr int EPI_BYTES = EPI_WARPS * 2 * EPI_BOX_BYTES;  // double-buffered
constexpr int GROUP = 8;

struct alignas(8) PairControl {
  uint64_t full[STAGES];      // used in the even CTA only
  uint64_t empty[STAGES];
  uint64_t acc_full[NUM_ACC];
  uint64_t acc_empty[NUM_ACC];  // used in the even CTA only (8 arrivals)
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// One unit of work: a 256-row tile of C, columns [n0, n0 + width).
struct Unit {
  int m0;
  int n0;
  int width;
};

__device__ __forceinline__ Unit unit_of(int unit, int num_full, int split,
                                        int tiles_m, int tiles_n) {
  int tile = unit, piece = 0, width = BN;
  if (unit >= num_full) {
    tile = num_full + (unit - num_full) / split;
    piece = (unit - num_full) % split;
    width = BN / split;
  }
  const TileCoord tc = tile_order(tile, tiles_m, tiles_n, GROUP);
  Unit u;
  u.m0 = tc.m * PAIR_M;
  u.n0 = tc.n * BN + piece * width;
  u.width = width;
  return u;
}

__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort, uint64_t tmo) {
  return mbar_wait(bar, parity, abort, tmo);
}

__device__ __forceinline__ void raise_abort(volatile int* abort,
                                            uint32_t peer_abort_addr,
                                            unsigned int* status) {
  *abort = 1;
  st_cluster_u32(peer_abort_addr, 1u);
  atomicOr(status, 1u);
}

// Position in the shared-memory ring (stage, and the parity of its uses).
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance() {
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// Producer for one unit of width W: per k-slice, wait for the stage to be
// free, arm the even CTA's "full" barrier (even CTA only), copy this CTA's
// 128 rows of A and W/2 columns of B.
template <int W>
__device__ __forceinline__ bool produce_unit(const Unit& u, Ring& ring,
                                             int num_kb, uint8_t* smem,
                                             PairControl* ctl,
                                             const CUtensorMap* tmA,
                                             const CUtensorMap* tmB,
                                             uint32_t rank, int* last_phase,
                                             volatile int* abort, uint64_t tmo,
                                             bool skip_first) {
  constexpr int BOXES = W / 2 / B_BOX_COLS;
  constexpr uint32_t TX = 2u * (A_STAGE_BYTES + BOXES * B_BOX_BYTES);
  const int a_row = u.m0 + static_cast<int>(rank) * CTA_M;
  const int b_col = u.n0 + static_cast<int>(rank) * (W / 2);
  for (int kb = 0; kb < num_kb; ++kb) {
    if (!mbar_wait(&ctl->empty[ring.stage], ring.phase ^ 1u, abort, tmo)) return false;
    if (skip_first && kb == 0) {
      // Test fault: this k-slice is never copied, so the MMA's wait for it
      // runs out and the kernel unwinds with a timeout status.
      ring.advance();
      continue;
    }
    if (rank == 0) {
      mbar_arrive_expect_tx(&ctl->full[ring.stage], TX);
      last_phase[ring.stage] = static_cast<int>(ring.phase);
    }
    const uint32_t full0 = map_to_rank(smem_u32(&ctl->full[ring.stage]), 0);
    uint8_t* sa = smem + ring.stage * STAGE_BYTES;
    uint8_t* sb = sa + A_STAGE_BYTES;
    tma_load_2d_pair(sa, tmA, full0, kb * BK, a_row);
#pragma unroll
    for (int j = 0; j < BOXES; ++j)
      tma_load_2d_pair(sb + j * B_BOX_BYTES, tmB, full0, b_col + j * B_BOX_COLS,
                       kb * BK);
    ring.advance();
  }
  return true;
}

// MMA issue for one unit of width W into the accumulator at d_tmem.
template <int W>
__device__ __forceinline__ bool mma_unit(uint32_t d_tmem, Ring& ring,
                                         int num_kb, uint8_t* smem,
                                         PairControl* ctl,
                                         volatile int* abort, uint64_t tmo) {
  constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_M, W, /*a_mn_major=*/false,
                                            /*b_mn_major=*/true);
  for (int kb = 0; kb < num_kb; ++kb) {
    if (!mbar_wait(&ctl->full[ring.stage], ring.phase, abort, tmo)) return false;
    tc_fence_after_sync();
    const uint32_t a_addr = smem_u32(smem + ring.stage * STAGE_BYTES);
    const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / MMA_K; ++kk) {
      // A: K-major rows of 128 bytes; a 16-deep k step is 32 bytes in.
      const uint64_t adesc = sdesc_sw128(a_addr + kk * MMA_K * 2, 16, 1024);
      // B: N-major; 64-column boxes 8 KB apart (LBO), 8-row k groups 1 KB
      // apart (SBO); a 16-deep k step is 16 rows = 2 KB in.
      const uint64_t bdesc =
          sdesc_sw128(b_addr + kk * MMA_K * 128, B_BOX_BYTES, 1024);
      mma_f16_ss_pair(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
    }
    mma_commit_pair(&ctl->empty[ring.stage], 0x3);
    ring.advance();
  }
  return true;
}

// Epilogue of one unit: this thread's row, W columns from TMEM to C.
template <int W>
__device__ __forceinline__ void store_unit(uint32_t taddr, float* C,
                                           int64_t ldc, int row, int n0, int M,
                                           int N, int vec_c,
                                           const EpiParams& epi) {
  float* crow = C + static_cast<int64_t>(row) * ldc;
#pragma unroll 1
  for (int c = 0; c < W / 32; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    tmem_ld_wait();
    const int gn = n0 + c * 32;
    if (row < M) {
      if (vec_c && gn + 31 < N) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 old = make_float4(0.f, 0.f, 0.f, 0.f);
          if (epi.beta != 0.0f) old = *reinterpret_cast<const float4*>(crow + gn + j);
          const float o[4] = {old.x, old.y, old.z, old.w};
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[e] = epi_apply(epi, __uint_as_float(r[j + e]), o[e],
                             epi.bias ? epi.bias[gn + j + e] : 0.0f);
          *reinterpret_cast<float4*>(crow + gn + j) = make_float4(v[0], v[1], v[2], v[3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (gn + j < N)
            crow[gn + j] = epi_apply(epi, __uint_as_float(r[j]),
                                     epi.beta != 0.0f ? crow[gn + j] : 0.0f,
                                     epi.bias ? epi.bias[gn + j] : 0.0f);
      }
    }
  }
}

// Epilogue of one unit through shared memory and TMA stores: per 32-column
// chunk the warp writes its 32 x 32 block into a 128-byte-swizzled staging
// box (each lane one row, conflict-free 16-byte stores) and one lane stores
// the box with the copy engine, which writes whole lines and clips rows and
// columns outside C.  Two staging boxes per warp alternate.
template <int W>
__device__ __forceinline__ void store_unit_tma(uint32_t taddr,
                                               const CUtensorMap* tmC,
                                               uint8_t* ebuf, int row0, int n0,
                                               int M, int N, int lane,
                                               int& chunk, const float* C,
                                               int64_t ldc,
                                               const EpiParams& epi) {
#pragma unroll 1
  for (int c = 0; c < W / 32; ++c) {
    // Boxes wholly outside C are skipped (warp-uniform test); every other
    // chunk issues exactly one store group, which the buffer alternation
    // below relies on.
    if (row0 >= M || n0 + c * 32 >= N) continue;
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    uint8_t* buf = ebuf + (chunk++ & 1) * EPI_BOX_BYTES;
    if (lane == 0) bulk_wait_read<1>();  // the box's previous store has read it
    __syncwarp();
    tmem_ld_wait();
    if (epi.alpha != 1.0f || epi.beta != 0.0f || epi.bias != nullptr || epi.act != 0) {
      // Fused epilogue on this lane's row (N % 4 == 0 on this path, so each
      // 16-byte group is wholly inside or outside C).
      const int row = row0 + lane;
      const int gn = n0 + c * 32;
      const float* crow = C + static_cast<int64_t>(row) * ldc;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float4 old = make_float4(0.f, 0.f, 0.f, 0.f);
        if (epi.beta != 0.0f && row < M && gn + j < N)
          old = *reinterpret_cast<const float4*>(crow + gn + j);
        const float o[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool in = gn + j + e < N;
          r[j + e] = __float_as_uint(epi_apply(
              epi, __uint_as_float(r[j + e]), o[e],
              (epi.bias != nullptr && in) ? epi.bias[gn + j + e] : 0.0f));
        }
      }
    }
    uint8_t* rowp = buf + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
          make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    // partial boxes are clipped by the copy engine
    if (lane == 0) {
      tma_store_2d(tmC, buf, n0 + c * 32, row0);
      bulk_commit();
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC,
                      float* __restrict__ C, int64_t ldc, int M, int N, int K,
                      int tiles_m, int tiles_n, int num_full, int split,
                      int vec_c, int tma_c, unsigned int* __restrict__ status,
                      EpiParams epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* epi_smem = smem + STAGES * STAGE_BYTES;
  PairControl* ctl =
      reinterpret_cast<PairControl*>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int num_tiles = tiles_m * tiles_n;
  // Work units: tiles [0, num_full) at full width, then every remaining tile
  // as `split` column pieces of BN / split (the last, partial wave).
  const int num_units = num_full + (num_tiles - num_full) * split;
  const int num_kb = (K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < NUM_ACC; ++a) {
      mbar_init(&ctl->acc_full[a], 1);
      mbar_init(&ctl->acc_empty[a], 8);  // 4 epilogue warps x 2 CTAs
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl->tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after_sync();
  const uint32_t tmem_base = ctl->tmem_base;
  const uint64_t tmo = wait_limit_ns(status);
  const unsigned int fault = status[1];
  const uint32_t peer_abort = map_to_rank(smem_u32(&ctl->abort), rank ^ 1u);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring ring;
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = -1;
      bool ok = true;
      for (int unit = pair; ok && unit < num_units; unit += num_pairs) {
        const Unit u = unit_of(unit, num_full, split, tiles_m, tiles_n);
        const bool skip = fault == 1 && unit == pair;
        ok = u.width == BN
                 ? produce_unit<BN>(u, ring, num_kb, smem, ctl, &tmA, &tmB, rank,
                                    last_phase, abort, tmo, skip)
                 : produce_unit<BN / 2>(u, ring, num_kb, smem, ctl, &tmA, &tmB,
                                        rank, last_phase, abort, tmo, skip);
      }
      if (!ok) raise_abort(abort, peer_abort, status);
      // The even CTA's "full" barriers count both CTAs' copies: every phase
      // it armed must complete before the pair may exit.
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (last_phase[s] >= 0 &&
            !mbar_wait(&ctl->full[s], static_cast<uint32_t>(last_phase[s]),
                       &never, tmo))
          raise_abort(abort, peer_abort, status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (even && lane == 0) {
      Ring ring;
      bool ok = true;
      bool issued = false;
      int t = 0;
      for (int unit = pair; ok && unit < num_units; unit += num_pairs, ++t) {
        const Unit u = unit_of(unit, num_full, split, tiles_m, tiles_n);
        const int acc = t % NUM_ACC;
        const uint32_t acc_phase = static_cast<uint32_t>(t / NUM_ACC) & 1u;
        if (!pair_wait(&ctl->acc_empty[acc], acc_phase ^ 1u, abort, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        issued |= num_kb > 0;
        ok = u.width == BN ? mma_unit<BN>(d_tmem, ring, num_kb, smem, ctl, abort, tmo)
                           : mma_unit<BN / 2>(d_tmem, ring, num_kb, smem, ctl, abort, tmo);
        if (!ok) break;
        mma_commit_pair(&ctl->acc_full[acc], 0x3);
      }
      if (!ok) raise_abort(abort, peer_abort, status);
      if (issued) {
        mma_commit_pair(&ctl->drain, 0x1);
        volatile int never = 0;
        if (!mbar_wait(&ctl->drain, 0u, &never, tmo))
          raise_abort(abort, peer_abort, status);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    uint8_t* ebuf = epi_smem + (warp - 2) * 2 * EPI_BOX_BYTES;
    int chunk = 0;
    int t = 0;
    for (int unit = pair; unit < num_units; unit += num_pairs, ++t) {
      const int acc = t % NUM_ACC;
      const uint32_t acc_phase = static_cast<uint32_t>(t / NUM_ACC) & 1u;
      int ok = 0;
      if (lane == 0) ok = pair_wait(&ctl->acc_full[acc], acc_phase, abort, tmo) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) raise_abort(abort, peer_abort, status);
        break;
      }
      tc_fence_after_sync();
      const Unit u = unit_of(unit, num_full, split, tiles_m, tiles_n);
      const int row = u.m0 + static_cast<int>(rank) * CTA_M + q * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int row0 = row - lane;
      if (tma_c) {
        if (u.width == BN)
          store_unit_tma<BN>(taddr, &tmC, ebuf, row0, u.n0, M, N, lane, chunk,
                             C, ldc, epi);
        else
          store_unit_tma<BN / 2>(taddr, &tmC, ebuf, row0, u.n0, M, N, lane,
                                 chunk, C, ldc, epi);
      } else if (u.width == BN) {
        store_unit<BN>(taddr, C, ldc, row, u.n0, M, N, vec_c, epi);
      } else {
        store_unit<BN / 2>(taddr, C, ldc, row, u.n0, M, N, vec_c, epi);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0)
        mbar_arrive_cluster(map_to_rank(smem_u32(&ctl->acc_empty[acc]), 0));
    }
    // Every store issued must have completed before the CTA exits.
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

struct LaunchInfo {
  int ready = 0;
  int max_pairs = 0;
};
LaunchInfo g_info[64];

}  // namespace

size_t pair_smem_bytes() {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + EPI_BYTES +
         sizeof(PairControl);
}

int pair_max_active(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  LaunchInfo& li = g_info[dev];
  if (!li.ready) {
    const size_t smem = pair_smem_bytes();
    if (cudaFuncSetAttribute(gemm_bf16_pair_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_bf16_pair_kernel, &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    li.max_pairs = clusters;
    li.ready = 1;
  }
  return li.max_pairs;
}

cudaError_t launch_gemm_bf16_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const CUtensorMap* tmC, float* C, int64_t ldc,
                                  int M, int N, int K, bool vec_c, int max_pairs,
                                  unsigned int* status, const EpiParams& epi,
                                  cudaStream_t stream) {
  const int tiles_m = (M + PAIR_M - 1) / PAIR_M;
  const int tiles_n = (N + BN - 1) / BN;
  const int tiles = tiles_m * tiles_n;
  // A last wave that fills at most half of the pairs runs as half-width
  // units instead, so it takes half as long.
  const int tail = tiles % max_pairs;
  const int split = (tail > 0 && 2 * tail <= max_pairs) ? 2 : 1;
  const int num_full = split == 2 ? tiles - tail : tiles;
  const int units = num_full + (tiles - num_full) * split;
  const int pairs = units < max_pairs ? units : max_pairs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes();
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  CUtensorMap unused;
  if (tmC == nullptr) std::memset(&unused, 0, sizeof(unused));
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, gemm_bf16_pair_kernel, tmA, tmB, tmC ? *tmC : unused, C, ldc, M, N,
      K, tiles_m, tiles_n, num_full, split, vec_c ? 1 : 0, tmC ? 1 : 0, status,
      epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace g07
