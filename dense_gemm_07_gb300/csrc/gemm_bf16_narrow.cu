// gemm_bf16_narrow.cu -- BF16 x BF16 -> FP32 GEMM for narrow N (N <= 128)
// and M > 128; also for wider N when there are few tiles and a long K.
//
// With few columns the product does few FLOPs per byte of A and is bound by
// reading A, as a small-M product is bound by reading B ("How a Matrix
// Multiply Runs on a GPU", "Shapes that run slowly": skinny GEMMs, and
// split-K for too few output tiles; "A06", section 3, "Split-K /
// Stream-K").  The 256 x 256 tiles of the paired kernel would leave at
// least half of every MMA on columns outside C, and give few tiles to
// share out; here every SM streams its own slice of A once instead:
//   * a tile is 128 rows of C by all N columns: D (128 x NN) = A_tile
//     (128 x K, A read K-major as stored) x B (K x NN, B read N-major as
//     stored), NN = 64 or 128 (tcgen05.mma M=128, N=NN; columns of B past
//     N read as zeros).  Wider N is cut into tiles of 128 columns; with at
//     most half as many such tiles as SMs, K still splits over clusters of
//     two or more and every SM streams its own operands, where 256 x 256
//     tiles on SM pairs would leave most pairs idle;
//   * one cluster of CS CTAs per tile splits K into CS contiguous ranges;
//     each CTA runs a TMA -> mbarrier ring -> tcgen05.mma pipeline over its
//     range;
//   * the CTAs park their partial accumulators (128 x NN FP32, rows NN + 4
//     words apart) in their own shared memory, and after a cluster
//     barrier CTA r sums rows r, r + CS, ... over all CS partials in rank
//     order through distributed shared memory, four columns per thread,
//     and writes them to C (consecutive threads, consecutive columns).  The
//     order is fixed, so the results are deterministic; no global workspace
//     is needed.
// Every mbarrier wait is bounded as in the other tensor-core kernels.
#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace g07 {
namespace {

constexpr int TILE_M = kTcTileM;                  // 128: MMA M, rows of C per tile
constexpr int BK = kTcTileK;                      // 64
constexpr int A_STAGE_BYTES = TILE_M * BK * 2;    // 16 KB, K-major rows of 128 B
constexpr int B_BOX_COLS = 64;
constexpr int B_BOX_BYTES = BK * B_BOX_COLS * 2;  // 64 k x 64 columns, 8 KB
constexpr int MMA_K = 16;
constexpr int THREADS = 192;
constexpr int RING_BYTES = 192 * 1024;

template <int NN>
struct NarrowShape {
  static constexpr int B_BOXES = NN / B_BOX_COLS;
  static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_BOXES * B_BOX_BYTES;
  static constexpr int STAGES =
      RING_BYTES / STAGE_BYTES < 8 ? RING_BYTES / STAGE_BYTES : 8;
  static constexpr int TMEM_COLS = NN;
  // Parked rows NN + 4 words apart: 16-byte aligned, and the 8 rows a
  // quarter-warp parks with one 16-byte store each fall in 8 different
  // 4-bank groups; a row stays contiguous for the reduction's remote reads.
  static constexpr int PART_STRIDE = NN + 4;
  static constexpr int PARTIAL_BYTES = TILE_M * PART_STRIDE * 4;
  static_assert(PARTIAL_BYTES <= STAGES * STAGE_BYTES, "partials reuse the ring");
};

template <int STAGES>
struct alignas(8) NarrowControl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(volatile int* abort, unsigned int* status) {
  *abort = 1;
  atomicOr(status, 1u);
}

// Arm stage `stage`'s "full" barrier and copy k-slice kb into it: the
// 128 x 64 box of A's rows, then B's 64-column boxes of that slice.
template <int NN>
__device__ __forceinline__ void issue_stage(uint8_t* smem, uint64_t* full, int stage,
                                            const CUtensorMap* tmA, const CUtensorMap* tmB,
                                            int m0, int n0, int kb) {
  using S = NarrowShape<NN>;
  uint8_t* sa = smem + stage * S::STAGE_BYTES;
  uint8_t* sb = sa + A_STAGE_BYTES;
  mbar_arrive_expect_tx(&full[stage], S::STAGE_BYTES);
  tma_load_2d(sa, tmA, &full[stage], kb * BK, m0);
#pragma unroll
  for (int j = 0; j < S::B_BOXES; ++j)
    tma_load_2d(sb + j * B_BOX_BYTES, tmB, &full[stage], n0 + j * B_BOX_COLS, kb * BK);
}

// GELU: whether the GELU activation is compiled in (epi_apply); the copy
// without it serves every other epilogue.
template <int NN, bool GELU>
__global__ void __launch_bounds__(THREADS, 1)
gemm_bf16_narrow_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, float* __restrict__ C,
                        int64_t ldc, int M, int N, int K, int cs,
                        unsigned int* __restrict__ status, EpiParams epi) {
  using S = NarrowShape<NN>;
  constexpr int STAGES = S::STAGES;
  constexpr uint32_t IDESC =
      idesc_bf16_f32(TILE_M, NN, /*a_mn_major=*/false, /*b_mn_major=*/true);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  auto* ctl = reinterpret_cast<NarrowControl<STAGES>*>(smem + STAGES * S::STAGE_BYTES);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  // tiles in column-major order: consecutive clusters share B's columns
  const int tile = blockIdx.x / cs;
  const int tiles_m = (M + TILE_M - 1) / TILE_M;
  const int m0 = (tile % tiles_m) * TILE_M;
  const int n0 = (tile / tiles_m) * NN;
  const int num_kb_total = (K + BK - 1) / BK;
  const int kb_begin = static_cast<int>(static_cast<int64_t>(num_kb_total) * rank / cs);
  const int kb_end = static_cast<int>(static_cast<int64_t>(num_kb_total) * (rank + 1) / cs);
  const int num_kb = kb_end - kb_begin;
  // Nothing global has been touched yet: wait for the kernels before this
  // one, and let the next one be scheduled as SMs free up.
  grid_dependency_wait();
  grid_dependents_go();
  // Test fault (gemm_debug_inject mode 1): no CTA copies its first stage,
  // so the MMA issuer's wait for it runs out; every role unwinds and the
  // cluster still meets at its final barrier.
  const bool skip_first = status[1] == 1u;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // The ring is empty, so its first stages need no slot to be freed: their
    // copies go out now, while tensor memory is allocated and the block
    // meets (the barriers were initialised by this thread).
    const int pre = num_kb < STAGES ? num_kb : STAGES;
    for (int i = 0; i < pre; ++i)
      if (!(skip_first && i == 0))
        issue_stage<NN>(smem, ctl->full, i, &tmA, &tmB, m0, n0, kb_begin + i);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, S::TMEM_COLS);
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
      // continue after the stages issued before the block barrier
      const int pre = num_kb < STAGES ? num_kb : STAGES;
      int stage = pre % STAGES;
      uint32_t phase = pre == STAGES ? 1u : 0u;
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = s < pre && !(skip_first && s == 0) ? 0 : -1;
      for (int kb = kb_begin + pre; kb < kb_end; ++kb) {
        if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort, tmo)) {
          raise_abort(abort, status);
          break;
        }
        issue_stage<NN>(smem, ctl->full, stage, &tmA, &tmB, m0, n0, kb);
        last_phase[stage] = static_cast<int>(phase);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // every copy issued has landed before the block may leave
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (last_phase[s] >= 0 &&
            !mbar_wait(&ctl->full[s], static_cast<uint32_t>(last_phase[s]), &never, tmo))
          raise_abort(abort, status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(&ctl->full[stage], phase, abort, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(smem + stage * S::STAGE_BYTES);
        const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / MMA_K; ++kk) {
          // A: K-major rows of 128 bytes; a 16-deep k step is 32 bytes in.
          const uint64_t adesc = sdesc_sw128(a_addr + kk * MMA_K * 2, 16, 1024);
          // B: N-major; 64-column boxes 8 KB apart (LBO), 8-row k groups
          // 1 KB apart (SBO); a 16-deep k step is 16 rows = 2 KB in.
          const uint64_t bdesc = sdesc_sw128(b_addr + kk * MMA_K * 128, B_BOX_BYTES, 1024);
          mma_f16_ss(tmem_base, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        mma_commit(&ctl->empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) raise_abort(abort, status);
      // Signals the epilogue (also when this CTA had no k range: the drain
      // of nothing completes at once).
      mma_commit(&ctl->acc_full);
      volatile int never = 0;
      mma_commit(&ctl->drain);
      if (!mbar_wait(&ctl->drain, 0u, &never, tmo)) raise_abort(abort, status);
    }
  } else {
    // ------------------------------------------- epilogue: park the partial
    // TMEM lane = row of the tile; columns 16 at a time.
    const int q = warp & 3;
    const int m_local = q * 32 + lane;
    int ok = 0;
    if (lane == 0) ok = mbar_wait(&ctl->acc_full, 0u, abort, tmo) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) raise_abort(abort, status);
    tc_fence_after_sync();
    float* partial = reinterpret_cast<float*>(smem);
#pragma unroll 1
    for (int c = 0; c < NN / 16; ++c) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 16, r);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(partial + m_local * S::PART_STRIDE + c * 16);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = num_kb > 0 ? make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                          __uint_as_float(r[4 * j + 2]),
                                          __uint_as_float(r[4 * j + 3]))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    tc_fence_before_sync();
  }

  // All partials of the cluster are in place.
  __syncthreads();
  cluster_sync();

  if (warp >= 2) {
    // ---------------------------- reduction in rank order, write C rows
    // 128 threads, 4 columns each: a row takes NN / 4 threads, so 512 / NN
    // rows are summed at a time.
    constexpr int TPR = NN / 4;
    constexpr int PAR = TILE_M / TPR;
    const int t = (warp - 2) * 32 + lane;
    const int n = (t % TPR) * 4;  // column within the tile
    const int gn = n0 + n;        // column of C
    const int sub = t / TPR;
    const uint32_t local = smem_u32(smem);
    const int rows = M - m0 < TILE_M ? M - m0 : TILE_M;
    const bool vec_c = (ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(C) & 15u) == 0;
    // RB rows at a time: all their remote loads are issued before any sum
    // is formed, so their latencies overlap; each sum is then taken in rank
    // order 0, 1, ..., cs-1.
    constexpr int RB = 4;
    const int step = cs * PAR;
    for (int mb = rank + cs * sub; mb < rows; mb += RB * step) {
      float4 v[RB][8];
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const int m = mb + i * step;
        const uint32_t off =
            static_cast<uint32_t>(((m < rows ? m : 0) * S::PART_STRIDE + n) * 4);
#pragma unroll
        for (int qq = 0; qq < 8; ++qq)
          v[i][qq] = qq < cs ? ld_cluster_f32x4(map_to_rank(local + off, static_cast<uint32_t>(qq)))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const int m = mb + i * step;
        if (m >= rows || gn >= N) continue;
        float sum[4] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w};
#pragma unroll
        for (int qq = 1; qq < 8; ++qq)
          if (qq < cs) {
            sum[0] += v[i][qq].x;
            sum[1] += v[i][qq].y;
            sum[2] += v[i][qq].z;
            sum[3] += v[i][qq].w;
          }
        float* crow = C + static_cast<int64_t>(m0 + m) * ldc;
        if (vec_c && gn + 3 < N) {
          float4 old = make_float4(0.f, 0.f, 0.f, 0.f);
          if (epi.beta != 0.0f) old = *reinterpret_cast<const float4*>(crow + gn);
          const float o[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sum[e] = epi_apply<GELU>(epi, sum[e], o[e], epi.bias ? epi.bias[gn + e] : 0.0f);
          *reinterpret_cast<float4*>(crow + gn) = make_float4(sum[0], sum[1], sum[2], sum[3]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (gn + e < N)
              crow[gn + e] = epi_apply<GELU>(epi, sum[e],
                                             epi.beta != 0.0f ? crow[gn + e] : 0.0f,
                                             epi.bias ? epi.bias[gn + e] : 0.0f);
        }
      }
    }
  }

  // No CTA leaves while others may still read its shared memory.
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

std::atomic<int> g_attr_done[64][2];
// Clusters of c CTAs that can be resident at once, per device, column class
// and c (0: not asked yet).
std::atomic<int> g_max_clusters[64][2][9];

template <int NN>
size_t narrow_smem_bytes() {
  using S = NarrowShape<NN>;
  return 1024 + static_cast<size_t>(S::STAGES) * S::STAGE_BYTES + sizeof(NarrowControl<S::STAGES>);
}

template <int NN>
cudaError_t set_attrs_nn(int dev, int slot) {
  if (g_attr_done[dev][slot].load()) return cudaSuccess;
  const size_t smem = narrow_smem_bytes<NN>();
  for (auto k : {gemm_bf16_narrow_kernel<NN, false>, gemm_bf16_narrow_kernel<NN, true>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  g_attr_done[dev][slot].store(1);
  return cudaSuccess;
}

// How many clusters of cs CTAs fit on the device at once (a cluster sits
// within one GPC).  -1: the query failed.
template <int NN>
int max_clusters_nn(int cs, int dev, int slot) {
  const int known = g_max_clusters[dev][slot][cs].load();
  if (known != 0) return known;
  if (set_attrs_nn<NN>(dev, slot) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = narrow_smem_bytes<NN>();
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_narrow_kernel<NN, false>, &cfg) !=
          cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    return -1;
  }
  g_max_clusters[dev][slot][cs].store(n);
  return n;
}

template <int NN>
cudaError_t launch_nn(const CUtensorMap& tmA, const CUtensorMap& tmB, float* C, int64_t ldc,
                      int M, int N, int K, int cs, unsigned int* status, const EpiParams& epi,
                      cudaStream_t stream, int dev, int slot) {
  const size_t smem = narrow_smem_bytes<NN>();
  auto kernel = epi.act == kActGelu ? gemm_bf16_narrow_kernel<NN, true>
                                     : gemm_bf16_narrow_kernel<NN, false>;
  const cudaError_t ea = set_attrs_nn<NN>(dev, slot);
  if (ea != cudaSuccess) return ea;
  const int tiles = ((M + TILE_M - 1) / TILE_M) * ((N + NN - 1) / NN);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * cs), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, C, ldc, M, N, K, cs, status, epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace

int narrow_cols(int N) { return N <= 64 ? 64 : 128; }

int64_t narrow_tiles(int64_t M, int64_t N) {
  const int64_t nn = N <= 64 ? 64 : 128;
  return ((M + TILE_M - 1) / TILE_M) * ((N + nn - 1) / nn);
}

int narrow_split(int M, int N, int K, int sms) {
  const int64_t tiles = narrow_tiles(M, N);
  const int kb = (K + BK - 1) / BK;
  int cs = static_cast<int>(sms / (tiles > 0 ? tiles : 1));
  if (cs > 8) cs = 8;
  if (cs > kb) cs = kb;
  return cs < 1 ? 1 : cs;
}

int narrow_split_resident(int M, int N, int K, int sms) {
  int cs = narrow_split(M, N, K, sms);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return cs;
  }
  const int64_t tiles = narrow_tiles(M, N);
  // The largest split whose clusters all fit at once (a split that does not
  // leaves some clusters for a second round); with more tiles than fit at
  // once, the split is 1 anyway.
  for (; cs > 1; --cs) {
    const int fit = narrow_cols(N) == 64 ? max_clusters_nn<64>(cs, dev, 0)
                                         : max_clusters_nn<128>(cs, dev, 1);
    if (fit < 0 || tiles <= fit) break;
  }
  return cs;
}

cudaError_t launch_gemm_bf16_narrow(const CUtensorMap& tmA, const CUtensorMap& tmB, float* C,
                                    int64_t ldc, int M, int N, int K, int cs,
                                    unsigned int* status, const EpiParams& epi,
                                    cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || cs < 1 || cs > 8 || N < 1 || M < 1 ||
      narrow_tiles(M, N) * cs > 0x7FFFFFFF)
    return cudaErrorInvalidValue;
  return narrow_cols(N) == 64
             ? launch_nn<64>(tmA, tmB, C, ldc, M, N, K, cs, status, epi, stream, dev, 0)
             : launch_nn<128>(tmA, tmB, C, ldc, M, N, K, cs, status, epi, stream, dev, 1);
}

}  // namespace g07
