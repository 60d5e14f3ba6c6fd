// gemm_bf16_skinny.cu -- BF16 x BF16 -> FP32 GEMM for small M (M <= 128).
//
// When M is small the product is close to a matrix-vector product: it does
// few FLOPs per byte of B and is bound by reading B from memory ("How a
// Matrix Multiply Runs on a GPU", "Shapes that run slowly": skinny GEMMs, and
// split-K for too few output tiles; "A06", section 3, "Split-K / Stream-K").
// The aim is therefore to have every SM streaming its own slice of B once.
//
// sm_103a realisation:
//   * operand roles are swapped so the long dimension N fills the 128 lanes
//     of the MMA: D^T (128 x NM) = B_tile^T (128 x K, B read N-major as
//     stored) x A^T (K x NM, A read K-major as stored), NM = M rounded up to
//     16, 32, 64 or 128 (tcgen05.mma M=128, N=NM);
//   * one cluster of CS CTAs per 128-column tile of C splits K into CS
//     contiguous ranges (split-K); each CTA runs a TMA -> mbarrier ring ->
//     tcgen05.mma pipeline over its range;
//   * the CTAs park their partial accumulators (NM x 128 FP32) in their own
//     shared memory, and after a cluster barrier CTA r sums rows
//     m = r, r + CS, ... over all CS partials in rank order through
//     distributed shared memory and writes them to C (consecutive threads,
//     consecutive columns).  The sum order is fixed, so results are
//     deterministic; no global workspace and no second kernel are needed.
// Every mbarrier wait is bounded as in the other tensor-core kernels.
#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace g07 {
namespace {

constexpr int TILE_N = 128;                       // MMA M: columns of C per tile
constexpr int BK = 64;
constexpr int B_BOX_BYTES = BK * 64 * 2;           // 64 columns x 64 k, 8 KB
constexpr int B_STAGE_BYTES = 2 * B_BOX_BYTES;     // 128 columns, 16 KB
constexpr int MMA_K = 16;
constexpr int THREADS = 192;
constexpr int RING_BYTES = 192 * 1024;

template <int NM>
struct SkinnyShape {
  static constexpr int A_STAGE_BYTES = NM * BK * 2;  // NM rows x 128 B
  static constexpr int STAGE_BYTES = B_STAGE_BYTES + A_STAGE_BYTES;
  static constexpr int STAGES =
      RING_BYTES / STAGE_BYTES < 8 ? RING_BYTES / STAGE_BYTES : 8;
  static constexpr int TMEM_COLS = NM < 32 ? 32 : NM;
  static constexpr int PARTIAL_BYTES = NM * TILE_N * 4;
  static_assert(PARTIAL_BYTES <= STAGES * STAGE_BYTES, "partials reuse the ring");
};

template <int STAGES>
struct alignas(8) SkinnyControl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(volatile int* abort,
                                            unsigned int* status) {
  *abort = 1;
  atomicOr(status, 1u);
}

// Arm stage `stage`'s "full" barrier and copy k-slice kb into it: the two
// 64-column boxes of B's 128-column tile and the NM x 64 box of A.
template <int NM>
__device__ __forceinline__ void issue_stage(uint8_t* smem, uint64_t* full, int stage,
                                            const CUtensorMap* tmA, const CUtensorMap* tmB,
                                            int n0, int kb) {
  using S = SkinnyShape<NM>;
  uint8_t* sb = smem + stage * S::STAGE_BYTES;
  uint8_t* sa = sb + B_STAGE_BYTES;
  mbar_arrive_expect_tx(&full[stage], S::STAGE_BYTES);
  tma_load_2d(sb, tmB, &full[stage], n0, kb * BK);
  tma_load_2d(sb + B_BOX_BYTES, tmB, &full[stage], n0 + 64, kb * BK);
  tma_load_2d(sa, tmA, &full[stage], kb * BK, 0);
}

// GELU: whether the GELU activation is compiled in (epi_apply); the copy
// without it serves every other epilogue.
template <int NM, bool GELU>
__global__ void __launch_bounds__(THREADS, 1)
gemm_bf16_skinny_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        float* __restrict__ C, int64_t ldc, int M, int N,
                        int K, int cs, unsigned int* __restrict__ status,
                        EpiParams epi) {
  using S = SkinnyShape<NM>;
  constexpr int STAGES = S::STAGES;
  constexpr uint32_t IDESC =
      idesc_bf16_f32(TILE_N, NM, /*a_mn_major=*/true, /*b_mn_major=*/false);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  auto* ctl = reinterpret_cast<SkinnyControl<STAGES>*>(smem + STAGES * S::STAGE_BYTES);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int tile = blockIdx.x / cs;
  const int n0 = tile * TILE_N;
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
        issue_stage<NM>(smem, ctl->full, i, &tmA, &tmB, n0, kb_begin + i);
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
        issue_stage<NM>(smem, ctl->full, stage, &tmA, &tmB, n0, kb);
        last_phase[stage] = static_cast<int>(phase);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
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
        const uint32_t b_addr = smem_u32(smem + stage * S::STAGE_BYTES);
        const uint32_t a_addr = b_addr + B_STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / MMA_K; ++kk) {
          // MMA A operand = 128 columns of B, N-major: 64-column boxes 8 KB
          // apart (LBO), 8-row k groups 1 KB apart (SBO), k step 2 KB.
          const uint64_t bdesc =
              sdesc_sw128(b_addr + kk * MMA_K * 128, B_BOX_BYTES, 1024);
          // MMA B operand = NM rows of A, K-major: k step of 32 bytes.
          const uint64_t adesc = sdesc_sw128(a_addr + kk * MMA_K * 2, 16, 1024);
          mma_f16_ss(tmem_base, bdesc, adesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
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
    const int q = warp & 3;
    const int n_local = q * 32 + lane;  // TMEM lane = column of the tile
    int ok = 0;
    if (lane == 0) ok = mbar_wait(&ctl->acc_full, 0u, abort, tmo) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) raise_abort(abort, status);
    tc_fence_after_sync();
    float* partial = reinterpret_cast<float*>(smem);  // [NM][TILE_N]
#pragma unroll 1
    for (int c = 0; c < NM / 16; ++c) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 16, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        partial[(c * 16 + j) * TILE_N + n_local] =
            num_kb > 0 ? __uint_as_float(r[j]) : 0.0f;
    }
    tc_fence_before_sync();
  }

  // All partials of the cluster are in place.
  __syncthreads();
  cluster_sync();

  if (warp >= 2) {
    // ---------------------------- reduction in rank order, write C rows
    const int n_local = (warp - 2) * 32 + lane;
    const int n = n0 + n_local;
    const uint32_t local = smem_u32(smem);
    const int rows = M < NM ? M : NM;
    // Four rows at a time: all their remote loads are issued before any sum
    // is formed, so their latencies overlap; each sum is then taken in rank
    // order 0, 1, ..., cs-1.
    constexpr int RB = 4;
    for (int m0 = rank; m0 < rows; m0 += RB * cs) {
      float v[RB][8];
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const int m = m0 + i * cs;
        const uint32_t off = static_cast<uint32_t>(((m < rows ? m : 0) * TILE_N + n_local) * 4);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[i][q] = q < cs ? ld_cluster_f32(map_to_rank(local + off, static_cast<uint32_t>(q)))
                           : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const int m = m0 + i * cs;
        float sum = v[i][0];
#pragma unroll
        for (int q = 1; q < 8; ++q)
          if (q < cs) sum += v[i][q];
        if (m < rows && n < N) {
          float* p = C + static_cast<int64_t>(m) * ldc + n;
          *p = epi_apply<GELU>(epi, sum, epi.beta != 0.0f ? *p : 0.0f,
                         epi.bias ? epi.bias[n] : 0.0f);
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

std::atomic<int> g_attr_done[64][4];
// Clusters of c CTAs that can be resident at once, per device, row class
// and c (0: not asked yet).
std::atomic<int> g_max_clusters[64][4][9];

template <int NM>
size_t skinny_smem_bytes() {
  using S = SkinnyShape<NM>;
  return 1024 + static_cast<size_t>(S::STAGES) * S::STAGE_BYTES + sizeof(SkinnyControl<S::STAGES>);
}

template <int NM>
cudaError_t set_attrs_nm(int dev, int slot) {
  if (g_attr_done[dev][slot].load()) return cudaSuccess;
  const size_t smem = skinny_smem_bytes<NM>();
  for (auto k : {gemm_bf16_skinny_kernel<NM, false>, gemm_bf16_skinny_kernel<NM, true>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  g_attr_done[dev][slot].store(1);
  return cudaSuccess;
}

// How many clusters of cs CTAs fit on the device at once.  A cluster must
// sit within one GPC, so this can be less than the SM count / cs (clusters
// of 4 reach only 144 of a GB300's 152 SMs).  -1: the query failed.
template <int NM>
int max_clusters_nm(int cs, int dev, int slot) {
  const int known = g_max_clusters[dev][slot][cs].load();
  if (known != 0) return known;
  if (set_attrs_nm<NM>(dev, slot) != cudaSuccess) {
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
  cfg.dynamicSmemBytes = skinny_smem_bytes<NM>();
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_skinny_kernel<NM, false>, &cfg) !=
          cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    return -1;
  }
  g_max_clusters[dev][slot][cs].store(n);
  return n;
}

template <int NM>
cudaError_t launch_nm(const CUtensorMap& tmA, const CUtensorMap& tmB, float* C,
                      int64_t ldc, int M, int N, int K, int cs,
                      unsigned int* status, const EpiParams& epi,
                      cudaStream_t stream, int dev, int slot) {
  const size_t smem = skinny_smem_bytes<NM>();
  auto kernel = epi.act == kActGelu ? gemm_bf16_skinny_kernel<NM, true>
                                     : gemm_bf16_skinny_kernel<NM, false>;
  const cudaError_t ea = set_attrs_nm<NM>(dev, slot);
  if (ea != cudaSuccess) return ea;
  const int tiles = (N + TILE_N - 1) / TILE_N;
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, C, ldc, M, N, K, cs,
                                           status, epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace

int skinny_rows(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

int skinny_split(int N, int K, int sms) {
  const int tiles = (N + TILE_N - 1) / TILE_N;
  const int kb = (K + BK - 1) / BK;
  int cs = sms / (tiles > 0 ? tiles : 1);
  if (cs > 8) cs = 8;
  if (cs > kb) cs = kb;
  return cs < 1 ? 1 : cs;
}

int skinny_split_resident(int M, int N, int K, int sms) {
  int cs = skinny_split(N, K, sms);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return cs;
  }
  const int tiles = (N + TILE_N - 1) / TILE_N;
  // The largest split whose clusters all fit at once: one that does not
  // leaves some clusters for a second round, about doubling the time
  // (16 x 4864 x 4096 in clusters of 4: 24.1 us against 17.2 us for
  // N = 4096).
  for (; cs > 1; --cs) {
    int fit = 0;
    switch (skinny_rows(M)) {
      case 16: fit = max_clusters_nm<16>(cs, dev, 0); break;
      case 32: fit = max_clusters_nm<32>(cs, dev, 1); break;
      case 64: fit = max_clusters_nm<64>(cs, dev, 2); break;
      default: fit = max_clusters_nm<128>(cs, dev, 3); break;
    }
    if (fit < 0 || tiles <= fit) break;
  }
  return cs;
}

cudaError_t launch_gemm_bf16_skinny(const CUtensorMap& tmA,
                                    const CUtensorMap& tmB, float* C,
                                    int64_t ldc, int M, int N, int K, int cs,
                                    unsigned int* status, const EpiParams& epi,
                                    cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  switch (skinny_rows(M)) {
    case 16:
      return launch_nm<16>(tmA, tmB, C, ldc, M, N, K, cs, status, epi, stream, dev, 0);
    case 32:
      return launch_nm<32>(tmA, tmB, C, ldc, M, N, K, cs, status, epi, stream, dev, 1);
    case 64:
      return launch_nm<64>(tmA, tmB, C, ldc, M, N, K, cs, status, epi, stream, dev, 2);
    default:
      return launch_nm<128>(tmA, tmB, C, ldc, M, N, K, cs, status, epi, stream, dev, 3);
  }
}

}  // namespace g07
