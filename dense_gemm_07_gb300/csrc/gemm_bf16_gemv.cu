// gemm_bf16_gemv.cu -- BF16 x BF16 -> FP32 product for M = 1: one row of A
// (a vector x) times B.
//
// With a single row of A the product does 2 FLOPs per 2-byte element of B:
// it is bound by reading B from memory, not by arithmetic ("How a Matrix
// Multiply Runs on a GPU", section "Shapes that run slowly, and why": skinny
// products are memory-bound; "A06 -- Tiled Matrix Multiply (GEMM)", section
// "2. First Principles": intensity against the ridge point).  Tensor cores
// would do nothing useful here, so the kernel streams B through shared
// memory and multiplies on the CUDA cores:
//   * columns of C are cut into blocks of 1024 (2 KB of every row of B) and
//     the rows of B into KS contiguous ranges, one block of 288 threads per
//     (column block, range), about one per SM;
//   * a producer warp copies its range into a ring of shared-memory stages
//     with TMA, 16 rows x 1024 columns of B (four 256-column boxes, 2 KB of
//     each row contiguous, so DRAM reads whole row segments) plus the 16
//     matching elements of x per stage;
//   * 8 consumer warps each own 4 columns per thread and add x[k] * B[k][n]
//     in FP32, k increasing (BF16 products are exact in FP32);
//   * with KS > 1 each range publishes its 1024 sums to a workspace and
//     counts itself in; the launch is cooperative (all blocks resident), so
//     each range then waits, bounded, for the other ranges of its column
//     block and finishes its own 1/KS slice of the columns: it adds that
//     slice of every range's sums in range order 0, 1, ..., applies the
//     output step and writes C.  The order is fixed, so the result does not
//     depend on timing, and the final additions are spread over all KS SMs
//     instead of one SM reading every range's sums.
// Every mbarrier wait is bounded as in the tensor-core kernels.
#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace g07 {
namespace {

constexpr int COLS = kGemvCols;                       // columns of C per block
constexpr int BOX_COLS = 256;                         // columns per TMA box
constexpr int ROWS = kGemvRows;                       // rows of B per stage
constexpr int STAGES = kGemvStages;
constexpr int B_BOX_BYTES = ROWS * BOX_COLS * 2;      // 8 KB
constexpr int B_STAGE_BYTES = (COLS / BOX_COLS) * B_BOX_BYTES;  // 32 KB
constexpr int X_BYTES = ROWS * 2;                     // x[k .. k + 15]
constexpr int STAGE_STRIDE = B_STAGE_BYTES + 128;
constexpr int CONSUMERS = COLS / 4;                   // 4 columns per thread
constexpr int THREADS = CONSUMERS + 32;               // + one producer warp
static_assert(COLS % BOX_COLS == 0 && BOX_COLS % 4 == 0, "column blocking");

struct alignas(8) GemvControl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  int abort;
};

__device__ __forceinline__ void raise_abort(volatile int* abort, unsigned int* status) {
  *abort = 1;
  atomicOr(status, 1u);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Arm stage `stage` and copy rows [k, k + ROWS) of the block's 1024 columns
// of B, and x[k, k + ROWS), into it.  Out-of-range rows and columns read 0.
__device__ __forceinline__ void issue_stage(uint8_t* smem, uint64_t* full, int stage,
                                            const CUtensorMap* tmA, const CUtensorMap* tmB,
                                            int n0, int k) {
  uint8_t* st = smem + stage * STAGE_STRIDE;
  mbar_arrive_expect_tx(&full[stage], B_STAGE_BYTES + X_BYTES);
#pragma unroll
  for (int j = 0; j < COLS / BOX_COLS; ++j)
    tma_load_2d(st + j * B_BOX_BYTES, tmB, &full[stage], n0 + j * BOX_COLS, k);
  tma_load_2d(st + B_STAGE_BYTES, tmA, &full[stage], k, 0);
}

// C[0][n .. n + 3] := epilogue of the four sums (n may run past N).
template <bool GELU>
__device__ __forceinline__ void store_out(float* C, int n, int N, const float (&v)[4],
                                          const EpiParams& epi) {
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (n + e < N)
      C[n + e] = epi_apply<GELU>(epi, v[e], epi.beta != 0.0f ? C[n + e] : 0.0f,
                                 epi.bias ? epi.bias[n + e] : 0.0f);
}

// GELU: whether the GELU activation is compiled in (epi_apply); the copy
// without it serves every other epilogue.
template <bool GELU>
__global__ void __launch_bounds__(THREADS, 1)
gemm_bf16_gemv_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, float* __restrict__ C,
                      int N, int K, int ranges, float* __restrict__ ws,
                      unsigned int* __restrict__ counters, unsigned int* __restrict__ status,
                      EpiParams epi) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  auto* ctl = reinterpret_cast<GemvControl*>(smem + STAGES * STAGE_STRIDE);
  volatile int* abort = &ctl->abort;

  // nothing global is touched before this: wait for the kernels before this
  // one, and let the next one be scheduled as SMs free up
  grid_dependency_wait();
  grid_dependents_go();
  const int tid = threadIdx.x;
  const int nb = blockIdx.x / ranges;
  const int rg = blockIdx.x % ranges;
  const int n0 = nb * COLS;
  const int groups = (K + ROWS - 1) / ROWS;
  const int g_begin = static_cast<int>(static_cast<int64_t>(groups) * rg / ranges);
  const int g_end = static_cast<int>(static_cast<int64_t>(groups) * (rg + 1) / ranges);
  const int num_g = g_end - g_begin;
  const int pre = num_g < STAGES ? num_g : STAGES;
  // Test fault (gemm_debug_inject mode 1): the first stage is never copied,
  // so the consumers' wait for it runs out and the block unwinds.
  const bool skip_first = status[1] == 1u;

  if (tid == CONSUMERS) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], CONSUMERS / 32);
    }
    ctl->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // The ring is empty: its first stages go out at once.
    for (int i = 0; i < pre; ++i)
      if (!(skip_first && i == 0))
        issue_stage(smem, ctl->full, i, &tmA, &tmB, n0, (g_begin + i) * ROWS);
  }
  __syncthreads();
  const uint64_t tmo = wait_limit_ns(status);

  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (tid >= CONSUMERS) {
    // ------------------------------------------------------------ producer
    if (tid == CONSUMERS) {
      int stage = pre % STAGES;
      uint32_t phase = pre == STAGES ? 1u : 0u;
      int last_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) last_phase[s] = s < pre && !(skip_first && s == 0) ? 0 : -1;
      for (int g = pre; g < num_g; ++g) {
        if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort, tmo)) {
          raise_abort(abort, status);
          break;
        }
        issue_stage(smem, ctl->full, stage, &tmA, &tmB, n0, (g_begin + g) * ROWS);
        last_phase[stage] = static_cast<int>(phase);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // No copy may still be landing in shared memory when the block exits.
      volatile int never = 0;
      for (int s = 0; s < STAGES; ++s)
        if (last_phase[s] >= 0 &&
            !mbar_wait(&ctl->full[s], static_cast<uint32_t>(last_phase[s]), &never, tmo))
          raise_abort(abort, status);
    }
  } else {
    // ----------------------------------------------------------- consumers
    // Thread t owns columns n0 + 4t .. n0 + 4t + 3: box t / 64, 8 bytes at
    // (t % 64) * 8 within each of its 512-byte rows.
    const int box = tid / (BOX_COLS / 4);
    const int off = (tid % (BOX_COLS / 4)) * 8;
    int stage = 0;
    uint32_t phase = 0;
    for (int g = 0; g < num_g; ++g) {
      if (!mbar_wait(&ctl->full[stage], phase, abort, tmo)) {
        raise_abort(abort, status);
        break;
      }
      const uint8_t* st = smem + stage * STAGE_STRIDE;
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(st + B_STAGE_BYTES);
      const uint8_t* bp = st + box * B_BOX_BYTES + off;
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        const float x = __uint_as_float(static_cast<uint32_t>(xs[r]) << 16);
        const uint2 v = *reinterpret_cast<const uint2*>(bp + r * BOX_COLS * 2);
        acc[0] = fmaf(x, bf16_lo(v.x), acc[0]);
        acc[1] = fmaf(x, bf16_hi(v.x), acc[1]);
        acc[2] = fmaf(x, bf16_lo(v.y), acc[2]);
        acc[3] = fmaf(x, bf16_hi(v.y), acc[3]);
      }
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive(&ctl->empty[stage]);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }

  const int n = n0 + 4 * tid;
  if (ranges == 1) {
    if (tid < CONSUMERS) store_out<GELU>(C, n, N, acc, epi);
    return;
  }
  // Publish this range's sums, then count the range in.
  if (tid < CONSUMERS)
    __stcg(reinterpret_cast<float4*>(ws + (static_cast<int64_t>(nb) * ranges + rg) * COLS) + tid,
           make_float4(acc[0], acc[1], acc[2], acc[3]));
  __threadfence();
  __syncthreads();
  unsigned int* arrived = counters + 2 * nb;
  unsigned int* departed = arrived + 1;
  if (tid == 0) {
    atomicAdd(arrived, 1u);
    // The launch is cooperative, so every range of this column block is
    // resident: wait (bounded) until all of them have published.
    if (!wait_count_gpu(arrived, static_cast<unsigned>(ranges), tmo)) raise_abort(abort, status);
  }
  __syncthreads();
  // Each range then finishes its own slice of the block's columns: it loads
  // that slice of every range's sums into the idle ring in one batch and
  // adds them in range order 0, 1, ..., ranges - 1.
  const int per = ((COLS + ranges - 1) / ranges + 3) & ~3;  // columns per slice
  const int s0 = rg * per;
  const int cols = s0 < COLS ? (per < COLS - s0 ? per : COLS - s0) : 0;
  float* slice = reinterpret_cast<float*>(smem);             // [ranges][cols]
  if (cols > 0) {
    const int vec = cols / 4;
    const float4* src =
        reinterpret_cast<const float4*>(ws + static_cast<int64_t>(nb) * ranges * COLS + s0);
    for (int i = tid; i < ranges * vec; i += THREADS)
      reinterpret_cast<float4*>(slice)[i] = __ldcg(src + (i / vec) * (COLS / 4) + i % vec);
  }
  __syncthreads();
  for (int c = tid; c < cols; c += THREADS) {
    // in range order; eight terms are loaded before they are added
    float sum = 0.0f;
    int q = 0;
    for (; q + 8 <= ranges; q += 8) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = slice[(q + i) * cols + c];
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += v[i];
    }
    for (; q < ranges; ++q) sum += slice[q * cols + c];
    const int nn = n0 + s0 + c;
    if (nn < N)
      C[nn] = epi_apply<GELU>(epi, sum, epi.beta != 0.0f ? C[nn] : 0.0f,
                              epi.bias ? epi.bias[nn] : 0.0f);
  }
  // Count the range out; the last one leaves both counters at zero for the
  // next launch (every range has passed its wait by then).
  if (tid == 0 && atomicAdd(departed, 1u) == static_cast<unsigned>(ranges - 1)) {
    *arrived = 0u;
    *departed = 0u;
  }
}

size_t gemv_smem_bytes() {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_STRIDE + sizeof(GemvControl);
}

std::atomic<int> g_gemv_attr[64];

}  // namespace

int gemv_ranges(int N, int K, int sms) {
  const int blocks = (N + COLS - 1) / COLS;
  const int groups = (K + ROWS - 1) / ROWS;
  int r = sms / (blocks > 0 ? blocks : 1);
  if (r > groups / 2) r = groups / 2;  // at least two stages per range
  return r < 1 ? 1 : r;
}

int64_t gemv_workspace_bytes(int N, int ranges) {
  if (ranges <= 1) return 0;
  const int64_t blocks = (N + COLS - 1) / COLS;
  return blocks * ranges * COLS * 4;
}

cudaError_t launch_gemm_bf16_gemv(const CUtensorMap& tmA, const CUtensorMap& tmB, float* C,
                                  int N, int K, int ranges, float* ws, unsigned int* counters,
                                  unsigned int* status, const EpiParams& epi,
                                  cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (ranges < 1 || (ranges > 1 && (ws == nullptr || counters == nullptr)))
    return cudaErrorInvalidValue;
  const size_t smem = gemv_smem_bytes();
  if (!g_gemv_attr[dev].load()) {
    for (auto k : {gemm_bf16_gemv_kernel<false>, gemm_bf16_gemv_kernel<true>}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    g_gemv_attr[dev].store(1);
  }
  const int blocks = (N + COLS - 1) / COLS;
  auto kernel = epi.act == kActGelu ? gemm_bf16_gemv_kernel<true> : gemm_bf16_gemv_kernel<false>;
  // With split rows the ranges of a column block wait for one another, so
  // the launch is cooperative: every block is resident at once (the grid,
  // one block per SM, never exceeds the SM count then) or it fails.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = ranges > 1 ? 1 : 0;
  attr[1] = pdl_attribute();
  cfg.gridDim = dim3(static_cast<unsigned>(blocks * ranges), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, C, N, K, ranges, ws, counters, status, epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace g07
