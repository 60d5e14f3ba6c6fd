// kernels.h -- internal launch interface between the C-ABI layer (api.cu)
// and the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "stream_k.cuh"

namespace g07 {

// ---- programmatic dependent launch.  A kernel launched with
// pdl_attribute() may be scheduled while the kernel before it on the stream
// is still finishing; it calls grid_dependency_wait() before its first
// access to global memory, which returns once every earlier kernel has
// completed and its writes are visible (at once when there is nothing to
// wait for).  grid_dependents_go() lets the next such kernel be scheduled
// before this one ends; that kernel's own wait keeps it correct.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_go() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}
// A plain launch (no cluster) with that attribute.
template <typename... P, typename... Args>
cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Records `n` kernel launches by this library (defined in api.cu); the total
// is exported through gemm_launch_count().
void note_launches(int n);

// ---- FP32 SIMT path (gemm_f32.cu)
constexpr int kF32TileM = 128;
constexpr int kF32TileN = 128;
constexpr int kF32TileK = 32;
// Tile-rows per band of the grouped raster (rows of 128 x 128 tiles).
// Measured at 4096^3 (time, DRAM bytes per launch): 8 rows 2197 us, 422.7 MB
// (with the split-K partials written back); 12: 2186 us, 378 MB; 16: 2193 us,
// 351.5 MB; 24: 2192 us, 408 MB; 32: 2209 us, 581 MB.  10 to 14 are equally
// fast, also at 8192 x 8192 x 4096 and 4096 x 4096 x 8192 (0.4-0.7 % ahead
// of 16).
constexpr int kF32Group = 12;
constexpr int kF32Stages = 2;

// Launch plan: `full` tiles in whole waves, then `tail` tiles split into
// `split` k-ranges each (split-K; needs workspace_bytes of partials and
// counter_bytes of zeroed counters).
struct F32Plan {
  int tiles_m = 0, tiles_n = 0;
  int full = 0, tail = 0, split = 1;
  int64_t workspace_bytes = 0, counter_bytes = 0;
  bool small = false;  // 64 x 64 tiles (f32_small_problem), all split `split` ways
};
// Small problems (at most 16 tiles of 128 x 128 and 2^29 multiply-adds) run
// as 64 x 64 tiles split along K, so that they spread over the SMs.
constexpr int kF32SmallTile = 64;
inline bool f32_small_problem(int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = ((M + kF32TileM - 1) / kF32TileM) * ((N + kF32TileN - 1) / kF32TileN);
  return tiles <= 16 && M * N * K <= (int64_t(1) << 29);
}
// Resident blocks of the FP32 kernel on the current device (0: cannot run).
int64_t f32_slots();
F32Plan f32_plan(int M, int N, int K, int64_t slots);
cudaError_t launch_gemm_f32(int M, int N, int K, const float* A, int64_t lda,
                            const float* B, int64_t ldb, float* C, int64_t ldc,
                            bool vec_b, bool vec_c, const F32Plan& plan,
                            float* ws, unsigned int* counters,
                            const EpiParams& epi, cudaStream_t stream);

// ---- BF16, small problems on the CUDA cores (gemm_bf16_small.cu): 64 x 64
// tiles split along K, operands read in place at any alignment.
constexpr int kBf16SmallTile = 64;
constexpr int kBf16SmallMaxSplit = 16;
struct Bf16SmallPlan {
  int tiles_m = 0, tiles_n = 0, split = 1;
  int64_t workspace_bytes = 0;  // partial tiles (after kBf16SmallCounterBytes of counters)
};
// Problems run there (measured crossovers on a GB300, CUDA events):
//   * M >= 2 (M = 1 keeps the small-M tensor-core kernel, which streams B);
//   * M >= 64 or B of at most 2^19 elements (for few rows and a larger B
//     the small-M tensor-core kernel streams B much faster);
//   * at most the set limit of multiply-adds (by default kBf16SmallMaxMacs)
//     and at most kBf16SmallCopyMacs when an operand would have to be
//     copied to an aligned layout for the tensor-core kernels and K is at
//     most kBf16SmallShortK, else at most kBf16SmallAlignedMacs: past those
//     the tensor-core kernels (small-M, narrow-N or paired) are faster,
//     copy included (1000 x 127 x 1000: 10.2 against 17.5 us; 1000 x 1000 x
//     127: 9.7 against 13.4; 127 x 127 x 3001: 14.3 against 17.8), below
//     them slower (3001 x 127 x 127: 14.0 against 10.3; 127 x 3001 x 127:
//     14.0 against 11.8).
constexpr int64_t kBf16SmallMaxMacs = int64_t(1) << 27;
constexpr int64_t kBf16SmallCopyMacs = int64_t(1) << 26;
constexpr int64_t kBf16SmallShortK = 512;
constexpr int64_t kBf16SmallAlignedMacs = int64_t(1) << 24;
bool bf16_small_problem(int64_t M, int64_t N, int64_t K, bool needs_copy);
// Fixed counter area at the start of the scratch block (one counter per
// tile, so at most 1024 split tiles), the partial tiles after it.
constexpr int64_t kBf16SmallCounterBytes = 4096;
Bf16SmallPlan bf16_small_plan(int M, int N, int K, int sms);
cudaError_t launch_gemm_bf16_small(int M, int N, int K, const uint16_t* A, int64_t lda,
                                   const uint16_t* B, int64_t ldb, float* C, int64_t ldc,
                                   bool vec_c, const Bf16SmallPlan& p, float* ws,
                                   unsigned int* counters, const EpiParams& epi,
                                   cudaStream_t stream);

// ---- BF16 tensor-core path: shared tile constants.  One CTA of a pair
// stages kTcTileM rows of A per k-slice of kTcTileK; M <= kTcTileM runs on
// the small-M kernel, larger M on the paired-SM kernel.
constexpr int kTcTileM = 128;
constexpr int kTcTileK = 64;

// ---- BF16 tensor-core path on SM pairs (gemm_bf16_tc2.cu): 256 x 256 tiles
constexpr int kPairTileM = 256;
constexpr int kPairTileN = 256;
constexpr int kPairTileK = 64;
constexpr int kPairStages = 6;

size_t pair_smem_bytes();
// Clusters of two CTAs that can be resident at once (0 if the pair kernel
// cannot run on this device).
int pair_max_active(cudaStream_t stream);
// tmA: box {64, 128}, tmB: box {64, 64}, both 128-byte swizzled.  tmC: FP32
// map of C (box 32 x 32, 128-byte swizzle) for TMA stores, or nullptr to
// store row segments from the staging boxes with ordinary stores.  sched: work sharing from pair_schedule()
// (stream_k.cuh); sched.pairs clusters are launched.  When sched.sk_tiles >
// 0: tmW maps the partial-sum workspace (FP32, 256 columns,
// sched.sk_pairs * 512 rows, box 32 x 32, 128-byte swizzle), sk_sync points
// at sk_sync_words(sched) 64-bit words of any content, and sk_tag is this
// launch's tag (nonzero, below 2^56, not used by an earlier launch on the
// same words).
cudaError_t launch_gemm_bf16_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const CUtensorMap* tmC, const CUtensorMap* tmW,
                                  float* C, int64_t ldc, int M, int N,
                                  const PairSchedule& sched,
                                  unsigned long long* sk_sync,
                                  unsigned long long sk_tag,
                                  unsigned int* status, const EpiParams& epi,
                                  cudaStream_t stream);

// ---- BF16 narrow-N path (gemm_bf16_narrow.cu), N <= kNarrowMaxN and
// M > kSkinnyMaxM: 128-row tiles of C by all N columns, split-K over a
// cluster, partial sums reduced through distributed shared memory.  The
// kernel also takes N > kNarrowMaxN, as 128 x 128 tiles.
constexpr int kNarrowMaxN = 128;
// Wider N also runs on this kernel when its 128 x 128 tiles number at most
// half the SMs and K is at least this long (the automatic schedule only).
constexpr int kNarrowTiledMinK = 1536;
// MMA N used for N columns (64 or 128; 128 for every N > 64).
int narrow_cols(int N);
// Tiles of an M x N problem (128 rows by narrow_cols(N) columns).
int64_t narrow_tiles(int64_t M, int64_t N);
// CTAs per cluster (k split) for an M x N x K problem on `sms` SMs (1..8).
int narrow_split(int M, int N, int K, int sms);
// The same, lowered until every cluster of the launch fits on the current
// device at once (host code).
int narrow_split_resident(int M, int N, int K, int sms);
// tmA: box {64, 128} (kTcTileM rows); tmB: the usual box {64, 64}.
cudaError_t launch_gemm_bf16_narrow(const CUtensorMap& tmA, const CUtensorMap& tmB, float* C,
                                    int64_t ldc, int M, int N, int K, int cs,
                                    unsigned int* status, const EpiParams& epi,
                                    cudaStream_t stream);

// ---- BF16 small-M path (gemm_bf16_skinny.cu): swap-AB, split-K over a
// cluster, partial sums reduced through distributed shared memory.
constexpr int kSkinnyMaxM = 128;
constexpr int kSkinnyTileN = 128;

// MMA N used for M rows (16, 32, 64 or 128).
int skinny_rows(int M);
// CTAs per cluster (k split) for an N x K problem on `sms` SMs (1..8).
int skinny_split(int N, int K, int sms);
// The same, lowered until every cluster of the launch fits on the current
// device at once (checked with the occupancy calculator; host code).
int skinny_split_resident(int M, int N, int K, int sms);
// tmA: box {64, skinny_rows(M)}; tmB: the usual box {64, 64}.
cudaError_t launch_gemm_bf16_skinny(const CUtensorMap& tmA,
                                    const CUtensorMap& tmB, float* C,
                                    int64_t ldc, int M, int N, int K, int cs,
                                    unsigned int* status, const EpiParams& epi,
                                    cudaStream_t stream);

// ---- FP32 teaching rungs (gemm_f32_ladder.cu): 0 naive, 1 smem-tiled,
// 2 one-dimensional register tiling.
cudaError_t launch_gemm_f32_ladder(int rung, int M, int N, int K, const float* A,
                                   int64_t lda, const float* B, int64_t ldb,
                                   float* C, int64_t ldc, cudaStream_t stream);

// ---- small helpers (gemm_aux.cu)
// K == 0: C := act(beta * C + bias) (zeros for the identity epilogue).
cudaError_t launch_zero_fill_f32(float* C, int64_t ldc, int M, int N,
                                 const EpiParams& epi, cudaStream_t stream);
// Copy a rows x cols matrix of 16-bit elements to dst with row stride ld_dst
// (a multiple of 8; dst 16-byte aligned); columns cols..round_up(cols, 8)-1
// of dst are zeroed.  Up to two copies run in one launch.
struct PackJob {
  const uint16_t* src;
  int64_t ld_src;
  uint16_t* dst;
  int64_t ld_dst;
  int rows, cols;
};
struct PackJobs {
  PackJob job[2];
};
cudaError_t launch_pack_u16(const PackJob* jobs, int count, cudaStream_t stream);

}  // namespace g07
