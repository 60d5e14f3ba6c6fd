// api.cu -- the C ABI declared in include/gemm07.h: argument checking, path
// selection, tensor-map encoding, per-device state and the kernel launches.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <chrono>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gemm07.h"
#include "kernels.h"
#include "tile_order.cuh"

namespace g07 {

std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

// Largest M * N * K sent to the CUDA-core small-problem kernel (M >= 2).
std::atomic<int64_t> g_small_limit{kBf16SmallMaxMacs};
bool bf16_small_problem(int64_t M, int64_t N, int64_t K, bool needs_copy) {
  const int64_t lim = g_small_limit.load();
  const int64_t cap = needs_copy && K <= kBf16SmallShortK ? kBf16SmallCopyMacs
                                                          : kBf16SmallAlignedMacs;
  const int64_t max_macs = lim < cap ? lim : cap;
  // M, N, K < 2^31: M * N and N * K fit 64 bits, M * N * K need not
  return M >= 2 && K > 0 && (M >= 64 || N * K <= (int64_t(1) << 19)) &&
         M * N <= max_macs / K;
}

namespace {

// Device status block: [0] status bits (bit 0: a bounded wait ran out),
// [1] test fault mode, [2..3] bounded-wait limit in ns (0: default 2 s).
__device__ unsigned int g_status_word[4];

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 0x7FFFFFFF;  // M, N, K < 2^31

// Scratch kept between calls for one stream and one use: calls on a stream
// run in order, so they can share it without allocating each time (a
// stream-ordered allocate/free pair costs about 2 us of GPU time per call).
enum ScratchUse {
  kScratchStreamK = 0,  // BF16 stream-K partial sums + tagged sync words
  kScratchSplitK = 1,   // FP32 split-K counters (kept zero) + partial sums
  kScratchPack = 2,     // BF16 operands copied to aligned rows
  kScratchSmall = 3,    // BF16 small problems: counters (kept zero) + partial tiles
  kScratchUses = 4
};
struct StreamScratch {
  cudaStream_t stream = nullptr;
  int use = 0;
  void* ptr = nullptr;
  int64_t bytes = 0;
  uint64_t last_use = 0;
};
constexpr int kScratchEntries = 8 * kScratchUses;
// Scratch blocks of one use above this size are allocated per call instead.
constexpr int64_t kScratchKeepMax = int64_t(1) << 30;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  unsigned int* status = nullptr;  // address of g_status_word on this device
  cudaMemPool_t pool = nullptr;
  cudaStream_t up = nullptr;    // host-variant uploads
  cudaStream_t down = nullptr;  // host-variant downloads
  StreamScratch scratch[kScratchEntries];
  uint64_t scratch_clock = 0;
  uint64_t launch_tags = 0;     // stream-K launches so far (tag source)
  uint64_t tag_salt = 0;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

// How the BF16 paired-SM kernel shares a partial last wave (a
// gemm_schedule_t; the values match PairScheduleMode).
std::atomic<int> g_schedule{GEMM_SCHEDULE_AUTO};
static_assert(static_cast<int>(GEMM_SCHEDULE_AUTO) == kScheduleAuto &&
                  static_cast<int>(GEMM_SCHEDULE_STREAM_K) == kScheduleStreamK &&
                  static_cast<int>(GEMM_SCHEDULE_COLUMN_SPLIT) == kScheduleNoSplitK,
              "schedule values");

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType,
                                   cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// C can take the TMA-store epilogue (FP32 rows of whole 16-byte groups).
bool tma_store_ok(const void* C, int64_t N, int64_t ldc) {
  return aligned16(C) && ldc % 4 == 0 && N % 4 == 0;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// The elements a matrix spans (rows x leading dimension) stay at most
// 2^60, so that byte offsets and workspace sizes fit 64 bits.
bool span_ok(int64_t rows, int64_t ld) {
  return rows == 0 || ld <= (int64_t(1) << 60) / rows;
}

gemm_status_t check_args(int64_t M, int64_t N, int64_t K, const void* A,
                         int64_t lda, const void* B, int64_t ldb,
                         const void* C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_ARG;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return GEMM_ERR_INVALID_ARG;
  if (!span_ok(M, lda) || !span_ok(K, ldb) || !span_ok(M, ldc)) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr) return GEMM_ERR_INVALID_ARG;
  if (K > 0 && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_ARG;
  return GEMM_OK;
}

// Scratch of the copies that make A and B readable by the copy engine.
int64_t pack_bytes(int64_t M, int64_t N, int64_t K, bool pack_a, bool pack_b) {
  int64_t ws = 0;
  if (pack_a) ws += round_up(M * round_up(K, 8) * 2, 256);
  if (pack_b) ws += round_up(K * round_up(N, 8) * 2, 256);
  return ws;
}

// Copy the operands the tensor-memory accelerator cannot read in place into
// `cursor` (packed A first, then packed B, each on a 256-byte boundary, row
// strides rounded up to 8 elements), both in one launch; the operand
// pointers and strides are replaced by the copies'.
cudaError_t pack_operands(const gemm_plan_t& plan, const uint16_t* A, int64_t lda,
                          const uint16_t* B, int64_t ldb, int64_t M, int64_t N,
                          int64_t K, uint8_t* cursor, const uint16_t** a_op,
                          int64_t* lda_op, const uint16_t** b_op, int64_t* ldb_op,
                          cudaStream_t stream) {
  PackJob jobs[2];
  int n = 0;
  if (plan.pack_a) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(cursor);
    *lda_op = round_up(K, 8);
    cursor += round_up(M * *lda_op * 2, 256);
    jobs[n++] = PackJob{A, lda, dst, *lda_op, static_cast<int>(M), static_cast<int>(K)};
    *a_op = dst;
  }
  if (plan.pack_b) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(cursor);
    *ldb_op = round_up(N, 8);
    jobs[n++] = PackJob{B, ldb, dst, *ldb_op, static_cast<int>(K), static_cast<int>(N)};
    *b_op = dst;
  }
  return launch_pack_u16(jobs, n, stream);
}

// Scratch of a stream-K schedule: partial sums, then synchronisation words.
int64_t sk_bytes(const PairSchedule& ps) {
  if (ps.sk_tiles == 0) return 0;
  return round_up(sk_partial_bytes(ps), 256) + round_up(sk_sync_words(ps) * 8, 256);
}

void plan_clear(gemm_plan_t* p) {
  std::memset(p, 0, sizeof(*p));
  p->split_k = 1;
}

gemm_status_t plan_f32(int64_t M, int64_t N, int64_t K, const void* A,
                       int64_t lda, const void* B, int64_t ldb, const void* C,
                       int64_t ldc, gemm_plan_t* p) {
  plan_clear(p);
  const gemm_status_t s = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) {
    p->path = GEMM_PATH_NONE;
    return GEMM_OK;
  }
  if (K == 0) {
    p->path = GEMM_PATH_ZERO_FILL;
    return GEMM_OK;
  }
  p->path = GEMM_PATH_F32_SIMT;
  const bool small = f32_small_problem(M, N, K);
  p->tile_m = small ? kF32SmallTile : kF32TileM;
  p->tile_n = small ? kF32SmallTile : kF32TileN;
  p->tile_k = kF32TileK;
  p->stages = 2;
  p->tiles = ((M + p->tile_m - 1) / p->tile_m) * ((N + p->tile_n - 1) / p->tile_n);
  if (p->tiles > kMaxDim) return GEMM_ERR_INVALID_ARG;
  return GEMM_OK;
}

gemm_status_t plan_bf16(int64_t M, int64_t N, int64_t K, const void* A,
                        int64_t lda, const void* B, int64_t ldb, const void* C,
                        int64_t ldc, gemm_plan_t* p, bool allow_small = true) {
  plan_clear(p);
  const gemm_status_t s = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) {
    p->path = GEMM_PATH_NONE;
    return GEMM_OK;
  }
  if (K == 0) {
    p->path = GEMM_PATH_ZERO_FILL;
    return GEMM_OK;
  }
  // The tensor-memory accelerator reads an operand in place when its base is
  // 16-byte aligned and its row stride is a multiple of 16 bytes (8 BF16).
  // (one row of A has no row stride to speak of: only its base counts)
  p->pack_a = (aligned16(A) && (lda % 8 == 0 || M == 1)) ? 0 : 1;
  p->pack_b = (aligned16(B) && ldb % 8 == 0) ? 0 : 1;
  p->path = (p->pack_a || p->pack_b) ? GEMM_PATH_BF16_PACKED : GEMM_PATH_BF16_TMA;
  p->workspace_bytes = pack_bytes(M, N, K, p->pack_a, p->pack_b);
  if (allow_small && bf16_small_problem(M, N, K, p->pack_a || p->pack_b)) {
    // Few multiply-adds: one launch on the CUDA cores, operands read in
    // place (the K split is reported for the 152 SMs of a GB300).
    const Bf16SmallPlan sp = bf16_small_plan(static_cast<int>(M), static_cast<int>(N),
                                             static_cast<int>(K), 152);
    p->path = GEMM_PATH_BF16_SMALL;
    p->pack_a = p->pack_b = 0;
    p->tile_m = p->tile_n = kBf16SmallTile;
    p->tile_k = 32;
    p->stages = 2;
    p->split_k = sp.split;
    p->tiles = static_cast<int64_t>(sp.tiles_m) * sp.tiles_n * sp.split;
    p->workspace_bytes = sp.split > 1 ? kBf16SmallCounterBytes + sp.workspace_bytes : 0;
    return GEMM_OK;
  }
  if (M <= kSkinnyMaxM) {
    // Small M (M = 1 included): 128-column tiles of C, K split over a
    // cluster (the split is
    // reported for the 152 SMs of a GB300; launches use the device's count
    // and lower the split until every cluster is resident at once).
    p->path = GEMM_PATH_BF16_SKINNY;
    p->tile_m = skinny_rows(static_cast<int>(M));
    p->tile_n = kSkinnyTileN;
    p->tile_k = kTcTileK;
    p->stages = 0;
    p->split_k = skinny_split(static_cast<int>(N), static_cast<int>(K), 152);
    p->tiles = ((N + kSkinnyTileN - 1) / kSkinnyTileN) * p->split_k;
    return GEMM_OK;
  }
  // Few tiles and a long K (automatic schedule only: the others describe
  // the paired kernel's work sharing): 128 x 128 tiles with K split over
  // clusters of at least two CTAs keep more SMs busy than 256 x 256 tiles on
  // SM pairs (512x512x4096 11.8 against 20.0 us, 512x1024x8192 16.0
  // against 28.3, 1024x1024x4096 17.2 against 20.1, 1000x1000x3001 19.8
  // against 21.8).
  const bool few_tiles = narrow_tiles(M, N) * 2 <= 152 &&
                         K >= kNarrowTiledMinK && g_schedule.load() == GEMM_SCHEDULE_AUTO;
  if (N <= kNarrowMaxN || few_tiles) {
    // Narrow N: 128-row tiles of C by all N columns (128 x 128 tiles when N
    // is wider), K split over a cluster (the split is reported for the 152
    // SMs of a GB300; launches use the device's count and lower the split
    // until every cluster is resident).
    p->path = GEMM_PATH_BF16_NARROW;
    p->tile_m = kTcTileM;
    p->tile_n = narrow_cols(static_cast<int>(N));
    p->tile_k = kTcTileK;
    p->stages = 0;
    p->split_k = narrow_split(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), 152);
    p->tiles = narrow_tiles(M, N) * p->split_k;
    return GEMM_OK;
  }
  // 256 x 256 tiles on SM pairs (the work sharing is reported for the 76
  // pairs of a 152-SM GB300; launches use the device's resident count).
  p->tile_m = kPairTileM;
  p->tile_n = kPairTileN;
  p->tile_k = kPairTileK;
  p->stages = kPairStages;
  p->tiles = ((M + p->tile_m - 1) / p->tile_m) * ((N + p->tile_n - 1) / p->tile_n);
  if (p->tiles > kMaxDim) return GEMM_ERR_INVALID_ARG;
  const PairSchedule ps =
      pair_schedule(M, N, K, 76, g_schedule.load(), tma_store_ok(C, N, ldc));
  p->dp_tiles = ps.dp_tiles;
  p->sk_tiles = ps.sk_tiles;
  p->sk_pairs = ps.sk_pairs;
  p->pairs = ps.pairs;
  p->workspace_bytes += sk_bytes(ps);
  return GEMM_OK;
}

// The caller's epilogue description as kernel parameters (NULL: identity).
gemm_status_t to_epi(const gemm_epilogue_t* e, EpiParams* out) {
  *out = epi_identity();
  if (e == nullptr) return GEMM_OK;
  if (e->activation != GEMM_ACT_NONE && e->activation != GEMM_ACT_RELU &&
      e->activation != GEMM_ACT_GELU)
    return GEMM_ERR_INVALID_ARG;
  out->alpha = e->alpha;
  out->beta = e->beta;
  out->bias = e->bias;
  out->act = e->activation;
  return GEMM_OK;
}

gemm_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GEMM_OK;
  if (e == cudaErrorMemoryAllocation) return GEMM_ERR_NO_MEMORY;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ||
      e == cudaErrorNoKernelImageForDevice)
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  return GEMM_ERR_LAUNCH;
}

// Per-device set-up, once: capability check, status word, memory pool.
gemm_status_t device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
      d.status = static_cast<unsigned int*>(addr);
      cudaMemPoolProps props;
      std::memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_NO_MEMORY;
      }
      uint64_t keep = ~0ull;  // keep freed blocks for the next call
      cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
      // tags of different processes or library loads sharing leftover
      // memory differ
      d.tag_salt = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(&d)) ^
                   (static_cast<uint64_t>(std::chrono::steady_clock::now()
                                              .time_since_epoch()
                                              .count()) *
                    0x9E3779B97F4A7C15ull);
    }
    d.ready = true;
  }
  if (!d.supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return GEMM_OK;
}

// The two helper streams of the host-buffer variants (created once).
gemm_status_t host_streams(DeviceState* d) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (d->up == nullptr &&
      cudaStreamCreateWithFlags(&d->up, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    d->up = nullptr;
    return GEMM_ERR_LAUNCH;
  }
  if (d->down == nullptr &&
      cudaStreamCreateWithFlags(&d->down, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    d->down = nullptr;
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

gemm_status_t encoder(EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = g_encode;
  return GEMM_OK;
}

// 2-D BF16 tensor map: dims {inner, outer}, row stride ld elements, box
// {box_inner, box_outer}, 128-byte swizzle, zero fill out of range.
gemm_status_t make_map_typed(CUtensorMap* map, CUtensorMapDataType type,
                             int64_t elem_bytes, const void* base, int64_t inner,
                             int64_t outer, int64_t ld, uint32_t box_inner,
                             uint32_t box_outer,
                             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = nullptr;
  gemm_status_t s = encoder(&enc);
  if (s != GEMM_OK) return s;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner),
                              static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * elem_bytes)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, type, 2,
                         const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INTERNAL;
}

gemm_status_t make_map(CUtensorMap* map, const void* base, int64_t inner,
                       int64_t outer, int64_t ld, uint32_t box_inner,
                       uint32_t box_outer) {
  return make_map_typed(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner,
                        outer, ld, box_inner, box_outer);
}

// BF16 operand maps: A boxes of 64 k x `a_rows` rows, B boxes of 64
// columns x 64 k, both 128-byte swizzled.
gemm_status_t make_operand_maps(CUtensorMap* tmA, CUtensorMap* tmB,
                                const uint16_t* a, int64_t lda,
                                const uint16_t* b, int64_t ldb, int64_t M,
                                int64_t N, int64_t K, uint32_t a_rows) {
  // A single row is read in place whatever its stride (boxes cover rows the
  // map holds as out of range, which read 0), so any 16-byte multiple will do.
  gemm_status_t s = make_map(tmA, a, K, M, M == 1 ? round_up(lda, 8) : lda, kTcTileK, a_rows);
  if (s == GEMM_OK) s = make_map(tmB, b, N, K, ldb, 64, kTcTileK);
  return s;
}

// The TMA-store epilogue needs C 16-byte aligned with rows a multiple of 16
// bytes apart, and N a multiple of 4: the copy engine clips the inner
// dimension of a store in 16-byte units, so a row that ends mid-unit would
// be written past column N-1.
// FP32 map of C for the TMA-store epilogue: 32 x 32 boxes, 128-byte swizzle.
gemm_status_t make_map_c(CUtensorMap* map, const float* C, int64_t M,
                         int64_t N, int64_t ldc) {
  return make_map_typed(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, ldc,
                        32, 32);
}

gemm_status_t pool_alloc(DeviceState* d, void** p, int64_t bytes,
                         cudaStream_t stream) {
  *p = nullptr;
  if (bytes <= 0) return GEMM_OK;
  if (cudaMallocFromPoolAsync(p, static_cast<size_t>(bytes), d->pool, stream) !=
      cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return GEMM_ERR_NO_MEMORY;
  }
  return GEMM_OK;
}

void pool_free(void* p, cudaStream_t stream) {
  if (p) cudaFreeAsync(p, stream);
}

std::mutex g_scratch_mutex;

// At least `bytes` of scratch of one use for work queued on `stream`, kept
// for later calls on the same stream.  *fresh is set when the block is new
// (its contents are undefined).  Growing frees the old block in stream
// order; taking over another stream's entry (all entries in use) first
// waits for the device, since that stream's work may still use the block.
gemm_status_t stream_scratch(DeviceState* d, cudaStream_t stream, int use,
                             int64_t bytes, void** out, bool* fresh) {
  *out = nullptr;
  *fresh = false;
  if (bytes <= 0) return GEMM_OK;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  StreamScratch* e = nullptr;
  for (StreamScratch& x : d->scratch)
    if (x.ptr && x.stream == stream && x.use == use) e = &x;
  if (e == nullptr) {
    for (StreamScratch& x : d->scratch)
      if (!x.ptr) {
        e = &x;
        break;
      }
  }
  if (e == nullptr) {
    e = &d->scratch[0];
    for (StreamScratch& x : d->scratch)
      if (x.last_use < e->last_use) e = &x;
    if (cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    cudaFreeAsync(e->ptr, stream);
    *e = StreamScratch();
  }
  if (e->ptr && e->bytes < bytes) {
    cudaFreeAsync(e->ptr, stream);
    e->ptr = nullptr;
  }
  if (!e->ptr) {
    const int64_t want = round_up(bytes, int64_t(1) << 20);
    if (cudaMallocFromPoolAsync(&e->ptr, static_cast<size_t>(want), d->pool,
                                stream) != cudaSuccess) {
      cudaGetLastError();
      *e = StreamScratch();
      return GEMM_ERR_NO_MEMORY;
    }
    e->bytes = want;
    *fresh = true;
  }
  e->stream = stream;
  e->use = use;
  e->last_use = ++d->scratch_clock;
  *out = e->ptr;
  return GEMM_OK;
}

// Scratch for one call: the stream's kept block when small enough, else a
// block from the pool for this call only (*owned: free it after the call).
// While the stream is being captured into a CUDA graph and its kept block is
// missing or too small, the block is allocated for the call too (inside the
// graph, which owns it), never kept: memory allocated during a capture
// belongs to the graph.
gemm_status_t call_scratch(DeviceState* d, cudaStream_t stream, int use,
                           int64_t bytes, void** out, bool* fresh, bool* owned) {
  *owned = false;
  *out = nullptr;
  *fresh = false;
  if (bytes <= 0) return GEMM_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  if (cap != cudaStreamCaptureStatusNone) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    for (StreamScratch& x : d->scratch)
      if (x.ptr && x.stream == stream && x.use == use && x.bytes >= bytes) {
        x.last_use = ++d->scratch_clock;
        *out = x.ptr;
        return GEMM_OK;
      }
  }
  if (bytes > kScratchKeepMax || cap != cudaStreamCaptureStatusNone) {
    *owned = true;
    *fresh = true;
    return pool_alloc(d, out, bytes, stream);
  }
  return stream_scratch(d, stream, use, bytes, out, fresh);
}

// A fresh 56-bit nonzero tag for one stream-K launch.
unsigned long long next_launch_tag(DeviceState* d) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  uint64_t z = ++d->launch_tags + d->tag_salt;
  // splitmix64 finaliser
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  z &= (1ull << 56) - 1;
  return z ? z : 1ull;
}

// Map of the stream-K partial-sum workspace (see gemm_bf16_tc2.cu).
gemm_status_t make_map_partials(CUtensorMap* map, float* ws,
                                const PairSchedule& ps) {
  return make_map_typed(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, 256,
                        static_cast<int64_t>(ps.sk_pairs) * 512, 256, 32, 32);
}

gemm_status_t run_f32(int64_t M, int64_t N, int64_t K, const float* A,
                      int64_t lda, const float* B, int64_t ldb, float* C,
                      int64_t ldc, cudaStream_t stream,
                      const EpiParams& epi = epi_identity()) {
  gemm_plan_t plan;
  gemm_status_t s = plan_f32(M, N, K, A, lda, B, ldb, C, ldc, &plan);
  if (s != GEMM_OK || plan.path == GEMM_PATH_NONE) return s;
  DeviceState* d = nullptr;
  s = device_state(&d);
  if (s != GEMM_OK) return s;
  if (plan.path == GEMM_PATH_ZERO_FILL)
    return from_cuda(launch_zero_fill_f32(C, ldc, static_cast<int>(M),
                                          static_cast<int>(N), epi, stream));
  const bool vec_b = aligned16(B) && ldb % 4 == 0;
  const bool vec_c = aligned16(C) && ldc % 4 == 0;
  const int m = static_cast<int>(M), n = static_cast<int>(N),
            k = static_cast<int>(K);
  const int64_t slots = f32_slots();
  if (slots <= 0) return GEMM_ERR_LAUNCH;
  const F32Plan fp = f32_plan(m, n, k, slots);
  // Split-K scratch: one counter per resident slot first (zero between
  // launches: the last block of each split tile puts its counter back to
  // zero, so they are cleared only when the block is new), then partials.
  const int64_t counter_area = round_up(slots * 4, 256);
  void* ws = nullptr;
  bool fresh = false, owned = false;
  if (fp.split > 1) {
    s = call_scratch(d, stream, kScratchSplitK, counter_area + fp.workspace_bytes, &ws,
                     &fresh, &owned);
    if (s != GEMM_OK) return s;
    if (fresh) s = from_cuda(cudaMemsetAsync(ws, 0, counter_area, stream));
  }
  unsigned int* counters = static_cast<unsigned int*>(ws);
  float* partials =
      ws ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + counter_area) : nullptr;
  if (s == GEMM_OK)
    s = from_cuda(launch_gemm_f32(m, n, k, A, lda, B, ldb, C, ldc, vec_b, vec_c,
                                  fp, partials, counters, epi, stream));
  if (owned) pool_free(ws, stream);
  return s;
}

gemm_status_t run_bf16(int64_t M, int64_t N, int64_t K, const uint16_t* A,
                       int64_t lda, const uint16_t* B, int64_t ldb, float* C,
                       int64_t ldc, cudaStream_t stream,
                       const EpiParams& epi = epi_identity()) {
  gemm_plan_t plan;
  gemm_status_t s = plan_bf16(M, N, K, A, lda, B, ldb, C, ldc, &plan);
  if (s != GEMM_OK || plan.path == GEMM_PATH_NONE) return s;
  DeviceState* d = nullptr;
  s = device_state(&d);
  if (s != GEMM_OK) return s;
  if (plan.path == GEMM_PATH_ZERO_FILL)
    return from_cuda(launch_zero_fill_f32(C, ldc, static_cast<int>(M),
                                          static_cast<int>(N), epi, stream));

  const int m = static_cast<int>(M), n = static_cast<int>(N),
            k = static_cast<int>(K);
  if (plan.path == GEMM_PATH_BF16_SMALL) {
    // A fixed area of counters first, so that every call finds its counters
    // zero whatever the size of earlier calls (zero when new; each launch's
    // last blocks put them back), then the partial tiles.
    const Bf16SmallPlan sp = bf16_small_plan(m, n, k, d->sms);
    const int64_t counter_area = kBf16SmallCounterBytes;
    void* ws = nullptr;
    bool fresh = false, owned = false;
    if (sp.split > 1) {
      s = call_scratch(d, stream, kScratchSmall, counter_area + sp.workspace_bytes, &ws,
                       &fresh, &owned);
      if (s != GEMM_OK) return s;
      if (fresh) s = from_cuda(cudaMemsetAsync(ws, 0, counter_area, stream));
    }
    if (s == GEMM_OK)
      s = from_cuda(launch_gemm_bf16_small(
          m, n, k, A, lda, B, ldb, C, ldc, aligned16(C) && ldc % 4 == 0, sp,
          ws ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + counter_area) : nullptr,
          static_cast<unsigned int*>(ws), epi, stream));
    if (owned) pool_free(ws, stream);
    return s;
  }
  const bool skinny = plan.path == GEMM_PATH_BF16_SKINNY;
  const bool narrow = plan.path == GEMM_PATH_BF16_NARROW;
  const bool paired = !skinny && !narrow;
  const int max_pairs = paired ? pair_max_active(stream) : 0;
  // The paired-SM kernel is the only kernel for M > 128: a device on which
  // no pair of its CTAs can be resident cannot run this GEMM.
  if (paired && max_pairs <= 0) return GEMM_ERR_LAUNCH;
  PairSchedule ps;
  if (max_pairs > 0)
    ps = pair_schedule(M, N, K, max_pairs, g_schedule.load(),
                       tma_store_ok(C, N, ldc) && epi.beta == 0.0f && epi.bias == nullptr &&
                           epi.act == 0);
  const int64_t pack_ws = pack_bytes(M, N, K, plan.pack_a, plan.pack_b);
  void* ws = nullptr;
  bool fresh = false, owned = false;
  s = call_scratch(d, stream, kScratchPack, pack_ws, &ws, &fresh, &owned);
  if (s != GEMM_OK) return s;
  // stream-K scratch: partial sums, then tagged synchronisation words (any
  // contents will do)
  void* sk = nullptr;
  bool sk_fresh = false, sk_owned = false;
  if (s == GEMM_OK)
    s = call_scratch(d, stream, kScratchStreamK, sk_bytes(ps), &sk, &sk_fresh,
                     &sk_owned);
  float* sk_ws = static_cast<float*>(sk);
  unsigned long long* sk_sync = nullptr;
  CUtensorMap tmW;
  if (s == GEMM_OK && ps.sk_tiles > 0) {
    sk_sync = reinterpret_cast<unsigned long long*>(
        static_cast<uint8_t*>(sk) + round_up(sk_partial_bytes(ps), 256));
    s = make_map_partials(&tmW, sk_ws, ps);
  }
  const uint16_t* a_op = A;
  const uint16_t* b_op = B;
  int64_t lda_op = lda, ldb_op = ldb;
  uint8_t* cursor = static_cast<uint8_t*>(ws);
  if (s == GEMM_OK)
    s = from_cuda(pack_operands(plan, A, lda, B, ldb, M, N, K, cursor, &a_op, &lda_op,
                                &b_op, &ldb_op, stream));
  CUtensorMap tmA, tmB;
  if (s == GEMM_OK)
    s = make_operand_maps(&tmA, &tmB, a_op, lda_op, b_op, ldb_op, M, N, K,
                          skinny ? static_cast<uint32_t>(skinny_rows(m)) : kTcTileM);
  if (s == GEMM_OK && skinny) {
    s = from_cuda(launch_gemm_bf16_skinny(tmA, tmB, C, ldc, m, n, k,
                                          skinny_split_resident(m, n, k, d->sms), d->status,
                                          epi, stream));
  } else if (s == GEMM_OK && narrow) {
    s = from_cuda(launch_gemm_bf16_narrow(tmA, tmB, C, ldc, m, n, k,
                                          narrow_split_resident(m, n, k, d->sms), d->status,
                                          epi, stream));
  } else if (s == GEMM_OK) {
    CUtensorMap tmC;
    const bool tma_c = tma_store_ok(C, N, ldc) && make_map_c(&tmC, C, M, N, ldc) == GEMM_OK;
    const unsigned long long tag = ps.sk_tiles > 0 ? next_launch_tag(d) : 0;
    s = from_cuda(launch_gemm_bf16_pair(
        tmA, tmB, tma_c ? &tmC : nullptr, ps.sk_tiles > 0 ? &tmW : nullptr, C,
        ldc, m, n, ps, sk_sync, tag, d->status, epi, stream));
  }
  if (owned) pool_free(ws, stream);
  if (sk_owned) pool_free(sk, stream);
  return s;
}

// Rows of the largest block of whole tile rows, within [lo, hi] of M, whose
// tiles fill whole waves of `slots` resident blocks; 0 if there is none.
int64_t whole_wave_rows(int64_t M, int64_t N, int tile_m, int tile_n, int64_t slots,
                        double lo, double hi) {
  if (slots <= 0) return 0;
  const int64_t tm = (M + tile_m - 1) / tile_m, tn = (N + tile_n - 1) / tile_n;
  for (int64_t r = static_cast<int64_t>(hi * static_cast<double>(tm));
       r >= 1 && static_cast<double>(r) >= lo * static_cast<double>(tm); --r)
    if ((r * tn) % slots == 0 && r * tile_m < M) return r * tile_m;
  return 0;
}

// Host-buffer variant: stage through pool memory and overlap the copies with
// the GEMM.  A is split into `chunks` row blocks; each block's GEMM runs on
// the caller's stream as soon as its rows (and B) have arrived, and each
// block of C goes back on an internal download stream while the next block
// computes, so both directions of the link are busy at once.
//
// Every output row needs all of B, so the first block would wait for the
// whole of B.  Instead, with `max_parts` > 1, several blocks and a long K, B
// and the first block of A go up in pieces along K, and the first block's
// product is accumulated piece by piece (C := A_k B_k, then
// C := A_k B_k + C): its first GEMM starts once one piece of the operands
// has arrived.  The first rows' sums are then added in that order.  This
// pays when the GEMM, not the link, takes the time (FP32).
//
// With `head_rows` > 0 there are two blocks, rows [0, head_rows) and the
// rest: a head block that is a whole number of waves of resident tiles
// keeps the block GEMMs from adding partial waves of their own.
template <typename T, typename Run>
gemm_status_t run_host(int64_t M, int64_t N, int64_t K, const T* A,
                       int64_t lda, const T* B, int64_t ldb, float* C,
                       int64_t ldc, cudaStream_t stream, int max_chunks,
                       int64_t min_chunk_rows, int max_parts, int64_t head_rows,
                       Run run) {
  gemm_status_t s = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (s != GEMM_OK || M == 0 || N == 0) return s;
  DeviceState* d = nullptr;
  s = device_state(&d);
  if (s != GEMM_OK) return s;
  s = host_streams(d);
  if (s != GEMM_OK) return s;
  const int64_t eb = static_cast<int64_t>(sizeof(T));
  int64_t chunks = M / (min_chunk_rows > 0 ? min_chunk_rows : 1);
  if (chunks > max_chunks) chunks = max_chunks;
  if (chunks < 1 || K == 0) chunks = 1;
  constexpr int kMaxChunks = 8;
  if (chunks > kMaxChunks) chunks = kMaxChunks;
  if (head_rows <= 0 || head_rows >= M || K == 0) head_rows = 0;
  if (head_rows > 0) chunks = 2;
  constexpr int kParts = 8;          // at most this many pieces of K
  constexpr int64_t kMinPartK = 512;
  int k_parts = max_parts < kParts ? max_parts : kParts;
  if (k_parts < 1 || chunks < 2 || K < k_parts * kMinPartK) k_parts = 1;

  void *dA = nullptr, *dB = nullptr, *dC = nullptr;
  // events: start, one per piece of the first block, then a_ready / c_ready
  // per block
  constexpr int kMaxEvents = 1 + kParts + 2 * kMaxChunks;
  cudaEvent_t ev[kMaxEvents] = {};
  const int want_ev = 1 + k_parts + 2 * static_cast<int>(chunks);
  int n_ev = 0;
  for (; n_ev < want_ev; ++n_ev)
    if (cudaEventCreateWithFlags(&ev[n_ev], cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      s = GEMM_ERR_LAUNCH;
      break;
    }
  cudaEvent_t start = ev[0];
  cudaEvent_t* piece_ready = ev + 1;
  cudaEvent_t* block_ev = ev + 1 + k_parts;
  if (s == GEMM_OK) s = pool_alloc(d, &dA, M * K * eb, stream);
  if (s == GEMM_OK) s = pool_alloc(d, &dB, K * N * eb, stream);
  if (s == GEMM_OK) s = pool_alloc(d, &dC, M * N * 4, stream);
  // the helper streams start after everything already queued on `stream`
  if (s == GEMM_OK) s = from_cuda(cudaEventRecord(start, stream));
  if (s == GEMM_OK) s = from_cuda(cudaStreamWaitEvent(d->up, start, 0));
  if (s == GEMM_OK) s = from_cuda(cudaStreamWaitEvent(d->down, start, 0));
  uint8_t* dA8 = static_cast<uint8_t*>(dA);
  uint8_t* dB8 = static_cast<uint8_t*>(dB);
  // Uploads, in the order they are needed, on the upload stream: B (in
  // k_parts pieces, each with its columns of the first block of A), then the
  // other blocks of A.
  // block i covers rows [row_at(i), row_at(i + 1)): equal shares, boundaries
  // on whole 128-row tiles where the rows allow
  auto row_at = [&](int64_t i) -> int64_t {
    if (i >= chunks) return M;
    if (head_rows > 0) return i == 0 ? 0 : head_rows;
    const int64_t r = M * i / chunks;
    const int64_t q = (r + 64) / 128 * 128;
    return q > 0 && q < M ? q : r;
  };
  const int64_t rows0 = row_at(1);
  // piece p covers k in [piece_k(p), piece_k(p + 1)), on 64-element bounds
  auto piece_k = [&](int p) -> int64_t {
    return p >= k_parts ? K : (K * p / k_parts) / 64 * 64;
  };
  for (int p = 0; s == GEMM_OK && K > 0 && p < k_parts; ++p) {
    const int64_t k0 = piece_k(p), k1 = piece_k(p + 1);
    s = from_cuda(cudaMemcpy2DAsync(dB8 + k0 * N * eb, N * eb, B + k0 * ldb, ldb * eb,
                                    N * eb, k1 - k0, cudaMemcpyHostToDevice, d->up));
    if (s == GEMM_OK)
      s = from_cuda(cudaMemcpy2DAsync(dA8 + k0 * eb, K * eb, A + k0, lda * eb,
                                      (k1 - k0) * eb, rows0, cudaMemcpyHostToDevice,
                                      d->up));
    if (s == GEMM_OK) s = from_cuda(cudaEventRecord(piece_ready[p], d->up));
  }
  for (int64_t i = 1; s == GEMM_OK && K > 0 && i < chunks; ++i) {
    const int64_t r0 = row_at(i), r1 = row_at(i + 1);
    s = from_cuda(cudaMemcpy2DAsync(dA8 + r0 * K * eb, K * eb, A + r0 * lda, lda * eb,
                                    K * eb, r1 - r0, cudaMemcpyHostToDevice, d->up));
    if (s == GEMM_OK) s = from_cuda(cudaEventRecord(block_ev[2 * i], d->up));
  }
  // GEMMs on the caller's stream, downloads on the download stream.
  EpiParams accumulate = epi_identity();
  accumulate.beta = 1.0f;
  for (int64_t i = 0; s == GEMM_OK && i < chunks; ++i) {
    const int64_t r0 = row_at(i), r1 = row_at(i + 1), rows = r1 - r0;
    const T* a_blk = reinterpret_cast<const T*>(dA8 + r0 * K * eb);
    float* c_blk = static_cast<float*>(dC) + r0 * N;
    if (i == 0) {
      for (int p = 0; s == GEMM_OK && p < k_parts; ++p) {
        const int64_t k0 = piece_k(p), k1 = piece_k(p + 1);
        if (K > 0) s = from_cuda(cudaStreamWaitEvent(stream, piece_ready[p], 0));
        if (s == GEMM_OK)
          s = run(rows, N, k1 - k0, a_blk + k0, K > 0 ? K : 1,
                  reinterpret_cast<const T*>(dB8 + k0 * N * eb), N, c_blk, N,
                  p == 0 ? epi_identity() : accumulate, stream);
      }
    } else {
      s = from_cuda(cudaStreamWaitEvent(stream, block_ev[2 * i], 0));
      if (s == GEMM_OK)
        s = run(rows, N, K, a_blk, K, reinterpret_cast<const T*>(dB8), N, c_blk, N,
                epi_identity(), stream);
    }
    cudaEvent_t c_ready = block_ev[2 * i + 1];
    if (s == GEMM_OK) s = from_cuda(cudaEventRecord(c_ready, stream));
    if (s == GEMM_OK) s = from_cuda(cudaStreamWaitEvent(d->down, c_ready, 0));
    if (s == GEMM_OK)
      s = from_cuda(cudaMemcpy2DAsync(C + r0 * ldc, ldc * 4, c_blk, N * 4, N * 4, rows,
                                      cudaMemcpyDeviceToHost, d->down));
  }
  // Every copy is done before the buffers go back to the pool.
  if (s == GEMM_OK) s = from_cuda(cudaEventRecord(ev[0], d->down));
  if (s == GEMM_OK) s = from_cuda(cudaStreamWaitEvent(stream, ev[0], 0));
  pool_free(dA, stream);
  pool_free(dB, stream);
  pool_free(dC, stream);
  const cudaError_t e1 = cudaStreamSynchronize(stream);
  const cudaError_t e2 = cudaStreamSynchronize(d->down);
  const cudaError_t e3 = cudaStreamSynchronize(d->up);
  for (int j = 0; j < n_ev; ++j) cudaEventDestroy(ev[j]);
  if (s == GEMM_OK) s = from_cuda(e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3));
  return s;
}

// ----------------------------------------------------------------------
// No-allocation variant of the BF16 entry point.  Its operand copies go into
// a fixed array in device memory instead of the memory pool.

constexpr int64_t kNoallocScratchBytes =
    static_cast<int64_t>(GEMM07_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) uint8_t g_noalloc_scratch[GEMM07_NOALLOC_SCRATCH_BYTES];

struct NoallocState {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  unsigned int* status = nullptr;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch
  uint64_t launch_tags = 0;    // stream-K launches so far (tag source)
};
NoallocState g_noalloc[kMaxDevices];

// A fresh 56-bit nonzero tag for one stream-K launch on the fixed scratch.
unsigned long long next_noalloc_tag(NoallocState* d) {
  static std::mutex m;
  std::lock_guard<std::mutex> lock(m);
  uint64_t z = ++d->launch_tags + 0x5851F42D4C957F2Dull *
                                      static_cast<uint64_t>(reinterpret_cast<uintptr_t>(d));
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  z &= (1ull << 56) - 1;
  return z ? z : 1ull;
}

// Once per device, with that device current: capability check and the device
// addresses of the status word and of the scratch array.  Allocates nothing.
gemm_status_t noalloc_device(NoallocState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  NoallocState& d = g_noalloc[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* status = nullptr;
      void* scratch = nullptr;
      if (cudaGetSymbolAddress(&status, g_status_word) != cudaSuccess ||
          cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
      }
      d.status = static_cast<unsigned int*>(status);
      d.scratch = static_cast<uint8_t*>(scratch);
    }
    d.ready = true;
  }
  if (!d.supported) return GEMM_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return GEMM_OK;
}

gemm_status_t run_bf16_noalloc(int64_t M, int64_t N, int64_t K,
                               const uint16_t* A, int64_t lda,
                               const uint16_t* B, int64_t ldb, float* C,
                               int64_t ldc, cudaStream_t stream) {
  gemm_plan_t plan;
  gemm_status_t s = plan_bf16(M, N, K, A, lda, B, ldb, C, ldc, &plan, /*allow_small=*/false);
  if (s != GEMM_OK || plan.path == GEMM_PATH_NONE) return s;
  const int64_t pack_ws = pack_bytes(M, N, K, plan.pack_a, plan.pack_b);
  if (pack_ws > kNoallocScratchBytes) return GEMM_ERR_SCRATCH_TOO_SMALL;
  NoallocState* d = nullptr;
  s = noalloc_device(&d);
  if (s != GEMM_OK) return s;
  if (plan.path == GEMM_PATH_ZERO_FILL)
    return from_cuda(launch_zero_fill_f32(C, ldc, static_cast<int>(M),
                                          static_cast<int>(N), epi_identity(), stream));
  const int m = static_cast<int>(M), n = static_cast<int>(N),
            k = static_cast<int>(K);
  // Same layout as the pooled path: packed A first, then packed B, each
  // starting on a 256-byte boundary.  Only the copied extent is ever read.
  const uint16_t* a_op = A;
  const uint16_t* b_op = B;
  int64_t lda_op = lda, ldb_op = ldb;
  uint8_t* cursor = d->scratch;
  s = from_cuda(pack_operands(plan, A, lda, B, ldb, M, N, K, cursor, &a_op, &lda_op,
                              &b_op, &ldb_op, stream));
  CUtensorMap tmA, tmB;
  // The small-M and narrow-N kernels reduce through distributed shared
  // memory: they put nothing in the array beyond the copies.
  const bool skinny = plan.path == GEMM_PATH_BF16_SKINNY;
  const bool narrow = plan.path == GEMM_PATH_BF16_NARROW;
  const int max_pairs = skinny || narrow ? 0 : pair_max_active(stream);
  if (!skinny && !narrow && max_pairs <= 0) return GEMM_ERR_LAUNCH;
  if (s == GEMM_OK)
    s = make_operand_maps(&tmA, &tmB, a_op, lda_op, b_op, ldb_op, M, N, K,
                          skinny ? static_cast<uint32_t>(skinny_rows(m)) : kTcTileM);
  if (s != GEMM_OK) return s;
  if (skinny)
    return from_cuda(launch_gemm_bf16_skinny(tmA, tmB, C, ldc, m, n, k,
                                             skinny_split_resident(m, n, k, d->sms),
                                             d->status, epi_identity(), stream));
  if (narrow)
    return from_cuda(launch_gemm_bf16_narrow(tmA, tmB, C, ldc, m, n, k,
                                             narrow_split_resident(m, n, k, d->sms),
                                             d->status, epi_identity(), stream));
  // Stream-K only when its scratch fits after the packed operands.
  PairSchedule ps =
      pair_schedule(M, N, K, max_pairs, g_schedule.load(), tma_store_ok(C, N, ldc));
  if (pack_ws + sk_bytes(ps) > kNoallocScratchBytes)
    ps = pair_schedule(M, N, K, max_pairs, kScheduleNoSplitK);
  float* sk_ws = nullptr;
  unsigned long long* sk_sync = nullptr;
  CUtensorMap tmW;
  unsigned long long tag = 0;
  if (ps.sk_tiles > 0) {
    sk_ws = reinterpret_cast<float*>(d->scratch + pack_ws);
    sk_sync = reinterpret_cast<unsigned long long*>(
        d->scratch + pack_ws + round_up(sk_partial_bytes(ps), 256));
    s = make_map_partials(&tmW, sk_ws, ps);
    if (s != GEMM_OK) return s;
    tag = next_noalloc_tag(d);
  }
  CUtensorMap tmC;
  const bool tma_c = tma_store_ok(C, N, ldc) && make_map_c(&tmC, C, M, N, ldc) == GEMM_OK;
  return from_cuda(launch_gemm_bf16_pair(
      tmA, tmB, tma_c ? &tmC : nullptr, ps.sk_tiles > 0 ? &tmW : nullptr, C,
      ldc, m, n, ps, sk_sync, tag, d->status, epi_identity(), stream));
}

}  // namespace
}  // namespace g07

using namespace g07;

extern "C" {

gemm_status_t gemm_f32(int64_t M, int64_t N, int64_t K, const float* A,
                       int64_t lda, const float* B, int64_t ldb, float* C,
                       int64_t ldc, void* stream) {
  return run_f32(M, N, K, A, lda, B, ldb, C, ldc,
                 static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_bf16_f32acc(int64_t M, int64_t N, int64_t K,
                               const uint16_t* A, int64_t lda,
                               const uint16_t* B, int64_t ldb, float* C,
                               int64_t ldc, void* stream) {
  return run_bf16(M, N, K, A, lda, B, ldb, C, ldc,
                  static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f32_ex(int64_t M, int64_t N, int64_t K, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float* C,
                          int64_t ldc, const gemm_epilogue_t* epilogue,
                          void* stream) {
  EpiParams epi;
  const gemm_status_t s = to_epi(epilogue, &epi);
  if (s != GEMM_OK) return s;
  return run_f32(M, N, K, A, lda, B, ldb, C, ldc,
                 static_cast<cudaStream_t>(stream), epi);
}

gemm_status_t gemm_bf16_f32acc_ex(int64_t M, int64_t N, int64_t K,
                                  const uint16_t* A, int64_t lda,
                                  const uint16_t* B, int64_t ldb, float* C,
                                  int64_t ldc, const gemm_epilogue_t* epilogue,
                                  void* stream) {
  EpiParams epi;
  const gemm_status_t s = to_epi(epilogue, &epi);
  if (s != GEMM_OK) return s;
  return run_bf16(M, N, K, A, lda, B, ldb, C, ldc,
                  static_cast<cudaStream_t>(stream), epi);
}

gemm_status_t gemm_bf16_f32acc_noalloc(int64_t M, int64_t N, int64_t K,
                                        const uint16_t* A, int64_t lda,
                                        const uint16_t* B, int64_t ldb,
                                        float* C, int64_t ldc, void* stream) {
  return run_bf16_noalloc(M, N, K, A, lda, B, ldb, C, ldc,
                          static_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_f32_ladder(int rung, int64_t M, int64_t N, int64_t K,
                              const float* A, int64_t lda, const float* B,
                              int64_t ldb, float* C, int64_t ldc, void* stream) {
  if (rung < 0 || rung > 2) return GEMM_ERR_INVALID_ARG;
  gemm_status_t s = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (s != GEMM_OK || M == 0 || N == 0) return s;
  // grid.y of the rungs is M / 8 at most rows per block: keep it in range
  if (M > 65535LL * 8) return GEMM_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  s = device_state(&d);
  if (s != GEMM_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (K == 0)
    return from_cuda(launch_zero_fill_f32(C, ldc, static_cast<int>(M),
                                          static_cast<int>(N), epi_identity(), st));
  return from_cuda(launch_gemm_f32_ladder(rung, static_cast<int>(M),
                                          static_cast<int>(N), static_cast<int>(K),
                                          A, lda, B, ldb, C, ldc, st));
}

gemm_status_t gemm_f32_host(int64_t M, int64_t N, int64_t K, const float* A,
                            int64_t lda, const float* B, int64_t ldb, float* C,
                            int64_t ldc, void* stream) {
  // A head block of whole waves of 128 x 128 tiles, 30-60 % of the rows, if
  // one exists (4096 x 4096: 2432 rows, two waves of 304 tiles).
  const int64_t head =
      M >= 2048 && N > 0 ? whole_wave_rows(M, N, kF32TileM, kF32TileN, f32_slots(), 0.3, 0.6)
                         : 0;
  return run_host<float>(
      M, N, K, A, lda, B, ldb, C, ldc, static_cast<cudaStream_t>(stream),
      /*max_chunks=*/3, /*min_chunk_rows=*/1024, /*max_parts=*/4, head,
      [](int64_t m, int64_t n, int64_t k, const float* a, int64_t la, const float* b,
         int64_t lb, float* c, int64_t lc, const EpiParams& e, cudaStream_t st) {
        return run_f32(m, n, k, a, la, b, lb, c, lc, st, e);
      });
}

gemm_status_t gemm_bf16_f32acc_host(int64_t M, int64_t N, int64_t K,
                                    const uint16_t* A, int64_t lda,
                                    const uint16_t* B, int64_t ldb, float* C,
                                    int64_t ldc, void* stream) {
  return run_host<uint16_t>(
      M, N, K, A, lda, B, ldb, C, ldc, static_cast<cudaStream_t>(stream),
      /*max_chunks=*/4, /*min_chunk_rows=*/512, /*max_parts=*/1, /*head_rows=*/0,
      [](int64_t m, int64_t n, int64_t k, const uint16_t* a, int64_t la,
         const uint16_t* b, int64_t lb, float* c, int64_t lc, const EpiParams& e,
         cudaStream_t st) { return run_bf16(m, n, k, a, la, b, lb, c, lc, st, e); });
}

const char* gemm_status_string(gemm_status_t status) {
  switch (status) {
    case GEMM_OK: return "success";
    case GEMM_ERR_INVALID_ARG: return "invalid argument (size, leading dimension or pointer)";
    case GEMM_ERR_MISALIGNED: return "misaligned operand (reserved: not returned by this library)";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "no CUDA device of compute capability 10.3 (sm_103a) is current";
    case GEMM_ERR_LAUNCH: return "a CUDA call or kernel launch failed";
    case GEMM_ERR_TIMEOUT: return "a device-side bounded wait ran out; the output is incomplete";
    case GEMM_ERR_NO_MEMORY: return "device workspace allocation failed";
    case GEMM_ERR_INTERNAL: return "internal error (tensor map encoding)";
    case GEMM_ERR_SCRATCH_TOO_SMALL: return "the operand copies need more than the fixed no-allocation scratch";
  }
  return "unknown status";
}

gemm_status_t gemm_get_device_status(void* stream) {
  DeviceState* d = nullptr;
  gemm_status_t s = device_state(&d);
  if (s != GEMM_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  unsigned int v = 0;
  e = cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(d->status, 0, sizeof(v));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return (v & 1u) ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

void gemm_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int cur = -1;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (int i = 0; i < kMaxDevices; ++i) {
    DeviceState& d = g_dev[i];
    if (d.pool || d.up || d.down) {
      if (cudaSetDevice(i) == cudaSuccess) {
        cudaDeviceSynchronize();
        for (StreamScratch& x : d.scratch)
          if (x.ptr) cudaFreeAsync(x.ptr, 0);
        cudaDeviceSynchronize();
        if (d.pool) cudaMemPoolDestroy(d.pool);
        if (d.up) cudaStreamDestroy(d.up);
        if (d.down) cudaStreamDestroy(d.down);
      }
    }
    d = DeviceState();
  }
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
}

int gemm_abi_version(void) { return 5; }

int64_t gemm_set_bf16_small_limit(int64_t max_macs) {
  if (max_macs < 0) return -1;
  return g_small_limit.exchange(max_macs);
}

int gemm_set_bf16_schedule(int schedule) {
  if (schedule < GEMM_SCHEDULE_AUTO || schedule > GEMM_SCHEDULE_COLUMN_SPLIT)
    return -1;
  return g_schedule.exchange(schedule);
}

int64_t gemm_pair_units(int64_t M, int64_t N, int64_t K, int32_t max_pairs,
                        int32_t schedule, int32_t pair, int64_t* out,
                        int64_t cap) {
  if (M < 0 || N < 0 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return -1;
  if (max_pairs < 1 || pair < 0 || pair >= max_pairs) return -1;
  if (schedule < GEMM_SCHEDULE_AUTO || schedule > GEMM_SCHEDULE_COLUMN_SPLIT)
    return -1;
  if (cap > 0 && out == nullptr) return -1;
  const PairSchedule ps = pair_schedule(M, N, K, max_pairs, schedule);
  if (pair >= ps.pairs) return 0;
  WorkIter wi;
  wi.init(ps, pair);
  WorkUnit w;
  int64_t n = 0;
  while (wi.next(ps, ps.pairs, w)) {
    if (n < cap) {
      int64_t* o = out + 9 * n;
      o[6] = w.tile >= ps.dp_tiles ? 1 : 0;
      o[7] = w.n_off;
      o[8] = w.width;
      o[0] = w.tile;
      o[1] = w.k0;
      o[2] = w.k1;
      const bool whole = w.k0 == 0 && w.k1 == ps.num_kb;
      if (whole) {
        o[3] = -1;
        o[4] = pair;
        o[5] = 1;
      } else {
        const SkTile st = sk_tile(ps, w.tile);
        o[3] = sk_slot(ps, pair, w.tile);
        o[4] = st.q_first;
        o[5] = st.nseg;
      }
    }
    ++n;
  }
  return n;
}

gemm_status_t gemm_debug_inject(int mode, uint64_t wait_ns) {
  if (mode < 0 || mode > 1) return GEMM_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  const gemm_status_t s = device_state(&d);
  if (s != GEMM_OK) return s;
  const unsigned int words[3] = {static_cast<unsigned int>(mode),
                                 static_cast<unsigned int>(wait_ns & 0xFFFFFFFFull),
                                 static_cast<unsigned int>(wait_ns >> 32)};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(d->status + 1, words, sizeof(words), cudaMemcpyHostToDevice) !=
          cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

uint64_t gemm_launch_count(void) { return g_launches.load(); }

gemm_status_t gemm_tile_order(int64_t tiles_m, int64_t tiles_n, int64_t group,
                              int64_t linear, int64_t* tile_m,
                              int64_t* tile_n) {
  if (tiles_m <= 0 || tiles_n <= 0 || group <= 0 || tiles_m > kMaxDim ||
      tiles_n > kMaxDim || group > kMaxDim || tile_m == nullptr ||
      tile_n == nullptr || linear < 0 || linear >= tiles_m * tiles_n)
    return GEMM_ERR_INVALID_ARG;
  const TileCoord t = tile_order(linear, static_cast<int32_t>(tiles_m),
                                 static_cast<int32_t>(tiles_n),
                                 static_cast<int32_t>(group));
  *tile_m = t.m;
  *tile_n = t.n;
  return GEMM_OK;
}

gemm_status_t gemm_plan_bf16(int64_t M, int64_t N, int64_t K, const void* A,
                             int64_t lda, const void* B, int64_t ldb,
                             const void* C, int64_t ldc, gemm_plan_t* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  return plan_bf16(M, N, K, A, lda, B, ldb, C, ldc, plan);
}

gemm_status_t gemm_plan_f32(int64_t M, int64_t N, int64_t K, const void* A,
                            int64_t lda, const void* B, int64_t ldb,
                            const void* C, int64_t ldc, gemm_plan_t* plan) {
  if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
  return plan_f32(M, N, K, A, lda, B, ldb, C, ldc, plan);
}

}  // extern "C"
