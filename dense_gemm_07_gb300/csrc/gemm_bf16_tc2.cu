// gemm_bf16_tc2.cu -- BF16 x BF16 -> FP32 GEMM on pairs of SMs.
//
// The tensor-core rung of "GEMM, step by step" (section "Concept": BF16
// inputs, FP32 sums, large tiles, neighbouring blocks on the same
// rows/columns; multi-stage prefetch as in "GEMM Optimization", section 5),
// with the output tile grown to 256 x 256 and computed by two SMs together
// ("Production tensor-core kernels use larger tiles", same section of "GEMM,
// step by step").  This kernel serves every M > 128.
//
// Work sharing (stream_k.cuh): whole tiles round-robin over the resident
// pairs while they fill whole waves.  A last wave that fills at most half of
// the pairs runs as 256 x 128 units (an N = 128 pair MMA, one 64-column box
// of B per CTA) on twice as many pairs.  On sm_103a an N = 128 pair MMA
// takes about as long per k-slice as an N = 256 one, so this mainly halves
// the last epilogue (measured: 4 us of 93 at 4096^3).  In a stream-K
// schedule the tiles of the last whole wave and of the partial one are
// instead cut into equal runs of k-slices, one per pair, which every pair
// computes after its whole tiles.  A tile cut into segments is finished by
// the epilogue warp that arrives last on the tile's ticket: the others store
// their partial sums to a workspace and raise a ready flag; the last one
// adds all segments in k order (its own from tensor memory) and applies the
// output step.  No warp waits for work that has not started: a flag is only
// awaited after its writer has taken its ticket.  A tile of two segments
// whose output step is alpha * A.B into a C open to TMA is finished in C
// itself instead: the pair holding its first segment clears the tile's rows
// of C when the kernel starts, and each segment adds its sums there with
// TMA reductions as soon as it is done.  Partial sums move by the
// copy engine; when the finishing unit is the pair's last, its operand ring
// is idle and each warp loads its 32 x 256 partial sums there in one batch.
//
// sm_103a realisation: clusters of two CTAs, one per SM.  CTA r of the pair
// owns rows [128r, 128r+128) of the 256-row tile and stages only those rows
// of A (128 x 64 per k-slice) plus columns [128r, 128r+128) of B (64 x 128);
// one tcgen05.mma.cta_group::2 (M=256, N=256, K=16), issued by the even CTA,
// reads A and B from both CTAs' shared memory and writes each CTA's 128 rows
// of D into that CTA's tensor memory.  Per SM this halves the bytes that
// have to be copied into shared memory per FLOP compared with one SM
// computing a 128 x 256 tile.
//
// Roles (192 threads per CTA):
//   warp 0 (both CTAs)  TMA producer.  Both CTAs' copies count their bytes on
//                       the even CTA's "full" barrier; the even CTA arms it
//                       for 64 KB per stage.
//   warp 1 (even CTA)   MMA issuer: waits on "full", issues 4 pair MMAs per
//                       stage, commits to "empty" in both CTAs, and after the
//                       last slice of a unit to "accumulator full" in both.
//   warps 2-5 (both)    epilogue: TMEM -> registers -> swizzled shared
//                       staging box -> TMA tensor store of C (whole lines;
//                       rows/columns outside C are clipped), or guarded
//                       row stores from the same staging box when C's
//                       layout does not allow TMA;
//                       then arrive on the even CTA's "accumulator empty"
//                       (8 arrivals per unit).
// Tensor memory: NUM_ACC 256-column FP32 accumulators per CTA; with two, a
// unit's epilogue overlaps the next unit's MMAs.  Every wait is bounded; on
// expiry the CTA raises its own and its peer's abort flag and the status
// word, all roles unwind, copies and MMAs in flight are drained, and both
// CTAs meet at a final cluster barrier before tensor memory is released.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "sm103_ptx.cuh"
#include "stream_k.cuh"
#include "tile_order.cuh"

namespace g07 {
namespace {

constexpr int PAIR_M = 256;                       // rows per pair tile
constexpr int CTA_M = 128;                        // rows per CTA
constexpr int BN = 256;                           // columns per pair tile
constexpr int CTA_N = 128;                        // B columns staged per CTA
constexpr int BK = kPairTileK;                    // 64: one 128-byte A row
constexpr int STAGES = kPairStages;               // 6
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
static_assert(BK == kSkSliceK, "stream-K slices are pipeline k-slices");

struct alignas(8) PairControl {
  uint64_t full[STAGES];      // used in the even CTA only
  uint64_t empty[STAGES];
  uint64_t acc_full[NUM_ACC];
  uint64_t acc_empty[NUM_ACC];  // used in the even CTA only (8 arrivals)
  uint64_t drain;
  uint64_t part[EPI_WARPS];     // per epilogue warp: partial-sum box loaded
  uint32_t tmem_base;
  int abort;
};

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

// Producer for one unit of width W: per k-slice in [k0, k1), wait for the
// stage to be free, arm the even CTA's "full" barrier (even CTA only), copy
// this CTA's 128 rows of A and W / 2 columns of B.
template <int W>
__device__ __forceinline__ bool produce_unit(int m0, int n0, int k0, int k1,
                                             Ring& ring, uint8_t* smem,
                                             PairControl* ctl,
                                             const CUtensorMap* tmA,
                                             const CUtensorMap* tmB,
                                             uint32_t rank, int* last_phase,
                                             volatile int* abort, uint64_t tmo,
                                             bool skip_first) {
  constexpr int BOXES = W / 2 / B_BOX_COLS;
  constexpr uint32_t TX = 2u * (A_STAGE_BYTES + BOXES * B_BOX_BYTES);
  const int a_row = m0 + static_cast<int>(rank) * CTA_M;
  const int b_col = n0 + static_cast<int>(rank) * (W / 2);
  for (int kb = k0; kb < k1; ++kb) {
    if (!mbar_wait(&ctl->empty[ring.stage], ring.phase ^ 1u, abort, tmo)) return false;
    if (skip_first && kb == k0) {
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

// MMA issue for k-slices [k0, k1) of one unit of width W into the
// accumulator at d_tmem (the first slice overwrites it).
template <int W>
__device__ __forceinline__ bool mma_unit(uint32_t d_tmem, int k0, int k1,
                                         Ring& ring, uint8_t* smem,
                                         PairControl* ctl,
                                         volatile int* abort, uint64_t tmo) {
  constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_M, W, /*a_mn_major=*/false,
                                            /*b_mn_major=*/true);
  for (int kb = k0; kb < k1; ++kb) {
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
      mma_f16_ss_pair(d_tmem, adesc, bdesc, IDESC,
                      (kb != k0 || kk != 0) ? 1u : 0u);
    }
    mma_commit_pair(&ctl->empty[ring.stage], 0x3);
    ring.advance();
  }
  return true;
}

// ------------------------------------------------------ stream-K fix-up
//
// Partial sums live in an FP32 workspace of 256 columns whose rows are, per
// stream-K pair q, slot (0: its first segment, 1: its last), CTA rank and
// epilogue warp, the warp's 32 rows of the accumulator:
//   row = ((q * 2 + slot) * 2 + rank) * 128 + warp * 32 + lane.
// It is read and written in 32 x 32 boxes by the copy engine (tensor map
// tmW, same box and swizzle as C's).
__device__ __forceinline__ int sk_row(int q, int slot, uint32_t rank, int wq) {
  return ((q * 2 + slot) * 2 + static_cast<int>(rank)) * CTA_M + wq * 32;
}

// Synchronisation words, 64-bit, tagged with the launch so that nothing has
// to be cleared between launches: ticket counters [sk_tiles][rank 2][warp 4]
// hold (tag << 8) | arrivals, ready flags [sk_pairs][slot 2][rank 2][warp 4]
// hold the tag once the slot's partial sums are stored.  A word with another
// tag counts as zero.  The finishing warp of a tile also puts its ticket and
// the flags it consumed back to zero, so a launch replayed with the same tag
// (a CUDA graph) starts from clean words.
__device__ __forceinline__ unsigned long long* sk_ticket(
    unsigned long long* sync, const PairSchedule& s, int tile, uint32_t rank,
    int wq) {
  return sync + (static_cast<int64_t>(tile - s.dp_tiles) * 2 + rank) * 4 + wq;
}
__device__ __forceinline__ unsigned long long* sk_ready(
    unsigned long long* sync, const PairSchedule& s, int q, int slot,
    uint32_t rank, int wq) {
  return sync + static_cast<int64_t>(s.sk_tiles) * 8 +
         ((static_cast<int64_t>(q) * 2 + slot) * 2 + rank) * 4 + wq;
}

// Take this launch's next ticket of a counter (0 = first arrival).  At most
// kSkMaxSeg warps contend, so the exchange loop ends after a few rounds; it
// is bounded all the same (-1: gave up).
__device__ __forceinline__ int sk_take_ticket(unsigned long long* w,
                                              unsigned long long tag) {
  unsigned long long cur = atomicAdd(w, 0ull);
  for (int i = 0; i < 1024; ++i) {
    const bool same = (cur >> 8) == tag;
    const unsigned long long want = same ? cur + 1 : ((tag << 8) | 1ull);
    const unsigned long long prev = atomicCAS(w, cur, want);
    if (prev == cur) return same ? static_cast<int>(cur & 0xFFull) : 0;
    cur = prev;
  }
  return -1;
}

// Wait (bounded) until a ready flag holds this launch's tag.
__device__ __forceinline__ bool sk_wait_ready(const unsigned long long* f,
                                              unsigned long long tag,
                                              volatile int* abort,
                                              uint64_t limit_ns) {
  if (ld_acquire_gpu_u64(f) == tag) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire_gpu_u64(f) == tag) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// What the finishing warp needs to add up one tile's segments.
struct SkCombine {
  const CUtensorMap* tmW;
  const PairSchedule* sched;
  int tile, q_first, nseg, mine;
  uint32_t rank;
  int wq;
  uint64_t* bar;        // this warp's "partial box loaded" barrier
  uint32_t* bar_uses;   // its completed phases
  volatile int* abort;
  uint64_t tmo;
  // Two segments, loaded in advance: the other segment's 8 boxes (one per
  // 32-column chunk, 4 KB each, as the copy engine lays them out), or null
  // to load each box when its chunk is combined.
  const uint8_t* stash;
};

// Row `lane` of a swizzled 32 x 32 FP32 staging box (the layout both the
// epilogue writes and TMA loads produce).
__device__ __forceinline__ void box_read_row(const uint8_t* buf, int lane,
                                             float (&v)[32]) {
  const uint8_t* rowp = buf + lane * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 x = *reinterpret_cast<const float4*>(rowp + ((j ^ (lane & 7)) << 4));
    v[4 * j] = x.x;
    v[4 * j + 1] = x.y;
    v[4 * j + 2] = x.z;
    v[4 * j + 3] = x.w;
  }
}

// Replace this lane's 32 accumulator values of column chunk c by the sum of
// every segment's values in segment (k) order, loading the other segments'
// boxes through `buf` (free on entry).  False: a wait ran out.
__device__ __forceinline__ bool combine_chunk(uint32_t (&r)[32],
                                              const SkCombine& cb, int c,
                                              uint8_t* buf, int lane) {
  if (cb.nseg == 2 && cb.stash) {
    // Two segments, the other's already in shared memory: a + b == b + a
    // exactly, so adding it to this segment's sums gives the k-order sum.
    float v[32];
    box_read_row(cb.stash + c * EPI_BOX_BYTES, lane, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + v[i]);
    return true;
  }
  float acc[32];
#pragma unroll 1
  for (int s = 0; s < cb.nseg; ++s) {
    float v[32];
    if (s == cb.mine) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    } else if (cb.stash) {
      box_read_row(cb.stash + c * EPI_BOX_BYTES, lane, v);
    } else {
      const int q = cb.q_first + s;
      const uint32_t parity = *cb.bar_uses & 1u;
      if (lane == 0) {
        mbar_arrive_expect_tx(cb.bar, EPI_BOX_BYTES);
        tma_load_2d(buf, cb.tmW, cb.bar, c * 32,
                    sk_row(q, sk_slot(*cb.sched, q, cb.tile), cb.rank, cb.wq));
      }
      ++*cb.bar_uses;
      int ok = 0;
      if (lane == 0) ok = mbar_wait(cb.bar, parity, cb.abort, cb.tmo) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return false;
      box_read_row(buf, lane, v);
      // all lanes have read the box before the copy engine refills it
      fence_proxy_async_smem();
      __syncwarp();
    }
    if (s == 0) {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = v[i];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] += v[i];
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(acc[i]);
  return true;
}

// ------------------------------------------------------------ output step

// Epilogue of one unit through shared memory and TMA stores: per 32-column
// chunk the warp writes its 32 x 32 block into a 128-byte-swizzled staging
// box (each lane one row, conflict-free 16-byte stores) and one lane stores
// the box with the copy engine, which writes whole lines and clips rows and
// columns outside the tensor.  Two staging boxes per warp alternate.  With
// cb set, each chunk is first combined with the other segments' partial
// sums (loaded into the same box); tmOut is C's map, or the workspace's
// when a segment leaves its partial sums (identity epilogue, M = N = the
// workspace's extent).  With `reduce`, the boxes are added to tmOut's
// elements instead of stored.  W: the unit's width.  False: a wait ran out.
template <int W, bool GELU>
__device__ __forceinline__ bool store_unit_tma(uint32_t taddr,
                                               const CUtensorMap* tmOut,
                                               uint8_t* ebuf, int row0, int n0,
                                               int M, int N, int lane,
                                               int& chunk, const float* C,
                                               int64_t ldc,
                                               const EpiParams& epi,
                                               const SkCombine* cb,
                                               bool reduce = false,
                                               uint8_t* wide = nullptr) {
#pragma unroll 1
  for (int c = 0; c < W / 32; ++c) {
    // Boxes wholly outside C are skipped (warp-uniform test); every other
    // chunk issues exactly one store group, which the buffer alternation
    // below relies on.
    if (row0 >= M || n0 + c * 32 >= N) continue;
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    uint8_t* buf;
    if (wide) {
      buf = wide + c * EPI_BOX_BYTES;  // a box per chunk: nothing to wait for
    } else {
      buf = ebuf + (chunk++ & 1) * EPI_BOX_BYTES;
      if (lane == 0) bulk_wait_read<1>();  // the box's previous store has read it
    }
    __syncwarp();
    tmem_ld_wait();
    if (cb && !combine_chunk(r, *cb, c, buf, lane)) return false;
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
          r[j + e] = __float_as_uint(epi_apply<GELU>(
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
      if (reduce)
        tma_reduce_add_2d(tmOut, buf, n0 + c * 32, row0);
      else
        tma_store_2d(tmOut, buf, n0 + c * 32, row0);
      bulk_commit();
    }
  }
  return true;
}

// (wide: W / 32 staging boxes of this warp's own, one per chunk, so no chunk
// waits for an earlier store to have read its box; used for a pair's last
// unit, whose operand ring is idle.)

// Epilogue of one unit when C's layout does not allow TMA stores (a row
// stride that is not a multiple of 16 bytes, or an unaligned base).  Per
// 32-column chunk the warp writes its 32 x 32 block into a swizzled staging
// box with one row per lane, as the TMA path does, then reads it back by
// columns and stores it one row at a time: lane j writes column j, so each
// store instruction writes 128 contiguous bytes (the fused epilogue's reads
// of C and of the bias are coalesced the same way).  With cb set, each chunk
// is first combined with the other segments' partial sums, loaded through
// the same box.  False: a wait ran out.
template <int W, bool GELU>
__device__ __forceinline__ bool store_unit_rows(uint32_t taddr, float* C,
                                                int64_t ldc, int row0, int n0,
                                                int M, int N,
                                                const EpiParams& epi,
                                                const SkCombine* cb,
                                                uint8_t* ebuf, int lane,
                                                int& chunk) {
  const bool plain = epi.alpha == 1.0f && epi.beta == 0.0f && epi.bias == nullptr &&
                     epi.act == 0;
  const int rows = M - row0 < 32 ? M - row0 : 32;
#pragma unroll 1
  for (int c = 0; c < W / 32; ++c) {
    if (rows <= 0 || n0 + c * 32 >= N) continue;
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    uint8_t* buf = ebuf + (chunk++ & 1) * EPI_BOX_BYTES;
    // the box may still be read by an earlier TMA store of this warp (the
    // partial sums of a stream-K segment)
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    tmem_ld_wait();
    if (cb && !combine_chunk(r, *cb, c, buf, lane)) return false;
    uint8_t* rowp = buf + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
          make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    __syncwarp();
    const int gn = n0 + c * 32 + lane;
    if (gn < N) {
      const float bias = epi.bias != nullptr ? epi.bias[gn] : 0.0f;
      // column `lane` of box row rr: 16-byte group lane / 4, swizzled by rr
      const uint32_t in_group = static_cast<uint32_t>(lane & 3) * 4;
      const uint32_t group = static_cast<uint32_t>(lane >> 2);
      float* cp = C + static_cast<int64_t>(row0) * ldc + gn;
#pragma unroll 4
      for (int rr = 0; rr < rows; ++rr) {
        const float v = *reinterpret_cast<const float*>(
            buf + rr * 128 + (((group ^ static_cast<uint32_t>(rr & 7)) << 4) | in_group));
        float* dst = cp + static_cast<int64_t>(rr) * ldc;
        *dst = plain ? v : epi_apply<GELU>(epi, v, epi.beta != 0.0f ? *dst : 0.0f, bias);
      }
    }
    // every lane has read the box before it is written again, by this
    // loop's generic stores or by the copy engine (partial-sum loads)
    fence_proxy_async_smem();
    __syncwarp();
  }
  return true;
}

// The same for a pair's last unit, whose operand ring is idle: all W / 32
// chunks are first staged, each in a box of this warp's own in `wide` (no
// chunk waits for another's stores), then the rows are stored chunk after
// chunk with nothing between the stores.  Never a stream-K finish.
template <int W, bool GELU>
__device__ __forceinline__ void store_unit_rows_wide(uint32_t taddr, float* C, int64_t ldc,
                                                     int row0, int n0, int M, int N,
                                                     const EpiParams& epi, uint8_t* wide,
                                                     int lane) {
  const bool plain = epi.alpha == 1.0f && epi.beta == 0.0f && epi.bias == nullptr &&
                     epi.act == 0;
  const int rows = M - row0 < 32 ? M - row0 : 32;
  if (rows <= 0) return;
  int chunks = 0;  // chunks with columns inside C
#pragma unroll 1
  for (int c = 0; c < W / 32; ++c) {
    if (n0 + c * 32 >= N) break;
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr + c * 32, r);
    tmem_ld_wait();
    uint8_t* rowp = wide + c * EPI_BOX_BYTES + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
          make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    ++chunks;
  }
  __syncwarp();
  // column `lane` of a box row rr: 16-byte group lane / 4, swizzled by rr
  const uint32_t in_group = static_cast<uint32_t>(lane & 3) * 4;
  const uint32_t group = static_cast<uint32_t>(lane >> 2);
#pragma unroll 1
  for (int c = 0; c < chunks; ++c) {
    const int gn = n0 + c * 32 + lane;
    if (gn >= N) continue;
    const float bias = epi.bias != nullptr ? epi.bias[gn] : 0.0f;
    const uint8_t* box = wide + c * EPI_BOX_BYTES;
    float* cp = C + static_cast<int64_t>(row0) * ldc + gn;
#pragma unroll 8
    for (int rr = 0; rr < rows; ++rr) {
      const float v = *reinterpret_cast<const float*>(
          box + rr * 128 + (((group ^ static_cast<uint32_t>(rr & 7)) << 4) | in_group));
      float* dst = cp + static_cast<int64_t>(rr) * ldc;
      *dst = plain ? v : epi_apply<GELU>(epi, v, epi.beta != 0.0f ? *dst : 0.0f, bias);
    }
  }
}

// GELU: whether the GELU activation is compiled in (epi_apply); the copy
// without it serves every other epilogue.
template <bool GELU>
__global__ void __launch_bounds__(THREADS, 1)
gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmW,
                      float* __restrict__ C, int64_t ldc, int M, int N,
                      const PairSchedule sched,
                      unsigned long long* __restrict__ sk_sync,
                      unsigned long long sk_tag, int tma_c,
                      unsigned int* __restrict__ status, EpiParams epi) {
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
    for (int w = 0; w < EPI_WARPS; ++w) mbar_init(&ctl->part[w], 1);
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
  // Set-up done (it touched no global memory): wait for the kernels before
  // this one, and let the next one be scheduled as SMs free up.
  grid_dependency_wait();
  grid_dependents_go();
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
      WorkIter wi;
      wi.init(sched, pair);
      WorkUnit w;
      for (bool first = true; ok && wi.next(sched, num_pairs, w); first = false) {
        const TileCoord tc = tile_order(w.tile, sched.tiles_m, sched.tiles_n, GROUP);
        const int m0 = tc.m * PAIR_M, n0 = tc.n * BN + w.n_off;
        const bool skip = fault == 1 && first;
        ok = w.width == BN
                 ? produce_unit<BN>(m0, n0, w.k0, w.k1, ring, smem, ctl, &tmA, &tmB,
                                    rank, last_phase, abort, tmo, skip)
                 : produce_unit<BN / 2>(m0, n0, w.k0, w.k1, ring, smem, ctl, &tmA,
                                        &tmB, rank, last_phase, abort, tmo, skip);
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
      WorkIter wi;
      wi.init(sched, pair);
      WorkUnit w;
      for (int t = 0; ok && wi.next(sched, num_pairs, w); ++t) {
        const int acc = t % NUM_ACC;
        const uint32_t acc_phase = static_cast<uint32_t>(t / NUM_ACC) & 1u;
        if (!pair_wait(&ctl->acc_empty[acc], acc_phase ^ 1u, abort, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        issued |= w.k1 > w.k0;
        ok = w.width == BN
                 ? mma_unit<BN>(d_tmem, w.k0, w.k1, ring, smem, ctl, abort, tmo)
                 : mma_unit<BN / 2>(d_tmem, w.k0, w.k1, ring, smem, ctl, abort, tmo);
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
    uint32_t part_uses = 0;
    WorkIter wi;
    wi.init(sched, pair);
    // Tiles cut into two segments, with C open to TMA and no term besides
    // alpha * A.B, are finished directly in C: each segment adds its sums
    // there with TMA reductions, so those rows of C must read zero first.
    // The pair holding a tile's first segment clears its rows of the tile
    // before its first unit and raises its ready flag; the other segment's
    // warp waits for that flag before it adds.  (0 + a) + b == (0 + b) + a,
    // so the bits do not depend on which segment finishes first, and neither
    // waits for the other's MMAs.
    const bool direct_ok = tma_c && epi.beta == 0.0f && epi.bias == nullptr && epi.act == 0;
    if (direct_ok && pair < sched.sk_pairs) {
      const int64_t I = sk_total(sched);
      const int64_t b0 = sk_begin(pair, sched.sk_pairs, I);
      const int64_t b1 = sk_begin(pair + 1, sched.sk_pairs, I);
      // A first segment of a two-segment tile ends this pair's range.
      const int tile = sched.dp_tiles + static_cast<int>((b1 > b0 ? b1 - 1 : b0) / sched.num_kb);
      const SkTile st = b1 > b0 ? sk_tile(sched, tile) : SkTile{-1, 0};
      if (st.q_first == pair && st.nseg == 2) {
        const TileCoord tc = tile_order(tile, sched.tiles_m, sched.tiles_n, GROUP);
        const int row0 = tc.m * PAIR_M + static_cast<int>(rank) * CTA_M + q * 32;
        const int n0 = tc.n * BN;
        uint4* zrow = reinterpret_cast<uint4*>(ebuf + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j) zrow[j] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (row0 < M)
            for (int c = 0; c < BN / 32; ++c)
              if (n0 + c * 32 < N) tma_store_2d(&tmC, ebuf, n0 + c * 32, row0);
          bulk_commit();
          // The zeros are in C (and the box is free again) before the flag
          // says so.
          bulk_wait_all();
          fence_proxy_async_global();
          __threadfence();
          st_release_gpu_u64(sk_ready(sk_sync, sched, pair, sk_slot(sched, pair, tile), rank, q),
                             sk_tag);
        }
        __syncwarp();
      }
    }
    WorkUnit w;
    for (int t = 0; wi.next(sched, num_pairs, w); ++t) {
      const int acc = t % NUM_ACC;
      const uint32_t acc_phase = static_cast<uint32_t>(t / NUM_ACC) & 1u;
      WorkIter peek = wi;
      WorkUnit after;
      const bool last_unit = !peek.next(sched, num_pairs, after);
      // Everything that depends only on the unit is done while its MMAs
      // run: coordinates, the split-tile lookup and, for a segment finished
      // in C, the wait for the tile's cleared rows.
      const TileCoord tc = tile_order(w.tile, sched.tiles_m, sched.tiles_n, GROUP);
      const int m0 = tc.m * PAIR_M, n0 = tc.n * BN + w.n_off;
      const int row = m0 + static_cast<int>(rank) * CTA_M + q * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int row0 = row - lane;
      const bool segment = w.k0 != 0 || w.k1 != sched.num_kb;
      const SkTile st = segment ? sk_tile(sched, w.tile) : SkTile{pair, 1};
      const bool in_c = segment && direct_ok && st.nseg == 2;
      int ok = 1;
      if (in_c && lane == 0 && pair != st.q_first) {
        // A segment finished directly in C (above): it may add once the
        // tile's rows of C have been cleared.
        unsigned long long* f =
            sk_ready(sk_sync, sched, st.q_first, sk_slot(sched, st.q_first, w.tile), rank, q);
        ok = sk_wait_ready(f, sk_tag, abort, tmo) ? 1 : 0;
        // the flag was read by this thread; C will be updated by the copy
        // engine
        fence_proxy_async_global();
        // the only reader of this flag puts it back to zero for a replay of
        // this launch with the same tag
        if (ok) *f = 0ull;
      }
      if (lane == 0 && ok) ok = pair_wait(&ctl->acc_full[acc], acc_phase, abort, tmo) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) raise_abort(abort, peer_abort, status);
        break;
      }
      tc_fence_after_sync();

      int ready_slot = -1;  // >= 0: this segment's flag goes up after its stores
      SkCombine cb;
      const SkCombine* cbp = nullptr;
      bool reduce_c = in_c;  // add this segment into C (cleared at the start)
      bool good = true;
      if (segment && !in_c) {
        // A stream-K segment: take a ticket; the last of the tile's
        // segments finishes it, the others leave their partial sums.
        int ticket = 0;
        if (lane == 0)
          ticket = sk_take_ticket(sk_ticket(sk_sync, sched, w.tile, rank, q), sk_tag);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket < 0) {
          good = false;
        } else if (ticket + 1 < st.nseg) {
          ready_slot = sk_slot(sched, pair, w.tile);
          good = store_unit_tma<BN, GELU>(taddr, &tmW, ebuf, sk_row(pair, ready_slot, rank, q),
                                          0, 0x7FFFFFFF, BN, lane, chunk, nullptr, 0,
                                          epi_identity(), nullptr);
        } else {
          cb.tmW = &tmW;
          cb.sched = &sched;
          cb.tile = w.tile;
          cb.q_first = st.q_first;
          cb.nseg = st.nseg;
          cb.mine = pair - st.q_first;
          cb.rank = rank;
          cb.wq = q;
          cb.bar = &ctl->part[q];
          cb.bar_uses = &part_uses;
          cb.abort = abort;
          cb.tmo = tmo;
          cb.stash = nullptr;
          // Every other segment's writer has taken its ticket, so it is
          // running; wait (bounded) until its partial sums are stored.
          int got = 1;
          if (lane == 0) {
            for (int sg = 0; got && sg < st.nseg; ++sg) {
              if (sg == cb.mine) continue;
              const int qq = st.q_first + sg;
              got = sk_wait_ready(sk_ready(sk_sync, sched, qq, sk_slot(sched, qq, w.tile), rank, q),
                                  sk_tag, abort, tmo) ? 1 : 0;
            }
            // the flags were read by this thread; the boxes will be read by
            // the copy engine
            fence_proxy_async_global();
            if (got) {
              // Every segment has taken its ticket and raised its flag: put
              // the words back to zero, so that a replay of this launch
              // (same tag, e.g. from a CUDA graph) finds them clean.
              *sk_ticket(sk_sync, sched, w.tile, rank, q) = 0ull;
              for (int sg = 0; sg < st.nseg; ++sg)
                if (sg != cb.mine) {
                  const int qq = st.q_first + sg;
                  *sk_ready(sk_sync, sched, qq, sk_slot(sched, qq, w.tile), rank, q) = 0ull;
                }
            }
          }
          got = __shfl_sync(0xffffffffu, got, 0);
          good = got != 0;
          if (good && last_unit && st.nseg == 2) {
            // This CTA's operand ring is idle: every MMA of the pair has
            // completed (this unit's accumulator is full) and no copy is
            // left to issue.  Load the other segment's 8 boxes at once into
            // this warp's 32 KB of it.
            uint8_t* stash = smem + q * (BN / 32) * EPI_BOX_BYTES;
            const int oq = st.q_first + (1 - cb.mine);
            const int orow = sk_row(oq, sk_slot(sched, oq, w.tile), rank, q);
            const uint32_t parity = part_uses & 1u;
            if (lane == 0) {
              mbar_arrive_expect_tx(&ctl->part[q], (BN / 32) * EPI_BOX_BYTES);
              for (int c = 0; c < BN / 32; ++c)
                tma_load_2d(stash + c * EPI_BOX_BYTES, &tmW, &ctl->part[q], c * 32, orow);
            }
            ++part_uses;
            int ld = 0;
            if (lane == 0) ld = mbar_wait(&ctl->part[q], parity, abort, tmo) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, ld, 0) != 0;
            cb.stash = stash;
          }
          cbp = &cb;
        }
      }
      // The pair's last unit: its operand ring is idle (every MMA of the
      // pair has completed and no copy is left to issue), so unless it holds
      // the other segment's sums, this warp's quarter of it stages a box per
      // chunk.
      uint8_t* wide = last_unit && cbp == nullptr ? smem + q * (BN / 32) * EPI_BOX_BYTES : nullptr;
      if (good && ready_slot < 0) {
        if (w.width != BN) {
          // a column-split unit of the last wave (never a stream-K segment)
          if (tma_c)
            store_unit_tma<BN / 2, GELU>(taddr, &tmC, ebuf, row0, n0, M, N, lane,
                                   chunk, C, ldc, epi, nullptr, false, wide);
          else if (wide)
            store_unit_rows_wide<BN / 2, GELU>(taddr, C, ldc, row0, n0, M, N, epi, wide, lane);
          else
            store_unit_rows<BN / 2, GELU>(taddr, C, ldc, row0, n0, M, N, epi, nullptr,
                                    ebuf, lane, chunk);
        } else if (tma_c) {
          good = store_unit_tma<BN, GELU>(taddr, &tmC, ebuf, row0, n0, M, N, lane, chunk, C,
                                          ldc, epi, cbp, reduce_c, wide);
        } else if (wide) {
          store_unit_rows_wide<BN, GELU>(taddr, C, ldc, row0, n0, M, N, epi, wide, lane);
        } else {
          good = store_unit_rows<BN, GELU>(taddr, C, ldc, row0, n0, M, N, epi, cbp, ebuf,
                                           lane, chunk);
        }
      }
      if (!good) {
        if (lane == 0) raise_abort(abort, peer_abort, status);
        break;
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(map_to_rank(smem_u32(&ctl->acc_empty[acc]), 0));
        if (ready_slot >= 0) {
          // The segment's sums are in global memory (copies complete)
          // before the flag says so.
          bulk_wait_all();
          fence_proxy_async_global();
          __threadfence();
          st_release_gpu_u64(sk_ready(sk_sync, sched, pair, ready_slot, rank, q), sk_tag);
        }
      }
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

// Per device: 0 until the shared-memory attribute is set and the occupancy
// known, then the number of resident pairs + 1.  One atomic word, so that
// a thread that finds it set also finds the attribute set (calls may come
// from several host threads at once).
std::atomic<int> g_pairs_plus1[64];

}  // namespace

size_t pair_smem_bytes() {
  return 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + EPI_BYTES +
         sizeof(PairControl);
}

int pair_max_active(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int known = g_pairs_plus1[dev].load(std::memory_order_acquire);
  if (known > 0) return known - 1;
  {
    const size_t smem = pair_smem_bytes();
    if (cudaFuncSetAttribute(gemm_bf16_pair_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_bf16_pair_kernel<true>,
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
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_bf16_pair_kernel<false>, &cfg) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    g_pairs_plus1[dev].store(clusters + 1, std::memory_order_release);
    return clusters;
  }
}

cudaError_t launch_gemm_bf16_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const CUtensorMap* tmC, const CUtensorMap* tmW,
                                  float* C, int64_t ldc, int M, int N,
                                  const PairSchedule& sched,
                                  unsigned long long* sk_sync,
                                  unsigned long long sk_tag,
                                  unsigned int* status, const EpiParams& epi,
                                  cudaStream_t stream) {
  if (sched.pairs <= 0) return cudaErrorInvalidValue;
  if (sched.sk_tiles > 0 &&
      (tmW == nullptr || sk_sync == nullptr || sk_tag == 0 || (sk_tag >> 56) != 0))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.gridDim = dim3(static_cast<unsigned>(2 * sched.pairs), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes();
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  const cudaError_t e =
      epi.act == kActGelu
          ? cudaLaunchKernelEx(&cfg, gemm_bf16_pair_kernel<true>, tmA, tmB,
                               tmC ? *tmC : unused, tmW ? *tmW : unused, C, ldc, M, N,
                               sched, sk_sync, sk_tag, tmC ? 1 : 0, status, epi)
          : cudaLaunchKernelEx(&cfg, gemm_bf16_pair_kernel<false>, tmA, tmB,
                               tmC ? *tmC : unused, tmW ? *tmW : unused, C, ldc, M, N,
                               sched, sk_sync, sk_tag, tmC ? 1 : 0, status, epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace g07
