// stream_k.cuh -- how the paired-SM BF16 kernel shares its work among the
// resident pairs: whole tiles in full waves, and a partial last wave either
// split along N (each tile as two 256 x 128 units on twice as many pairs)
// or, in stream-K schedules, split along K.
//
// Stream-K part ("GEMM Optimization", section "L2 Cache and Wave Analysis":
// a partial last wave leaves SMs idle; spreading the k-iterations of the
// last tiles evenly over the SMs removes that tail): the
// I = sk_tiles * num_kb k-slices of tiles [dp_tiles, dp_tiles + sk_tiles),
// taken tile after tile and k-slice after k-slice, are cut into sk_pairs
// contiguous ranges of nearly equal length; pair p computes the slices
// [sk_begin(p), sk_begin(p + 1)).  A tile whose slices fall into several
// ranges is finished by combining the partial sums of its segments in
// segment order (k order), so the result does not depend on timing.
//
// Data-parallel part: tiles [0, dp_tiles) of the tile order as units, pair p
// taking units p, p + pairs, p + 2 * pairs, ...: tiles [0, num_full) whole,
// each later one as `split` units of 256 / split columns.
//
// Each pair does its data-parallel units first and its stream-K range last.
// When the ranges span several tiles, a split tile's first segment is the
// end of one pair's range and its second the start of the next pair's: the
// second is computed early and leaves its partial sums, the first is
// computed last and adds them, as the pair's final unit, when its operand
// ring is idle and can hold them.  When each tile is halved over two pairs,
// both halves are their pairs' final units and run at the same time; the
// later one to finish adds them.
//
// Everything here is plain integer arithmetic shared by the kernel and by
// the host (planning, and a host-side listing used by the tests).
#pragma once

#include <cstdint>

namespace g07 {

struct PairSchedule {
  int tiles_m = 0, tiles_n = 0;
  int num_kb = 0;     // k-slices per tile
  int dp_tiles = 0;   // tiles computed by single pairs, round-robin
  int num_full = 0;   // of those, tiles [0, num_full) at full width
  int split = 1;      // the rest as `split` column units (1 or 2)
  int sk_tiles = 0;   // tiles after them, split by k-slices
  int sk_pairs = 0;   // pairs sharing the stream-K slices (pairs [0, sk_pairs))
  int pairs = 0;      // pairs launched
};

// How the last, partial wave is shared.
enum PairScheduleMode {
  kScheduleAuto = 0,     // the estimated fastest (pair_schedule_cost)
  kScheduleStreamK = 1,  // stream-K wherever it applies
  kScheduleNoSplitK = 2  // never stream-K (column split only)
};

// Depth of one k-slice (the kernel's pipeline stage).
constexpr int kSkSliceK = 64;

// Most segments one stream-K tile can be split into (the planner keeps every
// range at least half a tile long, which bounds it by 3; whole-wave
// schedules and aligned halves give 2).
constexpr int kSkMaxSeg = 3;
// Shortest k extent (in slices) worth splitting at all.
constexpr int kSkMinSlices = 8;

__host__ __device__ inline int64_t sk_total(const PairSchedule& s) {
  return static_cast<int64_t>(s.sk_tiles) * s.num_kb;
}

// First stream-K slice of pair p (p in [0, sk_pairs]; p == sk_pairs gives I).
__host__ __device__ inline int64_t sk_begin(int p, int P, int64_t I) {
  return static_cast<int64_t>(p) * I / P;
}

// The pair whose range holds slice x (0 <= x < I): the largest p with
// sk_begin(p) <= x, i.e. p * I < (x + 1) * P.
__host__ __device__ inline int sk_owner(int64_t x, int P, int64_t I) {
  return static_cast<int>(((x + 1) * P + I - 1) / I - 1);
}

// One unit of work: k-slices [k0, k1) of columns [n_off, n_off + width) of
// tile `tile` (tile-order index).
struct WorkUnit {
  int tile;
  int k0, k1;
  int n_off, width;
};

// Walks one pair's units: its data-parallel units, then its stream-K range.
struct WorkIter {
  int next_dp;
  int64_t it, end;  // stream-K range [it, end) still to walk, from the end

  __host__ __device__ void init(const PairSchedule& s, int pair) {
    next_dp = pair;
    if (pair < s.sk_pairs) {
      const int64_t I = sk_total(s);
      it = sk_begin(pair, s.sk_pairs, I);
      end = sk_begin(pair + 1, s.sk_pairs, I);
    } else {
      it = end = 0;
    }
  }

  __host__ __device__ bool next(const PairSchedule& s, int num_pairs, WorkUnit& u) {
    const int units = s.num_full + (s.dp_tiles - s.num_full) * s.split;
    if (next_dp < units) {
      const int v = next_dp;
      next_dp += num_pairs;
      u.k0 = 0;
      u.k1 = s.num_kb;
      if (v < s.num_full) {
        u.tile = v;
        u.n_off = 0;
        u.width = 256;
      } else {
        u.tile = s.num_full + (v - s.num_full) / s.split;
        u.width = 256 / s.split;
        u.n_off = ((v - s.num_full) % s.split) * u.width;
      }
      return true;
    }
    if (end > it) {
      // The range is walked from its end: its last tile first, from k = 0,
      // so that the pairs start their runs in step along K (their first
      // slices are shared in L2, as whole tiles' are) rather than each at
      // its own depth.
      const int64_t t = (end - 1) / s.num_kb;
      const int64_t x0 = t * s.num_kb;
      const int64_t lo = it > x0 ? it : x0;
      u.tile = s.dp_tiles + static_cast<int>(t);
      u.k0 = static_cast<int>(lo - x0);
      u.k1 = static_cast<int>(end - x0);
      u.n_off = 0;
      u.width = 256;
      end = lo;
      return true;
    }
    return false;
  }
};

// The segments of stream-K tile `tile`: pairs q_first .. q_first + nseg - 1
// hold its slices, in k order.
struct SkTile {
  int q_first;
  int nseg;
};

__host__ __device__ inline SkTile sk_tile(const PairSchedule& s, int tile) {
  const int64_t I = sk_total(s);
  const int64_t x0 = static_cast<int64_t>(tile - s.dp_tiles) * s.num_kb;
  SkTile r;
  r.q_first = sk_owner(x0, s.sk_pairs, I);
  r.nseg = sk_owner(x0 + s.num_kb - 1, s.sk_pairs, I) - r.q_first + 1;
  return r;
}

// Which of pair q's two partial-sum slots its segment of `tile` uses: 0 when
// the segment is the first of q's range, 1 when it is the last (a range
// holds at most one partial segment at each end; one lying inside a single
// tile is its first).
__host__ __device__ inline int sk_slot(const PairSchedule& s, int q, int tile) {
  const int64_t x0 = static_cast<int64_t>(tile - s.dp_tiles) * s.num_kb;
  return sk_begin(q, s.sk_pairs, sk_total(s)) >= x0 ? 0 : 1;
}

// Plan for an M x N x K problem with 256 x 256 tiles, 64-deep k-slices and
// `max_pairs` (P) resident pairs.  With W whole waves and a last wave of T
// tiles (0 < T):
//   column split (every mode but kScheduleStreamK, when 2T <= P): the T
//     tiles run as 2T units of 256 x 128;
//   stream-K (kScheduleStreamK):
//   - W >= 1: the last whole wave and the partial one (P + T tiles) are
//     shared by all P pairs after W - 1 whole waves (at least a tile's worth
//     each, so a tile has at most two segments);
//   - W == 0: each tile is halved over 2T pairs (if 2T <= P);
//   halving (kScheduleAuto only): each tile of the last wave is halved along
//     K over 2T pairs (2T <= P), after the W whole waves;
//   kScheduleAuto takes whichever of these (or the plain or column-split
//     last wave) has the lowest estimated time, pair_schedule_cost().
// A last wave more than 85 % full, or fewer than kSkMinSlices k-slices, is
// never split along K.
// Estimated time of a schedule in units of one k-slice of one pair (about
// 0.3 us on a GB300), for W whole waves of P pairs, a last wave of T tiles
// and kb k-slices per tile, fitted to measurements of the paired kernel: a
// 256 x 128 unit takes as long as a whole tile (operand delivery, not the
// MMA, paces it), so the column split saves only epilogue time.  Finishing
// a tile halved along K costs about 20 + kb / 16 slices after its main loop
// when the halves are added in C itself (in_c: two segments, a plain
// alpha * A.B output step and a C open to TMA), 58 when they meet in the
// partial-sum workspace; a stream-K run over the last whole wave and the
// partial one costs 38 + kb / 16 slices, or 75 + kb / 16 through the
// workspace (its pairs' runs end at different k, so fewer operand reads are
// shared in L2 near the end, and the shortest segments pay a tile's
// start-up).
enum PairScheduleKind { kPlainTail = 0, kColumnTail = 1, kHalvedTail = 2, kStreamKTail = 3 };
inline int64_t pair_schedule_cost(int kind, int64_t W, int64_t T, int64_t P, int64_t kb,
                                  bool in_c) {
  switch (kind) {
    case kPlainTail: return (W + 1) * kb + 16;
    case kColumnTail: return (W + 1) * kb + 8;
    case kHalvedTail: return W * kb + (kb + 1) / 2 + (in_c ? 20 + kb / 16 : 58);
    default:
      return (W - 1) * kb + ((P + T) * kb + P - 1) / P +
             (in_c ? 38 + kb / 16 : 75 + kb / 16);
  }
}

// Operands larger than this (bytes of A and B) are not shared out as
// stream-K runs by the automatic schedule: with pairs at different k, L2 no
// longer holds what they read (2048 x 4096 x 11008, 135 MB: 138 against
// 116 us for whole tiles).
constexpr int64_t kSkAutoMaxOperandBytes = 96ll << 20;

// in_c: tiles cut into two segments can be finished in C itself (C open to
// TMA stores and an output step of alpha * A.B alone); it only changes
// the automatic choice.
inline PairSchedule pair_schedule(int64_t M, int64_t N, int64_t K,
                                  int max_pairs, int mode, bool in_c = true) {
  PairSchedule s;
  s.tiles_m = static_cast<int>((M + 255) / 256);
  s.tiles_n = static_cast<int>((N + 255) / 256);
  s.num_kb = static_cast<int>((K + kSkSliceK - 1) / kSkSliceK);
  const int64_t tiles = static_cast<int64_t>(s.tiles_m) * s.tiles_n;
  const int64_t P = max_pairs > 0 ? max_pairs : 1;
  const int64_t waves = tiles / P, tail = tiles % P;
  s.dp_tiles = static_cast<int>(tiles);
  s.num_full = static_cast<int>(tiles);
  s.pairs = static_cast<int>(tiles < P ? tiles : P);
  // column split of a partial last wave that fills at most half the pairs
  const bool col_split = tail > 0 && 2 * tail <= P;
  auto column_split = [&]() {
    if (col_split) {
      s.num_full = static_cast<int>(tiles - tail);
      s.split = 2;
      const int64_t units = s.num_full + 2 * tail;
      s.pairs = static_cast<int>(units < P ? units : P);
    }
    return s;
  };
  const bool sk_ok = tiles > 0 && tail > 0 && s.num_kb >= kSkMinSlices &&
                     20 * tail <= 17 * P;
  if (mode == kScheduleNoSplitK || !sk_ok) return column_split();
  bool full_sk = waves >= 1 && mode == kScheduleStreamK;
  if (mode == kScheduleAuto) {
    // The simpler schedule unless a split along K is estimated to save more
    // than 8 slices (about 2.5 us).
    const int64_t kb = s.num_kb;
    const int64_t base =
        pair_schedule_cost(col_split ? kColumnTail : kPlainTail, waves, tail, P, kb, in_c);
    const int64_t halved =
        2 * tail <= P ? pair_schedule_cost(kHalvedTail, waves, tail, P, kb, in_c) : INT64_MAX;
    const bool fits = 2 * (M * K + K * N) <= kSkAutoMaxOperandBytes;
    const int64_t streamk = waves >= 1 && fits
                                ? pair_schedule_cost(kStreamKTail, waves, tail, P, kb, in_c)
                                : INT64_MAX;
    const int64_t best_k = halved < streamk ? halved : streamk;
    if (best_k >= base - 8) return column_split();
    full_sk = streamk < halved;
  }
  int64_t sk_tiles = 0, sk_pairs = 0;
  if (full_sk) {
    sk_tiles = P + tail;
    sk_pairs = P;
  } else {
    // the last wave's tiles, each halved over two pairs
    if (2 * tail > P) return column_split();
    sk_tiles = tail;
    sk_pairs = 2 * tail;
  }
  s.sk_tiles = static_cast<int>(sk_tiles);
  s.sk_pairs = static_cast<int>(sk_pairs);
  s.dp_tiles = static_cast<int>(tiles - sk_tiles);
  s.num_full = s.dp_tiles;
  s.pairs = static_cast<int>(waves >= 1 ? P : sk_pairs);
  return s;
}

// Device workspace of a schedule: per stream-K pair two slots (first and last
// segment) per CTA of 128 x 256 FP32 partial sums, then the 64-bit
// synchronisation words (per stream-K tile one ticket counter per CTA rank
// and epilogue warp, per slot one ready flag per CTA rank and warp).  The
// words carry a per-launch tag, so they need no clearing.
constexpr int64_t kSkSlotBytes = 128 * 256 * 4;
inline int64_t sk_partial_bytes(const PairSchedule& s) {
  return static_cast<int64_t>(s.sk_pairs) * 2 * 2 * kSkSlotBytes;
}
inline int64_t sk_sync_words(const PairSchedule& s) {
  return static_cast<int64_t>(s.sk_tiles) * 2 * 4 +
         static_cast<int64_t>(s.sk_pairs) * 2 * 2 * 4;
}
inline int64_t sk_workspace_bytes(const PairSchedule& s) {
  if (s.sk_tiles == 0) return 0;
  return sk_partial_bytes(s) + sk_sync_words(s) * 8;
}

}  // namespace g07
