// gemm_aux.cu -- the small memory-bound kernels around the GEMMs:
//   * C for K == 0 (the empty sum): zeros, or act(beta * C + bias) when an
//     epilogue is given;
//   * a row copy of a 16-bit matrix into a buffer with a different row
//     stride, used to give the tensor-memory accelerator an operand whose
//     base is 16-byte aligned and whose row stride is a multiple of 16 bytes.
// The fill is a grid-stride loop over rows x columns (consecutive threads,
// consecutive columns).  The copy gives each thread one 16-byte group of a
// destination row: the source (2-byte aligned, any offset) is read as the
// one or two aligned 16-byte chunks that hold the group and shifted into
// place in registers, then stored with one 16-byte store; zeros in the
// padding columns up to the destination stride.
#include <cstdint>

#include "kernels.h"

namespace g07 {
namespace {

__global__ void zero_fill_f32_kernel(float* __restrict__ C, int64_t ldc, int M,
                                     int N, EpiParams epi) {
  grid_dependency_wait();
  grid_dependents_go();
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < total; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N;
    const int64_t c = i - r * N;
    float* p = C + r * ldc + c;
    *p = epi_apply(epi, 0.0f, epi.beta != 0.0f ? *p : 0.0f,
                   epi.bias ? epi.bias[c] : 0.0f);
  }
}

// Bytes d .. d + 15 of the 32 bytes lo:hi (d even, 0 .. 14).
__device__ __forceinline__ uint4 bytes_at(const uint4& lo, const uint4& hi, int d) {
  const int sh = (d & 3) * 8;
  uint32_t w0, w1, w2, w3, w4;
  switch (d >> 2) {
    case 0: w0 = lo.x; w1 = lo.y; w2 = lo.z; w3 = lo.w; w4 = hi.x; break;
    case 1: w0 = lo.y; w1 = lo.z; w2 = lo.w; w3 = hi.x; w4 = hi.y; break;
    case 2: w0 = lo.z; w1 = lo.w; w2 = hi.x; w3 = hi.y; w4 = hi.z; break;
    default: w0 = lo.w; w1 = hi.x; w2 = hi.y; w3 = hi.z; w4 = hi.w; break;
  }
  return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                    __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// One 16-byte group of a destination row: source elements c0 .. c0 + n - 1
// (n <= 8, the rest of the group zero).  The source is read as the one or
// two aligned 16-byte chunks that hold those elements, so every load stays
// inside a 16-byte granule that holds data of the source row.
__device__ __forceinline__ uint4 load_group(const uint16_t* s, int n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(s);
  const int d = static_cast<int>(a & 15u);
  const uint4* base = reinterpret_cast<const uint4*>(a - d);
  const uint4 lo = __ldg(base);
  const uint4 hi = d + 2 * n > 16 ? __ldg(base + 1) : make_uint4(0u, 0u, 0u, 0u);
  uint4 v = d ? bytes_at(lo, hi, d) : lo;
  if (n < 8) {
    // clear the elements past the end of the row (word i holds elements
    // 2i and 2i + 1)
    auto keep = [n](int i) {
      return (2 * i < n ? 0x0000FFFFu : 0u) | (2 * i + 1 < n ? 0xFFFF0000u : 0u);
    };
    v.x &= keep(0);
    v.y &= keep(1);
    v.z &= keep(2);
    v.w &= keep(3);
  }
  return v;
}

// grid: x over 16-byte groups of a row (blockDim.x threads each), y over
// rows (grid-stride, four rows' loads in flight per thread), z over the
// copies; each ld_dst is a multiple of 8 and each dst 16-byte aligned.
__global__ void copy_rows_u16_kernel(PackJobs jobs) {
  // (a select, not an index: indexing the parameter array by blockIdx.z
  // would copy it to local memory)
  const PackJob j = blockIdx.z == 0 ? jobs.job[0] : jobs.job[1];
  // the operands may come from the kernel before this one; the GEMM after
  // this one waits for the whole copy before it reads it
  grid_dependency_wait();
  grid_dependents_go();
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  const int c0 = g * 8;
  if (c0 >= j.cols) return;
  const int n = j.cols - c0 < 8 ? j.cols - c0 : 8;
  constexpr int R = 4;
  const int step = static_cast<int>(gridDim.y);
  for (int r0 = blockIdx.y; r0 < j.rows; r0 += R * step) {
    uint4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int r = r0 + i * step;
      if (r < j.rows) v[i] = load_group(j.src + static_cast<int64_t>(r) * j.ld_src + c0, n);
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int r = r0 + i * step;
      if (r < j.rows)
        *reinterpret_cast<uint4*>(j.dst + static_cast<int64_t>(r) * j.ld_dst + c0) = v[i];
    }
  }
}

int grid_for(int64_t total, int threads) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_zero_fill_f32(float* C, int64_t ldc, int M, int N,
                                 const EpiParams& epi, cudaStream_t stream) {
  const int threads = 256;
  const cudaError_t e =
      launch_pdl(zero_fill_f32_kernel,
                 dim3(static_cast<unsigned>(grid_for(static_cast<int64_t>(M) * N, threads))),
                 dim3(threads), 0, stream, C, ldc, M, N, epi);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

cudaError_t launch_pack_u16(const PackJob* jobs, int count, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  if (count > 2) return cudaErrorInvalidValue;
  PackJobs p = {};
  int gx = 1, max_rows = 1;
  const int threads = 128;
  for (int i = 0; i < count; ++i) {
    const PackJob& j = jobs[i];
    if (j.rows < 0 || j.cols < 0 || j.ld_dst % 8 != 0 || j.ld_dst < j.cols ||
        (reinterpret_cast<uintptr_t>(j.dst) & 15u) != 0)
      return cudaErrorInvalidValue;
    p.job[i] = j;
    const int groups = (j.cols + 7) / 8;
    const int x = (groups + threads - 1) / threads;
    if (x > gx) gx = x;
    if (j.rows > max_rows) max_rows = j.rows;
  }
  // about 16 blocks of 128 threads per SM for each copy; each walks its rows
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t gy = (static_cast<int64_t>(sms) * 16 + gx - 1) / gx;
  if (gy > max_rows) gy = max_rows;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const cudaError_t e = launch_pdl(copy_rows_u16_kernel,
                                   dim3(gx, static_cast<unsigned>(gy), count), dim3(threads),
                                   0, stream, p);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace g07
