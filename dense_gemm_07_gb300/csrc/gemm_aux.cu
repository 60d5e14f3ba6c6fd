// gemm_aux.cu -- the small memory-bound kernels around the GEMMs:
//   * C for K == 0 (the empty sum): zeros, or act(beta * C + bias) when an
//     epilogue is given;
//   * a row copy of a 16-bit matrix into a buffer with a different row
//     stride, used to give the tensor-memory accelerator an operand whose
//     base is 16-byte aligned and whose row stride is a multiple of 16 bytes.
// The fill is a grid-stride loop over rows x columns (consecutive threads,
// consecutive columns).  The copy gives each thread one 16-byte group of a
// destination row: eight 2-byte loads from the source (any alignment; a
// warp's loads cover 512 contiguous bytes, so they are served by a few
// cache lines) and one 16-byte store, zeros in the padding columns up to
// the destination stride.
#include <cstdint>

#include "kernels.h"

namespace g07 {
namespace {

__global__ void zero_fill_f32_kernel(float* __restrict__ C, int64_t ldc, int M,
                                     int N, EpiParams epi) {
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

// grid: x over 16-byte groups of a row (blockDim.x threads each), y over
// rows (grid-stride), z over the copies; each ld_dst is a multiple of 8 and
// each dst 16-byte aligned.
__global__ void copy_rows_u16_kernel(PackJobs jobs) {
  const PackJob& j = jobs.job[blockIdx.z];
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  const int c0 = g * 8;
  if (c0 >= j.cols) return;
  const bool whole = c0 + 8 <= j.cols;
  for (int r = blockIdx.y; r < j.rows; r += gridDim.y) {
    const uint16_t* s = j.src + static_cast<int64_t>(r) * j.ld_src + c0;
    uint16_t v[8];
    if (whole) {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = s[e];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = c0 + e < j.cols ? s[e] : uint16_t(0);
    }
    uint4 w;
    w.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
    w.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
    w.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
    w.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
    *reinterpret_cast<uint4*>(j.dst + static_cast<int64_t>(r) * j.ld_dst + c0) = w;
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
  zero_fill_f32_kernel<<<grid_for(static_cast<int64_t>(M) * N, threads),
                         threads, 0, stream>>>(C, ldc, M, N, epi);
  note_launches(1);
  return cudaGetLastError();
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
  copy_rows_u16_kernel<<<dim3(gx, static_cast<unsigned>(gy), count), threads, 0,
                         stream>>>(p);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace g07
