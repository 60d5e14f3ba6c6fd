// gemm_aux.cu -- the small memory-bound kernels around the GEMMs:
//   * C for K == 0 (the empty sum): zeros, or act(beta * C + bias) when an
//     epilogue is given;
//   * a row copy of a 16-bit matrix into a buffer with a different row
//     stride, used to give the tensor-memory accelerator an operand whose
//     base is 16-byte aligned and whose row stride is a multiple of 16 bytes.
// Both are grid-stride loops over rows x columns; consecutive threads touch
// consecutive columns of one row, so reads and writes are coalesced.
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

__global__ void copy_rows_u16_kernel(const uint16_t* __restrict__ src,
                                     int64_t ld_src, uint16_t* __restrict__ dst,
                                     int64_t ld_dst, int rows, int cols) {
  const int64_t total = static_cast<int64_t>(rows) * cols;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < total; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / cols;
    const int64_t c = i - r * cols;
    dst[r * ld_dst + c] = src[r * ld_src + c];
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

cudaError_t launch_copy_rows_u16(const uint16_t* src, int64_t ld_src,
                                 uint16_t* dst, int64_t ld_dst, int rows,
                                 int cols, cudaStream_t stream) {
  const int threads = 256;
  copy_rows_u16_kernel<<<grid_for(static_cast<int64_t>(rows) * cols, threads),
                         threads, 0, stream>>>(src, ld_src, dst, ld_dst, rows,
                                               cols);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace g07
