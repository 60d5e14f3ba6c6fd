// epilogue.cuh -- the fused output step of every kernel:
//   C := act(alpha * (A*B) + beta * C + bias[col])
// ("How a Matrix Multiply Runs on a GPU", "Level 2" pseudocode: the output is
// alpha * acc + beta * C, plus a bias and an activation, applied while the
// accumulators are still in registers).  With alpha = 1, beta = 0, no bias
// and no activation the value is the accumulator itself, bit for bit, and C
// is not read.
#pragma once

#include <cstdint>

namespace g07 {

struct EpiParams {
  float alpha;
  float beta;          // 0: the prior contents of C are not read
  const float* bias;   // N floats (device) or nullptr
  int act;             // 0 identity, 1 ReLU, 2 GELU
};

__host__ __device__ inline EpiParams epi_identity() {
  return EpiParams{1.0f, 0.0f, nullptr, 0};
}

// kGelu = false compiles the GELU case out: the main kernels are built
// twice, and the copy without it is used for every other activation (the
// erff code, even unused, changes the register allocation of the main loops
// around it).
template <bool kGelu = true>
__device__ __forceinline__ float epi_apply(const EpiParams& e, float acc,
                                           float c_old, float bias) {
  float v = e.alpha * acc;
  if (e.beta != 0.0f) v = fmaf(e.beta, c_old, v);
  if (e.bias != nullptr) v += bias;
  if (e.act == 1) v = fmaxf(v, 0.0f);
  // GELU: x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), with CUDA's erff
  if (kGelu && e.act == 2) v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  return v;
}

constexpr int kActGelu = 2;

}  // namespace g07
