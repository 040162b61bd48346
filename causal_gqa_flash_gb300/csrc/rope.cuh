// rope.cuh — parameters and launchers of the rotary-embedding kernels (rope.cu).
#pragma once

#include <cuda_runtime.h>

#include "attn_common.cuh"

namespace gqa {

constexpr int kRopeThreads = 128;
constexpr int kRopeHeads = 4;  // heads of one token per thread
constexpr int kRopeMaxHalfD = 64;  // d <= 128

struct RopeTableParams {
  float* table;                  // [T, d/2] of (cos, sin), fp32
  int T, half_d;
  double theta[kRopeMaxHalfD];   // base^(-2i/d)
};

// y[b,t,h] = rotation of x[b,t,h]; bf16 views with packed heads (head stride d).
struct RopeParams {
  const void* x;
  void* y;
  long long x_st16, x_sb16;   // token / batch strides of x in 16-byte units
  long long y_st16, y_sb16;
  const float* table;         // [T, d/2] of (cos, sin), or null: angles from freq
  int B, T, H;
  int inverse;                // rotate by minus the angle
  RopeFreq freq;              // with table == null
};

cudaError_t launch_rope_table(const RopeTableParams& p, cudaStream_t stream);
cudaError_t launch_rope(const RopeParams& p, int d, cudaStream_t stream);

}  // namespace gqa
