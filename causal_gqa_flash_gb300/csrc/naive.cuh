// naive.cuh — the plain attention kernels that write the whole score matrix
// (naive.cu): the reference the flash kernels are checked against on the GPU.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace gqa {

struct NaiveShape {
  int B, T, Hq, Hkv, d;
};

struct NaiveFwdArgs {
  NaiveShape s;
  const void *q, *k, *v;
  void* o;
  float* lse;
  void* workspace;  // naive_workspace_bytes(s)
  float scale;
  int causal;
};

struct NaiveBwdArgs {
  NaiveShape s;
  const void *q, *k, *v, *o, *dO;
  const float* lse;
  void *dq, *dk, *dv;
  void* workspace;  // naive_workspace_bytes(s)
  float scale;
  int causal;
};

size_t naive_workspace_bytes(const NaiveShape& s);
cudaError_t launch_naive_fwd(const NaiveFwdArgs& a, cudaStream_t stream);
cudaError_t launch_naive_bwd(const NaiveBwdArgs& a, cudaStream_t stream);

}  // namespace gqa
