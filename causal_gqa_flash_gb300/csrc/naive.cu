// naive.cu — the "naive bf16" attention of "A transformer in PTX" (§Three ways
// to run it: plain kernels on bf16 activations, the reference the fast kernels
// are checked against; §Flash attention: the naive kernels write the whole T x T
// score matrix of every head). Plain CUDA, no tensor cores, nothing shared with
// the flash kernels: 16 x 16 shared-memory tiles, fp32 products and sums.
//
// Per (batch b, query head h), kv head h / (Hq/Hkv):
//   S  = scale Q K^T                  fp32 [T, T], -inf above the diagonal (causal)
//   LSE_i = ln sum_j exp(S_ij);  P = exp(S - LSE)   stored as bf16
//   O  = P V                          bf16
// and for the loss sum(O * dO):
//   dP = dO V^T (fp32);  D_i = dO_i . O_i;  dS = P (dP - D)   stored as bf16
//   dQ = scale dS K;  dK = scale sum_{h in group} dS^T Q;  dV = sum_{h in group} P^T dO
// q, o, dO, dq are [B,T,Hq,d], k, v, dk, dv [B,T,Hkv,d], lse [B,Hq,T], row-major.
#include <cuda_bf16.h>

#include "naive.cuh"

namespace gqa {
namespace {

constexpr int kT = 16;  // tile edge

__device__ __forceinline__ float ld_bf16(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// out[bh][i][j] = scale * sum_c X[b,i,h,c] Y[b,j,h/G,c]; -inf where masked (j > i, causal).
__global__ void rowdot_kernel(const __nv_bfloat16* X, const __nv_bfloat16* Y, float* out, NaiveShape s, float scale,
                              int mask) {
  __shared__ float xs[kT][kT + 1], ys[kT][kT + 1];
  const int bh = blockIdx.z, b = bh / s.Hq, h = bh % s.Hq, kvh = h / (s.Hq / s.Hkv);
  const int i = blockIdx.y * kT + threadIdx.y, j = blockIdx.x * kT + threadIdx.x;
  const int jy = blockIdx.x * kT + threadIdx.y;  // row of Y this thread loads
  float acc = 0.f;
  for (int c0 = 0; c0 < s.d; c0 += kT) {
    const int c = c0 + threadIdx.x;
    xs[threadIdx.y][threadIdx.x] = (i < s.T) ? ld_bf16(X + ((static_cast<size_t>(b) * s.T + i) * s.Hq + h) * s.d + c) : 0.f;
    ys[threadIdx.y][threadIdx.x] =
        (jy < s.T) ? ld_bf16(Y + ((static_cast<size_t>(b) * s.T + jy) * s.Hkv + kvh) * s.d + c) : 0.f;
    __syncthreads();
    for (int cc = 0; cc < kT; ++cc) acc = fmaf(xs[threadIdx.y][cc], ys[threadIdx.x][cc], acc);
    __syncthreads();
  }
  if (i < s.T && j < s.T)
    out[(static_cast<size_t>(bh) * s.T + i) * s.T + j] = (mask && j > i) ? -INFINITY : scale * acc;
}

// One block per (bh, row i). Forward (lse_in == nullptr): LSE_i from the row,
// written to lse_out; P = exp(S - LSE) as bf16. Backward: P from the given LSE.
__global__ void softmax_rows_kernel(const float* S, const float* lse_in, float* lse_out, __nv_bfloat16* P,
                                    NaiveShape s) {
  __shared__ float red[256];
  const size_t row = blockIdx.x;  // bh * T + i
  const float* sr = S + row * s.T;
  float lse;
  if (lse_in) {
    lse = lse_in[row];
  } else {
    float m = -INFINITY;
    for (int j = threadIdx.x; j < s.T; j += blockDim.x) m = fmaxf(m, sr[j]);
    red[threadIdx.x] = m;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + w]);
      __syncthreads();
    }
    m = red[0];
    __syncthreads();
    float l = 0.f;
    for (int j = threadIdx.x; j < s.T; j += blockDim.x) l += expf(sr[j] - m);
    red[threadIdx.x] = l;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    lse = m + logf(red[0]);
    if (threadIdx.x == 0) lse_out[row] = lse;
  }
  for (int j = threadIdx.x; j < s.T; j += blockDim.x) P[row * s.T + j] = __float2bfloat16_rn(expf(sr[j] - lse));
}

// out[b,i,h,c] = scale * sum_j A[bh][i][j] Y[b,j,h/G,c]  (A bf16 [T,T]), bf16 out.
__global__ void amul_kernel(const __nv_bfloat16* A, const __nv_bfloat16* Y, __nv_bfloat16* out, NaiveShape s,
                            float scale) {
  __shared__ float as[kT][kT + 1], ys[kT][kT + 1];
  const int bh = blockIdx.z, b = bh / s.Hq, h = bh % s.Hq, kvh = h / (s.Hq / s.Hkv);
  const int i = blockIdx.y * kT + threadIdx.y, c = blockIdx.x * kT + threadIdx.x;
  float acc = 0.f;
  for (int j0 = 0; j0 < s.T; j0 += kT) {
    const int ja = j0 + threadIdx.x, jy = j0 + threadIdx.y;
    as[threadIdx.y][threadIdx.x] = (i < s.T && ja < s.T) ? ld_bf16(A + (static_cast<size_t>(bh) * s.T + i) * s.T + ja) : 0.f;
    ys[threadIdx.y][threadIdx.x] =
        (jy < s.T) ? ld_bf16(Y + ((static_cast<size_t>(b) * s.T + jy) * s.Hkv + kvh) * s.d + c) : 0.f;
    __syncthreads();
    for (int jj = 0; jj < kT; ++jj) acc = fmaf(as[threadIdx.y][jj], ys[jj][threadIdx.x], acc);
    __syncthreads();
  }
  if (i < s.T) out[((static_cast<size_t>(b) * s.T + i) * s.Hq + h) * s.d + c] = __float2bfloat16_rn(scale * acc);
}

// out[b,j,g,c] = scale * sum_{h in group g} sum_i A[bh][i][j] X[b,i,h,c], bf16 out.
__global__ void atmul_group_kernel(const __nv_bfloat16* A, const __nv_bfloat16* X, __nv_bfloat16* out, NaiveShape s,
                                   float scale) {
  __shared__ float as[kT][kT + 1], xs[kT][kT + 1];
  const int bg = blockIdx.z, b = bg / s.Hkv, g = bg % s.Hkv, G = s.Hq / s.Hkv;
  const int j = blockIdx.y * kT + threadIdx.y, c = blockIdx.x * kT + threadIdx.x;
  float acc = 0.f;
  for (int h = g * G; h < (g + 1) * G; ++h) {
    const size_t bh = static_cast<size_t>(b) * s.Hq + h;
    for (int i0 = 0; i0 < s.T; i0 += kT) {
      const int ia = i0 + threadIdx.x, ix = i0 + threadIdx.y;
      // as[y][x] = A[i0 + x][j]: row j of A^T
      as[threadIdx.y][threadIdx.x] = (j < s.T && ia < s.T) ? ld_bf16(A + (bh * s.T + ia) * s.T + j) : 0.f;
      xs[threadIdx.y][threadIdx.x] = (ix < s.T) ? ld_bf16(X + ((static_cast<size_t>(b) * s.T + ix) * s.Hq + h) * s.d + c) : 0.f;
      __syncthreads();
      for (int ii = 0; ii < kT; ++ii) acc = fmaf(as[threadIdx.y][ii], xs[ii][threadIdx.x], acc);
      __syncthreads();
    }
  }
  if (j < s.T) out[((static_cast<size_t>(b) * s.T + j) * s.Hkv + g) * s.d + c] = __float2bfloat16_rn(scale * acc);
}

// One block per (bh, row i): D_i = dO_i . O_i, then dS = P (dP - D) as bf16.
__global__ void ds_rows_kernel(const float* dP, const __nv_bfloat16* P, const __nv_bfloat16* O,
                               const __nv_bfloat16* dO, __nv_bfloat16* dS, NaiveShape s) {
  __shared__ float red[256];
  const size_t row = blockIdx.x;  // bh * T + i
  const int bh = static_cast<int>(row / s.T), i = static_cast<int>(row % s.T);
  const int b = bh / s.Hq, h = bh % s.Hq;
  const size_t off = ((static_cast<size_t>(b) * s.T + i) * s.Hq + h) * s.d;
  float part = 0.f;
  for (int c = threadIdx.x; c < s.d; c += blockDim.x) part += ld_bf16(O + off + c) * ld_bf16(dO + off + c);
  red[threadIdx.x] = part;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  const float D = red[0];
  for (int j = threadIdx.x; j < s.T; j += blockDim.x)
    dS[row * s.T + j] = __float2bfloat16_rn(__bfloat162float(P[row * s.T + j]) * (dP[row * s.T + j] - D));
}

dim3 tiles(int cols, int rows, int z) { return dim3((cols + kT - 1) / kT, (rows + kT - 1) / kT, z); }

}  // namespace

size_t naive_workspace_bytes(const NaiveShape& s) {
  const size_t tt = static_cast<size_t>(s.B) * s.Hq * s.T * s.T;
  return tt * sizeof(float) + 2 * tt * sizeof(__nv_bfloat16);  // S or dP (fp32), P and dS (bf16)
}

cudaError_t launch_naive_fwd(const NaiveFwdArgs& a, cudaStream_t st) {
  const NaiveShape& s = a.s;
  const size_t tt = static_cast<size_t>(s.B) * s.Hq * s.T * s.T;
  float* S = static_cast<float*>(a.workspace);
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(S + tt);
  const auto* q = static_cast<const __nv_bfloat16*>(a.q);
  const auto* k = static_cast<const __nv_bfloat16*>(a.k);
  const auto* v = static_cast<const __nv_bfloat16*>(a.v);
  rowdot_kernel<<<tiles(s.T, s.T, s.B * s.Hq), dim3(kT, kT), 0, st>>>(q, k, S, s, a.scale, a.causal);
  softmax_rows_kernel<<<static_cast<unsigned>(s.B * s.Hq * s.T), 256, 0, st>>>(S, nullptr, a.lse, P, s);
  amul_kernel<<<tiles(s.d, s.T, s.B * s.Hq), dim3(kT, kT), 0, st>>>(P, v, static_cast<__nv_bfloat16*>(a.o), s, 1.f);
  return cudaGetLastError();
}

cudaError_t launch_naive_bwd(const NaiveBwdArgs& a, cudaStream_t st) {
  const NaiveShape& s = a.s;
  const size_t tt = static_cast<size_t>(s.B) * s.Hq * s.T * s.T;
  float* SdP = static_cast<float*>(a.workspace);  // S, then dP
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(SdP + tt);
  __nv_bfloat16* dS = P + tt;
  const auto* q = static_cast<const __nv_bfloat16*>(a.q);
  const auto* k = static_cast<const __nv_bfloat16*>(a.k);
  const auto* v = static_cast<const __nv_bfloat16*>(a.v);
  const auto* o = static_cast<const __nv_bfloat16*>(a.o);
  const auto* dO = static_cast<const __nv_bfloat16*>(a.dO);
  const unsigned rows = static_cast<unsigned>(s.B * s.Hq * s.T);
  rowdot_kernel<<<tiles(s.T, s.T, s.B * s.Hq), dim3(kT, kT), 0, st>>>(q, k, SdP, s, a.scale, a.causal);
  softmax_rows_kernel<<<rows, 256, 0, st>>>(SdP, a.lse, nullptr, P, s);
  rowdot_kernel<<<tiles(s.T, s.T, s.B * s.Hq), dim3(kT, kT), 0, st>>>(dO, v, SdP, s, 1.f, 0);
  ds_rows_kernel<<<rows, 256, 0, st>>>(SdP, P, o, dO, dS, s);
  amul_kernel<<<tiles(s.d, s.T, s.B * s.Hq), dim3(kT, kT), 0, st>>>(dS, k, static_cast<__nv_bfloat16*>(a.dq), s,
                                                                     a.scale);
  atmul_group_kernel<<<tiles(s.d, s.T, s.B * s.Hkv), dim3(kT, kT), 0, st>>>(
      dS, q, static_cast<__nv_bfloat16*>(a.dk), s, a.scale);
  atmul_group_kernel<<<tiles(s.d, s.T, s.B * s.Hkv), dim3(kT, kT), 0, st>>>(
      P, dO, static_cast<__nv_bfloat16*>(a.dv), s, 1.f);
  return cudaGetLastError();
}

}  // namespace gqa
