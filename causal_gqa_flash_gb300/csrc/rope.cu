// rope.cu — rotary position embedding of the queries and keys (and its inverse
// for their gradients), as the trainer of "A transformer in PTX" applies it
// between the fused QKV matmul and attention (§The model). The page names the
// operation without a formula; this is the textbook rotation: feature pair
// (2i, 2i+1) of token t turns by t * base^(-2i/d).
//
// Two kernels, both bound by memory:
//  * rope_table_kernel fills a [T, d/2] table of (cos, sin) pairs, angles and
//    their sine and cosine taken in double and stored as fp32 (one pass, reusable
//    by every layer and step with the same T, d and base);
//  * rope_kernel rotates a [B, T, H, d] bf16 view (in place or into another
//    view): one thread per 16-byte chunk (4 pairs) of a token and group of up to
//    kRopeHeads heads, its table entries read once for the group; the group's
//    loads are all issued before its stores (no chunk is touched by two threads,
//    so this holds in place too), which keeps kRopeHeads loads in flight per
//    thread. Products and sums in fp32, each result rounded once to bf16.
//    Without a table (FREQ) the cosines and sines come from rope_cos_sin, the
//    angles the attention kernels' fused rotation uses.
#include "attn_common.cuh"
#include "rope.cuh"

namespace gqa {
namespace {

__global__ void rope_table_kernel(const RopeTableParams p) {
  const long long n = static_cast<long long>(p.T) * p.half_d;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / p.half_d);
    const int k = static_cast<int>(i - static_cast<long long>(t) * p.half_d);
    double s, c;
    sincos(static_cast<double>(t) * p.theta[k], &s, &c);
    reinterpret_cast<float2*>(p.table)[i] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

template <int D, bool FREQ>
__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const RopeParams p) {
  constexpr int kChunks = D / 8;  // 16-byte chunks (4 pairs) of one head's row
  pdl_launch_dependents();
  pdl_wait_previous();
  // thread -> (token bt, head group hg, chunk): chunks of one head row are adjacent lanes
  const long long gid = blockIdx.x * static_cast<long long>(kRopeThreads) + threadIdx.x;
  const int n_hg = (p.H + kRopeHeads - 1) / kRopeHeads;
  const long long rest = gid / kChunks;
  const long long bt = rest / n_hg;
  if (bt >= static_cast<long long>(p.B) * p.T) return;
  const int chunk = static_cast<int>(gid - rest * kChunks);
  const int h0 = static_cast<int>(rest - bt * n_hg) * kRopeHeads;
  const int nh = min(kRopeHeads, p.H - h0);
  const int b = static_cast<int>(bt / p.T), t = static_cast<int>(bt - static_cast<long long>(b) * p.T);
  // (cos, sin) of the chunk's four pairs
  const float sg = p.inverse ? -1.f : 1.f;
  float c[4], s[4];
  if (FREQ) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      rope_cos_sin(static_cast<uint32_t>(t), p.freq.lo[chunk * 4 + j], p.freq.hi[chunk * 4 + j], c[j], s[j]);
      s[j] *= sg;
    }
  } else {
    const float4* tab = reinterpret_cast<const float4*>(p.table) + (static_cast<long long>(t) * (D / 2) + chunk * 4) / 2;
    const float4 e01 = tab[0], e23 = tab[1];
    c[0] = e01.x, c[1] = e01.z, c[2] = e23.x, c[3] = e23.z;
    s[0] = sg * e01.y, s[1] = sg * e01.w, s[2] = sg * e23.y, s[3] = sg * e23.w;
  }
  const uint4* src = reinterpret_cast<const uint4*>(p.x) + (b * p.x_sb16 + t * p.x_st16 + h0 * kChunks + chunk);
  uint4* dst = reinterpret_cast<uint4*>(p.y) + (b * p.y_sb16 + t * p.y_st16 + h0 * kChunks + chunk);
  uint4 v[kRopeHeads];
#pragma unroll
  for (int j = 0; j < kRopeHeads; ++j)
    if (j < nh) v[j] = src[j * kChunks];
#pragma unroll
  for (int j = 0; j < kRopeHeads; ++j)
    if (j < nh)
      dst[j * kChunks] = make_uint4(rope_rotate_bf16x2(v[j].x, c[0], s[0]), rope_rotate_bf16x2(v[j].y, c[1], s[1]),
                                    rope_rotate_bf16x2(v[j].z, c[2], s[2]), rope_rotate_bf16x2(v[j].w, c[3], s[3]));
}

}  // namespace

cudaError_t launch_rope_table(const RopeTableParams& p, cudaStream_t stream) {
  const long long n = static_cast<long long>(p.T) * p.half_d;
  const int blocks = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  rope_table_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rope(const RopeParams& p, int d, cudaStream_t stream) {
  const long long threads =
      static_cast<long long>(p.B) * p.T * ((p.H + kRopeHeads - 1) / kRopeHeads) * (d / 8);
  const unsigned grid = static_cast<unsigned>((threads + kRopeThreads - 1) / kRopeThreads);
  cudaError_t e;
  if (p.table)
    e = d == 64 ? launch_pdl(rope_kernel<64, false>, grid, kRopeThreads, 0, stream, p)
                : launch_pdl(rope_kernel<128, false>, grid, kRopeThreads, 0, stream, p);
  else
    e = d == 64 ? launch_pdl(rope_kernel<64, true>, grid, kRopeThreads, 0, stream, p)
                : launch_pdl(rope_kernel<128, true>, grid, kRopeThreads, 0, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqa
