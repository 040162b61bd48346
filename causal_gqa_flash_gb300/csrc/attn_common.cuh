// attn_common.cuh — parameters and tile geometry shared by the attention kernels
// and the host code that launches them.
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace gqa {

// Query and key tiles are 128 rows: one row per TMEM lane, M = 128 MMAs.
constexpr int kTile = 128;
// One 128-byte swizzle atom column block: 64 bf16 of the head dim, 128 rows.
constexpr int kHalfTileBytes = kTile * 128;
// Bytes at the end of the backward workspace that hold the persistent launch's
// task counters.
constexpr size_t kBwdSchedBytes = 256;

enum KernelId : unsigned int {
  kKidFwd = 1,
  kKidBwdPre = 2,
  kKidBwdMain = 3,
  kKidProbe = 8,
  kKidSelfTest = 9,
};

// Division of a non-negative int below 2^31 by a divisor fixed for the launch, as a
// multiply-high, an add and a shift instead of the tens of instructions of a
// division by a runtime value (Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(n, m) + n) >> l, and the sum
// stays below 2^32 because umulhi(n, m) < n < 2^31. The work-item decodes sit on
// the path between one task and the next, where these divisions showed.
struct FastDiv {
  uint32_t d, m, s;
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
  return FastDiv{d, static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  const uint32_t u = static_cast<uint32_t>(n);
  return static_cast<int>((__umulhi(u, f.m) + u) >> f.s);
}

// Rotary frequencies as fixed-point turns: feature pair i of token t turns by
// t * f_i turns, f_i = base^(-2i/d) / (2 pi), held to 64 bits (hi and lo words).
// The fraction t * f_i mod 1 then comes out of two 32-bit integer multiplies,
// exact to 2^-32 of a turn for any t, so the angle needs no floating-point range
// reduction and no table in memory.
struct RopeFreq {
  uint32_t lo[64], hi[64];
};

// Forward: work items of one 128-query tile of one (query head, batch).
// Tensors [B,T,H,d] bf16 are reached through TMA maps or through element strides
// (token, batch) with the heads of one token packed (head stride d).
struct FwdParams {
  CUtensorMap tmap_q;  // [B,T,Hq,d] bf16, box 64 x 1 x 128 x 1, 128B swizzle
  CUtensorMap tmap_k;  // [B,T,Hkv,d]
  CUtensorMap tmap_v;  // [B,T,Hkv,d]
  CUtensorMap tmap_o;  // [B,T,Hq,d], box 64 x 1 x 32 x 1 (epilogue stores)
  CUtensorMap tmap_qrot;  // rotary only: [B,T,Hq,d] rotated Q out, boxes as tmap_q
  int rope;              // 1: q is rotated in the kernel (rope_f) and stored to tmap_qrot
  RopeFreq rope_f;
  float* lse;          // [B,Hq,T] fp32, natural log
  int B, T, Hq, Hkv, G, nT;
  FastDiv fd_bh, fd_hq, fd_g;  // divisors B*Hq, Hq, G of the work-item decode
  int causal;
  float scale_log2;    // (1/sqrt(d)) * log2(e)
  DevStatusWord* status;
  unsigned long long budget_ns;
};

// Backward preprocess: D = rowsum(dO * O), LSE2 = LSE * log2(e), both [B,Hq,Tpad].
struct BwdPreParams {
  const void* o;             // [B,T,Hq,d] bf16
  const void* dO;            // [B,T,Hq,d] bf16
  long long o_st16, o_sb16;    // strides of O between tokens / batch entries, in 16-byte units
  long long do_st16, do_sb16;  // the same for dO
  const float* lse;
  float* Dvec;   // [B,Hq,Tpad]
  float* lse2;   // [B,Hq,Tpad]
  unsigned* sched;  // [2] task counters of the dQ / dK/dV launch, zeroed here
  int B, T, Hq, Tpad;
};

// Backward dQ (one task per query tile) and dK/dV (one task per key tile), one persistent launch.
struct BwdParams {
  CUtensorMap tmap_q;
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  CUtensorMap tmap_do;
  CUtensorMap tmap_dq;  // d = 64 only: epilogue stores (32-row boxes)
  CUtensorMap tmap_dk;
  CUtensorMap tmap_dv;
  const float* Dvec;   // [B,Hq,Tpad]
  const float* lse2;   // [B,Hq,Tpad]
  unsigned* sched;     // [2] next task, finished CTAs; zero on entry, left zero on exit
  void* dq;            // [B,T,Hq,d]
  void* dk;            // [B,T,Hkv,d]
  void* dv;            // [B,T,Hkv,d]
  int rope;            // 1: dq, dk leave inverse-rotated by rope_f's angles
  RopeFreq rope_f;
  long long dq_st, dq_sb, dk_st, dk_sb, dv_st, dv_sb;  // element strides (token, batch) of the outputs
  int B, T, Hq, Hkv, G, nT, Tpad;
  int causal;
  int n_dkv_tasks;     // tasks [0, n_dkv_tasks) compute dK/dV (0 = none)
  int n_dq_tasks;      // the next n_dq_tasks tasks compute dQ (0 = none)
  int dkv_group_major;  // dK/dV task order: 1 = per (batch, kv head) group, 0 = key tile outermost
  int dq_group_major;   // dQ task order: 1 = per (batch, kv head) group, 0 = query tile outermost
  // divisors of the task decode: nT, B*Hkv, Hkv, B*Hq, Hq, G, nT*G
  FastDiv fd_nt, fd_bk, fd_hkv, fd_bh, fd_hq, fd_g, fd_ntg;
  float scale;         // 1/sqrt(d)
  float scale_log2;    // scale * log2(e)
  DevStatusWord* status;
  unsigned long long budget_ns;
};

// Rotary embedding of one bf16 pair (x0, x1) = (low, high half of w) by the angle
// with cosine c and sine s: (x0 c - x1 s, x0 s + x1 c), products and sums in fp32,
// each result rounded once to bf16. The standalone rotation and the forward's
// fused one both call this, so they produce the same bits.
__device__ __forceinline__ uint32_t rope_rotate_bf16x2(uint32_t w, float c, float s) {
  const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xffff0000u);
  return pack_bf16x2(fmaf(x0, c, -x1 * s), fmaf(x0, s, x1 * c));
}

// cos and sin of token t's angle for the pair with frequency (lo, hi) (see RopeFreq):
// the turn fraction as a signed 32-bit fixed-point number in [-1/2, 1/2), scaled to
// radians in [-pi, pi), where the hardware sine and cosine are accurate to ~2^-21.
__device__ __forceinline__ void rope_cos_sin(uint32_t t, uint32_t lo, uint32_t hi, float& c, float& s) {
  const int32_t turns = static_cast<int32_t>(__umulhi(t, lo) + t * hi);
  __sincosf(static_cast<float>(turns) * 1.4629180792671596e-09f, &s, &c);  // 2 pi / 2^32
}

// The same rotation of an fp32 pair in place (the backward passes -s: the inverse).
__device__ __forceinline__ void rope_rotate_f32(float& x0, float& x1, float c, float s) {
  const float y0 = fmaf(x0, c, -x1 * s), y1 = fmaf(x0, s, x1 * c);
  x0 = y0;
  x1 = y1;
}

// Number of SMs of the current device (cached per device).
inline cudaError_t sm_count(int* n) {
  static int cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    *n = cache[dev];
    return cudaSuccess;
  }
  e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = *n;
  return cudaSuccess;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Launch `kernel` on `stream` with programmatic stream serialization, so it can
// be scheduled while the previous kernel of the stream finishes; the kernel
// itself waits (pdl_wait_previous) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host-side launchers (defined next to their kernels).
cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdPreParams& p, int d, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream);
cudaError_t launch_selftest_timeout(DevStatusWord* status, unsigned long long budget_ns, cudaStream_t stream);
cudaError_t launch_mma_probe(int n, int a_tmem, int chains, int iters, void* out, DevStatusWord* status,
                             unsigned long long budget_ns, int grid, cudaStream_t stream);
cudaError_t launch_ex2_probe(int iters, unsigned long long* cycles, float* sink, int grid, cudaStream_t stream);
cudaError_t launch_tma_probe(const CUtensorMap& map, int n_tiles, int stages, int ctas_per_sm, int iters,
                             unsigned long long* out, DevStatusWord* status, unsigned long long budget_ns, int sms,
                             cudaStream_t stream);

}  // namespace gqa
