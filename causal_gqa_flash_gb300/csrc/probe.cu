// probe.cu — rate probes for the units the attention kernels lean on: the tcgen05
// tensor core (bf16 x bf16 -> fp32 MMAs, M = 128), the ex2 unit of the softmax, and
// the TMA path that fills their operand rings (16 KB tiles into shared memory).
//
// "Talking to the GPU", §The real tensor core peak: the page measures its GPU's
// real MMA peak with enough independent work per SM to keep the unit busy, over one
// wave, timed on the device, instead of trusting the data sheet. The same idea here
// for sm_103a: one CTA per SM, one elected thread issuing a long chain of tcgen05
// MMAs into TMEM (the tensor core works through them in order; the issuing thread
// only waits once, at the end), timed with the SM's cycle counter and the global
// nanosecond timer, so the result is FLOP per cycle per SM and the clock it ran at.
// Operands are zeros: the rate does not depend on the values.
#include "attn_common.cuh"

namespace gqa {
namespace {

constexpr int kProbeThreads = 128;

struct MmaProbeOut {
  unsigned long long cycles;  // SM cycles of the MMA chain (issue of the first to completion of the last)
  unsigned long long ns;      // the same interval in global-timer nanoseconds
};

// n: MMA N (64, 128 or 256); a_tmem: A operand from TMEM (TS) instead of shared memory (SS);
// chains: 1 = every MMA accumulates into one accumulator (each waits for the previous
// one's result), 2 = alternate between two accumulators (independent neighbours).
// TMEM: accumulators at columns 0 and (n <= 128 ? 128 : 256); A at 256 (TS: n <= 128
// when chains == 2).
__global__ void __launch_bounds__(kProbeThreads, 1) mma_probe_kernel(int n, int a_tmem, int chains, int iters,
                                                                     MmaProbeOut* out,
                                                                     DevStatusWord* status,
                                                                     unsigned long long budget_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);  // A: 128 x 64 bf16 (16 KB), B: 256 x 64 bf16 (32 KB)
  __shared__ uint64_t bar_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (48 * 1024) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bar_done, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // A in TMEM: columns [256, 264) hold 128 lanes x 16 bf16 (one K-step), zeroed here
  {
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    tmem_st8(tmem + lane_base + 256, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const WaitCtx ctx{&abort_sh, status, budget_ns, kKidProbe};
  if (warp == 0) {
    const uint64_t a_desc = sdesc_sw128(smem_u32(smem), 16, 1024);
    const uint64_t b_desc = sdesc_sw128(smem_u32(smem + 16 * 1024), 16, 1024);
    const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(n), 0, 0);
    const uint32_t d1 = chains == 2 ? (n <= 128 ? 128u : 256u) : 0u;  // second accumulator
    uint64_t c0 = 0, t0 = 0;
    if (elect_one()) {
      c0 = clock64();
      t0 = globaltimer_ns();
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t off = static_cast<uint32_t>(kk * 32) >> 4;
          const uint32_t d = (kk & 1) ? d1 : 0u;
          const uint32_t acc = (it > 0 || kk > 1 || (chains == 1 && kk > 0)) ? 1u : 0u;
          if (a_tmem)
            mma_ts(tmem + d, tmem + 256, b_desc + off, idesc, acc);
          else
            mma_ss(tmem + d, a_desc + off, b_desc + off, idesc, acc);
        }
      }
      mma_commit(&bar_done);
    }
    __syncwarp();
    const bool ok = mbar_wait(&bar_done, 0, ctx, 1);
    if (elect_one() && ok) {
      const uint64_t c1 = clock64(), t1 = globaltimer_ns();
      out[blockIdx.x].cycles = c1 - c0;
      out[blockIdx.x].ns = t1 - t0;
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// Every thread runs 8 independent chains of ex2.approx for `iters` rounds.
__global__ void __launch_bounds__(1024, 1) ex2_probe_kernel(int iters, unsigned long long* cycles, float* sink) {
  float x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = -1.0f - 0.001f * (threadIdx.x & 7) - 0.01f * i;
  __syncthreads();
  const uint64_t c0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = ex2_approx(x[i]) - 1.5f;  // stays in (-1.5, -0.5): no under/overflow
  }
  __syncthreads();
  const uint64_t c1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += x[i];
  if (s == 12345.f) sink[0] = s;  // keeps the chains alive
  if (threadIdx.x == 0) cycles[blockIdx.x] = c1 - c0;
}

// TMA tile loads: each CTA keeps `stages` loads of one 128-row x 128-byte tile
// (16 KB, the attention kernels' d = 64 operand tile) in flight, each into its own
// shared-memory slot with its own mbarrier, for `iters` tiles picked by a per-CTA
// linear congruential sequence over the tensor's n_tiles tiles. Record per CTA: the
// global-timer nanoseconds from the first request to the last arrival. With the
// tensor in the L2 the rate shows the load path; over a tensor far larger than the
// L2, HBM. Bytes in flight per SM divided by the per-SM rate is the load latency
// under that load.
constexpr int kTmaProbeMaxStages = 8;
constexpr int kTmaTileBytes = 16384;

__global__ void __launch_bounds__(32) tma_probe_kernel(const __grid_constant__ CUtensorMap map, int n_tiles,
                                                       int stages, int iters, unsigned long long* out,
                                                       DevStatusWord* status, unsigned long long budget_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t full[kTmaProbeMaxStages];
  __shared__ int abort_sh;
  if (threadIdx.x != 0) return;
  for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
  abort_sh = 0;
  fence_mbar_init();
  const WaitCtx ctx{&abort_sh, status, budget_ns, kKidProbe};
  uint32_t seed = blockIdx.x * 2654435761u + 12345u;
  const uint64_t t0 = globaltimer_ns();
  int issued = 0;
  bool ok = true;
  for (int i = 0; i < iters + stages && ok; ++i) {
    const int s = i % stages;
    // slot s last held request i - stages: it must have landed before the slot is reused
    if (i >= stages) ok = mbar_wait(&full[s], ((i / stages) - 1) & 1, ctx, 1);
    if (ok && i < iters) {
      seed = seed * 1664525u + 1013904223u;
      const int tile = static_cast<int>((seed >> 8) % static_cast<uint32_t>(n_tiles));
      mbar_arrive_expect_tx(&full[s], kTmaTileBytes);
      tma_load_4d(smem + s * kTmaTileBytes, &map, &full[s], 0, 0, tile * 128, 0);
      ++issued;
    }
  }
  if (!ok) {
    // let every request already made land before the CTA leaves
    for (int s = 0; s < stages; ++s) {
      const int uses = issued / stages + (s < issued % stages ? 1 : 0);
      if (uses > 0) mbar_wait_drain(&full[s], (uses - 1) & 1, budget_ns);
    }
    return;
  }
  out[blockIdx.x] = globaltimer_ns() - t0;
}

}  // namespace

// Both probes request more shared memory than two CTAs could share, so each SM
// runs exactly one CTA (grid = the SM count).
constexpr int kProbeSmem = 120 * 1024;

cudaError_t launch_mma_probe(int n, int a_tmem, int chains, int iters, void* out, DevStatusWord* status,
                             unsigned long long budget_ns, int grid, cudaStream_t stream) {
  constexpr int smem = kProbeSmem;
  cudaError_t e = cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_probe_kernel<<<grid, kProbeThreads, smem, stream>>>(n, a_tmem, chains, iters, static_cast<MmaProbeOut*>(out),
                                                          status, budget_ns);
  return cudaGetLastError();
}

cudaError_t launch_tma_probe(const CUtensorMap& map, int n_tiles, int stages, int ctas_per_sm, int iters,
                             unsigned long long* out, DevStatusWord* status, unsigned long long budget_ns, int sms,
                             cudaStream_t stream) {
  const int smem = stages * kTmaTileBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(tma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tma_probe_kernel<<<sms * ctas_per_sm, 32, smem, stream>>>(map, n_tiles, stages, iters, out, status, budget_ns);
  return cudaGetLastError();
}

cudaError_t launch_ex2_probe(int iters, unsigned long long* cycles, float* sink, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(ex2_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return e;
  ex2_probe_kernel<<<grid, 1024, kProbeSmem, stream>>>(iters, cycles, sink);
  return cudaGetLastError();
}

}  // namespace gqa
