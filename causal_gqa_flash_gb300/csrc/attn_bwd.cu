// attn_bwd.cu — backward kernels of causal grouped-query flash attention for sm_103a.
//
// "A transformer in PTX", §The same bits every time: the attention backward is
// two kernels, one per block of queries (dQ) and one per block of keys (dK,
// dV) that loops over every query head sharing that key/value head; both
// recompute the scores from the saved log-sum-exp, and no float atomic is
// used, so every output element has one writer and one summation order.
//
// Before them, a preprocess pass (not on the page; the standard companion of a
// recompute backward) writes, per query row, D_i = rowsum(dO_i * O_i) and the
// LSE in log2 units, into the caller's workspace, padded to whole 128-row tiles.
//
// Both main kernels use the forward's warp layout: warp 0 TMA, warp 1 tcgen05
// MMA issue (one thread) and TMEM owner, warps 2-5 one thread per TMEM lane.
//   dQ kernel (per 128-query tile of one query head), key tiles in ascending order:
//     S = Q K^T, dP = dO V^T                  (SS MMAs into TMEM)
//     P = 2^(S*scale*log2e - LSE2), dS = P (dP - D)   (per row, bf16 into TMEM)
//     dQ += dS K                              (TS MMA, K as MN-major operand)
//   dK/dV kernel (per 128-key tile of one kv head), query heads of the group in
//   ascending order, query tiles from the diagonal on:
//     S^T = K Q^T, dP^T = V dO^T              (SS MMAs)
//     P^T, dS^T per key row                   (bf16 into TMEM)
//     dV += P^T dO, dK += dS^T Q              (TS MMAs, dO/Q as MN-major operands)
// dQ and dK carry the score scale once, in the epilogue.
#include "attn_common.cuh"

namespace gqa {
namespace {

constexpr int kBwdThreads = 192;
constexpr uint32_t kBwdTmemCols = 512;
// Requesting at least this much dynamic shared memory keeps one CTA per SM,
// which the 512-column TMEM allocation needs anyway.
constexpr int kOneCtaPerSmSmem = 120 * 1024;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& c, unsigned where) {
  bool ok = mbar_wait(bar, parity, c, where);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ============================================================================
// Preprocess: D = rowsum(dO * O), LSE2 = LSE * log2(e); padded rows get 0.
// Rows are visited in memory order (b, t, h); D/8 threads read one row with
// 16-byte loads, so a warp reads contiguous bytes.
// ============================================================================
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdPreParams p) {
  constexpr int TPR = D / 8;
  const long long nrows = static_cast<long long>(p.B) * p.T * p.Hq;
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = gtid / TPR;
  const int part = static_cast<int>(gtid % TPR);
  float acc = 0.f;
  if (r < nrows) {
    const uint4 a = reinterpret_cast<const uint4*>(p.o)[r * TPR + part];
    const uint4 c = reinterpret_cast<const uint4*>(p.dO)[r * TPR + part];
    acc = bf16lo(a.x) * bf16lo(c.x);
    acc = fmaf(bf16hi(a.x), bf16hi(c.x), acc);
    acc = fmaf(bf16lo(a.y), bf16lo(c.y), acc);
    acc = fmaf(bf16hi(a.y), bf16hi(c.y), acc);
    acc = fmaf(bf16lo(a.z), bf16lo(c.z), acc);
    acc = fmaf(bf16hi(a.z), bf16hi(c.z), acc);
    acc = fmaf(bf16lo(a.w), bf16lo(c.w), acc);
    acc = fmaf(bf16hi(a.w), bf16hi(c.w), acc);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0 && r < nrows) {
    const int h = static_cast<int>(r % p.Hq);
    const long long bt = r / p.Hq;
    const int t = static_cast<int>(bt % p.T);
    const int b = static_cast<int>(bt / p.T);
    const size_t idx = (static_cast<size_t>(b) * p.Hq + h) * p.Tpad + t;
    p.Dvec[idx] = acc;
    p.lse2[idx] = p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.T + t] * 1.4426950408889634f;
  }
  // Zero the padding rows [T, Tpad) of every (b, h).
  const int pad = p.Tpad - p.T;
  if (pad > 0) {
    const long long npad = static_cast<long long>(p.B) * p.Hq * pad;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long x = gtid; x < npad; x += stride) {
      const long long bh = x / pad;
      const size_t idx = static_cast<size_t>(bh) * p.Tpad + p.T + static_cast<int>(x % pad);
      p.Dvec[idx] = 0.f;
      p.lse2[idx] = 0.f;
    }
  }
}

// ============================================================================
// dQ kernel
// ============================================================================
template <int D>
struct DqCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfTileBytes;
  static constexpr int kKStages = 2;
  static constexpr int kVStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTileBytes;
  static constexpr int kOffK = kOffDO + kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kUsed = kOffV + kVStages * kTileBytes + 1024;
  static constexpr int kSmemBytes = kUsed > kOneCtaPerSmSmem ? kUsed : kOneCtaPerSmSmem;
};

constexpr uint32_t kDqColS = 0;     // S fp32; dS bf16 aliases [0, 64)
constexpr uint32_t kDqColDP = 128;  // dP fp32
constexpr uint32_t kDqColDQ = 256;  // dQ fp32 [128 x D]

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = DqCfg<D>;
  constexpr int KS = Cfg::kKStages;
  constexpr int VS = Cfg::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_qdo, bar_kf[KS], bar_ke[KS], bar_vf[VS], bar_ve[VS], bar_s, bar_ds, bar_fin, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nbh = p.B * p.Hq;
  const int qt = p.nT - 1 - static_cast<int>(blockIdx.x) / nbh;  // heaviest first
  const int bh = static_cast<int>(blockIdx.x) % nbh;
  const int b = bh / p.Hq;
  const int h = bh % p.Hq;
  const int kvh = h / p.G;
  const int n_kv = p.causal ? qt + 1 : p.nT;

  if (threadIdx.x == 0) {
    mbar_init(&bar_qdo, 1);
    for (int s = 0; s < KS; ++s) { mbar_init(&bar_kf[s], 1); mbar_init(&bar_ke[s], 1); }
    for (int s = 0; s < VS; ++s) { mbar_init(&bar_vf[s], 1); mbar_init(&bar_ve[s], 1); }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_ds, 128);
    mbar_init(&bar_fin, 1);
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const WaitCtx ctx{&abort_sh, p.status, p.budget_ns, kKidBwdDq};

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
      tma_prefetch_desc(&p.tmap_v);
      tma_prefetch_desc(&p.tmap_do);
      mbar_arrive_expect_tx(&bar_qdo, 2 * Cfg::kTileBytes);
      for (int hf = 0; hf < Cfg::kHalves; ++hf) {
        tma_load_4d(smem + Cfg::kOffQ + hf * kHalfTileBytes, &p.tmap_q, &bar_qdo, hf * 64, h, qt * kTile, b);
        tma_load_4d(smem + Cfg::kOffDO + hf * kHalfTileBytes, &p.tmap_do, &bar_qdo, hf * 64, h, qt * kTile, b);
      }
      int issued_k[KS] = {}, issued_v[VS] = {};
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int ks = j % KS, kn = j / KS;
        if (kn > 0) ok = mbar_wait(&bar_ke[ks], (kn - 1) & 1, ctx, 1);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_kf[ks], Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_4d(smem + Cfg::kOffK + ks * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_k, &bar_kf[ks],
                      hf * 64, kvh, j * kTile, b);
        issued_k[ks]++;
        const int vs = j % VS, vn = j / VS;
        if (vn > 0) ok = mbar_wait(&bar_ve[vs], (vn - 1) & 1, ctx, 2);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_vf[vs], Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_4d(smem + Cfg::kOffV + vs * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_v, &bar_vf[vs],
                      hf * 64, kvh, j * kTile, b);
        issued_v[vs]++;
      }
      if (ok) {
        for (int s = 0; s < KS && ok; ++s)
          if (issued_k[s] > 0) ok = mbar_wait(&bar_ke[s], (issued_k[s] - 1) & 1, ctx, 3);
        for (int s = 0; s < VS && ok; ++s)
          if (issued_v[s] > 0) ok = mbar_wait(&bar_ve[s], (issued_v[s] - 1) & 1, ctx, 4);
      }
      if (!ok) {
        mbar_wait_drain(&bar_qdo, 0, p.budget_ns);
        for (int s = 0; s < KS; ++s)
          if (issued_k[s] > 0) mbar_wait_drain(&bar_kf[s], (issued_k[s] - 1) & 1, p.budget_ns);
        for (int s = 0; s < VS; ++s)
          if (issued_v[s] > 0) mbar_wait_drain(&bar_vf[s], (issued_v[s] - 1) & 1, p.budget_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_q = idesc_bf16_f32(128, D, 0, 1);
      const uint32_t sQ = smem_u32(smem + Cfg::kOffQ);
      const uint32_t sDO = smem_u32(smem + Cfg::kOffDO);
      const uint32_t sK = smem_u32(smem + Cfg::kOffK);
      const uint32_t sV = smem_u32(smem + Cfg::kOffV);
      bool issued = false;
      auto issue_dq = [&](int jj) -> bool {
        if (!mbar_wait(&bar_ds, jj & 1, ctx, 12)) return false;
        tc_fence_after();
        const int ks = jj % KS;
        const uint32_t kbase = sK + ks * Cfg::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bdesc = sdesc_sw128(kbase + kk * 2048, kHalfTileBytes, 1024);
          mma_ts(tmem + kDqColDQ, tmem + kDqColS + kk * 8, bdesc, idesc_q, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_ke[ks]);
        return true;
      };
      bool ok = mbar_wait(&bar_qdo, 0, ctx, 10);
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j > 0) {
          ok = issue_dq(j - 1);
          if (!ok) break;
        }
        const int ks = j % KS, vs = j % VS;
        ok = mbar_wait(&bar_kf[ks], (j / KS) & 1, ctx, 11);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kbase = sK + ks * Cfg::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
          mma_ss(tmem + kDqColS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        issued = true;
        ok = mbar_wait(&bar_vf[vs], (j / VS) & 1, ctx, 13);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vbase = sV + vs * Cfg::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
          mma_ss(tmem + kDqColDP, sdesc_sw128(sDO + off, 16, 1024), sdesc_sw128(vbase + off, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_ve[vs]);
        mma_commit(&bar_s);
      }
      if (ok) ok = issue_dq(n_kv - 1);
      if (ok) {
        mma_commit(&bar_fin);
      } else if (issued) {
        mma_commit(&bar_drain);
        mbar_wait_drain(&bar_drain, 0, p.budget_ns);
      }
    }
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q_idx = qt * kTile + row;
    const bool valid = q_idx < p.T;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + kDqColS;
    const uint32_t tDP = tmem + lane_base + kDqColDP;
    const uint32_t tDQ = tmem + lane_base + kDqColDQ;
    const size_t vec_idx = (static_cast<size_t>(b) * p.Hq + h) * p.Tpad + q_idx;  // < B*Hq*Tpad
    const float lse2_r = p.lse2[vec_idx];
    const float D_r = p.Dvec[vec_idx];
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = warp_wait(&bar_s, j & 1, ctx, 20);
      if (!ok) break;
      tc_fence_after();
      // Columns visible to this row in tile j: [0, lim).
      int lim = kTile;
      if (p.causal && j == qt) lim = row + 1;
      if (!p.causal && (j + 1) * kTile > p.T) lim = p.T - j * kTile;
      if (!valid) lim = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rs[32], rp[32];
        tmem_ld32(tS + c * 32, rs);
        tmem_ld32(tDP + c * 32, rp);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = c * 32 + 2 * i;
          float p0 = ex2_approx(fmaf(__uint_as_float(rs[2 * i]), sl2, -lse2_r));
          float p1 = ex2_approx(fmaf(__uint_as_float(rs[2 * i + 1]), sl2, -lse2_r));
          p0 = col < lim ? p0 : 0.f;
          p1 = col + 1 < lim ? p1 : 0.f;
          const float ds0 = p0 * (__uint_as_float(rp[2 * i]) - D_r);
          const float ds1 = p1 * (__uint_as_float(rp[2 * i + 1]) - D_r);
          pk[i] = pack_bf16x2(ds0, ds1);
        }
        tmem_st16(tS + c * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_ds);
    }
    if (ok) ok = warp_wait(&bar_fin, 0, ctx, 21);
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.dq) +
                           ((static_cast<size_t>(b) * p.T + (valid ? q_idx : 0)) * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tDQ + c * 32, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * p.scale, __uint_as_float(r[2 * i + 1]) * p.scale);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// ============================================================================
// dK / dV kernel
// ============================================================================
template <int D>
struct DkvCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfTileBytes;
  static constexpr int kQStages = 2;
  // stage = [Q tile][dO tile][LSE2 x128 fp32][D x128 fp32]
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffStage = kOffV + kTileBytes;
  static constexpr int kUsed = kOffStage + kQStages * kStageBytes + 1024;
  static constexpr int kSmemBytes = kUsed > kOneCtaPerSmSmem ? kUsed : kOneCtaPerSmSmem;
};

constexpr uint32_t kDkvColS = 0;     // S^T fp32; P^T bf16 aliases [0, 64)
constexpr uint32_t kDkvColDP = 128;  // dP^T fp32; dS^T bf16 aliases [128, 192)
constexpr uint32_t kDkvColDV = 256;  // dV fp32 [128 x D]
// dK follows dV at 256 + D

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkv_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = DkvCfg<D>;
  constexpr int QS = Cfg::kQStages;
  constexpr uint32_t kColDK = kDkvColDV + D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t bar_kv, bar_qf[QS], bar_qe[QS], bar_s, bar_pds, bar_fin, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nbk = p.B * p.Hkv;
  const int kt = static_cast<int>(blockIdx.x) / nbk;  // causal cost falls with the key tile: heaviest first
  const int bk = static_cast<int>(blockIdx.x) % nbk;
  const int b = bk / p.Hkv;
  const int kvh = bk % p.Hkv;
  const int i0 = p.causal ? kt : 0;
  const int ni = p.nT - i0;        // query tiles per head
  const int n_it = p.G * ni;       // (head, query tile) pairs, head-major

  if (threadIdx.x == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < QS; ++s) { mbar_init(&bar_qf[s], 1); mbar_init(&bar_qe[s], 1); }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_pds, 128);
    mbar_init(&bar_fin, 1);
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const WaitCtx ctx{&abort_sh, p.status, p.budget_ns, kKidBwdDkv};

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
      tma_prefetch_desc(&p.tmap_v);
      tma_prefetch_desc(&p.tmap_do);
      mbar_arrive_expect_tx(&bar_kv, 2 * Cfg::kTileBytes);
      for (int hf = 0; hf < Cfg::kHalves; ++hf) {
        tma_load_4d(smem + Cfg::kOffK + hf * kHalfTileBytes, &p.tmap_k, &bar_kv, hf * 64, kvh, kt * kTile, b);
        tma_load_4d(smem + Cfg::kOffV + hf * kHalfTileBytes, &p.tmap_v, &bar_kv, hf * 64, kvh, kt * kTile, b);
      }
      int issued[QS] = {};
      bool ok = true;
      for (int it = 0; it < n_it && ok; ++it) {
        const int st = it % QS, n = it / QS;
        if (n > 0) ok = mbar_wait(&bar_qe[st], (n - 1) & 1, ctx, 1);
        if (!ok) break;
        const int h = kvh * p.G + it / ni;
        const int qt = i0 + it % ni;
        uint8_t* stage = smem + Cfg::kOffStage + st * Cfg::kStageBytes;
        mbar_arrive_expect_tx(&bar_qf[st], 2 * Cfg::kTileBytes + 1024);
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(stage + hf * kHalfTileBytes, &p.tmap_q, &bar_qf[st], hf * 64, h, qt * kTile, b);
          tma_load_4d(stage + Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_do, &bar_qf[st], hf * 64, h,
                      qt * kTile, b);
        }
        const size_t vec = (static_cast<size_t>(b) * p.Hq + h) * p.Tpad + static_cast<size_t>(qt) * kTile;
        bulk_load(stage + 2 * Cfg::kTileBytes, p.lse2 + vec, 512, &bar_qf[st]);
        bulk_load(stage + 2 * Cfg::kTileBytes + 512, p.Dvec + vec, 512, &bar_qf[st]);
        issued[st]++;
      }
      if (ok) {
        for (int s = 0; s < QS && ok; ++s)
          if (issued[s] > 0) ok = mbar_wait(&bar_qe[s], (issued[s] - 1) & 1, ctx, 3);
      }
      if (!ok) {
        mbar_wait_drain(&bar_kv, 0, p.budget_ns);
        for (int s = 0; s < QS; ++s)
          if (issued[s] > 0) mbar_wait_drain(&bar_qf[s], (issued[s] - 1) & 1, p.budget_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);
      const uint32_t sK = smem_u32(smem + Cfg::kOffK);
      const uint32_t sV = smem_u32(smem + Cfg::kOffV);
      const uint32_t sStage = smem_u32(smem + Cfg::kOffStage);
      bool issued = false;
      bool ok = mbar_wait(&bar_kv, 0, ctx, 10);
      for (int it = 0; it < n_it && ok; ++it) {
        const int st = it % QS;
        ok = mbar_wait(&bar_qf[st], (it / QS) & 1, ctx, 11);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sQ = sStage + st * Cfg::kStageBytes;
        const uint32_t sDO = sQ + Cfg::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
          mma_ss(tmem + kDkvColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
          mma_ss(tmem + kDkvColDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        issued = true;
        mma_commit(&bar_s);
        ok = mbar_wait(&bar_pds, it & 1, ctx, 12);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + kDkvColDV, tmem + kDkvColS + kk * 8, sdesc_sw128(sDO + kk * 2048, kHalfTileBytes, 1024),
                 idesc_g, acc);
          mma_ts(tmem + kColDK, tmem + kDkvColDP + kk * 8, sdesc_sw128(sQ + kk * 2048, kHalfTileBytes, 1024),
                 idesc_g, acc);
        }
        mma_commit(&bar_qe[st]);
      }
      if (ok) {
        mma_commit(&bar_fin);
      } else if (issued) {
        mma_commit(&bar_drain);
        mbar_wait_drain(&bar_drain, 0, p.budget_ns);
      }
    }
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // key row within the tile
    const int k_idx = kt * kTile + row;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + kDkvColS;
    const uint32_t tDP = tmem + lane_base + kDkvColDP;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % QS;
      const int qt = i0 + it % ni;
      ok = warp_wait(&bar_s, it & 1, ctx, 20);
      if (!ok) break;
      ok = warp_wait(&bar_qf[st], (it / QS) & 1, ctx, 22);  // LSE2/D vectors of this stage
      if (!ok) break;
      tc_fence_after();
      const float* vlse2 = reinterpret_cast<const float*>(smem + Cfg::kOffStage + st * Cfg::kStageBytes +
                                                          2 * Cfg::kTileBytes);
      const float* vD = vlse2 + kTile;
      // Query columns visible to this key row in tile qt: [lo, hi).
      int lo = 0;
      int hi = p.T - qt * kTile;
      if (hi > kTile) hi = kTile;
      if (p.causal && qt == kt) lo = row;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rs[32], rp[32];
        tmem_ld32(tS + c * 32, rs);
        tmem_ld32(tDP + c * 32, rp);
        tmem_wait_ld();
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = c * 32 + 2 * i;
          float p0 = ex2_approx(fmaf(__uint_as_float(rs[2 * i]), sl2, -vlse2[col]));
          float p1 = ex2_approx(fmaf(__uint_as_float(rs[2 * i + 1]), sl2, -vlse2[col + 1]));
          p0 = (col >= lo && col < hi) ? p0 : 0.f;
          p1 = (col + 1 >= lo && col + 1 < hi) ? p1 : 0.f;
          const float ds0 = p0 * (__uint_as_float(rp[2 * i]) - vD[col]);
          const float ds1 = p1 * (__uint_as_float(rp[2 * i + 1]) - vD[col + 1]);
          pk[i] = pack_bf16x2(p0, p1);
          dk[i] = pack_bf16x2(ds0, ds1);
        }
        tmem_st16(tS + c * 16, pk);
        tmem_st16(tDP + c * 16, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_pds);
    }
    if (ok) ok = warp_wait(&bar_fin, 0, ctx, 21);
    if (ok) {
      tc_fence_after();
      const bool valid = k_idx < p.T;
      const size_t off = ((static_cast<size_t>(b) * p.T + (valid ? k_idx : 0)) * p.Hkv + kvh) * D;
      __nv_bfloat16* dv_row = reinterpret_cast<__nv_bfloat16*>(p.dv) + off;
      __nv_bfloat16* dk_row = reinterpret_cast<__nv_bfloat16*>(p.dk) + off;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        uint32_t pk[16];
        tmem_ld32(tmem + lane_base + kDkvColDV + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dv_row + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
        tmem_ld32(tmem + lane_base + kColDK + c * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * p.scale, __uint_as_float(r[2 * i + 1]) * p.scale);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(dk_row + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

int g_attr_done[64][4] = {};

template <typename K>
cudaError_t ensure_smem_attr(K kernel, int smem, int slot) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !g_attr_done[dev][slot]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    g_attr_done[dev][slot] = 1;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, int d, cudaStream_t stream) {
  const long long nrows = static_cast<long long>(p.B) * p.T * p.Hq;
  const int tpr = d / 8;
  const long long threads = nrows * tpr;
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  if (d == 64)
    bwd_pre_kernel<64><<<grid, 256, 0, stream>>>(p);
  else
    bwd_pre_kernel<128><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, int d, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.B) * p.Hq * p.nT;
  cudaError_t e;
  if (d == 64) {
    if ((e = ensure_smem_attr(bwd_dq_kernel<64>, DqCfg<64>::kSmemBytes, 0)) != cudaSuccess) return e;
    bwd_dq_kernel<64><<<grid, kBwdThreads, DqCfg<64>::kSmemBytes, stream>>>(p);
  } else {
    if ((e = ensure_smem_attr(bwd_dq_kernel<128>, DqCfg<128>::kSmemBytes, 1)) != cudaSuccess) return e;
    bwd_dq_kernel<128><<<grid, kBwdThreads, DqCfg<128>::kSmemBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkv(const BwdParams& p, int d, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.B) * p.Hkv * p.nT;
  cudaError_t e;
  if (d == 64) {
    if ((e = ensure_smem_attr(bwd_dkv_kernel<64>, DkvCfg<64>::kSmemBytes, 2)) != cudaSuccess) return e;
    bwd_dkv_kernel<64><<<grid, kBwdThreads, DkvCfg<64>::kSmemBytes, stream>>>(p);
  } else {
    if ((e = ensure_smem_attr(bwd_dkv_kernel<128>, DkvCfg<128>::kSmemBytes, 3)) != cudaSuccess) return e;
    bwd_dkv_kernel<128><<<grid, kBwdThreads, DkvCfg<128>::kSmemBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gqa
