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
// The dQ and dK/dV passes are two kinds of task of one launch (ordered so the
// heaviest tasks start first), each task owning its outputs:
//   dQ task (per 128-query tile of one query head), key tiles in ascending order:
//     S = Q K^T, dP = dO V^T                  (SS MMAs into TMEM)
//     P = 2^(S*scale*log2e - LSE2), dS = P (dP - D)   (per row, bf16 into TMEM)
//     dQ += dS K                              (TS MMA, K as MN-major operand)
//   dK/dV task (per 128-key tile of one kv head), query heads of the group in
//   ascending order, query tiles from the diagonal on:
//     S^T = K Q^T, dP^T = V dO^T              (SS MMAs)
//     P^T, dS^T per key row                   (bf16 into TMEM)
//     dV += P^T dO, dK += dS^T Q              (TS MMAs, dO/Q as MN-major operands)
// dQ and dK carry the score scale once, in the epilogue.
#include "attn_common.cuh"

namespace gqa {
namespace {

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
// dQ and dK/dV: one launch, two kinds of task.
//
// CTA = 10 warps: warp 0 issues TMA, warp 1 issues tcgen05 MMAs and owns TMEM,
// warps 2-9 are two compute warpgroups; each thread of a warpgroup owns one
// TMEM lane (one row) and the warpgroup owns half of the 128 score columns.
// Blocks [0, n_dkv) are dK/dV tasks (one per key tile, kv head, batch; key tile
// ascending = causal cost descending), blocks [n_dkv, n_dkv + n_dq) are dQ
// tasks (one per query tile, head, batch; query tile descending). Both kinds
// need the 512-column TMEM allocation, so one CTA runs per SM, and the
// heaviest tasks start first.
//
// TMEM columns: [0,128) S (dQ) or S^T (dK/dV), fp32; [128,256) dP or dP^T.
// Warpgroup g writes its bf16 P/dS (64 columns -> 32 packed) over the first
// half of its own fp32 columns: [g*64, g*64+32) and [128+g*64, 128+g*64+32).
// [256, 256+D) dQ or dV; [256+D, 256+2D) dK.
// ============================================================================
constexpr int kMainThreads = 320;
constexpr int kComputeThreads = 256;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColDP = 128;
constexpr uint32_t kColAcc = 256;

template <int D>
struct MainCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfTileBytes;
  // dQ task: [Q][dO] then K ring (2) then V ring (2)
  static constexpr int kDqOffQ = 0;
  static constexpr int kDqOffDO = kTileBytes;
  static constexpr int kDqOffK = 2 * kTileBytes;
  static constexpr int kDqOffV = 4 * kTileBytes;
  static constexpr int kDqBytes = 6 * kTileBytes;
  // dK/dV task: [K][V] then 2 stages of [Q][dO][LSE2 x128][D x128]
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kKvOffK = 0;
  static constexpr int kKvOffV = kTileBytes;
  static constexpr int kKvOffStage = 2 * kTileBytes;
  static constexpr int kKvBytes = 2 * kTileBytes + 2 * kStageBytes;
  static constexpr int kUsed = (kDqBytes > kKvBytes ? kDqBytes : kKvBytes) + 1024;
  static constexpr int kSmemBytes = kUsed > kOneCtaPerSmSmem ? kUsed : kOneCtaPerSmSmem;
};

// TMEM column of the bf16 A operand (P, P^T, dS or dS^T) for K-step kk (16 rows
// of the reduction each); `base` is kColS or kColDP.
__device__ __forceinline__ uint32_t packed_col(uint32_t base, int kk) {
  return base + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
}

// Store 32 packed bf16x2 columns (two x16 stores).
__device__ __forceinline__ void tmem_st_packed32(uint32_t taddr, const uint32_t (&v)[32]) {
  uint32_t a[16], b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = v[i];
    b[i] = v[16 + i];
  }
  tmem_st16(taddr, a);
  tmem_st16(taddr + 16, b);
}

// Store `ncols` (multiple of 32) fp32 columns of this thread's row as bf16 to dst.
template <int NCOLS>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, __nv_bfloat16* dst, float scale, bool valid) {
#pragma unroll
  for (int c = 0; c < NCOLS / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * scale, __uint_as_float(r[2 * i + 1]) * scale);
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kMainThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = MainCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // Barriers. dQ task: fixed = Q+dO, ring[0..1] = K full/empty, ring[2..3] = V full/empty.
  // dK/dV task: fixed = K+V, ring[0..1] = stage full/empty.
  __shared__ uint64_t bar_fixed, bar_full[4], bar_empty[4], bar_s, bar_p, bar_fin, bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_dkv = p.n_dkv_tasks;
  const bool is_dkv = static_cast<int>(blockIdx.x) < n_dkv;

  if (threadIdx.x == 0) {
    mbar_init(&bar_fixed, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_p, kComputeThreads);
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
  const WaitCtx ctx{&abort_sh, p.status, p.budget_ns, kKidBwdMain};
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: N = 128 keys/queries
  constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);    // gradient MMAs: N = D, B MN-major

  // ---------------------------------------------------------------- task decode
  int b, kvh, h = 0, tile, n_it;
  int i0 = 0, ni = 1;  // dK/dV: first query tile and query tiles per head
  if (is_dkv) {
    const int nbk = p.B * p.Hkv;
    tile = static_cast<int>(blockIdx.x) / nbk;
    const int bk = static_cast<int>(blockIdx.x) % nbk;
    b = bk / p.Hkv;
    kvh = bk % p.Hkv;
    i0 = p.causal ? tile : 0;
    ni = p.nT - i0;
    n_it = p.G * ni;
  } else {
    const int t = static_cast<int>(blockIdx.x) - n_dkv;
    const int nbh = p.B * p.Hq;
    tile = p.nT - 1 - t / nbh;
    const int bh = t % nbh;
    b = bh / p.Hq;
    h = bh % p.Hq;
    kvh = h / p.G;
    n_it = p.causal ? tile + 1 : p.nT;
  }

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
      tma_prefetch_desc(&p.tmap_v);
      tma_prefetch_desc(&p.tmap_do);
      int issued[4] = {0, 0, 0, 0};
      bool ok = true;
      if (is_dkv) {
        mbar_arrive_expect_tx(&bar_fixed, 2 * Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(smem + Cfg::kKvOffK + hf * kHalfTileBytes, &p.tmap_k, &bar_fixed, hf * 64, kvh, tile * kTile, b);
          tma_load_4d(smem + Cfg::kKvOffV + hf * kHalfTileBytes, &p.tmap_v, &bar_fixed, hf * 64, kvh, tile * kTile, b);
        }
        for (int it = 0; it < n_it && ok; ++it) {
          const int st = it & 1, n = it >> 1;
          if (n > 0) ok = mbar_wait(&bar_empty[st], (n - 1) & 1, ctx, 1);
          if (!ok) break;
          const int hq = kvh * p.G + it / ni;
          const int qt = i0 + it % ni;
          uint8_t* stage = smem + Cfg::kKvOffStage + st * Cfg::kStageBytes;
          mbar_arrive_expect_tx(&bar_full[st], 2 * Cfg::kTileBytes + 1024);
          for (int hf = 0; hf < Cfg::kHalves; ++hf) {
            tma_load_4d(stage + hf * kHalfTileBytes, &p.tmap_q, &bar_full[st], hf * 64, hq, qt * kTile, b);
            tma_load_4d(stage + Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_do, &bar_full[st], hf * 64, hq,
                        qt * kTile, b);
          }
          const size_t vec = (static_cast<size_t>(b) * p.Hq + hq) * p.Tpad + static_cast<size_t>(qt) * kTile;
          bulk_load(stage + 2 * Cfg::kTileBytes, p.lse2 + vec, 512, &bar_full[st]);
          bulk_load(stage + 2 * Cfg::kTileBytes + 512, p.Dvec + vec, 512, &bar_full[st]);
          issued[st]++;
        }
      } else {
        mbar_arrive_expect_tx(&bar_fixed, 2 * Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(smem + Cfg::kDqOffQ + hf * kHalfTileBytes, &p.tmap_q, &bar_fixed, hf * 64, h, tile * kTile, b);
          tma_load_4d(smem + Cfg::kDqOffDO + hf * kHalfTileBytes, &p.tmap_do, &bar_fixed, hf * 64, h, tile * kTile, b);
        }
        for (int j = 0; j < n_it && ok; ++j) {
          const int st = j & 1, n = j >> 1;
          if (n > 0) ok = mbar_wait(&bar_empty[st], (n - 1) & 1, ctx, 1);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_full[st], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kDqOffK + st * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_k, &bar_full[st],
                        hf * 64, kvh, j * kTile, b);
          issued[st]++;
          if (n > 0) ok = mbar_wait(&bar_empty[2 + st], (n - 1) & 1, ctx, 2);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_full[2 + st], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kDqOffV + st * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_v,
                        &bar_full[2 + st], hf * 64, kvh, j * kTile, b);
          issued[2 + st]++;
        }
      }
      // Wait until every stage is released, so no MMA commit arrives after exit.
      for (int s = 0; s < 4 && ok; ++s)
        if (issued[s] > 0) ok = mbar_wait(&bar_empty[s], (issued[s] - 1) & 1, ctx, 3);
      if (!ok) {
        mbar_wait_drain(&bar_fixed, 0, p.budget_ns);
        for (int s = 0; s < 4; ++s)
          if (issued[s] > 0) mbar_wait_drain(&bar_full[s], (issued[s] - 1) & 1, p.budget_ns);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      bool issued = false;
      bool ok = mbar_wait(&bar_fixed, 0, ctx, 10);
      if (is_dkv) {
        const uint32_t sK = smem_u32(smem + Cfg::kKvOffK);
        const uint32_t sV = smem_u32(smem + Cfg::kKvOffV);
        for (int it = 0; it < n_it && ok; ++it) {
          const int st = it & 1;
          ok = mbar_wait(&bar_full[st], (it >> 1) & 1, ctx, 11);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sQ = smem_u32(smem + Cfg::kKvOffStage + st * Cfg::kStageBytes);
          const uint32_t sDO = sQ + Cfg::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
            mma_ss(tmem + kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
            mma_ss(tmem + kColDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
          issued = true;
          mma_commit(&bar_s);
          ok = mbar_wait(&bar_p, it & 1, ctx, 12);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + kColAcc, tmem + packed_col(kColS, kk),
                   sdesc_sw128(sDO + kk * 2048, kHalfTileBytes, 1024), idesc_g, acc);
            mma_ts(tmem + kColAcc + D, tmem + packed_col(kColDP, kk),
                   sdesc_sw128(sQ + kk * 2048, kHalfTileBytes, 1024), idesc_g, acc);
          }
          mma_commit(&bar_empty[st]);
        }
      } else {
        const uint32_t sQ = smem_u32(smem + Cfg::kDqOffQ);
        const uint32_t sDO = smem_u32(smem + Cfg::kDqOffDO);
        auto issue_dq = [&](int jj) -> bool {
          if (!mbar_wait(&bar_p, jj & 1, ctx, 12)) return false;
          tc_fence_after();
          const int st = jj & 1;
          const uint32_t kbase = smem_u32(smem + Cfg::kDqOffK + st * Cfg::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tmem + kColAcc, tmem + packed_col(kColS, kk), sdesc_sw128(kbase + kk * 2048, kHalfTileBytes, 1024),
                   idesc_g, (jj > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar_empty[st]);
          return true;
        };
        for (int j = 0; j < n_it && ok; ++j) {
          if (j > 0) {
            ok = issue_dq(j - 1);
            if (!ok) break;
          }
          const int st = j & 1;
          ok = mbar_wait(&bar_full[st], (j >> 1) & 1, ctx, 11);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kbase = smem_u32(smem + Cfg::kDqOffK + st * Cfg::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
            mma_ss(tmem + kColS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
          issued = true;
          ok = mbar_wait(&bar_full[2 + st], (j >> 1) & 1, ctx, 13);
          if (!ok) break;
          tc_fence_after();
          const uint32_t vbase = smem_u32(smem + Cfg::kDqOffV + st * Cfg::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
            mma_ss(tmem + kColDP, sdesc_sw128(sDO + off, 16, 1024), sdesc_sw128(vbase + off, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(&bar_empty[2 + st]);
          mma_commit(&bar_s);
        }
        if (ok) ok = issue_dq(n_it - 1);
      }
      if (ok) {
        mma_commit(&bar_fin);
      } else if (issued) {
        mma_commit(&bar_drain);
        mbar_wait_drain(&bar_drain, 0, p.budget_ns);
      }
    }
  } else {
    // ============================================================ compute warpgroups
    const int wg = (warp - 2) >> 2;  // 0 or 1: score columns [wg*64, wg*64+64)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + wg * 64;
    const uint32_t tDP = tmem + lane_base + kColDP + wg * 64;
    const uint64_t sl2x2 = f2_make(p.scale_log2, p.scale_log2);
    bool ok = true;
    if (is_dkv) {
      const int k_idx = tile * kTile + row;
      for (int it = 0; it < n_it; ++it) {
        const int st = it & 1;
        const int qt = i0 + it % ni;
        ok = warp_wait(&bar_s, it & 1, ctx, 20);
        if (!ok) break;
        ok = warp_wait(&bar_full[st], (it >> 1) & 1, ctx, 22);  // LSE2 / D vectors of this stage
        if (!ok) break;
        tc_fence_after();
        uint32_t rs[64], rp[64];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&rs[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&rs[32]));
        tmem_ld32(tDP, *reinterpret_cast<uint32_t(*)[32]>(&rp[0]));
        tmem_ld32(tDP + 32, *reinterpret_cast<uint32_t(*)[32]>(&rp[32]));
        tmem_wait_ld();
        const float* vl = reinterpret_cast<const float*>(smem + Cfg::kKvOffStage + st * Cfg::kStageBytes +
                                                         2 * Cfg::kTileBytes) + wg * 64;
        const float* vd = vl + kTile;
        // Query columns visible to this key row: [lo, hi) relative to this warpgroup's 64 columns.
        const int hi_tile = min(kTile, p.T - qt * kTile);
        const bool masked = (p.causal && qt == tile) || hi_tile < kTile;
        const int lo = ((p.causal && qt == tile) ? row : 0) - wg * 64;
        const int hi = hi_tile - wg * 64;
        uint32_t pk[32], dk[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float4 l4 = *reinterpret_cast<const float4*>(vl + 2 * i);
          const float4 d4 = *reinterpret_cast<const float4*>(vd + 2 * i);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 2 * (i + u);
            const float la = u ? l4.z : l4.x, lb = u ? l4.w : l4.y;
            const float da = u ? d4.z : d4.x, db = u ? d4.w : d4.y;
            const uint64_t sarg = f2_fma(f2_make(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])), sl2x2,
                                         f2_make(-la, -lb));
            float a0, a1;
            f2_split(sarg, a0, a1);
            float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            if (masked) {
              p0 = (c >= lo && c < hi) ? p0 : 0.f;
              p1 = (c + 1 >= lo && c + 1 < hi) ? p1 : 0.f;
            }
            const uint64_t pp = f2_make(p0, p1);
            const uint64_t ds = f2_mul(pp, f2_sub(f2_make(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1])),
                                                  f2_make(da, db)));
            float d0, d1;
            f2_split(ds, d0, d1);
            pk[i + u] = pack_bf16x2(p0, p1);
            dk[i + u] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st_packed32(tS, pk);
        tmem_st_packed32(tDP, dk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p);
      }
      if (ok) ok = warp_wait(&bar_fin, 0, ctx, 21);
      if (ok) {
        tc_fence_after();
        const bool valid = k_idx < p.T;
        const size_t off = ((static_cast<size_t>(b) * p.T + (valid ? k_idx : 0)) * p.Hkv + kvh) * D;
        if (wg == 0)
          store_row_bf16<D>(tmem + lane_base + kColAcc, reinterpret_cast<__nv_bfloat16*>(p.dv) + off, 1.f, valid);
        else
          store_row_bf16<D>(tmem + lane_base + kColAcc + D, reinterpret_cast<__nv_bfloat16*>(p.dk) + off, p.scale,
                            valid);
      }
    } else {
      const int q_idx = tile * kTile + row;
      const bool valid = q_idx < p.T;
      const size_t vec_idx = (static_cast<size_t>(b) * p.Hq + h) * p.Tpad + q_idx;  // < B*Hq*Tpad
      const float lse2_r = p.lse2[vec_idx];
      const float D_r = p.Dvec[vec_idx];
      const uint64_t neg_l2 = f2_make(-lse2_r, -lse2_r);
      const uint64_t Dx2 = f2_make(D_r, D_r);
      for (int j = 0; j < n_it; ++j) {
        ok = warp_wait(&bar_s, j & 1, ctx, 20);
        if (!ok) break;
        tc_fence_after();
        uint32_t rs[64], rp[64];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&rs[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&rs[32]));
        tmem_ld32(tDP, *reinterpret_cast<uint32_t(*)[32]>(&rp[0]));
        tmem_ld32(tDP + 32, *reinterpret_cast<uint32_t(*)[32]>(&rp[32]));
        tmem_wait_ld();
        // Key columns visible to this query row: [0, lim) relative to this warpgroup's 64 columns.
        int lim_tile = kTile;
        if (p.causal && j == tile) lim_tile = row + 1;
        if (!p.causal && (j + 1) * kTile > p.T) lim_tile = p.T - j * kTile;
        const bool masked = (p.causal && j == tile) || (!p.causal && (j + 1) * kTile > p.T) ||
                            (tile + 1) * kTile > p.T;
        const int lim = (valid ? lim_tile : 0) - wg * 64;
        uint32_t dk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = 2 * i;
          const uint64_t sarg =
              f2_fma(f2_make(__uint_as_float(rs[c]), __uint_as_float(rs[c + 1])), sl2x2, neg_l2);
          float a0, a1;
          f2_split(sarg, a0, a1);
          float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
          if (masked) {
            p0 = c < lim ? p0 : 0.f;
            p1 = c + 1 < lim ? p1 : 0.f;
          }
          const uint64_t ds =
              f2_mul(f2_make(p0, p1), f2_sub(f2_make(__uint_as_float(rp[c]), __uint_as_float(rp[c + 1])), Dx2));
          float d0, d1;
          f2_split(ds, d0, d1);
          dk[i] = pack_bf16x2(d0, d1);
        }
        tmem_st_packed32(tS, dk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p);
      }
      if (ok) ok = warp_wait(&bar_fin, 0, ctx, 21);
      if (ok) {
        tc_fence_after();
        const size_t off = ((static_cast<size_t>(b) * p.T + (valid ? q_idx : 0)) * p.Hq + h) * D;
        store_row_bf16<D / 2>(tmem + lane_base + kColAcc + wg * (D / 2),
                              reinterpret_cast<__nv_bfloat16*>(p.dq) + off + wg * (D / 2), p.scale, valid);
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

cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.n_dkv_tasks + p.n_dq_tasks);
  if (grid == 0) return cudaSuccess;
  cudaError_t e;
  if (d == 64) {
    if ((e = ensure_smem_attr(bwd_main_kernel<64>, MainCfg<64>::kSmemBytes, 0)) != cudaSuccess) return e;
    bwd_main_kernel<64><<<grid, kMainThreads, MainCfg<64>::kSmemBytes, stream>>>(p);
  } else {
    if ((e = ensure_smem_attr(bwd_main_kernel<128>, MainCfg<128>::kSmemBytes, 1)) != cudaSuccess) return e;
    bwd_main_kernel<128><<<grid, kMainThreads, MainCfg<128>::kSmemBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gqa
