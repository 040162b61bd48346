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
// negated LSE in log2 units, into the caller's workspace, padded to whole
// 128-row tiles.
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

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// ============================================================================
// Preprocess: D = rowsum(dO * O), -LSE2 = -LSE * log2(e); padded rows get 0.
// Rows are visited in (b, h, t) order: D/8 threads read one 128- or 256-byte
// row of O and dO with 16-byte loads, and the LSE read and the D / -LSE2
// writes of consecutive rows are consecutive in memory.
// ============================================================================
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdPreParams p) {
  constexpr int TPR = D / 8;
  pdl_launch_dependents();
  pdl_wait_previous();
  const long long nrows = static_cast<long long>(p.B) * p.Hq * p.T;
  const long long gtid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = gtid / TPR;  // ((b * Hq + h) * T + t)
  const int part = static_cast<int>(gtid % TPR);
  float acc = 0.f;
  int t = 0;
  long long bh = 0;
  if (r < nrows) {
    t = static_cast<int>(r % p.T);
    bh = r / p.T;
    const int h = static_cast<int>(bh % p.Hq);
    const long long b = bh / p.Hq;
    const long long row = (b * p.T + t) * p.Hq + h;  // memory row of O / dO
    const uint4 a = reinterpret_cast<const uint4*>(p.o)[row * TPR + part];
    const uint4 c = reinterpret_cast<const uint4*>(p.dO)[row * TPR + part];
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
    const size_t idx = static_cast<size_t>(bh) * p.Tpad + t;
    p.Dvec[idx] = acc;
    p.lse2[idx] = -p.lse[static_cast<size_t>(r)] * 1.4426950408889634f;
  }
  // Zero the padding rows [T, Tpad) of every (b, h).
  const int pad = p.Tpad - p.T;
  if (pad > 0) {
    const long long npad = static_cast<long long>(p.B) * p.Hq * pad;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long x = gtid; x < npad; x += stride) {
      const long long pbh = x / pad;
      const size_t idx = static_cast<size_t>(pbh) * p.Tpad + p.T + static_cast<int>(x % pad);
      p.Dvec[idx] = 0.f;
      p.lse2[idx] = 0.f;
    }
  }
}

// ============================================================================
// dQ and dK/dV: one launch, two kinds of task.
//
// CTA = 19 warps: warp 0 issues TMA, warp 1 issues the S and dP MMAs and owns
// TMEM, warps 2-17 are four compute warpgroups, warp 18 issues the gradient MMAs. Each compute thread owns one TMEM lane
// (one row) and its warpgroup owns 32 of the 128 score columns.
//
// Blocks [0, n_dkv) are dK/dV tasks (one per key tile, kv head, batch; key tile
// ascending = causal cost descending); the following n_dq blocks are dQ tasks
// (query tile descending). Both kinds allocate all 512 TMEM columns, so one CTA
// runs per SM and the heaviest tasks start first.
//
// Pipeline per iteration `it` (one 128x128 score tile):
//   compute: load its 32 columns of S(it) and dP(it) into registers and release
//            both accumulators at once (sdp_free); P = 2^(S*scale*log2e - LSE2),
//            dS = P (dP - D) in registers; bf16 P and dS into their own TMEM
//            region once the gradient MMAs of it-1 have read it (pds_free), then
//            pds_full.
//   MMA:     S(it+1), dP(it+1) as soon as sdp_free(it) | gradient MMAs of it on
//            pds_full(it).
// so the tensor core computes the scores of it+1 while the compute warps work on
// it, and the compute warps never wait for a half-read accumulator.
//
// TMEM columns (S and dP are 128 fp32 columns; P and dS 64 columns of bf16 pairs):
//   dQ:        S [0,128) dP [128,256) dS [256,320) dQ [320,320+D)
//   dK/dV 64:  S [0,128) dP [128,256) P [256,320) dS [320,384) dV [384,448) dK [448,512)
//   dK/dV 128: S [0,128) dP [128,256) dV [256,384) dK [384,512); no room for a separate
//              P/dS region, so P goes to S columns [0,64) and dS to [64,128) once every
//              warpgroup has read S (sdp_free), and S(it+1) follows the gradient MMAs.
// Warpgroup g writes the bf16 pairs of its score columns [32g, 32g+32) to columns
// [16g, 16g+16) of the P (dS) region, so the A operand of K-step kk is at 8*kk.
// ============================================================================
constexpr int kMainThreads = 608;
constexpr int kComputeThreads = 512;
constexpr int kGradWarp = 18;  // second MMA issuer (gradient MMAs)

template <int D>
struct MainCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfTileBytes;
  static constexpr int kAuxBytes = 4096;  // 128 rows x 16 bf16, unswizzled K-major (one K-step)
  // dQ task: [Q][dO][QX][DX][ONES], K ring, V ring
  static constexpr int kDqKStages = 3;
  static constexpr int kDqVStages = (D == 64) ? 2 : 1;
  static constexpr int kDqOffQ = 0;
  static constexpr int kDqOffDO = kTileBytes;
  static constexpr int kDqOffQX = 2 * kTileBytes;
  static constexpr int kDqOffDX = kDqOffQX + kAuxBytes;
  static constexpr int kDqOffOnes = kDqOffDX + kAuxBytes;
  static constexpr int kDqOffK = kDqOffOnes + kAuxBytes;
  static constexpr int kDqOffV = kDqOffK + kDqKStages * kTileBytes;
  static constexpr int kDqBytes = kDqOffV + kDqVStages * kTileBytes;
  // dK/dV task: [K][V][ONES], stages of [Q][dO][QX][DX] (d = 128) or
  // [dO][ZERO][Q][QX][DX] (d = 64). At d = 64 the gradient MMAs compute [dV | dK]
  // as one N = 128 chain over the block-diagonal operand [dO | 0] (P steps) and
  // [0 | Q] (dS steps): the zero tile sits between dO and Q so one LBO spans both.
  // N = 64 MMAs run well below the tensor peak when the compute warps stream
  // TMEM at the same time; N = 128 ones do not.
  static constexpr bool kBlockDiag = (D == 64);
  static constexpr int kKvStages = (D == 64) ? 3 : 2;   // Q/dO stages
  static constexpr int kStOffDO = kBlockDiag ? 0 : kTileBytes;
  static constexpr int kStOffZ = kTileBytes;             // d = 64 only
  static constexpr int kStOffQ = kBlockDiag ? 2 * kTileBytes : 0;
  static constexpr int kStOffQX = kBlockDiag ? 3 * kTileBytes : 2 * kTileBytes;
  static constexpr int kStOffDX = kStOffQX + kAuxBytes;
  static constexpr int kStageBytes = kStOffDX + kAuxBytes;
  static constexpr int kKvOffK = 0;
  static constexpr int kKvOffV = kTileBytes;
  static constexpr int kKvOffOnes = 2 * kTileBytes;
  static constexpr int kKvOffStage = 2 * kTileBytes + kAuxBytes;
  static constexpr int kKvBytes = kKvOffStage + kKvStages * kStageBytes;
  static constexpr int kUsed = (kDqBytes > kKvBytes ? kDqBytes : kKvBytes) + 1024;
  static constexpr int kSmemBytes = kUsed > kOneCtaPerSmSmem ? kUsed : kOneCtaPerSmSmem;
  // TMEM columns
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kDqColDS = 256;
  static constexpr uint32_t kDqColAcc = 320;
  static constexpr bool kKvSepPdS = (D == 64);  // dK/dV: P/dS region of its own
  static constexpr uint32_t kKvColP = kKvSepPdS ? 256 : 0;
  static constexpr uint32_t kKvColDS = kKvSepPdS ? 320 : 64;
  static constexpr uint32_t kKvColDV = kKvSepPdS ? 384 : 256;
  static constexpr uint32_t kKvColDK = kKvColDV + D;
  static_assert(kDqColAcc + D <= 512 && kKvColDK + D <= 512, "TMEM columns");
};

// Unswizzled K-major layout of a 128 x 16 bf16 operand: byte offset of (row, 8-column half).
__device__ __forceinline__ uint32_t aux_off(int row, int half) {
  return static_cast<uint32_t>((row >> 3) * 256 + half * 128 + (row & 7) * 16);
}

// The extra K-step that folds a per-row value into an accumulator: a row of this
// operand is [hi(x), lo(x), 0, ...] with hi + lo = x to ~2^-17 relative, and it
// meets a row [1, 1, 0, ...] of the ONES operand, adding x.
__device__ __forceinline__ void write_aux_row(uint8_t* tile, int row, float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
  const uint32_t w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                      (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
  *reinterpret_cast<uint4*>(tile + aux_off(row, 0)) = make_uint4(w0, 0u, 0u, 0u);
  *reinterpret_cast<uint4*>(tile + aux_off(row, 1)) = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ void write_ones_row(uint8_t* tile, int row) {
  const uint32_t one2 = 0x3F803F80u;  // bf16 1.0 in both halves
  *reinterpret_cast<uint4*>(tile + aux_off(row, 0)) = make_uint4(one2, 0u, 0u, 0u);
  *reinterpret_cast<uint4*>(tile + aux_off(row, 1)) = make_uint4(0u, 0u, 0u, 0u);
}

// Store NCOLS (16 or a multiple of 32) fp32 columns of this thread's row as bf16 to dst.
template <int NCOLS>
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, __nv_bfloat16* dst, float scale, bool valid) {
  if constexpr (NCOLS == 16) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * scale, __uint_as_float(r[2 * i + 1]) * scale);
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  } else {
    static_assert(NCOLS % 32 == 0, "NCOLS");
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
}

// This thread's 32 score columns of one tile. The accumulators already hold
// S - LSE2/c and dP - D, so P = 2^(c * s') and dS = P * dp'. Columns outside
// [lo, hi) of the warpgroup's frame are masked (MASKED only). Writes the bf16
// pairs of P (dK/dV only) and dS.
template <bool DKV, bool MASKED>
__device__ __forceinline__ void score_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[32], float sl2, int lo,
                                            int hi, uint32_t (&pk)[16], uint32_t (&dk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float p0 = ex2_approx(__uint_as_float(s[2 * i]) * sl2);
    float p1 = ex2_approx(__uint_as_float(s[2 * i + 1]) * sl2);
    if (MASKED) {
      p0 = (2 * i >= lo && 2 * i < hi) ? p0 : 0.f;
      p1 = (2 * i + 1 >= lo && 2 * i + 1 < hi) ? p1 : 0.f;
    }
    if (DKV) pk[i] = pack_bf16x2(p0, p1);
    dk[i] = pack_bf16x2(p0 * __uint_as_float(dp[2 * i]), p1 * __uint_as_float(dp[2 * i + 1]));
  }
}

// Barriers of one task. Every one of them is at most one phase ahead of any
// waiter: sdp_full(it+1) is committed only after sdp_free(it) completed, which
// needs every compute thread to have passed sdp_full(it); pds_full(it+1) needs
// pds_free(it), which the MMA thread commits only after it saw pds_full(it);
// and the reverse pairs likewise.
struct MainBars {
  uint64_t fixed, full[3], empty[3], vfull[2], vempty[2];
  uint64_t sdp_full;  // MMA -> compute: S(it) and dP(it) are in TMEM
  uint64_t sdp_free;  // compute -> MMA: every thread has S(it), dP(it) in registers
  uint64_t pds_full;  // compute -> MMA: bf16 P/dS of it are in TMEM
  uint64_t pds_free;  // MMA -> compute: the gradient MMAs of it have completed
  uint64_t fin, drain, drain2;
};

struct TaskInfo {
  int b, kvh, h, tile, n_it, i0, ni;
};

// Descriptor offset (in 16-byte units) of K-step kk inside a K-major tile of
// 64-wide halves: 32 bytes per step inside a 128-byte row, a new half every 4 steps.
__device__ __forceinline__ constexpr uint32_t kmaj_step(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * kHalfTileBytes + (kk & 3) * 32) >> 4);
}

// One task of either kind, all roles. Every pipeline depth is a compile-time
// constant and every MMA descriptor is a base plus a constant, so the single
// issuing thread spends a few instructions per MMA.
template <int D, bool DKV>
__device__ __forceinline__ void run_task(const BwdParams& p, uint8_t* smem, MainBars& bars, uint32_t tmem,
                                         const WaitCtx& ctx, const TaskInfo& t, int warp, int lane) {
  using Cfg = MainCfg<D>;
  constexpr bool kSep = DKV ? Cfg::kKvSepPdS : true;           // P/dS region separate from S
  constexpr uint32_t colP = DKV ? Cfg::kKvColP : 0;
  constexpr uint32_t colDS = DKV ? Cfg::kKvColDS : Cfg::kDqColDS;
  constexpr int NST = DKV ? Cfg::kKvStages : Cfg::kDqKStages;  // main ring depth
  constexpr int NV = Cfg::kDqVStages;                         // dQ V ring depth
  constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: N = 128
  constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);    // gradients: N = D, B MN-major
  constexpr uint32_t kTileD = Cfg::kTileBytes >> 4;             // tile stride, descriptor units
  constexpr uint32_t kStageD = Cfg::kStageBytes >> 4;
  const int n_it = t.n_it;
  const float inv_sl2 = 1.f / p.scale_log2;

  if (warp == 0) {
    // ============================================================ producer warp
    // Lane 0 issues TMA and waits; all 32 lanes write the unswizzled ONES / QX / DX
    // operands (4 rows each) from the workspace's -LSE2 and D.
    if (lane == 0) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
      tma_prefetch_desc(&p.tmap_v);
      tma_prefetch_desc(&p.tmap_do);
    }
    int issued[3] = {0, 0, 0}, vissued[2] = {0, 0};
    bool ok = true;
    const size_t vec_bh0 = (static_cast<size_t>(t.b) * p.Hq) * p.Tpad;
    if (lane == 0) mbar_arrive_expect_tx(&bars.fixed, 2 * Cfg::kTileBytes);
    if (DKV) {
      if (lane == 0)
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(smem + Cfg::kKvOffK + hf * kHalfTileBytes, &p.tmap_k, &bars.fixed, hf * 64, t.kvh,
                      t.tile * kTile, t.b);
          tma_load_4d(smem + Cfg::kKvOffV + hf * kHalfTileBytes, &p.tmap_v, &bars.fixed, hf * 64, t.kvh,
                      t.tile * kTile, t.b);
        }
      // -LSE2 and D of the next stage's 128 query rows, 4 per lane, fetched one
      // stage ahead so their latency hides behind the wait for a free stage.
      float vnl[4], vd[4];
      auto fetch = [&](int it) {
        const int hq = t.kvh * p.G + it / t.ni;
        const int qt = t.i0 + it % t.ni;
        const size_t vec = vec_bh0 + static_cast<size_t>(hq) * p.Tpad + static_cast<size_t>(qt) * kTile + lane;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          vnl[k] = __ldg(p.lse2 + vec + 32 * k);
          vd[k] = __ldg(p.Dvec + vec + 32 * k);
        }
      };
      if (n_it > 0) fetch(0);
      for (int r = lane; r < kTile; r += 32) write_ones_row(smem + Cfg::kKvOffOnes, r);
      if (Cfg::kBlockDiag) {
        // the zero tile of every stage (never written by TMA)
        for (int st = 0; st < NST; ++st) {
          uint4* z = reinterpret_cast<uint4*>(smem + Cfg::kKvOffStage + st * Cfg::kStageBytes + Cfg::kStOffZ);
          for (int i = lane; i < Cfg::kTileBytes / 16; i += 32) z[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.fixed);
      for (int it = 0; it < n_it && ok; ++it) {
        const int st = it % NST, n = it / NST;
        if (n > 0 && lane == 0) ok = mbar_wait(&bars.empty[st], (n - 1) & 1, ctx, 1);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int hq = t.kvh * p.G + it / t.ni;
        const int qt = t.i0 + it % t.ni;
        uint8_t* stage = smem + Cfg::kKvOffStage + st * Cfg::kStageBytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.full[st], 2 * Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf) {
            tma_load_4d(stage + Cfg::kStOffQ + hf * kHalfTileBytes, &p.tmap_q, &bars.full[st], hf * 64, hq,
                        qt * kTile, t.b);
            tma_load_4d(stage + Cfg::kStOffDO + hf * kHalfTileBytes, &p.tmap_do, &bars.full[st], hf * 64, hq,
                        qt * kTile, t.b);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          write_aux_row(stage + Cfg::kStOffQX, lane + 32 * k, vnl[k] * inv_sl2);
          write_aux_row(stage + Cfg::kStOffDX, lane + 32 * k, -vd[k]);
        }
        if (it + 1 < n_it) fetch(it + 1);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.full[st]);
        issued[st]++;
      }
    } else {
      if (lane == 0)
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(smem + Cfg::kDqOffQ + hf * kHalfTileBytes, &p.tmap_q, &bars.fixed, hf * 64, t.h,
                      t.tile * kTile, t.b);
          tma_load_4d(smem + Cfg::kDqOffDO + hf * kHalfTileBytes, &p.tmap_do, &bars.fixed, hf * 64, t.h,
                      t.tile * kTile, t.b);
        }
      const size_t vec = vec_bh0 + static_cast<size_t>(t.h) * p.Tpad + static_cast<size_t>(t.tile) * kTile + lane;
      float vnl[4], vd[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        vnl[k] = __ldg(p.lse2 + vec + 32 * k);
        vd[k] = __ldg(p.Dvec + vec + 32 * k);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        write_ones_row(smem + Cfg::kDqOffOnes, lane + 32 * k);
        write_aux_row(smem + Cfg::kDqOffQX, lane + 32 * k, vnl[k] * inv_sl2);
        write_aux_row(smem + Cfg::kDqOffDX, lane + 32 * k, -vd[k]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.fixed);
        for (int j = 0; j < n_it && ok; ++j) {
          const int st = j % NST, n = j / NST;
          if (n > 0) ok = mbar_wait(&bars.empty[st], (n - 1) & 1, ctx, 1);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars.full[st], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kDqOffK + st * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_k, &bars.full[st],
                        hf * 64, t.kvh, j * kTile, t.b);
          issued[st]++;
          const int vs = j % NV, vn = j / NV;
          if (vn > 0) ok = mbar_wait(&bars.vempty[vs], (vn - 1) & 1, ctx, 2);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars.vfull[vs], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kDqOffV + vs * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_v,
                        &bars.vfull[vs], hf * 64, t.kvh, j * kTile, t.b);
          vissued[vs]++;
        }
      }
    }
    if (lane != 0) return;
    // Wait until every stage is released, so no MMA commit arrives after exit.
    for (int s2 = 0; s2 < 3 && ok; ++s2)
      if (issued[s2] > 0) ok = mbar_wait(&bars.empty[s2], (issued[s2] - 1) & 1, ctx, 3);
    for (int s2 = 0; s2 < 2 && ok; ++s2)
      if (vissued[s2] > 0) ok = mbar_wait(&bars.vempty[s2], (vissued[s2] - 1) & 1, ctx, 4);
    if (!ok) {
      mbar_wait_drain(&bars.fixed, 0, p.budget_ns);
      for (int s2 = 0; s2 < 3; ++s2)
        if (issued[s2] > 0) mbar_wait_drain(&bars.full[s2], (issued[s2] - 1) & 1, p.budget_ns);
      for (int s2 = 0; s2 < 2; ++s2)
        if (vissued[s2] > 0) mbar_wait_drain(&bars.vfull[s2], (vissued[s2] - 1) & 1, p.budget_ns);
    }
  } else if (warp == 1 || warp == kGradWarp) {
    // ============================================================ MMA issuers
    // All 32 lanes of an issuing warp run its loop; the elected lane (always lane
    // 0 of the converged warp) issues every MMA and commit, so commits track its
    // MMAs. With a separate P/dS region, warp 1 issues S and dP and warp kGradWarp
    // the gradient MMAs, so neither chain of barrier checks and issues holds up the
    // other; otherwise (dK/dV at d = 128) S(it+1) must follow the gradient MMAs of
    // it and warp 1 issues everything.
    constexpr bool kTwoIssuers = kSep;
    if (!kTwoIssuers && warp == kGradWarp) return;
    // Base descriptors (stage / slot 0); a stage or K-step moves the start address only.
    uint64_t dA_S, dA_P, dB_S, dB_P, dG1, dG2, dXA_S, dXA_P, dXB_S, dXB_P;
    uint32_t strideB_S, strideB_P, strideX;
    if (DKV) {
      const uint32_t st0 = smem_u32(smem + Cfg::kKvOffStage);
      const uint64_t ones = sdesc_noswz(smem_u32(smem + Cfg::kKvOffOnes), 128, 256);
      dA_S = sdesc_sw128(smem_u32(smem + Cfg::kKvOffK), 16, 1024);             // K
      dA_P = sdesc_sw128(smem_u32(smem + Cfg::kKvOffV), 16, 1024);             // V
      dB_S = sdesc_sw128(st0 + Cfg::kStOffQ, 16, 1024);                        // Q   (K-major)
      dB_P = sdesc_sw128(st0 + Cfg::kStOffDO, 16, 1024);                       // dO  (K-major)
      if (Cfg::kBlockDiag) {
        dG1 = sdesc_sw128(st0 + Cfg::kStOffDO, Cfg::kTileBytes, 1024);         // [dO | 0] (MN-major, N = 128)
        dG2 = sdesc_sw128(st0 + Cfg::kStOffZ, Cfg::kTileBytes, 1024);          // [0 | Q]
      } else {
        dG1 = sdesc_sw128(st0 + Cfg::kStOffDO, kHalfTileBytes, 1024);          // dO  (MN-major) for dV
        dG2 = sdesc_sw128(st0 + Cfg::kStOffQ, kHalfTileBytes, 1024);           // Q   (MN-major) for dK
      }
      dXA_S = ones;                                                            // ONES x QX^T  -> -LSE2/c
      dXA_P = ones;                                                            // ONES x DX^T  -> -D
      dXB_S = sdesc_noswz(st0 + Cfg::kStOffQX, 128, 256);
      dXB_P = sdesc_noswz(st0 + Cfg::kStOffDX, 128, 256);
      strideB_S = kStageD;
      strideB_P = kStageD;
      strideX = kStageD;
    } else {
      const uint64_t ones = sdesc_noswz(smem_u32(smem + Cfg::kDqOffOnes), 128, 256);
      dA_S = sdesc_sw128(smem_u32(smem + Cfg::kDqOffQ), 16, 1024);             // Q
      dA_P = sdesc_sw128(smem_u32(smem + Cfg::kDqOffDO), 16, 1024);            // dO
      dB_S = sdesc_sw128(smem_u32(smem + Cfg::kDqOffK), 16, 1024);             // K slot 0 (K-major)
      dB_P = sdesc_sw128(smem_u32(smem + Cfg::kDqOffV), 16, 1024);             // V slot 0 (K-major)
      dG1 = sdesc_sw128(smem_u32(smem + Cfg::kDqOffK), kHalfTileBytes, 1024);  // K slot 0 (MN-major) for dQ
      dG2 = 0;
      dXA_S = sdesc_noswz(smem_u32(smem + Cfg::kDqOffQX), 128, 256);           // QX x ONES^T -> -LSE2/c
      dXA_P = sdesc_noswz(smem_u32(smem + Cfg::kDqOffDX), 128, 256);           // DX x ONES^T -> -D
      dXB_S = ones;
      dXB_P = ones;
      strideB_S = kTileD;
      strideB_P = kTileD;
      strideX = 0;
    }
    bool issued_any = false;
    // S(i); waits for its stage unless the caller already did (dK/dV: one stage carries Q and dO).
    auto issue_S = [&](int i, bool wait_stage) -> bool {
      const int st = i % NST;
      if (wait_stage) {
        if (!warp_wait(&bars.full[st], (i / NST) & 1, ctx, 11)) return false;
        tc_fence_after();
      }
      const uint32_t dst = tmem + Cfg::kColS;
      const uint64_t b0 = dB_S + st * strideB_S;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(dst, dA_S + kmaj_step(kk), b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_ss(dst, dXA_S, dXB_S + st * strideX, idesc_s, 1u);
      }
      __syncwarp();
      issued_any = true;
      return true;
    };
    auto issue_dP = [&](int i, bool wait_stage) -> bool {
      int slot, xst;
      if (DKV) {
        slot = i % NST;
        xst = slot;
        if (wait_stage) {
          if (!warp_wait(&bars.full[slot], (i / NST) & 1, ctx, 13)) return false;
          tc_fence_after();
        }
      } else {
        slot = i % NV;
        xst = 0;
        if (!warp_wait(&bars.vfull[slot], (i / NV) & 1, ctx, 13)) return false;
        tc_fence_after();
      }
      const uint64_t b0 = dB_P + slot * strideB_P;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + Cfg::kColDP, dA_P + kmaj_step(kk), b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
        mma_ss(tmem + Cfg::kColDP, dXA_P, dXB_P + xst * strideX, idesc_s, 1u);
        if (!DKV) mma_commit(&bars.vempty[slot]);
      }
      __syncwarp();
      issued_any = true;
      return true;
    };
    auto issue_grad = [&](int i) {
      const int st = i % NST;
      const uint32_t tP = tmem + colP, tDS = tmem + colDS;
      if (elect_one()) {
        if (DKV && Cfg::kBlockDiag) {
          // [dV | dK] (128 columns) += [P^T | dS^T] x blockdiag(dO, Q): 16 N = 128 steps
          constexpr uint32_t idesc_bd = idesc_bf16_f32(128, 128, 0, 1);
          const uint64_t g1 = dG1 + st * kStageD, g2 = dG2 + st * kStageD;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tmem + Cfg::kKvColDV, tP + kk * 8, g1 + kk * 128, idesc_bd, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tmem + Cfg::kKvColDV, tDS + kk * 8, g2 + kk * 128, idesc_bd, 1u);
        } else if (DKV) {
          const uint64_t g1 = dG1 + st * kStageD, g2 = dG2 + st * kStageD;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + Cfg::kKvColDV, tP + kk * 8, g1 + kk * 128, idesc_g, acc);
            mma_ts(tmem + Cfg::kKvColDK, tDS + kk * 8, g2 + kk * 128, idesc_g, acc);
          }
        } else {
          const uint64_t g1 = dG1 + st * kTileD;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tmem + Cfg::kDqColAcc, tDS + kk * 8, g1 + kk * 128, idesc_g, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars.pds_free);
        mma_commit(&bars.empty[st]);
      }
      __syncwarp();
      issued_any = true;
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };

    bool ok = true;
    if (warp == 1) {
      ok = warp_wait(&bars.fixed, 0, ctx, 10);
      if (ok) {
        tc_fence_after();
        ok = issue_S(0, true);
      }
      if (ok) ok = issue_dP(0, !DKV);
      if (ok) commit(&bars.sdp_full);
    }
    if (kTwoIssuers && warp == 1) {
      // S and dP of it+1 as soon as every compute thread holds S(it), dP(it)
      for (int it = 0; it + 1 < n_it && ok; ++it) {
        ok = warp_wait(&bars.sdp_free, it & 1, ctx, 14);
        if (!ok) break;
        ok = issue_S(it + 1, true);
        if (ok) ok = issue_dP(it + 1, !DKV);
        if (!ok) break;
        commit(&bars.sdp_full);
      }
    } else if (kTwoIssuers) {
      // gradient MMAs of it once its bf16 P/dS are in TMEM
      for (int it = 0; it < n_it && ok; ++it) {
        ok = warp_wait(&bars.pds_full, it & 1, ctx, 12);
        if (!ok) break;
        tc_fence_after();
        issue_grad(it);
      }
      // every S/dP MMA completed before the last P/dS was written
      if (ok) commit(&bars.fin);
    } else {
      for (int it = 0; it < n_it && ok; ++it) {
        const bool has_next = it + 1 < n_it;
        ok = warp_wait(&bars.sdp_free, it & 1, ctx, 14);
        if (!ok) break;
        if (has_next) {
          ok = issue_dP(it + 1, true);
          if (!ok) break;
        }
        ok = warp_wait(&bars.pds_full, it & 1, ctx, 12);
        if (!ok) break;
        tc_fence_after();
        issue_grad(it);
        if (has_next) {
          // P/dS of it live in the S columns: S(it+1) after the gradient MMAs
          ok = issue_S(it + 1, false);
          if (!ok) break;
          commit(&bars.sdp_full);
        }
      }
      if (ok) commit(&bars.fin);
    }
    if (!ok && issued_any) {
      uint64_t* dr = warp == 1 ? &bars.drain : &bars.drain2;
      commit(dr);
      mbar_wait_drain(dr, 0, p.budget_ns);
    }
  } else {
    // ============================================================ compute warpgroups
    const int wg = (warp - 2) >> 2;  // 0..3: score columns [wg*32, wg*32+32)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + Cfg::kColS + wg * 32;
    const uint32_t tDP = tmem + lane_base + Cfg::kColDP + wg * 32;
    const uint32_t tP = tmem + lane_base + colP + wg * 16;
    const uint32_t tDS = tmem + lane_base + colDS + wg * 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    // One tile: S, dP -> registers -> sdp_free; P, dS -> TMEM -> pds_full.
    auto tile = [&](int it, bool masked, int lo, int hi) -> bool {
      if (!warp_wait(&bars.sdp_full, it & 1, ctx, 20)) return false;
      tc_fence_after();
      uint32_t s[32], dp[32];
      tmem_ld32(tS, s);
      tmem_ld32(tDP, dp);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars.sdp_free);
      uint32_t pk[16], dk[16];
      if (masked)
        score_chunk<DKV, true>(s, dp, sl2, lo, hi, pk, dk);
      else
        score_chunk<DKV, false>(s, dp, sl2, lo, hi, pk, dk);
      // The P/dS region must be free: read by the gradient MMAs of it-1 (separate
      // region), or S(it) read by every warpgroup (region inside S).
      if (kSep) {
        if (it > 0 && !warp_wait(&bars.pds_free, (it - 1) & 1, ctx, 22)) return false;
      } else {
        if (!warp_wait(&bars.sdp_free, it & 1, ctx, 23)) return false;
      }
      tc_fence_after();
      if (DKV) tmem_st16(tP, pk);
      tmem_st16(tDS, dk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars.pds_full);
      return true;
    };
    if (DKV) {
      const int k_idx = t.tile * kTile + row;
      for (int it = 0; it < n_it && ok; ++it) {
        const int qt = t.i0 + it % t.ni;
        // Query columns visible to this key row: [lo, hi) in this warpgroup's 32-column frame.
        const int hi_tile = min(kTile, p.T - qt * kTile);
        const bool diag = p.causal && qt == t.tile;
        const int lo = (diag ? row : 0) - wg * 32;
        const int hi = hi_tile - wg * 32;
        ok = tile(it, diag || hi_tile < kTile, lo, hi);
      }
      if (ok) ok = warp_wait(&bars.fin, 0, ctx, 21);
      if (ok) {
        tc_fence_after();
        const bool valid = k_idx < p.T;
        const size_t off = ((static_cast<size_t>(t.b) * p.T + (valid ? k_idx : 0)) * p.Hkv + t.kvh) * D;
        // warpgroups 0, 1: dV halves; 2, 3: dK halves
        const int part = wg & 1;
        if (wg < 2)
          store_row_bf16<D / 2>(tmem + lane_base + Cfg::kKvColDV + part * (D / 2),
                                reinterpret_cast<__nv_bfloat16*>(p.dv) + off + part * (D / 2), 1.f, valid);
        else
          store_row_bf16<D / 2>(tmem + lane_base + Cfg::kKvColDK + part * (D / 2),
                                reinterpret_cast<__nv_bfloat16*>(p.dk) + off + part * (D / 2), p.scale, valid);
      }
    } else {
      const int q_idx = t.tile * kTile + row;
      const bool valid = q_idx < p.T;
      const bool tile_ragged = (t.tile + 1) * kTile > p.T;
      for (int j = 0; j < n_it && ok; ++j) {
        // Key columns visible to this query row: [0, lim) in this warpgroup's 32-column frame.
        const bool diag = p.causal && j == t.tile;
        const bool kv_ragged = !p.causal && (j + 1) * kTile > p.T;
        int lim_tile = kTile;
        if (diag) lim_tile = row + 1;
        if (kv_ragged) lim_tile = p.T - j * kTile;
        const int lim = (valid ? lim_tile : 0) - wg * 32;
        ok = tile(j, diag || kv_ragged || tile_ragged, 0, lim);
      }
      if (ok) ok = warp_wait(&bars.fin, 0, ctx, 21);
      if (ok) {
        tc_fence_after();
        const size_t off = ((static_cast<size_t>(t.b) * p.T + (valid ? q_idx : 0)) * p.Hq + t.h) * D;
        store_row_bf16<D / 4>(tmem + lane_base + Cfg::kDqColAcc + wg * (D / 4),
                              reinterpret_cast<__nv_bfloat16*>(p.dq) + off + wg * (D / 4), p.scale, valid);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kMainThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ MainBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_dkv = p.n_dkv_tasks;
  const bool is_dkv = static_cast<int>(blockIdx.x) < n_dkv;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bars.fixed, 2);  // TMA bytes + the producer warp's aux operands
    for (int s = 0; s < 3; ++s) {
      mbar_init(&bars.full[s], is_dkv ? 2 : 1);  // dK/dV stages also carry aux operands
      mbar_init(&bars.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vempty[s], 1);
    }
    mbar_init(&bars.sdp_full, 1);
    mbar_init(&bars.sdp_free, kComputeThreads);
    mbar_init(&bars.pds_full, kComputeThreads);
    mbar_init(&bars.pds_free, 1);
    mbar_init(&bars.fin, 1);
    mbar_init(&bars.drain, 1);
    mbar_init(&bars.drain2, 1);
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
  pdl_wait_previous();  // the workspace is written by the preprocess kernel

  TaskInfo t;
  t.h = 0;
  t.i0 = 0;
  t.ni = 1;
  if (is_dkv) {
    const int nbk = p.B * p.Hkv;
    t.tile = static_cast<int>(blockIdx.x) / nbk;
    const int bk = static_cast<int>(blockIdx.x) % nbk;
    t.b = bk / p.Hkv;
    t.kvh = bk % p.Hkv;
    t.i0 = p.causal ? t.tile : 0;
    t.ni = p.nT - t.i0;
    t.n_it = p.G * t.ni;
  } else {
    const int q = static_cast<int>(blockIdx.x) - n_dkv;
    const int nbh = p.B * p.Hq;
    t.tile = p.nT - 1 - q / nbh;
    const int bh = q % nbh;
    t.b = bh / p.Hq;
    t.h = bh % p.Hq;
    t.kvh = t.h / p.G;
    t.n_it = p.causal ? t.tile + 1 : p.nT;
  }
  if (is_dkv)
    run_task<D, true>(p, smem, bars, tmem, ctx, t, warp, lane);
  else
    run_task<D, false>(p, smem, bars, tmem, ctx, t, warp, lane);

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
  cudaError_t e = d == 64 ? launch_pdl(bwd_pre_kernel<64>, grid, 256, 0, stream, p)
                          : launch_pdl(bwd_pre_kernel<128>, grid, 256, 0, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.n_dkv_tasks + p.n_dq_tasks);
  if (grid == 0) return cudaSuccess;
  cudaError_t e;
  if (d == 64) {
    if ((e = ensure_smem_attr(bwd_main_kernel<64>, MainCfg<64>::kSmemBytes, 0)) != cudaSuccess) return e;
    e = launch_pdl(bwd_main_kernel<64>, grid, kMainThreads, MainCfg<64>::kSmemBytes, stream, p);
    if (e != cudaSuccess) return e;
  } else {
    if ((e = ensure_smem_attr(bwd_main_kernel<128>, MainCfg<128>::kSmemBytes, 1)) != cudaSuccess) return e;
    e = launch_pdl(bwd_main_kernel<128>, grid, kMainThreads, MainCfg<128>::kSmemBytes, stream, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace gqa
