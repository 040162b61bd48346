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
//     S = Q K^T, dP = dO V^T                  (MMAs into TMEM; at d = 128 S is a
//                                              TS MMA with Q copied to TMEM)
//     P = 2^(S*scale*log2e - LSE2), dS = P (dP - D)   (per row, bf16 into TMEM)
//     dQ += dS K                              (TS MMA, K as MN-major operand)
//   dK/dV task (per 128-key tile of one kv head), query heads of the group in
//   ascending order, query tiles from the diagonal on:
//     S^T = K Q^T, dP^T = V dO^T              (SS MMAs)
//     P^T, dS^T per key row                   (bf16 into TMEM)
//     dV += P^T dO, dK += dS^T Q              (TS MMAs, dO/Q as MN-major operands)
// dQ and dK carry the score scale once, in the epilogue; with the rotary
// embedding (a separate template instance) the epilogue also turns them back by
// the inverse rotation, since the kernel differentiates with respect to the
// rotated q and k.
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
// A block covers PreCfg<D>::kRows consecutive rows t of one (b, h), a row being
// read as D/8 16-byte chunks by as many threads (each thread takes two rows, so
// four loads are in flight; O and dO are addressed through their token and batch
// strides), so the block's rows of D / -LSE2 are consecutive in memory; the rows
// [T, Tpad) of the last block are written as zeros.
// ============================================================================
constexpr int kPreThreads = 256;

template <int D>
struct PreCfg {
  static constexpr int kTPR = D / 8;                        // threads per row
  static constexpr int kRows = 2 * (kPreThreads / kTPR);    // rows per block
};

template <int D>
__global__ void __launch_bounds__(kPreThreads) bwd_pre_kernel(const BwdPreParams p) {
  constexpr int TPR = PreCfg<D>::kTPR;
  constexpr int RPB = PreCfg<D>::kRows;
  pdl_launch_dependents();
  pdl_wait_previous();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.sched[0] = 0u;  // task counters of the dQ / dK/dV launch
    p.sched[1] = 0u;
  }
  const int n_tb = (p.Tpad + RPB - 1) / RPB;  // row blocks per (b, h)
  const int bh = static_cast<int>(blockIdx.x) / n_tb;
  const int t0 = (static_cast<int>(blockIdx.x) - bh * n_tb) * RPB + static_cast<int>(threadIdx.x) / TPR;
  const int part = static_cast<int>(threadIdx.x) % TPR;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  constexpr int kHalf = RPB / 2;  // a thread's second row is kHalf further
  // this thread's 16 bytes of row (b, t0, h) of O and dO; its second row is kHalf tokens on
  const uint4* po = reinterpret_cast<const uint4*>(p.o) + (b * p.o_sb16 + t0 * p.o_st16 + h * TPR + part);
  const uint4* pd = reinterpret_cast<const uint4*>(p.dO) + (b * p.do_sb16 + t0 * p.do_st16 + h * TPR + part);
  uint4 a[2], c[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = t0 + i * kHalf;
    a[i] = c[i] = make_uint4(0u, 0u, 0u, 0u);
    if (t < p.T) {
      a[i] = po[i * kHalf * p.o_st16];
      c[i] = pd[i * kHalf * p.do_st16];
    }
  }
  float lse[2] = {0.f, 0.f};
  if (part == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = t0 + i * kHalf;
      if (t < p.T) lse[i] = p.lse[static_cast<size_t>(bh) * p.T + t];
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float acc = bf16lo(a[i].x) * bf16lo(c[i].x);
    acc = fmaf(bf16hi(a[i].x), bf16hi(c[i].x), acc);
    acc = fmaf(bf16lo(a[i].y), bf16lo(c[i].y), acc);
    acc = fmaf(bf16hi(a[i].y), bf16hi(c[i].y), acc);
    acc = fmaf(bf16lo(a[i].z), bf16lo(c[i].z), acc);
    acc = fmaf(bf16hi(a[i].z), bf16hi(c[i].z), acc);
    acc = fmaf(bf16lo(a[i].w), bf16lo(c[i].w), acc);
    acc = fmaf(bf16hi(a[i].w), bf16hi(c[i].w), acc);
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int t = t0 + i * kHalf;
    if (part == 0 && t < p.Tpad) {
      // rows past T: zeros (acc is 0 there, and so is lse)
      const size_t idx = static_cast<size_t>(bh) * p.Tpad + t;
      p.Dvec[idx] = acc;
      p.lse2[idx] = t < p.T ? -lse[i] * 1.4426950408889634f : 0.f;
    }
  }
}

// ============================================================================
// dQ and dK/dV: one persistent launch, two kinds of task.
//
// One CTA per SM (all 512 TMEM columns) loops over tasks taken from a counter
// in the workspace, heaviest first: tasks [0, n_dkv) are dK/dV tasks (one per
// key tile, kv head, batch; key tile ascending = causal cost descending), the
// following n_dq are dQ tasks (query tile descending). Every output element is
// written by the one task that owns it, so which CTA runs a task does not
// change any result.
//
// CTA = 19 warps: warp 0 fetches tasks and issues TMA, warp 1 issues the S and
// dP MMAs and owns TMEM, warps 2-17 are four compute warpgroups, warp 18 issues
// the gradient MMAs. Each compute thread owns one TMEM lane (one row) and its
// warpgroup owns 32 of the 128 score columns.
//
// Pipeline per score tile (global index G, counted over all tasks of the CTA):
//   compute: load its 32 columns of S(G) and dP(G) into registers and release
//            both accumulators at once (sdp_free); P = 2^(S*scale*log2e - LSE2),
//            dS = P (dP - D) in registers; bf16 P and dS into their own TMEM
//            region once the gradient MMAs of G-1 have read it (pds_free), then
//            pds_full.
//   MMA:     S(G+1), dP(G+1) as soon as sdp_free(G) | gradient MMAs of G on
//            pds_full(G).
// so the tensor core computes the scores of G+1 while the compute warps work on
// G. d = 128 dK/dV tiles have no TMEM room for a P/dS region of their own: P and
// dS go over dP's columns, S(G+1) still follows sdp_free(G) (which there means
// "every thread holds S(G)"), dP(G+1) follows the gradient MMAs of G on warp 18,
// and the compute warps form P from S before they wait for dP (dp_full), then write
// P and dS over their warpgroup's own dP columns (no wait: each thread overwrites
// only the cells it has just read). Across a task
// boundary the next task is published (and its operands start loading) while this
// task's last tiles run; its first scores follow its fixed
// operands and first K (or Q/dO) tile.
// Per task: fixed_full (its fixed operands are in shared memory), fixed_free
// (its last S/dP MMAs are done, the fixed operands may be replaced), acc_full
// (its last gradient MMAs are done), acc_free (the epilogue has read its
// accumulators, the next task's first gradient MMA may overwrite them).
// The dK/dV stages at d = 128 (two stages of 72 KB: no room for a third) have a
// barrier pair for dO and one for Q: the gradient MMAs run as a dV chain then a dK
// chain, and dO's slot is refilled as soon as the dV chain is done, so the next
// tile's dP MMA no longer waits for the whole stage to be reloaded (a clock trace
// put that load on the tile loop's critical path; the kernel is 6.7% faster at
// T = 8192 with identical results).
//
// TMEM columns (S and dP are 128 fp32 columns; P and dS 64 columns of bf16 pairs):
//   dQ:        S [0,128) dP [128,256) dS [256,320) dQ [320,320+D)
//   dK/dV 64:  S [0,128) dP [128,256) P [256,320) dS [320,384) dV [384,448) dK [448,512)
//   dK/dV 128: S [0,128) dP [128,256) dV [256,384) dK [384,512); no room for a separate
//              P/dS region, so warpgroup g puts its P pairs in dP columns
//              [128+32g, 128+32g+16) and its dS pairs in the next 16 (its own dP
//              columns), and dP(G+1) follows the gradient MMAs of G (warp 18 issues it
//              right after them; warp 1 issues S).
// Elsewhere warpgroup g writes the bf16 pairs of its score columns [32g, 32g+32) to
// columns [16g, 16g+16) of the P (dS) region, so the A operand of K-step kk is at 8*kk.
// ============================================================================
constexpr int kMainThreads = 608;
constexpr int kComputeThreads = 512;
constexpr int kGradWarp = 18;       // second MMA issuer (gradient MMAs)
constexpr int kTaskConsumers = 18;  // warps 1..18 each take every task from the producer

// Ring depths the barrier arrays of MainBars hold.
constexpr int kMaxKvStages = 4, kMaxDqKStages = 4, kMaxDqVStages = 3;

template <int D>
struct MainCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfTileBytes;
  static constexpr int kAuxBytes = 4096;  // 128 rows x 16 bf16, unswizzled K-major (one K-step)
  // d = 64: one row-term tile per dK/dV stage carries both terms (-LSE2/c in its
  // columns 0-1, -D in 2-3), and two ONES operands pick one pair each; d = 128 keeps
  // a tile per term (its Q and dO slots are freed at different times) and one ONES.
  static constexpr bool kCombAux = (D == 64);
  static constexpr int kOffOnes = 0;      // both layouts: the ONES operand(s), written once
  static constexpr int kOffOnesP = kCombAux ? kAuxBytes : kOffOnes;
  static constexpr int kAuxRegion = kCombAux ? 2 * kAuxBytes : kAuxBytes;
  // Fixed operands of a task (dQ: Q, dO, QX, DX; dK/dV: K, V) are double-buffered
  // at d = 64, so the next task's are loaded while this task runs.
  static constexpr int kNF = (D == 64) ? 2 : 1;
  // dQ task: fixed buffers [Q][dO], K ring, V ring (its row terms stay in registers).
  // At d = 64 the rings take the room the dK/dV layout needs anyway (four K and
  // three V stages: 0.7-1.2% faster than three and two at T = 3000-4096).
  static constexpr int kDqKStages = (D == 64) ? 4 : 3;
  static constexpr int kDqVStages = (D == 64) ? 3 : 2;
  static constexpr int kDqFixBytes = 2 * kTileBytes;
  // A CTA takes its tasks in index order, every dK/dV task before any dQ task, so
  // the dQ layout may reuse the ONES region, which only dK/dV tasks read: at d = 128
  // that makes room for a second V stage. At d = 64 its fixed buffers stay where the
  // dK/dV ones are, since an epilogue's output rows are staged in them.
  static constexpr int kDqBase = (D == 64) ? kAuxRegion : 0;
  static constexpr int kDqOffQ = kDqBase;  // buffer 0; buffer f adds f * kDqFixBytes
  static constexpr int kDqOffDO = kDqOffQ + kTileBytes;
  static constexpr int kDqOffK = kDqBase + kNF * kDqFixBytes;
  static constexpr int kDqOffV = kDqOffK + kDqKStages * kTileBytes;
  static constexpr int kDqBytes = kDqOffV + kDqVStages * kTileBytes;
  // dK/dV task: fixed buffers [K][V], then the ring of stages [Q][dO][QX][DX].
  // The two gradient chains (dV += P^T dO, dK += dS^T Q) are separate N = D MMAs:
  // at d = 64 a single N = 128 chain over block-diagonal operands (half of it
  // multiplying zeros) measured 8-10% slower overall.
  // Q/dO stages. At d = 64 a stage is busy from its load (~1.6 us from the L2 under
  // load, attn_probe_tma) until the tile's gradient MMAs finish, about two tile
  // periods later: two stages measured 18% slower than three, and the fourth (room
  // made by the shared row-term tile and the staging in the fixed buffers) 6% faster.
  static constexpr int kKvStages = (D == 64) ? 4 : 2;
  // d = 128: each stage's dO and Q have their own barriers (see MainBars)
  static constexpr bool kSplitStage = (D == 128);
  static constexpr int kKvFixBytes = 2 * kTileBytes;
  static constexpr int kKvOffK = kAuxRegion;            // buffer 0; buffer f adds f * kKvFixBytes
  static constexpr int kKvOffV = kKvOffK + kTileBytes;
  static constexpr int kKvOffStages = kAuxRegion + kNF * kKvFixBytes;
  static constexpr int kStageBytes = 2 * kTileBytes + (kCombAux ? 1 : 2) * kAuxBytes;
  static constexpr int kKvBytes = kKvOffStages + kKvStages * kStageBytes;
  static_assert(kKvStages <= kMaxKvStages && kDqKStages <= kMaxDqKStages && kDqVStages <= kMaxDqVStages &&
                    kNF <= 2,
                "a ring is deeper than its barrier arrays");
  __host__ __device__ static constexpr int st_q(int s) { return kKvOffStages + s * kStageBytes; }
  __host__ __device__ static constexpr int st_do(int s) { return st_q(s) + kTileBytes; }
  __host__ __device__ static constexpr int st_qx(int s) { return st_q(s) + 2 * kTileBytes; }
  __host__ __device__ static constexpr int st_dx(int s) { return kCombAux ? st_qx(s) : st_qx(s) + kAuxBytes; }
  // d = 64 epilogue: each compute warp stages its 32 rows of bf16 output (dK/dV:
  // 32 columns, dQ: 16) in a region of its own and stores them with one TMA box.
  // The regions lie in the task's own fixed buffer, which no MMA reads once the
  // task's accumulators are complete; the producer reloads that buffer only after
  // the stores have read it (stg_free). At d = 128 rows are stored directly from
  // registers.
  static constexpr bool kTmaStore = (D == 64);
  static constexpr int kOutWarpBytes = 2048;
  static_assert(!kTmaStore || (kNF == 2 && 16 * kOutWarpBytes <= kKvFixBytes && 16 * kOutWarpBytes <= kDqFixBytes),
                "the staging regions fit in a fixed buffer");
  __host__ __device__ static constexpr int stage_out(bool dkv, int f, int warp) {
    return (dkv ? kKvOffK + f * kKvFixBytes : kDqOffQ + f * kDqFixBytes) + warp * kOutWarpBytes;
  }
  static constexpr int kUsed = (kDqBytes > kKvBytes ? kDqBytes : kKvBytes) + 1024;
  static constexpr int kSmemBytes = kUsed > kOneCtaPerSmSmem ? kUsed : kOneCtaPerSmSmem;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // TMEM columns
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kDqColDS = 256;
  static constexpr uint32_t kDqColAcc = 320;
  // d = 128 dQ tasks: Q is copied to the 64 free columns at the end of TMEM once per
  // task and S runs as a TS MMA (SS MMAs with N = 128 reach ~60% of the tensor
  // rate, TS ~86%). Measured 0.8% faster at d = 128; at d = 64, Q and dO in TMEM
  // and both S and dP as TS gave the same bits but no gain, so d = 64 keeps SS.
  static constexpr bool kDqTsS = (D == 128);
  static constexpr uint32_t kDqColQA = 448;
  static constexpr bool kKvSepPdS = (D == 64);  // dK/dV: P/dS region of its own
  // d = 128 dK/dV: P and dS go over dP's columns, so S(G+1) can be computed as soon
  // as every compute thread holds S(G); dP(G+1) follows the gradient MMAs of G
  // (warp 18), and the compute warps start the exponentials of G+1 before dP(G+1)
  // has landed.
  static constexpr bool kLateDP = !kKvSepPdS;
  // (d = 128: P and dS are interleaved per warpgroup over the dP columns, see
  // grad_mmas_split; these two name the region for the other paths)
  static constexpr uint32_t kKvColP = kKvSepPdS ? 256 : kColDP;
  static constexpr uint32_t kKvColDS = kKvSepPdS ? 320 : kColDP + 64;
  static constexpr uint32_t kKvColDV = kKvSepPdS ? 384 : 256;
  static constexpr uint32_t kKvColDK = kKvColDV + D;
  static_assert(kDqColAcc + D <= 512 && kKvColDK + D <= 512, "TMEM columns");
  static_assert(!kDqTsS || (kDqColAcc + D <= kDqColQA && kDqColQA + D / 2 <= 512), "TMEM columns of Q");
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

// A row of a ONES operand: bf16 1.0 in columns 2*pair and 2*pair + 1, zeros elsewhere.
__device__ __forceinline__ void write_ones_row(uint8_t* tile, int row, int pair = 0) {
  const uint32_t one2 = 0x3F803F80u;  // bf16 1.0 in both halves
  *reinterpret_cast<uint4*>(tile + aux_off(row, 0)) =
      make_uint4(pair == 0 ? one2 : 0u, pair == 1 ? one2 : 0u, 0u, 0u);
  *reinterpret_cast<uint4*>(tile + aux_off(row, 1)) = make_uint4(0u, 0u, 0u, 0u);
}

// Two row terms in one row of a row-term operand: x in columns 0-1, y in 2-3 (each
// as hi + lo), met by the ONES operand with pair 0 or pair 1.
__device__ __forceinline__ void write_aux_row2(uint8_t* tile, int row, float x, float y) {
  auto split = [](float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    return static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
  };
  *reinterpret_cast<uint4*>(tile + aux_off(row, 0)) = make_uint4(split(x), split(y), 0u, 0u);
  *reinterpret_cast<uint4*>(tile + aux_off(row, 1)) = make_uint4(0u, 0u, 0u, 0u);
}

// Load NC (16 or a multiple of 32) fp32 accumulator columns of this thread's row.
template <int NC>
__device__ __forceinline__ void load_acc(uint32_t taddr, uint32_t (&r)[NC]) {
  if constexpr (NC == 16) {
    tmem_ld16(taddr, r);
  } else {
    static_assert(NC % 32 == 0, "NC");
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) tmem_ld32(taddr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
  }
}

// Store NC accumulator values of one row as bf16 (times scale) to dst.
template <int NC>
__device__ __forceinline__ void store_acc_bf16(const uint32_t (&r)[NC], __nv_bfloat16* dst, float scale) {
#pragma unroll
  for (int v = 0; v < NC / 8; ++v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * i]) * scale, __uint_as_float(r[8 * v + 2 * i + 1]) * scale);
    reinterpret_cast<uint4*>(dst)[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// This thread's 32 score columns of one tile. dK/dV tasks: the accumulators
// already hold S - LSE2/c and dP - D (the row terms differ per column there and
// were folded in by an extra K-step), so P = 2^(c * s') and dS = P * dp'. dQ
// tasks: the thread's row is fixed for the whole task, so its row terms come in
// as nl = -LSE2 and nd = -D and P = 2^(c * s + nl), dS = P * (dp + nd): no fold
// MMA. Columns outside [lo, hi) of the warpgroup's frame are masked (MASKED
// only). Writes the bf16 pairs of P (dK/dV only) and dS.
template <bool DKV, bool MASKED>
__device__ __forceinline__ void score_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[32], float sl2, int lo,
                                            int hi, uint32_t (&pk)[16], uint32_t (&dk)[16], float nl = 0.f,
                                            float nd = 0.f) {
  // column pairs through packed fp32 multiplies (same rounding as scalar ones)
  const uint64_t c2 = f2_make(sl2, sl2);
  const uint64_t nl2 = f2_make(nl, nl), nd2 = f2_make(nd, nd);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0, x1;
    if (DKV)
      f2_split(f2_mul(f2_make(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2), x0, x1);
    else
      f2_split(f2_fma(f2_make(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, nl2), x0, x1);
    float p0 = ex2_approx(x0);
    float p1 = ex2_approx(x1);
    if (MASKED) {
      p0 = (2 * i >= lo && 2 * i < hi) ? p0 : 0.f;
      p1 = (2 * i + 1 >= lo && 2 * i + 1 < hi) ? p1 : 0.f;
    }
    if (DKV) pk[i] = pack_bf16x2(p0, p1);
    float d0, d1;
    if (DKV)
      f2_split(f2_mul(f2_make(p0, p1), f2_make(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1]))), d0, d1);
    else
      f2_split(f2_mul(f2_make(p0, p1), f2_add(f2_make(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), nd2)),
               d0, d1);
    dk[i] = pack_bf16x2(d0, d1);
  }
}

// score_chunk<true, MASKED> in two halves, for d = 128 dK/dV tiles, whose dP lands
// after S: P (fp32, kept for dS, and its bf16 pairs) from S alone, then dS from P
// and dP. The same operations per element as score_chunk, so the same bits.
template <bool MASKED>
__device__ __forceinline__ void score_p(const uint32_t (&s)[32], float sl2, int lo, int hi, float (&pf)[32],
                                        uint32_t (&pk)[16]) {
  const uint64_t c2 = f2_make(sl2, sl2);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float x0, x1;
    f2_split(f2_mul(f2_make(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2), x0, x1);
    float p0 = ex2_approx(x0);
    float p1 = ex2_approx(x1);
    if (MASKED) {
      p0 = (2 * i >= lo && 2 * i < hi) ? p0 : 0.f;
      p1 = (2 * i + 1 >= lo && 2 * i + 1 < hi) ? p1 : 0.f;
    }
    pk[i] = pack_bf16x2(p0, p1);
    pf[2 * i] = p0;
    pf[2 * i + 1] = p1;
  }
}

// dS of column pairs [8h, 8h + 8) from their 16 dP values.
__device__ __forceinline__ void score_ds_half(const float (&pf)[32], const uint32_t (&dp)[16], int h,
                                              uint32_t (&dk)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float d0, d1;
    f2_split(f2_mul(f2_make(pf[16 * h + 2 * i], pf[16 * h + 2 * i + 1]),
                    f2_make(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1]))),
             d0, d1);
    dk[8 * h + i] = pack_bf16x2(d0, d1);
  }
}

// Every barrier is at most one phase ahead of any waiter: sdp_full(G+1) is
// committed only after sdp_free(G) completed, which needs every compute thread
// to have passed sdp_full(G); pds_full(G+1) needs pds_free(G), which is committed
// only after pds_full(G) was seen; fixed_full of a buffer is produced again only
// after its fixed_free was seen, which needs that fixed_full; acc_free(n) needs acc_full(n)
// and acc_full(n+1) needs acc_free(n); task_full(n+2) needs task_empty(n); dp_full(G+1)
// follows the gradient MMAs of G, which need pds_full(G), given only after dp_full(G)
// was seen; stg_free(n+2) needs task n+2's fixed operands, loaded only after
// stg_free(n) was seen.
struct alignas(16) MainBars {
  uint64_t task_full[2], task_empty[2];   // producer <-> every other warp: next task index
  uint64_t fixed_full[2], fixed_free[2];   // per fixed buffer: operands loaded / no longer read
  uint64_t stg_free[2];  // per fixed buffer (d = 64): the epilogue's TMA stores have read their rows there
  // dK/dV stage ring. d = 64: q_full/q_empty cover the whole stage (Q, dO and their
  // row terms). d = 128: q_* cover Q and -LSE2, do_* cover dO and -D, so the dO slot
  // is refilled once the dV MMAs are done while the dK MMAs still read Q.
  uint64_t q_full[kMaxKvStages], q_empty[kMaxKvStages];
  uint64_t do_full[kMaxKvStages], do_empty[kMaxKvStages];
  uint64_t k_full[kMaxDqKStages], k_empty[kMaxDqKStages];  // dQ K and V rings
  uint64_t v_full[kMaxDqVStages], v_empty[kMaxDqVStages];
  uint64_t sdp_full;  // MMA -> compute: S(G) and dP(G) are in TMEM
  uint64_t sdp_free;  // compute -> MMA: every thread has S(G), dP(G) in registers (d = 128 dK/dV: S(G))
  uint64_t dp_full;   // d = 128 dK/dV: MMA (warp 18) -> compute: dP(G) is in TMEM
  uint64_t pds_full;  // compute -> MMA: bf16 P/dS of G are in TMEM
  uint64_t pds_free;  // MMA -> compute: the gradient MMAs of G have completed
  uint64_t acc_full;  // MMA -> compute (and producer): every MMA of the task is done
  uint64_t acc_free;  // compute -> MMA: the task's accumulators are in registers
  uint64_t drain, drain2;
};

struct TaskInfo {
  int dkv, b, kvh, h, tile, n_it, i0, ni;
};

__device__ __forceinline__ TaskInfo decode_task(const BwdParams& p, int id) {
  TaskInfo t;
  t.h = 0;
  t.i0 = 0;
  t.ni = 1;
  if (id < p.n_dkv_tasks) {
    t.dkv = 1;
    // key tile ascending = causal cost descending, within a group or over all groups
    int bk;
    if (p.dkv_group_major) {
      bk = fdiv(id, p.fd_nt);
      t.tile = id - bk * p.nT;
    } else {
      t.tile = fdiv(id, p.fd_bk);
      bk = id - t.tile * (p.B * p.Hkv);
    }
    t.b = fdiv(bk, p.fd_hkv);
    t.kvh = bk - t.b * p.Hkv;
    t.i0 = p.causal ? t.tile : 0;
    t.ni = p.nT - t.i0;
    t.n_it = p.G * t.ni;
  } else {
    t.dkv = 0;
    const int q = id - p.n_dkv_tasks;
    if (p.dq_group_major) {
      // group (b, kv head), then query tile descending, then the group's query heads
      const int grp = fdiv(q, p.fd_ntg);
      const int rem = q - grp * (p.nT * p.G);
      const int qt = fdiv(rem, p.fd_g);
      t.tile = p.nT - 1 - qt;
      t.b = fdiv(grp, p.fd_hkv);
      t.kvh = grp - t.b * p.Hkv;
      t.h = t.kvh * p.G + (rem - qt * p.G);
    } else {
      const int qt = fdiv(q, p.fd_bh);
      t.tile = p.nT - 1 - qt;
      const int bh = q - qt * (p.B * p.Hq);
      t.b = fdiv(bh, p.fd_hq);
      t.h = bh - t.b * p.Hq;
      t.kvh = fdiv(t.h, p.fd_g);
    }
    t.n_it = p.causal ? t.tile + 1 : p.nT;
  }
  return t;
}

// Descriptor offset (in 16-byte units) of K-step kk inside a K-major tile of
// 64-wide halves: 32 bytes per step inside a 128-byte row, a new half every 4 steps.
__device__ __forceinline__ constexpr uint32_t kmaj_step(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * kHalfTileBytes + (kk & 3) * 32) >> 4);
}

// Lane 0 waits, the warp agrees on the outcome.
__device__ __forceinline__ bool lane0_wait(uint64_t* bar, uint32_t parity, const WaitCtx& c, unsigned where,
                                           int lane) {
  bool ok = true;
  if (lane == 0) ok = mbar_wait(bar, parity, c, where);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Task n of this CTA as published by the producer (-1: no more); every consumer
// warp arrives once on task_empty after reading it.
__device__ __forceinline__ int recv_task(MainBars& bars, const volatile int* slot, int n, const WaitCtx& ctx,
                                         int lane, bool& ok) {
  ok = warp_wait(&bars.task_full[n & 1], (n >> 1) & 1, ctx, 40);
  const int id = ok ? slot[n & 1] : -1;
  __syncwarp();
  if (ok && lane == 0) mbar_arrive(&bars.task_empty[n & 1]);
  return id;
}

// ============================================================================ producer
template <int D>
__device__ __forceinline__ void producer_role(const BwdParams& p, uint8_t* smem, MainBars& bars, volatile int* slot,
                                              TaskInfo* ring,
                                              const WaitCtx& ctx, int lane) {
  using Cfg = MainCfg<D>;
  constexpr int NKV = Cfg::kKvStages, NK = Cfg::kDqKStages, NV = Cfg::kDqVStages, NF = Cfg::kNF;
  const int n_tasks = p.n_dkv_tasks + p.n_dq_tasks;
  const float inv_sl2 = 1.f / p.scale_log2;
  if (lane == 0) {
    tma_prefetch_desc(&p.tmap_q);
    tma_prefetch_desc(&p.tmap_k);
    tma_prefetch_desc(&p.tmap_v);
    tma_prefetch_desc(&p.tmap_do);
  }
  for (int r = lane; r < kTile; r += 32) {
    write_ones_row(smem + Cfg::kOffOnes, r);
    if (Cfg::kCombAux) write_ones_row(smem + Cfg::kOffOnesP, r, 1);
  }
  fence_proxy_async_smem();
  __syncwarp();
  int kv_used = 0, q_used = 0, n = 0, n_fixed = 0, prev_kind = -1;
  bool ok = true;
  for (;; ++n) {
    int id = -1;
    if (lane == 0) {
      const int x = static_cast<int>(atomicAdd(p.sched, 1u));
      id = x < n_tasks ? x : -1;
    }
    id = __shfl_sync(0xffffffffu, id, 0);
    // Decoded once here (FastDiv divisions by the launch's sizes); the other warps
    // read it from the ring.
    TaskInfo t{};
    if (id >= 0) t = decode_task(p, id);
    // dK/dV task: row terms (-LSE2, D; 4 rows per lane) of its first stage's query
    // tile. Their loads are issued here so the latency overlaps the waits below
    // instead of holding up the task's first operand loads. (A dQ task's compute
    // threads read their own row's terms.)
    float vnl[4], vd[4];
    const size_t vec_bh0 = (static_cast<size_t>(t.b) * p.Hq) * p.Tpad;
    if (id >= 0 && t.dkv) {
      const size_t vec = vec_bh0 + static_cast<size_t>(t.kvh * p.G) * p.Tpad + static_cast<size_t>(t.i0) * kTile + lane;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        vnl[k] = __ldg(p.lse2 + vec + 32 * k);
        vd[k] = __ldg(p.Dvec + vec + 32 * k);
      }
    }
    if (n >= 2) ok = lane0_wait(&bars.task_empty[n & 1], ((n - 2) >> 1) & 1, ctx, 41, lane);
    // Pace on acc_free: the compute warps finish the epilogue of n-1 only after
    // they received task n, so waiting for epilogue n-2 here keeps this warp in
    // step with that barrier for the wait on n-1 below.
    if (ok && n >= 2) ok = lane0_wait(&bars.acc_free, (n - 2) & 1, ctx, 44, lane);
    if (!ok) break;
    if (lane == 0) {
      if (id >= 0) ring[n & 3] = t;
      slot[n & 1] = id;
      mbar_arrive(&bars.task_full[n & 1]);
    }
    if (id < 0) break;
    // Fixed buffer f held task n-NF, free once that task's last S/dP MMAs are
    // done; a change of layout needs every MMA of the previous task done (its
    // epilogue has read the accumulators, so they are).
    const int f = n % NF, fu = n / NF;
    if (fu > 0) ok = lane0_wait(&bars.fixed_free[f], (fu - 1) & 1, ctx, 42, lane);
    // (its task's epilogue staged its output rows there: their stores must have read them)
    if (Cfg::kTmaStore && ok && fu > 0) ok = lane0_wait(&bars.stg_free[f], (fu - 1) & 1, ctx, 45, lane);
    if (ok && n > 0 && t.dkv != prev_kind) ok = lane0_wait(&bars.acc_free, (n - 1) & 1, ctx, 43, lane);
    if (!ok) break;
    uint64_t* fbar = &bars.fixed_full[f];
    if (lane == 0) mbar_arrive_expect_tx(fbar, 2 * Cfg::kTileBytes);
    ++n_fixed;
    if (t.dkv) {
      uint8_t* fix = smem + f * Cfg::kKvFixBytes;
      if (lane == 0)
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(fix + Cfg::kKvOffK + hf * kHalfTileBytes, &p.tmap_k, fbar, hf * 64, t.kvh, t.tile * kTile, t.b);
          tma_load_4d(fix + Cfg::kKvOffV + hf * kHalfTileBytes, &p.tmap_v, fbar, hf * 64, t.kvh, t.tile * kTile, t.b);
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(fbar);
      // -LSE2 and D of the next stage's 128 query rows, 4 per lane, fetched one
      // stage ahead so their latency hides behind the wait for a free stage (the
      // first stage's above).
      // (query head, query tile) of stages it and it + 1 as running counters:
      // it = (hq - kvh * G) * ni + (qt - i0)
      int hq = t.kvh * p.G, qt = t.i0, hq_n = hq, qt_n = qt;
      auto fetch = [&]() {
        const size_t vec = vec_bh0 + static_cast<size_t>(hq_n) * p.Tpad + static_cast<size_t>(qt_n) * kTile + lane;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          vnl[k] = __ldg(p.lse2 + vec + 32 * k);
          vd[k] = __ldg(p.Dvec + vec + 32 * k);
        }
      };
      for (int it = 0; it < t.n_it && ok; ++it, ++kv_used) {
        const int st = kv_used % NKV, u = kv_used / NKV;
        if constexpr (Cfg::kSplitStage) {
          // dO and its row term first (the dP MMA needs them first, and their slot is
          // freed by the dV MMAs), then Q and its row term (freed by the dK MMAs)
          if (u > 0) ok = lane0_wait(&bars.do_empty[st], (u - 1) & 1, ctx, 1, lane);
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars.do_full[st], Cfg::kTileBytes);
            for (int hf = 0; hf < Cfg::kHalves; ++hf)
              tma_load_4d(smem + Cfg::st_do(st) + hf * kHalfTileBytes, &p.tmap_do, &bars.do_full[st], hf * 64, hq,
                          qt * kTile, t.b);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) write_aux_row(smem + Cfg::st_dx(st), lane + 32 * k, -vd[k]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.do_full[st]);
          if (u > 0) ok = lane0_wait(&bars.q_empty[st], (u - 1) & 1, ctx, 5, lane);
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars.q_full[st], Cfg::kTileBytes);
            for (int hf = 0; hf < Cfg::kHalves; ++hf)
              tma_load_4d(smem + Cfg::st_q(st) + hf * kHalfTileBytes, &p.tmap_q, &bars.q_full[st], hf * 64, hq,
                          qt * kTile, t.b);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) write_aux_row(smem + Cfg::st_qx(st), lane + 32 * k, vnl[k] * inv_sl2);
        } else {
          if (u > 0) ok = lane0_wait(&bars.q_empty[st], (u - 1) & 1, ctx, 1, lane);
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars.q_full[st], 2 * Cfg::kTileBytes);
            for (int hf = 0; hf < Cfg::kHalves; ++hf) {
              tma_load_4d(smem + Cfg::st_q(st) + hf * kHalfTileBytes, &p.tmap_q, &bars.q_full[st], hf * 64, hq,
                          qt * kTile, t.b);
              tma_load_4d(smem + Cfg::st_do(st) + hf * kHalfTileBytes, &p.tmap_do, &bars.q_full[st], hf * 64, hq,
                          qt * kTile, t.b);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (Cfg::kCombAux) {
              write_aux_row2(smem + Cfg::st_qx(st), lane + 32 * k, vnl[k] * inv_sl2, -vd[k]);
            } else {
              write_aux_row(smem + Cfg::st_qx(st), lane + 32 * k, vnl[k] * inv_sl2);
              write_aux_row(smem + Cfg::st_dx(st), lane + 32 * k, -vd[k]);
            }
          }
        }
        if (++qt_n == p.nT) {
          qt_n = t.i0;
          ++hq_n;
        }
        if (it + 1 < t.n_it) fetch();
        hq = hq_n;
        qt = qt_n;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.q_full[st]);
      }
    } else {
      uint8_t* fix = smem + f * Cfg::kDqFixBytes;
      if (lane == 0)
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tma_load_4d(fix + Cfg::kDqOffQ + hf * kHalfTileBytes, &p.tmap_q, fbar, hf * 64, t.h, t.tile * kTile, t.b);
          tma_load_4d(fix + Cfg::kDqOffDO + hf * kHalfTileBytes, &p.tmap_do, fbar, hf * 64, t.h, t.tile * kTile, t.b);
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(fbar);
      for (int j = 0; j < t.n_it && ok; ++j, ++q_used) {
        const int ks = q_used % NK, ku = q_used / NK;
        if (ku > 0) ok = lane0_wait(&bars.k_empty[ks], (ku - 1) & 1, ctx, 1, lane);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.k_full[ks], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kDqOffK + ks * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_k,
                        &bars.k_full[ks], hf * 64, t.kvh, j * kTile, t.b);
        }
        const int vs = q_used % NV, vu = q_used / NV;
        if (vu > 0) ok = lane0_wait(&bars.v_empty[vs], (vu - 1) & 1, ctx, 2, lane);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.v_full[vs], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kDqOffV + vs * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_v,
                        &bars.v_full[vs], hf * 64, t.kvh, j * kTile, t.b);
        }
      }
    }
    if (!ok) break;
    prev_kind = t.dkv;
  }
  if (lane != 0) return;
  // Let every commit on a barrier of this CTA land before it exits: the last
  // fixed_free and the last release of every ring slot.
  for (int f = 0; f < NF && ok; ++f) {
    const int uses = n_fixed / NF + (f < n_fixed % NF ? 1 : 0);
    if (uses > 0) ok = mbar_wait(&bars.fixed_free[f], (uses - 1) & 1, ctx, 3);
  }
  for (int s2 = 0; s2 < NKV && ok; ++s2) {
    const int uses = kv_used / NKV + (s2 < kv_used % NKV ? 1 : 0);
    if (uses > 0) ok = mbar_wait(&bars.q_empty[s2], (uses - 1) & 1, ctx, 4);
    if (Cfg::kSplitStage && ok && uses > 0) ok = mbar_wait(&bars.do_empty[s2], (uses - 1) & 1, ctx, 4);
  }
  for (int s2 = 0; s2 < NK && ok; ++s2) {
    const int uses = q_used / NK + (s2 < q_used % NK ? 1 : 0);
    if (uses > 0) ok = mbar_wait(&bars.k_empty[s2], (uses - 1) & 1, ctx, 4);
  }
  for (int s2 = 0; s2 < NV && ok; ++s2) {
    const int uses = q_used / NV + (s2 < q_used % NV ? 1 : 0);
    if (uses > 0) ok = mbar_wait(&bars.v_empty[s2], (uses - 1) & 1, ctx, 4);
  }
  if (!ok) {
    // Abort path: let every load already issued land before the CTA exits.
    for (int f = 0; f < NF; ++f) {
      const int uses = n_fixed / NF + (f < n_fixed % NF ? 1 : 0);
      if (uses > 0) mbar_wait_drain(&bars.fixed_full[f], (uses - 1) & 1, p.budget_ns);
    }
    for (int s2 = 0; s2 < NKV; ++s2) {
      const int uses = kv_used / NKV + (s2 < kv_used % NKV ? 1 : 0);
      if (uses > 0) mbar_wait_drain(&bars.q_full[s2], (uses - 1) & 1, p.budget_ns);
      if (Cfg::kSplitStage && uses > 0) mbar_wait_drain(&bars.do_full[s2], (uses - 1) & 1, p.budget_ns);
    }
    for (int s2 = 0; s2 < NK; ++s2) {
      const int uses = q_used / NK + (s2 < q_used % NK ? 1 : 0);
      if (uses > 0) mbar_wait_drain(&bars.k_full[s2], (uses - 1) & 1, p.budget_ns);
    }
    for (int s2 = 0; s2 < NV; ++s2) {
      const int uses = q_used / NV + (s2 < q_used % NV ? 1 : 0);
      if (uses > 0) mbar_wait_drain(&bars.v_full[s2], (uses - 1) & 1, p.budget_ns);
    }
  }
}

// ============================================================================ MMA issuers
// All 32 lanes of an issuing warp run its loop; the elected lane (always lane 0
// of the converged warp) issues every MMA and commit, so commits track its MMAs.
template <int D>
struct MmaCtx {
  using Cfg = MainCfg<D>;
  static constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: N = 128
  static constexpr uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);    // gradients: N = D, B MN-major
  static constexpr uint32_t kTileD = Cfg::kTileBytes >> 4;  // descriptor units (16 bytes)
  // every dK/dV stage operand moves by one stage stride
  static constexpr uint32_t kStQ = Cfg::kStageBytes >> 4, kStDO = kStQ, kStX = kStQ, kStG1 = kStQ, kStG2 = kStQ;
  uint32_t tmem;
  // dK/dV descriptors (fixed buffer 0, stage 0)
  uint64_t kvA_S, kvA_P, kvB_S, kvB_P, kvG1, kvG2, kvXB_S, kvXB_P;
  // dQ descriptors (fixed buffer 0, ring slot 0)
  uint64_t qA_S, qA_P, qB_S, qB_P, qG1;
  uint64_t ones, ones_p;  // ONES operands of the S and dP folds (the same at d = 128)

  __device__ __forceinline__ void init(uint8_t* smem, uint32_t tm) {
    tmem = tm;
    const uint32_t b = smem_u32(smem);
    ones = sdesc_noswz(b + Cfg::kOffOnes, 128, 256);
    ones_p = sdesc_noswz(b + Cfg::kOffOnesP, 128, 256);
    kvA_S = sdesc_sw128(b + Cfg::kKvOffK, 16, 1024);  // K
    kvA_P = sdesc_sw128(b + Cfg::kKvOffV, 16, 1024);  // V
    kvB_S = sdesc_sw128(b + Cfg::st_q(0), 16, 1024);   // Q  (K-major)
    kvB_P = sdesc_sw128(b + Cfg::st_do(0), 16, 1024);  // dO (K-major)
    kvG1 = sdesc_sw128(b + Cfg::st_do(0), kHalfTileBytes, 1024);  // dO (MN-major) for dV
    kvG2 = sdesc_sw128(b + Cfg::st_q(0), kHalfTileBytes, 1024);   // Q  (MN-major) for dK
    kvXB_S = sdesc_noswz(b + Cfg::st_qx(0), 128, 256);  // ONES x QX^T -> -LSE2/c
    kvXB_P = sdesc_noswz(b + Cfg::st_dx(0), 128, 256);  // ONES x DX^T -> -D
    qA_S = sdesc_sw128(b + Cfg::kDqOffQ, 16, 1024);             // Q
    qA_P = sdesc_sw128(b + Cfg::kDqOffDO, 16, 1024);            // dO
    qB_S = sdesc_sw128(b + Cfg::kDqOffK, 16, 1024);             // K slot 0 (K-major)
    qB_P = sdesc_sw128(b + Cfg::kDqOffV, 16, 1024);             // V slot 0 (K-major)
    qG1 = sdesc_sw128(b + Cfg::kDqOffK, kHalfTileBytes, 1024);  // K slot 0 (MN-major) for dQ
  }
  // S = A_S B_S^T (+ the row-term step for dK/dV) into columns [0,128); f: fixed
  // buffer, bslot: ring slot of B.
  template <bool DKV>
  __device__ __forceinline__ void s_mmas(int f, int bslot) const {
    const uint32_t dst = tmem + Cfg::kColS;
    if (DKV) {
      const uint64_t a = kvA_S + f * (Cfg::kKvFixBytes >> 4);
      const uint64_t b0 = kvB_S + bslot * kStQ;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) mma_ss(dst, a + kmaj_step(kk), b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
      mma_ss(dst, ones, kvXB_S + bslot * kStX, idesc_s, 1u);
    } else {
      const uint64_t fo = f * (Cfg::kDqFixBytes >> 4);
      const uint64_t b0 = qB_S + bslot * kTileD;
      if constexpr (Cfg::kDqTsS) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(dst, tmem + Cfg::kDqColQA + kk * 8, b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
      } else {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(dst, qA_S + fo + kmaj_step(kk), b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
      }
    }
  }
  template <bool DKV>
  __device__ __forceinline__ void dp_mmas(int f, int bslot) const {
    const uint32_t dst = tmem + Cfg::kColDP;
    if (DKV) {
      const uint64_t a = kvA_P + f * (Cfg::kKvFixBytes >> 4);
      const uint64_t b0 = kvB_P + bslot * kStDO;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) mma_ss(dst, a + kmaj_step(kk), b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
      mma_ss(dst, ones_p, kvXB_P + bslot * kStX, idesc_s, 1u);
    } else {
      const uint64_t fo = f * (Cfg::kDqFixBytes >> 4);
      const uint64_t b0 = qB_P + bslot * kTileD;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(dst, qA_P + fo + kmaj_step(kk), b0 + kmaj_step(kk), idesc_s, kk > 0 ? 1u : 0u);
    }
  }
  // d = 128 dQ task: its Q into TMEM (one fixed buffer), ahead of its S MMAs. The
  // columns were last read by the previous dQ task's S MMAs (done: this task's
  // fixed operands were loaded only after its fixed_free) or written by a dK/dV
  // task's dK accumulator (read out: a change of task kind waits for acc_free).
  __device__ __forceinline__ void copy_q_to_tmem(int f) const {
    const uint64_t fo = f * (Cfg::kDqFixBytes >> 4);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) tmem_cp_128x256b(tmem + Cfg::kDqColQA + kk * 8, qA_S + fo + kmaj_step(kk));
  }
  // dK/dV gradient MMAs as two chains, dV first, with a commit on `do_free` between
  // them so that the dO slot is refilled while the dK chain still reads Q.
  // d = 128: warpgroup g's P pairs (query columns [32g, 32g+32)) sit in dP columns
  // [32g, 32g+16) and its dS pairs in [32g+16, 32g+32), so K-step kk reads warpgroup kk/2.
  __device__ __forceinline__ void grad_mmas_split(int bslot, bool first, uint64_t* do_free) const {
    static_assert(Cfg::kLateDP, "P and dS over dP's columns");
    const uint32_t tBase = tmem + Cfg::kColDP;
    const uint64_t g1 = kvG1 + bslot * kStG1, g2 = kvG2 + bslot * kStG2;
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      mma_ts(tmem + Cfg::kKvColDV, tBase + 32 * (kk >> 1) + 8 * (kk & 1), g1 + kk * 128, idesc_g,
             (!first || kk > 0) ? 1u : 0u);
    mma_commit(do_free);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      mma_ts(tmem + Cfg::kKvColDK, tBase + 32 * (kk >> 1) + 16 + 8 * (kk & 1), g2 + kk * 128, idesc_g,
             (!first || kk > 0) ? 1u : 0u);
  }
  // Gradient MMAs of one tile; `first` starts the task's accumulators.
  template <bool DKV>
  __device__ __forceinline__ void grad_mmas(int bslot, bool first) const {
    if (DKV) {
      const uint32_t tP = tmem + Cfg::kKvColP, tDS = tmem + Cfg::kKvColDS;
      const uint64_t g1 = kvG1 + bslot * kStG1, g2 = kvG2 + bslot * kStG2;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
        mma_ts(tmem + Cfg::kKvColDV, tP + kk * 8, g1 + kk * 128, idesc_g, acc);
        mma_ts(tmem + Cfg::kKvColDK, tDS + kk * 8, g2 + kk * 128, idesc_g, acc);
      }
    } else {
      const uint32_t tDS = tmem + Cfg::kDqColDS;
      const uint64_t g1 = qG1 + bslot * kTileD;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_ts(tmem + Cfg::kDqColAcc, tDS + kk * 8, g1 + kk * 128, idesc_g, (!first || kk > 0) ? 1u : 0u);
    }
  }
};

__device__ __forceinline__ void commit_one(uint64_t* bar) {
  if (elect_one()) mma_commit(bar);
  __syncwarp();
}

// Position in an operand ring of N slots: slot and phase parity of the next use.
template <int N>
struct RingPos {
  int slot, phase;
  __device__ __forceinline__ explicit RingPos(int used) : slot(used % N), phase((used / N) & 1) {}
  __device__ __forceinline__ void next() {
    if (++slot == N) {
      slot = 0;
      phase ^= 1;
    }
  }
};

// Warp 1, one task: S and dP of every tile (only S of dK/dV tiles at d = 128,
// where the dP MMA must follow the gradient MMAs of the previous tile and warp 18
// issues it). sdp_full and fixed_free expect two arrivals per phase: warp 1 gives
// both when it issued both S and dP; for a d = 128 dK/dV tile sdp_full reports S
// alone (two commits after it) and fixed_free gets one arrival from each warp.
template <int D, bool DKV>
__device__ __forceinline__ bool sdp_task(const MmaCtx<D>& m, MainBars& bars, const WaitCtx& ctx, int n_it, int f,
                                         int& G, int used, bool& issued) {
  using Cfg = MainCfg<D>;
  constexpr bool dp_here = !DKV || !Cfg::kLateDP;  // this warp issues dP as well as S
  RingPos<DKV ? Cfg::kKvStages : Cfg::kDqKStages> rb(used);
  RingPos<Cfg::kDqVStages> rv(used);
  bool ok = true;
  for (int it = 0; it < n_it && ok; ++it, ++G, rb.next(), rv.next()) {
    // S(G), dP(G) as soon as the compute warps hold S(G-1), dP(G-1). The K (or
    // Q/dO stage) operand is waited for first; in dQ tasks V only before dP, so
    // a late V tile (its ring is refilled only when dP(G-1) completes) does not
    // hold up S.
    // dK/dV: the S MMA needs Q and its row term (d = 128: their own barrier), at d = 64 the
    // dP MMA dO as well (one barrier for the stage)
    ok = warp_wait(DKV ? &bars.q_full[rb.slot] : &bars.k_full[rb.slot], rb.phase, ctx, 11);
    if (ok && G > 0) ok = warp_wait(&bars.sdp_free, (G - 1) & 1, ctx, 14);
    if (!ok) break;
    tc_fence_after();
    if (elect_one()) {
      m.template s_mmas<DKV>(f, rb.slot);
      mma_commit(&bars.sdp_full);
      if (DKV) {
        if (dp_here) m.template dp_mmas<DKV>(f, rb.slot);
        mma_commit(&bars.sdp_full);  // (d = 128: the phase's second arrival, S alone)
      }
    }
    __syncwarp();
    if (!DKV) {
      ok = warp_wait(&bars.v_full[rv.slot], rv.phase, ctx, 13);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        m.template dp_mmas<DKV>(f, rv.slot);
        mma_commit(&bars.v_empty[rv.slot]);
        mma_commit(&bars.sdp_full);
      }
      __syncwarp();
    }
    issued = true;
  }
  if (!ok) return false;
  // every S/dP MMA of this warp for the task is issued: the fixed operands are
  // free once they complete
  if (elect_one()) {
    mma_commit(&bars.fixed_free[f]);
    if (dp_here) mma_commit(&bars.fixed_free[f]);
  }
  __syncwarp();
  return true;
}

template <int D>
__device__ __forceinline__ void sdp_issuer_role(const BwdParams& p, uint8_t* smem, MainBars& bars,
                                                const volatile int* slot, const TaskInfo* ring, uint32_t tmem,
                                                const WaitCtx& ctx, int lane) {
  using Cfg = MainCfg<D>;
  MmaCtx<D> m;
  m.init(smem, tmem);
  int n = 0, G = 0, kv_used = 0, q_used = 0;
  bool ok = true, issued = false;
  for (;; ++n) {
    const int id = recv_task(bars, slot, n, ctx, lane, ok);
    if (!ok || id < 0) break;
    const TaskInfo t = ring[n & 3];
    const int f = n % Cfg::kNF;
    ok = warp_wait(&bars.fixed_full[f], (n / Cfg::kNF) & 1, ctx, 10);
    if (!ok) break;
    tc_fence_after();
    if (Cfg::kDqTsS && !t.dkv) {
      if (elect_one()) m.copy_q_to_tmem(f);
      __syncwarp();
    }
    if (t.dkv) {
      ok = sdp_task<D, true>(m, bars, ctx, t.n_it, f, G, kv_used, issued);
      kv_used += t.n_it;
    } else {
      ok = sdp_task<D, false>(m, bars, ctx, t.n_it, f, G, q_used, issued);
      q_used += t.n_it;
    }
    if (!ok) break;
  }
  if (!ok && issued) {
    commit_one(&bars.drain);
    mbar_wait_drain(&bars.drain, 0, p.budget_ns);
  }
}

// Warp 18, one task: the gradient MMAs of every tile, and at d = 128 the dP MMAs
// of dK/dV tiles, issued right after the gradient MMAs of the previous tile that
// read P and dS from the same TMEM columns. Steps it = 0..n_it: gradient MMAs of
// tile it-1, then (dP here) dP of tile it.
template <int D, bool DKV>
__device__ __forceinline__ bool grad_task(const MmaCtx<D>& m, MainBars& bars, const WaitCtx& ctx, int n_it, int f,
                                          int n, int G, int used, bool& issued) {
  using Cfg = MainCfg<D>;
  constexpr bool dp_here = DKV && Cfg::kLateDP;
  RingPos<DKV ? Cfg::kKvStages : Cfg::kDqKStages> rg(used);  // stage of tile it-1 (gradient operands)
  RingPos<Cfg::kKvStages> rs(used);                          // stage of tile it (dP operands)
  bool ok = true;
  if (dp_here) {
    ok = warp_wait(&bars.fixed_full[f], (n / Cfg::kNF) & 1, ctx, 17);
    if (!ok) return false;
  }
  for (int it = 0; it <= n_it && ok; ++it) {
    if (it > 0) {
      const int g = G + it - 1;
      ok = warp_wait(&bars.pds_full, g & 1, ctx, 12);
      if (ok && it == 1 && n > 0) ok = warp_wait(&bars.acc_free, (n - 1) & 1, ctx, 15);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        if constexpr (DKV && Cfg::kSplitStage)
          m.grad_mmas_split(rg.slot, it == 1, &bars.do_empty[rg.slot]);
        else
          m.template grad_mmas<DKV>(rg.slot, it == 1);
        mma_commit(&bars.pds_free);
        mma_commit(DKV ? &bars.q_empty[rg.slot] : &bars.k_empty[rg.slot]);
        if (it == n_it) mma_commit(&bars.acc_full);
      }
      __syncwarp();
      issued = true;
      rg.next();
    }
    if (ok && dp_here && it < n_it) {
      // dP(it) overwrites the columns the gradient MMAs above read: same thread, in order
      ok = warp_wait(&bars.do_full[rs.slot], rs.phase, ctx, 18);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        m.template dp_mmas<true>(f, rs.slot);
        mma_commit(&bars.dp_full);
        if (it + 1 == n_it) mma_commit(&bars.fixed_free[f]);
      }
      __syncwarp();
      issued = true;
      rs.next();
    }
  }
  return ok;
}

template <int D>
__device__ __forceinline__ void grad_issuer_role(const BwdParams& p, uint8_t* smem, MainBars& bars,
                                                 const volatile int* slot, const TaskInfo* ring, uint32_t tmem,
                                                 const WaitCtx& ctx, int lane) {
  using Cfg = MainCfg<D>;
  MmaCtx<D> m;
  m.init(smem, tmem);
  int n = 0, G = 0, kv_used = 0, q_used = 0;
  bool ok = true, issued = false;
  for (;; ++n) {
    const int id = recv_task(bars, slot, n, ctx, lane, ok);
    if (!ok || id < 0) break;
    const TaskInfo t = ring[n & 3];
    const int f = n % Cfg::kNF;
    if (t.dkv) {
      ok = grad_task<D, true>(m, bars, ctx, t.n_it, f, n, G, kv_used, issued);
      kv_used += t.n_it;
    } else {
      ok = grad_task<D, false>(m, bars, ctx, t.n_it, f, n, G, q_used, issued);
      q_used += t.n_it;
    }
    if (!ok) break;
    G += t.n_it;
  }
  if (!ok && issued) {
    commit_one(&bars.drain2);
    mbar_wait_drain(&bars.drain2, 0, p.budget_ns);
  }
}

// ============================================================================ compute warpgroups
// Score tiles [it0, it1) of task t (global index of tile 0: G0).
template <int D, bool DKV>
__device__ __forceinline__ bool compute_tiles(const BwdParams& p, MainBars& bars, uint32_t tmem, const WaitCtx& ctx,
                                              const TaskInfo& t, int G0, int it0, int it1, int warp, int lane) {
  using Cfg = MainCfg<D>;
  constexpr bool kSep = DKV ? Cfg::kKvSepPdS : true;
  constexpr uint32_t colP = DKV ? Cfg::kKvColP : 0;
  constexpr uint32_t colDS = DKV ? Cfg::kKvColDS : Cfg::kDqColDS;
  const int wg = (warp - 2) >> 2;  // 0..3: score columns [wg*32, wg*32+32)
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_base + Cfg::kColS + wg * 32;
  const uint32_t tDP = tmem + lane_base + Cfg::kColDP + wg * 32;
  const uint32_t tP = tmem + lane_base + colP + wg * 16;
  const uint32_t tDS = tmem + lane_base + colDS + wg * 16;
  const float sl2 = p.scale_log2;
  // dQ tasks: this thread's query row's -LSE2 and -D, applied in the score math
  float nl = 0.f, nd = 0.f;
  if (!DKV) {
    const size_t idx = (static_cast<size_t>(t.b) * p.Hq + t.h) * p.Tpad + static_cast<size_t>(t.tile) * kTile + row;
    nl = __ldg(p.lse2 + idx);
    nd = -__ldg(p.Dvec + idx);
  }
  // One tile: S, dP -> registers -> sdp_free; P, dS -> TMEM -> pds_full.
  auto tile = [&](int g, bool masked, int lo, int hi) -> bool {
    if constexpr (DKV && Cfg::kLateDP) {
      // S -> registers -> sdp_free (S(g+1) may start); P; dP -> registers; dS; P and
      // dS over the warpgroup's own dP columns -> pds_full.
      if (!warp_wait(&bars.sdp_full, g & 1, ctx, 20)) return false;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tS, sv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars.sdp_free);
      float pf[32];
      uint32_t pk[16], dk[16];
      if (masked)
        score_p<true>(sv, sl2, lo, hi, pf, pk);
      else
        score_p<false>(sv, sl2, lo, hi, pf, pk);
      if (!warp_wait(&bars.dp_full, g & 1, ctx, 24)) return false;
      tc_fence_after();
      // dP in two halves of 16 columns: fewer live registers next to P's 48
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t dp[16];
        tmem_ld16(tDP + 16 * h, dp);
        tmem_wait_ld();
        score_ds_half(pf, dp, h, dk);
      }
      // P and dS over this warpgroup's own 32 dP columns, which this thread has just
      // read in its own lane: no other thread's data is overwritten, so no barrier
      tmem_st16(tDP, pk);
      tmem_st16(tDP + 16, dk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars.pds_full);
      return true;
    }
    if (!warp_wait(&bars.sdp_full, g & 1, ctx, 20)) return false;
    tc_fence_after();
    uint32_t s[32], dp[32];
    tmem_ld32(tS, s);
    tmem_ld32(tDP, dp);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars.sdp_free);
    uint32_t pk[16], dk[16];
    if (masked)
      score_chunk<DKV, true>(s, dp, sl2, lo, hi, pk, dk, nl, nd);
    else
      score_chunk<DKV, false>(s, dp, sl2, lo, hi, pk, dk, nl, nd);
    // The P/dS region must be free: read by the gradient MMAs of g-1 (separate
    // region), or S(g) read by every warpgroup (region inside S; the gradient
    // MMAs of g-1 are complete there, since S(g) was issued after them by the
    // same thread and has completed).
    if (kSep) {
      if (g > 0 && !warp_wait(&bars.pds_free, (g - 1) & 1, ctx, 22)) return false;
    } else {
      if (!warp_wait(&bars.sdp_free, g & 1, ctx, 23)) return false;
    }
    tc_fence_after();
    if (DKV) tmem_st16(tP, pk);
    tmem_st16(tDS, dk);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars.pds_full);
    return true;
  };
  bool ok = true;
  if (DKV) {
    // query tile of step it: i0 + it % ni, kept as a running counter (ni = nT - i0)
    int qt = t.i0 + it0 % t.ni;
    for (int it = it0; it < it1 && ok; ++it, qt = (qt + 1 == p.nT) ? t.i0 : qt + 1) {
      // Query columns visible to this key row: [lo, hi) in this warpgroup's 32-column frame.
      const int hi_tile = min(kTile, p.T - qt * kTile);
      const bool diag = p.causal && qt == t.tile;
      const int lo = (diag ? row : 0) - wg * 32;
      const int hi = hi_tile - wg * 32;
      ok = tile(G0 + it, diag || hi_tile < kTile, lo, hi);
    }
  } else {
    const int q_idx = t.tile * kTile + row;
    const bool valid = q_idx < p.T;
    const bool tile_ragged = (t.tile + 1) * kTile > p.T;
    for (int j = it0; j < it1 && ok; ++j) {
      // Key columns visible to this query row: [0, lim) in this warpgroup's 32-column frame.
      const bool diag = p.causal && j == t.tile;
      const bool kv_ragged = !p.causal && (j + 1) * kTile > p.T;
      int lim_tile = kTile;
      if (diag) lim_tile = row + 1;
      if (kv_ragged) lim_tile = p.T - j * kTile;
      const int lim = (valid ? lim_tile : 0) - wg * 32;
      ok = tile(G0 + j, diag || kv_ragged || tile_ragged, 0, lim);
    }
  }
  return ok;
}

// Epilogue of task t (the n-th of this CTA): accumulators -> registers, released
// to the next task's gradient MMAs, then bf16 to memory.
// d = 64: this warp's 32 rows of NC bf16 columns (NC/8 16-byte chunks a row, 64 or
// 32 bytes) into its staging region, swizzled as its store map expects (chunk c of
// row r at c ^ ((r >> 1) & 3) with 64-byte rows, c ^ ((r >> 2) & 1) with 32-byte
// rows), then one TMA store of the box at column x, row r0. The warp's previous
// store must have read the region first.
template <int NC>
__device__ __forceinline__ void tma_store_rows(const uint32_t (&r)[NC], float scale, uint8_t* stg,
                                               const CUtensorMap* map, int x, int h, int r0, int b, int T,
                                               int lane) {
  constexpr int NCH = NC / 8;
  static_assert(NCH == 2 || NCH == 4, "row bytes");
  if (lane == 0) tma_store_wait_read();
  __syncwarp();
  const int sw = NCH == 4 ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
#pragma unroll
  for (int v = 0; v < NCH; ++v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = pack_bf16x2(__uint_as_float(r[8 * v + 2 * i]) * scale, __uint_as_float(r[8 * v + 2 * i + 1]) * scale);
    *reinterpret_cast<uint4*>(stg + lane * (NCH * 16) + ((v ^ sw) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && r0 < T) {
    tma_store_4d(map, stg, x, h, r0, b);
    tma_store_commit();
  }
}

// Rotary embedding fused into the epilogue: the kernel differentiates with respect
// to the rotated q and k, and the gradient of a rotation is the inverse rotation,
// so NC accumulator columns of one row (feature pairs pair0, pair0 + 1, ...) turn
// by minus the angles of its token `tok`, in fp32, before the one rounding to
// bf16. The angles come from rope_cos_sin, in registers: a table lookup here sat
// on the compute warps' path between two tasks.
template <int NC>
__device__ __forceinline__ void unrotate_acc(uint32_t (&r)[NC], int tok, int pair0, const RopeFreq& f) {
  const uint32_t t = static_cast<uint32_t>(tok);
#pragma unroll
  for (int i = 0; i < NC / 2; ++i) {
    float cs, sn;
    rope_cos_sin(t, f.lo[pair0 + i], f.hi[pair0 + i], cs, sn);
    float x0 = __uint_as_float(r[2 * i]), x1 = __uint_as_float(r[2 * i + 1]);
    rope_rotate_f32(x0, x1, cs, -sn);
    r[2 * i] = __float_as_uint(x0);
    r[2 * i + 1] = __float_as_uint(x1);
  }
}

template <int D, bool DKV, bool ROPE>
__device__ __forceinline__ bool compute_epilogue(const BwdParams& p, MainBars& bars, uint32_t tmem, uint8_t* smem,
                                                 const WaitCtx& ctx, const TaskInfo& t, int n, int warp, int lane) {
  using Cfg = MainCfg<D>;
  const int wg = (warp - 2) >> 2;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  // columns of this thread's row: dK/dV NC = D/2 (part wg & 1), dQ NC = D/4 (wg)
  constexpr int NC = DKV ? D / 2 : D / 4;
  const int c0 = (DKV ? (wg & 1) : wg) * NC;
  const bool unrot = ROPE && (!DKV || wg >= 2);  // dQ and dK, not dV
  if (!warp_wait(&bars.acc_full, n & 1, ctx, 21)) return false;
  tc_fence_after();
  if (DKV) {
    // warpgroups 0, 1: dV halves; 2, 3: dK halves
    const int part = wg & 1;
    uint32_t r[NC];
    load_acc<NC>(tmem + lane_base + (wg < 2 ? Cfg::kKvColDV : Cfg::kKvColDK) + part * NC, r);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars.acc_free);
    if (unrot) unrotate_acc<NC>(r, t.tile * kTile + row, c0 / 2, p.rope_f);
    if constexpr (Cfg::kTmaStore) {
      tma_store_rows<NC>(r, wg < 2 ? 1.f : p.scale, smem + Cfg::stage_out(true, n % Cfg::kNF, warp - 2),
                         wg < 2 ? &p.tmap_dv : &p.tmap_dk, part * NC, t.kvh, t.tile * kTile + quarter * 32, t.b,
                         p.T, lane);
      return true;
    }
    const int k_idx = t.tile * kTile + row;
    if (k_idx < p.T) {
      const long long st = wg < 2 ? p.dv_st : p.dk_st, sb = wg < 2 ? p.dv_sb : p.dk_sb;
      const long long off = t.b * sb + k_idx * st + t.kvh * D + part * NC;
      store_acc_bf16<NC>(r, reinterpret_cast<__nv_bfloat16*>(wg < 2 ? p.dv : p.dk) + off, wg < 2 ? 1.f : p.scale);
    }
  } else {
    uint32_t r[NC];
    load_acc<NC>(tmem + lane_base + Cfg::kDqColAcc + wg * NC, r);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars.acc_free);
    if (unrot) unrotate_acc<NC>(r, t.tile * kTile + row, c0 / 2, p.rope_f);
    if constexpr (Cfg::kTmaStore) {
      tma_store_rows<NC>(r, p.scale, smem + Cfg::stage_out(false, n % Cfg::kNF, warp - 2), &p.tmap_dq, wg * NC,
                         t.h, t.tile * kTile + quarter * 32, t.b, p.T, lane);
      return true;
    }
    const int q_idx = t.tile * kTile + row;
    if (q_idx < p.T) {
      const long long off = t.b * p.dq_sb + q_idx * p.dq_st + t.h * D + wg * NC;
      store_acc_bf16<NC>(r, reinterpret_cast<__nv_bfloat16*>(p.dq) + off, p.scale);
    }
  }
  return true;
}

// ROPE: dq and dk leave inverse-rotated (p.rope_f); a separate instance so that
// the plain kernel's code is untouched by it.
template <int D, bool ROPE>
__global__ void __launch_bounds__(kMainThreads, 1) bwd_main_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ MainBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ volatile int task_slot[2];
  // Decoded tasks by per-CTA task index n (entry n & 3): written by the producer
  // before it publishes task n, which needs every consumer to have received task
  // n - 2, so the compute warps can still read task n - 1 for its epilogue.
  __shared__ TaskInfo task_ring[4];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.task_full[s], 1);
      mbar_init(&bars.task_empty[s], kTaskConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.fixed_full[s], 2);  // TMA bytes + the producer warp's arrival once all are issued
      mbar_init(&bars.fixed_free[s], 2);  // one commit from each MMA issuer
      mbar_init(&bars.stg_free[s], 16);   // lane 0 of each compute warp
    }
    for (int s = 0; s < kMaxKvStages; ++s) {
      mbar_init(&bars.q_full[s], 2);  // TMA bytes + the producer warp's aux operands
      mbar_init(&bars.q_empty[s], 1);
      mbar_init(&bars.do_full[s], 2);
      mbar_init(&bars.do_empty[s], 1);
    }
    for (int s = 0; s < kMaxDqKStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < kMaxDqVStages; ++s) {
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.sdp_full, 2);  // one commit from each MMA issuer (or two from warp 1)
    mbar_init(&bars.sdp_free, kComputeThreads);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.pds_full, kComputeThreads);
    mbar_init(&bars.pds_free, 1);
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.acc_free, kComputeThreads);
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

  if (warp == 0) {
    producer_role<D>(p, smem, bars, task_slot, task_ring, ctx, lane);
  } else if (warp == 1) {
    sdp_issuer_role<D>(p, smem, bars, task_slot, task_ring, tmem, ctx, lane);
  } else if (warp == kGradWarp) {
    grad_issuer_role<D>(p, smem, bars, task_slot, task_ring, tmem, ctx, lane);
  } else {
    // With one fixed buffer (d = 128) each task's epilogue runs after the next
    // task's first tile, so its wait for the last gradient MMAs overlaps the next
    // task's first score MMAs; at a change of kind it runs first (the dQ dS
    // columns hold dV of dK/dV tasks). With two fixed buffers the next task's
    // operands are already loaded and the epilogue simply runs first.
    int n = 0, G = 0, prev_id = -1;  // the previous task is read again from the ring for its epilogue
    bool ok = true;
    auto epilogue = [&](int tn) {
      const TaskInfo t = task_ring[tn & 3];
      return t.dkv ? compute_epilogue<D, true, ROPE>(p, bars, tmem, smem, ctx, t, tn, warp, lane)
                   : compute_epilogue<D, false, ROPE>(p, bars, tmem, smem, ctx, t, tn, warp, lane);
    };
    auto tiles = [&](const TaskInfo& t, int i0, int i1) {
      return t.dkv ? compute_tiles<D, true>(p, bars, tmem, ctx, t, G, i0, i1, warp, lane)
                   : compute_tiles<D, false>(p, bars, tmem, ctx, t, G, i0, i1, warp, lane);
    };
    for (;; ++n) {
      const int id = recv_task(bars, task_slot, n, ctx, lane, ok);
      if (!ok) break;
      if (id < 0) {
        if (prev_id >= 0) ok = epilogue(n - 1);
        break;
      }
      const TaskInfo t = task_ring[n & 3];
      const bool early = prev_id >= 0 && (MainCfg<D>::kNF > 1 || (prev_id < p.n_dkv_tasks) != (t.dkv != 0));
      if (early) ok = epilogue(n - 1);
      if (ok) ok = tiles(t, 0, 1);
      if (MainCfg<D>::kTmaStore && ok && prev_id >= 0 && lane == 0) {
        // a tile after the epilogue of n-1: its stores have long read the staged rows
        tma_store_wait_read();
        mbar_arrive(&bars.stg_free[(n - 1) % MainCfg<D>::kNF]);
      }
      if (ok && prev_id >= 0 && !early) ok = epilogue(n - 1);
      if (ok) ok = tiles(t, 1, t.n_it);
      if (!ok) break;
      prev_id = id;
      G += t.n_it;
    }
    // the staging regions must stay until the TMA stores have finished
    if (MainCfg<D>::kTmaStore && lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
  if (threadIdx.x == 0) {
    // The last CTA to finish (every CTA has taken its last task by then) leaves
    // the task counters at zero for the next launch.
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
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


template <int D, bool ROPE>
cudaError_t launch_main(const BwdParams& p, unsigned grid, int attr_slot, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(bwd_main_kernel<D, ROPE>, MainCfg<D>::kSmemBytes, attr_slot);
  if (e != cudaSuccess) return e;
  return launch_pdl(bwd_main_kernel<D, ROPE>, grid, kMainThreads, MainCfg<D>::kSmemBytes, stream, p);
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPreParams& p, int d, cudaStream_t stream) {
  const int rpb = d == 64 ? PreCfg<64>::kRows : PreCfg<128>::kRows;
  const long long n_tb = (p.Tpad + rpb - 1) / rpb;
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hq * n_tb);
  cudaError_t e = d == 64 ? launch_pdl(bwd_pre_kernel<64>, grid, kPreThreads, 0, stream, p)
                          : launch_pdl(bwd_pre_kernel<128>, grid, kPreThreads, 0, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream) {
  const int n_tasks = p.n_dkv_tasks + p.n_dq_tasks;
  if (n_tasks == 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(n_tasks < sms ? n_tasks : sms);
  const bool rope = p.rope != 0;
  if (d == 64)
    e = rope ? launch_main<64, true>(p, grid, 2, stream) : launch_main<64, false>(p, grid, 0, stream);
  else
    e = rope ? launch_main<128, true>(p, grid, 3, stream) : launch_main<128, false>(p, grid, 1, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace gqa
