// attn_fwd.cu — forward kernel of causal grouped-query flash attention for sm_103a.
//
// "A transformer in PTX", §Flash attention: a block of queries walks the key
// blocks up to the diagonal keeping each row's running max and sum (online
// softmax); scores are scaled once by log2(e)/sqrt(d) so each probability is
// 2^(s - max) through the hardware ex2; P never goes to memory; the row's
// log-sum-exp is saved for the backward.
//
// GB300 design (not the page's mma.sync/ldmatrix/cp.async design):
//  * work item = one 128-query tile of one (batch, query head), heaviest first;
//    two CTAs per SM. At d = 64 the launch is persistent: each CTA runs a fixed
//    list of items in a snake order over the CTAs (CTA c takes items c,
//    2C-1-c, 2C+c, ...), so the causal cost evens out and the light items fill
//    the end of every list. At d = 128 each CTA runs one item;
//  * warp 0 issues TMA loads (Q per item, a K ring and a V ring that run on
//    across items, 128B swizzle), warp 1 issues tcgen05 MMAs (all lanes run the
//    loop, one elected lane issues) and owns the TMEM allocation, warps 2-5 are
//    the softmax warpgroup: one thread per query row, which is one TMEM lane, so
//    row max and row sum need no shuffles;
//  * S = Q K^T (SS MMA, fp32 in TMEM columns [0,128)) and O += P V (TS MMA, P
//    as bf16 pairs from TMEM, V as an MN-major smem operand). At d = 64, P has
//    columns of its own: the softmax loads the whole S row into registers and
//    releases S at once, so S(j+1) is computed while P(j) is; at d = 128 (no
//    TMEM room for two CTAs otherwise) P is written over S's first 64 columns
//    and S(j+1) follows PV(j);
//  * item boundaries overlap (d = 64): the next item's Q is loaded once the
//    last S MMA of the current one has read Q, its first S is computed while
//    the softmax warps run the epilogue, and only its first PV waits for the
//    epilogue to have read O out of TMEM;
//  * the epilogue stages bf16 O in shared memory, 32 rows per softmax warp with
//    the 128-byte swizzle, and stores them with TMA boxes: in a region of its
//    own at d = 64, in the item's dead Q buffer at d = 128;
//  * the running max is rescaled lazily: O and l are only rescaled when a
//    row's max grows by more than 2^8, otherwise p = 2^(s - m_stale) <= 256;
//  * causal tiles past the diagonal are never visited; only the diagonal tile
//    is masked; ragged T relies on TMA zero fill plus the causal mask;
//  * with the rotary embedding (a separate template instance) the softmax warps
//    rotate their rows of each Q tile in shared memory right after its load, and
//    the MMA warp stores the rotated tile for the backward before the first S.
#include "attn_common.cuh"

namespace gqa {
namespace {

constexpr int kFwdThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int kFwdCtasPerSm = 2;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;     // S fp32 [128 x 128]
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdCfg {
  // TMEM: d = 64: S [0,128) P [128,192) O [192,256); d = 128: S [0,128) with P
  // over [0,64), O [128,256).
  static constexpr bool kSepP = (D == 64);
  static constexpr uint32_t kColP = kSepP ? 128 : 0;
  static constexpr uint32_t kColO = kSepP ? 192 : 128;
  static_assert(kColO + D <= kTmemCols, "TMEM columns");
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfTileBytes;  // 128 rows x D bf16
  static constexpr int kKStages = (D == 64) ? 2 : 1;
  static constexpr int kVStages = (D == 64) ? 2 : 1;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  // d = 64: per softmax warp, 32 rows x 128 bytes of bf16 O for its TMA store.
  // d = 128: two CTAs leave no room for a region of its own; each CTA runs one
  // item, so the epilogue stages its rows (32 x 256 bytes per warp, two 64-column
  // halves) in the Q buffer, which no MMA reads once the item's last PV is done.
  static constexpr bool kTmaStore = (D == 64);
  static constexpr bool kStageInQ = (D == 128);
  // d = 64: persistent CTAs with lists of items; d = 128: one item per CTA.
  static constexpr bool kPersistent = (D == 64);
  static constexpr int kMaxRounds = kPersistent ? 0x7fffffff : 1;
  static_assert(kTmaStore || !kPersistent, "only the staged epilogue releases O for a next item");
  static_assert(kTmaStore || kStageInQ, "O leaves through TMA stores");
  static constexpr int kOffOut = kOffV + kVStages * kTileBytes;
  static constexpr int kOutBytes = kTmaStore ? 4 * 32 * 128 : 0;
  static constexpr int kSmemBytes = kOffOut + kOutBytes + 1024;  // + alignment slack
};

// Whole S row of this thread's lane (128 columns) in one TMEM load, and the 64
// columns of bf16 P pairs in one store: at d = 64 one instruction each in place of
// four measured 5-7% faster, with fewer live registers; at d = 128 the same time
// (168 -> 157 registers).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
        "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};"
      :
      : "r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]),
        "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]),
        "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]),
        "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]),
        "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}

// Wait with a warp-uniform outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& c, unsigned where) {
  bool ok = mbar_wait(bar, parity, c, where);
  return __all_sync(0xffffffffu, ok);
}

// Work item of round r for CTA c of C: snake order over the heaviest-first items.
__device__ __forceinline__ int item_of(int r, unsigned c, unsigned C) {
  return r * static_cast<int>(C) + ((r & 1) ? static_cast<int>(C - 1 - c) : static_cast<int>(c));
}

struct FwdItem {
  int qt, b, h, kvh, n_kv;
};

__device__ __forceinline__ FwdItem decode_item(const FwdParams& p, int id) {
  // heaviest query tiles first (causal cost grows with the tile index)
  FwdItem it;
  const int r = fdiv(id, p.fd_bh);
  it.qt = p.nT - 1 - r;
  const int bh = id - r * (p.B * p.Hq);
  it.b = fdiv(bh, p.fd_hq);
  it.h = bh - it.b * p.Hq;
  it.kvh = fdiv(it.h, p.fd_g);
  it.n_kv = p.causal ? it.qt + 1 : p.nT;
  return it;
}

// Rotary embedding fused into the Q load: this thread's query row of the Q tile in
// shared memory (128-byte swizzle: 16-byte chunk c of row r at c ^ (r & 7), one
// 128-row box per 64 columns) turned by the angles of its token `tok`, computed in
// registers (rope_cos_sin: nothing is read from memory on this path). Rows past T
// hold TMA's zero fill and are left as they are (the rotated tile's store skips them).
template <int D>
__device__ __forceinline__ void rotate_q_row(uint8_t* q_tile, int row, int tok, int T, const RopeFreq& f) {
  if (tok >= T) return;
  const uint32_t t = static_cast<uint32_t>(tok);
#pragma unroll
  for (int hf = 0; hf < D / 64; ++hf) {
    uint8_t* base = q_tile + hf * kHalfTileBytes + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4* ptr = reinterpret_cast<uint4*>(base + ((c ^ (row & 7)) * 16));
      uint4 v = *ptr;
      uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = hf * 32 + c * 4 + j;  // feature pair (2i, 2i+1)
        float cs, sn;
        rope_cos_sin(t, f.lo[i], f.hi[i], cs, sn);
        w[j] = rope_rotate_bf16x2(w[j], cs, sn);
      }
      *ptr = v;
    }
  }
}

// The forward's mbarriers, each in a 128-byte line of its own: packed next to one
// another the d = 128 forward measured 3.4% slower (c4) and the d = 64 one 2%
// (c3, c5), the polling of one barrier getting in the way of arrivals on its
// neighbours. Each ring's stages share a line.
template <int KS, int VS>
struct FwdBars {
  alignas(128) uint64_t q;
  alignas(128) uint64_t qrot;
  alignas(128) uint64_t qfree;
  alignas(128) uint64_t kf[KS];
  alignas(128) uint64_t ke[KS];
  alignas(128) uint64_t vf[VS];
  alignas(128) uint64_t ve[VS];
  alignas(128) uint64_t s;
  alignas(128) uint64_t sfree;
  alignas(128) uint64_t p;
  alignas(128) uint64_t pfree;
  alignas(128) uint64_t o;
  alignas(128) uint64_t ofree;
  alignas(128) uint64_t drain;
};

// ROPE: q is rotated in the kernel (p.rope_f) and stored to p.tmap_qrot; a separate
// instance, so the plain kernel's code is untouched by it.
template <int D, bool ROPE>
__global__ void __launch_bounds__(kFwdThreads, kFwdCtasPerSm) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using Cfg = FwdCfg<D>;
  constexpr int KS = Cfg::kKStages;
  constexpr int VS = Cfg::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr bool kSepP = Cfg::kSepP;
  constexpr uint32_t kColP = Cfg::kColP, kColO = Cfg::kColO;
  // Per item: bar_q (Q loaded), bar_qfree (its last S MMA is done), bar_o (its
  // last PV is done), bar_ofree (the softmax holds O in registers). Per tile,
  // counted over the CTA's items: bar_s (S in TMEM), bar_sfree (every softmax
  // thread holds S; d = 64), bar_p (P in TMEM), bar_pfree (PV done; d = 64).
  // With the rotary embedding, bar_qrot (every softmax thread has rotated its
  // row of Q) takes bar_q's place for the MMA warp.
  __shared__ FwdBars<KS, VS> fb;
  uint64_t &bar_q = fb.q, &bar_qrot = fb.qrot, &bar_qfree = fb.qfree, &bar_s = fb.s, &bar_sfree = fb.sfree,
           &bar_p = fb.p, &bar_pfree = fb.pfree, &bar_o = fb.o, &bar_ofree = fb.ofree, &bar_drain = fb.drain;
  uint64_t *bar_kf = fb.kf, *bar_ke = fb.ke, *bar_vf = fb.vf, *bar_ve = fb.ve;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // This CTA's items: item_of(r) for r = 0, 1, ... while below n_items (a prefix:
  // item_of grows with r). Roles re-derive an item's fields from its index when
  // they need them, which keeps the softmax loop's live registers down.
  const int n_items = p.B * p.Hq * p.nT;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1);
    if (ROPE) mbar_init(&bar_qrot, 128);
    mbar_init(&bar_qfree, 1);
    for (int s = 0; s < KS; ++s) { mbar_init(&bar_kf[s], 1); mbar_init(&bar_ke[s], 1); }
    for (int s = 0; s < VS; ++s) { mbar_init(&bar_vf[s], 1); mbar_init(&bar_ve[s], 1); }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_sfree, 128);
    mbar_init(&bar_p, 128);
    mbar_init(&bar_pfree, 1);
    mbar_init(&bar_o, 1);
    mbar_init(&bar_ofree, 128);
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const WaitCtx ctx{&abort_sh, p.status, p.budget_ns, kKidFwd};
  constexpr bool rope = ROPE;
  pdl_wait_previous();  // inputs may be written by the previous kernel; outputs may still be read by it

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tmap_q);
      tma_prefetch_desc(&p.tmap_k);
      tma_prefetch_desc(&p.tmap_v);
      int issued_k[KS] = {}, issued_v[VS] = {}, n_q = 0;
      bool ok = true;
      int gk = 0;  // K/V tiles loaded so far, over all items
      for (int r = 0; r < Cfg::kMaxRounds && ok; ++r) {
        const int id = item_of(r, blockIdx.x, gridDim.x);
        if (id >= n_items) break;
        const FwdItem it = decode_item(p, id);
        // Q of the previous item is read until its last S MMA is done
        if (r > 0) ok = mbar_wait(&bar_qfree, (r - 1) & 1, ctx, 5);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar_q, Cfg::kTileBytes);
        for (int hf = 0; hf < Cfg::kHalves; ++hf)
          tma_load_4d(smem + Cfg::kOffQ + hf * kHalfTileBytes, &p.tmap_q, &bar_q, hf * 64, it.h, it.qt * kTile,
                      it.b);
        ++n_q;
        for (int j = 0; j < it.n_kv && ok; ++j, ++gk) {
          const int ks = gk % KS, kn = gk / KS;
          if (kn > 0) ok = mbar_wait(&bar_ke[ks], (kn - 1) & 1, ctx, 1);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_kf[ks], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kOffK + ks * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_k, &bar_kf[ks],
                        hf * 64, it.kvh, j * kTile, it.b);
          issued_k[ks]++;
          const int vs = gk % VS, vn = gk / VS;
          if (vn > 0) ok = mbar_wait(&bar_ve[vs], (vn - 1) & 1, ctx, 2);
          if (!ok) break;
          mbar_arrive_expect_tx(&bar_vf[vs], Cfg::kTileBytes);
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_load_4d(smem + Cfg::kOffV + vs * Cfg::kTileBytes + hf * kHalfTileBytes, &p.tmap_v, &bar_vf[vs],
                        hf * 64, it.kvh, j * kTile, it.b);
          issued_v[vs]++;
        }
      }
      if (ok) {
        // Wait for the MMA side to release every stage and the last Q, so that no
        // commit arrives on a barrier of this CTA after it has left.
        for (int s = 0; s < KS && ok; ++s)
          if (issued_k[s] > 0) ok = mbar_wait(&bar_ke[s], (issued_k[s] - 1) & 1, ctx, 3);
        for (int s = 0; s < VS && ok; ++s)
          if (issued_v[s] > 0) ok = mbar_wait(&bar_ve[s], (issued_v[s] - 1) & 1, ctx, 4);
        if (Cfg::kPersistent && ok && n_q > 0) ok = mbar_wait(&bar_qfree, (n_q - 1) & 1, ctx, 6);
      }
      if (!ok) {
        // Abort path: let every load already issued land before the CTA exits.
        if (n_q > 0) mbar_wait_drain(&bar_q, (n_q - 1) & 1, p.budget_ns);
        for (int s = 0; s < KS; ++s)
          if (issued_k[s] > 0) mbar_wait_drain(&bar_kf[s], (issued_k[s] - 1) & 1, p.budget_ns);
        for (int s = 0; s < VS; ++s)
          if (issued_v[s] > 0) mbar_wait_drain(&bar_vf[s], (issued_v[s] - 1) & 1, p.budget_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
    const uint64_t dQ = sdesc_sw128(smem_u32(smem + Cfg::kOffQ), 16, 1024);
    const uint64_t dK = sdesc_sw128(smem_u32(smem + Cfg::kOffK), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(smem + Cfg::kOffV), kHalfTileBytes, 1024);
    constexpr uint32_t kTileD = Cfg::kTileBytes >> 4;  // descriptor units
    if (rope && lane == 0) tma_prefetch_desc(&p.tmap_qrot);
    bool issued = false;
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit(bar);
      __syncwarp();
    };
    // S(g) into columns [0,128); d = 64: once the softmax holds S(g-1).
    auto issue_s = [&](int g, bool last_of_item) -> bool {
      if (kSepP && g > 0 && !warp_wait(&bar_sfree, (g - 1) & 1, ctx, 14)) return false;
      const int ks = g % KS;
      if (!warp_wait(&bar_kf[ks], (g / KS) & 1, ctx, 11)) return false;
      tc_fence_after();
      const uint64_t kb = dK + ks * kTileD;
      if (rope && Cfg::kPersistent && last_of_item) {
        // the next item's Q load overwrites the tile: its rotated copy must have left
        if (lane == 0) tma_store_wait_read();
        __syncwarp();
      }
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kHalfTileBytes + (kk & 3) * 32) >> 4);
          mma_ss(tmem + kColS, dQ + off, kb + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s);
        mma_commit(&bar_ke[ks]);
        if (Cfg::kPersistent && last_of_item) mma_commit(&bar_qfree);
      }
      __syncwarp();
      issued = true;
      return true;
    };
    // PV(g); the first of item r overwrites O once the epilogue of item r-1 has read it.
    auto issue_pv = [&](int g, bool first_of_item, int r) -> bool {
      const int vs = g % VS;
      if (!warp_wait(&bar_p, g & 1, ctx, 12)) return false;
      if (first_of_item && r > 0 && !warp_wait(&bar_ofree, (r - 1) & 1, ctx, 15)) return false;
      if (!warp_wait(&bar_vf[vs], (g / VS) & 1, ctx, 13)) return false;
      tc_fence_after();
      const uint64_t vb = dV + vs * kTileD;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts(tmem + kColO, tmem + kColP + kk * 8, vb + kk * 128, idesc_o, (!first_of_item || kk > 0) ? 1u : 0u);
        if (kSepP) mma_commit(&bar_pfree);
        mma_commit(&bar_ve[vs]);
      }
      __syncwarp();
      issued = true;
      return true;
    };
    bool ok = true;
    int g0 = 0;  // global index of the item's first tile
    for (int r = 0; r < Cfg::kMaxRounds && ok; ++r) {
      const int id = item_of(r, blockIdx.x, gridDim.x);
      if (id >= n_items) break;
      // (the full decode, integer divisions by runtime sizes, only where it is used:
      // ahead of the first MMA it measured 2.4% of the d = 128 forward)
      const int n_kv = decode_item(p, id).n_kv;
      const FwdItem itm = ROPE ? decode_item(p, id) : FwdItem{};
      ok = warp_wait(rope ? &bar_qrot : &bar_q, r & 1, ctx, 10);
      if (!ok) break;
      if (rope) {
        // the rotated Q tile goes out once, for the backward
        if (lane == 0) {
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tma_store_4d(&p.tmap_qrot, smem + Cfg::kOffQ + hf * kHalfTileBytes, hf * 64, itm.h, itm.qt * kTile,
                         itm.b);
          tma_store_commit();
        }
        __syncwarp();
      }
      if (kSepP) {
        // S(j+1) as soon as the softmax holds S(j); PV(j) once P(j) is written.
        ok = issue_s(g0, n_kv == 1);
        for (int j = 0; j < n_kv && ok; ++j) {
          if (j + 1 < n_kv) ok = issue_s(g0 + j + 1, j + 2 == n_kv);
          if (ok) ok = issue_pv(g0 + j, j == 0, r);
        }
      } else {
        for (int j = 0; j < n_kv && ok; ++j) {
          // O += P_{j-1} V_{j-1} must be issued before S_j overwrites P_{j-1}.
          if (j > 0) ok = issue_pv(g0 + j - 1, j == 1, r);
          if (ok) ok = issue_s(g0 + j, j + 1 == n_kv);
        }
        if (ok) ok = issue_pv(g0 + n_kv - 1, n_kv == 1, r);
      }
      if (ok && rope) {
        // d = 128 stages O in the Q buffer once bar_o completes
        if (lane == 0) tma_store_wait_read();
        __syncwarp();
      }
      if (ok) commit(&bar_o);
      g0 += n_kv;
    }
    if (!ok && issued) {
      commit(&bar_drain);
      mbar_wait_drain(&bar_drain, 0, p.budget_ns);
    }
    if (rope && lane == 0) tma_store_wait_all();
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tP = tmem + lane_base + kColP;
    const uint32_t tO = tmem + lane_base + kColO;
    const float sl2 = p.scale_log2;
    bool ok = true;
    // Rotary embedding: rotate this thread's row of round rr's Q tile once it has
    // landed (no-op past the CTA's last item).
    auto rotate_round = [&](int rr) -> bool {
      if (rr >= Cfg::kMaxRounds) return true;
      const int id2 = item_of(rr, blockIdx.x, gridDim.x);
      if (id2 >= n_items) return true;
      const int tok = (p.nT - 1 - fdiv(id2, p.fd_bh)) * kTile + row;
      if (!warp_wait(&bar_q, rr & 1, ctx, 23)) return false;
      rotate_q_row<D>(smem + Cfg::kOffQ, row, tok, p.T, p.rope_f);
      fence_proxy_async_smem();
      mbar_arrive(&bar_qrot);
      return true;
    };
    int g = 0;  // tiles seen so far, over all items
    for (int r = 0; r < Cfg::kMaxRounds && ok; ++r) {
      const int id = item_of(r, blockIdx.x, gridDim.x);
      if (id >= n_items) break;
      if (rope && r == 0 && !(ok = rotate_round(0))) break;
      const int qt = p.nT - 1 - fdiv(id, p.fd_bh);
      const int n_kv = p.causal ? qt + 1 : p.nT;
      float m_used = -INFINITY;  // running max in log2 units (possibly stale by <= 8)
      float l = 0.f;   // row sum of the fp32 probabilities (for the LSE)
      float lo = 0.f;  // the same less each tile's top term's bf16 rounding (for O, see below)
      for (int j = 0; j < n_kv; ++j, ++g) {
        ok = warp_wait(&bar_s, g & 1, ctx, 20);
        if (!ok) break;
        tc_fence_after();
        float s[kTile];
        {
          // one batched load of the whole row, one wait
          uint32_t rr[kTile];
          tmem_ld128(tS, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kTile; ++i) s[i] = __uint_as_float(rr[i]);
        }
        if (kSepP) {
          // S is in registers: the MMA may compute S(g+1) into the same columns.
          tc_fence_before();
          mbar_arrive(&bar_sfree);
        }
        if (p.causal && j == qt) {
#pragma unroll
          for (int cc = 0; cc < kTile; ++cc)
            if (cc > row) s[cc] = -INFINITY;
        } else if (!p.causal && (j + 1) * kTile > p.T) {
          const int lim = p.T - j * kTile;
#pragma unroll
          for (int cc = 0; cc < kTile; ++cc)
            if (cc >= lim) s[cc] = -INFINITY;
        }
        // row max: a tree of 3-input maxima (independent chains, half the instructions)
        float m8[8];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          float a = max3(s[q8 * 16 + 0], s[q8 * 16 + 1], s[q8 * 16 + 2]);
          float b = max3(s[q8 * 16 + 3], s[q8 * 16 + 4], s[q8 * 16 + 5]);
          float cc = max3(s[q8 * 16 + 6], s[q8 * 16 + 7], s[q8 * 16 + 8]);
          float d = max3(s[q8 * 16 + 9], s[q8 * 16 + 10], s[q8 * 16 + 11]);
          float e = max3(s[q8 * 16 + 12], s[q8 * 16 + 13], s[q8 * 16 + 14]);
          m8[q8] = max3(max3(a, b, cc), max3(d, e, s[q8 * 16 + 15]), a);
        }
        const float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        const float m_tile = mx * sl2;
        const bool need = m_tile > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_used - m_tile);
          m_used = m_tile;
          l *= alpha;
          lo *= alpha;
        }
        // p = 2^(s*c - m) two columns at a time (packed fp32 FMA and add), bf16 pairs kept
        // in registers until the P columns are free.
        const uint64_t c2 = f2_make(sl2, sl2), nm2 = f2_make(-m_used, -m_used);
        uint64_t lsum[4] = {0ull, 0ull, 0ull, 0ull};  // independent partial sums of pairs
        uint32_t pk[kTile / 2];
#pragma unroll
        for (int i = 0; i < kTile / 2; ++i) {
          float x0, x1;
          f2_split(f2_fma(f2_make(s[2 * i], s[2 * i + 1]), c2, nm2), x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          lsum[i & 3] = f2_add(lsum[i & 3], f2_make(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        {
          float a0, a1;
          f2_split(f2_add(f2_add(lsum[0], lsum[1]), f2_add(lsum[2], lsum[3])), a0, a1);
          l += a0 + a1;
          // The PV MMA weighs each key by its bf16-rounded probability. With m_used up to
          // 2^8 stale the largest term of a tile is not a power of two, and in a row one
          // key dominates its rounding (up to 2^-9 relative) would move O by that much of
          // the key's value when O is divided by the fp32 sum: O's divisor therefore
          // counts each tile's largest term as the MMA sees it (the same FMA and ex2 as
          // in the loop above, then the same rounding).
          const float ptop = ex2_approx(fmaf(mx, sl2, -m_used));
          lo += (a0 + a1) - (ptop - __bfloat162float(__float2bfloat16_rn(ptop)));
        }
        // d = 64: P(g-1) (possibly of the previous item) must no longer be read by PV(g-1).
        if (kSepP && g > 0) {
          ok = warp_wait(&bar_pfree, (g - 1) & 1, ctx, 22);
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st64(tP, pk);
        // Rescale O (complete: PV_{j-1} has finished) when any row of this warp needs it.
        if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t rr[32];
            tmem_ld32(tO + cc * 32, rr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st32(tO + cc * 32, rr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar_p);
      }
      // the next item's Q is rotated before this item's epilogue, so its first S can
      // be computed while the epilogue runs
      if (ok && rope) ok = rotate_round(r + 1);
      if (ok) ok = warp_wait(&bar_o, r & 1, ctx, 21);
      if (!ok) break;
      // ---- epilogue: O / l as bf16, and the row's log-sum-exp
      tc_fence_after();
      const FwdItem it = decode_item(p, id);
      const int q_idx = qt * kTile + row;
      const float inv_l = 1.f / lo;
      const bool valid = q_idx < p.T;
      if constexpr (Cfg::kTmaStore) {
        // O / l as bf16 pairs, then O's columns are free; 32 rows x 128 bytes per
        // warp staged with the 128-byte swizzle (chunk c of row r at c ^ (r & 7))
        // and stored with one TMA box
        uint32_t o_pk[D / 2];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tO + cc * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o_pk[cc * 16 + i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l, __uint_as_float(rr[2 * i + 1]) * inv_l);
        }
        tc_fence_before();
        mbar_arrive(&bar_ofree);  // the next item's first PV may overwrite O
        uint8_t* stg = smem + Cfg::kOffOut + (warp - 2) * 32 * 128;
        if (lane == 0) tma_store_wait_read();
        __syncwarp();
#pragma unroll
        for (int v = 0; v < D / 8; ++v)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((v ^ (lane & 7)) * 16)) =
              make_uint4(o_pk[4 * v], o_pk[4 * v + 1], o_pk[4 * v + 2], o_pk[4 * v + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        const int r0 = qt * kTile + quarter * 32;
        if (lane == 0 && r0 < p.T) {
          tma_store_4d(&p.tmap_o, stg, 0, it.h, r0, it.b);
          tma_store_commit();
        }
      } else if constexpr (Cfg::kStageInQ) {
        static_assert(!Cfg::kPersistent, "the Q buffer is reloaded by persistent CTAs");
        // 32 rows per warp, each 64-column half a 128-byte-swizzled 4 KB box
        uint8_t* stg = smem + Cfg::kOffQ + (warp - 2) * (32 * 256);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tO + cc * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w[i] = pack_bf16x2(__uint_as_float(rr[8 * v + 2 * i]) * inv_l,
                                 __uint_as_float(rr[8 * v + 2 * i + 1]) * inv_l);
            const int ch = cc * 4 + v;  // 16-byte chunk of the row, 0..15
            *reinterpret_cast<uint4*>(stg + (ch >> 3) * 4096 + lane * 128 + (((ch & 7) ^ (lane & 7)) * 16)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int r0 = qt * kTile + quarter * 32;
        if (lane == 0 && r0 < p.T) {
          tma_store_4d(&p.tmap_o, stg, 0, it.h, r0, it.b);
          tma_store_4d(&p.tmap_o, stg + 4096, 64, it.h, r0, it.b);
          tma_store_commit();
        }
      }
      if (valid)
        p.lse[(static_cast<size_t>(it.b) * p.Hq + it.h) * p.T + q_idx] = (m_used + log2f(l)) * 0.69314718055994531f;
    }
    // the staging rows must stay until the TMA stores have finished
    if ((Cfg::kTmaStore || Cfg::kStageInQ) && lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool ROPE>
cudaError_t launch_fwd_d(const FwdParams& p, cudaStream_t stream) {
  constexpr int smem = FwdCfg<D>::kSmemBytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // d = 64: persistent, two CTAs per SM. d = 128: one item per CTA (the grid
  // covers every item, so each CTA's list is its own index): without room for
  // the staged epilogue its item boundaries gain little from persistence, and
  // the hardware's dispatch of CTAs to whichever SM frees first balanced the
  // per-SM speed differences better than the fixed lists (measured 5% faster).
  const long long n_items = static_cast<long long>(p.B) * p.Hq * p.nT;
  long long slots = n_items;
  if (FwdCfg<D>::kPersistent) {
    int sms = 0;
    if ((e = sm_count(&sms)) != cudaSuccess) return e;
    slots = static_cast<long long>(sms) * kFwdCtasPerSm;
  }
  const unsigned grid = static_cast<unsigned>(n_items < slots ? n_items : slots);
  e = launch_pdl(attn_fwd_kernel<D, ROPE>, grid, kFwdThreads, smem, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t stream) {
  if (p.rope) return d == 64 ? launch_fwd_d<64, true>(p, stream) : launch_fwd_d<128, true>(p, stream);
  return d == 64 ? launch_fwd_d<64, false>(p, stream) : launch_fwd_d<128, false>(p, stream);
}

}  // namespace gqa
