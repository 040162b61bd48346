/*
 * gqa_attn.h — C ABI of the causal grouped-query flash-attention library for
 * GB300 (sm_103a): forward and backward, bf16 inputs, fp32 accumulation.
 *
 * The operation is the attention of "A transformer in PTX" (mnemonic-site,
 * 5-transformer):
 *  - §The model: a causal decoder whose attention is grouped-query — query
 *    head h reads key/value head h / (Hq/Hkv), several query heads per kv head.
 *  - §Flash attention: O = softmax(scale * Q K^T, masked so key j is visible to
 *    query i only when j <= i) V, with scale = 1/sqrt(d), computed block by
 *    block without writing the T x T score matrix, and the log-sum-exp of each
 *    row saved so that the backward can recompute the probabilities.
 *  - §The same bits every time: the backward is a dQ pass per block of
 *    queries and a dK/dV pass per block of keys that loops over every query
 *    head sharing the kv head; no float atomics, every sum has one owner and
 *    one order, so repeated calls give identical bits.
 *
 * Conventions shared by every entry point:
 *  - Tensors are device pointers, row-major, contiguous, 16-byte aligned
 *    (the *_strided entry points take views with free token and batch strides):
 *      q, o, dO, dq     bf16 [B, T, Hq,  d]
 *      k, v, dk, dv     bf16 [B, T, Hkv, d]
 *      lse              fp32 [B, Hq, T]   natural-log log-sum-exp of each query row
 *  - d is 64 or 128; Hq % Hkv == 0; B, T, Hq, Hkv >= 1.
 *  - The caller owns every buffer. The library never allocates device memory;
 *    it keeps only a per-device status word and a small host-side cache.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    asynchronous on it and never synchronise.
 *  - Outputs are overwritten, never accumulated into.
 *  - Errors: a non-zero gqa_status_t is returned before anything is launched
 *    when an argument is invalid; attn_last_error() then describes it.
 *    Kernels never trap: a pipeline wait that exceeds its time budget makes
 *    the CTA leave cleanly and records GQA_ERR_TIMEOUT in the device status
 *    word, which attn_sync_status() reports.
 *  - Requires a device of compute capability 10.3 (GB300).
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int gqa_status_t;

#define GQA_OK 0
#define GQA_ERR_INVALID_ARG 1       /* null/misaligned pointer, bad shape, d not 64/128, small workspace */
#define GQA_ERR_UNSUPPORTED_DEVICE 2 /* current device is not compute capability 10.3 */
#define GQA_ERR_LAUNCH 3            /* a CUDA runtime/driver call or kernel launch failed */
#define GQA_ERR_TIMEOUT 4           /* a kernel gave up waiting on its pipeline (device status word) */

/*
 * Forward pass ("A transformer in PTX", §Flash attention).
 *   q [B,T,Hq,d], k/v [B,T,Hkv,d] bf16 in; o [B,T,Hq,d] bf16 out;
 *   lse [B,Hq,T] fp32 out (natural log).
 *   causal != 0: key j is visible to query i iff j <= i; causal == 0: all keys.
 *   The score scale is 1/sqrt(d).
 */
gqa_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int Hq,
                      int Hkv, int d, int causal, void* stream);

/*
 * Bytes of scratch the backward needs: two fp32 arrays [B, Hq, T rounded up
 * to 128] (D_i = rowsum(dO * O) and the LSE in log2 units) followed by 256
 * bytes of task counters. The caller allocates it; nothing in it needs to be
 * initialised (the preprocess writes all of it) or preserved.
 * Ownership follows the CPU reference of "ptx_sass.cu" (Day 46: reading PTX
 * and SASS, decayFoldCpu): the library never allocates, the caller owns every
 * buffer, scratch included. Returns 0 when B, T or Hq is not positive.
 */
size_t attn_bwd_workspace_bytes(int B, int T, int Hq);

/*
 * Backward pass of L = sum(O * dO) ("A transformer in PTX", §The same bits
 * every time): a rowsum(dO * O) preprocess, then dQ tasks (one per block of
 * queries) and dK/dV tasks (one per block of keys, looping over the query heads
 * of its kv head in ascending order), run by one persistent launch.
 *   q, k, v, o, lse: as produced/consumed by attn_fwd; dO [B,T,Hq,d] bf16 in;
 *   dq [B,T,Hq,d], dk/dv [B,T,Hkv,d] bf16 out.
 *   workspace: device memory of at least attn_bwd_workspace_bytes(B,T,Hq)
 *   bytes, 16-byte aligned, not shared with a concurrent call.
 * Results are bit-identical from call to call for the same inputs.
 */
gqa_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                      int B, int T, int Hq, int Hkv, int d, int causal, void* stream);

/*
 * The stages of attn_bwd, callable one by one: attn_bwd is exactly
 * attn_bwd_preprocess followed by attn_bwd_dq_dkv on one stream. The dQ and
 * dK/dV passes read D and the LSE from the workspace and take their tasks from
 * its counters, which the preprocess zeroes and each pass leaves at zero (so
 * the pointer is declared const although those counters change during the
 * call); attn_bwd_dq_dkv runs both kinds of task in one launch (heaviest
 * first), attn_bwd_dq and attn_bwd_dkv one kind each.
 *
 * attn_bwd_preprocess: workspace <- D_i = rowsum(dO_i * O_i) and LSE_i*log2(e),
 *   fp32 [B, Hq, T rounded up to 128] each, rows past T set to 0; counters 0.
 * attn_bwd_dq:  dq [B,T,Hq,d] <- scale * sum_j dS_ij k_j, one task per query tile.
 * attn_bwd_dkv: dk, dv [B,T,Hkv,d] <- sums over the query heads sharing each kv
 *   head, one task per key tile, heads and query tiles in ascending order.
 * Arguments mean what they mean in attn_bwd.
 */
gqa_status_t attn_bwd_preprocess(const void* o, const float* lse, const void* dO, void* workspace,
                                 size_t workspace_bytes, int B, int T, int Hq, int d, void* stream);
gqa_status_t attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq,
                         const void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                         int causal, void* stream);
gqa_status_t attn_bwd_dkv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv,
                          const void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                          int causal, void* stream);
gqa_status_t attn_bwd_dq_dkv(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk,
                             void* dv, const void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                             int d, int causal, void* stream);

/*
 * Backward pass that allocates nothing, not even a workspace from the caller.
 * The pages have no counterpart to this entry point; it exists for callers
 * that may not allocate device memory where they run the backward (a loop
 * whose device memory is all handed out up front by a pool it does not own,
 * or a latency-critical loop that avoids cudaMalloc/cudaFree because they can
 * synchronise the device). Inputs and outputs are still the caller's and mean
 * what they mean in attn_bwd; the scratch lives in a fixed array of
 * GQA_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.
 *  - Limit: attn_bwd_workspace_bytes(B, T, Hq) must not exceed
 *    GQA_NOALLOC_SCRATCH_BYTES (B * Hq * roundup(T, 128) <= 1,048,544);
 *    larger problems get GQA_ERR_INVALID_ARG before anything is launched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents. Every element the kernels read is rewritten by the call itself,
 *    so stale contents do no harm, but two calls whose work overlaps on the
 *    GPU (different streams, or different host threads on one device) race.
 */
#define GQA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
gqa_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int d,
                              int causal, void* stream);

/*
 * Strided views ("A transformer in PTX", §The model: one fused matmul computes
 * the queries, keys and values of a layer into one buffer, which attention
 * reads, and attention's output is the input of the output projection).
 *
 * A gqa_view_t describes a bf16 [B, T, H, d] tensor whose element (b, t, h, c)
 * lives at ptr + b*stride_b + t*stride_t + h*d + c (counted in elements): the
 * H heads of one token are packed, while the token and batch strides are free.
 * So q, k and v can be the three parts of a fused [B, T, Hq + 2*Hkv, d]
 * projection (stride_t = (Hq + 2*Hkv)*d; k starting at head Hq, v at head
 * Hq + Hkv), a sequence-first [T, B, H, d] tensor can be read in place
 * (stride_b = H*d, stride_t = B*H*d), and o or the gradients can be written
 * into parts of wider buffers.
 *  - ptr: device pointer, 16-byte aligned.
 *  - stride_t, stride_b: positive multiples of 8 elements (16 bytes), below
 *    2^39. A stride whose dimension has size 1 is not used (T == 1: stride_t;
 *    B == 1: stride_b) and may hold any value.
 *  - An output view must not overlap itself: either stride_t >= H*d and
 *    stride_b >= T*stride_t, or stride_b >= H*d and stride_t >= B*stride_b
 *    (checked). Outputs must not overlap each other or an input (not checked).
 * Results are bit-identical to those of the same tensors stored contiguously.
 */
typedef struct gqa_view {
  void* ptr;
  long long stride_t;
  long long stride_b;
} gqa_view_t;

/* attn_fwd over views: q [B,T,Hq,d], k/v [B,T,Hkv,d] in, o [B,T,Hq,d] out;
 * lse [B,Hq,T] fp32 contiguous as in attn_fwd. */
gqa_status_t attn_fwd_strided(gqa_view_t q, gqa_view_t k, gqa_view_t v, gqa_view_t o, float* lse, int B, int T,
                              int Hq, int Hkv, int d, int causal, void* stream);

/* attn_bwd over views: q, k, v, o, dO in; dq [B,T,Hq,d], dk/dv [B,T,Hkv,d] out;
 * lse and the workspace as in attn_bwd. */
gqa_status_t attn_bwd_strided(gqa_view_t q, gqa_view_t k, gqa_view_t v, gqa_view_t o, const float* lse,
                              gqa_view_t dO, gqa_view_t dq, gqa_view_t dk, gqa_view_t dv, void* workspace,
                              size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal,
                              void* stream);

/*
 * Rotary position embedding ("A transformer in PTX", §The model: the trainer
 * rotates the queries and keys with RoPE between the fused QKV matmul and
 * attention). The page gives no formula; the rotation is the textbook one:
 * feature pair (2i, 2i+1) of token t turns by angle t * base^(-2i/d),
 *     y[2i] = x[2i] cos - x[2i+1] sin,   y[2i+1] = x[2i] sin + x[2i+1] cos,
 * and its inverse (minus the angle) is also its gradient, so the gradients of
 * the unrotated q and k are the inverse rotation of attn_bwd's dq and dk.
 *
 * attn_rope_table_bytes: bytes of the table for T tokens and head dim d:
 *   T * d/2 (cos, sin) pairs of fp32 (0 for a bad T or d).
 * attn_rope_table: fills `table` (device, 16-byte aligned, at least
 *   attn_rope_table_bytes(T, d) bytes) with cos and sin of every angle, each
 *   taken in double and rounded to fp32. base > 0 (10000 in the usual setting);
 *   d is 64 or 128. One table serves every call with the same T, d and base.
 * attn_rope: y = rotation of x (inverse != 0: by minus the angle) for every
 *   (b, t, h) of the bf16 [B, T, H, d] views x and y (gqa_view_t); the angle of
 *   token t is read from `table` (T tokens or more). y may be x itself (same
 *   pointer and strides: in place); otherwise y must not overlap x (not
 *   checked). To rotate q and k of a fused [B, T, Hq + 2*Hkv, d] projection in
 *   one call, pass the view of its first Hq + Hkv heads.
 */
size_t attn_rope_table_bytes(int T, int d);
gqa_status_t attn_rope_table(float* table, int T, int d, double base, void* stream);
gqa_status_t attn_rope(gqa_view_t x, gqa_view_t y, const float* table, int B, int T, int H, int d, int inverse,
                       void* stream);

/*
 * Attention with the rotary embedding fused in ("A transformer in PTX", §The
 * model: q and k are rotated between the fused QKV matmul and attention). The
 * rotation of attn_rope with base `base` (> 0, finite; 10000 in the usual
 * setting); the attention is attn_fwd / attn_bwd of the rotated q and k.
 * No table: each kernel computes its angles in registers. The turn count of
 * token t, t * base^(-2i/d) / (2 pi) mod 1, is taken exactly to 2^-32 of a turn
 * with integer multiplies, and the hardware sine and cosine of the reduced angle
 * (in [-pi, pi)) are within ~1e-6 of the exact values (attn_rope's fp32 table:
 * ~6e-8); a rotated element may therefore differ from attn_rope's by one bf16
 * rounding step.
 *
 * attn_fwd_rope: q [B,T,Hq,d] and k [B,T,Hkv,d] are the UNROTATED projections.
 *   The keys are rotated once into k_rot (one pass: every key tile is read by
 *   all query tiles of its group). The forward kernel rotates each query tile in
 *   shared memory as it arrives and writes the rotated tile to q_rot, so the
 *   queries make one trip through HBM. o, lse as in attn_fwd; q_rot and k_rot
 *   are what attn_bwd_rope takes, and o and lse are bit-identical to attn_fwd of
 *   q_rot and k_rot. q_rot may be q itself (same pointer and strides: rotated in
 *   place, as the page's trainer does on its QKV buffer), and k_rot may be k;
 *   otherwise they must not overlap any other argument (not checked).
 * attn_bwd_rope: q_rot, k_rot from attn_fwd_rope (same base); v, o, lse, dO, the
 *   workspace and dv as in attn_bwd (dv bit-identical to attn_bwd of q_rot and
 *   k_rot). dq and dk are the gradients of the UNROTATED q and k: the kernel's
 *   fp32 gradients of q_rot and k_rot are turned back by the inverse rotation in
 *   its epilogue, before the one rounding to bf16.
 * All tensors are views (gqa_view_t); errors as in attn_fwd_strided and
 * attn_bwd_strided, plus GQA_ERR_INVALID_ARG for a bad base; nothing is
 * launched when an argument is refused.
 */
gqa_status_t attn_fwd_rope(gqa_view_t q, gqa_view_t k, gqa_view_t v, gqa_view_t o, float* lse, gqa_view_t q_rot,
                           gqa_view_t k_rot, double base, int B, int T, int Hq, int Hkv, int d, int causal,
                           void* stream);
gqa_status_t attn_bwd_rope(gqa_view_t q_rot, gqa_view_t k_rot, gqa_view_t v, gqa_view_t o, const float* lse,
                           gqa_view_t dO, gqa_view_t dq, gqa_view_t dk, gqa_view_t dv, double base,
                           void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal,
                           void* stream);

/*
 * Naive attention ("A transformer in PTX", §Three ways to run it: the same
 * operations as plain kernels on bf16 activations, the reference the fast
 * kernels are checked against; §Flash attention: the naive kernels write the
 * whole T x T score matrix of every head). Slow and memory-hungry by design:
 * a check of the flash kernels at full size, not a fast path. Plain CUDA cores,
 * fp32 products and sums; scores and dP are kept in fp32, P and dS in bf16.
 *
 * attn_naive_workspace_bytes: bytes of scratch for both calls,
 *   B * Hq * T * T * (4 + 2 + 2).
 * attn_fwd_naive / attn_bwd_naive: the same arguments and layouts as attn_fwd
 *   and attn_bwd (contiguous tensors), with a workspace of at least
 *   attn_naive_workspace_bytes(B, T, Hq) bytes, 16-byte aligned.
 */
size_t attn_naive_workspace_bytes(int B, int T, int Hq);
gqa_status_t attn_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal, void* stream);
gqa_status_t attn_bwd_naive(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            int B, int T, int Hq, int Hkv, int d, int causal, void* stream);

/*
 * Description of the last error returned on this host thread ("" if none).
 * "Talking to the GPU", §One macro for every call: every driver call is
 * checked, and a failure is reported with the call's name and the driver's
 * own words for the error. Here the message names the entry point, the CUDA
 * call or argument that failed and cudaGetErrorString / cudaGetErrorName of
 * the code, and the caller gets it back instead of the process exiting.
 * The string stays valid until the next call of this library on the thread.
 */
const char* attn_last_error(void);

/*
 * Synchronise `stream`, then read and clear the device status word of the
 * current device. Returns GQA_OK, GQA_ERR_TIMEOUT (a kernel gave up waiting;
 * attn_last_error() names the kernel and wait), or GQA_ERR_LAUNCH if the
 * synchronisation itself failed.
 * The check after the work, as in "Talking to the GPU", §One macro for every
 * call (each call's result is tested before going on), extended to what the
 * kernels report: a bounded wait inside a kernel cannot return an error code,
 * so it writes one into the status word that this call reads.
 */
gqa_status_t attn_sync_status(void* stream);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nobody arrives at, with a budget of `budget_ns` nanoseconds, so
 * the wait must run out, record GQA_ERR_TIMEOUT in the status word and
 * return. Nothing faults or hangs. Read the result with attn_sync_status().
 */
gqa_status_t attn_selftest_timeout(unsigned long long budget_ns, void* stream);

/*
 * Rate probes ("Talking to the GPU", §The real tensor core peak: measure the
 * unit's real rate with enough independent work per SM, over one wave, timed on
 * the device). Each runs one CTA on every SM of the current device; `out` is a
 * caller-owned device buffer with one record per SM (cudaDevAttrMultiProcessorCount
 * records); nothing is allocated. Read the records after attn_sync_status().
 *
 * attn_probe_mma: one thread per SM issues `iters` x 4 tcgen05 MMAs (bf16 x bf16 ->
 *   fp32, M = 128, N = n in {64, 128, 256}, K = 16 each; A from shared memory, or
 *   from tensor memory when a_tmem != 0) and waits once for the last. chains = 1:
 *   all into one accumulator (each MMA needs the previous one's result); chains =
 *   2: alternately into two (not with a_tmem at n = 256: no TMEM room). Record per
 *   SM: {u64 SM cycles, u64 global-timer ns} of the chain, so FLOP/cycle/SM =
 *   iters * 4 * 2*128*n*16 / cycles and the clock = cycles / ns.
 *   iters in [1, 2^20]; out 16 bytes per SM, 16-byte aligned.
 * attn_probe_ex2: 1024 threads per SM each run 8 independent chains of
 *   ex2.approx.f32 for `iters` rounds. Record per SM: u64 SM cycles; ex2
 *   lanes/cycle/SM = 1024 * 8 * iters / cycles. sink: 4 bytes of device memory
 *   (written only to keep the chains alive).
 */
/*
 * attn_probe_tma: the TMA path that feeds the attention kernels' operand rings.
 *   ctas_per_sm (1 or 2) CTAs on every SM each keep `stages` (1..8 with one CTA per
 *   SM, 1..6 with two) requests in flight for one 128-row x 128-byte tile (16 KB,
 *   128-byte swizzle) of `buf`, each into its own shared-memory slot, `iters` tiles
 *   in all, picked by a per-CTA linear congruential sequence over the buffer's
 *   bytes / 16384 tiles. buf: caller-owned device memory, `bytes` a multiple of
 *   16384, 16-byte aligned; its contents are only read. Record per CTA (SMs x
 *   ctas_per_sm of them, 8 bytes each): u64 global-timer ns from the first request
 *   to the last arrival. Rate = CTAs * iters * 16384 / ns; a buffer that fits the
 *   L2 measures the load path from the L2, one far larger than it HBM; the bytes a
 *   SM holds in flight divided by its share of the rate give the load latency.
 *   iters in [1, 2^20].
 */
gqa_status_t attn_probe_mma(int n, int a_tmem, int chains, int iters, void* out, void* stream);
gqa_status_t attn_probe_ex2(int iters, void* out, void* sink, void* stream);
gqa_status_t attn_probe_tma(const void* buf, long long bytes, int stages, int ctas_per_sm, int iters, void* out,
                            void* stream);

/*
 * Time budget of every pipeline wait, in nanoseconds (default 2e9). Applies
 * to launches made after the call, on every device. 0 restores the default.
 */
void attn_set_wait_budget_ns(unsigned long long budget_ns);

/*
 * Order in which the backward's persistent launch hands out its tasks (a
 * performance choice only: every output element has one owner and a fixed
 * summation order, so the results are the same bits in any order).
 *   0 (default): per task kind, group-major when the tiles its tasks stream
 *      (Q and dO for dK/dV tasks, K and V for dQ tasks) exceed 45% of the
 *      device's L2, otherwise tile-major;
 *   1: tile-major (heaviest tiles first over all (batch, kv head) groups);
 *   2: group-major (one (batch, kv head) group after another, heaviest first
 *      within it).
 * Applies to launches made after the call. Returns GQA_ERR_INVALID_ARG for any
 * other value (the setting is then unchanged).
 */
gqa_status_t attn_set_task_order(int order);

/* Library version as "major.minor.patch". */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
