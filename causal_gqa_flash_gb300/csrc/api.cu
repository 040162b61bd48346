// api.cu — the C ABI (include/gqa_attn.h): argument checks, TMA tensor maps,
// the per-device status word, and kernel launches on the caller's stream.
//
// Error convention after "Talking to the GPU", §One macro for every call: every
// CUDA call is checked, and a failure is reported with the call's name and the
// runtime's own words — here as a return code plus attn_last_error(), never by
// exiting the process.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/gqa_attn.h"
#include "attn_common.cuh"
#include "naive.cuh"
#include "rope.cuh"

namespace gqa {

__device__ DevStatusWord g_status_word;

__global__ void selftest_timeout_kernel(DevStatusWord* status, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx ctx{&abort_sh, status, budget_ns, kKidSelfTest};
  // Nobody arrives on `bar`: the wait must run out and record a timeout.
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, ctx, 1);
  __syncthreads();
}

cudaError_t launch_selftest_timeout(DevStatusWord* status, unsigned long long budget_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, budget_ns);
  return cudaGetLastError();
}

}  // namespace gqa

using namespace gqa;

namespace {

thread_local std::string t_last_error;

}  // namespace

namespace gqa {
// Lets other translation units of the library report through attn_last_error().
void set_last_error_message(const char* msg) { t_last_error = msg ? msg : ""; }
}  // namespace gqa

namespace {

std::atomic<unsigned long long> g_budget_ns{2000000000ull};
std::atomic<int> g_task_order{0};  // attn_set_task_order
constexpr unsigned long long kDefaultBudgetNs = 2000000000ull;

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool ready = false;
  bool supported = false;
  DevStatusWord* status = nullptr;
  long long l2_bytes = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

gqa_status_t fail(gqa_status_t code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

gqa_status_t cuda_fail(const char* fn, const char* what, cudaError_t e) {
  return fail(GQA_ERR_LAUNCH, "%s: %s failed: %s (%s)", fn, what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// Per-device setup: capability check, status-word address, tensor-map encoder.
gqa_status_t device_state(const char* fn, DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return fail(GQA_ERR_UNSUPPORTED_DEVICE, "%s: device %d out of range", fn, dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return cuda_fail(fn, "cudaDeviceGetAttribute", e);
    e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(fn, "cudaDeviceGetAttribute", e);
    st.supported = (major == 10 && minor == 3);
    int l2 = 0;
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return cuda_fail(fn, "cudaDeviceGetAttribute", e);
    st.l2_bytes = l2;
    if (st.supported) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_status_word);
      if (e != cudaSuccess) return cuda_fail(fn, "cudaGetSymbolAddress(status word)", e);
      st.status = static_cast<DevStatusWord*>(addr);
      if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
          return fail(GQA_ERR_LAUNCH, "%s: cannot resolve cuTensorMapEncodeTiled", fn);
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
      }
    }
    st.ready = true;
  }
  if (!st.supported)
    return fail(GQA_ERR_UNSUPPORTED_DEVICE, "%s: device %d is not compute capability 10.3 (GB300)", fn, dev);
  *out = &st;
  return GQA_OK;
}

}  // namespace

namespace gqa {
// The per-device check of every entry point, for other translation units: GQA_OK
// when the current device is in range and of compute capability 10.3, otherwise
// the error code with attn_last_error() set, naming `fn`.
gqa_status_t check_current_device(const char* fn) {
  DeviceState* ds = nullptr;
  return device_state(fn, &ds);
}
}  // namespace gqa

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gqa_status_t check_shape(const char* fn, int B, int T, int Hq, int Hkv, int d) {
  if (B <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0)
    return fail(GQA_ERR_INVALID_ARG, "%s: B, T, Hq, Hkv must be positive (got %d, %d, %d, %d)", fn, B, T, Hq, Hkv);
  if (d != 64 && d != 128) return fail(GQA_ERR_INVALID_ARG, "%s: d must be 64 or 128 (got %d)", fn, d);
  if (Hq % Hkv != 0) return fail(GQA_ERR_INVALID_ARG, "%s: Hq (%d) must be a multiple of Hkv (%d)", fn, Hq, Hkv);
  // Index arithmetic inside the kernels uses 32-bit tile coordinates and
  // 64-bit element offsets; keep every TMA coordinate and grid size in range.
  const long long tiles = (long long)B * Hq * ((T + kTile - 1) / kTile);
  if (tiles > 0x7fffffffLL || (long long)T > (1LL << 30))
    return fail(GQA_ERR_INVALID_ARG, "%s: problem too large (B*Hq*ceil(T/128) = %lld)", fn, tiles);
  return GQA_OK;
}

gqa_status_t check_ptr(const char* fn, const char* name, const void* p) {
  if (!p) return fail(GQA_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
  if (!aligned16(p)) return fail(GQA_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, name);
  return GQA_OK;
}

// A bf16 [B, T, H, d] tensor with packed heads: element (b, t, h, c) at
// ptr + b*sb + t*st + h*d + c (elements).
struct View {
  const void* ptr;
  long long st, sb;
};

View packed(const void* ptr, int T, int H, int d) {
  return View{ptr, (long long)H * d, (long long)T * H * d};
}

// Checks a caller's strided view (see gqa_view_t) and fills `out`; strides of a
// dimension of size 1 are replaced by the packed ones, since they are never used.
gqa_status_t check_view(const char* fn, const char* name, const gqa_view_t& v, int B, int T, int H, int d,
                        bool output, View* out) {
  gqa_status_t s;
  if ((s = check_ptr(fn, name, v.ptr))) return s;
  const long long row = (long long)H * d;
  long long st = T == 1 ? row : v.stride_t;
  long long sb = B == 1 ? st * T : v.stride_b;
  const long long kMax = 1LL << 39;
  for (long long x : {st, sb})
    if (x <= 0 || x % 8 != 0 || x >= kMax)
      return fail(GQA_ERR_INVALID_ARG,
                  "%s: %s strides (t %lld, b %lld) must be positive multiples of 8 elements below 2^39", fn, name,
                  v.stride_t, v.stride_b);
  if (output) {
    const bool t_major = st >= row && sb >= st * T;  // [B, T, H, d]-like
    const bool b_major = sb >= row && st >= sb * B;  // [T, B, H, d]-like
    if (!t_major && !b_major)
      return fail(GQA_ERR_INVALID_ARG, "%s: output %s overlaps itself (stride_t %lld, stride_b %lld, H*d %lld)", fn,
                  name, v.stride_t, v.stride_b, row);
  }
  *out = View{v.ptr, st, sb};
  return GQA_OK;
}

// 4D tiled map over a [B, T, H, d] bf16 view: box = box_c (d) x 1 (head) x box_rows x 1 (batch),
// swizzled over the box's inner bytes (box_c = 64: 128-byte swizzle, 32: 64-byte, 16: 32-byte);
// loads read rows past T as zero, stores skip them. The operand loads use 64 x 128 boxes.
gqa_status_t make_map(const char* fn, const char* name, CUtensorMap* m, const View& t, int B, int T, int H,
                      int d, int box_c = 64, int box_rows = kTile) {
  const void* ptr = t.ptr;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)t.st * 2, (cuuint64_t)t.sb * 2};
  cuuint32_t box[4] = {(cuuint32_t)box_c, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle swz = box_c == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : box_c == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GQA_ERR_INVALID_ARG, "%s: cuTensorMapEncodeTiled(%s) failed (%d)", fn, name, (int)r);
  return GQA_OK;
}

size_t round_up_tile(int T) { return ((size_t)T + kTile - 1) / kTile * kTile; }

// Fixed-point rotary frequencies (RopeFreq) of head dim d: pair i turns by
// base^(-2i/d) / (2 pi) per token, the same angles as attn_rope_table's.
gqa_status_t rope_freq(const char* fn, double base, int d, RopeFreq* rf) {
  if (!(base > 0.0) || !std::isfinite(base))
    return fail(GQA_ERR_INVALID_ARG, "%s: base must be positive and finite (got %g)", fn, base);
  memset(rf, 0, sizeof(*rf));
  for (int i = 0; i < d / 2; ++i) {
    const double turns = pow(base, -2.0 * i / d) / 6.283185307179586;  // per token, below 1/(2 pi)
    const uint64_t f = static_cast<uint64_t>(ldexp(turns, 64));
    rf->lo[i] = static_cast<uint32_t>(f);
    rf->hi[i] = static_cast<uint32_t>(f >> 32);
  }
  return GQA_OK;
}
// Task counters of the persistent dQ / dK/dV launch, after the two fp32 arrays.
constexpr size_t kSchedBytes = kBwdSchedBytes;

}  // namespace

extern "C" {

const char* attn_version(void) { return "0.1.0"; }

const char* attn_last_error(void) { return t_last_error.c_str(); }

void attn_set_wait_budget_ns(unsigned long long budget_ns) {
  g_budget_ns.store(budget_ns ? budget_ns : kDefaultBudgetNs);
}

gqa_status_t attn_set_task_order(int order) {
  t_last_error.clear();
  if (order < 0 || order > 2)
    return fail(GQA_ERR_INVALID_ARG, "attn_set_task_order: order must be 0 (by size), 1 (tile-major) or 2 "
                                     "(group-major) (got %d)", order);
  g_task_order.store(order);
  return GQA_OK;
}

size_t attn_bwd_workspace_bytes(int B, int T, int Hq) {
  if (B <= 0 || T <= 0 || Hq <= 0) return 0;
  return 2 * (size_t)B * (size_t)Hq * round_up_tile(T) * sizeof(float) + kSchedBytes;
}

}  // extern "C"

namespace {

// Shape, pointers and views already checked. Rotary (rf != null): q is the
// unrotated query, rotated in the kernel and written to q_rot; k is already rotated.
gqa_status_t fwd_impl(const char* fn, const View& q, const View& k, const View& v, const View& o, float* lse, int B,
                      int T, int Hq, int Hkv, int d, int causal, cudaStream_t stream, const View* q_rot = nullptr,
                      const RopeFreq* rf = nullptr) {
  gqa_status_t s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  if ((s = make_map(fn, "q", &p.tmap_q, q, B, T, Hq, d)) || (s = make_map(fn, "k", &p.tmap_k, k, B, T, Hkv, d)) ||
      (s = make_map(fn, "v", &p.tmap_v, v, B, T, Hkv, d)))
    return s;
  if ((s = make_map(fn, "o", &p.tmap_o, o, B, T, Hq, d, 64, 32))) return s;  // epilogue stores (32-row boxes)
  if (rf) {
    // the rotated Q tile leaves in the same 128-row boxes it arrived in
    if ((s = make_map(fn, "q_rot", &p.tmap_qrot, *q_rot, B, T, Hq, d))) return s;
    p.rope = 1;
    p.rope_f = *rf;
  }
  p.lse = lse;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.nT = (T + kTile - 1) / kTile;
  p.fd_bh = make_fastdiv((uint32_t)(B * Hq));
  p.fd_hq = make_fastdiv((uint32_t)Hq);
  p.fd_g = make_fastdiv((uint32_t)p.G);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p.status = ds->status;
  p.budget_ns = g_budget_ns.load();
  cudaError_t e = launch_fwd(p, d, stream);
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int Hq,
                      int Hkv, int d, int causal, void* stream) {
  const char* fn = "attn_fwd";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  if ((s = check_ptr(fn, "q", q)) || (s = check_ptr(fn, "k", k)) || (s = check_ptr(fn, "v", v)) ||
      (s = check_ptr(fn, "o", o)) || (s = check_ptr(fn, "lse", lse)))
    return s;
  return fwd_impl(fn, packed(q, T, Hq, d), packed(k, T, Hkv, d), packed(v, T, Hkv, d), packed(o, T, Hq, d), lse, B,
                  T, Hq, Hkv, d, causal, static_cast<cudaStream_t>(stream));
}

gqa_status_t attn_fwd_strided(gqa_view_t q, gqa_view_t k, gqa_view_t v, gqa_view_t o, float* lse, int B, int T,
                              int Hq, int Hkv, int d, int causal, void* stream) {
  const char* fn = "attn_fwd_strided";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  View vq, vk, vv, vo;
  if ((s = check_view(fn, "q", q, B, T, Hq, d, false, &vq)) || (s = check_view(fn, "k", k, B, T, Hkv, d, false, &vk)) ||
      (s = check_view(fn, "v", v, B, T, Hkv, d, false, &vv)) || (s = check_view(fn, "o", o, B, T, Hq, d, true, &vo)) ||
      (s = check_ptr(fn, "lse", lse)))
    return s;
  return fwd_impl(fn, vq, vk, vv, vo, lse, B, T, Hq, Hkv, d, causal, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Checks shared by the backward stages; fills the workspace pointers.
gqa_status_t check_workspace(const char* fn, const void* workspace, size_t workspace_bytes, int B, int T, int Hq,
                             float** Dvec, float** lse2, int* Tpad, unsigned** sched) {
  gqa_status_t s;
  if ((s = check_ptr(fn, "workspace", workspace))) return s;
  const size_t need = attn_bwd_workspace_bytes(B, T, Hq);
  if (workspace_bytes < need)
    return fail(GQA_ERR_INVALID_ARG, "%s: workspace_bytes %zu < required %zu", fn, workspace_bytes, need);
  *Tpad = (int)round_up_tile(T);
  *Dvec = static_cast<float*>(const_cast<void*>(workspace));
  *lse2 = *Dvec + (size_t)B * Hq * (*Tpad);
  *sched = reinterpret_cast<unsigned*>(*lse2 + (size_t)B * Hq * (*Tpad));
  return GQA_OK;
}

// Parameters of the dQ and dK/dV kernels (shape, pointers and tensor maps already checked by the caller).
gqa_status_t make_bwd_params(const char* fn, BwdParams* p, const View& q, const View& k, const View& v,
                             const View& dO, float* Dvec, float* lse2, unsigned* sched, int Tpad, int B, int T,
                             int Hq, int Hkv,
                             int d, int causal, DeviceState* ds) {
  memset(p, 0, sizeof(*p));
  gqa_status_t s;
  if ((s = make_map(fn, "q", &p->tmap_q, q, B, T, Hq, d)) || (s = make_map(fn, "k", &p->tmap_k, k, B, T, Hkv, d)) ||
      (s = make_map(fn, "v", &p->tmap_v, v, B, T, Hkv, d)) ||
      (s = make_map(fn, "dO", &p->tmap_do, dO, B, T, Hq, d)))
    return s;
  p->Dvec = Dvec;
  p->lse2 = lse2;
  p->sched = sched;
  p->B = B;
  p->T = T;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->G = Hq / Hkv;
  p->nT = (T + kTile - 1) / kTile;
  p->Tpad = Tpad;
  p->fd_nt = make_fastdiv((uint32_t)p->nT);
  p->fd_bk = make_fastdiv((uint32_t)(B * Hkv));
  p->fd_hkv = make_fastdiv((uint32_t)Hkv);
  p->fd_bh = make_fastdiv((uint32_t)(B * Hq));
  p->fd_hq = make_fastdiv((uint32_t)Hq);
  p->fd_g = make_fastdiv((uint32_t)p->G);
  p->fd_ntg = make_fastdiv((uint32_t)(p->nT * p->G));
  p->causal = causal ? 1 : 0;
  p->scale = (float)(1.0 / sqrt((double)d));
  p->scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
  p->status = ds->status;
  p->budget_ns = g_budget_ns.load();
  return GQA_OK;
}

// Shape and pointers of o, lse, dO already checked.
gqa_status_t bwd_preprocess_impl(const char* fn, const View& o, const float* lse, const View& dO, void* workspace,
                                 size_t workspace_bytes, int B, int T, int Hq, int d, cudaStream_t st) {
  gqa_status_t s;
  float *Dvec, *lse2;
  unsigned* sched;
  int Tpad;
  if ((s = check_workspace(fn, workspace, workspace_bytes, B, T, Hq, &Dvec, &lse2, &Tpad, &sched))) return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  BwdPreParams pp;
  pp.o = o.ptr;
  pp.dO = dO.ptr;
  pp.o_st16 = o.st / 8;  // strides are multiples of 8 elements (16 bytes)
  pp.o_sb16 = o.sb / 8;
  pp.do_st16 = dO.st / 8;
  pp.do_sb16 = dO.sb / 8;
  pp.lse = lse;
  pp.Dvec = Dvec;
  pp.lse2 = lse2;
  pp.sched = sched;
  pp.B = B;
  pp.T = T;
  pp.Hq = Hq;
  pp.Tpad = Tpad;
  cudaError_t e = launch_bwd_pre(pp, d, st);
  if (e != cudaSuccess) return cuda_fail(fn, "preprocess launch", e);
  return GQA_OK;
}

// which: 1 = dQ tasks, 2 = dK/dV tasks, 3 = both (one launch). Shape and the
// pointers of the views it uses already checked.
gqa_status_t bwd_main_impl(const char* fn, int which, const View& q, const View& k, const View& v, const View& dO,
                           const View& dq, const View& dk, const View& dv, const void* workspace,
                           size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal, cudaStream_t st,
                           const RopeFreq* rf = nullptr) {
  gqa_status_t s;
  float *Dvec, *lse2;
  unsigned* sched;
  int Tpad;
  if ((s = check_workspace(fn, workspace, workspace_bytes, B, T, Hq, &Dvec, &lse2, &Tpad, &sched))) return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  BwdParams p;
  if ((s = make_bwd_params(fn, &p, q, k, v, dO, Dvec, lse2, sched, Tpad, B, T, Hq, Hkv, d, causal, ds))) return s;
  p.dq = const_cast<void*>(dq.ptr);
  p.dk = const_cast<void*>(dk.ptr);
  p.dv = const_cast<void*>(dv.ptr);
  p.dq_st = dq.st;
  p.dq_sb = dq.sb;
  p.dk_st = dk.st;
  p.dk_sb = dk.sb;
  p.dv_st = dv.st;
  p.dv_sb = dv.sb;
  if (rf) {
    p.rope = 1;
    p.rope_f = *rf;
  }
  if (d == 64) {
    // d = 64 epilogues store through TMA, one 32-row box per compute warp: dQ 16
    // columns of a warpgroup, dK / dV 32 columns.
    if ((which & 1) && (s = make_map(fn, "dq", &p.tmap_dq, dq, B, T, Hq, d, 16, 32))) return s;
    if ((which & 2) && ((s = make_map(fn, "dk", &p.tmap_dk, dk, B, T, Hkv, d, 32, 32)) ||
                        (s = make_map(fn, "dv", &p.tmap_dv, dv, B, T, Hkv, d, 32, 32))))
      return s;
  }
  p.n_dkv_tasks = (which & 2) ? B * Hkv * p.nT : 0;
  p.n_dq_tasks = (which & 1) ? B * Hq * p.nT : 0;
  // Task order (results are the same bits either way: every output has one owner and
  // a fixed summation order). Tile-major, heaviest first over all (batch, kv head)
  // groups, has the ~one-task-per-SM tasks in flight read the streamed tiles of every
  // group; once those tiles (Q and dO for dK/dV tasks, K and V for dQ tasks) take
  // about half the L2 they are re-read from DRAM, and group-major order (one group's
  // tasks together, heaviest first within it) keeps the working set to a few groups.
  // Measured: group-major dK/dV tasks 1.7% faster with 74 MB of Q + dO (57% of the
  // L2), group-major dQ tasks 0.5% faster with 67 MB of K + V (52%; DRAM reads of the
  // T = 8192 workload 4.9x -> 2.0x the algorithmic bytes with both), but group-major
  // was slower with 17 MB (dQ, 2.7%) and neutral with 50 MB (dK/dV, 39%), where
  // tile-major balances the end of the launch better. The switch sits at 45%.
  const long long limit = ds->l2_bytes * 9 / 20;
  const long long qdo_bytes = 2LL * B * T * Hq * d * 2, kv_bytes = 2LL * B * T * Hkv * d * 2;
  const int order = g_task_order.load();
  p.dkv_group_major = order == 2 || (order == 0 && qdo_bytes > limit) ? 1 : 0;
  p.dq_group_major = order == 2 || (order == 0 && kv_bytes > limit) ? 1 : 0;
  cudaError_t e = launch_bwd_main(p, d, st);
  if (e != cudaSuccess) return cuda_fail(fn, "backward kernel launch", e);
  return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status_t attn_bwd_preprocess(const void* o, const float* lse, const void* dO, void* workspace,
                                 size_t workspace_bytes, int B, int T, int Hq, int d, void* stream) {
  const char* fn = "attn_bwd_preprocess";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, 1, d))) return s;
  if ((s = check_ptr(fn, "o", o)) || (s = check_ptr(fn, "lse", lse)) || (s = check_ptr(fn, "dO", dO))) return s;
  return bwd_preprocess_impl(fn, packed(o, T, Hq, d), lse, packed(dO, T, Hq, d), workspace, workspace_bytes, B, T,
                             Hq, d, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// attn_bwd_dq, attn_bwd_dkv and attn_bwd_dq_dkv on contiguous tensors.
gqa_status_t bwd_stage(const char* fn, int which, const void* q, const void* k, const void* v, const void* dO,
                       void* dq, void* dk, void* dv, const void* workspace, size_t workspace_bytes, int B, int T,
                       int Hq, int Hkv, int d, int causal, void* stream) {
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  if ((s = check_ptr(fn, "q", q)) || (s = check_ptr(fn, "k", k)) || (s = check_ptr(fn, "v", v)) ||
      (s = check_ptr(fn, "dO", dO)))
    return s;
  if ((which & 1) && (s = check_ptr(fn, "dq", dq))) return s;
  if ((which & 2) && ((s = check_ptr(fn, "dk", dk)) || (s = check_ptr(fn, "dv", dv)))) return s;
  return bwd_main_impl(fn, which, packed(q, T, Hq, d), packed(k, T, Hkv, d), packed(v, T, Hkv, d),
                       packed(dO, T, Hq, d), packed(dq, T, Hq, d), packed(dk, T, Hkv, d), packed(dv, T, Hkv, d),
                       workspace, workspace_bytes, B, T, Hq, Hkv, d, causal, static_cast<cudaStream_t>(stream));
}

// The whole backward on checked views: everything is validated before the first launch.
gqa_status_t bwd_impl(const char* fn, const View& q, const View& k, const View& v, const View& o, const float* lse,
                      const View& dO, const View& dq, const View& dk, const View& dv, void* workspace,
                      size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal, void* stream,
                      const RopeFreq* rf = nullptr) {
  gqa_status_t s;
  float *Dvec, *lse2;
  unsigned* sched;
  int Tpad;
  if ((s = check_workspace(fn, workspace, workspace_bytes, B, T, Hq, &Dvec, &lse2, &Tpad, &sched))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = bwd_preprocess_impl(fn, o, lse, dO, workspace, workspace_bytes, B, T, Hq, d, st))) return s;
  return bwd_main_impl(fn, 3, q, k, v, dO, dq, dk, dv, workspace, workspace_bytes, B, T, Hq, Hkv, d, causal, st,
                       rf);
}

}  // namespace

extern "C" {

gqa_status_t attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq,
                         const void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                         int causal, void* stream) {
  return bwd_stage("attn_bwd_dq", 1, q, k, v, dO, dq, nullptr, nullptr, workspace, workspace_bytes, B, T, Hq, Hkv,
                   d, causal, stream);
}

gqa_status_t attn_bwd_dkv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv,
                          const void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                          int causal, void* stream) {
  return bwd_stage("attn_bwd_dkv", 2, q, k, v, dO, nullptr, dk, dv, workspace, workspace_bytes, B, T, Hq, Hkv, d,
                   causal, stream);
}

gqa_status_t attn_bwd_dq_dkv(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk,
                             void* dv, const void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                             int d, int causal, void* stream) {
  return bwd_stage("attn_bwd_dq_dkv", 3, q, k, v, dO, dq, dk, dv, workspace, workspace_bytes, B, T, Hq, Hkv, d,
                   causal, stream);
}

gqa_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                      void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int T, int Hq,
                      int Hkv, int d, int causal, void* stream) {
  const char* fn = "attn_bwd";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  if ((s = check_ptr(fn, "q", q)) || (s = check_ptr(fn, "k", k)) || (s = check_ptr(fn, "v", v)) ||
      (s = check_ptr(fn, "o", o)) || (s = check_ptr(fn, "lse", lse)) || (s = check_ptr(fn, "dO", dO)) ||
      (s = check_ptr(fn, "dq", dq)) || (s = check_ptr(fn, "dk", dk)) || (s = check_ptr(fn, "dv", dv)))
    return s;
  return bwd_impl(fn, packed(q, T, Hq, d), packed(k, T, Hkv, d), packed(v, T, Hkv, d), packed(o, T, Hq, d), lse,
                  packed(dO, T, Hq, d), packed(dq, T, Hq, d), packed(dk, T, Hkv, d), packed(dv, T, Hkv, d), workspace,
                  workspace_bytes, B, T, Hq, Hkv, d, causal, stream);
}

gqa_status_t attn_bwd_strided(gqa_view_t q, gqa_view_t k, gqa_view_t v, gqa_view_t o, const float* lse,
                              gqa_view_t dO, gqa_view_t dq, gqa_view_t dk, gqa_view_t dv, void* workspace,
                              size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal,
                              void* stream) {
  const char* fn = "attn_bwd_strided";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  View vq, vk, vv, vo, vdo, vdq, vdk, vdv;
  if ((s = check_view(fn, "q", q, B, T, Hq, d, false, &vq)) || (s = check_view(fn, "k", k, B, T, Hkv, d, false, &vk)) ||
      (s = check_view(fn, "v", v, B, T, Hkv, d, false, &vv)) || (s = check_view(fn, "o", o, B, T, Hq, d, false, &vo)) ||
      (s = check_ptr(fn, "lse", lse)) || (s = check_view(fn, "dO", dO, B, T, Hq, d, false, &vdo)) ||
      (s = check_view(fn, "dq", dq, B, T, Hq, d, true, &vdq)) ||
      (s = check_view(fn, "dk", dk, B, T, Hkv, d, true, &vdk)) ||
      (s = check_view(fn, "dv", dv, B, T, Hkv, d, true, &vdv)))
    return s;
  return bwd_impl(fn, vq, vk, vv, vo, lse, vdo, vdq, vdk, vdv, workspace, workspace_bytes, B, T, Hq, Hkv, d, causal,
                  stream);
}

gqa_status_t attn_fwd_rope(gqa_view_t q, gqa_view_t k, gqa_view_t v, gqa_view_t o, float* lse, gqa_view_t q_rot,
                           gqa_view_t k_rot, double base, int B, int T, int Hq, int Hkv, int d, int causal,
                           void* stream) {
  const char* fn = "attn_fwd_rope";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  View vq, vk, vv, vo, vqr, vkr;
  if ((s = check_view(fn, "q", q, B, T, Hq, d, false, &vq)) || (s = check_view(fn, "k", k, B, T, Hkv, d, false, &vk)) ||
      (s = check_view(fn, "v", v, B, T, Hkv, d, false, &vv)) || (s = check_view(fn, "o", o, B, T, Hq, d, true, &vo)) ||
      (s = check_ptr(fn, "lse", lse)) || (s = check_view(fn, "q_rot", q_rot, B, T, Hq, d, true, &vqr)) ||
      (s = check_view(fn, "k_rot", k_rot, B, T, Hkv, d, true, &vkr)))
    return s;
  RopeFreq rf;
  if ((s = rope_freq(fn, base, d, &rf))) return s;
  if (vqr.ptr == vq.ptr && (vqr.st != vq.st || vqr.sb != vq.sb))
    return fail(GQA_ERR_INVALID_ARG, "%s: in place (q_rot == q) needs the same strides for q and q_rot", fn);
  if (vkr.ptr == vk.ptr && (vkr.st != vk.st || vkr.sb != vk.sb))
    return fail(GQA_ERR_INVALID_ARG, "%s: in place (k_rot == k) needs the same strides for k and k_rot", fn);
  if ((long long)B * T * ((Hkv + kRopeHeads - 1) / kRopeHeads) > 0x7fffffffLL / (d / 8))
    return fail(GQA_ERR_INVALID_ARG, "%s: problem too large for the key rotation (B*T = %lld)", fn, (long long)B * T);
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Keys: one rotation pass (each key tile is read by every query tile of its
  // group, so rotating it once beats rotating it at every load). Queries: rotated
  // in the attention kernel as each tile arrives, and stored from there.
  RopeParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.x = vk.ptr;
  rp.y = const_cast<void*>(vkr.ptr);
  rp.x_st16 = vk.st / 8;
  rp.x_sb16 = vk.sb / 8;
  rp.y_st16 = vkr.st / 8;
  rp.y_sb16 = vkr.sb / 8;
  rp.table = nullptr;  // angles from rf, as in the attention kernels
  rp.freq = rf;
  rp.B = B;
  rp.T = T;
  rp.H = Hkv;
  rp.inverse = 0;
  cudaError_t e = launch_rope(rp, d, st);
  if (e != cudaSuccess) return cuda_fail(fn, "key rotation launch", e);
  return fwd_impl(fn, vq, vkr, vv, vo, lse, B, T, Hq, Hkv, d, causal, st, &vqr, &rf);
}

gqa_status_t attn_bwd_rope(gqa_view_t q_rot, gqa_view_t k_rot, gqa_view_t v, gqa_view_t o, const float* lse,
                           gqa_view_t dO, gqa_view_t dq, gqa_view_t dk, gqa_view_t dv, double base,
                           void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal,
                           void* stream) {
  const char* fn = "attn_bwd_rope";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  View vq, vk, vv, vo, vdo, vdq, vdk, vdv;
  if ((s = check_view(fn, "q_rot", q_rot, B, T, Hq, d, false, &vq)) ||
      (s = check_view(fn, "k_rot", k_rot, B, T, Hkv, d, false, &vk)) ||
      (s = check_view(fn, "v", v, B, T, Hkv, d, false, &vv)) || (s = check_view(fn, "o", o, B, T, Hq, d, false, &vo)) ||
      (s = check_ptr(fn, "lse", lse)) || (s = check_view(fn, "dO", dO, B, T, Hq, d, false, &vdo)) ||
      (s = check_view(fn, "dq", dq, B, T, Hq, d, true, &vdq)) ||
      (s = check_view(fn, "dk", dk, B, T, Hkv, d, true, &vdk)) ||
      (s = check_view(fn, "dv", dv, B, T, Hkv, d, true, &vdv)))
    return s;
  RopeFreq rf;
  if ((s = rope_freq(fn, base, d, &rf))) return s;
  return bwd_impl(fn, vq, vk, vv, vo, lse, vdo, vdq, vdk, vdv, workspace, workspace_bytes, B, T, Hq, Hkv, d, causal,
                  stream, &rf);
}

size_t attn_naive_workspace_bytes(int B, int T, int Hq) {
  if (B <= 0 || T <= 0 || Hq <= 0) return 0;
  return naive_workspace_bytes(NaiveShape{B, T, Hq, 1, 64});
}

}  // extern "C"

namespace {

gqa_status_t naive_checks(const char* fn, const void* workspace, size_t workspace_bytes, int B, int T, int Hq,
                          int Hkv, int d) {
  gqa_status_t s;
  if ((s = check_shape(fn, B, T, Hq, Hkv, d))) return s;
  // one block per score row and (T/16)^2 tiles per head: keep the grids in range
  if ((long long)B * Hq * T > 0x7fffffffLL || (long long)B * Hq > 65535)
    return fail(GQA_ERR_INVALID_ARG, "%s: problem too large for the naive kernels", fn);
  if ((s = check_ptr(fn, "workspace", workspace))) return s;
  const size_t need = attn_naive_workspace_bytes(B, T, Hq);
  if (workspace_bytes < need)
    return fail(GQA_ERR_INVALID_ARG, "%s: workspace_bytes %zu < required %zu", fn, workspace_bytes, need);
  return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status_t attn_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, int causal, void* stream) {
  const char* fn = "attn_fwd_naive";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = naive_checks(fn, workspace, workspace_bytes, B, T, Hq, Hkv, d))) return s;
  if ((s = check_ptr(fn, "q", q)) || (s = check_ptr(fn, "k", k)) || (s = check_ptr(fn, "v", v)) ||
      (s = check_ptr(fn, "o", o)) || (s = check_ptr(fn, "lse", lse)))
    return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  NaiveFwdArgs a;
  a.s = NaiveShape{B, T, Hq, Hkv, d};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.workspace = workspace;
  a.scale = (float)(1.0 / sqrt((double)d));
  a.causal = causal ? 1 : 0;
  cudaError_t e = launch_naive_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

gqa_status_t attn_bwd_naive(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            int B, int T, int Hq, int Hkv, int d, int causal, void* stream) {
  const char* fn = "attn_bwd_naive";
  t_last_error.clear();
  gqa_status_t s;
  if ((s = naive_checks(fn, workspace, workspace_bytes, B, T, Hq, Hkv, d))) return s;
  if ((s = check_ptr(fn, "q", q)) || (s = check_ptr(fn, "k", k)) || (s = check_ptr(fn, "v", v)) ||
      (s = check_ptr(fn, "o", o)) || (s = check_ptr(fn, "lse", lse)) || (s = check_ptr(fn, "dO", dO)) ||
      (s = check_ptr(fn, "dq", dq)) || (s = check_ptr(fn, "dk", dk)) || (s = check_ptr(fn, "dv", dv)))
    return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  NaiveBwdArgs a;
  a.s = NaiveShape{B, T, Hq, Hkv, d};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.scale = (float)(1.0 / sqrt((double)d));
  a.causal = causal ? 1 : 0;
  cudaError_t e = launch_naive_bwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

size_t attn_rope_table_bytes(int T, int d) {
  if (T <= 0 || (d != 64 && d != 128)) return 0;
  return (size_t)T * (size_t)(d / 2) * 2 * sizeof(float);
}

gqa_status_t attn_rope_table(float* table, int T, int d, double base, void* stream) {
  const char* fn = "attn_rope_table";
  t_last_error.clear();
  gqa_status_t s;
  if (T <= 0 || T > (1 << 30)) return fail(GQA_ERR_INVALID_ARG, "%s: T must be in [1, 2^30] (got %d)", fn, T);
  if (d != 64 && d != 128) return fail(GQA_ERR_INVALID_ARG, "%s: d must be 64 or 128 (got %d)", fn, d);
  if (!(base > 0.0) || !std::isfinite(base))
    return fail(GQA_ERR_INVALID_ARG, "%s: base must be positive and finite (got %g)", fn, base);
  if ((s = check_ptr(fn, "table", table))) return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  RopeTableParams p;
  memset(&p, 0, sizeof(p));
  p.table = table;
  p.T = T;
  p.half_d = d / 2;
  for (int i = 0; i < d / 2; ++i) p.theta[i] = pow(base, -2.0 * i / d);
  cudaError_t e = launch_rope_table(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

gqa_status_t attn_rope(gqa_view_t x, gqa_view_t y, const float* table, int B, int T, int H, int d, int inverse,
                       void* stream) {
  const char* fn = "attn_rope";
  t_last_error.clear();
  gqa_status_t s;
  if (B <= 0 || T <= 0 || H <= 0)
    return fail(GQA_ERR_INVALID_ARG, "%s: B, T, H must be positive (got %d, %d, %d)", fn, B, T, H);
  if (d != 64 && d != 128) return fail(GQA_ERR_INVALID_ARG, "%s: d must be 64 or 128 (got %d)", fn, d);
  if ((long long)B * T * ((H + kRopeHeads - 1) / kRopeHeads) > 0x7fffffffLL / (d / 8))
    return fail(GQA_ERR_INVALID_ARG, "%s: problem too large (B*T = %lld, H = %d)", fn, (long long)B * T, H);
  View vx, vy;
  if ((s = check_view(fn, "x", x, B, T, H, d, false, &vx)) || (s = check_view(fn, "y", y, B, T, H, d, true, &vy)) ||
      (s = check_ptr(fn, "table", table)))
    return s;
  if (vx.ptr == vy.ptr && (vx.st != vy.st || vx.sb != vy.sb))
    return fail(GQA_ERR_INVALID_ARG, "%s: in place (y == x) needs the same strides for x and y", fn);
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  RopeParams p;
  memset(&p, 0, sizeof(p));
  p.x = vx.ptr;
  p.y = const_cast<void*>(vy.ptr);
  p.x_st16 = vx.st / 8;
  p.x_sb16 = vx.sb / 8;
  p.y_st16 = vy.st / 8;
  p.y_sb16 = vy.sb / 8;
  p.table = table;
  p.B = B;
  p.T = T;
  p.H = H;
  p.inverse = inverse ? 1 : 0;
  cudaError_t e = launch_rope(p, d, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

gqa_status_t attn_sync_status(void* stream) {
  const char* fn = "attn_sync_status";
  t_last_error.clear();
  DeviceState* ds = nullptr;
  gqa_status_t s;
  if ((s = device_state(fn, &ds))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaStreamSynchronize", e);
  DevStatusWord w;
  e = cudaMemcpy(&w, ds->status, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaMemcpy(status word)", e);
  if (w.code == kDevOk) return GQA_OK;
  static const char* names[] = {"?", "attn_fwd", "bwd_preprocess", "bwd_main", "?", "?", "?", "?", "probe",
                                "selftest"};
  const char* kname = w.kernel < 10 ? names[w.kernel] : "?";
  DevStatusWord zero;
  memset(&zero, 0, sizeof(zero));
  e = cudaMemcpy(ds->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaMemcpy(clear status word)", e);
  return fail(GQA_ERR_TIMEOUT, "%s: kernel %s gave up waiting (wait %u, block %u)", fn, kname, w.where, w.block);
}

gqa_status_t attn_probe_mma(int n, int a_tmem, int chains, int iters, void* out, void* stream) {
  const char* fn = "attn_probe_mma";
  t_last_error.clear();
  if (n != 64 && n != 128 && n != 256) return fail(GQA_ERR_INVALID_ARG, "%s: n must be 64, 128 or 256 (got %d)", fn, n);
  if (chains != 1 && chains != 2) return fail(GQA_ERR_INVALID_ARG, "%s: chains must be 1 or 2 (got %d)", fn, chains);
  if (chains == 2 && a_tmem && n == 256)
    return fail(GQA_ERR_INVALID_ARG, "%s: two accumulators of N = 256 leave no TMEM columns for A", fn);
  if (iters <= 0 || iters > (1 << 20)) return fail(GQA_ERR_INVALID_ARG, "%s: iters must be in [1, 2^20]", fn);
  gqa_status_t s;
  if ((s = check_ptr(fn, "out", out))) return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaDeviceGetAttribute", e);
  e = launch_mma_probe(n, a_tmem ? 1 : 0, chains, iters, out, ds->status, g_budget_ns.load(), sms,
                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

gqa_status_t attn_probe_ex2(int iters, void* out, void* sink, void* stream) {
  const char* fn = "attn_probe_ex2";
  t_last_error.clear();
  if (iters <= 0 || iters > (1 << 20)) return fail(GQA_ERR_INVALID_ARG, "%s: iters must be in [1, 2^20]", fn);
  gqa_status_t s;
  if ((s = check_ptr(fn, "out", out)) || (s = check_ptr(fn, "sink", sink))) return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaDeviceGetAttribute", e);
  e = launch_ex2_probe(iters, static_cast<unsigned long long*>(out), static_cast<float*>(sink), sms,
                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

gqa_status_t attn_probe_tma(const void* buf, long long bytes, int stages, int ctas_per_sm, int iters, void* out,
                            void* stream) {
  const char* fn = "attn_probe_tma";
  t_last_error.clear();
  if (bytes < 16384 || bytes % 16384 != 0 || bytes / 16384 > 0x7fffffffLL)
    return fail(GQA_ERR_INVALID_ARG, "%s: bytes must be a positive multiple of 16384 (got %lld)", fn, bytes);
  if (ctas_per_sm != 1 && ctas_per_sm != 2)
    return fail(GQA_ERR_INVALID_ARG, "%s: ctas_per_sm must be 1 or 2 (got %d)", fn, ctas_per_sm);
  const int max_stages = ctas_per_sm == 1 ? 8 : 6;  // 16 KB slots a CTA, two CTAs sharing an SM's 228 KB
  if (stages < 1 || stages > max_stages)
    return fail(GQA_ERR_INVALID_ARG, "%s: stages must be in [1, %d] with %d CTA(s) per SM (got %d)", fn, max_stages,
                ctas_per_sm, stages);
  if (iters <= 0 || iters > (1 << 20)) return fail(GQA_ERR_INVALID_ARG, "%s: iters must be in [1, 2^20]", fn);
  gqa_status_t s;
  if ((s = check_ptr(fn, "buf", buf)) || (s = check_ptr(fn, "out", out))) return s;
  DeviceState* ds = nullptr;
  if ((s = device_state(fn, &ds))) return s;
  // the buffer as bf16 rows of 64 (128 bytes), read in boxes of 128 rows
  const cuuint64_t rows = static_cast<cuuint64_t>(bytes / 128);
  CUtensorMap map;
  cuuint64_t dims[4] = {64, 1, rows, 1};
  cuuint64_t strides[3] = {128, 128, rows * 128};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(buf), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GQA_ERR_INVALID_ARG, "%s: cuTensorMapEncodeTiled failed (%d)", fn, (int)r);
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return cuda_fail(fn, "cudaDeviceGetAttribute", e);
  e = launch_tma_probe(map, static_cast<int>(bytes / 16384), stages, ctas_per_sm, iters,
                       static_cast<unsigned long long*>(out), ds->status, g_budget_ns.load(), sms,
                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

gqa_status_t attn_selftest_timeout(unsigned long long budget_ns, void* stream) {
  const char* fn = "attn_selftest_timeout";
  t_last_error.clear();
  DeviceState* ds = nullptr;
  gqa_status_t s;
  if ((s = device_state(fn, &ds))) return s;
  cudaError_t e = launch_selftest_timeout(ds->status, budget_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(fn, "kernel launch", e);
  return GQA_OK;
}

}  // extern "C"
