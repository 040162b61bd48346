// api_noalloc.cu — attn_bwd_noalloc: the backward pass with its scratch held
// in a fixed array inside the library instead of a buffer from the caller.
//
// Who needs this: code that is not allowed to allocate device memory at the
// point where it runs the backward. Examples are a serving or training loop
// whose device memory is all handed out up front by a pool it does not own
// (a stray cudaMalloc there either fails or fragments that pool), and
// latency-sensitive loops where cudaMalloc/cudaFree are avoided because they
// can synchronise the whole device. Such callers still own their inputs and
// outputs; only the backward's scratch (D and the log2-unit LSE, two fp32
// arrays of [B, Hq, T rounded up to 128]) moves into this array.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds its kNoallocScratchBytes until the process exits, whether or
// not this entry point is used. Host code cannot use the array's name as a
// device address: it asks the runtime for the address once per device and
// passes that pointer to the kernels through the ordinary workspace argument
// of the existing backward stages.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/gqa_attn.h"
#include "attn_common.cuh"

namespace gqa {
void set_last_error_message(const char* msg);        // defined in api.cu
gqa_status_t check_current_device(const char* fn);   // defined in api.cu
}

namespace {

constexpr size_t kNoallocScratchBytes = GQA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

extern "C" gqa_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                         const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                                         int T, int Hq, int Hkv, int d, int causal, void* stream) {
  char msg[256];
  const size_t need = attn_bwd_workspace_bytes(B, T, Hq);
  if (need == 0) {
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc: B, T, Hq must be positive (got %d, %d, %d)", B, T, Hq);
    gqa::set_last_error_message(msg);
    return GQA_ERR_INVALID_ARG;
  }
  if (need > kNoallocScratchBytes) {
    // D and LSE2 take 8 bytes per padded row; the task counters take the rest
    snprintf(msg, sizeof(msg),
             "attn_bwd_noalloc: problem needs %zu bytes of scratch, more than the library's fixed %zu "
             "(B*Hq*roundup(T,128) must be <= %zu); use attn_bwd with a caller workspace",
             need, kNoallocScratchBytes, (kNoallocScratchBytes - gqa::kBwdSchedBytes) / 8);
    gqa::set_last_error_message(msg);
    return GQA_ERR_INVALID_ARG;
  }
  // Device range and compute capability first (GQA_ERR_UNSUPPORTED_DEVICE), so the
  // symbol lookup below only ever runs on a device this library has code for.
  const gqa_status_t ds = gqa::check_current_device("attn_bwd_noalloc");
  if (ds != GQA_OK) return ds;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    gqa::set_last_error_message(msg);
    return GQA_ERR_LAUNCH;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(msg, sizeof(msg), "attn_bwd_noalloc: device %d out of range", dev);
    gqa::set_last_error_message(msg);
    return GQA_ERR_UNSUPPORTED_DEVICE;
  }
  void* scratch = nullptr;
  {
    // First call on this device, with it current: look up where the array lives on it.
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
      if (e != cudaSuccess || !ptr) {
        snprintf(msg, sizeof(msg), "attn_bwd_noalloc: cudaGetSymbolAddress(scratch) failed: %s",
                 cudaGetErrorString(e));
        gqa::set_last_error_message(msg);
        return GQA_ERR_LAUNCH;
      }
      g_scratch_ptr[dev] = ptr;
    }
    scratch = g_scratch_ptr[dev];
  }
  // The preprocess rewrites every element the dQ and dK/dV kernels read
  // (padding rows included), so the previous call's contents never leak in
  // and nothing needs clearing first.
  return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, kNoallocScratchBytes, B, T, Hq, Hkv, d, causal,
                  stream);
}
