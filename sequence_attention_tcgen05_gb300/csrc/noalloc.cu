// usp_attention_noalloc: usp_attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code embedded in a host application that owns
// every device allocation (its allocator is not reachable from here), or latency-critical paths
// where cudaMalloc's implicit device synchronisation is not acceptable.  For them this entry point
// uses a fixed scratch array compiled into the library instead of a caller-provided workspace.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU on which the library's
// device code is loaded holds it until the process exits.  In host code the array's name is only a
// host-side stand-in, so its device address is looked up with cudaGetSymbolAddress, with the
// device current, on the first call on each device and cached.  The cache entry remembers the
// CUDA context it was taken in: if the device's context changes (cudaDeviceReset and a new
// context, where the module and its array are loaded again), the next call looks the address up
// again instead of using a stale one.
//
// All calls share the one array and it keeps the previous call's contents.  Only the status word
// at its start must begin at zero, and each call clears it.  Calls that overlap on the GPU (other
// streams, other host threads on the same device) race on the array and must be serialised by the
// caller.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(128) << 20;  // 128 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_usp_scratch[kScratchBytes];

std::mutex g_scratch_mu;
struct ScratchEntry {
  void* ctx = nullptr;   // CUcontext the address was looked up in
  void* addr = nullptr;  // device address of g_usp_scratch in that context
};
ScratchEntry g_scratch[kMaxDevices];

// The driver's cuCtxGetCurrent, reached through the runtime's entry-point query so that the library
// does not link the driver library itself.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

usp_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return usp::fail(USP_ERR_NO_DEVICE, "usp_attention_noalloc: no CUDA device is current");
  }
  if (dev < 0 || dev >= kMaxDevices)
    return usp::fail(USP_ERR_UNSUPPORTED, "usp_attention_noalloc: device ordinal %d >= %d", dev, kMaxDevices);
  // The current context (null before the runtime has created it); the lookup below creates it.
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (!get_ctx) return usp::fail(USP_ERR_CUDA, "usp_attention_noalloc: cuCtxGetCurrent is not available");
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (!ent.addr || !ctx || ent.ctx != static_cast<void*>(ctx)) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_usp_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return usp::fail(USP_ERR_CUDA, "usp_attention_noalloc: cudaGetSymbolAddress of the scratch array: %s",
                       cudaGetErrorString(e));
    }
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
      return usp::fail(USP_ERR_CUDA, "usp_attention_noalloc: no current CUDA context on device %d", dev);
    ent.ctx = ctx;
    ent.addr = p;
  }
  *out = ent.addr;
  return USP_OK;
}

}  // namespace

extern "C" usp_status_t usp_attention_noalloc(const void* q, const void* k, const void* v, int B,
                                              int S, int H, int D, float scale, int causal,
                                              int ulysses_degree, int ring_degree,
                                              const int32_t* seq_lens, const int32_t* head_counts,
                                              usp_order_t order, void* o, usp_dtype_t o_dt,
                                              float* lse, uint32_t* status, usp_stream_t stream) {
  const size_t need = usp_attention_workspace_size(B, S, H, D, causal, ulysses_degree, ring_degree, order, o_dt);
  if (need == 0) {
    // invalid arguments: let usp_attention's validation report the precise error (it returns
    // before any launch when an argument is invalid)
    return usp_attention(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, seq_lens,
                         head_counts, order, o, o_dt, lse, nullptr, 0, stream);
  }
  // the pointer checks usp_attention makes, before the status word is cleared in the stream
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (!q || !k || !v || !o) return usp::fail(USP_ERR_INVALID_ARG, "NULL q, k, v or o");
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      (lse && misaligned(lse, 4)))
    return usp::fail(USP_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (need > kScratchBytes)
    return usp::fail(USP_ERR_WORKSPACE,
                     "usp_attention_noalloc: this problem needs %zu bytes of scratch, more than the "
                     "%zu-byte (128 MiB) array built into the library; use usp_attention with a "
                     "workspace instead",
                     need, kScratchBytes);
  void* scratch = nullptr;
  if (usp_status_t st = scratch_for_current_device(&scratch)) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);  // the status word
  if (e != cudaSuccess)
    return usp::fail(USP_ERR_CUDA, "usp_attention_noalloc: clearing the status word: %s", cudaGetErrorString(e));
  usp_status_t st = usp_attention(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree,
                                  seq_lens, head_counts, order, o, o_dt, lse, scratch, kScratchBytes,
                                  stream);
  if (st != USP_OK) return st;
  if (status) {
    e = cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess)
      return usp::fail(USP_ERR_CUDA, "usp_attention_noalloc: copying the status word: %s", cudaGetErrorString(e));
  }
  return USP_OK;
}
