// usp_attention_noalloc: usp_attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: code embedded in a host application that owns
// every device allocation (its allocator is not reachable from here), or latency-critical paths
// where cudaMalloc's implicit device synchronisation is not acceptable.  For them this entry point
// uses a fixed scratch array compiled into the library instead of a caller-provided workspace.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU on which the library's
// device code is loaded holds it until the process exits.  In host code the array's name is only a
// host-side stand-in, so its device address is looked up with cudaGetSymbolAddress once per
// device (on that device's first call, with the device current) and cached.
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
void* g_scratch_addr[kMaxDevices] = {};

usp_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return usp::fail(USP_ERR_NO_DEVICE, "usp_attention_noalloc: no CUDA device is current");
  }
  if (dev < 0 || dev >= kMaxDevices)
    return usp::fail(USP_ERR_UNSUPPORTED, "usp_attention_noalloc: device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_usp_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return usp::fail(USP_ERR_CUDA, "usp_attention_noalloc: cudaGetSymbolAddress of the scratch array: %s",
                       cudaGetErrorString(e));
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return USP_OK;
}

}  // namespace

extern "C" usp_status_t usp_attention_noalloc(const void* q, const void* k, const void* v, int B,
                                              int S, int H, int D, float scale, int causal,
                                              int ulysses_degree, int ring_degree,
                                              const int32_t* seq_lens, const int32_t* head_counts,
                                              usp_order_t order, void* o, usp_dtype_t o_dt,
                                              float* lse, uint32_t* status, usp_stream_t stream) {
  const size_t need = usp_attention_workspace_size(B, S, H, D, ulysses_degree, ring_degree, order, o_dt);
  if (need == 0) {
    // invalid arguments: let usp_attention's validation report the precise error (it returns
    // before any launch when an argument is invalid)
    return usp_attention(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, seq_lens,
                         head_counts, order, o, o_dt, lse, nullptr, 0, stream);
  }
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
