// Re-layout kernels: the Ulysses all-to-alls as local permutations ([CP] Ulysses Attention;
// [UAA] arbitrary per-rank lengths), ring-chunk reordering ([YC] contiguous / zigzag / stripe)
// and their fusion.  Pure data movement, bit-exact, HBM-bound.
//
// Every (tensor, row, head group) moves one contiguous block of h_g * D elements on both sides
// (h_g * D * elem bytes: 3 KB for 12 bf16 heads of 128).  One warp copies one block: its lanes
// issue every 16-byte (or narrower, when an offset is not aligned) vector load of the block, up
// to kNV per lane, before the first store, so a warp keeps the whole block in flight and waits
// for one memory latency per block.  Blocks are numbered tensor-major, then row, then head
// group, so the warps of a CTA read neighbouring memory on the sequence side; with one block per
// warp the hardware's CTA scheduler balances the work.
#include <algorithm>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace usp {
namespace {

template <int VEC>
struct Vec;
template <>
struct Vec<16> { using T = uint4; };
template <>
struct Vec<8> { using T = uint2; };
template <>
struct Vec<4> { using T = uint32_t; };
template <>
struct Vec<2> { using T = uint16_t; };

// Position of ring-local row `row` (of all tensors' row space) on both sides: its ring group r,
// batch b, ring-local row l, and the element offset of its first element on the sequence side.
struct RowPlace {
  int r, b, l;
  long long seq_elem;
};

__device__ __forceinline__ RowPlace place_row(const RelayoutParams& p, long long row) {
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.row0[mid] <= row) lo = mid; else hi = mid - 1;
  }
  RowPlace x;
  x.r = lo;
  const int Sr = p.S_r[lo];
  const long long rr = row - p.row0[lo];
  x.b = static_cast<int>(rr / Sr);
  x.l = static_cast<int>(rr - static_cast<long long>(x.b) * Sr);
  const long long HD = p.seq_rs;
  if (p.seq_mode == 0) {
    const int base = x.r * p.U;
    int a = 0, z = p.U - 1;
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (p.c_off[base + mid] <= x.l) a = mid; else z = mid - 1;
    }
    const int c = base + a;
    x.seq_elem = p.c_base[c] + (static_cast<long long>(x.b) * p.c_len[c] + (x.l - p.c_off[c])) * HD;
  } else {
    const long long pos = x.l < p.p_len0[x.r]
                              ? p.p_start0[x.r] + static_cast<long long>(x.l) * p.p_stride[x.r]
                              : p.p_start1[x.r] + static_cast<long long>(x.l - p.p_len0[x.r]) * p.p_stride[x.r];
    x.seq_elem = (static_cast<long long>(x.b) * p.S + pos) * HD;
  }
  return x;
}

constexpr int kNV = 8;  // vectors in flight per lane (4 KB per warp with 16-byte vectors)

// One warp per (tensor, row, head group) block: the lanes issue every vector load of the block
// (up to kNV per lane per batch) before the first store.  Under programmatic dependent launch a
// warp places its first block before it waits for the previous kernel of the stream: at 57 MB a
// launch, that moved the head->seq re-layout of O from 5.34 to 5.78 TB/s back to back.
template <int VEC>
__global__ void __launch_bounds__(256) relayout_block_kernel(const __grid_constant__ RelayoutParams p,
                                                             long long n_blocks) {
  using T = typename Vec<VEC>::T;
  pdl_launch_dependents();
  bool waited = false;  // the first block's addresses come from the parameters before the wait
  const int lane = threadIdx.x & 31;
  const long long rows = p.row0[p.R];
  const long long per_tensor = rows * p.U;
  const long long step = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long blk = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       blk < n_blocks; blk += step) {
    const int tensor = static_cast<int>(blk / per_tensor);
    const long long rest = blk - tensor * per_tensor;
    const long long row = rest / p.U;
    const int g = static_cast<int>(rest - row * p.U);
    const RowPlace x = place_row(p, row);
    const long long hg = static_cast<long long>(p.h[g]) * p.D;
    const long long head_elem = p.hbase[x.r * p.U + g] + (static_cast<long long>(x.b) * p.S_r[x.r] + x.l) * hg;
    const long long seq_g = x.seq_elem + static_cast<long long>(p.hoff[g]) * p.D;
    const int nvec = static_cast<int>(hg * p.elem / VEC);
    const T* __restrict__ src = reinterpret_cast<const T*>(p.src[tensor] + (p.dir == 0 ? seq_g : head_elem) * p.elem);
    T* __restrict__ dst = reinterpret_cast<T*>(p.dst[tensor] + (p.dir == 0 ? head_elem : seq_g) * p.elem);
    if (!waited) {  // warp-uniform
      pdl_wait();
      waited = true;
    }
    for (int v0 = 0; v0 < nvec; v0 += 32 * kNV) {
      T buf[kNV];
#pragma unroll
      for (int i = 0; i < kNV; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < nvec) buf[i] = __ldcs(src + v);
      }
#pragma unroll
      for (int i = 0; i < kNV; ++i) {
        const int v = v0 + i * 32 + lane;
        if (v < nvec) dst[v] = buf[i];
      }
    }
  }
}

// Small rows (fewer than 32 vectors, e.g. an LSE row of H floats): one thread per token row, which
// places the row once and copies its vectors with all loads issued before the stores.
template <int VEC>
__global__ void __launch_bounds__(256) relayout_small_kernel(const __grid_constant__ RelayoutParams p) {
  using T = typename Vec<VEC>::T;
  constexpr int kBatch = 8;
  pdl_prologue();
  const char* __restrict__ src = p.src[blockIdx.y];
  char* __restrict__ dst = p.dst[blockIdx.y];
  const long long total = p.row0[p.R];
  for (long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; row < total;
       row += static_cast<long long>(gridDim.x) * blockDim.x) {
    const RowPlace x = place_row(p, row);
    const int r = x.r, b = x.b, l = x.l;
    const int Sr = p.S_r[r];
    const long long seq_elem = x.seq_elem;
    for (int g = 0; g < p.U; ++g) {
      const long long hg = static_cast<long long>(p.h[g]) * p.D;
      const long long head_elem = p.hbase[r * p.U + g] + (static_cast<long long>(b) * Sr + l) * hg;
      const long long seq_g = seq_elem + static_cast<long long>(p.hoff[g]) * p.D;
      const int nvec = static_cast<int>(hg * p.elem / VEC);
      const T* s = reinterpret_cast<const T*>(src + (p.dir == 0 ? seq_g : head_elem) * p.elem);
      T* d = reinterpret_cast<T*>(dst + (p.dir == 0 ? head_elem : seq_g) * p.elem);
      for (int v0 = 0; v0 < nvec; v0 += kBatch) {
        T buf[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (v0 + i < nvec) buf[i] = __ldcs(s + v0 + i);
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (v0 + i < nvec) d[v0 + i] = buf[i];
      }
    }
  }
}

}  // namespace

usp_status_t launch_relayout(RelayoutParams& p, cudaStream_t stream) {
  const long long total = p.row0[p.R];
  if (total == 0) return USP_OK;
  // widest vector every byte offset allows
  long long g = 16;
  auto fold = [&](long long x) {
    while (g > p.elem && (x % g) != 0) g >>= 1;
  };
  fold(static_cast<long long>(p.H) * p.D * p.elem);
  fold(p.seq_rs * p.elem);
  for (int u = 0; u < p.U; ++u) {
    fold(static_cast<long long>(p.h[u]) * p.D * p.elem);
    fold(static_cast<long long>(p.hoff[u]) * p.D * p.elem);
  }
  for (int i = 0; i < p.R * p.U; ++i) {
    fold(p.hbase[i] * p.elem);
    if (p.seq_mode == 0) fold(p.c_base[i] * p.elem);
  }
  for (int t = 0; t < p.n_tensors; ++t) {
    fold(static_cast<long long>(reinterpret_cast<uintptr_t>(p.src[t]) & 15));
    fold(static_cast<long long>(reinterpret_cast<uintptr_t>(p.dst[t]) & 15));
  }
  const long long nv = static_cast<long long>(p.H) * p.D * p.elem / g;  // vectors per row
  const long long sms = sm_count();
  if (nv < 32) {
    long long blocks = (total + 255) / 256;
    if (blocks > sms * 16) blocks = sms * 16;
    dim3 grid(static_cast<unsigned>(blocks), p.n_tensors);
    cudaError_t e;
    switch (g) {
      case 16: e = launch_pdl(relayout_small_kernel<16>, grid, dim3(256), 0, stream, p); break;
      case 8: e = launch_pdl(relayout_small_kernel<8>, grid, dim3(256), 0, stream, p); break;
      case 4: e = launch_pdl(relayout_small_kernel<4>, grid, dim3(256), 0, stream, p); break;
      default: e = launch_pdl(relayout_small_kernel<2>, grid, dim3(256), 0, stream, p); break;
    }
    if (e != cudaSuccess) return fail(USP_ERR_CUDA, "relayout kernel: %s", cudaGetErrorString(e));
    return check_launch("relayout kernel");
  }
  // one warp per (tensor, row, head group) block, 8 warps per CTA; the hardware hands CTAs to the
  // SMs as slots free up (a grid-stride loop takes over beyond 2^24 CTAs)
  const long long n_blocks = total * p.U * p.n_tensors;
  long long ctas = (n_blocks + 7) / 8;
  if (ctas > (1LL << 24)) ctas = 1LL << 24;
  const unsigned grid = static_cast<unsigned>(ctas);
  cudaError_t e;
  switch (g) {
    case 16: e = launch_pdl(relayout_block_kernel<16>, dim3(grid), dim3(256), 0, stream, p, n_blocks); break;
    case 8: e = launch_pdl(relayout_block_kernel<8>, dim3(grid), dim3(256), 0, stream, p, n_blocks); break;
    case 4: e = launch_pdl(relayout_block_kernel<4>, dim3(grid), dim3(256), 0, stream, p, n_blocks); break;
    default: e = launch_pdl(relayout_block_kernel<2>, dim3(grid), dim3(256), 0, stream, p, n_blocks); break;
  }
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "relayout kernel: %s", cudaGetErrorString(e));
  return check_launch("relayout kernel");
}

}  // namespace usp
