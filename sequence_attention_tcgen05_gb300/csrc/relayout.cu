// Re-layout kernels: the Ulysses all-to-alls as local permutations ([CP] Ulysses Attention;
// [UAA] arbitrary per-rank lengths), ring-chunk reordering ([YC] contiguous / zigzag / stripe)
// and their fusion.  Pure data movement, bit-exact, HBM-bound.
//
// Every (row, head group) moves one contiguous block of h_g * D elements on both sides, so the
// kernel copies whole blocks with the widest vector (16, 8, 4 or 2 bytes) that every offset
// allows.  One warp walks one row; its lanes stride over the row's vectors with four loads in
// flight per lane.
#include <cstdio>

#include "internal.h"

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

template <int VEC>
__device__ __forceinline__ void copy_block(char* __restrict__ d, const char* __restrict__ s,
                                           int nvec, int lane) {
  using T = typename Vec<VEC>::T;
  const T* src = reinterpret_cast<const T*>(s);
  T* dst = reinterpret_cast<T*>(d);
  int v = lane;
  for (; v + 96 < nvec; v += 128) {
    T a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64), e = __ldg(src + v + 96);
    dst[v] = a;
    dst[v + 32] = b;
    dst[v + 64] = c;
    dst[v + 96] = e;
  }
  for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
}

template <int VEC>
__global__ void __launch_bounds__(256) relayout_kernel(const __grid_constant__ RelayoutParams p) {
  const int tensor = blockIdx.y;
  const char* __restrict__ src = p.src[tensor];
  char* __restrict__ dst = p.dst[tensor];
  const int lane = threadIdx.x & 31;
  const long long total = p.row0[p.R];
  const long long step = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long HD = static_cast<long long>(p.H) * p.D;
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < total; row += step) {
    int lo = 0, hi = p.R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.row0[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int Sr = p.S_r[r];
    const long long rr = row - p.row0[r];
    const int b = static_cast<int>(rr / Sr);
    const int l = static_cast<int>(rr - static_cast<long long>(b) * Sr);
    long long seq_elem;
    if (p.seq_mode == 0) {
      const int base = r * p.U;
      int a = 0, z = p.U - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (p.c_off[base + mid] <= l) a = mid; else z = mid - 1;
      }
      const int c = base + a;
      seq_elem = p.c_base[c] + (static_cast<long long>(b) * p.c_len[c] + (l - p.c_off[c])) * HD;
    } else {
      const long long pos = l < p.p_len0[r]
                                ? p.p_start0[r] + static_cast<long long>(l) * p.p_stride[r]
                                : p.p_start1[r] + static_cast<long long>(l - p.p_len0[r]) * p.p_stride[r];
      seq_elem = (static_cast<long long>(b) * p.S + pos) * HD;
    }
    for (int g = 0; g < p.U; ++g) {
      const long long hg = static_cast<long long>(p.h[g]) * p.D;
      const long long head_elem = p.hbase[r * p.U + g] + (static_cast<long long>(b) * Sr + l) * hg;
      const long long seq_g = seq_elem + static_cast<long long>(p.hoff[g]) * p.D;
      const int nvec = static_cast<int>(hg * p.elem / VEC);
      const long long s_off = (p.dir == 0 ? seq_g : head_elem) * p.elem;
      const long long d_off = (p.dir == 0 ? head_elem : seq_g) * p.elem;
      copy_block<VEC>(dst + d_off, src + s_off, nvec, lane);
    }
  }
}

// Small rows (fewer than 32 vectors, e.g. an LSE row of H floats): one thread per token row, which
// places the row once and copies its vectors with all loads issued before the stores.
template <int VEC>
__global__ void __launch_bounds__(256) relayout_small_kernel(const __grid_constant__ RelayoutParams p) {
  using T = typename Vec<VEC>::T;
  constexpr int kBatch = 8;
  const char* __restrict__ src = p.src[blockIdx.y];
  char* __restrict__ dst = p.dst[blockIdx.y];
  const long long total = p.row0[p.R];
  const long long HD = static_cast<long long>(p.H) * p.D;
  for (long long row = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; row < total;
       row += static_cast<long long>(gridDim.x) * blockDim.x) {
    int lo = 0, hi = p.R - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.row0[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int Sr = p.S_r[r];
    const long long rr = row - p.row0[r];
    const int b = static_cast<int>(rr / Sr);
    const int l = static_cast<int>(rr - static_cast<long long>(b) * Sr);
    long long seq_elem;
    if (p.seq_mode == 0) {
      const int base = r * p.U;
      int a = 0, z = p.U - 1;
      while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (p.c_off[base + mid] <= l) a = mid; else z = mid - 1;
      }
      const int c = base + a;
      seq_elem = p.c_base[c] + (static_cast<long long>(b) * p.c_len[c] + (l - p.c_off[c])) * HD;
    } else {
      const long long pos = l < p.p_len0[r]
                                ? p.p_start0[r] + static_cast<long long>(l) * p.p_stride[r]
                                : p.p_start1[r] + static_cast<long long>(l - p.p_len0[r]) * p.p_stride[r];
      seq_elem = (static_cast<long long>(b) * p.S + pos) * HD;
    }
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
  if (nv < 32) {
    long long blocks = (total + 255) / 256;
    if (blocks > 152LL * 16) blocks = 152LL * 16;
    dim3 grid(static_cast<unsigned>(blocks), p.n_tensors);
    switch (g) {
      case 16: relayout_small_kernel<16><<<grid, 256, 0, stream>>>(p); break;
      case 8: relayout_small_kernel<8><<<grid, 256, 0, stream>>>(p); break;
      case 4: relayout_small_kernel<4><<<grid, 256, 0, stream>>>(p); break;
      default: relayout_small_kernel<2><<<grid, 256, 0, stream>>>(p); break;
    }
    return check_launch("relayout kernel");
  }
  const int warps = 8;
  long long blocks = (total + warps - 1) / warps;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  dim3 grid(static_cast<unsigned>(blocks), p.n_tensors);
  switch (g) {
    case 16: relayout_kernel<16><<<grid, warps * 32, 0, stream>>>(p); break;
    case 8: relayout_kernel<8><<<grid, warps * 32, 0, stream>>>(p); break;
    case 4: relayout_kernel<4><<<grid, warps * 32, 0, stream>>>(p); break;
    default: relayout_kernel<2><<<grid, warps * 32, 0, stream>>>(p); break;
  }
  return check_launch("relayout kernel");
}

}  // namespace usp
