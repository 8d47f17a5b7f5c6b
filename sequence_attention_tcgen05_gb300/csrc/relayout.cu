// Re-layout kernels: the Ulysses all-to-alls as local permutations ([CP] Ulysses Attention;
// [UAA] arbitrary per-rank lengths), ring-chunk reordering ([YC] contiguous / zigzag / stripe)
// and their fusion.  Pure data movement, bit-exact, HBM-bound.
//
// Every (tensor, row, head group) moves one contiguous block of h_g * D elements on both sides
// (h_g * D * elem bytes: 3 KB for 12 bf16 heads of 128).  The blocks are cut into sub-blocks of
// 32 vectors (512 bytes with 16-byte vectors; the widest vector every offset allows), numbered
// tensor-major, then row, head group and position in the block.  The grid is persistent (as many
// CTAs as fit on the GPU at once) and every warp takes an equal, contiguous range of sub-blocks,
// so all warps finish together whatever the block count.  A warp issues the loads of up to kNV
// sub-blocks of one row (one vector per lane each) before their stores, so it keeps 4 KB in
// flight and places each row once.
#include <algorithm>
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

constexpr int kNV = 8;  // sub-blocks (one vector per lane each) in flight per warp

template <int VEC>
__global__ void __launch_bounds__(256) relayout_kernel(const __grid_constant__ RelayoutParams p,
                                                       long long n_sb) {
  using T = typename Vec<VEC>::T;
  const int lane = threadIdx.x & 31;
  const long long W = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  long long s = n_sb * w / W;  // this warp's sub-blocks [s, e)
  const long long e = n_sb * (w + 1) / W;
  const int sbpr = p.sb_off[p.U];  // sub-blocks per row (all groups)
  const long long rows = p.row0[p.R];
  while (s < e) {
    const long long q = s / sbpr;  // tensor * rows + row
    int j = static_cast<int>(s - q * sbpr);
    const int tensor = static_cast<int>(q / rows);
    const long long row = q - tensor * rows;
    const int nb = static_cast<int>(min(static_cast<long long>(min(kNV, sbpr - j)), e - s));
    const RowPlace x = place_row(p, row);
    const long long row_in_r = static_cast<long long>(x.b) * p.S_r[x.r] + x.l;
    int g = 0;
    while (p.sb_off[g + 1] <= j) ++g;
    T buf[kNV];
    T* dp[kNV];
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      dp[i] = nullptr;
      if (i < nb) {
        while (p.sb_off[g + 1] <= j) ++g;
        const long long hg = static_cast<long long>(p.h[g]) * p.D;
        const long long head_elem = p.hbase[x.r * p.U + g] + row_in_r * hg;
        const long long seq_g = x.seq_elem + static_cast<long long>(p.hoff[g]) * p.D;
        const int v = (j - p.sb_off[g]) * 32 + lane;
        if (v < static_cast<int>(hg * p.elem / VEC)) {
          const T* src = reinterpret_cast<const T*>(p.src[tensor] + (p.dir == 0 ? seq_g : head_elem) * p.elem);
          buf[i] = __ldcs(src + v);
          dp[i] = reinterpret_cast<T*>(p.dst[tensor] + (p.dir == 0 ? head_elem : seq_g) * p.elem) + v;
        }
        ++j;
      }
    }
#pragma unroll
    for (int i = 0; i < kNV; ++i)
      if (dp[i]) *dp[i] = buf[i];
    s += nb;
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
    switch (g) {
      case 16: relayout_small_kernel<16><<<grid, 256, 0, stream>>>(p); break;
      case 8: relayout_small_kernel<8><<<grid, 256, 0, stream>>>(p); break;
      case 4: relayout_small_kernel<4><<<grid, 256, 0, stream>>>(p); break;
      default: relayout_small_kernel<2><<<grid, 256, 0, stream>>>(p); break;
    }
    return check_launch("relayout kernel");
  }
  // sub-blocks of 32 vectors per (row, group): prefix over the groups of a row
  p.sb_off[0] = 0;
  for (int u = 0; u < p.U; ++u)
    p.sb_off[u + 1] = p.sb_off[u] + static_cast<int>((static_cast<long long>(p.h[u]) * p.D * p.elem / g + 31) / 32);
  const long long n_sb = total * p.sb_off[p.U] * p.n_tensors;
  // persistent grid: the CTAs that fit on the GPU at once, never more warps than sub-blocks
  const int threads = 256;
  auto go = [&](auto kern) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    long long ctas = std::min<long long>(static_cast<long long>(per_sm) * sms, (n_sb + 7) / 8);
    kern<<<static_cast<unsigned>(std::max(1LL, ctas)), threads, 0, stream>>>(p, n_sb);
  };
  switch (g) {
    case 16: go(relayout_kernel<16>); break;
    case 8: go(relayout_kernel<8>); break;
    case 4: go(relayout_kernel<4>); break;
    default: go(relayout_kernel<2>); break;
  }
  return check_launch("relayout kernel");
}

}  // namespace usp
