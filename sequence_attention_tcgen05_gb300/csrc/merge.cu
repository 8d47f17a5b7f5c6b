// LSE merge of ring partials ([USP] TemplatedRingAttention forward: the fp32 sigmoid /
// log-sigmoid combine of (prev_out, prev_lse) with (out, lse)).  All partials of one
// (row, head) vector are combined in one pass with the equivalent max-shifted weights,
//   m = max_k lse_k,  w_k = 2^((lse_k - m) log2 e),  out = sum w_k out_k / sum w_k,
//   lse = m + ln(sum w_k),
// which is exact in real arithmetic and equal to applying the pairwise form in ring order.
// Partials with lse = -inf saw no key: they get weight 0 and their out is never used.  The
// public merge loads each partial's out together with its LSE (one memory latency per batch);
// the rows variant of the causal path loads an out only once its LSE shows a visible key.
//
// HBM-bound: each thread owns float4 slots of D-vectors (a warp reads 512 contiguous bytes of each
// partial for D = 128; the LSE loads of a vector are warp-uniform broadcasts).  The partial count
// is a template parameter so that all loads of an iteration are issued before any is used.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace usp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// An LSE value of a partial: read by every lane that merges one of its vector's 16-byte slots, so
// the load keeps L1's default caching; a coherent load (not ld.global.nc), because the kernel may
// start while the kernel that wrote the partials is still running (see pdl_wait in ptx.cuh).
__device__ __forceinline__ float ld_lse(const float* p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// NP partials, U vectors' worth of float4 slots per thread per iteration: every LSE and partial
// load of the iteration is issued before the first is used (a partial whose LSE turns out to be
// -inf was loaded for nothing but is ignored), so U x NP independent 16-byte loads are in flight.
template <int NP, bool OUT_BF16, int U>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* __restrict__ o_parts,
                                                        long long o_stride,
                                                        const float* __restrict__ lse_parts,
                                                        long long lse_stride, long long n_vec,
                                                        int D, void* __restrict__ o_out,
                                                        float* __restrict__ lse_out) {
  pdl_launch_dependents();
  bool waited = false;  // the first iteration's indices come before the wait
  const int qpv = D >> 2;  // float4 per vector
  const long long total = n_vec * qpv;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
       base += stride * U) {
    long long vec[U];
    int q[U];
    bool valid[U];
    float l[U][NP];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = base + u * stride;
      valid[u] = i < total;
      vec[u] = valid[u] ? i / qpv : 0;
      q[u] = static_cast<int>(i - vec[u] * qpv);
    }
    if (!waited) {
      pdl_wait();
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int k = 0; k < NP; ++k)
        l[u][k] = valid[u] ? ld_lse(lse_parts + k * lse_stride + vec[u]) : -INFINITY;
    }
    float4 o[U][NP];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NP; ++k)
        if (valid[u])
          o[u][k] = __ldcs(reinterpret_cast<const float4*>(o_parts + k * o_stride + vec[u] * D) + q[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!valid[u]) continue;
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < NP; ++k) m = fmaxf(m, l[u][k]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float lse = -INFINITY;
      if (m != -INFINITY) {
        float den = 0.f;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          if (l[u][k] != -INFINITY) {
            const float w = ex2_approx((l[u][k] - m) * kLog2e);
            den += w;
            acc.x = fmaf(w, o[u][k].x, acc.x);
            acc.y = fmaf(w, o[u][k].y, acc.y);
            acc.z = fmaf(w, o[u][k].z, acc.z);
            acc.w = fmaf(w, o[u][k].w, acc.w);
          }
        }
        const float inv = 1.0f / den;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        lse = m + lg2_approx(den) * kLn2;
      }
      const long long ov = vec[u];
      if (OUT_BF16) {
        const uint2 packed = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        reinterpret_cast<uint2*>(static_cast<char*>(o_out) + (ov * D) * 2)[q[u]] = packed;
      } else {
        reinterpret_cast<float4*>(static_cast<float*>(o_out) + ov * D)[q[u]] = acc;
      }
      if (q[u] == 0 && lse_out) lse_out[ov] = lse;
    }
  }
}


// Merge with the result placed in the global layout (MergeMap): one warp per token row of one
// head-sharded block, i.e. h_u contiguous D-vectors on both sides.  The row's placement is decoded
// once; the lanes then stream the row's h_u * D / 4 float4 slots in batches of kB per lane (4 for
// up to 2 partials, 2 for up to 4, else 1, so that the NP x kB float4 loads a lane keeps in flight
// fit a register budget that leaves several blocks per SM), issuing the partials' loads of a batch
// before combining them.  Without a causal mask (ALL_SEEN) every partial slot holds a result, so a
// partial's loads go out together with its LSE load; otherwise a partial is loaded only once its
// LSE shows that its rows saw a key.
template <int NP, bool OUT_BF16, bool ALL_SEEN>
__global__ void __launch_bounds__(256) lse_merge_rows_kernel(const float* __restrict__ o_parts,
                                                             long long o_stride,
                                                             const float* __restrict__ lse_parts,
                                                             long long lse_stride, int D,
                                                             void* __restrict__ o_out,
                                                             float* __restrict__ lse_out,
                                                             const __grid_constant__ MergeMap m) {
  constexpr int kB = NP <= 2 ? 4 : (NP <= 4 ? 2 : 1);  // float4 slots per lane per batch
  pdl_launch_dependents();
  bool waited = false;  // the first row's placement comes from the parameters before the wait
  const int lane = threadIdx.x & 31;
  const long long total = m.row0[m.n_blocks];
  const long long step = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int qpv = D >> 2;
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < total; row += step) {
    int lo = 0, hi = m.n_blocks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (m.row0[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const long long rr = row - m.row0[lo];
    const int Sr = m.S_r[lo];
    const long long b = rr / Sr;
    const int l = static_cast<int>(rr - b * Sr);
    const long long pos = l < m.p_len0[lo] ? m.p_start0[lo] + static_cast<long long>(l) * m.p_stride[lo]
                                           : m.p_start1[lo] + static_cast<long long>(l - m.p_len0[lo]) * m.p_stride[lo];
    const int hh = m.h[lo];
    const long long src_vec = m.vec0[lo] + rr * hh;          // W vector of (row, head 0)
    const long long dst_vec = (b * m.S + pos) * m.H + m.hoff[lo];
    const int nf4 = hh * qpv;
    if (!waited) {  // warp-uniform
      pdl_wait();
      waited = true;
    }
    for (int f0 = 0; f0 < nf4; f0 += 32 * kB) {
      float l_[kB][NP];
      float4 o_[kB][NP];
      int head[kB], q[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const int f = f0 + i * 32 + lane;
        head[i] = f / qpv;
        q[i] = f - head[i] * qpv;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          l_[i][k] = f < nf4 ? ld_lse(lse_parts + k * lse_stride + src_vec + head[i]) : -INFINITY;
          if (ALL_SEEN && f < nf4)  // every slot was written: load it with its LSE, not after
            o_[i][k] = __ldcs(reinterpret_cast<const float4*>(o_parts + k * o_stride +
                                                              (src_vec + head[i]) * D) + q[i]);
        }
      }
      if (!ALL_SEEN) {
#pragma unroll
        for (int i = 0; i < kB; ++i)
#pragma unroll
          for (int k = 0; k < NP; ++k)
            if (l_[i][k] != -INFINITY)
              o_[i][k] = __ldcs(reinterpret_cast<const float4*>(o_parts + k * o_stride +
                                                                (src_vec + head[i]) * D) + q[i]);
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (f0 + i * 32 + lane >= nf4) continue;
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < NP; ++k) mx = fmaxf(mx, l_[i][k]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse = -INFINITY;
        if (mx != -INFINITY) {
          float den = 0.f;
#pragma unroll
          for (int k = 0; k < NP; ++k) {
            if (l_[i][k] != -INFINITY) {
              const float w = ex2_approx((l_[i][k] - mx) * kLog2e);
              den += w;
              acc.x = fmaf(w, o_[i][k].x, acc.x);
              acc.y = fmaf(w, o_[i][k].y, acc.y);
              acc.z = fmaf(w, o_[i][k].z, acc.z);
              acc.w = fmaf(w, o_[i][k].w, acc.w);
            }
          }
          const float inv = 1.0f / den;
          acc.x *= inv;
          acc.y *= inv;
          acc.z *= inv;
          acc.w *= inv;
          lse = mx + lg2_approx(den) * kLn2;
        }
        const long long ov = dst_vec + head[i];
        if (OUT_BF16) {
          const uint2 packed = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
          reinterpret_cast<uint2*>(static_cast<char*>(o_out) + (ov * D) * 2)[q[i]] = packed;
        } else {
          reinterpret_cast<float4*>(static_cast<float*>(o_out) + ov * D)[q[i]] = acc;
        }
        if (q[i] == 0 && lse_out) lse_out[ov] = lse;
      }
    }
  }
}

template <int NP>
cudaError_t launch_np(bool out_bf16, const MergeMap* map, cudaStream_t stream, const float* o_parts,
               long long o_stride, const float* lse_parts, long long lse_stride, long long n_vec,
               int D, void* o_out, float* lse_out) {
  constexpr int U = NP <= 4 ? 2 : 1;  // 2: 48 registers, 5 CTAs per SM (4 measured slower: 72, 3)
  if (map) {
    long long rb = (map->row0[map->n_blocks] + 7) / 8;
    const long long cap = static_cast<long long>(sm_count()) * 32;
    if (rb > cap) rb = cap;
    const unsigned nb = static_cast<unsigned>(std::max(1LL, rb));
    auto go = [&](auto kern) {
      return launch_pdl(kern, dim3(nb), dim3(256), 0, stream, o_parts, o_stride, lse_parts,
                        lse_stride, D, o_out, lse_out, *map);
    };
    if (map->all_seen)
      return out_bf16 ? go(lse_merge_rows_kernel<NP, true, true>) : go(lse_merge_rows_kernel<NP, false, true>);
    return out_bf16 ? go(lse_merge_rows_kernel<NP, true, false>) : go(lse_merge_rows_kernel<NP, false, false>);
  }
  // persistent grid: the CTAs that fit on the GPU at once (each thread then takes an equal share of
  // the float4 slots, U at a time), never more threads than slots need
  auto go = [&](auto kern) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    const long long slots = n_vec * (D / 4);
    const long long need = (slots + 256LL * U - 1) / (256LL * U);
    const long long ctas = std::max(1LL, std::min<long long>(static_cast<long long>(per_sm) * sm_count(), need));
    return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(256), 0, stream, o_parts,
                      o_stride, lse_parts, lse_stride, n_vec, D, o_out, lse_out);
  };
  return out_bf16 ? go(lse_merge_kernel<NP, true, U>) : go(lse_merge_kernel<NP, false, U>);
}

}  // namespace

usp_status_t launch_lse_merge(int n_parts, const float* o_parts, int64_t o_part_stride,
                              const float* lse_parts, int64_t lse_part_stride, int64_t n_vec,
                              int D, void* o_out, bool out_bf16, float* lse_out,
                              const MergeMap* map, cudaStream_t stream) {
  if (n_vec == 0) return USP_OK;
  cudaError_t e = cudaSuccess;
#define USP_MERGE_CASE(N)                                                                        \
  case N:                                                                                        \
    e = launch_np<N>(out_bf16, map, stream, o_parts, o_part_stride, lse_parts, lse_part_stride,   \
                     n_vec, D, o_out, lse_out);                                                  \
    break;
  switch (n_parts) {
    USP_MERGE_CASE(1) USP_MERGE_CASE(2) USP_MERGE_CASE(3) USP_MERGE_CASE(4) USP_MERGE_CASE(5)
    USP_MERGE_CASE(6) USP_MERGE_CASE(7) USP_MERGE_CASE(8) USP_MERGE_CASE(9) USP_MERGE_CASE(10)
    USP_MERGE_CASE(11) USP_MERGE_CASE(12) USP_MERGE_CASE(13) USP_MERGE_CASE(14)
    USP_MERGE_CASE(15) USP_MERGE_CASE(16)
    default:
      return fail(USP_ERR_INVALID_ARG, "n_parts %d outside [1, 16]", n_parts);
  }
#undef USP_MERGE_CASE
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "lse merge kernel: %s", cudaGetErrorString(e));
  return check_launch("lse merge kernel");
}

}  // namespace usp
