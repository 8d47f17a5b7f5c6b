// LSE merge of ring partials ([USP] TemplatedRingAttention forward: the fp32 sigmoid /
// log-sigmoid combine of (prev_out, prev_lse) with (out, lse)).  All partials of one
// (row, head) vector are combined in one pass with the equivalent max-shifted weights,
//   m = max_k lse_k,  w_k = 2^((lse_k - m) log2 e),  out = sum w_k out_k / sum w_k,
//   lse = m + ln(sum w_k),
// which is exact in real arithmetic and equal to applying the pairwise form in ring order.
// Partials with lse = -inf saw no key: they get weight 0 and their out is never read.
//
// HBM-bound: each thread owns one float4 of a D-vector, so a warp reads 512 contiguous bytes of
// each partial for D = 128 and the LSE loads of a vector are warp-uniform broadcasts.
#include "internal.h"
#include "ptx.cuh"

namespace usp {
namespace {

constexpr int kMaxParts = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <bool OUT_BF16>
__global__ void __launch_bounds__(256) lse_merge_kernel(int n_parts, const float* __restrict__ o_parts,
                                                        long long o_stride,
                                                        const float* __restrict__ lse_parts,
                                                        long long lse_stride, long long n_vec,
                                                        int D, void* __restrict__ o_out,
                                                        float* __restrict__ lse_out) {
  const int qpv = D >> 2;  // float4 per vector
  const long long total = n_vec * qpv;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long vec = i / qpv;
    const int q = static_cast<int>(i - vec * qpv);
    float l[kMaxParts];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMaxParts; ++k) {
      if (k < n_parts) {
        l[k] = __ldg(lse_parts + k * lse_stride + vec);
        m = fmaxf(m, l[k]);
      }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (m != -INFINITY) {
      float den = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxParts; ++k) {
        if (k < n_parts && l[k] != -INFINITY) {
          const float w = ex2_approx((l[k] - m) * kLog2e);
          const float4 o = __ldcs(reinterpret_cast<const float4*>(o_parts + k * o_stride + vec * D) + q);
          den += w;
          acc.x = fmaf(w, o.x, acc.x);
          acc.y = fmaf(w, o.y, acc.y);
          acc.z = fmaf(w, o.z, acc.z);
          acc.w = fmaf(w, o.w, acc.w);
        }
      }
      const float inv = 1.0f / den;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      lse = m + lg2_approx(den) * kLn2;
    }
    if (OUT_BF16) {
      uint2 packed = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
      reinterpret_cast<uint2*>(static_cast<char*>(o_out) + (vec * D) * 2)[q] = packed;
    } else {
      reinterpret_cast<float4*>(static_cast<float*>(o_out) + vec * D)[q] = acc;
    }
    if (q == 0 && lse_out) lse_out[vec] = lse;
  }
}

}  // namespace

usp_status_t launch_lse_merge(int n_parts, const float* o_parts, int64_t o_part_stride,
                              const float* lse_parts, int64_t lse_part_stride, int64_t n_vec,
                              int D, void* o_out, bool out_bf16, float* lse_out,
                              cudaStream_t stream) {
  if (n_vec == 0) return USP_OK;
  const long long total = n_vec * (D / 4);
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (out_bf16)
    lse_merge_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        n_parts, o_parts, o_part_stride, lse_parts, lse_part_stride, n_vec, D, o_out, lse_out);
  else
    lse_merge_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        n_parts, o_parts, o_part_stride, lse_parts, lse_part_stride, n_vec, D, o_out, lse_out);
  return check_launch("lse merge kernel");
}

}  // namespace usp
