// Partial attention on the 5th-generation tensor cores: for every (chunk pair, batch, head,
// 256-row query block) work unit, O = softmax(scale Q K^T + mask) V and its natural-log LSE
// ([USP] the backend's (out, lse) for one ring step; [CP] Ring Attention).
//
// One persistent CTA per SM, five warpgroups (640 threads):
//   WG0  warp 0: TMA producer — the unit's two 128-row Q tiles, then K and V tiles into a
//                STAGES-deep ring (K and V of a key tile serve both query tiles).
//        warp 1: MMA issuer (one thread) and TMEM owner.  Per key tile j, in this order:
//                  S_a = Q_a K_j^T,  O_b += P_b(j-1) V_{j-1},  S_b = Q_b K_j^T,  O_a += P_a(j) V_j
//                (SS MMA M=128 N=128 for the scores; TS MMA with P read from TMEM for P V), so the
//                softmax of each query tile overlaps a score MMA and a P V MMA of the other tile.
//        warps 2-3 idle.  The warpgroup gives registers away (setmaxnreg) to the softmax groups.
//   WG1..WG4  softmax of query tile x = (wg-1)/2, key columns h*64..h*64+63 with h = (wg-1)%2:
//                thread = query row = TMEM lane.  One 64-column tcgen05.ld of its half of the S row,
//                masking on boundary tiles, partial row max, exchanged with the other half through
//                shared memory (one mbarrier per tile), then 2^(s * scale log2e - m) with packed
//                fp32x2 fused multiply-adds and MUFU ex2, bf16 P written over the first 32 columns
//                of its own S half, partial row sum in registers.  The running max m is raised only
//                when a tile's max exceeds it by more than 8 (log2 units); then each half rescales
//                its half of O in TMEM.  Otherwise the stale max stays, which bounds P by 2^8 and
//                is exact after the final division by the row sum.  Epilogue: the two partial
//                row sums are combined, each half stores its half of O / l (fp32 or bf16) and the
//                first half the lse = (m + log2 l) ln 2.
// Splitting each tile's softmax over two warpgroups halves the softmax term of the chain
// S_x(j) -> softmax -> O_x += P V -> S_x(j+1), which sets the kernel's period per key tile.
// TMEM (512 columns): S_a [0,128) S_b [128,256) O_a [256,256+D) O_b [256+D,256+2D); P_x columns
// [0,32) and [64,96) of S_x.  MMAs issued by one thread execute in issue order, so a completed
// S_x(j) implies P V of tile j-1 of the same query tile has completed: S_x may then be read, P_x
// rewritten and O_x rescaled without another wait.
//
// Shared memory tiles are the canonical 128-byte-swizzled layouts TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B: rows of 64 bf16 (128 B), 8-row atoms of 1024 B.  Q and K are
// K-major operands (head dim contiguous); V is the MN-major B operand of P V.
//
// Every mbarrier wait is bounded (see ptx.cuh); on a timeout all roles stop, drain their
// in-flight copies and MMAs, free TMEM and exit, and the status word records the error.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace usp {
namespace {

constexpr float kTau = 8.0f;  // lazy-rescale threshold, log2 units
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = 640;
constexpr int kSoftmaxThreads = 256;  // the two warpgroups of one query tile
// Register split: 640 threads x 96 at launch = 61440 >= 128 x 56 (WG0) + 512 x 104 (softmax).
constexpr uint32_t kRegsLaunch = 96;
constexpr uint32_t kRegsWG0 = 56;
constexpr uint32_t kRegsSoftmax = 104;
static_assert(128 * kRegsWG0 + 512 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");

template <int D, int STAGES>
struct Layout {
  static constexpr int kQTile = kAttnBM * D * 2;  // one 128-row Q tile
  static constexpr int kKBytes = kAttnBN * D * 2;
  static constexpr int kVBytes = kAttnBN * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kQTile;
  static constexpr int kV = kK + STAGES * kKBytes;
  static constexpr int kBar = kV + STAGES * kVBytes;
  // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done[2],
  // o_empty[2], xch[2], xl[2], mma_done
  static constexpr int kNumBars = 2 + 2 * STAGES + 13;
  static constexpr int kXmax = kBar + kNumBars * 8;        // float [2 parity][2 tile][2 half][128]
  static constexpr int kXsum = kXmax + 2 * 2 * 2 * 128 * 4;  // float [2 tile][2 half][128]
  static constexpr int kTmemSlot = kXsum + 2 * 2 * 128 * 4;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kEnd = kAbort + 4;
  static constexpr int kAlloc = kEnd + 1024;  // slack to align the base to 1024 B
};

struct Unit {
  const AttnSeg* seg;
  int b, h, q0, n_kv;
  int qv[2];  // valid rows of tiles a and b
};

__device__ __forceinline__ Unit decode_unit(const AttnParams& p, int unit) {
  int lo = 0, hi = p.n_segs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.segs[mid].unit0 <= unit) lo = mid; else hi = mid - 1;
  }
  const AttnSeg& s = p.segs[lo];
  const int local = unit - s.unit0;
  const int qi = local % s.n_qblk;
  const int hb = local / s.n_qblk;
  Unit u;
  u.seg = &s;
  const int qb = s.rev ? s.n_qblk - 1 - qi : qi;
  u.h = hb % s.n_heads;
  u.b = hb / s.n_heads;
  u.q0 = qb * kAttnUnitRows;
  u.qv[0] = max(0, min(kAttnBM, s.q_len - u.q0));
  u.qv[1] = max(0, min(kAttnBM, s.q_len - u.q0 - kAttnBM));
  const int last_row = u.q0 + u.qv[0] + u.qv[1] - 1;
  int max_c = s.kv_len - 1;
  if (s.diag != kNoDiag) max_c = min(max_c, last_row + s.diag);
  u.n_kv = max_c < 0 ? 0 : max_c / kAttnBN + 1;
  return u;
}

// 2^(s * c + nb) for the 64 columns of one half row: bf16 P written as 32 packed columns at t_p
// (two 16-column stores); returns the fp32 sum.
__device__ __forceinline__ float exp_half(const uint32_t (&r)[64], uint64_t c2, float nb,
                                          uint32_t t_p) {
  const uint64_t nb2 = f2_pack(nb, nb);
  uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
  for (int chunk = 0; chunk < 2; ++chunk) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = chunk * 32 + 2 * i;
      const uint64_t a2 =
          f2_fma(f2_pack(__uint_as_float(r[col]), __uint_as_float(r[col + 1])), c2, nb2);
      float e0, e1;
      f2_unpack(a2, e0, e1);
      const float p0 = ex2_approx(e0);
      const float p1 = ex2_approx(e1);
      sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
      pk[i] = pack_bf16x2(p0, p1);
    }
    tmem_st16(t_p + chunk * 16, pk);
  }
  float s0, s1, s2, s3;
  f2_unpack(sum2[0], s0, s1);
  f2_unpack(sum2[1], s2, s3);
  return (s0 + s1) + (s2 + s3);
}

__device__ __forceinline__ float half_max(const uint32_t (&r)[64]) {
  float m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m8[i] = __uint_as_float(r[i]);
#pragma unroll
  for (int i = 8; i < 64; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      m8[k] = fmax3(m8[k], __uint_as_float(r[i + 2 * k]), __uint_as_float(r[i + 2 * k + 1]));
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

template <int D, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;  // K and V of a stage, one transaction count
  uint64_t* kv_empty = kv_full + STAGES;
  uint64_t* s_full = kv_empty + STAGES;  // [2]: query tile a, b
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_empty = pv_done + 2;
  uint64_t* xch = o_empty + 2;      // [2]: partial row max exchanged (per key tile)
  uint64_t* xl = xch + 2;           // [2]: partial row sum exchanged (per unit)
  uint64_t* mma_done = xl + 2;
  float* xmax = reinterpret_cast<float*>(sm + L::kXmax);
  float* xsum = reinterpret_cast<float*>(sm + L::kXsum);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  const uint64_t budget = p.budget_ns;
  const uint64_t drain_budget = budget < 200000000ull ? budget : 200000000ull;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxThreads);
      mbar_init(&pv_done[i], 1);
      mbar_init(&o_empty[i], kSoftmaxThreads);
      mbar_init(&xch[i], kSoftmaxThreads);
      mbar_init(&xl[i], kSoftmaxThreads);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (wg == 0) {
    regs_dec<kRegsWG0>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      uint32_t stage = 0, phase = 0, q_iter = 0;
      uint32_t fills[STAGES];
      for (int s = 0; s < STAGES; ++s) fills[s] = 0;
      for (int unit = blockIdx.x; unit < p.n_units; unit += gridDim.x) {
        const Unit u = decode_unit(p, unit);
        if (u.n_kv == 0) continue;
        const AttnSeg& s = *u.seg;
        if (q_iter > 0 && !mbar_wait(q_empty, (q_iter - 1) & 1, abort_flag, p.status, budget)) break;
        mbar_arrive_expect_tx(q_full, 2 * L::kQTile);
        const int qrow = s.q_row0 + u.q0;
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(sm + L::kQ + x * L::kQTile + blk * kAttnBM * 128, &p.maps[s.q_map], blk * 64,
                        u.h, qrow + x * kAttnBM, u.b, q_full);
        ++q_iter;
        const int kvrow = s.kv_row0;
        bool ok = true;
        for (int j = 0; j < u.n_kv; ++j) {
          if (!mbar_wait(&kv_empty[stage], phase ^ 1, abort_flag, p.status, budget)) { ok = false; break; }
          mbar_arrive_expect_tx(&kv_full[stage], L::kKBytes + L::kVBytes);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(sm + L::kK + stage * L::kKBytes + blk * kAttnBN * 128, &p.maps[s.k_map],
                        blk * 64, u.h, kvrow + j * kAttnBN, u.b, &kv_full[stage]);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(sm + L::kV + stage * L::kVBytes + blk * kAttnBN * 128, &p.maps[s.v_map],
                        blk * 64, u.h, kvrow + j * kAttnBN, u.b, &kv_full[stage]);
          ++fills[stage];
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      for (int s = 0; s < STAGES; ++s) {
        if (fills[s]) {
          mbar_drain(&kv_full[s], (fills[s] - 1) & 1, drain_budget);
        }
      }
      if (q_iter) mbar_drain(q_full, (q_iter - 1) & 1, drain_budget);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kAttnBM, kAttnBN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kAttnBM, D, 1);
      const uint32_t q_base = smem_u32(sm + L::kQ);
      const uint32_t k_base = smem_u32(sm + L::kK);
      const uint32_t v_base = smem_u32(sm + L::kV);
      static_assert(L::kAlloc < (1 << 18), "descriptor start addresses are 14-bit fields of addr >> 4");
      uint32_t stage = 0, phase = 0, q_iter = 0, units_done = 0;
      uint32_t gp[2] = {0, 0};  // P V count per query tile
      bool ok = true;
      // Shared-memory descriptors (128-byte swizzle, SBO 1024 B, version 1): constant high word;
      // low word = start address >> 4 | LBO field (1 for the K-major Q and K, 16384 B for V).
      constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
      const uint32_t q_lo = (q_base >> 4) | (1u << 16);
      const uint32_t k_lo = (k_base >> 4) | (1u << 16);
      const uint32_t v_lo = (v_base >> 4) | ((static_cast<uint32_t>(kAttnBN * 128) >> 4) << 16);
      auto qk = [&](int x, uint32_t st) {
        const uint32_t a = q_lo + x * (L::kQTile >> 4);
        const uint32_t b = k_lo + st * (L::kKBytes >> 4);
        if (D == 128) mma_group_qk8(tmem + x * 128, a, b, kDescHi, idesc_qk);
        else mma_group_qk4(tmem + x * 128, a, b, kDescHi, idesc_qk);
        mma_commit(&s_full[x]);
      };
      // O_x += P_x V(st); `first` = first key tile of the unit (overwrites O_x), `last` = its last
      // one (pv_done tells the epilogue that O_x is final).  P_x: keys 0-63 packed in S_x columns
      // [0,32), keys 64-127 in [64,96).  V(st) arrived with K(st): the S MMA of this stage waited.
      auto pv = [&](int x, uint32_t st, bool first, bool last) -> bool {
        if (!mbar_wait(&p_full[x], gp[x] & 1, abort_flag, p.status, budget)) return false;
        if (first && units_done > 0 &&
            !mbar_wait(&o_empty[x], (units_done - 1) & 1, abort_flag, p.status, budget))
          return false;
        tc_fence_after();
        mma_group_pv(tmem + 256 + x * D, tmem + x * 128, v_lo + st * (L::kVBytes >> 4), kDescHi,
                     idesc_pv, first ? 0u : 1u);
        if (last) mma_commit(&pv_done[x]);
        ++gp[x];
        return true;
      };
      for (int unit = blockIdx.x; unit < p.n_units && ok; unit += gridDim.x) {
        const Unit u = decode_unit(p, unit);
        if (u.n_kv == 0) continue;
        // Q and K/V come from TMA (async proxy, like the MMAs): the barrier waits order them, no
        // tcgen05 fence is needed; P comes from tcgen05.st of other threads (fence in pv()).
        if (!mbar_wait(q_full, q_iter & 1, abort_flag, p.status, budget)) break;
        ++q_iter;
        uint32_t prev_stage = 0;
        for (int j = 0; j < u.n_kv; ++j) {
          if (!mbar_wait(&kv_full[stage], phase, abort_flag, p.status, budget)) { ok = false; break; }
          qk(0, stage);
          if (j > 0) {
            if (!pv(1, prev_stage, j == 1, false)) { ok = false; break; }
            mma_commit(&kv_empty[prev_stage]);
          }
          qk(1, stage);
          if (j == u.n_kv - 1) mma_commit(q_empty);
          if (!pv(0, stage, j == 0, j == u.n_kv - 1)) { ok = false; break; }
          prev_stage = stage;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (!pv(1, prev_stage, u.n_kv == 1, true)) { ok = false; break; }
        mma_commit(&kv_empty[prev_stage]);
        ++units_done;
      }
      // drain: all issued MMAs complete before TMEM is freed
      mma_commit(mma_done);
      mbar_drain(mma_done, 0, drain_budget);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    regs_inc<kRegsSoftmax>();
    const int x = (wg - 1) >> 1;   // query tile a (0) or b (1)
    const int hf = (wg - 1) & 1;   // key columns [hf*64, hf*64+64) of each tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t t_s = t_lane + x * 128 + hf * 64;           // this half of S_x, and its P
    const uint32_t t_o = t_lane + 256 + x * D + hf * (D / 2);  // this half of O_x
    const float c = p.scale_log2;  // > 0 (checked on the host)
    const uint64_t c2 = f2_pack(c, c);
    uint32_t g = 0, units = 0;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = mbar_wait(bar, parity, abort_flag, p.status, budget);
      return __all_sync(0xffffffffu, r);
    };
    for (int unit = blockIdx.x; unit < p.n_units && ok; unit += gridDim.x) {
      const Unit u = decode_unit(p, unit);
      const AttnSeg& s = *u.seg;
      const int q0 = u.q0 + x * kAttnBM;  // first local row of this query tile
      const bool row_valid = row < u.qv[x];
      const int ol = s.o_row0 + q0 + row;  // output-side local row
      const long long opos = ol < s.o_len0
                                 ? static_cast<long long>(s.o_start0) + static_cast<long long>(ol) * s.o_stride
                                 : static_cast<long long>(s.o_start1) + static_cast<long long>(ol - s.o_len0) * s.o_stride;
      const long long orow = static_cast<long long>(u.b) * s.o_bstride + opos;
      const long long o_elem = (orow * s.o_heads + u.h) * D + hf * (D / 2);
      if (u.n_kv == 0) {
        if (row_valid) {
          if (p.o_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(s.o) + o_elem);
            for (int i = 0; i < D / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(s.o) + o_elem);
            for (int i = 0; i < D / 8; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          if (hf == 0 && s.lse) s.lse[orow * s.o_heads + u.h] = -INFINITY;
        }
        continue;
      }
      const int lim = s.diag == kNoDiag ? INT_MAX : q0 + row + s.diag;  // visible key c <= lim
      float m_ref = -INFINITY;  // running max of scale*log2e*s, raised lazily (same in both halves)
      float l = 0.f;            // row sum over this half's columns
      for (int j = 0; j < u.n_kv; ++j, ++g) {
        if (!wait_all(&s_full[x], g & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64(t_s, r);
        tmem_wait_ld();
        const int c0 = j * kAttnBN + hf * 64;  // local key index of r[0]
        const bool need_mask = (c0 + 64 > s.kv_len) || (s.diag != kNoDiag && c0 + 63 > q0 + s.diag);
        if (need_mask) {
          const int last = min(s.kv_len - 1, lim) - c0;  // visible columns of this half: i <= last
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > last) r[i] = 0xff800000u;  // -inf
        }
        // exchange the partial row max with the other half of the tile
        const float pm = half_max(r);
        float* xm = xmax + ((g & 1) * 4 + x * 2) * 128;
        xm[hf * 128 + row] = pm;
        mbar_arrive(&xch[x]);
        if (!wait_all(&xch[x], g & 1)) { ok = false; break; }
        const float mx = fmaxf(pm, xm[(1 - hf) * 128 + row]) * c;
        float alpha = 1.f;
        bool resc = false;
        if (mx > m_ref + kTau) {
          if (m_ref != -INFINITY) {
            alpha = ex2_approx(m_ref - mx);
            resc = true;
          }
          m_ref = mx;
        }
        const float nb = (m_ref == -INFINITY) ? 0.f : -m_ref;
        const float sum = exp_half(r, c2, nb, t_s);
        l = l * alpha + sum;
        if (__any_sync(0xffffffffu, resc)) {
          // S_x(j) complete => P V of tile j-1 complete: O_x is stable
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t w[32];
            tmem_ld32(t_o + cc * 32, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
            tmem_st32(t_o + cc * 32, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
      }
      if (!ok) break;
      // epilogue: combine the two partial row sums, then each half stores its half of O
      float* xs = xsum + x * 2 * 128;
      xs[hf * 128 + row] = l;
      mbar_arrive(&xl[x]);
      if (!wait_all(&xl[x], units & 1)) { ok = false; break; }
      const float lt = l + xs[(1 - hf) * 128 + row];
      if (!wait_all(&pv_done[x], units & 1)) { ok = false; break; }  // committed once per unit
      ++units;
      tc_fence_after();
      const float inv_l = lt > 0.f ? 1.0f / lt : 0.f;
      const float lse = lt > 0.f ? (m_ref + lg2_approx(lt)) * kLn2 : -INFINITY;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t o[32];
        tmem_ld32(t_o + cc * 32, o);
        tmem_wait_ld();
        if (cc == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(&o_empty[x]);
        }
        if (row_valid) {
          if (p.o_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(s.o) + o_elem + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(
                  pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l),
                  pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l));
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(s.o) + o_elem + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i + 0]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                   __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
          }
        }
      }
      if (row_valid && hf == 0 && s.lse) s.lse[orow * s.o_heads + u.h] = lse;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int STAGES>
usp_status_t launch_one(const AttnParams& p, cudaStream_t stream) {
  using L = Layout<D, STAGES>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  auto kern = attn_fwd_kernel<D, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::max(1, std::min(p.n_units, sms));
  kern<<<grid, kThreads, L::kAlloc, stream>>>(p);
  return check_launch("attention kernel");
}

}  // namespace

usp_status_t make_qkv_map(CUtensorMap* map, const void* base, int n_heads, int D, int64_t rows,
                          int B, int64_t row_stride, int64_t batch_stride) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<EncodeFn>(fn);
  }();
  if (!encode) return fail(USP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(n_heads),
                              static_cast<cuuint64_t>(std::max<int64_t>(rows, 1)),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(row_stride) * 2,
                                 static_cast<cuuint64_t>(std::max<int64_t>(batch_stride, row_stride)) * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kAttnBM), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(USP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return USP_OK;
}

usp_status_t launch_attention(AttnParams& p, std::vector<AttnSeg>& segs, int D,
                              cudaStream_t stream) {
  if (!(p.scale_log2 > 0.f)) return fail(USP_ERR_INVALID_ARG, "the softmax scale must be positive");
  // Longest units first: sort segments by the keys a full query block visits.
  auto cost = [](const AttnSeg& s) {
    return s.diag == kNoDiag ? s.kv_len : std::min(s.kv_len, s.q_len + s.diag);
  };
  std::stable_sort(segs.begin(), segs.end(),
                   [&](const AttnSeg& a, const AttnSeg& b) { return cost(a) > cost(b); });
  size_t at = 0;
  while (at < segs.size()) {
    const size_t n = std::min<size_t>(kAttnMaxSegs, segs.size() - at);
    int units = 0, used = 0;
    for (size_t i = 0; i < n; ++i) {
      AttnSeg s = segs[at + i];
      s.n_qblk = (s.q_len + kAttnUnitRows - 1) / kAttnUnitRows;
      s.unit0 = units;
      const long long add = static_cast<long long>(s.n_qblk) * s.n_heads * p.B;
      if (add == 0) continue;
      if (units + add > INT_MAX / 2) return fail(USP_ERR_UNSUPPORTED, "too many attention work units");
      units += static_cast<int>(add);
      p.segs[used++] = s;
    }
    p.n_segs = used;
    p.n_units = units;
    if (units > 0) {
      usp_status_t st = D == 64 ? launch_one<64, 4>(p, stream) : launch_one<128, 2>(p, stream);
      if (st != USP_OK) return st;
    }
    at += n;
  }
  return USP_OK;
}

}  // namespace usp
