// Attention on the 5th-generation tensor cores: for every (segment, batch, head, 256-row query
// block) work unit, O = softmax(scale Q K^T + mask) V and its natural-log LSE ([USP] the backend's
// (out, lse) for one ring step; [CP] Ring Attention).  A segment's keys are one or more links
// (key ranges of K/V chunks): with one link a unit is one ring step's chunk pair and may write an
// fp32 partial; with several, the unit's online softmax runs across the K/V chunks of every ring
// step in ring order (the LSE-weighted merge done in registers) and writes the final O and LSE.
//
// Work units are numbered per unit group (one per Ulysses rank), head-major over the group's
// segments (longest first), so that CTAs running at the same time share one or two heads' K/V in
// L2.  The host picks each launch's deal of units to CTAs from a time model: a static order
// (snake or round-robin) that every role computes alone, or a dynamic one, where each CTA takes
// the next unit from a counter in global memory when it is ready for one (the DYN kernels).
//
// One persistent CTA per SM, five warpgroups (640 threads):
//   WG0  warp 0: TMA producer — the unit's two 128-row Q tiles, then K and V tiles into a
//                STAGES-deep ring (K and V of a key tile serve both query tiles).  K and V have
//                their own full and empty barriers: a K slot is released when both score MMAs of
//                its tile complete, a V slot when both P V MMAs do, so the next K load starts
//                about a period before the V load.
//        warp 1: MMA issuer and TMEM owner.  The whole warp runs the issuing loop (its state
//                stays warp-uniform); one elected lane issues each tcgen05.mma and commit.  Per
//                key tile j, in this order:
//                  S_a = Q_a K_j^T,  O_b += P_b(j-1) V_{j-1},  S_b = Q_b K_j^T,  O_a += P_a(j) V_j
//                (SS MMA M=128 N=128 for the scores; TS MMA with P read from TMEM for P V), so the
//                softmax of each query tile overlaps a score MMA and a P V MMA of the other tile.
//                The waits for V_j and K_{j+1} come just before the wait for P_a(j), the long one,
//                so that O_a += P_a(j) V_j is followed at once by S_a = Q_a K_{j+1}^T.
//        warps 2-3 idle.  The warpgroup gives registers away (setmaxnreg) to the softmax groups.
//   WG1..WG4  softmax of query tile x = (wg-1)/2 over lane half h = (wg-1)%2 of every 32-lane TMEM
//                quadrant: each thread owns two rows of the tile (quadrant lanes 16h + t/4 and that
//                + 8) and a quarter of their 128 key columns (8k + 2(t%4) + {0,1}), read with one
//                16-lane tcgen05.ld (.16x256b.x16).  Row maxima and sums combine over the four
//                threads of a row with two warp shuffles, so the two warpgroups of a tile never
//                wait for each other.  A tile that needs a mask (past a link's last key, or past
//                the causal diagonal) first gets -inf written into its hidden S columns in TMEM by
//                a small pre-pass; launches without such tiles use a kernel instantiation without
//                that code.  2^(s * scale log2e - m) with packed
//                fp32x2 fused multiply-adds and MUFU ex2; each thread's column pair becomes one
//                bf16x2 P word that a .16x128b tcgen05.st puts exactly at P column 4k + t%4, so P
//                for the tile's 128 keys is packed over S_x columns [0, 64).  Once a warp's rows
//                have a finite running max m, a tile is exponentiated against that (stale) m with
//                no max over the tile; only when a thread's partial row sum exceeds 2^16 (or is not
//                finite) does the warp take the slow path: row maxima, m raised where the tile's
//                max exceeds it by more than 8 (log2 units), its part of O rescaled in TMEM and
//                the exponentials redone.  P stays bounded by 2^16, and the stale m is exact after
//                the final division by the row sum.  Epilogue: O / l (fp32 or bf16) and
//                lse = (m + log2 l) ln 2 from the same fragments; bf16 O words are first
//                transposed across the four threads of each row (two shuffle rounds), so that
//                each thread writes whole 8-column groups as 16-byte stores.
// Without a max exchange between the warpgroups the softmax term of the chain
// S_x(j) -> softmax -> O_x += P V -> S_x(j+1), which sets the kernel's period per key tile, is
// one warpgroup's own work.
// TMEM (512 columns): S_a [0,128) S_b [128,256) O_a [256,256+D) O_b [256+D,256+2D); P_x packed in
// columns [0,64) of S_x.  MMAs issued by the one issuing lane execute in issue order, so a completed
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
#include <cstdlib>
#include <cstring>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace usp {
namespace {

constexpr float kTau = 8.0f;          // slow path: raise m by at least this much (log2 units)
constexpr float kFastSum = 65536.0f;  // fast path: a thread's partial row sum of one tile
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = 640;
constexpr int kSoftmaxThreads = 256;  // the two warpgroups of one query tile
// Register split: 640 threads x 96 at launch = 61440 >= 128 x 56 (WG0) + 512 x 104 (softmax).
constexpr uint32_t kRegsLaunch = 96;
constexpr uint32_t kRegsWG0 = 56;
constexpr uint32_t kRegsSoftmax = 104;
static_assert(128 * kRegsWG0 + 512 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
// Dynamic deal: slots of the unit queue from the producer thread to the other roles, and the
// warps that read each slot (the MMA warp and the 16 softmax warps).
constexpr int kUnitQ = 4;
constexpr int kUnitReaders = 1 + (kThreads - 128) / 32;

template <int D, int STAGES>
struct Layout {
  static constexpr int kQTile = kAttnBM * D * 2;  // one 128-row Q tile
  static constexpr int kKBytes = kAttnBN * D * 2;
  static constexpr int kVBytes = kAttnBN * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kQTile;
  static constexpr int kV = kK + STAGES * kKBytes;
  static constexpr int kBar = kV + STAGES * kVBytes;
  // q_full, q_empty, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_full[2],
  // pv_done[2], o_empty[2], mma_done
  static constexpr int kNumBars = 2 + 4 * STAGES + 9;
  // unit queue: full[kUnitQ], empty[kUnitQ] barriers, then int[kUnitQ] slots
  static constexpr int kUnitQueue = kBar + kNumBars * 8;
  static constexpr int kTmemSlot = kUnitQueue + 2 * kUnitQ * 8 + 4 * kUnitQ;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kEnd = kAbort + 4;
  static constexpr int kAlloc = kEnd + 1024;  // slack to align the base to 1024 B
};

struct Unit {
  const AttnSeg* seg;
  int b, h, q0, n_kv;
  int last_row;  // last valid segment-local query row of the unit
  int qv[2];     // valid rows of tiles a and b
};

__device__ __forceinline__ Unit decode_unit(const AttnParams& p, int unit) {
  int gl = 0, gh = p.n_groups - 1;
  while (gl < gh) {
    const int mid = (gl + gh + 1) >> 1;
    if (p.groups[mid].unit0 <= unit) gl = mid; else gh = mid - 1;
  }
  const AttnGroup& G = p.groups[gl];
  const int local = unit - G.unit0;
  const int hb = local / G.blocks;
  const int rem = deal_block(local - hb * G.blocks, G.blocks, hb, p.deal);  // over the segments
  int lo = G.seg0, hi = G.seg0 + G.n_segs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.segs[mid].qb0 <= rem) lo = mid; else hi = mid - 1;
  }
  const AttnSeg& s = p.segs[lo];
  const int qi = rem - s.qb0;
  Unit u;
  u.seg = &s;
  const int qb = s.rev ? s.n_qblk - 1 - qi : qi;
  u.h = hb % s.n_heads;
  u.b = hb / s.n_heads;
  u.q0 = qb * kAttnUnitRows;
  u.qv[0] = max(0, min(kAttnBM, s.q_len - u.q0));
  u.qv[1] = max(0, min(kAttnBM, s.q_len - u.q0 - kAttnBM));
  u.last_row = u.q0 + u.qv[0] + u.qv[1] - 1;
  int n = 0;
  for (int i = 0; i < s.n_links; ++i) n += link_tiles(p.links[s.link0 + i], u.last_row);
  u.n_kv = n;
  return u;
}

// The unit this CTA takes in round t under the launch's deal.  By default the snake order: in
// round t CTA c takes unit t*G + c for even t and t*G + G-1-c for odd t.  The host lists units
// longest first, so each CTA's total stays close to the mean (a longest-processing-time deal)
// while neighbouring CTAs still work on the same head's K/V at the same time, which keeps those
// tiles in L2.  Every role walks the same sequence.
__device__ __forceinline__ int unit_of_round(const AttnParams& p, int t) {
  return deal_unit(t, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), p.deal);
}

// Under the dynamic deal the producer thread takes each next unit from the launch's counter in
// global memory (units in their numbering order, each to the CTA that asks first) and passes it
// to the MMA warp and the softmax warps through a kUnitQ-slot queue in shared memory: `full[s]`
// completes when the producer has written slot s, `empty[s]` when every reading warp has read
// it.  A unit index >= n_units ends the walk.  Under a static deal every role computes its k-th
// unit alone.

// Shared-memory address OFF bytes into the kernel's 1024-aligned shared memory (the unit queue:
// full[kUnitQ], empty[kUnitQ] barriers, then kUnitQ int slots; or the abort flag), recomputed
// from the dynamic shared memory base where it is used so that no register holds it across a
// role's unit loop.
template <int OFF>
__device__ __forceinline__ uint32_t shared_at() {
  extern __shared__ uint8_t smem_raw[];
  return ((smem_u32(smem_raw) + 1023u) & ~1023u) + OFF;
}
__device__ __forceinline__ uint32_t uq_full(uint32_t q, int s) { return q + 8 * s; }
__device__ __forceinline__ uint32_t uq_empty(uint32_t q, int s) { return q + 8 * (kUnitQ + s); }
__device__ __forceinline__ uint32_t uq_slot(uint32_t q, int s) { return q + 16 * kUnitQ + 4 * s; }

// The producer thread's k-th unit under the dynamic deal; false if a wait gave up.
template <int OFF>
__device__ __forceinline__ bool produce_unit(const AttnParams& p, int k, volatile int* abort_flag,
                                             uint64_t budget, int& unit) {
  const uint32_t q = shared_at<OFF>();
  const int s = k & (kUnitQ - 1);
  if (k >= kUnitQ && !mbar_wait_at(uq_empty(q, s), ((k / kUnitQ) - 1) & 1, abort_flag, p.status, budget))
    return false;
  unit = static_cast<int>(atomicAdd(p.counter, 1u));
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(uq_slot(q, s)), "r"(unit) : "memory");
  mbar_arrive_at(uq_full(q, s));  // release: the slot's value is visible to whoever waits on it
  return true;
}

// Wait of the softmax warps for a queue slot, lighter than mbar_wait (their registers are all
// taken across the unit loop): the abort flag is read through its shared address, and instead
// of a clock the wait counts its polls.  The producer fills each slot well before the softmax
// warps get to it (after issuing the loads of the unit before, while the MMA warp and the
// softmax are still on that unit), and the MMA warp waits for the same slot with a timed wait
// that raises the abort flag, so the count only bounds a failure: after 2^22 polls the wait
// raises the abort flag and the timeout status itself.
__device__ __forceinline__ bool queue_wait_polls(uint32_t bar, uint32_t parity, uint32_t abort_at,
                                                 uint32_t* status) {
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_at(bar, parity)) return true;
    if ((it & 63u) == 0) {
      uint32_t aborted;
      asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(aborted) : "r"(abort_at) : "memory");
      if (aborted) return false;
      if (it == (1u << 22)) {
        asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(abort_at), "r"(1u) : "memory");
        if (status) atomicOr(status, kErrTimeout);
        return false;
      }
    }
  }
}

// A reading warp's k-th unit under the dynamic deal (every lane takes part); false if a wait
// gave up.  TIMED: the MMA warp's wait (mbar_wait); otherwise the softmax warps'
// (queue_wait_polls).
template <int OFF, int ABORT, bool TIMED>
__device__ __forceinline__ bool consume_unit(const AttnParams& p, int k, int lane, volatile int* abort_flag,
                                             uint64_t budget, int& unit) {
  const uint32_t q = shared_at<OFF>();
  const int s = k & (kUnitQ - 1);
  const bool ready = TIMED ? mbar_wait_at(uq_full(q, s), (k / kUnitQ) & 1, abort_flag, p.status, budget)
                           : queue_wait_polls(uq_full(q, s), (k / kUnitQ) & 1, shared_at<ABORT>(), p.status);
  if (!__all_sync(0xffffffffu, ready)) return false;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(unit) : "r"(uq_slot(q, s)) : "memory");
  __syncwarp();
  if (lane == 0) mbar_arrive_at(uq_empty(q, s));
  return true;
}

// Max over one row's 32 values of a 16x256b.x16 load (registers 4k + 2i + {0,1}, k < 16), then
// over the four threads that share the row.
__device__ __forceinline__ float row_max4(const uint32_t (&r)[64], int i) {
  float m8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    m8[k] = fmax3(__uint_as_float(r[4 * k + 2 * i]), __uint_as_float(r[4 * k + 2 * i + 1]),
                  __uint_as_float(r[4 * (k + 8) + 2 * i]));
#pragma unroll
  for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], __uint_as_float(r[4 * (k + 8) + 2 * i + 1]));
  float m = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
}

// P = 2^(s * c + nb_i) for the thread's 64 values (row i uses nb_i), as bf16 pairs: the pair of
// columns 8k + 2(t%4) + {0,1} (registers 4k + 2i + {0,1}, adjacent, so each packed fp32x2 op
// reads a register pair as it is) is P column 4k + t%4, which is where a 16x128b store puts
// register 2k + i.  PARTS stores of 64 / PARTS P columns (PARTS = 4 keeps fewer P words live, for
// the kernels whose registers are tightest); returns the fp32 row sums of the unrounded values.
template <int PARTS>
__device__ __forceinline__ void exp_tile(const uint32_t (&r)[64], uint64_t c2, float nb0, float nb1,
                                         uint32_t t_p, float (&sum)[2]) {
  constexpr int KP = 16 / PARTS;
  const uint64_t nbr[2] = {f2_pack(nb0, nb0), f2_pack(nb1, nb1)};
  uint64_t acc[2] = {0ull, 0ull};  // row 0, row 1
#pragma unroll
  for (int quarter = 0; quarter < PARTS; ++quarter) {
    uint32_t pk[2 * KP];
#pragma unroll
    for (int kk = 0; kk < KP; ++kk) {
      const int k = quarter * KP + kk;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint64_t a2 = f2_fma(f2_pack(__uint_as_float(r[4 * k + 2 * i]), __uint_as_float(r[4 * k + 2 * i + 1])),
                                   c2, nbr[i]);
        float e0, e1;
        f2_unpack(a2, e0, e1);
        const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
        acc[i] = f2_add(acc[i], f2_pack(p0, p1));
        pk[2 * kk + i] = pack_bf16x2(p0, p1);
      }
    }
    if constexpr (PARTS == 4) tmem_st_16x128b_x4(t_p + quarter * 16, pk);
    else tmem_st_16x128b_x8(t_p + quarter * 32, pk);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float s0, s1;
    f2_unpack(acc[i], s0, s1);
    sum[i] = s0 + s1;
  }
}

// 4 x 4 transpose of 32-bit words across the four threads of a row (lanes 4r .. 4r+3): on entry
// thread c holds w[j] = its word of group j, on return w[j] = thread j's word of group c.  Two
// butterfly rounds; in each, a thread keeps the words whose index bit matches its lane bit and
// trades the other with its partner.
__device__ __forceinline__ void quad_transpose4(uint32_t* w, int lane) {
#pragma unroll
  for (int bit = 1; bit <= 2; bit <<= 1) {
    const bool hi = (lane & bit) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j & bit) continue;
      const uint32_t send = hi ? w[j] : w[j + bit];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, bit);
      if (hi) w[j] = recv; else w[j + bit] = recv;
    }
  }
}

// MASKS = false: the launch has no tile that needs a mask (every link whole key tiles, no causal
// diagonal), so the kernel carries only the unmasked tile loop.  DYN: the launch deals its units
// dynamically (kDealDynamic); the static deals' kernels carry no queue code.
template <int D, int STAGES, bool MASKS, bool DYN>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using L = Layout<D, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = k_full + STAGES;
  uint64_t* k_empty = v_full + STAGES;  // K slot free: both score MMAs of its tile completed
  uint64_t* v_empty = k_empty + STAGES;  // V slot free: both P V MMAs of its tile completed
  uint64_t* s_full = v_empty + STAGES;  // [2]: query tile a, b
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_empty = pv_done + 2;
  uint64_t* mma_done = o_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);  // uniform
  const int lane = threadIdx.x & 31;
  const int wg = warp >> 2;
  const uint64_t budget = p.budget_ns;
  const uint64_t drain_budget = budget < 200000000ull ? budget : 200000000ull;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxThreads);
      mbar_init(&pv_done[i], 1);
      mbar_init(&o_empty[i], kSoftmaxThreads);
    }
    mbar_init(mma_done, 1);
    uint64_t* uq = reinterpret_cast<uint64_t*>(sm + L::kUnitQueue);
    for (int i = 0; i < kUnitQ; ++i) {
      mbar_init(uq + i, 1);                     // full: the producer's arrive
      mbar_init(uq + kUnitQ + i, kUnitReaders);  // empty: one arrive per reading warp
    }
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
      uint32_t kfills[STAGES], vfills[STAGES];
      for (int s = 0; s < STAGES; ++s) kfills[s] = vfills[s] = 0;
      // a static deal's CTA has `rounds` units or fewer; a dynamic one's walk ends at the first
      // index past the last unit
      const int rounds = p.withhold_loads ? 0 : (p.n_units + gridDim.x - 1) / gridDim.x;
      for (int t = 0; DYN ? !p.withhold_loads : t < rounds; ++t) {
        int unit;
        if constexpr (DYN) {
          if (!produce_unit<L::kUnitQueue>(p, t, abort_flag, budget, unit) || unit >= p.n_units) break;
        } else {
          unit = unit_of_round(p, t);
          if (unit >= p.n_units) continue;
        }
        const Unit u = decode_unit(p, unit);
        if (u.n_kv == 0) continue;
        const AttnSeg& s = *u.seg;
        if (q_iter > 0 && !mbar_wait(q_empty, (q_iter - 1) & 1, abort_flag, p.status, budget)) break;
        mbar_arrive_expect_tx(q_full, 2 * L::kQTile);
        const int qrow = s.q_row0 + u.q0;
        const int qn = p.map_rows[s.q_map];  // 0: one piece (4-D map)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int row = qrow + x * kAttnBM;  // 128-row tiles never straddle two pieces
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk) {
            uint8_t* dst = sm + L::kQ + x * L::kQTile + blk * kAttnBM * 128;
            if (qn == 0) tma_load_4d(dst, &p.maps[s.q_map], blk * 64, u.h, row, u.b, q_full);
            else tma_load_5d(dst, &p.maps[s.q_map], blk * 64, u.h, row % qn, row / qn, u.b, q_full);
          }
        }
        ++q_iter;
        bool ok = true;
        // the unit's key tiles: every link in order, each from its own K/V maps
        for (int li = 0; li < s.n_links && ok; ++li) {
          const AttnLink& lk = p.links[s.link0 + li];
          const int nl = link_tiles(lk, u.last_row);
          const int kn = p.map_rows[lk.k_map];  // the K and V maps of a link have the same pieces
          int kr = kn ? lk.kv_row0 % kn : lk.kv_row0, kp = kn ? lk.kv_row0 / kn : 0;  // row, piece
          for (int j = 0; j < nl; ++j) {
            // K(j) may overwrite K(j - STAGES) once its score MMAs are done, well before the P V
            // MMAs release V(j - STAGES).
            if (!mbar_wait(&k_empty[stage], phase ^ 1, abort_flag, p.status, budget)) { ok = false; break; }
            mbar_arrive_expect_tx(&k_full[stage], L::kKBytes);
#pragma unroll
            for (int blk = 0; blk < D / 64; ++blk) {
              uint8_t* dk = sm + L::kK + stage * L::kKBytes + blk * kAttnBN * 128;
              if (kn == 0) tma_load_4d(dk, &p.maps[lk.k_map], blk * 64, u.h, kr, u.b, &k_full[stage]);
              else tma_load_5d(dk, &p.maps[lk.k_map], blk * 64, u.h, kr, kp, u.b, &k_full[stage]);
            }
            ++kfills[stage];
            if (!mbar_wait(&v_empty[stage], phase ^ 1, abort_flag, p.status, budget)) { ok = false; break; }
            mbar_arrive_expect_tx(&v_full[stage], L::kVBytes);
#pragma unroll
            for (int blk = 0; blk < D / 64; ++blk) {
              uint8_t* dv = sm + L::kV + stage * L::kVBytes + blk * kAttnBN * 128;
              if (kn == 0) tma_load_4d(dv, &p.maps[lk.v_map], blk * 64, u.h, kr, u.b, &v_full[stage]);
              else tma_load_5d(dv, &p.maps[lk.v_map], blk * 64, u.h, kr, kp, u.b, &v_full[stage]);
            }
            ++vfills[stage];
            kr += kAttnBN;
            if (kn && kr >= kn) { kr -= kn; ++kp; }
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
          }
        }
        if (!ok) break;
      }
      for (int s = 0; s < STAGES; ++s) {
        if (kfills[s]) mbar_drain(&k_full[s], (kfills[s] - 1) & 1, drain_budget);
        if (vfills[s]) mbar_drain(&v_full[s], (vfills[s] - 1) & 1, drain_budget);
      }
      if (q_iter) mbar_drain(q_full, (q_iter - 1) & 1, drain_budget);
    } else if (warp == 1) {
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
      // Every lane waits; the vote keeps the warp's control flow uniform even if a wait times out
      // on some lanes only.
      auto wait_w = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status, budget));
      };
      // Shared-memory matrix descriptors (tcgen05 descriptor version 1): bits 0-13 start address
      // >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte offset >> 4 (1024 B: 8-row atoms),
      // 46-47 version 1, 49-51 base offset 0 (atoms 1024-byte aligned), 61-63 layout 2 (128-byte
      // swizzle).  The high word is the same for every operand; low word = start address >> 4 |
      // LBO field (1 for the K-major Q and K, 16384 B between V's 64-column blocks).
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
      // [0,32), keys 64-127 in [64,96).  V(st) was waited for before the first P V of its tile.
      auto pv = [&](int x, uint32_t st, bool first, bool last) -> bool {
        if (!wait_w(&p_full[x], gp[x] & 1)) return false;
        if (first && units_done > 0 &&
            !wait_w(&o_empty[x], (units_done - 1) & 1))
          return false;
        tc_fence_after();
        mma_group_pv(tmem + 256 + x * D, tmem + x * 128, v_lo + st * (L::kVBytes >> 4), kDescHi,
                     idesc_pv, first ? 0u : 1u);
        if (last) mma_commit(&pv_done[x]);
        ++gp[x];
        return true;
      };
      const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
      for (int t = 0; (DYN || t < rounds) && ok; ++t) {
        int unit;
        if constexpr (DYN) {
          if (!consume_unit<L::kUnitQueue, L::kAbort, true>(p, t, lane, abort_flag, budget, unit) ||
              unit >= p.n_units)
            break;
        } else {
          unit = unit_of_round(p, t);
          if (unit >= p.n_units) continue;
        }
        const Unit u = decode_unit(p, unit);
        if (u.n_kv == 0) continue;
        // Q and K/V come from TMA (async proxy, like the MMAs): the barrier waits order them, no
        // tcgen05 fence is needed; P comes from tcgen05.st of other threads (fence in pv()).
        if (!wait_w(q_full, q_iter & 1)) break;
        ++q_iter;
        uint32_t prev_stage = 0;
        if (!wait_w(&k_full[stage], phase)) break;
        // K(j) was waited for before this iteration; V(j) and K(j+1) are waited for just before the
        // wait for P_a(j), which is the long one, so that O_a += P_a V is followed directly by
        // S_a = Q_a K(j+1)^T.
        for (int j = 0; j < u.n_kv; ++j) {
          qk(0, stage);
          if (j > 0) {
            if (!pv(1, prev_stage, j == 1, false)) { ok = false; break; }
            mma_commit(&v_empty[prev_stage]);
          }
          qk(1, stage);
          mma_commit(&k_empty[stage]);
          if (j == u.n_kv - 1) mma_commit(q_empty);
          const uint32_t ns = stage + 1 == STAGES ? 0 : stage + 1;
          const uint32_t nph = ns == 0 ? phase ^ 1 : phase;
          if (!wait_w(&v_full[stage], phase)) { ok = false; break; }
          if (j + 1 < u.n_kv && !wait_w(&k_full[ns], nph)) { ok = false; break; }
          if (!pv(0, stage, j == 0, j == u.n_kv - 1)) { ok = false; break; }
          prev_stage = stage;
          stage = ns;
          phase = nph;
        }
        if (!ok) break;
        if (!pv(1, prev_stage, u.n_kv == 1, true)) { ok = false; break; }
        mma_commit(&v_empty[prev_stage]);
        ++units_done;
      }
      // drain: all issued MMAs complete before TMEM is freed
      mma_commit(mma_done);
      mbar_drain(mma_done, 0, drain_budget);
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    // Warpgroup wg (1..4) serves query tile x = (wg-1)/2 and, within every 32-lane quadrant of
    // TMEM, lane half hl = (wg-1)%2 (lanes 16*hl .. 16*hl+15 of the quadrant).  A thread owns
    // two rows, lanes q*32 + 16*hl + lane/4 and that + 8, and one quarter of their columns:
    // 16-lane loads give it columns 8k + 2(lane%4) + {0,1}; the four threads of a row combine
    // their maxima and sums with two shuffles.
    regs_inc<kRegsSoftmax>();
    const int x = (wg - 1) >> 1;   // query tile a (0) or b (1)
    const int hl = (wg - 1) & 1;   // lane half of each quadrant
    const int wq = warp & 3;
    const int lane_base = wq * 32 + hl * 16;
    const int rw[2] = {lane_base + (lane >> 2), lane_base + (lane >> 2) + 8};  // tile rows
    const int cq = 2 * (lane & 3);  // first of this thread's two columns in every 8-column group
    const uint32_t t_base = tmem + (static_cast<uint32_t>(lane_base) << 16);
    const uint32_t t_s = t_base + x * 128;  // S_x; P_x packed over its columns [0, 64)
    const uint32_t t_o = t_base + 256 + x * D;
    const float c = p.scale_log2;  // > 0 (checked on the host)
    const uint64_t c2 = f2_pack(c, c);
    uint32_t g = 0, units = 0;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool r = mbar_wait(bar, parity, abort_flag, p.status, budget);
      return __all_sync(0xffffffffu, r);
    };
    const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
    for (int t = 0; (DYN || t < rounds) && ok; ++t) {
      int unit;
      if constexpr (DYN) {
        if (!consume_unit<L::kUnitQueue, L::kAbort, false>(p, t, lane, abort_flag, budget, unit) ||
            unit >= p.n_units)
          break;
      } else {
        unit = unit_of_round(p, t);
        if (unit >= p.n_units) continue;
      }
      const Unit u = decode_unit(p, unit);
      const AttnSeg& s = *u.seg;
      const int q0 = u.q0 + x * kAttnBM;  // first local row of this query tile
      auto row_valid_at = [&](int i) { return rw[i] < min(kAttnBM, s.q_len - q0); };
      // output element of row i's column 0 and its LSE index (computed where used, so that they
      // are not live across the key-tile loop)
      auto out_at = [&](int i, long long& oe, long long& la) {
        const int ol = s.o_row0 + q0 + rw[i];  // output-side local row
        const long long opos = ol < s.o_len0
                                   ? static_cast<long long>(s.o_start0) + static_cast<long long>(ol) * s.o_stride
                                   : static_cast<long long>(s.o_start1) + static_cast<long long>(ol - s.o_len0) * s.o_stride;
        const long long orow = static_cast<long long>(u.b) * s.o_bstride + opos;
        la = orow * s.o_heads + u.h;
        oe = la * D;
      };
      if (u.n_kv == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (!row_valid_at(i)) continue;
          long long o_elem_i, lse_at_i;
          out_at(i, o_elem_i, lse_at_i);
          for (int k = 0; k < D / 8; ++k) {
            if (s.o_bf16) {
              reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(s.o) + o_elem_i + 8 * k + cq)[0] = 0u;
            } else {
              reinterpret_cast<float2*>(static_cast<float*>(s.o) + o_elem_i + 8 * k + cq)[0] = make_float2(0.f, 0.f);
            }
          }
          if ((lane & 3) == 0 && s.lse) s.lse[lse_at_i] = -INFINITY;
        }
        continue;
      }
      float m_ref[2] = {-INFINITY, -INFINITY};  // running max of scale*log2e*s, raised lazily
      float l[2] = {0.f, 0.f};                  // row sums over this thread's columns
      // One key tile: scores from TMEM, the online softmax update, P back to TMEM.  The
      // mask-free kernel (MASKS = false) runs `tile` on every tile; the other runs `tile_masked`,
      // which first writes -inf into the hidden columns of a tile that needs a mask (a small
      // TMEM pre-pass, so the tile body itself carries no mask code).  The two bodies are kept
      // apart because each instantiation's register allocation is at its limit.
      auto tile = [&]() -> bool {
        if (!wait_all(&s_full[x], g & 1)) return false;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld_16x256b_x16(t_s, r);
        tmem_wait_ld();
        float alpha[2] = {1.f, 1.f};
        bool resc = false;
        float sum[2];
        // Fast path: exponentials against the running max as it stands.  A partial sum above
        // kFastSum (or inf / NaN) means some score rose more than 11 log2 units above m: wait
        // for the P stores, then redo the tile after raising m.
        bool fast = __all_sync(0xffffffffu, m_ref[0] != -INFINITY && m_ref[1] != -INFINITY);
        if (fast) {
          exp_tile<2>(r, c2, -m_ref[0], -m_ref[1], t_s, sum);
          fast = __all_sync(0xffffffffu, sum[0] <= kFastSum && sum[1] <= kFastSum);
          if (!fast) tmem_wait_st();
        }
        if (!fast) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float mx = row_max4(r, i) * c;
            if (mx > m_ref[i] + kTau) {
              if (m_ref[i] != -INFINITY) {
                alpha[i] = ex2_approx(m_ref[i] - mx);
                resc = true;
              }
              m_ref[i] = mx;
            }
          }
          const float nb0 = m_ref[0] == -INFINITY ? 0.f : -m_ref[0];
          const float nb1 = m_ref[1] == -INFINITY ? 0.f : -m_ref[1];
          exp_tile<2>(r, c2, nb0, nb1, t_s, sum);
        }
        l[0] = l[0] * alpha[0] + sum[0];
        l[1] = l[1] * alpha[1] + sum[1];
        if (__any_sync(0xffffffffu, resc)) {
          // S_x(j) complete => P V of tile j-1 complete: O_x is stable
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t w[32];
            tmem_ld_16x256b_x8(t_o + cc * 64, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha[(i >> 1) & 1]);
            tmem_st_16x256b_x8(t_o + cc * 64, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
        ++g;
        return true;
      };
      auto tile_masked = [&](int li, int j, bool masked) -> bool {
        if (!wait_all(&s_full[x], g & 1)) return false;
        tc_fence_after();
        if (masked) {
          const int kv_len = p.links[li].kv_len, diag = p.links[li].diag;
          const int c0 = j * kAttnBN;  // link-local key index of column 0
          uint32_t m[64];
          tmem_ld_16x256b_x16(t_s, m);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int lim = diag == kNoDiag ? kv_len - 1 : min(kv_len - 1, q0 + rw[i] + diag);
            const int last = lim - c0 - cq;
#pragma unroll
            for (int k = 0; k < 16; ++k)
#pragma unroll
              for (int e = 0; e < 2; ++e)
                if (8 * k + e > last) m[4 * k + 2 * i + e] = 0xff800000u;  // -inf
          }
          tmem_st_16x256b_x16(t_s, m);
          tmem_wait_st();
        }
        uint32_t r[64];
        tmem_ld_16x256b_x16(t_s, r);
        tmem_wait_ld();
        float alpha[2] = {1.f, 1.f};
        bool resc = false;
        float sum[2];
        // Fast path: exponentials against the running max as it stands.  A partial sum above
        // kFastSum (or inf / NaN) means some score rose more than 11 log2 units above m: wait
        // for the P stores, then redo the tile after raising m.
        bool fast = __all_sync(0xffffffffu, m_ref[0] != -INFINITY && m_ref[1] != -INFINITY);
        if (fast) {
          exp_tile<D == 64 ? 4 : 2>(r, c2, -m_ref[0], -m_ref[1], t_s, sum);
          fast = __all_sync(0xffffffffu, sum[0] <= kFastSum && sum[1] <= kFastSum);
          if (!fast) tmem_wait_st();
        }
        if (!fast) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float mx = row_max4(r, i) * c;
            if (mx > m_ref[i] + kTau) {
              if (m_ref[i] != -INFINITY) {
                alpha[i] = ex2_approx(m_ref[i] - mx);
                resc = true;
              }
              m_ref[i] = mx;
            }
          }
          const float nb0 = m_ref[0] == -INFINITY ? 0.f : -m_ref[0];
          const float nb1 = m_ref[1] == -INFINITY ? 0.f : -m_ref[1];
          exp_tile<D == 64 ? 4 : 2>(r, c2, nb0, nb1, t_s, sum);
        }
        l[0] = l[0] * alpha[0] + sum[0];
        l[1] = l[1] * alpha[1] + sum[1];
        if (__any_sync(0xffffffffu, resc)) {
          // S_x(j) complete => P V of tile j-1 complete: O_x is stable
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t w[32];
            tmem_ld_16x256b_x8(t_o + cc * 64, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha[(i >> 1) & 1]);
            tmem_st_16x256b_x8(t_o + cc * 64, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[x]);
        ++g;
        return true;
      };
      // one online softmax over the key tiles of every link of the segment, in link order; a
      // link's length and diagonal are re-read from the parameters where needed, so that only
      // the link index and the tile counters stay live across the tiles
      for (int li = s.link0; li < s.link0 + s.n_links && ok; ++li) {
        // the unit's last valid row, from values that are live anyway
        const int last_row = min(s.q_len, q0 - x * kAttnBM + kAttnUnitRows) - 1;
        // tiles [0, mf) need no mask: whole tiles of keys that every row of this query tile sees
        int mf = min(link_tiles(p.links[li], last_row), p.links[li].kv_len / kAttnBN);
        if (p.links[li].diag != kNoDiag) {
          const int d1 = q0 + p.links[li].diag + 1;  // keys [0, d1) are visible to the tile's first row
          mf = min(mf, d1 <= 0 ? 0 : d1 / kAttnBN);
        }
        int j = 0;
        if constexpr (!MASKS) {
          for (; j < mf; ++j)
            if (!tile()) { ok = false; break; }
          if (!ok) break;
        } else {
          // tiles j >= mf get their hidden columns set to -inf in TMEM first
          const int nl = link_tiles(p.links[li], last_row);
          for (; j < nl; ++j)
            if (!tile_masked(li, j, j >= mf)) { ok = false; break; }
        }
      }
      if (!ok) break;
      // epilogue: full row sums from the four threads of each row, then O / l and the lse
      float inv_l[2], lse[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float lt = l[i];
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        inv_l[i] = lt > 0.f ? 1.0f / lt : 0.f;
        lse[i] = lt > 0.f ? (m_ref[i] + lg2_approx(lt)) * kLn2 : -INFINITY;
      }
      if (!wait_all(&pv_done[x], units & 1)) { ok = false; break; }  // committed once per unit
      ++units;
      tc_fence_after();
      long long o_elem[2], lse_at[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) out_at(i, o_elem[i], lse_at[i]);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t o[32];
        tmem_ld_16x256b_x8(t_o + cc * 64, o);
        tmem_wait_ld();
        if (cc == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(&o_empty[x]);
        }
        if (s.o_bf16) {
          // The four threads of a row hold one bf16 pair of each 8-column group; a 4 x 4 word
          // transpose across them (two shuffle rounds) gives thread lane%4 all of groups
          // 4g + lane%4, which it writes as one 16-byte store per group.
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(__uint_as_float(o[4 * k + 2 * i]) * inv_l[i],
                                 __uint_as_float(o[4 * k + 2 * i + 1]) * inv_l[i]);
            quad_transpose4(w, lane);
            quad_transpose4(w + 4, lane);
            if (row_valid_at(i)) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(s.o) + o_elem[i] + cc * 64 +
                                                    4 * cq);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);  // group lane%4
              dst[4] = make_uint4(w[4], w[5], w[6], w[7]);  // group 4 + lane%4
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (!row_valid_at(i)) continue;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float v0 = __uint_as_float(o[4 * k + 2 * i]) * inv_l[i];
              const float v1 = __uint_as_float(o[4 * k + 2 * i + 1]) * inv_l[i];
              reinterpret_cast<float2*>(static_cast<float*>(s.o) + o_elem[i] + cc * 64 + 8 * k + cq)[0] =
                  make_float2(v0, v1);
            }
          }
        }
      }
      if ((lane & 3) == 0 && s.lse) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (row_valid_at(i)) s.lse[lse_at[i]] = lse[i];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (DYN && threadIdx.x == 0) {
    // Every role of this CTA is past its last take of a unit.  The last CTA to get here returns
    // the counter (and this count of finished CTAs) to zero for the next launch.
    __threadfence();
    if (atomicAdd(p.counter + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.counter, 0u);
      atomicExch(p.counter + 1, 0u);
    }
  }
}

template <int D, int STAGES, bool MASKS, bool DYN>
usp_status_t launch_one(const AttnParams& p, cudaStream_t stream) {
  using L = Layout<D, STAGES>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  auto kern = attn_fwd_kernel<D, STAGES, MASKS, DYN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const int grid = std::max(1, std::min(p.n_units, sm_count()));
  kern<<<grid, kThreads, L::kAlloc, stream>>>(p);
  return check_launch("attention kernel");
}

}  // namespace

usp_status_t make_qkv_map(CUtensorMap* map, const void* base, int n_heads, int D, int64_t piece_rows,
                          int n_pieces, int B, int64_t row_stride, int64_t piece_stride,
                          int64_t batch_stride) {
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
  const int64_t rows = std::max<int64_t>(piece_rows, 1);
  const int64_t pstride = std::max<int64_t>(piece_stride, rows * row_stride);
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(n_heads),
                              static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(std::max(n_pieces, 1)),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(row_stride) * 2,
                                 static_cast<cuuint64_t>(pstride) * 2,
                                 static_cast<cuuint64_t>(std::max<int64_t>(batch_stride, row_stride)) * 2};
  const cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(kAttnBM), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r;
  if (n_pieces <= 1) {  // {D, heads, rows, B}: the piece dimension dropped
    const cuuint64_t dims4[4] = {dims[0], dims[1], dims[2], dims[4]};
    const cuuint64_t strides3[3] = {strides[0], strides[1], strides[3]};
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims4, strides3, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(USP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return USP_OK;
}

int deal_env() {
  const char* env = std::getenv("USP_UNIT_DEAL");
  if (!env || !*env) return -1;
  return std::atoi(env) & (kDealCount - 1);
}

namespace {
// The deals worth modelling: the static four and, with a counter, dynamic with either block order.
constexpr int kDealChoices[] = {0, kDealRoundRobin, kDealAlternate, kDealRoundRobin | kDealAlternate,
                                kDealDynamic, kDealDynamic | kDealAlternate};
}  // namespace

double deal_periods(const AttnParams& p, int deal, int ctas) {
  std::vector<double> load(ctas, 0.0), cost;
  // dynamic: CTAs by (time free, index); the first free one takes the next unit
  std::priority_queue<std::pair<double, int>, std::vector<std::pair<double, int>>,
                      std::greater<std::pair<double, int>>> free_at;
  if (deal & kDealDynamic)
    for (int c = 0; c < ctas; ++c) free_at.push({0.0, c});
  for (int gi = 0; gi < p.n_groups; ++gi) {
    const AttnGroup& G = p.groups[gi];
    cost.clear();  // key tiles + epilogue of every block of the group, in block order
    for (int si = G.seg0; si < G.seg0 + G.n_segs; ++si) {
      const AttnSeg& s = p.segs[si];
      for (int qi = 0; qi < s.n_qblk; ++qi) {
        const int qb = s.rev ? s.n_qblk - 1 - qi : qi;
        const int last = std::min(s.q_len, (qb + 1) * kAttnUnitRows) - 1;
        int n = 0;
        for (int l = 0; l < s.n_links; ++l) n += link_tiles(p.links[s.link0 + l], last);
        cost.push_back(n + (s.o_bf16 ? 2.0 : 2.5));
      }
    }
    const int n = G.blocks * p.segs[G.seg0].n_heads * p.B;
    for (int i = 0; i < n; ++i) {
      const int unit = G.unit0 + i, t = unit / ctas;
      const int hb = i / G.blocks;
      const double c = cost[deal_block(i - hb * G.blocks, G.blocks, hb, deal)];
      if (deal & kDealDynamic) {
        const auto [at, cta] = free_at.top();
        free_at.pop();
        load[cta] = at + c;
        free_at.push({at + c, cta});
      } else {
        load[deal_unit(t, unit - t * ctas, ctas, deal) - t * ctas] += c;
      }
    }
  }
  return *std::max_element(load.begin(), load.end());
}

usp_status_t pack_attention(const AttnParams& base, std::vector<AttnSeg>& segs,
                            const std::vector<AttnLink>& links, std::vector<AttnLaunch>& out, int sms) {
  out.clear();
  if (!(base.scale_log2 > 0.f)) return fail(USP_ERR_INVALID_ARG, "the softmax scale must be positive");
  // Segments grouped by unit group, longest first within a group: sort by the key tiles their
  // longest query block visits.
  auto cost = [&](const AttnSeg& s) {
    long long c = 0;
    for (int i = 0; i < s.n_links; ++i) c += link_tiles(links[s.link0 + i], s.q_len - 1);
    return c;
  };
  std::stable_sort(segs.begin(), segs.end(), [&](const AttnSeg& a, const AttnSeg& b) {
    return a.grp != b.grp ? a.grp < b.grp : cost(a) > cost(b);
  });
  size_t at = 0;
  while (at < segs.size()) {
    out.emplace_back();
    AttnLaunch& L = out.back();
    L.params = base;
    AttnParams& p = L.params;
    long long units = 0;
    int used = 0, n_links = 0, n_groups = 0;
    for (; at < segs.size() && used < kAttnMaxSegs; ++at) {
      AttnSeg s = segs[at];
      if (s.n_links > kAttnMaxLinks) return fail(USP_ERR_UNSUPPORTED, "too many links in one segment");
      if (n_links + s.n_links > kAttnMaxLinks) break;
      s.n_qblk = (s.q_len + kAttnUnitRows - 1) / kAttnUnitRows;
      if (s.n_qblk == 0) continue;  // (a segment whose links see no key still writes o = 0, lse = -inf)
      const bool new_group = n_groups == 0 || p.segs[used - 1].grp != s.grp;
      if (new_group) {
        if (n_groups == kAttnMaxGroups) break;
        if (n_groups > 0) {  // close the previous group
          AttnGroup& G = p.groups[n_groups - 1];
          units += static_cast<long long>(G.blocks) * p.segs[G.seg0].n_heads * p.B;
        }
        p.groups[n_groups++] = {static_cast<int>(units), 0, used, 0};
      }
      AttnGroup& G = p.groups[n_groups - 1];
      s.qb0 = G.blocks;
      G.blocks += s.n_qblk;
      ++G.n_segs;
      for (int i = 0; i < s.n_links; ++i) p.links[n_links + i] = links[s.link0 + i];
      s.link0 = n_links;
      n_links += s.n_links;
      p.segs[used++] = s;
    }
    if (n_groups > 0) {
      AttnGroup& G = p.groups[n_groups - 1];
      units += static_cast<long long>(G.blocks) * p.segs[G.seg0].n_heads * p.B;
    }
    if (units > INT_MAX / 2) return fail(USP_ERR_UNSUPPORTED, "too many attention work units");
    p.n_segs = used;
    p.n_groups = n_groups;
    p.n_units = static_cast<int>(units);
    // the unit deal with the shortest modelled launch, if it beats the default by more than 0.5 %
    p.deal = 0;
    const bool dynamic_ok = p.counter != nullptr;
    if (const int forced = deal_env(); forced >= 0) {
      p.deal = dynamic_ok ? forced : forced & ~kDealDynamic;
    } else if (units > 0) {
      const int ctas = std::max(1, std::min(p.n_units, sms > 0 ? sms : sm_count()));
      const double t0 = deal_periods(p, 0, ctas);
      double best = t0;
      for (int d : kDealChoices) {
        if (d == 0 || ((d & kDealDynamic) && !dynamic_ok)) continue;
        const double t = deal_periods(p, d, ctas);
        if (t < best && t < 0.995 * t0) { best = t; p.deal = d; }
      }
    }
    // the mask-free kernel when every link is whole key tiles without a causal diagonal
    L.masks = false;
    for (int i = 0; i < n_links; ++i)
      L.masks = L.masks || p.links[i].diag != kNoDiag || p.links[i].kv_len % kAttnBN != 0;
    if (units == 0) out.pop_back();
  }
  return USP_OK;
}

usp_status_t run_attention(const std::vector<AttnLaunch>& launches, int D, cudaStream_t stream) {
  for (const AttnLaunch& L : launches) {
    const AttnParams& p = L.params;
    const bool dyn = (p.deal & kDealDynamic) != 0;
    usp_status_t st;
    if (D == 64)
      st = L.masks ? (dyn ? launch_one<64, 4, true, true>(p, stream) : launch_one<64, 4, true, false>(p, stream))
                   : (dyn ? launch_one<64, 4, false, true>(p, stream) : launch_one<64, 4, false, false>(p, stream));
    else
      st = L.masks ? (dyn ? launch_one<128, 2, true, true>(p, stream) : launch_one<128, 2, true, false>(p, stream))
                   : (dyn ? launch_one<128, 2, false, true>(p, stream) : launch_one<128, 2, false, false>(p, stream));
    if (st != USP_OK) return st;
  }
  return USP_OK;
}

usp_status_t launch_attention(AttnParams& p, std::vector<AttnSeg>& segs,
                              const std::vector<AttnLink>& links, int D, cudaStream_t stream,
                              int* n_launched) {
  if (n_launched) *n_launched = 0;
  static thread_local std::vector<AttnLaunch> launches;
  if (usp_status_t st = pack_attention(p, segs, links, launches)) return st;
  if (usp_status_t st = run_attention(launches, D, stream)) return st;
  if (n_launched) *n_launched = static_cast<int>(launches.size());
  return USP_OK;
}

}  // namespace usp
