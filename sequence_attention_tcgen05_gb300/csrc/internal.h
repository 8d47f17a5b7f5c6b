// Host-side declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <vector>

#include "usp.h"

namespace usp {

// ------------------------------------------------------------------------------------------
// Errors: the thread-local message behind usp_last_error().
// ------------------------------------------------------------------------------------------
usp_status_t fail(usp_status_t s, const char* fmt, ...);
usp_status_t check_launch(const char* what);
usp_status_t check_device();  // current device must be sm_103
int sm_count();               // SMs of the current device (cached per device; 152 on a GB300)

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Launch with programmatic stream serialization (for kernels that start with pdl_prologue()):
// the kernel may be scheduled while the previous kernel of the stream finishes, which hides the
// launch latency between back-to-back bandwidth-bound kernels.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Default split of n items over P parts: floor(n/P) + (p < n mod P).
std::vector<int> default_split(int n, int P);

// Global positions of ring rank r's local rows under an ordering (piecewise affine, <= 2 pieces).
struct Positions {
  int n_seg = 1;
  int start[2] = {0, 0};
  int len[2] = {0, 0};
  int stride = 1;
  int rows() const { return len[0] + (n_seg > 1 ? len[1] : 0); }
  int64_t at(int i) const {
    return i < len[0] ? int64_t(start[0]) + int64_t(i) * stride
                      : int64_t(start[1]) + int64_t(i - len[0]) * stride;
  }
};
std::vector<Positions> ring_positions(usp_order_t order, int S, int R);

// ------------------------------------------------------------------------------------------
// Re-layout (Ulysses all-to-all as a permutation, reorder, and their fusion).
// Rows are enumerated as (ring group r, batch b, ring-local row l).  The "head side" is a set of
// per-(r, head group g) buffers [B][S_r][h_g][D]; the "sequence side" is either packed chunks
// (mode 0: chunk (r, u) = [B][len][H][D] holding ring-local rows [off, off + len)) or a global
// [B][S][H][D] tensor addressed through the ordering's positions (mode 1).
// ------------------------------------------------------------------------------------------
constexpr int kRelayoutMaxR = 64;
constexpr int kRelayoutMaxU = 64;
constexpr int kRelayoutMaxRU = 256;

struct RelayoutParams {
  const char* src[3];
  char* dst[3];
  int n_tensors;
  int B, H, D, elem;  // D = elements per head, elem = bytes per element
  int R, U;
  int seq_mode;  // 0 packed chunks, 1 global through positions
  int dir;       // 0 sequence side -> head side, 1 head side -> sequence side
  int S;         // global sequence length (mode 1)
  long long seq_rs;  // elements from one sequence-side row to the next (H * D unless packed)
  long long row0[kRelayoutMaxR + 1];
  int S_r[kRelayoutMaxR];
  int h[kRelayoutMaxU];
  int hoff[kRelayoutMaxU];
  long long hbase[kRelayoutMaxRU];  // element offset of head-side block (r, g)
  int c_off[kRelayoutMaxRU];        // mode 0: chunk (r, u)
  int c_len[kRelayoutMaxRU];
  long long c_base[kRelayoutMaxRU];
  int p_start0[kRelayoutMaxR], p_len0[kRelayoutMaxR], p_start1[kRelayoutMaxR],
      p_stride[kRelayoutMaxR];  // mode 1
};

usp_status_t launch_relayout(RelayoutParams& p, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// LSE merge.
// ------------------------------------------------------------------------------------------
// Optional output placement for the merge: the partials are in the head-sharded layout of
// usp_attention (blocks (r, u) of [B][S_r][h_u] vectors, back to back); the merged vector of block k,
// batch b, ring-local row l, head h' goes to global row b*S + pos_k(l), head hoff_k + h'.
constexpr int kMergeMaxBlocks = 16;
struct MergeMap {
  int n_blocks;
  int H, S;
  long long vec0[kMergeMaxBlocks + 1];  // first vector of each block; vec0[n_blocks] = total
  long long row0[kMergeMaxBlocks + 1];  // first row (B * S_r rows per block); row0[n_blocks] = total
  int S_r[kMergeMaxBlocks], h[kMergeMaxBlocks], hoff[kMergeMaxBlocks];
  int p_start0[kMergeMaxBlocks], p_len0[kMergeMaxBlocks], p_start1[kMergeMaxBlocks],
      p_stride[kMergeMaxBlocks];
  int all_seen;  // no partial can be empty (non-causal): load every partial with its LSE
};

usp_status_t launch_lse_merge(int n_parts, const float* o_parts, int64_t o_part_stride,
                              const float* lse_parts, int64_t lse_part_stride, int64_t n_vec,
                              int D, void* o_out, bool out_bf16, float* lse_out,
                              const MergeMap* map, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// Partial attention (tcgen05).
// ------------------------------------------------------------------------------------------
constexpr int kAttnBM = 128;  // query rows per tile (one TMEM lane each)
constexpr int kAttnBN = 128;  // key rows per tile
constexpr int kAttnUnitRows = 2 * kAttnBM;  // query rows per work unit (two tiles per CTA)
constexpr int kAttnMaxMaps = 48;
constexpr int kAttnMaxSegs = 96;
constexpr int kAttnMaxLinks = 256;
constexpr int kNoDiag = INT_MAX;

// One key range of a unit's online softmax: keys c (0 <= c < kv_len) of the K/V maps, map rows
// kv_row0 + c; key c is visible to segment-local query row i iff c <= i + diag (diag == kNoDiag:
// no limit).  A segment of one link is one ring step's (Q chunk, K/V chunk) pair; a segment of
// several links is a chain: its query rows carry one online softmax across the K/V chunks of
// every ring step (the ring merge done in registers), and it writes the final O and LSE.
struct AttnLink {
  int k_map, v_map;
  int kv_row0, kv_len;
  int diag;
};

// One run of query rows against the links [link0, link0 + n_links).  Q tiles come from 4-D (or
// 5-D, two-piece) tensor maps {D, heads, rows, batch}; rows of this run are map rows q_row0 + i.
// Output row of query i of batch b:
//   row = b * o_bstride + pos(o_row0 + i),  pos(l) = l < o_len0 ? o_start0 + l * o_stride
//                                                               : o_start1 + (l - o_len0) * o_stride
// and element (row * o_heads + h) * D of `o` (LSE: row * o_heads + h of `lse`); `o` and `lse` are
// already offset to the run's first head.  Identity pos (o_len0 = INT_MAX) for a dense output.
struct AttnSeg {
  void* o;        // bf16 when o_bf16, else fp32
  float* lse;     // may be null
  int o_bf16;     // 1: bf16 O (a final output); 0: fp32 O (a final output or a ring partial)
  int q_map;
  int q_row0, q_len;
  int link0, n_links;
  int n_heads;    // heads of the maps (the same for every segment of a group)
  int o_row0, o_bstride, o_heads;
  int o_start0, o_len0, o_start1, o_stride;
  int grp;        // unit group (one per Ulysses rank): its segments share n_heads
  int n_qblk;     // 256-row query blocks (set at launch)
  int qb0;        // first block of this segment within its group (set at launch)
  int rev;        // 1: visit query blocks last first (causal: longest first)
};

// Work units of one group are numbered head-major: for every (batch, head), the query blocks of
// all the group's segments (segments longest first, blocks in their visiting order).  All CTAs
// working at the same time then share one or two heads' K/V, which stays in L2.
constexpr int kAttnMaxGroups = 16;
struct AttnGroup {
  int unit0;      // first unit
  int blocks;     // query blocks per (batch, head): sum of the segments' n_qblk
  int seg0, n_segs;
};

// Unit deals: which CTA of a G-CTA grid takes which unit, and in which order each (batch, head)
// of a group visits its blocks.  Every role of the kernel walks the same sequence, and each unit
// computes the same values wherever it runs, so the deal changes timing only.
//   default: snake order (round t: CTA c takes unit t*G + c, or t*G + G-1-c for odd t), every
//            (batch, head) visiting its blocks in the group's order (longest first);
//   kDealRoundRobin: round t, CTA c takes unit t*G + c;
//   kDealAlternate:  odd (batch, head) indices of a group visit their blocks in reverse order;
//   kDealDynamic:    units in numbering order, each to the CTA that asks first (a counter in
//                    global memory, AttnParams::counter); kDealRoundRobin has no effect then.
constexpr int kDealRoundRobin = 1;
constexpr int kDealAlternate = 2;
constexpr int kDealDynamic = 4;
constexpr int kDealCount = 8;
// The unit CTA c takes in round t (the map is its own inverse within a round: the CTA that takes
// unit u is deal_unit(u / G, u % G, G, deal) - (u / G) * G).
__host__ __device__ inline int deal_unit(int t, int c, int G, int deal) {
  const bool flip = !(deal & kDealRoundRobin) && (t & 1);
  return t * G + (flip ? G - 1 - c : c);
}
// The block (index over the group's segments) that a (batch, head) index hb visits rem-th.
__host__ __device__ inline int deal_block(int rem, int blocks, int hb, int deal) {
  return (deal & kDealAlternate) && (hb & 1) ? blocks - 1 - rem : rem;
}

struct AttnParams {
  CUtensorMap maps[kAttnMaxMaps];
  int map_rows[kAttnMaxMaps];  // two-piece maps: rows per piece (row l = piece l / n, row l % n); 0: one piece
  AttnSeg segs[kAttnMaxSegs];
  AttnLink links[kAttnMaxLinks];
  AttnGroup groups[kAttnMaxGroups];
  int n_groups;
  int n_segs;
  int n_units;
  int deal;            // kDealRoundRobin | kDealAlternate | kDealDynamic bits
  // kDealDynamic: {next unit, finished CTAs}, zero at launch; the last CTA to finish zeroes both
  uint32_t* counter;
  int B;
  float scale_log2;
  uint32_t* status;
  unsigned long long budget_ns;
  int withhold_loads;  // test hook: the producer issues no loads, so every wait runs out
};

// A run of query rows produced by the chunk-pair planner.
struct Run {
  int q0, q_len, kv_len, diag;
};
// Runs for query rows with positions qp against key rows with positions kp (both increasing).
// causal = false gives one run covering everything.
std::vector<Run> plan_runs(const Positions& qp, const Positions& kp, bool causal);

// 5-D tensor map {D, n_heads, piece_rows, n_pieces, B} over bf16 data: heads adjacent (D elements
// apart), rows row_stride elements apart, pieces piece_stride apart, batches batch_stride apart.
// Map row l is row l % piece_rows of piece l / piece_rows: one piece (encoded as the 4-D map
// {D, n_heads, rows, B}) for a chunk that is one run of rows, two for a zigzag chunk (its two
// half-chunks) addressed in place.  Box: 64 x 1 x 128 (x 1) x 1.
usp_status_t make_qkv_map(CUtensorMap* map, const void* base, int n_heads, int D, int64_t piece_rows,
                          int n_pieces, int B, int64_t row_stride, int64_t piece_stride,
                          int64_t batch_stride);

// One kernel launch's parameters (segments, links and groups packed) and which instantiation runs
// it (masks = false: no link needs a mask).
struct AttnLaunch {
  AttnParams params;
  bool masks;
};
// Packs the segments (sorted in place) and their links into launches, each starting from `base`
// (maps, scale, status, budget, counter), with the unit deal chosen for a grid of
// min(units, sms) CTAs (sms = 0: the current device's SM count; dynamic deals only with a
// counter); run_attention runs them.
usp_status_t pack_attention(const AttnParams& base, std::vector<AttnSeg>& segs,
                            const std::vector<AttnLink>& links, std::vector<AttnLaunch>& out,
                            int sms = 0);
// Modelled time of one packed launch over `ctas` CTAs in key-tile periods under a unit deal: each
// unit costs its key tiles plus an epilogue (2 periods for bf16 rows, 2.5 for fp32) and runs on
// the CTA the deal gives it (dynamic: the CTA that becomes free first, the lowest index among
// equals).  pack_attention gives each launch the deal with the shortest modelled time when it
// beats the default by more than 0.5 %; USP_UNIT_DEAL=0..7 in the environment (read at each call)
// forces one (a dynamic one falls back to its static bits without a counter).
double deal_periods(const AttnParams& p, int deal, int ctas);
int deal_env();  // -1 when USP_UNIT_DEAL is unset
usp_status_t run_attention(const std::vector<AttnLaunch>& launches, int D, cudaStream_t stream);

// Launch over all segments, each with its own links (split into several launches if there are
// more than fit; `n_launched`, if not null, receives how many).  The links of segs[i] are
// links[segs[i].link0 .. + n_links) of `links`.
usp_status_t launch_attention(AttnParams& p, std::vector<AttnSeg>& segs,
                              const std::vector<AttnLink>& links, int D, cudaStream_t stream,
                              int* n_launched);

// Key tiles of a link visited by a 256-row query block whose last segment-local row is
// `last_row` (host and device).
__host__ __device__ inline int link_tiles(const AttnLink& lk, int last_row) {
  int max_c = lk.kv_len - 1;
  if (lk.diag != kNoDiag) max_c = max_c < last_row + lk.diag ? max_c : last_row + lk.diag;
  return max_c < 0 ? 0 : max_c / kAttnBN + 1;
}

}  // namespace usp

// Kernel parameters are passed by value; CUDA 12.1+ allows up to 32764 bytes of them.
static_assert(sizeof(usp::AttnParams) <= 32764, "attention kernel parameters too large");
static_assert(sizeof(usp::RelayoutParams) <= 32764, "relayout kernel parameters too large");
