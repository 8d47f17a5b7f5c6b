// C ABI entry points: argument validation, the chunk-pair planner, workspace layout and the
// launch sequence of usp_attention.  Nothing here allocates device memory or synchronises,
// except usp_check_status.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>

#include "internal.h"

namespace usp {

namespace {
thread_local std::string g_last_error;
constexpr unsigned long long kDefaultBudgetNs = 2000000000ull;  // 2 s per bounded wait

unsigned long long wait_budget_ns() {
  const char* s = std::getenv("USP_WAIT_BUDGET_MS");
  if (s && *s) {
    const long long ms = std::atoll(s);
    if (ms > 0) return static_cast<unsigned long long>(ms) * 1000000ull;
  }
  return kDefaultBudgetNs;
}

// Test hook for the failure path: USP_TEST_WITHHOLD_LOADS=1 makes the attention kernel's producer
// issue no loads, so the other roles' bounded waits run out and the status word reports it.
int withhold_loads() {
  const char* s = std::getenv("USP_TEST_WITHHOLD_LOADS");
  return (s && s[0] == '1' && s[1] == 0) ? 1 : 0;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

usp_status_t fail(usp_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

usp_status_t check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return USP_OK;
}

usp_status_t check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(USP_ERR_NO_DEVICE, "no CUDA device is current");
  }
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(USP_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                major, minor);
  return USP_OK;
}

int sm_count() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return 152;
  }
  if (cached[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

std::vector<int> default_split(int n, int P) {
  std::vector<int> out(P);
  for (int p = 0; p < P; ++p) out[p] = n / P + (p < n % P ? 1 : 0);
  return out;
}

std::vector<Positions> ring_positions(usp_order_t order, int S, int R) {
  std::vector<Positions> pos(R);
  if (order == USP_ORDER_CONTIGUOUS) {
    auto len = default_split(S, R);
    int off = 0;
    for (int r = 0; r < R; ++r) {
      pos[r].n_seg = 1;
      pos[r].start[0] = off;
      pos[r].len[0] = len[r];
      pos[r].stride = 1;
      off += len[r];
    }
  } else if (order == USP_ORDER_ZIGZAG) {
    auto len = default_split(S, 2 * R);
    std::vector<int> off(2 * R + 1, 0);
    for (int i = 0; i < 2 * R; ++i) off[i + 1] = off[i] + len[i];
    for (int r = 0; r < R; ++r) {
      pos[r].n_seg = 2;
      pos[r].start[0] = off[r];
      pos[r].len[0] = len[r];
      pos[r].start[1] = off[2 * R - 1 - r];
      pos[r].len[1] = len[2 * R - 1 - r];
      pos[r].stride = 1;
    }
  } else {
    for (int r = 0; r < R; ++r) {
      pos[r].n_seg = 1;
      pos[r].start[0] = r;
      pos[r].len[0] = S > r ? (S - r + R - 1) / R : 0;
      pos[r].stride = R;
    }
  }
  return pos;
}

// Number of keys with position <= x.
static int64_t visible_count(const Positions& kp, int64_t x) {
  int64_t v = 0;
  for (int s = 0; s < kp.n_seg; ++s) {
    const int64_t len = kp.len[s];
    if (len == 0 || x < kp.start[s]) continue;
    v += std::min<int64_t>(len, (x - kp.start[s]) / kp.stride + 1);
  }
  return v;
}

// Greedy partition of the query rows into runs whose visible-key count has the form
// V(i) = clamp(i - q0 + e, 0, L): zeros, then +1 per row, then a plateau.  Causal chunk pairs of
// the contiguous, zigzag and stripe orderings need one run per contiguous query piece.
std::vector<Run> plan_runs(const Positions& qp, const Positions& kp, bool causal) {
  const int nq = qp.rows(), nk = kp.rows();
  std::vector<Run> runs;
  if (nq == 0) return runs;
  if (!causal) {
    runs.push_back({0, nq, nk, kNoDiag});
    return runs;
  }
  std::vector<int64_t> V(nq);
  for (int i = 0; i < nq; ++i) V[i] = visible_count(kp, qp.at(i));
  int i = 0;
  while (i < nq) {
    const int s = i;
    // phase 0: zeros; 1: slope +1; 2: plateau
    int phase = V[s] == 0 ? 0 : -1;
    int64_t e = 0, L = V[s];
    bool slope_seen = false;
    ++i;
    if (phase == -1) {
      // first row non-zero: the next row decides between a slope (e = V[s]) and a plateau
      if (i < nq && V[i] == V[s] + 1) { phase = 1; e = V[s]; slope_seen = true; }
      else phase = 2;
    }
    while (i < nq) {
      const int64_t v = V[i], prev = V[i - 1];
      if (phase == 0) {
        if (v == 0) { ++i; continue; }
        if (v == 1) { phase = 1; e = 1 - (i - s); slope_seen = true; ++i; continue; }
        break;
      }
      if (phase == 1) {
        if (v == prev + 1) { ++i; continue; }
        if (v == prev) { phase = 2; L = v; ++i; continue; }
        break;
      }
      // plateau
      if (v == L) { ++i; continue; }
      break;
    }
    Run r;
    r.q0 = s;
    r.q_len = i - s;
    if (phase == 0) {
      r.kv_len = 0;
      r.diag = kNoDiag;
    } else if (!slope_seen) {
      r.kv_len = static_cast<int>(L);
      r.diag = kNoDiag;
    } else {
      r.kv_len = static_cast<int>(phase == 2 ? L : V[i - 1]);
      r.diag = static_cast<int>(e - 1);
    }
    runs.push_back(r);
  }
  return runs;
}

}  // namespace usp

using namespace usp;

namespace {

// A ring chunk of two runs of rows that are not adjacent in the global tensor (zigzag with several
// ring ranks); one ring rank's two zigzag pieces are adjacent and form one run.
bool two_pieces(const Positions& ps) {
  return ps.n_seg > 1 && ps.len[0] > 0 && ps.len[1] > 0 &&
         int64_t(ps.start[1]) != int64_t(ps.start[0]) + int64_t(ps.len[0]) * ps.stride;
}

struct Grid {
  int B = 0, S = 0, H = 0, D = 0, U = 0, R = 0;
  bool causal = false;
  // Ring mode (several ring ranks): fused = each query block's online softmax runs across the K/V
  // chunks of every ring step and writes the final O and LSE (the merge happens in registers);
  // otherwise every ring step writes an fp32 partial and a merge pass combines them.
  bool fused_ring = false;
  usp_order_t order = USP_ORDER_CONTIGUOUS;
  std::vector<Positions> pos;  // per ring group
  std::vector<int> S_r;        // ring chunk lengths
  std::vector<int> h, hoff;    // head groups
  // Q/K/V of every virtual rank are addressed in place in the global tensor.  A ring chunk that is
  // one affine run of rows has a 4-D map over it; a zigzag chunk of two equal half-chunks of
  // whole 128-row tiles a 5-D map with a piece dimension; any other zigzag chunk a 4-D "span" map
  // over the global rows from its first half-chunk's start to its second's end, in which its
  // second half-chunk starts at map row span_off[r] (0: no span map).  Query runs and key ranges
  // of a span-mapped chunk never cross its half-chunk boundary (the planner cuts them there), so
  // the rows of other ranks inside the span are never read as its rows.
  std::vector<int> span_off;
  bool span(int r) const { return span_off[r] > 0; }
  int maprow(int r, int l) const {  // map row of ring-local row l of chunk r
    return span(r) && l >= pos[r].len[0] ? span_off[r] + (l - pos[r].len[0]) : l;
  }
  // Split of a fused ring (non-causal only): query rows [split_row, S_r) of ring chunk split_r in
  // Ulysses group split_u run as separate ring steps, writing fp32 partials into slots of their
  // own ([R][B][split_rows][h][D]) that a merge pass combines after the attention.  Their units
  // form a unit group of their own, dealt after every chain, so that these shorter units fill
  // the last round of equal-length chains.  split_r = -1: no split.
  int split_r = -1, split_u = 0, split_row = 0;
  int split_rows() const { return split_r < 0 ? 0 : S_r[split_r] - split_row; }
  int64_t split_vec() const { return split_r < 0 ? 0 : int64_t(B) * split_rows() * h[split_u]; }
  // workspace layout (bytes)
  size_t off_opart = 0, off_lpart = 0, off_spart = 0, off_slpart = 0, total = 0;
  int64_t elems = 0;  // B*S*H*D
  int64_t woff(int r, int u, int d) const {  // element offset of block (r, u) in the W layout
    int64_t off = 0;
    for (int rr = 0; rr < r; ++rr) off += int64_t(B) * S_r[rr] * H * d;
    for (int uu = 0; uu < u; ++uu) off += int64_t(B) * S_r[r] * h[uu] * d;
    return off;
  }
};

bool choose_fused_ring(const Grid& g, usp_dtype_t o_dt);

// USP_RING_MERGE (environment, read at each call): 1 = "fused", 2 = "separate", 0 = unset/other.
int ring_env() {
  const char* env = std::getenv("USP_RING_MERGE");
  if (env && std::strcmp(env, "fused") == 0) return 1;
  if (env && std::strcmp(env, "separate") == 0) return 2;
  return 0;
}

// USP_RING_SPLIT (environment, read at each call): "0" = never split a fused ring, a positive
// number k = split the last k 256-row blocks of the last ring chunk of the last Ulysses group
// (non-causal fused rings; for tests), unset = the model decides.
int split_env() {
  const char* env = std::getenv("USP_RING_SPLIT");
  if (!env || !*env) return -1;
  return std::max(0, std::atoi(env));
}

void choose_split(Grid& g, usp_dtype_t o_dt);

usp_status_t build_grid(Grid& g, int B, int S, int H, int D, int causal, int U, int R,
                        usp_order_t order, const int32_t* seq_lens, const int32_t* head_counts,
                        usp_dtype_t o_dt) {
  if (B < 1 || S < 0 || H < 1) return fail(USP_ERR_INVALID_ARG, "need B >= 1, S >= 0, H >= 1");
  if (D != 64 && D != 128) return fail(USP_ERR_UNSUPPORTED, "head dim D=%d: only 64 and 128 are built", D);
  if (U < 1 || R < 1 || U > 16 || R > 16 || U * R > 16)
    return fail(USP_ERR_INVALID_ARG, "need 1 <= ulysses_degree, ring_degree and their product <= 16");
  if (order != USP_ORDER_CONTIGUOUS && order != USP_ORDER_ZIGZAG && order != USP_ORDER_STRIPE)
    return fail(USP_ERR_INVALID_ARG, "unknown order %d", static_cast<int>(order));
  if (o_dt != USP_BF16 && o_dt != USP_FP32) return fail(USP_ERR_INVALID_ARG, "o_dt must be BF16 or FP32");
  if (int64_t(B) * S * H * D >= (int64_t(1) << 40)) return fail(USP_ERR_INVALID_ARG, "tensor too large");
  g.B = B; g.S = S; g.H = H; g.D = D; g.U = U; g.R = R; g.order = order;
  g.causal = causal != 0;
  g.pos = ring_positions(order, S, R);
  g.S_r.resize(R);
  for (int r = 0; r < R; ++r) g.S_r[r] = g.pos[r].rows();
  if (seq_lens) {
    for (int r = 0; r < R; ++r) {
      int64_t sum = 0;
      for (int u = 0; u < U; ++u) {
        if (seq_lens[r * U + u] < 0) return fail(USP_ERR_INVALID_ARG, "seq_lens[%d] < 0", r * U + u);
        sum += seq_lens[r * U + u];
      }
      if (sum != g.S_r[r])
        return fail(USP_ERR_INVALID_ARG, "seq_lens of ring group %d sum to %lld, its ring chunk has %d rows",
                    r, static_cast<long long>(sum), g.S_r[r]);
    }
  }
  if (head_counts) {
    int64_t sum = 0;
    for (int u = 0; u < U; ++u) {
      if (head_counts[u] < 1) return fail(USP_ERR_INVALID_ARG, "head_counts[%d] < 1", u);
      sum += head_counts[u];
    }
    if (sum != H) return fail(USP_ERR_INVALID_ARG, "head_counts sum to %lld, H = %d", static_cast<long long>(sum), H);
    g.h.assign(head_counts, head_counts + U);
  } else {
    if (H < U) return fail(USP_ERR_INVALID_ARG, "H=%d < ulysses_degree=%d", H, U);
    g.h = default_split(H, U);
  }
  g.hoff.assign(U, 0);
  for (int u = 1; u < U; ++u) g.hoff[u] = g.hoff[u - 1] + g.h[u - 1];
  // span maps for the zigzag chunks whose half-chunks differ in length or are not whole 128-row
  // tiles (a tile of a 5-D map must not straddle them)
  g.span_off.assign(R, 0);
  for (int r = 0; r < R; ++r) {
    const Positions& ps = g.pos[r];
    if (two_pieces(ps) && !(ps.len[0] == ps.len[1] && ps.len[0] % kAttnBM == 0))
      g.span_off[r] = ps.start[1] - ps.start[0];
  }
  g.elems = int64_t(B) * S * H * D;
  const int64_t rowsH = int64_t(B) * S * H;
  size_t at = 256;  // status word
  auto take = [&](size_t bytes) {
    const size_t o = at;
    at = static_cast<size_t>(align_up(static_cast<int64_t>(at + bytes), 256));
    return o;
  };
  g.fused_ring = R > 1 && choose_fused_ring(g, o_dt);
  if (R > 1 && !g.fused_ring) {
    g.off_opart = take(size_t(R) * g.elems * 4);
    g.off_lpart = take(size_t(R) * rowsH * 4);
  }
  if (g.fused_ring && !g.causal && S > 0) choose_split(g, o_dt);
  if (g.split_r >= 0) {
    g.off_spart = take(size_t(R) * g.split_vec() * D * 4);
    g.off_slpart = take(size_t(R) * g.split_vec() * 4);
  }
  g.total = at;
  return USP_OK;
}

// ------------------------------------------------------------------------------------------------
// Attention work lists.  Output placement of a segment: ring partial slot k of block (r, u) (the W
// layout, fp32), or the final global [B][S][H] layout through ring chunk r's positions.
// ------------------------------------------------------------------------------------------------
// Where a segment writes: byte offsets from the caller's o and lse (the final output), or from the
// workspace (a ring partial slot).  Plans hold offsets, not pointers, so that they can be reused
// across calls with other buffers.
struct SegOut {
  bool partial;
  int64_t o_off, lse_off;  // bytes
};

struct AttnPlan {
  std::vector<AttnSeg> segs;  // o and lse are filled in per call from `outs`
  std::vector<SegOut> outs;
  std::vector<AttnLink> links;
};

int map_index(const Grid& g, int r, int u, int t) { return (r * g.U + u) * 3 + t; }

SegOut set_final_output(AttnSeg& s, const Grid& g, int r, int u, int oel) {
  s.o_bstride = g.S; s.o_heads = g.H;
  s.o_start0 = g.pos[r].start[0]; s.o_len0 = g.pos[r].n_seg > 1 ? g.pos[r].len[0] : INT_MAX;
  s.o_start1 = g.pos[r].start[1]; s.o_stride = g.pos[r].stride;
  return {false, int64_t(g.hoff[u]) * g.D * oel, int64_t(g.hoff[u]) * 4};
}

// A zigzag chunk read through a 5-D map is two pieces of whole tiles: every run must start on a
// 128-row tile so that no tile straddles its half-chunks (runs start at 0 or at the second half
// for these orderings).
usp_status_t check_run_start(const Grid& g, int r, const Run& run) {
  if (two_pieces(g.pos[r]) && !g.span(r) && run.q0 % kAttnBM != 0)
    return fail(USP_ERR_UNSUPPORTED, "zigzag run at row %d does not start on a 128-row tile", run.q0);
  return USP_OK;
}

// The links of one ring step for a segment of q_len query rows: the visible keys of K/V chunk r2
// are its ring-local keys [0, kv_len), key c visible to segment-local query i iff c <= i + diag
// (kNoDiag: no limit).  One link, or two when chunk r2 has a span map: its first half-chunk's
// keys, and its second's from their own map row with the diagonal shifted by the first half's
// length.  A link that no query row sees is left out.
void add_links(const Grid& g, int r2, int u, int kv_len, int diag, int q_len,
               std::vector<AttnLink>& links) {
  const int km = map_index(g, r2, u, 1), vm = map_index(g, r2, u, 2);
  auto seen = [&](int len, int d) { return len > 0 && (d == kNoDiag || (q_len - 1) + d >= 0); };
  if (!g.span(r2)) {
    if (seen(kv_len, diag)) links.push_back({km, vm, 0, kv_len, diag});
    return;
  }
  const int len0 = g.pos[r2].len[0];
  const int n0 = std::min(kv_len, len0), n1 = kv_len - len0;
  const int d1 = diag == kNoDiag ? kNoDiag : diag - len0;
  if (seen(n0, diag)) links.push_back({km, vm, 0, n0, diag});
  if (seen(n1, d1)) links.push_back({km, vm, g.span_off[r2], n1, d1});
}

// Causal pieces whose length is not a multiple of the 256-row block: cut the remainder off the
// piece's start, so that the short block holds the rows that see the fewest keys (at the end it
// would hold the rows that see the most, and cost as much as a whole block).  Chunks read
// through a 5-D map have pieces of whole 128-row tiles, so the cut stays on a tile.
void front_remainders(const Grid& g, std::vector<int>& cuts) {
  if (!g.causal) return;
  const size_t n = cuts.size();
  for (size_t i = 0; i + 1 < n; ++i) {
    const int len = cuts[i + 1] - cuts[i], rem = len % kAttnUnitRows;
    if (len > kAttnUnitRows && rem != 0) cuts.push_back(cuts[i] + rem);
  }
  std::sort(cuts.begin(), cuts.end());
}

// The same for runs (separate ring steps): a run's remainder rows become a run of their own.
std::vector<Run> front_remainders(const Grid& g, const std::vector<Run>& runs) {
  if (!g.causal) return runs;
  std::vector<Run> out;
  for (const Run& run : runs) {
    const int rem = run.q_len % kAttnUnitRows;
    if (run.q_len > kAttnUnitRows && rem != 0) {
      Run a = run, b = run;
      a.q_len = rem;
      b.q0 = run.q0 + rem;
      b.q_len = run.q_len - rem;
      if (b.diag != kNoDiag) b.diag += rem;
      out.push_back(a);
      out.push_back(b);
    } else {
      out.push_back(run);
    }
  }
  return out;
}

// The runs of ring chunk r, cut where a span-mapped chunk's second half-chunk starts.
std::vector<Run> cut_at_span(const Grid& g, int r, const std::vector<Run>& runs) {
  if (!g.span(r)) return runs;
  const int len0 = g.pos[r].len[0];
  std::vector<Run> out;
  for (const Run& run : runs) {
    if (run.q0 < len0 && run.q0 + run.q_len > len0) {
      Run a = run, b = run;
      a.q_len = len0 - run.q0;
      b.q0 = len0;
      b.q_len = run.q0 + run.q_len - len0;
      if (b.diag != kNoDiag) b.diag += len0 - run.q0;
      out.push_back(a);
      out.push_back(b);
    } else {
      out.push_back(run);
    }
  }
  return out;
}

// One segment per (ring rank r, ring step k, Ulysses rank u, run of query rows), one link each.
usp_status_t plan_separate(const Grid& g, int oel, AttnPlan& pl) {
  const int64_t slot_o = g.elems * 4, slot_l = int64_t(g.B) * g.S * g.H;
  for (int r = 0; r < g.R; ++r) {
    for (int kstep = 0; kstep < g.R; ++kstep) {
      const int r2 = (r - kstep + g.R) % g.R;
      const std::vector<Run> runs =
          front_remainders(g, cut_at_span(g, r, plan_runs(g.pos[r], g.pos[r2], g.causal)));
      for (const Run& run : runs)
        if (usp_status_t st = check_run_start(g, r, run)) return st;
      for (int u = 0; u < g.U; ++u) {
        for (const Run& run : runs) {
          AttnSeg s{};
          s.q_map = map_index(g, r, u, 0);
          s.q_row0 = g.maprow(r, run.q0); s.q_len = run.q_len;
          // every (ring step, run) segment writes its partial slot, with no link at all if no
          // row sees a key (o = 0, lse = -inf)
          s.link0 = static_cast<int>(pl.links.size());
          add_links(g, r2, u, run.kv_len, run.diag, run.q_len, pl.links);
          s.n_links = static_cast<int>(pl.links.size()) - s.link0;
          s.n_heads = g.h[u];
          s.grp = u;
          s.o_row0 = run.q0;
          s.rev = g.causal;
          if (g.R > 1) {
            pl.outs.push_back({true, int64_t(g.off_opart) + kstep * slot_o + g.woff(r, u, g.D) * 4,
                               int64_t(g.off_lpart) + (kstep * slot_l + g.woff(r, u, 1)) * 4});
            s.o_bstride = g.S_r[r]; s.o_heads = g.h[u];
            s.o_start0 = 0; s.o_len0 = INT_MAX; s.o_start1 = 0; s.o_stride = 1;
          } else {
            pl.outs.push_back(set_final_output(s, g, r, u, oel));
          }
          pl.segs.push_back(s);
        }
      }
    }
  }
  return USP_OK;
}

// Ring steps fused: the query rows of ring chunk r are cut at every run boundary of every ring
// step, so that within a piece each step's visible keys keep the run form (clamp(i + e, 0, L));
// a piece is one segment whose links are the ring steps k = 0..R-1 in ring order (K/V chunk
// (r - k) mod R), skipping steps that no row of the piece sees.
usp_status_t plan_fused(const Grid& g, int oel, AttnPlan& pl) {
  for (int r = 0; r < g.R; ++r) {
    const int Sr = g.S_r[r];
    if (Sr == 0) continue;
    std::vector<std::vector<Run>> runs(g.R);
    std::vector<int> cuts = {0, Sr};
    if (g.span(r)) cuts.push_back(g.pos[r].len[0]);  // pieces never cross the half-chunks
    if (r == g.split_r && g.split_row > 0) cuts.push_back(g.split_row);
    for (int kstep = 0; kstep < g.R; ++kstep) {
      runs[kstep] = plan_runs(g.pos[r], g.pos[(r - kstep + g.R) % g.R], g.causal);
      for (const Run& run : runs[kstep]) {
        if (usp_status_t st = check_run_start(g, r, run)) return st;
        cuts.push_back(run.q0);
      }
    }
    std::sort(cuts.begin(), cuts.end());
    cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());
    front_remainders(g, cuts);
    for (size_t ci = 0; ci + 1 < cuts.size(); ++ci) {
      const int a = cuts[ci], b = cuts[ci + 1];
      for (int u = 0; u < g.U; ++u) {
        if (r == g.split_r && u == g.split_u && a >= g.split_row) {
          // split rows: one segment per ring step, each writing its fp32 partial slot
          const int64_t slot_o = g.split_vec() * g.D * 4, slot_l = g.split_vec() * 4;
          for (int kstep = 0; kstep < g.R; ++kstep) {
            const int r2 = (r - kstep + g.R) % g.R;
            AttnSeg s{};
            s.q_map = map_index(g, r, u, 0);
            s.q_row0 = g.maprow(r, a); s.q_len = b - a;
            s.link0 = static_cast<int>(pl.links.size());
            for (const Run& x : runs[kstep])
              if (x.q0 <= a && a < x.q0 + x.q_len)
                add_links(g, r2, u, x.kv_len, x.diag == kNoDiag ? kNoDiag : x.diag + (a - x.q0), b - a,
                          pl.links);
            s.n_links = static_cast<int>(pl.links.size()) - s.link0;
            s.n_heads = g.h[u];
            s.grp = g.U;  // dealt after every chain
            s.rev = g.causal;
            s.o_row0 = a - g.split_row; s.o_bstride = g.split_rows(); s.o_heads = g.h[u];
            s.o_start0 = 0; s.o_len0 = INT_MAX; s.o_start1 = 0; s.o_stride = 1;
            pl.outs.push_back({true, int64_t(g.off_spart) + kstep * slot_o, int64_t(g.off_slpart) + kstep * slot_l});
            pl.segs.push_back(s);
          }
          continue;
        }
        AttnSeg s{};
        s.q_map = map_index(g, r, u, 0);
        s.q_row0 = g.maprow(r, a); s.q_len = b - a;
        s.link0 = static_cast<int>(pl.links.size());
        for (int kstep = 0; kstep < g.R; ++kstep) {
          const int r2 = (r - kstep + g.R) % g.R;
          const Run* run = nullptr;
          for (const Run& x : runs[kstep])
            if (x.q0 <= a && a < x.q0 + x.q_len) run = &x;
          if (!run) continue;
          const int diag = run->diag == kNoDiag ? kNoDiag : run->diag + (a - run->q0);
          add_links(g, r2, u, run->kv_len, diag, b - a, pl.links);  // none if no row sees a key
        }
        s.n_links = static_cast<int>(pl.links.size()) - s.link0;
        s.n_heads = g.h[u];
        s.grp = u;
        s.o_row0 = a;
        s.rev = g.causal;
        pl.outs.push_back(set_final_output(s, g, r, u, oel));
        pl.segs.push_back(s);
      }
    }
  }
  return USP_OK;
}

// Modelled time of one launch in key-tile periods: units dealt as the kernel deals them (per unit
// group, head-major over the group's segments taken longest first; snake order over the CTAs),
// each costing its key tiles plus an epilogue overhead.
double launch_periods(std::vector<AttnSeg> segs, const std::vector<AttnLink>& links, int B,
                      double overhead, int ctas) {
  auto seg_cost = [&](const AttnSeg& s) {
    long long c = 0;
    for (int i = 0; i < s.n_links; ++i) c += link_tiles(links[s.link0 + i], s.q_len - 1);
    return c;
  };
  std::stable_sort(segs.begin(), segs.end(), [&](const AttnSeg& a, const AttnSeg& b) {
    return a.grp != b.grp ? a.grp < b.grp : seg_cost(a) > seg_cost(b);
  });
  std::vector<double> load(ctas, 0.0);
  long long unit = 0;
  size_t g0 = 0;
  while (g0 < segs.size()) {
    size_t g1 = g0;
    while (g1 < segs.size() && segs[g1].grp == segs[g0].grp) ++g1;
    std::vector<int> tiles;  // the group's blocks in visiting order, per (batch, head)
    for (size_t i = g0; i < g1; ++i) {
      const AttnSeg& s = segs[i];
      const int n_qblk = (s.q_len + kAttnUnitRows - 1) / kAttnUnitRows;
      for (int qi = 0; qi < n_qblk; ++qi) {
        const int qb = s.rev ? n_qblk - 1 - qi : qi;
        const int last = std::min(s.q_len, (qb + 1) * kAttnUnitRows) - 1;
        int n = 0;
        for (int l = 0; l < s.n_links; ++l) n += link_tiles(links[s.link0 + l], last);
        tiles.push_back(n);
      }
    }
    for (long long hb = 0; hb < int64_t(segs[g0].n_heads) * B; ++hb) {
      for (int n : tiles) {
        const long long t = unit / ctas, c = unit % ctas;
        load[(t & 1) ? ctas - 1 - c : c] += n + overhead;
        ++unit;
      }
    }
    g0 = g1;
  }
  return *std::max_element(load.begin(), load.end());
}

// Fused or separate ring steps, from the modelled time of both: the separate mode also pays its
// merge pass (bytes at about 6 TB/s; one key-tile period is about 1.55 us) and a larger epilogue
// per unit (fp32 partial rows).  The same arguments always give the same answer (no device
// query), so usp_attention_workspace_size and usp_attention agree.  USP_RING_MERGE=fused or
// =separate (environment, read at each call) overrides the model.
bool choose_fused_ring(const Grid& g, usp_dtype_t o_dt) {
  if (const int env = ring_env()) return env == 1;
  constexpr int kModelCtas = 152;
  constexpr double kPeriodBytes = 6.0e12 * 1.55e-6;  // merge bytes per key-tile period
  AttnPlan sep, fus;
  if (plan_separate(g, 4, sep) != USP_OK) return false;
  if (plan_fused(g, 4, fus) != USP_OK) return false;
  const double t_sep = launch_periods(sep.segs, sep.links, g.B, 2.5, kModelCtas);
  const double t_fus = launch_periods(fus.segs, fus.links, g.B, o_dt == USP_BF16 ? 2.0 : 2.5, kModelCtas);
  // merge bytes: every partial LSE, the O of partials whose rows saw a key, the final O and LSE
  double seen_vec = 0;
  for (const AttnSeg& s : sep.segs) {
    if (s.n_links == 0) continue;  // no row sees a key (a later link never sees more rows)
    const AttnLink& lk = sep.links[s.link0];
    const int rows = lk.diag == kNoDiag ? s.q_len : std::max(0, s.q_len - std::max(0, -lk.diag));
    seen_vec += double(rows) * s.n_heads * g.B;
  }
  const double rows_h = double(g.B) * g.S * g.H;
  const double merge_bytes = g.R * rows_h * 4 + seen_vec * g.D * 4 +
                             rows_h * (g.D * (o_dt == USP_BF16 ? 2 : 4) + 4);
  return t_fus <= t_sep + merge_bytes / kPeriodBytes;
}

// Split of a fused non-causal ring (see Grid): the chains of a ring are all equally long there,
// and when their count is not a multiple of the SMs the last round runs part-empty.  Running the
// last k 256-row blocks of one ring chunk as separate ring steps turns those units into R
// shorter ones dealt after every chain; they fill the last round, at the price of their fp32
// partials and a merge pass over their rows.  The model deals the units as the kernel does
// (launch_periods) for every ring chunk of the last Ulysses group and every k, adds the merge's
// bytes at ~6 TB/s and a launch, and keeps the best split if it saves more than 1 %.
// USP_RING_SPLIT overrides it.
void choose_split(Grid& g, usp_dtype_t o_dt) {
  g.split_r = -1;
  const int env = split_env();
  if (env == 0) return;
  const int u = g.U - 1;
  auto set = [&](int r, int k) {
    const int nblk = (g.S_r[r] + kAttnUnitRows - 1) / kAttnUnitRows;
    k = std::min(k, nblk);
    g.split_r = r; g.split_u = u; g.split_row = (nblk - k) * kAttnUnitRows;
  };
  if (env > 0) {
    set(g.R - 1, env);
    return;
  }
  constexpr int kModelCtas = 152;
  constexpr double kPeriodBytes = 6.0e12 * 1.55e-6;  // merge bytes per key-tile period
  const int oel = o_dt == USP_BF16 ? 2 : 4;
  auto model = [&]() -> double {
    AttnPlan pl;
    if (plan_fused(g, oel, pl) != USP_OK) return 1e30;
    double t = launch_periods(pl.segs, pl.links, g.B, 2.0, kModelCtas);
    if (g.split_r >= 0) {
      const double vec = double(g.split_vec());
      t += (g.R * vec * (g.D * 4 + 4) + vec * (g.D * oel + 4)) / kPeriodBytes + 2.0;
    }
    return t;
  };
  const double t0 = model();
  double best = t0;
  int best_r = -1, best_k = 0;
  for (int r = 0; r < g.R; ++r) {
    const int nblk = (g.S_r[r] + kAttnUnitRows - 1) / kAttnUnitRows;
    for (int k = 1; k <= nblk; ++k) {
      set(r, k);
      const double t = model();
      if (t < best) { best = t; best_r = r; best_k = k; }
    }
  }
  g.split_r = -1;
  if (best_r >= 0 && best < 0.99 * t0) set(best_r, best_k);
}

// ------------------------------------------------------------------------------------------------
// Plan cache.  Planning a long ring (the chunk-pair runs of every ring step, the ring-mode time
// model) takes milliseconds on the host; a caller running the same shapes step after step gets
// the plan from here, and each call only binds its buffers and encodes its tensor maps.  Keyed by
// every argument that shapes the plan (and the USP_RING_MERGE override); the last kPlanCache
// plans are kept.
// ------------------------------------------------------------------------------------------------
struct PlanKey {
  int B, S, H, D, causal, U, R, order, o_dt, ring_env, split_env, deal_env;
  std::vector<int32_t> seq_lens, head_counts;
  bool operator==(const PlanKey& o) const {
    return B == o.B && S == o.S && H == o.H && D == o.D && causal == o.causal && U == o.U &&
           R == o.R && order == o.order && o_dt == o.o_dt && ring_env == o.ring_env &&
           split_env == o.split_env && deal_env == o.deal_env &&
           seq_lens == o.seq_lens && head_counts == o.head_counts;
  }
};

struct PlanEntry {
  PlanKey key;
  Grid g;
  AttnPlan plan;
};

constexpr size_t kPlanCache = 16;
std::mutex g_plan_mu;
std::vector<std::shared_ptr<const PlanEntry>> g_plan_cache;  // most recent first

// The validated grid and attention plan for these arguments (built and cached on first use).
usp_status_t get_plan(int B, int S, int H, int D, int causal, int U, int R, usp_order_t order,
                      const int32_t* seq_lens, const int32_t* head_counts, usp_dtype_t o_dt,
                      std::shared_ptr<const PlanEntry>& out) {
  PlanKey key{B, S, H, D, causal != 0, U, R, static_cast<int>(order), static_cast<int>(o_dt), ring_env(),
              split_env(), deal_env(), {}, {}};
  if (seq_lens && U >= 1 && R >= 1 && U <= 16 && R <= 16) key.seq_lens.assign(seq_lens, seq_lens + U * R);
  if (head_counts && U >= 1 && U <= 16) key.head_counts.assign(head_counts, head_counts + U);
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    for (size_t i = 0; i < g_plan_cache.size(); ++i) {
      if (g_plan_cache[i]->key == key) {
        out = g_plan_cache[i];
        if (i > 0) {
          g_plan_cache.erase(g_plan_cache.begin() + i);
          g_plan_cache.insert(g_plan_cache.begin(), out);
        }
        return USP_OK;
      }
    }
  }
  auto e = std::make_shared<PlanEntry>();
  e->key = key;
  if (usp_status_t st = build_grid(e->g, B, S, H, D, causal, U, R, order, seq_lens, head_counts, o_dt))
    return st;
  const int oel = o_dt == USP_BF16 ? 2 : 4;
  if (S > 0) {
    usp_status_t st = e->g.fused_ring ? plan_fused(e->g, oel, e->plan) : plan_separate(e->g, oel, e->plan);
    if (st) return st;
  }
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plan_cache.insert(g_plan_cache.begin(), e);
  if (g_plan_cache.size() > kPlanCache) g_plan_cache.pop_back();
  out = e;
  return USP_OK;
}

void fill_relayout_grid(RelayoutParams& rp, const Grid& g, int d, int elem) {
  std::memset(&rp, 0, sizeof(rp));
  rp.B = g.B; rp.H = g.H; rp.D = d; rp.elem = elem; rp.R = g.R; rp.U = g.U;
  rp.seq_mode = 1; rp.S = g.S;
  rp.seq_rs = int64_t(g.H) * d;
  int64_t row = 0;
  for (int r = 0; r < g.R; ++r) {
    rp.row0[r] = row;
    row += int64_t(g.B) * g.S_r[r];
    rp.S_r[r] = g.S_r[r];
    rp.p_start0[r] = g.pos[r].start[0];
    rp.p_len0[r] = g.pos[r].len[0];
    rp.p_start1[r] = g.pos[r].start[1];
    rp.p_stride[r] = g.pos[r].stride;
  }
  rp.row0[g.R] = row;
  for (int u = 0; u < g.U; ++u) { rp.h[u] = g.h[u]; rp.hoff[u] = g.hoff[u]; }
  for (int r = 0; r < g.R; ++r)
    for (int u = 0; u < g.U; ++u) rp.hbase[r * g.U + u] = g.woff(r, u, d);
}

usp_status_t relayout_public(int n_tensors, const void* const* src, void* const* dst, usp_dtype_t dt,
                             int B, int H, int D, int P, const int32_t* seq_lens,
                             const int32_t* head_counts, int dir, cudaStream_t stream) {
  if (n_tensors < 1 || n_tensors > 3) return fail(USP_ERR_INVALID_ARG, "need 1 <= n_tensors <= 3");
  if (!src || !dst || !seq_lens) return fail(USP_ERR_INVALID_ARG, "NULL src, dst or seq_lens");
  for (int t = 0; t < n_tensors; ++t)
    if (!src[t] || !dst[t]) return fail(USP_ERR_INVALID_ARG, "NULL src[%d] or dst[%d]", t, t);
  if (dt != USP_BF16 && dt != USP_FP32) return fail(USP_ERR_INVALID_ARG, "dt must be BF16 or FP32");
  if (B < 1 || H < 1 || D < 1) return fail(USP_ERR_INVALID_ARG, "need B, H, D >= 1");
  if (P < 1 || P > kRelayoutMaxU) return fail(USP_ERR_INVALID_ARG, "need 1 <= P <= %d", kRelayoutMaxU);
  RelayoutParams rp;
  std::memset(&rp, 0, sizeof(rp));
  const int elem = dt == USP_BF16 ? 2 : 4;
  int64_t S = 0;
  for (int q = 0; q < P; ++q) {
    if (seq_lens[q] < 0) return fail(USP_ERR_INVALID_ARG, "seq_lens[%d] < 0", q);
    rp.c_off[q] = static_cast<int>(S);
    rp.c_len[q] = seq_lens[q];
    rp.c_base[q] = int64_t(B) * S * H * D;
    S += seq_lens[q];
  }
  if (S > INT_MAX / 2 || int64_t(B) * S * H * D >= (int64_t(1) << 40))
    return fail(USP_ERR_INVALID_ARG, "tensor too large");
  std::vector<int> h;
  if (head_counts) {
    int64_t sum = 0;
    for (int p = 0; p < P; ++p) {
      if (head_counts[p] < 1) return fail(USP_ERR_INVALID_ARG, "head_counts[%d] < 1", p);
      sum += head_counts[p];
    }
    if (sum != H) return fail(USP_ERR_INVALID_ARG, "head_counts sum to %lld, H = %d", static_cast<long long>(sum), H);
    h.assign(head_counts, head_counts + P);
  } else {
    if (H < P) return fail(USP_ERR_INVALID_ARG, "H=%d < P=%d with default head counts", H, P);
    h = default_split(H, P);
  }
  if (S == 0) return USP_OK;
  if (usp_status_t st = check_device()) return st;
  for (int t = 0; t < n_tensors; ++t) {
    rp.src[t] = static_cast<const char*>(src[t]);
    rp.dst[t] = static_cast<char*>(dst[t]);
  }
  rp.n_tensors = n_tensors;
  rp.B = B; rp.H = H; rp.D = D; rp.elem = elem; rp.R = 1; rp.U = P;
  rp.seq_mode = 0; rp.dir = dir; rp.S = static_cast<int>(S);
  rp.seq_rs = int64_t(H) * D;
  rp.row0[0] = 0;
  rp.row0[1] = int64_t(B) * S;
  rp.S_r[0] = static_cast<int>(S);
  int off = 0;
  for (int p = 0; p < P; ++p) {
    rp.h[p] = h[p];
    rp.hoff[p] = off;
    rp.hbase[p] = int64_t(B) * S * off * D;
    off += h[p];
  }
  return launch_relayout(rp, stream);
}

}  // namespace

extern "C" {

usp_status_t usp_relayout_seq2head(const void* src, void* dst, usp_dtype_t dt, int B, int H, int D,
                                   int P, const int32_t* seq_lens, const int32_t* head_counts,
                                   usp_stream_t stream) {
  void* d = dst;
  return relayout_public(1, &src, &d, dt, B, H, D, P, seq_lens, head_counts, 0,
                         reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_relayout_head2seq(const void* src, void* dst, usp_dtype_t dt, int B, int H, int D,
                                   int P, const int32_t* seq_lens, const int32_t* head_counts,
                                   usp_stream_t stream) {
  void* d = dst;
  return relayout_public(1, &src, &d, dt, B, H, D, P, seq_lens, head_counts, 1,
                         reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_relayout_seq2head_multi(int n_tensors, const void* const* src, void* const* dst,
                                         usp_dtype_t dt, int B, int H, int D, int P,
                                         const int32_t* seq_lens, const int32_t* head_counts,
                                         usp_stream_t stream) {
  return relayout_public(n_tensors, src, dst, dt, B, H, D, P, seq_lens, head_counts, 0,
                         reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_relayout_head2seq_multi(int n_tensors, const void* const* src, void* const* dst,
                                         usp_dtype_t dt, int B, int H, int D, int P,
                                         const int32_t* seq_lens, const int32_t* head_counts,
                                         usp_stream_t stream) {
  return relayout_public(n_tensors, src, dst, dt, B, H, D, P, seq_lens, head_counts, 1,
                         reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_reorder(const void* src, void* dst, usp_dtype_t dt, int B, int S, int H, int D,
                         int R, usp_order_t order, int inverse, usp_stream_t stream) {
  if (!src || !dst) return fail(USP_ERR_INVALID_ARG, "NULL src or dst");
  if (dt != USP_BF16 && dt != USP_FP32) return fail(USP_ERR_INVALID_ARG, "dt must be BF16 or FP32");
  if (B < 1 || H < 1 || D < 1 || S < 0) return fail(USP_ERR_INVALID_ARG, "need B, H, D >= 1 and S >= 0");
  if (R < 1 || R > kRelayoutMaxR) return fail(USP_ERR_INVALID_ARG, "need 1 <= R <= %d", kRelayoutMaxR);
  if (order != USP_ORDER_CONTIGUOUS && order != USP_ORDER_ZIGZAG && order != USP_ORDER_STRIPE)
    return fail(USP_ERR_INVALID_ARG, "unknown order");
  if (int64_t(B) * S * H * D >= (int64_t(1) << 40)) return fail(USP_ERR_INVALID_ARG, "tensor too large");
  if (S == 0) return USP_OK;
  if (usp_status_t st = check_device()) return st;
  Grid g;
  g.B = B; g.S = S; g.H = H; g.D = D; g.U = 1; g.R = R; g.order = order;
  g.pos = ring_positions(order, S, R);
  g.S_r.resize(R);
  for (int r = 0; r < R; ++r) g.S_r[r] = g.pos[r].rows();
  g.h = {H};
  g.hoff = {0};
  RelayoutParams rp;
  fill_relayout_grid(rp, g, D, dt == USP_BF16 ? 2 : 4);
  rp.src[0] = static_cast<const char*>(src);
  rp.dst[0] = static_cast<char*>(dst);
  rp.n_tensors = 1;
  rp.dir = inverse ? 1 : 0;
  return launch_relayout(rp, reinterpret_cast<cudaStream_t>(stream));
}

static bool positions_ok(const usp_positions_t* p, int rows) {
  if (p->n_seg != 1 && p->n_seg != 2) return false;
  if (p->stride < 1 || p->len[0] < 0) return false;
  if (p->n_seg == 2 && p->len[1] < 0) return false;
  const int64_t total = int64_t(p->len[0]) + (p->n_seg == 2 ? p->len[1] : 0);
  if (total != rows) return false;
  if (p->n_seg == 2 && p->len[0] > 0 && p->len[1] > 0 &&
      int64_t(p->start[1]) <= int64_t(p->start[0]) + int64_t(p->len[0] - 1) * p->stride)
    return false;
  return true;
}

usp_status_t usp_attn_partial(const void* q, const void* k, const void* v, int B, int H, int Sq,
                              int Sk, int D, int64_t q_row_stride, int64_t kv_row_stride,
                              float scale, const usp_positions_t* q_pos,
                              const usp_positions_t* k_pos, void* o, usp_dtype_t o_dt, float* lse,
                              uint32_t* status, usp_stream_t stream) {
  if (!q || !k || !v || !o) return fail(USP_ERR_INVALID_ARG, "NULL q, k, v or o");
  if (B < 1 || H < 1 || Sq < 0 || Sk < 0) return fail(USP_ERR_INVALID_ARG, "need B, H >= 1 and Sq, Sk >= 0");
  if (D != 64 && D != 128) return fail(USP_ERR_UNSUPPORTED, "head dim D=%d: only 64 and 128 are built", D);
  if (o_dt != USP_BF16 && o_dt != USP_FP32) return fail(USP_ERR_INVALID_ARG, "o_dt must be BF16 or FP32");
  if (q_row_stride < int64_t(H) * D || kv_row_stride < int64_t(H) * D ||
      (q_row_stride * 2) % 16 || (kv_row_stride * 2) % 16)
    return fail(USP_ERR_INVALID_ARG, "row strides must be >= H*D and a multiple of 8 elements");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(USP_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if ((q_pos == nullptr) != (k_pos == nullptr))
    return fail(USP_ERR_INVALID_ARG, "give both q_pos and k_pos (causal) or neither");
  if (q_pos && (!positions_ok(q_pos, Sq) || !positions_ok(k_pos, Sk)))
    return fail(USP_ERR_INVALID_ARG, "positions must have 1 or 2 increasing segments covering the chunk");
  if (int64_t(B) * Sq >= INT_MAX / 2 || int64_t(B) * Sk >= INT_MAX / 2)
    return fail(USP_ERR_INVALID_ARG, "too many rows");
  if (Sq == 0) return USP_OK;
  if (usp_status_t st = check_device()) return st;
  static thread_local AttnParams params;
  AttnParams& p = params;
  std::memset(&p, 0, sizeof(p));
  usp_status_t st;
  if ((st = make_qkv_map(&p.maps[0], q, H, D, Sq, 1, B, q_row_stride, 0, int64_t(Sq) * q_row_stride))) return st;
  if ((st = make_qkv_map(&p.maps[1], k, H, D, Sk, 1, B, kv_row_stride, 0, int64_t(Sk) * kv_row_stride))) return st;
  if ((st = make_qkv_map(&p.maps[2], v, H, D, Sk, 1, B, kv_row_stride, 0, int64_t(Sk) * kv_row_stride))) return st;

  p.B = B;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.budget_ns = wait_budget_ns();
  p.withhold_loads = withhold_loads();
  Positions qp, kp;
  if (q_pos) {
    qp.n_seg = q_pos->n_seg; kp.n_seg = k_pos->n_seg;
    for (int i = 0; i < 2; ++i) {
      qp.start[i] = q_pos->start[i]; qp.len[i] = q_pos->len[i];
      kp.start[i] = k_pos->start[i]; kp.len[i] = k_pos->len[i];
    }
    if (qp.n_seg == 1) qp.len[1] = 0;
    if (kp.n_seg == 1) kp.len[1] = 0;
    qp.stride = q_pos->stride; kp.stride = k_pos->stride;
  } else {
    qp.len[0] = Sq;
    kp.len[0] = Sk;
  }
  std::vector<AttnSeg> segs;
  std::vector<AttnLink> links;
  for (const Run& r : plan_runs(qp, kp, q_pos != nullptr)) {
    AttnSeg s{};
    s.o = o; s.lse = lse;
    s.o_bf16 = o_dt == USP_BF16;
    s.q_map = 0;
    s.q_row0 = r.q0; s.q_len = r.q_len;
    s.link0 = static_cast<int>(links.size()); s.n_links = 1;
    links.push_back({1, 2, 0, r.kv_len, r.diag});
    s.n_heads = H;
    s.o_row0 = r.q0; s.o_bstride = Sq; s.o_heads = H;
    s.o_start0 = 0; s.o_len0 = INT_MAX; s.o_start1 = 0; s.o_stride = 1;
    s.rev = q_pos != nullptr;
    segs.push_back(s);
  }
  return launch_attention(p, segs, links, D, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

usp_status_t usp_lse_merge(int n_parts, const float* o_parts, int64_t o_part_stride,
                           const float* lse_parts, int64_t lse_part_stride, int64_t n_rows, int H,
                           int D, void* o_out, usp_dtype_t out_dt, float* lse_out,
                           usp_stream_t stream) {
  if (n_parts < 1 || n_parts > 16) return fail(USP_ERR_INVALID_ARG, "need 1 <= n_parts <= 16");
  if (!o_parts || !lse_parts || !o_out) return fail(USP_ERR_INVALID_ARG, "NULL o_parts, lse_parts or o_out");
  if (H < 1 || n_rows < 0 || D < 4 || D > 256 || D % 4)
    return fail(USP_ERR_INVALID_ARG, "need H >= 1, n_rows >= 0, D a multiple of 4 in [4, 256]");
  if (out_dt != USP_BF16 && out_dt != USP_FP32) return fail(USP_ERR_INVALID_ARG, "out_dt must be BF16 or FP32");
  if (!aligned(o_parts, 16) || !aligned(o_out, out_dt == USP_BF16 ? 8 : 16) || (o_part_stride % 4))
    return fail(USP_ERR_INVALID_ARG, "o_parts and o_out must be vector aligned, o_part_stride a multiple of 4");
  if (n_parts > 1 && (o_part_stride < n_rows * H * D || lse_part_stride < n_rows * H))
    return fail(USP_ERR_INVALID_ARG, "part strides smaller than one part");
  if (n_rows == 0) return USP_OK;
  if (usp_status_t st = check_device()) return st;
  return launch_lse_merge(n_parts, o_parts, o_part_stride, lse_parts, lse_part_stride, n_rows * H, D,
                          o_out, out_dt == USP_BF16, lse_out, nullptr,
                          reinterpret_cast<cudaStream_t>(stream));
}

size_t usp_attention_workspace_size(int B, int S, int H, int D, int causal, int ulysses_degree,
                                    int ring_degree, usp_order_t order, usp_dtype_t o_dt) {
  std::shared_ptr<const PlanEntry> pe;
  if (get_plan(B, S, H, D, causal, ulysses_degree, ring_degree, order, nullptr, nullptr, o_dt, pe) != USP_OK)
    return 0;
  return pe->g.total;
}

static usp_status_t attention_impl(const void* q, const void* k, const void* v, int B, int S, int H,
                                   int D, float scale, int causal, int ulysses_degree,
                                   int ring_degree, const int32_t* seq_lens,
                                   const int32_t* head_counts, usp_order_t order, void* o,
                                   usp_dtype_t o_dt, float* lse, void* workspace,
                                   size_t workspace_bytes, void* const* events, int* launches,
                                   int64_t in_rs, cudaStream_t stream) {
  // in_rs: elements from one token's row of q (k, v) to the next: H*D, or 3*H*D for packed QKV
  int n_launch[4] = {0, 0, 0, 0};
  auto mark = [&](int i) -> usp_status_t {
    if (events && events[i]) {
      cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream);
      if (e != cudaSuccess) return fail(USP_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    }
    return USP_OK;
  };
  if (launches) for (int i = 0; i < 4; ++i) launches[i] = 0;
  if (!q || !k || !v || !o) return fail(USP_ERR_INVALID_ARG, "NULL q, k, v or o");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
    return fail(USP_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  std::shared_ptr<const PlanEntry> pe;
  if (usp_status_t st = get_plan(B, S, H, D, causal, ulysses_degree, ring_degree, order, seq_lens,
                                 head_counts, o_dt, pe))
    return st;
  const Grid& g = pe->g;
  if (!workspace || !aligned(workspace, 256)) return fail(USP_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (workspace_bytes < g.total)
    return fail(USP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, g.total);
  if (S == 0) return USP_OK;
  if (usp_status_t st = check_device()) return st;
  char* ws = static_cast<char*>(workspace);
  const int U = g.U, R = g.R;
  usp_status_t st;

  // The attention launch's parameters are prepared on the host before anything is launched, so
  // that a call failing on the host leaves nothing in the stream.  A thread that repeats its
  // previous call (same plan, buffers and settings) reuses the parameters it built then, without
  // encoding the tensor maps again.
  struct CallMemo {
    std::shared_ptr<const PlanEntry> pe;
    const void *q, *k, *v, *o, *lse, *ws;
    int64_t in_rs;
    float scale;
    unsigned long long budget;
    int withhold;
    std::vector<AttnLaunch> launches;
  };
  static thread_local CallMemo memo;
  const unsigned long long budget = wait_budget_ns();
  const int withhold = withhold_loads();
  const bool partials = R > 1 && !g.fused_ring;
  bool clear_counter = false;
  if (!(memo.pe == pe && memo.q == q && memo.k == k && memo.v == v && memo.o == o &&
        memo.lse == lse && memo.ws == workspace && memo.in_rs == in_rs && memo.scale == scale &&
        memo.budget == budget && memo.withhold == withhold)) {
    memo.pe.reset();
    static thread_local AttnParams params;
    AttnParams& p = params;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < R; ++r) {
      for (int u = 0; u < U; ++u) {
        // virtual rank (r, u)'s head-sharded view, in place: the chunk's rows from its first,
        // heads [hoff_u, hoff_u + h_u)
        int64_t piece_rows = std::max(1, g.S_r[r]), piece_stride = 0;
        int n_pieces = 1;
        const int64_t e0 = int64_t(g.pos[r].start[0]) * in_rs + int64_t(g.hoff[u]) * D;
        const void* base[3] = {static_cast<const uint16_t*>(q) + e0, static_cast<const uint16_t*>(k) + e0,
                               static_cast<const uint16_t*>(v) + e0};
        const int64_t row_stride = int64_t(g.pos[r].stride) * in_rs;
        int64_t batch_stride = int64_t(S) * in_rs;
        if (g.span(r)) {  // zigzag chunk with ragged half-chunks: the span of global rows over both
          piece_rows = g.span_off[r] + g.pos[r].len[1];
        } else if (two_pieces(g.pos[r])) {  // zigzag chunk: its two half-chunks as two pieces
          piece_rows = g.pos[r].len[0];
          n_pieces = 2;
          piece_stride = int64_t(g.pos[r].start[1] - g.pos[r].start[0]) * in_rs;
        }
        if (B == 1) batch_stride = piece_rows * n_pieces * row_stride;
        for (int t = 0; t < 3; ++t) {
          const int mi = map_index(g, r, u, t);
          if ((st = make_qkv_map(&p.maps[mi], base[t], g.h[u], D, piece_rows, n_pieces, B, row_stride,
                                 piece_stride, batch_stride)))
            return st;
          p.map_rows[mi] = n_pieces > 1 ? static_cast<int>(piece_rows) : 0;
        }
      }
    }
    p.B = B;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = reinterpret_cast<uint32_t*>(ws);
    p.counter = reinterpret_cast<uint32_t*>(ws) + 2;  // bytes 8-15: the dynamic deal's counter
    p.budget_ns = budget;
    p.withhold_loads = withhold;
    // the cached plan's segments, bound to this call's output and workspace
    std::vector<AttnSeg> segs = pe->plan.segs;
    for (size_t i = 0; i < segs.size(); ++i) {
      const SegOut& so = pe->plan.outs[i];
      segs[i].o_bf16 = !so.partial && o_dt == USP_BF16;
      if (so.partial) {
        segs[i].o = ws + so.o_off;
        segs[i].lse = reinterpret_cast<float*>(ws + so.lse_off);
      } else {
        segs[i].o = static_cast<char*>(o) + so.o_off;
        segs[i].lse = lse ? reinterpret_cast<float*>(reinterpret_cast<char*>(lse) + so.lse_off) : nullptr;
      }
    }
    if ((st = pack_attention(p, segs, pe->plan.links, memo.launches))) return st;
    memo.pe = pe;
    memo.q = q; memo.k = k; memo.v = v; memo.o = o; memo.lse = lse; memo.ws = workspace;
    memo.in_rs = in_rs; memo.scale = scale; memo.budget = budget; memo.withhold = withhold;
    for (const AttnLaunch& L : memo.launches) clear_counter = clear_counter || (L.params.deal & kDealDynamic);
  }
  // A dynamic deal's counter returns to zero at the end of every launch; it is set to zero here
  // whenever this thread binds a new plan or workspace, so a workspace whose bytes 8-15 were not
  // zeroed still starts from zero.
  if (clear_counter) {
    const cudaError_t e = cudaMemsetAsync(ws + 8, 0, 8, stream);
    if (e != cudaSuccess) return fail(USP_ERR_CUDA, "clearing the unit counter: %s", cudaGetErrorString(e));
  }
  if ((st = mark(0))) return st;

  // 1. Q, K, V of virtual rank (r, u) are read in place (the first all-to-all and the reorder are
  //    the tensor maps' addressing): no pass.
  if ((st = mark(1))) return st;

  // 2. attention over every (Ulysses rank, q ring chunk, ring step) pair in one launch: one
  //    segment per chunk pair (ring partials or, with one ring rank, the final output), or one
  //    chain per piece of query rows across all ring steps (fused ring: the final output).
  if ((st = run_attention(memo.launches, D, stream))) return st;
  n_launch[1] = static_cast<int>(memo.launches.size());
  if ((st = mark(2))) return st;

  // 3. merge the ring partials straight into the global layout (the head -> seq all-to-all and the
  //    inverse reorder are the merge's store addressing)
  if (partials) {
    MergeMap mm;
    std::memset(&mm, 0, sizeof(mm));
    mm.n_blocks = R * U;
    mm.H = H;
    mm.S = S;
    for (int r = 0; r < R; ++r) {
      for (int u = 0; u < U; ++u) {
        const int kb = r * U + u;
        mm.vec0[kb] = g.woff(r, u, 1);
        mm.row0[kb] = kb == 0 ? 0 : mm.row0[kb - 1] + int64_t(B) * g.S_r[(kb - 1) / U];
        mm.S_r[kb] = std::max(1, g.S_r[r]);
        mm.h[kb] = g.h[u];
        mm.hoff[kb] = g.hoff[u];
        mm.p_start0[kb] = g.pos[r].start[0];
        mm.p_len0[kb] = g.pos[r].n_seg > 1 ? g.pos[r].len[0] : INT_MAX;
        mm.p_start1[kb] = g.pos[r].start[1];
        mm.p_stride[kb] = g.pos[r].stride;
      }
    }
    mm.all_seen = causal ? 0 : 1;
    mm.vec0[R * U] = int64_t(B) * S * H;
    mm.row0[R * U] = mm.row0[R * U - 1] + int64_t(B) * g.S_r[R - 1];
    if ((st = launch_lse_merge(R, reinterpret_cast<const float*>(ws + g.off_opart), g.elems,
                               reinterpret_cast<const float*>(ws + g.off_lpart), int64_t(B) * S * H,
                               int64_t(B) * S * H, D, o, o_dt == USP_BF16, lse, &mm, stream)))
      return st;
    ++n_launch[2];
  }
  // 3'. a split fused ring: merge the split rows' partials into the global layout (the rows
  //    [split_row, S_r) of ring chunk split_r, heads of Ulysses group split_u)
  if (g.split_r >= 0) {
    const Positions& ps = g.pos[g.split_r];
    const int c = g.split_row;
    MergeMap mm;
    std::memset(&mm, 0, sizeof(mm));
    mm.n_blocks = 1;
    mm.H = H;
    mm.S = S;
    mm.vec0[0] = 0;
    mm.vec0[1] = g.split_vec();
    mm.row0[0] = 0;
    mm.row0[1] = int64_t(B) * g.split_rows();
    mm.S_r[0] = std::max(1, g.split_rows());
    mm.h[0] = g.h[g.split_u];
    mm.hoff[0] = g.hoff[g.split_u];
    if (ps.n_seg > 1 && c >= ps.len[0]) {  // the split rows lie in the second piece
      mm.p_start0[0] = ps.start[1] + (c - ps.len[0]) * ps.stride;
      mm.p_len0[0] = INT_MAX;
    } else {
      mm.p_start0[0] = ps.start[0] + c * ps.stride;
      mm.p_len0[0] = ps.n_seg > 1 ? ps.len[0] - c : INT_MAX;
      mm.p_start1[0] = ps.start[1];
    }
    mm.p_stride[0] = ps.stride;
    mm.all_seen = causal ? 0 : 1;
    const int64_t vec = g.split_vec();
    if ((st = launch_lse_merge(R, reinterpret_cast<const float*>(ws + g.off_spart), vec * D,
                               reinterpret_cast<const float*>(ws + g.off_slpart), vec, vec, D, o,
                               o_dt == USP_BF16, lse, &mm, stream)))
      return st;
    ++n_launch[2];
  }
  if ((st = mark(3))) return st;
  if ((st = mark(4))) return st;
  if (launches) for (int i = 0; i < 4; ++i) launches[i] = n_launch[i];
  return USP_OK;
}

usp_status_t usp_attention(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                           float scale, int causal, int ulysses_degree, int ring_degree,
                           const int32_t* seq_lens, const int32_t* head_counts, usp_order_t order,
                           void* o, usp_dtype_t o_dt, float* lse, void* workspace,
                           size_t workspace_bytes, usp_stream_t stream) {
  return attention_impl(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, seq_lens,
                        head_counts, order, o, o_dt, lse, workspace, workspace_bytes, nullptr,
                        nullptr, int64_t(H) * D, reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_attention_qkvpacked(const void* qkv, int B, int S, int H, int D, float scale,
                                     int causal, int ulysses_degree, int ring_degree,
                                     const int32_t* seq_lens, const int32_t* head_counts,
                                     usp_order_t order, void* o, usp_dtype_t o_dt, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     usp_stream_t stream) {
  if (!qkv) return fail(USP_ERR_INVALID_ARG, "NULL qkv");
  const int64_t hd = int64_t(std::max(H, 0)) * std::max(D, 0);
  const uint16_t* base = static_cast<const uint16_t*>(qkv);
  return attention_impl(base, base + hd, base + 2 * hd, B, S, H, D, scale, causal, ulysses_degree,
                        ring_degree, seq_lens, head_counts, order, o, o_dt, lse, workspace,
                        workspace_bytes, nullptr, nullptr, 3 * hd,
                        reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_attention_events(const void* q, const void* k, const void* v, int B, int S, int H,
                                  int D, float scale, int causal, int ulysses_degree,
                                  int ring_degree, const int32_t* seq_lens,
                                  const int32_t* head_counts, usp_order_t order, void* o,
                                  usp_dtype_t o_dt, float* lse, void* workspace,
                                  size_t workspace_bytes, void* const* events, int* launches,
                                  usp_stream_t stream) {
  return attention_impl(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, seq_lens,
                        head_counts, order, o, o_dt, lse, workspace, workspace_bytes, events,
                        launches, int64_t(H) * D, reinterpret_cast<cudaStream_t>(stream));
}

int usp_attention_ring_mode(int B, int S, int H, int D, int causal, int ulysses_degree,
                            int ring_degree, usp_order_t order, usp_dtype_t o_dt) {
  std::shared_ptr<const PlanEntry> pe;
  if (get_plan(B, S, H, D, causal, ulysses_degree, ring_degree, order, nullptr, nullptr, o_dt, pe) != USP_OK)
    return -1;
  return pe->g.R == 1 ? 0 : (pe->g.fused_ring ? 2 : 1);
}

int usp_plan_deals(int B, int S, int H, int D, int causal, int ulysses_degree, int ring_degree,
                   usp_order_t order, usp_dtype_t o_dt, int sms, int32_t* out, int cap) {
  if (sms < 1) {
    fail(USP_ERR_INVALID_ARG, "need sms >= 1");
    return -1;
  }
  std::shared_ptr<const PlanEntry> pe;
  if (get_plan(B, S, H, D, causal, ulysses_degree, ring_degree, order, nullptr, nullptr, o_dt, pe) != USP_OK)
    return -1;
  std::vector<AttnSeg> segs = pe->plan.segs;
  for (size_t i = 0; i < segs.size(); ++i) segs[i].o_bf16 = !pe->plan.outs[i].partial && o_dt == USP_BF16;
  AttnParams base;
  std::memset(&base, 0, sizeof(base));
  base.B = B;
  base.scale_log2 = 1.f;
  static uint32_t no_counter[2];  // usp_attention has a counter, so dynamic deals are allowed; never read
  base.counter = no_counter;
  std::vector<AttnLaunch> launches;
  if (pack_attention(base, segs, pe->plan.links, launches, sms) != USP_OK) return -1;
  const int n = static_cast<int>(launches.size());
  for (int i = 0; i < n && out && i < cap; ++i) {
    const AttnParams& p = launches[i].params;
    const int ctas = std::max(1, std::min(p.n_units, sms));
    int32_t* rec = out + 4 * i;
    rec[0] = p.n_units;
    rec[1] = p.deal;
    rec[2] = static_cast<int32_t>(std::lround(1000.0 * deal_periods(p, p.deal, ctas)));
    rec[3] = static_cast<int32_t>(std::lround(1000.0 * deal_periods(p, 0, ctas)));
  }
  return n;
}

usp_status_t usp_check_status(void* status, usp_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
  if (!status) return USP_OK;
  uint32_t word = 0;
  e = cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(USP_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (word) {
    e = cudaMemset(status, 0, sizeof(word));
    if (e != cudaSuccess) return fail(USP_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
    return fail(USP_ERR_TIMEOUT, "a bounded device wait gave up (status 0x%x)", word);
  }
  return USP_OK;
}

int usp_plan_pairs(int S, int ulysses_degree, int ring_degree, int causal, usp_order_t order,
                   int32_t* out, int cap) {
  std::shared_ptr<const PlanEntry> pe;
  if (get_plan(1, S, std::max(1, ulysses_degree), 64, causal, ulysses_degree, ring_degree, order,
               nullptr, nullptr, USP_FP32, pe) != USP_OK)
    return -1;
  const Grid& g = pe->g;
  int n = 0;
  for (int u = 0; u < g.U; ++u) {
    for (int r = 0; r < g.R; ++r) {
      for (int kstep = 0; kstep < g.R; ++kstep) {
        const int r2 = (r - kstep + g.R) % g.R;
        for (const Run& run : plan_runs(g.pos[r], g.pos[r2], causal != 0)) {
          if (out && n < cap) {
            int32_t* rec = out + 8 * n;
            rec[0] = u; rec[1] = r; rec[2] = kstep; rec[3] = r2;
            rec[4] = run.q0; rec[5] = run.q_len; rec[6] = run.kv_len; rec[7] = run.diag;
          }
          ++n;
        }
      }
    }
  }
  return n;
}

int usp_plan_chains(int S, int ulysses_degree, int ring_degree, int causal, usp_order_t order,
                    int32_t* out, int cap) {
  Grid g;
  if (build_grid(g, 1, S, std::max(1, ulysses_degree), 64, causal, ulysses_degree, ring_degree,
                 order, nullptr, nullptr, USP_FP32) != USP_OK)
    return -1;
  AttnPlan pl;
  if (plan_fused(g, 4, pl) != USP_OK) return -1;
  // one record per (piece, ring step): the two links of a span-mapped K/V chunk (its half-chunks)
  // are reported as the one key range [0, kv_len) of the chunk they split
  int n = 0;
  for (const AttnSeg& s : pl.segs) {
    const int r = s.q_map / (3 * g.U), u = (s.q_map / 3) % g.U;
    for (int i = 0; i < s.n_links;) {
      const AttnLink& lk = pl.links[s.link0 + i];
      const int r2 = lk.k_map / (3 * g.U);
      int kv_len = lk.kv_len, j = i + 1;
      for (; j < s.n_links && pl.links[s.link0 + j].k_map == lk.k_map; ++j) kv_len += pl.links[s.link0 + j].kv_len;
      if (out && n < cap) {
        int32_t* rec = out + 8 * n;
        // chunk-local first row (a split segment's o_row0 counts from the split row)
        rec[0] = u; rec[1] = r; rec[2] = s.grp == g.U ? g.split_row + s.o_row0 : s.o_row0;
        rec[3] = s.q_len;
        rec[4] = (r - r2 + g.R) % g.R; rec[5] = r2; rec[6] = kv_len; rec[7] = lk.diag;
      }
      ++n;
      i = j;
    }
  }
  return n;
}

const char* usp_status_string(usp_status_t s) {
  switch (s) {
    case USP_OK: return "ok";
    case USP_ERR_INVALID_ARG: return "invalid argument";
    case USP_ERR_UNSUPPORTED: return "unsupported";
    case USP_ERR_CUDA: return "CUDA error";
    case USP_ERR_TIMEOUT: return "device wait timed out";
    case USP_ERR_WORKSPACE: return "workspace missing or too small";
    case USP_ERR_NO_DEVICE: return "no sm_103 device";
  }
  return "unknown status";
}

const char* usp_last_error(void) { return g_last_error.c_str(); }

int usp_version(void) { return 100; }

}  // extern "C"
