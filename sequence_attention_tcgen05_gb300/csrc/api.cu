// C ABI entry points: argument validation, the chunk-pair planner, workspace layout and the
// launch sequence of usp_attention.  Nothing here allocates device memory or synchronises,
// except usp_check_status.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
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
  usp_order_t order = USP_ORDER_CONTIGUOUS;
  std::vector<Positions> pos;  // per ring group
  std::vector<int> S_r;        // ring chunk lengths
  std::vector<int> h, hoff;    // head groups
  // Q/K/V of every virtual rank can be addressed in place in the global tensor (each ring chunk is
  // one affine run of rows, or two equal half-chunks of whole 128-row tiles under zigzag); otherwise
  // they are first re-laid into the head-sharded workspace copies.
  bool fused_in = true;
  // workspace layout (bytes)
  size_t off_q = 0, off_k = 0, off_v = 0, off_opart = 0, off_lpart = 0, total = 0;
  int64_t elems = 0;  // B*S*H*D
  int64_t woff(int r, int u, int d) const {  // element offset of block (r, u) in the W layout
    int64_t off = 0;
    for (int rr = 0; rr < r; ++rr) off += int64_t(B) * S_r[rr] * H * d;
    for (int uu = 0; uu < u; ++uu) off += int64_t(B) * S_r[r] * h[uu] * d;
    return off;
  }
};

usp_status_t build_grid(Grid& g, int B, int S, int H, int D, int U, int R, usp_order_t order,
                        const int32_t* seq_lens, const int32_t* head_counts, usp_dtype_t o_dt) {
  if (B < 1 || S < 0 || H < 1) return fail(USP_ERR_INVALID_ARG, "need B >= 1, S >= 0, H >= 1");
  if (D != 64 && D != 128) return fail(USP_ERR_UNSUPPORTED, "head dim D=%d: only 64 and 128 are built", D);
  if (U < 1 || R < 1 || U > 16 || R > 16 || U * R > 16)
    return fail(USP_ERR_INVALID_ARG, "need 1 <= ulysses_degree, ring_degree and their product <= 16");
  if (order != USP_ORDER_CONTIGUOUS && order != USP_ORDER_ZIGZAG && order != USP_ORDER_STRIPE)
    return fail(USP_ERR_INVALID_ARG, "unknown order %d", static_cast<int>(order));
  if (o_dt != USP_BF16 && o_dt != USP_FP32) return fail(USP_ERR_INVALID_ARG, "o_dt must be BF16 or FP32");
  if (int64_t(B) * S * H * D >= (int64_t(1) << 40)) return fail(USP_ERR_INVALID_ARG, "tensor too large");
  g.B = B; g.S = S; g.H = H; g.D = D; g.U = U; g.R = R; g.order = order;
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
  // Q/K/V are addressed in place unless a zigzag chunk's two half-chunks differ in length or are not
  // whole 128-row tiles (a tile must not straddle them); then they are re-laid into the workspace.
  g.fused_in = true;
  for (int r = 0; r < R; ++r) {
    const Positions& ps = g.pos[r];
    if (two_pieces(ps) && !(ps.len[0] == ps.len[1] && ps.len[0] % kAttnBM == 0)) g.fused_in = false;
  }
  g.elems = int64_t(B) * S * H * D;
  const int64_t rowsH = int64_t(B) * S * H;
  size_t at = 256;  // status word
  auto take = [&](size_t bytes) {
    const size_t o = at;
    at = static_cast<size_t>(align_up(static_cast<int64_t>(at + bytes), 256));
    return o;
  };
  if (!g.fused_in) {
    g.off_q = take(g.elems * 2);
    g.off_k = take(g.elems * 2);
    g.off_v = take(g.elems * 2);
  }
  if (R > 1) {
    g.off_opart = take(size_t(R) * g.elems * 4);
    g.off_lpart = take(size_t(R) * rowsH * 4);
  }
  g.total = at;
  return USP_OK;
}

void fill_relayout_grid(RelayoutParams& rp, const Grid& g, int d, int elem) {
  std::memset(&rp, 0, sizeof(rp));
  rp.B = g.B; rp.H = g.H; rp.D = d; rp.elem = elem; rp.R = g.R; rp.U = g.U;
  rp.seq_mode = 1; rp.S = g.S;
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

usp_status_t relayout_public(const void* src, void* dst, usp_dtype_t dt, int B, int H, int D, int P,
                             const int32_t* seq_lens, const int32_t* head_counts, int dir,
                             cudaStream_t stream) {
  if (!src || !dst || !seq_lens) return fail(USP_ERR_INVALID_ARG, "NULL src, dst or seq_lens");
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
  rp.src[0] = static_cast<const char*>(src);
  rp.dst[0] = static_cast<char*>(dst);
  rp.n_tensors = 1;
  rp.B = B; rp.H = H; rp.D = D; rp.elem = elem; rp.R = 1; rp.U = P;
  rp.seq_mode = 0; rp.dir = dir; rp.S = static_cast<int>(S);
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
  return relayout_public(src, dst, dt, B, H, D, P, seq_lens, head_counts, 0,
                         reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_relayout_head2seq(const void* src, void* dst, usp_dtype_t dt, int B, int H, int D,
                                   int P, const int32_t* seq_lens, const int32_t* head_counts,
                                   usp_stream_t stream) {
  return relayout_public(src, dst, dt, B, H, D, P, seq_lens, head_counts, 1,
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
  p.o_bf16 = o_dt == USP_BF16;
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
  for (const Run& r : plan_runs(qp, kp, q_pos != nullptr)) {
    AttnSeg s{};
    s.o = o; s.lse = lse;
    s.q_map = 0; s.k_map = 1; s.v_map = 2;
    s.q_row0 = r.q0; s.q_len = r.q_len;
    s.kv_row0 = 0; s.kv_len = r.kv_len;
    s.diag = r.diag; s.n_heads = H;
    s.o_row0 = r.q0; s.o_bstride = Sq; s.o_heads = H;
    s.o_start0 = 0; s.o_len0 = INT_MAX; s.o_start1 = 0; s.o_stride = 1;
    s.rev = q_pos != nullptr;
    segs.push_back(s);
  }
  return launch_attention(p, segs, D, reinterpret_cast<cudaStream_t>(stream));
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

size_t usp_attention_workspace_size(int B, int S, int H, int D, int ulysses_degree,
                                    int ring_degree, usp_order_t order, usp_dtype_t o_dt) {
  Grid g;
  if (build_grid(g, B, S, H, D, ulysses_degree, ring_degree, order, nullptr, nullptr, o_dt) != USP_OK)
    return 0;
  return g.total;
}

static usp_status_t attention_impl(const void* q, const void* k, const void* v, int B, int S, int H,
                                   int D, float scale, int causal, int ulysses_degree,
                                   int ring_degree, const int32_t* seq_lens,
                                   const int32_t* head_counts, usp_order_t order, void* o,
                                   usp_dtype_t o_dt, float* lse, void* workspace,
                                   size_t workspace_bytes, void* const* events, int* n_launches,
                                   cudaStream_t stream) {
  int launches = 0;
  auto mark = [&](int i) -> usp_status_t {
    if (events && events[i]) {
      cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream);
      if (e != cudaSuccess) return fail(USP_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    }
    return USP_OK;
  };
  if (n_launches) *n_launches = 0;
  if (!q || !k || !v || !o) return fail(USP_ERR_INVALID_ARG, "NULL q, k, v or o");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || (lse && !aligned(lse, 4)))
    return fail(USP_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  Grid g;
  if (usp_status_t st = build_grid(g, B, S, H, D, ulysses_degree, ring_degree, order, seq_lens,
                                   head_counts, o_dt))
    return st;
  if (!workspace || !aligned(workspace, 256)) return fail(USP_ERR_WORKSPACE, "workspace NULL or not 256-byte aligned");
  if (workspace_bytes < g.total)
    return fail(USP_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, g.total);
  if (S == 0) return USP_OK;
  if (usp_status_t st = check_device()) return st;
  if (usp_status_t st = mark(0)) return st;
  char* ws = static_cast<char*>(workspace);
  const int U = g.U, R = g.R;
  const int oel = o_dt == USP_BF16 ? 2 : 4;
  usp_status_t st;

  // 1. Q, K, V of virtual rank (r, u): in place in the global tensor when ring chunk r is one affine
  //    run of rows (the head-sharded view is then pure addressing); otherwise a fused reorder +
  //    seq -> head re-layout into the workspace first.
  if (!g.fused_in) {
    RelayoutParams rp;
    fill_relayout_grid(rp, g, D, 2);
    rp.n_tensors = 3;
    rp.src[0] = static_cast<const char*>(q); rp.dst[0] = ws + g.off_q;
    rp.src[1] = static_cast<const char*>(k); rp.dst[1] = ws + g.off_k;
    rp.src[2] = static_cast<const char*>(v); rp.dst[2] = ws + g.off_v;
    rp.dir = 0;
    if ((st = launch_relayout(rp, stream))) return st;
    ++launches;
  }
  if ((st = mark(1))) return st;

  // 2. partial attention over every (Ulysses rank, q ring chunk, ring step) pair in one launch
  static thread_local AttnParams params;
  AttnParams& p = params;
  std::memset(&p, 0, sizeof(p));
  auto map_index = [&](int r, int u, int t) { return (r * U + u) * 3 + t; };
  for (int r = 0; r < R; ++r) {
    for (int u = 0; u < U; ++u) {
      const void* base[3];
      int64_t row_stride, batch_stride;
      int64_t piece_rows = std::max(1, g.S_r[r]), piece_stride = 0;
      int n_pieces = 1;
      if (g.fused_in) {
        const int64_t e0 = (int64_t(g.pos[r].start[0]) * H + g.hoff[u]) * D;
        base[0] = static_cast<const uint16_t*>(q) + e0;
        base[1] = static_cast<const uint16_t*>(k) + e0;
        base[2] = static_cast<const uint16_t*>(v) + e0;
        row_stride = int64_t(g.pos[r].stride) * H * D;
        batch_stride = int64_t(S) * H * D;
        if (two_pieces(g.pos[r])) {  // zigzag chunk: its two half-chunks
          piece_rows = g.pos[r].len[0];
          n_pieces = 2;
          piece_stride = int64_t(g.pos[r].start[1] - g.pos[r].start[0]) * H * D;
        }
      } else {
        const int64_t off = g.woff(r, u, D) * 2;
        base[0] = ws + g.off_q + off;
        base[1] = ws + g.off_k + off;
        base[2] = ws + g.off_v + off;
        row_stride = int64_t(g.h[u]) * D;
        batch_stride = int64_t(g.S_r[r]) * row_stride;
      }
      if (B == 1) batch_stride = std::max<int64_t>(1, g.S_r[r]) * row_stride;
      for (int t = 0; t < 3; ++t) {
        if ((st = make_qkv_map(&p.maps[map_index(r, u, t)], base[t], g.h[u], D, piece_rows, n_pieces, B,
                               row_stride, piece_stride, batch_stride)))
          return st;
        p.map_rows[map_index(r, u, t)] = n_pieces > 1 ? static_cast<int>(piece_rows) : 0;
      }
    }
  }
  p.B = B;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = reinterpret_cast<uint32_t*>(ws);
  p.budget_ns = wait_budget_ns();
  p.withhold_loads = withhold_loads();
  // ring partials (fp32, head-sharded W layout) when R > 1; else the final output in place
  const int64_t slot_o = g.elems * 4, slot_l = int64_t(B) * S * H;
  p.o_bf16 = R > 1 ? 0 : (o_dt == USP_BF16);
  std::vector<AttnSeg> segs;
  for (int r = 0; r < R; ++r) {
    for (int kstep = 0; kstep < R; ++kstep) {
      const int r2 = (r - kstep + R) % R;
      const std::vector<Run> runs = plan_runs(g.pos[r], g.pos[r2], causal != 0);
      // a zigzag chunk addressed in place is two maps' worth of pieces: every run must start on a
      // 128-row tile so that no tile straddles its half-chunks (runs start at 0 or at the second
      // half for these orderings)
      if (g.fused_in && two_pieces(g.pos[r]))
        for (const Run& run : runs)
          if (run.q0 % kAttnBM != 0)
            return fail(USP_ERR_UNSUPPORTED, "zigzag run at row %d does not start on a 128-row tile", run.q0);
      for (int u = 0; u < U; ++u) {
        for (const Run& run : runs) {
          AttnSeg s{};
          s.q_map = map_index(r, u, 0);
          s.k_map = map_index(r2, u, 1);
          s.v_map = map_index(r2, u, 2);
          s.q_row0 = run.q0; s.q_len = run.q_len;
          s.kv_row0 = 0; s.kv_len = run.kv_len;
          s.diag = run.diag; s.n_heads = g.h[u];
          s.o_row0 = run.q0;
          s.rev = causal != 0;
          if (R > 1) {
            s.o = ws + g.off_opart + kstep * slot_o + g.woff(r, u, D) * 4;
            s.lse = reinterpret_cast<float*>(ws + g.off_lpart) + kstep * slot_l + g.woff(r, u, 1);
            s.o_bstride = g.S_r[r]; s.o_heads = g.h[u];
            s.o_start0 = 0; s.o_len0 = INT_MAX; s.o_start1 = 0; s.o_stride = 1;
          } else {
            s.o = static_cast<char*>(o) + int64_t(g.hoff[u]) * D * oel;
            s.lse = lse ? lse + g.hoff[u] : nullptr;
            s.o_bstride = S; s.o_heads = H;
            s.o_start0 = g.pos[r].start[0]; s.o_len0 = g.pos[r].n_seg > 1 ? g.pos[r].len[0] : INT_MAX;
            s.o_start1 = g.pos[r].start[1]; s.o_stride = g.pos[r].stride;
          }
          segs.push_back(s);
        }
      }
    }
  }
  if ((st = launch_attention(p, segs, D, stream))) return st;
  launches += static_cast<int>((segs.size() + kAttnMaxSegs - 1) / kAttnMaxSegs);
  if ((st = mark(2))) return st;

  // 3. merge the ring partials straight into the global layout (the head -> seq all-to-all and the
  //    inverse reorder are the merge's store addressing)
  if (R > 1) {
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
    ++launches;
  }
  if ((st = mark(3))) return st;
  if ((st = mark(4))) return st;
  if (n_launches) *n_launches = launches;
  return USP_OK;
}

usp_status_t usp_attention(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                           float scale, int causal, int ulysses_degree, int ring_degree,
                           const int32_t* seq_lens, const int32_t* head_counts, usp_order_t order,
                           void* o, usp_dtype_t o_dt, float* lse, void* workspace,
                           size_t workspace_bytes, usp_stream_t stream) {
  return attention_impl(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, seq_lens,
                        head_counts, order, o, o_dt, lse, workspace, workspace_bytes, nullptr,
                        nullptr, reinterpret_cast<cudaStream_t>(stream));
}

usp_status_t usp_attention_events(const void* q, const void* k, const void* v, int B, int S, int H,
                                  int D, float scale, int causal, int ulysses_degree,
                                  int ring_degree, const int32_t* seq_lens,
                                  const int32_t* head_counts, usp_order_t order, void* o,
                                  usp_dtype_t o_dt, float* lse, void* workspace,
                                  size_t workspace_bytes, void* const* events, int* n_launches,
                                  usp_stream_t stream) {
  return attention_impl(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, seq_lens,
                        head_counts, order, o, o_dt, lse, workspace, workspace_bytes, events,
                        n_launches, reinterpret_cast<cudaStream_t>(stream));
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
  Grid g;
  if (build_grid(g, 1, S, std::max(1, ulysses_degree), 64, ulysses_degree, ring_degree, order,
                 nullptr, nullptr, USP_FP32) != USP_OK)
    return -1;
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
