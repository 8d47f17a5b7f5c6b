/*
 * usp.h — C ABI of libusp_gb300.so: context-parallel exact softmax attention with all
 * sequence chunks ("virtual ranks") on one NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (web pages on context parallelism):
 *   [UAA]   diffusers issue #12706, "UAA: Ulysses Anything Attention" — Ulysses with arbitrary
 *           per-rank sequence lengths, no padding, per-rank seq_len gathered on the host.
 *   [CP]    Hugging Face diffusers docs, "Context parallelism" — sections Ring Attention,
 *           Ulysses Attention, Unified Attention, Ulysses Anything Attention, Ring Anything.
 *   [USP]   diffusers PR #12693, "Add Unified Sequence Parallel attention" — the ring step's
 *           (out, lse) merge and the lse layout (B, S, H_LOCAL).
 *   [YC]    sourcepulse summary of USP / yunchang, "Highlighted Details" — ring orderings
 *           "basic" (contiguous), "zigzag" and "stripe".
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major.  Q, K, V, O are [B][S][H][D]; the log-sum-exp (LSE) is fp32
 *     [B][S][H], natural log, softmax scale included ([USP]: "the lse is of shape
 *     (B, S, H_LOCAL)").
 *   - All pointers named src/dst/q/k/v/o/lse/workspace/status are DEVICE pointers owned by the
 *     caller.  seq_lens, head_counts and usp_positions_t are HOST memory, read during the call
 *     only ([UAA]: the per-rank lengths travel on the host, which avoids forced device syncs).
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream) and never
 *     synchronises the host with the device, except usp_check_status.
 *   - The library allocates no device memory (usp_attention_noalloc's scratch is a static array
 *     compiled into the library).  On the host it caches the plans of recent argument sets
 *     (thread-safe); calls on different streams are independent if their buffers are.
 *   - Errors are return codes; usp_last_error() gives a thread-local message for the last
 *     failing call of the calling thread.  Argument and workspace errors are found before
 *     anything is launched (except that usp_attention_noalloc has cleared its status word when
 *     a plan exceeds this library's limits); a CUDA error from a launch leaves the call's earlier
 *     launches in the stream.
 *   - Stream order holds for every kernel.  The re-layout and merge kernels use programmatic
 *     dependent launch: they may be scheduled while the previous kernel of the stream drains,
 *     but touch no memory before it has completed.
 *   - Head dimension D must be 64 or 128 for attention; re-layout accepts any D >= 1.
 */
#ifndef USP_GB300_H
#define USP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (declared here without including the CUDA headers). */
typedef struct CUstream_st* usp_stream_t;

typedef enum usp_status {
  USP_OK = 0,
  USP_ERR_INVALID_ARG = 1, /* bad size, split, pointer alignment or NULL pointer */
  USP_ERR_UNSUPPORTED = 2, /* valid request this library does not implement (e.g. D = 96) */
  USP_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed (launch, tensor-map encode) */
  USP_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (from usp_check_status) */
  USP_ERR_WORKSPACE = 5,   /* workspace NULL, misaligned or smaller than required */
  USP_ERR_NO_DEVICE = 6    /* the current device is not an sm_103 GPU */
} usp_status_t;

typedef enum usp_dtype { USP_BF16 = 0, USP_FP32 = 1 } usp_dtype_t;

/* Ring chunk ordering [YC].  Readings (the pages name them without a definition):
 *   CONTIGUOUS: ring rank r holds piece r of the default split of S into R pieces.
 *   ZIGZAG:     split S into 2R pieces (default split); rank r holds piece r then piece 2R-1-r.
 *   STRIPE:     token t goes to rank t mod R, local index t / R.
 * Default split of n items into P parts: part p has floor(n/P) + (p < n mod P) items. */
typedef enum usp_order {
  USP_ORDER_CONTIGUOUS = 0,
  USP_ORDER_ZIGZAG = 1,
  USP_ORDER_STRIPE = 2
} usp_order_t;

/* Global token positions of a chunk's rows, used by the causal mask: row i of the chunk has
 * position start[0] + i*stride for i < len[0], else start[1] + (i - len[0])*stride.
 * n_seg is 1 or 2.  Positions must increase with the row index.  This covers a contiguous chunk
 * (1 segment, stride 1), a zigzag chunk (2 segments) and a stripe chunk (stride R). */
typedef struct usp_positions {
  int32_t n_seg;
  int32_t start[2];
  int32_t len[2];
  int32_t stride;
} usp_positions_t;

/* ---------------------------------------------------------------------------------------------
 * usp_relayout_seq2head — the first Ulysses all-to-all as a local permutation.
 * [CP] Ulysses Attention: the first all-to-all regroups the data so that each rank holds every
 * token for a subset of heads.  [UAA]: per-rank lengths are arbitrary and nothing is padded.
 *
 *   src: P sequence chunks back to back; chunk q is [B][seq_lens[q]][H][D].
 *   dst: P head-sharded buffers back to back; buffer p is [B][S][head_counts[p]][D] with
 *        S = sum(seq_lens), and dst_p[b][o_q + t][h][d] = src_q[b][t][g_p + h][d] where
 *        o_q = sum of seq_lens before q and g_p = sum of head_counts before p.
 *   dt: element type (2-byte BF16 or 4-byte FP32; the copy is bit-exact either way).
 *   seq_lens: host int32[P], each >= 0.  head_counts: host int32[P], each >= 1, summing to H, or
 *   NULL for the default split of H over P (ranks may then hold different head counts: [CP]
 *   Ulysses Anything Attention removes the head-divisibility requirement).
 *   1 <= P <= 64.  src and dst must not overlap.
 *   Errors: INVALID_ARG for P out of range, B/H/D < 1, a negative length, head counts not
 *   summing to H, H < P with head_counts NULL, NULL buffers.
 * ------------------------------------------------------------------------------------------- */
usp_status_t usp_relayout_seq2head(const void* src, void* dst, usp_dtype_t dt, int B, int H, int D,
                                   int P, const int32_t* seq_lens, const int32_t* head_counts,
                                   usp_stream_t stream);

/* usp_relayout_head2seq — the second Ulysses all-to-all, the exact inverse of seq2head: src is
 * the P head-sharded buffers, dst the P sequence chunks (same layouts and arguments as above).
 * [CP] Ulysses Attention: a second all-to-all regroups the results by token; [USP] sends the
 * lse through the same exchange (use dt = USP_FP32 and D = 1 for an LSE [B][S][H]). */
usp_status_t usp_relayout_head2seq(const void* src, void* dst, usp_dtype_t dt, int B, int H, int D,
                                   int P, const int32_t* seq_lens, const int32_t* head_counts,
                                   usp_stream_t stream);

/* The same two re-layouts for n_tensors (1..3) tensors of one shape in ONE launch — Q, K and V
 * before the attention ([CP] Ulysses Attention: the first all-to-all moves the query, key and
 * value projections), or O and a second output after it.  src and dst are HOST arrays of
 * n_tensors device pointers, read during the call; tensor t moves from src[t] to dst[t] exactly
 * as in usp_relayout_seq2head / usp_relayout_head2seq.  Errors: as those, plus INVALID_ARG for
 * n_tensors outside [1, 3] or a NULL entry. */
usp_status_t usp_relayout_seq2head_multi(int n_tensors, const void* const* src, void* const* dst,
                                         usp_dtype_t dt, int B, int H, int D, int P,
                                         const int32_t* seq_lens, const int32_t* head_counts,
                                         usp_stream_t stream);
usp_status_t usp_relayout_head2seq_multi(int n_tensors, const void* const* src, void* const* dst,
                                         usp_dtype_t dt, int B, int H, int D, int P,
                                         const int32_t* seq_lens, const int32_t* head_counts,
                                         usp_stream_t stream);

/* usp_reorder — global sequence <-> ring-rank chunks under an ordering [YC].
 *   inverse = 0: src is global [B][S][H][D]; dst is R chunks back to back, chunk r is
 *                [B][s_r][H][D] holding rank r's tokens in local order (see usp_order_t).
 *   inverse = 1: the reverse copy.
 *   Bit-exact.  1 <= R <= 64.  Errors: INVALID_ARG for R out of range, S < 0, B/H/D < 1, NULL
 *   buffers. */
usp_status_t usp_reorder(const void* src, void* dst, usp_dtype_t dt, int B, int S, int H, int D,
                         int R, usp_order_t order, int inverse, usp_stream_t stream);

/* usp_attn_partial — one ring step: exact attention of one Q chunk against one K/V chunk,
 * returning the partial output and its log-sum-exp ([USP]: the backend returns "out, lse";
 * [CP] Ring Attention: each rank attends to the K/V block it holds).
 *
 *   q: bf16, B*Sq rows of q_row_stride elements (batch-major: row b*Sq + i), head h of a row at
 *      element h*D.  k, v: bf16, B*Sk rows of kv_row_stride elements, same head layout.
 *      Row strides are in elements, >= H*D, and row_stride*2 must be a multiple of 16 bytes;
 *      q, k, v must be 16-byte aligned.
 *   scale: softmax scale (1/sqrt(D) for standard attention).
 *   q_pos, k_pos: host descriptions of the chunks' global positions; both NULL = non-causal.
 *      Causal: key j visible to query i iff kpos(j) <= qpos(i) (diagonal included).
 *   o: [B][Sq][H][D] of o_dt (USP_FP32 for a partial; USP_BF16 allowed), 16-byte aligned.
 *   lse: fp32 [B][Sq][H]; a query that sees no key gets o = 0 and lse = -inf.
 *   status: device uint32 the kernel ORs error bits into (bounded waits), or NULL.
 *   Errors: INVALID_ARG (sizes, alignment, positions not increasing, only one of q_pos/k_pos),
 *   UNSUPPORTED (D not 64 or 128), CUDA (tensor-map encode or launch failure). */
usp_status_t usp_attn_partial(const void* q, const void* k, const void* v, int B, int H, int Sq,
                              int Sk, int D, int64_t q_row_stride, int64_t kv_row_stride,
                              float scale, const usp_positions_t* q_pos,
                              const usp_positions_t* k_pos, void* o, usp_dtype_t o_dt, float* lse,
                              uint32_t* status, usp_stream_t stream);

/* usp_lse_merge — the ring step's LSE-weighted combine over n_parts partials ([USP]:
 * out = prev_out - sigmoid(lse - prev_lse) * (prev_out - out),
 * lse = prev_lse - logsigmoid(prev_lse - lse), in fp32).  This kernel merges all partials of a
 * row in one pass with the equivalent max-shifted form (exact in real arithmetic):
 * m = max_k lse_k, w_k = exp(lse_k - m), out = sum_k w_k out_k / sum_k w_k,
 * lse = m + ln sum_k w_k.  Partials with lse = -inf contribute nothing: their out is loaded
 * with the LSE but never used, so it may hold any bits (NaN included) as long as the memory is
 * readable; a row whose partials are all -inf gets out = 0, lse = -inf.
 *
 *   o_parts: fp32, part k at o_parts + k*o_part_stride (elements), each [n_rows][H][D].
 *   lse_parts: fp32, part k at lse_parts + k*lse_part_stride, each [n_rows][H].
 *   o_out: [n_rows][H][D] of out_dt; lse_out: fp32 [n_rows][H] (may be NULL).
 *   1 <= n_parts <= 16; D a multiple of 4 and <= 256; 16-byte aligned o pointers and strides.
 *   Errors: INVALID_ARG otherwise. */
usp_status_t usp_lse_merge(int n_parts, const float* o_parts, int64_t o_part_stride,
                           const float* lse_parts, int64_t lse_part_stride, int64_t n_rows, int H,
                           int D, void* o_out, usp_dtype_t out_dt, float* lse_out,
                           usp_stream_t stream);

/* usp_attention — the whole method end to end on one GPU ([CP] Unified Attention: an all-to-all
 * inside each Ulysses group, Ring Attention on the result, the reverse all-to-all; with
 * ulysses_degree = 1 it is Ring Attention, with ring_degree = 1 Ulysses (Anything) Attention).
 *
 *   q, k, v: bf16 global [B][S][H][D] (16-byte aligned).  Virtual rank c = r*ulysses_degree + u
 *   (ring group r, Ulysses index u) holds rows [o, o + seq_lens[c]) of ring chunk r, whose tokens
 *   the ordering fixes; seq_lens (host, ulysses_degree*ring_degree entries) must sum per ring
 *   group to that ring chunk's length, or be NULL for the default split.  head_counts (host,
 *   ulysses_degree entries summing to H) or NULL for the default split of H.
 *   ulysses_degree >= 1, ring_degree >= 1, their product <= 16, ulysses_degree <= H.
 *   causal: key j visible to query i iff j <= i (global positions).
 *   o: [B][S][H][D] of o_dt; lse: fp32 [B][S][H] or NULL.
 *   workspace: device scratch of at least usp_attention_workspace_size(...) bytes, 256-byte
 *   aligned.  Its first 4 bytes are the status word usp_check_status reads and clears; zero
 *   them once before the first call (e.g. allocate the workspace zeroed).  Bytes 8-15 hold the
 *   counter of a dynamic unit deal (see usp_plan_deals): every launch that uses it leaves it
 *   zero when it ends, and the library clears it in the stream whenever a thread calls with a
 *   workspace, plan or buffers other than its previous call's.  Leave bytes 0-15 to the library
 *   between calls.
 *   Steps (one stream): (1) the seq->head re-layout of Q, K, V (with the ring ordering) is
 *   addressing, not a pass: each virtual rank's head-sharded view is read in place by the
 *   attention's tensor maps, one map over its ring chunk when that is one affine run of global
 *   rows (contiguous or stripe order, one ring rank), a map with a piece dimension over a zigzag
 *   chunk's two equal half-chunks of whole 128-row tiles (S divisible by 256 * ring_degree), and
 *   otherwise a map over the global rows spanning both half-chunks, of which only the chunk's
 *   own rows are read as keys and written as outputs.
 *   (2) One attention launch over every (ring step, chunk pair, head, query block), with fully
 *   masked causal tiles skipped.  With several ring ranks the ring steps are either
 *     - fused: each 256-row query block carries one online softmax across the visible K/V chunks
 *       of all ring steps, in ring order ([CP] Ring Attention: K/V blocks pass around the ring;
 *       the running (max, sum, output) is the LSE-weighted merge of [USP] done in registers),
 *       and writes the final O and LSE; or
 *     - separate: every ring step writes an fp32 partial (O, LSE) into the workspace and
 *       (3) an LSE merge pass combines them.
 *   The library picks the mode with the shorter modelled time (the merge pass and per-step
 *   epilogues against the load balance of fewer, longer units); the choice depends only on the
 *   arguments, so usp_attention_workspace_size and usp_attention agree.  USP_RING_MERGE=fused or
 *   =separate in the environment (read at each call) overrides it.  A fused non-causal ring may
 *   also run the last 256-row blocks of one ring chunk as separate ring steps, whose units are
 *   dealt after all the chains and fill the last round of the launch, with their own partials
 *   and (3) a merge over those rows only (USP_RING_SPLIT=0 never does, =k splits the last k
 *   blocks of the last ring chunk; for tests).  The head->seq re-layout and inverse reorder of O
 *   and LSE are the store addressing of (2) (one ring rank, or fused) or (3): the result lands
 *   in the global layout directly.
 *   Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA as above. */
usp_status_t usp_attention(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                           float scale, int causal, int ulysses_degree, int ring_degree,
                           const int32_t* seq_lens, const int32_t* head_counts, usp_order_t order,
                           void* o, usp_dtype_t o_dt, float* lse, void* workspace,
                           size_t workspace_bytes, usp_stream_t stream);

/* usp_attention on a QKV-packed input ([YC]: yunchang ships QKV-packed variants of its
 * attention functions, which outperform the unpacked ones): qkv is bf16 [B][S][3][H][D], i.e.
 * token t of batch b holds its query heads, then its key heads, then its value heads, in one row
 * of 3*H*D elements (the layout a fused QKV projection writes).  The attention's tensor maps read
 * the three tensors in place with a 3*H*D row stride, so nothing is unpacked.  All other
 * arguments, outputs, workspace and errors are those of usp_attention (qkv must be 16-byte
 * aligned). */
usp_status_t usp_attention_qkvpacked(const void* qkv, int B, int S, int H, int D, float scale,
                                     int causal, int ulysses_degree, int ring_degree,
                                     const int32_t* seq_lens, const int32_t* head_counts,
                                     usp_order_t order, void* o, usp_dtype_t o_dt, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     usp_stream_t stream);

/* usp_attention with phase timing: identical work, and additionally records the caller's CUDA
 * events (cudaEvent_t handles, created by the caller) on `stream`:
 *   events[0] before the first launch, events[1] after the Q/K/V re-layout, events[2] after the
 *   partial-attention launch(es), events[3] after the merge, events[4] after the output
 *   re-layout.  A skipped phase records its event at the same point as the previous one.
 *   `events` must hold 5 handles (entries may be NULL to skip a record).  If `launches` is not
 *   NULL it receives 4 counts: kernels launched for the Q/K/V re-layout, the attention, the merge
 *   and the output re-layout (0 for a phase that did not run; both re-layouts are addressing in
 *   this library, so their counts are 0).  Errors as usp_attention. */
usp_status_t usp_attention_events(const void* q, const void* k, const void* v, int B, int S, int H,
                                  int D, float scale, int causal, int ulysses_degree,
                                  int ring_degree, const int32_t* seq_lens,
                                  const int32_t* head_counts, usp_order_t order, void* o,
                                  usp_dtype_t o_dt, float* lse, void* workspace,
                                  size_t workspace_bytes, void* const* events, int* launches,
                                  usp_stream_t stream);

/* usp_attention_noalloc — usp_attention without a workspace, for callers that cannot allocate
 * device memory: code embedded in a host application that owns every device allocation, or
 * latency-critical paths where cudaMalloc's implicit synchronisation is not acceptable.  The pages
 * have no counterpart to this entry point; it is a library convenience.
 *
 *   Same arguments and results as usp_attention, minus the workspace.  The scratch is a 128 MiB
 *   array compiled into the library (a file-scope __device__ array): every GPU that loads the
 *   library's device code holds it until the process exits.  Problems whose
 *   usp_attention_workspace_size exceeds 128 MiB are rejected with USP_ERR_WORKSPACE and a message
 *   giving both sizes; nothing is launched then.
 *   The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current) and caches it with the device's current CUDA context; make that
 *   first call before any stream capture.  If the context changes (after cudaDeviceReset the
 *   library's module is loaded again), the next call looks the address up again.
 *   Every call shares the array and finds the previous call's data in it; each call clears the
 *   status word it needs zeroed.  Calls that overlap on the GPU (several streams or host threads
 *   on one device) race on the array: serialise them.
 *   status: optional device uint32 that receives this call's bounded-wait status word (pass it to
 *   usp_check_status).  With status = NULL a timed-out wait is not reported: the array's own
 *   status word is cleared by the next call and has no address the caller can read.
 *   This entry point calls no cudaMalloc or cudaFree and no allocating library routine. */
usp_status_t usp_attention_noalloc(const void* q, const void* k, const void* v, int B, int S, int H,
                                   int D, float scale, int causal, int ulysses_degree,
                                   int ring_degree, const int32_t* seq_lens,
                                   const int32_t* head_counts, usp_order_t order, void* o,
                                   usp_dtype_t o_dt, float* lse, uint32_t* status,
                                   usp_stream_t stream);

/* Bytes of workspace usp_attention needs for these arguments (0 on invalid arguments): a 256-byte
 * status word, plus ring_degree fp32 partial slots of O and LSE when the ring steps run
 * separately, or for the split rows of a split fused ring (see usp_attention). */
size_t usp_attention_workspace_size(int B, int S, int H, int D, int causal, int ulysses_degree,
                                    int ring_degree, usp_order_t order, usp_dtype_t o_dt);

/* Host-only query (no device needed): how usp_attention runs the ring steps for these arguments.
 * Returns 0 with one ring rank, 1 when every ring step writes an fp32 partial and a merge pass
 * combines them, 2 when the ring steps are fused into one online softmax per query block (see
 * usp_attention), or -1 on invalid arguments (usp_last_error says why). */
int usp_attention_ring_mode(int B, int S, int H, int D, int causal, int ulysses_degree,
                            int ring_degree, usp_order_t order, usp_dtype_t o_dt);

/* Synchronises `stream`, reads the device status word at `status` (a usp_attention workspace or
 * the uint32 given to usp_attn_partial), clears it, and returns USP_ERR_TIMEOUT if a bounded wait
 * gave up since the last check, USP_ERR_CUDA if the stream reports an error, else USP_OK.
 * Every device-side wait of the attention kernel gives up after USP_WAIT_BUDGET_MS milliseconds
 * (environment, read at each call; default 2000); all its roles then stop, finish their copies
 * and MMAs in flight, free their tensor memory and exit, so the context stays usable.
 * USP_TEST_WITHHOLD_LOADS=1 (environment, read at each call) is a test hook for that path: the
 * kernel's producer issues no loads, so the waits run out. */
usp_status_t usp_check_status(void* status, usp_stream_t stream);

/* Host-only planning query (no device needed): the chunk-pair work list usp_attention launches
 * when the ring steps run separately, for B = 1, as the causal pair schedule's runs (the launch
 * may cut a run further, at a zigzag chunk's half-chunk boundary or after a causal run's first
 * (length mod 256) rows, without changing which keys any row sees).  Writes up to `cap` records
 * of 8 int32 each into `out`:
 *   {ulysses index u, q ring chunk r, ring step k, kv ring chunk r2, q local row0, q rows,
 *    visible kv rows, diag}
 * where key c (0 <= c < visible kv rows, local to ring chunk r2) is visible to q local row i
 * (row0 <= i < row0 + q rows) iff c <= i - row0 + diag (diag = INT32_MAX: no causal limit).
 * Returns the total record count (which may exceed cap), or -1 on invalid arguments. */
int usp_plan_pairs(int S, int ulysses_degree, int ring_degree, int causal, usp_order_t order,
                   int32_t* out, int cap);

/* Host-only planning query for the fused ring (no device needed): the links usp_attention runs
 * when the ring steps are fused, for B = 1, whichever mode the library would pick.  Writes up to
 * `cap` records of 8 int32 each into `out`:
 *   {ulysses index u, q ring chunk r, piece row0, piece rows, ring step k, kv ring chunk r2,
 *    visible kv rows, diag}
 * one per visible ring step of each piece of query rows; key c (0 <= c < visible kv rows, local to
 * ring chunk r2) is visible to piece row i (0 <= i < piece rows, local row row0 + i of chunk r)
 * iff c <= i + diag (diag = INT32_MAX: no causal limit).  Returns the total record count (which
 * may exceed cap), or -1 on invalid arguments. */
int usp_plan_chains(int S, int ulysses_degree, int ring_degree, int causal, usp_order_t order,
                    int32_t* out, int cap);

/* Host-only planning query for the order of work units (no device needed): the attention
 * launches usp_attention runs for these arguments (default seq_lens and head_counts) on a GPU
 * with `sms` SMs.  Each launch runs one CTA per SM over its work units (one per head, batch and
 * 256-row query block of a segment; numbered per Ulysses rank, head-major, longest first), and a
 * deal fixes which CTA takes which unit.  By default a snake order: round t, CTA c takes unit
 * t*G + c, or t*G + G-1-c for odd t (G CTAs).  A deal with (deal & 1) takes t*G + c in every
 * round; one with (deal & 4) is dynamic: each CTA takes the next unit in numbering order from a
 * counter in the workspace when it is ready for one; one with (deal & 2) makes every odd
 * (batch, head) index b * heads + h of a Ulysses rank visit its query blocks in reverse order.
 * The library models each deal's launch time (every unit costs its key tiles plus an epilogue of
 * 2 tile periods for bf16 rows, 2.5 for fp32; static deals put it on the CTA the deal names,
 * the dynamic one on the CTA free first, the lowest index among equals; the busiest CTA's total
 * is the time) and keeps the fastest when it saves more than 0.5 % against the default.  The deal
 * changes only the timing: each unit computes the same values wherever it runs.
 * USP_UNIT_DEAL=0..7 in the environment (read at each call) forces a deal (usp_attn_partial,
 * which has no workspace, drops the dynamic bit).  Writes up to `cap` records of 4 int32 each
 * into `out`, one per launch:
 *   {work units, deal, modelled time of that deal, modelled time of the default deal}
 * with times in thousandths of a key-tile period.  Returns the launch count (which may exceed
 * cap), or -1 on invalid arguments (sms < 1, or as usp_attention_ring_mode). */
int usp_plan_deals(int B, int S, int H, int D, int causal, int ulysses_degree, int ring_degree,
                   usp_order_t order, usp_dtype_t o_dt, int sms, int32_t* out, int cap);

const char* usp_status_string(usp_status_t s);
const char* usp_last_error(void);
int usp_version(void); /* major*10000 + minor*100 + patch */

#ifdef __cplusplus
}
#endif

#endif /* USP_GB300_H */
