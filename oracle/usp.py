"""fp64 oracle for context-parallel attention.  Test infrastructure only (see ``oracle/__init__``).

Conventions, fixed once for the whole library and its oracle:

* Q, K, V, O are ``[B][S][H][D]`` (batch, sequence, head, head dim); the log-sum-exp is
  ``[B][S][H]`` (diffusers PR #12693 "Add Unified Sequence Parallel attention": "the lse is of shape
  (B, S, H_LOCAL)").
* The log-sum-exp is natural-log and includes the softmax scale: ``lse = ln sum_j exp(scale q.k_j)``.
  The pages' merge uses ``sigmoid`` / ``logsigmoid``, which are natural-exponential functions, so
  only a natural-log LSE makes that merge exact.
* Causal masking compares GLOBAL token positions: key j is visible to query i iff
  ``pos_k(j) <= pos_q(i)`` (diagonal included).  The pages never define the mask; global
  positions leave no top-left / bottom-right ambiguity when a chunk pair is not square.
* A query that sees no key has ``out = 0`` and ``lse = -inf``.
"""
from __future__ import annotations

import numpy as np

NEG_INF = float("-inf")


# ------------------------------------------------------------------------------------------------
# Inputs
# ------------------------------------------------------------------------------------------------

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact bfloat16 -> float64 widening of raw uint16 bit patterns."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def default_split(S: int, P: int) -> list[int]:
    """Default split of S tokens over P ranks: ``floor(S/P) + (p < S mod P)``.

    The pages give no rule (diffusers issue #12706 only says UAA supports arbitrary lengths with
    zero padding); this is the plainest one and it reproduces every split the workloads print
    (1000 -> 334/333/333, 4481 -> 2241/2240 and 1494/1494/1493)."""
    if P < 1 or S < 0:
        raise ValueError("need P >= 1 and S >= 0")
    base, extra = divmod(S, P)
    return [base + (1 if p < extra else 0) for p in range(P)]


# ------------------------------------------------------------------------------------------------
# Attention with log-sum-exp (one ring step's (out, lse))
# ------------------------------------------------------------------------------------------------

def _attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                    allowed: np.ndarray | None):
    """One (batch, head): q [Sq, D], k/v [Sk, D]; ``allowed`` [Sq, Sk] bool or None (all)."""
    Sq = q.shape[0]
    D = v.shape[1]
    if k.shape[0] == 0:
        return np.zeros((Sq, D)), np.full(Sq, NEG_INF)
    s = scale * (q @ k.T)                      # scores s_ij = scale * q_i . k_j
    if allowed is not None:
        s = np.where(allowed, s, NEG_INF)
    m = s.max(axis=1)                          # row max over the allowed set
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(s - m_safe[:, None])            # exp(s_ij - m_i); exp(-inf) = 0 for masked keys
    l = w.sum(axis=1)
    out = (w @ v) / np.where(empty, 1.0, l)[:, None]
    lse = m_safe + np.log(np.where(empty, 1.0, l))
    out[empty] = 0.0
    lse[empty] = NEG_INF
    return out, lse


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool = False,
              q_pos: np.ndarray | None = None, k_pos: np.ndarray | None = None,
              row_block: int = 4096):
    """Exact softmax attention returning ``(out, lse)``.

    q: ``[B][Sq][H][D]``, k and v: ``[B][Sk][H][D]`` (float64).  Returns out ``[B][Sq][H][D]`` and
    lse ``[B][Sq][H]``.  With ``causal`` the visible keys of query i are ``{j : k_pos[j] <=
    q_pos[i]}`` (positions default to ``0..S-1``).  This is the backend call each ring step makes,
    "out, lse" with ``return_lse`` (diffusers PR #12693, TemplatedRingAttention forward).

    Query rows are processed ``row_block`` at a time only to bound memory; every output row is
    computed exactly as the definition states."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if causal:
        q_pos = np.arange(Sq) if q_pos is None else np.asarray(q_pos)
        k_pos = np.arange(Sk) if k_pos is None else np.asarray(k_pos)
    out = np.zeros((B, Sq, H, v.shape[3]))
    lse = np.full((B, Sq, H), NEG_INF)
    for b in range(B):
        for h in range(H):
            kb, vb = k[b, :, h, :], v[b, :, h, :]
            for i0 in range(0, Sq, row_block):
                i1 = min(Sq, i0 + row_block)
                allowed = (k_pos[None, :] <= q_pos[i0:i1, None]) if causal else None
                o, l = _attention_head(q[b, i0:i1, h, :], kb, vb, scale, allowed)
                out[b, i0:i1, h, :] = o
                lse[b, i0:i1, h] = l
    return out, lse


def attention_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   causal: bool = False, q_pos: np.ndarray | None = None,
                   k_pos: np.ndarray | None = None):
    """Attention for a sample of query rows of ONE (batch, head): q_rows [n][D], k/v [Sk][D].

    Same definition as ``attention``; used to check full-size runs row by row."""
    allowed = None
    if causal:
        k_pos = np.arange(k.shape[0]) if k_pos is None else np.asarray(k_pos)
        allowed = k_pos[None, :] <= np.asarray(q_pos)[:, None]
    return _attention_head(q_rows, k, v, scale, allowed)


# ------------------------------------------------------------------------------------------------
# Ring step merge (the pages' formula)
# ------------------------------------------------------------------------------------------------

def _sigmoid(x: np.ndarray) -> np.ndarray:
    return np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))),
                    np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))


def _logsigmoid(x: np.ndarray) -> np.ndarray:
    return np.where(x >= 0, -np.log1p(np.exp(-np.abs(x))), x - np.log1p(np.exp(-np.abs(x))))


def merge(prev_out: np.ndarray, prev_lse: np.ndarray, out: np.ndarray, lse: np.ndarray):
    """Merge a new partial ``(out, lse)`` into the running ``(prev_out, prev_lse)``.

    The pages' ring step (diffusers PR #12693, TemplatedRingAttention forward, in fp32 there and
    fp64 here)::

        out = prev_out - sigmoid(lse - prev_lse) * (prev_out - out)
        lse = prev_lse - logsigmoid(prev_lse - lse)

    ``out``: ``[..., D]``, ``lse``: ``[...]``.  The sigmoid form is undefined when both LSEs are
    -inf; reading: a partial with lse = -inf saw no key and contributes nothing, so the result is
    the other operand exactly (and stays out = 0, lse = -inf when both are empty)."""
    prev_out = np.asarray(prev_out, dtype=np.float64)
    out = np.asarray(out, dtype=np.float64)
    prev_lse = np.asarray(prev_lse, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    prev_empty = ~np.isfinite(prev_lse)
    new_empty = ~np.isfinite(lse)
    both = ~(prev_empty | new_empty)
    with np.errstate(invalid="ignore"):
        d_new = np.where(both, lse - prev_lse, 0.0)
    res_out = prev_out - _sigmoid(d_new)[..., None] * (prev_out - out)
    res_lse = prev_lse - _logsigmoid(-d_new)
    res_out = np.where(new_empty[..., None], prev_out, res_out)
    res_lse = np.where(new_empty, prev_lse, res_lse)
    res_out = np.where((prev_empty & ~new_empty)[..., None], out, res_out)
    res_lse = np.where(prev_empty & ~new_empty, lse, res_lse)
    return res_out, res_lse


# ------------------------------------------------------------------------------------------------
# Ulysses all-to-all as index loops
# ------------------------------------------------------------------------------------------------

def _offsets(lengths) -> list[int]:
    off = [0]
    for n in lengths:
        off.append(off[-1] + int(n))
    return off


def seq2head(src: np.ndarray, B: int, H: int, D: int, seq_lens, head_counts=None) -> np.ndarray:
    """Ulysses all-to-all #1 (sequence-sharded -> head-sharded) on flat buffers.

    ``src`` holds the P ranks' sequence chunks back to back: chunk q is ``[B][s_q][H][D]``.
    The result holds the P ranks' head-sharded buffers back to back: buffer p is
    ``[B][S][h_p][D]`` with ``S = sum s_q``, and ``Y_p[b][o_q + t][h'][d] = X_q[b][t][g_p + h'][d]``
    where ``o_q`` are the sequence offsets and ``g_p`` the head offsets.  After it "each GPU
    holds every token for a subset of attention heads" (HF docs "Context parallelism", Ulysses
    Attention).  Uneven ``seq_lens`` with no padding is the Ulysses Anything case (diffusers
    issue #12706); uneven ``head_counts`` is the other requirement UAA removes (HF docs, Ulysses
    Anything Attention).  ``head_counts`` defaults to ``default_split(H, P)``."""
    P = len(seq_lens)
    head_counts = default_split(H, P) if head_counts is None else list(head_counts)
    so, ho = _offsets(seq_lens), _offsets(head_counts)
    S = so[-1]
    src = np.asarray(src).reshape(-1)
    dst = np.empty(B * S * H * D, dtype=src.dtype)
    chunks = []
    for q in range(P):
        base = B * so[q] * H * D
        chunks.append(src[base: base + B * seq_lens[q] * H * D].reshape(B, seq_lens[q], H, D))
    for p in range(P):
        base = B * S * ho[p] * D
        Y = dst[base: base + B * S * head_counts[p] * D].reshape(B, S, head_counts[p], D)
        for q in range(P):
            for b in range(B):
                Y[b, so[q]: so[q + 1], :, :] = chunks[q][b, :, ho[p]: ho[p + 1], :]
    return dst


def head2seq(src: np.ndarray, B: int, H: int, D: int, seq_lens, head_counts=None) -> np.ndarray:
    """Ulysses all-to-all #2 (head-sharded -> sequence-sharded), the exact inverse of
    ``seq2head`` ("a second all-to-all regroups the results by token", HF docs "Context
    parallelism", Ulysses Attention).  Also used for the LSE with ``D = 1`` (diffusers PR #12693
    sends the lse through the same all-to-all, scatter on heads, gather on sequence)."""
    P = len(seq_lens)
    head_counts = default_split(H, P) if head_counts is None else list(head_counts)
    so, ho = _offsets(seq_lens), _offsets(head_counts)
    S = so[-1]
    src = np.asarray(src).reshape(-1)
    dst = np.empty(B * S * H * D, dtype=src.dtype)
    for q in range(P):
        base = B * so[q] * H * D
        X = dst[base: base + B * seq_lens[q] * H * D].reshape(B, seq_lens[q], H, D)
        for p in range(P):
            pbase = B * S * ho[p] * D
            Y = src[pbase: pbase + B * S * head_counts[p] * D].reshape(B, S, head_counts[p], D)
            for b in range(B):
                X[b, :, ho[p]: ho[p + 1], :] = Y[b, so[q]: so[q + 1], :, :]
    return dst


# ------------------------------------------------------------------------------------------------
# Chunk orderings
# ------------------------------------------------------------------------------------------------

def ring_positions(order: str, S: int, ring_degree: int) -> list[np.ndarray]:
    """Global token positions held by each ring rank, in the rank's local order.

    * ``contiguous`` (yunchang's "basic" ring): rank r holds the r-th piece of
      ``default_split(S, R)``.
    * ``zigzag``: split S into 2R pieces by ``default_split(S, 2R)``; rank r holds piece r then
      piece 2R-1-r.  (Reading: the pages only name zigzag as a causal load balance; this is the
      layout that balances causal work and gives "16 half-chunks of 4096" for R = 8, S = 65536.)
    * ``stripe``: token t goes to rank ``t mod R`` at local index ``t // R``.

    Positions increase with the local index in all three, which the chunk-pair schedule uses."""
    R = ring_degree
    if order == "contiguous":
        off = _offsets(default_split(S, R))
        return [np.arange(off[r], off[r + 1], dtype=np.int64) for r in range(R)]
    if order == "zigzag":
        off = _offsets(default_split(S, 2 * R))
        return [np.concatenate([np.arange(off[r], off[r + 1]),
                                np.arange(off[2 * R - 1 - r], off[2 * R - r])]).astype(np.int64)
                for r in range(R)]
    if order == "stripe":
        return [np.arange(r, S, R, dtype=np.int64) for r in range(R)]
    raise ValueError(f"unknown order {order!r}")


def virtual_rank_lengths(order: str, S: int, ulysses_degree: int, ring_degree: int,
                         seq_lens=None) -> list[int]:
    """Per virtual rank chunk lengths; rank ``c = r * ulysses_degree + u`` (ring group r, Ulysses
    index u) holds local rows ``[o, o + s_c)`` of ring chunk r.  Default: ``default_split`` of the
    ring chunk over the Ulysses group.  Given ``seq_lens`` must sum, per ring group, to the ring
    chunk length the ordering fixes."""
    ring_len = [len(p) for p in ring_positions(order, S, ring_degree)]
    if seq_lens is None:
        out = []
        for r in range(ring_degree):
            out += default_split(ring_len[r], ulysses_degree)
        return out
    seq_lens = [int(x) for x in seq_lens]
    if len(seq_lens) != ulysses_degree * ring_degree or min(seq_lens) < 0:
        raise ValueError("seq_lens must have ulysses_degree * ring_degree non-negative entries")
    for r in range(ring_degree):
        if sum(seq_lens[r * ulysses_degree:(r + 1) * ulysses_degree]) != ring_len[r]:
            raise ValueError("seq_lens of a ring group must sum to its ring chunk length")
    return seq_lens


# ------------------------------------------------------------------------------------------------
# The whole method
# ------------------------------------------------------------------------------------------------

def usp_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool,
                  ulysses_degree: int, ring_degree: int, order: str = "contiguous",
                  seq_lens=None, head_counts=None):
    """Unified sequence-parallel attention over ``ulysses_degree x ring_degree`` virtual ranks.

    Follows HF docs "Context parallelism", section Unified Attention: an all-to-all inside each
    Ulysses group redistributes heads and tokens, Ring Attention runs on the result, and the
    all-to-all is reversed (for out and for lse, as in diffusers PR #12693).  Ring Attention
    (same docs, Ring Attention section): at step k rank r attends to the K/V block of rank
    ``(r - k) mod R`` and merges the partial into its running result with ``merge``.

    Inputs are global ``[B][S][H][D]`` float64; returns global ``(out, lse)``."""
    B, S, H, D = q.shape
    U, R = ulysses_degree, ring_degree
    pos = ring_positions(order, S, R)
    lens = virtual_rank_lengths(order, S, U, R, seq_lens)
    hc = default_split(H, U) if head_counts is None else list(head_counts)
    ho = _offsets(hc)
    out = np.zeros((B, S, H, D))
    lse = np.full((B, S, H), NEG_INF)
    # Ulysses all-to-all inside each ring group: every rank of group r ends with all rows of
    # ring chunk r for its head subset.
    heads = {}
    for r in range(R):
        rl = lens[r * U:(r + 1) * U]
        for name, x in (("q", q), ("k", k), ("v", v)):
            src = np.concatenate([x[:, pos[r][o:o + n]].reshape(-1)
                                  for o, n in zip(_offsets(rl)[:-1], rl)])
            y = seq2head(src, B, H, D, rl, hc)
            Sr = len(pos[r])
            for u in range(U):
                base = B * Sr * ho[u] * D
                heads[(name, r, u)] = y[base: base + B * Sr * hc[u] * D].reshape(B, Sr, hc[u], D)
    for r in range(R):
        rl = lens[r * U:(r + 1) * U]
        Sr = len(pos[r])
        y_out = np.empty(B * Sr * H * D)
        y_lse = np.empty(B * Sr * H)
        for u in range(U):
            run_o = run_l = None
            for step in range(R):
                r2 = (r - step) % R
                o, l = attention(heads[("q", r, u)], heads[("k", r2, u)], heads[("v", r2, u)],
                                 scale, causal, pos[r], pos[r2])
                if run_o is None:
                    run_o, run_l = o, l
                else:
                    run_o, run_l = merge(run_o, run_l, o, l)
            base = B * Sr * ho[u]
            y_out[base * D: (base + B * Sr * hc[u]) * D] = run_o.reshape(-1)
            y_lse[base: base + B * Sr * hc[u]] = run_l.reshape(-1)
        # reverse all-to-all, then scatter the ring chunk back to its global positions
        xo = head2seq(y_out, B, H, D, rl, hc)
        xl = head2seq(y_lse, B, H, 1, rl, hc)
        so = _offsets(rl)
        for u in range(U):
            rows = pos[r][so[u]:so[u + 1]]
            base = B * so[u]
            out[:, rows] = xo[base * H * D:(base + B * rl[u]) * H * D].reshape(B, rl[u], H, D)
            lse[:, rows] = xl[base * H:(base + B * rl[u]) * H].reshape(B, rl[u], H)
    return out, lse
