"""Thin ctypes binding of ``libusp_gb300.so`` (the C ABI in ``include/usp.h``).

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
Functions keep the C names.  Tensor arguments may be torch tensors (their ``data_ptr()`` is
passed) or raw integer device addresses; ``stream=None`` means torch's current CUDA stream.
If the library is not built, the first call raises ``RuntimeError``: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libusp_gb300.so")

USP_OK, USP_ERR_INVALID_ARG, USP_ERR_UNSUPPORTED, USP_ERR_CUDA, USP_ERR_TIMEOUT, \
    USP_ERR_WORKSPACE, USP_ERR_NO_DEVICE = range(7)
USP_BF16, USP_FP32 = 0, 1
ORDERS = {"contiguous": 0, "zigzag": 1, "stripe": 2}

EXPORTED = [
    "usp_relayout_seq2head", "usp_relayout_head2seq", "usp_relayout_seq2head_multi",
    "usp_relayout_head2seq_multi", "usp_reorder", "usp_attn_partial",
    "usp_lse_merge", "usp_attention", "usp_attention_qkvpacked", "usp_attention_events",
    "usp_attention_noalloc",
    "usp_attention_workspace_size", "usp_attention_ring_mode",
    "usp_check_status",
    "usp_plan_pairs", "usp_plan_chains", "usp_plan_deals", "usp_status_string", "usp_last_error",
    "usp_version",
]


class UspError(RuntimeError):
    def __init__(self, status: int, func: str, message: str):
        super().__init__(f"{func}: status {status}: {message}")
        self.status = status


class Positions(ctypes.Structure):
    """usp_positions_t: global positions of a chunk's rows (1 or 2 affine segments)."""
    _fields_ = [("n_seg", ctypes.c_int32), ("start", ctypes.c_int32 * 2),
                ("len", ctypes.c_int32 * 2), ("stride", ctypes.c_int32)]

    @classmethod
    def make(cls, segments, stride: int = 1) -> "Positions":
        """segments: [(start, len)] with 1 or 2 entries."""
        p = cls()
        p.n_seg = len(segments)
        for i, (s, n) in enumerate(segments):
            p.start[i] = s
            p.len[i] = n
        p.stride = stride
        return p


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    i32p = ctypes.POINTER(ctypes.c_int32)
    posp = ctypes.POINTER(Positions)
    sig = {
        "usp_relayout_seq2head": [vp, vp, i32, i32, i32, i32, i32, i32p, i32p, vp],
        "usp_relayout_head2seq": [vp, vp, i32, i32, i32, i32, i32, i32p, i32p, vp],
        "usp_relayout_seq2head_multi": [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, i32, i32,
                                        i32, i32, i32p, i32p, vp],
        "usp_relayout_head2seq_multi": [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i32, i32, i32,
                                        i32, i32, i32p, i32p, vp],
        "usp_reorder": [vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp],
        "usp_attn_partial": [vp, vp, vp, i32, i32, i32, i32, i32, i64, i64, f32, posp, posp, vp,
                             i32, vp, vp, vp],
        "usp_lse_merge": [i32, vp, i64, vp, i64, i64, i32, i32, vp, i32, vp, vp],
        "usp_attention": [vp, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, i32p, i32p, i32, vp,
                          i32, vp, vp, sz, vp],
        "usp_attention_qkvpacked": [vp, i32, i32, i32, i32, f32, i32, i32, i32, i32p, i32p, i32, vp,
                                    i32, vp, vp, sz, vp],
        "usp_attention_events": [vp, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, i32p, i32p,
                                 i32, vp, i32, vp, vp, sz, ctypes.POINTER(vp),
                                 ctypes.POINTER(ctypes.c_int), vp],
        "usp_attention_noalloc": [vp, vp, vp, i32, i32, i32, i32, f32, i32, i32, i32, i32p, i32p,
                                  i32, vp, i32, vp, vp, vp],
        "usp_attention_workspace_size": [i32, i32, i32, i32, i32, i32, i32, i32, i32],
        "usp_attention_ring_mode": [i32, i32, i32, i32, i32, i32, i32, i32, i32],
        "usp_check_status": [vp, vp],
        "usp_plan_pairs": [i32, i32, i32, i32, i32, i32p, i32],
        "usp_plan_chains": [i32, i32, i32, i32, i32, i32p, i32],
        "usp_plan_deals": [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32p, i32],
        "usp_status_string": [i32],
        "usp_last_error": [],
        "usp_version": [],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.usp_attention_workspace_size.restype = ctypes.c_size_t
    L.usp_status_string.restype = ctypes.c_char_p
    L.usp_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _i32(seq):
    if seq is None:
        return None
    seq = [int(x) for x in seq]
    return (ctypes.c_int32 * max(1, len(seq)))(*seq)


def _check(status: int, func: str) -> None:
    if status != USP_OK:
        raise UspError(status, func, lib().usp_last_error().decode())


def _dtype(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return USP_BF16
    if t.dtype == torch.float32:
        return USP_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


# --------------------------------------------------------------------------------------------
# One function per C entry point
# --------------------------------------------------------------------------------------------

def usp_relayout_seq2head(src, dst, B, H, D, seq_lens, head_counts=None, dt=None, stream=None):
    dt = _dtype(src) if dt is None else dt
    _check(lib().usp_relayout_seq2head(_ptr(src), _ptr(dst), dt, B, H, D, len(seq_lens),
                                       _i32(seq_lens), _i32(head_counts), _stream(stream)),
           "usp_relayout_seq2head")


def usp_relayout_head2seq(src, dst, B, H, D, seq_lens, head_counts=None, dt=None, stream=None):
    dt = _dtype(src) if dt is None else dt
    _check(lib().usp_relayout_head2seq(_ptr(src), _ptr(dst), dt, B, H, D, len(seq_lens),
                                       _i32(seq_lens), _i32(head_counts), _stream(stream)),
           "usp_relayout_head2seq")


def _ptr_array(xs):
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def usp_relayout_seq2head_multi(srcs, dsts, B, H, D, seq_lens, head_counts=None, dt=None,
                                stream=None):
    """seq->head re-layout of up to 3 same-shaped tensors (e.g. Q, K, V) in one launch."""
    dt = _dtype(srcs[0]) if dt is None else dt
    _check(lib().usp_relayout_seq2head_multi(len(srcs), _ptr_array(srcs), _ptr_array(dsts), dt, B,
                                             H, D, len(seq_lens), _i32(seq_lens),
                                             _i32(head_counts), _stream(stream)),
           "usp_relayout_seq2head_multi")


def usp_relayout_head2seq_multi(srcs, dsts, B, H, D, seq_lens, head_counts=None, dt=None,
                                stream=None):
    """head->seq re-layout of up to 3 same-shaped tensors in one launch."""
    dt = _dtype(srcs[0]) if dt is None else dt
    _check(lib().usp_relayout_head2seq_multi(len(srcs), _ptr_array(srcs), _ptr_array(dsts), dt, B,
                                             H, D, len(seq_lens), _i32(seq_lens),
                                             _i32(head_counts), _stream(stream)),
           "usp_relayout_head2seq_multi")


def usp_reorder(src, dst, B, S, H, D, R, order="contiguous", inverse=False, dt=None, stream=None):
    dt = _dtype(src) if dt is None else dt
    _check(lib().usp_reorder(_ptr(src), _ptr(dst), dt, B, S, H, D, R, ORDERS[order],
                             int(bool(inverse)), _stream(stream)), "usp_reorder")


def usp_attn_partial(q, k, v, B, H, Sq, Sk, D, q_row_stride, kv_row_stride, scale, o, lse,
                     q_pos: Positions | None = None, k_pos: Positions | None = None,
                     o_dt=None, status=None, stream=None):
    o_dt = _dtype(o) if o_dt is None else o_dt
    qp = ctypes.byref(q_pos) if q_pos is not None else None
    kp = ctypes.byref(k_pos) if k_pos is not None else None
    _check(lib().usp_attn_partial(_ptr(q), _ptr(k), _ptr(v), B, H, Sq, Sk, D, q_row_stride,
                                  kv_row_stride, float(scale), qp, kp, _ptr(o), o_dt, _ptr(lse),
                                  _ptr(status), _stream(stream)), "usp_attn_partial")


def usp_lse_merge(n_parts, o_parts, o_part_stride, lse_parts, lse_part_stride, n_rows, H, D,
                  o_out, lse_out=None, out_dt=None, stream=None):
    out_dt = _dtype(o_out) if out_dt is None else out_dt
    _check(lib().usp_lse_merge(n_parts, _ptr(o_parts), o_part_stride, _ptr(lse_parts),
                               lse_part_stride, n_rows, H, D, _ptr(o_out), out_dt, _ptr(lse_out),
                               _stream(stream)), "usp_lse_merge")


def usp_attention_workspace_size(B, S, H, D, ulysses_degree, ring_degree, order="contiguous",
                                 o_dt=USP_FP32, causal=False) -> int:
    return int(lib().usp_attention_workspace_size(B, S, H, D, int(causal), ulysses_degree,
                                                  ring_degree, ORDERS[order], o_dt))


RING_MODES = {0: "none", 1: "separate", 2: "fused"}


def usp_attention_ring_mode(B, S, H, D, causal, ulysses_degree, ring_degree, order="contiguous",
                            o_dt=USP_FP32) -> str:
    """How usp_attention runs the ring steps: "none" (one ring rank), "separate" (per-step fp32
    partials and a merge pass) or "fused" (one online softmax per query block across all steps)."""
    m = int(lib().usp_attention_ring_mode(B, S, H, D, int(causal), ulysses_degree, ring_degree,
                                          ORDERS[order], o_dt))
    if m < 0:
        raise UspError(USP_ERR_INVALID_ARG, "usp_attention_ring_mode", lib().usp_last_error().decode())
    return RING_MODES[m]


def usp_attention(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, o, lse,
                  workspace, workspace_bytes, seq_lens=None, head_counts=None, order="contiguous",
                  o_dt=None, stream=None):
    o_dt = _dtype(o) if o_dt is None else o_dt
    _check(lib().usp_attention(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, float(scale), int(causal),
                               ulysses_degree, ring_degree, _i32(seq_lens), _i32(head_counts),
                               ORDERS[order], _ptr(o), o_dt, _ptr(lse), _ptr(workspace),
                               workspace_bytes, _stream(stream)), "usp_attention")


def usp_attention_qkvpacked(qkv, B, S, H, D, scale, causal, ulysses_degree, ring_degree, o, lse,
                            workspace, workspace_bytes, seq_lens=None, head_counts=None,
                            order="contiguous", o_dt=None, stream=None):
    """usp_attention on a packed bf16 input qkv [B][S][3][H][D]."""
    o_dt = _dtype(o) if o_dt is None else o_dt
    _check(lib().usp_attention_qkvpacked(_ptr(qkv), B, S, H, D, float(scale), int(causal),
                                         ulysses_degree, ring_degree, _i32(seq_lens),
                                         _i32(head_counts), ORDERS[order], _ptr(o), o_dt,
                                         _ptr(lse), _ptr(workspace), workspace_bytes,
                                         _stream(stream)), "usp_attention_qkvpacked")


def usp_attention_events(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, o, lse,
                         workspace, workspace_bytes, events, seq_lens=None, head_counts=None,
                         order="contiguous", o_dt=None, stream=None) -> list[int]:
    """usp_attention that records 5 caller events between its phases; returns the kernels it
    launched per phase: [Q/K/V re-layout, attention, merge, output re-layout].
    ``events``: 5 raw cudaEvent_t handles (ints) or None entries."""
    o_dt = _dtype(o) if o_dt is None else o_dt
    ev = (ctypes.c_void_p * 5)(*[e or None for e in events])
    n = (ctypes.c_int * 4)()
    _check(lib().usp_attention_events(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, float(scale),
                                      int(causal), ulysses_degree, ring_degree, _i32(seq_lens),
                                      _i32(head_counts), ORDERS[order], _ptr(o), o_dt, _ptr(lse),
                                      _ptr(workspace), workspace_bytes, ev, n,
                                      _stream(stream)), "usp_attention_events")
    return list(n)


def usp_attention_noalloc(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, o, lse,
                          seq_lens=None, head_counts=None, order="contiguous", o_dt=None,
                          status=None, stream=None):
    """usp_attention on the library's built-in scratch (no workspace argument, no allocation)."""
    o_dt = _dtype(o) if o_dt is None else o_dt
    _check(lib().usp_attention_noalloc(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, float(scale),
                                       int(causal), ulysses_degree, ring_degree, _i32(seq_lens),
                                       _i32(head_counts), ORDERS[order], _ptr(o), o_dt, _ptr(lse),
                                       _ptr(status), _stream(stream)), "usp_attention_noalloc")


def usp_check_status(status, stream=None) -> int:
    """Returns the status code (USP_OK or USP_ERR_TIMEOUT/...) without raising."""
    return int(lib().usp_check_status(_ptr(status), _stream(stream)))


def usp_plan_pairs(S, ulysses_degree, ring_degree, causal, order="contiguous"):
    n = lib().usp_plan_pairs(S, ulysses_degree, ring_degree, int(causal), ORDERS[order], None, 0)
    if n < 0:
        raise UspError(USP_ERR_INVALID_ARG, "usp_plan_pairs", lib().usp_last_error().decode())
    buf = (ctypes.c_int32 * (8 * max(1, n)))()
    lib().usp_plan_pairs(S, ulysses_degree, ring_degree, int(causal), ORDERS[order], buf, n)
    return [tuple(buf[8 * i: 8 * i + 8]) for i in range(n)]


def usp_plan_chains(S, ulysses_degree, ring_degree, causal, order="contiguous"):
    """The fused ring's links: (u, r, row0, rows, step, r2, kv_rows, diag) per visible ring step of
    each piece of query rows."""
    n = lib().usp_plan_chains(S, ulysses_degree, ring_degree, int(causal), ORDERS[order], None, 0)
    if n < 0:
        raise UspError(USP_ERR_INVALID_ARG, "usp_plan_chains", lib().usp_last_error().decode())
    buf = (ctypes.c_int32 * (8 * max(1, n)))()
    lib().usp_plan_chains(S, ulysses_degree, ring_degree, int(causal), ORDERS[order], buf, n)
    return [tuple(buf[8 * i: 8 * i + 8]) for i in range(n)]


def usp_plan_deals(B, S, H, D, causal, ulysses_degree, ring_degree, order="contiguous",
                   o_dt=USP_BF16, sms=152):
    """Per attention launch: (work units, deal, modelled periods of that deal, modelled periods of
    the default deal), periods as floats."""
    args = (B, S, H, D, int(causal), ulysses_degree, ring_degree, ORDERS[order], o_dt, sms)
    n = lib().usp_plan_deals(*args, None, 0)
    if n < 0:
        raise UspError(USP_ERR_INVALID_ARG, "usp_plan_deals", lib().usp_last_error().decode())
    buf = (ctypes.c_int32 * (4 * max(1, n)))()
    lib().usp_plan_deals(*args, buf, n)
    return [(buf[4 * i], buf[4 * i + 1], buf[4 * i + 2] / 1000.0, buf[4 * i + 3] / 1000.0)
            for i in range(n)]


def usp_version() -> int:
    return int(lib().usp_version())


# --------------------------------------------------------------------------------------------
# Convenience wrapper: torch allocates the outputs and the workspace (device memory plumbing).
# --------------------------------------------------------------------------------------------

def attention(q, k, v, causal=False, ulysses_degree=1, ring_degree=1, order="contiguous",
              seq_lens=None, head_counts=None, scale=None, out_dtype=None, workspace=None,
              stream=None):
    """q, k, v: CUDA bf16 tensors [B][S][H][D].  Returns (out [B][S][H][D], lse fp32 [B][S][H])."""
    import torch
    B, S, H, D = q.shape
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    o_dt = USP_FP32 if out_dtype == torch.float32 else USP_BF16
    scale = D ** -0.5 if scale is None else scale
    o = torch.empty((B, S, H, D), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, S, H), dtype=torch.float32, device=q.device)
    nbytes = usp_attention_workspace_size(B, S, H, D, ulysses_degree, ring_degree, order, o_dt,
                                          causal)
    if nbytes == 0:
        raise UspError(USP_ERR_INVALID_ARG, "usp_attention_workspace_size",
                       lib().usp_last_error().decode())
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    usp_attention(q, k, v, B, S, H, D, scale, causal, ulysses_degree, ring_degree, o, lse,
                  workspace, nbytes, seq_lens, head_counts, order, o_dt, stream)
    return o, lse
