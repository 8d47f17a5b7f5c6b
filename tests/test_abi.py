"""The C ABI on the CPU: the library builds and loads, exports every declared symbol, validates
arguments without touching a GPU, and its chunk-pair planner agrees with the oracle's orderings."""
import ctypes
import heapq
import os
import re

import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import build, usp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INT32_MAX = 2**31 - 1


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return usp.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "usp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(usp_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert sorted(usp.EXPORTED) == names


def test_status_strings_and_version(L):
    assert usp.usp_version() == 100
    for s in range(7):
        assert L.usp_status_string(s)


def test_invalid_arguments_rejected_on_host(L):
    lens = (ctypes.c_int32 * 2)(3, 4)
    assert L.usp_relayout_seq2head(256, 512, 0, 1, 4, 8, 0, lens, None, None) == usp.USP_ERR_INVALID_ARG
    neg = (ctypes.c_int32 * 2)(3, -1)
    assert L.usp_relayout_seq2head(256, 512, 0, 1, 4, 8, 2, neg, None, None) == usp.USP_ERR_INVALID_ARG
    bad_heads = (ctypes.c_int32 * 2)(1, 1)
    assert L.usp_relayout_head2seq(256, 512, 0, 1, 4, 8, 2, lens, bad_heads, None) == usp.USP_ERR_INVALID_ARG
    assert "head_counts" in L.usp_last_error().decode()
    # D = 96 is valid but not built
    assert L.usp_attn_partial(256, 256, 256, 1, 1, 8, 8, 96, 96, 96, 1.0, None, None, 256, 1,
                              256, None, None) == usp.USP_ERR_UNSUPPORTED
    # misaligned q
    assert L.usp_attn_partial(258, 256, 256, 1, 1, 8, 8, 64, 64, 64, 1.0, None, None, 256, 1,
                              256, None, None) == usp.USP_ERR_INVALID_ARG
    # seq_lens not summing to the ring chunk
    sl = (ctypes.c_int32 * 2)(5, 5)
    assert L.usp_attention(256, 256, 256, 1, 11, 4, 64, 1.0, 0, 2, 1, sl, None, 0, 256, 1, 256,
                           256, 1 << 30, None) == usp.USP_ERR_INVALID_ARG
    # workspace too small
    assert L.usp_attention(256, 256, 256, 1, 10, 4, 64, 1.0, 0, 2, 1, sl, None, 0, 256, 1, 256,
                           256, 16, None) == usp.USP_ERR_WORKSPACE
    assert L.usp_lse_merge(0, 256, 0, 256, 0, 1, 1, 4, 256, 1, 256, None) == usp.USP_ERR_INVALID_ARG
    assert L.usp_lse_merge(17, 256, 0, 256, 0, 1, 1, 4, 256, 1, 256, None) == usp.USP_ERR_INVALID_ARG


def test_new_entry_points_validate_on_host(L):
    """The packed-QKV and multi-tensor entry points reject bad arguments before any launch."""
    lens = (ctypes.c_int32 * 2)(3, 4)
    two = (ctypes.c_void_p * 2)(256, 512)
    with_null = (ctypes.c_void_p * 2)(256, None)
    for f in (L.usp_relayout_seq2head_multi, L.usp_relayout_head2seq_multi):
        assert f(0, two, two, 0, 1, 4, 8, 2, lens, None, None) == usp.USP_ERR_INVALID_ARG
        assert f(4, two, two, 0, 1, 4, 8, 2, lens, None, None) == usp.USP_ERR_INVALID_ARG
        assert f(2, two, with_null, 0, 1, 4, 8, 2, lens, None, None) == usp.USP_ERR_INVALID_ARG
        assert "dst[1]" in L.usp_last_error().decode()
    # packed QKV: NULL input, misaligned input, D not built, workspace too small
    assert L.usp_attention_qkvpacked(None, 1, 10, 4, 64, 1.0, 0, 1, 1, None, None, 0, 256, 1, 256,
                                     256, 1 << 20, None) == usp.USP_ERR_INVALID_ARG
    assert L.usp_attention_qkvpacked(258, 1, 10, 4, 64, 1.0, 0, 1, 1, None, None, 0, 256, 1, 256,
                                     256, 1 << 20, None) == usp.USP_ERR_INVALID_ARG
    assert L.usp_attention_qkvpacked(256, 1, 10, 4, 96, 1.0, 0, 1, 1, None, None, 0, 256, 1, 256,
                                     256, 1 << 20, None) == usp.USP_ERR_UNSUPPORTED
    assert L.usp_attention_qkvpacked(256, 1, 10, 4, 64, 1.0, 0, 1, 2, None, None, 0, 256, 1, 256,
                                     256, 16, None) == usp.USP_ERR_WORKSPACE


def test_plans_are_reused_and_follow_the_override(L, monkeypatch):
    """Planning a long ring takes milliseconds; the library caches plans per argument set, so a
    repeated query is fast, and the USP_RING_MERGE override is part of the key."""
    import time
    monkeypatch.delenv("USP_RING_MERGE", raising=False)
    args = (1, 69632, 32, 128, 1, 1, 8, 1, 0)  # a shape no other test plans (16 half-chunks of 4352)
    t0 = time.perf_counter()
    first = L.usp_attention_ring_mode(*args)
    t1 = time.perf_counter()
    for _ in range(20):
        assert L.usp_attention_ring_mode(*args) == first
    t2 = time.perf_counter()
    assert (t2 - t1) / 20 < max(1e-3, (t1 - t0) / 10)
    monkeypatch.setenv("USP_RING_MERGE", "separate")
    assert L.usp_attention_ring_mode(*args) == 1
    assert L.usp_attention_workspace_size(*args) > 8 * 69632 * 32 * 128 * 4
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    assert L.usp_attention_ring_mode(*args) == 2
    assert L.usp_attention_workspace_size(*args) == 256


def test_split_fused_ring_choice(L, monkeypatch):
    """Qwen-Image 1328^2 over Ulysses 2 x ring 2 (non-causal, fused): 672 equal chains are 4.42
    rounds of 152 CTAs, and the model splits the last 6 blocks (rows 2048..3571) of the second
    ring chunk of the second Ulysses group into ring steps, whose fp32 partial slots are the
    whole workspace beyond the status word; USP_RING_SPLIT=0 turns the split off."""
    monkeypatch.delenv("USP_RING_MERGE", raising=False)
    monkeypatch.delenv("USP_RING_SPLIT", raising=False)
    args = (1, 7145, 24, 128, 2, 2, "contiguous", usp.USP_BF16, False)
    vec = 1524 * 12  # split rows x heads of the group
    align = lambda x: (x + 255) // 256 * 256
    assert usp.usp_attention_ring_mode(1, 7145, 24, 128, False, 2, 2, "contiguous", usp.USP_BF16) == "fused"
    assert usp.usp_attention_workspace_size(*args) == 256 + align(2 * vec * 128 * 4) + align(2 * vec * 4)
    monkeypatch.setenv("USP_RING_SPLIT", "0")
    assert usp.usp_attention_workspace_size(*args) == 256
    # causal rings are never split
    monkeypatch.delenv("USP_RING_SPLIT")
    assert usp.usp_attention_workspace_size(1, 65536, 32, 128, 1, 8, "zigzag", usp.USP_BF16, True) == 256


def test_workspace_size(L, monkeypatch):
    B, S, H, D = 1, 4608, 24, 128
    # contiguous Ulysses: Q/K/V are addressed in place and O is written in place -> status only
    assert usp.usp_attention_workspace_size(B, S, H, D, 2, 1) == 256
    # ring of 3 with separate ring steps: R fp32 partials of O and LSE
    monkeypatch.setenv("USP_RING_MERGE", "separate")
    r = usp.usp_attention_workspace_size(1, 1000, 4, 64, 1, 3)
    assert 3 * 1000 * 4 * 64 * 4 + 3 * 1000 * 4 * 4 <= r <= 3 * 1000 * 4 * 64 * 4 + 3 * 1000 * 4 * 4 + 1024
    # every ordering is addressed in place: zigzag needs no copies of Q, K, V, whether its
    # half-chunks are whole 128-row tiles (64K tokens, ring 8: 16 x 4096: a piece dimension) or
    # not (1000 tokens over 6 half-chunks; 65535 tokens: a span map per chunk)
    assert usp.usp_attention_workspace_size(1, 1000, 4, 64, 1, 3, "zigzag") == r
    zc = usp.usp_attention_workspace_size(1, 65536, 32, 128, 1, 8, "contiguous")
    assert usp.usp_attention_workspace_size(1, 65536, 32, 128, 1, 8, "zigzag") == zc > 8 * 65536 * 32 * 128 * 4
    assert (usp.usp_attention_workspace_size(1, 65535, 32, 128, 1, 8, "zigzag") ==
            usp.usp_attention_workspace_size(1, 65535, 32, 128, 1, 8, "contiguous"))
    # fused ring steps write the final output directly: no partial slots
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    assert usp.usp_attention_workspace_size(1, 1000, 4, 64, 1, 3) == 256
    assert usp.usp_attention_workspace_size(1, 65536, 32, 128, 1, 8, "zigzag", causal=True) == 256
    assert usp.usp_attention_workspace_size(1, 65535, 32, 128, 1, 8, "zigzag", causal=True) == 256
    assert usp.usp_attention_workspace_size(1, 1000, 4, 64, 1, 3, "zigzag") == 256
    assert usp.usp_attention_workspace_size(1, 10, 4, 96, 1, 1) == 0
    assert usp.usp_attention_workspace_size(1, 10, 4, 64, 5, 4) == 0


def test_ring_mode_choice(L, monkeypatch):
    """The ring mode follows the override, and without one the library's time model picks the
    fused ring for the long causal zigzag ring (no 6.7 GB partial round trip, 8192 long units) and
    the separate steps for a tiny ring whose units would not fill the GPU."""
    monkeypatch.delenv("USP_RING_MERGE", raising=False)
    assert usp.usp_attention_ring_mode(1, 4608, 24, 128, False, 2, 1) == "none"
    assert usp.usp_attention_ring_mode(1, 65536, 32, 128, True, 1, 8, "zigzag", usp.USP_BF16) == "fused"
    assert usp.usp_attention_ring_mode(1, 1000, 4, 64, False, 1, 3) == "separate"
    for mode in ("fused", "separate"):
        monkeypatch.setenv("USP_RING_MERGE", mode)
        assert usp.usp_attention_ring_mode(1, 1000, 4, 64, False, 1, 3) == mode
        assert usp.usp_attention_ring_mode(1, 1000, 4, 64, False, 1, 1) == "none"
    with pytest.raises(usp.UspError):
        usp.usp_attention_ring_mode(1, 10, 4, 96, False, 1, 2)


@pytest.mark.parametrize("S,U,R,causal,order", [
    (1000, 1, 3, False, "contiguous"), (65536, 1, 8, True, "zigzag"), (61, 1, 5, True, "zigzag"),
    (61, 1, 4, True, "stripe"), (7145, 2, 2, True, "contiguous"), (47, 2, 3, True, "stripe"),
    (19, 1, 8, True, "contiguous"), (5, 1, 8, True, "zigzag"), (300, 3, 1, True, "contiguous"),
])
def test_planner_matches_oracle_visibility(L, S, U, R, causal, order):
    """Every planned run reproduces, row by row, the number of visible keys the oracle's global
    positions give, and the runs of each (u, r, step) tile the ring chunk exactly."""
    pos = oracle.ring_positions(order, S, R)
    recs = usp.usp_plan_pairs(S, U, R, causal, order)
    cover = {}
    for (u, r, k, r2, q0, qlen, kvlen, diag) in recs:
        assert r2 == (r - k) % R
        qp = pos[r][q0:q0 + qlen]
        vis = (pos[r2][None, :] <= qp[:, None]).sum(axis=1) if causal else np.full(qlen, len(pos[r2]))
        i = np.arange(qlen)
        if diag == INT32_MAX:
            want = np.full(qlen, kvlen)
        else:
            want = np.clip(i + diag + 1, 0, kvlen)
        assert np.array_equal(vis, want), (u, r, k, q0)
        cover.setdefault((u, r, k), []).append((q0, qlen))
    assert len(cover) == U * R * sum(1 for p in pos if len(p) > 0)
    for (u, r, k), runs in cover.items():
        runs.sort()
        at = 0
        for q0, qlen in runs:
            assert q0 == at
            at += qlen
        assert at == len(pos[r])


@pytest.mark.parametrize("S,U,R,causal,order,split", [
    (65536, 1, 8, True, "zigzag", ""), (61, 1, 5, True, "zigzag", ""), (61, 1, 4, True, "stripe", ""),
    (7145, 2, 2, False, "contiguous", ""), (47, 2, 3, True, "stripe", ""), (19, 1, 8, True, "contiguous", ""),
    (5, 1, 8, True, "zigzag", ""), (1537, 1, 3, True, "zigzag", ""), (1000, 1, 3, False, "zigzag", ""),
    (32771, 1, 4, True, "stripe", ""), (65793, 1, 8, True, "zigzag", ""),
    # forced splits of non-causal fused rings: the split rows' ring-step segments
    (1000, 2, 2, False, "contiguous", "1"), (4481, 1, 3, False, "zigzag", "3"),
    (1537, 2, 4, False, "stripe", "2"), (7145, 2, 2, False, "contiguous", "0"),
])
def test_fused_chains_match_oracle_visibility(L, S, U, R, causal, order, split, monkeypatch):
    """The fused ring's pieces tile every ring chunk's query rows, each piece has at most one link
    per ring step, in ring order, and for every row the links' visible keys are exactly the keys
    of that ring step's chunk that the oracle's global positions allow (also for the rows of a
    split fused ring, whose ring steps are separate segments)."""
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    if split:
        monkeypatch.setenv("USP_RING_SPLIT", split)
    pos = oracle.ring_positions(order, S, R)
    recs = usp.usp_plan_chains(S, U, R, causal, order)
    pieces = {}
    for (u, r, row0, rows, k, r2, kvlen, diag) in recs:
        assert r2 == (r - k) % R
        pieces.setdefault((u, r, row0, rows), []).append((k, r2, kvlen, diag))
    for (u, r, row0, rows), links in pieces.items():
        steps = [k for k, *_ in links]
        assert steps == sorted(set(steps))  # ring order, each step once
        qp = pos[r][row0:row0 + rows]
        i = np.arange(rows)
        got = {k: (np.full(rows, kvlen) if diag == INT32_MAX else np.clip(i + diag + 1, 0, kvlen))
               for k, r2, kvlen, diag in links}
        for k in range(R):
            r2 = (r - k) % R
            want = ((pos[r2][None, :] <= qp[:, None]).sum(axis=1) if causal
                    else np.full(rows, len(pos[r2])))
            assert np.array_equal(got.get(k, np.zeros(rows, dtype=int)), want), (u, r, row0, k)
    for u in range(U):
        for r in range(R):
            spans = sorted((row0, rows) for (uu, rr, row0, rows) in pieces if uu == u and rr == r)
            at = 0
            for row0, rows in spans:
                assert row0 == at
                at += rows
            assert at == len(pos[r])


def test_planner_counts_every_causal_pair_once(L):
    """Across all ring steps, the planned runs see each causal (query, key) pair exactly once:
    sum over runs of the visible-key counts is S(S+1)/2, the count the FLOP figure uses."""
    for S, U, R, order in [(65536, 1, 8, "zigzag"), (7145, 2, 2, "contiguous"), (999, 1, 4, "stripe")]:
        total = 0
        for (u, r, k, r2, q0, qlen, kvlen, d) in usp.usp_plan_pairs(S, U, R, True, order):
            i = np.arange(qlen, dtype=np.int64)
            vis = np.full(qlen, kvlen) if d == INT32_MAX else np.clip(i + d + 1, 0, kvlen)
            if u == 0:
                total += int(vis.sum())
        assert total == S * (S + 1) // 2


def test_binding_signatures_match_header(L):
    """The ctypes argument list of every entry point has as many parameters as its declaration."""
    text = open(os.path.join(ROOT, "include", "usp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    for name in declared_functions():
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(getattr(L, name).argtypes) == len(params), name


def modelled_deal_periods(B, S, H, U, R, causal, order, bf16, deal, sms=152):
    """The unit-deal time model restated from the header over the fused ring's pieces: per Ulysses
    rank, the pieces longest first (by the key tiles of their longest block), every (batch, head)
    visiting their 256-row blocks in order (causal: last block first), reversed for odd (batch,
    head) indices under deal & 2; a unit costs its key tiles + 2 (bf16 O) or 2.5 (fp32 O).  Under
    deal & 4 each unit in turn goes to the CTA free first (lowest index among equals); otherwise
    unit i goes to CTA i % G in even rounds and, unless deal & 1, to G-1 - i % G in odd ones.
    With sms=None: the unit costs in numbering order instead."""
    pieces = {}
    for (u, r, row0, rows, k, r2, kvlen, diag) in usp.usp_plan_chains(S, U, R, causal, order):
        pieces.setdefault((u, r, row0, rows), []).append((kvlen, diag))

    def tiles(links, last):
        n = 0
        for kv, diag in links:
            m = kv - 1 if diag == INT32_MAX else min(kv - 1, last + diag)
            n += 0 if m < 0 else m // 128 + 1
        return n

    units = []
    for u in range(U):
        mine = sorted(((key[3], links) for key, links in pieces.items() if key[0] == u),
                      key=lambda p: -tiles(p[1], p[0] - 1))
        blocks = []
        for rows, links in mine:
            nb = -(-rows // 256)
            for qi in range(nb):
                qb = nb - 1 - qi if causal else qi
                blocks.append(tiles(links, min(rows, 256 * (qb + 1)) - 1) + (2.0 if bf16 else 2.5))
        for hb in range(B * H // U):
            units += blocks[::-1] if (deal & 2) and hb % 2 else blocks
    if sms is None:
        return units
    ctas = min(len(units), sms)
    load = [0.0] * ctas
    if deal & 4:
        free = [(0.0, c) for c in range(ctas)]
        for c in units:
            at, cta = heapq.heappop(free)
            load[cta] = at + c
            heapq.heappush(free, (at + c, cta))
        return max(load)
    for i, c in enumerate(units):
        t, pos = divmod(i, ctas)
        load[ctas - 1 - pos if not (deal & 1) and t % 2 else pos] += c
    return max(load)


@pytest.mark.parametrize("B,S,H,U,R,causal,order", [
    (1, 65536, 32, 1, 8, True, "zigzag"), (2, 1085, 3, 1, 4, True, "contiguous"),
    (2, 1536, 3, 1, 3, True, "zigzag"), (1, 32771, 32, 1, 4, True, "stripe"),
    (1, 12289, 4, 1, 2, True, "contiguous"), (2, 4481, 6, 2, 2, True, "stripe"),
    (1, 7145, 24, 2, 2, False, "contiguous"), (3, 3000, 10, 2, 3, False, "stripe"),
])
def test_unit_deal_model(L, B, S, H, U, R, causal, order, monkeypatch):
    """usp_plan_deals against the model restated over usp_plan_chains for every deal (forced with
    USP_UNIT_DEAL), and the library's own pick: among the snake, round-robin and dynamic deals,
    each with either block order, the one of least modelled time when it saves more than 0.5 %
    against the default (the first in that order among equals), else the default."""
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    monkeypatch.setenv("USP_RING_SPLIT", "0")
    for bf16 in (False, True):
        dt = usp.USP_BF16 if bf16 else usp.USP_FP32
        want = [modelled_deal_periods(B, S, H, U, R, causal, order, bf16, d) for d in range(8)]
        for d in range(8):
            monkeypatch.setenv("USP_UNIT_DEAL", str(d))
            ((n, deal, t, t0),) = usp.usp_plan_deals(B, S, H, 128, causal, U, R, order, dt)
            assert deal == d and abs(t - want[d]) < 1e-3 and abs(t0 - want[0]) < 1e-3, (d, t, want)
        monkeypatch.delenv("USP_UNIT_DEAL")
        ((n, deal, t, t0),) = usp.usp_plan_deals(B, S, H, 128, causal, U, R, order, dt)
        pick, best = 0, want[0]
        for d in (1, 2, 3, 4, 6):
            if want[d] < best and want[d] < 0.995 * want[0]:
                pick, best = d, want[d]
        assert deal == pick and abs(t - want[deal]) < 1e-3


def random_deal_cases(n, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        U, R = int(rng.integers(1, 4)), int(rng.integers(1, 6))
        H = U * int(rng.integers(1, 6))
        S = int(rng.integers(max(U * R, 2), 9000))
        out.append((int(rng.integers(1, 3)), S, H, U, R, bool(rng.integers(0, 2)),
                    ["contiguous", "zigzag", "stripe"][int(rng.integers(0, 3))]))
    return out


@pytest.mark.parametrize("B,S,H,U,R,causal,order", random_deal_cases(16))
def test_unit_deal_model_random_grids(L, B, S, H, U, R, causal, order, monkeypatch):
    """The same restatement on random grids (sequence lengths that split unevenly, 1-5 ring
    ranks, 1-3 Ulysses ranks, both batch sizes): every deal's modelled time matches, and none is
    below the mean CTA's work (the sum of all unit costs over the CTAs)."""
    monkeypatch.setenv("USP_RING_MERGE", "fused")
    monkeypatch.setenv("USP_RING_SPLIT", "0")
    for d in range(8):
        monkeypatch.setenv("USP_UNIT_DEAL", str(d))
        recs = usp.usp_plan_deals(B, S, H, 128, causal, U, R, order, usp.USP_BF16)
        if len(recs) != 1:
            continue  # more than one launch: the restatement covers one
        ((n, deal, t, t0),) = recs
        want = modelled_deal_periods(B, S, H, U, R, causal, order, True, d)
        assert deal == d and abs(t - want) < 1e-3, (d, t, want)
        units = modelled_deal_periods(B, S, H, U, R, causal, order, True, d, sms=None)
        assert n == len(units)
        assert t >= max(max(units), sum(units) / min(n, 152)) - 1e-6


def test_unit_deal_choices(L, monkeypatch):
    """The deals the model picks for the long causal rings: the dynamic deal for the 65793-token
    zigzag ring of 8 (its half-chunks of 4112 and 4111 rows end in short blocks, so each head's
    blocks differ in cost and the snake piles the long ones onto the same CTAs: 8 % shorter
    modelled) and for the 64K ring (1 %); the snake for the 16K ring (0.4 % is within the
    model's margin) and for FLUX (equal units: every deal models the same).  The query rejects
    a GPU without SMs."""
    for var in ("USP_UNIT_DEAL", "USP_RING_MERGE", "USP_RING_SPLIT"):
        monkeypatch.delenv(var, raising=False)
    ((n, deal, t, t0),) = usp.usp_plan_deals(1, 65793, 32, 128, True, 1, 8, "zigzag")
    assert deal == 4 and t < 0.95 * t0
    ((n, deal, t, t0),) = usp.usp_plan_deals(1, 65536, 32, 128, True, 1, 8, "zigzag")
    assert n == 8192 and deal == 4 and 0.985 * t0 < t < 0.995 * t0
    ((n, deal, t, t0),) = usp.usp_plan_deals(1, 16384, 32, 128, True, 1, 8, "zigzag")
    assert deal == 0 and t == t0
    ((n, deal, t, t0),) = usp.usp_plan_deals(1, 4608, 24, 128, False, 2, 1, "contiguous")
    assert n == 432 and deal == 0 and t == t0
    with pytest.raises(usp.UspError):
        usp.usp_plan_deals(1, 65536, 32, 128, True, 1, 8, "zigzag", sms=0)
    # the deal moves work between CTAs only: the workspace is the same under every forced deal
    sizes = set()
    for d in ("", "0", "3", "4", "6"):
        monkeypatch.setenv("USP_UNIT_DEAL", d)
        for args in ((1, 65793, 32, 128, 1, 8, "zigzag"), (1, 7145, 24, 128, 2, 2, "contiguous")):
            sizes.add((args, usp.usp_attention_workspace_size(*args, usp.USP_BF16, True)))
    assert len(sizes) == 2
