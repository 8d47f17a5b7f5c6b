"""Back-to-back launches that depend on each other.  The re-layout and merge kernels are launched
with programmatic dependent launch: each may be scheduled while the previous kernel of the stream
drains, computes its first addresses, and only then waits for that kernel to complete.  These
chains check, without any host synchronisation between the launches, that every kernel reads
what the kernel before it wrote (read after write) and writes nothing the kernel before it still
reads (write after read)."""
import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import usp

from gpu_util import bits_of, torch

pytestmark = pytest.mark.gpu

# Ulysses splits of S = 4608 tokens and H = 24 heads: the head-side layout differs for each, so a
# head->seq launch that read its input early (the previous split's layout) would scramble the
# round trip, and a seq->head launch that wrote early would overwrite the input of the head->seq
# launch still running before it.
SPLITS = [
    ([2304, 2304], None),
    ([1536, 1536, 1536], None),
    ([1000, 3608], [10, 14]),
    ([1152, 1152, 1152, 1152], [6, 6, 6, 6]),
    ([921, 921, 922, 922, 922], [5, 5, 5, 5, 4]),
]


def test_relayout_chain_round_trips():
    t = torch()
    B, S, H, D = 1, 4608, 24, 128
    rng = np.random.default_rng(21)
    src = rng.integers(0, 2**16, size=B * S * H * D, dtype=np.uint64).astype(np.uint16)
    x = t.from_numpy(src.view(np.int16).copy()).view(t.bfloat16).cuda()
    y = t.empty_like(x)
    t.cuda.synchronize()
    for lens, heads in SPLITS * 2:  # 20 launches, each consuming the previous one's output
        usp.usp_relayout_seq2head(x, y, B, H, D, lens, heads)
        usp.usp_relayout_head2seq(y, x, B, H, D, lens, heads)
    t.cuda.synchronize()
    assert np.array_equal(bits_of(x), src)
    lens, heads = SPLITS[-1]
    assert np.array_equal(bits_of(y), oracle.seq2head(src, B, H, D, lens, heads))


def test_copy_then_merge_chain():
    """Each round: an identity re-layout (one part) copies fresh partials into the buffer that
    the merge reads, and the merge writes its own output buffer.  A merge that read early would
    see the previous round's partials; a copy that wrote early would change the partials under
    the previous round's merge."""
    t = torch()
    NP, rows, H, D = 2, 4608, 24, 128
    rng = np.random.default_rng(22)
    rounds = 4
    o_src = [rng.standard_normal((NP, rows, H, D)).astype(np.float32) for _ in range(rounds)]
    l_src = [(rng.standard_normal((NP, rows, H)) * 3).astype(np.float32) for _ in range(rounds)]
    o_dev = [t.from_numpy(a).cuda() for a in o_src]
    l_dev = [t.from_numpy(a).cuda() for a in l_src]
    o_parts = t.empty((NP, rows, H, D), dtype=t.float32, device="cuda")
    l_parts = t.empty((NP, rows, H), dtype=t.float32, device="cuda")
    outs = [(t.empty((rows, H, D), dtype=t.float32, device="cuda"),
             t.empty((rows, H), dtype=t.float32, device="cuda")) for _ in range(rounds)]
    t.cuda.synchronize()
    for i in range(rounds):
        usp.usp_relayout_seq2head(o_dev[i], o_parts, NP, H, D, [rows])
        usp.usp_relayout_seq2head(l_dev[i], l_parts, NP, H, 1, [rows])
        usp.usp_lse_merge(NP, o_parts, rows * H * D, l_parts, rows * H, rows, H, D, outs[i][0],
                          outs[i][1])
    t.cuda.synchronize()
    for i in range(rounds):
        run_o, run_l = o_src[i][0].astype(np.float64), l_src[i][0].astype(np.float64)
        for k in range(1, NP):
            run_o, run_l = oracle.merge(run_o, run_l, o_src[i][k], l_src[i][k])
        got_o = outs[i][0].cpu().numpy().astype(np.float64)
        got_l = outs[i][1].cpu().numpy().astype(np.float64)
        assert np.abs(got_o - run_o).max() <= 1e-5 * max(1.0, np.abs(run_o).max()), i
        assert np.abs(got_l - run_l).max() <= 2e-5 * max(1.0, np.abs(run_l).max()), i
