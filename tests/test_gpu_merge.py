"""GPU LSE merge against the oracle's pairwise ring-order merge (the pages' sigmoid form)."""
import numpy as np
import pytest

import oracle
from sequence_attention_tcgen05_gb300 import usp

from gpu_util import Guarded, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_parts,rows,H,D", [(1, 64, 2, 64), (2, 7145, 12, 128), (3, 1000, 4, 64),
                                              (8, 513, 3, 128), (16, 31, 2, 128)])
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_merge_matches_oracle(n_parts, rows, H, D, out):
    t = torch()
    rng = np.random.default_rng(n_parts * 1000 + rows)
    o = rng.standard_normal((n_parts, rows, H, D)).astype(np.float32)
    lse = (rng.standard_normal((n_parts, rows, H)) * 3).astype(np.float32)
    # empty partials: some (row, head) entries see no key in some parts, a few in all parts
    lse[rng.random(lse.shape) < 0.2] = -np.inf
    lse[:, :3, 0] = -np.inf
    o[np.isinf(lse)] = np.nan  # must never be read
    run_o, run_l = o[0].astype(np.float64), lse[0].astype(np.float64)
    for k in range(1, n_parts):
        run_o, run_l = oracle.merge(run_o, run_l, o[k], lse[k])
    run_o[~np.isfinite(run_l)] = 0.0
    dt = t.float32 if out == "fp32" else t.bfloat16
    oo = Guarded((rows, H, D), dt)
    ll = Guarded((rows, H), t.float32)
    usp.usp_lse_merge(n_parts, t.from_numpy(o).cuda(), rows * H * D, t.from_numpy(lse).cuda(),
                      rows * H, rows, H, D, oo.view, ll.view)
    t.cuda.synchronize()
    oo.check()
    ll.check()
    got_o = oo.view.float().cpu().numpy().astype(np.float64)
    got_l = ll.view.cpu().numpy().astype(np.float64)
    fin = np.isfinite(run_l)
    assert np.array_equal(np.isfinite(got_l), fin)
    assert np.all(got_o[~fin] == 0)
    tol = 1e-5 if out == "fp32" else 8e-3
    assert np.abs(got_o - run_o).max() <= tol * max(1.0, np.abs(run_o).max())
    assert np.abs(got_l[fin] - run_l[fin]).max() <= 2e-5 * max(1.0, np.abs(run_l[fin]).max())
