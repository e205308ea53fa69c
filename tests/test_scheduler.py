"""Hybrid scheduling simulator on the CPU, driven through the oracle
backend: host mirrors agree with the cache every step, every request
finishes, the hybrid policy preempts, compresses at the trigger and at
admission, and keeps more requests decoding than the strict policy."""
from __future__ import annotations

import numpy as np

from compressed_paged_kv_gb300 import scheduler as S
from tests.sched_oracle_backend import Draws, OracleBackend


def small_requests(n, seed):
    return S.synthetic_requests(n, seed, prompt=(10, 40), out_median=90, out_sigma=0.7,
                                out_max=300)


def run(orc, strict, slots=2, n=14, blocks=46):
    cfg = S.SimConfig(num_blocks=blocks, max_rows=16, n_max=4, w=4, query_slots=slots,
                      strict=strict, seed=1)
    be = OracleBackend(orc, cfg, L=1, Hkv=1, Hq=2, d=64, stride=24, draws=Draws(2))
    sch = S.Scheduler(cfg, be, small_requests(n, 3))

    def check(s):
        assert be.free_count() == s.free_blocks, "free blocks: mirror and cache differ"
        lengths = be.s["lengths"]
        for r in s.running:
            assert lengths[r.row] == r.length
            assert np.count_nonzero(be.s["tables"][r.row] >= 0) == r.held
        idle = [row for row in range(cfg.max_rows) if row in s.free_rows]
        assert np.all(lengths[idle] == 0) and np.all(be.s["tables"][idle] == -1)

    out = sch.run(max_steps=5000, check=check)
    assert out["finished"] == n
    assert be.free_count() == cfg.num_blocks and np.all(be.s["refcount"] == 0)
    return out


def test_hybrid_schedule_runs_to_completion(orc):
    h = run(orc, strict=False)
    assert h["preemptions"] > 0 and h["compressions"] > 0 and h["prefill_compressions"] > 0
    assert h["stalls"] > 0  # two query slots are a real limit


def test_hybrid_keeps_more_requests_decoding_than_strict(orc):
    """Same slot pool: strict runs at most 3 requests (one slot each), hybrid
    as many as the blocks allow."""
    h = run(orc, strict=False, slots=3)
    s = run(orc, strict=True, slots=3)
    assert s["preemptions"] == 0
    assert h["mean_decoding"] > s["mean_decoding"]
    assert h["steps"] < s["steps"]
