"""The reference arm of bench.py (the fp64 oracle on the host cores) keeps the
bench line's contract, without a GPU: one JSON line from rank 0 with the
product arm's metric, unit and direction, the steps it timed, a cpu_baseline
describing the run and an e2e block with no host-device bytes; other ranks
print nothing and exit 0."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(rank=0, world=1):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    return [ln for ln in p.stdout.splitlines() if ln.strip()]


def test_reference_line_keeps_the_contract():
    sys.path.insert(0, ROOT)
    import bench
    lines = run_bench()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    from compressed_paged_kv_gb300 import workloads as W
    wl = W.WORKLOADS["tiny"]
    assert d["config"] == bench.bench_config(wl, wl.R, 1)  # the GPU arm's config, key by key
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_other_ranks_print_nothing():
    assert run_bench(rank=1, world=2) == []
    lines = run_bench(rank=0, world=2)
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2


def test_samples_of_the_oracle_legs():
    """The CPU baseline of the shared-prefix workload times two whole sharing
    groups on every layer (>= 1,024 units); a reference step is a bounded
    slice (whole requests of one group, a subset of layers) that rotates."""
    sys.path.insert(0, ROOT)
    import bench
    from compressed_paged_kv_gb300 import workloads as W
    wl = W.WORKLOADS["qwen3_36l"]
    rows, layers = bench.baseline_sample(wl)
    assert len(rows) == 2 * wl.group and layers == list(range(wl.L))
    assert {r // wl.group for r in rows} == {0, wl.R // wl.group - 1}
    assert len(rows) * len(layers) * wl.Hkv >= 1024
    seen = set()
    for i in range(8):
        rows, layers = bench.reference_step_sample(wl, i)
        assert len({r // wl.group for r in rows}) == 1 and len(rows) == wl.group
        assert 0 < len(rows) * len(layers) * wl.Hkv <= 1024
        seen.add((rows[0], tuple(layers)))
    assert len(seen) == 8
    for name in ("qwen3_1l", "long4k"):
        wl = W.WORKLOADS[name]
        rows, layers = bench.baseline_sample(wl)
        assert len(rows) * len(layers) * wl.Hkv >= min(1024, wl.units())
        rows, layers = bench.reference_step_sample(wl, 3)
        assert len(rows) * len(layers) * wl.Hkv <= 1024


def test_moved_rows_count_of_the_algorithmic_bytes():
    """The bench's algorithmic bytes count 3 row copies per moved row: a row
    moves unless it keeps its position in the same physical block.  Hand-made
    kept sets over N = 3 blocks of b = 4 (8 destination rows, 4 evicted)."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    from compressed_paged_kv_gb300 import workloads as W
    wl = W.scaled(W.WORKLOADS["tiny"], b=4, N=3)
    src = torch.tensor([[10, 11, 12], [20, 21, 22]], dtype=torch.int32)
    kept = torch.tensor([[[[0, 1, 2, 3, 4, 5, 6, 7]],       # nothing evicted before row 8
                          [[0, 2, 3, 5, 6, 8, 9, 11]]],     # shifts from row 1 on: 7 move
                         ], dtype=torch.int32)
    # request 0 compacts in place; request 1 into two fresh blocks: all 8 move
    dst_in_place = src[:, :2].clone()
    assert bench.count_moved(kept[:, :1], src[:1], dst_in_place[:1], wl) == 0
    assert bench.count_moved(kept[:, 1:], src[1:], dst_in_place[1:], wl) == 7
    fresh = torch.tensor([[10, 11], [30, 31]], dtype=torch.int32)
    assert bench.count_moved(kept, src, fresh, wl) == 0 + 8
    # a row kept at its position but in a different destination block moves
    half = torch.tensor([[10, 99], [20, 21]], dtype=torch.int32)
    assert bench.count_moved(kept[:, :1], src[:1], half[:1], wl) == 4


def test_bench_parity_leg_matches_units_through_both_tables():
    """The bench's parity leg compares the oracle's compaction of a sampled
    snapshot (blocks renumbered) with a compaction of the full cache through
    that cache's own tables.  Here both sides are the oracle, so every unit
    must be byte-identical; a corrupted row must be counted as different."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from compressed_paged_kv_gb300 import workloads as W
    orc = oracle.load()
    wl = W.scaled(W.WORKLOADS["qwen3_36l"], name="parity_leg", L=2, R=8, group=4,
                  prefix_blocks=2, N=6, spare_blocks=24)
    st = W.build_cache(wl, "cpu")
    full = W.snapshot(st)
    fres = orc.compress(full["k_pools"], full["v_pools"], full["block_tables"], full["lengths"],
                        full["window_q"], wl.N, wl.w, wl.lam, full["free_ids"], full["free_count"],
                        full["refcount"], Hq=wl.Hq, want_scores=False, want_kept=False)
    assert fres["status"] == 0

    def rows_of(r, l):
        tab = fres["tables"][r, :wl.N - 1]
        return fres["kpools"][l][tab], fres["vpools"][l][tab]

    snap = W.sample_snapshot(wl, [0, 1, 2, 3], [0, 1], device="cpu", spare=16)
    _, _, sres = bench.oracle_step(orc, wl, snap, 2)
    par = bench.compacted_parity(wl, snap, sres, rows_of, [0, 1])
    assert par["units"] == 4 * 2 * wl.Hkv and par["byte_identical"] == par["units"]

    def corrupted(r, l):
        k, v = rows_of(r, l)
        k = k.copy()
        if r == 2 and l == 1:
            k[3, 1, 5, 0] ^= np.uint16(1)
        return k, v

    par = bench.compacted_parity(wl, snap, sres, corrupted, [0, 1], orc)
    assert par["byte_identical"] == par["units"] - 1
    assert par["near_ties"] == 0 and par["mismatches"] == 1


def test_bench_parity_near_tie_rule():
    """The bench's reading of a differing unit: the kept positions are read
    back from the compacted rows, and the unit is a near-tie only when every
    token in the symmetric difference scores within 1e-5 of the cut."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    rng = np.random.default_rng(5)
    Ks = rng.integers(0, 1 << 16, (12, 4), dtype=np.uint16)
    Vs = rng.integers(0, 1 << 16, (12, 4), dtype=np.uint16)
    kept = np.array([0, 1, 3, 4, 6, 8, 9, 10, 11])
    assert np.array_equal(bench.kept_of_rows(Ks, Vs, Ks[kept], Vs[kept]), kept)
    Kg = Ks[kept].copy()
    Kg[2, 1] ^= np.uint16(1)
    assert bench.kept_of_rows(Ks, Vs, Kg, Vs[kept]) is None
    # 10 candidates (w = 2), 3 evicted; the cut is the 3rd lowest score
    s = np.array([0.5, 0.4, 0.1, 0.3, 0.9, 0.2, 0.8, 0.6, 0.7, 0.95])
    imp, red = np.full(10, 0.1), np.full(12, 0.2)
    s_tie = s.copy()
    s_tie[3] = 0.3
    s_tie[1] = 0.3 + 1e-9                                   # tokens 1 and 3 tie at the cut
    # the oracle keeps 1 (higher), evicts 2, 5, 3; a GPU keeping 3 and evicting 1 differs
    kept_o = np.array([0, 1, 4, 6, 7, 8, 9, 10, 11])
    kept_g = np.array([0, 3, 4, 6, 7, 8, 9, 10, 11])
    assert bench.near_tie(s_tie, imp, red, 0.5, kept_o, kept_g, 3)
    s_far = s_tie.copy()
    s_far[1] = 0.35                                         # far from the cut
    assert not bench.near_tie(s_far, imp, red, 0.5, kept_o, kept_g, 3)
    assert bench.near_tie(s_tie, imp, red, 0.5, kept_o, kept_o, 3)


def test_packed_buffers_hold_each_tensor_at_an_aligned_offset():
    """The end-to-end loop's packed copies: one flat buffer, every tensor at a
    256-byte aligned offset, views that read back what was written."""
    sys.path.insert(0, ROOT)
    import torch
    import bench
    ts = [torch.arange(7, dtype=torch.int32), torch.randn(3, 5).to(torch.bfloat16),
          torch.arange(300, dtype=torch.int32).view(10, 30)]
    flat, views = bench.packed(torch, ts, "cpu")
    for v, t in zip(views, ts):
        v.copy_(t)
    for v, t in zip(views, ts):
        assert torch.equal(v, t) and v.shape == t.shape and v.dtype == t.dtype
        assert (v.data_ptr() - flat.data_ptr()) % 256 == 0
    assert flat.numel() == 256 + 256 + 1280
