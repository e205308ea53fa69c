"""A compression without the debug outputs against one with them and the oracle.

The score and kept-index outputs are optional; asking for them must not change
what the call does.  Each case compresses the same state twice, without and
with the score output, and requires identical kept indices, pool bytes and
tables; the run without scores is also checked against the oracle (kept sets
exact or near-ties, compacted rows exact).  Degenerate inputs (all keys equal,
zero keys, exact ties from a handful of distinct keys, lambda 0 and negative,
a window of b tokens) are among the cases."""
import gc

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from compressed_paged_kv_gb300 import _build
    _build.build()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _snapshot(st):
    return ([t.clone() for t in st.k_pools + st.v_pools],
            [t.clone() for t in (st.block_tables, st.lengths, st.refcount, st.free_ids,
                                 st.free_count)])


def _restore(st, snap):
    pools, ints = snap
    for a, b in zip(st.k_pools + st.v_pools, pools):
        a.copy_(b)
    for a, b in zip((st.block_tables, st.lengths, st.refcount, st.free_ids, st.free_count), ints):
        a.copy_(b)


def _run(st, with_scores, cache):
    run = H.CompressRun(st, cache=cache, with_scores=with_scores)
    rc, dev = run.run()
    assert rc == zp.OK and dev == zp.OK, (rc, dev)
    torch.cuda.synchronize()
    return (run.kept.clone(), [t.view(torch.int16).clone() for t in st.k_pools + st.v_pools],
            H.int_state(st))


def without_equals_with_scores(st):
    """Runs the compression of `st` twice from the same state, without and with
    the score output, and requires identical results; returns the snapshot of
    the state before (`st` is left compressed)."""
    cache = H.make_cache(st)
    snap = _snapshot(st)
    kp, pp, ip = _run(st, False, cache)
    _restore(st, snap)
    kf, pf, i_f = _run(st, True, cache)
    assert torch.equal(kp, kf), "kept indices depend on the score output"
    for a, b in zip(pp, pf):
        assert torch.equal(a, b), "pool bytes depend on the score output"
    H.check_ints(ip, i_f)
    cache.close()
    return snap


ONE_CTA = [
    ("qwen3_1l", {}),
    ("T128_w4", dict(N=8, R=4, w=4)),
    ("T128_w16", dict(N=8, R=4, w=16)),
    ("T384", dict(N=24, R=2)),
    ("T512", dict(N=32, R=3)),
    ("d64_rows64", dict(d=64, N=32, w=16, R=2)),
    ("w1_G1", dict(Hq=8, w=1, N=16, R=3)),
    ("G8_rows64", dict(Hkv=2, Hq=16, N=16, w=8, R=2)),
    ("ar1_heavy_hitters", dict(N=32, R=4, rho=0.95, hh_prob=0.05)),
    ("shared_prefix", dict(N=16, R=6, group=3, prefix_blocks=5, spare_blocks=40)),
    ("lambda0", dict(N=16, R=2, lam=0.0)),
    ("lambda_big", dict(N=16, R=2, lam=50.0)),
    ("lambda_negative", dict(N=16, R=2, lam=-0.5)),
]


@pytest.mark.parametrize("name,changes", ONE_CTA, ids=[s[0] for s in ONE_CTA])
def test_without_scores_equals_with_and_oracle(orc, name, changes):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name=name, **changes)
    st = W.build_cache(wl, DEV, with_decode_q=False)
    snap = without_equals_with_scores(st)
    _restore(st, snap)
    rows = None if wl.R * wl.Hkv <= 64 else list(range(0, wl.R, 4))
    H.check_compress(orc, st, sample_rows=rows, with_scores=False)
    del st
    gc.collect()
    torch.cuda.empty_cache()


def test_cluster_without_scores_matches_oracle(orc):
    """Above 2048 tokens a cluster of CTAs owns a unit."""
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="T4096_no_scores", N=256, R=2)
    st = W.build_cache(wl, DEV, with_decode_q=False)
    without_equals_with_scores(st)


def test_qwen3_36l_sampled_without_scores(orc):
    wl = W.WORKLOADS["qwen3_36l"]
    st = W.build_cache(wl, DEV, with_decode_q=False)
    rng = np.random.default_rng(17)
    rows = sorted(set(range(0, 8)) | set(rng.choice(wl.R, 8, replace=False).tolist()))
    H.check_compress(orc, st, sample_rows=rows, sample_layers=[0, 35], with_scores=False)
    del st
    gc.collect()
    torch.cuda.empty_cache()


def _small(**changes):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="edge", **{**dict(N=8, R=3, spare_blocks=16),
                                                           **changes})
    return W.build_cache(wl, DEV, with_decode_q=False)


def test_all_equal_keys_without_scores(orc):
    """Every key equal: all scores tie and the b highest indices before the
    window are evicted."""
    st = _small()
    wl = st.wl
    row0 = st.block_tables[0].long()
    for l in range(wl.L):
        st.k_pools[l][row0] = st.k_pools[l][row0[0], :, :1].clone()
    snap = without_equals_with_scores(st)
    _restore(st, snap)
    run = H.CompressRun(st, with_scores=False)
    rc, dev = run.run()
    assert rc == zp.OK and dev == zp.OK
    kept = run.kept[0, 0].cpu().numpy()
    C, b = wl.C, wl.b
    for h in range(wl.Hkv):
        assert kept[h].tolist() == list(range(C - b)) + list(range(C, wl.T))


def test_zero_keys_without_scores(orc):
    """Zero keys have redundancy 0 and equal logits: ties throughout."""
    st = _small(R=2)
    for l in range(st.wl.L):
        st.k_pools[l][st.block_tables[1].long()] = 0
    snap = without_equals_with_scores(st)
    _restore(st, snap)
    H.check_compress(orc, st, with_scores=False)


def test_quantised_keys_many_ties(orc):
    """Keys drawn from 8 distinct vectors: many exactly equal scores."""
    st = _small(N=16, R=3)
    wl = st.wl
    g = torch.Generator(device="cpu").manual_seed(5)
    for l in range(wl.L):
        for r in range(wl.R):
            blk = st.block_tables[r, :wl.N].long()
            basis = torch.randn(8, wl.d, generator=g).to(torch.bfloat16)
            pick = torch.randint(0, 8, (wl.N, wl.Hkv, wl.b), generator=g)
            st.k_pools[l][blk] = basis[pick].to(DEV)
    snap = without_equals_with_scores(st)
    _restore(st, snap)
    H.check_compress(orc, st, with_scores=False)
