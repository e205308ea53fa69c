"""The seeded synthetic inputs follow their stated recipe (CPU only): the
SplitMix64 seed derivation against the generator's published output
sequence, AR(1) keys (lag-1 correlation rho, unit variance), heavy hitters
(rate and scale), shared prompt prefixes (the same physical blocks, one
reference per holder, the recursion continued per request), block
conservation, and determinism in the seed."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W

GAMMA = 0x9E3779B97F4A7C15
MASK = (1 << 64) - 1


def test_splitmix64_matches_the_published_sequence():
    # the first three outputs of SplitMix64 from state 0 (Steele, Lea, Flood;
    # the reference C code by S. Vigna)
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [W.splitmix64((i * GAMMA) & MASK) for i in range(3)]
    assert got == want


def test_seed_derivation_separates_tensors_and_layers():
    seeds = {W.derive_seed(20260001, t, l) for t in range(7) for l in range(36)}
    assert len(seeds) == 7 * 36
    assert all(0 <= s < (1 << 63) for s in seeds)


def keys_f64(st, r, h):
    """Request r's keys of kv head h in token order, from the pools."""
    wl = st.wl
    T = int(st.lengths[r])
    n = -(-T // wl.b)
    blocks = st.block_tables[r, :n].long()
    K = st.k_pools[0][blocks, h].reshape(n * wl.b, wl.d)[:T]
    return K.double().numpy()


def small(**kw):
    base = W.scaled(W.WORKLOADS["qwen3_36l"], L=1, R=8, N=32, group=1, prefix_blocks=0,
                    rho=0.0, hh_prob=0.0, spare_blocks=4)
    return W.scaled(base, **kw)


def test_ar1_keys_have_the_stated_correlation_and_unit_variance():
    st = W.build_cache(small(rho=0.9), "cpu", with_decode_q=False)
    lag1, var = [], []
    for r in range(st.wl.R):
        for h in range(st.wl.Hkv):
            K = keys_f64(st, r, h)
            a, b = K[:-1], K[1:]
            lag1.append((a * b).mean() / np.sqrt((a * a).mean() * (b * b).mean()))
            var.append(K.var(axis=0).mean())
    assert abs(np.mean(lag1) - 0.9) < 0.01
    assert abs(np.mean(var) - 1.0) < 0.05


def test_iid_keys_are_uncorrelated():
    st = W.build_cache(small(rho=0.0), "cpu", with_decode_q=False)
    K = keys_f64(st, 0, 0)
    a, b = K[:-1], K[1:]
    assert abs((a * b).mean()) < 0.02


def test_heavy_hitters_have_the_stated_rate_and_scale():
    wl = small(hh_prob=0.05)
    st = W.build_cache(wl, "cpu", with_decode_q=False)
    norms = np.concatenate([np.linalg.norm(keys_f64(st, r, h), axis=1)
                            for r in range(wl.R) for h in range(wl.Hkv)])
    heavy = norms > 4 * np.sqrt(wl.d)  # plain rows are near sqrt(d), heavy ones near 8 sqrt(d)
    n = norms.size
    assert abs(heavy.mean() - 0.05) < 4 * np.sqrt(0.05 * 0.95 / n)
    ratio = norms[heavy].mean() / norms[~heavy].mean()
    assert abs(ratio - wl.hh_scale) < 0.3


def test_shared_prefixes_are_one_set_of_blocks_per_group():
    wl = small(R=8, group=4, prefix_blocks=3, rho=0.9)
    st = W.build_cache(wl, "cpu", with_decode_q=False)
    tab, rc = st.block_tables, st.refcount
    for g0 in (0, 4):
        members = range(g0, g0 + 4)
        shared = tab[g0, :3]
        for r in members:
            assert torch.equal(tab[r, :3], shared)
        assert (rc[shared.long()] == 4).all()
        # past the prefix every member has blocks of its own and its own keys
        own = [set(tab[r, 3:].tolist()) for r in members]
        for i in range(4):
            for j in range(i + 1, 4):
                assert not own[i] & own[j]
        Ka, Kb = keys_f64(st, g0, 0), keys_f64(st, g0 + 1, 0)
        P = 3 * wl.b
        assert np.array_equal(Ka[:P], Kb[:P])
        assert not np.array_equal(Ka[P:], Kb[P:])
    assert not torch.equal(tab[0, :3], tab[4, :3])


def test_blocks_are_conserved():
    wl = small(R=8, group=4, prefix_blocks=3)
    st = W.build_cache(wl, "cpu", with_decode_q=False)
    tab = st.block_tables
    used = tab[tab >= 0]
    refs = torch.bincount(used.long(), minlength=st.num_blocks)
    assert torch.equal(refs.to(torch.int32), st.refcount)
    free = st.free_ids[:int(st.free_count)]
    assert (st.refcount[free.long()] == 0).all()
    assert int(st.free_count) + int((st.refcount > 0).sum()) == st.num_blocks


@pytest.mark.parametrize("seed_same", [True, False])
def test_inputs_are_determined_by_the_seed(seed_same):
    wl = small(R=2, N=8)
    a = W.build_cache(wl, "cpu")
    b = W.build_cache(wl, "cpu", seed=wl.seed if seed_same else wl.seed + 1)
    same = all(torch.equal(x, y) for x, y in zip(a.k_pools + a.v_pools + [a.window_q, a.decode_q],
                                                 b.k_pools + b.v_pools + [b.window_q, b.decode_q]))
    assert same == seed_same


def test_sample_snapshot_equals_the_full_build():
    """A sampled snapshot holds exactly the full build's rows, queries and
    per-request block structure (shared prefixes included), renumbered."""
    import numpy as np
    wl = W.scaled(W.WORKLOADS["qwen3_36l"], name="sample", L=3, R=12, group=4, prefix_blocks=2,
                  N=8, spare_blocks=10)
    st = W.build_cache(wl, "cpu")
    rows = [4, 5, 6, 7, 10]
    snap = W.sample_snapshot(wl, rows, [0, 2], device="cpu")
    tab = st.block_tables.numpy()
    for j, r in enumerate(rows):
        for li, l in enumerate([0, 2]):
            full_k = W.bf16_bits(st.k_pools[l])[tab[r]]
            full_v = W.bf16_bits(st.v_pools[l])[tab[r]]
            assert np.array_equal(snap["k_pools"][li][snap["block_tables"][j]], full_k)
            assert np.array_equal(snap["v_pools"][li][snap["block_tables"][j]], full_v)
            assert np.array_equal(snap["window_q"][li][j], W.bf16_bits(st.window_q[l][r]))
            assert np.array_equal(snap["decode_q"][li][j], W.bf16_bits(st.decode_q[l][r]))
    # rows 4..7 form a whole sharing group: its prefix blocks keep refcount 4
    pre = snap["block_tables"][0, :2]
    assert (snap["refcount"][pre] == 4).all()
    assert np.array_equal(snap["block_tables"][1, :2], pre)
    assert snap["free_count"] == len(rows) * wl.N
    used = np.unique(snap["block_tables"][snap["block_tables"] >= 0])
    assert np.array_equal(used, np.arange(used.size))
    assert snap["lengths"].tolist() == [wl.T] * len(rows)
