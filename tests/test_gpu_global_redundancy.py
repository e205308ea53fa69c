"""GPU parity of the all-keys redundancy ablation against the oracle's
pair-by-pair definition, for both kernels: zp_global_redundancy (sums of the
normalised keys) and zp_global_redundancy_gram (the dense Gram of every unit
on the tensor cores).  Per unit, |r_gpu - r_orc| <= 1e-4 * max(|r_orc|,
mean |r_orc|) (fp32 against fp64 pairwise cosines)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
RTOL = 1e-4


def gather(pool, table_row, T, h):
    n = -(-T // 16)
    x = pool[table_row[:n].long(), h]
    return W.bf16_bits(x.reshape(n * 16, -1)[:T])


@pytest.mark.parametrize("gram", [False, True], ids=["sum_of_keys", "dense_gram"])
@pytest.mark.parametrize("lens,d", [([2048, 1000, 17, 16, 1, 300], 128), ([700, 64, 5], 64),
                                    ([4096, 257, 255, 129, 128], 128), ([4200, 130], 128),
                                    ([4500, 4097, 200], 64)])
def test_global_redundancy_matches_pairwise(orc, lens, d, gram):
    c = W.prefill_cache(500 + d, lens, 8, L=2, Hkv=2, Hq=4, d=d, w=4, device=DEV)
    # a few zero keys: cosine 0 with everything, redundancy 0
    c["k_pools"][0][c["tables"][1, 0], 0, 3] = 0
    c["k_pools"][1][c["tables"][0, 2], 1, 0] = 0
    # the slots past each length in its last block hold NaN bits: never keys
    for r, T in enumerate(lens):
        if T % 16:
            for l in range(2):
                c["k_pools"][l][c["tables"][r, T // 16], :, T % 16:] = float("nan")
    cache = zp.Cache(c["k_pools"], c["v_pools"], c["Hq"], max_requests=len(lens),
                     max_blocks_per_req=c["stride"])
    red = torch.full((2, len(lens), 2, c["stride"] * 16), float("nan"), device=DEV)
    cache.global_redundancy(c["tables"], c["lengths"], red, gram=gram)
    assert cache.status() == zp.OK
    got = red.cpu().numpy()
    worst = 0.0
    for l in range(2):
        for r, T in enumerate(lens):
            for h in range(2):
                K = gather(c["k_pools"][l], c["tables"][r], T, h)
                want = orc.redundancy_global(K)
                g = got[l, r, h, :T].astype(np.float64)
                scale = max(float(np.mean(np.abs(want))), 1e-30)
                err = np.abs(g - want) / np.maximum(np.abs(want), scale)
                worst = max(worst, float(err.max()))
                assert np.all(np.isnan(got[l, r, h, T:])), "written past the length"
                if T <= 16:  # one block: the block-local score
                    assert np.allclose(want, orc.redundancy(K, 16), atol=1e-12)
    print(f"[parity] global redundancy ({'dense Gram' if gram else 'sum of keys'}): "
          f"max rel err {worst:.2e}")
    assert worst <= RTOL


def test_dense_gram_agrees_with_sum_of_keys_at_scale():
    """The two kernels on the bench workload's 512 units (T = 2048, d = 128)."""
    wl = W.WORKLOADS["qwen3_1l"]
    st = W.build_cache(wl, DEV, with_decode_q=False)
    cache = zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=wl.R,
                     max_blocks_per_req=st.block_tables.shape[1])
    shape = (wl.L, wl.R, wl.Hkv, st.block_tables.shape[1] * 16)
    a = torch.full(shape, float("nan"), device=DEV)
    b = torch.full(shape, float("nan"), device=DEV)
    cache.global_redundancy(st.block_tables, st.lengths, a)
    cache.global_redundancy(st.block_tables, st.lengths, b, gram=True)
    assert cache.status() == zp.OK
    T = wl.T
    x, y = a[..., :T].double(), b[..., :T].double()
    scale = x.abs().mean(dim=-1, keepdim=True)
    rel = ((x - y).abs() / torch.maximum(x.abs(), scale)).max().item()
    print(f"[parity] dense Gram vs sum of keys, 512 units: max rel diff {rel:.2e}")
    assert rel <= 2 * RTOL


@pytest.mark.parametrize("gram", [False, True], ids=["sum_of_keys", "dense_gram"])
def test_global_redundancy_bad_length_is_flagged(gram):
    c = W.prefill_cache(510, [100], 8, L=1, Hkv=2, Hq=2, d=64, w=1, device=DEV)
    c["lengths"][0] = c["stride"] * 16 + 1
    cache = zp.Cache(c["k_pools"], c["v_pools"], 2, max_requests=1, max_blocks_per_req=c["stride"])
    red = torch.zeros(1, 1, 2, c["stride"] * 16, device=DEV)
    cache.global_redundancy(c["tables"], c["lengths"], red, gram=gram)
    assert cache.status() == zp.ERR_DEVICE_CHECK
    assert torch.count_nonzero(red) == 0


def test_dense_gram_many_items_per_cta(orc):
    """Ragged lengths over more work items than the persistent kernel has CTAs
    (384 units x 6 row tiles: about 15 items per CTA, items past a unit's
    length skipped, odd tile counts): a seeded sample of units against the
    oracle, every unit against the sum-of-keys kernel, nothing written past a
    length."""
    rng = np.random.default_rng(515)
    lens = [int(x) for x in rng.integers(1, 1500, size=24)]
    lens[0], lens[1] = 1500, 129
    c = W.prefill_cache(515, lens, 8, L=2, Hkv=8, Hq=8, d=128, w=4, device=DEV)
    cache = zp.Cache(c["k_pools"], c["v_pools"], c["Hq"], max_requests=len(lens),
                     max_blocks_per_req=c["stride"])
    shape = (2, len(lens), 8, c["stride"] * 16)
    a = torch.full(shape, float("nan"), device=DEV)
    b = torch.full(shape, float("nan"), device=DEV)
    cache.global_redundancy(c["tables"], c["lengths"], a, gram=True)
    cache.global_redundancy(c["tables"], c["lengths"], b)
    assert cache.status() == zp.OK
    worst = 0.0
    for r, T in enumerate(lens):
        x, y = a[:, r, :, :T].double(), b[:, r, :, :T].double()
        scale = x.abs().mean(dim=-1, keepdim=True).clamp_min(1e-30)
        worst = max(worst, ((x - y).abs() / torch.maximum(x.abs(), scale)).max().item())
        assert torch.isnan(a[:, r, :, T:]).all(), "written past the length"
    assert worst <= 2 * RTOL, worst
    got = a.cpu().numpy()
    picks = [(0, 0, 0), (1, 0, 7), (0, 1, 3)] + [
        (int(rng.integers(2)), int(rng.integers(len(lens))), int(rng.integers(8)))
        for _ in range(9)]
    worst = 0.0
    for l, r, h in picks:
        T = lens[r]
        K = gather(c["k_pools"][l], c["tables"][r], T, h)
        want = orc.redundancy_global(K)
        g = got[l, r, h, :T].astype(np.float64)
        scale = max(float(np.mean(np.abs(want))), 1e-30)
        worst = max(worst, float((np.abs(g - want) / np.maximum(np.abs(want), scale)).max()))
    print(f"[parity] dense Gram, {len(lens) * 16} units ragged: max rel err {worst:.2e}")
    assert worst <= RTOL
