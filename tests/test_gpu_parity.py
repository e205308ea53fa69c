"""GPU parity of compression and decode attention against the CPU oracle,
through the C ABI.  Workload sizes: the tiny and single-layer Qwen3-8B cases in
full, the 36-layer, long-budget and mixed cases at full size on sampled units,
plus edge cases (ragged and degenerate shapes, ties, shared blocks, errors)."""
import gc
import math

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


def _free():
    gc.collect()
    torch.cuda.empty_cache()


# ------------------------------------------------------------ the workloads

def test_tiny_compress_then_decode(orc):
    wl = W.WORKLOADS["tiny"]
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    rep = H.check_compress(orc, st)
    assert rep.units == wl.units()
    # one decode step: a new token in the first slot of the reserved block
    N, b = wl.N, wl.b
    assert st.lengths.tolist() == [(N - 1) * b] * wl.R
    g = torch.Generator().manual_seed(W.derive_seed(wl.seed, 99))
    for l in range(wl.L):
        for r in range(wl.R):
            blk = int(st.block_tables[r, N - 1])
            st.k_pools[l][blk, :, 0] = torch.randn(wl.Hkv, wl.d, generator=g).to(torch.bfloat16).to(DEV)
            st.v_pools[l][blk, :, 0] = torch.randn(wl.Hkv, wl.d, generator=g).to(torch.bfloat16).to(DEV)
    st.lengths += 1
    H.check_decode(orc, st, 0, cache=cache)


def test_qwen3_1l_full(orc):
    wl = W.WORKLOADS["qwen3_1l"]
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    rep = H.check_compress(orc, st)
    assert rep.units == 512
    H.check_decode(orc, st, 0, cache=cache)
    del st, cache
    _free()


def test_qwen3_36l_shared_sampled(orc):
    wl = W.WORKLOADS["qwen3_36l"]
    st = W.build_cache(wl, DEV, with_decode_q=False)
    rng = np.random.default_rng(7)
    groups = [0, 31]
    rows = sorted(set(r for gi in groups for r in range(gi * 8, gi * 8 + 8))
                  | set(rng.choice(wl.R, 8, replace=False).tolist()))
    H.check_compress(orc, st, sample_rows=rows, sample_layers=[0, 17, 35])
    del st
    _free()


def test_long4k_sampled(orc):
    wl = W.WORKLOADS["long4k"]
    st = W.build_cache(wl, DEV, with_decode_q=False)
    rng = np.random.default_rng(8)
    rows = sorted(rng.choice(wl.R, 12, replace=False).tolist())
    H.check_compress(orc, st, sample_rows=rows, sample_layers=[0, 35])
    del st
    _free()


def test_mixed_sampled(orc):
    wl = W.WORKLOADS["mixed"]
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    rng = np.random.default_rng(9)
    H.check_compress(orc, st, sample_rows=sorted(rng.choice(51, 10, replace=False).tolist()),
                     sample_layers=[0, 31])
    dec = st.decode_rows[torch.as_tensor(sorted(rng.choice(461, 48, replace=False).tolist()),
                                         device=DEV).long()]
    H.check_decode(orc, st, 5, rows=dec, cache=cache)
    del st, cache
    _free()


# --------------------------------------------------------------- edge cases

SHAPES = [
    # (name, changes) on top of the single-layer Qwen3-8B workload
    # up to 2048 tokens one CTA owns a unit; beyond, a cluster of T / 2048 CTAs
    # (rank merge of the candidates up to 4 CTAs, k-way merge above)
    ("T512_one_cta", dict(N=32, R=3)),
    ("T1024_one_cta", dict(N=64, R=2)),
    ("T4096_cluster2", dict(N=256, R=2)),
    ("T6144_cluster3", dict(N=384, R=1)),
    ("T8192_cluster4", dict(N=512, R=1)),
    ("T10240_cluster5_kway", dict(N=640, R=1)),
    ("T16384_cluster8_kway", dict(N=1024, R=1, Hkv=2, Hq=8)),
    ("T32768_cluster16_kway", dict(N=2048, R=1, Hkv=2, Hq=8)),
    ("T384_one_cta", dict(N=24, R=2)),
    ("d64_rows64", dict(d=64, N=32, w=16, R=2)),
    ("w1_G1", dict(Hq=8, w=1, N=16, R=3)),
    ("G8_rows64", dict(Hkv=2, Hq=16, N=16, w=8, R=2)),
    ("L3_two_layers_more", dict(L=3, N=16, R=2)),
    ("ar1_heavy_hitters", dict(N=32, R=4, rho=0.95, hh_prob=0.05)),
    ("shared_prefix", dict(N=16, R=6, group=3, prefix_blocks=5, spare_blocks=40)),
    ("lambda0", dict(N=16, R=2, lam=0.0)),
    ("lambda_big", dict(N=16, R=2, lam=50.0)),
]


@pytest.mark.parametrize("name,changes", SHAPES, ids=[s[0] for s in SHAPES])
def test_shapes(orc, name, changes):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name=name, **changes)
    st = W.build_cache(wl, DEV)
    H.check_compress(orc, st)
    H.check_decode(orc, st, wl.L - 1)


def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("kind", ["tail_few", "tail_many", "T256", "d64_T512"])
@pytest.mark.parametrize("with_scores", [True, False])
def test_more_units_than_sms(orc, kind, with_scores):
    """More one-CTA units than SMs, not a multiple of them (several waves,
    the first-wave pairing on every SM, a ragged last wave): every unit is
    checked against the oracle."""
    S = _num_sms()
    Hkv = 8
    if kind == "tail_few":
        R, changes = S // Hkv + 1, {}
    elif kind == "tail_many":
        R, changes = (2 * S - 8) // Hkv, {}
    elif kind == "T256":
        R, changes = S // Hkv + 3, dict(N=16)
    else:
        R, changes = S // Hkv + 2, dict(N=32, d=64)
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name=f"units_{kind}", R=R, Hkv=Hkv, **changes)
    units = wl.units()
    assert units >= S and units % S != 0
    st = W.build_cache(wl, DEV, with_decode_q=False)
    rep = H.check_compress(orc, st, with_scores=with_scores)
    assert rep.units == units
    del st
    _free()


def _small_state(**changes):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="edge", **{**dict(N=8, R=3, spare_blocks=16),
                                                           **changes})
    return W.build_cache(wl, DEV)


def test_all_equal_keys_evicts_highest_indices(orc):
    st = _small_state()
    wl = st.wl
    row0 = st.block_tables[0].long()
    for l in range(wl.L):
        st.k_pools[l][row0] = st.k_pools[l][row0[0], :, :1].clone()  # one key everywhere
    run = H.CompressRun(st)
    rc, dev = run.run()
    assert rc == zp.OK and dev == zp.OK
    kept = run.kept[0, 0].cpu().numpy()
    C, b = wl.C, wl.b
    for h in range(wl.Hkv):
        assert kept[h].tolist() == list(range(C - b)) + list(range(C, wl.T))


def test_fully_shared_request(orc):
    """Two requests with identical tables (every block refcount 2, the
    reserved one included): both compress into fresh blocks, the old blocks
    are all freed and stay byte-identical."""
    st = _small_state(R=2, spare_blocks=40)
    shared = st.block_tables[0].clone()
    old1 = st.block_tables[1].clone()
    st.block_tables[1] = st.block_tables[0]
    st.refcount[st.block_tables[0].long()] = 2
    st.refcount[old1.long()] = 0
    fc = int(st.free_count.item())
    st.free_ids[fc:fc + old1.numel()] = old1
    st.free_count += old1.numel()
    H.check_compress(orc, st)
    assert int(st.refcount[shared.long()].sum()) == 0


def test_partial_holders(orc):
    """Refcount 3 on a prefix with only two of its holders compressing."""
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="partial", N=8, R=6, group=3, prefix_blocks=2,
                  spare_blocks=32, mixed=True, mixed_compress=3, mixed_len_lo=128)
    st = W.build_cache(wl, DEV)
    # force a deterministic compressing set: rows 0, 1 (group 0) and 4 (group 1)
    rows = torch.tensor([0, 1, 4], dtype=torch.int32, device=DEV)
    st.lengths[:] = wl.N * wl.b
    st.compress_rows = rows
    st.window_q = st.window_q[:, :3].contiguous()
    H.check_compress(orc, st)


def _assert_unchanged(st, before_pools, before_ints):
    after = H.int_state(st)
    for k in ("tables", "lengths", "refcount", "free_ids"):
        assert np.array_equal(after[k], before_ints[k]), k
    assert after["free_count"] == before_ints["free_count"]
    for l in range(st.wl.L):
        assert torch.equal(st.k_pools[l], before_pools[l][0])
        assert torch.equal(st.v_pools[l], before_pools[l][1])


def _snap(st):
    return [(k.clone(), v.clone()) for k, v in zip(st.k_pools, st.v_pools)], H.int_state(st)


@pytest.mark.parametrize("fault", ["out_of_blocks", "bad_length", "bad_block_id",
                                   "duplicate_row", "row_out_of_range"])
def test_device_errors_leave_state_unchanged(orc, fault):
    wl = W.scaled(W.WORKLOADS["tiny"], name="faults")
    st = W.build_cache(wl, DEV)
    req_idx = None
    expect = zp.ERR_INVALID_ARG
    if fault == "out_of_blocks":
        st.free_count.fill_(1)  # two targets are needed
        expect = zp.ERR_OUT_OF_BLOCKS
    elif fault == "bad_length":
        st.lengths[1] -= 1
    elif fault == "bad_block_id":
        st.block_tables[1, 3] = st.refcount.numel() + 5
    elif fault == "duplicate_row":
        req_idx = torch.tensor([1, 1], dtype=torch.int32, device=DEV)
    elif fault == "row_out_of_range":
        req_idx = torch.tensor([0, 7], dtype=torch.int32, device=DEV)
    pools, ints = _snap(st)
    cache = H.make_cache(st)
    rc = cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam,
                        st.free_ids, st.free_count, st.refcount, req_idx=req_idx)
    assert rc == zp.OK
    assert cache.status() == expect
    assert cache.status() == zp.OK  # reading clears the sticky word
    _assert_unchanged(st, pools, ints)


def test_host_argument_errors():
    wl = W.WORKLOADS["tiny"]
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    pool = zp.zp_block_pool(st.free_ids.data_ptr(), st.free_count.data_ptr(),
                            st.refcount.data_ptr(), st.free_ids.numel())
    h = cache.handle
    args = dict(block_tables=st.block_tables.data_ptr(), bt_stride=wl.N, num_rows=wl.R,
                lengths=st.lengths.data_ptr(), req_idx=0, R=wl.R,
                window_q=st.window_q.data_ptr(), n_max=wl.N, window=wl.w, lam=0.5, pool=pool,
                stream=torch.cuda.current_stream().cuda_stream)
    assert zp.zp_compress(h, **{**args, "window": 0}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "window": 17}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "n_max": 1}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "bt_stride": wl.N - 1}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "n_max": 7, "bt_stride": 8}) == zp.ERR_UNSUPPORTED
    assert zp.zp_compress(h, **{**args, "window_q": 0}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "window_q": st.window_q.data_ptr() + 2}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "lam": float("nan")}) == zp.ERR_INVALID_ARG
    assert zp.zp_compress(h, **{**args, "R": 0}) == zp.OK
    q = torch.zeros((wl.R, wl.Hq, wl.d), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros_like(q)
    dargs = dict(layer=0, q=q.data_ptr(), block_tables=st.block_tables.data_ptr(), bt_stride=wl.N,
                 num_rows=wl.R, lengths=st.lengths.data_ptr(), req_idx=0, R=wl.R, scale=0.125,
                 out=out.data_ptr(), stream=torch.cuda.current_stream().cuda_stream)
    assert zp.zp_paged_decode_attn(h, **{**dargs, "layer": 1}) == zp.ERR_INVALID_ARG
    assert zp.zp_paged_decode_attn(h, **{**dargs, "q": 0}) == zp.ERR_INVALID_ARG
    assert zp.zp_paged_decode_attn(h, **{**dargs, "R": wl.R + 1}) == zp.ERR_INVALID_ARG
    assert cache.status() == zp.OK


# ------------------------------------------------------------------- decode

@pytest.mark.parametrize("d,Hkv,Hq", [(128, 8, 32), (64, 2, 4), (128, 4, 4), (64, 1, 16)])
def test_decode_ragged_lengths(orc, d, Hkv, Hq):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="ragged", d=d, Hkv=Hkv, Hq=Hq, N=20, R=9,
                  spare_blocks=8)
    st = W.build_cache(wl, DEV)
    lens = torch.tensor([0, 1, 15, 16, 17, 100, 255, 319, 320], dtype=torch.int32, device=DEV)
    H.check_decode(orc, st, 0, lengths=lens)
    H.check_decode(orc, st, 0, lengths=lens, scale=0.05)


def test_decode_ignores_slots_past_the_length(orc):
    """NaN bits in the K and V slots past each length in its last block: the
    output stays finite and equal to the oracle's."""
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="nan_tail", N=20, R=9, spare_blocks=8)
    st = W.build_cache(wl, DEV)
    lens = torch.tensor([0, 1, 15, 16, 17, 100, 255, 319, 320], dtype=torch.int32, device=DEV)
    for r, T in enumerate(lens.tolist()):
        if T % 16:
            blk = st.block_tables[r, T // 16]
            st.k_pools[0][blk, :, T % 16:] = float("nan")
            st.v_pools[0][blk, :, T % 16:] = float("inf")
    H.check_decode(orc, st, 0, lengths=lens)


def test_decode_bad_length_is_flagged(orc):
    wl = W.scaled(W.WORKLOADS["tiny"], name="badlen")
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    lens = torch.tensor([5, wl.N * wl.b + 1], dtype=torch.int32, device=DEV)
    q = st.decode_q[0].contiguous()
    out = torch.zeros_like(q)
    assert cache.decode(0, q, st.block_tables, lens, 0.125, out) == zp.OK
    assert cache.status() == zp.ERR_DEVICE_CHECK


def test_overlapped_compress_and_decode_match_serial(orc):
    """Compression of the requests at N_max on one stream while the others
    decode on a second stream (disjoint requests) gives exactly the results of
    running the two calls one after the other."""
    wl = W.scaled(W.WORKLOADS["mixed"], name="overlap", L=3, R=40, mixed_compress=6)

    def run(overlap):
        st = W.build_cache(wl, DEV)
        cache = H.make_cache(st)
        drows = st.decode_rows
        outs = [torch.empty((drows.numel(), wl.Hq, wl.d), dtype=torch.bfloat16, device=DEV)
                for _ in range(wl.L)]
        main = torch.cuda.current_stream()
        s_dec = torch.cuda.Stream(priority=-1) if overlap else main
        s_cmp = torch.cuda.Stream() if overlap else main
        # the queries exist before the fork and live until the synchronisation
        qs = [st.decode_q[l][drows.long()].contiguous() for l in range(wl.L)]
        ev = torch.cuda.Event()
        ev.record(main)
        s_dec.wait_event(ev)
        s_cmp.wait_event(ev)
        for l in range(wl.L):
            cache.decode(l, qs[l], st.block_tables, st.lengths, 1.0 / math.sqrt(wl.d), outs[l],
                         req_idx=drows, stream=s_dec)
        cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam,
                       st.free_ids, st.free_count, st.refcount, req_idx=st.compress_rows,
                       stream=s_cmp)
        torch.cuda.synchronize()
        assert cache.status() == zp.OK
        return st, outs

    st_o, out_o = run(True)
    st_s, out_s = run(False)
    for a, b in zip(out_o, out_s):
        assert torch.equal(a, b)
    for a, b in zip(st_o.k_pools + st_o.v_pools, st_s.k_pools + st_s.v_pools):
        assert torch.equal(a, b)
    for name in ("block_tables", "lengths", "refcount", "free_ids", "free_count"):
        assert torch.equal(getattr(st_o, name), getattr(st_s, name)), name
