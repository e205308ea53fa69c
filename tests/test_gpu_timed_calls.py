"""The calls the bench times, checked against the oracle exactly as timed.

1. zp_compress with both debug outputs NULL (scores_out and kept_out), as a
   production caller and the bench call it.  The kept sets are read back from
   the compacted pool rows (output row j is the copy of source row kept[j]),
   and everything is compared with the oracle: kept sets (exact or a counted
   near-tie), compacted K/V rows bit-exact, block tables, lengths, refcounts
   and free stack exact, shared blocks untouched.  Cases: every unit of the
   single-layer Qwen3-8B workload, cluster shapes (T 4096 and 8192), the
   36-layer shared-prefix workload and the long-budget workload at full size
   on sampled units (two complete sharing groups included).

2. The asynchronous step (Zipage, Dutch summary, "Methodologie" §4; Korean
   summary, "방법론" D: requests that decode do not wait for others'
   compression): the decoding requests reserve their next slot, then on one
   stream every layer writes their new K/V rows and runs decode attention
   while the requests at N_max compress on a second stream.  The oracle runs
   the same operations one after the other (reservation, compression, new
   rows, attention) from the same inputs; the overlapped GPU run must equal
   it: integer state exact, every pool byte exact (compressed units: exact or
   a near-tie), decode outputs within 2e-2.  Once on a reduced mixed step
   with every byte compared, once at the mixed workload's full size on
   sampled units, rows and layers.
"""
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


# ------------------------------------------- compression without debug outputs

def test_qwen3_1l_every_unit_without_debug_outputs(orc):
    st = W.build_cache(W.WORKLOADS["qwen3_1l"], DEV, with_decode_q=False)
    rep = H.check_compress(orc, st, debug=False)
    assert rep.units == 512
    del st
    _free()


@pytest.mark.parametrize("N,R", [(256, 2), (512, 1)], ids=["T4096_cluster2", "T8192_cluster4"])
def test_cluster_without_debug_outputs(orc, N, R):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name=f"T{N * 16}_no_debug", N=N, R=R)
    st = W.build_cache(wl, DEV, with_decode_q=False)
    H.check_compress(orc, st, debug=False)


def test_qwen3_36l_sampled_without_debug_outputs(orc):
    wl = W.WORKLOADS["qwen3_36l"]
    st = W.build_cache(wl, DEV, with_decode_q=False)
    rng = np.random.default_rng(23)
    groups = [3, 30]
    rows = sorted(set(r for gi in groups for r in range(gi * 8, gi * 8 + 8))
                  | set(rng.choice(wl.R, 8, replace=False).tolist()))
    H.check_compress(orc, st, sample_rows=rows, sample_layers=[0, 11, 35], debug=False)
    del st
    _free()


def test_long4k_sampled_without_debug_outputs(orc):
    wl = W.WORKLOADS["long4k"]
    st = W.build_cache(wl, DEV, with_decode_q=False)
    rng = np.random.default_rng(24)
    rows = sorted(rng.choice(wl.R, 10, replace=False).tolist())
    H.check_compress(orc, st, sample_rows=rows, sample_layers=[0, 35], debug=False)
    del st
    _free()


# ------------------------------------------------------- the asynchronous step

def _new_rows(wl, n, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    k = [torch.randn(n, wl.Hkv, wl.d, generator=g, device=device).to(torch.bfloat16)
         for _ in range(wl.L)]
    v = [torch.randn(n, wl.Hkv, wl.d, generator=g, device=device).to(torch.bfloat16)
         for _ in range(wl.L)]
    return k, v


def _overlapped_step(st, cache, k_new, v_new, outs, compress):
    """The step as the bench times it: the reservation on the current stream,
    then new rows + attention per layer on a high-priority stream while
    `compress(stream)` runs on a second stream."""
    wl = st.wl
    drows = st.decode_rows
    main = torch.cuda.current_stream()
    s_dec = torch.cuda.Stream(priority=-1)
    s_cmp = torch.cuda.Stream()
    # every layer's queries exist before the streams fork and stay alive until
    # the synchronisation below (a temporary freed on this stream while the
    # decode stream still reads it could be handed to the next allocation)
    qs = [st.decode_q[l][drows.long()].contiguous() for l in range(wl.L)]
    cache.append_slots(st.block_tables, st.lengths, wl.N, st.free_ids, st.free_count,
                       st.refcount, req_idx=drows, stream=main)
    ev = torch.cuda.Event()
    ev.record(main)
    s_dec.wait_event(ev)
    s_cmp.wait_event(ev)
    scale = 1.0 / math.sqrt(wl.d)
    for l in range(wl.L):
        cache.append_kv(l, k_new[l], v_new[l], st.block_tables, st.lengths, req_idx=drows,
                        stream=s_dec)
        cache.decode(l, qs[l], st.block_tables, st.lengths, scale, outs[l], req_idx=drows,
                     stream=s_dec)
    compress(s_cmp)
    torch.cuda.synchronize()
    del qs
    assert cache.status() == zp.OK


def test_overlapped_step_matches_oracle_every_byte(orc):
    wl = W.scaled(W.WORKLOADS["mixed"], name="async_step", L=3, R=24, mixed_compress=4)
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    drows = st.decode_rows
    crows = st.compress_rows.cpu().numpy()
    k_new, v_new = _new_rows(wl, drows.numel(), 31, DEV)
    snap = W.snapshot(st)
    outs = [torch.full((drows.numel(), wl.Hq, wl.d), float("nan"), dtype=torch.bfloat16,
                       device=DEV) for _ in range(wl.L)]

    def compress(stream):
        cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam,
                       st.free_ids, st.free_count, st.refcount, req_idx=st.compress_rows,
                       stream=stream)

    _overlapped_step(st, cache, k_new, v_new, outs, compress)

    # the oracle, one operation after the other
    dr = drows.cpu().numpy()
    a = orc.append_slots(snap["k_pools"], snap["v_pools"], snap["block_tables"],
                         snap["lengths"], snap["free_ids"], snap["free_count"], snap["refcount"],
                         wl.N, req_idx=dr)
    assert a["status"] == 0
    c = orc.compress(a["kpools"], a["vpools"], a["tables"], a["lengths"], snap["window_q"],
                     wl.N, wl.w, wl.lam, a["free_ids"], a["free_count"], a["refcount"], Hq=wl.Hq,
                     req_idx=crows)
    assert c["status"] == 0
    want = dict(tables=c["tables"], lengths=c["lengths"], refcount=c["refcount"],
                free_ids=c["free_ids"], free_count=c["free_count"])
    H.check_ints(H.int_state(st), want)

    scale = 1.0 / math.sqrt(wl.d)
    kq = [H.bits(x) for x in k_new]
    vq = [H.bits(x) for x in v_new]
    worst = 0.0
    comp_blocks = np.unique(c["tables"][crows, :wl.N - 1])
    for l in range(wl.L):
        s1, kp, vp = orc.append_kv(c["kpools"][l], c["vpools"][l], c["tables"], c["lengths"],
                                   kq[l], vq[l], req_idx=dr)
        assert s1 == 0
        gk, gv = H.bits(st.k_pools[l]), H.bits(st.v_pools[l])
        if not (np.array_equal(gk, kp) and np.array_equal(gv, vp)):
            # only a near-tie in a compressed unit may differ: every block outside
            # the compressed rows' destinations must still be byte-identical
            other = np.setdiff1d(np.arange(gk.shape[0]), comp_blocks)
            assert np.array_equal(gk[other], kp[other]), f"layer {l}: K bytes differ"
            assert np.array_equal(gv[other], vp[other]), f"layer {l}: V bytes differ"
            Kn = H.bits(H.gather_units(st.k_pools[l], st.block_tables[:, :wl.N - 1],
                                       torch.as_tensor(crows, device=DEV).long()))
            Vn = H.bits(H.gather_units(st.v_pools[l], st.block_tables[:, :wl.N - 1],
                                       torch.as_tensor(crows, device=DEV).long()))
            src_tab = a["tables"][crows]
            for j, r in enumerate(crows):
                for h in range(wl.Hkv):
                    Ks = np.concatenate([a["kpools"][l][blk, h] for blk in src_tab[j, :wl.N]])
                    Vs = np.concatenate([a["vpools"][l][blk, h] for blk in src_tab[j, :wl.N]])
                    Q = snap["window_q"][l, j, h * wl.G:(h + 1) * wl.G].reshape(-1, wl.d)
                    H.check_unit(orc, wl, Ks, Vs, Q, None, None, Kn[j, h], Vn[j, h])
        q = H.bits(st.decode_q[l][drows.long()])
        ost, o64, _ = orc.decode_attn(q, kp, vp, c["tables"][dr], c["lengths"][dr], scale)
        assert ost == 0
        got = outs[l].float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        err = float(np.abs(got - o64).max())
        worst = max(worst, err)
        assert err <= H.DECODE_ATOL, (l, err)
    print(f"[parity] overlapped step {wl.name}: {len(dr)} decoding x {wl.L} layers "
          f"(max abs err {worst:.2e}), {len(crows)} compressing, every pool byte compared")
    cache.close()


def test_mixed_full_size_overlapped_sampled(orc):
    """The mixed workload at full size (32 layers, 461 decoding, 51 compressing),
    overlapped as timed; compression checked on sampled units, attention of
    sampled decoding rows in two layers, both against the oracle."""
    wl = W.WORKLOADS["mixed"]
    st = W.build_cache(wl, DEV)
    cache = H.make_cache(st)
    drows = st.decode_rows
    rng = np.random.default_rng(41)
    layers = [0, 31]
    chk = H.CompressCheck(orc, st, sample_rows=sorted(rng.choice(51, 8, replace=False).tolist()),
                          sample_layers=layers, debug=False, cache=cache)
    pick = np.sort(rng.choice(drows.numel(), 40, replace=False))
    pre = {l: (H.bits(st.k_pools[l]), H.bits(st.v_pools[l])) for l in layers}
    pre_ints = H.int_state(st)
    k_new, v_new = _new_rows(wl, drows.numel(), 32, DEV)
    outs = [torch.full((drows.numel(), wl.Hq, wl.d), float("nan"), dtype=torch.bfloat16,
                       device=DEV) for _ in range(wl.L)]
    dr = drows.cpu().numpy()

    # the reservation comes first in the step: the compression's expected
    # integer state starts from the oracle's reservation
    nb = pre_ints["refcount"].shape[0]
    dummy = [np.zeros((nb, 1, wl.b, 8), dtype=np.uint16)]  # integer state only
    a_ints = orc.append_slots(dummy, dummy, pre_ints["tables"], pre_ints["lengths"],
                              pre_ints["free_ids"], pre_ints["free_count"], pre_ints["refcount"],
                              wl.N, req_idx=dr)
    assert a_ints["status"] == 0
    chk.before = dict(tables=a_ints["tables"], lengths=a_ints["lengths"],
                      refcount=a_ints["refcount"], free_ids=a_ints["free_ids"],
                      free_count=a_ints["free_count"])
    _overlapped_step(st, cache, k_new, v_new, outs, chk.launch)
    chk.verify()

    scale = 1.0 / math.sqrt(wl.d)
    for l in layers:
        kq, vq = H.bits(k_new[l]), H.bits(v_new[l])
        pk, pv = pre[l]
        # attention of the picked rows over the oracle's reservation + new rows
        sub = dr[pick]
        s1, kp, vp = orc.append_kv(pk, pv, a_ints["tables"], a_ints["lengths"], kq[pick],
                                   vq[pick], req_idx=sub)
        assert s1 == 0
        q = H.bits(st.decode_q[l][torch.as_tensor(sub, device=DEV).long()])
        ost, o64, _ = orc.decode_attn(q, kp, vp, a_ints["tables"][sub], a_ints["lengths"][sub],
                                      scale)
        assert ost == 0
        got = outs[l][torch.as_tensor(pick, device=DEV).long()].float().cpu().numpy()
        err = float(np.abs(got.astype(np.float64) - o64).max())
        assert np.all(np.isfinite(got)) and err <= H.DECODE_ATOL, (l, err)
        print(f"[parity] overlapped mixed layer {l}: {len(sub)} decoding rows, max abs err "
              f"{err:.2e}")
    cache.close()
    del st, pre
    _free()
