"""GPU parity of the decode-side append path and of the whole decode ->
trigger -> compress loop, through the C ABI, against the CPU oracle.

Integers (tables, lengths, refcounts, free stack, trigger lists) and pool
bytes are compared exactly; decode attention within 2e-2 absolute; a
compression inside the loop by the criteria of gpu_helpers (here the kept
sets must match exactly, since the loop continues from the compacted state).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DECODE_ATOL = 2e-2


class Fork:
    """A forked cache on the GPU plus its host mirror for the oracle."""

    def __init__(self, c, Hq):
        self.c = c
        self.Hq = Hq
        self.kp = [k.to(DEV) for k in c["k_pools"]]
        self.vp = [v.to(DEV) for v in c["v_pools"]]
        self.tables = torch.tensor(c["tables"], device=DEV)
        self.lengths = torch.tensor(c["lengths"], device=DEV)
        self.rc = torch.tensor(c["rc"], device=DEV)
        self.free = torch.tensor(c["free"], device=DEV)
        self.fc = torch.tensor([c["nfree"]], dtype=torch.int32, device=DEV)
        self.cache = zp.Cache(self.kp, self.vp, Hq, max_requests=self.tables.shape[0],
                              max_blocks_per_req=max(2, self.tables.shape[1]))
        R = self.tables.shape[0]
        self.trig_rows = torch.full((R,), -7, dtype=torch.int32, device=DEV)
        self.trig_count = torch.full((1,), -7, dtype=torch.int32, device=DEV)

    def host(self):
        return dict(kpools=[W.bf16_bits(k).copy() for k in self.kp],
                    vpools=[W.bf16_bits(v).copy() for v in self.vp],
                    tables=self.tables.cpu().numpy(), lengths=self.lengths.cpu().numpy(),
                    refcount=self.rc.cpu().numpy(), free_ids=self.free.cpu().numpy(),
                    free_count=int(self.fc.item()))

    def append_slots(self, n_max, req_idx=None):
        ri = None if req_idx is None else torch.tensor(req_idx, dtype=torch.int32, device=DEV)
        st = self.cache.append_slots(self.tables, self.lengths, n_max, self.free, self.fc,
                                     self.rc, req_idx=ri, trigger_rows=self.trig_rows,
                                     trigger_count=self.trig_count, check=False)
        dev = self.cache.status()
        n = int(self.trig_count.item())
        return st, dev, self.trig_rows[:max(n, 0)].cpu().numpy()


def assert_state(g, o, what):
    for key in ("tables", "lengths", "refcount"):
        assert np.array_equal(g[key], o[key]), f"{what}: {key} differs"
    assert g["free_count"] == o["free_count"], f"{what}: free count"
    assert np.array_equal(g["free_ids"][:g["free_count"]], o["free_ids"][:o["free_count"]]), \
        f"{what}: free stack"
    for l in range(len(g["kpools"])):
        assert np.array_equal(g["kpools"][l], o["kpools"][l]), f"{what}: K pool of layer {l}"
        assert np.array_equal(g["vpools"][l], o["vpools"][l]), f"{what}: V pool of layer {l}"


def oracle_append(orc, h, n_max, req_idx=None):
    return orc.append_slots(h["kpools"], h["vpools"], h["tables"], h["lengths"], h["free_ids"],
                            h["free_count"], h["refcount"], n_max,
                            req_idx=None if req_idx is None else np.array(req_idx, np.int32))


def test_append_fork_example(orc):
    """The hand-worked fork of the golden fixture restated at block size 16
    (positions 6, 6, 4, 7 of 4-token blocks become 18, 18, 16, 31): two
    samples share a partial block, one row opens an unallocated block, one
    reaches N_max = 2 full blocks."""
    with open(os.path.join(GOLDEN, "append_fork_handworked.json")) as f:
        gd = json.load(f)
    for case in gd["cases"]:
        c = dict(tables=np.array(gd["tables"], np.int32),
                 lengths=np.array([18, 18, 16, 31], np.int32),
                 rc=np.array(gd["refcount"], np.int32),
                 free=np.array(gd["free_ids"], np.int32), nfree=len(gd["free_ids"]),
                 k_pools=[torch.randn(gd["num_blocks"], 2, 16, 64).to(torch.bfloat16)
                          for _ in range(2)],
                 v_pools=[torch.randn(gd["num_blocks"], 2, 16, 64).to(torch.bfloat16)
                          for _ in range(2)])
        f_ = Fork(c, Hq=4)
        before = f_.host()
        o = oracle_append(orc, before, gd["n_max"], case["req_idx"])
        st, dev, trig = f_.append_slots(gd["n_max"], case["req_idx"])
        assert st == 0 and dev == 0 and o["status"] == 0
        assert o["tables"].tolist() == case["tables"]
        assert o["refcount"].tolist() == case["refcount"]
        assert trig.tolist() == o["triggers"].tolist() == case["triggers"]
        assert_state(f_.host(), o, "fork example")
        src, dst, _ = case["copied"][0]
        for l in range(2):
            assert np.array_equal(W.bf16_bits(f_.kp[l])[dst, :, :2], before["kpools"][l][src, :, :2])


@pytest.mark.parametrize("seed,d,R,perm", [(200, 128, 40, False), (201, 64, 40, True),
                                           (202, 128, 300, True), (203, 128, 1500, True)])
def test_append_random_forks(orc, seed, d, R, perm):
    c = W.fork_cache(seed, R, n_max=6, L=2, Hkv=2, d=d, spare=R // 2 + 8)
    f_ = Fork(c, Hq=4)
    before = f_.host()
    req = np.random.default_rng(seed).permutation(R).astype(np.int32) if perm else None
    if perm:
        req = req[: R - R // 5]                      # some rows sit this step out
    o = oracle_append(orc, before, 6, req)
    st, dev, trig = f_.append_slots(6, req)
    assert o["status"] == 0 and st == 0 and dev == 0
    assert np.array_equal(trig, o["triggers"])
    assert_state(f_.host(), o, f"random forks seed {seed}")
    pops = c["nfree"] - o["free_count"]
    assert pops > 0


def test_append_out_of_free_blocks_changes_nothing(orc):
    c = W.fork_cache(210, 64, n_max=6, L=1, Hkv=2, d=128, spare=0)
    c["nfree"] = 0
    f_ = Fork(c, Hq=4)
    before = f_.host()
    o = oracle_append(orc, before, 6)
    st, dev, trig = f_.append_slots(6)
    assert o["status"] == zp.ERR_OUT_OF_BLOCKS
    assert st == 0 and dev == zp.ERR_OUT_OF_BLOCKS
    assert len(trig) == 0
    assert_state(f_.host(), before, "out of blocks")


@pytest.mark.parametrize("what", ["full_row", "partial_no_block", "duplicate_row",
                                  "writers_exceed_refs", "bad_block"])
def test_append_device_errors(orc, what):
    c = W.fork_cache(220, 12, n_max=4, L=1, Hkv=2, d=64, spare=16, max_fan=1, len_lo=33)
    req = None
    if what == "full_row":
        c["lengths"][3] = 4 * 16
    elif what == "partial_no_block":
        c["lengths"][2] = 17
        c["tables"][2, 1] = -1
        c["tables"][2, 2:] = -1
    elif what == "duplicate_row":
        req = [0, 1, 1]
    elif what == "writers_exceed_refs":
        c["lengths"][4] = c["lengths"][5] = 20
        c["tables"][4] = c["tables"][5]
        c["rc"][:] = 0
        for x in c["tables"].reshape(-1):
            if x >= 0:
                c["rc"][x] += 1
        c["rc"][c["tables"][5, 1]] = 1
    elif what == "bad_block":
        c["lengths"][6] = 20
        c["tables"][6, 1] = c["num_blocks"] + 5
    f_ = Fork(c, Hq=4)
    before = f_.host()
    o = oracle_append(orc, before, 4, req)
    st, dev, trig = f_.append_slots(4, req)
    assert o["status"] == zp.ERR_INVALID_ARG, o["status"]
    assert st == 0 and dev == zp.ERR_INVALID_ARG
    assert len(trig) == 0
    assert_state(f_.host(), before, what)


def test_append_kv_then_decode(orc):
    """Slots, then each layer's new K/V rows, then decode attention over the
    grown cache: pools bit-exact, attention within tolerance."""
    R, L, Hkv, G, d = 96, 2, 2, 4, 128
    c = W.fork_cache(230, R, n_max=6, L=L, Hkv=Hkv, d=d, spare=80)
    f_ = Fork(c, Hq=Hkv * G)
    h = f_.host()
    o = oracle_append(orc, h, 6)
    st, dev, _ = f_.append_slots(6)
    assert st == 0 and dev == 0 and o["status"] == 0
    g = torch.Generator(device=DEV)
    g.manual_seed(231)
    scale = 1.0 / math.sqrt(d)
    for l in range(L):
        kn = torch.randn(R, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
        vn = torch.randn(R, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
        q = torch.randn(R, Hkv * G, d, generator=g, device=DEV).to(torch.bfloat16)
        f_.cache.append_kv(l, kn, vn, f_.tables, f_.lengths)
        out = torch.empty(R, Hkv * G, d, dtype=torch.bfloat16, device=DEV)
        f_.cache.decode(l, q, f_.tables, f_.lengths, scale, out)
        assert f_.cache.status() == 0
        sto, kpo, vpo = orc.append_kv(o["kpools"][l], o["vpools"][l], o["tables"], o["lengths"],
                                      W.bf16_bits(kn), W.bf16_bits(vn))
        assert sto == 0
        assert np.array_equal(W.bf16_bits(f_.kp[l]), kpo)
        assert np.array_equal(W.bf16_bits(f_.vp[l]), vpo)
        std, o64, _ = orc.decode_attn(W.bf16_bits(q), kpo, vpo, o["tables"], o["lengths"], scale)
        assert std == 0
        err = np.abs(out.float().cpu().numpy() - o64).max()
        assert err <= DECODE_ATOL, err


def test_append_kv_bad_length_is_flagged():
    c = W.fork_cache(240, 8, n_max=4, L=1, Hkv=2, d=64, spare=8)
    c["lengths"][:] = 0                               # no slot reserved
    f_ = Fork(c, Hq=2)
    kn = torch.zeros(8, 2, 64, dtype=torch.bfloat16, device=DEV)
    before = W.bf16_bits(f_.kp[0]).copy()
    f_.cache.append_kv(0, kn, kn, f_.tables, f_.lengths)
    assert f_.cache.status() == zp.ERR_DEVICE_CHECK
    assert np.array_equal(W.bf16_bits(f_.kp[0]), before)


def test_decode_compress_loop(orc):
    """Eight decode steps over a forked cache close to N_max: every step
    reserves slots (copy-on-write of shared tails), writes each layer's new
    K/V, runs decode attention, and compresses the requests the step listed
    as due; the GPU and the oracle advance in lockstep from the same inputs."""
    R, L, Hkv, G, d, N, w, lam = 24, 2, 2, 4, 128, 8, 8, 0.5
    b = 16
    c = W.fork_cache(250, R, n_max=N, L=L, Hkv=Hkv, d=d, spare=96, len_lo=N * b - 7)
    f_ = Fork(c, Hq=Hkv * G)
    h = f_.host()
    g = torch.Generator(device=DEV)
    g.manual_seed(251)
    scale = 1.0 / math.sqrt(d)
    compressed = 0
    for step in range(8):
        o = oracle_append(orc, h, N)
        st, dev, trig = f_.append_slots(N)
        assert o["status"] == 0 and st == 0 and dev == 0, (step, o["status"], dev)
        assert np.array_equal(trig, o["triggers"]), step
        h = {k: o[k] for k in ("kpools", "vpools", "tables", "lengths", "refcount", "free_ids",
                               "free_count")}
        for l in range(L):
            kn = torch.randn(R, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
            vn = torch.randn(R, Hkv, d, generator=g, device=DEV).to(torch.bfloat16)
            q = torch.randn(R, Hkv * G, d, generator=g, device=DEV).to(torch.bfloat16)
            f_.cache.append_kv(l, kn, vn, f_.tables, f_.lengths)
            out = torch.empty(R, Hkv * G, d, dtype=torch.bfloat16, device=DEV)
            f_.cache.decode(l, q, f_.tables, f_.lengths, scale, out)
            sto, h["kpools"][l], h["vpools"][l] = orc.append_kv(
                h["kpools"][l], h["vpools"][l], h["tables"], h["lengths"], W.bf16_bits(kn),
                W.bf16_bits(vn))
            assert sto == 0
            std, o64, _ = orc.decode_attn(W.bf16_bits(q), h["kpools"][l], h["vpools"][l],
                                          h["tables"], h["lengths"], scale)
            assert std == 0
            err = np.abs(out.float().cpu().numpy() - o64).max()
            assert err <= DECODE_ATOL, (step, l, err)
        assert f_.cache.status() == 0
        assert_state(f_.host(), h, f"step {step} after append")
        if len(trig):
            Rc = len(trig)
            wq = torch.randn(L, Rc, Hkv * G, w, d, generator=g, device=DEV).to(torch.bfloat16)
            ri = torch.tensor(trig, dtype=torch.int32, device=DEV)
            kept = torch.full((L, Rc, Hkv, (N - 1) * b), -1, dtype=torch.int32, device=DEV)
            f_.cache.compress(f_.tables, f_.lengths, wq, N, w, lam, f_.free, f_.fc, f_.rc,
                              req_idx=ri, kept_out=kept)
            assert f_.cache.status() == 0
            oc = orc.compress(h["kpools"], h["vpools"], h["tables"], h["lengths"],
                              W.bf16_bits(wq), N, w, lam, h["free_ids"], h["free_count"],
                              h["refcount"], Hq=Hkv * G, req_idx=trig, want_scores=False)
            assert oc["status"] == 0
            assert np.array_equal(kept.cpu().numpy(), oc["kept"]), f"step {step}: kept sets"
            h = {k: oc[k] for k in ("kpools", "vpools", "tables", "lengths", "refcount",
                                    "free_ids", "free_count")}
            assert_state(f_.host(), h, f"step {step} after compress")
            compressed += Rc
    assert compressed >= R // 2
