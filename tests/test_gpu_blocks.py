"""GPU parity of whole-request block allocation and release (zp_alloc_rows,
zp_release_rows) against the oracle: tables, lengths, refcounts and the free
stack exact, failed calls changing nothing."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


class Pool:
    def __init__(self, tables, lengths, free, fc, rc, L=1, Hkv=2, d=64):
        nb = rc.shape[0]
        self.kp = [torch.zeros(nb, Hkv, 16, d, dtype=torch.bfloat16, device=DEV) for _ in range(L)]
        self.vp = [torch.zeros_like(x) for x in self.kp]
        self.tables = torch.tensor(tables, dtype=torch.int32, device=DEV)
        self.lengths = torch.tensor(lengths, dtype=torch.int32, device=DEV)
        self.free = torch.tensor(free, dtype=torch.int32, device=DEV)
        self.fc = torch.tensor([fc], dtype=torch.int32, device=DEV)
        self.rc = torch.tensor(rc, dtype=torch.int32, device=DEV)
        self.cache = zp.Cache(self.kp, self.vp, Hkv, max_requests=self.tables.shape[0],
                              max_blocks_per_req=max(2, self.tables.shape[1]))

    def host(self):
        return dict(tables=self.tables.cpu().numpy(), lengths=self.lengths.cpu().numpy(),
                    free_ids=self.free.cpu().numpy(), free_count=int(self.fc.item()),
                    refcount=self.rc.cpu().numpy())

    def alloc(self, counts, req=None):
        ri = None if req is None else torch.tensor(req, dtype=torch.int32, device=DEV)
        ct = torch.tensor(counts, dtype=torch.int32, device=DEV)
        st = self.cache.alloc_rows(self.tables, self.lengths, ct, self.free, self.fc, self.rc,
                                   req_idx=ri, check=False)
        return st, self.cache.status()

    def release(self, req=None):
        ri = None if req is None else torch.tensor(req, dtype=torch.int32, device=DEV)
        st = self.cache.release_rows(self.tables, self.lengths, self.free, self.fc, self.rc,
                                     req_idx=ri, check=False)
        return st, self.cache.status()


def same(g, o, what):
    for k in ("tables", "lengths", "refcount"):
        assert np.array_equal(g[k], o[k]), f"{what}: {k}"
    assert g["free_count"] == o["free_count"], what
    fc = o["free_count"]
    assert np.array_equal(g["free_ids"][:fc], o["free_ids"][:fc]), f"{what}: free stack"


@pytest.mark.parametrize("seed", [600, 601, 602])
def test_release_then_alloc_random(orc, seed):
    c = W.fork_cache(seed, 200, n_max=6, L=1, Hkv=2, d=64, spare=300)
    p = Pool(c["tables"], c["lengths"], c["free"], c["nfree"], c["rc"])
    g = np.random.default_rng(seed)
    req = g.permutation(200)[:120].astype(np.int32)
    o = orc.release_rows(c["tables"], c["lengths"], c["free"], c["nfree"], c["rc"], req_idx=req)
    assert o["status"] == 0
    assert p.release(req) == (zp.OK, zp.OK)
    same(p.host(), o, "release")
    counts = g.integers(0, 6 * 16 + 1, 120).astype(np.int32)
    o2 = orc.alloc_rows(o["tables"], o["lengths"], o["free_ids"], o["free_count"], o["refcount"],
                        counts, 16, req_idx=req)
    assert o2["status"] == 0
    assert p.alloc(counts, req) == (zp.OK, zp.OK)
    same(p.host(), o2, "alloc")
    # everything back: the pool is whole again
    assert p.release() == (zp.OK, zp.OK)
    h = p.host()
    assert h["free_count"] == c["num_blocks"] and np.all(h["refcount"] == 0)
    assert sorted(h["free_ids"].tolist()) == list(range(c["num_blocks"]))


@pytest.mark.parametrize("what", ["alloc_nonempty", "alloc_short", "alloc_dup", "release_dup",
                                  "release_overheld"])
def test_block_call_errors_change_nothing(orc, what):
    tables = np.full((4, 3), -1, dtype=np.int32)
    tables[0, :2] = [0, 1]
    tables[1, :1] = [0]
    lengths = np.array([20, 5, 0, 0], np.int32)
    rc = np.array([2, 1, 0, 0, 0, 0], np.int32)
    free = np.array([5, 4, 3, 2, -1, -1], np.int32)
    p = Pool(tables, lengths, free, 4, rc)
    before = p.host()
    if what == "alloc_nonempty":
        st = p.alloc([16], req=[1])
        o = orc.alloc_rows(tables, lengths, free, 4, rc, [16], 16, req_idx=np.array([1], np.int32))
    elif what == "alloc_short":
        st = p.alloc([40, 33], req=[2, 3])
        o = orc.alloc_rows(tables, lengths, free, 4, rc, [40, 33], 16,
                           req_idx=np.array([2, 3], np.int32))
    elif what == "alloc_dup":
        st = p.alloc([4, 4], req=[2, 2])
        o = orc.alloc_rows(tables, lengths, free, 4, rc, [4, 4], 16,
                           req_idx=np.array([2, 2], np.int32))
    elif what == "release_dup":
        st = p.release(req=[0, 0])
        o = orc.release_rows(tables, lengths, free, 4, rc, req_idx=np.array([0, 0], np.int32))
    else:
        rc2 = rc.copy()
        rc2[0] = 1
        p = Pool(tables, lengths, free, 4, rc2)
        before = p.host()
        st = p.release(req=[0, 1])
        o = orc.release_rows(tables, lengths, free, 4, rc2, req_idx=np.array([0, 1], np.int32))
    assert o["status"] != 0
    assert st == (zp.OK, o["status"]), (st, o["status"])
    same(p.host(), before, what)
