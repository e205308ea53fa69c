"""Randomised lockstep stress of the whole library against the oracle.

Seeded sequences of operations -- allocate empty rows, allocate a long prompt
and compress it at admission, fork a request, a decode step (slot
reservation with copy-on-write, new K/V rows and attention in every layer),
compress the requests that reached N_max, release rows -- run on the GPU
through the C ABI and on the CPU oracle from the same inputs.  After every
operation the statuses agree and the block tables, lengths, refcounts, free
stack and every pool byte are equal; attention agrees within 2e-2.
Operations that the oracle refuses (too few free blocks) must be refused by
the GPU with the same status and change nothing.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import zp
from tests.sched_oracle_backend import bf16_draw

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
L, HKV, HQ, D, N, W, B = 2, 2, 4, 64, 8, 4, 16
ROWS, STRIDE, NBLK = 24, 40, 260


class Twin:
    def __init__(self, orc, seed, NBLK=NBLK):
        self.orc = orc
        g = np.random.default_rng(seed)
        self.g = g
        self.h = dict(
            kpools=[bf16_draw(g, (NBLK, HKV, B, D)) for _ in range(L)],
            vpools=[bf16_draw(g, (NBLK, HKV, B, D)) for _ in range(L)],
            tables=np.full((ROWS, STRIDE), -1, np.int32), lengths=np.zeros(ROWS, np.int32),
            free_ids=np.arange(NBLK - 1, -1, -1, dtype=np.int32), free_count=NBLK,
            refcount=np.zeros(NBLK, np.int32))
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(
            torch.bfloat16).to(DEV)
        self.t = t
        self.kp = [t(x) for x in self.h["kpools"]]
        self.vp = [t(x) for x in self.h["vpools"]]
        i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=DEV)
        self.i32 = i32
        self.tables = i32(self.h["tables"])
        self.lengths = i32(self.h["lengths"])
        self.free = i32(self.h["free_ids"])
        self.fc = i32([NBLK])
        self.rc = i32(self.h["refcount"])
        self.cache = zp.Cache(self.kp, self.vp, HQ, max_requests=ROWS, max_blocks_per_req=STRIDE)
        self.ws = torch.empty(self.cache.prefill_workspace_bytes(ROWS, STRIDE), dtype=torch.uint8,
                              device=DEV)
        self.trig = torch.zeros(ROWS, dtype=torch.int32, device=DEV)
        self.ntrig = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.worst = 0.0

    # -- helpers ----------------------------------------------------------
    def take(self, res, keys):
        if res["status"] == 0:
            for k in keys:
                self.h[k] = res[k]
        return res["status"]

    def check(self, what, want_status):
        got = self.cache.status()
        assert got == want_status, f"{what}: GPU status {got}, oracle {want_status}"
        h = self.h
        assert np.array_equal(self.tables.cpu().numpy(), h["tables"]), f"{what}: tables"
        assert np.array_equal(self.lengths.cpu().numpy(), h["lengths"]), f"{what}: lengths"
        assert np.array_equal(self.rc.cpu().numpy(), h["refcount"]), f"{what}: refcounts"
        fc = h["free_count"]
        assert int(self.fc.item()) == fc, f"{what}: free count"
        assert np.array_equal(self.free.cpu().numpy()[:fc], h["free_ids"][:fc]), f"{what}: stack"
        for l in range(L):
            bits = lambda x: x.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(bits(self.kp[l]), h["kpools"][l]), f"{what}: K pool {l}"
            assert np.array_equal(bits(self.vp[l]), h["vpools"][l]), f"{what}: V pool {l}"

    def empty_rows(self):
        return [r for r in range(ROWS) if self.h["lengths"][r] == 0
                and np.all(self.h["tables"][r] < 0)]

    def live_rows(self):
        return [r for r in range(ROWS) if self.h["lengths"][r] > 0]

    # -- operations -----------------------------------------------------------
    def alloc(self, rows, counts):
        h = self.h
        res = self.orc.alloc_rows(h["tables"], h["lengths"], h["free_ids"], h["free_count"],
                                  h["refcount"], counts, B, req_idx=np.array(rows, np.int32))
        want = self.take(res, ("tables", "lengths", "free_ids", "free_count", "refcount"))
        self.cache.alloc_rows(self.tables, self.lengths, self.i32(counts), self.free, self.fc,
                              self.rc, req_idx=self.i32(rows))
        self.check("alloc", want)
        return want

    def prefill(self, rows):
        h = self.h
        wq = bf16_draw(self.g, (L, len(rows), HQ, W, D))
        res = self.orc.compress_prefill(h["kpools"], h["vpools"], h["tables"], h["lengths"], wq,
                                        N, W, 0.5, h["free_ids"], h["free_count"], h["refcount"],
                                        Hq=HQ, req_idx=np.array(rows, np.int32),
                                        want_scores=False, want_kept=False)
        want = self.take(res, ("kpools", "vpools", "tables", "lengths", "free_ids", "free_count",
                               "refcount"))
        self.cache.compress_prefill(self.tables, self.lengths, self.t(wq), N, W, 0.5, self.free,
                                    self.fc, self.rc, self.ws, req_idx=self.i32(rows))
        self.check("prefill", want)

    def fork(self, src, dst):
        h = self.h
        res = self.orc.fork_rows(h["tables"], h["lengths"], h["refcount"], src, dst)
        want = self.take(res, ("tables", "lengths", "refcount"))
        self.cache.fork_rows(self.tables, self.lengths, self.rc, self.i32(src), self.i32(dst))
        self.check("fork", want)

    def decode_step(self, rows):
        h = self.h
        res = self.orc.append_slots(h["kpools"], h["vpools"], h["tables"], h["lengths"],
                                    h["free_ids"], h["free_count"], h["refcount"], N,
                                    req_idx=np.array(rows, np.int32))
        want = self.take(res, ("kpools", "vpools", "tables", "lengths", "free_ids", "free_count",
                               "refcount"))
        self.cache.append_slots(self.tables, self.lengths, N, self.free, self.fc, self.rc,
                                req_idx=self.i32(rows), trigger_rows=self.trig,
                                trigger_count=self.ntrig)
        self.check("append", want)
        if want != 0:
            return want, []
        trig = res["triggers"].tolist()
        assert self.trig[:int(self.ntrig.item())].tolist() == trig
        ri = np.array(rows, np.int32)
        for l in range(L):
            kn, vn = bf16_draw(self.g, (len(rows), HKV, D)), bf16_draw(self.g, (len(rows), HKV, D))
            q = bf16_draw(self.g, (len(rows), HQ, D))
            st, h["kpools"][l], h["vpools"][l] = self.orc.append_kv(
                h["kpools"][l], h["vpools"][l], h["tables"], h["lengths"], kn, vn, req_idx=ri)
            assert st == 0
            self.cache.append_kv(l, self.t(kn), self.t(vn), self.tables, self.lengths,
                                 req_idx=self.i32(rows))
            out = torch.empty(len(rows), HQ, D, dtype=torch.bfloat16, device=DEV)
            self.cache.decode(l, self.t(q), self.tables, self.lengths, 1 / math.sqrt(D), out,
                              req_idx=self.i32(rows))
            st, o64, _ = self.orc.decode_attn(q, h["kpools"][l], h["vpools"][l], h["tables"][ri],
                                              h["lengths"][ri], 1 / math.sqrt(D))
            assert st == 0
            self.worst = max(self.worst, float(np.abs(out.float().cpu().numpy() - o64).max()))
        self.check("decode", 0)
        return 0, trig

    def compress(self, rows):
        h = self.h
        wq = bf16_draw(self.g, (L, len(rows), HQ, W, D))
        res = self.orc.compress(h["kpools"], h["vpools"], h["tables"], h["lengths"], wq, N, W,
                                0.5, h["free_ids"], h["free_count"], h["refcount"], Hq=HQ,
                                req_idx=np.array(rows, np.int32), want_scores=False)
        want = self.take(res, ("kpools", "vpools", "tables", "lengths", "free_ids", "free_count",
                               "refcount"))
        kept = torch.full((L, len(rows), HKV, (N - 1) * B), -1, dtype=torch.int32, device=DEV)
        self.cache.compress(self.tables, self.lengths, self.t(wq), N, W, 0.5, self.free, self.fc,
                            self.rc, req_idx=self.i32(rows), kept_out=kept)
        if want == 0:
            assert np.array_equal(kept.cpu().numpy(), res["kept"]), "kept sets (a near-tie?)"
        self.check("compress", want)

    def release(self, rows):
        h = self.h
        res = self.orc.release_rows(h["tables"], h["lengths"], h["free_ids"], h["free_count"],
                                    h["refcount"], req_idx=np.array(rows, np.int32))
        want = self.take(res, ("tables", "lengths", "free_ids", "free_count", "refcount"))
        self.cache.release_rows(self.tables, self.lengths, self.free, self.fc, self.rc,
                                req_idx=self.i32(rows))
        self.check("release", want)


@pytest.mark.parametrize("seed,nblk,ops", [(900, NBLK, 60), (901, NBLK, 60), (902, 70, 90)])
def test_random_operation_sequences(orc, seed, nblk, ops):
    """The third case runs a pool of 70 blocks, so allocations and decode steps
    are refused for lack of blocks along the way."""
    tw = Twin(orc, seed, NBLK=nblk)
    g = np.random.default_rng(seed + 1)
    counts = dict(alloc=0, prefill=0, fork=0, decode=0, compress=0, release=0, refused=0)
    for _ in range(ops):
        op = g.choice(["alloc", "prefill", "fork", "decode", "decode", "decode", "release"])
        empty, live = tw.empty_rows(), tw.live_rows()
        if op == "alloc" and empty:
            rows = list(g.choice(empty, size=min(len(empty), int(g.integers(1, 4))), replace=False))
            st = tw.alloc(rows, [int(g.integers(1, N * B)) for _ in rows])
            counts["refused" if st else "alloc"] += 1
        elif op == "prefill" and empty:
            row = int(g.choice(empty))
            if tw.alloc([row], [int(g.integers(N * B, STRIDE * B + 1))]) == 0:
                tw.prefill([row])
                counts["prefill"] += 1
            else:
                counts["refused"] += 1
        elif op == "fork" and empty:
            src = [r for r in live if tw.h["lengths"][r] < N * B]
            if src:
                tw.fork([int(g.choice(src))], [int(g.choice(empty))])
                counts["fork"] += 1
        elif op == "decode":
            rows = [r for r in live if tw.h["lengths"][r] < N * B]
            if rows:
                st, trig = tw.decode_step(rows)
                counts["refused" if st else "decode"] += 1
                if trig:
                    tw.compress(trig)
                    counts["compress"] += 1
        elif op == "release" and live:
            rows = list(g.choice(live, size=min(len(live), int(g.integers(1, 4))), replace=False))
            tw.release([int(r) for r in rows])
            counts["release"] += 1
    print(f"[stress] seed {seed}: {counts}, max attention err {tw.worst:.2e}")
    assert tw.worst <= 2e-2
    assert counts["fork"] > 0 and counts["decode"] > 0 and counts["prefill"] > 0
    if nblk < NBLK:
        assert counts["refused"] > 0
