"""An oracle-backed twin of ``scheduler.GpuBackend`` (test infrastructure):
the same operations on host copies of the cache, through the CPU oracle, and
seeded host draws for the new tokens' K/V, queries and window queries, so that
a GPU run fed the same draws can be compared with it step by step."""
from __future__ import annotations

import math

import numpy as np
import torch

from compressed_paged_kv_gb300 import workloads as W


def bf16_draw(g, shape):
    t = torch.as_tensor(g.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


class Draws:
    """One seeded stream of bf16 draws shared by a pair of backends."""

    def __init__(self, seed):
        self.g = np.random.default_rng(seed)
        self.log = []

    def take(self, shape):
        x = bf16_draw(self.g, shape)
        self.log.append(x)
        return x


class OracleBackend:
    def __init__(self, orc, cfg, L, Hkv, Hq, d, stride, draws, pools_seed=0):
        self.orc, self.cfg, self.L, self.Hkv, self.Hq, self.d = orc, cfg, L, Hkv, Hq, d
        self.stride = stride
        self.draws = draws
        g = np.random.default_rng(pools_seed)
        nb = cfg.num_blocks
        self.s = dict(
            kpools=[bf16_draw(g, (nb, Hkv, cfg.b, d)) for _ in range(L)],
            vpools=[bf16_draw(g, (nb, Hkv, cfg.b, d)) for _ in range(L)],
            tables=np.full((cfg.max_rows, stride), -1, np.int32),
            lengths=np.zeros(cfg.max_rows, np.int32),
            free_ids=np.arange(nb - 1, -1, -1, dtype=np.int32), free_count=nb,
            refcount=np.zeros(nb, np.int32))
        self.scale = 1.0 / math.sqrt(d)
        self.outputs = []

    def _upd(self, res, keys):
        assert res["status"] == 0, res["status"]
        for k in keys:
            self.s[k] = res[k]

    def alloc(self, rows, counts):
        s = self.s
        r = self.orc.alloc_rows(s["tables"], s["lengths"], s["free_ids"], s["free_count"],
                                s["refcount"], counts, self.cfg.b, req_idx=np.array(rows, np.int32))
        self._upd(r, ("tables", "lengths", "free_ids", "free_count", "refcount"))

    def prefill(self, rows):
        s = self.s
        wq = self.draws.take((self.L, len(rows), self.Hq, self.cfg.w, self.d))
        r = self.orc.compress_prefill(s["kpools"], s["vpools"], s["tables"], s["lengths"], wq,
                                      self.cfg.n_max, self.cfg.w, 0.5, s["free_ids"],
                                      s["free_count"], s["refcount"], Hq=self.Hq,
                                      req_idx=np.array(rows, np.int32), want_scores=False,
                                      want_kept=False)
        self._upd(r, ("kpools", "vpools", "tables", "lengths", "free_ids", "free_count",
                      "refcount"))

    def append(self, rows):
        s = self.s
        r = self.orc.append_slots(s["kpools"], s["vpools"], s["tables"], s["lengths"],
                                  s["free_ids"], s["free_count"], s["refcount"], self.cfg.n_max,
                                  req_idx=np.array(rows, np.int32))
        self._upd(r, ("kpools", "vpools", "tables", "lengths", "free_ids", "free_count",
                      "refcount"))
        return r["triggers"].tolist()

    def write_and_attend(self, rows):
        s = self.s
        ri = np.array(rows, np.int32)
        outs = []
        for l in range(self.L):
            kn = self.draws.take((len(rows), self.Hkv, self.d))
            vn = self.draws.take((len(rows), self.Hkv, self.d))
            q = self.draws.take((len(rows), self.Hq, self.d))
            st, s["kpools"][l], s["vpools"][l] = self.orc.append_kv(
                s["kpools"][l], s["vpools"][l], s["tables"], s["lengths"], kn, vn, req_idx=ri)
            assert st == 0
            st, o64, _ = self.orc.decode_attn(q, s["kpools"][l], s["vpools"][l], s["tables"][ri],
                                              s["lengths"][ri], self.scale)
            assert st == 0
            outs.append(o64)
        self.outputs.append(outs)

    def compress(self, rows):
        s = self.s
        wq = self.draws.take((self.L, len(rows), self.Hq, self.cfg.w, self.d))
        r = self.orc.compress(s["kpools"], s["vpools"], s["tables"], s["lengths"], wq,
                              self.cfg.n_max, self.cfg.w, 0.5, s["free_ids"], s["free_count"],
                              s["refcount"], Hq=self.Hq, req_idx=np.array(rows, np.int32),
                              want_scores=False, want_kept=False)
        self._upd(r, ("kpools", "vpools", "tables", "lengths", "free_ids", "free_count",
                      "refcount"))

    def release(self, rows):
        s = self.s
        r = self.orc.release_rows(s["tables"], s["lengths"], s["free_ids"], s["free_count"],
                                  s["refcount"], req_idx=np.array(rows, np.int32))
        self._upd(r, ("tables", "lengths", "free_ids", "free_count", "refcount"))

    def free_count(self):
        return self.s["free_count"]
