"""The hybrid-scheduling simulator driving the GPU library and the CPU
oracle in lockstep: the same requests, the same decisions, the same seeded
draws; after every step the block tables, lengths, refcounts and free stack
are equal, decode attention agrees within 2e-2, and the pools are
byte-identical at the end."""
from __future__ import annotations

import copy

import numpy as np
import torch

import pytest

from compressed_paged_kv_gb300 import scheduler as S
from tests.sched_oracle_backend import Draws, OracleBackend

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


class LockstepGpuBackend(S.GpuBackend):
    def __init__(self, cfg, L, Hkv, Hq, d, stride, draws, host_pools):
        super().__init__(cfg, L=L, Hkv=Hkv, Hq=Hq, d=d, device=DEV, max_row_blocks=stride)
        self.draws = draws
        for t, h in zip(self.kp + self.vp, host_pools):
            t.copy_(self._dev(h))

    def _dev(self, x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(DEV)

    def _rand(self, shape):
        return self._dev(self.draws.take(shape))


@pytest.mark.parametrize("strict", [False, True])
def test_scheduler_gpu_matches_oracle_in_lockstep(orc, strict):
    cfg = S.SimConfig(num_blocks=90, max_rows=20, n_max=8, w=8, query_slots=3, strict=strict,
                      seed=5)
    L, Hkv, Hq, d, stride = 1, 2, 4, 64, 48
    reqs = S.synthetic_requests(16, 7, prompt=(20, 80), out_median=170, out_sigma=0.6,
                                out_max=600)
    ob = OracleBackend(orc, cfg, L, Hkv, Hq, d, stride, Draws(11), pools_seed=12)
    gb = LockstepGpuBackend(cfg, L, Hkv, Hq, d, stride, Draws(11),
                            ob.s["kpools"] + ob.s["vpools"])
    so = S.Scheduler(cfg, ob, copy.deepcopy(reqs))
    sg = S.Scheduler(cfg, gb, copy.deepcopy(reqs))
    steps = 0
    worst = 0.0
    while so.waiting or so.running:
        a, b = so.step(), sg.step()
        assert a == b, f"step {steps}: decisions differ"
        assert gb.status() == 0, f"step {steps}: device error"
        for k in ("tables", "lengths", "refcount"):
            assert np.array_equal(ob.s[k], getattr(gb, {"refcount": "rc"}.get(k, k)).cpu().numpy()), \
                f"step {steps}: {k}"
        fc = ob.s["free_count"]
        assert int(gb.fc.item()) == fc == so.free_blocks
        assert np.array_equal(ob.s["free_ids"][:fc], gb.free.cpu().numpy()[:fc])
        if b.decoding:
            for o64, og in zip(ob.outputs[-1], gb.last_out):
                worst = max(worst, float(np.abs(og.float().cpu().numpy() - o64).max()))
        steps += 1
        assert steps < 4000
    assert worst <= 2e-2, worst
    for l in range(L):
        assert np.array_equal(ob.s["kpools"][l], gb.kp[l].view(torch.int16).cpu().numpy().view(np.uint16))
        assert np.array_equal(ob.s["vpools"][l], gb.vp[l].view(torch.int16).cpu().numpy().view(np.uint16))
    summ = sg.summary()
    print(f"[sched] strict={strict} {summ} max attention err {worst:.2e}")
    assert summ["finished"] == 16 and summ["compressions"] > 0
