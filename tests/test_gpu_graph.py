"""The C ABI under CUDA graph capture: every entry point only enqueues work on
the caller's stream (no allocation, no synchronisation), so a decode step and
a compression can be captured once and replayed.  Each replay must equal an
eager run from the same state (ints and pool bytes exact, attention outputs
bit-identical: the same kernels run on the same inputs)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


class State:
    def __init__(self, c, Hq):
        self.kp = [k.to(DEV) for k in c["k_pools"]]
        self.vp = [v.to(DEV) for v in c["v_pools"]]
        self.tables = torch.tensor(c["tables"], device=DEV)
        self.lengths = torch.tensor(c["lengths"], device=DEV)
        self.rc = torch.tensor(c["rc"], device=DEV)
        self.free = torch.tensor(c["free"], device=DEV)
        self.fc = torch.tensor([c["nfree"]], dtype=torch.int32, device=DEV)
        self.cache = zp.Cache(self.kp, self.vp, Hq, max_requests=self.tables.shape[0],
                              max_blocks_per_req=self.tables.shape[1])
        R = self.tables.shape[0]
        self.trig = torch.zeros(R, dtype=torch.int32, device=DEV)
        self.ntrig = torch.zeros(1, dtype=torch.int32, device=DEV)

    def tensors(self):
        return self.kp + self.vp + [self.tables, self.lengths, self.rc, self.free, self.fc]

    def load(self, other):
        for a, b in zip(self.tensors(), other.tensors()):
            a.copy_(b)


def assert_same(a: State, b: State, what):
    for x, y in zip(a.tensors(), b.tensors()):
        assert torch.equal(x, y), what


def test_decode_step_graph_replays_match_eager():
    R, L, Hkv, G, d, N = 48, 2, 2, 4, 128, 8
    steps = 4
    # lengths up to N*16 - steps: the rows at exactly that length reach N_max
    # blocks on the last step and are listed as due for compression
    c = W.fork_cache(300, R, n_max=N, L=L, Hkv=Hkv, d=d, spare=64, len_lo=N * 16 - 12,
                     len_hi=N * 16 - steps + 1)
    due = int(np.count_nonzero(c["lengths"] == N * 16 - steps))
    eager = State(c, Hkv * G)
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator(device=DEV)
    g.manual_seed(301)
    inputs = [[(torch.randn(R, Hkv, d, generator=g, device=DEV).to(torch.bfloat16),
                torch.randn(R, Hkv, d, generator=g, device=DEV).to(torch.bfloat16),
                torch.randn(R, Hkv * G, d, generator=g, device=DEV).to(torch.bfloat16))
               for _ in range(L)] for _ in range(steps)]

    def step(st: State, ins, outs):
        st.cache.append_slots(st.tables, st.lengths, N, st.free, st.fc, st.rc,
                              trigger_rows=st.trig, trigger_count=st.ntrig)
        for l in range(L):
            kn, vn, q = ins[l]
            st.cache.append_kv(l, kn, vn, st.tables, st.lengths)
            st.cache.decode(l, q, st.tables, st.lengths, scale, outs[l])

    # static input/output buffers of the graph
    s_in = [tuple(torch.empty_like(x) for x in ins) for ins in inputs[0]]
    s_out = [torch.empty(R, Hkv * G, d, dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    e_out = [torch.empty_like(x) for x in s_out]
    # capturing records the launches without running them: the captured
    # state is still the initial one afterwards
    scratch = State(c, Hkv * G)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(scratch, s_in, s_out)
    torch.cuda.synchronize()
    assert_same(scratch, eager, "state after capture")
    triggered = 0
    for i in range(steps):
        for dst, src in zip(s_in, inputs[i]):
            for a, b in zip(dst, src):
                a.copy_(b)
        graph.replay()
        step(eager, inputs[i], e_out)
        torch.cuda.synchronize()
        assert eager.cache.status() == 0 and scratch.cache.status() == 0, f"step {i}"
        assert_same(scratch, eager, f"state after replay {i}")
        for a, b in zip(s_out, e_out):
            assert torch.equal(a, b), f"attention after replay {i}"
        assert torch.equal(scratch.ntrig, eager.ntrig)
        n = int(eager.ntrig.item())
        assert torch.equal(scratch.trig[:n], eager.trig[:n])
        triggered += n
    assert triggered == due


@pytest.mark.parametrize("many", [False, True], ids=["few_units", "more_units_than_sms"])
def test_compress_graph_replays_match_eager(many):
    """One captured compression replayed on restored inputs: every replay
    gives the eager result (this also checks that the duplicate-row stamps
    advance on the device, not in the captured launch arguments, and that the
    per-SM pairing words are reset between replays)."""
    R = torch.cuda.get_device_properties(0).multi_processor_count // 8 + 3 if many else 12
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="graph", N=16, R=R, group=3, prefix_blocks=2,
                  spare_blocks=128)
    st0 = W.build_cache(wl, DEV)
    base = [t.clone() for t in st0.k_pools + st0.v_pools +
            [st0.block_tables, st0.lengths, st0.refcount, st0.free_ids, st0.free_count]]

    def fresh():
        ts = [t.clone() for t in base]
        L = wl.L
        return ts[:L], ts[L:2 * L], ts[2 * L:]

    kp_e, vp_e, ints_e = fresh()
    cache_e = zp.Cache(kp_e, vp_e, wl.Hq, max_requests=wl.R, max_blocks_per_req=wl.N)
    kept_e = torch.empty(wl.L, wl.R, wl.Hkv, (wl.N - 1) * wl.b, dtype=torch.int32, device=DEV)
    cache_e.compress(ints_e[0], ints_e[1], st0.window_q, wl.N, wl.w, wl.lam, ints_e[3],
                     ints_e[4], ints_e[2], kept_out=kept_e)
    assert cache_e.status() == 0

    kp_g, vp_g, ints_g = fresh()
    cache_g = zp.Cache(kp_g, vp_g, wl.Hq, max_requests=wl.R, max_blocks_per_req=wl.N)
    kept_g = torch.empty_like(kept_e)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cache_g.compress(ints_g[0], ints_g[1], st0.window_q, wl.N, wl.w, wl.lam, ints_g[3],
                         ints_g[4], ints_g[2], kept_out=kept_g)
    torch.cuda.synchronize()
    for rep in range(3):
        for a, b in zip(kp_g + vp_g + ints_g, base):
            a.copy_(b)
        kept_g.fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        assert cache_g.status() == 0, f"replay {rep}"
        assert torch.equal(kept_g, kept_e), f"kept sets, replay {rep}"
        for a, b in zip(kp_g + vp_g + ints_g, kp_e + vp_e + ints_e):
            assert torch.equal(a, b), f"state after replay {rep}"
