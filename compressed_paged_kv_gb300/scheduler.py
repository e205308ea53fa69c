"""Hybrid scheduling of Compressed PagedAttention requests: a step-level
simulator that drives the library's kernels.

Zipage (gist.science summaries: Dutch "Methodologie" §2, Korean "방법론" B):
every request may hold at most N_max blocks; query slots (storage for the
window queries a compression needs) go only to requests that need
compression; requests that are short or not yet near N_max decode without
one; when blocks run out, requests without a query slot are preempted first.
Without the hybrid policy ("strict" below) every running request holds a
query slot from admission on and may grow to N_max blocks, so concurrency is
capped by the slot pool and by num_blocks / N_max.

Readings where the pages are silent (each is a choice of this simulator):
  * a request needs its slot from the decode step of token N_max*b - w (its
    query is the first window query) until the compression at N_max*b, and
    gives it back then; a request that needs a slot while none is free skips
    the step (it cannot proceed past N_max blocks without compressing);
  * admission is first-come first-served while the free blocks cover the
    prompt's blocks plus the next decode step's new blocks;
  * the preemption victim is the most recently admitted request without a
    slot, then the most recently admitted with one; a preempted request
    releases every block and is queued again at the front, to be recomputed
    (prompt + tokens generated so far) -- compressed at admission when that
    is longer than N_max*b;
  * every decode step writes each decoding request's new K/V row and runs
    paged decode attention in every layer, so the kernels see the real
    workload; the values are seeded random draws (no model).

The scheduler decides from host-side mirrors (lengths, blocks held, slots),
which evolve deterministically; a backend carries the device (or oracle)
state.  ``GpuBackend`` calls the C ABI; ``tests`` hold an oracle backend with
the same interface, so the two can run in lockstep and be compared.
"""
from __future__ import annotations

import dataclasses
import math
from collections import deque

import numpy as np


@dataclasses.dataclass
class SimConfig:
    num_blocks: int        # physical blocks in the pool
    max_rows: int          # table rows (the largest batch the engine tracks)
    n_max: int             # blocks per request at compression
    w: int = 8             # observation window
    b: int = 16            # block size
    query_slots: int = 1   # the pool of query slots (window-query storage)
    strict: bool = False
    seed: int = 0


@dataclasses.dataclass(eq=False)
class Request:
    rid: int
    prompt: int
    output: int
    generated: int = 0
    row: int = -1
    length: int = 0        # tokens cached
    held: int = 0          # blocks in the table row (a reserved empty block counts)
    slot: bool = False
    admitted_at: int = -1
    preemptions: int = 0


@dataclasses.dataclass
class StepStats:
    decoding: int = 0
    stalled: int = 0
    admitted: int = 0
    preempted: int = 0
    compressed: int = 0
    prefill_compressed: int = 0
    finished: int = 0
    blocks_held: int = 0


class Scheduler:
    def __init__(self, cfg: SimConfig, backend, requests):
        if cfg.query_slots < 1:
            raise ValueError("scheduling needs at least one query slot")
        self.cfg = cfg
        self.be = backend
        self.waiting = deque(requests)
        self.running: list[Request] = []
        self.done: list[Request] = []
        self.free_rows = list(range(cfg.max_rows - 1, -1, -1))
        self.free_blocks = cfg.num_blocks
        self.slots_free = cfg.query_slots
        self.step_no = 0
        self.history: list[StepStats] = []
        self.strict_cap = min(cfg.query_slots, cfg.num_blocks // cfg.n_max)

    # -- host mirrors -------------------------------------------------------
    def _blocks_for(self, tokens: int) -> int:
        return -(-tokens // self.cfg.b)

    def _needs_block(self, r: Request) -> bool:
        """Whether the next token opens a block the row does not hold yet."""
        return r.length % self.cfg.b == 0 and r.held <= r.length // self.cfg.b

    def _window_start(self) -> int:
        return self.cfg.n_max * self.cfg.b - self.cfg.w

    # -- policy -------------------------------------------------------------
    def _admit(self, st: StepStats):
        cfg = self.cfg
        demand = sum(self._needs_block(r) for r in self.running)
        rows, counts, long_rows = [], [], []
        while self.waiting and self.free_rows:
            r = self.waiting[0]
            tokens = r.prompt + r.generated
            nb = self._blocks_for(tokens)  # all of them until compression at admission
            if cfg.strict and len(self.running) + 1 > self.strict_cap:
                break
            if nb + demand + 1 > self.free_blocks:
                break
            self.waiting.popleft()
            r.row = self.free_rows.pop()
            r.length = tokens
            r.held = nb
            r.admitted_at = self.step_no
            if cfg.strict:
                r.slot = True
            self.free_blocks -= nb
            rows.append(r.row)
            counts.append(tokens)
            if tokens >= cfg.n_max * cfg.b:
                long_rows.append(r)
            self.running.append(r)
            st.admitted += 1
            if tokens < cfg.n_max * cfg.b:
                demand += self._needs_block(r)
        if rows:
            self.be.alloc(rows, counts)
        if long_rows:
            self.be.prefill([r.row for r in long_rows])
            for r in long_rows:
                # kept (N-1)*b tokens + the reserved block; the excess went back
                self.free_blocks += r.held - cfg.n_max
                r.held = cfg.n_max
                r.length = (cfg.n_max - 1) * cfg.b
            st.prefill_compressed += len(long_rows)

    def _release(self, reqs):
        if not reqs:
            return
        self.be.release([r.row for r in reqs])
        for r in reqs:
            self.free_blocks += r.held
            self.free_rows.append(r.row)
            if r.slot and not self.cfg.strict:
                self.slots_free += 1
            r.row, r.length, r.held, r.slot = -1, 0, 0, False

    def _preempt(self, need: int, decoders: list, st: StepStats):
        """Frees blocks until `need` fit: requests without a slot first, the
        most recently admitted first."""
        order = sorted(self.running, key=lambda r: (r.slot, -r.admitted_at, -r.rid))
        victims = []
        for r in order:
            if need <= self.free_blocks + sum(v.held for v in victims):
                break
            victims.append(r)
        if need > self.free_blocks + sum(v.held for v in victims):
            victims = list(self.running)
        self._release(victims)
        for r in victims:
            self.running.remove(r)
            if r in decoders:
                decoders.remove(r)
            r.preemptions += 1
            st.preempted += 1
        for r in reversed(sorted(victims, key=lambda r: r.rid)):
            self.waiting.appendleft(r)

    def step(self) -> StepStats:
        cfg = self.cfg
        st = StepStats()
        self._admit(st)

        # who decodes: near N_max a request needs a query slot
        decoders = []
        for r in sorted(self.running, key=lambda r: r.row):
            if r.length >= self._window_start() and not r.slot:
                if self.slots_free > 0:
                    self.slots_free -= 1
                    r.slot = True
                else:
                    st.stalled += 1
                    continue
            decoders.append(r)
        need = sum(self._needs_block(r) for r in decoders)
        if need > self.free_blocks:
            self._preempt(need, decoders, st)
            need = sum(self._needs_block(r) for r in decoders)

        if decoders:
            decoders.sort(key=lambda r: r.row)
            triggers = self.be.append([r.row for r in decoders])
            self.be.write_and_attend([r.row for r in decoders])
            for r in decoders:
                if self._needs_block(r):
                    r.held += 1
                    self.free_blocks -= 1
                r.length += 1
                r.generated += 1
            full = [r for r in decoders if r.length == cfg.n_max * cfg.b]
            assert sorted(triggers) == sorted(r.row for r in full), "trigger list differs"
            st.decoding = len(decoders)
            # finished requests leave before compressing
            finished = [r for r in decoders if r.generated >= r.output]
            if finished:
                self._release(finished)
                for r in finished:
                    self.running.remove(r)
                    self.done.append(r)
                st.finished = len(finished)
            full = [r for r in full if r.row >= 0]
            if full:
                self.be.compress([r.row for r in full])
                for r in full:
                    r.length = (cfg.n_max - 1) * cfg.b  # the reserved block stays held
                    if not cfg.strict:
                        r.slot = False
                        self.slots_free += 1
                st.compressed = len(full)
        st.blocks_held = sum(r.held for r in self.running)
        assert st.blocks_held + self.free_blocks == cfg.num_blocks
        self.history.append(st)
        self.step_no += 1
        return st

    def run(self, max_steps: int = 10**9, check=None):
        """Steps until every request finished; `check(scheduler)` (optional)
        runs after each step."""
        while (self.waiting or self.running) and self.step_no < max_steps:
            before = (len(self.waiting), len(self.running), len(self.done))
            st = self.step()
            if check is not None:
                check(self)
            if st.decoding == 0 and st.admitted == 0 and before == (
                    len(self.waiting), len(self.running), len(self.done)):
                raise RuntimeError("scheduler made no progress (all running requests stalled)")
        return self.summary()

    def summary(self) -> dict:
        h = self.history
        n = max(len(h), 1)
        return dict(
            steps=len(h), finished=len(self.done),
            tokens=sum(s.decoding for s in h),
            mean_decoding=sum(s.decoding for s in h) / n,
            peak_decoding=max((s.decoding for s in h), default=0),
            mean_block_use=sum(s.blocks_held for s in h) / n / self.cfg.num_blocks,
            preemptions=sum(s.preempted for s in h),
            stalls=sum(s.stalled for s in h),
            compressions=sum(s.compressed for s in h),
            prefill_compressions=sum(s.prefill_compressed for s in h))


def synthetic_requests(n: int, seed: int, prompt=(64, 512), out_median=3000, out_sigma=0.8,
                       out_max=16384):
    """Seeded requests: prompts uniform in `prompt`, outputs log-normal (long
    reasoning traces, median `out_median`, clipped to [16, out_max])."""
    g = np.random.default_rng(seed)
    p = g.integers(prompt[0], prompt[1] + 1, n)
    o = np.clip(np.exp(math.log(out_median) + out_sigma * g.standard_normal(n)), 16, out_max)
    return [Request(rid=i, prompt=int(p[i]), output=int(o[i])) for i in range(n)]


class GpuBackend:
    """Drives the C ABI on one GPU: a zp_cache over L layers of pools, block
    tables of ``max_rows`` rows, seeded random K/V/queries for new tokens."""

    def __init__(self, cfg: SimConfig, L=2, Hkv=2, Hq=8, d=128, device="cuda", max_row_blocks=None):
        import torch

        from . import zp
        self.torch, self.zp = torch, zp
        self.cfg, self.L, self.Hkv, self.Hq, self.d = cfg, L, Hkv, Hq, d
        dev = torch.device(device)
        self.dev = dev
        nb = cfg.num_blocks
        self.stride = max_row_blocks or max(cfg.n_max, 2)
        g = torch.Generator(device=dev)
        g.manual_seed(cfg.seed)
        self.g = g
        self.kp = [torch.randn(nb, Hkv, cfg.b, d, generator=g, device=dev).to(torch.bfloat16)
                   for _ in range(L)]
        self.vp = [torch.randn(nb, Hkv, cfg.b, d, generator=g, device=dev).to(torch.bfloat16)
                   for _ in range(L)]
        i32 = dict(dtype=torch.int32, device=dev)
        self.tables = torch.full((cfg.max_rows, self.stride), -1, **i32)
        self.lengths = torch.zeros(cfg.max_rows, **i32)
        self.free = torch.arange(nb - 1, -1, -1, **i32)
        self.fc = torch.tensor([nb], **i32)
        self.rc = torch.zeros(nb, **i32)
        self.trig = torch.zeros(cfg.max_rows, **i32)
        self.ntrig = torch.zeros(1, **i32)
        self.cache = zp.Cache(self.kp, self.vp, Hq, max_requests=cfg.max_rows,
                              max_blocks_per_req=self.stride)
        self.ws = None
        self.scale = 1.0 / math.sqrt(d)

    def _rows(self, rows):
        return self.torch.tensor(rows, dtype=self.torch.int32, device=self.dev)

    def _rand(self, shape):
        """bf16 N(0,1) draws for new tokens and window queries."""
        torch = self.torch
        return torch.randn(shape, generator=self.g, device=self.dev).to(torch.bfloat16)

    def alloc(self, rows, counts):
        self.cache.alloc_rows(self.tables, self.lengths, self._rows(counts), self.free, self.fc,
                              self.rc, req_idx=self._rows(rows))

    def prefill(self, rows):
        torch = self.torch
        R = len(rows)
        wq = self._rand((self.L, R, self.Hq, self.cfg.w, self.d))
        need = self.cache.prefill_workspace_bytes(R, self.stride)
        if self.ws is None or self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.dev)
        self.cache.compress_prefill(self.tables, self.lengths, wq, self.cfg.n_max, self.cfg.w,
                                    0.5, self.free, self.fc, self.rc, self.ws,
                                    req_idx=self._rows(rows))

    def append(self, rows):
        self.cache.append_slots(self.tables, self.lengths, self.cfg.n_max, self.free, self.fc,
                                self.rc, req_idx=self._rows(rows), trigger_rows=self.trig,
                                trigger_count=self.ntrig)
        n = int(self.ntrig.item())
        return self.trig[:n].tolist()

    def write_and_attend(self, rows):
        torch = self.torch
        ri = self._rows(rows)
        R = len(rows)
        self.last_out = []
        for l in range(self.L):
            kn = self._rand((R, self.Hkv, self.d))
            vn = self._rand((R, self.Hkv, self.d))
            q = self._rand((R, self.Hq, self.d))
            out = torch.empty_like(q)
            self.cache.append_kv(l, kn, vn, self.tables, self.lengths, req_idx=ri)
            self.cache.decode(l, q, self.tables, self.lengths, self.scale, out, req_idx=ri)
            self.last_out.append(out)

    def compress(self, rows):
        wq = self._rand((self.L, len(rows), self.Hq, self.cfg.w, self.d))
        self.cache.compress(self.tables, self.lengths, wq, self.cfg.n_max, self.cfg.w, 0.5,
                            self.free, self.fc, self.rc, req_idx=self._rows(rows))

    def release(self, rows):
        self.cache.release_rows(self.tables, self.lengths, self.free, self.fc, self.rc,
                                req_idx=self._rows(rows))

    def free_count(self) -> int:
        return int(self.fc.item())

    def status(self) -> int:
        return self.cache.status()
