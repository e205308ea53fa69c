#!/usr/bin/env python3
"""Benchmark of the compression + decode-attention hot path on one GB300.

A step = one zp_compress call over every request, layer and kv head of the
workload (plan, fused score/select/compact kernel, finalize) followed by
paged decode attention over the compacted tables, one call per layer.
Default workload: Qwen3-8B-shaped, 36 layers (8/32 heads, d 128, b 16,
N_max 128, w 8, lambda 0.5), 256 requests at N_max in 32 groups of 8 sharing
a 4-block prompt prefix (the shared blocks compress into fresh target
blocks), K AR(1) rho 0.9 with 1% heavy hitters.

Before each step (outside the timed events) the KV pools, block tables,
lengths, refcounts and free stack are restored from a pristine device copy and
a 256 MiB buffer is written and another read to flush L2, so every step
compresses the workload's own data from HBM (the read leaves L2 holding clean
lines: the write-back of the written buffer's lines is not timed as part of
the step).

`--impl reference` times the CPU oracle (plain fp64 C, all host cores) on
bounded slices of the same workload instead (the same config, steps and
warm-up).  Under torchrun each rank runs its own replica
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV tokens compressed/s and decode-attn HBM GB/s (fraction of ~8 TB/s), 1 GB300"
UNIT = "request-tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


class L2Flush:
    """Evicts the workload's data from L2 between steps: a buffer twice its
    size is written, then another one read, so L2 ends up holding clean lines
    of the second (nothing of the flush is written back inside the next timed
    region)."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="qwen3_36l")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-ablations", action="store_true",
                   help="skip the all-keys redundancy ablations timed after the step")
    p.add_argument("--e2e-steps", type=int, default=None,
                   help="steps of the end-to-end measurement (default: --steps)")
    p.add_argument("--layers", type=int, default=None,
                   help="run the workload with fewer layers (small profiling captures only; "
                        "the bench line then names the reduced workload)")
    p.add_argument("--prefill-layers", type=int, default=None,
                   help="layers of the prefill8k workload (default: the model's 36)")
    return p.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed alone."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the files the compression kernel is compiled from: the recorded DRAM
# traffic stays valid while none of them changes
COMPRESS_KERNEL_SOURCES = ["zp_compress_stream.cuh", "zp_internal.cuh", "zp_compress_d64.cu",
                           "zp_compress_d128.cu", "zp_tmap.cu"]


def kernel_source_digest():
    from compressed_paged_kv_gb300 import _build
    h = hashlib.sha256()
    paths = [os.path.join(_build.CSRC, n) for n in COMPRESS_KERNEL_SOURCES]
    for path in paths:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, units):
    """DRAM bytes per launch of the compression kernel, from a committed ncu
    summary taken on the current kernel sources (else None).  A capture of a
    reduced case of the same workload (fewer layers: the same per-unit work)
    is scaled to `units` by its DRAM bytes per unit."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_digest") == kernel_source_digest():
            if "dram_bytes_per_unit" in e:
                return float(e["dram_bytes_per_unit"]) * units
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            for n, v in zip(names, r[4:8]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.rows)}


def device_index(torch):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    idx = torch.cuda.current_device()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if idx < len(ids):
            return ids[idx]
    return idx


# ------------------------------------------------------------ multi-rank
def replica_seed(wl, rank: int) -> int:
    """Each rank compresses its own replica of the workload (units are
    independent: no collective on the data path)."""
    return wl.seed + 7919 * rank


def reduce_max(values, world: int, device=None):
    """Max over ranks of a list of floats (the step timings); identity for 1."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# ------------------------------------------------------------------ GPU arm

def run_mixed(args, world, rank, local):
    """The mixed decode step: the decoding requests reserve their next slot,
    then, on a high-priority stream, every layer writes their new K/V rows and
    runs paged decode attention, while the requests that reached N_max
    compress on a second stream; timed overlapped and serialised, with each
    stream's interval recorded."""
    import torch
    import torch.distributed as dist

    from compressed_paged_kv_gb300 import _build
    from compressed_paged_kv_gb300 import workloads as W
    from compressed_paged_kv_gb300 import zp

    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    wl = W.WORKLOADS[args.workload]
    if args.layers:
        wl = W.scaled(wl, L=args.layers)
    seed = replica_seed(wl, rank)
    # room for a fresh target block per block of every compressing request
    # (the pipelined end-to-end loop below compresses into fresh targets)
    st = W.build_cache(W.scaled(wl, spare_blocks=wl.spare_blocks + wl.mixed_compress * wl.N),
                       dev, seed=seed)
    cache = zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=st.block_tables.shape[0],
                     max_blocks_per_req=st.block_tables.shape[1])
    scale = 1.0 / math.sqrt(wl.d)
    live = [st.block_tables, st.lengths, st.refcount, st.free_ids, st.free_count]
    pristine = [t.clone() for t in live]
    flush = L2Flush(torch, dev)
    drows = st.decode_rows
    q = [st.decode_q[l][drows.long()].contiguous() for l in range(wl.L)]
    out = [torch.empty_like(x) for x in q]
    # the new token's K/V rows of every decoding request (seeded, per layer)
    k_new, v_new = mixed_new_rows(wl, drows.numel(), seed + 7, dev)
    s_dec = torch.cuda.Stream(device=dev, priority=-1)
    s_cmp = torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream()

    def compress(stream, kept=None):
        cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam, st.free_ids,
                       st.free_count, st.refcount, req_idx=st.compress_rows, stream=stream,
                       kept_out=kept)

    def append_slots(stream):
        cache.append_slots(st.block_tables, st.lengths, wl.N, st.free_ids, st.free_count,
                           st.refcount, req_idx=drows, stream=stream)

    def decode(stream):
        for l in range(wl.L):
            cache.append_kv(l, k_new[l], v_new[l], st.block_tables, st.lengths, req_idx=drows,
                            stream=stream)
            cache.decode(l, q[l], st.block_tables, st.lengths, scale, out[l], req_idx=drows,
                         stream=stream)

    # the compressing requests' blocks are rewritten in place: keep pristine
    # copies of just those slabs (every layer) and restore them before each
    # step (the decoding requests' new rows land past their restored lengths)
    blk = st.block_tables[st.compress_rows.long()].flatten().long()
    pristine_slabs = [p[blk].clone() for p in st.k_pools + st.v_pools]

    def restore():
        for a, b in zip(live, pristine):
            a.copy_(b)
        for p, saved in zip(st.k_pools + st.v_pools, pristine_slabs):
            p.index_copy_(0, blk, saved)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def step(overlap):
        restore()
        flush()
        t = {k: ev() for k in ("e0", "ea", "d0", "d1", "c0", "c1", "e1")}
        t["e0"].record(main)
        # slot reservation and compression both update the free stack and the
        # refcounts: the reservation goes first, then the two streams fork
        append_slots(main)
        t["ea"].record(main)
        if overlap:
            s_dec.wait_event(t["ea"])
            s_cmp.wait_event(t["ea"])
            t["d0"].record(s_dec)
            decode(s_dec)
            t["d1"].record(s_dec)
            t["c0"].record(s_cmp)
            compress(s_cmp)
            t["c1"].record(s_cmp)
            main.wait_event(t["d1"])
            main.wait_event(t["c1"])
        else:
            t["d0"].record(main)
            decode(main)
            t["d1"].record(main)
            t["c0"].record(main)
            compress(main)
            t["c1"].record(main)
        t["e1"].record(main)
        return t

    for _ in range(args.warmup):
        step(True)
        step(False)
    torch.cuda.synchronize()
    assert cache.status() == zp.OK
    K = args.steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    res_o, res_s = [], []
    with ClockSampler(device_index(torch)) as clk:
        for _ in range(K):
            res_o.append(step(True))
            res_s.append(step(False))
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    assert cache.status() == zp.OK

    def avg(res, a, b):
        return sum(t[a].elapsed_time(t[b]) for t in res) / len(res)

    ov, se = avg(res_o, "e0", "e1"), avg(res_s, "e0", "e1")
    slot_ms = avg(res_s, "e0", "ea")
    dec_ms, cmp_ms = avg(res_s, "d0", "d1"), avg(res_s, "c0", "c1")
    o_dec = [avg(res_o, "e0", "d0"), avg(res_o, "e0", "d1")]
    o_cmp = [avg(res_o, "e0", "c0"), avg(res_o, "e0", "c1")]
    # time both streams had work in flight: the intersection of their intervals
    concurrent = sum(max(0.0, min(t["e0"].elapsed_time(t["c1"]), t["e0"].elapsed_time(t["d1"]))
                         - max(t["e0"].elapsed_time(t["c0"]), t["e0"].elapsed_time(t["d0"])))
                     for t in res_o) / len(res_o)
    inside = sum(1 for t in res_o
                 if t["e0"].elapsed_time(t["c0"]) >= t["e0"].elapsed_time(t["d0"]) - 1e-3
                 and t["e0"].elapsed_time(t["c1"]) <= t["e0"].elapsed_time(t["d1"]) + 1e-3)
    ov_dec, ov_cmp = o_dec[1] - o_dec[0], o_cmp[1] - o_cmp[0]

    # moved rows of the compression (from its kept indices), outside the timing
    restore()
    append_slots(main)
    Rc = st.window_q.shape[1]
    kept = torch.empty((wl.L, Rc, wl.Hkv, (wl.N - 1) * wl.b), dtype=torch.int32, device=dev)
    src_tab = st.block_tables[st.compress_rows.long(), :wl.N].clone()
    compress(main, kept)
    torch.cuda.synchronize()
    moved = count_moved(kept, src_tab, st.block_tables[st.compress_rows.long(), :wl.N - 1], wl)
    row = wl.d * 2
    cmp_units = wl.units(Rc)
    cmp_bytes = cmp_units * (wl.T * row + wl.w * wl.G * row) + 3 * moved * row
    # attention reads every cached K and V row, the new token included; the
    # append reads and writes one K and one V row per (request, layer, kv head)
    dec_len = int(pristine[1][drows.long()].sum().item()) + drows.numel()
    dec_bytes = dec_len * wl.L * wl.Hkv * row * 2 + drows.numel() * wl.L * wl.Hkv * row * 4

    # e2e through host buffers: the step's inputs (window queries of the
    # compressing requests, decode queries, new K/V rows, block state) from
    # pinned host memory, the attention outputs and new block state back
    h_wq = st.window_q.cpu().pin_memory()
    h_q = [x.cpu().pin_memory() for x in q]
    h_kv = [x.cpu().pin_memory() for x in k_new + v_new]
    h_state = [t.cpu().pin_memory() for t in pristine]
    h_out = [torch.empty_like(x, device="cpu").pin_memory() for x in out]
    h_tab = torch.empty_like(st.block_tables, device="cpu").pin_memory()
    h_len = torch.empty_like(st.lengths, device="cpu").pin_memory()
    h2d = (h_wq.numel() * 2 + sum(x.numel() * 2 for x in h_q + h_kv)
           + sum(t.numel() * 4 for t in h_state))
    d2h = sum(x.numel() * 2 for x in h_out) + h_tab.numel() * 4 + h_len.numel() * 4
    E = args.e2e_steps or K
    e2e = []
    for i in range(E + 2):
        restore()
        flush()
        a0, a1 = ev(), ev()
        a0.record(main)
        st.window_q.copy_(h_wq, non_blocking=True)
        for x, h in zip(live, h_state):
            x.copy_(h, non_blocking=True)
        for x, h in zip(q + k_new + v_new, h_q + h_kv):
            x.copy_(h, non_blocking=True)
        ea = ev()
        append_slots(main)
        ea.record(main)
        s_dec.wait_event(ea)
        s_cmp.wait_event(ea)
        decode(s_dec)
        compress(s_cmp)
        dd, cc = ev(), ev()
        dd.record(s_dec)
        cc.record(s_cmp)
        main.wait_event(dd)
        main.wait_event(cc)
        for h, x in zip(h_out, out):
            h.copy_(x, non_blocking=True)
        h_tab.copy_(st.block_tables, non_blocking=True)
        h_len.copy_(st.lengths, non_blocking=True)
        a1.record(main)
        a1.synchronize()
        if i >= 2:
            e2e.append(a0.elapsed_time(a1))
    e2e_serial_ms = sum(e2e) / len(e2e)
    # as a serving loop runs it: the next step's inputs cross on a copy stream
    # into the other of two device buffer sets while this step computes (the
    # pools stay resident: no restore between steps)
    # Without a restore of the pools between its steps, each step would
    # compress what the previous one compacted, the same window queries over
    # data already thinned by them (the moved rows drift from ~1,900 to under
    # 900 per unit).  So in the block state each step's inputs restore, every
    # block of a compressing request is held twice (refcount 2): its
    # compaction goes to fresh target blocks and leaves the sources as they
    # were, and every step compresses the same data -- writing all (N_max-1)*b
    # rows of a unit, more than the device-timed step's in-place compaction.
    h_state_ft = [t.clone().pin_memory() for t in h_state]
    crows_blk = pristine[0][st.compress_rows.long()].flatten().long()
    h_state_ft[2][crows_blk.cpu()] += 1
    cp = torch.cuda.Stream(device=dev)
    # a step's inputs, and its results, each cross as one copy of one packed
    # buffer (pinned on the host) rather than as one copy per tensor
    h_src = [h_wq] + list(h_q) + list(h_kv) + list(h_state_ft)
    h_inp, hv = packed(torch, h_src, "cpu", pin=True)
    for v, t in zip(hv, h_src):
        v.copy_(t)
    nq = len(h_q) + len(h_kv)
    d_flat, d_wq, d_in, d_state = [], [], [], []
    for _ in range(2):
        flat, views = packed(torch, hv, dev)
        d_flat.append(flat)
        d_wq.append(views[0])
        d_in.append(views[1:1 + nq])
        d_state.append(views[1 + nq:])
    h_res, _ = packed(torch, list(h_out) + [h_tab, h_len], "cpu", pin=True)
    d_res, d_out, d_tab, d_len = [], [], [], []
    for _ in range(2):
        flat, views = packed(torch, list(out) + [st.block_tables, st.lengths], dev)
        d_res.append(flat)
        d_out.append(views[:len(out)])
        d_tab.append(views[len(out)])
        d_len.append(views[len(out) + 1])
    ready = [torch.cuda.Event() for _ in range(2)]   # inputs of set b landed
    free = [torch.cuda.Event() for _ in range(2)]    # step on set b computed
    back = [torch.cuda.Event() for _ in range(2)]    # results of set b on the host
    L = wl.L

    def bring(i):
        b = i % 2
        if i >= 2:
            cp.wait_event(free[b])
        with torch.cuda.stream(cp):
            d_flat[b].copy_(h_inp, non_blocking=True)
        ready[b].record(cp)

    def run(i):
        b = i % 2
        main.wait_event(ready[b])
        if i >= 2:
            main.wait_event(back[b])  # set b's previous results have left
        for x, y in zip(live, d_state[b]):
            x.copy_(y, non_blocking=True)
        append_slots(main)
        ea = ev()
        ea.record(main)
        s_dec.wait_event(ea)
        s_cmp.wait_event(ea)
        dq, dk, dv = d_in[b][:L], d_in[b][L:2 * L], d_in[b][2 * L:]
        for l in range(L):
            cache.append_kv(l, dk[l], dv[l], st.block_tables, st.lengths, req_idx=drows,
                            stream=s_dec)
            cache.decode(l, dq[l], st.block_tables, st.lengths, scale, d_out[b][l],
                         req_idx=drows, stream=s_dec)
        cache.compress(st.block_tables, st.lengths, d_wq[b], wl.N, wl.w, wl.lam, st.free_ids,
                       st.free_count, st.refcount, req_idx=st.compress_rows, stream=s_cmp)
        dd, cc = ev(), ev()
        dd.record(s_dec)
        cc.record(s_cmp)
        main.wait_event(dd)
        main.wait_event(cc)
        d_tab[b].copy_(st.block_tables, non_blocking=True)
        d_len[b].copy_(st.lengths, non_blocking=True)
        free[b].record(main)

    def take(i):
        # step i's results cross back on the copy stream while step i+1 runs
        b = i % 2
        cp.wait_event(free[b])
        with torch.cuda.stream(cp):
            h_res.copy_(d_res[b], non_blocking=True)
        back[b].record(cp)

    def loop(steps):
        bring(0)
        for i in range(steps):
            if i + 1 < steps:
                bring(i + 1)
            run(i)
            take(i)

    loop(2)
    torch.cuda.synchronize()
    p0, p1 = ev(), ev()
    p0.record(main)
    cp.wait_event(p0)
    loop(E)
    main.wait_stream(cp)  # the last step's results have reached the host
    p1.record(main)
    p1.synchronize()
    e2e_ms = p0.elapsed_time(p1) / E
    assert cache.status() == zp.OK
    # the rows an end-to-end step moves (one untimed compression from the
    # block state its inputs restore)
    for a, b in zip(live, h_state_ft):
        a.copy_(b)
    append_slots(main)
    compress(main, kept)
    torch.cuda.synchronize()
    e2e_moved = count_moved(kept, src_tab, st.block_tables[st.compress_rows.long(), :wl.N - 1], wl)

    ov, se, slot_ms, dec_ms, cmp_ms, e2e_ms, e2e_serial_ms = reduce_max(
        [ov, se, slot_ms, dec_ms, cmp_ms, e2e_ms, e2e_serial_ms], world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    peak, peak_src = peaks()
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    cmp_gbs = cmp_bytes / (cmp_ms * 1e-3) / 1e9
    step_bytes = dec_bytes + cmp_bytes
    res = {
        "metric": METRIC, "value": world * Rc * wl.T / (ov * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ov,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the named model, no weights)",
        "config": {"workload": f"{wl.name}: L={wl.L} decode step of {drows.numel()} requests "
                               f"(lengths {wl.mixed_len_lo}..{wl.T - 1}: slot reservation, then "
                               f"new K/V rows + attention per layer) on a high-priority stream, "
                               f"{Rc} requests at N_max={wl.N} compressing on a second stream",
                   "global_batch": world * wl.R, "seq_len": wl.T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read) after restoring the "
                         "compressed blocks"},
        "overlap_ms": ov, "serial_ms": se, "overlap_gain": se / ov,
        "slot_reservation_ms": slot_ms, "decode_ms": dec_ms, "compress_ms": cmp_ms,
        "compression_share_of_serial_step": cmp_ms / se,
        "compression_over_decode": cmp_ms / dec_ms,
        "streams_overlapped": {
            "decode_interval_ms": o_dec, "compress_interval_ms": o_cmp,
            "decode_ms_overlapped": ov_dec, "compress_ms_overlapped": ov_cmp,
            "concurrent_ms": concurrent,
            "compress_inside_decode_steps": inside, "of_steps": K,
            "what": "mean start/end of each stream's work from the step start, overlapped run; "
                    "concurrent_ms = mean time both streams had work in flight"},
        "roofline": {"kernel": "zp_decode_kernel (+ zp_append_kv), serial run: the dominant "
                               "part of the step", "bound": "hbm", "achieved": dec_gbs,
                     "peak": peak, "unit": "GB/s", "frac": dec_gbs / peak, "traffic": None,
                     "peak_source": peak_src, "algorithmic_bytes_per_step": dec_bytes},
        "compress_roofline": {"kernel": "zp_compress_stream_kernel (its zp_compress call), "
                                        "serial run", "bound": "hbm", "achieved": cmp_gbs,
                              "peak": peak, "unit": "GB/s", "frac": cmp_gbs / peak,
                              "algorithmic_bytes_per_call": cmp_bytes, "moved_rows": moved},
        "step_gbs_overlapped": step_bytes / (ov * 1e-3) / 1e9,
        "step_frac_overlapped": step_bytes / (ov * 1e-3) / 1e9 / peak,
        "e2e": {"value": world * Rc * wl.T / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms,
                "how": "C ABI calls, overlapped as above; each step's inputs (window queries, "
                       "decode queries, new K/V rows, block state) cross from pinned host memory "
                       "on a copy stream into one of two device buffer sets while the previous "
                       "step computes, and its outputs (attention, tables, lengths) cross back on "
                       "it while the next step computes; every copy inside the timed region; the "
                       "KV pools stay resident",
                "moved_rows_per_unit": e2e_moved / cmp_units,
                "device_step_moved_rows_per_unit": moved / cmp_units,
                "work": "the pools are not restored between end-to-end steps; the block state "
                        "each step's inputs restore holds every block of a compressing request "
                        "twice, so its compaction goes to fresh targets and every step "
                        "compresses the same data, moving all rows of a unit (above, against "
                        "the device-timed step's in-place compaction)",
                "serial_ms_per_step": e2e_serial_ms,
                "serial_value": world * Rc * wl.T / (e2e_serial_ms * 1e-3)},
        "gpu_launches": 2 * K * (2 + 3 + wl.L * (
            2 if cache_splits_one(wl, drows.numel(), cache) else 3)),
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu_baseline and not args.layers:
        res["cpu_baseline"] = mixed_cpu_baseline(wl, seed, dev)
    if world > 1:
        dist.destroy_process_group()
    return res


def mixed_new_rows(wl, n, seed, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    k = [torch.randn(n, wl.Hkv, wl.d, generator=g, device=device).to(torch.bfloat16)
         for _ in range(wl.L)]
    v = [torch.randn(n, wl.Hkv, wl.d, generator=g, device=device).to(torch.bfloat16)
         for _ in range(wl.L)]
    return k, v


def count_moved(kept, src_tab, dst_tab, wl):
    """Rows a compaction moves: destination j of a unit takes source kept[j];
    it moves unless kept[j] == j in the same physical block."""
    import torch
    L, Rc, Hkv, KT = kept.shape
    j = torch.arange(KT, device=kept.device)
    k = kept.long()
    src_blk = torch.gather(src_tab.long()[None, :, None, :].expand(L, Rc, Hkv, -1), 3,
                           k // wl.b)
    dst_blk = dst_tab.long()[None, :, None, :].repeat_interleave(wl.b, dim=3)
    return int(((k != j) | (src_blk != dst_blk)).sum().item())


def mixed_cpu_baseline(wl, seed, device):
    """The oracle on a proportional slice of the mixed step: 4 of the
    compressing requests and as many decoding requests as the same fraction
    of the decoding ones, all layers; the reservation, compression, new rows
    and attention run one after the other."""
    import numpy as np

    import oracle
    from compressed_paged_kv_gb300 import workloads as W
    orc = oracle.load()
    cores = os.cpu_count() or 1
    lay = W.layout(wl, seed)
    comp = lay.compress_rows.tolist()
    decs = lay.decode_rows.tolist()
    nc = min(4, len(comp))
    frac = nc / len(comp)
    nd = max(1, round(frac * len(decs)))
    rows = sorted(comp[:nc] + decs[:nd])
    snap = W.sample_snapshot(wl, rows, list(range(wl.L)), device=device, seed=seed,
                             spare=len(rows) * 2)
    k_new, v_new = mixed_new_rows(wl, nd, seed + 11, device)
    kq = [W.bf16_bits(x) for x in k_new]
    vq = [W.bf16_bits(x) for x in v_new]
    dr = snap["decode_rows"]
    cr = snap["compress_rows"]
    t0 = time.perf_counter()
    a = orc.append_slots(snap["k_pools"], snap["v_pools"], snap["block_tables"], snap["lengths"],
                         snap["free_ids"], snap["free_count"], snap["refcount"], wl.N,
                         req_idx=dr)
    assert a["status"] == 0
    c = orc.compress(a["kpools"], a["vpools"], a["tables"], a["lengths"], snap["window_q"], wl.N,
                     wl.w, wl.lam, a["free_ids"], a["free_count"], a["refcount"], Hq=wl.Hq,
                     req_idx=cr, want_scores=False, want_kept=False, nthreads=cores)
    assert c["status"] == 0
    for l in range(wl.L):
        s1, kp, vp = orc.append_kv(c["kpools"][l], c["vpools"][l], c["tables"], c["lengths"],
                                   kq[l], vq[l], req_idx=dr)
        assert s1 == 0
        s2, _, _ = orc.decode_attn(np.ascontiguousarray(snap["decode_q"][l][dr]), kp, vp,
                                   c["tables"][dr], c["lengths"][dr], 1.0 / math.sqrt(wl.d))
        assert s2 == 0
    secs = time.perf_counter() - t0
    full_s = secs / frac
    return {"value": len(comp) * wl.T / full_s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{nc} of {len(comp)} compressing and {nd} of {len(decs)} decoding "
                      f"requests of {wl.name}, all {wl.L} layers (reservation, compression, new "
                      f"rows, attention one after the other), fp64 C oracle on {cores} threads "
                      f"(compression and attention; the rest single-threaded), {secs:.1f} s "
                      f"wall; scaled by {len(comp)}/{nc} to the full step ({full_s:.0f} s)"}


# Compression at admission: Qwen3-8B-shaped prompts longer than the 2048-token
# budget (lengths uniform in [4096, 8192], seeded), compressed to 2032 tokens.
PREFILL = dict(name="prefill8k", R=16, L=36, Hkv=8, Hq=32, d=128, N=128, w=8, lam=0.5,
               len_lo=4096, len_hi=8192, seed=2024)


def run_prefill(args, world, rank, local):
    """One zp_compress_prefill over every request, layer and kv head; pools
    and allocator state restored and L2 flushed before each step, outside the
    timed events."""
    import torch
    import torch.distributed as dist

    from compressed_paged_kv_gb300 import _build
    from compressed_paged_kv_gb300 import workloads as W
    from compressed_paged_kv_gb300 import zp

    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    P = dict(PREFILL)
    if args.prefill_layers:
        P["L"] = args.prefill_layers
    g = torch.Generator()
    g.manual_seed(P["seed"] + rank)
    lens = torch.randint(P["len_lo"], P["len_hi"] + 1, (P["R"],), generator=g).tolist()
    c = W.prefill_cache(P["seed"] + 1000 * rank, lens, P["N"], L=P["L"], Hkv=P["Hkv"],
                        Hq=P["Hq"], d=P["d"], w=P["w"], spare=64, device=dev)
    cache = zp.Cache(c["k_pools"], c["v_pools"], P["Hq"], max_requests=P["R"],
                     max_blocks_per_req=c["stride"])
    live = [c["tables"], c["lengths"], c["refcount"], c["free_ids"], c["free_count"]]
    pristine = [t.clone() for t in live]
    pools = c["k_pools"] + c["v_pools"]
    pristine_pools = [t.clone() for t in pools]
    ws = torch.empty(cache.prefill_workspace_bytes(P["R"], c["stride"]), dtype=torch.uint8,
                     device=dev)
    flush = L2Flush(torch, dev)
    units = P["R"] * P["L"] * P["Hkv"]
    KT = (P["N"] - 1) * 16
    kept = torch.empty(P["L"], P["R"], P["Hkv"], KT, dtype=torch.int32, device=dev)

    def restore():
        for a, b in zip(live, pristine):
            a.copy_(b)
        for a, b in zip(pools, pristine_pools):
            a.copy_(b)

    def step(k=None):
        cache.compress_prefill(c["tables"], c["lengths"], c["window_q"], P["N"], P["w"], P["lam"],
                               c["free_ids"], c["free_count"], c["refcount"], ws, kept_out=k)

    for _ in range(args.warmup):
        restore()
        flush()
        step()
    torch.cuda.synchronize()
    assert cache.status() == zp.OK
    K = min(args.steps, 20)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    if world > 1:
        dist.barrier()
    with ClockSampler(device_index(torch)) as clk:
        for e0, e1 in evs:
            restore()
            flush()
            e0.record()
            step()
            e1.record()
        torch.cuda.synchronize()
    assert cache.status() == zp.OK
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / K

    # moved rows (from the kept positions) for the algorithmic bytes
    restore()
    src_tab = c["tables"][:, :P["N"] - 1].clone().long()
    step(kept)
    torch.cuda.synchronize()
    dst_tab = c["tables"][:, :P["N"] - 1].long()
    j = torch.arange(KT, device=dev)
    kk = kept.long()
    src_blk = torch.gather(pristine[0].long()[None, :, None, :].expand(P["L"], P["R"], P["Hkv"], -1),
                           3, kk // 16)
    dst_blk = dst_tab[None, :, None, :].repeat_interleave(16, dim=3)
    moved = int(((kk != j) | (src_blk != dst_blk)).sum().item())
    del src_tab
    ms, = reduce_max([ms], world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    row = P["d"] * 2
    tokens = sum(lens)
    alg = P["L"] * P["Hkv"] * tokens * row + units * P["w"] * (P["Hq"] // P["Hkv"]) * row \
        + 3 * moved * row
    peak, peak_src = peaks()
    gbs = alg / (ms * 1e-3) / 1e9
    res = {
        "metric": "prompt tokens compressed at admission/s (request-tokens)",
        "value": world * tokens / (ms * 1e-3), "unit": "request-tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the named model, no weights)",
        "config": {"workload": f"{P['name']}: L={P['L']}, 8/32 heads, d 128, {P['R']} requests "
                               f"with prompts of {min(lens)}..{max(lens)} tokens compressed to "
                               f"N_max={P['N']} blocks (2032 tokens + reserved block)",
                   "global_batch": world * P["R"], "seq_len": max(lens),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "traffic": None, "peak_source": peak_src},
        "algorithmic_bytes": alg, "moved_rows": moved, "units": units,
        "clocks": clk.summary(),
        "gpu_launches": K * 6,
    }
    if world > 1:
        dist.destroy_process_group()
    return res


# Hybrid vs strict scheduling of long reasoning requests through the library.
SCHED = dict(name="sched", R=192, L=4, Hkv=8, Hq=32, d=128, N=128, w=8, num_blocks=6144,
             query_slots=32, prompt=(128, 512), out_median=3000, out_sigma=0.6, out_max=8192,
             seed=77)


def run_sched(args, world, rank, local):
    """The step-level simulator (compressed_paged_kv_gb300.scheduler) under
    both policies on the same requests, every step running the kernels:
    admission allocation (and compression at admission after a preemption),
    slot reservation, new K/V and decode attention per layer, compression at
    N_max, release."""
    import torch

    from compressed_paged_kv_gb300 import _build
    from compressed_paged_kv_gb300 import scheduler as S

    _build.build()
    torch.cuda.set_device(local)
    P = SCHED
    res = {}
    for policy in ("hybrid", "strict"):
        reqs = S.synthetic_requests(P["R"], P["seed"] + rank, prompt=P["prompt"],
                                    out_median=P["out_median"], out_sigma=P["out_sigma"],
                                    out_max=P["out_max"])
        cfg = S.SimConfig(num_blocks=P["num_blocks"], max_rows=P["R"], n_max=P["N"], w=P["w"],
                          query_slots=P["query_slots"], strict=policy == "strict",
                          seed=P["seed"])
        stride = -(-(P["prompt"][1] + P["out_max"]) // 16)
        be = S.GpuBackend(cfg, L=P["L"], Hkv=P["Hkv"], Hq=P["Hq"], d=P["d"],
                          device=f"cuda:{local}", max_row_blocks=stride)
        sch = S.Scheduler(cfg, be, reqs)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        out = sch.run()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        assert be.status() == 0 and be.free_count() == cfg.num_blocks
        out["wall_s"] = wall
        out["tokens_per_s"] = out["tokens"] / wall
        res[policy] = out
        del sch, be
        torch.cuda.empty_cache()
    if rank != 0:
        return None
    h, s = res["hybrid"], res["strict"]
    return {
        "metric": "generated tokens/s of a simulated serving run (real kernels every step)",
        "value": world * h["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": h["steps"], "warmup": 0, "ms_per_step": 1e3 * h["wall_s"] / h["steps"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded request lengths; random K/V/queries, no model)",
        "config": {"workload": f"{P['name']}: {P['R']} requests, prompts {P['prompt']}, outputs "
                               f"log-normal median {P['out_median']} (max {P['out_max']}); "
                               f"L={P['L']}, 8/32 heads, d 128, N_max={P['N']}, "
                               f"{P['num_blocks']} blocks, {P['query_slots']} query slots",
                   "global_batch": world * P["R"], "seq_len": P["N"] * 16,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "hybrid": h, "strict": s,
        "hybrid_over_strict_steps": s["steps"] / h["steps"],
        "hybrid_over_strict_concurrency": h["mean_decoding"] / s["mean_decoding"],
    }


def run_gpu(args, world, rank, local):
    import torch
    import torch.distributed as dist

    from compressed_paged_kv_gb300 import _build
    from compressed_paged_kv_gb300 import workloads as W
    from compressed_paged_kv_gb300 import zp

    _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    wl = W.WORKLOADS[args.workload]
    if args.layers:
        wl = W.scaled(wl, L=args.layers)
    # The pipelined end-to-end loop below does not restore the pools between
    # its steps.  Where the room is affordable, the block state its steps
    # restore holds every block of a compressing request twice, so that the
    # compaction goes to fresh target blocks and every step compresses the
    # same data; the workload is then built with a fresh target per block.
    fresh_targets = wl.R * wl.N * wl.Hkv * wl.b * wl.d * 2 * 2 * wl.L <= (16 << 30)
    st = W.build_cache(W.scaled(wl, spare_blocks=wl.spare_blocks + wl.R * wl.N)
                       if fresh_targets else wl, dev, seed=replica_seed(wl, rank))
    cache = zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=st.block_tables.shape[0],
                     max_blocks_per_req=st.block_tables.shape[1])
    req_idx = st.compress_rows if wl.mixed else None
    dec_rows = st.compress_rows  # decode the compacted requests
    Rc = st.window_q.shape[1]
    T = wl.T
    scale = 1.0 / math.sqrt(wl.d)
    pristine = [t.clone() for t in (st.block_tables, st.lengths, st.refcount, st.free_ids,
                                    st.free_count)]
    live = [st.block_tables, st.lengths, st.refcount, st.free_ids, st.free_count]
    pristine_pools = [t.clone() for t in st.k_pools + st.v_pools]
    live_pools = st.k_pools + st.v_pools
    flush = L2Flush(torch, dev)
    q = [st.decode_q[l][dec_rows.long()].contiguous() for l in range(wl.L)]
    out = [torch.empty_like(x) for x in q]

    def restore(pools=True):
        for a, b in zip(live, pristine):
            a.copy_(b)
        if pools:
            for a, b in zip(live_pools, pristine_pools):
                a.copy_(b)

    def compress(scores=None, kept=None):
        cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam,
                       st.free_ids, st.free_count, st.refcount, req_idx=req_idx,
                       scores_out=scores, kept_out=kept)

    def decode():
        for l in range(wl.L):
            cache.decode(l, q[l], st.block_tables, st.lengths, scale, out[l], req_idx=dec_rows)

    K, Wm = args.steps, args.warmup
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for _ in range(Wm):
        restore()
        flush()
        compress()
        decode()
    torch.cuda.synchronize()
    assert cache.status() == zp.OK, "device error during warm-up"

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device_index(torch)) as clk:
        t_wall0 = time.perf_counter()
        for i in range(K):
            restore()
            flush()
            ev[i][0].record()
            compress()
            ev[i][1].record()
            decode()
            ev[i][2].record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    status = cache.status()
    comp_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    step_ms = sum(c + d for c, d in zip(comp_ms, dec_ms)) / K
    comp_avg = sum(comp_ms) / K
    dec_avg = sum(dec_ms) / K

    # the attention alone, after a flush that leaves L2 clean: inside the step
    # its interval also carries the write-back of the compression's last dirty
    # L2 lines (up to the L2's size), which belongs to the step, not to decode
    dec_alone = []
    for i in range(K + 3):
        flush()
        ev[0][0].record()
        decode()
        ev[0][1].record()
        ev[0][1].synchronize()
        if i >= 3:
            dec_alone.append(ev[0][0].elapsed_time(ev[0][1]))
    dec_alone_ms = sum(dec_alone) / len(dec_alone)

    # moved rows of a step (from the kept indices), for the algorithmic bytes
    restore()
    scores_dbg = None
    kept_dbg = torch.empty((wl.L, Rc, wl.Hkv, (wl.N - 1) * wl.b), dtype=torch.int32, device=dev)
    src_tab = st.block_tables[st.compress_rows.long(), :wl.N].clone()
    compress(scores_dbg, kept_dbg)
    moved = count_moved(kept_dbg, src_tab, st.block_tables[st.compress_rows.long(), :wl.N - 1], wl)
    del kept_dbg
    units = wl.units(Rc)
    row = wl.d * 2
    comp_bytes = units * (T * row + wl.w * wl.G * row) + 3 * moved * row
    comp_bytes_bound = units * wl.unit_bytes()
    dec_tokens = wl.L * Rc * (wl.N - 1) * wl.b
    dec_bytes = dec_tokens * wl.Hkv * row * 2 + 2 * wl.L * Rc * wl.Hq * row

    # e2e through host buffers: per-step inputs H2D from pinned memory,
    # decode outputs and the new block tables back to the host
    restore()
    h_wq = st.window_q.cpu().pin_memory()
    h_q = [x.cpu().pin_memory() for x in q]
    h_state = [t.cpu().pin_memory() for t in pristine]
    h_out = [torch.empty_like(x, device="cpu").pin_memory() for x in out]
    h_tab = torch.empty_like(st.block_tables, device="cpu").pin_memory()
    h_len = torch.empty_like(st.lengths, device="cpu").pin_memory()
    h2d = h_wq.numel() * 2 + sum(x.numel() * 2 for x in h_q) + sum(t.numel() * 4 for t in h_state)
    d2h = sum(x.numel() * 2 for x in h_out) + h_tab.numel() * 4 + h_len.numel() * 4
    E = args.e2e_steps or K
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # (a) one step at a time: copies, compression, attention, copies back
    e2e_ms_total = 0.0
    for i in range(E + 3):
        restore()
        flush()
        e0.record()
        st.window_q.copy_(h_wq, non_blocking=True)
        for a, b in zip(live, h_state):
            a.copy_(b, non_blocking=True)
        for a, b in zip(q, h_q):
            a.copy_(b, non_blocking=True)
        compress()
        decode()
        for a, b in zip(h_out, out):
            a.copy_(b, non_blocking=True)
        h_tab.copy_(st.block_tables, non_blocking=True)
        h_len.copy_(st.lengths, non_blocking=True)
        e1.record()
        e1.synchronize()
        if i >= 3:
            e2e_ms_total += e0.elapsed_time(e1)
    e2e_serial_ms = e2e_ms_total / E
    # the host link's rates on this machine (pinned buffers, one large copy each
    # way: the window queries there and back, the same bytes), which set what
    # the copies of a step cost
    xfer = []
    for src, dst in ((h_wq, st.window_q), (st.window_q, h_wq)):
        dst.copy_(src, non_blocking=True)
        e0.record()
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        e1.record()
        e1.synchronize()
        xfer.append(3 * src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    # (b) as a serving loop runs it: step i+1's inputs cross on a copy stream
    # into the other of two device buffer sets while step i computes; every
    # step's inputs and results still cross inside the timed region.  The
    # pools stay resident (no restore between steps): with fresh targets each
    # step compresses the same data, else the cache the previous one left,
    # its block state restored from that step's host inputs.
    h_state_e2e = h_state
    if fresh_targets:
        h_state_e2e = [t.clone().pin_memory() for t in h_state]
        held = torch.unique(pristine[0][st.compress_rows.long()].flatten().long()).cpu()
        h_state_e2e[2][held] += 1
    e2e_ms = pipelined_e2e(torch, cache, st, wl, q, out, pristine, live, h_wq, h_q, h_state_e2e,
                           h_out, h_tab, h_len, req_idx, dec_rows, scale, E)
    status2 = cache.status()
    # the rows an end-to-end step moves (one untimed compression from the
    # block state its inputs restore, on the pools the loop ended with)
    for a, b in zip(live, h_state_e2e):
        a.copy_(b)
    kept_dbg = torch.empty((wl.L, Rc, wl.Hkv, (wl.N - 1) * wl.b), dtype=torch.int32, device=dev)
    src_tab = st.block_tables[st.compress_rows.long(), :wl.N].clone()
    compress(None, kept_dbg)
    torch.cuda.synchronize()
    e2e_moved = count_moved(kept_dbg, src_tab, st.block_tables[st.compress_rows.long(), :wl.N - 1],
                            wl)
    del kept_dbg

    # ablation: the redundancy of every key against all keys of its unit (the
    # score the block-local one replaces), timed alone on the same units
    abl_ms = gram_ms = float("nan")
    if not args.no_ablations:
        restore()
        red_all = torch.empty((wl.L, Rc, wl.Hkv, st.block_tables.shape[1] * wl.b), device=dev)
        abl = []
        for i in range(6):
            flush()
            e0.record()
            cache.global_redundancy(st.block_tables, st.lengths, red_all, req_idx=req_idx, R=Rc)
            e1.record()
            e1.synchronize()
            if i >= 2:
                abl.append(e0.elapsed_time(e1))
        abl_ms = sum(abl) / len(abl)
        # ... and the same score from the dense T x T Gram of every unit on the
        # tensor cores (the cost of the original method)
        gram = []
        for i in range(6):
            flush()
            e0.record()
            cache.global_redundancy(st.block_tables, st.lengths, red_all, req_idx=req_idx, R=Rc,
                                    gram=True)
            e1.record()
            e1.synchronize()
            if i >= 2:
                gram.append(e0.elapsed_time(e1))
        gram_ms = sum(gram) / len(gram)
        assert cache.status() == zp.OK
        del red_all

    # max over ranks
    (step_ms, comp_avg, dec_avg, e2e_ms, e2e_serial_ms, t_wall, abl_ms, gram_ms,
     dec_alone_ms) = reduce_max([step_ms, comp_avg, dec_avg, e2e_ms, e2e_serial_ms, t_wall, abl_ms,
                                 gram_ms, dec_alone_ms], world, dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    req_tokens = Rc * T  # request-tokens compressed per step (per rank)
    peak, peak_src = peaks()
    comp_gbs = comp_bytes / (comp_avg * 1e-3) / 1e9
    dec_gbs = dec_bytes / (dec_avg * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": world * req_tokens / (step_ms * 1e-3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the named model, no weights)",
        "config": bench_config(wl, Rc, world),
        "compress_ms": comp_avg,
        "decode_ms": dec_avg,
        "compress_tokens_per_s": world * req_tokens / (comp_avg * 1e-3),
        "compress_gbs": comp_gbs,
        "compress_bytes_per_call": comp_bytes,
        "compress_bytes_upper_bound": comp_bytes_bound,
        "moved_rows": moved,
        "decode_gbs": dec_gbs,
        "decode_frac_of_8tbs": dec_gbs / NOMINAL_HBM_GBS,
        "decode_frac_of_measured": dec_gbs / peak,
        "compress_frac_of_8tbs": comp_gbs / NOMINAL_HBM_GBS,
        "roofline": {
            "kernel": "zp_compress_stream_kernel (timed over its zp_compress call: plan + fused + "
                      "finalize launches)",
            "bound": "hbm",
            "achieved": comp_gbs,
            "peak": peak,
            "unit": "GB/s",
            "frac": comp_gbs / peak,
            "traffic": recorded_traffic(wl.name, units),
            "peak_source": peak_src,
            "algorithmic_bytes": "per unit T*d*2 (K read) + w*G*d*2 (window q) + 3*M*d*2 "
                                 "(V read, K and V write of the M moved rows, M counted from "
                                 "the kept indices)",
            "algorithmic_bytes_per_launch": comp_bytes,
            "frac_of_8tbs": comp_gbs / NOMINAL_HBM_GBS,
            "upper_bound_bytes": {"bytes_per_launch": comp_bytes_bound,
                                  "achieved": comp_bytes_bound / (comp_avg * 1e-3) / 1e9,
                                  "frac": comp_bytes_bound / (comp_avg * 1e-3) / 1e9 / peak,
                                  "frac_of_8tbs": comp_bytes_bound / (comp_avg * 1e-3) / 1e9
                                  / NOMINAL_HBM_GBS,
                                  "what": "M = (N_max-1)*b for every unit"},
        },
        "decode_roofline": {"kernel": "zp_decode_kernel (+ its combine when split), one "
                                      "zp_paged_decode_attn call per layer",
                            "bound": "hbm", "achieved": dec_gbs, "peak": peak, "unit": "GB/s",
                            "frac": dec_gbs / peak, "bytes_per_step": dec_bytes,
                            "what": "every cached K and V row of the compacted requests, "
                                    "plus q and out",
                            "alone": {"ms": dec_alone_ms,
                                      "achieved": dec_bytes / (dec_alone_ms * 1e-3) / 1e9,
                                      "frac": dec_bytes / (dec_alone_ms * 1e-3) / 1e9 / peak,
                                      "what": "the same calls timed alone after an L2 flush that "
                                              "leaves L2 clean (in the step, the decode "
                                              "interval also carries the write-back of the "
                                              "compression's dirty L2 lines)"}},
        "e2e": {"value": world * req_tokens / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms,
                "how": "C ABI calls; each step's inputs (window and decode queries, block state) "
                       "cross from pinned host memory on a copy stream into one of two device "
                       "buffer sets while the previous step computes, and each step's outputs "
                       "(attention, tables, lengths) cross back on it while the next step "
                       "computes; every copy inside the timed region; the KV pools stay "
                       "resident",
                "serial_ms_per_step": e2e_serial_ms,
                "serial_value": world * req_tokens / (e2e_serial_ms * 1e-3),
                "moved_rows_per_unit": e2e_moved / units,
                "device_step_moved_rows_per_unit": moved / units,
                "work": ("the pools are not restored between end-to-end steps; the block state "
                         "each step's inputs restore holds every block of a compressing request "
                         "twice, so its compaction goes to fresh targets and every step "
                         "compresses the same data, moving all rows of a unit"
                         if fresh_targets else
                         "the pools are not restored between end-to-end steps (a fresh target "
                         "per block would not fit beside the pools), so each step compresses "
                         "what the previous one left") +
                        " (moved rows above, from one untimed compression, against the "
                        "device-timed step's)",
                "host_link_gbs": {"h2d": xfer[0], "d2h": xfer[1],
                                  "what": "pinned host <-> device copy rates measured beside "
                                          "the e2e loop (one large copy each way)"}},
        "gpu_launches": K * (3 + wl.L * (1 if cache_splits_one(wl, Rc, cache) else 2)),
        "wall_s_timed_loop": t_wall,
        "ablation_all_keys_redundancy": None if args.no_ablations else {
            "ms": abl_ms, "gbs": 2 * units * T * row / (abl_ms * 1e-3) / 1e9,
            "what": "zp_global_redundancy on the same units (two passes over K), outside the "
                    "timed step"},
        "ablation_dense_gram": None if args.no_ablations else {
            "ms": gram_ms, "tflops": 2.0 * units * T * T * wl.d / (gram_ms * 1e-3) / 1e12,
            "peak_tflops": bf16_peak()[0], "peak_source": bf16_peak()[1],
            "frac": 2.0 * units * T * T * wl.d / (gram_ms * 1e-3) / 1e12 / bf16_peak()[0],
            "what": "zp_global_redundancy_gram: the same score from each unit's dense T x T Gram "
                    "(tcgen05, 2 T^2 d FLOP per unit), outside the timed step"},
        "device_status": [status, status2],
    }
    res["clocks"] = clk.summary()
    if world == 1 and not args.no_cpu_baseline and not args.layers:
        # one untimed call exactly as timed, from the pristine state, for the
        # oracle's comparison on its sample
        restore()
        compress()
        torch.cuda.synchronize()
        assert cache.status() == zp.OK

        def gpu_rows(r, l):
            tab = st.block_tables[r, :wl.N - 1].long()
            return W.bf16_bits(st.k_pools[l][tab]), W.bf16_bits(st.v_pools[l][tab])

        res["cpu_baseline"] = cpu_baseline(wl, replica_seed(wl, rank), dev, gpu_rows)
        res["speedup_vs_oracle"] = res["value"] / res["cpu_baseline"]["value"]
        res["parity"] = res["cpu_baseline"].pop("parity")
    if world > 1:
        dist.destroy_process_group()
    return res


def packed(torch, tensors, device, pin=False):
    """One flat byte buffer with room for `tensors` (each at a 256-byte
    aligned offset) and views of it shaped like them."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    flat = torch.empty(n, dtype=torch.uint8, device=device)
    if pin:
        flat = flat.pin_memory()
    views = [flat[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for o, t in zip(offs, tensors)]
    return flat, views


def pipelined_e2e(torch, cache, st, wl, q, out, pristine, live, h_wq, h_q, h_state, h_out, h_tab,
                  h_len, req_idx, dec_rows, scale, E):
    """Steps through the C ABI as a serving loop runs them: a copy stream
    brings step i+1's inputs into one of two device buffer sets while the
    compute stream runs step i's attention on the other (after its
    compression, whose K re-reads through L2 the copies would churn), and
    takes step i's results (its attention outputs, block tables and lengths,
    snapshotted on the compute stream) back to the host while step i+1
    computes.  ms per step over E
    timed steps (after 2 warm-up steps; the first timed step's inputs and the
    last one's results are not overlapped, and every copy is inside the timed
    region)."""
    comp = torch.cuda.current_stream()
    cp = torch.cuda.Stream()
    L = wl.L
    # a step's inputs, and its results, each cross as one copy of one packed
    # buffer (pinned on the host) rather than as one copy per tensor
    h_in, hv = packed(torch, [h_wq] + list(h_q) + list(h_state), "cpu", pin=True)
    for v, t in zip(hv, [h_wq] + list(h_q) + list(h_state)):
        v.copy_(t)
    d_in, d_wq, d_q, d_state = [], [], [], []
    for _ in range(2):
        flat, views = packed(torch, hv, st.window_q.device)
        d_in.append(flat)
        d_wq.append(views[0])
        d_q.append(views[1:1 + L])
        d_state.append(views[1 + L:])
    h_res, _ = packed(torch, list(h_out) + [h_tab, h_len], "cpu", pin=True)
    d_res, d_out, d_tab, d_len = [], [], [], []
    for _ in range(2):
        flat, views = packed(torch, list(out) + [st.block_tables, st.lengths], st.window_q.device)
        d_res.append(flat)
        d_out.append(views[:L])
        d_tab.append(views[L])
        d_len.append(views[L + 1])
    ready = [torch.cuda.Event() for _ in range(2)]   # inputs of set b landed
    done = [torch.cuda.Event() for _ in range(2)]    # step on set b computed
    back = [torch.cuda.Event() for _ in range(2)]    # results of set b on the host
    cdone = [torch.cuda.Event() for _ in range(2)]   # compression of the step on set b done

    def bring(i):
        b = i % 2
        if i >= 2:
            cp.wait_event(done[b])
        if i >= 1:
            # the inputs cross while the previous step runs its attention: the
            # compression re-reads K through L2, which the copies would churn
            cp.wait_event(cdone[1 - b])
        with torch.cuda.stream(cp):
            d_in[b].copy_(h_in, non_blocking=True)
        ready[b].record(cp)

    def run(i):
        b = i % 2
        comp.wait_event(ready[b])
        if i >= 2:
            comp.wait_event(back[b])  # set b's previous results have left
        for x, y in zip(live, d_state[b]):
            x.copy_(y, non_blocking=True)
        cache.compress(st.block_tables, st.lengths, d_wq[b], wl.N, wl.w, wl.lam, st.free_ids,
                       st.free_count, st.refcount, req_idx=req_idx)
        cdone[b].record(comp)
        for l in range(wl.L):
            cache.decode(l, d_q[b][l], st.block_tables, st.lengths, scale, d_out[b][l],
                         req_idx=dec_rows)
        d_tab[b].copy_(st.block_tables, non_blocking=True)
        d_len[b].copy_(st.lengths, non_blocking=True)
        done[b].record(comp)

    def take(i):
        b = i % 2
        cp.wait_event(done[b])
        with torch.cuda.stream(cp):
            h_res.copy_(d_res[b], non_blocking=True)
        back[b].record(cp)

    def loop(steps):
        bring(0)
        for i in range(steps):
            run(i)
            if i + 1 < steps:
                bring(i + 1)
            take(i)

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    loop(2)  # warm-up
    torch.cuda.synchronize()
    t0.record(comp)
    cp.wait_event(t0)  # the first step's inputs too cross inside the timed region
    loop(E)
    comp.wait_stream(cp)  # the last step's results have reached the host
    t1.record(comp)
    t1.synchronize()
    return t0.elapsed_time(t1) / E


def cache_splits_one(wl, R, cache):
    """Mirror of the library's split choice (one decode launch when 1)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    pairs = R * wl.Hkv
    splits = min(16, max(1, (sms + pairs - 1) // pairs))
    splits = min(splits, max(1, wl.N // 4))
    bps = (wl.N + splits - 1) // splits
    return (wl.N + bps - 1) // bps == 1


# ------------------------------------------------------------- CPU oracle

def baseline_sample(wl):
    """(table rows, layers) of the sample the CPU baseline times: every unit
    of the small workloads; two whole prefix-sharing groups on every layer
    (so the block accounting of shared blocks is covered) where requests
    share; else enough whole requests for >= 1,024 units."""
    if wl.units() <= 1024:
        return list(range(wl.R)), list(range(wl.L))
    if wl.group > 1:
        n_groups = (wl.R + wl.group - 1) // wl.group
        rows = list(range(wl.group)) + list(range((n_groups - 1) * wl.group, wl.R))
        return rows, list(range(wl.L))
    per_req = wl.L * wl.Hkv
    n = max(1, -(-1024 // per_req))
    return list(range(0, wl.R, max(1, wl.R // n)))[:n], list(range(wl.L))


def reference_step_sample(wl, i):
    """(table rows, layers) of reference step i: a bounded slice of the
    workload (about 600 units), rotating over the requests and layers."""
    if wl.units() <= 1024:
        return list(range(wl.R)), list(range(wl.L))
    n_layers = max(1, min(wl.L, 600 // (max(wl.group, 1) * wl.Hkv)))
    stride = max(1, wl.L // n_layers)
    layers = sorted({(i % stride) + stride * k for k in range(n_layers)} & set(range(wl.L)))
    if wl.group > 1:
        n_groups = (wl.R + wl.group - 1) // wl.group
        g = (7 * i) % n_groups
        rows = list(range(g * wl.group, min((g + 1) * wl.group, wl.R)))
    else:
        n = max(1, 600 // (len(layers) * wl.Hkv))
        rows = [((7 * i) * n + k) % wl.R for k in range(n)]
        rows = sorted(set(rows))
    return rows, layers


def oracle_step(orc, wl, snap, nthreads):
    """One oracle step on a host snapshot (whole or sampled): compression of
    its compressing requests on its layers, then decode attention of the
    compacted requests on each of those layers.  Returns (seconds,
    request-tokens: compressing requests x T x the fraction of the model's
    layers the snapshot holds, the oracle's compacted state)."""
    layers = snap.get("layers", list(range(wl.L)))
    req = snap["compress_rows"] if (wl.mixed or "rows" in snap) else None
    t0 = time.perf_counter()
    res = orc.compress(snap["k_pools"], snap["v_pools"], snap["block_tables"], snap["lengths"],
                       snap["window_q"], wl.N, wl.w, wl.lam, snap["free_ids"],
                       snap["free_count"], snap["refcount"], Hq=wl.Hq, req_idx=req,
                       want_scores=False, want_kept=False, nthreads=nthreads)
    assert res["status"] == 0
    rows = snap["compress_rows"]
    dq = snap.get("decode_q")
    for li in range(len(layers)):
        q = dq[li][rows] if dq is not None else _oracle_q(wl, len(rows))
        st, _, _ = orc.decode_attn(q, res["kpools"][li], res["vpools"][li],
                                   res["tables"][rows], res["lengths"][rows],
                                   1.0 / math.sqrt(wl.d))
        assert st == 0
    secs = time.perf_counter() - t0
    return secs, len(rows) * wl.T * len(layers) / wl.L, res


def _oracle_q(wl, n):
    import numpy as np
    rng = np.random.default_rng(0)
    q = rng.standard_normal((n, wl.Hq, wl.d)).astype(np.float32)
    return (q.view(np.uint32) >> 16).astype(np.uint16)


def _gen_device():
    import torch
    return "cuda" if torch.cuda.is_available() else "cpu"


def kept_of_rows(Ks, Vs, Kg, Vg):
    """The source positions of compacted rows (ascending, as the compaction
    keeps the order): for each destination row the next source position whose
    K and V rows are byte-identical to it; None if some row is no such copy."""
    import numpy as np
    kept, p = [], 0
    for j in range(Kg.shape[0]):
        while p < Ks.shape[0] and not (np.array_equal(Ks[p], Kg[j]) and np.array_equal(Vs[p], Vg[j])):
            p += 1
        if p == Ks.shape[0]:
            return None
        kept.append(p)
        p += 1
    return np.asarray(kept)


def near_tie(s, imp, red, lam, kept_o, kept_g, evicted, tie_rtol=1e-5):
    """Whether two kept sets differ only at a near-tie: every token in their
    symmetric difference has a score within tie_rtol * max(|cut|, D) of the
    cut (the evicted-th lowest candidate score; D = mean of |imp| + lam |red|
    over the candidates)."""
    import numpy as np
    C = s.shape[0]
    cut = np.sort(s)[evicted - 1]
    D = float(np.mean(np.abs(imp[:C]) + lam * np.abs(red[:C])))
    diff = np.setxor1d(kept_o, kept_g)
    diff = diff[diff < C]
    return bool(np.all(np.abs(s[diff] - cut) <= tie_rtol * max(abs(cut), D)))


def compacted_parity(wl, snap, res, gpu_rows, check_layers, orc=None):
    """Compares, unit by unit, the compacted K and V rows of the oracle's run on
    a sample (`res`, its tables over the sample's renumbered blocks) with the
    GPU's (`gpu_rows(row, layer)` -> ([N-1][Hkv][b][d], same for V) as uint16,
    through the GPU's own tables).  Counts the units compared, those whose
    rows are byte-identical and, with the oracle `orc`, those that differ only
    at a near-tie of the scores (the GPU's kept set read back from its rows);
    any other unit is counted as a mismatch."""
    import numpy as np
    rows = snap["rows"]
    layers = snap["layers"]
    G, T, b, d = wl.G, wl.T, wl.b, wl.d
    n, same, ties, bad = 0, 0, 0, 0
    for l in check_layers:
        li = layers.index(l)
        for k, i in enumerate(snap["compress_rows"]):
            tab = res["tables"][i][:wl.N - 1]
            ko, vo = res["kpools"][li][tab], res["vpools"][li][tab]
            kg, vg = gpu_rows(rows[i], l)
            for h in range(wl.Hkv):
                n += 1
                if np.array_equal(ko[:, h], kg[:, h]) and np.array_equal(vo[:, h], vg[:, h]):
                    same += 1
                    continue
                if orc is None:
                    bad += 1
                    continue
                src = snap["block_tables"][i][:wl.N]
                Ks = snap["k_pools"][li][src][:, h].reshape(T, d)
                Vs = snap["v_pools"][li][src][:, h].reshape(T, d)
                Q = snap["window_q"][li][k][h * G:(h + 1) * G].reshape(-1, d)
                imp, red, sc = orc.unit_scores(Ks, Q, b, wl.w, G, wl.lam)
                kept_o = orc.select(sc, wl.w, wl.n_keep)
                kept_g = kept_of_rows(Ks, Vs, kg[:, h].reshape(-1, d), vg[:, h].reshape(-1, d))
                if kept_g is not None and near_tie(sc, imp, red, wl.lam, kept_o, kept_g, b):
                    ties += 1
                else:
                    bad += 1
    return {"units": n, "byte_identical": same, "near_ties": ties, "mismatches": bad,
            "layers": list(check_layers),
            "what": "compacted K/V rows of the sampled units, the bench's own call (no debug "
                    "outputs) against the oracle on the same inputs; a unit that differs only "
                    "where oracle scores tie within 1e-5 of the cut is a near-tie"}


def cpu_baseline(wl, seed, device, gpu_rows=None):
    import oracle
    from compressed_paged_kv_gb300 import workloads as W
    orc = oracle.load()
    cores = os.cpu_count() or 1
    rows, layers = baseline_sample(wl)
    snap = W.sample_snapshot(wl, rows, layers, device=device, seed=seed,
                             spare=len(rows) * (wl.prefix_blocks + 2))
    secs, toks, ores = oracle_step(orc, wl, snap, cores)
    parity = None
    if gpu_rows is not None:
        check = sorted({layers[0], layers[len(layers) // 2], layers[-1]})
        parity = compacted_parity(wl, snap, ores, gpu_rows, check, orc)
    units = len(snap["compress_rows"]) * len(layers) * wl.Hkv
    v = toks / secs
    full_s = wl.R * wl.T / v
    return {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "units_per_s": units / secs, "full_step_s_extrapolated": full_s, "parity": parity,
            "sample": f"{units} of {wl.units()} units of {wl.name} ({len(rows)} whole requests"
                      f"{' = 2 whole sharing groups' if wl.group > 1 and units < wl.units() else ''}"
                      f", {len(layers)} layers, compression + decode of the compacted requests),"
                      f" fp64 C oracle on {cores} threads, {secs:.1f} s wall; the full step "
                      f"extrapolates to {full_s:.0f} s"}


def bench_config(wl, Rc, world, layers=None):
    """The `config` of the bench line (the same for both arms)."""
    L = wl.L if layers is None else layers
    return {
        "workload": f"{wl.name}: L={L} Hkv={wl.Hkv} Hq={wl.Hq} d={wl.d} b={wl.b} "
                    f"N_max={wl.N} w={wl.w} lambda={wl.lam} R={Rc}"
                    + (f", {wl.R // wl.group} groups of {wl.group} sharing a "
                       f"{wl.prefix_blocks}-block prefix" if wl.group > 1 else "")
                    + (f", K AR(1) rho={wl.rho}" if wl.rho else "")
                    + (f" + {wl.hh_prob:.0%} heavy hitters x{wl.hh_scale:g}" if wl.hh_prob
                       else ""),
        "global_batch": world * Rc,
        "seq_len": wl.T,
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "l2": "flushed between steps (256 MiB write, then 256 MiB read) after restoring the pools",
        "step": "zp_compress (all layers/heads) + zp_paged_decode_attn per layer",
    }


def run_reference(args, world, rank):
    """The CPU oracle as it stands, on the host cores: each step one bounded
    sample of the workload (built outside the timed region), timed as
    compression + decode; value = request-tokens of the samples / time."""
    if rank != 0:
        return None
    import oracle
    from compressed_paged_kv_gb300 import workloads as W
    oracle.build()
    orc = oracle.load()
    wl = W.WORKLOADS[args.workload]
    dev = _gen_device()
    cores = os.cpu_count() or 1
    Rc = len(W.layout(wl, wl.seed).compress_rows)

    def sample(i):
        rows, layers = reference_step_sample(wl, i)
        return W.sample_snapshot(wl, rows, layers, device=dev,
                                 spare=len(rows) * (wl.prefix_blocks + 2))

    for i in range(args.warmup):
        oracle_step(orc, wl, sample(i), cores)
    secs, toks, units = 0.0, 0.0, 0
    for i in range(args.steps):
        snap = sample(args.warmup + i)
        s_, t_, _ = oracle_step(orc, wl, snap, cores)
        secs += s_
        toks += t_
        units += len(snap["compress_rows"]) * len(snap["layers"]) * wl.Hkv
    v = toks / secs
    per = units // max(args.steps, 1)
    sample_txt = (f"{args.steps} steps, each a slice of {wl.name} of about {per} units "
                  f"(whole requests{' of one sharing group' if wl.group > 1 else ''} on a "
                  f"rotating subset of layers; compression + decode of the compacted requests)"
                  if per < wl.units() else f"{args.steps} full {wl.name} steps")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the named model, no weights)",
        "config": bench_config(wl, Rc, world),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample_txt + f", fp64 C oracle on {cores} threads"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    elif args.workload == "mixed":
        res = run_mixed(args, world, rank, local)
    elif args.workload == PREFILL["name"]:
        res = run_prefill(args, world, rank, local)
    elif args.workload == SCHED["name"]:
        res = run_sched(args, world, rank, local)
    else:
        res = run_gpu(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
