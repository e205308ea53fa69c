#!/usr/bin/env python3
"""Benchmark of the compression + decode-attention hot path on one GB300.

A step = one zp_compress call over every request, layer and kv head of the
workload (plan, fused score/select/compact kernel, finalize) followed by
paged decode attention over the compacted tables, one call per layer.
Default workload: Qwen3-8B-shaped single layer (8/32 heads, d 128, b 16,
N_max 128, w 8, lambda 0.5, 64 requests at N_max, no sharing).

Before each step (outside the timed events) the KV pools, block tables,
lengths, refcounts and free stack are restored from a pristine device copy and
a 256 MiB buffer is written to flush L2, so every step compresses the
workload's own data from HBM.

`--impl reference` times the CPU oracle (plain fp64 C, all host cores) on
the same workload instead.  Under torchrun each rank runs its own replica
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


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="qwen3_1l")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
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
                           "zp_compress_d128.cu"]


def kernel_source_digest():
    from compressed_paged_kv_gb300 import _build
    h = hashlib.sha256()
    paths = [os.path.join(_build.CSRC, n) for n in COMPRESS_KERNEL_SOURCES]
    for path in paths:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_digest") == kernel_source_digest():
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
    compress on a second stream; timed overlapped and serialised."""
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
    st = W.build_cache(wl, dev, seed=replica_seed(wl, rank))
    cache = zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=st.block_tables.shape[0],
                     max_blocks_per_req=st.block_tables.shape[1])
    scale = 1.0 / math.sqrt(wl.d)
    live = [st.block_tables, st.lengths, st.refcount, st.free_ids, st.free_count]
    pristine = [t.clone() for t in live]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    drows = st.decode_rows
    q = [st.decode_q[l][drows.long()].contiguous() for l in range(wl.L)]
    out = [torch.empty_like(x) for x in q]
    # the new token's K/V rows of every decoding request (seeded, per layer)
    gkv = torch.Generator(device=dev)
    gkv.manual_seed(replica_seed(wl, rank) + 7)
    k_new = [torch.randn(drows.numel(), wl.Hkv, wl.d, generator=gkv, device=dev)
             .to(torch.bfloat16) for _ in range(wl.L)]
    v_new = [torch.randn(drows.numel(), wl.Hkv, wl.d, generator=gkv, device=dev)
             .to(torch.bfloat16) for _ in range(wl.L)]
    s_dec = torch.cuda.Stream(device=dev, priority=-1)
    s_cmp = torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream()

    def compress(stream):
        cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam, st.free_ids,
                       st.free_count, st.refcount, req_idx=st.compress_rows, stream=stream)

    def append_slots(stream):
        cache.append_slots(st.block_tables, st.lengths, wl.N, st.free_ids, st.free_count,
                           st.refcount, req_idx=drows, stream=stream)

    def decode(stream):
        for l in range(wl.L):
            cache.append_kv(l, k_new[l], v_new[l], st.block_tables, st.lengths, req_idx=drows,
                            stream=stream)
            cache.decode(l, q[l], st.block_tables, st.lengths, scale, out[l], req_idx=drows,
                         stream=stream)

    # the compressing requests' blocks are rewritten in place: keep a pristine
    # copy of just those slabs (every layer) and restore them before each step
    cblk = st.block_tables[st.compress_rows.long()].flatten().long()
    pristine_slabs = [p[cblk].clone() for p in st.k_pools + st.v_pools]

    def step(overlap):
        for a, b in zip(live, pristine):
            a.copy_(b)
        for p, saved in zip(st.k_pools + st.v_pools, pristine_slabs):
            p.index_copy_(0, cblk, saved)
        flush.zero_()
        e0, ea, ed, ec, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(5))
        e0.record(main)
        # slot reservation and compression both update the free stack and the
        # refcounts: the reservation goes first, then the two streams fork
        append_slots(main)
        ea.record(main)
        if overlap:
            s_dec.wait_event(ea)
            s_cmp.wait_event(ea)
            decode(s_dec)
            ed.record(s_dec)
            compress(s_cmp)
            ec.record(s_cmp)
            main.wait_event(ed)
            main.wait_event(ec)
        else:
            decode(main)
            ed.record(main)
            compress(main)
            ec.record(main)
        e1.record(main)
        return e0, ea, ed, ec, e1

    for _ in range(args.warmup):
        step(True)
        step(False)
    torch.cuda.synchronize()
    K = min(args.steps, 20)
    res_o, res_s = [], []
    for _ in range(K):
        res_o.append(step(True))
        res_s.append(step(False))
    torch.cuda.synchronize()
    assert cache.status() == zp.OK
    ov = sum(e0.elapsed_time(e1) for e0, _, _, _, e1 in res_o) / K
    se = sum(e0.elapsed_time(e1) for e0, _, _, _, e1 in res_s) / K
    slot_ms = sum(e0.elapsed_time(ea) for e0, ea, _, _, _ in res_s) / K
    dec_ms = sum(ea.elapsed_time(ed) for _, ea, ed, _, _ in res_s) / K
    cmp_ms = sum(ed.elapsed_time(ec) for _, _, ed, ec, _ in res_s) / K
    ov, se, slot_ms, dec_ms, cmp_ms = reduce_max([ov, se, slot_ms, dec_ms, cmp_ms], world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    Rc = st.window_q.shape[1]
    row = wl.d * 2
    # attention reads every cached K and V row, the new token included; the
    # append reads and writes one K and one V row per (request, layer, kv head)
    dec_len = int(pristine[1][drows.long()].sum().item()) + drows.numel()
    dec_bytes = dec_len * wl.L * wl.Hkv * row * 2 + drows.numel() * wl.L * wl.Hkv * row * 4
    peak, peak_src = peaks()
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
                   "l2": "flushed between steps"},
        "overlap_ms": ov, "serial_ms": se, "slot_reservation_ms": slot_ms,
        "decode_ms": dec_ms, "compress_ms": cmp_ms,
        "overlap_gain": se / ov, "decode_gbs": dec_bytes / (dec_ms * 1e-3) / 1e9,
        "decode_frac_of_measured": dec_bytes / (dec_ms * 1e-3) / 1e9 / peak,
        "compression_share_of_serial_step": cmp_ms / se,
        "gpu_launches": 2 * K * (2 + 3 + wl.L * (
            2 if cache_splits_one(wl, drows.numel(), cache) else 3)),
    }
    if world > 1:
        dist.destroy_process_group()
    return res


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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
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
        flush.zero_()
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
            flush.zero_()
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
                   "l2": "flushed between steps"},
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
    st = W.build_cache(wl, dev, seed=replica_seed(wl, rank))
    host_snap = W.snapshot(st) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
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
        flush.zero_()
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
            flush.zero_()
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

    # moved rows of a step (from the kept indices), for the algorithmic bytes
    restore()
    scores_dbg = None
    kept_dbg = torch.empty((wl.L, Rc, wl.Hkv, (wl.N - 1) * wl.b), dtype=torch.int32, device=dev)
    src_tab = st.block_tables[st.compress_rows.long(), :wl.N].clone()
    compress(scores_dbg, kept_dbg)
    dst_tab = st.block_tables[st.compress_rows.long(), :wl.N - 1]
    j = torch.arange((wl.N - 1) * wl.b, device=dev, dtype=torch.int32)
    k = kept_dbg.long()
    src_blk = torch.gather(src_tab.long()[None, :, None, :].expand(wl.L, Rc, wl.Hkv, wl.N), 3,
                           k // wl.b)
    dst_blk = dst_tab.long()[None, :, None, :].repeat_interleave(wl.b, dim=3)
    moved = int(((k != j) | (src_blk != dst_blk)).sum().item())
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
    E = args.e2e_steps
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms_total = 0.0
    for i in range(E + 3):
        restore()
        flush.zero_()
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
    e2e_ms = e2e_ms_total / E
    status2 = cache.status()

    # ablation: the redundancy of every key against all keys of its unit (the
    # score the block-local one replaces), timed alone on the same units
    restore()
    red_all = torch.empty((wl.L, Rc, wl.Hkv, st.block_tables.shape[1] * wl.b), device=dev)
    abl = []
    for i in range(6):
        flush.zero_()
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
        flush.zero_()
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
    step_ms, comp_avg, dec_avg, e2e_ms, t_wall, abl_ms, gram_ms = reduce_max(
        [step_ms, comp_avg, dec_avg, e2e_ms, t_wall, abl_ms, gram_ms], world, dev)

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
        "config": {
            "workload": f"{wl.name}: L={wl.L} Hkv={wl.Hkv} Hq={wl.Hq} d={wl.d} b={wl.b} "
                        f"N_max={wl.N} w={wl.w} lambda={wl.lam} R={Rc}",
            "global_batch": world * Rc,
            "seq_len": T,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed between steps (256 MiB write) after restoring the pools",
            "step": "zp_compress (all layers/heads) + zp_paged_decode_attn per layer",
        },
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
            "traffic": recorded_traffic(wl.name),
            "peak_source": peak_src,
            "algorithmic_bytes": "per unit T*d*2 (K read) + w*G*d*2 (window q) + 3*M*d*2 "
                                 "(V read, K and V write of the M moved rows)",
        },
        "e2e": {"value": world * req_tokens / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": e2e_ms},
        "gpu_launches": K * (3 + wl.L * (1 if cache_splits_one(wl, Rc, cache) else 2)),
        "wall_s_timed_loop": t_wall,
        "ablation_all_keys_redundancy": {
            "ms": abl_ms, "gbs": 2 * units * T * row / (abl_ms * 1e-3) / 1e9,
            "what": "zp_global_redundancy on the same units (two passes over K), outside the "
                    "timed step"},
        "ablation_dense_gram": {
            "ms": gram_ms, "tflops": 2.0 * units * T * T * wl.d / (gram_ms * 1e-3) / 1e12,
            "peak_tflops": bf16_peak()[0], "peak_source": bf16_peak()[1],
            "frac": 2.0 * units * T * T * wl.d / (gram_ms * 1e-3) / 1e12 / bf16_peak()[0],
            "what": "zp_global_redundancy_gram: the same score from each unit's dense T x T Gram "
                    "(tcgen05, 2 T^2 d FLOP per unit), outside the timed step"},
        "device_status": [status, status2],
    }
    res["clocks"] = clk.summary()
    if host_snap is not None:
        res["cpu_baseline"] = cpu_baseline(wl, host_snap, req_tokens)
    if world > 1:
        dist.destroy_process_group()
    return res


def cache_splits_one(wl, R, cache):
    """Mirror of the library's split choice (one decode launch when 1)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    pairs = R * wl.Hkv
    splits = min(16, max(1, (4 * sms + pairs - 1) // pairs))
    splits = min(splits, max(1, wl.N // 4))
    bps = (wl.N + splits - 1) // splits
    return (wl.N + bps - 1) // bps == 1


# ------------------------------------------------------------- CPU oracle

def oracle_step(orc, wl, snap, nthreads):
    """One oracle step on host copies: whole compression, then decode of the
    compacted requests on every layer.  Returns seconds."""
    import numpy as np
    t0 = time.perf_counter()
    req = snap["compress_rows"] if wl.mixed else None
    res = orc.compress(snap["k_pools"], snap["v_pools"], snap["block_tables"], snap["lengths"],
                       snap["window_q"], wl.N, wl.w, wl.lam, snap["free_ids"],
                       snap["free_count"], snap["refcount"], Hq=wl.Hq, req_idx=req,
                       want_scores=False, want_kept=False, nthreads=nthreads)
    assert res["status"] == 0
    rows = snap["compress_rows"]
    rng = np.random.default_rng(0)
    for l in range(wl.L):
        q = rng.standard_normal((len(rows), wl.Hq, wl.d)).astype(np.float32)
        qb = (q.view(np.uint32) >> 16).astype(np.uint16)
        st, _, _ = orc.decode_attn(qb, res["kpools"][l], res["vpools"][l],
                                   res["tables"][rows], res["lengths"][rows],
                                   1.0 / math.sqrt(wl.d))
        assert st == 0
    return time.perf_counter() - t0


def cpu_baseline(wl, snap, req_tokens):
    import oracle
    orc = oracle.load()
    cores = os.cpu_count() or 1
    secs = oracle_step(orc, wl, snap, cores)
    return {"value": req_tokens / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one full step of {wl.name} (all {wl.units(snap['window_q'].shape[1])} "
                      f"units + decode of the compacted requests), fp64 C oracle, "
                      f"{secs:.1f} s wall"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    from compressed_paged_kv_gb300 import workloads as W
    oracle.build()
    orc = oracle.load()
    wl = W.WORKLOADS[args.workload]
    st = W.build_cache(wl, "cpu")
    snap = W.snapshot(st)
    del st
    cores = os.cpu_count() or 1
    Rc = snap["window_q"].shape[1]
    req_tokens = Rc * wl.T
    for _ in range(args.warmup if args.warmup < 3 else 3):
        oracle_step(orc, wl, snap, cores)
    t = [oracle_step(orc, wl, snap, cores) for _ in range(min(args.steps, 5))]
    step_s = sum(t) / len(t)
    v = req_tokens / step_s
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": len(t), "warmup": min(args.warmup, 3), "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "global_batch": Rc, "seq_len": wl.T,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"full {wl.name} steps (compress + decode), "
                                   f"{len(t)} timed"},
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
