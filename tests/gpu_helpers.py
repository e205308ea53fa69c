"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs.

Parity criteria (per unit = request x layer x kv head):
  * scores:  |s_gpu - s_orc| <= 1e-4 * max(|s_orc|, D), D = mean_j(|imp_j| +
             lambda |red_j|) over the candidates (a purely relative test is
             ill-posed where imp and lambda*red cancel);
  * kept set: identical, or every token of the symmetric difference has an
             oracle score within 1e-5 * max(|s_cut|, D) of the cut (the b-th
             lowest candidate score) -- a near-tie, counted and reported;
  * compacted K/V rows: bit-exact copies of the source rows at the kept
             indices (the GPU's own kept set at a near-tie);
  * block tables, lengths, refcounts, free stack: exact (oracle plan+commit);
  * decode attention: within 2e-2 absolute of the oracle (bf16 output, fp32
             accumulation).
"""
from __future__ import annotations

import concurrent.futures
import math
import os

import numpy as np
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

SCORE_RTOL = 1e-4
TIE_RTOL = 1e-5
DECODE_ATOL = 2e-2


def bits(t):
    return W.bf16_bits(t)


def gather_units(pool, tables, rows):
    """K (or V) rows of requests `rows` in token order: [n, Hkv, T', d]."""
    x = pool[tables[rows].long()]  # [n, N', Hkv, 16, d]
    n, Np, Hkv, b, d = x.shape
    return x.permute(0, 2, 1, 3, 4).reshape(n, Hkv, Np * b, d)


def make_cache(st: W.CacheState):
    wl = st.wl
    return zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=st.block_tables.shape[0],
                    max_blocks_per_req=st.block_tables.shape[1])


class CompressRun:
    """One GPU compression of a cache state, with debug outputs."""

    def __init__(self, st: W.CacheState, cache=None, debug=True, with_scores=True):
        """debug: ask for the kept indices; with_scores: also for the scores.
        debug=False passes NULL for both outputs, as a production caller
        (and the bench) does."""
        wl = st.wl
        self.st = st
        self.cache = cache or make_cache(st)
        self.req_idx = st.compress_rows if wl.mixed else None
        Rc = st.window_q.shape[1]
        self.Rc = Rc
        dev = st.block_tables.device
        self.scores = (torch.full((wl.L, Rc, wl.Hkv, wl.T), float("nan"), device=dev)
                       if debug and with_scores else None)
        self.kept = (torch.full((wl.L, Rc, wl.Hkv, (wl.N - 1) * wl.b), -1, dtype=torch.int32,
                                device=dev) if debug else None)

    def launch(self, stream=None):
        st, wl = self.st, self.st.wl
        return self.cache.compress(st.block_tables, st.lengths, st.window_q, wl.N, wl.w, wl.lam,
                                   st.free_ids, st.free_count, st.refcount, req_idx=self.req_idx,
                                   scores_out=self.scores, kept_out=self.kept, stream=stream)

    def run(self):
        rc = self.launch()
        return rc, self.cache.status()


def int_state(st: W.CacheState):
    return dict(tables=st.block_tables.cpu().numpy().copy(), lengths=st.lengths.cpu().numpy().copy(),
                refcount=st.refcount.cpu().numpy().copy(), free_ids=st.free_ids.cpu().numpy().copy(),
                free_count=int(st.free_count.cpu().item()))


def oracle_int_update(orc, before, wl, req_idx):
    s = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in before.items()}
    st, dst, pops = orc.plan(s["tables"], s["lengths"], s["refcount"], s["free_ids"],
                             s["free_count"], wl.N, wl.b, s["refcount"].shape[0],
                             req_idx=req_idx)
    if st != 0:
        return st, s
    s["free_count"] = orc.commit(s["tables"], s["lengths"], s["refcount"], s["free_ids"],
                                 s["free_count"], dst, pops, wl.N, wl.b, req_idx=req_idx)
    return st, s


def check_ints(got, want):
    assert np.array_equal(got["tables"], want["tables"]), "block tables differ"
    assert np.array_equal(got["lengths"], want["lengths"]), "lengths differ"
    assert np.array_equal(got["refcount"], want["refcount"]), "refcounts differ"
    assert got["free_count"] == want["free_count"], (got["free_count"], want["free_count"])
    fc = want["free_count"]
    assert np.array_equal(got["free_ids"][:fc], want["free_ids"][:fc]), "free stacks differ"


class UnitReport:
    def __init__(self):
        self.units = 0
        self.exact = 0
        self.near_ties = 0
        self.max_score_err = 0.0  # relative to max(|s|, D)


def kept_from_rows(Ksrc, Vsrc, Kout, Vout, b):
    """The kept positions a compaction used, read back from its output rows:
    output row j is the copy of source row kept[j], kept strictly increasing
    with j <= kept[j] <= j + b (exactly b candidates are evicted).  Matching
    each output (K, V) row pair to the first unused source position whose
    bytes equal it gives a kept set that reproduces the output exactly (the
    kept set itself wherever source rows are distinct).  None when some
    output row is not such a copy."""
    n = Kout.shape[0]
    kept = np.empty(n, dtype=np.int64)
    i = 0
    for j in range(n):
        while i <= j + b and i < Ksrc.shape[0] and not (
                np.array_equal(Ksrc[i], Kout[j]) and np.array_equal(Vsrc[i], Vout[j])):
            i += 1
        if i > j + b or i >= Ksrc.shape[0]:
            return None
        kept[j] = i
        i += 1
    return kept


def check_unit(orc, wl, Ksrc, Vsrc, Q, s_gpu, kept_gpu, Kout, Vout):
    """Ksrc/Vsrc: [T, d] uint16 source rows; Q: [G*w, d]; s_gpu [T] fp32 (None:
    not asked for); kept_gpu [(N-1)b] (None: not asked for -- the kept set is
    then read back from the compacted rows); Kout/Vout [(N-1)b, d] uint16
    compacted rows.  Returns (kept set identical to the oracle's, worst
    relative score error)."""
    C, b = wl.C, wl.b
    imp, red, s = orc.unit_scores(Ksrc, Q, b, wl.w, wl.G, wl.lam)
    D = float(np.mean(np.abs(imp) + wl.lam * np.abs(red[:C])))
    worst = 0.0
    if s_gpu is not None:
        sg = s_gpu.astype(np.float64)
        assert np.all(np.isposinf(sg[C:])), "window positions must hold +inf"
        rel = np.abs(sg[:C] - s) / np.maximum(np.abs(s), D)
        worst = float(rel.max())
        assert worst <= SCORE_RTOL, f"score error {worst:.3e} > {SCORE_RTOL}"
    kept_o = orc.select(s, wl.w, wl.n_keep)
    if kept_gpu is None:
        if np.array_equal(Kout, Ksrc[kept_o]) and np.array_equal(Vout, Vsrc[kept_o]):
            return True, worst
        kept_gpu = kept_from_rows(Ksrc, Vsrc, Kout, Vout, b)
        assert kept_gpu is not None, "a compacted row is not a copy of a source row"
    kg = kept_gpu.astype(np.int64)
    assert kg.shape == kept_o.shape
    assert np.all(np.diff(kg) > 0), "GPU kept indices not strictly increasing"
    assert np.array_equal(kg[-wl.w:], np.arange(C, wl.T)), "window not kept"
    exact = bool(np.array_equal(kg, kept_o))
    if not exact:
        cut = np.sort(s)[b - 1]
        diff = np.setxor1d(kg, kept_o)
        tol = TIE_RTOL * max(abs(cut), D)
        assert np.all(np.abs(s[diff] - cut) <= tol), (
            f"kept sets differ beyond a near-tie: {diff.tolist()[:8]} "
            f"dev {np.abs(s[diff] - cut).max():.3e} tol {tol:.3e}")
    assert np.array_equal(Kout, Ksrc[kg]), "compacted K rows differ"
    assert np.array_equal(Vout, Vsrc[kg]), "compacted V rows differ"
    return exact, worst


class CompressCheck:
    """A GPU compression checked against the oracle, in three steps so that a
    caller can launch it on a stream of its choice next to other work:
    __init__ records the state before (integer state, the source rows of the
    sampled units, the shared blocks), launch() enqueues the compression,
    verify() (after the caller synchronised) compares everything with the
    oracle.

    sample_rows: compress-batch indices (all when None); sample_layers: layers
    (all when None); with_scores: ask for the score output; debug=False passes
    NULL for both debug outputs, as the bench's timed call does -- the kept
    sets are then read back from the compacted rows."""

    def __init__(self, orc, st: W.CacheState, sample_rows=None, sample_layers=None,
                 with_scores=True, debug=True, cache=None):
        wl = st.wl
        self.orc, self.st, self.wl = orc, st, wl
        Rc = st.window_q.shape[1]
        self.rows_c = np.arange(Rc) if sample_rows is None else np.asarray(sample_rows)
        self.layers = list(range(wl.L)) if sample_layers is None else list(sample_layers)
        self.comp_rows = st.compress_rows.cpu().numpy()
        self.tab_rows = torch.as_tensor(self.comp_rows[self.rows_c],
                                        device=st.block_tables.device).long()
        self.before = int_state(st)
        self.src = {}
        for l in self.layers:
            self.src[l] = (bits(gather_units(st.k_pools[l], st.block_tables, self.tab_rows)),
                           bits(gather_units(st.v_pools[l], st.block_tables, self.tab_rows)))
        self.wq = bits(st.window_q[self.layers][:, torch.as_tensor(self.rows_c).long()])
        self.shared = torch.nonzero(st.refcount > 1).flatten()
        self.shared_before = [(bits(st.k_pools[l][self.shared]), bits(st.v_pools[l][self.shared]))
                              for l in self.layers]
        self.with_scores = with_scores and debug
        self.run = CompressRun(st, cache=cache, debug=debug, with_scores=with_scores)

    def launch(self, stream=None):
        rc = self.run.launch(stream=stream)
        assert rc == zp.OK, rc

    def verify(self, threads=None):
        st, wl, orc, run = self.st, self.wl, self.orc, self.run
        dev = run.cache.status()
        assert dev == zp.OK, dev
        after = int_state(st)
        ost, want = oracle_int_update(orc, self.before, wl, self.comp_rows if wl.mixed else None)
        assert ost == 0
        check_ints(after, want)
        for i, l in enumerate(self.layers):
            assert np.array_equal(bits(st.k_pools[l][self.shared]), self.shared_before[i][0]), \
                "shared K block written"
            assert np.array_equal(bits(st.v_pools[l][self.shared]), self.shared_before[i][1]), \
                "shared V block written"

        new_tab = st.block_tables[:, :wl.N - 1]
        scores = run.scores.cpu().numpy() if self.with_scores else None
        kept = run.kept.cpu().numpy() if run.kept is not None else None
        rep = UnitReport()
        jobs = []
        for i, l in enumerate(self.layers):
            Kn = bits(gather_units(st.k_pools[l], new_tab, self.tab_rows))
            Vn = bits(gather_units(st.v_pools[l], new_tab, self.tab_rows))
            Ks, Vs = self.src[l]
            for j, rcmp in enumerate(self.rows_c):
                for h in range(wl.Hkv):
                    Q = self.wq[i, j, h * wl.G:(h + 1) * wl.G].reshape(-1, wl.d)
                    jobs.append((Ks[j, h], Vs[j, h], Q,
                                 None if scores is None else scores[l, rcmp, h],
                                 None if kept is None else kept[l, rcmp, h], Kn[j, h], Vn[j, h]))
        nthreads = threads or min(32, os.cpu_count() or 1)
        with concurrent.futures.ThreadPoolExecutor(nthreads) as ex:
            futs = [ex.submit(check_unit, orc, wl, *job) for job in jobs]
            for f in futs:
                exact, worst = f.result()
                rep.units += 1
                rep.exact += exact
                rep.near_ties += not exact
                rep.max_score_err = max(rep.max_score_err, worst)
        assert rep.units == len(jobs)
        print(f"[parity] {wl.name}: units {rep.units} exact {rep.exact} near-ties "
              f"{rep.near_ties} max score err {rep.max_score_err:.2e}"
              + ("" if run.kept is not None else " (no debug outputs: kept sets from the rows)"))
        return rep


def check_compress(orc, st: W.CacheState, sample_rows=None, sample_layers=None, threads=None,
                   with_scores=True, debug=True):
    """Runs one GPU compression of `st` and checks it against the oracle on the
    units of `sample_rows` (compress-batch indices) x `sample_layers` x all kv
    heads (all units when None).  with_scores=False runs it without the score
    output; debug=False without the score and the kept-index outputs (both
    NULL).  Returns the UnitReport."""
    chk = CompressCheck(orc, st, sample_rows, sample_layers, with_scores=with_scores,
                        debug=debug)
    chk.launch()
    torch.cuda.synchronize()
    return chk.verify(threads)


def check_decode(orc, st: W.CacheState, layer, rows=None, lengths=None, scale=None, cache=None,
                 out_offset=0):
    """GPU decode attention for table rows `rows` (all when None) vs the oracle.
    out_offset: elements between a 16-byte boundary and the output (1 puts it
    on a 2-byte boundary only)."""
    wl = st.wl
    dev = st.block_tables.device
    cache = cache or make_cache(st)
    nrows = st.block_tables.shape[0]
    rows = torch.arange(nrows, device=dev, dtype=torch.int32) if rows is None else rows
    lens = st.lengths if lengths is None else lengths
    q = st.decode_q[layer][rows.long()].contiguous()
    buf = torch.full((q.numel() + out_offset,), float("nan"), dtype=q.dtype, device=dev)
    out = buf[out_offset:].view(q.shape)
    scale = 1.0 / math.sqrt(wl.d) if scale is None else scale
    cache.decode(layer, q, st.block_tables, lens, scale, out, req_idx=rows)
    assert cache.status() == zp.OK
    tab = st.block_tables[rows.long()].cpu().numpy()
    ln = lens[rows.long()].cpu().numpy()
    ost, o64, o16 = orc.decode_attn(bits(q), bits(st.k_pools[layer]), bits(st.v_pools[layer]),
                                    tab, ln, scale)
    assert ost == 0
    got = out.float().cpu().numpy().astype(np.float64)
    err = float(np.abs(got - o64).max()) if got.size else 0.0
    assert np.all(np.isfinite(got)), "non-finite decode output"
    assert err <= DECODE_ATOL, f"decode error {err:.3e} > {DECODE_ATOL}"
    print(f"[parity] decode {wl.name} layer {layer}: rows {len(ln)} max abs err {err:.2e}")
    return err
