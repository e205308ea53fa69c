"""GPU parity of compression at admission (zp_compress_prefill) against the
oracle, through the C ABI.

Per unit (request, layer, kv head): scores within 1e-4 of max(|s|, D) (D =
mean |imp| + lambda |red| of the unit); kept sets identical, or differing only
at a near-tie (oracle scores within 1e-5 max(|cut|, D) of the cut between the
kept and the evicted); compacted K/V rows bit-exact copies of the source rows
at the GPU's kept positions.  Tables, lengths, refcounts and the free stack
exact; shared blocks byte-identical; decode attention over the result within
2e-2.
"""
from __future__ import annotations

import concurrent.futures
import math
import os

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SCORE_RTOL = 1e-4
TIE_RTOL = 1e-5
DECODE_ATOL = 2e-2
LAM = 0.5


def bits(t):
    return W.bf16_bits(t)


def ints(c):
    return dict(tables=c["tables"].cpu().numpy().copy(), lengths=c["lengths"].cpu().numpy().copy(),
                refcount=c["refcount"].cpu().numpy().copy(),
                free_ids=c["free_ids"].cpu().numpy().copy(),
                free_count=int(c["free_count"].item()))


def run_prefill(c, req_idx=None, workspace=None, want=True):
    cache = zp.Cache(c["k_pools"], c["v_pools"], c["Hq"], max_requests=c["tables"].shape[0],
                     max_blocks_per_req=c["stride"])
    R = c["window_q"].shape[1]
    L, Hkv, N, b = c["L"], c["Hkv"], c["n_max"], c["b"]
    scores = torch.full((L, R, Hkv, c["stride"] * b), float("nan"), device=DEV) if want else None
    kept = (torch.full((L, R, Hkv, (N - 1) * b), -1, dtype=torch.int32, device=DEV)
            if want else None)
    if workspace is None:
        workspace = torch.empty(cache.prefill_workspace_bytes(R, c["stride"]), dtype=torch.uint8,
                                device=DEV)
    st = cache.compress_prefill(c["tables"], c["lengths"], c["window_q"], N, c["w"], LAM,
                                c["free_ids"], c["free_count"], c["refcount"], workspace,
                                req_idx=req_idx, scores_out=scores, kept_out=kept, check=False)
    return cache, st, cache.status(), scores, kept


def check_unit(orc, T, w, G, b, n_keep, K, V, Q, s_gpu, kept_gpu, Kout, Vout, strict=False):
    C = T - w
    imp, red, s = orc.unit_scores(K, Q, b, w, G, LAM)
    D = float(np.mean(np.abs(imp) + LAM * np.abs(red[:C])))
    sg = s_gpu[:T].astype(np.float64)
    assert np.all(np.isposinf(sg[C:])), "window positions must hold +inf"
    worst = float((np.abs(sg[:C] - s) / np.maximum(np.abs(s), D)).max())
    assert worst <= SCORE_RTOL, f"score error {worst:.3e}"
    kept_o = orc.select(s, w, n_keep)
    kg = kept_gpu.astype(np.int64)
    assert np.all(np.diff(kg) > 0) and np.array_equal(kg[-w:], np.arange(C, T))
    exact = bool(np.array_equal(kg, kept_o))
    assert exact or not strict, f"kept set differs: {np.setxor1d(kg, kept_o).tolist()[:8]}"
    if not exact:
        cut = np.sort(s)[C - n_keep - 1]          # the best evicted score
        diff = np.setxor1d(kg, kept_o)
        tol = TIE_RTOL * max(abs(cut), D)
        assert np.all(np.abs(s[diff] - cut) <= tol), f"kept sets differ: {diff.tolist()[:8]}"
    assert np.array_equal(Kout, K[kg]), "compacted K rows differ"
    assert np.array_equal(Vout, V[kg]), "compacted V rows differ"
    return exact, worst


def gather(pool, table_row, T, h):
    n = -(-T // 16)
    x = pool[table_row[:n].long(), h]              # [n, 16, d]
    return bits(x.reshape(n * 16, -1)[:T])


def check_prefill(orc, c, req_idx=None, sample=None, strict=False):
    """Runs one GPU prefill compression of `c` and checks it (all units, or a
    sample of (layer, request) pairs)."""
    L, Hkv, N, b, w = c["L"], c["Hkv"], c["n_max"], c["b"], c["w"]
    G = c["Hq"] // Hkv
    R = c["window_q"].shape[1]
    rows = list(range(R)) if req_idx is None else list(req_idx)
    before = ints(c)
    pairs = [(l, r) for l in range(L) for r in range(R)] if sample is None else sample
    src = {}
    for l, r in pairs:
        T = int(before["lengths"][rows[r]])
        for h in range(Hkv):
            src[l, r, h] = (gather(c["k_pools"][l], c["tables"][rows[r]], T, h),
                            gather(c["v_pools"][l], c["tables"][rows[r]], T, h))
    shared = torch.nonzero(c["refcount"] > 1).flatten()
    shared_before = [(k[shared].clone(), v[shared].clone())
                     for k, v in zip(c["k_pools"], c["v_pools"])]
    ri = None if req_idx is None else torch.tensor(req_idx, dtype=torch.int32, device=DEV)
    cache, st, dev, scores, kept = run_prefill(c, req_idx=ri)
    assert st == zp.OK and dev == zp.OK, (st, dev)
    after = ints(c)

    # the block accounting of the oracle (independent of the kept sets)
    zero = [np.zeros((before["refcount"].shape[0], Hkv, b, c["d"]), np.uint16)]
    wq0 = np.zeros((1, R, c["Hq"], w, c["d"]), np.uint16)
    o = orc.compress_prefill(zero, zero, before["tables"], before["lengths"], wq0, N, w, LAM,
                             before["free_ids"], before["free_count"], before["refcount"],
                             Hq=c["Hq"], req_idx=req_idx, want_scores=False, want_kept=False)
    assert o["status"] == 0
    for key in ("tables", "lengths", "refcount"):
        assert np.array_equal(after[key], o[key]), key
    assert after["free_count"] == o["free_count"]
    fc = o["free_count"]
    assert np.array_equal(after["free_ids"][:fc], o["free_ids"][:fc]), "free stack"
    for (k0, v0), k, v in zip(shared_before, c["k_pools"], c["v_pools"]):
        assert torch.equal(k[shared], k0) and torch.equal(v[shared], v0), "shared block written"

    sc = scores.cpu().numpy()
    kp = kept.cpu().numpy()
    wq = bits(c["window_q"])
    n_keep = (N - 1) * b - w
    jobs = []
    for l, r in pairs:
        T = int(before["lengths"][rows[r]])
        for h in range(Hkv):
            Kout = gather(c["k_pools"][l], c["tables"][rows[r]], (N - 1) * b, h)
            Vout = gather(c["v_pools"][l], c["tables"][rows[r]], (N - 1) * b, h)
            Q = wq[l, r, h * G:(h + 1) * G].reshape(-1, c["d"])
            jobs.append((T, w, G, b, n_keep, *src[l, r, h], Q, sc[l, r, h], kp[l, r, h], Kout,
                         Vout, strict))
    with concurrent.futures.ThreadPoolExecutor(min(32, os.cpu_count() or 1)) as ex:
        res = [f.result() for f in [ex.submit(check_unit, orc, *j) for j in jobs]]
    exact = sum(e for e, _ in res)
    print(f"[parity] prefill: units {len(res)} exact {exact} near-ties {len(res) - exact} "
          f"max score err {max(wv for _, wv in res):.2e}")
    return cache


@pytest.mark.parametrize("case", [
    dict(lens=[128, 128, 128], n_max=8, d=128, w=8, Hq=8),                    # exactly N*b
    dict(lens=[131, 150, 207, 256, 300, 511], n_max=8, d=128, w=8, Hq=8),     # ragged, 1 chunk
    dict(lens=[600, 1000, 1337, 1500], n_max=8, d=64, w=4, Hq=4, group=2, prefix_blocks=3),
    dict(lens=[129, 140], n_max=8, d=128, w=1, Hq=2),                         # w 1, G 1
    dict(lens=[333, 700], n_max=8, d=128, w=16, Hq=8),                        # 64 window rows
    dict(lens=[2500, 4096, 3001], n_max=128, d=128, w=8, Hq=8),               # budget 2048
    # prompts of the bench's admission workload: several 2048-token chunks
    dict(lens=[7534, 4108], n_max=128, d=128, w=8, Hq=8),
    dict(lens=[8192, 5000, 2049], n_max=128, d=128, w=8, Hq=8, group=3, prefix_blocks=6),
    dict(lens=[8200, 9001], n_max=128, d=128, w=8, Hq=8),                     # 5 chunks
    dict(lens=[3100, 4000], n_max=128, d=128, w=16, Hq=8),                    # 64 rows
    dict(lens=[40, 77, 200], n_max=2, d=128, w=16, Hq=8),                     # keep 0: window only
    # prompts of 8.5 K (d 64) and 17 K tokens
    dict(lens=[8500, 3000], n_max=128, d=64, w=8, Hq=8),
    dict(lens=[17000, 5000], n_max=128, d=128, w=8, Hq=8),
])
def test_prefill_parity(orc, case):
    case = dict(case)
    lens = case.pop("lens")
    n_max = case.pop("n_max")
    c = W.prefill_cache(400 + len(lens) + n_max, lens, n_max, L=2, Hkv=2, device=DEV, **case)
    check_prefill(orc, c)


@pytest.mark.parametrize("keys", ["equal", "zero", "eight_distinct"])
def test_prefill_ties_keep_the_lower_indices(orc, keys):
    """Tie-heavy scores.  Every key equal, or every key zero: all candidates
    tie exactly on both sides, the lower indices are kept, and the kept sets
    must equal the oracle's exactly.  Eight keys repeated block after block:
    a key and its twin in the same block sum the same cosines in a different
    order, so their scores differ by rounding on both sides and only the
    near-tie rule applies."""
    c = W.prefill_cache(471, [1000, 2600, 333], 8, L=1, Hkv=2, device=DEV)
    k = c["k_pools"][0]
    if keys == "equal":
        k.fill_(0.5)
    elif keys == "zero":
        k.zero_()
    else:
        base = k[:1, :, :8].clone()                # 8 key rows per kv head
        k.copy_(base.repeat(1, 1, 2, 1).expand_as(k))
    check_prefill(orc, c, strict=keys != "eight_distinct")


def test_prefill_ignores_slots_past_the_length(orc):
    """NaN bits in the unfilled slots of each prompt's last block (K and V)
    change nothing: those slots are neither keys nor moved rows."""
    lens = [131, 150, 207, 300, 511]
    c = W.prefill_cache(431, lens, 8, L=2, Hkv=2, d=128, w=8, Hq=8, device=DEV)
    for r, T in enumerate(lens):
        if T % 16:
            for l in range(2):
                blk = c["tables"][r, T // 16]
                c["k_pools"][l][blk, :, T % 16:] = float("nan")
                c["v_pools"][l][blk, :, T % 16:] = float("nan")
    check_prefill(orc, c)


def test_prefill_subset_of_rows_then_decode(orc):
    """Only some rows compress (req_idx, in shuffled order); decode attention
    of every row afterwards matches the oracle."""
    lens = [300, 140, 477, 210, 160]
    c = W.prefill_cache(410, lens, 8, L=2, Hkv=2, Hq=8, d=128, w=8, group=2, prefix_blocks=2,
                        device=DEV)
    # rows 1 and 4 stay as they are, but must stay within N_max blocks to decode later
    req = [3, 0, 2]
    c["window_q"] = c["window_q"][:, req].contiguous()
    cache = check_prefill(orc, c, req_idx=req, sample=[(l, r) for l in range(2) for r in range(3)])
    g = torch.Generator(device=DEV)
    g.manual_seed(411)
    q = torch.randn(len(lens), c["Hq"], c["d"], generator=g, device=DEV).to(torch.bfloat16)
    out = torch.empty_like(q)
    scale = 1.0 / math.sqrt(c["d"])
    for l in range(2):
        cache.decode(l, q, c["tables"], c["lengths"], scale, out)
        assert cache.status() == 0
        st, o64, _ = orc.decode_attn(bits(q), bits(c["k_pools"][l]), bits(c["v_pools"][l]),
                                     c["tables"].cpu().numpy(), c["lengths"].cpu().numpy(), scale)
        assert st == 0
        assert float(np.abs(out.float().cpu().numpy() - o64).max()) <= DECODE_ATOL


@pytest.mark.parametrize("what", ["short", "beyond_row", "missing_block", "out_of_blocks"])
def test_prefill_device_errors_change_nothing(orc, what):
    c = W.prefill_cache(420, [200, 150], 8, L=1, Hkv=2, Hq=4, d=64, w=4, group=2,
                        prefix_blocks=2, spare=2, device=DEV)
    if what == "short":
        c["lengths"][1] = 127
    elif what == "beyond_row":
        c["lengths"][0] = c["stride"] * 16 + 1
    elif what == "missing_block":
        c["tables"][0, 5] = -1
    elif what == "out_of_blocks":
        c["free_count"].fill_(1)
    before = ints(c)
    pools = [t.clone() for t in c["k_pools"] + c["v_pools"]]
    _, st, dev, _, _ = run_prefill(c)
    assert st == zp.OK
    assert dev == (zp.ERR_OUT_OF_BLOCKS if what == "out_of_blocks" else zp.ERR_INVALID_ARG), dev
    after = ints(c)
    for k in before:
        assert np.array_equal(np.asarray(after[k]), np.asarray(before[k])), k
    for a, b in zip(c["k_pools"] + c["v_pools"], pools):
        assert torch.equal(a, b)


def test_prefill_host_checks():
    """A workspace smaller than the size query is refused before any launch."""
    c = W.prefill_cache(430, [200], 8, L=1, Hkv=2, Hq=4, d=64, w=4, device=DEV)
    cache = zp.Cache(c["k_pools"], c["v_pools"], c["Hq"], max_requests=1,
                     max_blocks_per_req=c["stride"])
    need = cache.prefill_workspace_bytes(1, c["stride"])
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    st = cache.compress_prefill(c["tables"], c["lengths"], c["window_q"], 8, 4, LAM, c["free_ids"],
                                c["free_count"], c["refcount"], small, check=False)
    assert st == zp.ERR_INVALID_ARG
