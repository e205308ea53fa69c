"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` function takes a loaded oracle (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with a closed form, a brute-force
enumeration, an independent library routine (torch fp64), a hand-worked
value, or an invariant the pages state.  ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle
with one planted mistake each and requires that some pin fails.

Sources: "Zipage: Maintain High Request Concurrency for LLM Reasoning through
Compressed PagedAttention" (gist.science summaries: Dutch "Methodologie" §1,
§3, §5; Korean "방법론" A, C, E) and "Paged KV cache and continuous batching
for LLMs" ("How it works").
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch

from compressed_paged_kv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers

def bf16(x) -> np.ndarray:
    """uint16 bf16 bit patterns of float data (rounded by torch)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def widen(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rng(seed):
    return np.random.default_rng(seed)


def close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


def torch_importance(K, Q, w, G):
    """Observation-window importance with torch's fp64 softmax (independent)."""
    Kd = torch.tensor(widen(K))
    Qd = torch.tensor(widen(Q))
    T, d = Kd.shape
    C = T - w
    logits = (Qd @ Kd.T) / math.sqrt(d)            # [G*w, T]
    rows = torch.arange(G * w) % w                  # window slot of each row
    mask = torch.arange(T)[None, :] > (C + rows)[:, None]
    logits = logits.masked_fill(mask, float("-inf"))
    P = torch.softmax(logits, dim=-1)
    return P[:, :C].mean(dim=0).numpy()


def torch_redundancy(K, b):
    Kd = torch.tensor(widen(K))
    T, d = Kd.shape
    out = np.zeros(T)
    for base in range(0, T, b):
        blk = Kd[base:base + b]
        cos = torch.nn.functional.cosine_similarity(blk[:, None, :], blk[None, :, :], dim=-1,
                                                    eps=1e-300)
        norms = blk.norm(dim=-1)
        zero = norms == 0
        cos[zero, :] = 0.0
        cos[:, zero] = 0.0
        cos.fill_diagonal_(0.0)
        f = blk.shape[0]                            # filled slots (a partial last block)
        out[base:base + f] = (cos.sum(dim=1) / (f - 1)).numpy() if f > 1 else 0.0
    return out


# --------------------------------------------------------------- importance

def pin_importance_uniform_zero_queries(orc):
    """q = 0: every visible logit is 0, so window row i spreads 1/(C+i+1) over
    keys 0..C+i and imp_j = (1/w) sum_i 1/(C+i+1) for every candidate."""
    T, d, w, G = 48, 16, 4, 2
    C = T - w
    K = bf16(rng(1).standard_normal((T, d)))
    Q = np.zeros((G * w, d), dtype=np.uint16)
    imp = orc.importance(K, Q, w, G)
    expect = sum(1.0 / (C + i + 1) for i in range(w)) / w
    close(imp, np.full(C, expect), 1e-15, "importance with q = 0")


def pin_importance_equal_keys(orc):
    """All keys equal: logits are equal on each row; same closed form."""
    T, d, w, G = 40, 8, 5, 3
    C = T - w
    row = rng(2).standard_normal(d)
    K = bf16(np.tile(row, (T, 1)))
    Q = bf16(rng(3).standard_normal((G * w, d)))
    imp = orc.importance(K, Q, w, G)
    expect = sum(1.0 / (C + i + 1) for i in range(w)) / w
    close(imp, np.full(C, expect), 1e-14, "importance with equal keys")


def pin_importance_dominant_key(orc):
    """One key aligned with every query and 8x longer: its logit exceeds the
    others by ~32, so it takes all of the probability mass (imp -> 1)."""
    T, d, w, G = 64, 16, 4, 2
    u = np.where(rng(4).standard_normal(d) > 0, 1.0, -1.0)
    K = 0.01 * rng(5).standard_normal((T, d))
    jstar = 17
    K[jstar] = 8.0 * u
    Q = np.tile(u, (G * w, 1))
    imp = orc.importance(bf16(K), bf16(Q), w, G)
    assert abs(imp[jstar] - 1.0) < 1e-11, imp[jstar]
    others = np.delete(imp, jstar)
    assert np.all(others < 1e-12) and np.all(others >= 0.0)


def pin_importance_torch_softmax(orc):
    """Random keys and queries against torch's fp64 softmax with the causal
    window mask (query i of the window sees keys up to C+i)."""
    for seed, (T, d, w, G) in enumerate([(64, 16, 8, 4), (48, 32, 5, 1), (33, 8, 3, 2)]):
        K = bf16(2.0 * rng(10 + seed).standard_normal((T, d)))
        Q = bf16(2.0 * rng(20 + seed).standard_normal((G * w, d)))
        close(orc.importance(K, Q, w, G), torch_importance(K, Q, w, G), 1e-13,
              f"importance vs torch softmax {T, d, w, G}")


# --------------------------------------------------------------- redundancy

def pin_redundancy_identical_keys(orc):
    b, d = 8, 16
    K = bf16(np.tile(rng(6).standard_normal(d), (3 * b, 1)))
    close(orc.redundancy(K, b), np.ones(3 * b), 1e-14, "redundancy of identical keys")


def pin_redundancy_orthogonal_keys(orc):
    b, d = 8, 16
    K = np.zeros((b, d))
    for j in range(b):
        K[j, (3 * j) % d] = 1.0 + j
    close(orc.redundancy(bf16(K), b), np.zeros(b), 1e-15, "redundancy of orthogonal keys")


def pin_redundancy_opposite_halves(orc):
    """b/2 copies of u and b/2 of -u: each key has b/2-1 cosines of +1 and
    b/2 of -1, so red = -1/(b-1)."""
    b, d = 16, 8
    u = rng(7).standard_normal(d)
    K = np.vstack([np.tile(u, (b // 2, 1)), np.tile(-u, (b // 2, 1))])
    close(orc.redundancy(bf16(K), b), np.full(b, -1.0 / (b - 1)), 1e-14,
          "redundancy of opposite halves")


def pin_redundancy_zero_key(orc):
    """A zero key has cosine 0 with everything: its own red is 0, and each
    other (identical) key sees b-2 cosines of 1, so red = (b-2)/(b-1)."""
    b, d = 8, 4
    K = np.tile(rng(8).standard_normal(d), (b, 1))
    K[3] = 0.0
    red = orc.redundancy(bf16(K), b)
    expect = np.full(b, (b - 2) / (b - 1))
    expect[3] = 0.0
    close(red, expect, 1e-14, "redundancy with a zero key")


def pin_redundancy_handworked(orc):
    with open(os.path.join(GOLDEN, "lrs_handworked.json")) as f:
        g = json.load(f)
    red = orc.redundancy(bf16(np.array(g["keys"], dtype=np.float64)), g["b"])
    close(red, g["red"], 1e-14, "hand-worked redundancy")


def pin_redundancy_torch_cosine(orc):
    for seed, (T, b, d) in enumerate([(64, 16, 32), (48, 4, 8), (30, 6, 5)]):
        K = bf16(rng(30 + seed).standard_normal((T, d)))
        close(orc.redundancy(K, b), torch_redundancy(K, b), 1e-13,
              f"redundancy vs torch cosine {T, b, d}")


def pin_redundancy_block_locality(orc):
    """Only keys of the same block are compared: changing block 1 leaves the
    values of block 0 unchanged."""
    b, d = 8, 8
    K = rng(40).standard_normal((3 * b, d))
    r0 = orc.redundancy(bf16(K), b)
    K2 = K.copy()
    K2[b:2 * b] = rng(41).standard_normal((b, d))
    r1 = orc.redundancy(bf16(K2), b)
    close(r0[:b], r1[:b], 0.0, "block 0 redundancy after changing block 1")
    close(r0[2 * b:], r1[2 * b:], 0.0, "block 2 redundancy after changing block 1")


# -------------------------------------------------------------------- score

def pin_redundancy_global_one_block_is_lrs(orc):
    """With a single block (T = b) the global redundancy is the Lightning
    Redundancy Score; partial blocks too (T < b)."""
    g = rng(160)
    for T in (16, 9):
        K = bf16(g.standard_normal((T, 8)))
        close(orc.redundancy_global(K), orc.redundancy(K, 16), 1e-12, "one block")


def pin_redundancy_global_closed_forms(orc):
    """Identical keys: 1; mutually orthogonal keys: 0; m copies of u and m of
    -u: (m - 1 - m)/(2m - 1) = -1/(2m - 1); a zero key: 0 for it, and it
    counts as a cosine of 0 for the others."""
    u = np.ones(4)
    close(orc.redundancy_global(bf16(np.tile(u, (7, 1)))), np.ones(7), 1e-12, "identical")
    close(orc.redundancy_global(bf16(np.eye(6))), np.zeros(6), 1e-12, "orthogonal")
    m = 3
    K = bf16(np.vstack([np.tile(u, (m, 1)), np.tile(-u, (m, 1))]))
    close(orc.redundancy_global(K), np.full(2 * m, -1.0 / (2 * m - 1)), 1e-12, "+-u")
    K = bf16(np.vstack([np.tile(u, (3, 1)), np.zeros((1, 4))]))
    close(orc.redundancy_global(K), [2 / 3, 2 / 3, 2 / 3, 0.0], 1e-12, "zero key")


def pin_redundancy_global_torch(orc):
    """Against torch fp64: the mean of each row of the cosine-similarity
    matrix without its diagonal."""
    K = bf16(rng(161).standard_normal((70, 16)))
    Kd = torch.tensor(widen(K))
    cos = torch.nn.functional.cosine_similarity(Kd[:, None, :], Kd[None, :, :], dim=-1)
    cos.fill_diagonal_(0.0)
    close(orc.redundancy_global(K), (cos.sum(dim=1) / 69).numpy(), 1e-12, "torch")


def pin_score_lambda_zero_is_importance(orc):
    T, d, b, w, G = 64, 16, 8, 4, 2
    K = bf16(rng(50).standard_normal((T, d)))
    Q = bf16(rng(51).standard_normal((G * w, d)))
    imp, red, score = orc.unit_scores(K, Q, b, w, G, 0.0)
    close(score, torch_importance(K, Q, w, G), 1e-13, "score at lambda 0")


def pin_score_large_lambda_evicts_most_redundant(orc):
    """As lambda grows the importance term becomes negligible: the b evicted
    candidates are the b most redundant ones."""
    N, b, d, w, G = 6, 4, 8, 2, 2
    T = N * b
    K = bf16(rng(52).standard_normal((T, d)))
    Q = bf16(rng(53).standard_normal((G * w, d)))
    _, red, score = orc.unit_scores(K, Q, b, w, G, 1e6)
    C = T - w
    kept = orc.select(score, w, C - b)
    evicted = sorted(set(range(C)) - set(kept.tolist()))
    most = sorted(np.argsort(-red[:C], kind="stable")[:b].tolist())
    assert evicted == most, (evicted, most)
    close(score, torch_importance(K, Q, w, G) - 1e6 * torch_redundancy(K, b)[:C], 1e-7,
          "score at lambda 1e6")


def pin_score_mixture(orc):
    """score = imp - lambda * red against the torch versions of both terms."""
    T, d, b, w, G = 96, 16, 16, 8, 4
    K = bf16(rng(54).standard_normal((T, d)))
    Q = bf16(rng(55).standard_normal((G * w, d)))
    _, _, score = orc.unit_scores(K, Q, b, w, G, 0.5)
    C = T - w
    close(score, torch_importance(K, Q, w, G) - 0.5 * torch_redundancy(K, b)[:C], 1e-13,
          "score vs torch terms")


# ------------------------------------------------------------------- select

def _brute_force_keep(score, n_keep):
    """Among all size-n_keep subsets, the ones with the largest total score;
    of those the lexicographically smallest sorted index tuple."""
    best = None
    for sub in itertools.combinations(range(len(score)), n_keep):
        s = sum(score[i] for i in sub)
        key = (-s, sub)
        if best is None or key < best:
            best = key
    return list(best[1])


def pin_select_brute_force(orc):
    """Integer scores with deliberate ties, every subset enumerated."""
    b, w = 4, 3
    for seed, C in enumerate([12, 16, 20]):
        score = rng(60 + seed).integers(0, 5, size=C).astype(np.float64)
        kept = orc.select(score, w, C - b)
        assert kept[:C - b].tolist() == _brute_force_keep(score.tolist(), C - b), seed
        assert kept[C - b:].tolist() == list(range(C, C + w))


def pin_select_all_equal(orc):
    """All scores equal: the higher indices lose the tie, so the b highest
    candidates are evicted."""
    C, b, w = 40, 8, 4
    kept = orc.select(np.zeros(C), w, C - b)
    assert kept.tolist() == list(range(C - b)) + list(range(C, C + w))


def pin_select_invariants(orc):
    """Window kept, exactly (N-1)*b entries, strictly increasing."""
    N, b, w = 8, 16, 8
    C = N * b - w
    score = rng(61).standard_normal(C)
    kept = orc.select(score, w, (N - 1) * b - w)
    assert kept.size == (N - 1) * b
    assert np.all(np.diff(kept) > 0)
    assert kept[-w:].tolist() == list(range(C, C + w))
    evicted = sorted(set(range(C)) - set(kept.tolist()))
    assert evicted == sorted(np.argsort(score)[:b].tolist())


# ------------------------------------------------------------ block accounting

def _state(tables, refcount, free_ids, N, b):
    tables = np.asarray(tables, dtype=np.int32)
    R = tables.shape[0]
    return dict(tables=tables.copy(), lengths=np.full(R, N * b, dtype=np.int32),
                refcount=np.asarray(refcount, dtype=np.int32).copy(),
                free_ids=np.asarray(free_ids, dtype=np.int32).copy())


def _apply(orc, s, free_count, N, b, num_blocks, req_idx=None):
    st, dst, pops = orc.plan(s["tables"], s["lengths"], s["refcount"], s["free_ids"],
                             free_count, N, b, num_blocks, req_idx=req_idx)
    if st != 0:
        return st, free_count, dst
    fc = orc.commit(s["tables"], s["lengths"], s["refcount"], s["free_ids"], free_count, dst,
                    pops, N, b, req_idx=req_idx)
    return st, fc, dst


def pin_blocks_no_sharing(orc):
    N, b = 4, 4
    tables = [[0, 1, 2, 3], [4, 5, 6, 7]]
    rc = [1] * 8 + [0] * 4
    free = [8, 9, 10, 11]
    s = _state(tables, rc, free, N, b)
    st, fc, dst = _apply(orc, s, 4, N, b, 12)
    assert st == 0 and fc == 4
    assert s["tables"].tolist() == tables and s["refcount"].tolist() == rc
    assert s["lengths"].tolist() == [(N - 1) * b] * 2


def pin_blocks_shared_prefix(orc):
    """Block 0 shared by both requests (refcount 2): both compress into fresh
    targets popped from the top of the stack (request 0 first); block 0 drops
    to refcount 0 on its last holder and is pushed after the pops."""
    N, b = 3, 4
    tables = [[0, 1, 2], [0, 3, 4]]
    rc = [2, 1, 1, 1, 1, 0, 0, 0]
    free = [5, 6, 7, -1, -1, -1, -1, -1]
    s = _state(tables, rc, free, N, b)
    st, fc, dst = _apply(orc, s, 3, N, b, 8)
    assert st == 0
    assert dst.tolist() == [[7, 1, 2], [6, 3, 4]]
    assert s["tables"].tolist() == [[7, 1, 2], [6, 3, 4]]
    assert s["refcount"].tolist() == [0, 1, 1, 1, 1, 0, 1, 1]
    assert fc == 2 and s["free_ids"][:fc].tolist() == [5, 0]


def pin_blocks_partial_holders(orc):
    """Refcount 3 with only two compressing holders: the block keeps one
    reference and is not freed; a shared reserved block is replaced too."""
    N, b = 2, 4
    tables = [[0, 9], [0, 9], [0, 2]]
    rc = [3, 0, 1, 0, 0, 0, 0, 0, 0, 2]
    free = [1, 3, 4, 5, 6, 7, 8, -1, -1, -1]
    s = _state(tables, rc, free, N, b)
    st, fc, dst = _apply(orc, s, 7, N, b, 10, req_idx=np.array([0, 1], dtype=np.int32))
    assert st == 0
    assert dst.tolist() == [[8, 7], [6, 5]]
    assert s["tables"].tolist() == [[8, 7], [6, 5], [0, 2]]
    assert s["refcount"][0] == 1 and s["refcount"][9] == 0
    assert fc == 7 - 4 + 1 and s["free_ids"][:fc].tolist() == [1, 3, 4, 9]


def pin_blocks_conservation(orc):
    """On a random valid cache: free + blocks in use = capacity, the sum of
    refcounts equals the number of table references, targets are unique per
    request, and shared-at-start blocks are never destinations."""
    g = rng(70)
    N, b, R, group, pb = 6, 4, 12, 3, 2
    num_blocks = 200
    perm = g.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((R, N), dtype=np.int32)
    rc = np.zeros(num_blocks, dtype=np.int32)
    nxt = 0
    for gi in range(R // group):
        shared = perm[nxt:nxt + pb]
        nxt += pb
        for r in range(gi * group, (gi + 1) * group):
            tables[r, :pb] = shared
            tables[r, pb:] = perm[nxt:nxt + N - pb]
            nxt += N - pb
    for x in tables.reshape(-1):
        rc[x] += 1
    free = np.full(num_blocks, -1, dtype=np.int32)
    nfree = num_blocks - nxt
    free[:nfree] = perm[nxt:]
    shared_at_start = set(np.nonzero(rc > 1)[0].tolist())
    req = np.array([0, 1, 2, 4, 7, 9, 10], dtype=np.int32)
    s = _state(tables, rc, free, N, b)
    st, fc, dst = _apply(orc, s, nfree, N, b, num_blocks, req_idx=req)
    assert st == 0
    assert fc + int(np.count_nonzero(s["refcount"] >= 1)) == num_blocks
    assert int(s["refcount"].sum()) == s["tables"].size
    for r in range(dst.shape[0]):
        assert len(set(dst[r].tolist())) == N
        assert not (set(dst[r].tolist()) & shared_at_start)
    assert len(set(s["free_ids"][:fc].tolist())) == fc
    assert np.all(s["refcount"][s["free_ids"][:fc]] == 0)


def pin_blocks_out_of_blocks(orc):
    """Too few free blocks: status 'out of blocks' and nothing modified."""
    N, b = 2, 4
    tables = [[0, 1], [0, 2]]
    rc = [2, 1, 1, 0]
    free = [3, -1, -1, -1]
    s = _state(tables, rc, free, N, b)
    before = {k: v.copy() for k, v in s.items()}
    st, fc, _ = _apply(orc, s, 1, N, b, 4)
    assert st == -3 and fc == 1
    for k in s:
        assert np.array_equal(s[k], before[k]), k


def pin_blocks_invalid(orc):
    """A length other than N*b (the trigger needs a full last block) or a
    block id out of range is rejected."""
    N, b = 2, 4
    s = _state([[0, 1]], [1, 1, 0], [2, -1, -1], N, b)
    s["lengths"][0] = N * b - 1
    assert _apply(orc, s, 1, N, b, 3)[0] == -1
    s = _state([[0, 5]], [1, 1, 0], [2, -1, -1], N, b)
    assert _apply(orc, s, 1, N, b, 3)[0] == -1


# ------------------------------------------------------------ whole compress

def _tiny_cache(seed, N=6, b=4, d=8, Hkv=2, G=2, L=2, R=3, share=True, w=3):
    """A tiny random cache: request 0 and 1 share their first block."""
    g = rng(seed)
    num_blocks = R * N + 8
    perm = g.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((R, N), dtype=np.int32)
    nxt = 0
    for r in range(R):
        tables[r] = perm[nxt:nxt + N]
        nxt += N
    if share:
        tables[1, 0] = tables[0, 0]
        nxt_free = perm[nxt:]
        nxt_free = np.concatenate([nxt_free, [perm[N]]])  # request 1's old block 0 is free
    else:
        nxt_free = perm[nxt:]
    rc = np.zeros(num_blocks, dtype=np.int32)
    for x in tables.reshape(-1):
        rc[x] += 1
    free = np.full(num_blocks, -1, dtype=np.int32)
    free[:len(nxt_free)] = nxt_free
    kp = [bf16(g.standard_normal((num_blocks, Hkv, b, d))) for _ in range(L)]
    vp = [bf16(g.standard_normal((num_blocks, Hkv, b, d))) for _ in range(L)]
    wq = bf16(g.standard_normal((L, R, Hkv * G, w, d)))
    return dict(kp=kp, vp=vp, tables=tables, lengths=np.full(R, N * b, dtype=np.int32),
                rc=rc, free=free, free_count=len(nxt_free), wq=wq, N=N, b=b, d=d, Hkv=Hkv,
                G=G, L=L, R=R, w=w)


def _gather(pool, row, h, b):
    return np.concatenate([pool[blk, h] for blk in row], axis=0)


def pin_compress_rows_and_shared_blocks(orc):
    """Every compacted row byte-equals the input row at its kept index; the
    shared block is byte-identical afterwards; (N-1)*b rows per head; the
    kept indices match a fresh select on the oracle's own scores."""
    c = _tiny_cache(80)
    N, b, w, L, R, Hkv = c["N"], c["b"], c["w"], c["L"], c["R"], c["Hkv"]
    res = orc.compress(c["kp"], c["vp"], c["tables"], c["lengths"], c["wq"], N, w, 0.5,
                       c["free"], c["free_count"], c["rc"], Hq=Hkv * c["G"])
    assert res["status"] == 0
    shared = c["tables"][0, 0]
    for l in range(L):
        assert np.array_equal(res["kpools"][l][shared], c["kp"][l][shared])
        assert np.array_equal(res["vpools"][l][shared], c["vp"][l][shared])
        for r in range(R):
            for h in range(Hkv):
                kept = res["kept"][l, r, h]
                assert kept.size == (N - 1) * b and np.all(np.diff(kept) > 0)
                src_k = _gather(c["kp"][l], c["tables"][r], h, b)
                src_v = _gather(c["vp"][l], c["tables"][r], h, b)
                new_row = res["tables"][r, :N - 1]
                got_k = _gather(res["kpools"][l], new_row, h, b)
                got_v = _gather(res["vpools"][l], new_row, h, b)
                assert np.array_equal(got_k, src_k[kept])
                assert np.array_equal(got_v, src_v[kept])
                C = N * b - w
                K = src_k
                Q = c["wq"][l, r, h * c["G"]:(h + 1) * c["G"]].reshape(-1, c["d"])
                _, _, score = orc.unit_scores(K, Q, b, w, c["G"], 0.5)
                close(res["scores"][l, r, h, :C], score, 0.0, "scores_out")
                assert kept.tolist() == orc.select(score, w, (N - 1) * b - w).tolist()
    assert res["lengths"].tolist() == [(N - 1) * b] * R
    assert res["tables"][0, 0] != shared and res["tables"][1, 0] != shared
    assert res["refcount"][shared] == 0


# ------------------------------------------------------------------ prefill

def _prefill_cache(seed, lens, N=3, b=4, d=8, Hkv=2, G=2, L=2, w=2, share=0, spare=12):
    """Requests of the given lengths in random blocks (entries beyond a
    request's blocks -1); requests 0 and 1 share their first `share` blocks."""
    g = rng(seed)
    R = len(lens)
    nblk = [-(-T // b) for T in lens]
    stride = max(nblk)
    num_blocks = sum(nblk) + spare
    perm = g.permutation(num_blocks).astype(np.int32)
    tables = np.full((R, stride), -1, dtype=np.int32)
    nxt = 0
    for r, n in enumerate(nblk):
        s0 = share if r == 1 else 0
        tables[r, :s0] = tables[0, :s0]
        tables[r, s0:n] = perm[nxt:nxt + n - s0]
        nxt += n - s0
    rc = np.zeros(num_blocks, dtype=np.int32)
    for x in tables.reshape(-1):
        if x >= 0:
            rc[x] += 1
    free = np.full(num_blocks, -1, dtype=np.int32)
    free[:num_blocks - nxt] = perm[nxt:]
    kp = [bf16(g.standard_normal((num_blocks, Hkv, b, d))) for _ in range(L)]
    vp = [bf16(g.standard_normal((num_blocks, Hkv, b, d))) for _ in range(L)]
    wq = bf16(g.standard_normal((L, R, Hkv * G, w, d)))
    return dict(kp=kp, vp=vp, tables=tables, lengths=np.array(lens, dtype=np.int32), rc=rc,
                free=free, free_count=num_blocks - nxt, wq=wq, N=N, b=b, d=d, Hkv=Hkv, G=G, L=L,
                R=R, w=w, num_blocks=num_blocks)


def _run_prefill(orc, c, lam=0.5, **kw):
    return orc.compress_prefill(c["kp"], c["vp"], c["tables"], c["lengths"], c["wq"], c["N"],
                                c["w"], lam, c["free"], c["free_count"], c["rc"],
                                Hq=c["Hkv"] * c["G"], **kw)


def pin_prefill_handworked_release(orc):
    """The hand-worked release of tests/golden/prefill_release_handworked.json."""
    with open(os.path.join(GOLDEN, "prefill_release_handworked.json")) as f:
        gd = json.load(f)
    b, N, w, nb = gd["b"], gd["N"], gd["w"], gd["num_blocks"]
    g = rng(150)
    kp = [bf16(g.standard_normal((nb, 1, b, 4)))]
    vp = [bf16(g.standard_normal((nb, 1, b, 4)))]
    wq = bf16(g.standard_normal((1, 2, 1, w, 4)))
    res = orc.compress_prefill(kp, vp, gd["tables"], gd["lengths"], wq, N, w, 0.5,
                               gd["free_ids"], gd["free_count"], gd["refcount"], Hq=1)
    assert res["status"] == 0
    ex = gd["expect"]
    assert res["tables"].tolist() == ex["tables"]
    assert res["lengths"].tolist() == ex["lengths"]
    assert res["refcount"].tolist() == ex["refcount"]
    assert res["free_count"] == len(ex["free_ids"])
    assert res["free_ids"][:res["free_count"]].tolist() == ex["free_ids"]


def pin_prefill_at_budget_equals_compress(orc):
    """Requests of exactly N*b tokens: compression at admission is the
    decode-time compression, byte for byte."""
    c = _tiny_cache(151)
    N, b, w = c["N"], c["b"], c["w"]
    a = orc.compress(c["kp"], c["vp"], c["tables"], c["lengths"], c["wq"], N, w, 0.5, c["free"],
                     c["free_count"], c["rc"], Hq=c["Hkv"] * c["G"])
    p = orc.compress_prefill(c["kp"], c["vp"], c["tables"], c["lengths"], c["wq"], N, w, 0.5,
                             c["free"], c["free_count"], c["rc"], Hq=c["Hkv"] * c["G"])
    assert a["status"] == p["status"] == 0
    for k in ("tables", "lengths", "refcount", "free_ids", "kept"):
        assert np.array_equal(a[k], p[k]), k
    assert a["free_count"] == p["free_count"]
    assert np.array_equal(a["scores"], p["scores"][..., :N * b])
    for l in range(c["L"]):
        assert np.array_equal(a["kpools"][l], p["kpools"][l])
        assert np.array_equal(a["vpools"][l], p["vpools"][l])


def pin_prefill_partial_block_redundancy(orc):
    """A partial last block compares only its filled keys: two keys (1,0) and
    (1,1) have redundancy cos = 1/sqrt2 each, a single key 0."""
    K = bf16([[1, 0], [0, 1], [1, 1], [-1, 0], [1, 0], [1, 1]])
    red = orc.redundancy(K, 4)
    close(red[4:], [2 ** -0.5] * 2, 1e-12, "two-key block")
    red5 = orc.redundancy(K[:5], 4)
    close(red5[4:], [0.0], 0.0, "one-key block")
    close(red5[:4], red[:4], 0.0, "full block unchanged")


def pin_prefill_rows_scores_and_release(orc):
    """Ragged requests longer than the budget, two sharing a prefix: the
    scores equal torch's fp64 importance and cosine redundancy over each
    request's own T tokens, the kept set is the top of a library sort by
    (score desc, index asc) plus the window, every compacted row equals its
    source row, shared blocks keep their bytes, every excess block loses one
    reference, and blocks are conserved."""
    lens = [23, 17, 12, 30]
    c = _prefill_cache(152, lens, N=3, b=4, d=8, w=2, share=2)
    N, b, w, G, d = c["N"], c["b"], c["w"], c["G"], c["d"]
    res = _run_prefill(orc, c)
    assert res["status"] == 0
    n_keep = (N - 1) * b - w
    for l in range(c["L"]):
        for r, T in enumerate(lens):
            C = T - w
            n = -(-T // b)
            for h in range(c["Hkv"]):
                K = _gather(c["kp"][l], c["tables"][r, :n], h, b)[:T]
                V = _gather(c["vp"][l], c["tables"][r, :n], h, b)[:T]
                Q = c["wq"][l, r, h * G:(h + 1) * G].reshape(-1, d)
                score = torch_importance(K, Q, w, G) - 0.5 * torch_redundancy(K, b)[:C]
                close(res["scores"][l, r, h, :C], score, 1e-12, "prefill scores")
                assert np.all(np.isinf(res["scores"][l, r, h, C:T]))
                order = np.lexsort((np.arange(C), -res["scores"][l, r, h, :C]))
                want = sorted(order[:n_keep].tolist()) + list(range(C, T))
                kept = res["kept"][l, r, h]
                assert kept.tolist() == want
                new_row = res["tables"][r, :N - 1]
                assert np.array_equal(_gather(res["kpools"][l], new_row, h, b), K[kept])
                assert np.array_equal(_gather(res["vpools"][l], new_row, h, b), V[kept])
    shared = c["tables"][0, :2]
    for l in range(c["L"]):
        assert np.array_equal(res["kpools"][l][shared], c["kp"][l][shared])
    assert res["lengths"].tolist() == [(N - 1) * b] * len(lens)
    assert np.all(res["tables"][:, N:] == -1)
    ref = np.zeros_like(res["refcount"])
    for x in res["tables"].reshape(-1):
        if x >= 0:
            ref[x] += 1
    assert np.array_equal(ref, res["refcount"])
    fc = res["free_count"]
    assert fc + int(np.count_nonzero(res["refcount"])) == c["num_blocks"]
    assert np.all(res["refcount"][res["free_ids"][:fc]] == 0)
    assert len(set(res["free_ids"][:fc].tolist())) == fc


def pin_prefill_attention_masked(orc):
    """Attention over the cache compressed at admission equals attention over
    the original rows restricted to the kept indices."""
    lens = [29, 18]
    c = _prefill_cache(153, lens, N=3, b=4, d=8, L=1, w=2)
    res = _run_prefill(orc, c)
    assert res["status"] == 0
    q = bf16(rng(154).standard_normal((2, c["Hkv"] * c["G"], c["d"])))
    scale = 1.0 / math.sqrt(c["d"])
    st, o64, _ = orc.decode_attn(q, res["kpools"][0], res["vpools"][0], res["tables"],
                                 res["lengths"], scale)
    assert st == 0
    for r, T in enumerate(lens):
        n = -(-T // c["b"])
        for hq in range(c["Hkv"] * c["G"]):
            h = hq // c["G"]
            K = torch.tensor(widen(_gather(c["kp"][0], c["tables"][r, :n], h, c["b"])[:T]))
            V = torch.tensor(widen(_gather(c["vp"][0], c["tables"][r, :n], h, c["b"])[:T]))
            mask = torch.zeros(T, dtype=torch.bool)
            mask[torch.tensor(res["kept"][0, r, h], dtype=torch.long)] = True
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(widen(q[r, hq]))[None, None, :], K[None], V[None],
                attn_mask=mask[None, None, :], scale=scale)[0, 0]
            close(o64[r, hq], o.numpy(), 1e-12, "prefill compacted vs masked")


def pin_prefill_errors(orc):
    """All or nothing: a request shorter than N*b, longer than its table row,
    with a missing block, or too few free blocks changes nothing."""
    base = _prefill_cache(155, [20, 14], N=3, b=4, d=4, L=1, w=2, share=2, spare=2)

    def run(**ch):
        c = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in base.items()}
        c.update(ch)
        res = _run_prefill(orc, c)
        if res["status"] != 0:
            assert np.array_equal(res["tables"], c["tables"])
            assert np.array_equal(res["lengths"], c["lengths"])
            assert np.array_equal(res["refcount"], c["rc"])
            assert res["free_count"] == c["free_count"]
        return res["status"]

    assert run() == 0
    assert run(lengths=np.array([20, 11], dtype=np.int32)) == -1
    assert run(lengths=np.array([21, 14], dtype=np.int32)) == -1
    t = base["tables"].copy()
    t[0, 3] = -1
    assert run(tables=t) == -1
    assert run(free_count=1) == -3


# ------------------------------------------------------------------- decode

def torch_decode(q, kpool, vpool, tables, lengths, scale):
    """Dense gather + torch fp64 scaled_dot_product_attention."""
    qd = torch.tensor(widen(q))
    R, Hq, d = qd.shape
    Hkv, b = kpool.shape[1], kpool.shape[2]
    G = Hq // Hkv
    out = torch.zeros(R, Hq, d, dtype=torch.float64)
    for r in range(R):
        n = int(lengths[r])
        if n == 0:
            continue
        blocks = tables[r, :(n + b - 1) // b]
        K = torch.tensor(widen(np.concatenate([kpool[x] for x in blocks], axis=1)))[:, :n]
        V = torch.tensor(widen(np.concatenate([vpool[x] for x in blocks], axis=1)))[:, :n]
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qd[r][:, None, :], K, V, scale=scale)
        out[r] = o[:, 0, :]
    return out.numpy()


def _decode_case(seed, R=3, Hkv=2, G=3, d=16, b=4, nb=6, num_blocks=30):
    g = rng(seed)
    kpool = bf16(g.standard_normal((num_blocks, Hkv, b, d)))
    vpool = bf16(g.standard_normal((num_blocks, Hkv, b, d)))
    tables = np.stack([g.permutation(num_blocks)[:nb] for _ in range(R)]).astype(np.int32)
    q = bf16(g.standard_normal((R, Hkv * G, d)))
    return q, kpool, vpool, tables


def pin_decode_torch_sdpa(orc):
    q, kp, vp, tables = _decode_case(90)
    lengths = np.array([24, 13, 1], dtype=np.int32)
    scale = 1.0 / math.sqrt(q.shape[-1])
    st, o64, o16 = orc.decode_attn(q, kp, vp, tables, lengths, scale)
    assert st == 0
    close(o64, torch_decode(q, kp, vp, tables, lengths, scale), 1e-13, "decode vs torch sdpa")
    close(widen(o16), torch.tensor(o64).to(torch.bfloat16).to(torch.float64).numpy(), 0.0,
          "bf16 rounding of the decode output")


def pin_decode_closed_forms(orc):
    """All keys equal -> uniform weights -> the mean of the V rows; a zero
    length gives zeros."""
    q, kp, vp, tables = _decode_case(91, R=2)
    kp = np.broadcast_to(kp[:1, :, :1, :], kp.shape).copy()
    lengths = np.array([10, 0], dtype=np.int32)
    st, o64, _ = orc.decode_attn(q, kp, vp, tables, lengths, 0.25)
    assert st == 0
    b = kp.shape[2]
    Hkv = kp.shape[1]
    G = q.shape[1] // Hkv
    V = widen(np.concatenate([vp[x] for x in tables[0, :3]], axis=1))[:, :10]
    expect = np.repeat(V.mean(axis=1), G, axis=0)
    close(o64[0], expect, 1e-14, "decode with equal keys")
    close(o64[1], np.zeros_like(o64[1]), 0.0, "decode with zero length")


def pin_decode_dominant_key(orc):
    """One key aligned with the query and much longer: its V row comes out."""
    q, kp, vp, tables = _decode_case(92, R=1, Hkv=1, G=1, d=16)
    qv = np.where(widen(q)[0, 0] > 0, 1.0, -1.0)
    q = bf16(qv[None, None, :])
    kf = 0.01 * widen(kp)
    blk, slot = tables[0, 2], 1
    kf[blk, 0, slot] = 8.0 * qv
    kp = bf16(kf)
    st, o64, _ = orc.decode_attn(q, kp, vp, tables, np.array([20], dtype=np.int32), 1.0)
    assert st == 0
    close(o64[0, 0], widen(vp[blk, 0, slot]), 1e-30, "decode dominant key")


def pin_decode_compacted_equals_masked(orc):
    """Attention over the compacted cache equals full attention over the
    original cache restricted to the kept indices."""
    c = _tiny_cache(93, L=1, R=2)
    N, b, w, Hkv, G, d = c["N"], c["b"], c["w"], c["Hkv"], c["G"], c["d"]
    res = orc.compress(c["kp"], c["vp"], c["tables"], c["lengths"], c["wq"], N, w, 0.5,
                       c["free"], c["free_count"], c["rc"], Hq=Hkv * G)
    assert res["status"] == 0
    q = bf16(rng(94).standard_normal((c["R"], Hkv * G, d)))
    scale = 1.0 / math.sqrt(d)
    st, o64, _ = orc.decode_attn(q, res["kpools"][0], res["vpools"][0], res["tables"],
                                 res["lengths"], scale)
    assert st == 0
    for r in range(c["R"]):
        for hq in range(Hkv * G):
            h = hq // G
            kept = res["kept"][0, r, h]
            K = torch.tensor(widen(_gather(c["kp"][0], c["tables"][r], h, b)))
            V = torch.tensor(widen(_gather(c["vp"][0], c["tables"][r], h, b)))
            mask = torch.zeros(N * b, dtype=torch.bool)
            mask[torch.tensor(kept, dtype=torch.long)] = True
            qq = torch.tensor(widen(q[r, hq]))
            o = torch.nn.functional.scaled_dot_product_attention(
                qq[None, None, :], K[None], V[None], attn_mask=mask[None, None, :],
                scale=scale)[0, 0]
            close(o64[r, hq], o.numpy(), 1e-12, "compacted vs masked attention")


# ------------------------------------------------------------ decode append

def _logical(pool, table, length, h, b):
    """Rows 0 .. length-1 of kv head h, gathered through a block table."""
    return np.stack([pool[table[t // b], h, t % b] for t in range(length)]) if length else \
        np.zeros((0, pool.shape[3]), dtype=pool.dtype)


def pin_append_fork_handworked(orc):
    """The hand-worked fork of tests/golden/append_fork_handworked.json."""
    with open(os.path.join(GOLDEN, "append_fork_handworked.json")) as f:
        gd = json.load(f)
    b, nb, L, Hkv, d = gd["b"], gd["num_blocks"], 2, 2, 3
    g = rng(110)
    kp = [bf16(g.standard_normal((nb, Hkv, b, d))) for _ in range(L)]
    vp = [bf16(g.standard_normal((nb, Hkv, b, d))) for _ in range(L)]
    for case in gd["cases"]:
        res = orc.append_slots(kp, vp, gd["tables"], gd["lengths"], gd["free_ids"],
                               len(gd["free_ids"]), gd["refcount"], gd["n_max"],
                               req_idx=np.array(case["req_idx"], dtype=np.int32))
        assert res["status"] == 0
        assert res["tables"].tolist() == case["tables"]
        assert res["lengths"].tolist() == case["lengths"]
        assert res["refcount"].tolist() == case["refcount"]
        assert res["free_count"] == case["free_count"]
        assert res["free_ids"][:res["free_count"]].tolist() == gd["free_ids"][:case["free_count"]]
        assert res["triggers"].tolist() == case["triggers"]
        for src, dst, rows in case["copied"]:
            for l in range(L):
                assert np.array_equal(res["kpools"][l][dst, :, :rows], kp[l][src, :, :rows])
                assert np.array_equal(res["vpools"][l][dst, :, :rows], vp[l][src, :, :rows])
                assert np.array_equal(res["kpools"][l][src], kp[l][src])
                assert np.array_equal(res["vpools"][l][src], vp[l][src])


def _fork_cache(seed, R=10, b=4, nmax=5, L=2, Hkv=2, d=4, spare=40):
    """A small forked decode-time cache from the shared input generator, with
    the pools as bf16 bit patterns."""
    c = W.fork_cache(seed, R, nmax, L=L, Hkv=Hkv, d=d, b=b, spare=spare)
    c["kp"] = [W.bf16_bits(k).copy() for k in c.pop("k_pools")]
    c["vp"] = [W.bf16_bits(v).copy() for v in c.pop("v_pools")]
    c["nmax"] = c.pop("n_max")
    return c


def pin_append_invariants(orc):
    """On random forked caches: the logical content of every row is unchanged,
    a row writes only unshared blocks, refcounts equal table references, free
    and used blocks partition the pool, and the number of copies of a block
    with m writers in the call and refcount c at the start is min(m, c - 1)
    (every writer but the last copies unless other holders remain)."""
    for seed in range(120, 126):
        c = _fork_cache(seed)
        b, nmax = c["b"], c["nmax"]
        R = c["tables"].shape[0]
        req = rng(seed + 1000).permutation(R).astype(np.int32)
        res = orc.append_slots(c["kp"], c["vp"], c["tables"], c["lengths"], c["free"],
                               c["nfree"], c["rc"], nmax, req_idx=req)
        assert res["status"] == 0
        writers = {}
        unalloc = 0
        for r in req:
            p = int(c["lengths"][r])
            x = int(c["tables"][r, p // b])
            if x < 0:
                unalloc += 1
            else:
                writers[x] = writers.get(x, 0) + 1
        copies = sum(min(m, int(c["rc"][x]) - 1) for x, m in writers.items())
        assert c["nfree"] - res["free_count"] == unalloc + copies
        for x, m in writers.items():
            assert res["refcount"][x] == c["rc"][x] - min(m, int(c["rc"][x]) - 1)
        for r in range(R):
            p = int(c["lengths"][r])
            assert res["lengths"][r] == p + 1
            for l in range(c["L"]):
                for h in range(c["Hkv"]):
                    assert np.array_equal(_logical(res["kpools"][l], res["tables"][r], p, h, b),
                                          _logical(c["kp"][l], c["tables"][r], p, h, b))
                    assert np.array_equal(_logical(res["vpools"][l], res["tables"][r], p, h, b),
                                          _logical(c["vp"][l], c["tables"][r], p, h, b))
        # the block each row will write is exclusively its own
        tails = [int(res["tables"][r, int(c["lengths"][r]) // b]) for r in range(R)]
        assert len(set(tails)) == R
        assert all(res["refcount"][x] == 1 for x in tails)
        ref = np.zeros_like(res["refcount"])
        for x in res["tables"].reshape(-1):
            if x >= 0:
                ref[x] += 1
        assert np.array_equal(ref, res["refcount"])
        fc = res["free_count"]
        assert fc + int(np.count_nonzero(res["refcount"] >= 1)) == c["num_blocks"]
        assert np.all(res["refcount"][res["free_ids"][:fc]] == 0)
        for l in range(c["L"]):                       # blocks still referenced are untouched
            used = [x for x in range(c["num_blocks"]) if c["rc"][x] > 0]
            assert np.array_equal(res["kpools"][l][used], c["kp"][l][used])
            assert np.array_equal(res["vpools"][l][used], c["vp"][l][used])
        trig = [int(r) for r in req if c["lengths"][r] + 1 == nmax * b]
        assert res["triggers"].tolist() == trig


def pin_append_errors(orc):
    """All or nothing: a row already holding N_max full blocks, a partial tail
    with no block, a duplicate row or too few free blocks change nothing."""
    b, nmax = 4, 2
    kp = [bf16(np.ones((6, 1, b, 2)))]
    vp = [bf16(np.ones((6, 1, b, 2)))]
    base = dict(tables=np.array([[0, 1, -1], [0, 2, -1]], dtype=np.int32),
                lengths=np.array([6, 6], dtype=np.int32),
                rc=np.array([2, 1, 1, 0, 0, 0], dtype=np.int32),
                free=np.array([5, 4, 3, -1, -1, -1], dtype=np.int32))

    def run(tables=None, lengths=None, rc=None, fc=3, req=None):
        t = base["tables"] if tables is None else np.array(tables, dtype=np.int32)
        ln = base["lengths"] if lengths is None else np.array(lengths, dtype=np.int32)
        r = base["rc"] if rc is None else np.array(rc, dtype=np.int32)
        res = orc.append_slots(kp, vp, t, ln, base["free"], fc, r, nmax,
                               req_idx=None if req is None else np.array(req, dtype=np.int32))
        if res["status"] != 0:
            assert np.array_equal(res["tables"], t) and np.array_equal(res["lengths"], ln)
            assert np.array_equal(res["refcount"], r) and res["free_count"] == fc
        return res["status"]

    assert run() == 0
    assert run(lengths=[8, 6]) == -1          # due for compression first
    assert run(lengths=[6, 9]) == -1          # beyond the table row
    assert run(tables=[[0, 1, -1], [0, -1, -1]], rc=[2, 1, 0, 0, 0, 0]) == -1  # partial, no block
    assert run(req=[1, 1]) == -1              # duplicate row
    assert run(rc=[2, 0, 1, 0, 0, 0]) == -1   # a tail block with no reference
    assert run(tables=[[0, 1, -1], [0, 1, -1]], rc=[2, 1, 0, 0, 0, 0]) == -1  # 2 writers, 1 ref
    # two new blocks needed (row 0's tail 1 is shared with nothing; make it shared)
    t = [[0, 1, -1], [0, 1, -1]]
    assert run(tables=t, rc=[2, 2, 0, 0, 0, 0], lengths=[4, 5], fc=0) == -3
    assert run(tables=t, rc=[2, 2, 0, 0, 0, 0], lengths=[5, 5], fc=0) == -3


def pin_alloc_release_handworked(orc):
    """b = 4, free stack [5, 4, 3, 2, 1, 0] (top 0).  Rows 0 and 1 get 5 and 3
    tokens: row 0 pops 0 then 1, row 1 pops 2; lengths 5 and 3, three blocks
    left.  Releasing rows 1 then 0 pushes 2, then 0 and 1: the stack reads
    [5, 4, 3, 2, 0, 1] and every refcount is 0 again."""
    tables = np.full((3, 4), -1, dtype=np.int32)
    free = np.array([5, 4, 3, 2, 1, 0], dtype=np.int32)
    rc = np.zeros(6, dtype=np.int32)
    a = orc.alloc_rows(tables, np.zeros(3, np.int32), free, 6, rc, [5, 3], 4,
                       req_idx=np.array([0, 1], np.int32))
    assert a["status"] == 0
    assert a["tables"][:2].tolist() == [[0, 1, -1, -1], [2, -1, -1, -1]]
    assert a["lengths"].tolist() == [5, 3, 0] and a["free_count"] == 3
    assert a["refcount"].tolist() == [1, 1, 1, 0, 0, 0]
    r = orc.release_rows(a["tables"], a["lengths"], a["free_ids"], a["free_count"],
                         a["refcount"], req_idx=np.array([1, 0], np.int32))
    assert r["status"] == 0
    assert r["free_ids"].tolist() == [5, 4, 3, 2, 0, 1] and r["free_count"] == 6
    assert np.all(r["tables"] == -1) and np.all(r["lengths"] == 0)
    assert np.all(r["refcount"] == 0)


def pin_release_shared_and_lifecycle(orc):
    """Releasing forked requests drops one reference per holder and frees a
    block at its last holder, in request-then-entry order; a whole life cycle
    (alloc, append, compress, release of everything) returns every block to
    the pool with refcount 0."""
    c = _fork_cache(170, R=9, b=4, nmax=5)
    req = np.array([4, 0, 7, 2], dtype=np.int32)
    r = orc.release_rows(c["tables"], c["lengths"], c["free"], c["nfree"], c["rc"], req_idx=req)
    assert r["status"] == 0
    rc = c["rc"].copy()
    pushed = []
    for row in req:
        for x in c["tables"][row]:
            if x >= 0:
                rc[x] -= 1
                if rc[x] == 0:
                    pushed.append(int(x))
    assert np.array_equal(r["refcount"], rc)
    assert r["free_ids"][c["nfree"]:r["free_count"]].tolist() == pushed
    assert np.all(r["tables"][req] == -1) and np.all(r["lengths"][req] == 0)
    others = np.setdiff1d(np.arange(9), req)
    assert np.array_equal(r["tables"][others], c["tables"][others])

    # life cycle on an empty pool
    b, N, L, Hkv, d = 4, 3, 1, 2, 4
    nb = 40
    kp = [bf16(rng(171).standard_normal((nb, Hkv, b, d)))]
    vp = [bf16(rng(172).standard_normal((nb, Hkv, b, d)))]
    tables = np.full((4, N), -1, dtype=np.int32)
    st = orc.alloc_rows(tables, np.zeros(4, np.int32), np.arange(nb, dtype=np.int32), nb,
                        np.zeros(nb, np.int32), [9, 11, 4, 0], b)
    assert st["status"] == 0
    cur = dict(kpools=kp, vpools=vp, tables=st["tables"], lengths=st["lengths"],
               free_ids=st["free_ids"], free_count=st["free_count"], refcount=st["refcount"])
    a = orc.append_slots(cur["kpools"], cur["vpools"], cur["tables"], cur["lengths"],
                         cur["free_ids"], cur["free_count"], cur["refcount"], N)
    assert a["status"] == 0 and a["triggers"].tolist() == [1]   # 11 -> 12 = N*b
    wq = bf16(rng(173).standard_normal((L, 1, Hkv, 2, d)))
    cmp_ = orc.compress(a["kpools"], a["vpools"], a["tables"], a["lengths"], wq, N, 2, 0.5,
                        a["free_ids"], a["free_count"], a["refcount"], Hq=Hkv,
                        req_idx=a["triggers"])
    assert cmp_["status"] == 0
    a = orc.append_slots(cmp_["kpools"], cmp_["vpools"], cmp_["tables"], cmp_["lengths"],
                         cmp_["free_ids"], cmp_["free_count"], cmp_["refcount"], N)
    assert a["status"] == 0 and a["lengths"].tolist() == [11, 9, 6, 2]
    rel = orc.release_rows(a["tables"], a["lengths"], a["free_ids"], a["free_count"],
                           a["refcount"])
    assert rel["status"] == 0
    assert rel["free_count"] == nb and np.all(rel["refcount"] == 0)
    assert sorted(rel["free_ids"].tolist()) == list(range(nb))


def pin_fork_then_append_then_release(orc):
    """Forking a request of 6 tokens (b 4) into two samples shares both blocks
    (refcount 3); each sample's next token copies the partial tail on write
    (the last writer keeps it); releasing the three rows returns every block."""
    b = 4
    kp = [bf16(rng(180).standard_normal((8, 1, b, 2)))]
    vp = [bf16(rng(181).standard_normal((8, 1, b, 2)))]
    tables = np.full((3, 3), -1, np.int32)
    a = orc.alloc_rows(tables, np.zeros(3, np.int32), np.arange(8, dtype=np.int32), 8,
                       np.zeros(8, np.int32), [6], b, req_idx=np.array([0], np.int32))
    assert a["tables"][0].tolist() == [7, 6, -1]
    f = orc.fork_rows(a["tables"], a["lengths"], a["refcount"], [0, 0], [1, 2])
    assert f["status"] == 0
    assert f["tables"].tolist() == [[7, 6, -1]] * 3 and f["lengths"].tolist() == [6, 6, 6]
    assert f["refcount"][[7, 6]].tolist() == [3, 3]
    s = orc.append_slots(kp, vp, f["tables"], f["lengths"], a["free_ids"], a["free_count"],
                         f["refcount"], 3)
    assert s["status"] == 0
    # rows 0 and 1 copy block 6 (to 5, then 4); row 2, the last writer, keeps it
    assert s["tables"][:, 1].tolist() == [5, 4, 6]
    assert s["refcount"][[7, 6, 5, 4]].tolist() == [3, 1, 1, 1]
    assert np.array_equal(s["kpools"][0][5, :, :2], kp[0][6, :, :2])
    r = orc.release_rows(s["tables"], s["lengths"], s["free_ids"], s["free_count"], s["refcount"])
    assert r["status"] == 0 and r["free_count"] == 8 and np.all(r["refcount"] == 0)
    # errors: a destination that holds tokens, or a row forked from itself
    assert orc.fork_rows(f["tables"], f["lengths"], f["refcount"], [0], [1])["status"] == -1
    assert orc.fork_rows(a["tables"], a["lengths"], a["refcount"], [1], [1])["status"] == -1


def pin_alloc_release_errors(orc):
    """All or nothing: allocating into a row that holds tokens or blocks, too
    few free blocks, a repeated row, or releasing a block more often than it
    is referenced changes nothing."""
    tables = np.full((2, 3), -1, dtype=np.int32)
    free = np.arange(4, dtype=np.int32)
    rc = np.zeros(4, np.int32)
    assert orc.alloc_rows(tables, np.array([1, 0], np.int32), free, 4, rc, [4, 4], 4)["status"] == -1
    t2 = tables.copy()
    t2[1, 0] = 3
    assert orc.alloc_rows(t2, np.zeros(2, np.int32), free, 4, rc, [4, 4], 4)["status"] == -1
    assert orc.alloc_rows(tables, np.zeros(2, np.int32), free, 4, rc, [9, 8], 4)["status"] == -3
    assert orc.alloc_rows(tables, np.zeros(2, np.int32), free, 4, rc, [4, 4], 4,
                          req_idx=np.array([0, 0], np.int32))["status"] == -1
    held = np.array([[0, 1, -1], [0, -1, -1]], dtype=np.int32)
    rc2 = np.array([1, 1, 0, 0], np.int32)   # block 0 is in two rows but counted once
    r = orc.release_rows(held, np.array([5, 2], np.int32), np.array([2, 3, -1, -1], np.int32), 2,
                         rc2)
    assert r["status"] == -1
    assert np.array_equal(r["tables"], held) and r["free_count"] == 2


def pin_append_kv_then_decode(orc):
    """After the slots are reserved and each layer's new K/V row written, the
    new row sits at position p of the row's table, nothing else moved, and
    decode attention over the grown cache equals torch SDPA over the old
    logical rows with the new one appended."""
    c = _fork_cache(140, R=8, L=2, Hkv=2, d=8)
    b, nmax, Hkv, d = c["b"], c["nmax"], c["Hkv"], 8
    R = c["tables"].shape[0]
    res = orc.append_slots(c["kp"], c["vp"], c["tables"], c["lengths"], c["free"], c["nfree"],
                           c["rc"], nmax)
    assert res["status"] == 0
    g = rng(141)
    G = 2
    scale = 1.0 / math.sqrt(d)
    for l in range(c["L"]):
        kn = bf16(g.standard_normal((R, Hkv, d)))
        vn = bf16(g.standard_normal((R, Hkv, d)))
        st, kpool, vpool = orc.append_kv(res["kpools"][l], res["vpools"][l], res["tables"],
                                         res["lengths"], kn, vn)
        assert st == 0
        q = bf16(g.standard_normal((R, Hkv * G, d)))
        st, o64, _ = orc.decode_attn(q, kpool, vpool, res["tables"], res["lengths"], scale)
        assert st == 0
        for r in range(R):
            p = int(c["lengths"][r])
            for h in range(Hkv):
                K = _logical(kpool, res["tables"][r], p + 1, h, b)
                V = _logical(vpool, res["tables"][r], p + 1, h, b)
                assert np.array_equal(K[:p], _logical(c["kp"][l], c["tables"][r], p, h, b))
                assert np.array_equal(V[:p], _logical(c["vp"][l], c["tables"][r], p, h, b))
                assert np.array_equal(K[p], kn[r, h]) and np.array_equal(V[p], vn[r, h])
                for gq in range(G):
                    hq = h * G + gq
                    o = torch.nn.functional.scaled_dot_product_attention(
                        torch.tensor(widen(q[r, hq]))[None, None, :], torch.tensor(widen(K))[None],
                        torch.tensor(widen(V))[None], scale=scale)[0, 0]
                    close(o64[r, hq], o.numpy(), 1e-12, "decode after append")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
