"""Seeded synthetic inputs for the compression / decode-attention hot path.

This module builds INPUTS only: random K/V/Q tensors, block tables, refcounts
and free stacks with the shapes and structure of the workloads below.  It holds
none of the method's arithmetic (no scores, no selection, no compaction, no
attention), so both the CUDA path and the CPU oracle can be fed from it.

Workloads (shapes of the models the Zipage summaries evaluate: Qwen3-8B and
DeepSeek-R1-Distill-Llama-8B, KV budget 2048 tokens):

  tiny         1 layer, 2/4 heads, d 64, b 16, N_max 8, 2 requests sharing
               block 0 (refcount 2); K, V, Q i.i.d. N(0,1).
  qwen3_1l     1 layer, 8/32 heads, d 128, b 16, N_max 128, 64 requests, no
               sharing; K, V, Q i.i.d. N(0,1).
  qwen3_36l    36 layers, 256 requests in 32 groups of 8 sharing a 4-block
               prompt prefix (refcount 8); K AR(1) rho 0.9 + 1% heavy hitters
               (x8); V, Q N(0,1).
  long4k       36 layers, N_max 256, 128 requests, K AR(1) rho 0.95, V N(0,1).
  mixed        32 layers, 512 requests, lengths uniform in [1024, 2048); 51
               of them forced to 2048 (they compress); the rest decode.

All tensors are generated in fp32 from torch generators seeded per (tensor,
layer) from a master seed, then rounded once to bf16.  Physical block ids are
a seeded permutation, so block tables are not contiguous.
"""
from __future__ import annotations

import dataclasses
import math

import torch

MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    """One step of the SplitMix64 generator (Steele, Lea, Flood 2014)."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def derive_seed(master: int, *keys: int) -> int:
    s = splitmix64(master & MASK64)
    for k in keys:
        s = splitmix64(s ^ (k & MASK64))
    return s & ((1 << 63) - 1)


TENSOR_K, TENSOR_V, TENSOR_Q, TENSOR_DQ, TENSOR_TABLE, TENSOR_HH, TENSOR_LEN = range(7)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    Hkv: int
    Hq: int
    d: int
    b: int
    N: int            # N_max: blocks per request at compression
    w: int            # observation window
    lam: float        # lambda
    R: int            # requests in the batch
    group: int = 1    # requests per prefix-sharing group
    prefix_blocks: int = 0
    rho: float = 0.0  # AR(1) coefficient of K along the sequence (0: i.i.d.)
    hh_prob: float = 0.0
    hh_scale: float = 8.0
    spare_blocks: int = 64
    mixed: bool = False
    mixed_compress: int = 0
    mixed_len_lo: int = 0
    seed: int = 0

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def T(self):
        return self.N * self.b

    @property
    def C(self):
        return self.T - self.w

    @property
    def n_keep(self):
        return (self.N - 1) * self.b - self.w

    def units(self, R=None):
        return (self.R if R is None else R) * self.L * self.Hkv

    def unit_bytes(self, moved=None):
        """Algorithmic bytes of one compression unit: K read once for scoring,
        V read + K write + V write of the moved rows, the window queries."""
        M = (self.N - 1) * self.b if moved is None else moved
        row = self.d * 2
        return self.T * row + 3 * M * row + self.w * self.G * row


WORKLOADS = {
    "tiny": Workload("tiny", L=1, Hkv=2, Hq=4, d=64, b=16, N=8, w=8, lam=0.5, R=2, group=2,
                     prefix_blocks=1, spare_blocks=16, seed=20260000),
    "qwen3_1l": Workload("qwen3_1l", L=1, Hkv=8, Hq=32, d=128, b=16, N=128, w=8, lam=0.5,
                         R=64, spare_blocks=64, seed=20260001),
    "qwen3_36l": Workload("qwen3_36l", L=36, Hkv=8, Hq=32, d=128, b=16, N=128, w=8, lam=0.5,
                          R=256, group=8, prefix_blocks=4, rho=0.9, hh_prob=0.01,
                          spare_blocks=1024 + 64, seed=20260002),
    "long4k": Workload("long4k", L=36, Hkv=8, Hq=32, d=128, b=16, N=256, w=8, lam=0.5, R=128,
                       rho=0.95, spare_blocks=64, seed=20260003),
    "mixed": Workload("mixed", L=32, Hkv=8, Hq=32, d=128, b=16, N=128, w=8, lam=0.5, R=512,
                      mixed=True, mixed_compress=51, mixed_len_lo=1024, spare_blocks=64,
                      seed=20260004),
}
# Index order used by the configuration list this library is measured on.
WORKLOAD_ORDER = ["tiny", "qwen3_1l", "qwen3_36l", "long4k", "mixed"]


def scaled(wl: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller test cases)."""
    return dataclasses.replace(wl, **changes)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, device, seed):
    return torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)


def _ar1(eps: torch.Tensor, rho: float) -> torch.Tensor:
    """x_0 = eps_0;  x_t = rho x_{t-1} + sqrt(1-rho^2) eps_t along dim -2.
    Evaluated in chunks: inside a chunk the recursion is a small lower-
    triangular matrix product; chunks are chained sequentially."""
    if rho == 0.0:
        return eps
    T = eps.shape[-2]
    CH = 64
    s = math.sqrt(1.0 - rho * rho)
    idx = torch.arange(CH, device=eps.device, dtype=torch.float32)
    expo = (idx[:, None] - idx[None, :]).clamp(min=0)
    tri = torch.where(idx[:, None] >= idx[None, :], rho ** expo, torch.zeros_like(expo))
    decay = rho ** (idx + 1.0)
    out = torch.empty_like(eps)
    prev = None
    for c0 in range(0, T, CH):
        e = eps[..., c0:c0 + CH, :]
        n = e.shape[-2]
        inject = e.clone()
        if c0 == 0:
            inject[..., 1:, :] *= s  # x_0 = eps_0 exactly
        else:
            inject *= s
        x = torch.matmul(tri[:n, :n], inject)
        if prev is not None:
            x = x + decay[:n, None] * prev[..., None, :]
        out[..., c0:c0 + n, :] = x
        prev = x[..., -1, :]
    return out


@dataclasses.dataclass
class CacheState:
    """A paged KV cache and its block accounting (all tensors on one device)."""
    wl: Workload
    k_pools: list          # L x [num_blocks][Hkv][b][d] bf16
    v_pools: list
    block_tables: torch.Tensor  # [rows][max_blocks] int32
    lengths: torch.Tensor       # [rows] int32
    refcount: torch.Tensor      # [num_blocks] int32
    free_ids: torch.Tensor      # [num_blocks] int32 (capacity = num_blocks)
    free_count: torch.Tensor    # [1] int32
    window_q: torch.Tensor      # [L][Rc][Hq][w][d] bf16 (compressing requests)
    decode_q: torch.Tensor      # [L][rows][Hq][d] bf16
    compress_rows: torch.Tensor  # [Rc] int32: rows that compress
    decode_rows: torch.Tensor    # [Rd] int32: rows that decode only

    @property
    def num_blocks(self):
        return self.refcount.shape[0]


@dataclasses.dataclass
class Layout:
    """Lengths, block tables and block accounting of a workload (host)."""
    lengths: torch.Tensor        # [R] int64
    compress_rows: torch.Tensor  # [Rc] int64
    decode_rows: torch.Tensor    # [Rd] int64
    nblk: torch.Tensor           # [R] blocks held
    tables: torch.Tensor         # [R][N] int32, -1 past a row's blocks
    refcount: torch.Tensor       # [num_blocks] int32
    free_list: torch.Tensor      # spare block ids, bottom of the stack first
    num_blocks: int
    pb: int                      # shared prefix blocks per group (0: none)
    group: int


def layout(wl: Workload, master: int) -> Layout:
    b, N, R = wl.b, wl.N, wl.R
    gcpu = _gen("cpu", derive_seed(master, TENSOR_LEN))
    if wl.mixed:
        # decoding requests are never full (a full request is due for
        # compression) unless the workload asks for full lengths only
        hi = N * b if wl.mixed_len_lo < N * b else N * b + 1
        lengths = torch.randint(wl.mixed_len_lo, hi, (R,), generator=gcpu, dtype=torch.int64)
        perm = torch.randperm(R, generator=gcpu)
        compress_rows = torch.sort(perm[:wl.mixed_compress]).values
        lengths[compress_rows] = N * b
        mask = torch.ones(R, dtype=torch.bool)
        mask[compress_rows] = False
        decode_rows = torch.arange(R)[mask]
    else:
        lengths = torch.full((R,), N * b, dtype=torch.int64)
        compress_rows = torch.arange(R)
        decode_rows = torch.arange(0)
    nblk = (lengths + b - 1) // b

    # physical block assignment: shared prefix blocks once per group
    group = max(wl.group, 1)
    pb = wl.prefix_blocks if group > 1 else 0
    n_groups = (R + group - 1) // group
    used = int(nblk.sum().item()) - (R - n_groups) * pb
    num_blocks = used + wl.spare_blocks
    gperm = _gen("cpu", derive_seed(master, TENSOR_TABLE))
    phys = torch.randperm(num_blocks, generator=gperm).to(torch.int32)
    tables = torch.full((R, N), -1, dtype=torch.int32)  # -1: no block (yet)
    refcount = torch.zeros(num_blocks, dtype=torch.int32)
    nxt = 0
    for gi in range(n_groups):
        members = list(range(gi * group, min((gi + 1) * group, R)))
        shared = phys[nxt:nxt + pb]
        nxt += pb
        for r in members:
            tables[r, :pb] = shared
            own = int(nblk[r].item()) - pb
            tables[r, pb:pb + own] = phys[nxt:nxt + own]
            nxt += own
        if pb:
            refcount[shared.long()] = len(members)
    assert nxt == used
    for r in range(R):
        own = tables[r, pb:int(nblk[r].item())]
        refcount[own.long()] += 1
    return Layout(lengths, compress_rows, decode_rows, nblk, tables, refcount,
                  phys[used:].clone(), num_blocks, pb, group)


def layer_kv(wl: Workload, master: int, l: int, pb: int, group: int, device, rows=None):
    """K and V of layer l for every request (or the requests `rows`), token
    order: two bf16 tensors [R'][Hkv][T][d].  The draws are always made for
    all R requests (one generator per tensor and layer), so a subset holds
    exactly the values of the full build."""
    R, Hkv, T, d, b = wl.R, wl.Hkv, wl.T, wl.d, wl.b
    eps = _normal((R, Hkv, T, d), device, derive_seed(master, TENSOR_K, l))
    veps = _normal((R, Hkv, T, d), device, derive_seed(master, TENSOR_V, l))
    u = None
    if wl.hh_prob > 0:
        u = torch.rand((R, Hkv, T), generator=_gen(device, derive_seed(master, TENSOR_HH, l)),
                       device=device)
    if pb:
        # prefix tokens are generated once per group (from its first member)
        P = pb * b
        lead = (torch.arange(R, device=device) // group) * group
        eps[:, :, :P] = eps[lead][:, :, :P]
        veps[:, :, :P] = veps[lead][:, :, :P]
        if u is not None:
            u[:, :, :P] = u[lead][:, :, :P]
    # the recursion runs over all requests even for a subset: its batched
    # products could round differently for another batch size
    K = _ar1(eps, wl.rho)
    del eps
    if rows is not None:
        sel = torch.as_tensor(rows, device=device).long()
        K, veps = K[sel], veps[sel]
        u = u[sel] if u is not None else None
    if u is not None:
        K = torch.where((u < wl.hh_prob)[..., None], K * wl.hh_scale, K)
    return K.to(torch.bfloat16), veps.to(torch.bfloat16)


def layer_window_q(wl: Workload, master: int, l: int, Rc: int, device):
    return _normal((Rc, wl.Hq, wl.w, wl.d), device,
                   derive_seed(master, TENSOR_Q, l)).to(torch.bfloat16)


def layer_decode_q(wl: Workload, master: int, l: int, device):
    return _normal((wl.R, wl.Hq, wl.d), device,
                   derive_seed(master, TENSOR_DQ, l)).to(torch.bfloat16)


def build_cache(wl: Workload, device="cpu", seed=None, with_decode_q=True) -> CacheState:
    """Builds the cache of a workload: every request's K/V rows written through
    its block table into per-layer pools, plus the queries of one step."""
    master = wl.seed if seed is None else seed
    b, N, d, Hkv, L = wl.b, wl.N, wl.d, wl.Hkv, wl.L
    R = wl.R
    lay = layout(wl, master)
    num_blocks, nblk, tables = lay.num_blocks, lay.nblk, lay.tables
    free_ids = torch.full((num_blocks,), -1, dtype=torch.int32)
    free_ids[:lay.free_list.numel()] = lay.free_list
    free_count = torch.tensor([lay.free_list.numel()], dtype=torch.int32)

    k_pools, v_pools = [], []
    flat_tables = tables.to(device).long()
    live = torch.arange(N, device=device)[None, :] < nblk.to(device)[:, None]
    for l in range(L):
        kb, vb = layer_kv(wl, master, l, lay.pb, lay.group, device)
        kpool = torch.zeros((num_blocks, Hkv, b, d), dtype=torch.bfloat16, device=device)
        vpool = torch.zeros((num_blocks, Hkv, b, d), dtype=torch.bfloat16, device=device)
        # [R][Hkv][N][b][d] -> rows of blocks; only the live blocks are written
        kb = kb.view(R, Hkv, N, b, d).permute(0, 2, 1, 3, 4)
        vb = vb.view(R, Hkv, N, b, d).permute(0, 2, 1, 3, 4)
        kpool[flat_tables[live]] = kb[live]
        vpool[flat_tables[live]] = vb[live]
        del kb, vb
        k_pools.append(kpool)
        v_pools.append(vpool)

    Rc = lay.compress_rows.numel()
    window_q = torch.empty((L, Rc, wl.Hq, wl.w, d), dtype=torch.bfloat16, device=device)
    for l in range(L):
        window_q[l] = layer_window_q(wl, master, l, Rc, device)
    if with_decode_q:
        decode_q = torch.empty((L, R, wl.Hq, d), dtype=torch.bfloat16, device=device)
        for l in range(L):
            decode_q[l] = layer_decode_q(wl, master, l, device)
    else:
        decode_q = torch.empty(0, dtype=torch.bfloat16, device=device)
    i32 = dict(dtype=torch.int32, device=device)
    return CacheState(
        wl=wl, k_pools=k_pools, v_pools=v_pools, block_tables=tables.to(**i32),
        lengths=lay.lengths.to(**i32), refcount=lay.refcount.to(**i32),
        free_ids=free_ids.to(**i32), free_count=free_count.to(**i32), window_q=window_q,
        decode_q=decode_q, compress_rows=lay.compress_rows.to(**i32),
        decode_rows=lay.decode_rows.to(**i32))


def sample_snapshot(wl: Workload, rows, layers, device="cpu", seed=None, spare=None) -> dict:
    """Host snapshot (the format of `snapshot`) of a sample of a workload: the
    requests `rows` (table rows) on the layers `layers`, with exactly the
    values the full build gives them, without building the full pools.  The
    sampled rows' blocks are renumbered 0..n-1 in ascending order of their
    ids in the full build; their refcounts count the sampled rows only (equal
    to the full ones when whole sharing groups are sampled); `spare` fresh
    blocks (default: a full request's worth per sampled row) form the free
    stack.  window_q / decode_q hold the sampled compressing rows' and all
    sampled rows' queries; compress_rows / decode_rows index the sample."""
    import numpy as np
    master = wl.seed if seed is None else seed
    rows = sorted(int(r) for r in rows)
    lay = layout(wl, master)
    tab = lay.tables[rows]
    used = torch.unique(tab[tab >= 0])
    remap = torch.full((lay.num_blocks,), -1, dtype=torch.int32)
    remap[used.long()] = torch.arange(used.numel(), dtype=torch.int32)
    spare = len(rows) * wl.N if spare is None else spare
    nb = used.numel() + spare
    new_tab = torch.where(tab >= 0, remap[tab.clamp(min=0).long()], tab)
    refcount = torch.zeros(nb, dtype=torch.int32)
    for r in range(len(rows)):
        held = new_tab[r][new_tab[r] >= 0].long()
        refcount[held] += 1
    free_ids = torch.full((nb,), -1, dtype=torch.int32)
    free_ids[:spare] = torch.arange(used.numel(), nb, dtype=torch.int32)
    comp_full = lay.compress_rows.tolist()
    pos_c = {r: i for i, r in enumerate(comp_full)}
    crow = [i for i, r in enumerate(rows) if r in pos_c]
    drow = [i for i, r in enumerate(rows) if r not in pos_c]
    b, N, Hkv, d = wl.b, wl.N, wl.Hkv, wl.d
    nblk = lay.nblk[rows]
    kp, vp, wq, dq = [], [], [], []
    live = torch.arange(N)[None, :] < nblk[:, None]
    for l in layers:
        kb, vb = layer_kv(wl, master, l, lay.pb, lay.group, device, rows=rows)
        kb = kb.view(len(rows), Hkv, N, b, d).permute(0, 2, 1, 3, 4).cpu()
        vb = vb.view(len(rows), Hkv, N, b, d).permute(0, 2, 1, 3, 4).cpu()
        kpool = torch.zeros((nb, Hkv, b, d), dtype=torch.bfloat16)
        vpool = torch.zeros((nb, Hkv, b, d), dtype=torch.bfloat16)
        kpool[new_tab.long()[live]] = kb[live]
        vpool[new_tab.long()[live]] = vb[live]
        kp.append(bf16_bits(kpool))
        vp.append(bf16_bits(vpool))
        q = layer_window_q(wl, master, l, len(comp_full), device)
        wq.append(bf16_bits(q[[pos_c[rows[i]] for i in crow]]))
        dq.append(bf16_bits(layer_decode_q(wl, master, l, device)[rows]))
    return dict(
        k_pools=kp, v_pools=vp, block_tables=new_tab.numpy().copy(),
        lengths=lay.lengths[rows].to(torch.int32).numpy().copy(),
        refcount=refcount.numpy().copy(), free_ids=free_ids.numpy().copy(), free_count=spare,
        window_q=np.stack(wq), decode_q=np.stack(dq),
        compress_rows=np.asarray(crow, dtype=np.int32),
        decode_rows=np.asarray(drow, dtype=np.int32), layers=list(layers), rows=rows)


def fork_cache(seed: int, R: int, n_max: int, L: int = 2, Hkv: int = 2, d: int = 128,
               b: int = 16, spare: int = 64, len_lo: int = 0, max_fan: int = 3,
               reserve_prob: float = 0.4, len_hi: int | None = None, device="cpu") -> dict:
    """A decode-time cache with parallel samples of shared prompts.

    Rows come in groups of 1..max_fan samples that share every block of one
    prompt (its last block possibly partial, so refcount = group size);
    lengths are uniform in [len_lo, len_hi) (len_hi defaults to n_max*b); a row whose length is a
    multiple of b may already hold its next, empty block (as zp_compress
    leaves it); table entries beyond a row's blocks are -1.  Physical ids are
    a seeded permutation, the rest of the pool is the free stack.  K/V pools
    [num_blocks][Hkv][b][d] are N(0,1) rounded to bf16.

    Returns dict(tables, lengths, rc, free, nfree: numpy int32 / int;
    k_pools, v_pools: lists of L bf16 tensors on `device`; plus the sizes).
    """
    import numpy as np
    g = np.random.default_rng(seed)
    num_blocks = R * n_max + spare
    perm = g.permutation(num_blocks).astype(np.int32)
    tables = np.full((R, n_max), -1, dtype=np.int32)
    lengths = np.zeros(R, dtype=np.int32)
    nxt = 0
    r = 0
    while r < R:
        fan = min(int(g.integers(1, max_fan + 1)), R - r)
        length = int(g.integers(len_lo, n_max * b if len_hi is None else len_hi))
        nblk = -(-length // b)
        tables[r:r + fan, :nblk] = perm[nxt:nxt + nblk]
        lengths[r:r + fan] = length
        nxt += nblk
        r += fan
    for r in range(R):
        p = int(lengths[r])
        if p % b == 0 and p // b < n_max and g.random() < reserve_prob:
            tables[r, p // b] = perm[nxt]
            nxt += 1
    rc = np.zeros(num_blocks, dtype=np.int32)
    for x in tables.reshape(-1):
        if x >= 0:
            rc[x] += 1
    free = np.full(num_blocks, -1, dtype=np.int32)
    nfree = num_blocks - nxt
    free[:nfree] = perm[nxt:]
    shape = (num_blocks, Hkv, b, d)
    k_pools = [_normal(shape, device, derive_seed(seed, 1, l)).to(torch.bfloat16) for l in range(L)]
    v_pools = [_normal(shape, device, derive_seed(seed, 2, l)).to(torch.bfloat16) for l in range(L)]
    return dict(tables=tables, lengths=lengths, rc=rc, free=free, nfree=nfree, k_pools=k_pools,
                v_pools=v_pools, num_blocks=num_blocks, b=b, n_max=n_max, L=L, Hkv=Hkv, d=d)


def prefill_cache(seed: int, lens, n_max: int, L: int = 2, Hkv: int = 2, Hq: int = 8,
                  d: int = 128, w: int = 8, group: int = 1, prefix_blocks: int = 0,
                  spare: int = 64, b: int = 16, device="cpu") -> dict:
    """Requests admitted with prompts longer than the budget.

    Request r holds lens[r] tokens (any count, the last block possibly
    partial) in a seeded permutation of physical blocks; consecutive groups of
    `group` requests share their first `prefix_blocks` blocks (one prompt
    prefix); table entries past a request's blocks are -1; the rest of the
    pool plus `spare` blocks form the free stack.  K/V pools
    [num_blocks][Hkv][b][d] and window queries [L][R][Hq][w][d] are N(0,1)
    rounded to bf16 (slots past a request's length hold draws too).

    Returns dict of torch tensors on `device` (tables, lengths, refcount,
    free_ids, free_count, k_pools, v_pools, window_q) and the sizes.
    """
    R = len(lens)
    nblk = [-(-int(T) // b) for T in lens]
    stride = max(max(nblk), n_max)
    g = _gen("cpu", derive_seed(seed, TENSOR_TABLE))
    n_groups = -(-R // group)
    pb = prefix_blocks if group > 1 else 0
    used = sum(nblk) - (R - n_groups) * pb
    num_blocks = used + spare
    phys = torch.randperm(num_blocks, generator=g).to(torch.int32)
    tables = torch.full((R, stride), -1, dtype=torch.int32)
    nxt = 0
    for gi in range(n_groups):
        members = range(gi * group, min((gi + 1) * group, R))
        shared = phys[nxt:nxt + pb]
        nxt += pb
        for r in members:
            assert nblk[r] >= pb
            tables[r, :pb] = shared
            tables[r, pb:nblk[r]] = phys[nxt:nxt + nblk[r] - pb]
            nxt += nblk[r] - pb
    assert nxt == used
    refcount = torch.zeros(num_blocks, dtype=torch.int32)
    ids = tables[tables >= 0].long()
    refcount.index_add_(0, ids, torch.ones_like(ids, dtype=torch.int32))
    free_ids = torch.full((num_blocks,), -1, dtype=torch.int32)
    free_ids[:num_blocks - used] = phys[used:]
    shape = (num_blocks, Hkv, b, d)
    k_pools = [_normal(shape, device, derive_seed(seed, TENSOR_K, l)).to(torch.bfloat16)
               for l in range(L)]
    v_pools = [_normal(shape, device, derive_seed(seed, TENSOR_V, l)).to(torch.bfloat16)
               for l in range(L)]
    window_q = torch.stack([_normal((R, Hq, w, d), device, derive_seed(seed, TENSOR_Q, l))
                            for l in range(L)]).to(torch.bfloat16)
    i32 = dict(dtype=torch.int32, device=device)
    return dict(tables=tables.to(device), lengths=torch.tensor([int(T) for T in lens], **i32),
                refcount=refcount.to(device), free_ids=free_ids.to(device),
                free_count=torch.tensor([num_blocks - used], **i32), k_pools=k_pools,
                v_pools=v_pools, window_q=window_q, num_blocks=num_blocks, stride=stride,
                n_max=n_max, L=L, Hkv=Hkv, Hq=Hq, d=d, w=w, b=b)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor, as a host numpy array."""
    import numpy as np
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def snapshot(st: CacheState) -> dict:
    """Host copy of every mutable piece of a cache state."""
    return dict(
        k_pools=[bf16_bits(k) for k in st.k_pools],
        v_pools=[bf16_bits(v) for v in st.v_pools],
        block_tables=st.block_tables.cpu().numpy().copy(),
        lengths=st.lengths.cpu().numpy().copy(),
        refcount=st.refcount.cpu().numpy().copy(),
        free_ids=st.free_ids.cpu().numpy().copy(),
        free_count=int(st.free_count.cpu().item()),
        window_q=bf16_bits(st.window_q),
        compress_rows=st.compress_rows.cpu().numpy().copy(),
    )
