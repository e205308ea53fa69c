"""The allocation-free decode-attention entry point.

Some callers cannot allocate device memory where they run decode attention:
an allocator or memory-pool callback (allocating there would re-enter the
allocator), a plug-in in a process whose host owns all device memory, a
real-time path that must not wait on the allocator.  For them the library
exports zp_paged_decode_attn_noalloc, which needs no handle and keeps its
split-K partials in a fixed array compiled into the library.

These tests call it through the C ABI, on two calls in a row (the second call
reuses the array the first one left behind), and check each output against
the CPU oracle within the decode tolerance used everywhere else (2e-2
absolute) and against the regular entry point (zp_paged_decode_attn), which
runs the same kernels with the same splits: bit for bit.  A permuted request
list and a length out of range (flagged in the status word, or in the
array's own word when no status word is passed) are covered too.  The file
name makes pytest collect it last.
"""
import math

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DECODE_ATOL = 2e-2


def _setup(d, Hkv, Hq):
    from compressed_paged_kv_gb300 import _build
    _build.build()
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="noalloc", d=d, Hkv=Hkv, Hq=Hq, N=20, R=9,
                  spare_blocks=8)
    st = W.build_cache(wl, "cuda")
    lens = torch.tensor([0, 1, 15, 16, 17, 100, 255, 319, 320], dtype=torch.int32, device="cuda")
    return wl, st, lens


def _noalloc(st, wl, q, lens, req_idx, out, status, scale):
    stream = torch.cuda.current_stream().cuda_stream
    return zp.zp_paged_decode_attn_noalloc(
        st.k_pools[0].data_ptr(), st.v_pools[0].data_ptr(), st.k_pools[0].shape[0], wl.Hkv,
        wl.Hq, wl.d, q.data_ptr(), st.block_tables.data_ptr(), st.block_tables.shape[1],
        st.block_tables.shape[0], lens.data_ptr(), 0 if req_idx is None else req_idx.data_ptr(),
        q.shape[0], scale, out.data_ptr(), 0 if status is None else status.data_ptr(), stream)


@pytest.mark.parametrize("d,Hkv,Hq", [(128, 8, 32), (64, 2, 4)])
@pytest.mark.parametrize("permuted", [False, True], ids=["rows_in_order", "permuted_rows"])
def test_noalloc_decode_matches_oracle_and_handle_path(orc, d, Hkv, Hq, permuted):
    wl, st, lens = _setup(d, Hkv, Hq)
    cache = zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=st.block_tables.shape[0],
                     max_blocks_per_req=st.block_tables.shape[1])
    scale = 1.0 / math.sqrt(d)
    nrows = st.block_tables.shape[0]
    rows = (torch.randperm(nrows, generator=torch.Generator().manual_seed(3)) if permuted
            else torch.arange(nrows)).to(torch.int32)
    req_idx = rows.cuda() if permuted else None
    tab = st.block_tables[rows.long()].cpu().numpy()
    ln = lens[rows.long()].cpu().numpy()
    kb, vb = W.bf16_bits(st.k_pools[0]), W.bf16_bits(st.v_pools[0])
    g = torch.Generator(device="cuda").manual_seed(5)
    for call in range(2):
        q = torch.randn(st.decode_q[0].shape, generator=g, device="cuda").to(torch.bfloat16)
        ref = torch.empty_like(q)
        cache.decode(0, q, st.block_tables, lens, scale, ref, req_idx=req_idx)
        out = torch.full_like(q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(st, wl, q, lens, req_idx, out, status, scale) == zp.OK
        torch.cuda.synchronize()
        assert int(status.item()) == zp.OK
        assert cache.status() == zp.OK
        ost, o64, _ = orc.decode_attn(W.bf16_bits(q), kb, vb, tab, ln, scale)
        assert ost == 0
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), call
        err_oracle = float(np.abs(got - o64).max())
        assert err_oracle <= DECODE_ATOL, (call, err_oracle)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), call
    cache.close()


def test_noalloc_length_out_of_range_is_flagged():
    wl, st, lens = _setup(128, 8, 32)
    bad = lens.clone()
    bad[4] = st.block_tables.shape[1] * 16 + 1
    q = st.decode_q[0].contiguous()
    out = torch.zeros_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(st, wl, q, bad, None, out, status, 0.125) == zp.OK
    torch.cuda.synchronize()
    assert int(status.item()) == zp.ERR_DEVICE_CHECK
    # without a status word the flag goes to the array's own word
    assert _noalloc(st, wl, q, bad, None, out, None, 0.125) == zp.OK
    torch.cuda.synchronize()
    # a valid call afterwards is unaffected by the earlier ones
    status.zero_()
    assert _noalloc(st, wl, q, lens, None, out, status, 0.125) == zp.OK
    torch.cuda.synchronize()
    assert int(status.item()) == zp.OK
