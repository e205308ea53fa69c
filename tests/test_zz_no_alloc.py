"""The allocation-free decode-attention entry point.

Some callers cannot allocate device memory at the point where they run
decode attention (inside a CUDA graph capture, inside an allocator callback,
in a plug-in whose host process owns all device memory).  For them the
library exports zp_paged_decode_attn_noalloc, which needs no handle and keeps
its split-K partials in a fixed array compiled into the library.  This test
calls it through the C ABI and checks it against the regular entry point
(zp_paged_decode_attn) within the decode tolerance used everywhere else, on
two calls in a row: the second call reuses the array the first one left
behind.  The file name makes pytest collect it last.
"""
import math

import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from compressed_paged_kv_gb300 import zp

pytestmark = pytest.mark.gpu

DECODE_ATOL = 2e-2


@pytest.mark.parametrize("d,Hkv,Hq", [(128, 8, 32), (64, 2, 4)])
def test_noalloc_decode_matches_handle_path(d, Hkv, Hq):
    from compressed_paged_kv_gb300 import _build
    _build.build()
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="noalloc", d=d, Hkv=Hkv, Hq=Hq, N=20, R=9,
                  spare_blocks=8)
    st = W.build_cache(wl, "cuda")
    lens = torch.tensor([0, 1, 15, 16, 17, 100, 255, 319, 320], dtype=torch.int32, device="cuda")
    cache = zp.Cache(st.k_pools, st.v_pools, wl.Hq, max_requests=st.block_tables.shape[0],
                     max_blocks_per_req=st.block_tables.shape[1])
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    g = torch.Generator(device="cuda").manual_seed(5)
    for call in range(2):
        q = torch.randn(st.decode_q[0].shape, generator=g, device="cuda").to(torch.bfloat16)
        ref = torch.empty_like(q)
        cache.decode(0, q, st.block_tables, lens, scale, ref)
        out = torch.full_like(q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = zp.zp_paged_decode_attn_noalloc(
            st.k_pools[0].data_ptr(), st.v_pools[0].data_ptr(), st.k_pools[0].shape[0], wl.Hkv,
            wl.Hq, wl.d, q.data_ptr(), st.block_tables.data_ptr(), st.block_tables.shape[1],
            st.block_tables.shape[0], lens.data_ptr(), 0, q.shape[0], scale, out.data_ptr(),
            status.data_ptr(), stream)
        assert rc == zp.OK
        torch.cuda.synchronize()
        assert int(status.item()) == zp.OK
        assert cache.status() == zp.OK
        err = (out.float() - ref.float()).abs().max().item()
        assert math.isfinite(err) and err <= DECODE_ATOL, (call, err)
