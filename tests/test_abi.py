"""The C ABI library loads without a GPU and exports every entry point that
include/*.h declares; host-side descriptor checks return before any CUDA call."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from compressed_paged_kv_gb300 import _build, zp
    _build.build()
    return zp.lib()


def declared_functions():
    names = []
    for path in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(path).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(zp_[a-z0-9_]+)\s*\(",
                            src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("zp_cache_create", "zp_cache_destroy", "zp_compress", "zp_paged_decode_attn",
              "zp_cache_status", "zp_status_string", "zp_append_slots", "zp_append_kv",
              "zp_compress_prefill", "zp_compress_prefill_workspace_size",
              "zp_global_redundancy", "zp_global_redundancy_gram", "zp_alloc_rows",
              "zp_release_rows",
              "zp_fork_rows"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    from compressed_paged_kv_gb300 import zp
    assert zp.status_string(zp.OK) == "ok"
    assert "free stack" in zp.status_string(zp.ERR_OUT_OF_BLOCKS)


def test_descriptor_checks_need_no_gpu(lib):
    from compressed_paged_kv_gb300 import zp
    P = ctypes.c_void_p
    dummy = (P * 1)(P(256))

    def create(**kw):
        base = dict(num_layers=1, num_kv_heads=2, num_q_heads=4, head_dim=64, block_size=16,
                    num_blocks=8, max_requests=2, max_blocks_per_req=8)
        base.update(kw)
        d = zp.zp_cache_desc(base["num_layers"], base["num_kv_heads"], base["num_q_heads"],
                             base["head_dim"], base["block_size"], base["num_blocks"],
                             base["max_requests"], base["max_blocks_per_req"], dummy, dummy)
        h = P()
        return lib.zp_cache_create(ctypes.byref(d), ctypes.byref(h))

    assert create(head_dim=96) == zp.ERR_UNSUPPORTED
    assert create(block_size=32) == zp.ERR_UNSUPPORTED
    assert create(num_q_heads=5) == zp.ERR_INVALID_ARG
    assert create(num_layers=0) == zp.ERR_INVALID_ARG
    assert create(max_blocks_per_req=1) == zp.ERR_INVALID_ARG
    assert create(num_kv_heads=1, num_q_heads=32) == zp.ERR_UNSUPPORTED
    assert lib.zp_cache_create(None, None) == zp.ERR_INVALID_ARG
    assert lib.zp_compress(None, None, 0, 0, None, None, 0, None, 0, 0, 0.0, None, None, None,
                           None) == zp.ERR_INVALID_ARG
    assert lib.zp_paged_decode_attn(None, 0, None, None, 0, 0, None, None, 0, 0.0, None,
                                    None) == zp.ERR_INVALID_ARG
    lib.zp_cache_destroy(None)


def test_every_handle_entry_refuses_a_null_cache(lib):
    """Each entry point that takes a cache handle returns ZP_ERR_INVALID_ARG
    for a null one (and null arrays), before any CUDA call."""
    from compressed_paged_kv_gb300 import zp
    skip = {"zp_cache_create", "zp_cache_destroy", "zp_status_string",
            "zp_paged_decode_attn_noalloc"}
    checked = 0
    for name in declared_functions():
        if name in skip:
            continue
        fn = getattr(lib, name)
        def zero(t):  # 0 for an integer, 0.0 for a float, NULL for a pointer
            code = getattr(t, "_type_", None)
            if code in ("f", "d"):
                return 0.0
            if isinstance(code, str) and code in "bBhHiIlLqQ?":
                return 0
            return None
        args = [zero(t) for t in fn.argtypes]
        assert fn(*args) == zp.ERR_INVALID_ARG, name
        checked += 1
    assert checked >= 12


def test_descriptor_and_size_limits_need_no_gpu(lib):
    """Pool alignment and the 2^31-row limit of cache creation, and the checks
    of the handle-free decode entry point, all answered on the host."""
    from compressed_paged_kv_gb300 import zp
    P = ctypes.c_void_p

    def create(ptr=256, **kw):
        base = dict(num_layers=1, num_kv_heads=2, num_q_heads=4, head_dim=64, block_size=16,
                    num_blocks=8, max_requests=2, max_blocks_per_req=8)
        base.update(kw)
        pools = (P * 1)(P(ptr))
        d = zp.zp_cache_desc(base["num_layers"], base["num_kv_heads"], base["num_q_heads"],
                             base["head_dim"], base["block_size"], base["num_blocks"],
                             base["max_requests"], base["max_blocks_per_req"], pools, pools)
        return lib.zp_cache_create(ctypes.byref(d), ctypes.byref(P()))

    assert create(ptr=264) == zp.ERR_INVALID_ARG          # pool not 16-byte aligned
    assert create(num_blocks=1 << 26) == zp.ERR_UNSUPPORTED  # 2^31 pool rows per layer

    buf = P(4096)

    def noalloc(R=1, Hkv=2, Hq=4, d=64, stride=8, scale=0.125, num_blocks=8):
        return lib.zp_paged_decode_attn_noalloc(buf, buf, num_blocks, Hkv, Hq, d, buf, buf,
                                                stride, 4, buf, None, R, scale, buf, None, None)

    assert noalloc(d=96) == zp.ERR_UNSUPPORTED
    assert noalloc(Hq=5) == zp.ERR_INVALID_ARG
    assert noalloc(scale=float("nan")) == zp.ERR_INVALID_ARG
    assert noalloc(num_blocks=0) == zp.ERR_INVALID_ARG
    assert noalloc(R=-1) == zp.ERR_INVALID_ARG
    assert noalloc(R=1 << 14, Hq=4) == zp.ERR_UNSUPPORTED  # more (request, head) pairs than slots
    assert noalloc(stride=1 << 27) == zp.ERR_UNSUPPORTED
    assert noalloc(R=0) == zp.OK                           # nothing to do, nothing launched
    assert lib.zp_paged_decode_attn_noalloc(None, buf, 8, 2, 4, 64, buf, buf, 8, 4, buf, None, 1,
                                            0.125, buf, None, None) == zp.ERR_INVALID_ARG
    assert lib.zp_paged_decode_attn_noalloc(buf, buf, 8, 2, 4, 64, P(4096 + 8), buf, 8, 4, buf,
                                            None, 1, 0.125, buf, None, None) == zp.ERR_INVALID_ARG
    assert noalloc(Hkv=1, Hq=32) == zp.ERR_UNSUPPORTED    # 32 query heads on one kv head
    odd = P(4096 + 8)  # pools are read 16 bytes at a time
    assert lib.zp_paged_decode_attn_noalloc(odd, buf, 8, 2, 4, 64, buf, buf, 8, 4, buf, None, 1,
                                            0.125, buf, None, None) == zp.ERR_INVALID_ARG
    assert lib.zp_paged_decode_attn_noalloc(buf, odd, 8, 2, 4, 64, buf, buf, 8, 4, buf, None, 1,
                                            0.125, buf, None, None) == zp.ERR_INVALID_ARG
    assert zp.status_string(12345) == "unknown status"


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from compressed_paged_kv_gb300 import zp
    monkeypatch.setattr(zp, "_lib", None)
    monkeypatch.setattr(zp, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        zp.lib()
