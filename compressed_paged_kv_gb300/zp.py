"""Thin ctypes binding of libzp.so (include/zp.h).  Argument marshalling only:
every step of compression and decode attention runs in the library's CUDA
kernels.  There is no fallback: if the library is missing or fails to load,
every call raises.

The functions keep the C names (``zp_cache_create``, ``zp_compress``,
``zp_paged_decode_attn``, ``zp_append_slots``, ``zp_append_kv``,
``zp_compress_prefill``, ``zp_compress_prefill_workspace_size``, ``zp_global_redundancy``,
``zp_global_redundancy_gram``,
``zp_alloc_rows``, ``zp_release_rows``, ``zp_fork_rows``,
``zp_cache_status``, ``zp_cache_destroy``, ``zp_status_string``) and take raw integers (device pointers, a cudaStream_t
as an int).  ``Cache`` wraps them for torch tensors: it reads ``data_ptr()``
and the current stream, and keeps the pool tensors alive.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_OUT_OF_BLOCKS = -3
ERR_DEVICE_CHECK = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6

P = ctypes.c_void_p
I32 = ctypes.c_int32


class zp_cache_desc(ctypes.Structure):
    _fields_ = [
        ("num_layers", I32), ("num_kv_heads", I32), ("num_q_heads", I32), ("head_dim", I32),
        ("block_size", I32), ("num_blocks", I32), ("max_requests", I32),
        ("max_blocks_per_req", I32), ("k_pools", ctypes.POINTER(P)),
        ("v_pools", ctypes.POINTER(P)),
    ]


class zp_block_pool(ctypes.Structure):
    _fields_ = [("free_ids", P), ("free_count", P), ("refcount", P), ("capacity", I32)]


class ZpError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libzp.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it first "
                              "(python -m compressed_paged_kv_gb300._build)")
        L = ctypes.CDLL(path)
        L.zp_cache_create.argtypes = [ctypes.POINTER(zp_cache_desc), ctypes.POINTER(P)]
        L.zp_cache_create.restype = I32
        L.zp_cache_destroy.argtypes = [P]
        L.zp_cache_destroy.restype = None
        L.zp_compress.argtypes = [P, P, I32, I32, P, P, I32, P, I32, I32, ctypes.c_float,
                                  ctypes.POINTER(zp_block_pool), P, P, P]
        L.zp_compress.restype = I32
        L.zp_paged_decode_attn.argtypes = [P, I32, P, P, I32, I32, P, P, I32, ctypes.c_float, P,
                                           P]
        L.zp_paged_decode_attn.restype = I32
        L.zp_paged_decode_attn_noalloc.argtypes = [P, P, I32, I32, I32, I32, P, P, I32, I32, P,
                                                   P, I32, ctypes.c_float, P, P, P]
        L.zp_paged_decode_attn_noalloc.restype = I32
        L.zp_append_slots.argtypes = [P, P, I32, I32, P, P, I32, I32,
                                      ctypes.POINTER(zp_block_pool), P, P, P]
        L.zp_append_slots.restype = I32
        L.zp_append_kv.argtypes = [P, I32, P, P, P, I32, I32, P, P, I32, P]
        L.zp_append_kv.restype = I32
        L.zp_compress_prefill_workspace_size.argtypes = [P, I32, I32,
                                                         ctypes.POINTER(ctypes.c_size_t)]
        L.zp_compress_prefill_workspace_size.restype = I32
        L.zp_compress_prefill.argtypes = [P, P, I32, I32, P, P, I32, P, I32, I32, ctypes.c_float,
                                          ctypes.POINTER(zp_block_pool), P, ctypes.c_size_t, P,
                                          P, P]
        L.zp_compress_prefill.restype = I32
        L.zp_alloc_rows.argtypes = [P, P, I32, I32, P, P, I32, P, ctypes.POINTER(zp_block_pool), P]
        L.zp_alloc_rows.restype = I32
        L.zp_release_rows.argtypes = [P, P, I32, I32, P, P, I32, ctypes.POINTER(zp_block_pool), P]
        L.zp_release_rows.restype = I32
        L.zp_fork_rows.argtypes = [P, P, I32, I32, P, P, P, I32, P, P]
        L.zp_fork_rows.restype = I32
        L.zp_global_redundancy.argtypes = [P, P, I32, I32, P, P, I32, P, P]
        L.zp_global_redundancy.restype = I32
        L.zp_global_redundancy_gram.argtypes = [P, P, I32, I32, P, P, I32, P, P]
        L.zp_global_redundancy_gram.restype = I32
        L.zp_cache_status.argtypes = [P, P, ctypes.POINTER(I32)]
        L.zp_cache_status.restype = I32
        L.zp_status_string.argtypes = [I32]
        L.zp_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


# ------------------------------------------------------------- raw C names

def status_string(status: int) -> str:
    return lib().zp_status_string(int(status)).decode()


zp_status_string = status_string


def zp_cache_create(desc: zp_cache_desc) -> int:
    """Returns the handle (an int) or raises ZpError."""
    h = P()
    st = lib().zp_cache_create(ctypes.byref(desc), ctypes.byref(h))
    if st != OK:
        raise ZpError(st, "zp_cache_create")
    return h.value


def zp_cache_destroy(handle: int) -> None:
    lib().zp_cache_destroy(P(handle))


def zp_compress(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R, window_q,
                n_max, window, lam, pool: zp_block_pool, stream, scores_out=0,
                kept_out=0) -> int:
    return lib().zp_compress(P(handle), P(block_tables), bt_stride, num_rows, P(lengths),
                             P(req_idx or None), R, P(window_q), n_max, window, float(lam),
                             ctypes.byref(pool), P(stream or None), P(scores_out or None),
                             P(kept_out or None))


def zp_compress_prefill_workspace_size(handle, R, bt_stride) -> int:
    n = ctypes.c_size_t(0)
    st = lib().zp_compress_prefill_workspace_size(P(handle), R, bt_stride, ctypes.byref(n))
    if st != OK:
        raise ZpError(st, "zp_compress_prefill_workspace_size")
    return n.value


def zp_compress_prefill(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R, window_q,
                        n_max, window, lam, pool: zp_block_pool, workspace, workspace_bytes,
                        stream, scores_out=0, kept_out=0) -> int:
    return lib().zp_compress_prefill(P(handle), P(block_tables), bt_stride, num_rows,
                                     P(lengths), P(req_idx or None), R, P(window_q), n_max,
                                     window, float(lam), ctypes.byref(pool), P(workspace or None),
                                     workspace_bytes, P(stream or None), P(scores_out or None),
                                     P(kept_out or None))


def zp_paged_decode_attn(handle, layer, q, block_tables, bt_stride, num_rows, lengths, req_idx,
                         R, scale, out, stream) -> int:
    return lib().zp_paged_decode_attn(P(handle), layer, P(q), P(block_tables), bt_stride,
                                      num_rows, P(lengths), P(req_idx or None), R, float(scale),
                                      P(out), P(stream or None))


def zp_paged_decode_attn_noalloc(k_pool, v_pool, num_blocks, num_kv_heads, num_q_heads, head_dim,
                                 q, block_tables, bt_stride, num_rows, lengths, req_idx, R, scale,
                                 out, status, stream) -> int:
    """Decode attention without a handle and without any allocation (for
    callers that cannot call cudaMalloc); see include/zp.h."""
    return lib().zp_paged_decode_attn_noalloc(
        P(k_pool), P(v_pool), num_blocks, num_kv_heads, num_q_heads, head_dim, P(q),
        P(block_tables), bt_stride, num_rows, P(lengths), P(req_idx or None), R, float(scale),
        P(out), P(status or None), P(stream or None))


def zp_append_slots(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R, n_max,
                    pool: zp_block_pool, stream, trigger_rows=0, trigger_count=0) -> int:
    return lib().zp_append_slots(P(handle), P(block_tables), bt_stride, num_rows, P(lengths),
                                 P(req_idx or None), R, n_max, ctypes.byref(pool),
                                 P(stream or None), P(trigger_rows or None),
                                 P(trigger_count or None))


def zp_append_kv(handle, layer, k_new, v_new, block_tables, bt_stride, num_rows, lengths,
                 req_idx, R, stream) -> int:
    return lib().zp_append_kv(P(handle), layer, P(k_new), P(v_new), P(block_tables), bt_stride,
                              num_rows, P(lengths), P(req_idx or None), R, P(stream or None))


def zp_alloc_rows(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R, counts,
                  pool: zp_block_pool, stream) -> int:
    return lib().zp_alloc_rows(P(handle), P(block_tables), bt_stride, num_rows, P(lengths),
                               P(req_idx or None), R, P(counts), ctypes.byref(pool),
                               P(stream or None))


def zp_release_rows(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R,
                    pool: zp_block_pool, stream) -> int:
    return lib().zp_release_rows(P(handle), P(block_tables), bt_stride, num_rows, P(lengths),
                                 P(req_idx or None), R, ctypes.byref(pool), P(stream or None))


def zp_fork_rows(handle, block_tables, bt_stride, num_rows, lengths, src_rows, dst_rows, n,
                 refcount, stream) -> int:
    return lib().zp_fork_rows(P(handle), P(block_tables), bt_stride, num_rows, P(lengths),
                              P(src_rows), P(dst_rows), n, P(refcount), P(stream or None))


def zp_global_redundancy(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R, red_out,
                         stream) -> int:
    return lib().zp_global_redundancy(P(handle), P(block_tables), bt_stride, num_rows,
                                      P(lengths), P(req_idx or None), R, P(red_out),
                                      P(stream or None))


def zp_global_redundancy_gram(handle, block_tables, bt_stride, num_rows, lengths, req_idx, R,
                              red_out, stream) -> int:
    return lib().zp_global_redundancy_gram(P(handle), P(block_tables), bt_stride, num_rows,
                                           P(lengths), P(req_idx or None), R, P(red_out),
                                           P(stream or None))


def zp_cache_status(handle, stream) -> tuple[int, int]:
    """(call status, device status) after synchronising the stream."""
    v = I32(0)
    st = lib().zp_cache_status(P(handle), P(stream or None), ctypes.byref(v))
    return st, v.value


# ------------------------------------------------------------ torch wrapper

def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Cache:
    """A zp_cache over per-layer torch pools ([num_blocks][Hkv][16][d] bf16)."""

    def __init__(self, k_pools, v_pools, num_q_heads, max_requests, max_blocks_per_req):
        import torch
        assert len(k_pools) == len(v_pools) >= 1
        for t in list(k_pools) + list(v_pools):
            if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
                raise ValueError("pools must be contiguous 4-D bf16 CUDA tensors")
        nb, hkv, b, d = k_pools[0].shape
        self.k_pools, self.v_pools = list(k_pools), list(v_pools)
        self.L, self.Hkv, self.Hq, self.d, self.b, self.num_blocks = (
            len(k_pools), hkv, num_q_heads, d, b, nb)
        kp = (P * self.L)(*[t.data_ptr() for t in k_pools])
        vp = (P * self.L)(*[t.data_ptr() for t in v_pools])
        desc = zp_cache_desc(self.L, hkv, num_q_heads, d, b, nb, max_requests,
                             max_blocks_per_req, kp, vp)
        self.handle = zp_cache_create(desc)

    def close(self):
        if getattr(self, "handle", None):
            zp_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def compress(self, block_tables, lengths, window_q, n_max, window, lam, free_ids,
                 free_count, refcount, req_idx=None, scores_out=None, kept_out=None,
                 stream=None, check=True):
        pool = zp_block_pool(free_ids.data_ptr(), free_count.data_ptr(), refcount.data_ptr(),
                             free_ids.numel())
        R = window_q.shape[1]
        st = zp_compress(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                         block_tables.shape[0], lengths.data_ptr(), _ptr(req_idx), R,
                         window_q.data_ptr(), n_max, window, lam, pool, _stream(stream),
                         _ptr(scores_out), _ptr(kept_out))
        if check and st != OK:
            raise ZpError(st, "zp_compress")
        return st

    def compress_prefill(self, block_tables, lengths, window_q, n_max, window, lam, free_ids,
                         free_count, refcount, workspace, req_idx=None, scores_out=None,
                         kept_out=None, stream=None, check=True):
        """``workspace``: a uint8 CUDA tensor of at least
        ``prefill_workspace_bytes(R, block_tables.shape[1])`` bytes."""
        pool = zp_block_pool(free_ids.data_ptr(), free_count.data_ptr(), refcount.data_ptr(),
                             free_ids.numel())
        R = window_q.shape[1]
        st = zp_compress_prefill(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                                 block_tables.shape[0], lengths.data_ptr(), _ptr(req_idx), R,
                                 window_q.data_ptr(), n_max, window, lam, pool,
                                 workspace.data_ptr(), workspace.numel(), _stream(stream),
                                 _ptr(scores_out), _ptr(kept_out))
        if check and st != OK:
            raise ZpError(st, "zp_compress_prefill")
        return st

    def prefill_workspace_bytes(self, R, bt_stride) -> int:
        return zp_compress_prefill_workspace_size(self.handle, R, bt_stride)

    def decode(self, layer, q, block_tables, lengths, scale, out, req_idx=None, stream=None,
               check=True):
        st = zp_paged_decode_attn(self.handle, layer, q.data_ptr(), block_tables.data_ptr(),
                                  block_tables.shape[1], block_tables.shape[0],
                                  lengths.data_ptr(), _ptr(req_idx), q.shape[0], scale,
                                  out.data_ptr(), _stream(stream))
        if check and st != OK:
            raise ZpError(st, "zp_paged_decode_attn")
        return st

    def append_slots(self, block_tables, lengths, n_max, free_ids, free_count, refcount,
                     req_idx=None, R=None, trigger_rows=None, trigger_count=None, stream=None,
                     check=True):
        pool = zp_block_pool(free_ids.data_ptr(), free_count.data_ptr(), refcount.data_ptr(),
                             free_ids.numel())
        if R is None:
            R = req_idx.numel() if req_idx is not None else block_tables.shape[0]
        st = zp_append_slots(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                             block_tables.shape[0], lengths.data_ptr(), _ptr(req_idx), R, n_max,
                             pool, _stream(stream), _ptr(trigger_rows), _ptr(trigger_count))
        if check and st != OK:
            raise ZpError(st, "zp_append_slots")
        return st

    def append_kv(self, layer, k_new, v_new, block_tables, lengths, req_idx=None, stream=None,
                  check=True):
        st = zp_append_kv(self.handle, layer, k_new.data_ptr(), v_new.data_ptr(),
                          block_tables.data_ptr(), block_tables.shape[1], block_tables.shape[0],
                          lengths.data_ptr(), _ptr(req_idx), k_new.shape[0], _stream(stream))
        if check and st != OK:
            raise ZpError(st, "zp_append_kv")
        return st

    def alloc_rows(self, block_tables, lengths, counts, free_ids, free_count, refcount,
                   req_idx=None, stream=None, check=True):
        pool = zp_block_pool(free_ids.data_ptr(), free_count.data_ptr(), refcount.data_ptr(),
                             free_ids.numel())
        st = zp_alloc_rows(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                           block_tables.shape[0], lengths.data_ptr(), _ptr(req_idx),
                           counts.numel(), counts.data_ptr(), pool, _stream(stream))
        if check and st != OK:
            raise ZpError(st, "zp_alloc_rows")
        return st

    def release_rows(self, block_tables, lengths, free_ids, free_count, refcount, req_idx=None,
                     R=None, stream=None, check=True):
        pool = zp_block_pool(free_ids.data_ptr(), free_count.data_ptr(), refcount.data_ptr(),
                             free_ids.numel())
        if R is None:
            R = req_idx.numel() if req_idx is not None else block_tables.shape[0]
        st = zp_release_rows(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                             block_tables.shape[0], lengths.data_ptr(), _ptr(req_idx), R, pool,
                             _stream(stream))
        if check and st != OK:
            raise ZpError(st, "zp_release_rows")
        return st

    def fork_rows(self, block_tables, lengths, refcount, src_rows, dst_rows, stream=None,
                  check=True):
        st = zp_fork_rows(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                          block_tables.shape[0], lengths.data_ptr(), src_rows.data_ptr(),
                          dst_rows.data_ptr(), src_rows.numel(), refcount.data_ptr(),
                          _stream(stream))
        if check and st != OK:
            raise ZpError(st, "zp_fork_rows")
        return st

    def global_redundancy(self, block_tables, lengths, red_out, req_idx=None, R=None,
                          stream=None, check=True, gram=False):
        """gram=False: zp_global_redundancy (O(T d)); gram=True:
        zp_global_redundancy_gram (the dense Gram on the tensor cores)."""
        if R is None:
            R = req_idx.numel() if req_idx is not None else block_tables.shape[0]
        fn = zp_global_redundancy_gram if gram else zp_global_redundancy
        st = fn(self.handle, block_tables.data_ptr(), block_tables.shape[1],
                block_tables.shape[0], lengths.data_ptr(), _ptr(req_idx), R,
                red_out.data_ptr(), _stream(stream))
        if check and st != OK:
            raise ZpError(st, fn.__name__)
        return st

    def status(self, stream=None) -> int:
        st, dev = zp_cache_status(self.handle, _stream(stream))
        if st != OK:
            raise ZpError(st, "zp_cache_status")
        return dev
