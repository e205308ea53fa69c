"""Plain fp64 CPU oracle for the Compressed PagedAttention hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and ``--impl reference`` arm) may import
this package.  It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``zp_oracle.c`` (plain loops in double, built with gcc
without fast-math and without FMA contraction).  This module compiles it on
first use and marshals numpy arrays through ctypes.  bf16 tensors are passed
as their raw uint16 bit patterns.

Sources are cited in ``zp_oracle.c``: the two gist.science summaries of
"Zipage: Maintain High Request Concurrency for LLM Reasoning through
Compressed PagedAttention" (Dutch "Methodologie", Korean "방법론") and the
"Paged KV cache and continuous batching for LLMs" concept page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libzp_oracle.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_OUT_OF_BLOCKS = -3
ERR_DEVICE_CHECK = -4

GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle source file into a shared library and return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm", "-lpthread"], check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    return compile_oracle()


def _declare(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.zpo_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.zpo_bf16_to_double.restype = D
    lib.zpo_double_to_bf16.argtypes = [D]
    lib.zpo_double_to_bf16.restype = ctypes.c_uint16
    lib.zpo_double_to_bf16_array.argtypes = [P, P, ctypes.c_long]
    lib.zpo_double_to_bf16_array.restype = None
    lib.zpo_importance.argtypes = [P, P, I, I, I, I, P]
    lib.zpo_importance.restype = None
    lib.zpo_redundancy.argtypes = [P, I, I, I, P]
    lib.zpo_redundancy.restype = None
    lib.zpo_redundancy_global.argtypes = [P, I, I, P]
    lib.zpo_redundancy_global.restype = None
    lib.zpo_unit_scores.argtypes = [P, P, I, I, I, I, I, D, P, P, P]
    lib.zpo_unit_scores.restype = None
    lib.zpo_select.argtypes = [P, I, I, I, P]
    lib.zpo_select.restype = None
    lib.zpo_plan.argtypes = [P, I, P, P, I, I, I, I, I, P, P, I, P, P]
    lib.zpo_plan.restype = I
    lib.zpo_commit.argtypes = [P, I, P, P, I, I, I, P, P, I, P, I]
    lib.zpo_commit.restype = I
    lib.zpo_compress.argtypes = [I, I, I, I, I, I, P, P, P, P, P, I, P, P, I, I, P, I, I, D,
                                 P, P, P, P, P, I]
    lib.zpo_compress.restype = I
    lib.zpo_decode_attn.argtypes = [P, P, P, P, I, P, I, I, I, I, I, I, D, P, P]
    lib.zpo_decode_attn.restype = I
    lib.zpo_plan_prefill.argtypes = [P, I, P, P, I, I, I, I, I, P, P, I, P, P]
    lib.zpo_plan_prefill.restype = I
    lib.zpo_commit_prefill.argtypes = [P, I, P, P, I, I, I, P, P, I, P, I]
    lib.zpo_commit_prefill.restype = I
    lib.zpo_compress_prefill.argtypes = [I, I, I, I, I, I, P, P, P, P, P, I, P, P, I, I, P, I, I,
                                         D, P, P, P, P, P, I]
    lib.zpo_compress_prefill.restype = I
    lib.zpo_alloc_rows.argtypes = [P, I, I, P, P, I, P, I, I, P, P, P, I]
    lib.zpo_alloc_rows.restype = I
    lib.zpo_release_rows.argtypes = [P, I, I, P, P, I, I, P, P, P, I]
    lib.zpo_release_rows.restype = I
    lib.zpo_fork_rows.argtypes = [P, I, I, P, P, P, I, I, P]
    lib.zpo_fork_rows.restype = I
    lib.zpo_append_slots.argtypes = [I, I, I, I, I, P, P, P, I, I, P, P, I, I, P, P, P, I, P, P]
    lib.zpo_append_slots.restype = I
    lib.zpo_append_kv.argtypes = [I, I, I, I, P, P, P, I, I, P, P, I, P, P]
    lib.zpo_append_kv.restype = I
    return lib


def load(path: str | None = None):
    """Load the oracle library (compiling it if needed).  With ``path``, load
    that library instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return Oracle(_declare(ctypes.CDLL(path)))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                compile_oracle()
            _lib = Oracle(_declare(ctypes.CDLL(_LIB_PATH)))
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class Oracle:
    """numpy front end of one loaded oracle library."""

    def __init__(self, lib):
        self.lib = lib

    # -- bf16 ---------------------------------------------------------------
    def bf16_to_f64(self, bits: np.ndarray) -> np.ndarray:
        bits = np.asarray(bits, dtype=np.uint16)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def f64_to_bf16(self, x) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.zpo_double_to_bf16_array(_p(x), _p(out), x.size)
        return out

    # -- unit scoring -------------------------------------------------------
    def importance(self, K, Q, w, G):
        K = _c(K, np.uint16)
        Q = _c(Q, np.uint16)
        T, d = K.shape
        imp = np.zeros(max(T - w, 0), dtype=np.float64)
        self.lib.zpo_importance(_p(K), _p(Q), T, d, w, G, _p(imp))
        return imp

    def redundancy(self, K, b):
        K = _c(K, np.uint16)
        T, d = K.shape
        red = np.zeros(T, dtype=np.float64)
        self.lib.zpo_redundancy(_p(K), T, d, b, _p(red))
        return red

    def redundancy_global(self, K):
        """Mean cosine of each key to every other key of the unit (O(T^2 d))."""
        K = _c(K, np.uint16)
        T, d = K.shape
        red = np.zeros(T, dtype=np.float64)
        self.lib.zpo_redundancy_global(_p(K), T, d, _p(red))
        return red

    def unit_scores(self, K, Q, b, w, G, lam):
        K = _c(K, np.uint16)
        Q = _c(Q, np.uint16)
        T, d = K.shape
        imp = np.zeros(T, dtype=np.float64)
        red = np.zeros(T, dtype=np.float64)
        score = np.zeros(T, dtype=np.float64)
        self.lib.zpo_unit_scores(_p(K), _p(Q), T, d, b, w, G, float(lam), _p(imp), _p(red),
                                 _p(score))
        C = T - w
        return imp[:C].copy(), red, score[:C].copy()

    def select(self, score, w, n_keep):
        score = _c(score, np.float64)
        C = score.shape[0]
        kept = np.zeros(n_keep + w, dtype=np.int32)
        self.lib.zpo_select(_p(score), C, w, n_keep, _p(kept))
        return kept

    # -- block accounting ---------------------------------------------------
    def plan(self, tables, lengths, refcount, free_ids, free_count, N, b, num_blocks,
             req_idx=None, R=None):
        tables = _c(tables, np.int32)
        lengths = _c(lengths, np.int32)
        refcount = _c(refcount, np.int32)
        free_ids = _c(free_ids, np.int32)
        num_rows, stride = tables.shape
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
            R = req_idx.shape[0]
        elif R is None:
            R = num_rows
        dst = np.zeros((max(R, 1), N), dtype=np.int32)
        pops = ctypes.c_int(0)
        st = self.lib.zpo_plan(_p(tables), stride, _p(lengths), _p(req_idx), R, num_rows, N, b,
                               num_blocks, _p(refcount), _p(free_ids), int(free_count), _p(dst),
                               ctypes.byref(pops))
        return st, dst[:R], pops.value

    def commit(self, tables, lengths, refcount, free_ids, free_count, dst, pops, N, b,
               req_idx=None):
        """Applies a plan in place on the given (contiguous int32) arrays."""
        for a in (tables, lengths, refcount, free_ids, dst):
            assert a.dtype == np.int32 and a.flags.c_contiguous
        stride = tables.shape[1]
        R = dst.shape[0]
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
        return self.lib.zpo_commit(_p(tables), stride, _p(lengths), _p(req_idx), R, N, b,
                                   _p(refcount), _p(free_ids), int(free_count), _p(dst), pops)

    # -- whole compression --------------------------------------------------
    def compress(self, kpools, vpools, tables, lengths, window_q, N, w, lam, free_ids,
                 free_count, refcount, Hq, req_idx=None, want_scores=True, want_kept=True,
                 nthreads=None):
        """Runs the whole compression on host copies.

        kpools/vpools: list of L uint16 arrays [num_blocks][Hkv][b][d] (read only).
        Returns dict(status, kpools, vpools, tables, lengths, free_ids, free_count,
        refcount, scores [L][R][Hkv][T], kept [L][R][Hkv][(N-1)b]).
        """
        L = len(kpools)
        num_blocks, Hkv, b, d = kpools[0].shape
        kin = [_c(k, np.uint16) for k in kpools]
        vin = [_c(v, np.uint16) for v in vpools]
        kout = [k.copy() for k in kin]
        vout = [v.copy() for v in vin]
        tables = _c(tables, np.int32).copy()
        lengths = _c(lengths, np.int32).copy()
        free_ids = _c(free_ids, np.int32).copy()
        refcount = _c(refcount, np.int32).copy()
        window_q = _c(window_q, np.uint16)
        num_rows, stride = tables.shape
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
            R = req_idx.shape[0]
        else:
            R = num_rows
        T = N * b
        scores = np.zeros((L, R, Hkv, T), dtype=np.float64) if want_scores else None
        kept = np.zeros((L, R, Hkv, (N - 1) * b), dtype=np.int32) if want_kept else None
        arr = ctypes.c_void_p * L
        kp = arr(*[k.ctypes.data for k in kin])
        vp = arr(*[v.ctypes.data for v in vin])
        ko = arr(*[k.ctypes.data for k in kout])
        vo = arr(*[v.ctypes.data for v in vout])
        fc = ctypes.c_int32(int(free_count))
        nthreads = nthreads or os.cpu_count() or 1
        st = self.lib.zpo_compress(L, Hkv, Hq, d, b, num_blocks, kp, vp, ko, vo, _p(tables),
                                   stride, _p(lengths), _p(req_idx), R, num_rows, _p(window_q),
                                   N, w, float(lam), _p(free_ids), ctypes.byref(fc),
                                   _p(refcount), _p(scores), _p(kept), int(nthreads))
        return dict(status=st, kpools=kout, vpools=vout, tables=tables, lengths=lengths,
                    free_ids=free_ids, free_count=fc.value, refcount=refcount, scores=scores,
                    kept=kept)

    def compress_prefill(self, kpools, vpools, tables, lengths, window_q, N, w, lam, free_ids,
                         free_count, refcount, Hq, req_idx=None, want_scores=True,
                         want_kept=True, nthreads=None):
        """Compression at admission on host copies (lengths >= N*b).

        Same inputs and dict as ``compress``; scores are [L][R][Hkv][stride*b]
        with NaN where nothing is written (positions at and beyond a request's
        length)."""
        L = len(kpools)
        num_blocks, Hkv, b, d = kpools[0].shape
        kin = [_c(k, np.uint16) for k in kpools]
        vin = [_c(v, np.uint16) for v in vpools]
        kout = [k.copy() for k in kin]
        vout = [v.copy() for v in vin]
        tables = _c(tables, np.int32).copy()
        lengths = _c(lengths, np.int32).copy()
        free_ids = _c(free_ids, np.int32).copy()
        refcount = _c(refcount, np.int32).copy()
        window_q = _c(window_q, np.uint16)
        num_rows, stride = tables.shape
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
            R = req_idx.shape[0]
        else:
            R = num_rows
        scores = (np.full((L, R, Hkv, stride * b), np.nan, dtype=np.float64)
                  if want_scores else None)
        kept = np.zeros((L, R, Hkv, (N - 1) * b), dtype=np.int32) if want_kept else None
        arr = ctypes.c_void_p * L
        kp = arr(*[k.ctypes.data for k in kin])
        vp = arr(*[v.ctypes.data for v in vin])
        ko = arr(*[k.ctypes.data for k in kout])
        vo = arr(*[v.ctypes.data for v in vout])
        fc = ctypes.c_int32(int(free_count))
        nthreads = nthreads or os.cpu_count() or 1
        st = self.lib.zpo_compress_prefill(L, Hkv, Hq, d, b, num_blocks, kp, vp, ko, vo,
                                           _p(tables), stride, _p(lengths), _p(req_idx), R,
                                           num_rows, _p(window_q), N, w, float(lam),
                                           _p(free_ids), ctypes.byref(fc), _p(refcount),
                                           _p(scores), _p(kept), int(nthreads))
        return dict(status=st, kpools=kout, vpools=vout, tables=tables, lengths=lengths,
                    free_ids=free_ids, free_count=fc.value, refcount=refcount, scores=scores,
                    kept=kept)

    # -- decode attention ---------------------------------------------------
    def decode_attn(self, q, kpool, vpool, tables, lengths, scale):
        q = _c(q, np.uint16)
        kpool = _c(kpool, np.uint16)
        vpool = _c(vpool, np.uint16)
        tables = _c(tables, np.int32)
        lengths = _c(lengths, np.int32)
        R, Hq, d = q.shape
        num_blocks, Hkv, b, _ = kpool.shape
        stride = tables.shape[1]
        out64 = np.zeros((R, Hq, d), dtype=np.float64)
        out16 = np.zeros((R, Hq, d), dtype=np.uint16)
        st = self.lib.zpo_decode_attn(_p(q), _p(kpool), _p(vpool), _p(tables), stride,
                                      _p(lengths), R, Hq, Hkv, d, b, num_blocks, float(scale),
                                      _p(out64), _p(out16))
        return st, out64, out16

    # -- decode-side append ---------------------------------------------------
    def append_slots(self, kpools, vpools, tables, lengths, free_ids, free_count, refcount,
                     n_max, req_idx=None):
        """Reserves each listed request's next slot on host copies.

        Returns dict(status, kpools, vpools, tables, lengths, free_ids,
        free_count, refcount, triggers) -- the inputs unchanged when status != 0.
        """
        L = len(kpools)
        num_blocks, Hkv, b, d = kpools[0].shape
        kout = [_c(k, np.uint16).copy() for k in kpools]
        vout = [_c(v, np.uint16).copy() for v in vpools]
        tables = _c(tables, np.int32).copy()
        lengths = _c(lengths, np.int32).copy()
        free_ids = _c(free_ids, np.int32).copy()
        refcount = _c(refcount, np.int32).copy()
        num_rows, stride = tables.shape
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
            R = req_idx.shape[0]
        else:
            R = num_rows
        arr = ctypes.c_void_p * L
        kp = arr(*[k.ctypes.data for k in kout])
        vp = arr(*[v.ctypes.data for v in vout])
        fc = ctypes.c_int32(int(free_count))
        trig = np.zeros(max(R, 1), dtype=np.int32)
        nt = ctypes.c_int32(0)
        st = self.lib.zpo_append_slots(L, Hkv, d, b, num_blocks, kp, vp, _p(tables), stride,
                                       num_rows, _p(lengths), _p(req_idx), R, int(n_max),
                                       _p(refcount), _p(free_ids), ctypes.byref(fc),
                                       free_ids.shape[0], _p(trig), ctypes.byref(nt))
        return dict(status=st, kpools=kout, vpools=vout, tables=tables, lengths=lengths,
                    free_ids=free_ids, free_count=fc.value, refcount=refcount,
                    triggers=trig[:nt.value].copy())

    def append_kv(self, kpool, vpool, tables, lengths, k_new, v_new, req_idx=None):
        """Writes one layer's new-token rows into copies of its pools; returns
        (status, kpool, vpool)."""
        kpool = _c(kpool, np.uint16).copy()
        vpool = _c(vpool, np.uint16).copy()
        tables = _c(tables, np.int32)
        lengths = _c(lengths, np.int32)
        k_new = _c(k_new, np.uint16)
        v_new = _c(v_new, np.uint16)
        num_blocks, Hkv, b, d = kpool.shape
        num_rows, stride = tables.shape
        R = k_new.shape[0]
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
        st = self.lib.zpo_append_kv(Hkv, d, b, num_blocks, _p(kpool), _p(vpool), _p(tables),
                                    stride, num_rows, _p(lengths), _p(req_idx), R, _p(k_new),
                                    _p(v_new))
        return st, kpool, vpool

    # -- whole-request allocation and release ---------------------------------
    def _ints(self, tables, lengths, free_ids, refcount, req_idx):
        tables = _c(tables, np.int32).copy()
        lengths = _c(lengths, np.int32).copy()
        free_ids = _c(free_ids, np.int32).copy()
        refcount = _c(refcount, np.int32).copy()
        if req_idx is not None:
            req_idx = _c(req_idx, np.int32)
        return tables, lengths, free_ids, refcount, req_idx

    def alloc_rows(self, tables, lengths, free_ids, free_count, refcount, counts, b,
                   req_idx=None):
        """Blocks for the first counts[i] tokens of empty rows; returns dict
        (status, tables, lengths, free_ids, free_count, refcount) of copies."""
        tables, lengths, free_ids, refcount, req_idx = self._ints(tables, lengths, free_ids,
                                                                  refcount, req_idx)
        counts = _c(counts, np.int32)
        num_rows, stride = tables.shape
        fc = ctypes.c_int32(int(free_count))
        st = self.lib.zpo_alloc_rows(_p(tables), stride, num_rows, _p(lengths), _p(req_idx),
                                     counts.shape[0], _p(counts), b, refcount.shape[0],
                                     _p(refcount), _p(free_ids), ctypes.byref(fc),
                                     free_ids.shape[0])
        return dict(status=st, tables=tables, lengths=lengths, free_ids=free_ids,
                    free_count=fc.value, refcount=refcount)

    def release_rows(self, tables, lengths, free_ids, free_count, refcount, req_idx=None, R=None):
        """Every block of the listed rows back to the pool; dict as alloc_rows."""
        tables, lengths, free_ids, refcount, req_idx = self._ints(tables, lengths, free_ids,
                                                                  refcount, req_idx)
        num_rows, stride = tables.shape
        if R is None:
            R = req_idx.shape[0] if req_idx is not None else num_rows
        fc = ctypes.c_int32(int(free_count))
        st = self.lib.zpo_release_rows(_p(tables), stride, num_rows, _p(lengths), _p(req_idx), R,
                                       refcount.shape[0], _p(refcount), _p(free_ids),
                                       ctypes.byref(fc), free_ids.shape[0])
        return dict(status=st, tables=tables, lengths=lengths, free_ids=free_ids,
                    free_count=fc.value, refcount=refcount)

    def fork_rows(self, tables, lengths, refcount, src, dst):
        """Rows dst[i] become copies of rows src[i] sharing their blocks;
        dict(status, tables, lengths, refcount) of copies."""
        tables = _c(tables, np.int32).copy()
        lengths = _c(lengths, np.int32).copy()
        refcount = _c(refcount, np.int32).copy()
        src = _c(src, np.int32)
        dst = _c(dst, np.int32)
        num_rows, stride = tables.shape
        st = self.lib.zpo_fork_rows(_p(tables), stride, num_rows, _p(lengths), _p(src), _p(dst),
                                    src.shape[0], refcount.shape[0], _p(refcount))
        return dict(status=st, tables=tables, lengths=lengths, refcount=refcount)
