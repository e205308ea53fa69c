"""Decode attention against the oracle on more shapes of the request list.

Ragged lengths with empty and one-token requests at three head
configurations (G up to 16), permuted and partial request lists, single
requests and lists of empty ones, an output that is only 2-byte aligned, and
2,100 requests in one call."""
import gc

import numpy as np
import pytest
import torch

from compressed_paged_kv_gb300 import workloads as W
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from compressed_paged_kv_gb300 import _build
    _build.build()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _ragged(R, N, seed, d=128, Hkv=8, Hq=32, zero_frac=0.1):
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name=f"ragged{R}", d=d, Hkv=Hkv, Hq=Hq, N=N, R=R,
                  spare_blocks=8)
    st = W.build_cache(wl, DEV)
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, N * 16 + 1, R)
    lens[rng.random(R) < zero_frac] = 0
    lens[rng.random(R) < 0.05] = 1
    return st, torch.as_tensor(lens, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("d,Hkv,Hq", [(128, 8, 32), (64, 2, 4), (128, 2, 32)])
def test_ragged_many_requests(orc, d, Hkv, Hq):
    st, lens = _ragged(96, 96, 1, d=d, Hkv=Hkv, Hq=Hq)
    H.check_decode(orc, st, 0, lengths=lens)


def test_permuted_partial_rows(orc):
    st, lens = _ragged(80, 64, 2)
    rows = torch.randperm(80, generator=torch.Generator().manual_seed(4))[:53].to(torch.int32)
    H.check_decode(orc, st, 0, rows=rows.to(DEV), lengths=lens)


@pytest.mark.parametrize("lengths", [[1], [16], [17], [2048], [0, 0, 0], [0, 5, 0]])
def test_small_calls(orc, lengths):
    R = len(lengths)
    wl = W.scaled(W.WORKLOADS["qwen3_1l"], name="small", N=128, R=R, spare_blocks=4)
    st = W.build_cache(wl, DEV)
    H.check_decode(orc, st, 0, lengths=torch.tensor(lengths, dtype=torch.int32, device=DEV))


def test_output_on_a_2_byte_boundary(orc):
    st, lens = _ragged(12, 96, 3)  # 96 (request, kv head) pairs: two splits per pair
    H.check_decode(orc, st, 0, lengths=lens, out_offset=1)


def test_2100_requests(orc):
    st, lens = _ragged(2100, 4, 5)
    H.check_decode(orc, st, 0, lengths=lens)
    del st
    gc.collect()
    torch.cuda.empty_cache()
