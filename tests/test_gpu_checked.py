"""The checked build (libumm_checked.so): every vector access of the copy
kernels is tested against the buffer it must lie in and against its
alignment, and a failing one is skipped and raises FLAG_ACCESS.  Here the
parity cases run through it: a result equal to the oracle with no flag shows
that no access left its buffer, at the small sizes and at the full sizes
bench.py times.  Faults are never provoked on the device; the flag's
handling on the host is checked by writing it into the status block."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import test_gpu_fuzz as fuzz
import test_gpu_parity as parity
import test_gpu_scale as scale
from gpu_helpers import DevUMM
from synth.workloads import FULL_SWITCH, TINY, WEIGHTS_H4096

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _checked():
    with umm.checked_library():
        yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", parity.W_CASES, ids=lambda w: w.name)
def test_checked_weights(w):
    parity.test_weights_full_buffer_parity(w, 0)


@pytest.mark.parametrize("w", parity.KV_CASES, ids=lambda w: w.name)
def test_checked_kv(w):
    parity.test_kv_full_buffer_parity(w)


@pytest.mark.parametrize("w", parity.ATTN_CASES, ids=lambda w: w.name)
def test_checked_attention(w):
    parity.test_attn_full_buffer_parity(w)


@pytest.mark.parametrize("seed", [0, 1, 5, 6, 11, 17, 100, 103])
def test_checked_fuzz(seed):
    """Fused and staged paths (odd seeds staged), 1 to 64 ranks."""
    ranks = (24, 32, 48, 64) if seed >= 100 else (1, 2, 3, 4, 6, 8, 16)
    fuzz._fuzz(*fuzz.random_case(seed, ranks=ranks), seed)


def test_checked_full_switch_fullsize():
    scale.test_kv_and_full_switch_fullsize(FULL_SWITCH, False, False)


def test_checked_weights_fullsize():
    scale.test_weights_fullsize(WEIGHTS_H4096)


def test_access_flag_reported_and_cleared():
    """FLAG_ACCESS and FLAG_TIMEOUT (a bounded wait of the TMA copy gave up),
    written into the status block from the host, come back as UMM_ERR_ACCESS
    and UMM_ERR_TIMEOUT ahead of the validation flags and are cleared by the
    read.  They do not roll the KV mode back (the switch ran), while a
    validation flag from the same call does (that switch never ran).  No
    wait is made to time out on the device."""
    from gpu_helpers import i32
    from helpers import initial_kv_state
    st_off = None
    for flags, want_code, want_kv in ((umm.FLAG_ACCESS, umm.UMM_ERR_ACCESS, umm.UMM_MODE_TP),
                                      (umm.FLAG_ACCESS | umm.FLAG_CAPACITY, umm.UMM_ERR_ACCESS, umm.UMM_MODE_EP),
                                      (umm.FLAG_CAPACITY, umm.UMM_ERR_CAPACITY, umm.UMM_MODE_EP),
                                      (umm.FLAG_TIMEOUT, umm.UMM_ERR_TIMEOUT, umm.UMM_MODE_TP),
                                      (umm.FLAG_TIMEOUT | umm.FLAG_CAPACITY, umm.UMM_ERR_TIMEOUT, umm.UMM_MODE_EP),
                                      (umm.FLAG_ACCESS | umm.FLAG_TIMEOUT, umm.UMM_ERR_ACCESS, umm.UMM_MODE_TP)):
        dev = DevUMM(TINY, seed=2)
        st = initial_kv_state(TINY, dev.d, dev.L, seed=2)
        st_off = dev.L["status_off"]
        umm.reshard_kv_ep2tp(dev.h, len(st.lens), st.ep_pt.shape[1], i32(st.lens), i32(st.owner), i32(st.ep_pt),
                             i32(st.tp_pt))
        torch.cuda.synchronize()
        assert umm.umm_get_modes(dev.h)[1] == umm.UMM_MODE_TP
        blk = dev.buf[st_off:st_off + 8].view(torch.int32)
        blk.copy_(torch.tensor([flags, 1], dtype=torch.int32, device="cuda"))   # flags, first failing call
        torch.cuda.synchronize()
        code, f = dev.status()
        assert code == want_code and f == flags
        assert umm.umm_get_modes(dev.h)[1] == want_kv
        assert dev.status() == (0, 0)
        assert np.all(dev.buf[st_off:st_off + 8].cpu().numpy() == 0)
        dev.close()
