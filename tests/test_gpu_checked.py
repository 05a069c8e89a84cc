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


@pytest.mark.parametrize("N", [2, 3])
def test_tma_wait_runs_out_on_the_device(N):
    """The bounded mbarrier wait of the TMA KV copy, made to run out on the
    GPU (checked-build hook umm_test_stall_tma_wait): every CTA of the call's
    last layer, after its tensor loads have landed, waits on a barrier that
    never completes, gives up after 64 polls and takes the timeout exit with
    no copy in flight.  Then:
      - umm_status_sync reports UMM_ERR_TIMEOUT (flag TIMEOUT only), and the
        KV mode stays TP (the call ran, incomplete);
      - a validating kernel enqueued after the call did nothing;
      - exactly the earlier layers were copied: the buffer equals its initial
        contents with the TP slots of those layers taken from the oracle's
        complete EP->TP, and nothing else written;
      - the handle recovers: once the flag is read, a new EP->TP call (the
        cache rebuilt first when a copied layer overwrote an EP slot) equals
        the oracle."""
    from gpu_helpers import fill_device, i32
    from helpers import initial_kv_state, kvslot
    import oracle
    w = TINY.with_(N=N)
    dev = DevUMM(w, seed=4)
    assert umm.umm_kv_copy_kernel(dev.dims, 0)[0] == umm.UMM_KV_COPY_TMA
    st = initial_kv_state(w, dev.d, dev.L, seed=4)
    R, maxp = len(st.lens), st.ep_pt.shape[1]
    args = (R, maxp, i32(st.lens), i32(st.owner), i32(st.ep_pt), i32(st.tp_pt))
    ref0 = dev.host()
    full = ref0.copy()
    assert oracle.kv_ep2tp(full, dev.d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    L, d = dev.L, dev.d
    umm.umm_test_stall_tma_wait(dev.h, N - 1, 64)
    umm.reshard_kv_ep2tp(dev.h, *args)
    tp_pos = torch.full((R,), -3, dtype=torch.int32, device="cuda")
    umm.gather_requests_ep2tp(dev.h, R, i32(st.owner), tp_pos)
    torch.cuda.synchronize()
    assert dev.status() == (umm.UMM_ERR_TIMEOUT, umm.FLAG_TIMEOUT)
    assert umm.umm_get_modes(dev.h)[1] == umm.UMM_MODE_TP
    assert (tp_pos.cpu() == -3).all()
    want = ref0.copy()
    for q in range(d.P):
        for layer in range(N - 1):
            a = kvslot(L, q, layer, 0)
            want[a:a + L["kvslot_stride"]] = full[a:a + L["kvslot_stride"]]
    np.testing.assert_array_equal(dev.host(), want)
    # recovery: the hook off, the flag read; the cache rebuilt when a copied
    # layer (l >= 1) overwrote EP slot l, then EP->TP again
    umm.umm_test_stall_tma_wait(dev.h, -1, 0)
    assert dev.status() == (0, 0)
    if N > 2:
        fill_device(dev.buf, L, w, 4)
    umm.umm_set_modes(dev.h, umm.UMM_MODE_EP, umm.UMM_MODE_EP)
    umm.reshard_kv_ep2tp(dev.h, *args)
    torch.cuda.synchronize()
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), full)
    dev.close()


def test_tma_wait_hook_range():
    dev = DevUMM(TINY, seed=4, fill=False)
    for bad in (-2, TINY.N):
        with pytest.raises(umm.UmmError) as ei:
            umm.umm_test_stall_tma_wait(dev.h, bad, 64)
        assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    umm.umm_test_stall_tma_wait(dev.h, 0, 0)       # polls 0: off
    dev.close()
