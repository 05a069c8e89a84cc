"""The allocation-free placement entry point, against the handle-based one.

place_requests_tp2ep_noalloc serves callers that cannot allocate device
memory (it keeps its scratch in a fixed array inside the library).  It must
give exactly what place_requests_tp2ep gives, call after call, and must not
change how much device memory is in use.  This file runs last on purpose."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import synth
from gpu_helpers import DevUMM, i32
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


def _reference(P, lens, list_pos):
    R = len(lens)
    w = Workload("place_ref", P=P, N=1, Hkv=P, D=8, ps=16, R=R, len_a=1, len_b=1)
    dev = DevUMM(w, fill=False, pages_tp=P, max_requests=R, max_pages=P)
    owner = torch.empty(R, dtype=torch.int32, device="cuda")
    local = torch.empty_like(owner)
    umm.place_requests_tp2ep(dev.h, R, i32(lens), None if list_pos is None else i32(list_pos), owner, local)
    assert umm.umm_status_sync(dev.h) == (0, 0)
    out = owner.cpu().numpy(), local.cpu().numpy()
    dev.close()
    return out


@pytest.mark.parametrize("P,R,keyed", [(8, 2048, True), (3, 17, False), (64, 300, True), (5, 16384, True)])
def test_noalloc_placement_equals_handle_placement_twice(P, R, keyed):
    rng = np.random.default_rng(P + R)
    lens = synth.lengths_lognormal(7, R, 2048, 1.0, 32768)
    lens[rng.integers(0, R, max(1, R // 8))] = 99           # ties
    list_pos = rng.permutation(R).astype(np.int32) if keyed else None
    ref_owner, ref_local = _reference(P, lens, list_pos)
    d_lens, d_pos = i32(lens), (None if list_pos is None else i32(list_pos))
    owner = torch.full((R,), -5, dtype=torch.int32, device="cuda")
    local = torch.full((R,), -5, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):                                    # the scratch is reused by the second call
        owner.fill_(-5)
        local.fill_(-5)
        status.fill_(-1)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        umm.place_requests_tp2ep_noalloc(P, R, d_lens, d_pos, owner, local, status)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert int(status.item()) == umm.UMM_OK
        np.testing.assert_array_equal(owner.cpu().numpy(), ref_owner)
        np.testing.assert_array_equal(local.cpu().numpy(), ref_local)


def test_noalloc_placement_limits_and_bad_input():
    with pytest.raises(umm.UmmError) as ei:
        umm.place_requests_tp2ep_noalloc(8, 16385, 1, None, 1, 1)
    assert ei.value.code == umm.UMM_ERR_CAPACITY
    with pytest.raises(umm.UmmError) as ei:
        umm.place_requests_tp2ep_noalloc(65, 10, 1, None, 1, 1)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    lens = i32([5, -1, 3])
    owner = torch.full((3,), -5, dtype=torch.int32, device="cuda")
    local = torch.full((3,), -5, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    umm.place_requests_tp2ep_noalloc(2, 3, lens, None, owner, local, status)
    torch.cuda.synchronize()
    assert int(status.item()) == umm.UMM_ERR_BAD_REQUEST
    assert (owner.cpu() == -5).all() and (local.cpu() == -5).all()
    umm.place_requests_tp2ep_noalloc(2, 3, i32([5, 1, 3]), i32([0, 0, 1]), owner, local, status)
    torch.cuda.synchronize()
    assert int(status.item()) == umm.UMM_ERR_BAD_REQUEST
