"""The allocation-free placement entry point, against the oracle and the
handle-based one.

place_requests_tp2ep_noalloc serves callers that cannot allocate device
memory (it keeps its scratch in fixed arrays inside the library).  It must
give exactly the oracle's greedy placement (§3.2: longest request first, to
the least-loaded rank) and what place_requests_tp2ep gives, call after call,
and calls after the first on a device must not change how much device memory
is in use.  This file runs last on purpose."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import oracle
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
    orc_owner, orc_local, _ = oracle.place(P, lens, key=list_pos)
    np.testing.assert_array_equal(ref_owner, orc_owner)
    np.testing.assert_array_equal(ref_local, orc_local)
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
        np.testing.assert_array_equal(owner.cpu().numpy(), orc_owner)
        np.testing.assert_array_equal(local.cpu().numpy(), orc_local)


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


_FRESH = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, ".")
import ep_tp_weight_gb300 as umm
import oracle
import synth
torch.cuda.init()
torch.zeros(1, device="cuda")                         # the context exists before anything is measured
R, P = 2048, 8
lens = synth.lengths_lognormal(3, R, 2048, 1.0, 32768)
d_lens = torch.from_numpy(lens.astype(np.int32)).cuda()
owner = torch.empty(R, dtype=torch.int32, device="cuda")
local = torch.empty_like(owner)
status = torch.empty(1, dtype=torch.int32, device="cuda")
torch.cuda.synchronize()
free = [torch.cuda.mem_get_info()[0]]
umm.place_requests_tp2ep_noalloc(P, 0, None, None, None, None)      # the first call on this device: set-up
torch.cuda.synchronize()
free.append(torch.cuda.mem_get_info()[0])
for _ in range(2):
    umm.place_requests_tp2ep_noalloc(P, R, d_lens, None, owner, local, status)
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
want_owner, want_local, _ = oracle.place(P, lens)
ok = (int(status.item()) == 0 and np.array_equal(owner.cpu().numpy(), want_owner)
      and np.array_equal(local.cpu().numpy(), want_local))
print(json.dumps({"free": free, "ok": bool(ok)}))
"""


def test_noalloc_first_call_in_a_fresh_process():
    """In a new process, the first call on the device (here with R = 0) does
    the set-up: it loads the library's placement code and scratch arrays on
    that device, which the CUDA driver may back with device memory.  After
    it, calls take no device memory at all (free memory is unchanged across
    them) and give the oracle's placement."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    got = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    free = got["free"]
    assert got["ok"]
    assert free[2] == free[1] and free[3] == free[1], free
    print(f"set-up call took {free[0] - free[1]} bytes of device memory; later calls took none")
