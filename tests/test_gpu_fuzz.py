"""Randomised parity of the CUDA path with the oracle: random rank counts,
expert and hidden sizes (including sizes that force 8-, 4- and 2-byte
vectors), head ratios, page sizes and request mixes (zero lengths, exact
page multiples, one-token requests), through the fused, staged and
attention entry points, whole buffers compared, both directions."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import oracle
import synth
from gpu_helpers import DevUMM, i32
from helpers import dims_of
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


def random_case(seed: int, ranks=(1, 2, 3, 4, 6, 8, 16)):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice(ranks))
    N = int(rng.integers(1, 4))
    E = P * int(rng.integers(1, 4))
    I = P * int(rng.integers(1, 7))
    H = int(rng.integers(1, 70))
    if rng.random() < 0.5:
        Hkv = P * int(rng.choice([1, 2, 4]))            # Hkv >= P
    else:
        divs = [h for h in range(1, P + 1) if P % h == 0]
        Hkv = int(rng.choice(divs))                      # Hkv <= P, a divisor
    D = int(rng.integers(1, 20))
    ps = int(rng.integers(1, 33))
    R = int(rng.integers(0, 40 if P <= 16 else 12))
    Hq = P * int(rng.integers(1, 4)) if rng.random() < 0.6 else 0
    len_b = int(rng.integers(1, (5 if P <= 16 else 2) * ps + 2))
    return rng, Workload(f"fuzz{seed}", P=P, N=N, E=E, H=H, I=I, Hkv=Hkv, D=D, ps=ps, R=max(R, 1),
                         len_kind="uniform", len_a=0, len_b=len_b, slack=1.0 + P, Hq=Hq), R


def pool_pages(w: Workload, R: int) -> int:
    """A TP pool large enough that every EP rank could hold all live pages."""
    m = w.Hkv // w.h_tp
    total = R * ((int(w.len_b) + w.ps - 1) // w.ps) + 1
    return m * total


def kv_state(rng, w: Workload, d, L: dict, R: int):
    """Random lengths (with zeros and exact multiples), greedy owners, random pages."""
    lens = rng.integers(0, int(w.len_b) + 1, R).astype(np.int32)
    if R > 2:
        lens[0] = 0
        lens[1] = w.ps * max(1, int(w.len_b) // w.ps)
    maxp = max(1, int(np.ceil(max(1, int(lens.max()) if R else 1) / w.ps)))
    owner, _, _ = oracle.place(w.P, lens)
    free_ep = synth.permutation(int(rng.integers(1 << 30)), 2, L["pages_ep"], rows=w.P)
    fl, ep_pt = oracle.assign_pages(w.P, lens, w.ps, maxp, free_ep, region=owner)
    pos = oracle.request_order(w.P, owner)
    fl2, tp_pt = oracle.assign_pages(1, lens, w.ps, maxp, synth.permutation(int(rng.integers(1 << 30)), 3,
                                                                             L["pages_tp"]), key=pos)
    owner2, _, _ = oracle.place(w.P, lens, key=pos)
    fl3, ep_pt2 = oracle.assign_pages(w.P, lens, w.ps, maxp, synth.permutation(int(rng.integers(1 << 30)), 4,
                                                                               L["pages_ep"], w.P),
                                      region=owner2, key=pos)
    ok = fl == 0 and fl2 == 0 and fl3 == 0
    return ok, lens, maxp, owner, ep_pt, tp_pt, owner2, ep_pt2


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_parity(seed):
    _fuzz(*random_case(seed), seed)


@pytest.mark.parametrize("seed", range(100, 106))
def test_fuzz_parity_wide_rank_counts(seed):
    """24 to 64 ranks: group scans and counts over up to 64 groups, one region
    per rank."""
    _fuzz(*random_case(seed, ranks=(24, 32, 48, 64)), seed)


def _fuzz(rng, w, R, seed):
    ptp = pool_pages(w, R)
    dev = DevUMM(w, seed=seed, pages_tp=ptp, max_requests=R, max_pages=ptp)
    L, d = dev.L, dev.d
    staged = bool(seed % 2)
    ok, lens, maxp, owner, ep_pt, tp_pt, owner2, ep_pt2 = kv_state(rng, w, d, L, R)
    assert ok
    ref = dev.host()
    g = i32
    stage_w = torch.empty(umm.umm_weights_stage_bytes(dev.h), dtype=torch.uint8, device="cuda")
    stage_k = torch.empty(umm.umm_kv_stage_bytes(dev.h), dtype=torch.uint8, device="cuda")
    # EP -> TP
    if staged:
        umm.reshard_weights_ep2tp_staged(dev.h, stage_w, stage_w.numel())
        umm.reshard_kv_ep2tp_staged(dev.h, stage_k, stage_k.numel(), R, maxp, g(lens), g(owner), g(ep_pt), g(tp_pt))
    else:
        umm.reshard_weights_ep2tp(dev.h)
        umm.reshard_kv_ep2tp(dev.h, R, maxp, g(lens), g(owner), g(ep_pt), g(tp_pt))
    if w.Hq:
        umm.reshard_attn_ep2tp(dev.h)
        oracle.attn_ep2tp(ref, d)
    oracle.weights_ep2tp(ref, d)
    assert oracle.kv_ep2tp(ref, d, lens, owner, ep_pt, tp_pt) == 0
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    # TP -> EP
    if staged:
        umm.reshard_weights_tp2ep_staged(dev.h, stage_w, stage_w.numel())
        umm.reshard_kv_tp2ep_staged(dev.h, stage_k, stage_k.numel(), R, maxp, g(lens), g(owner2), g(ep_pt2),
                                    g(tp_pt))
    else:
        umm.reshard_weights_tp2ep(dev.h)
        umm.reshard_kv_tp2ep(dev.h, R, maxp, g(lens), g(owner2), g(ep_pt2), g(tp_pt))
    if w.Hq:
        umm.reshard_attn_tp2ep(dev.h)
        oracle.attn_tp2ep(ref, d)
    oracle.weights_tp2ep(ref, d)
    assert oracle.kv_tp2ep(ref, d, lens, owner2, ep_pt2, tp_pt) == 0
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


def _code_of(flags: int) -> int:
    """The status a set of flags reports (highest first: bad request, capacity,
    page out of range, duplicate page), as include/umm.h documents."""
    for bit, code in ((oracle.F_BAD_REQUEST, umm.UMM_ERR_BAD_REQUEST), (oracle.F_CAPACITY, umm.UMM_ERR_CAPACITY),
                      (oracle.F_PAGE_OOB, umm.UMM_ERR_PAGE_OOB), (oracle.F_DUP_PAGE, umm.UMM_ERR_DUP_PAGE)):
        if flags & bit:
            return code
    return umm.UMM_OK


def _live(lens, ps):
    return [(k, p) for k in range(len(lens)) for p in range((int(lens[k]) + ps - 1) // ps)]


@pytest.mark.parametrize("seed", range(20))
def test_fuzz_invalid_metadata_is_refused(seed):
    """One to three random corruptions of a valid KV call (bad lengths or
    owners, page ids out of range, a destination or TP source page used twice):
    the device raises exactly the oracle's validation flags, writes nothing, and
    the handle works again after the status read."""
    rng = np.random.default_rng(5000 + seed)
    P = int(rng.choice([2, 3, 4, 8]))
    Hkv = int(rng.choice([h for h in (1, 2, 4, 8, 16) if h % P == 0 or P % h == 0]))
    w = Workload(f"bad{seed}", P=P, N=2, Hkv=Hkv, D=int(rng.choice([4, 8, 16])), ps=int(rng.integers(2, 9)),
                 R=int(rng.integers(4, 20)), len_kind="uniform", len_a=1, len_b=40, slack=1.0 + P)
    R = w.R
    ptp = pool_pages(w, R)
    dev = DevUMM(w, seed=seed, pages_tp=ptp, max_requests=R, max_pages=ptp)
    d, L = dev.d, dev.L
    ok, lens, maxp, owner, ep_pt, tp_pt, owner2, ep_pt2 = kv_state(rng, w, d, L, R)
    assert ok
    direction = int(rng.integers(2))
    a = {"lens": lens.copy(), "owner": (owner if direction == 0 else owner2).copy(),
         "ep_pt": (ep_pt if direction == 0 else ep_pt2).copy(), "tp_pt": tp_pt.copy()}
    live = _live(lens, w.ps)
    kinds = ["neg_len", "long_len", "bad_owner", "ep_oob", "tp_oob", "dup_dst"] + (["dup_tp"] if direction else [])
    for kind in rng.choice(kinds, size=int(rng.integers(1, 4))):
        k = int(rng.integers(R))
        if kind == "neg_len":
            a["lens"][k] = -int(rng.integers(1, 5))
        elif kind == "long_len":
            a["lens"][k] = maxp * w.ps + int(rng.integers(1, 5))
        elif kind == "bad_owner":
            a["owner"][k] = int(rng.choice([-1, P, P + 3]))
        elif kind in ("ep_oob", "tp_oob") and live:
            kk, p = live[int(rng.integers(len(live)))]
            pool = L["pages_ep"] if kind == "ep_oob" else L["pages_tp"]
            a["ep_pt" if kind == "ep_oob" else "tp_pt"][kk, p] = int(rng.choice([-1, pool, pool + 7]))
        elif kind in ("dup_dst", "dup_tp") and len(live) > 1:
            i, j = rng.choice(len(live), size=2, replace=False)
            (k1, p1), (k2, p2) = live[int(i)], live[int(j)]
            if kind == "dup_tp" or direction == 0:
                a["tp_pt"][k2, p2] = a["tp_pt"][k1, p1]
            elif a["owner"][k1] == a["owner"][k2]:
                a["ep_pt"][k2, p2] = a["ep_pt"][k1, p1]
    want = oracle.kv_validate(d, direction, a["lens"], a["owner"], a["ep_pt"], a["tp_pt"])
    ref = dev.host()
    if direction == 1:
        umm.umm_set_modes(dev.h, umm.UMM_MODE_EP, umm.UMM_MODE_TP)
    fn = umm.reshard_kv_ep2tp if direction == 0 else umm.reshard_kv_tp2ep
    fn(dev.h, R, maxp, i32(a["lens"]), i32(a["owner"]), i32(a["ep_pt"]), i32(a["tp_pt"]))
    assert dev.status() == (_code_of(want), want)
    assert dev.status() == (0, 0)
    if want:
        # refused: nothing written, and the KV mode is back to the call's source
        np.testing.assert_array_equal(dev.host(), ref)
        assert umm.umm_get_modes(dev.h)[1] == (umm.UMM_MODE_TP if direction else umm.UMM_MODE_EP)
        # the handle works again: the valid call of the same direction
        owner_ok = owner if direction == 0 else owner2
        ep_ok = ep_pt if direction == 0 else ep_pt2
        fn(dev.h, R, maxp, i32(lens), i32(owner_ok), i32(ep_ok), i32(tp_pt))
        (oracle.kv_ep2tp if direction == 0 else oracle.kv_tp2ep)(ref, d, lens, owner_ok, ep_ok, tp_pt)
        assert dev.status() == (0, 0)
        np.testing.assert_array_equal(dev.host(), ref)
    dev.close()
