"""Parity at the full workload sizes, in the launch configuration bench.py
times (same entry points, same sequence, same grid sizing).  The oracle
cannot hold these buffers, so outputs are checked (a) on random samples the
oracle maps one by one (its element maps + the generator's value at the
source), (b) whole, against properties that hold at any size: the TP shards
equal torch slices of the full EP tensors (§3.1 shapes), the EP->TP->EP
round trip is the identity (weights), and every live KV row of a few whole
requests, and (c) bytes outside every destination keep their contents."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import oracle
import synth
from gpu_helpers import DevUMM, i32
from helpers import attnslot, heads_of_rank
from synth.workloads import ATTN_QWEN3_SHAPE, FULL_SWITCH, KV_256REQ, TINY, WEIGHTS_H2048, WEIGHTS_H4096

pytestmark = pytest.mark.gpu

SAMPLES = 200_000


def _expect(dev: DevUMM, idx_u16: np.ndarray, kv: bool) -> np.ndarray:
    mode, sigma = dev.w.kv_mode() if kv else dev.w.w_mode()
    return synth.values_at(dev.seed, idx_u16.astype(np.uint64), mode, sigma).view(np.int16)


def _gather(dev: DevUMM, idx_u16: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(idx_u16.astype(np.int64)).cuda()
    return dev.u16()[t].cpu().numpy()


def _regen(dev: DevUMM, off_bytes: int, nbytes: int, kv: bool) -> torch.Tensor:
    """Initial contents of a byte range, regenerated on the device."""
    out = torch.empty(nbytes // 2, dtype=torch.int16, device="cuda")
    mode, sigma = dev.w.kv_mode() if kv else dev.w.w_mode()
    from gpu_helpers import table_dev
    synth.fill_device(out.data_ptr(), nbytes // 2, dev.seed, mode,
                      table_dev(sigma).data_ptr() if mode else 0, base=off_bytes // 2)
    return out


# ------------------------------------------------------------------ weights

def _check_weights_ep2tp(dev: DevUMM, rng):
    w, d, L = dev.w, dev.d, dev.L
    El, Ip = w.E // w.P, w.I // w.P
    # (a) sampled element maps from the oracle
    for part in ("w13", "w2"):
        n = SAMPLES // 2
        q = rng.integers(0, w.P, n)
        e = rng.integers(0, w.E, n)
        layer = rng.integers(0, w.N, n)
        src = np.empty(n, np.int64)
        dst = np.empty(n, np.int64)
        if part == "w13":
            row = rng.integers(0, 2 * Ip, n)
            h = rng.integers(0, w.H, n)
            for i in range(n):
                src[i], dst[i] = oracle.w13_tp_elem(d, int(q[i]), int(e[i]), int(row[i]), int(h[i]),
                                                    int(layer[i]) + 1, int(layer[i]))
        else:
            h = rng.integers(0, w.H, n)
            c = rng.integers(0, Ip, n)
            for i in range(n):
                src[i], dst[i] = oracle.w2_tp_elem(d, int(q[i]), int(e[i]), int(h[i]), int(c[i]),
                                                   int(layer[i]) + 1, int(layer[i]))
        np.testing.assert_array_equal(_gather(dev, dst // 2), _expect(dev, src // 2, False))
    # (b) whole layers against torch slices of the full EP tensors
    u = dev.u16()
    for layer in range(w.N):
        w13 = []
        w2 = []
        for r in range(w.P):
            base = r * L["region_stride"] + (layer + 1) * L["wslot_stride"]
            w13.append(_regen(dev, base + L["w13_off"], El * 2 * w.I * w.H * 2, False).view(El, 2 * w.I, w.H))
            w2.append(_regen(dev, base + L["w2_off"], El * w.H * w.I * 2, False).view(El, w.H, w.I))
        f13 = torch.cat(w13)
        f2 = torch.cat(w2)
        del w13, w2
        for q in range(w.P):
            base = (q * L["region_stride"] + layer * L["wslot_stride"]) // 2
            tp13 = u[base + L["w13_off"] // 2: base + L["w13_off"] // 2 + w.E * 2 * Ip * w.H].view(w.E, 2 * Ip, w.H)
            tp2 = u[base + L["w2_off"] // 2: base + L["w2_off"] // 2 + w.E * w.H * Ip].view(w.E, w.H, Ip)
            want13 = torch.cat([f13[:, q * Ip:(q + 1) * Ip], f13[:, w.I + q * Ip:w.I + (q + 1) * Ip]], dim=1)
            assert torch.equal(tp13, want13), (layer, q)
            assert torch.equal(tp2, f2[:, :, q * Ip:(q + 1) * Ip]), (layer, q)
        del f13, f2


def _check_weights_round_trip(dev: DevUMM):
    w, L = dev.w, dev.L
    for r in range(w.P):
        for s in range(1, w.N + 1):
            base = r * L["region_stride"] + s * L["wslot_stride"]
            n = L["wslot_stride"]
            got = dev.u16()[base // 2:(base + n) // 2]
            assert torch.equal(got, _regen(dev, base, n, False)), (r, s)


@pytest.mark.parametrize("w", [WEIGHTS_H2048, WEIGHTS_H4096], ids=lambda w: w.name)
def test_weights_fullsize(w):
    dev = DevUMM(w, seed=21)
    rng = np.random.default_rng(0)
    umm.umm_switch_ep2tp(dev.h, 0, 1, None, None, None, None, 0, None, None)    # as bench.py, no requests
    torch.cuda.synchronize()
    _check_weights_ep2tp(dev, rng)
    # slot N is not a destination of EP->TP: untouched
    L = dev.L
    for r in range(w.P):
        base = r * L["region_stride"] + w.N * L["wslot_stride"]
        assert torch.equal(dev.u16()[base // 2:(base + L["wslot_stride"]) // 2],
                           _regen(dev, base, L["wslot_stride"], False))
    umm.umm_switch_tp2ep(dev.h, 0, 1, None, None, None, None, 0, 0, None, None, None)
    torch.cuda.synchronize()
    _check_weights_round_trip(dev)
    dev.close()


# ------------------------------------------------------------------ KV, in the bench's call sequence

class KVRun:
    """The bench's EP->TP->EP KV sequence on the device, with the oracle's
    metadata computed beside it."""

    def __init__(self, dev: DevUMM):
        w, d, L = dev.w, dev.d, dev.L
        self.dev = dev
        self.lens = w.lengths()
        self.R = len(self.lens)
        self.maxp = w.max_pages_per_req()
        P = w.P
        self.owner0, _, _ = oracle.place(P, self.lens)
        self.ep_free = synth.permutation(w.seed, 2, L["pages_ep"], rows=P)
        _, self.ep_pt0 = oracle.assign_pages(P, self.lens, w.ps, self.maxp, self.ep_free, region=self.owner0)
        self.tp_free = synth.permutation(w.seed, 3, L["pages_tp"], rows=1)
        self.pos = oracle.request_order(P, self.owner0)
        _, self.tp_pt = oracle.assign_pages(1, self.lens, w.ps, self.maxp, self.tp_free, key=self.pos)
        self.owner1, self.local1, _ = oracle.place(P, self.lens, key=self.pos)
        _, self.ep_pt1 = oracle.assign_pages(P, self.lens, w.ps, self.maxp, self.ep_free, region=self.owner1,
                                             key=self.pos)

    def ep2tp(self, switch: bool = False):
        """switch=True: one umm_switch_ep2tp call (weights and attention too),
        exactly as bench.py times it; else the separate KV entry points."""
        dev, R, maxp = self.dev, self.R, self.maxp
        h, L = dev.h, dev.L
        self.d_lens = i32(self.lens)
        self.d_owner0 = i32(self.owner0)
        self.d_tp_pos = torch.empty(R, dtype=torch.int32, device="cuda")
        self.d_tp_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
        if switch:
            umm.umm_switch_ep2tp(h, R, maxp, self.d_lens, self.d_owner0, i32(self.ep_pt0), i32(self.tp_free),
                                 L["pages_tp"], self.d_tp_pos, self.d_tp_pt)
        else:
            umm.gather_requests_ep2tp(h, R, self.d_owner0, self.d_tp_pos)
            umm.umm_assign_pages(h, 1, R, self.d_lens, None, self.d_tp_pos, i32(self.tp_free), L["pages_tp"],
                                 L["pages_tp"], self.d_tp_pt, maxp)
            umm.reshard_kv_ep2tp(h, R, maxp, self.d_lens, self.d_owner0, i32(self.ep_pt0), self.d_tp_pt)
        assert dev.status() == (0, 0)
        assert np.array_equal(self.d_tp_pos.cpu().numpy(), self.pos)
        assert np.array_equal(self.d_tp_pt.cpu().numpy(), self.tp_pt)

    def tp2ep(self, switch: bool = False):
        dev, R, maxp = self.dev, self.R, self.maxp
        h, L, P = dev.h, dev.L, dev.w.P
        o1 = torch.empty(R, dtype=torch.int32, device="cuda")
        l1 = torch.empty_like(o1)
        pt1 = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
        if switch:
            umm.umm_switch_tp2ep(h, R, maxp, self.d_lens, self.d_tp_pos, self.d_tp_pt, i32(self.ep_free),
                                 L["pages_ep"], L["pages_ep"], o1, l1, pt1)
        else:
            umm.place_requests_tp2ep(h, R, self.d_lens, self.d_tp_pos, o1, l1)
            umm.umm_assign_pages(h, P, R, self.d_lens, o1, self.d_tp_pos, i32(self.ep_free), L["pages_ep"],
                                 L["pages_ep"], pt1, maxp)
            umm.reshard_kv_tp2ep(h, R, maxp, self.d_lens, o1, pt1, self.d_tp_pt)
        assert dev.status() == (0, 0)
        assert np.array_equal(o1.cpu().numpy(), self.owner1)
        assert np.array_equal(l1.cpu().numpy(), self.local1)
        assert np.array_equal(pt1.cpu().numpy(), self.ep_pt1)


def _kv_samples(run: KVRun, rng, n):
    w = run.dev.w
    k = rng.integers(0, run.R, n)
    tok = (rng.random(n) * run.lens[k]).astype(np.int64)
    c = rng.integers(0, 2, n)
    h = rng.integers(0, w.Hkv, n)
    e = rng.integers(0, w.D, n)
    layer = rng.integers(0, w.N, n)
    rep = max(1, w.P // w.Hkv)
    j = rng.integers(0, rep, n)
    q = np.where(w.Hkv >= w.P, h // max(1, w.Hkv // w.P), h * rep + j)
    return k, tok, c, h, e, layer, q


def _check_kv_ep2tp(run: KVRun, rng):
    dev, w, d = run.dev, run.dev.w, run.dev.d
    k, tok, c, h, e, layer, q = _kv_samples(run, rng, SAMPLES)
    src = np.empty(SAMPLES, np.int64)
    dst = np.empty(SAMPLES, np.int64)
    for i in range(SAMPLES):
        p, t = divmod(int(tok[i]), w.ps)
        src[i], dst[i] = oracle.kv_elem(d, int(run.owner0[k[i]]), int(q[i]), int(run.ep_pt0[k[i], p]),
                                        int(run.tp_pt[k[i], p]), t, int(c[i]), int(h[i]), int(e[i]),
                                        int(layer[i]) + 1, int(layer[i]))
    assert (src >= 0).all() and (dst >= 0).all()
    np.testing.assert_array_equal(_gather(dev, dst // 2), _expect(dev, src // 2, True))


def _check_kv_tp2ep(run: KVRun, rng):
    dev, w, d = run.dev, run.dev.w, run.dev.d
    k, tok, c, h, e, layer, _ = _kv_samples(run, rng, SAMPLES)
    src = np.empty(SAMPLES, np.int64)
    dst = np.empty(SAMPLES, np.int64)
    q0 = np.where(w.Hkv >= w.P, h // max(1, w.Hkv // w.P), h * max(1, w.P // w.Hkv))
    for i in range(SAMPLES):
        p, t = divmod(int(tok[i]), w.ps)
        # where the element started (EP of owner0) and where it must be now (EP of owner1)
        src[i], _ = oracle.kv_elem(d, int(run.owner0[k[i]]), int(q0[i]), int(run.ep_pt0[k[i], p]), 0, t,
                                   int(c[i]), int(h[i]), int(e[i]), int(layer[i]) + 1, 0)
        dst[i], _ = oracle.kv_elem(d, int(run.owner1[k[i]]), int(q0[i]), int(run.ep_pt1[k[i], p]), 0, t,
                                   int(c[i]), int(h[i]), int(e[i]), int(layer[i]) + 1, 0)
    np.testing.assert_array_equal(_gather(dev, dst // 2), _expect(dev, src // 2, True))


def _check_kv_whole_requests(run: KVRun, ks):
    """Every live row of a few whole requests (all layers, K and V, all
    heads) under TP, against the generator at their EP source rows."""
    dev, w, L = run.dev, run.dev.w, run.dev.L
    u = dev.u16()
    hd = w.D
    for k in ks:
        n = int(run.lens[k])
        t = np.arange(n)
        for layer in range(w.N):
            for c in range(2):
                ep_base = (int(run.owner0[k]) * L["region_stride"] + L["kvslots_off"] +
                           (layer + 1) * L["kvslot_stride"] + c * L["kv_v_off"]) // 2
                ep_rows = ep_base + (run.ep_pt0[k, t // w.ps].astype(np.int64) * w.ps + t % w.ps) * w.Hkv * hd
                want = _expect(dev, (ep_rows[:, None] + np.arange(w.Hkv * hd)[None, :]).ravel(),
                               True).reshape(n, w.Hkv, hd)
                for q in range(w.P):
                    heads = list(range(q * w.Hkv // w.P, (q + 1) * w.Hkv // w.P)) if w.Hkv >= w.P \
                        else [q * w.Hkv // w.P]
                    tp_base = (q * L["region_stride"] + L["kvslots_off"] + layer * L["kvslot_stride"] +
                               c * L["kv_v_off"]) // 2
                    tp_rows = tp_base + (run.tp_pt[k, t // w.ps].astype(np.int64) * w.ps + t % w.ps) * \
                        L["h_tp"] * hd
                    idx = torch.from_numpy((tp_rows[:, None] + np.arange(L["h_tp"] * hd)[None, :]).ravel()).cuda()
                    got = u[idx].cpu().numpy().reshape(n, L["h_tp"], hd)
                    np.testing.assert_array_equal(got, want[:, heads, :])


def _check_kv_untouched(run: KVRun, rng):
    """TP slot 0 pages that no request uses, and the rows past the end of
    every request's last page, keep their initial contents."""
    dev, w, L = run.dev, run.dev.w, run.dev.L
    used = np.zeros(L["pages_tp"], bool)
    for k in range(run.R):
        used[run.tp_pt[k, :int(synth.npages(run.lens[k:k + 1], w.ps)[0])]] = True
    free_pages = np.flatnonzero(~used)
    page_u16 = w.ps * L["h_tp"] * w.D
    for pg in rng.choice(free_pages, size=min(64, len(free_pages)), replace=False):
        for q in rng.choice(w.P, 2, replace=False):
            base = (int(q) * L["region_stride"] + L["kvslots_off"]) // 2 + int(pg) * page_u16
            idx = np.arange(base, base + page_u16)
            np.testing.assert_array_equal(_gather(dev, idx), _expect(dev, idx, True))
    tails = [k for k in range(run.R) if run.lens[k] % w.ps][:64]
    for k in tails:
        p = int(run.lens[k]) // w.ps
        base = (L["kvslots_off"]) // 2 + int(run.tp_pt[k, p]) * page_u16
        idx = np.arange(base + (int(run.lens[k]) % w.ps) * L["h_tp"] * w.D, base + page_u16)
        np.testing.assert_array_equal(_gather(dev, idx), _expect(dev, idx, True))


@pytest.mark.parametrize("w,timed,overlap", [(KV_256REQ, False, False), (FULL_SWITCH, False, False),
                                             (FULL_SWITCH, True, False), (FULL_SWITCH, False, True)],
                         ids=["kv_256req", "full_switch", "full_switch_timed", "full_switch_overlap"])
def test_kv_and_full_switch_fullsize(w, timed, overlap):
    """KV alone through the separate entry points; the full switch through
    umm_switch_ep2tp / umm_switch_tp2ep, the calls bench.py times, also with
    per-kernel timing on (timed: events around each call's chain of layer
    copies), as in bench.py's timed steps, and with the weight copies on the
    side stream (overlap), where KV EP->TP runs on the LSU copy instead of
    the TMA one."""
    dev = DevUMM(w, seed=w.seed)
    umm.umm_profile_enable(dev.h, timed)
    umm.umm_set_switch_overlap(dev.h, overlap)
    run = KVRun(dev)
    rng = np.random.default_rng(1)
    switch = bool(w.E)
    run.ep2tp(switch)
    torch.cuda.synchronize()
    _check_kv_ep2tp(run, rng)
    _check_kv_whole_requests(run, [int(np.argmax(run.lens)), int(np.argmin(run.lens)), 0])
    _check_kv_untouched(run, rng)
    if w.E:
        _check_weights_ep2tp(dev, rng)
    run.tp2ep(switch)
    torch.cuda.synchronize()
    _check_kv_tp2ep(run, rng)
    if w.E:
        _check_weights_round_trip(dev)
    dev.close()


def test_full_switch_soak_100_round_trips():
    """100 round trips of the full switch through umm_switch_*, on one handle,
    with new free lists on every trip (pages move each time).  Afterwards
    every weight slot that holds an EP layer is bit-identical to its start,
    and sampled KV elements of every layer sit in their requests' final EP
    pages with their original values."""
    w = FULL_SWITCH
    dev = DevUMM(w, seed=w.seed)
    run = KVRun(dev)
    h, L, d, P, R, maxp = dev.h, dev.L, dev.d, w.P, run.R, run.maxp
    d_lens = i32(run.lens)
    d_owner, d_ep_pt = i32(run.owner0), i32(run.ep_pt0)
    n_owner, n_ep_pt = torch.empty_like(d_owner), torch.empty_like(d_ep_pt)
    d_local = torch.empty_like(d_owner)
    d_pos = torch.empty(R, dtype=torch.int32, device="cuda")
    d_tp_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
    for trip in range(100):
        tp_free = i32(synth.permutation(1000 + trip, 3, L["pages_tp"], rows=1))
        ep_free = i32(synth.permutation(1000 + trip, 4, L["pages_ep"], rows=P))
        umm.umm_switch_ep2tp(h, R, maxp, d_lens, d_owner, d_ep_pt, tp_free, L["pages_tp"], d_pos, d_tp_pt)
        umm.umm_switch_tp2ep(h, R, maxp, d_lens, d_pos, d_tp_pt, ep_free, L["pages_ep"], L["pages_ep"], n_owner,
                             d_local, n_ep_pt)
        d_owner, n_owner = n_owner, d_owner
        d_ep_pt, n_ep_pt = n_ep_pt, d_ep_pt
    assert dev.status() == (0, 0)
    _check_weights_round_trip(dev)
    owner_t, ep_pt_t = d_owner.cpu().numpy(), d_ep_pt.cpu().numpy()
    rng = np.random.default_rng(9)
    k, tok, c, hh, e, layer, _ = _kv_samples(run, rng, SAMPLES)
    q0 = np.where(w.Hkv >= w.P, hh // max(1, w.Hkv // w.P), hh * max(1, w.P // w.Hkv))
    src = np.empty(SAMPLES, np.int64)
    dst = np.empty(SAMPLES, np.int64)
    for i in range(SAMPLES):
        p, t = divmod(int(tok[i]), w.ps)
        src[i], _ = oracle.kv_elem(d, int(run.owner0[k[i]]), int(q0[i]), int(run.ep_pt0[k[i], p]), 0, t,
                                   int(c[i]), int(hh[i]), int(e[i]), int(layer[i]) + 1, 0)
        dst[i], _ = oracle.kv_elem(d, int(owner_t[k[i]]), int(q0[i]), int(ep_pt_t[k[i], p]), 0, t,
                                   int(c[i]), int(hh[i]), int(e[i]), int(layer[i]) + 1, 0)
    np.testing.assert_array_equal(_gather(dev, dst // 2), _expect(dev, src // 2, True))
    dev.close()


def _attn_views(dev: DevUMM, r: int, slot: int, full: bool):
    """(QKV heads, Wo) of one attention slot as device tensors: EP (full) or
    TP (shard) view, the shapes of §3.1's attention part."""
    w, L = dev.w, dev.L
    base = attnslot(L, r, slot) // 2
    nh = w.Hq + 2 * w.Hkv if full else w.Hq // w.P + 2 * L["h_tp"]
    ncol = w.Hq * w.D if full else w.Hq // w.P * w.D
    u = dev.u16()
    qkv = u[base:base + nh * w.D * w.H].view(nh, w.D * w.H)
    wo_at = base + L["attn_wo_off"] // 2
    return qkv, u[wo_at:wo_at + w.H * ncol].view(w.H, ncol)


def _attn_initial(dev: DevUMM, r: int, slot: int):
    w, L = dev.w, dev.L
    nh = w.Hq + 2 * w.Hkv
    off = attnslot(L, r, slot)
    qkv = _regen(dev, off, 2 * nh * w.D * w.H, False).view(nh, w.D * w.H)
    wo = _regen(dev, off + L["attn_wo_off"], 2 * w.H * w.Hq * w.D, False).view(w.H, w.Hq * w.D)
    return qkv, wo


def test_attn_fullsize():
    """Attention weights of the page's model shape (64 query / 4 KV heads of
    128, hidden 4096, 8 layers) through umm_switch_*: every TP shard equals the
    torch slice of its own rank's full copy (memory-saving variant: EP->TP is a
    local extraction), and after TP->EP every rank holds the all-gather of the
    shards (KV heads from the lowest rank holding them)."""
    w = ATTN_QWEN3_SHAPE
    dev = DevUMM(w, seed=5)
    P, Hq, Hkv, D = w.P, w.Hq, w.Hkv, w.D
    qh = Hq // P
    umm.umm_switch_ep2tp(dev.h, 0, 1, None, None, None, None, 0, None, None)
    torch.cuda.synchronize()
    assert umm.umm_get_attn_mode(dev.h) == umm.UMM_MODE_TP
    for layer in range(w.N):
        for q in range(P):
            full, wo = _attn_initial(dev, q, layer + 1)
            kvh = heads_of_rank(P, Hkv, q)
            want = torch.cat([full[q * qh:(q + 1) * qh], full[[Hq + h for h in kvh]],
                              full[[Hq + Hkv + h for h in kvh]]])
            got_qkv, got_wo = _attn_views(dev, q, layer, full=False)
            assert torch.equal(got_qkv, want), (layer, q)
            assert torch.equal(got_wo, wo[:, q * qh * D:(q + 1) * qh * D]), (layer, q)
    # expected full copies after TP->EP, from the shards now in the TP slots
    want_full = []
    for layer in range(w.N):
        shards = [_attn_views(dev, q, layer, full=False) for q in range(P)]
        lowest = {}
        for q in range(P):
            for i, h in enumerate(heads_of_rank(P, Hkv, q)):
                lowest.setdefault(h, (q, i))
        h_tp = len(heads_of_rank(P, Hkv, 0))
        k_rows = [shards[lowest[h][0]][0][qh + lowest[h][1]] for h in range(Hkv)]
        v_rows = [shards[lowest[h][0]][0][qh + h_tp + lowest[h][1]] for h in range(Hkv)]
        qkv = torch.cat([torch.cat([s[0][:qh] for s in shards]), torch.stack(k_rows), torch.stack(v_rows)])
        wo = torch.cat([s[1] for s in shards], dim=1)
        want_full.append((qkv.clone(), wo.clone()))
    umm.umm_switch_tp2ep(dev.h, 0, 1, None, None, None, None, 0, 0, None, None, None)
    torch.cuda.synchronize()
    assert umm.umm_get_attn_mode(dev.h) == umm.UMM_MODE_EP
    for layer in range(w.N):
        for r in range(P):
            got_qkv, got_wo = _attn_views(dev, r, layer + 1, full=True)
            assert torch.equal(got_qkv, want_full[layer][0]), (layer, r)
            assert torch.equal(got_wo, want_full[layer][1]), (layer, r)
    dev.close()


def test_tiny_round_trip_matches_oracle_exactly_in_bench_sequence():
    """The same device sequence at the tiny size, compared whole with the oracle."""
    w = TINY
    dev = DevUMM(w, seed=w.seed)
    run = KVRun(dev)
    ref = dev.host()
    umm.reshard_weights_ep2tp(dev.h)
    run.ep2tp()
    umm.reshard_weights_tp2ep(dev.h)
    run.tp2ep()
    oracle.weights_ep2tp(ref, dev.d)
    assert oracle.kv_ep2tp(ref, dev.d, run.lens, run.owner0, run.ep_pt0, run.tp_pt) == 0
    oracle.weights_tp2ep(ref, dev.d)
    assert oracle.kv_tp2ep(ref, dev.d, run.lens, run.owner1, run.ep_pt1, run.tp_pt) == 0
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()
