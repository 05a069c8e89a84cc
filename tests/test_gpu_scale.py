"""Parity at the full workload sizes, in the launch configuration bench.py
times (same entry points, same sequence, same grid sizing).  The oracle
cannot hold these buffers, so outputs are checked (a) on random samples the
oracle maps one by one (its element maps + the generator's value at the
source), (b) whole, against properties that hold at any size: the TP shards
equal torch slices of the full EP tensors (§3.1 shapes), the EP->TP->EP
round trip is the identity (weights), and (c) every byte of every KV slot of
every region, after each direction, against contents rebuilt on the device
from the generator and the oracle's page tables (KVComplete), and bytes
outside every destination keep their contents."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import oracle
import synth
from gpu_helpers import DevUMM, i32
from helpers import attnslot, heads_of_rank
from synth.workloads import ATTN_QWEN3_SHAPE, FULL_SWITCH, KV_256REQ, TINY, WEIGHTS_H2048, WEIGHTS_H4096, Workload

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


@pytest.mark.parametrize("I", [10912, 10922], ids=["vec16", "vec2"])
def test_weights_largest_region(I):
    """The largest expert-weight region the handle accepts: 2 ranks, one expert
    each, H = 65,536, 3*I*H just under 2^31 - 2^16 elements per region (the
    bound that keeps the kernel's 32-bit vector indices and exact divisions
    valid), 16 GiB.  I = 10,912 runs 16-byte vectors; I = 10,922 (I/P odd)
    2-byte ones, whose highest vector index is 2,147,352,575.  Sampled oracle
    maps, whole-layer torch slices, then the round trip over every slot."""
    w = Workload(f"weights_p2_e2_h65536_i{I}_1layer", P=2, N=1, E=2, H=65536, I=I)
    dev = DevUMM(w, seed=17)
    rng = np.random.default_rng(I)
    umm.reshard_weights_ep2tp(dev.h)
    torch.cuda.synchronize()
    assert dev.status() == (0, 0)
    _check_weights_ep2tp(dev, rng)
    umm.reshard_weights_tp2ep(dev.h)
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


def _group(key: np.ndarray, n: int, a: np.ndarray, b: np.ndarray) -> list:
    """For each group g < n: (a[key == g], b[key == g]) as device tensors,
    in token order (one stable sort, then views of one device copy)."""
    order = np.argsort(key, kind="stable")
    bounds = np.searchsorted(key[order], np.arange(n + 1))
    da = torch.from_numpy(np.ascontiguousarray(a[order])).cuda()
    db = torch.from_numpy(np.ascontiguousarray(b[order])).cuda()
    return [(da[bounds[g]:bounds[g + 1]], db[bounds[g]:bounds[g + 1]]) for g in range(n)]


class KVComplete:
    """Every byte of every KV slot of every region, compared whole.

    The expected contents are rebuilt on the device, one (slot, half) at a
    time: the generator's initial values, with the rows each switch writes
    replaced by the generator's values at their sources (§3.2, Fig. 5: the
    page table maps logical page p of request k to a physical page; token t
    is row t % page_size of page table[k][t // page_size]; §4.2 Fig. 7: EP
    layer l in slot l+1, TP layer l in slot l).  Sources and destinations are
    the oracle's (owners, page tables); the row arithmetic below is pinned to
    the oracle's element map (kv_elem) on a sample before it is used.

    After EP->TP, slot l (l < N) of rank q holds TP layer l: its initial bytes
    with every live token row of TP page tp_pt[k][p] set to the row of the
    request's EP page in EP slot l+1 of its owner, heads of rank q only; slot
    N is untouched.  After TP->EP, slot l+1 holds that state (TP layer l+1
    for l+1 < N, else the initial bytes) with every live row of new EP page
    ep_pt1[k][p] of the new owner set to the original EP row; slot 0 keeps TP
    layer 0.  The page tails, unused pages and alignment padding of each slot
    are compared too: they must keep their initial bytes."""

    def __init__(self, run: KVRun, samples: int = 20_000):
        dev, w, L = run.dev, run.dev.w, run.dev.L
        self.run, self.dev, self.w, self.L = run, dev, w, L
        P, ps = w.P, w.ps
        lens = run.lens.astype(np.int64)
        k = np.repeat(np.arange(run.R), lens)
        t = np.arange(len(k)) - np.repeat(np.cumsum(lens) - lens, lens)
        p, row = t // ps, t % ps
        o0, o1 = run.owner0[k].astype(np.int64), run.owner1[k].astype(np.int64)
        src0 = run.ep_pt0[k, p].astype(np.int64) * ps + row
        tp = run.tp_pt[k, p].astype(np.int64) * ps + row
        dst1 = run.ep_pt1[k, p].astype(np.int64) * ps + row
        self.half_u16 = L["pages_tp"] * ps * L["h_tp"] * w.D
        assert self.half_u16 == L["pages_ep"] * ps * w.Hkv * w.D
        self._pin(k, t, o0, o1, src0, tp, dst1, samples)
        self.by_o0 = _group(o0, P, src0, tp)
        self.by_move = _group(o0 * P + o1, P * P, src0, dst1)
        self.heads = [heads_of_rank(P, w.Hkv, q) for q in range(P)]

    def slot_off(self, r: int, s: int) -> int:
        L = self.L
        return r * L["region_stride"] + L["kvslots_off"] + s * L["kvslot_stride"]

    def _pin(self, k, t, o0, o1, src0, tp, dst1, n):
        """The flat element offsets used below equal the oracle's kv_elem."""
        run, w, L, d = self.run, self.w, self.L, self.dev.d
        rng = np.random.default_rng(17)
        pick = rng.integers(0, len(k), n)
        c = rng.integers(0, 2, n)
        h = rng.integers(0, w.Hkv, n)
        e = rng.integers(0, w.D, n)
        layer = rng.integers(0, w.N, n)
        for i in range(n):
            j = int(pick[i])
            q = next(q for q in range(w.P) if h[i] in self.heads_of(q))
            hl = self.heads_of(q).index(int(h[i]))
            pg, tt = divmod(int(t[j]), w.ps)
            kk = int(k[j])
            a, b = oracle.kv_elem(d, int(o0[j]), q, int(run.ep_pt0[kk, pg]), int(run.tp_pt[kk, pg]), tt,
                                  int(c[i]), int(h[i]), int(e[i]), int(layer[i]) + 1, int(layer[i]))
            ep = self.slot_off(int(o0[j]), int(layer[i]) + 1) + c[i] * L["kv_v_off"] + \
                2 * ((int(src0[j]) * w.Hkv + int(h[i])) * w.D + int(e[i]))
            tpo = self.slot_off(q, int(layer[i])) + c[i] * L["kv_v_off"] + \
                2 * ((int(tp[j]) * L["h_tp"] + hl) * w.D + int(e[i]))
            assert (a, b) == (ep, tpo), i
            a1, _ = oracle.kv_elem(d, int(o1[j]), q, int(run.ep_pt1[kk, pg]), 0, tt, int(c[i]), int(h[i]),
                                   int(e[i]), int(layer[i]) + 1, 0)
            assert a1 == self.slot_off(int(o1[j]), int(layer[i]) + 1) + c[i] * L["kv_v_off"] + \
                2 * ((int(dst1[j]) * w.Hkv + int(h[i])) * w.D + int(e[i])), i

    def heads_of(self, q: int) -> list[int]:
        return heads_of_rank(self.w.P, self.w.Hkv, q)

    def _half(self, r: int, s: int, c: int) -> int:
        return (self.slot_off(r, s) + c * self.L["kv_v_off"]) // 2

    def got(self, r: int, s: int, c: int) -> torch.Tensor:
        o = self._half(r, s, c)
        return self.dev.u16()[o:o + self.half_u16]

    def initial(self, r: int, s: int, c: int) -> torch.Tensor:
        return _regen(self.dev, 2 * self._half(r, s, c), 2 * self.half_u16, True)

    def _tp_rows(self, exp: list, layer: int, c: int) -> None:
        """Write TP layer `layer` (from EP slot layer+1) into exp[q] (TP view)."""
        w, h_tp = self.w, self.L["h_tp"]
        for r in range(w.P):
            s_idx, t_idx = self.by_o0[r]
            if not len(s_idx):
                continue
            vals = self.initial(r, layer + 1, c).view(-1, w.Hkv, w.D)[s_idx]
            for q in range(w.P):
                exp[q].view(-1, h_tp, w.D)[t_idx] = vals[:, self.heads[q], :]
            del vals

    def _pads_intact(self, r: int, s: int) -> None:
        """Alignment padding after each half of a KV slot keeps its bytes."""
        L, u = self.L, self.dev.u16()
        for a, b in ((self.half_u16 * 2, L["kv_v_off"]), (L["kv_v_off"] + self.half_u16 * 2, L["kvslot_stride"])):
            if b > a:
                o = self.slot_off(r, s) + a
                assert torch.equal(u[o // 2:(o + b - a) // 2], _regen(self.dev, o, b - a, True)), (r, s)

    def check_after_ep2tp(self) -> None:
        w = self.w
        torch.cuda.empty_cache()
        for layer in range(w.N):
            for c in range(2):
                exp = [self.initial(q, layer, c) for q in range(w.P)]
                self._tp_rows(exp, layer, c)
                for q in range(w.P):
                    assert torch.equal(self.got(q, layer, c), exp[q]), ("ep2tp", layer, c, q)
                del exp
        for r in range(w.P):
            for c in range(2):
                assert torch.equal(self.got(r, w.N, c), self.initial(r, w.N, c)), ("slot N", r, c)
            for s in range(w.N + 1):
                self._pads_intact(r, s)
        torch.cuda.empty_cache()

    def check_live_ep(self, owner, ep_pt) -> None:
        """Every live element of every layer sits in EP page ep_pt[k][p] of
        owner[k] with its original value (the generator's value at the
        request's starting EP row: owner0, ep_pt0).  Bytes outside live rows
        are not compared here."""
        w, run, ps = self.w, self.run, self.w.ps
        lens = run.lens.astype(np.int64)
        k = np.repeat(np.arange(run.R), lens)
        t = np.arange(len(k)) - np.repeat(np.cumsum(lens) - lens, lens)
        p, row = t // ps, t % ps
        o0, ot = run.owner0[k].astype(np.int64), np.asarray(owner)[k].astype(np.int64)
        src0 = run.ep_pt0[k, p].astype(np.int64) * ps + row
        dst = np.asarray(ep_pt)[k, p].astype(np.int64) * ps + row
        moves = _group(o0 * w.P + ot, w.P * w.P, src0, dst)
        torch.cuda.empty_cache()
        for layer in range(w.N):
            for c in range(2):
                for a in range(w.P):
                    src = self.initial(a, layer + 1, c).view(-1, w.Hkv, w.D)
                    for b in range(w.P):
                        s_idx, d_idx = moves[a * w.P + b]
                        if len(s_idx):
                            got = self.got(b, layer + 1, c).view(-1, w.Hkv, w.D)[d_idx]
                            assert torch.equal(got, src[s_idx]), ("live", layer, c, a, b)
                    del src
        torch.cuda.empty_cache()

    def check_after_tp2ep(self) -> None:
        w = self.w
        torch.cuda.empty_cache()
        for layer in range(w.N):
            for c in range(2):
                exp = [self.initial(r, layer + 1, c) for r in range(w.P)]
                if layer + 1 < w.N:
                    self._tp_rows(exp, layer + 1, c)
                for a in range(w.P):
                    src = self.initial(a, layer + 1, c).view(-1, w.Hkv, w.D)
                    for b in range(w.P):
                        s_idx, d_idx = self.by_move[a * w.P + b]
                        if len(s_idx):
                            exp[b].view(-1, w.Hkv, w.D)[d_idx] = src[s_idx]
                    del src
                for r in range(w.P):
                    assert torch.equal(self.got(r, layer + 1, c), exp[r]), ("tp2ep", layer, c, r)
                del exp
        for c in range(2):
            exp = [self.initial(q, 0, c) for q in range(w.P)]
            self._tp_rows(exp, 0, c)
            for q in range(w.P):
                assert torch.equal(self.got(q, 0, c), exp[q]), ("slot 0", c, q)
            del exp
        for r in range(w.P):
            for s in range(w.N + 1):
                self._pads_intact(r, s)
        torch.cuda.empty_cache()


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
    full = KVComplete(run)
    rng = np.random.default_rng(1)
    switch = bool(w.E)
    run.ep2tp(switch)
    torch.cuda.synchronize()
    _check_kv_ep2tp(run, rng)
    full.check_after_ep2tp()
    if w.E:
        _check_weights_ep2tp(dev, rng)
    run.tp2ep(switch)
    torch.cuda.synchronize()
    _check_kv_tp2ep(run, rng)
    full.check_after_tp2ep()
    if w.E:
        _check_weights_round_trip(dev)
    dev.close()


# Shapes between the randomised small cases and the two full-size KV
# workloads: thousands of descriptors on other head/page/rank shapes, each
# compared byte for byte by KVComplete.  Pools with slack 5 leave the live
# pages under half the TP pool, so the copies walk the descriptor list
# instead of the TP-page schedule.
KV_SHAPES = [
    Workload("kv_p16_hkv16_d64_ps32", P=16, N=3, Hkv=16, D=64, ps=32, R=600, len_a=1, len_b=4096, slack=1.3),
    Workload("kv_p4_hkv8_d128", P=4, N=2, Hkv=8, D=128, ps=16, R=500, len_a=1, len_b=8192, slack=1.3),
    Workload("kv_p8_hkv1_d128_lognormal", P=8, N=2, Hkv=1, D=128, ps=16, R=400, len_kind="lognormal",
             len_a=1024, len_b=1.0, len_cap=16384, slack=1.3),
    Workload("kv_p2_hkv2_d72_ps8", P=2, N=3, Hkv=2, D=72, ps=8, R=300, len_a=1, len_b=3000, slack=1.3),
    Workload("kv_p64_hkv64_d16", P=64, N=2, Hkv=64, D=16, ps=16, R=2000, len_a=1, len_b=1024, slack=1.6),
    Workload("kv_p8_hkv4_d12_sparse", P=8, N=2, Hkv=4, D=12, ps=16, R=300, len_a=1, len_b=2048, slack=5.0),
    Workload("kv_p8_hkv4_d128_sparse", P=8, N=2, Hkv=4, D=128, ps=16, R=200, len_a=1, len_b=4096, slack=5.0),
    Workload("kv_p3_hkv3_d5_ps7", P=3, N=2, Hkv=3, D=5, ps=7, R=200, len_a=1, len_b=500, slack=1.5),
]


@pytest.mark.parametrize("w", KV_SHAPES, ids=lambda w: w.name)
def test_kv_shapes_complete(w):
    """EP->TP then TP->EP through the separate entry points; every byte of
    every KV slot compared after each direction (the TMA or LSU copy the
    shape selects, in TP-page or descriptor-list order)."""
    dev = DevUMM(w, seed=w.seed + 7)
    run = KVRun(dev)
    full = KVComplete(run, samples=3_000)
    run.ep2tp()
    torch.cuda.synchronize()
    full.check_after_ep2tp()
    run.tp2ep()
    torch.cuda.synchronize()
    full.check_after_tp2ep()
    dev.close()


@pytest.mark.parametrize("P,R", [(8, 1 << 15), (64, 30_001)])
def test_kv_many_requests_complete(P, R):
    """More requests than the other KV tests (2^15, and a ragged 30,001 on 64
    ranks), short requests (0..12 tokens, pages of 4), through the bench's
    call sequence.  The sizes stay where the oracle's quadratic request
    loops (local positions, page hand-out) finish in seconds.  The
    single-CTA metadata kernels run at that scale:
      - the request order and the TP page tables equal the oracle's;
      - the greedy owners, local positions and EP page tables equal it too
        (the placement sorts its keys in the workspace beyond 16,384
        requests);
      - the descriptor list of the EP->TP pass equals the oracle's;
      - every KV byte is compared after both directions."""
    w = Workload(f"kv_p{P}_{R}req_u0-12_ps4", P=P, N=1, Hkv=P, D=8, ps=4, R=R, len_a=0, len_b=12, slack=1.3)
    dev = DevUMM(w, seed=3)
    run = KVRun(dev)
    full = KVComplete(run, samples=1_000)
    L = dev.L
    nd = int(synth.npages(run.lens, w.ps).sum())

    def descriptors():
        assert int(dev.buf[L["status_off"] + 8:L["status_off"] + 16].view(torch.int64).item()) == nd
        return dev.buf[L["desc_off"]:L["desc_off"] + 32 * nd].view(torch.int32).view(nd, 8).cpu().numpy()

    run.ep2tp()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(descriptors(),
                                  oracle.kv_descriptors(dev.d, 0, run.lens, run.owner0, run.ep_pt0, run.tp_pt))
    full.check_after_ep2tp()
    run.tp2ep()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(descriptors(),
                                  oracle.kv_descriptors(dev.d, 1, run.lens, run.owner1, run.ep_pt1, run.tp_pt))
    full.check_after_tp2ep()
    dev.close()


def random_medium_kv(seed: int) -> Workload:
    """A random KV shape with hundreds of requests and thousands of pages,
    its pool sized so that the greedy placement's busiest rank fits, and the
    buffer kept under about 16 GiB."""
    rng = np.random.default_rng(5000 + seed)
    P = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 32, 64]))
    if rng.random() < 0.5:
        divs = [h for h in range(1, P + 1) if P % h == 0]
        Hkv = int(rng.choice(divs))                          # Hkv <= P: one head per TP rank
    else:
        Hkv = P * int(rng.choice([2, 4]))                    # Hkv > P: several heads per TP rank
    D = int(rng.choice([8, 16, 64, 128, int(rng.integers(1, 160)), int(rng.integers(1, 160))]))
    ps = int(rng.choice([1, 4, 7, 16, 32, 64]))
    N = int(rng.integers(1, 4))
    R = int(rng.integers(50, 800))
    len_b = int(rng.integers(ps, 400 * ps + 1))
    sparse = 5.0 if rng.random() < 0.3 else 1.0

    def sized(w: Workload) -> Workload:
        pages = synth.npages(w.lengths(), w.ps)
        used, m = max(1, int(pages.sum())), w.Hkv // w.h_tp
        bound = used / w.P + int(pages.max()) + w.R / w.P + 1   # busiest rank under the greedy rule
        return w.with_(slack=max(1.05, 1.02 * m * bound / used) * sparse)

    from gpu_helpers import lib_dims
    w = sized(Workload(f"kv_rand{seed}", P=P, N=N, Hkv=Hkv, D=D, ps=ps, R=R, len_a=0, len_b=len_b, seed=seed))
    while umm.umm_required_bytes(lib_dims(w)) > (16 << 30):
        if w.R > 10:
            w = sized(w.with_(R=w.R // 2))
        elif w.len_b > w.ps:
            w = sized(w.with_(len_b=max(w.ps, int(w.len_b) // 2)))
        else:
            break
    return w


@pytest.mark.parametrize("seed", range(12))
def test_kv_random_medium_complete(seed):
    """Random medium shapes, byte-complete after both directions."""
    w = random_medium_kv(seed)
    dev = DevUMM(w, seed=seed)
    run = KVRun(dev)
    full = KVComplete(run, samples=1_000)
    run.ep2tp()
    torch.cuda.synchronize()
    full.check_after_ep2tp()
    run.tp2ep()
    torch.cuda.synchronize()
    full.check_after_tp2ep()
    dev.close()


def test_kv_shapes_take_both_copies_and_both_walks():
    """The shapes above cover the TMA and the LSU copy, every LSU vector
    width, and both walks of the copies (TP-page schedule, descriptor list)."""
    from gpu_helpers import lib_dims
    kernels, walks = set(), set()
    for w in KV_SHAPES:
        k, vb = umm.umm_kv_copy_kernel(lib_dims(w), 0)
        kernels.add((k, vb))
        lens = w.lengths()
        pages_tp = w.pages_tp()
        most = min(pages_tp, len(lens) * w.max_pages_per_req())
        walks.add(2 * most >= pages_tp)
    assert {k for k, _ in kernels} == {umm.UMM_KV_COPY_TMA, umm.UMM_KV_COPY_LSU}
    assert {vb for k, vb in kernels if k == umm.UMM_KV_COPY_LSU} >= {32, 8, 2}
    assert walks == {True, False}


def test_full_switch_soak_100_round_trips():
    """100 round trips of the full switch through umm_switch_*, on one handle,
    with new free lists on every trip (pages move each time).  Afterwards
    every weight slot that holds an EP layer is bit-identical to its start,
    and every live KV element of every layer (and, independently, 200k
    oracle-mapped samples) sits in its request's final EP page with its
    original value."""
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
    KVComplete(run, samples=2_000).check_live_ep(owner_t, ep_pt_t)
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
