"""Pins of the CPU oracle to facts other than its own code (no GPU).

Each test checks the oracle against something the page or the mathematics
fixes: hand-worked examples (tests/golden), the functional equivalence the
page rests on ("one model, two layouts": EP and TP compute the same function on
the same bytes, "Moebius: Serving Mixture-of-Expert Models with Seamless
Runtime Parallelism Switch" (paper review) §3), round trips, exactly-once and
replication counts, special cases that reduce to numpy/torch slicing, the
byte accounting of §4.3 Table 1, the layer order of §4.2 Fig. 7, and brute
force for the greedy placement of §3.2.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import (bf16_to_f64, dims_of, fill_regions, gather_tokens, heads_of_rank,
                     initial_kv_state, ints, kv_ep, kv_tp, read_golden, w13_ep, w13_tp,
                     w2_ep, w2_tp, wslot)
from synth.workloads import TINY, Workload

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

SMALL_W = Workload("w_small", P=4, N=3, E=8, H=24, I=16, w_sigma=0.5)
SMALL_KV = Workload("kv_small", P=4, N=3, Hkv=2, D=8, ps=4, R=9, len_kind="uniform",
                    len_a=1, len_b=23, kv_sigma=1.0)


# ----------------------------------------------------------------------------- layout

@pytest.mark.parametrize("w", [TINY, SMALL_W, SMALL_KV, TINY.with_(Hkv=4, P=2, E=4), TINY.with_(Hq=4)])
def test_layout_parts_disjoint_and_aligned(w):
    d = dims_of(w)
    L = oracle.layout(d)
    El, Ip = d.E // d.P, d.I // d.P
    w13 = El * 2 * d.I * d.H * 2
    w2 = El * d.H * d.I * 2
    assert L["w2_off"] >= w13 and L["w2_off"] % 256 == 0
    if d.E:
        assert L["wslot_stride"] >= L["w2_off"] + w2 and L["wslot_stride"] % 4096 == 0
    # the same bytes per slot in both views (§3: only ownership changes)
    assert w13 == d.E * 2 * Ip * d.H * 2 and w2 == d.E * d.H * Ip * 2
    if d.Hkv:
        half_tp = L["pages_tp"] * d.ps * L["h_tp"] * d.D * 2
        half_ep = L["pages_ep"] * d.ps * d.Hkv * d.D * 2
        assert half_ep == half_tp
        assert L["kv_v_off"] >= half_tp and L["kv_v_off"] % 256 == 0
        assert L["kvslot_stride"] >= L["kv_v_off"] + half_tp
    assert L["kvslots_off"] == (d.N + 1) * L["wslot_stride"]
    # attention slots (memory-saving variant) after the KV slots, sized for the
    # full EP copy: Wqkv of Hq + 2 Hkv heads, then W_o (H x Hq*Dh)
    assert L["attnslots_off"] == (d.N + 1) * (L["wslot_stride"] + L["kvslot_stride"])
    if d.Hq:
        assert L["attn_wo_off"] >= (d.Hq + 2 * d.Hkv) * d.D * d.H * 2 and L["attn_wo_off"] % 256 == 0
        assert L["attnslot_stride"] >= L["attn_wo_off"] + d.H * d.Hq * d.D * 2
        assert L["attnslot_stride"] % 4096 == 0
    assert L["region_stride"] >= (d.N + 1) * (L["wslot_stride"] + L["kvslot_stride"] + L["attnslot_stride"])
    assert L["region_stride"] % (2 << 20) == 0
    assert L["ws_off"] == d.P * L["region_stride"]


# ----------------------------------------------------------------------------- weights

def _tagged_weights(d: oracle.Dims, L: dict, tag_w13, tag_w2, slot: int) -> np.ndarray:
    buf = np.zeros(L["ws_off"], dtype=np.uint8)
    for r in range(d.P):
        a = w13_ep(buf, L, d, r, slot)
        b = w2_ep(buf, L, d, r, slot)
        for el in range(d.E // d.P):
            e = r * (d.E // d.P) + el
            for j in range(2 * d.I):
                for h in range(d.H):
                    a[el, j, h] = tag_w13(e, j, h)
            for h in range(d.H):
                for i in range(d.I):
                    b[el, h, i] = tag_w2(e, h, i)
    return buf


def test_weights_golden_hand_worked():
    g = read_golden("w13_w2_p2_e2_h2_i4.txt")
    kv = {ln.split()[0]: int(ln.split()[1]) for ln in g if ln.split()[0] in ("P", "E", "H", "I")}
    d = oracle.Dims(P=kv["P"], E=kv["E"], H=kv["H"], I=kv["I"], N=1)
    L = oracle.layout(d)
    buf = _tagged_weights(d, L, lambda e, j, h: 100 * e + 10 * j + h,
                          lambda e, h, i: 1000 + 100 * e + 10 * h + i, slot=1)
    oracle.weights_ep2tp(buf, d)
    n = 0
    for ln in g:
        name, rest = ln.split(" ", 1)
        if name not in ("tp_w13", "tp_w2"):
            continue
        head, vals = rest.split(":")
        q, e = ints(head)
        got = (w13_tp if name == "tp_w13" else w2_tp)(buf, L, d, q, 0)[e].ravel().tolist()
        assert got == ints(vals), (name, q, e)
        n += 1
    assert n == 8


def _silu(x):
    return x / (1.0 + np.exp(-x))


@pytest.mark.parametrize("w", [SMALL_W, TINY.with_(w_sigma=0.3)])
def test_weights_tp_shards_compute_the_same_moe_ffn(w):
    """§3: EP and TP compute the same function on the same bytes.  For every
    expert, the EP owner's SwiGLU FFN  W2 (silu(W1 x) * (W3 x))  equals the sum
    over TP ranks of the same FFN on their shards (the All-Reduce of §2.1)."""
    d = dims_of(w)
    L = oracle.layout(d)
    buf = fill_regions(L, w, seed=11)
    before = buf.copy()
    oracle.weights_ep2tp(buf, d)
    rng = np.random.default_rng(5)
    El, Ip = d.E // d.P, d.I // d.P
    for layer in range(d.N):
        x = rng.normal(size=d.H)
        for e in range(d.E):
            r, el = divmod(e, El)
            w13 = bf16_to_f64(w13_ep(before, L, d, r, layer + 1)[el])
            w2 = bf16_to_f64(w2_ep(before, L, d, r, layer + 1)[el])
            y_ep = w2 @ (_silu(w13[:d.I] @ x) * (w13[d.I:] @ x))
            y_tp = np.zeros(d.H)
            for q in range(d.P):
                s13 = bf16_to_f64(w13_tp(buf, L, d, q, layer)[e])
                s2 = bf16_to_f64(w2_tp(buf, L, d, q, layer)[e])
                y_tp += s2 @ (_silu(s13[:Ip] @ x) * (s13[Ip:] @ x))
            np.testing.assert_allclose(y_tp, y_ep, rtol=1e-9, atol=1e-12)


def test_weights_contiguous_split_is_a_row_slice():
    """w13_split = 1: TP rank q keeps W13 rows [q*2I/P, (q+1)*2I/P) (numpy slice)."""
    w = SMALL_W
    d = dims_of(w, w13_split=1)
    L = oracle.layout(d)
    buf = fill_regions(L, w, seed=3)
    before = buf.copy()
    oracle.weights_ep2tp(buf, d)
    full = np.concatenate([w13_ep(before, L, d, r, 1) for r in range(d.P)])
    rows = 2 * d.I // d.P
    for q in range(d.P):
        np.testing.assert_array_equal(w13_tp(buf, L, d, q, 0), full[:, q * rows:(q + 1) * rows, :])


def test_weights_exactly_once_tagged():
    """Every EP element lands in exactly one TP place (unique 16-bit tags)."""
    w = TINY
    d = dims_of(w)
    L = oracle.layout(d)
    El = d.E // d.P
    n13 = d.E * 2 * d.I * d.H
    buf = _tagged_weights(d, L, lambda e, j, h: (e * 2 * d.I + j) * d.H + h,
                          lambda e, h, i: n13 + (e * d.H + h) * d.I + i, slot=2)
    assert n13 + d.E * d.H * d.I <= 65536
    oracle.weights_ep2tp(buf, d)
    got = np.concatenate([np.concatenate([w13_tp(buf, L, d, q, 1).ravel(), w2_tp(buf, L, d, q, 1).ravel()])
                          for q in range(d.P)])
    assert np.array_equal(np.sort(got), np.arange(n13 + d.E * d.H * d.I))
    # cross-region share: (P-1)/P of the moved elements change rank (§3); the
    # rank's own share moves too, from slot l+1 to slot l
    moved_from = []
    for q in range(d.P):
        t13 = w13_tp(buf, L, d, q, 1).astype(np.int64)
        e_of = t13 // (2 * d.I * d.H)
        moved_from.append(((e_of // El) != q).sum())
    assert sum(moved_from) == n13 * (d.P - 1) // d.P
    del El


@pytest.mark.parametrize("split", [0, 1])
def test_weights_round_trip_identity_and_untouched_bytes(split):
    """EP -> TP -> EP is the identity on every EP slot, for both W13 row
    splits (R-2), and bytes that are not a destination keep their contents."""
    w = SMALL_W.with_(w_sigma=None)
    d = dims_of(w, w13_split=split)
    L = oracle.layout(d)
    buf = fill_regions(L, w, seed=7)
    orig = buf.copy()
    oracle.weights_ep2tp(buf, d)
    # slot N still holds EP layer N-1: nothing writes it, and bytes that are
    # not a destination keep their contents
    for r in range(d.P):
        a = wslot(L, r, d.N)
        assert np.array_equal(buf[a:a + L["wslot_stride"]], orig[a:a + L["wslot_stride"]])
    oracle.weights_tp2ep(buf, d)
    for r in range(d.P):
        a, b = wslot(L, r, 1), wslot(L, r, d.N + 1)
        assert np.array_equal(buf[a:b], orig[a:b])
    # padding between W13 and W2, and after W2, never written
    for r in range(d.P):
        for s in range(d.N + 1):
            base = wslot(L, r, s)
            w13 = (d.E // d.P) * 2 * d.I * d.H * 2
            assert np.array_equal(buf[base + w13:base + L["w2_off"]], orig[base + w13:base + L["w2_off"]])


def test_weights_p1_is_a_slot_shift():
    """P = 1: both layouts coincide, so EP->TP is a plain copy slot l+1 -> slot l."""
    w = Workload("p1", P=1, N=3, E=3, H=8, I=6)
    d = dims_of(w)
    L = oracle.layout(d)
    buf = fill_regions(L, w, seed=1)
    orig = buf.copy()
    oracle.weights_ep2tp(buf, d)
    s = L["wslot_stride"]
    used = L["w2_off"] + d.E * d.H * d.I * 2
    for layer in range(d.N):
        np.testing.assert_array_equal(buf[layer * s + L["w13_off"]:layer * s + d.E * 2 * d.I * d.H * 2],
                                      orig[(layer + 1) * s:(layer + 1) * s + d.E * 2 * d.I * d.H * 2])
        np.testing.assert_array_equal(buf[layer * s + L["w2_off"]:layer * s + used],
                                      orig[(layer + 1) * s + L["w2_off"]:(layer + 1) * s + used])


def test_weights_w2_tp_is_a_column_slice():
    """TP W2 of rank q = columns [q*I/P, (q+1)*I/P) of the full W2 (numpy slice)."""
    w = SMALL_W
    d = dims_of(w)
    L = oracle.layout(d)
    buf = fill_regions(L, w, seed=9)
    before = buf.copy()
    oracle.weights_ep2tp(buf, d)
    Ip = d.I // d.P
    for layer in range(d.N):
        full = np.concatenate([w2_ep(before, L, d, r, layer + 1) for r in range(d.P)])
        for q in range(d.P):
            np.testing.assert_array_equal(w2_tp(buf, L, d, q, layer), full[:, :, q * Ip:(q + 1) * Ip])


def test_layer_order_makes_in_place_safe():
    """§4.2 Fig. 7: with the one-slot offset, EP->TP ascending and TP->EP
    descending in place equal the copy-from-snapshot definition; the other
    order overwrites layers before they are read."""
    w = SMALL_W.with_(w_sigma=None)
    d = dims_of(w)
    L = oracle.layout(d)
    orig = fill_regions(L, w, seed=2)
    ref = orig.copy()
    oracle.weights_ep2tp(ref, d, src=orig.copy())
    ip = orig.copy()
    oracle.weights_ep2tp(ip, d)
    assert np.array_equal(ip, ref)
    wrong = orig.copy()
    oracle.weights_ep2tp(wrong, d, order=-1)
    assert not np.array_equal(wrong, ref)
    ref2 = ref.copy()
    oracle.weights_tp2ep(ref2, d, src=ref.copy())
    ip2 = ref.copy()
    oracle.weights_tp2ep(ip2, d)
    assert np.array_equal(ip2, ref2)
    wrong2 = ref.copy()
    oracle.weights_tp2ep(wrong2, d, order=1)
    assert not np.array_equal(wrong2, ref2)


def test_weights_byte_accounting_table1():
    """§4.3 Table 1: the fused path writes every element once.  Written bytes
    per layer = 2 * P * (W13 + W2 bytes of one rank); nothing else changes."""
    w = SMALL_W.with_(w_sigma=None)
    d = dims_of(w)
    L = oracle.layout(d)
    src = fill_regions(L, w, seed=4)
    # destination pre-filled with a sentinel that the data never holds
    src.view(np.uint16)[src.view(np.uint16) == 0xFFFF] = 0
    dst = np.full_like(src, 0xFF)
    oracle.weights_ep2tp(dst, d, src=src)
    written = int((dst.view(np.uint16) != 0xFFFF).sum()) * 2
    per_rank = (d.E // d.P) * (2 * d.I * d.H + d.H * d.I) * 2
    assert written == d.N * d.P * per_rank


# ----------------------------------------------------------------------------- KV

def _kv_setup(w, seed=0):
    d = dims_of(w)
    L = oracle.layout(d)
    st = initial_kv_state(w, d, L, seed=seed)
    buf = fill_regions(L, w, seed=seed + 100)
    return d, L, st, buf


def _attention(Kt, Vt, qv):
    s = Kt @ qv / math.sqrt(len(qv))
    p = np.exp(s - s.max())
    p /= p.sum()
    return p @ Vt


@pytest.mark.parametrize("w", [TINY.with_(kv_sigma=1.0), SMALL_KV,
                               SMALL_KV.with_(Hkv=8, D=4), SMALL_KV.with_(Hkv=1)])
def test_kv_tp_heads_compute_the_same_attention(w):
    """§3, §3.2: after EP->TP every rank holding head h computes the same
    decode attention for every request and head as the EP owner did."""
    d, L, st, buf = _kv_setup(w)
    before = buf.copy()
    assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    rng = np.random.default_rng(1)
    for layer in range(d.N):
        for k in range(len(st.lens)):
            n, o = int(st.lens[k]), int(st.owner[k])
            Ke = gather_tokens(kv_ep(before, L, d, o, layer + 1, 0), st.ep_pt[k], n)
            Ve = gather_tokens(kv_ep(before, L, d, o, layer + 1, 1), st.ep_pt[k], n)
            for q in range(d.P):
                Kt = gather_tokens(kv_tp(buf, L, d, q, layer, 0), st.tp_pt[k], n)
                Vt = gather_tokens(kv_tp(buf, L, d, q, layer, 1), st.tp_pt[k], n)
                for hl, h in enumerate(heads_of_rank(d.P, d.Hkv, q)):
                    qv = rng.normal(size=d.D)
                    a_ep = _attention(bf16_to_f64(Ke[:, h]), bf16_to_f64(Ve[:, h]), qv)
                    a_tp = _attention(bf16_to_f64(Kt[:, hl]), bf16_to_f64(Vt[:, hl]), qv)
                    np.testing.assert_array_equal(a_tp, a_ep)


def test_kv_golden_head_groups():
    """§3.2 example: 4 KV heads at TP-8 -> each head on 2 ranks, and the other
    worked cases; checked by where tagged head data lands after EP->TP."""
    for ln in read_golden("kv_heads.txt"):
        head, rest = ln.split(":")
        Hkv, P = ints(head)[-2:]
        want = [ints(x) for x in rest.split(";")]
        w = Workload("g", P=P, N=1, Hkv=Hkv, D=2, ps=2, R=1, len_kind="uniform", len_a=3, len_b=3,
                     slack=8.0)
        d, L, st, buf = _kv_setup(w)
        u = buf.view(np.uint16)
        ep = kv_ep(buf, L, d, int(st.owner[0]), 1, 0)
        for h in range(Hkv):
            ep[:, :, h, :] = 1000 + h          # head tag
        u[u == 0] = 1                           # no tag collides with filler
        assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
        for h in range(Hkv):
            ranks = [q for q in range(P) if (kv_tp(buf, L, d, q, 0, 0) == 1000 + h).any()]
            assert ranks == want[h], (Hkv, P, h, ranks)


def test_kv_exactly_once_and_replication_tagged():
    """Every (request, token, head, dim) value appears exactly P/Hkv times
    under TP (once when Hkv >= P), and exactly once after returning to EP."""
    for w in (SMALL_KV.with_(kv_sigma=None), SMALL_KV.with_(Hkv=8, D=4, kv_sigma=None)):
        d, L, st, buf = _kv_setup(w)
        # unique tags on live EP elements (K half only; V half zero)
        tag = 1
        for k in range(len(st.lens)):
            o = int(st.owner[k])
            for c in range(2):
                pages = kv_ep(buf, L, d, o, 1, c)
                for t in range(int(st.lens[k])):
                    p, s = divmod(t, d.ps)
                    for h in range(d.Hkv):
                        pages[st.ep_pt[k, p], s, h, :] = np.arange(tag, tag + d.D) if c == 0 else 0
                        tag += d.D if c == 0 else 0
        ntag = tag - 1
        assert ntag < 65536
        for r in range(d.P):               # clear everything else in the TP slot
            for c in range(2):
                kv_tp(buf, L, d, r, 0, c)[:] = 0
        assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
        got = np.concatenate([kv_tp(buf, L, d, q, 0, 0).ravel() for q in range(d.P)])
        cnt = np.bincount(got.astype(np.int64), minlength=ntag + 1)[1:]
        assert (cnt == max(1, d.P // d.Hkv)).all()


def test_kv_round_trip_is_logically_identity():
    """EP -> TP -> EP with the greedy placement and fresh pages: every live
    (request, token, half, head, dim) value is back, now under its new owner's
    pages (§3.2: no request dropped, same position).  Head sharing (Hkv < P),
    one head per rank, and two heads per TP rank (Hkv = 2P: the TP page holds
    a rank's heads side by side)."""
    for w in (TINY, SMALL_KV.with_(kv_sigma=None), SMALL_KV.with_(Hkv=8, D=4, kv_sigma=None)):
        d, L, st, buf = _kv_setup(w)
        orig = buf.copy()
        assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
        owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
        ep_free2 = synth.permutation(9, 4, L["pages_ep"], rows=d.P)
        fl, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, st.ep_pt.shape[1], ep_free2,
                                         region=owner2, key=st.tp_pos)
        assert fl == 0
        assert oracle.kv_tp2ep(buf, d, st.lens, owner2, ep_pt2, st.tp_pt) == 0
        for layer in range(d.N):
            for k in range(len(st.lens)):
                n = int(st.lens[k])
                for c in range(2):
                    a = gather_tokens(kv_ep(orig, L, d, int(st.owner[k]), layer + 1, c), st.ep_pt[k], n)
                    b = gather_tokens(kv_ep(buf, L, d, int(owner2[k]), layer + 1, c), ep_pt2[k], n)
                    np.testing.assert_array_equal(a, b)


def test_kv_hkv_equals_p_is_a_head_transpose():
    """Hkv = P: TP rank q's page = the EP page's head q (numpy slice)."""
    w = SMALL_KV.with_(Hkv=4, kv_sigma=None)
    d, L, st, buf = _kv_setup(w)
    before = buf.copy()
    assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    for k in range(len(st.lens)):
        n = int(st.lens[k])
        for p in range(n // d.ps):              # full pages only
            src = kv_ep(before, L, d, int(st.owner[k]), 1, 0)[st.ep_pt[k, p]]
            for q in range(d.P):
                np.testing.assert_array_equal(kv_tp(buf, L, d, q, 0, 0)[st.tp_pt[k, p], :, 0, :],
                                              src[:, q, :])


def test_kv_single_request_matches_torch_index_select():
    """One request of whole pages: the TP K cache of the head-0 rank equals
    torch.index_select over the page-flattened EP cache."""
    torch = pytest.importorskip("torch")
    w = SMALL_KV.with_(R=1, len_a=12, len_b=12, kv_sigma=None, slack=4.0)   # 3 full pages of 4
    d, L, st, buf = _kv_setup(w)
    before = buf.copy()
    assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    ep = torch.from_numpy(kv_ep(before, L, d, int(st.owner[0]), 1, 0).astype(np.int32))
    tp = torch.from_numpy(kv_tp(buf, L, d, 0, 0, 0).astype(np.int32))
    npg = 3
    want = torch.index_select(ep, 0, torch.tensor(st.ep_pt[0, :npg], dtype=torch.long))[:, :, 0, :]
    got = torch.index_select(tp, 0, torch.tensor(st.tp_pt[0, :npg], dtype=torch.long))[:, :, 0, :]
    assert torch.equal(got, want)


def test_kv_untouched_bytes_and_byte_accounting():
    """Only live token rows are written; every other byte keeps its contents.
    Bytes written per layer EP->TP =
    tokens * max(P, Hkv) * D * 2 halves * 2 B; TP->EP = tokens * Hkv * D * 4 B."""
    w = SMALL_KV.with_(kv_sigma=None)
    d, L, st, src = _kv_setup(w)
    u = src.view(np.uint16)
    u[u == 0xFFFF] = 0
    dst = np.full_like(src, 0xFF)
    assert oracle.kv_ep2tp(dst, d, st.lens, st.owner, st.ep_pt, st.tp_pt, src=src) == 0
    T = int(st.lens.sum())
    written = int((dst.view(np.uint16) != 0xFFFF).sum()) * 2
    assert written == d.N * T * max(d.P, d.Hkv) * d.D * 4
    dst2 = np.full_like(src, 0xFF)
    assert oracle.kv_tp2ep(dst2, d, st.lens, st.owner, st.ep_pt, st.tp_pt, src=src) == 0
    written2 = int((dst2.view(np.uint16) != 0xFFFF).sum()) * 2
    assert written2 == d.N * T * d.Hkv * d.D * 4


def test_kv_layer_order_in_place():
    w = SMALL_KV.with_(kv_sigma=None)
    d, L, st, orig = _kv_setup(w)
    ref = orig.copy()
    oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, st.tp_pt, src=orig.copy())
    ip = orig.copy()
    oracle.kv_ep2tp(ip, d, st.lens, st.owner, st.ep_pt, st.tp_pt)
    assert np.array_equal(ip, ref)
    wrong = orig.copy()
    oracle.kv_ep2tp(wrong, d, st.lens, st.owner, st.ep_pt, st.tp_pt, order=-1)
    assert not np.array_equal(wrong, ref)


def test_kv_validation_flags():
    """§4.5 capacity check and §3.2 page tables: invalid inputs are refused
    before anything moves (buffer unchanged)."""
    w = SMALL_KV.with_(kv_sigma=None)
    d, L, st, buf = _kv_setup(w)
    orig = buf.copy()

    def run(**ch):
        a = dict(lens=st.lens.copy(), owner=st.owner.copy(), ep_pt=st.ep_pt.copy(), tp_pt=st.tp_pt.copy())
        for key, fn in ch.items():
            fn(a[key])
        b = orig.copy()
        fl = oracle.kv_ep2tp(b, d, a["lens"], a["owner"], a["ep_pt"], a["tp_pt"])
        if fl:
            assert np.array_equal(b, orig)
        return fl

    assert run() == 0
    assert run(lens=lambda x: x.__setitem__(0, -1)) == oracle.F_BAD_REQUEST
    assert run(owner=lambda x: x.__setitem__(1, d.P)) == oracle.F_BAD_REQUEST
    assert run(ep_pt=lambda x: x.__setitem__((0, 0), L["pages_ep"])) == oracle.F_PAGE_OOB
    assert run(tp_pt=lambda x: x.__setitem__((0, 0), -1)) == oracle.F_PAGE_OOB
    k2 = int(np.argmax(st.lens > d.ps))
    assert run(tp_pt=lambda x: x.__setitem__((k2, 1), x[0, 0])) == oracle.F_DUP_PAGE
    small = dims_of(w, pages_tp=int(synth.npages(st.lens, d.ps).sum()) - 2)
    assert oracle.kv_validate(small, 0, st.lens, st.owner, st.ep_pt, np.zeros_like(st.tp_pt)) \
        & oracle.F_CAPACITY
    # TP -> EP: two requests claiming the same TP page
    owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
    free2 = synth.permutation(8, 4, L["pages_ep"], rows=d.P)
    _, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, st.ep_pt.shape[1], free2, region=owner2, key=st.tp_pos)
    assert oracle.kv_validate(d, 1, st.lens, owner2, ep_pt2, st.tp_pt) == 0
    bad_tp = st.tp_pt.copy()
    bad_tp[k2, 1] = bad_tp[0, 0]
    assert oracle.kv_validate(d, 1, st.lens, owner2, ep_pt2, bad_tp) == oracle.F_DUP_PAGE
    # TP -> EP: one EP rank asked to hold more than its pool
    many = np.zeros_like(st.owner)
    fl = oracle.kv_validate(d, 1, st.lens, many, st.ep_pt, st.tp_pt)
    assert fl & oracle.F_CAPACITY or fl & oracle.F_DUP_PAGE


def test_kv_validation_boundaries():
    """The bounds of the §4.5 capacity check and of the §3.2 page ids, worked
    by hand: P = 2 ranks, Hkv = 2 (one head per TP rank), page size 4, a TP
    pool of 8 pages (so 8 * h_tp / Hkv = 4 EP pages per rank) and room for 8
    descriptors.  Lengths 9, 4, 7, 3, 2 take 3 + 1 + 2 + 1 + 1 = 8 pages; EP
    owners 0, 1, 1, 0, 1 give rank 0 pages 3 + 1 = 4 and rank 1 1 + 2 + 1 = 4:
    every pool exactly full, which both directions accept.  One token more on
    the last request (5 tokens, 2 pages) overflows the TP pool, the
    descriptor room and rank 1's EP pool; a page id equal to its pool size is
    out of range."""
    d = oracle.Dims(P=2, N=1, Hkv=2, D=4, ps=4, pages_tp=8, max_requests=5, max_pages=8)
    assert oracle.layout(d)["pages_ep"] == 4
    lens = np.array([9, 4, 7, 3, 2], np.int32)
    owner = np.array([0, 1, 1, 0, 1], np.int32)
    ep_pt = np.full((5, 3), -1, np.int32)
    tp_pt = np.full((5, 3), -1, np.int32)
    ep_pt[0, :3], ep_pt[3, 0] = [0, 1, 2], 3             # rank 0: EP pages 0..3
    ep_pt[1, 0], ep_pt[2, :2], ep_pt[4, 0] = 0, [1, 2], 3  # rank 1: EP pages 0..3
    tp_pt[0, :3], tp_pt[1, 0], tp_pt[2, :2], tp_pt[3, 0], tp_pt[4, 0] = [0, 1, 2], 3, [4, 5], 6, 7
    for direction in (0, 1):
        assert oracle.kv_validate(d, direction, lens, owner, ep_pt, tp_pt) == 0
        longer = lens.copy()
        longer[4] = 5
        ep2, tp2 = ep_pt.copy(), tp_pt.copy()
        ep2[4, 1], tp2[4, 1] = 0, 0                      # ids of the extra page (never reached)
        assert oracle.kv_validate(d, direction, longer, owner, ep2, tp2) == oracle.F_CAPACITY
        bad = tp_pt.copy()
        bad[3, 0] = 8                                     # = pages_tp
        assert oracle.kv_validate(d, direction, lens, owner, ep_pt, bad) == oracle.F_PAGE_OOB
        bad = ep_pt.copy()
        bad[3, 0] = 4                                     # = pages_ep
        assert oracle.kv_validate(d, direction, lens, owner, bad, tp_pt) == oracle.F_PAGE_OOB
    # TP -> EP only: rank 1 one page over its pool while the totals still fit
    owner2 = owner.copy()
    owner2[3] = 1                                         # rank 1: 4 + 1 = 5 > 4
    assert oracle.kv_validate(d, 1, lens, owner2, ep_pt, tp_pt) == oracle.F_CAPACITY
    assert oracle.kv_validate(d, 0, lens, owner2, ep_pt, tp_pt) == 0


def test_kv_descriptors_cover_every_live_token():
    w = SMALL_KV
    d, L, st, _ = _kv_setup(w)
    desc = oracle.kv_descriptors(d, 0, st.lens, st.owner, st.ep_pt, st.tp_pt)
    assert len(desc) == int(synth.npages(st.lens, d.ps).sum())
    assert int(desc[:, 6].sum()) == int(st.lens.sum())
    assert (np.diff(desc[:, 2]) >= 0).all()                  # grouped by source rank
    assert set(map(tuple, desc[:, :2].tolist())) == {(k, p) for k in range(len(st.lens))
                                                      for p in range(int(synth.npages(st.lens[k:k + 1], d.ps)[0]))}


# ----------------------------------------------------------------------------- requests

def test_placement_golden():
    for ln in read_golden("placement_lpt.txt"):
        head, lens, key, owner, local, mx = ln.split("|")[0].split(":")[0], *ln.split(":", 1)[1].split("|")
        P = ints(head.split("P=")[1])[0]
        lens_v = ints(lens)
        key_v = None if key.strip() == "-" else ints(key)
        o, lp, m = oracle.place(P, lens_v, key_v)
        assert o.tolist() == ints(owner), ln
        assert lp.tolist() == ints(local), ln
        assert m == ints(mx)[0], ln


def test_placement_deterministic_and_conserving():
    lens = synth.lengths_lognormal(0, 300, 2048, 1.0, 32768)
    a = oracle.place(8, lens)
    oracle.set_threads(4)
    b = oracle.place(8, lens)
    oracle.set_threads(1)
    assert all(np.array_equal(x, y) for x, y in zip(a[:2], b[:2]))
    owner, local, mx = a
    loads = np.bincount(owner, weights=lens, minlength=8)
    assert loads.sum() == lens.sum() and loads.max() == mx
    for q in range(8):                        # local positions are 0..n_q-1 in list order
        ks = np.flatnonzero(owner == q)
        assert local[ks].tolist() == list(range(len(ks)))


def test_placement_lpt_bound_against_brute_force():
    """Graham's bound for longest-processing-time-first list scheduling:
    max load <= (4/3 - 1/(3P)) * OPT, OPT found by enumerating all P^R."""
    rng = np.random.default_rng(3)
    for _ in range(40):
        P = int(rng.integers(2, 4))
        R = int(rng.integers(1, 8))
        lens = rng.integers(1, 50, R)
        _, _, mx = oracle.place(P, lens)
        opt = min(max(np.bincount(np.array(a), weights=lens, minlength=P))
                  for a in itertools.product(range(P), repeat=R))
        assert mx <= (4 / 3 - 1 / (3 * P)) * opt + 1e-9
        assert mx >= opt


def test_placement_matches_heap_list_scheduling():
    """Same result as a textbook min-heap list scheduler over the sorted list."""
    import heapq
    rng = np.random.default_rng(8)
    for _ in range(30):
        P = int(rng.integers(1, 9))
        R = int(rng.integers(0, 60))
        lens = rng.integers(1, 20, R)        # many ties on purpose
        key = rng.permutation(R)
        heap = [(0, q) for q in range(P)]
        want = np.zeros(R, dtype=np.int64)
        for k in sorted(range(R), key=lambda k: (-lens[k], key[k])):
            load, q = heapq.heappop(heap)
            want[k] = q
            heapq.heappush(heap, (load + lens[k], q))
        got, _, _ = oracle.place(P, lens, key)
        assert got.tolist() == want.tolist()


def test_request_order_golden():
    for ln in read_golden("request_order.txt"):
        head, rest = ln.split(":")
        P = ints(head)[0]
        owner, want = rest.split("|")
        assert oracle.request_order(P, ints(owner)).tolist() == ints(want)


def test_assign_pages_golden_and_capacity():
    g = {ln.split(":")[0].strip(): ln.split(":")[1] for ln in read_golden("assign_pages.txt")}
    fl, pt = oracle.assign_pages(1, ints(g["lens"]), 16, ints(g["maxp"])[0], ints(g["free"]),
                                 key=ints(g["key"]))
    assert fl == 0
    assert pt.tolist() == [ints(r) for r in g["table"].split("|")]
    fl, pt = oracle.assign_pages(1, [100, 100], 16, 8, list(range(13)))
    assert fl == oracle.F_CAPACITY and (pt == -7).all()      # nothing written


# ----------------------------------------------------------------------------- generator

def test_generator_normal_table_and_raw():
    t = synth.normal_table(0.02)
    v = bf16_to_f64(t)
    assert (np.diff(v) >= 0).all()
    assert abs(v.mean()) < 1e-4 and abs(v.std() - 0.02) < 2e-4
    x = synth.values_at(0, np.arange(1 << 16))
    assert len(np.unique(x)) > 40000
    a = synth.fill_host(1000, 5, base=123)
    assert np.array_equal(a, synth.values_at(5, np.arange(123, 1123)))


# ----------------------------------------------------------------------------- attention (memory-saving variant)

from helpers import attn_full_qkv, attn_full_wo, attn_shard_qkv, attn_shard_wo  # noqa: E402

ATTN = [Workload("attn_hkv2_p4", P=4, N=2, H=12, Hkv=2, D=4, Hq=8, w_sigma=0.5),
        Workload("attn_hkv8_p4", P=4, N=2, H=8, Hkv=8, D=2, Hq=4, w_sigma=0.5),
        Workload("attn_hkv4_p4", P=4, N=3, H=6, Hkv=4, D=3, Hq=12, w_sigma=0.5)]


def _attn_setup(w, seed):
    """EP state: the same full copy on every rank (DP attention replicas)."""
    d = dims_of(w)
    L = oracle.layout(d)
    buf = fill_regions(L, w, seed=seed)
    for r in range(1, d.P):
        for s in range(d.N + 1):
            a = L["attnslots_off"] + s * L["attnslot_stride"]
            buf[r * L["region_stride"] + a: r * L["region_stride"] + a + L["attnslot_stride"]] = \
                buf[a:a + L["attnslot_stride"]]
    return d, L, buf


def test_attn_golden_hand_worked():
    g = read_golden("attn_p2_hq2_hkv1.txt")
    kv = {ln.split()[0]: int(ln.split()[1]) for ln in g if ln.split()[0] in ("P", "Hq", "Hkv", "D", "H")}
    d = oracle.Dims(P=kv["P"], H=kv["H"], N=1, Hkv=kv["Hkv"], D=kv["D"], ps=1, pages_tp=1, Hq=kv["Hq"])
    L = oracle.layout(d)
    buf = np.zeros(L["ws_off"], dtype=np.uint8)
    for r in range(d.P):
        qkv = attn_full_qkv(buf, L, d, r, 1)
        for hh in range(d.Hq + 2 * d.Hkv):
            qkv[hh] = 10 * hh + np.arange(d.H)
        wo = attn_full_wo(buf, L, d, r, 1)
        for i in range(d.H):
            wo[i] = 100 + 10 * i + np.arange(d.Hq * d.D)
    oracle.attn_ep2tp(buf, d)
    n = 0
    for ln in g:
        name, rest = ln.split(" ", 1)
        if name not in ("shard_qkv", "shard_wo"):
            continue
        head, vals = rest.split(":")
        q = ints(head)[0]
        got = (attn_shard_qkv if name == "shard_qkv" else attn_shard_wo)(buf, L, d, q, 0).ravel().tolist()
        assert got == ints(vals), (name, q)
        n += 1
    assert n == 4


@pytest.mark.parametrize("w", ATTN, ids=lambda w: w.name)
def test_attn_tp_shards_compute_the_same_projections(w):
    """§3: the TP shards compute the same function.  Every rank's query/key/
    value projections equal the full copy's for its heads, and the sum over
    ranks of their output-projection partials equals the full output
    projection (the All-Reduce of row-parallel Wo)."""
    d, L, buf = _attn_setup(w, 3)
    before = buf.copy()
    oracle.attn_ep2tp(buf, d)
    rng = np.random.default_rng(2)
    hq = d.Hq // d.P
    for layer in range(d.N):
        x = rng.normal(size=d.H)
        u = rng.normal(size=(d.Hq, d.D))
        full_qkv = bf16_to_f64(attn_full_qkv(before, L, d, 0, layer + 1))
        full_wo = bf16_to_f64(attn_full_wo(before, L, d, 0, layer + 1))
        y_full = full_wo @ u.ravel()
        y_tp = np.zeros(d.H)
        for q in range(d.P):
            sq = bf16_to_f64(attn_shard_qkv(buf, L, d, q, layer))
            heads = list(range(q * hq, (q + 1) * hq))
            kvh = heads_of_rank(d.P, d.Hkv, q)
            want = [full_qkv[h] for h in heads] + [full_qkv[d.Hq + h] for h in kvh] + \
                   [full_qkv[d.Hq + d.Hkv + h] for h in kvh]
            for b, wrow in enumerate(want):      # one head: Dh rows of H
                np.testing.assert_array_equal(sq[b].reshape(d.D, d.H) @ x, wrow.reshape(d.D, d.H) @ x)
            wo_q = bf16_to_f64(attn_shard_wo(buf, L, d, q, layer))
            y_tp += wo_q @ u[heads].ravel()
        np.testing.assert_allclose(y_tp, y_full, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("w", ATTN, ids=lambda w: w.name)
def test_attn_round_trip_and_layer_order(w):
    """EP -> TP -> EP restores every rank's full copy (all-gather), the
    in-place layer orders equal the snapshot definition, and slot N is not a
    destination of EP->TP."""
    d, L, orig = _attn_setup(w.with_(w_sigma=None), 5)
    buf = orig.copy()
    oracle.attn_ep2tp(buf, d)
    snap = orig.copy()
    oracle.attn_ep2tp(snap, d, src=orig.copy())
    assert np.array_equal(buf, snap)
    for r in range(d.P):
        a = r * L["region_stride"] + L["attnslots_off"] + d.N * L["attnslot_stride"]
        assert np.array_equal(buf[a:a + L["attnslot_stride"]], orig[a:a + L["attnslot_stride"]])
    mid = buf.copy()
    oracle.attn_tp2ep(buf, d)
    snap2 = mid.copy()
    oracle.attn_tp2ep(snap2, d, src=mid.copy())
    assert np.array_equal(buf, snap2)
    for r in range(d.P):
        a = r * L["region_stride"] + L["attnslots_off"] + L["attnslot_stride"]
        b = r * L["region_stride"] + L["attnslots_off"] + (d.N + 1) * L["attnslot_stride"]
        assert np.array_equal(buf[a:b], orig[a:b]), r


# ----------------------------------------------------------------------------- element maps

# The element maps (w13_tp_elem, w2_tp_elem, kv_elem) name, for one element,
# its EP and TP byte offsets; the full-size GPU tests check samples and whole
# slots through them.  Here they are pinned to the whole-buffer switch
# functions above (themselves pinned by goldens, equivalence and brute
# force): on random 16-bit contents, the destination the map names must hold,
# after the switch, the value at the source it names, for every element.

@pytest.mark.parametrize("split", [0, 1])
@pytest.mark.parametrize("w", [TINY, SMALL_W], ids=lambda w: w.name)
def test_weight_element_maps_agree_with_the_switch(w, split):
    d = dims_of(w, w13_split=split)
    L = oracle.layout(d)
    before = fill_regions(L, w.with_(w_sigma=None), seed=11)
    after = before.copy()
    oracle.weights_ep2tp(after, d)
    b16, a16 = before.view(np.uint16), after.view(np.uint16)
    Ip = d.I // d.P
    dst_seen = set()
    for layer in range(d.N):
        for q in range(d.P):
            for e in range(d.E):
                for h in range(d.H):
                    for row in range(2 * Ip):
                        s, t = oracle.w13_tp_elem(d, q, e, row, h, layer + 1, layer)
                        assert a16[t // 2] == b16[s // 2], ("w13", layer, q, e, row, h)
                        dst_seen.add(t)
                    for c in range(Ip):
                        s, t = oracle.w2_tp_elem(d, q, e, h, c, layer + 1, layer)
                        assert a16[t // 2] == b16[s // 2], ("w2", layer, q, e, h, c)
                        dst_seen.add(t)
    # the maps name every TP element once: as many distinct destinations as
    # TP elements in the N destination slots
    assert len(dst_seen) == d.N * d.P * d.E * 3 * Ip * d.H


@pytest.mark.parametrize("w", [SMALL_KV.with_(kv_sigma=None), SMALL_KV.with_(Hkv=8, D=4, kv_sigma=None),
                               SMALL_KV.with_(P=8, Hkv=2, D=4, kv_sigma=None)],
                         ids=["hkv2_p4", "hkv8_p4", "hkv2_p8"])
def test_kv_element_map_agrees_with_the_switch(w):
    """EP->TP: every TP replica of every live element holds the value at the
    EP offset the map names.  TP->EP (greedy owners, new pages): every EP
    element holds the value at the TP offset (lowest replica) the map names."""
    d, L, st, buf = _kv_setup(w, seed=4)
    ep2tp = buf.copy()
    assert oracle.kv_ep2tp(ep2tp, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
    maxp = st.ep_pt.shape[1]
    _, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, maxp, synth.permutation(9, 4, L["pages_ep"], d.P),
                                    region=owner2, key=st.tp_pos)
    tp2ep = ep2tp.copy()
    assert oracle.kv_tp2ep(tp2ep, d, st.lens, owner2, ep_pt2, st.tp_pt) == 0
    b16, m16, a16 = buf.view(np.uint16), ep2tp.view(np.uint16), tp2ep.view(np.uint16)
    checked = 0
    for k in range(len(st.lens)):
        for t in range(int(st.lens[k])):
            p, s = divmod(t, d.ps)
            for layer in range(d.N):
                for c in range(2):
                    for h in range(d.Hkv):
                        holders = [q for q in range(d.P) if h in heads_of_rank(d.P, d.Hkv, q)]
                        for e in range(d.D):
                            for q in holders:
                                a, b = oracle.kv_elem(d, int(st.owner[k]), q, int(st.ep_pt[k, p]),
                                                      int(st.tp_pt[k, p]), s, c, h, e, layer + 1, layer)
                                assert m16[b // 2] == b16[a // 2], ("ep2tp", k, t, layer, c, h, e, q)
                                checked += 1
                            a, b = oracle.kv_elem(d, int(owner2[k]), holders[0], int(ep_pt2[k, p]),
                                                  int(st.tp_pt[k, p]), s, c, h, e, layer + 1, layer)
                            assert a16[a // 2] == m16[b // 2], ("tp2ep", k, t, layer, c, h, e)
    assert checked == int(st.lens.sum()) * d.N * 2 * max(d.P, d.Hkv) * d.D
    # a rank that does not hold the head gets no offsets
    q_not = next((q for q in range(d.P) if 0 not in heads_of_rank(d.P, d.Hkv, q)), None)
    if q_not is not None:
        assert oracle.kv_elem(d, 0, q_not, 0, 0, 0, 0, 0, 0, 1, 0) == (-1, -1)
