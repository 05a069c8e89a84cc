"""Test helpers: tensor views of a host copy of the unified buffer, bf16
decoding, and construction of seeded initial states with the oracle.

The views follow the shapes of §3.1 (weights) and §3.2 (paged KV, token-major
pages of [page_size][heads][head_dim]) of "Moebius: Serving Mixture-of-Expert
Models with Seamless Runtime Parallelism Switch" at the byte offsets of a
layout dictionary (from the oracle or from the library).
"""
from __future__ import annotations

import re
from dataclasses import dataclass
from pathlib import Path

import numpy as np

import oracle
import synth
from synth.workloads import Workload

GOLDEN = Path(__file__).parent / "golden"


def u16(buf: np.ndarray, off: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    assert off % 2 == 0
    return buf[off:off + 2 * n].view(np.uint16).reshape(shape)


def wslot(L: dict, r: int, s: int) -> int:
    return r * L["region_stride"] + s * L["wslot_stride"]


def kvslot(L: dict, r: int, s: int, c: int) -> int:
    return r * L["region_stride"] + L["kvslots_off"] + s * L["kvslot_stride"] + c * L["kv_v_off"]


def w13_ep(buf, L, d, r, s):
    return u16(buf, wslot(L, r, s) + L["w13_off"], (d.E // d.P, 2 * d.I, d.H))


def w2_ep(buf, L, d, r, s):
    return u16(buf, wslot(L, r, s) + L["w2_off"], (d.E // d.P, d.H, d.I))


def w13_tp(buf, L, d, q, s):
    return u16(buf, wslot(L, q, s) + L["w13_off"], (d.E, 2 * (d.I // d.P), d.H))


def w2_tp(buf, L, d, q, s):
    return u16(buf, wslot(L, q, s) + L["w2_off"], (d.E, d.H, d.I // d.P))


def kv_ep(buf, L, d, r, s, c):
    return u16(buf, kvslot(L, r, s, c), (L["pages_ep"], d.ps, d.Hkv, d.D))


def kv_tp(buf, L, d, q, s, c):
    return u16(buf, kvslot(L, q, s, c), (L["pages_tp"], d.ps, L["h_tp"], d.D))


def bf16_to_f64(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def heads_of_rank(P: int, Hkv: int, q: int) -> list[int]:
    """Heads rank q keeps under TP (reading of §3.2's head split)."""
    if Hkv >= P:
        per = Hkv // P
        return list(range(q * per, (q + 1) * per))
    return [q * Hkv // P]


def gather_tokens(pages: np.ndarray, pt_row: np.ndarray, n: int) -> np.ndarray:
    """Paged read (PagedAttention style): token t sits at page pt[t // ps],
    slot t % ps.  pages: [npages][ps][...]."""
    ps = pages.shape[1]
    t = np.arange(n)
    return pages[pt_row[t // ps], t % ps]


def dims_of(w: Workload, **over) -> oracle.Dims:
    kw = w.dims()
    kw.update(over)
    return oracle.Dims(**kw)


@dataclass
class KVState:
    lens: np.ndarray
    owner: np.ndarray
    ep_pt: np.ndarray
    tp_pt: np.ndarray
    tp_pos: np.ndarray


def initial_kv_state(w: Workload, d: oracle.Dims, L: dict, seed: int = 0) -> KVState:
    """EP owners by the greedy rule, EP pages from per-rank permutations of the
    pool (local order), TP pages from a permutation of the TP pool in all-gather
    order.  Built with the oracle (tests only)."""
    lens = w.lengths()
    maxp = w.max_pages_per_req()
    owner, _, _ = oracle.place(d.P, lens)
    ep_free = synth.permutation(seed, 2, L["pages_ep"], rows=d.P)
    fl, ep_pt = oracle.assign_pages(d.P, lens, d.ps, maxp, ep_free, region=owner)
    assert fl == 0
    tp_pos = oracle.request_order(d.P, owner)
    tp_free = synth.permutation(seed, 3, L["pages_tp"], rows=1)
    fl, tp_pt = oracle.assign_pages(1, lens, d.ps, maxp, tp_free, key=tp_pos)
    assert fl == 0
    return KVState(lens, owner, ep_pt, tp_pt, tp_pos)


def fill_regions(L: dict, w: Workload, seed: int) -> np.ndarray:
    """Host copy of the unified buffer: regions part filled from the generator
    (weights and KV slots in their modes), workspace zero."""
    total = L["ws_off"]
    buf = np.zeros(total, dtype=np.uint8)
    u = buf.view(np.uint16)
    for a, n, mode, sigma in fill_plan(L, w):
        u[a:a + n] = synth.fill_host(n, seed, mode, sigma, base=a)
    return buf


def fill_plan(L: dict, w: Workload):
    """(first u16 index, count, mode, sigma) ranges that make up the initial
    contents: the whole regions part in the weights' mode, then every region's
    KV slots in the KV mode.  Element i always holds synth value i."""
    mode, sigma = w.w_mode()
    plan = [(0, L["ws_off"] // 2, mode, sigma)]
    if w.Hkv:
        kmode, ksig = w.kv_mode()
        for r in range(w.P):
            a = (r * L["region_stride"] + L["kvslots_off"]) // 2
            plan.append((a, (w.N + 1) * L["kvslot_stride"] // 2, kmode, ksig))
    return plan


def read_golden(name: str) -> list[str]:
    lines = []
    for ln in (GOLDEN / name).read_text().splitlines():
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            lines.append(ln)
    return lines


def ints(s: str) -> list[int]:
    return [int(x) for x in re.findall(r"-?\d+", s)]


# ---- attention weights (memory-saving variant): views of one attention slot

def attnslot(L: dict, r: int, s: int) -> int:
    return r * L["region_stride"] + L["attnslots_off"] + s * L["attnslot_stride"]


def attn_full_qkv(buf, L, d, r, s):
    """EP view: [Hq + 2*Hkv heads][Dh * H] (each head Dh rows of H)."""
    return u16(buf, attnslot(L, r, s), (d.Hq + 2 * d.Hkv, d.D * d.H))


def attn_full_wo(buf, L, d, r, s):
    return u16(buf, attnslot(L, r, s) + L["attn_wo_off"], (d.H, d.Hq * d.D))


def attn_shard_qkv(buf, L, d, q, s):
    """TP view of rank q: [Hq/P + 2*h_tp heads][Dh * H]."""
    return u16(buf, attnslot(L, q, s), (d.Hq // d.P + 2 * L["h_tp"], d.D * d.H))


def attn_shard_wo(buf, L, d, q, s):
    return u16(buf, attnslot(L, q, s) + L["attn_wo_off"], (d.H, d.Hq // d.P * d.D))
