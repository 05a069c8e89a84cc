"""KV EP->TP through the TMA copy on an EP page pool of more than 2^31 token
rows (pages x page size), and back through the LSU copy.

Tensor-map coordinates are signed 32-bit.  The TMA copy addresses an EP page
by {element, head, row in page, page, region}, so the coordinate is the page
id (below 2^31 for every pool the handle accepts), never the page's first
row.  Here one rank (P = 1), one KV head of 8 elements and 16-token pages
give a pool of 2^27 + 64 pages = 2^31 + 1024 rows per half (about 129 GiB on
the device).  The requests' pages include the highest page ids and the ones
around row 2^31; every live element is checked against the oracle's element
map (§3.2 paged KV through the page tables), together with the tail rows of
last pages, which must keep their bytes."""
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

PAGES = 2**27 + 64
BIG = Workload("kv_p1_1layer_hkv1_d8_2p31rows", P=1, N=1, Hkv=1, D=8, ps=16, R=6)
LENS = np.array([16 * 5 + 3, 32, 7, 16 * 4 + 15, 1, 48], dtype=np.int32)


def _pages(first_high: int, seed: int) -> np.ndarray:
    """18 distinct page ids: the six highest of the pool, five around page
    2^27 (row 2^31), seven low ones; shuffled."""
    ids = [first_high - i for i in range(6)] + [2**27 + i for i in (-2, -1, 0, 1, 2)] + \
        [0, 1, 2, 1000, 99999, 2**26, 2**26 + 7]
    assert len(set(ids)) == 18 == int(synth.npages(LENS, 16).sum())
    return np.random.default_rng(seed).permutation(np.array(ids, dtype=np.int64))


def _table(ids: np.ndarray, maxp: int) -> np.ndarray:
    pt = np.full((len(LENS), maxp), -1, dtype=np.int32)
    i = 0
    for k, n in enumerate(synth.npages(LENS, 16)):
        pt[k, :n] = ids[i:i + n]
        i += n
    return pt


def _elements(d, ep_pt, tp_pt, ep_slot, tp_slot):
    """(source, destination) u16 offsets of every live element, from the oracle."""
    src, dst = [], []
    for k, n in enumerate(LENS):
        for t in range(int(n)):
            p, row = divmod(t, 16)
            for c in range(2):
                for e in range(8):
                    a, b = oracle.kv_elem(d, 0, 0, int(ep_pt[k, p]), int(tp_pt[k, p]), row, c, 0, e, ep_slot,
                                          tp_slot)
                    src.append(a // 2)
                    dst.append(b // 2)
    return np.array(src, np.int64), np.array(dst, np.int64)


def _gather(dev, idx):
    return dev.u16()[torch.from_numpy(idx).cuda()].cpu().numpy()


def _value(dev, idx):
    return synth.values_at(dev.seed, idx.astype(np.uint64)).view(np.int16)


@pytest.mark.parametrize("checked", [False, True], ids=["libumm", "libumm_checked"])
def test_tma_copy_past_2p31_ep_rows(checked):
    over = dict(pages_tp=PAGES, max_requests=len(LENS), max_pages=64)
    need = umm.umm_required_bytes(umm.make_dims(P=1, N=1, Hkv=1, D=8, ps=16, **over))
    torch.cuda.empty_cache()
    if torch.cuda.mem_get_info()[0] < need + (2 << 30):
        pytest.skip(f"needs {need / 2**30:.1f} GiB of free device memory")
    ctx = umm.checked_library() if checked else _null()
    with ctx:
        dev = DevUMM(BIG, seed=11, **over)
        L, d = dev.L, dev.d
        assert L["pages_ep"] == PAGES and L["pages_ep"] * 16 > 2**31
        O = oracle.layout(d)
        assert all(L[k] == O[k] for k in O)
        assert umm.umm_kv_copy_kernel(dev.dims, 0) == (umm.UMM_KV_COPY_TMA, 0)
        maxp = 6
        ep_pt = _table(_pages(PAGES - 1, 1), maxp)
        tp_pt = _table(_pages(PAGES - 1, 2), maxp)
        owner = np.zeros(len(LENS), np.int32)
        # EP slot 1 -> TP slot 0
        umm.reshard_kv_ep2tp(dev.h, len(LENS), maxp, i32(LENS), i32(owner), i32(ep_pt), i32(tp_pt))
        torch.cuda.synchronize()
        assert dev.status() == (0, 0)
        src, dst = _elements(d, ep_pt, tp_pt, 1, 0)
        assert src.max() * 2 > L["kvslots_off"] + L["kvslot_stride"] + 2**31 * 16   # rows past 2^31 were read
        np.testing.assert_array_equal(_gather(dev, dst), _value(dev, src))
        # tail rows of each last TP page keep their bytes
        for k, n in enumerate(LENS.tolist()):
            if n % 16:
                for c in range(2):
                    base = (L["kvslots_off"] + c * L["kv_v_off"]) // 2 + int(tp_pt[k, (n - 1) // 16]) * 16 * 8
                    idx = np.arange(base + (n % 16) * 8, base + 16 * 8)
                    np.testing.assert_array_equal(_gather(dev, idx), _value(dev, idx))
        # back: TP slot 0 -> EP slot 1, to new pages (the highest ones again)
        ep_pt1 = _table(_pages(PAGES - 1, 3), maxp)
        umm.reshard_kv_tp2ep(dev.h, len(LENS), maxp, i32(LENS), i32(owner), i32(ep_pt1), i32(tp_pt))
        torch.cuda.synchronize()
        assert dev.status() == (0, 0)
        # the same elements, now at their new EP pages, hold their original values
        at1, _ = _elements(d, ep_pt1, tp_pt, 1, 0)
        np.testing.assert_array_equal(_gather(dev, at1), _value(dev, src))
        dev.close()


class _null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False
