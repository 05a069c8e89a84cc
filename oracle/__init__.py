"""CPU oracle of the EP<->TP reshard data plane (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it, and
it never calls the product library: the two share no code.

The arithmetic lives in ``umm_oracle.c`` (plain C, element by element, each
function citing the passage of "Moebius: Serving Mixture-of-Expert Models with
Seamless Runtime Parallelism Switch" it follows); this module compiles it with
gcc and wraps it with ctypes over numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, fields

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "umm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# flag bits an invalid KV / page-assignment call raises (restated in the C file)
F_BAD_REQUEST = 1
F_CAPACITY = 2
F_PAGE_OOB = 4
F_DUP_PAGE = 8


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (OpenMP for the timed CPU baseline)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, u32 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
        vp = ctypes.c_void_p
        L.orc_set_threads.argtypes = [i32]
        L.orc_max_threads.restype = i32
        L.orc_layout.argtypes = [vp, vp]
        for f in ("orc_weights_ep2tp", "orc_weights_tp2ep"):
            getattr(L, f).argtypes = [vp, vp, vp, i32]
        for f in ("orc_attn_ep2tp", "orc_attn_tp2ep"):
            getattr(L, f).argtypes = [vp, vp, vp, i32]
        L.orc_w13_tp_elem.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp, vp]
        L.orc_w2_tp_elem.argtypes = [vp, i64, i64, i64, i64, i64, i64, vp, vp]
        L.orc_kv_validate.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp]
        L.orc_kv_validate.restype = u32
        for f in ("orc_kv_ep2tp", "orc_kv_tp2ep"):
            getattr(L, f).argtypes = [vp, vp, vp, i64, i64, vp, vp, vp, vp, i32]
            getattr(L, f).restype = u32
        L.orc_kv_elem.argtypes = [vp, i64, i64, i64, i64, i64, i64, i64, i64, i64, i64, vp, vp]
        L.orc_request_order.argtypes = [i64, i64, vp, vp]
        L.orc_place.argtypes = [i64, i64, vp, vp, vp, vp]
        L.orc_place.restype = i64
        L.orc_assign_pages.argtypes = [i64, i64, i64, i64, vp, vp, vp, vp, i64, i64, vp]
        L.orc_assign_pages.restype = u32
        L.orc_kv_descriptors.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp, vp]
        L.orc_kv_descriptors.restype = i64
        _lib = L
    return _lib


@dataclass
class Dims:
    """Problem sizes, in the page's notation (§3.1, §3.2)."""
    P: int
    E: int = 0
    H: int = 0
    I: int = 0
    N: int = 1
    Hkv: int = 0
    D: int = 0
    ps: int = 16
    pages_tp: int = 0
    max_requests: int = 0
    max_pages: int = 0
    w13_split: int = 0
    Hq: int = 0           # attention query heads (0 = no attention weights)

    def vec(self) -> np.ndarray:
        return np.array([getattr(self, f.name) for f in fields(self)], dtype=np.int64)

    @property
    def El(self) -> int:
        return self.E // self.P

    @property
    def Ip(self) -> int:
        return self.I // self.P


LAYOUT_KEYS = ("region_stride", "wslot_stride", "w13_off", "w2_off", "kvslot_stride",
               "kv_v_off", "kvslots_off", "ws_off", "pages_ep", "pages_tp", "h_tp",
               "attnslot_stride", "attn_wo_off", "attnslots_off")


def layout(d: Dims) -> dict:
    out = np.zeros(len(LAYOUT_KEYS), dtype=np.int64)
    lib().orc_layout(d.vec().ctypes.data, out.ctypes.data)
    return dict(zip(LAYOUT_KEYS, (int(x) for x in out)))


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def weights_ep2tp(buf: np.ndarray, d: Dims, src: np.ndarray | None = None, order: int = 1) -> None:
    """EP->TP weight switch on a host copy of the unified buffer (in place, or
    reading the snapshot ``src`` when given)."""
    dv = d.vec()
    lib().orc_weights_ep2tp(_ptr(src if src is not None else buf), _ptr(buf), dv.ctypes.data, order)


def weights_tp2ep(buf: np.ndarray, d: Dims, src: np.ndarray | None = None, order: int = -1) -> None:
    dv = d.vec()
    lib().orc_weights_tp2ep(_ptr(src if src is not None else buf), _ptr(buf), dv.ctypes.data, order)


def attn_ep2tp(buf: np.ndarray, d: Dims, src: np.ndarray | None = None, order: int = 1) -> None:
    """Attention weights EP -> TP (keep own shard), memory-saving variant."""
    dv = d.vec()
    lib().orc_attn_ep2tp(_ptr(src if src is not None else buf), _ptr(buf), dv.ctypes.data, order)


def attn_tp2ep(buf: np.ndarray, d: Dims, src: np.ndarray | None = None, order: int = -1) -> None:
    """Attention weights TP -> EP (all-gather of the shards)."""
    dv = d.vec()
    lib().orc_attn_tp2ep(_ptr(src if src is not None else buf), _ptr(buf), dv.ctypes.data, order)


def w13_tp_elem(d: Dims, q, e, row, h, ep_slot, tp_slot):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    dv = d.vec()
    lib().orc_w13_tp_elem(dv.ctypes.data, q, e, row, h, ep_slot, tp_slot, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def w2_tp_elem(d: Dims, q, e, h, c, ep_slot, tp_slot):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    dv = d.vec()
    lib().orc_w2_tp_elem(dv.ctypes.data, q, e, h, c, ep_slot, tp_slot, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def kv_elem(d: Dims, owner, q, ep_page, tp_page, tok_in_page, c, h, e, ep_slot, tp_slot):
    a, b = ctypes.c_int64(), ctypes.c_int64()
    dv = d.vec()
    lib().orc_kv_elem(dv.ctypes.data, owner, q, ep_page, tp_page, tok_in_page, c, h, e,
                      ep_slot, tp_slot, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def kv_validate(d: Dims, direction: int, lens, owner, ep_pt, tp_pt) -> int:
    lens, owner, ep_pt, tp_pt = _i32(lens), _i32(owner), _i32(ep_pt), _i32(tp_pt)
    dv = d.vec()
    return int(lib().orc_kv_validate(dv.ctypes.data, direction, len(lens), ep_pt.shape[1],
                                     _ptr(lens), _ptr(owner), _ptr(ep_pt), _ptr(tp_pt)))


def _kv(fn, buf, d, lens, owner, ep_pt, tp_pt, src, order):
    lens, owner, ep_pt, tp_pt = _i32(lens), _i32(owner), _i32(ep_pt), _i32(tp_pt)
    dv = d.vec()
    return int(fn(_ptr(src if src is not None else buf), _ptr(buf), dv.ctypes.data, len(lens),
                  ep_pt.shape[1], _ptr(lens), _ptr(owner), _ptr(ep_pt), _ptr(tp_pt), order))


def kv_ep2tp(buf, d: Dims, lens, owner, ep_pt, tp_pt, src=None, order: int = 1) -> int:
    """KV EP->TP on a host buffer; returns the error flags (0 = moved)."""
    return _kv(lib().orc_kv_ep2tp, buf, d, lens, owner, ep_pt, tp_pt, src, order)


def kv_tp2ep(buf, d: Dims, lens, owner, ep_pt, tp_pt, src=None, order: int = -1) -> int:
    """KV TP->EP on a host buffer (owner = new EP owner, ep_pt = new EP pages)."""
    return _kv(lib().orc_kv_tp2ep, buf, d, lens, owner, ep_pt, tp_pt, src, order)


def request_order(P: int, owner) -> np.ndarray:
    owner = _i32(owner)
    out = np.zeros(len(owner), dtype=np.int32)
    lib().orc_request_order(P, len(owner), _ptr(owner), _ptr(out))
    return out


def place(P: int, lens, key=None):
    """LPT placement; returns (owner, local_pos, max_load)."""
    lens = _i32(lens)
    key = None if key is None else _i32(key)
    owner = np.zeros(len(lens), dtype=np.int32)
    local = np.zeros(len(lens), dtype=np.int32)
    mx = lib().orc_place(P, len(lens), _ptr(lens), _ptr(key), _ptr(owner), _ptr(local))
    return owner, local, int(mx)


def assign_pages(npools: int, lens, ps: int, maxp: int, free_pages, region=None, key=None):
    """Page hand-out from free lists (one row per pool); returns (flags, table)."""
    lens = _i32(lens)
    free_pages = _i32(np.atleast_2d(free_pages))
    region = None if region is None else _i32(region)
    key = None if key is None else _i32(key)
    pt = np.full((len(lens), maxp), -7, dtype=np.int32)
    fl = lib().orc_assign_pages(npools, len(lens), ps, maxp, _ptr(lens), _ptr(region), _ptr(key),
                                _ptr(free_pages), free_pages.shape[1], free_pages.shape[1], _ptr(pt))
    return int(fl), pt


def kv_descriptors(d: Dims, direction: int, lens, owner, ep_pt, tp_pt) -> np.ndarray:
    lens, owner, ep_pt, tp_pt = _i32(lens), _i32(owner), _i32(ep_pt), _i32(tp_pt)
    total = int(sum((int(x) + d.ps - 1) // d.ps for x in lens))
    out = np.zeros((max(total, 1), 8), dtype=np.int32)
    dv = d.vec()
    n = lib().orc_kv_descriptors(dv.ctypes.data, direction, len(lens), ep_pt.shape[1], _ptr(lens),
                                 _ptr(owner), _ptr(ep_pt), _ptr(tp_pt), _ptr(out))
    return out[:n]
