"""Python binding of libumm (ctypes; argument marshalling only).

Every function here has the name of its C entry point in include/umm.h and
does nothing but convert arguments: torch tensors become device pointers,
torch streams become cudaStream_t handles, non-zero status codes become
``UmmError``.  Tensor arguments are checked first (a contiguous CUDA tensor
of int32, or bytes for buffers, large enough for the sizes passed), so a host
tensor or a short table is refused instead of reaching a kernel.  All work
runs in the library's CUDA kernels.  Importing this module fails loudly when
libumm.so has not been built.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libumm.so")
# the same ABI, built with every copy-kernel access checked (tests)
CHECKED_LIB_PATH = os.path.join(_HERE, "libumm_checked.so")

UMM_OK = 0
UMM_ERR_INVALID_ARG = 1
UMM_ERR_ALIGN = 2
UMM_ERR_MODE = 3
UMM_ERR_CAPACITY = 4
UMM_ERR_PAGE_OOB = 5
UMM_ERR_CUDA = 6
UMM_ERR_TIMEOUT = 7
UMM_ERR_DUP_PAGE = 8
UMM_ERR_BAD_REQUEST = 9
UMM_ERR_ACCESS = 10

UMM_MODE_EP = 0
UMM_MODE_TP = 1

UMM_KV_COPY_LSU = 0
UMM_KV_COPY_TMA = 1

FLAG_BAD_REQUEST = 1
FLAG_CAPACITY = 2
FLAG_PAGE_OOB = 4
FLAG_DUP_PAGE = 8
FLAG_ACCESS = 16
FLAG_TIMEOUT = 32

(K_WEIGHTS_EP2TP, K_WEIGHTS_TP2EP, K_KV_PREP, K_KV_EP2TP, K_KV_TP2EP, K_PLACE, K_ORDER, K_ASSIGN,
 K_ATTN_EP2TP, K_ATTN_TP2EP) = range(10)
K_COUNT = 10
KIND_NAMES = ("weights_ep2tp", "weights_tp2ep", "kv_prep", "kv_ep2tp", "kv_tp2ep", "place", "order", "assign",
              "attn_ep2tp", "attn_tp2ep")


class UmmDims(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int32), ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("kv_pages_tp", ctypes.c_int64), ("max_requests", ctypes.c_int32),
                ("w13_split", ctypes.c_int32), ("max_pages", ctypes.c_int64), ("weight_mode", ctypes.c_int32),
                ("kv_mode", ctypes.c_int32), ("attn_q_heads", ctypes.c_int32), ("attn_mode", ctypes.c_int32)]


class UmmLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("region_stride", "wslot_stride", "w13_off", "w2_off",
                                               "kvslot_stride", "kv_v_off", "kvslots_off", "ws_off",
                                               "ws_bytes", "total_bytes")] + \
               [(n, ctypes.c_int64) for n in ("pages_ep", "pages_tp", "h_tp")] + \
               [("status_off", ctypes.c_uint64), ("desc_off", ctypes.c_uint64), ("desc_capacity", ctypes.c_int64)] + \
               [(n, ctypes.c_uint64) for n in ("attnslot_stride", "attn_wo_off", "attnslots_off")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class UmmPolicyParams(ctypes.Structure):
    _fields_ = [("t_high", ctypes.c_double), ("t_low", ctypes.c_double), ("window", ctypes.c_int32),
                ("cooldown_s", ctypes.c_double), ("start_mode", ctypes.c_int32)]


POLICY_STAY, POLICY_TO_EP, POLICY_TO_TP, POLICY_CANCELLED = 0, 1, 2, 3


class UmmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libumm.so is not built ({LIB_PATH}); run ep_tp_weight_gb300.build.build()")

_vp, _i32, _i64, _u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
_P = ctypes.POINTER

_SIG = {
    "umm_required_bytes": [_P(UmmDims), _P(_u64)],
    "umm_layout_for_dims": [_P(UmmDims), _P(UmmLayout)],
    "umm_create": [_P(UmmDims), _vp, _u64, _P(_vp)],
    "umm_destroy": [_vp],
    "umm_layout": [_vp, _P(UmmLayout)],
    "umm_get_modes": [_vp, _P(_i32), _P(_i32)],
    "umm_set_modes": [_vp, _i32, _i32],
    "reshard_weights_ep2tp": [_vp, _vp],
    "reshard_weights_tp2ep": [_vp, _vp],
    "gather_requests_ep2tp": [_vp, _i32, _vp, _vp, _vp],
    "place_requests_tp2ep": [_vp, _i32, _vp, _vp, _vp, _vp, _vp],
    "umm_assign_pages": [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _i32, _vp],
    "reshard_kv_ep2tp": [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp],
    "reshard_kv_tp2ep": [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp],
    "umm_kv_check_capacity": [_vp, _i32, _i32, _vp, _vp],
    "umm_status_sync": [_vp, _vp, _P(_i32), _P(ctypes.c_uint32)],
    "umm_profile_enable": [_vp, _i32],
    "umm_profile_read": [_vp, _i32, _P(_i64), _P(ctypes.c_double)],
    "umm_profile_reset": [_vp],
    "umm_launch_count": [_vp, _P(_i64)],
    "place_requests_tp2ep_noalloc": [_i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp],
    "umm_weights_stage_bytes": [_vp, _P(_u64)],
    "reshard_weights_ep2tp_staged": [_vp, _vp, _u64, _vp],
    "reshard_weights_tp2ep_staged": [_vp, _vp, _u64, _vp],
    "umm_kv_stage_bytes": [_vp, _P(_u64)],
    "reshard_kv_ep2tp_staged": [_vp, _vp, _u64, _i32, _i32, _vp, _vp, _vp, _vp, _vp],
    "reshard_kv_tp2ep_staged": [_vp, _vp, _u64, _i32, _i32, _vp, _vp, _vp, _vp, _vp],
    "reshard_attn_ep2tp": [_vp, _vp],
    "reshard_attn_tp2ep": [_vp, _vp],
    "umm_get_attn_mode": [_vp, _P(_i32)],
    "umm_set_attn_mode": [_vp, _i32],
    "umm_switch_ep2tp": [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp],
    "umm_switch_tp2ep": [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp],
    "umm_set_switch_overlap": [_vp, _i32],
    "umm_kv_copy_kernel": [_P(UmmDims), _i32, _P(_i32), _P(_i32)],
    "umm_test_stall_tma_wait": [_vp, _i32, ctypes.c_uint32],
    "umm_policy_create": [_vp, _P(_vp)],
    "umm_policy_destroy": [_vp],
    "umm_policy_step": [_vp, _i64, ctypes.c_double, _i32, _P(_i32)],
    "umm_policy_state": [_vp, _P(_i32), _P(_i64), _P(_i64)],
}


def _bind(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name, args in _SIG.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.umm_strerror.argtypes = [ctypes.c_int]
    lib.umm_strerror.restype = ctypes.c_char_p
    return lib


_lib = _bind(LIB_PATH)


@contextlib.contextmanager
def checked_library():
    """Route every call of this module through libumm_checked.so inside the
    block (handles made inside must also be destroyed inside).  It swaps a
    module global: use it from one thread, as the tests do."""
    global _lib
    if not os.path.exists(CHECKED_LIB_PATH):
        raise ImportError(f"libumm_checked.so is not built ({CHECKED_LIB_PATH})")
    saved = _lib
    _lib = _bind(CHECKED_LIB_PATH)
    try:
        yield
    finally:
        _lib = saved

EXPORTED = tuple(_SIG) + ("umm_strerror",)


def strerror(code: int) -> str:
    return _lib.umm_strerror(int(code)).decode()


def _ck(rc: int, where: str) -> None:
    if rc != UMM_OK:
        raise UmmError(rc, where)


def _ptr(x):
    """Device pointer of a tensor (or an int address); None stays NULL."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    return int(x) or None


def _arr(x, n: int, where: str, what: str):
    """Device pointer of a caller array that the call reads or writes as n
    int32 elements.  A tensor must be a contiguous int32 CUDA tensor with at
    least n elements; anything else raises UmmError(UMM_ERR_INVALID_ARG) before
    the library is called, so a host tensor or a short table never reaches a
    kernel.  A raw int address is passed through: its size is the caller's
    responsibility, as in C.  None stays NULL."""
    if x is None or not hasattr(x, "data_ptr"):
        return _ptr(x)
    dev = getattr(x, "device", None)
    if (dev is None or dev.type != "cuda" or str(x.dtype) != "torch.int32" or not x.is_contiguous()
            or x.numel() < n):
        raise UmmError(UMM_ERR_INVALID_ARG, f"{where} ({what}: a contiguous int32 CUDA tensor of at least "
                                            f"{n} elements is required)")
    return x.data_ptr() or None


def _buf(x, nbytes: int, where: str, what: str):
    """Device pointer of a caller byte buffer of at least nbytes (a contiguous
    CUDA tensor of any dtype, or a raw int address); as _arr."""
    if x is None or not hasattr(x, "data_ptr"):
        return _ptr(x)
    dev = getattr(x, "device", None)
    if dev is None or dev.type != "cuda" or not x.is_contiguous() or x.numel() * x.element_size() < nbytes:
        raise UmmError(UMM_ERR_INVALID_ARG, f"{where} ({what}: a contiguous CUDA tensor of at least "
                                            f"{nbytes} bytes is required)")
    return x.data_ptr() or None


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def make_dims(P, E=0, H=0, I=0, N=1, Hkv=0, D=0, ps=16, pages_tp=0, max_requests=0, max_pages=0,
              w13_split=0, weight_mode=UMM_MODE_EP, kv_mode=UMM_MODE_EP, Hq=0,
              attn_mode=UMM_MODE_EP) -> UmmDims:
    """umm_dims from the page's notation (§3.1, §3.2)."""
    return UmmDims(P, E, H, I, N, Hkv, D, ps, pages_tp, max_requests, w13_split, max_pages,
                   weight_mode, kv_mode, Hq, attn_mode)


def umm_required_bytes(dims: UmmDims) -> int:
    out = ctypes.c_uint64()
    _ck(_lib.umm_required_bytes(ctypes.byref(dims), ctypes.byref(out)), "umm_required_bytes")
    return out.value


def umm_layout_for_dims(dims: UmmDims) -> dict:
    out = UmmLayout()
    _ck(_lib.umm_layout_for_dims(ctypes.byref(dims), ctypes.byref(out)), "umm_layout_for_dims")
    return out.as_dict()


# ranks (P) of the handles made through this module: the size checks of the
# per-rank free lists need it
_RANKS: dict[int, int] = {}


def umm_create(dims: UmmDims, d_base, nbytes: int) -> int:
    h = ctypes.c_void_p()
    base = _buf(d_base, int(nbytes), "umm_create", "d_base")
    _ck(_lib.umm_create(ctypes.byref(dims), base, int(nbytes), ctypes.byref(h)), "umm_create")
    _RANKS[h.value] = int(dims.P)
    return h.value


def umm_destroy(h: int) -> None:
    _ck(_lib.umm_destroy(h), "umm_destroy")
    _RANKS.pop(h, None)


def umm_layout(h: int) -> dict:
    out = UmmLayout()
    _ck(_lib.umm_layout(h, ctypes.byref(out)), "umm_layout")
    return out.as_dict()


def umm_get_modes(h: int) -> tuple[int, int]:
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _ck(_lib.umm_get_modes(h, ctypes.byref(a), ctypes.byref(b)), "umm_get_modes")
    return a.value, b.value


def umm_set_modes(h: int, weight_mode: int, kv_mode: int) -> None:
    _ck(_lib.umm_set_modes(h, weight_mode, kv_mode), "umm_set_modes")


def reshard_weights_ep2tp(h: int, stream=None) -> None:
    _ck(_lib.reshard_weights_ep2tp(h, _stream(stream)), "reshard_weights_ep2tp")


def reshard_weights_tp2ep(h: int, stream=None) -> None:
    _ck(_lib.reshard_weights_tp2ep(h, _stream(stream)), "reshard_weights_tp2ep")


def umm_weights_stage_bytes(h: int) -> int:
    out = ctypes.c_uint64()
    _ck(_lib.umm_weights_stage_bytes(h, ctypes.byref(out)), "umm_weights_stage_bytes")
    return out.value


def reshard_weights_ep2tp_staged(h: int, stage, stage_bytes: int, stream=None) -> None:
    w = "reshard_weights_ep2tp_staged"
    _ck(_lib.reshard_weights_ep2tp_staged(h, _buf(stage, int(stage_bytes), w, "stage"), int(stage_bytes),
                                          _stream(stream)), w)


def reshard_weights_tp2ep_staged(h: int, stage, stage_bytes: int, stream=None) -> None:
    w = "reshard_weights_tp2ep_staged"
    _ck(_lib.reshard_weights_tp2ep_staged(h, _buf(stage, int(stage_bytes), w, "stage"), int(stage_bytes),
                                          _stream(stream)), w)


def umm_kv_stage_bytes(h: int) -> int:
    out = ctypes.c_uint64()
    _ck(_lib.umm_kv_stage_bytes(h, ctypes.byref(out)), "umm_kv_stage_bytes")
    return out.value


def reshard_kv_ep2tp_staged(h: int, stage, stage_bytes: int, R: int, max_pages_per_req: int, seq_lens,
                            ep_owner, ep_page_table, tp_page_table, stream=None) -> None:
    w, n, t = "reshard_kv_ep2tp_staged", max(R, 0), max(R, 0) * max(max_pages_per_req, 0)
    _ck(_lib.reshard_kv_ep2tp_staged(h, _buf(stage, int(stage_bytes), w, "stage"), int(stage_bytes), R,
                                     max_pages_per_req, _arr(seq_lens, n, w, "seq_lens"),
                                     _arr(ep_owner, n, w, "ep_owner"), _arr(ep_page_table, t, w, "ep_page_table"),
                                     _arr(tp_page_table, t, w, "tp_page_table"), _stream(stream)), w)


def reshard_kv_tp2ep_staged(h: int, stage, stage_bytes: int, R: int, max_pages_per_req: int, seq_lens,
                            ep_owner, ep_page_table, tp_page_table, stream=None) -> None:
    w, n, t = "reshard_kv_tp2ep_staged", max(R, 0), max(R, 0) * max(max_pages_per_req, 0)
    _ck(_lib.reshard_kv_tp2ep_staged(h, _buf(stage, int(stage_bytes), w, "stage"), int(stage_bytes), R,
                                     max_pages_per_req, _arr(seq_lens, n, w, "seq_lens"),
                                     _arr(ep_owner, n, w, "ep_owner"), _arr(ep_page_table, t, w, "ep_page_table"),
                                     _arr(tp_page_table, t, w, "tp_page_table"), _stream(stream)), w)


def reshard_attn_ep2tp(h: int, stream=None) -> None:
    _ck(_lib.reshard_attn_ep2tp(h, _stream(stream)), "reshard_attn_ep2tp")


def reshard_attn_tp2ep(h: int, stream=None) -> None:
    _ck(_lib.reshard_attn_tp2ep(h, _stream(stream)), "reshard_attn_tp2ep")


def umm_get_attn_mode(h: int) -> int:
    m = ctypes.c_int32()
    _ck(_lib.umm_get_attn_mode(h, ctypes.byref(m)), "umm_get_attn_mode")
    return m.value


def umm_set_attn_mode(h: int, mode: int) -> None:
    _ck(_lib.umm_set_attn_mode(h, mode), "umm_set_attn_mode")


def gather_requests_ep2tp(h: int, R: int, ep_owner, tp_pos, stream=None) -> None:
    w, n = "gather_requests_ep2tp", max(R, 0)
    _ck(_lib.gather_requests_ep2tp(h, R, _arr(ep_owner, n, w, "ep_owner"), _arr(tp_pos, n, w, "tp_pos"),
                                   _stream(stream)), w)


def place_requests_tp2ep(h: int, R: int, seq_lens, list_pos, owner, local_pos, stream=None) -> None:
    w, n = "place_requests_tp2ep", max(R, 0)
    _ck(_lib.place_requests_tp2ep(h, R, _arr(seq_lens, n, w, "seq_lens"), _arr(list_pos, n, w, "list_pos"),
                                  _arr(owner, n, w, "owner"), _arr(local_pos, n, w, "local_pos"),
                                  _stream(stream)), w)


def place_requests_tp2ep_noalloc(P: int, R: int, seq_lens, list_pos, owner, local_pos, status=None,
                                 stream=None) -> None:
    """place_requests_tp2ep without a handle and without any allocation (for
    callers that cannot allocate device memory); R <= 16384."""
    w, n = "place_requests_tp2ep_noalloc", max(R, 0)
    _ck(_lib.place_requests_tp2ep_noalloc(P, R, _arr(seq_lens, n, w, "seq_lens"), _arr(list_pos, n, w, "list_pos"),
                                          _arr(owner, n, w, "owner"), _arr(local_pos, n, w, "local_pos"),
                                          _arr(status, 1, w, "status"), _stream(stream)), w)


def umm_assign_pages(h: int, npools: int, R: int, seq_lens, pool, key, free_pages, free_stride: int,
                     free_count: int, page_table, max_pages_per_req: int, stream=None) -> None:
    w, n = "umm_assign_pages", max(R, 0)
    nfree = max(npools - 1, 0) * max(int(free_stride), 0) + max(int(free_count), 0)
    _ck(_lib.umm_assign_pages(h, npools, R, _arr(seq_lens, n, w, "seq_lens"), _arr(pool, n, w, "pool"),
                              _arr(key, n, w, "key"), _arr(free_pages, nfree, w, "free_pages"),
                              int(free_stride), int(free_count),
                              _arr(page_table, n * max(int(max_pages_per_req), 0), w, "page_table"),
                              int(max_pages_per_req), _stream(stream)), w)


def reshard_kv_ep2tp(h: int, R: int, max_pages_per_req: int, seq_lens, ep_owner, ep_page_table,
                     tp_page_table, stream=None) -> None:
    w, n, t = "reshard_kv_ep2tp", max(R, 0), max(R, 0) * max(max_pages_per_req, 0)
    _ck(_lib.reshard_kv_ep2tp(h, R, max_pages_per_req, _arr(seq_lens, n, w, "seq_lens"),
                              _arr(ep_owner, n, w, "ep_owner"), _arr(ep_page_table, t, w, "ep_page_table"),
                              _arr(tp_page_table, t, w, "tp_page_table"), _stream(stream)), w)


def reshard_kv_tp2ep(h: int, R: int, max_pages_per_req: int, seq_lens, ep_owner, ep_page_table,
                     tp_page_table, stream=None) -> None:
    w, n, t = "reshard_kv_tp2ep", max(R, 0), max(R, 0) * max(max_pages_per_req, 0)
    _ck(_lib.reshard_kv_tp2ep(h, R, max_pages_per_req, _arr(seq_lens, n, w, "seq_lens"),
                              _arr(ep_owner, n, w, "ep_owner"), _arr(ep_page_table, t, w, "ep_page_table"),
                              _arr(tp_page_table, t, w, "tp_page_table"), _stream(stream)), w)


def umm_switch_ep2tp(h: int, R: int, max_pages_per_req: int, seq_lens, ep_owner, ep_page_table, tp_free_pages,
                     tp_free_count: int, tp_pos, tp_page_table, stream=None) -> None:
    w, n, t = "umm_switch_ep2tp", max(R, 0), max(R, 0) * max(max_pages_per_req, 0)
    _ck(_lib.umm_switch_ep2tp(h, R, max_pages_per_req, _arr(seq_lens, n, w, "seq_lens"),
                              _arr(ep_owner, n, w, "ep_owner"), _arr(ep_page_table, t, w, "ep_page_table"),
                              _arr(tp_free_pages, max(int(tp_free_count), 0), w, "tp_free_pages"),
                              int(tp_free_count), _arr(tp_pos, n, w, "tp_pos"),
                              _arr(tp_page_table, t, w, "tp_page_table"), _stream(stream)), w)


def umm_switch_tp2ep(h: int, R: int, max_pages_per_req: int, seq_lens, tp_pos, tp_page_table, ep_free_pages,
                     ep_free_stride: int, ep_free_count: int, ep_owner, local_pos, ep_page_table,
                     stream=None) -> None:
    # the library reads (P-1) * stride + count free-list entries; P is known
    # for handles made through this module (else one pool's count is checked)
    w, n, t = "umm_switch_tp2ep", max(R, 0), max(R, 0) * max(max_pages_per_req, 0)
    nfree = (_RANKS.get(h, 1) - 1) * max(int(ep_free_stride), 0) + max(int(ep_free_count), 0)
    _ck(_lib.umm_switch_tp2ep(h, R, max_pages_per_req, _arr(seq_lens, n, w, "seq_lens"),
                              _arr(tp_pos, n, w, "tp_pos"), _arr(tp_page_table, t, w, "tp_page_table"),
                              _arr(ep_free_pages, nfree, w, "ep_free_pages"),
                              int(ep_free_stride), int(ep_free_count), _arr(ep_owner, n, w, "ep_owner"),
                              _arr(local_pos, n, w, "local_pos"), _arr(ep_page_table, t, w, "ep_page_table"),
                              _stream(stream)), w)


def umm_set_switch_overlap(h: int, enable: bool = True) -> None:
    _ck(_lib.umm_set_switch_overlap(h, 1 if enable else 0), "umm_set_switch_overlap")


def umm_kv_copy_kernel(dims: UmmDims, direction: int) -> tuple[int, int]:
    """(UMM_KV_COPY_TMA or UMM_KV_COPY_LSU, LSU vector bytes or 0) that a KV
    reshard of these dims launches (host-only)."""
    k, vb = ctypes.c_int32(), ctypes.c_int32()
    _ck(_lib.umm_kv_copy_kernel(ctypes.byref(dims), int(direction), ctypes.byref(k), ctypes.byref(vb)),
        "umm_kv_copy_kernel")
    return k.value, vb.value


def umm_test_stall_tma_wait(h: int, layer: int, polls: int) -> None:
    """Checked build only: make the TMA copy of one KV EP->TP layer run out a
    wait (see include/umm.h)."""
    _ck(_lib.umm_test_stall_tma_wait(h, int(layer), int(polls)), "umm_test_stall_tma_wait")


def umm_kv_check_capacity(h: int, target_kv_mode: int, R: int, h_seq_lens, h_ep_owner=None) -> int:
    """Host-side capacity check; returns the status code (0 = fits)."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(h_seq_lens, dtype=np.int32))
    own = None if h_ep_owner is None else np.ascontiguousarray(np.asarray(h_ep_owner, dtype=np.int32))
    return int(_lib.umm_kv_check_capacity(h, target_kv_mode, R, lens.ctypes.data,
                                          None if own is None else own.ctypes.data))


def umm_status_sync(h: int, stream=None) -> tuple[int, int]:
    """(status code, flag bits) of the device checks since the last sync; clears them."""
    st, fl = ctypes.c_int32(), ctypes.c_uint32()
    _ck(_lib.umm_status_sync(h, _stream(stream), ctypes.byref(st), ctypes.byref(fl)), "umm_status_sync")
    return st.value, fl.value


def umm_strerror(code: int) -> str:
    return strerror(code)


def umm_profile_enable(h: int, enable: bool = True) -> None:
    _ck(_lib.umm_profile_enable(h, 1 if enable else 0), "umm_profile_enable")


def umm_profile_read(h: int, kind: int) -> tuple[int, float]:
    n, ms = ctypes.c_int64(), ctypes.c_double()
    _ck(_lib.umm_profile_read(h, kind, ctypes.byref(n), ctypes.byref(ms)), "umm_profile_read")
    return n.value, ms.value


def umm_profile_reset(h: int) -> None:
    _ck(_lib.umm_profile_reset(h), "umm_profile_reset")


def umm_launch_count(h: int) -> int:
    n = ctypes.c_int64()
    _ck(_lib.umm_launch_count(h, ctypes.byref(n)), "umm_launch_count")
    return n.value


def umm_policy_create(t_high: float, t_low: float, window: int, cooldown_s: float,
                      start_mode: int = UMM_MODE_TP) -> int:
    h = ctypes.c_void_p()
    prm = UmmPolicyParams(t_high, t_low, window, cooldown_s, start_mode)
    _ck(_lib.umm_policy_create(ctypes.byref(prm), ctypes.byref(h)), "umm_policy_create")
    return h.value


def umm_policy_destroy(h: int) -> None:
    _ck(_lib.umm_policy_destroy(h), "umm_policy_destroy")


def umm_policy_step(h: int, inflight: int, now_s: float, target_fits: bool = True) -> int:
    d = ctypes.c_int32()
    _ck(_lib.umm_policy_step(h, int(inflight), float(now_s), 1 if target_fits else 0, ctypes.byref(d)),
        "umm_policy_step")
    return d.value


def umm_policy_state(h: int) -> tuple[int, int, int]:
    m, sw, ca = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64()
    _ck(_lib.umm_policy_state(h, ctypes.byref(m), ctypes.byref(sw), ctypes.byref(ca)), "umm_policy_state")
    return m.value, sw.value, ca.value
