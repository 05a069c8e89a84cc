"""Host-side checks of the C-ABI library (no GPU): it loads, exports every
entry point include/umm.h declares, and its host logic (layout, argument
checks, capacity check, status strings) agrees with the header and with the
oracle's independent layout computation."""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import pytest

import oracle
from helpers import dims_of
from synth.workloads import ALL, TINY, Workload

HEADER = Path(__file__).resolve().parent.parent / "include" / "umm.h"


@pytest.fixture(scope="module")
def umm():
    import ep_tp_weight_gb300 as m
    return m


def declared_functions() -> list[str]:
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def header_defines() -> dict[str, int]:
    return {m.group(1): int(m.group(2), 0) for m in
            re.finditer(r"#define\s+(UMM_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?", HEADER.read_text())}


def test_library_exports_every_declared_entry_point(umm):
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(umm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(umm.EXPORTED)


@pytest.mark.parametrize("which", ["LIB_PATH", "CHECKED_LIB_PATH"])
def test_library_exports_nothing_undeclared(umm, which):
    """Both builds (normal and checked) export exactly the declared C ABI."""
    import shutil
    import subprocess
    if not shutil.which("nm"):
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", getattr(umm, which)], capture_output=True,
                         text=True).stdout
    c_symbols = {ln.split()[-1] for ln in out.splitlines()
                 if " T " in ln and not ln.split()[-1].startswith(("_Z", "cuda", "__", "_"))}
    assert c_symbols == set(declared_functions())


def test_checked_library_loads_with_the_same_signatures(umm):
    with umm.checked_library():
        assert umm._lib._name == umm.CHECKED_LIB_PATH
        for n in umm.EXPORTED:
            assert hasattr(umm._lib, n), n
        assert umm.strerror(umm.UMM_ERR_ACCESS).startswith("checked build")
    assert umm._lib._name == umm.LIB_PATH


def test_binding_constants_match_header(umm):
    d = header_defines()
    for k, v in d.items():
        if k.startswith(("UMM_ERR_", "UMM_MODE_", "UMM_OK")):
            assert getattr(umm, k) == v, k
        if k.startswith("UMM_FLAG_"):
            assert getattr(umm, k.replace("UMM_", "")) == v, k
        if k.startswith("UMM_K_") and k != "UMM_K_COUNT":
            assert getattr(umm, k.replace("UMM_", "")) == v, k
    # the oracle restates the same flag bits on its own
    assert (oracle.F_BAD_REQUEST, oracle.F_CAPACITY, oracle.F_PAGE_OOB, oracle.F_DUP_PAGE) == \
        (d["UMM_FLAG_BAD_REQUEST"], d["UMM_FLAG_CAPACITY"], d["UMM_FLAG_PAGE_OOB"], d["UMM_FLAG_DUP_PAGE"])


def test_struct_sizes_match_c_abi(umm):
    assert ctypes.sizeof(umm.UmmDims) == 72
    assert ctypes.sizeof(umm.UmmLayout) == 152


def lib_dims(umm, w: Workload, **over):
    d = w.dims()
    d.update(over)
    return umm.make_dims(P=d["P"], E=d["E"], H=d["H"], I=d["I"], N=d["N"], Hkv=d["Hkv"], D=d["D"],
                         ps=d["ps"], pages_tp=d["pages_tp"], max_requests=d["max_requests"],
                         max_pages=d["max_pages"], w13_split=d["w13_split"], Hq=d.get("Hq", 0))


@pytest.mark.parametrize("name", sorted(ALL))
def test_layout_matches_oracle(umm, name):
    w = ALL[name]
    L = umm.umm_layout_for_dims(lib_dims(umm, w))
    O = oracle.layout(dims_of(w))
    for k in ("region_stride", "wslot_stride", "w13_off", "w2_off", "kvslot_stride", "kv_v_off",
              "kvslots_off", "ws_off", "pages_ep", "pages_tp", "h_tp"):
        assert L[k] == O[k], (name, k)
    assert umm.umm_required_bytes(lib_dims(umm, w)) == L["total_bytes"] > L["ws_off"]
    assert L["status_off"] == L["ws_off"] and L["desc_off"] % 256 == 0


def test_layout_variants_match_oracle(umm):
    for w in (TINY.with_(Hkv=4, P=2), TINY.with_(Hkv=1, P=4, E=8, I=32), TINY.with_(E=0),
              TINY.with_(Hkv=0), Workload("odd", P=3, N=2, E=6, H=7, I=9, Hkv=6, D=5, ps=3, R=3,
                                          len_a=1, len_b=10)):
        L = umm.umm_layout_for_dims(lib_dims(umm, w))
        O = oracle.layout(dims_of(w))
        assert all(L[k] == O[k] for k in O), w.name


def test_full_switch_fits_one_gb300(umm):
    """The full-switch workload (weights of 128 experts x 8 layers + KV of
    2048 requests) must fit in 284,208 MiB with room for the CUDA context."""
    from synth.workloads import FULL_SWITCH
    need = umm.umm_required_bytes(lib_dims(umm, FULL_SWITCH))
    assert need < 270 * 2**30


@pytest.mark.parametrize("bad", [dict(P=0), dict(E=9), dict(I=31), dict(Hkv=3), dict(pages_tp=3),
                                 dict(D=0), dict(ps=0), dict(w13_split=2), dict(P=65, E=0, Hkv=0),
                                 dict(max_requests=-1)])
def test_bad_dims_rejected(umm, bad):
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_required_bytes(lib_dims(umm, TINY, **bad))
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG


def test_null_handle_and_strerror(umm):
    for code in range(0, 10):
        assert umm.strerror(code) and umm.strerror(code) != "unknown status"
    assert umm.strerror(99) == "unknown status"
    lib = ctypes.CDLL(umm.LIB_PATH)
    lib.reshard_weights_ep2tp.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert lib.reshard_weights_ep2tp(None, None) == umm.UMM_ERR_INVALID_ARG
    lib.umm_status_sync.argtypes = [ctypes.c_void_p] * 4
    assert lib.umm_status_sync(None, None, None, None) == umm.UMM_ERR_INVALID_ARG


def test_create_rejects_misaligned_and_small_buffers(umm):
    d = lib_dims(umm, TINY)
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_create(d, 0x1000 + 8, 1 << 30)
    assert ei.value.code == umm.UMM_ERR_ALIGN
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_create(d, 0x100000, 16)
    assert ei.value.code == umm.UMM_ERR_CAPACITY


def test_c_program_uses_the_abi(umm, tmp_path):
    """tests/c_abi_check.c, compiled as C99 with -Wall -Wextra -Werror against
    include/umm.h and linked with libumm.so, calls the host-side entry points;
    what it prints equals what the Python binding gets."""
    import shutil
    import subprocess
    from pathlib import Path
    if not shutil.which("gcc"):
        pytest.skip("gcc not available")
    root = Path(__file__).resolve().parent.parent
    lib_dir = Path(umm.LIB_PATH).parent
    exe = tmp_path / "c_abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", str(root / "include"),
                    str(root / "tests" / "c_abi_check.c"), "-L", str(lib_dir), "-lumm",
                    f"-Wl,-rpath,{lib_dir}", "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = dict(ln.split(" ", 1) for ln in out.splitlines())
    assert int(got["entry_points"]) == len(umm.EXPORTED)
    assert int(got["sizeof_dims"]) == ctypes.sizeof(umm.UmmDims)
    assert int(got["sizeof_layout"]) == ctypes.sizeof(umm.UmmLayout)
    dims = umm.make_dims(P=8, E=128, H=2048, I=768, N=8, Hkv=4, D=128, ps=16, pages_tp=441304,
                         max_requests=2048, max_pages=441304)
    assert int(got["required_bytes"]) == umm.umm_required_bytes(dims)
    L = umm.umm_layout_for_dims(dims)
    for k in ("region_stride", "wslot_stride", "kvslot_stride", "kvslots_off", "ws_off", "pages_ep", "h_tp"):
        assert int(got[k]) == L[k], k
    assert int(got["bad_experts"]) == umm.UMM_ERR_INVALID_ARG
    assert int(got["bad_heads"]) == umm.UMM_ERR_INVALID_ARG
    assert int(got["null_handle"]) == umm.UMM_ERR_INVALID_ARG
    assert got["strerror_capacity"] == umm.strerror(umm.UMM_ERR_CAPACITY)
    assert int(got["kv_copy_ep2tp_rc"]) == umm.UMM_OK and int(got["kv_copy_tp2ep_rc"]) == umm.UMM_OK
    assert tuple(int(x) for x in got["kv_copy_ep2tp"].split()) == umm.umm_kv_copy_kernel(dims, 0) == \
        (umm.UMM_KV_COPY_TMA, 0)
    assert tuple(int(x) for x in got["kv_copy_tp2ep"].split()) == umm.umm_kv_copy_kernel(dims, 1) == \
        (umm.UMM_KV_COPY_LSU, 32)
    assert int(got["stall_hook_null"]) == umm.UMM_ERR_INVALID_ARG
    assert (int(got["policy_last_decision"]), int(got["policy_mode"]), int(got["policy_switches"])) == \
        (umm.POLICY_TO_EP, umm.UMM_MODE_EP, 1)


class _FakeDevice:
    def __init__(self, kind):
        self.type = kind


class _FakeTensor:
    """Just enough of a tensor for the binding's argument checks."""

    def __init__(self, n, dtype="torch.int32", kind="cuda", contiguous=True, itemsize=4):
        self.n, self.dtype, self.device, self.contig, self.itemsize = n, dtype, _FakeDevice(kind), contiguous, itemsize

    def data_ptr(self):
        return 0x7f0000000000

    def numel(self):
        return self.n

    def element_size(self):
        return self.itemsize

    def is_contiguous(self):
        return self.contig


class _SpyLib:
    """Stands in for libumm: records which entry points were reached."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name == "umm_strerror":
            return lambda code: b"status text"

        def call(*args):
            self.calls.append(name)
            return 0
        return call


def test_binding_refuses_arrays_that_cannot_be_the_kernels_input(umm, monkeypatch):
    """A host tensor, another dtype, a strided view or a table shorter than
    R x max_pages_per_req is refused with UMM_ERR_INVALID_ARG before the library
    is called, so it never reaches a kernel as a device pointer; a contiguous
    int32 CUDA array of the right size, or a raw address, goes through."""
    import torch
    spy = _SpyLib()
    monkeypatch.setattr(umm, "_lib", spy)
    R, maxp = 6, 3
    ok_vec, ok_tab = _FakeTensor(R), _FakeTensor(R * maxp)

    def kv(seq_lens=ok_vec, ep_pt=ok_tab):
        umm.reshard_kv_ep2tp(0x1, R, maxp, seq_lens, ok_vec, ep_pt, ok_tab)

    kv()
    assert spy.calls == ["reshard_kv_ep2tp"]
    bad = [dict(seq_lens=torch.zeros(R, dtype=torch.int32)),          # host memory
           dict(seq_lens=_FakeTensor(R, dtype="torch.int64")),        # another dtype
           dict(seq_lens=_FakeTensor(R, contiguous=False)),          # strided view
           dict(seq_lens=_FakeTensor(R - 1)),                        # too short
           dict(ep_pt=_FakeTensor(R * maxp - 1))]                    # table too short
    for kw in bad:
        with pytest.raises(umm.UmmError) as ei:
            kv(**kw)
        assert ei.value.code == umm.UMM_ERR_INVALID_ARG, kw
    assert spy.calls == ["reshard_kv_ep2tp"]
    umm.reshard_kv_ep2tp(0x1, R, maxp, 0x1000, 0x2000, 0x3000, 0x4000)   # raw addresses: the caller's word
    umm.reshard_kv_ep2tp(0x1, 0, maxp, None, None, None, None)           # R = 0: nothing to check
    assert spy.calls == ["reshard_kv_ep2tp"] * 3
    with pytest.raises(umm.UmmError) as ei:                              # free list shorter than its count
        umm.umm_switch_ep2tp(0x1, R, maxp, ok_vec, ok_vec, ok_tab, _FakeTensor(9), 10, ok_vec, ok_tab)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    with pytest.raises(umm.UmmError) as ei:                              # pools 0..2 need 2*stride + count entries
        umm.umm_assign_pages(0x1, 3, R, ok_vec, ok_vec, ok_vec, _FakeTensor(2 * 8 + 4), 8, 5, ok_tab, maxp)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    umm.umm_assign_pages(0x1, 3, R, ok_vec, ok_vec, ok_vec, _FakeTensor(2 * 8 + 5), 8, 5, ok_tab, maxp)
    umm._RANKS[0x5] = 4                                                  # a handle of 4 ranks
    with pytest.raises(umm.UmmError) as ei:                              # 4 pools need 3*stride + count
        umm.umm_switch_tp2ep(0x5, R, maxp, ok_vec, ok_vec, ok_tab, _FakeTensor(3 * 10 + 6), 10, 7, ok_vec, ok_vec,
                             ok_tab)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    umm.umm_switch_tp2ep(0x5, R, maxp, ok_vec, ok_vec, ok_tab, _FakeTensor(3 * 10 + 7), 10, 7, ok_vec, ok_vec, ok_tab)
    del umm._RANKS[0x5]
    with pytest.raises(umm.UmmError) as ei:                              # buffer smaller than claimed
        umm.umm_create(lib_dims(umm, TINY), _FakeTensor(1000, dtype="torch.uint8", itemsize=1), 1001)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    with pytest.raises(umm.UmmError):
        umm.umm_create(lib_dims(umm, TINY), torch.zeros(64, dtype=torch.uint8), 64)
    assert spy.calls == ["reshard_kv_ep2tp"] * 3 + ["umm_assign_pages", "umm_switch_tp2ep"]


def _kv_dims(umm, P, Hkv, D, ps, pages_tp):
    return umm.make_dims(P=P, N=1, Hkv=Hkv, D=D, ps=ps, pages_tp=pages_tp, max_requests=16, max_pages=1024)


@pytest.mark.parametrize("ps,pages_tp", [(1, 2**31 - 1), (2, 2**30), (16, 2**27), (16, 2**27 + 64),
                                         (256, 2**27), (16, 2**31 - 16)])
def test_tma_copy_addresses_pages_not_rows(umm, ps, pages_tp):
    """The TMA KV EP->TP copy addresses an EP page by its page id (tensor
    coordinates {element, head, row in page, page, region}), so EP pools of
    2^31 - 1, 2^31 and more token rows (pages x page size) keep the TMA copy:
    no coordinate is ever page * page_size.  Every pool the handle accepts has
    page ids below 2^31, and one page more is refused."""
    d = _kv_dims(umm, 1, 1, 8, ps, pages_tp)
    L = umm.umm_layout_for_dims(d)
    assert L["pages_ep"] == pages_tp and L["pages_ep"] < 2**31
    assert umm.umm_kv_copy_kernel(d, 0) == (umm.UMM_KV_COPY_TMA, 0)
    assert umm.umm_kv_copy_kernel(d, 1) == (umm.UMM_KV_COPY_LSU, 16)


def test_page_ids_are_capped_below_2_31(umm):
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_required_bytes(_kv_dims(umm, 1, 1, 8, 16, 2**31))
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_kv_copy_kernel(_kv_dims(umm, 1, 1, 8, 16, 2**31), 0)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG


@pytest.mark.parametrize("P,Hkv,D,ps,want", [
    (8, 4, 128, 16, ("TMA", 0)),      # the full-switch shape: one head per TP rank
    (2, 2, 16, 16, ("TMA", 0)),
    (2, 4, 128, 16, ("LSU", 32)),     # two heads per TP rank
    (8, 4, 4, 16, ("LSU", 8)),        # 8-byte head rows: not a bulk-copy size
    (8, 4, 12, 16, ("LSU", 8)),       # 24-byte head rows
    (4, 4, 256, 32, ("LSU", 32)),     # 4 heads x 16 KiB tiles: over 48 KiB of shared memory
    (8, 1, 128, 512, ("LSU", 32)),    # a 512-row page: over the 256 box limit
    (3, 1, 5, 16, ("LSU", 2)),
    # tiles + 128 B alignment room + 1 KiB static shared memory within 48 KiB:
    (2, 1, 128, 187, ("TMA", 0)),     # 187 rows x 256 B = 47,872 B: 49,024 B in all, fits
    (2, 1, 128, 188, ("LSU", 32)),    # 188 rows: 49,280 B, over
    (2, 2, 128, 93, ("TMA", 0)),      # two heads of 93 rows: 47,616 B of tiles, fits
    (2, 2, 128, 94, ("LSU", 32)),
    (2, 1, 256, 16, ("TMA", 0)),      # head of 256 elements: the box limit
    (2, 1, 264, 16, ("LSU", 16)),     # 264: over it
    (2, 1, 8, 256, ("TMA", 0)),       # 256-row page: the box limit
    (2, 1, 8, 257, ("LSU", 16)),
])
def test_kv_copy_kernel_choice(umm, P, Hkv, D, ps, want):
    d = _kv_dims(umm, P, Hkv, D, ps, 64 * max(1, Hkv // max(1, Hkv // P)))
    k, vb = umm.umm_kv_copy_kernel(d, 0)
    assert ({umm.UMM_KV_COPY_TMA: "TMA", umm.UMM_KV_COPY_LSU: "LSU"}[k], vb) == want
    assert umm.umm_kv_copy_kernel(d, 1)[0] == umm.UMM_KV_COPY_LSU


def test_kv_copy_kernel_bad_arguments(umm):
    d = _kv_dims(umm, 8, 4, 128, 16, 64)
    for bad in (2, -1):
        with pytest.raises(umm.UmmError) as ei:
            umm.umm_kv_copy_kernel(d, bad)
        assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_kv_copy_kernel(umm.make_dims(P=8, E=8, H=8, I=8), 0)      # no KV cache
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG


def test_stall_hook_is_checked_build_only(umm):
    """The normal build refuses the TMA-wait test hook; the checked build
    accepts it only for a handle (the GPU test drives it)."""
    with pytest.raises(umm.UmmError) as ei:
        umm.umm_test_stall_tma_wait(0x1, 0, 64)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    with umm.checked_library():
        with pytest.raises(umm.UmmError) as ei:
            umm.umm_test_stall_tma_wait(None, 0, 64)
        assert ei.value.code == umm.UMM_ERR_INVALID_ARG
