"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by
element on whole buffers, at sizes the oracle finishes in seconds that still
span many tiles and ragged tails; plus error paths, address stability and
CUDA-graph capture.  Tolerance 0: the method is pure data movement."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ep_tp_weight_gb300 as umm
import oracle
import synth
from gpu_helpers import DevUMM, i32
from helpers import initial_kv_state
from synth.workloads import TINY, Workload

pytestmark = pytest.mark.gpu

# weights: 16 B vectors, 8 B vectors (I/P = 12), 4 B (I/P = 6), 2 B (odd H); split 1
W_CASES = [
    TINY,
    Workload("w_v8_ragged", P=4, N=3, E=8, H=200, I=48, w_sigma=0.02),
    Workload("w_v4", P=2, N=2, E=4, H=36, I=12),
    Workload("w_v2_oddh", P=3, N=2, E=6, H=35, I=9),
    Workload("w_p1", P=1, N=3, E=3, H=64, I=40),
    Workload("w_p8_tiles", P=8, N=2, E=16, H=256, I=128, w_sigma=0.02),
]

KV_CASES = [
    TINY,
    Workload("kv_hkv2_p4", P=4, N=3, Hkv=2, D=8, ps=4, R=9, len_a=1, len_b=23),
    Workload("kv_hkv8_p4_d12", P=4, N=2, Hkv=8, D=12, ps=5, R=13, len_a=1, len_b=41, slack=2.0),
    Workload("kv_hkv1_p4_d5", P=4, N=2, Hkv=1, D=5, ps=3, R=7, len_a=1, len_b=20),
    Workload("kv_hkv4_p8_d128", P=8, N=2, Hkv=4, D=128, ps=16, R=40, len_a=1, len_b=300, kv_sigma=1.0),
    Workload("kv_hkv4_p4_many_pages", P=4, N=2, Hkv=4, D=16, ps=8, R=300, len_a=1, len_b=200),
    # a pool much larger than the live pages: the copies walk the descriptor
    # list instead of the TP page pool
    Workload("kv_sparse_pool", P=4, N=2, Hkv=2, D=8, ps=4, R=9, len_a=1, len_b=23, slack=8.0),
]


@pytest.fixture(autouse=True)
def _sync():
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", W_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [0, 1])
def test_weights_full_buffer_parity(w, split):
    dev = DevUMM(w, seed=3, w13_split=split)
    d = oracle.Dims(**{**w.dims(), "w13_split": split})
    ref = dev.host()
    umm.reshard_weights_ep2tp(dev.h)
    oracle.weights_ep2tp(ref, d)
    np.testing.assert_array_equal(dev.host(), ref)
    assert umm.umm_get_modes(dev.h)[0] == umm.UMM_MODE_TP
    umm.reshard_weights_tp2ep(dev.h)
    oracle.weights_tp2ep(ref, d)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


def _kv_round(dev: DevUMM, w: Workload):
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=5)
    ref = dev.host()
    g = lambda a: i32(a)
    lens, owner, ep_pt, tp_pt = g(st.lens), g(st.owner), g(st.ep_pt), g(st.tp_pt)
    maxp = st.ep_pt.shape[1]
    umm.reshard_kv_ep2tp(dev.h, len(st.lens), maxp, lens, owner, ep_pt, tp_pt)
    assert oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    # a6 parity: the descriptors in the workspace
    nd = int(synth.npages(st.lens, d.ps).sum())
    want = oracle.kv_descriptors(d, 0, st.lens, st.owner, st.ep_pt, st.tp_pt)
    got = dev.buf[L["desc_off"]:L["desc_off"] + 32 * nd].view(torch.int32).reshape(nd, 8).cpu().numpy()
    np.testing.assert_array_equal(got, want)
    # TP -> EP with the greedy placement and new pages
    owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
    free2 = synth.permutation(8, 4, L["pages_ep"], rows=d.P)
    fl, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, maxp, free2, region=owner2, key=st.tp_pos)
    assert fl == 0
    umm.reshard_kv_tp2ep(dev.h, len(st.lens), maxp, lens, g(owner2), g(ep_pt2), tp_pt)
    assert oracle.kv_tp2ep(ref, d, st.lens, owner2, ep_pt2, st.tp_pt) == 0
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    want = oracle.kv_descriptors(d, 1, st.lens, owner2, ep_pt2, st.tp_pt)
    got = dev.buf[L["desc_off"]:L["desc_off"] + 32 * nd].view(torch.int32).reshape(nd, 8).cpu().numpy()
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("w", KV_CASES, ids=lambda w: w.name)
def test_kv_full_buffer_parity(w):
    dev = DevUMM(w, seed=4)
    _kv_round(dev, w)
    dev.close()


# Shapes at the limits of the TMA copy (one head per TP rank): the largest
# tiles that fit its 48 KiB of shared memory, and boxes of 256 elements and of
# 256 rows (the tensor-map box limit).  Whole buffers against the oracle.
TMA_EDGE_CASES = [
    Workload("kv_tma_tile_187rows_d128", P=2, N=2, Hkv=1, D=128, ps=187, R=5, len_a=1, len_b=600),
    Workload("kv_tma_two_heads_93rows_d128", P=2, N=2, Hkv=2, D=128, ps=93, R=5, len_a=1, len_b=400),
    Workload("kv_tma_head_256", P=2, N=2, Hkv=1, D=256, ps=16, R=6, len_a=1, len_b=90),
    Workload("kv_tma_page_256rows", P=2, N=2, Hkv=1, D=8, ps=256, R=6, len_a=1, len_b=1200),
]


@pytest.mark.parametrize("w", TMA_EDGE_CASES, ids=lambda w: w.name)
def test_kv_tma_edge_shapes(w):
    dev = DevUMM(w, seed=6)
    assert umm.umm_kv_copy_kernel(dev.dims, 0) == (umm.UMM_KV_COPY_TMA, 0)
    _kv_round(dev, w)
    dev.close()


def test_weights_and_kv_together_and_modes():
    w = TINY
    dev = DevUMM(w, seed=9)
    _kv_round(dev, w)
    ref = dev.host()
    umm.reshard_weights_ep2tp(dev.h)
    oracle.weights_ep2tp(ref, dev.d)
    np.testing.assert_array_equal(dev.host(), ref)
    with pytest.raises(umm.UmmError) as ei:
        umm.reshard_weights_ep2tp(dev.h)
    assert ei.value.code == umm.UMM_ERR_MODE
    with pytest.raises(umm.UmmError) as ei:
        umm.reshard_kv_tp2ep(dev.h, 0, 1, None, None, None, None)
    assert ei.value.code == umm.UMM_ERR_MODE
    dev.close()


# ------------------------------------------------------------------ request metadata

@pytest.mark.parametrize("P,R", [(2, 4), (8, 2048), (3, 1), (8, 5000), (16, 300), (5, 20000), (64, 100)])
def test_order_place_assign_parity(P, R):
    rng = np.random.default_rng(P * 1000 + R)
    lens = synth.lengths_lognormal(R, R, 2048, 1.0, 32768) if R > 50 else rng.integers(1, 60, R).astype(np.int32)
    if R > 100:
        lens[rng.integers(0, R, R // 10)] = 77      # many equal lengths: tie-breaks matter
    ps = 16
    maxp = int((lens.max() + ps - 1) // ps)
    w = Workload("meta", P=P, N=1, Hkv=P, D=8, ps=ps, R=R, len_a=1, len_b=1)
    pages_tp = (int(synth.npages(lens, ps).sum()) + 7 + P - 1) // P * P
    dev = DevUMM(w, fill=False, pages_tp=pages_tp, max_requests=R, max_pages=pages_tp)
    owner0 = rng.integers(0, P, R).astype(np.int32)
    dl, do = i32(lens), i32(owner0)
    tp_pos = torch.empty(R, dtype=torch.int32, device="cuda")
    umm.gather_requests_ep2tp(dev.h, R, do, tp_pos)
    want_pos = oracle.request_order(P, owner0)
    assert np.array_equal(tp_pos.cpu().numpy(), want_pos)
    owner = torch.empty(R, dtype=torch.int32, device="cuda")
    local = torch.empty(R, dtype=torch.int32, device="cuda")
    for key in (None, tp_pos):
        umm.place_requests_tp2ep(dev.h, R, dl, key, owner, local)
        wo, wl, _ = oracle.place(P, lens, None if key is None else want_pos)
        assert np.array_equal(owner.cpu().numpy(), wo)
        assert np.array_equal(local.cpu().numpy(), wl)
    # pages: one pool in list order, and per-rank pools in local order
    free = synth.permutation(1, 3, pages_tp, rows=1)
    pt = torch.full((R, maxp), -9, dtype=torch.int32, device="cuda")
    umm.umm_assign_pages(dev.h, 1, R, dl, None, tp_pos, i32(free), pages_tp, pages_tp, pt, maxp)
    fl, want = oracle.assign_pages(1, lens, ps, maxp, free, key=want_pos)
    assert fl == 0 and np.array_equal(pt.cpu().numpy(), want)
    n_ep = pages_tp                                  # generous per-rank free lists
    free_ep = synth.permutation(2, 4, n_ep, rows=P)
    wo, _, _ = oracle.place(P, lens, want_pos)
    fl, want = oracle.assign_pages(P, lens, ps, maxp, free_ep, region=wo, key=want_pos)
    umm.umm_assign_pages(dev.h, P, R, dl, i32(wo), tp_pos, i32(free_ep), n_ep, n_ep, pt, maxp)
    st = dev.status()
    if fl == 0:
        assert st == (0, 0) and np.array_equal(pt.cpu().numpy(), want)
    else:
        assert st[0] == umm.UMM_ERR_CAPACITY
    dev.close()


# (P, R, length range): together they reach every variant of the device
# greedy (8 or 16 ranks with 32-bit loads, 16 ranks with 64-bit loads, one
# rank per lane, loads in local memory) and every sort (registers with 1, 2
# and 4 keys per thread, the network in shared memory, the network over the
# workspace).  Totals of 2^27..2^29 tokens and more force the wide words.
PLACE_VARIANTS = [
    (8, 1000, (1, 4000)), (8, 4000, (1, 4000)), (7, 9000, (1, 4000)), (8, 17000, (1, 300)),
    (12, 2500, (1, 4000)), (12, 3000, (100_000, 200_000)), (6, 3000, (150_000, 250_000)),
    (24, 1500, (1, 4000)), (24, 1500, (100_000, 200_000)), (40, 800, (1, 4000)),
]


@pytest.mark.parametrize("P,R,lr", PLACE_VARIANTS, ids=lambda v: str(v))
def test_place_variants(P, R, lr):
    rng = np.random.default_rng(P * 7919 + R)
    lens = rng.integers(lr[0], lr[1] + 1, R).astype(np.int32)
    lens[rng.integers(0, R, R // 8)] = lr[0]              # ties on length
    w = Workload("meta", P=P, N=1, Hkv=P, D=8, ps=16, R=R, len_a=1, len_b=1)
    dev = DevUMM(w, fill=False, pages_tp=2 * P, max_requests=R, max_pages=2 * P)
    key = rng.permutation(R).astype(np.int32)
    owner = torch.empty(R, dtype=torch.int32, device="cuda")
    local = torch.empty_like(owner)
    for k in (None, key):
        umm.place_requests_tp2ep(dev.h, R, i32(lens), None if k is None else i32(k), owner, local)
        wo, wl, _ = oracle.place(P, lens, k)
        assert np.array_equal(owner.cpu().numpy(), wo)
        assert np.array_equal(local.cpu().numpy(), wl)
    assert dev.status() == (0, 0)
    dev.close()


def test_empty_and_degenerate_requests():
    w = Workload("deg", P=4, N=2, Hkv=4, D=8, ps=4, R=3, len_a=0, len_b=0)
    dev = DevUMM(w, seed=1, pages_tp=8, max_requests=8, max_pages=8)
    ref = dev.host()
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    umm.reshard_kv_ep2tp(dev.h, 0, 1, z, z, z, z)              # R = 0: nothing moves
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    lens = np.array([0, 0, 0], np.int32)                      # zero-length requests
    pt = np.full((3, 2), -1, np.int32)
    umm.reshard_kv_tp2ep(dev.h, 3, 2, i32(lens), i32([0, 1, 2]), i32(pt), i32(pt))
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


# ------------------------------------------------------------------ error paths (all-or-nothing)

@pytest.mark.parametrize("mode,sigma", [(synth.RAW, 1.0), (synth.NORMAL, 1.0), (synth.NORMAL, 0.02)])
def test_device_generator_equals_host_generator(mode, sigma):
    """The seeded inputs: the device fill (synth_fill.cu) writes exactly what
    the host generator defines, element i = value of index base + i, for odd
    bases and lengths and for a start that is not 16-byte aligned (the
    kernel's scalar path)."""
    from gpu_helpers import table_dev
    out = torch.zeros(1 << 21, dtype=torch.int16, device="cuda")
    for seed, base, n, skew in ((0, 0, 1 << 20, 0), (7, 12345, 999_997, 1), (1 << 40, 3, 8, 3), (5, 1 << 33, 17, 0)):
        out.zero_()
        synth.fill_device(out.data_ptr() + 2 * skew, n, seed, mode, table_dev(sigma).data_ptr() if mode else 0,
                          base=base)
        want = synth.fill_host(n, seed, mode, sigma, base=base).view(np.int16)
        got = out.cpu().numpy()
        np.testing.assert_array_equal(got[skew:skew + n], want)
        assert not got[:skew].any() and not got[skew + n:].any()


def test_largest_request_count():
    """R = 2^26, the most requests a handle accepts, through the single-CTA
    request-order and page hand-out kernels.  The oracle's definitions are
    quadratic in R, so the results are checked against what they reduce to
    here (§3.2 list order, page hand-out in list order): with every request on
    rank 0 the list position is the request index, and with one-token
    requests from one pool, request k takes the k-th free page."""
    R = 1 << 26
    dims = umm.make_dims(P=1, N=1, ps=16, max_requests=R)
    nbytes = umm.umm_required_bytes(dims)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    h = umm.umm_create(dims, buf, nbytes)
    owner = torch.zeros(R, dtype=torch.int32, device="cuda")
    tp_pos = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    umm.gather_requests_ep2tp(h, R, owner, tp_pos)
    lens = torch.ones(R, dtype=torch.int32, device="cuda")
    free = torch.randperm(R, device="cuda", generator=torch.Generator(device="cuda").manual_seed(3)).int()
    pt = torch.full((R, 1), -2, dtype=torch.int32, device="cuda")
    umm.umm_assign_pages(h, 1, R, lens, None, None, free, R, R, pt, 1)
    assert umm.umm_status_sync(h) == (0, 0)
    assert torch.equal(tp_pos, torch.arange(R, dtype=torch.int32, device="cuda"))
    assert torch.equal(pt[:, 0], free)
    umm.umm_destroy(h)
    del buf, owner, tp_pos, lens, free, pt
    torch.cuda.empty_cache()


def test_kv_device_errors_leave_buffer_untouched():
    w = KV_CASES[1]
    dev = DevUMM(w, seed=2)
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=5)
    ref = dev.host()
    maxp = st.ep_pt.shape[1]
    cases = []
    bad = st.ep_pt.copy(); bad[0, 0] = L["pages_ep"]; cases.append(("ep_pt", bad, umm.UMM_ERR_PAGE_OOB))
    bad = st.tp_pt.copy(); bad[0, 0] = -1; cases.append(("tp_pt", bad, umm.UMM_ERR_PAGE_OOB))
    k2 = int(np.argmax(st.lens > d.ps))
    bad = st.tp_pt.copy(); bad[k2, 1] = bad[0, 0]; cases.append(("tp_pt", bad, umm.UMM_ERR_DUP_PAGE))
    bad = st.lens.copy(); bad[1] = -3; cases.append(("lens", bad, umm.UMM_ERR_BAD_REQUEST))
    bad = st.owner.copy(); bad[2] = d.P; cases.append(("owner", bad, umm.UMM_ERR_BAD_REQUEST))
    for name, arr, code in cases:
        a = dict(lens=st.lens, owner=st.owner, ep_pt=st.ep_pt, tp_pt=st.tp_pt)
        a[name] = arr
        want = oracle.kv_validate(d, 0, a["lens"], a["owner"], a["ep_pt"], a["tp_pt"])
        umm.reshard_kv_ep2tp(dev.h, len(st.lens), maxp, i32(a["lens"]), i32(a["owner"]), i32(a["ep_pt"]),
                             i32(a["tp_pt"]))
        assert umm.umm_get_modes(dev.h)[1] == umm.UMM_MODE_TP      # flipped at enqueue ...
        code_got, flags = dev.status()
        assert (code_got, flags) == (code, want), name
        assert umm.umm_get_modes(dev.h)[1] == umm.UMM_MODE_EP      # ... restored by the sync
        np.testing.assert_array_equal(dev.host(), ref)
    # TP -> EP: two requests reading the same TP page
    umm.umm_set_modes(dev.h, umm.UMM_MODE_EP, umm.UMM_MODE_TP)
    owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
    free2 = synth.permutation(8, 4, L["pages_ep"], rows=d.P)
    _, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, maxp, free2, region=owner2, key=st.tp_pos)
    bad_tp = st.tp_pt.copy()
    bad_tp[k2, 1] = bad_tp[0, 0]
    want = oracle.kv_validate(d, 1, st.lens, owner2, ep_pt2, bad_tp)
    umm.reshard_kv_tp2ep(dev.h, len(st.lens), maxp, i32(st.lens), i32(owner2), i32(ep_pt2), i32(bad_tp))
    assert dev.status() == (umm.UMM_ERR_DUP_PAGE, want) and want == oracle.F_DUP_PAGE
    assert umm.umm_get_modes(dev.h)[1] == umm.UMM_MODE_TP
    np.testing.assert_array_equal(dev.host(), ref)
    umm.umm_set_modes(dev.h, umm.UMM_MODE_EP, umm.UMM_MODE_EP)
    # sticky: a failed page hand-out stops the following KV call too
    big = np.full(len(st.lens), 10**6, np.int32)
    pt = torch.zeros(st.tp_pt.shape, dtype=torch.int32, device="cuda")
    umm.umm_assign_pages(dev.h, 1, len(st.lens), i32(big), None, None, i32(np.arange(4)), 4, 4, pt, maxp)
    umm.reshard_kv_ep2tp(dev.h, len(st.lens), maxp, i32(st.lens), i32(st.owner), i32(st.ep_pt), i32(st.tp_pt))
    assert dev.status()[0] == umm.UMM_ERR_BAD_REQUEST
    np.testing.assert_array_equal(dev.host(), ref)
    assert umm.umm_get_modes(dev.h)[1] == umm.UMM_MODE_EP
    # capacity: more pages than the TP pool
    small = DevUMM(w, seed=2, pages_tp=int(synth.npages(st.lens, d.ps).sum()) // 2 // 2 * 2)
    ref2 = small.host()
    umm.reshard_kv_ep2tp(small.h, len(st.lens), maxp, i32(st.lens), i32(st.owner),
                         i32(np.zeros_like(st.ep_pt)), i32(st.tp_pt))
    assert small.status()[0] == umm.UMM_ERR_CAPACITY
    np.testing.assert_array_equal(small.host(), ref2)
    assert umm.umm_kv_check_capacity(small.h, umm.UMM_MODE_TP, len(st.lens), st.lens) == umm.UMM_ERR_CAPACITY
    assert umm.umm_kv_check_capacity(dev.h, umm.UMM_MODE_TP, len(st.lens), st.lens) == umm.UMM_OK
    small.close()
    dev.close()


# ------------------------------------------------------------------ fixed addresses, graphs, no allocation

def test_address_stability_graph_replay_and_no_allocation():
    """§4.2: tensors keep their addresses across switches, so a CUDA graph
    captured on the TP views before any switch reads the right data after
    EP->TP->EP->TP; and the switch path allocates no device memory."""
    w = Workload("gr", P=4, N=2, E=8, H=64, I=32, Hkv=4, D=16, ps=4, R=6, len_a=1, len_b=30, slack=3.0)
    dev = DevUMM(w, seed=6)
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=1)
    ref = dev.host()
    maxp = st.ep_pt.shape[1]
    lens, owner, ep_pt, tp_pt = i32(st.lens), i32(st.owner), i32(st.ep_pt), i32(st.tp_pt)
    # probe graph: copy TP slot 0 of every region (weights + KV) into a probe buffer
    spans = [(r * L["region_stride"], L["wslot_stride"]) for r in range(d.P)] + \
            [(r * L["region_stride"] + L["kvslots_off"], L["kvslot_stride"]) for r in range(d.P)]
    probe = torch.empty(sum(n for _, n in spans), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    views = [dev.buf[a:a + n] for a, n in spans]
    ptrs = [v.data_ptr() for v in views]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            torch.cat(views, out=probe)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    cur = torch.cuda.current_stream()
    owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
    free2 = synth.permutation(8, 4, L["pages_ep"], rows=d.P)
    _, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, maxp, free2, region=owner2, key=st.tp_pos)
    o2, e2 = i32(owner2), i32(ep_pt2)
    # EP -> TP -> EP -> TP, on the current stream, no allocation in between
    umm.reshard_weights_ep2tp(dev.h, cur); umm.reshard_kv_ep2tp(dev.h, len(st.lens), maxp, lens, owner, ep_pt, tp_pt, cur)
    umm.reshard_weights_tp2ep(dev.h, cur); umm.reshard_kv_tp2ep(dev.h, len(st.lens), maxp, lens, o2, e2, tp_pt, cur)
    umm.reshard_weights_ep2tp(dev.h, cur); umm.reshard_kv_ep2tp(dev.h, len(st.lens), maxp, lens, o2, e2, tp_pt, cur)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert dev.status() == (0, 0)
    g.replay()
    torch.cuda.synchronize()
    assert [v.data_ptr() for v in views] == ptrs
    oracle.weights_ep2tp(ref, d); oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, st.tp_pt)
    oracle.weights_tp2ep(ref, d); oracle.kv_tp2ep(ref, d, st.lens, owner2, ep_pt2, st.tp_pt)
    oracle.weights_ep2tp(ref, d); oracle.kv_ep2tp(ref, d, st.lens, owner2, ep_pt2, st.tp_pt)
    want = np.concatenate([ref[a:a + n] for a, n in spans])
    np.testing.assert_array_equal(probe.cpu().numpy(), want)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


def test_switch_captured_in_a_cuda_graph():
    """The switch itself enqueues only kernels on the given stream, so a whole
    EP->TP switch (weights + KV) can be captured once and replayed."""
    w = Workload("cap", P=4, N=2, E=8, H=64, I=32, Hkv=2, D=16, ps=4, R=5, len_a=1, len_b=25, slack=3.0)
    dev = DevUMM(w, seed=7)
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=2)
    maxp = st.ep_pt.shape[1]
    lens, owner, ep_pt, tp_pt = i32(st.lens), i32(st.owner), i32(st.ep_pt), i32(st.tp_pt)
    ref = dev.host()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            umm.reshard_weights_ep2tp(dev.h, s)
            umm.reshard_kv_ep2tp(dev.h, len(st.lens), maxp, lens, owner, ep_pt, tp_pt, s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dev.host(), ref)        # capture ran nothing
    g.replay()
    torch.cuda.synchronize()
    oracle.weights_ep2tp(ref, d)
    oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, st.tp_pt)
    np.testing.assert_array_equal(dev.host(), ref)
    assert dev.status() == (0, 0)
    dev.close()


def test_overlapped_switch_captured_in_a_cuda_graph():
    """With the side stream on, one call still forms one unit: a captured
    umm_switch_ep2tp (weights on the side stream, bookkeeping and KV on the
    capturing stream) replays to the oracle's result, and nothing ran during
    the capture."""
    w = Workload("cap_ovl", P=4, N=2, E=8, H=64, I=32, Hkv=2, D=16, ps=4, R=5, len_a=1, len_b=25, slack=3.0)
    dev = DevUMM(w, seed=8)
    umm.umm_set_switch_overlap(dev.h, True)
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=4)
    R, maxp = len(st.lens), st.ep_pt.shape[1]
    tp_free = synth.permutation(6, 3, L["pages_tp"], rows=1)
    d_pos = torch.empty(R, dtype=torch.int32, device="cuda")
    d_tp_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
    args = (i32(st.lens), i32(st.owner), i32(st.ep_pt), i32(tp_free))
    ref = dev.host()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            umm.umm_switch_ep2tp(dev.h, R, maxp, *args[:3], args[3], L["pages_tp"], d_pos, d_tp_pt, s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dev.host(), ref)        # capture ran nothing
    g.replay()
    torch.cuda.synchronize()
    pos = oracle.request_order(d.P, st.owner)
    _, tp_pt = oracle.assign_pages(1, st.lens, d.ps, maxp, tp_free, key=pos)
    oracle.weights_ep2tp(ref, d)
    assert oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, tp_pt) == 0
    np.testing.assert_array_equal(dev.host(), ref)
    np.testing.assert_array_equal(d_tp_pt.cpu().numpy(), tp_pt)
    assert dev.status() == (0, 0)
    dev.close()


# ------------------------------------------------------------------ staged (collective-style) comparison path

@pytest.mark.parametrize("w", [TINY, W_CASES[1], W_CASES[3], W_CASES[5]], ids=lambda w: w.name)
def test_weights_staged_equals_oracle(w):
    """The staged path (permute into per-peer blocks + exchange) lands the
    same bytes as the definition."""
    dev = DevUMM(w, seed=13)
    nb = umm.umm_weights_stage_bytes(dev.h)
    stage = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ref = dev.host()
    umm.reshard_weights_ep2tp_staged(dev.h, stage, nb)
    oracle.weights_ep2tp(ref, dev.d)
    np.testing.assert_array_equal(dev.host(), ref)
    umm.reshard_weights_tp2ep_staged(dev.h, stage, nb)
    oracle.weights_tp2ep(ref, dev.d)
    np.testing.assert_array_equal(dev.host(), ref)
    with pytest.raises(umm.UmmError) as ei:
        umm.reshard_weights_ep2tp_staged(dev.h, stage, nb - 16)
    assert ei.value.code == umm.UMM_ERR_CAPACITY
    dev.close()


@pytest.mark.parametrize("w", KV_CASES, ids=lambda w: w.name)
def test_kv_staged_equals_oracle(w):
    """The staged KV path (gather into per-peer blocks, exchange, scatter)
    lands the same bytes as the definition, both directions."""
    dev = DevUMM(w, seed=14)
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=5)
    nb = umm.umm_kv_stage_bytes(dev.h)
    stage = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ref = dev.host()
    maxp = st.ep_pt.shape[1]
    g = lambda a: i32(a)
    umm.reshard_kv_ep2tp_staged(dev.h, stage, nb, len(st.lens), maxp, g(st.lens), g(st.owner), g(st.ep_pt),
                                g(st.tp_pt))
    assert oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    owner2, _, _ = oracle.place(d.P, st.lens, key=st.tp_pos)
    free2 = synth.permutation(8, 4, L["pages_ep"], rows=d.P)
    _, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, maxp, free2, region=owner2, key=st.tp_pos)
    umm.reshard_kv_tp2ep_staged(dev.h, stage, nb, len(st.lens), maxp, g(st.lens), g(owner2), g(ep_pt2),
                                g(st.tp_pt))
    assert oracle.kv_tp2ep(ref, d, st.lens, owner2, ep_pt2, st.tp_pt) == 0
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


# ------------------------------------------------------------------ attention weights (memory-saving variant)

ATTN_CASES = [
    Workload("attn_p2_hq2_hkv1", P=2, N=2, H=64, Hkv=1, D=16, Hq=2),
    Workload("attn_p4_hq8_hkv2", P=4, N=3, H=96, Hkv=2, D=8, Hq=8, w_sigma=0.02),
    Workload("attn_p4_hq8_hkv8_odd", P=4, N=2, H=36, Hkv=8, D=6, Hq=8),           # 8-byte vectors
    Workload("attn_p8_hq64_hkv4_d128", P=8, N=2, H=512, Hkv=4, D=128, Hq=64, w_sigma=0.02),
    Workload("attn_p4_h7", P=4, N=2, H=7, Hkv=4, D=3, Hq=4),                       # 2-byte vectors
    Workload("attn_p4_hq4_d8", P=4, N=2, H=24, Hkv=2, D=8, Hq=4),                   # 16-byte vectors
]


@pytest.mark.parametrize("w", ATTN_CASES, ids=lambda w: w.name)
def test_attn_full_buffer_parity(w):
    dev = DevUMM(w, seed=15)
    ref = dev.host()
    umm.reshard_attn_ep2tp(dev.h)
    oracle.attn_ep2tp(ref, dev.d)
    np.testing.assert_array_equal(dev.host(), ref)
    assert umm.umm_get_attn_mode(dev.h) == umm.UMM_MODE_TP
    with pytest.raises(umm.UmmError) as ei:
        umm.reshard_attn_ep2tp(dev.h)
    assert ei.value.code == umm.UMM_ERR_MODE
    umm.reshard_attn_tp2ep(dev.h)
    oracle.attn_tp2ep(ref, dev.d)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


def test_attn_needs_attention_dims():
    dev = DevUMM(TINY, seed=1)
    with pytest.raises(umm.UmmError) as ei:
        umm.reshard_attn_ep2tp(dev.h)
    assert ei.value.code == umm.UMM_ERR_INVALID_ARG
    dev.close()


# ------------------------------------------------------------------ one call per direction

@pytest.mark.parametrize("w", [TINY.with_(Hq=4), Workload("switch_mid", P=4, N=3, E=8, H=40, I=24, Hkv=2, D=8, ps=4,
                                                            R=20, len_a=1, len_b=37, slack=3.0, Hq=8)],
                         ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ["serial", "overlap", "timed"])
def test_switch_entry_points_equal_oracle(w, mode):
    """umm_switch_ep2tp / umm_switch_tp2ep: weights, attention, request
    order, page hand-out and KV in one call each; the same bytes and metadata
    as the oracle's step-by-step definition, with the weights on the caller's
    stream or on the handle's side stream (overlap), and with per-kernel
    timing on (timed: one event pair around each call's chain of layer copies,
    one unit counted per layer): the same bytes each way."""
    dev = DevUMM(w, seed=17)
    umm.umm_set_switch_overlap(dev.h, mode == "overlap")
    umm.umm_profile_enable(dev.h, mode == "timed")
    d, L = dev.d, dev.L
    st = initial_kv_state(w, d, L, seed=3)
    R, maxp = len(st.lens), st.ep_pt.shape[1]
    ref = dev.host()
    tp_free = synth.permutation(5, 3, L["pages_tp"], rows=1)
    ep_free = synth.permutation(5, 4, L["pages_ep"], rows=d.P)
    d_pos = torch.empty(R, dtype=torch.int32, device="cuda")
    d_tp_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
    umm.umm_switch_ep2tp(dev.h, R, maxp, i32(st.lens), i32(st.owner), i32(st.ep_pt), i32(tp_free), L["pages_tp"],
                         d_pos, d_tp_pt)
    pos = oracle.request_order(d.P, st.owner)
    _, tp_pt = oracle.assign_pages(1, st.lens, d.ps, maxp, tp_free, key=pos)
    oracle.weights_ep2tp(ref, d)
    oracle.attn_ep2tp(ref, d)
    assert oracle.kv_ep2tp(ref, d, st.lens, st.owner, st.ep_pt, tp_pt) == 0
    assert dev.status() == (0, 0)
    assert np.array_equal(d_pos.cpu().numpy(), pos) and np.array_equal(d_tp_pt.cpu().numpy(), tp_pt)
    np.testing.assert_array_equal(dev.host(), ref)
    assert umm.umm_get_modes(dev.h) == (umm.UMM_MODE_TP, umm.UMM_MODE_TP)
    d_owner = torch.empty(R, dtype=torch.int32, device="cuda")
    d_local = torch.empty_like(d_owner)
    d_ep_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
    umm.umm_switch_tp2ep(dev.h, R, maxp, i32(st.lens), d_pos, d_tp_pt, i32(ep_free), L["pages_ep"], L["pages_ep"],
                         d_owner, d_local, d_ep_pt)
    owner2, local2, _ = oracle.place(d.P, st.lens, key=pos)
    _, ep_pt2 = oracle.assign_pages(d.P, st.lens, d.ps, maxp, ep_free, region=owner2, key=pos)
    oracle.weights_tp2ep(ref, d)
    oracle.attn_tp2ep(ref, d)
    assert oracle.kv_tp2ep(ref, d, st.lens, owner2, ep_pt2, tp_pt) == 0
    assert dev.status() == (0, 0)
    assert np.array_equal(d_owner.cpu().numpy(), owner2) and np.array_equal(d_local.cpu().numpy(), local2)
    assert np.array_equal(d_ep_pt.cpu().numpy(), ep_pt2)
    np.testing.assert_array_equal(dev.host(), ref)
    with pytest.raises(umm.UmmError) as ei:      # already EP: nothing enqueued
        umm.umm_switch_tp2ep(dev.h, R, maxp, i32(st.lens), d_pos, d_tp_pt, i32(ep_free), L["pages_ep"],
                             L["pages_ep"], d_owner, d_local, d_ep_pt)
    assert ei.value.code == umm.UMM_ERR_MODE
    if mode == "timed":
        launches = {umm.KIND_NAMES[k]: umm.umm_profile_read(dev.h, k)[0] for k in range(umm.K_COUNT)}
        for kind in ("weights_ep2tp", "weights_tp2ep", "kv_ep2tp", "kv_tp2ep", "attn_ep2tp", "attn_tp2ep"):
            assert launches[kind] == d.N, (kind, launches)
    dev.close()


@pytest.mark.parametrize("overlap", [False, True], ids=["serial", "overlap"])
def test_many_round_trips_stay_exact(overlap):
    """40 EP->TP->EP round trips through umm_switch_* on one handle, each with
    fresh free lists, the KV pool two-thirds full so that the copies walk it
    through the call-tagged TP-page schedule (stale entries of earlier calls
    must be ignored), and the status read only at the end: equal to the
    oracle step for step.  The layer copies launch chained; with overlap the
    weight chains run on the side stream beside the KV chains."""
    w = Workload("many_trips", P=4, N=2, E=8, H=32, I=16, Hkv=2, D=16, ps=4, R=24, len_a=1, len_b=30,
                 slack=1.5, Hq=8)
    lens = w.lengths().copy()
    trips = 40
    maxp = int((lens.max() + w.ps - 1) // w.ps)
    used = int(((lens + w.ps - 1) // w.ps).sum())
    m = w.Hkv // w.h_tp
    ptp = (int(1.5 * used) + m - 1) // m * m
    dev = DevUMM(w, seed=29, pages_tp=ptp, max_requests=len(lens), max_pages=ptp)
    umm.umm_set_switch_overlap(dev.h, overlap)
    d, L = dev.d, dev.L
    R, P = len(lens), d.P
    owner, _, _ = oracle.place(P, lens)
    _, ep_pt = oracle.assign_pages(P, lens, d.ps, maxp, synth.permutation(1, 2, L["pages_ep"], rows=P), region=owner)
    ref = dev.host()
    d_owner, d_ep_pt = i32(owner), i32(ep_pt)
    d_pos = torch.empty(R, dtype=torch.int32, device="cuda")
    d_tp_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
    d_local = torch.empty(R, dtype=torch.int32, device="cuda")
    for trip in range(trips):
        tp_free = synth.permutation(100 + trip, 3, L["pages_tp"], rows=1)
        ep_free = synth.permutation(100 + trip, 4, L["pages_ep"], rows=P)
        d_lens = i32(lens)
        umm.umm_switch_ep2tp(dev.h, R, maxp, d_lens, d_owner, d_ep_pt, i32(tp_free), L["pages_tp"], d_pos, d_tp_pt)
        pos = oracle.request_order(P, owner)
        _, tp_pt = oracle.assign_pages(1, lens, d.ps, maxp, tp_free, key=pos)
        oracle.weights_ep2tp(ref, d)
        oracle.attn_ep2tp(ref, d)
        assert oracle.kv_ep2tp(ref, d, lens, owner, ep_pt, tp_pt) == 0
        n_owner = torch.empty(R, dtype=torch.int32, device="cuda")
        n_ep_pt = torch.empty((R, maxp), dtype=torch.int32, device="cuda")
        umm.umm_switch_tp2ep(dev.h, R, maxp, d_lens, d_pos, d_tp_pt, i32(ep_free), L["pages_ep"], L["pages_ep"],
                             n_owner, d_local, n_ep_pt)
        owner, _, _ = oracle.place(P, lens, key=pos)
        _, ep_pt = oracle.assign_pages(P, lens, d.ps, maxp, ep_free, region=owner, key=pos)
        oracle.weights_tp2ep(ref, d)
        oracle.attn_tp2ep(ref, d)
        assert oracle.kv_tp2ep(ref, d, lens, owner, ep_pt, tp_pt) == 0
        d_owner, d_ep_pt = n_owner, n_ep_pt
    assert dev.status() == (0, 0)
    np.testing.assert_array_equal(d_owner.cpu().numpy(), owner)
    np.testing.assert_array_equal(d_ep_pt.cpu().numpy(), ep_pt)
    np.testing.assert_array_equal(dev.host(), ref)
    dev.close()


def test_request_metadata_errors_are_refused_on_device():
    """Bad owners, pools, list positions and pool shortage raise flags and
    leave the outputs untouched."""
    w = Workload("meta_err", P=4, N=1, Hkv=4, D=8, ps=4, R=6, len_a=1, len_b=9)
    dev = DevUMM(w, fill=False, pages_tp=64, max_requests=8, max_pages=64)
    lens = i32([3, 9, 1, 4, 8, 2])
    out = torch.full((6,), -7, dtype=torch.int32, device="cuda")
    umm.gather_requests_ep2tp(dev.h, 6, i32([0, 1, 4, 2, 3, 1]), out)          # owner 4 >= P
    assert dev.status()[0] == umm.UMM_ERR_BAD_REQUEST and (out.cpu() == -7).all()
    own = torch.full((6,), -7, dtype=torch.int32, device="cuda")
    loc = torch.full((6,), -7, dtype=torch.int32, device="cuda")
    umm.place_requests_tp2ep(dev.h, 6, lens, i32([0, 1, 2, 2, 4, 5]), own, loc)  # position 2 twice
    assert dev.status()[0] == umm.UMM_ERR_BAD_REQUEST
    assert (own.cpu() == -7).all() and (loc.cpu() == -7).all()
    umm.place_requests_tp2ep(dev.h, 6, i32([3, -1, 1, 4, 8, 2]), None, own, loc)  # negative length
    assert dev.status()[0] == umm.UMM_ERR_BAD_REQUEST and (own.cpu() == -7).all()
    pt = torch.full((6, 3), -7, dtype=torch.int32, device="cuda")
    free = i32(np.arange(40))
    umm.umm_assign_pages(dev.h, 2, 6, lens, i32([0, 1, 2, 0, 1, 0]), None, free, 20, 20, pt, 3)   # pool 2 >= 2
    assert dev.status()[0] == umm.UMM_ERR_BAD_REQUEST and (pt.cpu() == -7).all()
    umm.umm_assign_pages(dev.h, 1, 6, lens, None, i32([5, 4, 3, 2, 1, 7]), free, 40, 40, pt, 3)  # key 7 >= R
    assert dev.status()[0] == umm.UMM_ERR_BAD_REQUEST and (pt.cpu() == -7).all()
    umm.umm_assign_pages(dev.h, 1, 6, lens, None, None, free, 40, 8, pt, 3)      # 9 pages needed, 8 free
    assert dev.status()[0] == umm.UMM_ERR_CAPACITY and (pt.cpu() == -7).all()
    umm.umm_assign_pages(dev.h, 1, 6, lens, None, None, free, 40, 9, pt, 3)      # exactly enough
    assert dev.status() == (0, 0)
    fl, want = oracle.assign_pages(1, [3, 9, 1, 4, 8, 2], 4, 3, np.arange(9))
    assert fl == 0 and np.array_equal(pt.cpu().numpy(), want)
    dev.close()
