"""bench.py on the CPU: the reference arm's JSON line (the oracle, timed), the
silence of ranks other than 0, and the algorithmic byte model that every GB/s
figure divides by, checked against the elements the oracle actually writes."""
from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest

import bench
import oracle
import synth
from helpers import attnslot, dims_of, initial_kv_state, kvslot, wslot
from synth.workloads import TINY, Workload

ROOT = Path(__file__).resolve().parent.parent


def _run_bench(*args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def test_reference_arm_prints_one_complete_line():
    r = _run_bench("--impl", "reference", "--workload", TINY.name, "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == bench.METRIC and j["unit"] == bench.UNIT
    assert j["value"] > 0 and j["higher_is_better"] is True
    assert j["steps"] == 2 and j["warmup"] == 1
    assert j["config"]["workload"] == TINY.name
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    r = _run_bench("--impl", "reference", "--workload", TINY.name, "--steps", "1", "--warmup", "0",
                   env_extra={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


# ---------------------------------------------------------------- byte model

def _nonzero_u16(buf: np.ndarray, spans) -> int:
    u = buf.view(np.uint16)
    return int(sum(np.count_nonzero(u[a // 2:(a + n) // 2]) for a, n in spans))


BYTE_CASES = [
    TINY,                                                                     # Hkv = P: one copy per head
    Workload("bytes_rep", P=4, N=1, E=8, H=24, I=16, Hkv=2, D=8, ps=4, R=9, len_a=0, len_b=23, slack=3.0),
    Workload("bytes_wide", P=2, N=1, E=4, H=8, I=6, Hkv=4, D=4, ps=3, R=7, len_a=1, len_b=17, slack=3.0),
]


@pytest.mark.parametrize("w", BYTE_CASES, ids=lambda w: w.name)
def test_algorithmic_bytes_equal_elements_the_oracle_moves(w):
    """Zero the destination slot, make every source element nonzero, run the
    oracle, count destination elements that became nonzero: that count (x2
    bytes) is what bench.py charges as written, and the live source elements
    as read."""
    d = dims_of(w)
    L = oracle.layout(d)
    buf = np.zeros(L["ws_off"], dtype=np.uint8)
    lens = w.lengths()
    b = bench.algorithmic_bytes(w, lens)
    u = buf.view(np.uint16)
    # ---- weights EP -> TP: EP slot 1 -> TP slot 0
    for r in range(w.P):
        a = wslot(L, r, 1) // 2
        u[a:a + L["wslot_stride"] // 2] = 0x3f80
    oracle.weights_ep2tp(buf, d)
    written = _nonzero_u16(buf, [(wslot(L, r, 0), L["wslot_stride"]) for r in range(w.P)])
    assert 2 * 2 * written == b["weights_per_layer"]        # one read + one write per element moved
    # ---- KV EP -> TP: EP slot 1 -> TP slot 0 (replicas counted as written)
    st = initial_kv_state(w, d, L, seed=3)
    buf[:] = 0
    for r in range(w.P):
        a = kvslot(L, r, 1, 0) // 2
        u[a:a + L["kvslot_stride"] // 2] = 0x3f80
    assert oracle.kv_ep2tp(buf, d, st.lens, st.owner, st.ep_pt, st.tp_pt) == 0
    tp_spans = [(kvslot(L, r, 0, 0), L["kvslot_stride"]) for r in range(w.P)]
    wr = 2 * _nonzero_u16(buf, tp_spans)
    rd = 2 * int(st.lens.sum()) * w.Hkv * w.D * 2            # live K and V rows of the EP pages
    assert rd + wr == b["kv_ep2tp_per_layer"]
    # ---- KV TP -> EP: TP slot 0 -> EP slot 1, each head read once (lowest replica)
    owner2, _, _ = oracle.place(w.P, st.lens, key=st.tp_pos)
    maxp = w.max_pages_per_req()
    _, ep_pt2 = oracle.assign_pages(w.P, st.lens, w.ps, maxp,
                                    synth.permutation(5, 4, L["pages_ep"], w.P), region=owner2, key=st.tp_pos)
    for r in range(w.P):
        a = kvslot(L, r, 1, 0) // 2
        u[a:a + L["kvslot_stride"] // 2] = 0
    assert oracle.kv_tp2ep(buf, d, st.lens, owner2, ep_pt2, st.tp_pt) == 0
    wr2 = 2 * _nonzero_u16(buf, [(kvslot(L, r, 1, 0), L["kvslot_stride"]) for r in range(w.P)])
    assert 2 * wr2 == b["kv_tp2ep_per_layer"]               # read once, written once
    assert b["tokens"] == int(lens.sum())


def test_ceiling_program_compiles():
    """The read:write-mix ceiling program behind `bench.py --ceilings` builds
    for sm_103a (nvcc cross-compiles here; it runs only on a GPU)."""
    import shutil
    if shutil.which("nvcc") is None:
        pytest.skip("nvcc not on PATH")
    from ep_tp_weight_gb300 import build as umm_build
    exe = umm_build.build_ceiling()
    assert os.path.exists(exe) and os.access(exe, os.X_OK)


def test_kernel_table_rates_and_fractions():
    """The per-kernel rows of the bench line (full switch and `configs`):
    GB/s = algorithmic bytes of one layer copy / ms per layer, and its
    fractions of the measured peak and of the kernel's mix ceiling."""
    b = {"weights_per_layer": 2_000_000_000, "kv_ep2tp_per_layer": 6_000_000_000}
    prof = {"weights_ep2tp": (4, 1.0), "kv_ep2tp": (8, 8.0), "place": (2, 0.2), "order": (0, 0.0)}
    ceil = {"1R1W sequential": 8000.0, "1R2W shuffled reads": 6000.0}
    t = bench.kernel_table(prof, b, 7000.0, ceil)
    assert set(t) == {"weights_ep2tp", "kv_ep2tp", "place"}
    w = t["weights_ep2tp"]
    assert w["launches"] == 4 and w["ms_per_launch"] == 0.25
    assert w["GB_s"] == 8000.0 and w["frac_of_peak"] == round(8000 / 7000, 4) and w["frac_of_mix_ceiling"] == 1.0
    kv = t["kv_ep2tp"]
    assert kv["GB_s"] == 6000.0 and kv["frac_of_mix_ceiling"] == 1.0
    assert "GB_s" not in t["place"] and t["place"]["ms_per_launch"] == 0.1
    assert "frac_of_mix_ceiling" not in bench.kernel_table(prof, b, 7000.0, {})["weights_ep2tp"]


def test_configs_cover_the_other_workloads():
    """The `configs` object times the expert-weight sizes, the 256-request KV
    workload and the attention weights: every workload but the full switch
    (the line's own value) and the tiny parity case."""
    from synth.workloads import ATTN_QWEN3_SHAPE, KV_256REQ, WEIGHTS_H2048, WEIGHTS_H4096
    assert [w for _, w in bench.OTHER_CONFIGS] == [WEIGHTS_H2048, WEIGHTS_H4096, KV_256REQ, ATTN_QWEN3_SHAPE]


@pytest.mark.parametrize("w", [Workload("bytes_attn", P=4, N=1, H=16, Hkv=2, D=8, Hq=8),
                               Workload("bytes_attn_wide", P=2, N=1, H=8, Hkv=4, D=4, Hq=6)],
                         ids=lambda w: w.name)
def test_attention_bytes_equal_elements_the_oracle_moves(w):
    """Attention weights (memory-saving variant): EP->TP writes every rank's
    shard once (read once each), TP->EP reads each shard element once (key and
    value heads from their lowest replica) and writes it into all P full
    copies; counted from the oracle's writes into zeroed slots."""
    d = dims_of(w)
    L = oracle.layout(d)
    b = bench.algorithmic_bytes(w, [])
    nfull = ((d.Hq + 2 * d.Hkv) * d.D * d.H + d.H * d.Hq * d.D) * 2        # one full copy, bytes
    buf = np.zeros(L["ws_off"], dtype=np.uint8)
    u = buf.view(np.uint16)
    for r in range(d.P):                                                     # EP layer 0 = slot 1, nonzero
        a = attnslot(L, r, 1) // 2
        u[a:a + L["attnslot_stride"] // 2] = 0x3f80
    oracle.attn_ep2tp(buf, d)
    written = sum(int(np.count_nonzero(u[attnslot(L, q, 0) // 2:(attnslot(L, q, 0) + L["attnslot_stride"]) // 2]))
                  for q in range(d.P))
    assert 2 * 2 * written == b["attn_ep2tp_per_layer"]                     # read + write, 2 B each
    for r in range(d.P):                                                     # TP -> EP into zeroed EP slots
        a = attnslot(L, r, 1) // 2
        u[a:a + L["attnslot_stride"] // 2] = 0
    oracle.attn_tp2ep(buf, d)
    written2 = sum(int(np.count_nonzero(u[attnslot(L, r, 1) // 2:(attnslot(L, r, 1) + L["attnslot_stride"]) // 2]))
                   for r in range(d.P))
    assert 2 * written2 == d.P * nfull
    assert b["attn_tp2ep_per_layer"] == nfull + 2 * written2
