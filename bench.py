#!/usr/bin/env python3
"""Benchmark of the EP<->TP reshard data plane on one GB300 (or N replicas).

One step = one full switch round trip of the whole hot path on the
full-switch workload (expert weights P=8, E=128, H=2048, I=768 over 8 layers
+ paged KV of 2048 requests, lognormal lengths with median 2048 and sigma 1.0
capped at 32k, 4 KV heads of dim 128, page size 16, 8 layers):

  EP->TP: expert weights (8 launches, ascending), request list order,
          TP page hand-out, KV descriptors + gather/scatter (8 layers);
  TP->EP: greedy placement, EP page hand-out, expert weights (descending),
          KV descriptors + gather/scatter (descending).

Each step starts from the EP state the previous step left (new owners, new
pages).  The metric is reshard GB/s = algorithmic bytes read + written per
step (one read and one write of every moved element, plus the extra writes of
replicated KV heads) / device time.  Inputs (~260 GB) are far larger than L2,
so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl umm|reference]

Under torchrun each rank runs an independent replica on its own GPU (the
reshard does not shard across GPUs here); the value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth.workloads import ALL, ATTN_QWEN3_SHAPE, FULL_SWITCH, KV_256REQ, WEIGHTS_H2048, WEIGHTS_H4096  # noqa: E402

METRIC = "reshard GB/s (read+write) and % of HBM peak; ms per layer and per full switch"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="umm", choices=["umm", "reference"])
    ap.add_argument("--workload", default=FULL_SWITCH.name, choices=sorted(ALL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-staged", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="run the weight reshards of each switch on the handle's side stream "
                         "(umm_set_switch_overlap); per-kernel times then overlap")
    ap.add_argument("--phase-sweep", action="store_true",
                    help="instead of the benchmark line: the full-switch shape at several request counts, "
                         "one JSON line each with ms per phase (weights, request metadata, descriptor pass, KV)")
    ap.add_argument("--no-ceilings", action="store_true",
                    help="skip the read:write-mix ceilings measured after the timed region")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (expert weights of two sizes, KV of 256 requests, "
                         "attention weights) timed after the full switch for the `configs` object")
    ap.add_argument("--ceilings", action="store_true",
                    help="instead of the benchmark line: the HBM rate a plain streaming copy reaches for the "
                         "read:write mix of each reshard kernel, one JSON line per mix")
    args = ap.parse_args()
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps must be at least 1 and --warmup at least 0")
    return args


# ----------------------------------------------------------------------------- bytes model

def algorithmic_bytes(w, lens) -> dict:
    """Bytes the method must move (§4.3 Table 1: one read and one write per
    moved element; EP->TP KV writes each replicated head once per replica)."""
    out = {}
    if w.E:
        per_layer = 2 * w.P * (w.E // w.P) * 3 * w.I * w.H * 2      # read + write, W13 + W2
        out["weights_per_layer"] = per_layer
        out["weights_per_switch"] = per_layer * w.N
    if w.Hkv:
        T = int(np.asarray(lens, dtype=np.int64).sum())
        rd = T * w.Hkv * w.D * 2 * 2                                # K and V, 2 B
        wr = T * max(w.P, w.Hkv) * w.D * 2 * 2
        out["kv_ep2tp_per_layer"] = rd + wr
        out["kv_tp2ep_per_layer"] = 2 * rd
        out["tokens"] = T
    if w.Hq:
        hq, h_tp = w.Hq // w.P, w.h_tp
        shard = ((hq + 2 * h_tp) * w.D * w.H + w.H * hq * w.D) * 2          # one rank's TP shard, bytes
        full = ((w.Hq + 2 * w.Hkv) * w.D * w.H + w.H * w.Hq * w.D) * 2     # one full copy
        out["attn_ep2tp_per_layer"] = 2 * w.P * shard                       # every rank keeps its shard
        out["attn_tp2ep_per_layer"] = full + w.P * full                     # read each element once, write P copies
    step = 2 * out.get("weights_per_switch", 0) + w.N * (out.get("kv_ep2tp_per_layer", 0) +
                                                        out.get("kv_tp2ep_per_layer", 0) +
                                                        out.get("attn_ep2tp_per_layer", 0) +
                                                        out.get("attn_tp2ep_per_layer", 0))
    out["step"] = step
    return out


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.selector = None

    def _uuid(self):
        """The timed device's UUID as nvidia-smi names it ("GPU-..."): the
        index alone names another GPU when CUDA_VISIBLE_DEVICES remaps them."""
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.index).uuid)
        except Exception:
            return None
        return u if u.startswith("GPU-") else "GPU-" + u

    def _start(self, selector: str) -> bool:
        try:                                   # does nvidia-smi know this GPU?
            ok = subprocess.run(["nvidia-smi", "-i", selector, "--query-gpu=index", "--format=csv,noheader"],
                                capture_output=True, timeout=20).returncode == 0
        except subprocess.SubprocessError:
            ok = False
        if not ok:
            return False
        self.proc = subprocess.Popen(
            ["nvidia-smi", "-i", selector, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
             "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        time.sleep(0.3)
        self.selector = selector
        return True

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            uuid = self._uuid()
            if not (uuid and self._start(uuid)):
                self._start(str(self.index))
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if not self.proc or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(s):
            m = re.match(r"([\d.]+)", s)
            return float(m.group(1)) if m else None

        sm = [num(r[1]) for r in rows if num(r[1])]
        mx = max((num(r[2]) or 0) for r in rows)
        loaded = [x for x in sm if x >= 0.5 * mx] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows), "gpu": self.selector}


# ----------------------------------------------------------------------------- traffic from committed ncu summary

_CSRC = "ep_tp_weight_gb300/csrc/"
KERNEL_SOURCES = {"kv_copy_ep2tp": (_CSRC + "umm_kv.cu", _CSRC + "umm_scan.cuh", _CSRC + "umm_internal.cuh"),
                  "kv_copy_tp2ep": (_CSRC + "umm_kv.cu", _CSRC + "umm_scan.cuh", _CSRC + "umm_internal.cuh"),
                  "weights_kernel": (_CSRC + "umm_weights.cu", _CSRC + "umm_internal.cuh")}
# the ncu capture (small case of the same kernel) each traffic figure comes from
PROFILE_CASES = {"kv_copy_ep2tp": "kv_p8_2layers_8req_u1k-32k_hkv4_d128",
                 "kv_copy_tp2ep": "kv_p8_2layers_8req_u1k-32k_hkv4_d128",
                 "weights_kernel": "weights_p8_e128_h2048_i768_2layers"}


def source_digest(rels) -> str:
    """sha256 (16 hex) of the code of a kernel's source files (its .cu file and
    the headers it includes, in order): comments and whitespace are dropped,
    so edits to comments keep a profile valid and code edits do not."""
    if isinstance(rels, str):
        rels = (rels,)
    code = []
    for rel in rels:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code.append(re.sub(r"\s+", "", text))
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def committed_traffic(kernel: str, units: dict):
    """DRAM bytes per launch from the committed ncu summary of a small case of
    the same kernel, scaled by the units one launch of this workload moves
    (live tokens for KV, bytes for weights); None when the kernel source has
    changed since the capture."""
    case = PROFILE_CASES.get(kernel)
    path = os.path.join(ROOT, "profiles", f"{kernel}.{case}.md")
    if not case or not os.path.exists(path):
        return None
    txt = open(path).read()
    m_src = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m_src or m_src.group(1) != source_digest(KERNEL_SOURCES[kernel]):
        return None
    m_tok = re.search(r"dram_bytes_per_live_token:\s*([\d.]+)", txt)
    m_byte = re.search(r"dram_bytes_per_algorithmic_byte:\s*([\d.]+)", txt)
    if m_tok and units.get("tokens"):
        return int(float(m_tok.group(1)) * units["tokens"])
    if m_byte and units.get("bytes"):
        return int(float(m_byte.group(1)) * units["bytes"])
    return None


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (identity with one process); the
    step time every rank reports is the slowest rank's."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, ms_total_max: float, world: int) -> float:
    """Replicas: every rank moves the same bytes per step; the job's rate is
    all ranks' bytes over the slowest rank's time."""
    return world * bytes_per_step * steps / (ms_total_max / 1e3) / 1e9


# ----------------------------------------------------------------------------- the GPU run

def run_umm(args, rank, world, local_rank, w=None):
    import torch
    import ep_tp_weight_gb300 as umm
    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = w or ALL[args.workload]
    lens_h = w.lengths()
    R = len(lens_h)
    maxp = w.max_pages_per_req() if R else 1
    d = w.dims()
    dims = umm.make_dims(P=d["P"], E=d["E"], H=d["H"], I=d["I"], N=d["N"], Hkv=d["Hkv"], D=d["D"],
                         ps=d["ps"], pages_tp=d["pages_tp"], max_requests=d["max_requests"],
                         max_pages=d["max_pages"], Hq=d.get("Hq", 0))
    nbytes = umm.umm_required_bytes(dims)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)          # the one allocation (§4.2)
    h = umm.umm_create(dims, buf, nbytes)
    if getattr(args, "overlap", False):
        umm.umm_set_switch_overlap(h, True)
    L = umm.umm_layout(h)
    s = torch.cuda.Stream(device=dev)
    # initial contents: every element = synth value of its index
    tables = {}
    mode_w, sig_w = w.w_mode()
    plans = [(0, L["ws_off"] // 2, mode_w, sig_w)]
    if w.Hkv:
        mk, sk = w.kv_mode()
        for r in range(w.P):
            a = (r * L["region_stride"] + L["kvslots_off"]) // 2
            plans.append((a, (w.N + 1) * L["kvslot_stride"] // 2, mk, sk))
    for a, n, mode, sig in plans:
        if mode and sig not in tables:
            tables[sig] = torch.from_numpy(synth.normal_table(sig).view(np.int16).copy()).to(dev)
        synth.fill_device(buf.data_ptr() + 2 * a, n, w.seed, mode, tables[sig].data_ptr() if mode else 0,
                          base=a, stream=s.cuda_stream)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev)
    have_kv = w.Hkv > 0 and R > 0
    if have_kv:
        P = w.P
        lens = i32(lens_h)
        owner = torch.empty(R, dtype=torch.int32, device=dev)
        owner_n = torch.empty_like(owner)
        local = torch.empty_like(owner)
        tp_pos = torch.empty_like(owner)
        ep_pt = torch.empty((R, maxp), dtype=torch.int32, device=dev)
        ep_pt_n = torch.empty_like(ep_pt)
        tp_pt = torch.empty_like(ep_pt)
        tp_free = i32(synth.permutation(w.seed, 3, L["pages_tp"], rows=1))
        ep_free = i32(synth.permutation(w.seed, 2, L["pages_ep"], rows=P))
        # initial EP state: greedy owners, pages from each rank's free list
        umm.place_requests_tp2ep(h, R, lens, None, owner, local, s)
        umm.umm_assign_pages(h, P, R, lens, owner, None, ep_free, L["pages_ep"], L["pages_ep"], ep_pt, maxp, s)
    torch.cuda.synchronize()
    st = umm.umm_status_sync(h, s)
    if st[0] != 0:
        raise RuntimeError(f"setup failed: {umm.strerror(st[0])}")
    state = {"owner": owner, "owner_n": owner_n, "ep_pt": ep_pt, "ep_pt_n": ep_pt_n} if have_kv else {}

    ev_half = []

    def step(mark=False):
        """One round trip: umm_switch_ep2tp then umm_switch_tp2ep (weights,
        attention, request order, pages, KV; the state moves to the new EP
        owners and pages)."""
        e0 = torch.cuda.Event(enable_timing=True) if mark else None
        if mark:
            e0.record(s)
        if have_kv:
            umm.umm_switch_ep2tp(h, R, maxp, lens, state["owner"], state["ep_pt"], tp_free, L["pages_tp"], tp_pos,
                                 tp_pt, s)
        else:
            umm.umm_switch_ep2tp(h, 0, 1, None, None, None, None, 0, None, None, s)
        e1 = None
        if mark:
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(s)
        if have_kv:
            umm.umm_switch_tp2ep(h, R, maxp, lens, tp_pos, tp_pt, ep_free, L["pages_ep"], L["pages_ep"],
                                 state["owner_n"], local, state["ep_pt_n"], s)
            state["owner"], state["owner_n"] = state["owner_n"], state["owner"]
            state["ep_pt"], state["ep_pt_n"] = state["ep_pt_n"], state["ep_pt"]
        else:
            umm.umm_switch_tp2ep(h, 0, 1, None, None, None, None, 0, 0, None, None, None, s)
        if mark:
            e2 = torch.cuda.Event(enable_timing=True)
            e2.record(s)
            ev_half.append((e0, e1, e2))

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = umm.umm_status_sync(h, s)
    if st[0] != 0:
        raise RuntimeError(f"warm-up failed: {umm.strerror(st[0])}")
    bytes_model = algorithmic_bytes(w, lens_h)

    # ---------------- timed region (device time, CUDA events on the launching stream)
    umm.umm_profile_enable(h, True)
    umm.umm_profile_reset(h)
    n_launch0 = umm.umm_launch_count(h)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s)
        for _ in range(args.steps):
            step(mark=True)
        t1.record(s)
        torch.cuda.synchronize()
    barrier()
    ms_total = t0.elapsed_time(t1)
    launches = umm.umm_launch_count(h) - n_launch0
    prof = {umm.KIND_NAMES[k]: umm.umm_profile_read(h, k) for k in range(umm.K_COUNT)}
    umm.umm_profile_enable(h, False)
    st = umm.umm_status_sync(h, s)
    if st[0] != 0:
        raise RuntimeError(f"timed steps failed: {umm.strerror(st[0])}")
    ms_ep2tp = statistics.mean(a.elapsed_time(b) for a, b, _ in ev_half)
    ms_tp2ep = statistics.mean(b.elapsed_time(c) for _, b, c in ev_half)
    step_ms = [a.elapsed_time(c) for a, _, c in ev_half]
    ms_total = max_over_ranks(ms_total, dev)

    # ---------------- the same round trip replayed from a CUDA graph
    # Two steps are captured (EP state A -> B -> A), so each replay starts from
    # the state the previous one left; the host-side modes end where they began.
    graph = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                step()
                step()
        torch.cuda.synchronize()
        g.replay()                                   # warm-up replay
        torch.cuda.synchronize()
        reps = max(1, args.steps // 2)
        barrier()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(s)
        with torch.cuda.stream(s):
            for _ in range(reps):
                g.replay()
        g1.record(s)
        torch.cuda.synchronize()
        ms_g = max_over_ranks(g0.elapsed_time(g1), dev) / (2 * reps)
        code, _ = umm.umm_status_sync(h, s)
        if code:
            raise RuntimeError(f"graph replay failed: {umm.strerror(code)}")
        graph = {"ms_per_step": round(ms_g, 3), "value": round(whole_job_gbs(bytes_model["step"], 1, ms_g, world), 1),
                 "unit": UNIT, "steps": 2 * reps}
        del g

    # ---------------- the staged (collective-style) path, same steps, for comparison
    staged = None
    if not args.no_staged and (w.E or have_kv):
        wsb = umm.umm_weights_stage_bytes(h) if w.E else 0
        ksb = umm.umm_kv_stage_bytes(h) if have_kv else 0
        wsb_al = (wsb + 255) // 256 * 256
        stage_buf = torch.empty(wsb_al + ksb, dtype=torch.uint8, device=dev)
        w_stage, k_stage = stage_buf.data_ptr(), stage_buf.data_ptr() + wsb_al

        def step_staged():
            if w.E:
                umm.reshard_weights_ep2tp_staged(h, w_stage, wsb, s)
            if have_kv:
                umm.gather_requests_ep2tp(h, R, state["owner"], tp_pos, s)
                umm.umm_assign_pages(h, 1, R, lens, None, tp_pos, tp_free, L["pages_tp"], L["pages_tp"], tp_pt,
                                     maxp, s)
                umm.reshard_kv_ep2tp_staged(h, k_stage, ksb, R, maxp, lens, state["owner"], state["ep_pt"], tp_pt, s)
                umm.place_requests_tp2ep(h, R, lens, tp_pos, state["owner_n"], local, s)
                umm.umm_assign_pages(h, P, R, lens, state["owner_n"], tp_pos, ep_free, L["pages_ep"],
                                     L["pages_ep"], state["ep_pt_n"], maxp, s)
            if w.E:
                umm.reshard_weights_tp2ep_staged(h, w_stage, wsb, s)
            if have_kv:
                umm.reshard_kv_tp2ep_staged(h, k_stage, ksb, R, maxp, lens, state["owner_n"], state["ep_pt_n"],
                                            tp_pt, s)
                state["owner"], state["owner_n"] = state["owner_n"], state["owner"]
                state["ep_pt"], state["ep_pt_n"] = state["ep_pt_n"], state["ep_pt"]

        step_staged()                                   # warm-up
        torch.cuda.synchronize()
        umm.umm_profile_enable(h, True)
        umm.umm_profile_reset(h)
        reps = max(2, args.steps // 2)
        barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(s)
        for _ in range(reps):
            step_staged()
        s1.record(s)
        torch.cuda.synchronize()
        ms_s = max_over_ranks(s0.elapsed_time(s1), dev) / reps
        sprof = {umm.KIND_NAMES[k]: umm.umm_profile_read(h, k) for k in range(umm.K_COUNT)}
        umm.umm_profile_enable(h, False)
        code, _ = umm.umm_status_sync(h, s)
        if code:
            raise RuntimeError(f"staged steps failed: {umm.strerror(code)}")
        staged = {"ms_per_step": round(ms_s, 3),
                  "value": round(whole_job_gbs(bytes_model["step"], 1, ms_s, world), 1), "unit": UNIT,
                  "steps": reps, "stage_bytes": int(wsb_al + ksb)}
        if w.E and sprof["weights_ep2tp"][0]:
            staged["weights_ms_per_layer"] = round(
                (sprof["weights_ep2tp"][1] + sprof["weights_tp2ep"][1]) /
                (sprof["weights_ep2tp"][0] + sprof["weights_tp2ep"][0]), 4)
        if have_kv and sprof["kv_ep2tp"][0]:
            staged["kv_ep2tp_ms_per_switch"] = round(sprof["kv_ep2tp"][1] / reps, 3)
            staged["kv_tp2ep_ms_per_switch"] = round(sprof["kv_tp2ep"][1] / reps, 3)
        del stage_buf
        torch.cuda.empty_cache()

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and have_kv:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        h_lens = pin(lens_h.astype(np.int32))
        h_owner = pin(state["owner"].cpu().numpy())
        h_ep_pt = pin(state["ep_pt"].cpu().numpy())
        h_tp_free = pin(tp_free.cpu().numpy())
        h_ep_free = pin(ep_free.cpu().numpy())
        o_local = torch.empty(R, dtype=torch.int32).pin_memory()
        h2d = sum(x.numel() * 4 for x in (h_lens, h_owner, h_ep_pt, h_tp_free, h_ep_free))
        d2h = sum(x.numel() * 4 for x in (h_owner, o_local, h_ep_pt)) + 8   # + status word read
        barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for _ in range(args.steps):
            with torch.cuda.stream(s):
                lens.copy_(h_lens, non_blocking=True)
                state["owner"].copy_(h_owner, non_blocking=True)
                state["ep_pt"].copy_(h_ep_pt, non_blocking=True)
                tp_free.copy_(h_tp_free, non_blocking=True)
                ep_free.copy_(h_ep_free, non_blocking=True)
            step()
            with torch.cuda.stream(s):
                # the new EP owners and their pages come back into the host
                # arrays the next step sends (its EP state); local positions too
                h_owner.copy_(state["owner"], non_blocking=True)
                o_local.copy_(local, non_blocking=True)
                h_ep_pt.copy_(state["ep_pt"], non_blocking=True)
            code, _ = umm.umm_status_sync(h, s)                   # syncs the stream, reads status
            if code:
                raise RuntimeError(f"e2e step failed: {umm.strerror(code)}")
        wall = time.perf_counter() - wall0
        e2e_gbs = world * bytes_model["step"] * args.steps / wall / 1e9
        e2e = {"value": round(e2e_gbs, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": round(1e3 * wall / args.steps, 3)}

    umm.umm_destroy(h)
    del buf
    torch.cuda.empty_cache()
    return dict(w=w, lens=lens_h, ms_total=ms_total, graph=graph, staged=staged, launches=launches, prof=prof, clocks=clk.summary(),
                ms_ep2tp=ms_ep2tp, ms_tp2ep=ms_tp2ep, bytes=bytes_model, e2e=e2e, layout=L, nbytes=nbytes,
                step_ms=step_ms)


# ----------------------------------------------------------------------------- CPU oracle sample

class CpuSample:
    """The oracle, as it stands, on a bounded sample of the workload: the
    expert weights of every layer EP->TP->EP, and the KV cache of all requests
    (at most 2048) for one layer EP->TP->EP, four times (greedy placement,
    fresh pages each time).  Buffer contents do not change the oracle's speed,
    so they are left as allocated (touched once before timing)."""

    KV_REQUESTS = 2048
    KV_ROUNDS = 4

    def __init__(self, w, threads: int, kv_requests: int | None = None, kv_rounds: int | None = None,
                 weight_layers: int | None = None):
        import oracle
        self.oracle = oracle
        self.w = w
        oracle.set_threads(threads)
        self.threads = threads
        self.KV_REQUESTS = kv_requests or self.KV_REQUESTS
        self.KV_ROUNDS = kv_rounds or self.KV_ROUNDS
        self.weight_layers = min(weight_layers or w.N, w.N)
        self.wbuf = None
        self.kbuf = None
        self.abuf = None
        if w.Hq:
            aw = w.with_(E=0, R=0)
            self.ad = oracle.Dims(**aw.dims())
            self.abuf = np.ones(oracle.layout(self.ad)["ws_off"], dtype=np.uint8)
            b = algorithmic_bytes(aw, [])
            self.abytes = w.N * (b["attn_ep2tp_per_layer"] + b["attn_tp2ep_per_layer"])
        if w.E:
            ws = w.with_(Hkv=0, R=0, N=self.weight_layers)
            self.wd = oracle.Dims(**ws.dims())
            L = oracle.layout(self.wd)
            self.wbuf = np.ones(L["ws_off"], dtype=np.uint8)
            self.wbytes = 2 * algorithmic_bytes(ws, [])["weights_per_switch"]
        if w.Hkv and w.R:
            Rs = min(self.KV_REQUESTS, w.R)
            self.lens = w.lengths()[:Rs]
            used = int(synth.npages(self.lens, w.ps).sum())
            m = w.Hkv // w.h_tp
            ptp = (math.ceil(1.02 * used) + m - 1) // m * m
            kv = w.with_(E=0, R=Rs, N=1)
            self.kd = oracle.Dims(**dict(kv.dims(), pages_tp=ptp, max_requests=Rs, max_pages=ptp))
            self.kL = oracle.layout(self.kd)
            self.kbuf = np.ones(self.kL["ws_off"], dtype=np.uint8)
            self.maxp = w.max_pages_per_req()
            self.owner, _, _ = oracle.place(w.P, self.lens)
            _, self.ep_pt = oracle.assign_pages(w.P, self.lens, w.ps, self.maxp,
                                                synth.permutation(w.seed, 2, self.kL["pages_ep"], w.P),
                                                region=self.owner)
            b = algorithmic_bytes(kv, self.lens)
            self.kbytes = b["kv_ep2tp_per_layer"] + b["kv_tp2ep_per_layer"]
        self.n_runs = 0

    def describe(self) -> str:
        parts = []
        if self.abuf is not None:
            parts.append(f"attention weights of all {self.w.N} layers EP->TP->EP")
        if self.wbuf is not None:
            parts.append(f"expert weights of {self.weight_layers} of {self.w.N} layers EP->TP->EP")
        if self.kbuf is not None:
            parts.append(f"KV of {min(self.KV_REQUESTS, self.w.R)} of {self.w.R} requests for 1 layer "
                         f"EP->TP->EP, {self.KV_ROUNDS} times")
        return f"plain C oracle (element by element, OpenMP, {self.threads} threads): " + " + ".join(parts)

    def run(self):
        """One sample; returns (algorithmic bytes, seconds of oracle work)."""
        o, w = self.oracle, self.w
        moved, secs = 0, 0.0
        if self.abuf is not None:
            t = time.perf_counter()
            o.attn_ep2tp(self.abuf, self.ad)
            o.attn_tp2ep(self.abuf, self.ad)
            secs += time.perf_counter() - t
            moved += self.abytes
        if self.wbuf is not None:
            t = time.perf_counter()
            o.weights_ep2tp(self.wbuf, self.wd)
            o.weights_tp2ep(self.wbuf, self.wd)
            secs += time.perf_counter() - t
            moved += self.wbytes
        for _ in range(self.KV_ROUNDS if self.kbuf is not None else 0):
            L = self.kL
            self.n_runs += 1
            pos = o.request_order(w.P, self.owner)
            _, tp_pt = o.assign_pages(1, self.lens, w.ps, self.maxp,
                                      synth.permutation(w.seed + self.n_runs, 3, L["pages_tp"]), key=pos)
            owner2, _, _ = o.place(w.P, self.lens, key=pos)
            _, ep_pt2 = o.assign_pages(w.P, self.lens, w.ps, self.maxp,
                                       synth.permutation(w.seed + self.n_runs, 4, L["pages_ep"], w.P),
                                       region=owner2, key=pos)
            t = time.perf_counter()
            assert o.kv_ep2tp(self.kbuf, self.kd, self.lens, self.owner, self.ep_pt, tp_pt) == 0
            assert o.kv_tp2ep(self.kbuf, self.kd, self.lens, owner2, ep_pt2, tp_pt) == 0
            secs += time.perf_counter() - t
            moved += self.kbytes
            self.owner, self.ep_pt = owner2, ep_pt2
        return moved, secs


LAYER_BYTES = (("weights_ep2tp", "weights_per_layer"), ("weights_tp2ep", "weights_per_layer"),
               ("kv_ep2tp", "kv_ep2tp_per_layer"), ("kv_tp2ep", "kv_tp2ep_per_layer"),
               ("attn_ep2tp", "attn_ep2tp_per_layer"), ("attn_tp2ep", "attn_tp2ep_per_layer"))


def kernel_table(prof: dict, b: dict, peak: float, ceil: dict) -> dict:
    """Per kernel kind timed: launches (layer copies or calls), ms per launch,
    and for the copies GB/s of algorithmic bytes, its fraction of the measured
    copy peak and of the plain-copy ceiling of the kernel's read:write mix."""
    per_kind = {k: {"launches": n, "ms_per_launch": round(ms / n, 4) if n else None}
                for k, (n, ms) in prof.items() if n}
    for k, key in LAYER_BYTES:
        if k in per_kind and b.get(key):
            gbs = b[key] / (per_kind[k]["ms_per_launch"] / 1e3) / 1e9
            per_kind[k]["GB_s"] = round(gbs, 1)
            per_kind[k]["frac_of_peak"] = round(gbs / peak, 4)
            if MIX_OF_KIND.get(k) in ceil:
                per_kind[k]["mix_ceiling_GB_s"] = ceil[MIX_OF_KIND[k]]
                per_kind[k]["frac_of_mix_ceiling"] = round(gbs / ceil[MIX_OF_KIND[k]], 4)
    return per_kind


# the workloads timed after the full switch, for the `configs` object
OTHER_CONFIGS = (("weights_e128_h2048_i768", WEIGHTS_H2048), ("weights_e128_h4096_i1536", WEIGHTS_H4096),
                 ("kv_256req_u1k-32k", KV_256REQ), ("attention_hq64_hkv4_h4096", ATTN_QWEN3_SHAPE))


def other_configs(args, peak: float, ceil: dict) -> dict:
    """The other workloads on the same GPU, one after the other (each its own
    buffer), EP->TP->EP round trips timed exactly as the full switch: the
    same calls, per-kernel events around each call's chain of layer copies."""
    import copy
    sub = copy.copy(args)
    sub.no_graph = sub.no_staged = sub.no_e2e = True
    sub.overlap = False
    out = {}
    for label, w in OTHER_CONFIGS:
        r = run_umm(sub, 0, 1, int(os.environ.get("LOCAL_RANK", 0)), w=w)
        b = r["bytes"]
        n = args.steps
        ms_rt = r["ms_total"] / n
        gbs = b["step"] / (ms_rt / 1e3) / 1e9
        kern = kernel_table(r["prof"], b, peak, ceil)
        out[label] = {
            "workload": w.name, "layers": w.N, "steps": n, "warmup": args.warmup,
            "bytes_per_round_trip": b["step"], "ms_per_round_trip": round(ms_rt, 3),
            "ms_per_switch": {"ep2tp": round(r["ms_ep2tp"], 3), "tp2ep": round(r["ms_tp2ep"], 3)},
            "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "frac_of_8TBs_nominal": round(gbs / 8000.0, 4),
            "ms_per_layer": {k: v["ms_per_launch"] for k, v in kern.items() if "GB_s" in v},
            "kernels": {k: v for k, v in kern.items() if "GB_s" in v},
            "tokens": b.get("tokens"), "clocks": r["clocks"]}
    return out


def cpu_baseline(w):
    """The oracle on all host cores, plus a smaller sample on one core."""
    threads = os.cpu_count() or 1
    cs = CpuSample(w, threads)
    moved, secs = cs.run()
    one = CpuSample(w, 1, kv_requests=256, kv_rounds=1, weight_layers=1)
    m1, s1 = one.run()
    cs.oracle.set_threads(threads)
    return {"value": round(moved / secs / 1e9, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": cs.describe() + f"; {moved / 1e9:.1f} GB algorithmic in {secs:.2f} s",
            "one_core": {"value": round(m1 / s1 / 1e9, 3), "unit": UNIT, "cores": 1,
                         "sample": one.describe() + f"; {m1 / 1e9:.1f} GB algorithmic in {s1:.2f} s"}}


# ----------------------------------------------------------------------------- main

def phase_sweep(args):
    """The full-switch shape (weights + KV) at growing request counts, as the
    page's switch-cost breakdown by phase: the weights are a fixed floor, the
    KV grows with occupancy, the request metadata stays nearly flat."""
    args.no_graph = args.no_staged = args.no_e2e = True
    for R in (16, 128, 512, 1024, 2048):
        w = FULL_SWITCH.with_(name=f"{FULL_SWITCH.name}_{R}req", R=R)
        # a TP pool large enough that each rank's EP pool (pages_tp * h_tp / Hkv)
        # holds its share under the greedy rule: at most the mean plus the
        # longest request, plus one partial page per request
        pages = synth.npages(w.lengths(), w.ps)
        used, m = int(pages.sum()), w.Hkv // w.h_tp
        bound = used / w.P + int(pages.max()) + R / w.P + 1
        w = w.with_(slack=max(FULL_SWITCH.slack, 1.02 * m * bound / used))
        r = run_umm(args, 0, 1, 0, w=w)
        prof, n = r["prof"], args.steps

        def ms(*kinds):
            return round(sum(prof[k][1] for k in kinds) / n, 3)

        line = {"phase_sweep": True, "workload": w.name, "requests": R, "tokens": int(r["lens"].sum()),
                "switch_overlap": bool(args.overlap),
                "ms_per_round_trip": round(r["ms_total"] / n, 3),
                "ms_per_switch": {"ep2tp": round(r["ms_ep2tp"], 3), "tp2ep": round(r["ms_tp2ep"], 3)},
                "phases_ms_per_round_trip": {"weights": ms("weights_ep2tp", "weights_tp2ep"),
                                             "request_metadata": ms("order", "place", "assign"),
                                             "descriptor_pass": ms("kv_prep"),
                                             "kv": ms("kv_ep2tp", "kv_tp2ep")},
                "clocks": r["clocks"]}
        print(json.dumps(line), flush=True)


# the read:write mix of each kernel kind (ep_tp_weight_gb300/csrc/ceiling)
MIX_OF_KIND = {"weights_ep2tp": "1R1W sequential", "weights_tp2ep": "1R1W sequential",
               "kv_ep2tp": "1R2W shuffled reads", "kv_tp2ep": "1R1W shuffled writes",
               "attn_ep2tp": "1R1W sequential", "attn_tp2ep": "1R8W sequential"}


def run_ceilings(timeout_s: float = 180.0) -> list[dict]:
    """Runs the read:write-mix ceiling program (a plain streaming copy for
    each reshard kernel's access pattern, 8 GiB buffers) on this process's
    GPU; its JSON lines, or [] when it cannot be built or run here."""
    try:
        from ep_tp_weight_gb300 import build as umm_build
        exe = umm_build.build_ceiling()
        env = dict(os.environ)
        env.setdefault("CUDA_VISIBLE_DEVICES", os.environ.get("LOCAL_RANK", "0"))
        out = subprocess.run([exe, "8"], capture_output=True, text=True, timeout=timeout_s, check=True,
                             env=env).stdout
    except (OSError, subprocess.SubprocessError):
        return []
    return [json.loads(ln) for ln in out.splitlines() if ln.startswith("{")]


def ceilings():
    """`--ceilings`: the read:write-mix ceilings on this GPU, one JSON line
    each, then the clocks seen while they ran."""
    with ClockSampler(int(os.environ.get("LOCAL_RANK", 0))) as clk:
        rows = run_ceilings(timeout_s=600.0)
    if not rows:
        raise RuntimeError("the ceiling program could not be built or run")
    for row in rows:
        print(json.dumps(row), flush=True)
    print(json.dumps({"ceilings_clocks": clk.summary()}), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    w = ALL[args.workload]
    config = {"workload": w.name, "P": w.P, "layers": w.N, "experts": w.E, "hidden": w.H, "attn_q_heads": w.Hq,
              "intermediate": w.I, "requests": w.R, "kv_heads": w.Hkv, "head_dim": w.D, "page_size": w.ps,
              "l2": "inputs larger than L2 (no flush needed)", "parallelism": f"replicas{world}"}
    if args.overlap:
        config["switch_overlap"] = True

    if args.impl == "reference":
        if rank != 0:
            return
        threads = os.cpu_count() or 1
        cs = CpuSample(w, threads)
        for _ in range(args.warmup):
            cs.run()
        tot_b, tot_s = 0, 0.0
        for _ in range(args.steps):
            b, s = cs.run()
            tot_b += b
            tot_s += s
        val = tot_b / tot_s / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": UNIT, "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_s / args.steps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u16",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(val, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
                                 "sample": "each step: " + cs.describe()},
                "e2e": {"value": round(val, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if args.phase_sweep:
        if rank == 0:
            phase_sweep(args)
        return
    if args.ceilings:
        if rank == 0:
            ceilings()
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_umm(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return
    b = r["bytes"]
    ms_step = r["ms_total"] / args.steps
    value = whole_job_gbs(b["step"], args.steps, r["ms_total"], world)
    peak, peak_kind = peaks()
    # dominant kernel = most device time in the timed region
    prof = r["prof"]
    dom = max(prof, key=lambda k: prof[k][1])
    n_dom, ms_dom = prof[dom]
    per_launch_bytes = {"kv_ep2tp": b.get("kv_ep2tp_per_layer", 0), "kv_tp2ep": b.get("kv_tp2ep_per_layer", 0),
                        "weights_ep2tp": b.get("weights_per_layer", 0),
                        "weights_tp2ep": b.get("weights_per_layer", 0),
                        "attn_ep2tp": b.get("attn_ep2tp_per_layer", 0),
                        "attn_tp2ep": b.get("attn_tp2ep_per_layer", 0)}.get(dom, 0)
    achieved = per_launch_bytes / (ms_dom / n_dom / 1e3) / 1e9 if n_dom else 0.0
    kernel_name = {"kv_ep2tp": "kv_copy_ep2tp", "kv_tp2ep": "kv_copy_tp2ep", "weights_ep2tp": "weights_kernel",
                   "weights_tp2ep": "weights_kernel"}.get(dom)
    traffic = committed_traffic(kernel_name, {"tokens": b.get("tokens"), "bytes": per_launch_bytes}) \
        if kernel_name else None
    # the same kernels against a plain streaming copy of their own read:write
    # mix, measured on this GPU after the timed region (context beside peak)
    ceil = {} if args.no_ceilings else {row["ceiling"]: row["GB_s"] for row in run_ceilings()}
    per_kind = kernel_table(prof, b, peak, ceil)
    mix = None
    if ceil:
        if MIX_OF_KIND.get(dom) in ceil:
            c = ceil[MIX_OF_KIND[dom]]
            mix = {"mix": MIX_OF_KIND[dom], "GB_s": c, "frac": round(achieved / c, 4),
                   "source": "bench.py --ceilings program, same GPU, after the timed region"}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u16", "data": "synthetic (seeded; bf16 N(0,0.02) weights, N(0,1) KV)",
        "config": config,
        "ms_per_switch": {"ep2tp": round(r["ms_ep2tp"], 3), "tp2ep": round(r["ms_tp2ep"], 3)},
        "ms_per_step_spread": {"min": round(min(r["step_ms"]), 3), "median": round(statistics.median(r["step_ms"]), 3),
                               "max": round(max(r["step_ms"]), 3),
                               "source": "events around each timed step, on the launching stream"},
        "ms_per_layer": {k: per_kind[k]["ms_per_launch"] for k in ("weights_ep2tp", "weights_tp2ep", "kv_ep2tp",
                                                                   "kv_tp2ep", "attn_ep2tp", "attn_tp2ep")
                         if k in per_kind},
        "frac_of_hbm_peak": round(value / world / peak, 4),
        "frac_of_8TBs_nominal": round(value / world / 8000.0, 4),
        "bytes_per_step": b["step"], "tokens": b.get("tokens"),
        "kernels": per_kind,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} copy GB/s (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": per_launch_bytes,
                     "mix_ceiling": mix},
        "cuda_graph": r["graph"],
        "staged_comparison": None if r["staged"] is None else dict(
            r["staged"], fused_speedup=round(r["staged"]["ms_per_step"] / ms_step, 3)),
        "clocks": r["clocks"], "gpu_launches": r["launches"],
        "e2e": r["e2e"],
    }
    if not args.no_configs and world == 1 and args.workload == FULL_SWITCH.name:
        line["configs"] = other_configs(args, peak, ceil)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(r["w"])
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
