"""Checks that the oracle's pins catch plausible mistakes in the oracle.

Each mutation below plants one mistake in the oracle (a dropped factor, a
transposed index, an off-by-one bound, a reversed order, a rule read the other
way), and the CPU suite (`pytest -m "not gpu" -x`) must then fail.  It runs on
a temporary copy of the repository, so the oracle here is never touched.
Usage: python tests/mutate_oracle.py [ID ...]; exit status 1 if any mutation
survives.  About 10 s per mutation (too slow for the default suite).

The mutations name what they break in the terms of "Moebius: Serving
Mixture-of-Expert Models with Seamless Runtime Parallelism Switch" (paper
review): §3.1 layouts and gate/up split, §3.2 head groups, page tables, list
order and greedy placement, §4.2 slots and layer order, §4.5 capacity check
and switch policy.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C = "oracle/umm_oracle.c"
POL = "oracle/policy.py"

# (id, what it breaks, file, exact text, replacement); each text occurs once
MUTATIONS = [
    ("M1", "KV EP->TP ignores the local head slot (Hkv >= 2P)", C,
     "int64_t to = kvslot_at(L, q, l, c) + (((dp * ps + s) * h_tp + hl) * D + e) * 2;",
     "int64_t to = kvslot_at(L, q, l, c) + (((dp * ps + s) * h_tp + 0) * D + e) * 2;"),
    ("M2", "KV TP->EP ignores the local head slot (Hkv >= 2P)", C,
     "int64_t from = kvslot_at(L, q, l, c) + (((sp * ps + s) * h_tp + hl) * D + e) * 2;",
     "int64_t from = kvslot_at(L, q, l, c) + (((sp * ps + s) * h_tp + 0) * D + e) * 2;"),
    ("M3", "EP page table read with row stride page_size instead of maxp", C,
     "int64_t sp = ep_pt[k * maxp + p], dp = tp_pt[k * maxp + p];",
     "int64_t sp = ep_pt[k * ps + p], dp = tp_pt[k * maxp + p];"),
    ("M4", "KV TP->EP swaps the source and destination page tables", C,
     "int64_t sp = tp_pt[k * maxp + p], dp = ep_pt[k * maxp + p];",
     "int64_t sp = ep_pt[k * maxp + p], dp = tp_pt[k * maxp + p];"),
    ("M5", "validation refuses a request that fills its page-table row", C,
     "if (lens[k] < 0 || (int64_t)lens[k] > maxp * ps || owner[k] < 0",
     "if (lens[k] < 0 || (int64_t)lens[k] >= maxp * ps || owner[k] < 0"),
    ("M6", "pages of a length rounded wrongly", C,
     "static int64_t npages_of(int64_t len, int64_t ps) { return (len + ps - 1) / ps; }",
     "static int64_t npages_of(int64_t len, int64_t ps) { return len / ps + 1; }"),
    ("M7", "EP pool capacity check off by one", C,
     "if (per_region[r] > pages_ep) flags |= ORC_F_CAPACITY;",
     "if (per_region[r] >= pages_ep) flags |= ORC_F_CAPACITY;"),
    ("M8", "placement breaks length ties by descending list position", C,
     "if (x->key != y->key) return x->key < y->key ? -1 : 1;",
     "if (x->key != y->key) return x->key > y->key ? -1 : 1;"),
    ("M9", "placement load counts requests instead of tokens", C,
     "load[best] += it[n].len;", "load[best] += 1;"),
    ("M10", "local position by request index instead of list position", C,
     "if (owner[m] == owner[k] && km < kk) ++cnt;", "if (owner[m] == owner[k] && m < k) ++cnt;"),
    ("M11", "all-gather list starts from the last rank", C,
     "if (owner[k] == r) tp_pos[k] = (int32_t)pos++;", "if (owner[k] == P - 1 - r) tp_pos[k] = (int32_t)pos++;"),
    ("M12", "pages handed out in descending key order", C,
     "if (gm == g && km < kk) s += npages_of(lens[m], ps);", "if (gm == g && km > kk) s += npages_of(lens[m], ps);"),
    ("M13", "page hand-out capacity off by one", C,
     "if (s + npages_of(lens[k], ps) > free_count)", "if (s + npages_of(lens[k], ps) >= free_count)"),
    ("M14", "descriptors claim full last pages", C,
     "o[6] = (int32_t)(lens[k] - p * ps < ps ? lens[k] - p * ps : ps);", "o[6] = (int32_t)ps;"),
    ("M15", "KV EP->TP walks layers descending (in place)", C,
     "    int64_t l = (order >= 0) ? t : N - 1 - t;\n#pragma omp parallel for num_threads(g_threads) "
     "schedule(dynamic, 1) if (g_threads > 1)\n    for (int64_t k = 0; k < R; ++k) {\n      int64_t o = owner[k];\n"
     "      for (int64_t tok = 0; tok < lens[k]; ++tok) {\n        int64_t p = tok / ps, s = tok % ps;\n"
     "        int64_t sp = ep_pt",
     "    int64_t l = (order >= 0) ? N - 1 - t : t;\n#pragma omp parallel for num_threads(g_threads) "
     "schedule(dynamic, 1) if (g_threads > 1)\n    for (int64_t k = 0; k < R; ++k) {\n      int64_t o = owner[k];\n"
     "      for (int64_t tok = 0; tok < lens[k]; ++tok) {\n        int64_t p = tok / ps, s = tok % ps;\n"
     "        int64_t sp = ep_pt"),
    ("M16", "heads dealt round-robin instead of in contiguous groups (Hkv >= P)", C,
     "if (h >= q * per && h < (q + 1) * per) { *local = h - q * per; return 1; }",
     "if (h % P == q) { *local = h / P; return 1; }"),
    ("M17", "no duplicate check of the TP pages a TP->EP switch reads", C,
     "if (tp_used[tp]) flags |= ORC_F_DUP_PAGE;", "if (0) flags |= ORC_F_DUP_PAGE;"),
    ("M18", "TP page id bound off by one", C,
     "if (ep < 0 || ep >= pages_ep || tp < 0 || tp >= pages_tp) {",
     "if (ep < 0 || ep >= pages_ep || tp < 0 || tp > pages_tp) {"),
    ("M19", "token row inside a page off by one (TP->EP)", C,
     "        int64_t p = tok / ps, s = tok % ps;\n        int64_t sp = tp_pt",
     "        int64_t p = tok / ps, s = (tok + 1) % ps;\n        int64_t sp = tp_pt"),
    ("M20", "contiguous-row W13 split forgets the factor 2", C,
     "  return q * 2 * Ip + row;\n}", "  return q * Ip + row;\n}"),
    ("M21", "TP W2 rows transposed (hidden-major)", C,
     "int64_t to = wslot_at(L, q, tp_slot) + L[OL_W2_OFF] + ((e * H + h) * Ip + c) * 2;\n          copy2",
     "int64_t to = wslot_at(L, q, tp_slot) + L[OL_W2_OFF] + ((h * E + e) * Ip + c) * 2;\n          copy2"),
    ("M22", "TP->EP contiguous split takes the rank by modulo", C,
     "          q = j / (2 * Ip);\n          row = j % (2 * Ip);", "          q = j % P;\n          row = j / P;"),
    ("M23", "EP pages per rank computed without h_tp", C,
     "L[OL_PAGES_EP] = (Hkv > 0) ? pages_tp * h_tp / Hkv : 0;", "L[OL_PAGES_EP] = (Hkv > 0) ? pages_tp / Hkv : 0;"),
    ("M24", "region stride rounded to 1 MiB instead of 2 MiB", C,
     "round_up((N + 1) * (wslot + kvslot + attnslot), (int64_t)2 << 20)",
     "round_up((N + 1) * (wslot + kvslot + attnslot), (int64_t)1 << 20)"),
    ("M25", "attention KV heads of rank q taken round-robin (Hkv < P)", C,
     "int64_t h = (Hkv >= P) ? q * h_tp + kv : q * Hkv / P;", "int64_t h = (Hkv >= P) ? q * h_tp + kv : q % Hkv;"),
    ("M26", "attention TP->EP query head gathered from the wrong rank", C,
     "          q = hh / hq;\n          b = hh % hq;", "          q = hh % P;\n          b = hh / P;"),
    ("M27", "attention EP->TP keeps rank 0's W_o columns on every rank", C,
     "(row * Hq * D + q * hq * D + c) * 2", "(row * Hq * D + c) * 2"),
    ("M28", "weights TP->EP walks layers ascending (in place)", C,
     "    int64_t l = (order < 0) ? N - 1 - t : t;\n    weights_layer_tp2ep",
     "    int64_t l = (order < 0) ? t : N - 1 - t;\n    weights_layer_tp2ep"),
    ("M29", "attention slots placed over the KV slots", C,
     "L[OL_ATTNSLOTS_OFF] = (N + 1) * (wslot + kvslot);", "L[OL_ATTNSLOTS_OFF] = (N + 1) * wslot;"),
    ("M30", "gate and up rows interleaved instead of in halves", C,
     "    int64_t g = row / Ip;          /* 0 = gate (W1), 1 = up (W3) */\n    int64_t ii = row % Ip;",
     "    int64_t g = row % 2;          /* 0 = gate (W1), 1 = up (W3) */\n    int64_t ii = row / 2;"),
    ("M31", "KV element map: EP offset ignores the head", C,
     "(((ep_page * ps + tok_in_page) * Hkv + h) * D + e) * 2",
     "(((ep_page * ps + tok_in_page) * Hkv + 0) * D + e) * 2"),
    ("M32", "KV element map: TP offset ignores the local head (Hkv >= 2P)", C,
     "(((tp_page * ps + tok_in_page) * L[OL_H_TP] + hl) * D + e) * 2",
     "(((tp_page * ps + tok_in_page) * L[OL_H_TP] + 0) * D + e) * 2"),
    ("M33", "W2 element map: EP column ignores the TP rank's block", C,
     "((el * H + h) * I + q * Ip + c) * 2",
     "((el * H + h) * I + c) * 2"),
    ("M34", "W13 element map: EP row taken as the TP row", C,
     "int64_t j = ep_row_of_tp_row(d[OD_W13_SPLIT], I, Ip, q, row);",
     "int64_t j = row;"),
    ("P1", "policy: a count equal to T_h already switches to EP", POL,
     "want = n > t_high", "want = n >= t_high"),
    ("P2", "policy: a window mean equal to T_l already switches to TP", POL,
     "sum(recent) / window < t_low", "sum(recent) / window <= t_low"),
    ("P3", "policy: the mean of a window not yet full decides", POL,
     "want = len(recent) == window and sum(recent) / window < t_low", "want = sum(recent) / len(recent) < t_low"),
    ("P4", "policy: the cooldown also covers its last second", POL,
     "if last is not None and t - last < cooldown:", "if last is not None and t - last <= cooldown:"),
    ("P5", "policy: a cancelled switch does not restart the cooldown", POL,
     "        last = t\n        if not ok:\n            out.append(CANCELLED)\n            continue",
     "        if not ok:\n            out.append(CANCELLED)\n            continue\n        last = t"),
    ("P6", "policy: counts seen during a cooldown are not remembered", POL,
     "        history.append(n)\n        if last is not None and t - last < cooldown:\n            out.append(STAY)\n"
     "            continue",
     "        if last is not None and t - last < cooldown:\n            out.append(STAY)\n            continue\n"
     "        history.append(n)"),
    ("P7", "policy: TP->EP decided on the window mean", POL,
     "want = n > t_high", "want = sum(history[-window:]) / len(history[-window:]) > t_high"),
]


def main(argv: list[str]) -> int:
    chosen = [m for m in MUTATIONS if not argv or m[0] in argv]
    ignore = shutil.ignore_patterns(".git", "_work", "gpurun_out", "_build", "__pycache__", "baseline", "*.ncu-rep")
    survived = []
    with tempfile.TemporaryDirectory(prefix="mutate_oracle") as tmp:
        copy = os.path.join(tmp, "repo")
        shutil.copytree(ROOT, copy, ignore=ignore)
        for mid, what, rel, old, new in chosen:
            path = os.path.join(copy, rel)
            with open(path) as f:
                orig = f.read()
            if orig.count(old) != 1:
                print(f"{mid}: text found {orig.count(old)} times; the mutation list is out of date")
                survived.append(mid)
                continue
            with open(path, "w") as f:
                f.write(orig.replace(old, new))
            try:
                if rel == C:
                    subprocess.run([sys.executable, "-c", "import oracle; oracle.build(force=True)"], cwd=copy,
                                   check=True, capture_output=True)
                r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-q", "-x", "-m", "not gpu"], cwd=copy,
                                   capture_output=True, text=True)
            finally:
                with open(path, "w") as f:
                    f.write(orig)
                if rel == C:
                    subprocess.run([sys.executable, "-c", "import oracle; oracle.build(force=True)"], cwd=copy,
                                   check=True, capture_output=True)
            failed = [ln.split("::", 1)[1].split(" ")[0] for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
            caught = r.returncode != 0 and failed
            print(f"{mid:4s} {'caught' if caught else 'SURVIVED'}  {what}" + (f"  <- {failed[0]}" if failed else ""),
                  flush=True)
            if not caught:
                survived.append(mid)
    print(f"{len(chosen) - len(survived)} of {len(chosen)} mutations caught")
    return 1 if survived else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
