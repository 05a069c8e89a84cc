"""The switch policy (host C++ in libumm) against the hand-worked trace, an
independent Python restatement, and the properties §4.5 states (no GPU)."""
from __future__ import annotations

import numpy as np
import pytest

from helpers import ints, read_golden
from oracle import policy as ref


@pytest.fixture(scope="module")
def umm():
    import ep_tp_weight_gb300 as m
    return m


def run_lib(umm, t_high, t_low, window, cooldown, start_mode, counts, times, fits):
    h = umm.umm_policy_create(t_high, t_low, window, cooldown, start_mode)
    out = [umm.umm_policy_step(h, n, t, ok) for n, t, ok in zip(counts, times, fits)]
    state = umm.umm_policy_state(h)
    umm.umm_policy_destroy(h)
    return out, state


@pytest.mark.parametrize("name", ["policy_trace.txt", "policy_boundaries.txt"])
def test_policy_golden_trace(umm, name):
    """Hand-worked traces: the §6.1 settings over a burst, and the edges of
    each rule (thresholds met exactly, a window not yet full, the last step
    of a cooldown)."""
    lines = read_golden(name)
    p = lines[0].split(":")[1].split()
    t_high, t_low, window, cool = float(p[0]), float(p[1]), int(p[2]), float(p[3])
    start = umm.UMM_MODE_TP if p[4] == "TP" else umm.UMM_MODE_EP
    f = lines[1].split(":")[1].split()
    final = (umm.UMM_MODE_TP if f[0] == "TP" else umm.UMM_MODE_EP, int(f[1]), int(f[2]))
    rows = [ints(ln) for ln in lines[2:]]
    times = [r[0] for r in rows]
    counts = [r[1] for r in rows]
    fits = [bool(r[2]) for r in rows]
    want = [r[3] for r in rows]
    got, state = run_lib(umm, t_high, t_low, window, cool, start, counts, times, fits)
    assert got == want
    assert state == final
    assert ref.run(t_high, t_low, window, cool, ref.TP if p[4] == "TP" else ref.EP, counts, times, fits) == want


def bursty(seed, n):
    """In-flight counts of a bursty arrival curve: quiet periods of a few
    requests, bursts of thousands (the shape of the bursty trace of §6.2)."""
    rng = np.random.default_rng(seed)
    level = np.where((np.arange(n) // 150) % 2 == 1, 1500, 40)
    noise = rng.normal(0, 0.2, n)
    return np.maximum(0, level * np.exp(noise)).astype(np.int64)


@pytest.mark.parametrize("seed", range(6))
def test_policy_matches_restatement_and_properties(umm, seed):
    rng = np.random.default_rng(seed)
    n = 2000
    counts = bursty(seed, n)
    times = np.cumsum(rng.uniform(0.02, 0.2, n))
    fits = rng.random(n) > 0.05
    for (t_high, t_low, window, cool) in ((256, 204.8, 8, 5.0), (256, 256, 1, 5.0), (256, 100, 16, 1.0)):
        start = umm.UMM_MODE_TP
        got, (mode, switches, cancels) = run_lib(umm, t_high, t_low, window, cool, start, counts, times, fits)
        assert got == ref.run(t_high, t_low, window, cool, ref.TP, counts, times, fits)
        got = np.array(got)
        acted = np.flatnonzero(got != umm.POLICY_STAY)
        # the cooldown bounds the decision rate
        assert (np.diff(times[acted]) >= cool - 1e-9).all()
        # switches alternate direction, starting TP -> EP
        sw = got[(got == umm.POLICY_TO_EP) | (got == umm.POLICY_TO_TP)]
        assert (sw[0::2] == umm.POLICY_TO_EP).all() and (sw[1::2] == umm.POLICY_TO_TP).all()
        assert switches == len(sw) and cancels == int((got == umm.POLICY_CANCELLED).sum())
        # every switch to EP saw a count above T_h; every switch to TP a window mean below T_l
        for i in np.flatnonzero(got == umm.POLICY_TO_EP):
            assert counts[i] > t_high and fits[i]
        for i in np.flatnonzero(got == umm.POLICY_TO_TP):
            assert counts[max(0, i - window + 1):i + 1].mean() < t_low and fits[i]
        assert switches >= 2          # the bursts do cross the boundary


def test_policy_hysteresis_holds_between_thresholds(umm):
    """Counts that stay between T_l and T_h never switch back to TP."""
    counts = [300] + [230] * 500
    times = list(range(len(counts)))
    got, (mode, switches, _) = run_lib(umm, 256, 204.8, 8, 5, umm.UMM_MODE_TP, counts, times, [True] * len(counts))
    assert got[0] == umm.POLICY_TO_EP and switches == 1 and mode == umm.UMM_MODE_EP


def test_policy_rejects_bad_params(umm):
    for args in ((256, 300, 8, 5), (256, 200, 0, 5), (256, 200, 8, -1)):
        with pytest.raises(umm.UmmError):
            umm.umm_policy_create(*args)
