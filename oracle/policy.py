"""Plain restatement of the switch policy (test infrastructure only).

"Moebius: Serving Mixture-of-Expert Models with Seamless Runtime Parallelism
Switch" (paper review), §4.5: the coordinator samples the global in-flight
request count once per decode iteration.  In TP it moves to EP as soon as the
latest count exceeds T_h; in EP it moves back to TP only when the mean of the
last W counts falls below T_l; a cooldown C follows every switch; a switch
whose target layout cannot hold the live requests is cancelled and retried
after the cooldown.
"""
from __future__ import annotations

STAY, TO_EP, TO_TP, CANCELLED = 0, 1, 2, 3
EP, TP = 0, 1


def run(t_high, t_low, window, cooldown, start_mode, counts, times, fits):
    """Decisions for a whole trace (lists of equal length)."""
    mode = start_mode
    history = []
    last = None                       # time of the last switch or cancellation
    out = []
    for n, t, ok in zip(counts, times, fits):
        history.append(n)
        if last is not None and t - last < cooldown:
            out.append(STAY)
            continue
        if mode == TP:
            want = n > t_high
        else:
            recent = history[-window:]
            want = len(recent) == window and sum(recent) / window < t_low
        if not want:
            out.append(STAY)
            continue
        last = t
        if not ok:
            out.append(CANCELLED)
            continue
        mode = EP if mode == TP else TP
        out.append(TO_EP if mode == EP else TO_TP)
    return out
