"""Oracle: per-stage F/B/W orders and a unit-time simulator of all p stages.

TEST INFRASTRUCTURE (see the package docstring).  Pure Python, small inputs.

Model ("Zero-Bubble Pipeline Parallelism Guide for LLMs", section
"Mathematical Modeling: Bubble Fractions, Memory Bounds, and Speedups"):
every op takes one time unit (t_F = t_B = t_W), communication is free.
Dependencies, for stage s and microbatch i:
  F(s, i) after F(s-1, i)                       (activations flow down)
  B(s, i) after F(s, i) and after the backward of stage s+1 for i
  W(s, i) after B(s, i)                         (section "Core Innovation 1")
plus each stage's own program order.  When the backward is not split
(GPipe, 1F1B), stage s+1 sends its input gradient only once its whole
backward, B and W, is done, so B(s, i) then waits for W(s+1, i).

Orders:
* GPipe (section "1. The GPipe Bubble"): all m forwards, then all backwards.
* 1F1B (section "2. The 1F1B (One-Forward-One-Backward) Schedule" and the
  first diagram of "The Mechanics of Pipeline Bubbles"): stage s runs p-s
  forwards before its first backward, then alternates B and F, then drains
  the remaining B.  W is written right after its B.
* ZB-H1, the guide's ZB-1F1B (section "Core Innovation 2": same memory as
  1F1B, F and B prioritised, a W fills every slot that would otherwise be
  idle, steady F -> B -> W rhythm, the W left over are drained at the end;
  section "Memory Management & Activation Rollback": a hard ceiling on
  in-flight microbatches, and at the ceiling a W must run before the next F).
  Reading: the stage keeps the 1F1B order of its F and B; whenever it is free
  it runs that next F/B if its inputs are there, except that an F that would
  pass the ceiling (F issued minus W issued = ``limit``, default p) yields to
  the oldest pending W; when the next F/B is not ready it runs the oldest
  pending W; otherwise it idles.  The listing's fourth rule (an F past the
  ceiling) contradicts that hard ceiling and is not used.  The listing's
  first three rules alone do not give the section's own (p-1)/(3m) bubble
  (at p=4, m=8 they take 29 units where this reading takes 3m+p-1 = 27).
* ZB-2p (section "Core Innovation 2", item 2: the in-flight limit doubles to
  2p, the warm-up and cool-down bubbles vanish and every GPU computes without
  idle waiting).  Reading: the same policy with a ceiling of 2p and 2(p-s)-1
  forwards before the first B of stage s.  In the unit-time model every
  stage is then busy from its first op to its last (``window_idle`` = 0,
  for m >= 2p - 1) while holding up to 2p microbatches; over the common
  makespan nothing changes, since 3m + p - 1 is already the shortest
  possible when communication is free.
* Memory-limited orders ("Zero Bubble Pipeline Parallelism", the abstract: an
  algorithm that finds the best schedule for a given model configuration and
  memory limit; the guide's section "Core Innovation 2": ZB-H1 holds p
  microbatches, ZB-2p holds 2p).  Reading: the same policy with a ceiling L
  in [p, 2p] and min(L - s, 2(p - s) - 1) forwards before the first B of
  stage s (p - s at L = p, ZB-2p's count at L = 2p), run with measured integer
  durations t_F, t_B, t_W instead of unit times; the search takes the L no
  larger than the memory limit with the shortest makespan (the smallest such
  L on ties).
"""
from __future__ import annotations

F, B, W = "F", "B", "W"


def order_gpipe(s, p, m):
    """All forwards, then each backward as B followed by its W."""
    out = [(F, i) for i in range(m)]
    for i in range(m):
        out += [(B, i), (W, i)]
    return out


def order_1f1b(s, p, m):
    """1F1B for stage s: p-s forwards before the first B, then B/F alternate."""
    warm = min(p - s - 1, m)
    out = [(F, i) for i in range(warm)]
    for j in range(m - warm):
        out += [(F, warm + j), (B, j), (W, j)]
    for i in range(m - warm, m):
        out += [(B, i), (W, i)]
    return out


def _deps(kind, s, i, p, split):
    """Ops (kind, stage, mb) that must finish before (kind, s, i) may start."""
    if kind == F:
        return [(F, s - 1, i)] if s > 0 else []
    if kind == B:
        d = [(F, s, i)]
        if s < p - 1:
            d.append((B if split else W, s + 1, i))
        return d
    return [(B, s, i)]


def simulate_orders(orders, p, split):
    """Run fixed per-stage orders as early as the dependencies allow.

    Returns a dict (kind, stage, mb) -> start time.  Raises if the orders
    deadlock.
    """
    start = {}
    finish = {}
    ptr = [0] * p
    free_at = [0] * p
    total = sum(len(o) for o in orders)
    while len(start) < total:
        progressed = False
        for s in range(p):
            while ptr[s] < len(orders[s]):
                kind, i = orders[s][ptr[s]]
                deps = _deps(kind, s, i, p, split)
                if any(d not in finish for d in deps):
                    break
                t0 = max([free_at[s]] + [finish[d] for d in deps])
                start[(kind, s, i)] = t0
                finish[(kind, s, i)] = t0 + 1
                free_at[s] = t0 + 1
                ptr[s] += 1
                progressed = True
        if not progressed:
            raise RuntimeError("orders deadlock")
    return start


def fb_order(s, p, m, warm):
    """F/B order of stage s: `warm` forwards, then B and F alternate, then the last B."""
    warm = min(warm, m)
    out = [(F, i) for i in range(warm)]
    for j in range(m - warm):
        out += [(B, j), (F, warm + j)]
    out += [(B, i) for i in range(m - warm, m)]
    return out


def simulate_zbh1(p, m, limit=None, warm=None):
    """Time-stepped run of the ZB-H1 policy on all p stages.

    ``limit`` is the in-flight ceiling (default p) and ``warm(s)`` the number of
    forwards stage s runs before its first B (default p - s, as in 1F1B).
    Returns (orders, start): per-stage lists of (kind, mb) and the start time
    of every op.
    """
    if limit is None:
        limit = p
    if warm is None:
        warm = lambda s: p - s  # noqa: E731
    fb = [fb_order(s, p, m, warm(s)) for s in range(p)]
    ptr = [0] * p
    orders = [[] for _ in range(p)]
    start = {}
    finish = {}
    f_issued = [0] * p
    w_issued = [0] * p
    pending_w = [[] for _ in range(p)]  # oldest first
    busy_until = [0] * p
    t = 0
    total = 3 * m * p
    while len(start) < total:
        if t > 100 * (m + p) + 100:
            raise RuntimeError("zbh1 simulation did not finish")
        decided = []
        for s in range(p):
            if busy_until[s] > t:
                continue
            op = None
            if ptr[s] < len(fb[s]):
                kind, i = fb[s][ptr[s]]
                ready = all(d in finish and finish[d] <= t for d in _deps(kind, s, i, p, True))
                if ready:
                    if kind == F and f_issued[s] - w_issued[s] >= limit:
                        if pending_w[s]:
                            op = (W, pending_w[s][0])
                    else:
                        op = (kind, i)
                elif pending_w[s]:
                    op = (W, pending_w[s][0])
            elif pending_w[s]:
                op = (W, pending_w[s][0])
            if op is not None:
                decided.append((s, op))
        # all stages decide on the state at time t, then the ops are applied
        for s, (kind, i) in decided:
            start[(kind, s, i)] = t
            finish[(kind, s, i)] = t + 1
            busy_until[s] = t + 1
            orders[s].append((kind, i))
            if kind == W:
                pending_w[s].pop(0)
                w_issued[s] += 1
            else:
                ptr[s] += 1
                if kind == F:
                    f_issued[s] += 1
                else:
                    pending_w[s].append(i)
        t += 1
    return orders, start


def simulate_timed(p, m, limit, warm, t_f, t_b, t_w):
    """The ZB-H1 policy of simulate_zbh1 with op durations t_f, t_b, t_w (integers).

    Stages decide whenever they are free, all on the state at that moment, as
    in the unit-time run; time then jumps to the next end of an op.  Returns
    (orders, start, finish)."""
    dur = {F: t_f, B: t_b, W: t_w}
    fb = [fb_order(s, p, m, warm(s)) for s in range(p)]
    ptr = [0] * p
    orders = [[] for _ in range(p)]
    start, finish = {}, {}
    f_issued = [0] * p
    w_issued = [0] * p
    pending_w = [[] for _ in range(p)]
    busy_until = [0] * p
    t = 0
    total = 3 * m * p
    while len(start) < total:
        decided = []
        for s in range(p):
            if busy_until[s] > t:
                continue
            op = None
            if ptr[s] < len(fb[s]):
                kind, i = fb[s][ptr[s]]
                ready = all(d in finish and finish[d] <= t for d in _deps(kind, s, i, p, True))
                if ready:
                    if kind == F and f_issued[s] - w_issued[s] >= limit:
                        if pending_w[s]:
                            op = (W, pending_w[s][0])
                    else:
                        op = (kind, i)
                elif pending_w[s]:
                    op = (W, pending_w[s][0])
            elif pending_w[s]:
                op = (W, pending_w[s][0])
            if op is not None:
                decided.append((s, op))
        for s, (kind, i) in decided:
            start[(kind, s, i)] = t
            finish[(kind, s, i)] = t + dur[kind]
            busy_until[s] = t + dur[kind]
            orders[s].append((kind, i))
            if kind == W:
                pending_w[s].pop(0)
                w_issued[s] += 1
            else:
                ptr[s] += 1
                if kind == F:
                    f_issued[s] += 1
                else:
                    pending_w[s].append(i)
        if len(start) < total:
            later = [v for v in finish.values() if v > t]
            if not later:
                raise RuntimeError("timed simulation deadlocked")
            t = min(later)
    return orders, start, finish


def limited_warm(p, limit):
    """Forwards before the first B of stage s under a ceiling of `limit` held microbatches."""
    return lambda s: min(limit - s, 2 * (p - s) - 1)


def search_limit(p, m, mem_limit, t_f, t_b, t_w):
    """The ceiling L in [p, min(2p, mem_limit)] whose order runs shortest with the given
    durations (the smallest L on ties).  Returns (L, makespan, orders)."""
    best = None
    for limit in range(p, min(2 * p, mem_limit) + 1):
        orders, _, finish = simulate_timed(p, m, limit, limited_warm(p, limit), t_f, t_b, t_w)
        span = max(finish.values())
        if best is None or span < best[1]:
            best = (limit, span, orders)
    return best


def simulate_zb2p(p, m):
    """ZB-2p: the ZB-H1 policy with ceiling 2p and 2(p - s) - 1 warm-up forwards."""
    return simulate_zbh1(p, m, limit=2 * p, warm=lambda s: 2 * (p - s) - 1)


def orders_for(kind, p, m):
    """Per-stage orders for "gpipe", "1f1b" or "zbh1"."""
    if kind == "gpipe":
        return [order_gpipe(s, p, m) for s in range(p)]
    if kind == "1f1b":
        return [order_1f1b(s, p, m) for s in range(p)]
    if kind == "zbh1":
        return simulate_zbh1(p, m)[0]
    if kind == "zb2p":
        return simulate_zb2p(p, m)[0]
    raise ValueError(kind)


def timeline(kind, p, m):
    """(orders, start times) of a schedule under the unit-time model."""
    orders = orders_for(kind, p, m)
    split = kind in ("zbh1", "zb2p")
    return orders, simulate_orders(orders, p, split)


def makespan(start):
    return max(start.values()) + 1


def bubble(kind, p, m):
    """Idle time of the pipeline under the unit-time model.

    Returns (idle / compute, idle / wall): compute is the 3m units each stage
    works, wall is the makespan, both summed over the p stages.
    """
    _, start = timeline(kind, p, m)
    span = makespan(start)
    idle = p * span - 3 * m * p
    return idle / (3 * m * p), idle / (p * span)


def peak_in_flight(order):
    """Largest number of microbatches whose F has run and whose W has not."""
    cur = peak = 0
    for kind, _ in order:
        if kind == F:
            cur += 1
            peak = max(peak, cur)
        elif kind == W:
            cur -= 1
    return peak


def window_idle(kind, p, m):
    """Idle units inside each stage's own active window (its first op's start to
    its last op's end), summed over the stages."""
    orders, start = timeline(kind, p, m)
    idle = 0
    for s, order in enumerate(orders):
        ts = [start[(k, s, i)] for k, i in order]
        idle += (max(ts) + 1 - min(ts)) - len(order)
    return idle
