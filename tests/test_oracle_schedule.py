"""Pins for the schedule oracle (CPU only).

* the bubble values and the 1F1B diagram the pages print (``tests/golden/``);
* the closed forms of "Zero-Bubble Pipeline Parallelism Guide for LLMs":
  GPipe (p-1)/(m+p-1) (section "1. The GPipe Bubble"), 1F1B (p-1)/m of
  compute (section "2. The 1F1B ..."), (p-1)/(m+p-1) of wall time (section
  "Mathematical Modeling", item 1), ZB-1F1B (p-1)/(3m) (same section, item 2);
* the dependency rule (every W after its B, every B after its F) and the
  in-flight ceilings (section "Memory Management & Activation Rollback");
* a planted mistake in the simulator must break a pin.
"""
import os
from fractions import Fraction

import pytest

from oracle import schedule as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_bubble_table():
    rows = []
    with open(os.path.join(GOLDEN, "bubble_p8.txt")) as fh:
        for line in fh:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            kind, m, qty, pct = line.split()
            rows.append((kind, int(m), qty, float(pct)))
    return rows


def read_diagram():
    out = {}
    with open(os.path.join(GOLDEN, "diagram_1f1b_p4.txt")) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            s, ops = line.split(":")
            out[int(s)] = [(op[0], int(op[1:])) for op in ops.split()]
    return out


def test_printed_bubble_values():
    rows = read_bubble_table()
    assert len(rows) == 8
    for kind, m, qty, pct in rows:
        over_compute, over_wall = S.bubble(kind, 8, m)
        val = over_compute if qty == "idle_over_compute" else over_wall
        decimals = len(str(pct).split(".")[1])
        assert round(100 * val, decimals) == pct, (kind, m, qty, pct, val)


def test_printed_1f1b_diagram():
    diag = read_diagram()
    for s, ops in diag.items():
        fb = [op for op in S.order_1f1b(s, 4, 8) if op[0] != S.W]
        assert fb[: len(ops)] == ops, s


@pytest.mark.parametrize("p", [1, 2, 3, 4, 8, 12])
@pytest.mark.parametrize("m", [1, 2, 5, 8, 16, 24, 33])
def test_closed_forms(p, m):
    _, start = S.timeline("gpipe", p, m)
    span = S.makespan(start)
    assert Fraction(p * span - 3 * m * p, p * span) == Fraction(p - 1, m + p - 1)
    _, start = S.timeline("1f1b", p, m)
    span = S.makespan(start)
    assert Fraction(p * span - 3 * m * p, 3 * m * p) == Fraction(p - 1, m)
    assert Fraction(p * span - 3 * m * p, p * span) == Fraction(p - 1, m + p - 1)
    if m >= p:
        _, start = S.timeline("zbh1", p, m)
        span = S.makespan(start)
        assert span == 3 * m + p - 1
        assert Fraction(p * span - 3 * m * p, 3 * m * p) == Fraction(p - 1, 3 * m)


def test_zbh1_example_p8_m16():
    # (p-1)/(3m) = 7/48 at p = 8, m = 16
    c, _ = S.bubble("zbh1", 8, 16)
    assert abs(c - 7 / 48) < 1e-15


@pytest.mark.parametrize("kind", ["gpipe", "1f1b", "zbh1"])
@pytest.mark.parametrize("p,m", [(1, 1), (2, 1), (4, 2), (4, 8), (8, 3), (8, 16), (5, 13)])
def test_order_invariants(kind, p, m):
    orders, start = S.timeline(kind, p, m)
    for s, order in enumerate(orders):
        assert len(order) == 3 * m
        for k in (S.F, S.B, S.W):
            assert sorted(i for kk, i in order if kk == k) == list(range(m))
        pos = {op: j for j, op in enumerate(order)}
        for i in range(m):
            assert pos[(S.F, i)] < pos[(S.B, i)] < pos[(S.W, i)]
        # forwards and backwards run in microbatch order
        assert [i for k, i in order if k == S.F] == list(range(m))
        assert [i for k, i in order if k == S.B] == list(range(m))
        peak = S.peak_in_flight(order)
        if kind == "zbh1":
            assert peak <= p
        elif kind == "1f1b":
            assert peak == min(p - s, m)
    # cross-stage dependencies hold in the timeline
    split = kind == "zbh1"
    for (k, s, i), t in start.items():
        for d in S._deps(k, s, i, p, split):
            assert start[d] + 1 <= t


def test_zbh1_steady_rhythm():
    """Steady state runs B -> W -> F triples ("balanced 1F1B rhythm F -> B -> W")."""
    orders = S.orders_for("zbh1", 8, 16)
    s = 3
    order = orders[s]
    first_w = order.index((S.W, 0))
    steady = order[first_w - 1 : first_w - 1 + 3 * (16 - 8)]
    for j in range(0, len(steady), 3):
        assert [op[0] for op in steady[j : j + 3]] == [S.B, S.W, S.F]


def test_planted_simulator_mistake_is_caught(monkeypatch):
    real = S._deps

    def no_wait_downstream(kind, s, i, p, split):
        return [d for d in real(kind, s, i, p, split) if not (kind == S.B and d[1] == s + 1)]

    monkeypatch.setattr(S, "_deps", no_wait_downstream)
    with pytest.raises(AssertionError):
        test_printed_bubble_values()


@pytest.mark.parametrize("p", [1, 2, 3, 4, 5, 8])
def test_zb2p_claims(p):
    """"Zero-Bubble Pipeline Parallelism Guide for LLMs", section "Core Innovation 2",
    item 2 (ZB-2p): at most 2p microbatches held, and no GPU idles once m is large enough
    (here: no idle inside any stage's own window for m >= 2p - 1)."""
    for m in range(2 * p - 1, 2 * p + 12):
        orders = S.orders_for("zb2p", p, m)
        assert max(S.peak_in_flight(o) for o in orders) <= 2 * p
        assert S.window_idle("zb2p", p, m) == 0
        _, start = S.timeline("zb2p", p, m)
        assert S.makespan(start) == 3 * m + p - 1


def test_zbh1_window_idle_is_the_ramp():
    """ZB-H1 keeps idle inside the stages' windows: stage s waits s units for its first
    input or p-1-s units at the end, p(p-1)/2 in all; ZB-2p removes it."""
    for p in (2, 4, 8):
        for m in (2 * p, 3 * p):
            assert S.window_idle("zbh1", p, m) == p * (p - 1) // 2
            assert S.window_idle("zb2p", p, m) == 0


@pytest.mark.parametrize("p,m", [(1, 1), (2, 1), (4, 2), (4, 8), (8, 3), (8, 16), (5, 13)])
def test_zb2p_invariants(p, m):
    orders, start = S.timeline("zb2p", p, m)
    for order in orders:
        assert len(order) == 3 * m
        pos = {op: j for j, op in enumerate(order)}
        for i in range(m):
            assert pos[(S.F, i)] < pos[(S.B, i)] < pos[(S.W, i)]
    for (k, s, i), t in start.items():
        for d in S._deps(k, s, i, p, True):
            assert start[d] + 1 <= t


# ----------------------------------------------------------------------------
# memory-limited orders with measured durations
# ----------------------------------------------------------------------------

DURATIONS = [(1, 1, 1), (10, 12, 9), (3, 7, 2), (5, 5, 11)]


@pytest.mark.parametrize("p", [1, 2, 4, 8])
@pytest.mark.parametrize("m", [1, 3, 8, 16, 21])
def test_timed_run_with_unit_times_is_the_unit_policy(p, m):
    """With t_F = t_B = t_W = 1 the timed run is the unit-time ZB-H1 (L = p) and ZB-2p (L = 2p)."""
    orders, _, _ = S.simulate_timed(p, m, p, S.limited_warm(p, p), 1, 1, 1)
    assert orders == S.simulate_zbh1(p, m)[0]
    orders, _, _ = S.simulate_timed(p, m, 2 * p, S.limited_warm(p, 2 * p), 1, 1, 1)
    assert orders == S.simulate_zb2p(p, m)[0]


@pytest.mark.parametrize("t", [1, 3, 7])
def test_timed_equal_durations_scale_the_closed_form(t):
    """Equal durations t: ZB-H1 ends at t (3m + p - 1) for m >= p ("Mathematical Modeling")."""
    for p in (2, 4, 8):
        for m in (p, 2 * p + 1):
            _, _, finish = S.simulate_timed(p, m, p, S.limited_warm(p, p), t, t, t)
            assert max(finish.values()) == t * (3 * m + p - 1)


@pytest.mark.parametrize("tf,tb,tw", DURATIONS)
@pytest.mark.parametrize("p,m", [(2, 5), (4, 8), (4, 13), (8, 16)])
def test_timed_invariants(tf, tb, tw, p, m):
    dur = {S.F: tf, S.B: tb, S.W: tw}
    for limit in range(p, 2 * p + 1):
        orders, start, finish = S.simulate_timed(p, m, limit, S.limited_warm(p, limit), tf, tb, tw)
        for s, order in enumerate(orders):
            assert len(order) == 3 * m
            assert S.peak_in_flight(order) <= limit
            pos = {op: j for j, op in enumerate(order)}
            for i in range(m):
                assert pos[(S.F, i)] < pos[(S.B, i)] < pos[(S.W, i)]
            # one op at a time per stage, in program order
            ends = [start[(k, s, i)] + dur[k] for k, i in order]
            starts = [start[(k, s, i)] for k, i in order]
            assert all(ends[j] <= starts[j + 1] for j in range(len(order) - 1))
        for (k, s, i), t0 in start.items():
            assert finish[(k, s, i)] == t0 + dur[k]
            for d in S._deps(k, s, i, p, True):
                assert finish[d] <= t0
        span = max(finish.values())
        assert span >= m * (tf + tb + tw)        # every stage does all of its work
        assert span >= p * (tf + tb) + tw        # microbatch 0 down and back, then a W


@pytest.mark.parametrize("tf,tb,tw", DURATIONS)
def test_search_takes_the_best_limit_within_memory(tf, tb, tw):
    p, m = 4, 12
    spans = {}
    for limit in range(p, 2 * p + 1):
        _, _, finish = S.simulate_timed(p, m, limit, S.limited_warm(p, limit), tf, tb, tw)
        spans[limit] = max(finish.values())
    prev = None
    for mem in range(p, 2 * p + 3):
        limit, span, orders = S.search_limit(p, m, mem, tf, tb, tw)
        allowed = [l for l in spans if l <= mem]
        assert limit <= mem and span == min(spans[l] for l in allowed)
        assert limit == min(l for l in allowed if spans[l] == span)
        assert max(S.peak_in_flight(o) for o in orders) <= limit
        if prev is not None:
            assert span <= prev  # more memory never makes the best order slower
        prev = span


def test_planted_ceiling_mistake_is_caught(monkeypatch):
    """A run that ignores the ceiling must break the in-flight pin."""
    real = S.simulate_timed

    def no_ceiling(p, m, limit, warm, tf, tb, tw):
        return real(p, m, 10 ** 9, warm, tf, tb, tw)

    monkeypatch.setattr(S, "simulate_timed", no_ceiling)
    with pytest.raises(AssertionError):
        test_timed_invariants(10, 12, 9, 4, 8)
