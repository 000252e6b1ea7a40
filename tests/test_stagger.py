"""The staggering scheduler's host code (vc_stagger_plan / _simulate /
_horizon): no GPU.  Pinned by brute force (optimal phase loads on tiny
cases, Graham's bound for longest-processing-time-first), closed forms of the
staging model (unlimited link, no compute, one staging slot with layer-wise
landing, lock-step rounds) and the guide's horizon rule L_min =
ceil(swap time / draft-step time) in the case it covers ("VeriCache Guide",
"Best Practice 1")."""
import itertools
import math

import numpy as np
import pytest


@pytest.fixture(scope="module")
def vc():
    import __graft_entry__
    __graft_entry__._builder().build()
    import lossless_compressed_kv_gb300 as m
    return m


def test_plan_is_a_partition_with_exact_loads(vc):
    rng = np.random.default_rng(0)
    for _ in range(20):
        n, p = int(rng.integers(0, 40)), int(rng.integers(1, 12))
        sb = rng.integers(0, 1 << 40, n)
        ph, pb = vc.stagger_plan(sb, p)
        assert ph.shape == (n,) and ((ph >= 0) & (ph < p)).all()
        assert pb.tolist() == [int(sb[ph == q].sum()) for q in range(p)]


def test_plan_tie_rules(vc):
    # equal sizes: lower index first, each to the emptiest group (lower group
    # on ties); groups by load 0 (21), 1 (14), 2 (14) interleaved 0, 2, 1
    ph, pb = vc.stagger_plan([7] * 7, 3)
    assert ph.tolist() == [0, 2, 1, 0, 2, 1, 0]
    assert pb.tolist() == [21, 14, 14]
    # decreasing order is by size, not index: groups {1}, {2}, {0} with
    # loads 5, 3, 1, interleaved largest, smallest, middle
    ph, pb = vc.stagger_plan([1, 5, 3], 3)
    assert ph.tolist() == [1, 0, 2] and pb.tolist() == [5, 1, 3]
    # more phases than requests: one request per group, groups spread out
    ph, pb = vc.stagger_plan([4, 9], 5)
    assert ph.tolist() == [2, 0] and pb.tolist() == [9, 0, 4, 0, 0]


def test_plan_spreads_and_interleaves_when_phases_outnumber_requests(vc):
    rng = np.random.default_rng(5)
    for n, P in ((6, 13), (32, 65), (5, 5), (7, 100)):
        sb = rng.integers(1, 10 ** 6, n)
        ph, pb = vc.stagger_plan(sb, P)
        used = np.sort(ph)
        assert len(set(ph.tolist())) == n                      # one request per phase
        assert used.tolist() == [k * P // n for k in range(n)]  # evenly spaced
        seq = pb[used]                                          # bytes in phase order
        srt = np.sort(sb)[::-1]
        inter = [srt[i // 2] if i % 2 == 0 else srt[n - 1 - i // 2] for i in range(n)]
        assert seq.tolist() == [int(v) for v in inter]          # largest, smallest, ...


def test_plan_within_grahams_bound_of_brute_force(vc):
    """LPT makespan <= (4/3 - 1/(3p)) x the optimal makespan (Graham 1969),
    the optimum found by enumerating every assignment."""
    rng = np.random.default_rng(1)
    for _ in range(40):
        n, p = int(rng.integers(1, 8)), int(rng.integers(2, 4))
        sb = rng.integers(1, 100, n)
        _, pb = vc.stagger_plan(sb, p)
        best = min(max(np.bincount(a, weights=sb, minlength=p)) for a in
                   (np.array(t) for t in itertools.product(range(p), repeat=n)))
        assert pb.max() <= (4 / 3 - 1 / (3 * p)) * best + 1e-9
        assert pb.max() >= best


def test_simulate_unlimited_link_has_no_stall(vc):
    rng = np.random.default_rng(2)
    n, P = 10, 6
    sb = rng.integers(1, 1000, n)
    d, v = rng.random(n) * 5, rng.random(n) * 20
    ph, _ = vc.stagger_plan(sb, P)
    r = vc.stagger_simulate(ph, P, sb, d, v, link_bytes_per_ns=1e15, n_slots=2, n_layers=3, tick_ns=1.5)
    comp = P * (d.sum() + 1.5) + (v - d).sum()
    assert r["stall_ns"] == pytest.approx(0.0, abs=1e-6)
    assert r["compute_ns"] == pytest.approx(comp)
    assert r["cycle_ns"] == pytest.approx(comp)
    assert r["overlap"] == pytest.approx(1.0)
    assert r["draft_tokens_per_cycle"] == n * (P - 1)


def test_simulate_without_compute_is_link_bound(vc):
    sb = np.array([300, 100, 200, 400])
    ph, _ = vc.stagger_plan(sb, 4)
    r = vc.stagger_simulate(ph, 4, sb, np.zeros(4), np.zeros(4), link_bytes_per_ns=10.0, n_slots=2)
    assert r["cycle_ns"] == pytest.approx(100.0)     # 1000 bytes at 10 B/ns
    assert r["stage_ns"] == pytest.approx(100.0)
    assert r["stall_ns"] == pytest.approx(100.0)
    assert r["overlap"] == pytest.approx(0.0)
    assert r["peak_stage_bytes"] == 2 * 400


@pytest.mark.parametrize("L", [1, 2, 4])
def test_simulate_single_slot_closed_form(vc, L):
    """One request per phase, one staging slot, staging S >= compute T per
    tick: a job can start only when the previous tick ends, its layers land
    every S/L, so a tick lasts S + T/L and stalls S - T + T/L."""
    n = P = 5
    S, T = 50.0, 20.0
    sb = np.full(n, S * 10)                      # 10 B/ns
    d = np.full(n, T / n)                        # every tick: all draft ...
    v = d.copy()                                 # ... and the verifier costs the same
    ph = np.arange(n, dtype=np.int32)
    r = vc.stagger_simulate(ph, P, sb, d, v, link_bytes_per_ns=10.0, n_slots=1, n_layers=L)
    assert r["cycle_ns"] == pytest.approx(P * (S + T / L))
    assert r["stall_ns"] == pytest.approx(P * (S - T + T / L))
    # two slots: the link runs back to back, the cycle is link bound
    r2 = vc.stagger_simulate(ph, P, sb, d, v, link_bytes_per_ns=10.0, n_slots=2, n_layers=L)
    assert r2["cycle_ns"] == pytest.approx(P * S)
    assert r2["stall_ns"] < r["stall_ns"]


def test_simulate_lock_step_round(vc):
    """Lock step: every request verifies at the last tick of the cycle, all
    of KV_full is one job; with one slot the job overlaps only the x draft
    ticks: stall = max(0, S_all - x T_draft)."""
    n, x = 8, 6
    P = x + 1
    sb = np.full(n, 1000)
    d, v = np.full(n, 2.0), np.full(n, 5.0)
    ph = np.full(n, P - 1, np.int32)
    r = vc.stagger_simulate(ph, P, sb, d, v, link_bytes_per_ns=10.0, n_slots=1, n_layers=1)
    S_all, Td, Tv = 800.0, 16.0, 40.0
    assert r["stall_ns"] == pytest.approx(max(0.0, S_all - x * Td))
    assert r["cycle_ns"] == pytest.approx(x * Td + Tv + max(0.0, S_all - x * Td))
    assert r["peak_stage_bytes"] == 8000
    # the balanced staggered plan over the same cycle needs far less staging memory
    ph2, _ = vc.stagger_plan(sb, P)
    r2 = vc.stagger_simulate(ph2, P, sb, d, v, link_bytes_per_ns=10.0, n_slots=2, n_layers=1)
    assert r2["peak_stage_bytes"] == 2 * 2000
    assert r2["cycle_ns"] <= r["cycle_ns"]


@pytest.mark.parametrize("S,T", [(1000.0, 7.0), (640.0, 16.0), (90.0, 100.0), (5000.0, 3.0)])
def test_horizon_reduces_to_the_guides_rule(vc, S, T):
    """One request, verification free: the smallest stall-free horizon is
    ceil(T_swap / T_step)."""
    x, ph, r = vc.stagger_horizon([int(S * 4)], [T], [0.0], link_bytes_per_ns=4.0, x_lo=1, x_hi=4000)
    assert x == max(1, math.ceil(S / T))
    assert r["stall_ns"] == 0.0
    if x > 1:
        r1 = vc.stagger_simulate(ph, x, [int(S * 4)], [T], [0.0], link_bytes_per_ns=4.0)
        assert r1["stall_ns"] > 0.0       # one step shorter stalls


def test_horizon_caps_at_x_hi(vc):
    x, _, r = vc.stagger_horizon([10 ** 9] * 4, [1.0] * 4, [1.0] * 4, link_bytes_per_ns=1.0, x_lo=2, x_hi=9)
    assert x == 9 and r["stall_ns"] > 0.0 and 0.0 <= r["overlap"] < 1.0


def test_argument_errors(vc):
    with pytest.raises(vc.VCError):
        vc.stagger_plan([1, -2], 2)
    with pytest.raises(vc.VCError):
        vc.stagger_plan([1, 2], 0)
    with pytest.raises(vc.VCError):
        vc.stagger_simulate([0, 3], 3, [1, 1], [1, 1], [1, 1], 1.0)        # phase out of range
    with pytest.raises(vc.VCError):
        vc.stagger_simulate([0, 1], 2, [1, 1], [1, 1], [1, 1], 0.0)        # no link
    with pytest.raises(vc.VCError):
        vc.stagger_simulate([0, 1], 2, [1, 1], [1, 1], [1, 1], 1.0, n_slots=0)
    with pytest.raises(vc.VCError):
        vc.stagger_horizon([1], [1.0], [1.0], 1.0, x_lo=5, x_hi=4)
