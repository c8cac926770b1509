"""Pins of the planner oracle: hand-worked greedy orders, the invariants any
plan must satisfy, and optimality at the greedy's own breakpoints checked by
brute force over every assignment of tiny instances (damage per byte grows as
a block loses bits, so the greedy prefix is the fractional optimum there)."""
import itertools
import os

import numpy as np
import pytest

from oracle import planner

GOLD = os.path.join(os.path.dirname(__file__), "golden", "planner_hand.txt")


def _cases():
    out = []
    for line in open(GOLD):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, p, target, bits, res = (x.strip() for x in line.split("|"))
        out.append((name, [float(v) for v in p.split()], float(target),
                    [int(v) for v in bits.split()], int(res)))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_hand_worked_plans(case):
    name, mass, target, bits, res = case
    got, total = planner.plan_bits([1, 1], [64, 64], [1.0, 4.0], mass, 2, 0.5, 4, 3, 5, target)
    assert list(got) == bits and total == res


def test_resident_bytes_matches_the_layout():
    # q planes of R*K/8 bytes and tables of 2^b fp16 entries per row for b = 3..q
    assert planner.resident_bytes(2816, 2048, 6, 3) == 6 * 2816 * 2048 // 8 + 2816 * 2 * (8 + 16 + 32 + 64)
    for q in range(4, 9):
        assert (planner.resident_bytes(7, 96, q, 3) - planner.resident_bytes(7, 96, q - 1, 3)
                == planner.reduction_bytes(7, 96, q))


def _random_instance(rng, nb):
    R = rng.integers(1, 4, nb) * 8
    K = rng.integers(1, 4, nb) * 32
    sens = rng.lognormal(0.0, 1.0, nb)
    mass = rng.dirichlet(np.ones(nb))
    return list(R), list(K), list(sens), list(mass)


@pytest.mark.parametrize("seed", range(6))
def test_invariants_on_random_instances(seed):
    rng = np.random.default_rng(seed)
    R, K, sens, mass = _random_instance(rng, 9)
    full = sum(planner.resident_bytes(r, k, 8, 3) for r, k in zip(R, K))
    prev = None
    for frac in (1.0, 0.8, 0.6, 0.45, 0.3, 0.1):
        bits, total = planner.plan_bits(R, K, sens, mass, 9, 1.0 / 9, 6, 3, 8, frac * full)
        floors = [6 if m >= 1.0 / 9 else 3 for m in mass]
        assert all(f <= b <= 8 for f, b in zip(floors, bits))
        assert total == sum(planner.resident_bytes(r, k, int(b), 3) for r, k, b in zip(R, K, bits))
        assert total <= frac * full or all(b == f for b, f in zip(bits, floors))
        if prev is not None:                       # a smaller target never raises a block
            assert all(b <= p for b, p in zip(bits, prev))
        prev = bits


@pytest.mark.parametrize("seed", range(4))
def test_greedy_is_optimal_at_its_breakpoints(seed):
    rng = np.random.default_rng(100 + seed)
    R, K, sens, mass = _random_instance(rng, 3)
    E, bmin, n = 3, 3, 6
    levels = range(bmin, n + 1)
    full = sum(planner.resident_bytes(r, k, n, bmin) for r, k in zip(R, K))
    # every breakpoint the greedy passes through, by lowering the target one step at a time
    seen = set()
    target = full
    while True:
        bits, total = planner.plan_bits(R, K, sens, mass, E, 2.0, n, bmin, n, target)
        if total in seen:
            break
        seen.add(total)
        dmg = planner.total_damage(R, K, sens, mass, E, bits, n)
        best = min(planner.total_damage(R, K, sens, mass, E, a, n)
                   for a in itertools.product(levels, repeat=3)
                   if sum(planner.resident_bytes(r, k, q, bmin) for r, k, q in zip(R, K, a)) <= total)
        assert dmg <= best * (1 + 1e-12)
        target = total - 1


def test_prompt_residual_shifts_the_sensitivity():
    # block B's residual -3.5 makes its effective sensitivity 0.5 < A's 1: B goes first
    bits, _ = planner.plan_bits([1, 1], [64, 64], [1.0, 4.0], [0, 0], 2, 0.5, 4, 3, 5, 250,
                                resid=[0.0, -3.5])
    assert list(bits) == [5, 4]
    # a residual below -s clamps at zero damage
    bits, _ = planner.plan_bits([1, 1], [64, 64], [1.0, 4.0], [0, 0], 2, 0.5, 4, 3, 5, 120,
                                resid=[0.0, -9.0])
    assert list(bits) == [4, 3]
