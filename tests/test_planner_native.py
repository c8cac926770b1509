"""The native planner (pw_plan_bits, host code, no GPU) against the planner
oracle: the same bitwidths and resident bytes, bit for bit, on the hand-worked
cases and on random instances of the stack's shape."""
import numpy as np
import pytest

from oracle import planner as oplan

from test_oracle_planner import _cases


def test_hand_worked_cases():
    import any_precision_weight_gb300 as pw
    for name, mass, target, bits, res in _cases():
        got, total = pw.pw_plan_bits([1, 1], [64, 64], [1.0, 4.0], mass, 2, 0.5, 4, target, b_min=3, n_bits=5)
        assert list(got) == bits and total == res, name


@pytest.mark.parametrize("seed", range(5))
def test_matches_oracle_on_random_instances(seed):
    import any_precision_weight_gb300 as pw
    rng = np.random.default_rng(seed)
    E = 60
    nb = 2 * E * 3
    R = np.where(np.arange(nb) % 2 == 0, 2816, 2048)
    K = np.where(np.arange(nb) % 2 == 0, 2048, 1408)
    sens = rng.lognormal(0.0, 1.0, nb)
    resid = rng.normal(0.0, 0.3, nb) if seed % 2 else None
    p = rng.dirichlet(np.ones(E), size=3).reshape(-1)
    mass = np.repeat(p, 2)
    full = sum(oplan.resident_bytes(int(r), int(k), 8, 3) for r, k in zip(R, K))
    for frac in (0.9, 0.6, 0.4, 0.25):
        want, wt = oplan.plan_bits(list(R), list(K), list(sens), list(mass), E, 1.0 / E, 6, 3, 8,
                                   frac * full, resid=None if resid is None else list(resid))
        got, gt = pw.pw_plan_bits(R, K, sens, mass, E, 1.0 / E, 6, frac * full, resid=resid)
        assert np.array_equal(got, want) and gt == wt


def test_rejects_bad_floors():
    import any_precision_weight_gb300 as pw
    with pytest.raises(pw.PWError) as e:
        pw.pw_plan_bits([8], [64], [1.0], [0.0], 1, 0.5, 2, 100.0)   # hot floor below b_min
    assert e.value.code == pw.PW_EINVAL
