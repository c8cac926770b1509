"""The quality-aware bitwidth planner, restated plainly (oracle; test
infrastructure only).

Source: PagedWeight technical summary, core components section 2
("Quality-Aware Runtime Planner"): three signals decide which linear blocks
lose precision -- an offline Hessian-weighted sensitivity per block, online
routing statistics per expert (frequently routed "hot" experts get higher
bitwidth floors and damage multipliers) and a prompt-specific residual that
corrects the sensitivity; the planner scores the "damage" of each possible
bitwidth reduction and, when a memory target is triggered, greedily takes the
reductions of lowest damage per byte saved until the target is met.

The pages give the structure, not the formulas.  This build reads them as:

* effective sensitivity  s' = max(0, s + r)   (r: the prompt residual, 0 if none);
* damage multiplier      m  = 1 + E * p      (p: the routing mass of the
  block's expert, E experts: a uniformly routed expert has m = 2);
* hot expert             p >= hot_mass, bitwidth floor hot_floor (else b_min);
* damage of lowering a block from b to b - 1 bits:
      m * s' * R * K * (4^-(b-1) - 4^-b)
  (the mean squared error of a b-bit quantiser scales as 4^-b per weight);
* bytes saved by it: the plane R*K/8 plus the b-bit table R * 2^b * 2
  (a block at q bits holds planes 0..q-1 and the tables of b_min..q bits);
* start from every block at n bits; repeatedly take the candidate reduction
  with the smallest damage / bytes saved (ties: lower block index) until the
  resident bytes are at most the target or no block is above its floor.
"""
import numpy as np


def resident_bytes(R: int, K: int, q: int, b_min: int) -> int:
    """Bytes a block keeps on the device at q bits: q planes and tables b_min..q."""
    return R * K * q // 8 + R * 2 * sum(1 << c for c in range(b_min, q + 1))


def reduction_damage(R, K, s_eff, mult, b):
    """Damage of lowering a block from b to b - 1 bits."""
    return mult * s_eff * R * K * (4.0 ** -(b - 1) - 4.0 ** -b)


def reduction_bytes(R, K, b):
    """Bytes saved by lowering a block from b to b - 1 bits."""
    return R * K // 8 + R * 2 * (1 << b)


def plan_bits(R, K, sens, mass, E, hot_mass, hot_floor, b_min, n_bits, target, resid=None):
    """Greedy lowest-damage-per-byte bitwidths for a memory target.

    R, K, sens, mass (the routing mass of each block's expert), resid: one
    entry per block.  Returns (bits int array, resident bytes).
    """
    nb = len(R)
    s_eff = [max(0.0, float(sens[i]) + (float(resid[i]) if resid is not None else 0.0))
             for i in range(nb)]
    mult = [1.0 + E * float(mass[i]) for i in range(nb)]
    floor = [hot_floor if float(mass[i]) >= hot_mass else b_min for i in range(nb)]
    bits = [n_bits] * nb
    total = sum(resident_bytes(R[i], K[i], n_bits, b_min) for i in range(nb))
    while total > target:
        best = None
        for i in range(nb):                       # plain scan: smallest ratio, lowest index
            if bits[i] <= floor[i]:
                continue
            ratio = (reduction_damage(R[i], K[i], s_eff[i], mult[i], bits[i])
                     / reduction_bytes(R[i], K[i], bits[i]))
            if best is None or ratio < best[0]:
                best = (ratio, i)
        if best is None:
            break
        i = best[1]
        total -= reduction_bytes(R[i], K[i], bits[i])
        bits[i] -= 1
    return np.array(bits, dtype=np.int64), total


def total_damage(R, K, sens, mass, E, bits, n_bits, resid=None):
    """Sum over blocks of the damage of every reduction from n bits down to bits."""
    d = 0.0
    for i in range(len(R)):
        s = max(0.0, float(sens[i]) + (float(resid[i]) if resid is not None else 0.0))
        m = 1.0 + E * float(mass[i])
        for b in range(int(bits[i]) + 1, n_bits + 1):
            d += reduction_damage(R[i], K[i], s, m, b)
    return d
