// The quality-aware bitwidth planner (host).
//
// Source: PagedWeight technical summary, core components section 2
// ("Quality-Aware Runtime Planner"): an offline Hessian-weighted sensitivity
// per linear block, online routing statistics per expert (hot experts get
// higher bitwidth floors and damage multipliers) and a prompt-specific
// residual correction are combined into a "damage" score for every possible
// bitwidth reduction; under a memory target the planner greedily takes the
// reductions of lowest damage per byte saved until the target is met.
//
// The formulas are this library's reading (the pages give none):
//   s' = max(0, s + r), m = 1 + E * p, floor = hot_floor if p >= hot_mass else b_min,
//   damage(b -> b-1) = m * s' * R * K * (4^-(b-1) - 4^-b),
//   bytes saved      = R * K / 8 + R * 2^b * 2 (one plane and the b-bit table).
// Damage per byte grows as a block loses bits, so taking reductions in
// increasing damage-per-byte order never lowers a block out of turn, and the
// greedy's prefixes are the least-damage plans for their own byte counts.

#include <cmath>
#include <cstdint>
#include <queue>
#include <vector>

#include "pw_internal.h"

namespace {

int64_t resident(int64_t R, int64_t K, int q, int b_min) {
  int64_t tables = 0;
  for (int c = b_min; c <= q; ++c) tables += int64_t(1) << c;
  return R * K * q / 8 + R * 2 * tables;
}

struct Cand {
  double ratio;
  int block;
};
struct Worse {   // priority_queue puts the "largest" on top: the smallest ratio, then index
  bool operator()(const Cand& a, const Cand& b) const {
    if (a.ratio != b.ratio) return a.ratio > b.ratio;
    return a.block > b.block;
  }
};

}  // namespace

extern "C" int pw_plan_bits(int n_blocks, const int* R, const int* K, const double* sens,
                            const double* resid, const double* mass, int n_experts,
                            double hot_mass, int hot_floor, int b_min, int n_bits,
                            double target_bytes, int* bits_out, int64_t* resident_out) {
  if (n_blocks < 0 || (n_blocks > 0 && (!R || !K || !sens || !mass || !bits_out)))
    return pw::set_error(PW_EINVAL, "pw_plan_bits: bad count or null array");
  if (n_bits < 1 || n_bits > PW_MAX_BITS || b_min < 1 || b_min > n_bits || hot_floor < b_min ||
      hot_floor > n_bits || n_experts < 1)
    return pw::set_error(PW_EINVAL, "pw_plan_bits: need 1 <= b_min <= hot_floor <= n_bits <= 8, E >= 1");
  for (int i = 0; i < n_blocks; ++i)
    if (R[i] < 1 || K[i] < 8 || K[i] % 8)
      return pw::set_error(PW_EINVAL, "pw_plan_bits: block with R < 1 or K not a positive multiple of 8");

  std::vector<double> s_eff(n_blocks), mult(n_blocks);
  std::vector<int> floor(n_blocks);
  int64_t total = 0;
  for (int i = 0; i < n_blocks; ++i) {
    const double s = sens[i] + (resid ? resid[i] : 0.0);
    s_eff[i] = s > 0.0 ? s : 0.0;
    mult[i] = 1.0 + static_cast<double>(n_experts) * mass[i];
    floor[i] = mass[i] >= hot_mass ? hot_floor : b_min;
    bits_out[i] = n_bits;
    total += resident(R[i], K[i], n_bits, b_min);
  }
  auto saved = [&](int i, int b) { return int64_t(R[i]) * K[i] / 8 + int64_t(R[i]) * 2 * (int64_t(1) << b); };
  auto ratio = [&](int i, int b) {
    const double dmg = mult[i] * s_eff[i] * R[i] * K[i] * (std::ldexp(1.0, -2 * (b - 1)) - std::ldexp(1.0, -2 * b));
    return dmg / static_cast<double>(saved(i, b));
  };
  std::priority_queue<Cand, std::vector<Cand>, Worse> heap;
  for (int i = 0; i < n_blocks; ++i)
    if (bits_out[i] > floor[i]) heap.push({ratio(i, bits_out[i]), i});
  while (static_cast<double>(total) > target_bytes && !heap.empty()) {
    const int i = heap.top().block;
    heap.pop();
    total -= saved(i, bits_out[i]);
    --bits_out[i];
    if (bits_out[i] > floor[i]) heap.push({ratio(i, bits_out[i]), i});
  }
  if (resident_out) *resident_out = total;
  return PW_OK;
}
