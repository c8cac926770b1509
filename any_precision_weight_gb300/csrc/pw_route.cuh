// Routing + permutation shared by the kernels that run it (device code).
//
// Source: PagedWeight technical summary, problem statement (an MoE activates a
// subset of experts per token); the top-k softmax and the token -> expert
// gather with per-expert offsets are the routing steps of the fused layer.
#pragma once

#include "pw_device.cuh"

namespace pw {

constexpr int kMaxE = 256;

// Order of the top-k: larger logit first, ties to the lower expert index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Stable placement of a large batch's routed pairs by one CTA (blockDim.x a
// multiple of 32, at most 1024): per-expert counts, offsets, the active list,
// and perm / inv in (expert, token) order.  Warp w owns a contiguous chunk of
// the pair ids t*k + j (a token has distinct experts, so pair-id order within
// an expert is token order): it counts its chunk's pairs per expert, the
// per-expert counts of the chunks are scanned into each chunk's first
// position, and the warp places its pairs 32 at a time, a pair's rank among
// the lanes holding the same expert coming from a match.  s_c: shared
// [32][kMaxE] ints; s_off: shared kMaxE + 1 ints.  idx must be complete.
__device__ __forceinline__ void permute_block(const Fwd& p, int (*s_c)[kMaxE], int* s_off) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int E = p.E, P = p.T * p.k;
  const int chunk = (P + nwarp - 1) / nwarp;
  const int q0 = min(P, warp * chunk), q1 = min(P, q0 + chunk);
  for (int e = lane; e < E; e += 32) s_c[warp][e] = 0;
  __syncwarp();
  for (int q = q0 + lane; q < q1; q += 32) atomicAdd(&s_c[warp][p.idx[q]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {   // chunk bases within the expert, and its count
    int run = 0;
    for (int w = 0; w < nwarp; ++w) {
      const int c = s_c[w][e];
      s_c[w][e] = run;
      run += c;
    }
    s_off[e] = run;
    p.counts[e] = run;
  }
  __syncthreads();
  if (threadIdx.x < 32) {   // warp-level exclusive scan of the counts and of the active flags
    int run = 0, na = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + threadIdx.x;
      const int c = e < E ? s_off[e] : 0;
      int incl = c, actv = c > 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const int a = __shfl_up_sync(0xffffffffu, actv, o);
        if (threadIdx.x >= o) { incl += v; actv += a; }
      }
      if (e < E) {
        s_off[e] = run + incl - c;
        if (c) p.active[1 + na + actv - 1] = e;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      na += __shfl_sync(0xffffffffu, actv, 31);
    }
    if (threadIdx.x == 0) {
      s_off[E] = run;
      p.active[0] = na;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    p.offsets[e] = s_off[e];
    if (p.user_offsets) p.user_offsets[e] = s_off[e];
  }
  for (int i = threadIdx.x; i < nwarp * E; i += blockDim.x) s_c[i / E][i % E] += s_off[i % E];
  __syncthreads();
  for (int b = q0; b < q1; b += 32) {
    const int q = b + lane;
    const bool v = q < q1;
    const unsigned act = __ballot_sync(0xffffffffu, v);
    if (v) {
      const int e = p.idx[q];
      const unsigned same = __match_any_sync(act, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const int pos = s_c[warp][e] + rank;
      p.perm[pos] = q;
      p.inv[q] = pos;
      if (p.user_perm) p.user_perm[pos] = q;
      __syncwarp(act);   // every lane has read its expert's base
      if (rank == 0) s_c[warp][e] += __popc(same);
    }
    __syncwarp();
  }
  if (p.user_idx || p.user_w)
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
      if (p.user_idx) p.user_idx[i] = p.idx[i];
      if (p.user_w) p.user_w[i] = p.w[i];
    }
}

// ------------------------------------------------------------------ routing into shared memory

// Routing results of a decode batch held in one CTA's shared memory.
struct RouteSmem {
  int* idx;    // [T*k] expert of (t, j), descending logit
  float* w;    // [T*k] routing weight of (t, j)
  int* perm;   // [T*k] pair id t*k+j at each permuted position
  int* inv;    // [T*k] permuted position of each pair id
  int* cnt;    // [E]   tokens per expert
  int* off;    // [E+1] first permuted position of each expert
  int* act;    // [E+1] number of active experts, then their ids (expert order)
  int* lpt;    // [E+1] the same, largest gate_up cost first
  int* qgu;    // [E]   committed q of each expert's gate_up block
};
constexpr int kRouteSmemMaxPairs = 256;   // T*k bound of the fused decode path
__host__ __device__ constexpr int route_smem_bytes() {
  return (4 * kRouteSmemMaxPairs + 5 * (kMaxE + 1)) * 4;
}

// Top-k (larger logit first, ties to the lower expert index) and softmax
// weights over all E of the tokens t0, t0 + tstep, ..., one warp per token,
// with NPER logits per lane (E <= 32 * NPER); results into r.idx / r.w (shared
// or global memory).  A NaN logit counts as -inf and ORs 1 into *nan_flag.
template <int NPER>
__device__ __forceinline__ void route_tokens(const Fwd& p, const RouteSmem& r, int* nan_flag, int t0, int tstep) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, k = p.k, T = p.T;
  for (int t = t0; t < T; t += tstep) {
    float v[NPER];
    bool taken[NPER];
    bool nan_seen = false;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      const int e = lane + 32 * i;
      float z = -INFINITY;
      if (e < E) {
        z = p.logits[static_cast<size_t>(t) * E + e];
        if (isnan(z)) { nan_seen = true; z = -INFINITY; }
      }
      v[i] = z;
      taken[i] = (e >= E);
    }
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) atomicOr(nan_flag, 1);
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPER; ++i) m = fmaxf(m, v[i]);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NPER; ++i)
      if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    float wsum = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (!taken[i] && better(v[i], lane + 32 * i, bv, bi)) { bv = v[i]; bi = lane + 32 * i; }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (lane + 32 * i == bi) taken[i] = true;
      const float wj = expf(bv - m) / s;
      wsum += wj;
      if (lane == 0) {
        r.idx[t * k + j] = bi;
        r.w[t * k + j] = wj;
      }
    }
    __syncwarp();
    if (p.renorm)
      for (int j = lane; j < k; j += 32) r.w[t * k + j] /= wsum;
  }
}

// Routing of a decode batch into one CTA's shared memory: top-k and weights,
// counts, offsets, the active experts (in expert order and by gate_up cost,
// largest first), perm / inv.  Needs T*k <= kRouteSmemMaxPairs.  A NaN logit
// sets *nan_flag (shared memory); the caller raises the status bit.
__device__ __forceinline__ void route_local(const Fwd& p, const RouteSmem& r, int* nan_flag,
                                            int tok_cost) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int E = p.E, k = p.k, T = p.T;
  // each thread's share of the gate_up bitwidths: loads issued first, stored
  // after the tokens are routed, so their latency overlaps the logits'
  constexpr int kQPer = (kMaxE + 31) / 32;
  int qv[kQPer];
  const int nthr = blockDim.x;
#pragma unroll
  for (int j = 0; j < kQPer; ++j) {
    const int e = threadIdx.x + j * nthr;
    qv[j] = e < E ? p.desc[desc_index(p.layer, e, PW_KIND_GATE_UP, E)].q : 0;
  }
  for (int e = threadIdx.x; e < E; e += nthr) r.cnt[e] = 0;
  // every CTA of the fused layer routes the whole batch on its own (a few
  // hundred logits), so no CTA waits for another's results
  if (E <= 32) route_tokens<1>(p, r, nan_flag, warp, nwarp);
  else if (E <= 64) route_tokens<2>(p, r, nan_flag, warp, nwarp);
  else if (E <= 128) route_tokens<4>(p, r, nan_flag, warp, nwarp);
  else route_tokens<8>(p, r, nan_flag, warp, nwarp);
#pragma unroll
  for (int j = 0; j < kQPer; ++j) {
    const int e = threadIdx.x + j * nthr;
    if (e < E) r.qgu[e] = qv[j];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) atomicAdd(&r.cnt[r.idx[i]], 1);
  __syncthreads();
  if (threadIdx.x < 32) {   // warp-level exclusive scan of counts and of the active flags
    int run = 0, na = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + threadIdx.x;
      const int c = e < E ? r.cnt[e] : 0;
      int incl = c, actv = c > 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const int a = __shfl_up_sync(0xffffffffu, actv, o);
        if (threadIdx.x >= o) { incl += v; actv += a; }
      }
      if (e < E) {
        r.off[e] = run + incl - c;
        if (c) r.act[1 + na + actv - 1] = e;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      na += __shfl_sync(0xffffffffu, actv, 31);
    }
    if (threadIdx.x == 0) {
      r.off[E] = run;
      r.act[0] = na;
      r.lpt[0] = na;
    }
  }
  __syncthreads();
  if (T <= 16) {
    // small batches: one thread per pair; its place among the expert's pairs is
    // the number of earlier tokens routed to the same expert (a token's top-k
    // experts are distinct)
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
      const int t = i / k, e = r.idx[i];
      int rank = 0;
      for (int i2 = 0; i2 < t * k; ++i2) rank += (r.idx[i2] == e);
      const int pos = r.off[e] + rank;
      r.perm[pos] = i;
      r.inv[i] = pos;
    }
  } else {
    for (int e = warp; e < E; e += nwarp) {
      int run = 0;
      for (int base = 0; base < T; base += 32) {
        const int t = base + lane;
        int jsel = -1;
        if (t < T)
          for (int j = 0; j < k; ++j)
            if (r.idx[t * k + j] == e) jsel = j;
        const unsigned mask = __ballot_sync(0xffffffffu, jsel >= 0);
        if (jsel >= 0) {
          const int pos = r.off[e] + run + __popc(mask & ((1u << lane) - 1u));
          r.perm[pos] = t * k + jsel;
          r.inv[t * k + jsel] = pos;
        }
        run += __popc(mask);
      }
    }
  }
  // active experts by gate_up cost, largest first (ties keep expert order)
  const int na = r.act[0];
  for (int a = threadIdx.x; a < na; a += blockDim.x) {
    const int ea = r.act[1 + a];
    const int ca = (r.qgu[ea] + 2) * ((r.cnt[ea] + tok_cost - 1) / tok_cost);
    int rank = 0;
    for (int b = 0; b < na; ++b) {
      const int eb = r.act[1 + b];
      const int cb = (r.qgu[eb] + 2) * ((r.cnt[eb] + tok_cost - 1) / tok_cost);
      rank += (cb > ca) || (cb == ca && b < a);
    }
    r.lpt[1 + rank] = ea;
  }
  __syncthreads();
}

// Routing statistics, a by-product of the routing step (the runtime planner's
// routing-mass input): for each expert e, the batch mass
// M_e = (1/T) * sum of the routing weights of the pairs routed to e, and
// stats[layer][e] <- (1 - alpha) * stats[layer][e] + alpha * M_e.  One CTA; a warp
// per expert sums its pairs (expert order from the permutation) in a fixed
// order, so the result is the same on every run.  perm / w / off may live in
// global or shared memory; the caller synchronises the block before and after.
__device__ __forceinline__ void update_route_stats(const Fwd& p, const int* perm, const float* w,
                                                   const int* off) {
  if (!p.stats || p.T <= 0) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  float* m = p.stats + static_cast<size_t>(p.layer) * p.E;
  const float a = p.stats_alpha, invT = 1.f / static_cast<float>(p.T);
  for (int e = warp; e < p.E; e += nwarp) {
    float s = 0.f;
    for (int pos = off[e] + lane; pos < off[e + 1]; pos += 32) s += w[perm[pos]];
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) m[e] = (1.f - a) * m[e] + a * (s * invT);
  }
}

// out[t][r] = residual[t][r] + sum_j w[t][j] * y(t, j)[r] for r in [r0, r1) and
// t in [t0, t1), slots added in order j = 0..k-1 (deterministic), rounded once.
// w / inv may live in global or shared memory.
__device__ __forceinline__ void combine_rows(const Fwd& p, const float* w, const int* inv, int r0,
                                             int r1, int t0, int t1, int tid, int nthr) {
  const int n = r1 - r0;
  for (int q = tid; q < (t1 - t0) * n; q += nthr) {
    const int t = t0 + q / n, r = r0 + q % n;
    const float base = p.residual ? __half2float(p.residual[static_cast<size_t>(t) * p.H + r]) : 0.f;
    float mix = 0.f;
    for (int j = 0; j < p.k; ++j) {
      const int pos = inv[t * p.k + j];
      if (!PW_BOUNDS(p, pos >= 0 && pos < p.T * p.k, true)) continue;
      mix = fmaf(w[t * p.k + j], __ldcg(p.y + static_cast<size_t>(pos) * p.H + r), mix);   // L2: written by other SMs
    }
    p.out[static_cast<size_t>(t) * p.H + r] = __float2half_rn(base + mix);
  }
}

}  // namespace pw
