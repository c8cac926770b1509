// Routing + permutation shared by the kernels that run it (device code).
//
// Source: PagedWeight technical summary, problem statement (an MoE activates a
// subset of experts per token); the top-k softmax and the token -> expert
// gather with per-expert offsets are the routing steps of the fused layer.
#pragma once

#include "pw_device.cuh"

namespace pw {

constexpr int kMaxE = 256;
constexpr int kPerLane = kMaxE / 32;

// Order of the top-k: larger logit first, ties to the lower expert index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// x (fp16) -> xf (fp32), 8 elements per call.
__device__ __forceinline__ void convert8(const Fwd& p, int i) {
  const uint4 raw = reinterpret_cast<const uint4*>(p.x)[i];
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
  float4 a, b;
  float2 f;
  f = __half22float2(h2[0]); a.x = f.x; a.y = f.y;
  f = __half22float2(h2[1]); a.z = f.x; a.w = f.y;
  f = __half22float2(h2[2]); b.x = f.x; b.y = f.y;
  f = __half22float2(h2[3]); b.z = f.x; b.w = f.y;
  reinterpret_cast<float4*>(p.xf)[2 * i] = a;
  reinterpret_cast<float4*>(p.xf)[2 * i + 1] = b;
}

// Routing and permutation of the whole batch by one CTA (any block size that is
// a multiple of 32).  Phase 1: warp per token, top-k over the fp32 logits and
// softmax weights.  Phase 2: per-expert counts and offsets.  Phase 3: warp per
// expert, ballot ranks give the stable (expert, token) order.  s_cnt / s_off:
// shared scratch of kMaxE and kMaxE + 1 ints.  The caller resets the status word.
__device__ __forceinline__ void route_permute_block(const Fwd& p, int* s_cnt, int* s_off) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int E = p.E, k = p.k, T = p.T;

  for (int t = warp; t < T; t += nwarp) {
    float v[kPerLane];
    bool taken[kPerLane];
    bool nan_seen = false;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      float z = -INFINITY;
      if (e < E) {
        z = p.logits[static_cast<size_t>(t) * E + e];
        if (isnan(z)) { nan_seen = true; z = -INFINITY; }
      }
      v[i] = z;
      taken[i] = (e >= E);
    }
    if (__any_sync(0xffffffffu, nan_seen) && lane == 0) atomicOr(p.status, PW_STATUS_NAN_LOGIT);
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) m = fmaxf(m, v[i]);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
      if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    float wsum = 0.f, wsel = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i)
        if (!taken[i] && better(v[i], lane + 32 * i, bv, bi)) { bv = v[i]; bi = lane + 32 * i; }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
#pragma unroll
      for (int i = 0; i < kPerLane; ++i)
        if (lane + 32 * i == bi) taken[i] = true;
      const float wj = expf(bv - m) / s;
      wsum += wj;
      if ((j & 31) == lane) wsel = wj;
      if (lane == 0) p.idx[t * k + j] = bi;
      if ((j & 31) == 31 || j == k - 1) {   // flush slots [j & ~31, j]
        const int js = (j & ~31) + lane;
        if (js <= j) p.w[t * k + js] = wsel;
      }
    }
    if (p.renorm) {
      __syncwarp();
      for (int j = lane; j < k; j += 32) p.w[t * k + j] /= wsum;
    }
  }
  __syncthreads();

  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) atomicAdd(&s_cnt[p.idx[i]], 1);
  __syncthreads();
  if (threadIdx.x < 32) {   // warp-level exclusive scan of counts and of the active flags
    int run = 0, na = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + threadIdx.x;
      const int c = e < E ? s_cnt[e] : 0;
      int incl = c, act = c > 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        const int a = __shfl_up_sync(0xffffffffu, act, o);
        if (threadIdx.x >= o) { incl += v; act += a; }
      }
      if (e < E) {
        s_off[e] = run + incl - c;
        if (c) p.active[1 + na + act - 1] = e;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
      na += __shfl_sync(0xffffffffu, act, 31);
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
    if (e < E) p.counts[e] = s_cnt[e];
  }
  for (int e = warp; e < E; e += nwarp) {
    int run = 0;
    for (int base = 0; base < T; base += 32) {
      const int t = base + lane;
      int jsel = -1;
      if (t < T)
        for (int j = 0; j < k; ++j)
          if (p.idx[t * k + j] == e) jsel = j;
      const unsigned mask = __ballot_sync(0xffffffffu, jsel >= 0);
      if (jsel >= 0) {
        const int pos = s_off[e] + run + __popc(mask & ((1u << lane) - 1u));
        p.perm[pos] = t * k + jsel;
        p.inv[t * k + jsel] = pos;
        if (p.user_perm) p.user_perm[pos] = t * k + jsel;
      }
      run += __popc(mask);
    }
  }
  if (p.user_idx || p.user_w)
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
      if (p.user_idx) p.user_idx[i] = p.idx[i];
      if (p.user_w) p.user_w[i] = p.w[i];
    }
}

// out[t][r] = residual[t][r] + sum_j w[t][j] * y(t, j)[r] for r in [r0, r1) and
// t in [t0, t1), slots added in order j = 0..k-1 (deterministic), rounded once.
__device__ __forceinline__ void combine_rows(const Fwd& p, int r0, int r1, int t0, int t1, int tid,
                                             int nthr) {
  const int n = r1 - r0;
  for (int q = tid; q < (t1 - t0) * n; q += nthr) {
    const int t = t0 + q / n, r = r0 + q % n;
    const float base = p.residual ? __half2float(p.residual[static_cast<size_t>(t) * p.H + r]) : 0.f;
    float mix = 0.f;
    for (int j = 0; j < p.k; ++j) {
      const int pos = p.inv[t * p.k + j];
      mix = fmaf(p.w[t * p.k + j], __ldcg(p.y + static_cast<size_t>(pos) * p.H + r), mix);   // L2: written by other SMs
    }
    p.out[static_cast<size_t>(t) * p.H + r] = __float2half_rn(base + mix);
  }
}

}  // namespace pw
