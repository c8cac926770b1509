// Kernels of the fused APL MoE layer (sm_103a).
//
// Source: PagedWeight technical summary, core components section 3 ("Fused
// Mixed-Precision Kernel": a custom kernel that reads APL bit-planes and
// lookup tables directly, with a different bitwidth per linear block inside
// one fused operation), over the MoE layer of the problem statement (a subset
// of experts per token).
//
// Pipeline of one forward pass, all on the caller's stream:
//   k_route_permute  one CTA: top-k softmax routing per token, stable counting
//                    sort of the (token, slot) pairs by expert, active list;
//   gate_up          per active expert: dequantised gate/up rows . x, then
//                    h = silu(gate) * up (fp16);
//   down             per active expert: dequantised down rows . h (fp32 y);
//   k_combine        out[t] = residual[t] + sum_j w[t][j] * y(t, j) (fp16).
// The committed bitwidth of every block is read on the device from the page
// table's descriptor, so a commit needs no recompile.

#include <cuda_fp16.h>
#include <cstdint>

#include "pw_device.cuh"

namespace pw {

// ------------------------------------------------------------------ commit

__global__ void k_commit(BlockDesc* dst, BlockDesc v) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *dst = v;
}

cudaError_t launch_commit(BlockDesc* dst, const BlockDesc& value, cudaStream_t s) {
  k_commit<<<1, 32, 0, s>>>(dst, value);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ routing + permutation

constexpr int kRouteThreads = 1024;
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

constexpr int kConvertInRoute = 64;   // larger batches convert x in their own kernel

__global__ void k_convert_x(Fwd p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < p.T * p.H / 8) convert8(p, i);
}

// One CTA for the whole batch.  Phase 1: warp per token, top-k over the fp32
// logits and softmax weights.  Phase 2: per-expert counts and offsets.
// Phase 3: warp per expert, ballot ranks give the stable (expert, token) order.
__global__ void __launch_bounds__(kRouteThreads) k_route_permute(Fwd p) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int E = p.E, k = p.k, T = p.T;
  if (threadIdx.x < 4) p.status[threadIdx.x] = 0u;   // status word and work-queue counters
  if (T <= kConvertInRoute)
    for (int i = threadIdx.x; i < T * p.H / 8; i += blockDim.x) convert8(p, i);

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
  if (threadIdx.x == 0) {
    int run = 0, na = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = run;
      run += s_cnt[e];
      if (s_cnt[e]) p.active[1 + na++] = e;
    }
    s_off[E] = run;
    p.active[0] = na;
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

// ------------------------------------------------------------------ combine

__global__ void k_combine(Fwd p) {
  const int t = blockIdx.y;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= p.H) return;
  const float base = p.residual ? __half2float(p.residual[static_cast<size_t>(t) * p.H + r]) : 0.f;
  float mix = 0.f;
  for (int j = 0; j < p.k; ++j) {
    const int pos = p.inv[t * p.k + j];
    mix = fmaf(p.w[t * p.k + j], p.y[static_cast<size_t>(pos) * p.H + r], mix);
  }
  p.out[static_cast<size_t>(t) * p.H + r] = __float2half_rn(base + mix);
}

// ------------------------------------------------------------------ launcher

static Fwd make_fwd(const ForwardArgs& a) {
  Fwd p{};
  p.desc = a.desc;
  p.layer = a.layer;
  p.E = a.E;
  p.H = a.H;
  p.I = a.I;
  p.T = a.T;
  p.k = a.top_k;
  p.renorm = a.renorm;
  p.x = reinterpret_cast<const __half*>(a.x);
  p.logits = a.logits;
  p.residual = reinterpret_cast<const __half*>(a.residual);
  p.out = reinterpret_cast<__half*>(a.out);
  p.user_idx = a.user_idx;
  p.user_w = a.user_w;
  p.user_offsets = a.user_offsets;
  p.user_perm = a.user_perm;
  unsigned char* ws = a.ws;
  p.status = reinterpret_cast<uint32_t*>(ws + a.lay.status);
  p.idx = reinterpret_cast<int32_t*>(ws + a.lay.topk_idx);
  p.w = reinterpret_cast<float*>(ws + a.lay.topk_w);
  p.counts = reinterpret_cast<int32_t*>(ws + a.lay.counts);
  p.offsets = reinterpret_cast<int32_t*>(ws + a.lay.offsets);
  p.perm = reinterpret_cast<int32_t*>(ws + a.lay.perm);
  p.inv = reinterpret_cast<int32_t*>(ws + a.lay.inv);
  p.active = reinterpret_cast<int32_t*>(ws + a.lay.active);
  p.xf = reinterpret_cast<float*>(ws + a.lay.xf);
  p.hf = reinterpret_cast<float*>(ws + a.lay.hf);
  p.y = reinterpret_cast<float*>(ws + a.lay.y);
  return p;
}

static inline void mark(const ForwardArgs& a, int i, cudaStream_t s) {
  if (a.prof[i]) cudaEventRecord(a.prof[i], s);
}

cudaError_t launch_forward(const ForwardArgs& a, cudaStream_t s) {
  const Fwd p = make_fwd(a);
  mark(a, 0, s);
  if (p.T > kConvertInRoute) {
    const int n8 = p.T * p.H / 8;
    k_convert_x<<<(n8 + 255) / 256, 256, 0, s>>>(p);
  }
  k_route_permute<<<1, kRouteThreads, 0, s>>>(p);
  mark(a, 1, s);
  cudaError_t e = launch_decode(p, PW_KIND_GATE_UP, s);
  if (e != cudaSuccess) return e;
  mark(a, 2, s);
  e = launch_decode(p, PW_KIND_DOWN, s);
  if (e != cudaSuccess) return e;
  mark(a, 3, s);
  k_combine<<<dim3((p.H + 255) / 256, p.T), 256, 0, s>>>(p);
  mark(a, 4, s);
  return cudaGetLastError();
}

}  // namespace pw
