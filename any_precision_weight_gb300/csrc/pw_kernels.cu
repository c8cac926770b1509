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

#include "pw_internal.h"

namespace pw {

// ------------------------------------------------------------------ device params

struct Fwd {
  const BlockDesc* desc;
  int layer, E, H, I, T, k, renorm;
  const __half* x;
  const float* logits;
  const __half* residual;
  __half* out;
  int32_t* user_idx;
  float* user_w;
  int32_t* user_offsets;
  int32_t* user_perm;
  uint32_t* status;
  int32_t* idx;     // [T*k]
  float* w;         // [T*k]
  int32_t* counts;  // [E]
  int32_t* offsets; // [E+1]
  int32_t* perm;    // [T*k]
  int32_t* inv;     // [T*k]
  int32_t* active;  // [E+1]
  __half* h;        // [T*k][I]
  float* y;         // [T*k][H]
};

__device__ __forceinline__ const BlockDesc* block_desc(const Fwd& p, int e, int kind) {
  return p.desc + desc_index(p.layer, e, kind, p.E);
}

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

// One CTA for the whole batch.  Phase 1: warp per token, top-k over the fp32
// logits and softmax weights.  Phase 2: per-expert counts and offsets.
// Phase 3: warp per expert, ballot ranks give the stable (expert, token) order.
__global__ void __launch_bounds__(kRouteThreads) k_route_permute(Fwd p) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  const int E = p.E, k = p.k, T = p.T;
  if (threadIdx.x == 0) *p.status = 0u;

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

// ------------------------------------------------------------------ dequant GEMV (reference path)

constexpr int kGemvWarps = 8;
constexpr int kGemvTok = 8;      // tokens handled per pass over a row

// Dot products of one block row with up to kGemvTok input rows.
// Lane l handles plane words w = l, l+32, ...; element k = 32w + j takes the
// q-bit index assembled MSB first from the top q planes and looks up LUT_q.
__device__ __forceinline__ void row_dot(const BlockDesc& d, int row, const __half* const* xr, int nt,
                                        float* acc) {
  const int W = d.K >> 5;
  const int q = d.q;
  const uint16_t* lut = d.lut + (static_cast<size_t>(row) << q);
  for (int t = 0; t < kGemvTok; ++t) acc[t] = 0.f;
  for (int w = threadIdx.x & 31; w < W; w += 32) {
    uint32_t pw[PW_MAX_BITS];
#pragma unroll
    for (int pl = 0; pl < PW_MAX_BITS; ++pl)
      pw[pl] = (pl < q) ? __ldg(d.planes[pl] + static_cast<size_t>(row) * W + w) : 0u;
    for (int j = 0; j < 32; ++j) {
      uint32_t v = 0;
#pragma unroll
      for (int pl = 0; pl < PW_MAX_BITS; ++pl)
        if (pl < q) v = (v << 1) | ((pw[pl] >> j) & 1u);
      const float wt = __half2float(__ushort_as_half(__ldg(lut + v)));
      const int kk = 32 * w + j;
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t)
        if (t < nt) acc[t] = fmaf(wt, __half2float(xr[t][kk]), acc[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < kGemvTok; ++t)
#pragma unroll
    for (int o = 16; o; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
}

template <int kKind>
__global__ void __launch_bounds__(kGemvWarps * 32) k_gemv_ref(Fwd p) {
  const int e = blockIdx.y;
  const int cnt = p.counts[e];
  if (cnt == 0) return;
  const int off = p.offsets[e];
  const BlockDesc d = *block_desc(p, e, kKind);
  if (d.q < 1 || d.q > PW_MAX_BITS) {
    if (threadIdx.x == 0) atomicOr(p.status, PW_STATUS_BAD_DESC);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = (kKind == PW_KIND_GATE_UP) ? p.I : p.H;
  for (int r = blockIdx.x * kGemvWarps + warp; r < rows; r += gridDim.x * kGemvWarps) {
    for (int t0 = 0; t0 < cnt; t0 += kGemvTok) {
      const int nt = min(kGemvTok, cnt - t0);
      const __half* xr[kGemvTok];
#pragma unroll
      for (int t = 0; t < kGemvTok; ++t) {
        const int pos = off + t0 + min(t, nt - 1);
        xr[t] = (kKind == PW_KIND_GATE_UP) ? p.x + static_cast<size_t>(p.perm[pos] / p.k) * p.H
                                           : p.h + static_cast<size_t>(pos) * p.I;
      }
      if (kKind == PW_KIND_GATE_UP) {
        float g[kGemvTok], u[kGemvTok];
        row_dot(d, r, xr, nt, g);
        row_dot(d, p.I + r, xr, nt, u);
        if (lane < nt) {
          float gv = g[0], uv = u[0];
#pragma unroll
          for (int t = 1; t < kGemvTok; ++t)
            if (t == lane) { gv = g[t]; uv = u[t]; }
          const float hv = gv / (1.f + expf(-gv)) * uv;
          p.h[static_cast<size_t>(off + t0 + lane) * p.I + r] = __float2half_rn(hv);
        }
      } else {
        float a[kGemvTok];
        row_dot(d, r, xr, nt, a);
        if (lane < nt) {
          float av = a[0];
#pragma unroll
          for (int t = 1; t < kGemvTok; ++t)
            if (t == lane) av = a[t];
          p.y[static_cast<size_t>(off + t0 + lane) * p.H + r] = av;
        }
      }
    }
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
  p.h = reinterpret_cast<__half*>(ws + a.lay.h);
  p.y = reinterpret_cast<float*>(ws + a.lay.y);
  return p;
}

static inline void mark(const ForwardArgs& a, int i, cudaStream_t s) {
  if (a.prof[i]) cudaEventRecord(a.prof[i], s);
}

cudaError_t launch_forward(const ForwardArgs& a, cudaStream_t s) {
  const Fwd p = make_fwd(a);
  mark(a, 0, s);
  k_route_permute<<<1, kRouteThreads, 0, s>>>(p);
  mark(a, 1, s);
  const int gx_gu = (p.I + kGemvWarps - 1) / kGemvWarps;
  const int gx_dn = (p.H + kGemvWarps - 1) / kGemvWarps;
  k_gemv_ref<PW_KIND_GATE_UP><<<dim3(min(gx_gu, 1024), p.E), kGemvWarps * 32, 0, s>>>(p);
  mark(a, 2, s);
  k_gemv_ref<PW_KIND_DOWN><<<dim3(min(gx_dn, 1024), p.E), kGemvWarps * 32, 0, s>>>(p);
  mark(a, 3, s);
  k_combine<<<dim3((p.H + 255) / 256, p.T), 256, 0, s>>>(p);
  mark(a, 4, s);
  return cudaGetLastError();
}

}  // namespace pw
