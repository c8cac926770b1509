// Kernels of the fused APL MoE layer (sm_103a).
//
// Source: PagedWeight technical summary, core components section 3 ("Fused
// Mixed-Precision Kernel": a custom kernel that reads APL bit-planes and
// lookup tables directly, with a different bitwidth per linear block inside
// one fused operation), over the MoE layer of the problem statement (a subset
// of experts per token).
//
// Pipeline of one forward pass, all on the caller's stream:
//   k_route          top-k softmax routing, one warp per token over the grid;
//   k_permute        one CTA: stable counting sort of the (token, slot) pairs
//                    by expert, offsets, active list;
//   gate_up          per active expert: dequantised gate/up rows . x, then
//                    h = silu(gate) * up (fp16);
//   down             per active expert: dequantised down rows . h (fp32 y);
//   k_combine        out[t] = residual[t] + sum_j w[t][j] * y(t, j) (fp16).
// The committed bitwidth of every block is read on the device from the page
// table's descriptor, so a commit needs no recompile.

#include <cuda_fp16.h>
#include <atomic>
#include <cstdint>

#include "pw_route.cuh"

namespace pw {

// ------------------------------------------------------------------ commit

__global__ void k_commit(BlockDesc* dst, BlockDesc v) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *dst = v;
}

cudaError_t launch_commit(BlockDesc* dst, const BlockDesc& value, cudaStream_t s) {
  k_commit<<<1, 32, 0, s>>>(dst, value);
  return cudaGetLastError();
}

// Many descriptors in one launch: they travel in the kernel's parameter block
// (under the 32 KB limit), one warp per descriptor, one 4-byte word per lane.
__global__ void __launch_bounds__(32) k_commit_batch(BlockDesc* table, CommitBatch b) {
  const int i = blockIdx.x;
  if (i >= b.n) return;
  reinterpret_cast<uint32_t*>(table + b.index[i])[threadIdx.x] = b.words[i][threadIdx.x];
}

cudaError_t launch_commit_batch(BlockDesc* table, const CommitBatch& b, cudaStream_t s) {
  if (b.n <= 0) return cudaSuccess;
  k_commit_batch<<<b.n, 32, 0, s>>>(table, b);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ routing + permutation

// Routing of a large batch: one warp per token over the whole grid, results
// into the workspace (idx, w).  The status word was cleared before the launch;
// a NaN logit ORs PW_STATUS_NAN_LOGIT into it.
constexpr int kRouteWarps = 8;
template <int NPER>
__global__ void __launch_bounds__(kRouteWarps * 32) k_route(Fwd p) {
  static_assert(PW_STATUS_NAN_LOGIT == 1, "route_tokens ORs 1");
  RouteSmem r{};
  r.idx = p.idx;
  r.w = p.w;
  const int gw = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  route_tokens<NPER>(p, r, reinterpret_cast<int*>(p.status), gw, gridDim.x * kRouteWarps);
}

// Counts, offsets, perm / inv of the routed pairs (one CTA), then the routing
// statistics.
constexpr int kPermuteThreads = 1024;
__global__ void __launch_bounds__(kPermuteThreads) k_permute(Fwd p) {
  __shared__ int s_c[kPermuteThreads / 32][kMaxE];
  __shared__ int s_off[kMaxE + 1];
  permute_block(p, s_c, s_off);
  if (p.stats) {
    __syncthreads();
    update_route_stats(p, p.perm, p.w, p.offsets);
  }
}

// ------------------------------------------------------------------ combine

__global__ void k_combine(Fwd p) {
  const int r0 = blockIdx.x * 256, t0 = blockIdx.y * 16;
  combine_rows(p, p.w, p.inv, r0, min(r0 + 256, p.H), t0, min(t0 + 16, p.T), threadIdx.x, blockDim.x);
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
  p.sync = reinterpret_cast<unsigned long long*>(ws + a.lay.sync);
  p.hh = reinterpret_cast<__half*>(ws + a.lay.hh);
  p.xp = reinterpret_cast<__half*>(ws + a.lay.xp);
  p.y = reinterpret_cast<float*>(ws + a.lay.y);
  p.y_part = reinterpret_cast<float*>(ws + a.lay.y_part);
  p.ksplit = down_splits(a.H, a.I);
  p.stats = a.stats;
  p.stats_alpha = a.stats_alpha;
  return p;
}

static inline void mark(const ForwardArgs& a, int i, cudaStream_t s) {
  if (a.prof[i]) cudaEventRecord(a.prof[i], s);
}

// Forward counter of this process: each forward's tag is 0xA5 above it (the
// fused forward's ticket word, pw_device.cuh).
static std::atomic<uint32_t> g_forwards{0};

cudaError_t launch_forward(const ForwardArgs& a, cudaStream_t s) {
  Fwd p = make_fwd(a);
  p.tag = ((0xA5ull << 32) | ++g_forwards) << kTagShift;
  mark(a, 0, s);
  if (fused_batch(p.T, p.k)) {
    const cudaError_t e = launch_layer_fused(p, s);
    for (int i = 1; i < 5; ++i) mark(a, i, s);
    return e;
  }
  cudaError_t e0 = cudaMemsetAsync(p.status, 0, sizeof(uint32_t), s);
  if (e0 != cudaSuccess) return e0;
  const dim3 rgrid((p.T + kRouteWarps - 1) / kRouteWarps);
  if (p.E <= 32) k_route<1><<<rgrid, kRouteWarps * 32, 0, s>>>(p);
  else if (p.E <= 64) k_route<2><<<rgrid, kRouteWarps * 32, 0, s>>>(p);
  else if (p.E <= 128) k_route<4><<<rgrid, kRouteWarps * 32, 0, s>>>(p);
  else k_route<8><<<rgrid, kRouteWarps * 32, 0, s>>>(p);
  k_permute<<<1, kPermuteThreads, 0, s>>>(p);
  mark(a, 1, s);
  cudaError_t e = launch_prefill(p, PW_KIND_GATE_UP, s);
  if (e != cudaSuccess) return e;
  mark(a, 2, s);
  e = launch_prefill(p, PW_KIND_DOWN, s);
  if (e != cudaSuccess) return e;
  mark(a, 3, s);
  k_combine<<<dim3((p.H + 255) / 256, (p.T + 15) / 16), 256, 0, s>>>(p);
  mark(a, 4, s);
  return cudaGetLastError();
}

}  // namespace pw
