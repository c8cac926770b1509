// Decode-sized dequantised GEMV of the fused APL MoE layer (sm_103a, CUDA cores).
//
// Source: PagedWeight technical summary, core components section 3 ("Fused
// Mixed-Precision Kernel": reads APL bit-planes and lookup tables directly,
// a different committed bitwidth per linear block within one fused operation).
//
// Decode batches give each active expert a handful of tokens, so these
// kernels stream each active block's q bit-planes and q-bit table from HBM
// exactly once and keep the tokens on chip.  Design:
//
//  * persistent CTAs (two per SM) pull (active expert, 32-row tile) items from
//    a device work queue, so the committed q of each block is read from the
//    page table on the device and the grid never depends on the routing;
//  * a tile is 32 rows x all of K; lane l of each of the 8 warps owns row l,
//    the warps split K; the 32 rows' tables sit in shared memory as fp32
//    [v][row], so the 32 lanes of a warp always hit 32 different banks,
//    whatever their indices (conflict-free lookups at every q);
//  * bit-planes are staged global->shared with cp.async in 16-word (512-k)
//    chunks, double buffered, with the 16-byte chunks XOR-swizzled by row;
//    tokens are staged the same way (fp32), two tokens per pass;
//  * per 32-bit plane word a lane turns the q plane words into 32 q-bit
//    indices with an 8x8 bit-matrix transpose done four bytes at a time (delta
//    swaps), then one byte permute per element forms the table address
//    (index * 256 + row * 4);
//  * products accumulate in fp32 with packed two-wide FMAs; the eight K-warps'
//    partial sums are added in a fixed order (deterministic results).
// gate_up tiles hold 16 gate rows and the 16 matching up rows and finish with
// h = silu(gate) * up rounded to fp16; down tiles hold 32 rows of y (fp32).

#include <cuda_fp16.h>
#include <cstdint>

#include "pw_route.cuh"

namespace pw {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;        // two CTAs per SM overlap each other's item start-up
constexpr int kRows = 32;            // rows per tile: lane l of every warp owns row l
constexpr int kKW = 8;               // K-warps: each warp takes 2 of a stage's 16 words per row
constexpr int kStageWords = 16;      // plane words per row per stage
constexpr int kStageK = kStageWords * 32;
constexpr int kTok = 2;              // tokens per pass over a tile
constexpr int kLutBytes = 256 * 64 * 4;   // [v][64 slots] fp32; slot = row (byte-permute addressing)
constexpr int kPlaneStageBytes = PW_MAX_BITS * kRows * kStageWords * 4;
constexpr int kXStageBytes = kTok * kStageK * 4;
constexpr int kRedBytes = kKW * kTok * kRows * 4;
constexpr int kSmemBytes = kLutBytes + 2 * kPlaneStageBytes + 2 * kXStageBytes + kRedBytes + 64;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// a = a + w * x, two lanes at a time (packed fp32 FMA).
__device__ __forceinline__ void ffma2(float& ax, float& ay, float wx, float wy, float xx, float xy) {
  asm("{\n\t.reg .b64 a, w, x;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 w, {%2, %3};\n\tmov.b64 x, {%4, %5};\n\t"
      "fma.rn.f32x2 a, w, x, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(ax), "+f"(ay)
      : "f"(wx), "f"(wy), "f"(xx), "f"(xy));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & ~m) | (b & m) in one three-input logic op.
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(d) : "r"(m), "r"(b), "r"(a));
  return d;
}
// Exchange the bits of `hi` selected by `mask` with the bits of `lo` selected
// by `mask << s`: two shifts and two logic ops.
__device__ __forceinline__ void delta_swap(uint32_t& lo, uint32_t& hi, int s, uint32_t mask) {
  const uint32_t nlo = bitsel(lo, hi << s, mask << s);
  const uint32_t nhi = bitsel(hi, lo >> s, mask);
  lo = nlo;
  hi = nhi;
}

// 8x8 bit transposes, four byte lanes at once.  Row r of the input holds plane
// (q-1-r) (zero for r >= q); after the three rounds, byte bb of o[r] is the
// q-bit index (plane 0 most significant) of element 8*bb + r.
__device__ __forceinline__ void planes_to_indices(uint32_t (&o)[8]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) delta_swap(o[r], o[r + 4], 4, 0x0F0F0F0Fu);
#pragma unroll
  for (int r = 0; r < 8; r += 4) {
    delta_swap(o[r], o[r + 2], 2, 0x33333333u);
    delta_swap(o[r + 1], o[r + 3], 2, 0x33333333u);
  }
#pragma unroll
  for (int r = 0; r < 8; r += 2) delta_swap(o[r], o[r + 1], 1, 0x55555555u);
}

struct Item {
  int expert, tile, n, off;
};

// Global row of tile row i: gate_up tiles are 16 gate rows + the 16 matching
// up rows; down tiles are 32 consecutive rows.  Returns -1 past the block.
template <int KIND>
__device__ __forceinline__ int global_row(const Fwd& p, int tile, int i) {
  if (KIND == PW_KIND_GATE_UP) {
    const int r = tile * 16 + (i & 15);
    if (r >= p.I) return -1;
    return (i < 16) ? r : p.I + r;
  } else {
    const int r = tile * kRows + i;
    return (r < p.H) ? r : -1;
  }
}

template <int KIND>
__device__ __forceinline__ const float* token_row(const Fwd& p, int pos, int K) {
  if (KIND == PW_KIND_GATE_UP) return p.xf + static_cast<size_t>(p.perm[pos] / p.k) * K;
  return p.hf + static_cast<size_t>(pos) * K;
}

template <int KIND>
__device__ void run_tile(const Fwd& p, const BlockDesc& d, const Item& it, unsigned char* smem) {
  float* lut_s = reinterpret_cast<float*>(smem);
  uint32_t* pl_s = reinterpret_cast<uint32_t*>(smem + kLutBytes);
  float* x_s = reinterpret_cast<float*>(smem + kLutBytes + 2 * kPlaneStageBytes);
  float* red_s = reinterpret_cast<float*>(smem + kLutBytes + 2 * kPlaneStageBytes + 2 * kXStageBytes);

  const int tid = threadIdx.x, lane = tid & 31, kw = tid >> 5;
  const int K = d.K, W = K >> 5;
  const int Q = d.q, V = 1 << Q;
  const int nchunk = (W + kStageWords - 1) / kStageWords;

  // plane staging: threads 0..127 and 128..255 each cover the 32 rows x four
  // 16-byte chunks, taking even and odd planes; chunks are XOR-swizzled by row
  const int fr = (tid & 127) >> 2, fc = tid & 3, fpl = tid >> 7;
  const int fgr = global_row<KIND>(p, it.tile, fr);
  const int fdst = fr * kStageWords + ((fc ^ ((fr >> 1) & 3)) * 4);
  const size_t fsrc = (fgr >= 0 ? static_cast<size_t>(fgr) * W : 0) + fc * 4;

  const int row = lane;
  const uint32_t laneoff = static_cast<uint32_t>(row) * 4u;
  const int rsw = (((kw >> 1) ^ ((row >> 1) & 3)) * 4) + (kw & 1) * 2;
  const unsigned char* lut_bytes = reinterpret_cast<const unsigned char*>(lut_s);

  for (int t0 = 0; t0 < it.n; t0 += kTok) {
    const int nt = min(kTok, it.n - t0);
    const int xt = tid >> 7, xc = tid & 127;        // token staging: thread -> (token, 16 B)
    const float* trow = (xt < nt) ? token_row<KIND>(p, it.off + t0 + xt, K) : nullptr;

    auto fill = [&](int c, int s) {
      const int wsrc = c * kStageWords + fc * 4;
      if (fgr >= 0 && wsrc < W) {
        uint32_t* dst = pl_s + s * (kPlaneStageBytes / 4) + fdst;
#pragma unroll
        for (int j = 0; j < PW_MAX_BITS / 2; ++j) {   // static indices keep the descriptor in registers
          const int pl = 2 * j + fpl;
          const uint32_t* src = fpl ? d.planes[2 * j + 1] : d.planes[2 * j];
          if (pl < Q) cp_async16(dst + pl * kRows * kStageWords, src + fsrc + c * kStageWords);
        }
      }
      const int kk = c * kStageK + xc * 4;
      if (trow && kk < K) cp_async16(x_s + s * (kXStageBytes / 4) + xt * kStageK + xc * 4, trow + kk);
      cp_commit();
    };

    fill(0, 0);
    if (t0 == 0) {
      // this tile's tables: LUT_q[row][v] fp16 -> lut_s[v][row] fp32 (overlaps stage 0)
      const int i = tid & 31;
      const int gr = global_row<KIND>(p, it.tile, i);
      for (int vc = tid >> 5; vc * 8 < V; vc += kThreads / 32) {
        float f[8];
        if (gr >= 0) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(d.lut + static_cast<size_t>(gr) * V + vc * 8));
          const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 ff = __half22float2(h2[e]);
            f[2 * e] = ff.x;
            f[2 * e + 1] = ff.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) lut_s[(vc * 8 + e) * 64 + i] = f[e];
      }
    }

    // four independent accumulator pairs per token keep the FMA chains short
    float ax[kTok][4], ay[kTok][4];
#pragma unroll
    for (int t = 0; t < kTok; ++t)
#pragma unroll
      for (int m = 0; m < 4; ++m) ax[t][m] = ay[t][m] = 0.f;

    // one barrier per stage: it publishes stage c and proves every warp is done
    // with stage c-1, whose buffer the fill for stage c+1 then reuses
    for (int c = 0; c < nchunk; ++c) {
      const int s = c & 1;
      cp_wait<0>();
      __syncthreads();
      if (c + 1 < nchunk) fill(c + 1, s ^ 1);

      const int wbase = c * kStageWords + kw * 2;
      const int nw = min(2, W - wbase);
      if (nw > 0) {
        const uint32_t* ps = pl_s + s * (kPlaneStageBytes / 4) + row * kStageWords + rsw;
        uint2 pv[PW_MAX_BITS];
#pragma unroll
        for (int pl = 0; pl < PW_MAX_BITS; ++pl)   // pv[r] = plane (q-1-r)
          pv[pl] = (pl < Q) ? *reinterpret_cast<const uint2*>(ps + (Q - 1 - pl) * kRows * kStageWords)
                            : make_uint2(0u, 0u);
        const float* xs = x_s + s * (kXStageBytes / 4) + kw * 64;
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          if (wi < nw) {
            uint32_t o[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) o[r] = wi == 0 ? pv[r].x : pv[r].y;
            planes_to_indices(o);
            float wv[32];
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
#pragma unroll
              for (int r = 0; r < 8; ++r) {
                const uint32_t a = prmt(o[r], laneoff, 0x5504u | (static_cast<uint32_t>(bb) << 4));
                wv[8 * bb + r] = *reinterpret_cast<const float*>(lut_bytes + a);
              }
#pragma unroll
            for (int t = 0; t < kTok; ++t) {
              if (t < nt) {
                const float4* xr = reinterpret_cast<const float4*>(xs + t * kStageK + wi * 32);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                  const float4 xv = xr[j4];
                  const int m0 = (2 * j4) & 3, m1 = (2 * j4 + 1) & 3;
                  ffma2(ax[t][m0], ay[t][m0], wv[4 * j4], wv[4 * j4 + 1], xv.x, xv.y);
                  ffma2(ax[t][m1], ay[t][m1], wv[4 * j4 + 2], wv[4 * j4 + 3], xv.z, xv.w);
                }
              }
            }
          }
        }
      }
    }

    // ---- partial sums of the eight K-warps, added in a fixed order
#pragma unroll
    for (int t = 0; t < kTok; ++t)
      if (t < nt)
        red_s[(kw * kTok + t) * kRows + row] =
            ((ax[t][0] + ay[t][0]) + (ax[t][1] + ay[t][1])) + ((ax[t][2] + ay[t][2]) + (ax[t][3] + ay[t][3]));
    __syncthreads();
    if (KIND == PW_KIND_GATE_UP) {
      if (tid < nt * 16) {
        const int t = tid >> 4, i = tid & 15;
        const int r = it.tile * 16 + i;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < kKW; ++w8) {
          g += red_s[(w8 * kTok + t) * kRows + i];
          u += red_s[(w8 * kTok + t) * kRows + 16 + i];
        }
        if (r < p.I) {
          const float hv = g / (1.f + expf(-g)) * u;
          p.hf[static_cast<size_t>(it.off + t0 + t) * p.I + r] = __half2float(__float2half_rn(hv));
        }
      }
    } else {
      if (tid < nt * kRows) {
        const int t = tid >> 5, i = tid & 31;
        const int r = it.tile * kRows + i;
        float yv = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < kKW; ++w8) yv += red_s[(w8 * kTok + t) * kRows + i];
        if (r < p.H) p.y[static_cast<size_t>(it.off + t0 + t) * p.H + r] = yv;
      }
    }
    __syncthreads();
  }
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_decode(Fwd p) {
  extern __shared__ __align__(128) unsigned char smem[];
  int* s_item = reinterpret_cast<int*>(smem + kSmemBytes - 64);
  const int tiles = (KIND == PW_KIND_GATE_UP) ? p.I / 16 : (p.H + kRows - 1) / kRows;
  const int nact = p.active[0];
  const int total = nact * tiles;
  int* ctr = reinterpret_cast<int*>(p.status) + (KIND == PW_KIND_GATE_UP ? kCtrGateUp : kCtrDown);
  if (threadIdx.x == 0) s_item[0] = atomicAdd(ctr, 1);
  __syncthreads();
  for (int slot = 0;; slot ^= 1) {
    const int item = s_item[slot];
    if (item >= total) break;
    // claim the next item now; it is read after this item's barriers
    if (threadIdx.x == 0) s_item[slot ^ 1] = atomicAdd(ctr, 1);
    Item it;
    it.expert = p.active[1 + item / tiles];
    it.tile = item % tiles;
    it.n = p.counts[it.expert];
    it.off = p.offsets[it.expert];
    const BlockDesc d = *block_desc(p, it.expert, KIND);
    if (d.q >= 1 && d.q <= PW_MAX_BITS && d.K == (KIND == PW_KIND_GATE_UP ? p.H : p.I)) {
      run_tile<KIND>(p, d, it, smem);
    } else if (threadIdx.x == 0) {
      atomicOr(p.status, PW_STATUS_BAD_DESC);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ fused layer

constexpr int kSpinLimit = 1 << 22;   // ~0.3 s of polling before a wait gives up

__device__ __forceinline__ int ld_acquire(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* ptr, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
// Bounded wait (one thread): true once *ptr == want, false when the limit runs out.
__device__ bool wait_eq(const int* ptr, int want) {
  for (int i = 0; i < kSpinLimit; ++i) {
    if (ld_acquire(ptr) == want) return true;
    __nanosleep(64);
  }
  return false;
}

// Active experts ordered by the cost of their gate_up work, largest first
// (longest-processing-time order keeps the tail of the work queue short);
// ties keep expert order.  Thread a ranks active expert a (block-wide).
__device__ void build_lpt(const Fwd& p, int* s_cost) {
  const int na = p.active[0];
  for (int a = threadIdx.x; a < na; a += blockDim.x) {
    const int e = p.active[1 + a];
    s_cost[a] = (block_desc(p, e, PW_KIND_GATE_UP)->q + 2) * ((p.counts[e] + kTok - 1) / kTok);
  }
  __syncthreads();
  for (int a = threadIdx.x; a < na; a += blockDim.x) {
    const int c = s_cost[a];
    int rank = 0;
    for (int b = 0; b < na; ++b) rank += (s_cost[b] > c) || (s_cost[b] == c && b < a);
    p.act_lpt[1 + rank] = p.active[1 + a];
  }
  if (threadIdx.x == 0) p.act_lpt[0] = na;
}

// One persistent cooperative launch for the whole decode layer.
// CTA 0 routes the batch and publishes a ready epoch; then every CTA takes
// items from one queue: first all (expert, gate_up tile) items, then all
// (expert, down tile) items.  A down item first waits until its expert's
// gate_up tiles are all done; the last down item of a 64-row tile of H (over
// all active experts) combines that tile's output rows.  Every wait is bounded
// and reports PW_STATUS_TIMEOUT instead of hanging.
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_layer(Fwd p) {
  extern __shared__ __align__(128) unsigned char smem[];
  int* s_int = reinterpret_cast<int*>(smem + kSmemBytes - 64);
  const int tiles_gu = p.I / 16, tiles_dn = (p.H + kRows - 1) / kRows;
  int* queue = p.sync + 1;
  int* expert_done = p.sync + 2;
  int* tile_done = p.sync + 2 + p.E;

  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) p.status[0] = 0u;
    for (int i = threadIdx.x; i < 1 + p.E + tiles_dn; i += blockDim.x) queue[i] = 0;
    for (int i = threadIdx.x; i < p.T * p.H / 8; i += blockDim.x) convert8(p, i);
    __syncthreads();
    route_permute_block(p, reinterpret_cast<int*>(smem), reinterpret_cast<int*>(smem) + kMaxE);
    __syncthreads();
    build_lpt(p, reinterpret_cast<int*>(smem) + 2 * kMaxE + 2);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release(p.sync, static_cast<int>(p.epoch));
  } else {
    if (threadIdx.x == 0) {
      const bool ok = wait_eq(p.sync, static_cast<int>(p.epoch));
      if (!ok) atomicOr(p.status, PW_STATUS_TIMEOUT);
      s_int[2] = ok;
    }
    __syncthreads();
    if (!s_int[2]) return;
  }

  const int nact = p.act_lpt[0];
  const int n_gu = nact * tiles_gu, total = n_gu + nact * tiles_dn;
  if (threadIdx.x == 0) s_int[0] = atomicAdd(queue, 1);
  __syncthreads();
  for (int slot = 0;; slot ^= 1) {
    const int item = s_int[slot];
    if (item >= total) break;
    if (threadIdx.x == 0) s_int[slot ^ 1] = atomicAdd(queue, 1);   // claim the next one now
    const bool gu = item < n_gu;
    const int rank = gu ? item / tiles_gu : (item - n_gu) / tiles_dn;
    Item it;
    it.expert = p.act_lpt[1 + rank];
    it.tile = gu ? item % tiles_gu : (item - n_gu) % tiles_dn;
    it.n = p.counts[it.expert];
    it.off = p.offsets[it.expert];
    const int kind = gu ? PW_KIND_GATE_UP : PW_KIND_DOWN;
    const BlockDesc d = *block_desc(p, it.expert, kind);
    const bool ok = d.q >= 1 && d.q <= PW_MAX_BITS && d.K == (gu ? p.H : p.I);
    if (!gu) {
      if (threadIdx.x == 0 && !wait_eq(&expert_done[it.expert], tiles_gu))
        atomicOr(p.status, PW_STATUS_TIMEOUT);
      __syncthreads();
    }
    if (ok) {
      if (gu) run_tile<PW_KIND_GATE_UP>(p, d, it, smem);
      else run_tile<PW_KIND_DOWN>(p, d, it, smem);
    } else if (threadIdx.x == 0) {
      atomicOr(p.status, PW_STATUS_BAD_DESC);
    }
    __threadfence();   // this thread's h / y writes before the counters below
    __syncthreads();
    if (gu) {
      if (threadIdx.x == 0) atomicAdd(&expert_done[it.expert], 1);
    } else {
      if (threadIdx.x == 0) {
        s_int[2] = (atomicAdd(&tile_done[it.tile], 1) == nact - 1);
        __threadfence();
      }
      __syncthreads();
      if (s_int[2]) {
        __threadfence();
        const int r0 = it.tile * kRows;
        combine_rows(p, r0, min(r0 + kRows, p.H), 0, p.T, threadIdx.x, blockDim.x);
      }
    }
    __syncthreads();
  }
}

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};     // decode grid per device once configured (0: not yet)
int g_fused[kMaxDevices] = {};   // cooperative grid of the fused layer per device

}  // namespace

cudaError_t launch_decode(const Fwd& p, int kind, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (g_sms[dev] == 0) {   // once per device: opt in to > 48 KB of shared memory
    e = cudaFuncSetAttribute(k_decode<PW_KIND_GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_decode<PW_KIND_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    int sms = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_sms[dev] = (sms > 0 ? sms : 1) * kCtasPerSm;
  }
  if (kind == PW_KIND_GATE_UP)
    k_decode<PW_KIND_GATE_UP><<<g_sms[dev], kThreads, kSmemBytes, s>>>(p);
  else
    k_decode<PW_KIND_DOWN><<<g_sms[dev], kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_layer_fused(const Fwd& p, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (g_fused[dev] == 0) {   // once per device: shared-memory opt-in and co-resident grid size
    e = cudaFuncSetAttribute(k_layer, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    int per_sm = 0, sms = 0;
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_layer, kThreads, kSmemBytes);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    g_fused[dev] = per_sm * sms;
  }
  Fwd arg = p;
  void* args[] = {&arg};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(k_layer), dim3(g_fused[dev]),
                                     dim3(kThreads), args, kSmemBytes, s);
}

}  // namespace pw
