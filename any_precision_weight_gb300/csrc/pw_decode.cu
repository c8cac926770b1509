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
// Shared memory.  The tables take [v][64 slots] fp32 so that one byte permute
// forms index*256 + row*4; rows use slots 0..31, and the other 128 bytes of
// every 256-byte line ("pieces") hold the per-warp token scratch and the
// K-warp partial sums.
constexpr int kLutBytes = 256 * 64 * 4;
constexpr int kPlaneStageBytes = PW_MAX_BITS * kRows * kStageWords * 4;
constexpr int kXStageBytes = kTok * kStageK * 2;            // fp16 tokens
constexpr int kPieceRed = 0;                                // kKW * kTok pieces
constexpr int kPieceXw = kPieceRed + kKW * kTok;            // 2 per (warp, token)
constexpr int kSmemBytes = kLutBytes + 2 * kPlaneStageBytes + 2 * kXStageBytes + route_smem_bytes() + 64;

// The kernel's dynamic shared memory.  Table reads index this symbol directly,
// so its (link-time constant) shared address folds into the load's immediate
// offset instead of costing an add per looked-up weight.
extern __shared__ __align__(128) unsigned char g_smem[];

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }


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

// fp16 input row of permuted position pos: the token's x for gate_up, the
// pair's h for down.  perm may live in global or shared memory.
template <int KIND>
__device__ __forceinline__ const __half* token_row(const Fwd& p, const int* perm, int pos, int K) {
  if (KIND == PW_KIND_GATE_UP) return p.x + static_cast<size_t>(perm[pos] / p.k) * K;
  return p.hh + static_cast<size_t>(pos) * K;
}

// 128-byte piece n of the tables' unused half.
__device__ __forceinline__ float* piece(unsigned char* smem, int n) {
  return reinterpret_cast<float*>(smem + n * 256 + 128);
}

// mode: kTileWhole runs the tile; kTilePrologue only loads the tile's tables and
// its first stage of plane words (nothing that another kernel writes) and
// returns; kTileResume runs a tile whose prologue has been done.
constexpr int kTileWhole = 0, kTilePrologue = 1, kTileResume = 2;

template <int KIND>
__device__ void run_tile(const Fwd& p, const BlockDesc& d, const Item& it, unsigned char* smem,
                         const int* perm, int mode = kTileWhole) {
  float* lut_s = reinterpret_cast<float*>(smem);
  uint32_t* pl_s = reinterpret_cast<uint32_t*>(smem + kLutBytes);
  __half* x_s = reinterpret_cast<__half*>(smem + kLutBytes + 2 * kPlaneStageBytes);

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
  const unsigned char* lut_bytes = g_smem;   // lut_s == g_smem

  for (int t0 = 0; t0 < it.n; t0 += kTok) {
    const int nt = min(kTok, it.n - t0);
    const int xt = tid >> 6, xc = tid & 63;         // token staging: thread -> (token, 16 B)
    const __half* trow = (xt < nt) ? token_row<KIND>(p, perm, it.off + t0 + xt, K) : nullptr;

    auto fill = [&](int c, int s, bool planes = true, bool tokens = true) {
      const int wsrc = c * kStageWords + fc * 4;
      if (planes && fgr >= 0 && wsrc < W) {
        uint32_t* dst = pl_s + s * (kPlaneStageBytes / 4) + fdst;
#pragma unroll
        for (int j = 0; j < PW_MAX_BITS / 2; ++j) {   // static indices keep the descriptor in registers
          const int pl = 2 * j + fpl;
          const uint32_t* src = fpl ? d.planes[2 * j + 1] : d.planes[2 * j];
          if (pl < Q) cp_async16(dst + pl * kRows * kStageWords, src + fsrc + c * kStageWords);
        }
      }
      const int kk = c * kStageK + xc * 8;
      if (tokens && trow && kk < K) cp_async16(x_s + s * (kXStageBytes / 2) + xt * kStageK + xc * 8, trow + kk);
      cp_commit();
    };

    const bool first = t0 == 0;
    fill(0, 0, !(first && mode == kTileResume), !(first && mode == kTilePrologue));
    if (first && mode != kTileResume) {
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
    if (mode == kTilePrologue) return;

    // four independent packed (two-wide fp32) accumulators per token keep the
    // FMA chains short
    float2 acc[kTok][4];
#pragma unroll
    for (int t = 0; t < kTok; ++t)
#pragma unroll
      for (int m = 0; m < 4; ++m) acc[t][m] = make_float2(0.f, 0.f);

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
        // this warp's 64 token values of the stage, fp16 -> fp32 scratch
        __syncwarp();
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
          if (t < nt) {
            const __half2 h2 = reinterpret_cast<const __half2*>(x_s + s * (kXStageBytes / 2) + t * kStageK + kw * 64)[lane];
            *reinterpret_cast<float2*>(piece(smem, kPieceXw + 2 * (kw * kTok + t) + (lane >> 4)) + ((2 * lane) & 31)) =
                __half22float2(h2);
          }
        }
        __syncwarp();
        const uint32_t* ps = pl_s + s * (kPlaneStageBytes / 4) + row * kStageWords + rsw;
        uint2 pv[PW_MAX_BITS];
#pragma unroll
        for (int pl = 0; pl < PW_MAX_BITS; ++pl)   // pv[r] = plane (q-1-r)
          pv[pl] = (pl < Q) ? *reinterpret_cast<const uint2*>(ps + (Q - 1 - pl) * kRows * kStageWords)
                            : make_uint2(0u, 0u);
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          if (wi < nw) {
            uint32_t o[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) o[r] = wi == 0 ? pv[r].x : pv[r].y;
            planes_to_indices(o);
            // eight weights at a time (byte lane bb of the transposed words),
            // each multiplied into every token of the pass before the next eight
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              float w8[8];
#pragma unroll
              for (int r = 0; r < 8; ++r) {
                const uint32_t a = prmt(o[r], laneoff, 0x5504u | (static_cast<uint32_t>(bb) << 4));
                w8[r] = *reinterpret_cast<const float*>(lut_bytes + a);
              }
#pragma unroll
              for (int t = 0; t < kTok; ++t) {
                if (t < nt) {
                  const float4* xr = reinterpret_cast<const float4*>(piece(smem, kPieceXw + 2 * (kw * kTok + t) + wi));
                  const float4 x0 = xr[2 * bb], x1 = xr[2 * bb + 1];
                  acc[t][0] = __ffma2_rn(make_float2(w8[0], w8[1]), make_float2(x0.x, x0.y), acc[t][0]);
                  acc[t][1] = __ffma2_rn(make_float2(w8[2], w8[3]), make_float2(x0.z, x0.w), acc[t][1]);
                  acc[t][2] = __ffma2_rn(make_float2(w8[4], w8[5]), make_float2(x1.x, x1.y), acc[t][2]);
                  acc[t][3] = __ffma2_rn(make_float2(w8[6], w8[7]), make_float2(x1.z, x1.w), acc[t][3]);
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
        piece(smem, kPieceRed + kw * kTok + t)[row] =
            ((acc[t][0].x + acc[t][0].y) + (acc[t][1].x + acc[t][1].y)) +
            ((acc[t][2].x + acc[t][2].y) + (acc[t][3].x + acc[t][3].y));
    __syncthreads();
    if (KIND == PW_KIND_GATE_UP) {
      if (tid < nt * 16) {
        const int t = tid >> 4, i = tid & 15;
        const int r = it.tile * 16 + i;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < kKW; ++w8) {
          g += piece(smem, kPieceRed + w8 * kTok + t)[i];
          u += piece(smem, kPieceRed + w8 * kTok + t)[16 + i];
        }
        if (r < p.I) {
          const float hv = g / (1.f + expf(-g)) * u;
          p.hh[static_cast<size_t>(it.off + t0 + t) * p.I + r] = __float2half_rn(hv);
        }
      }
    } else {
      if (tid < nt * kRows) {
        const int t = tid >> 5, i = tid & 31;
        const int r = it.tile * kRows + i;
        float yv = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < kKW; ++w8) yv += piece(smem, kPieceRed + w8 * kTok + t)[i];
        if (r < p.H) p.y[static_cast<size_t>(it.off + t0 + t) * p.H + r] = yv;
      }
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

// One persistent launch (the co-resident grid) for the whole decode layer.
// CTA 0 clears the work-queue counters and publishes a ready epoch at once;
// every CTA routes the batch itself into shared memory (a few hundred logits,
// so no CTA waits for another's routing), then takes items from one queue:
// first all (expert, gate_up tile) items, largest gate_up cost first, then all
// (expert, down tile) items in the same expert order.  A down item first waits
// until its expert's gate_up tiles are all done; the last down item of a
// 32-row tile of H (over all active experts) combines that tile's output rows.
// Every wait is bounded and reports PW_STATUS_TIMEOUT instead of hanging.
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_layer(Fwd p) {
  unsigned char* smem = g_smem;
  int* s_int = reinterpret_cast<int*>(smem + kSmemBytes - 64);
  int* rs = reinterpret_cast<int*>(smem + kLutBytes + 2 * kPlaneStageBytes + 2 * kXStageBytes);
  RouteSmem r;
  r.idx = rs;
  r.w = reinterpret_cast<float*>(rs + kRouteSmemMaxPairs);
  r.perm = rs + 2 * kRouteSmemMaxPairs;
  r.inv = rs + 3 * kRouteSmemMaxPairs;
  r.cnt = rs + 4 * kRouteSmemMaxPairs;
  r.off = r.cnt + (kMaxE + 1);
  r.act = r.off + (kMaxE + 1);
  r.lpt = r.act + (kMaxE + 1);
  r.qgu = r.lpt + (kMaxE + 1);

  const int tiles_gu = p.I / 16, tiles_dn = (p.H + kRows - 1) / kRows;
  int* queue = p.sync + 1;
  int* expert_done = p.sync + 2;
  int* tile_done = p.sync + 2 + p.E;

  // The launch lets the next forward on the stream start on SMs this grid frees
  // (programmatic dependent launch): that forward routes its own batch while
  // this one finishes, and waits for it before touching the workspace.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) s_int[3] = 0;   // NaN logit seen
  __syncthreads();
  route_local(p, r, &s_int[3], kTok);   // reads only logits and descriptors
  const int nact = r.lpt[0];
  const int n_gu = nact * tiles_gu, total = n_gu + nact * tiles_dn;
  // Every CTA's first item is item blockIdx.x (later ones come from the queue).
  // A gate_up first item needs only weights, so its tables and first stage of
  // planes load before the wait below, overlapping the previous kernel's tail.
  auto make_item = [&](int item, int& kind) {
    const bool gu = item < n_gu;
    const int rank = gu ? item / tiles_gu : (item - n_gu) / tiles_dn;
    Item it;
    it.expert = r.lpt[1 + rank];
    it.tile = gu ? item % tiles_gu : (item - n_gu) % tiles_dn;
    it.n = r.cnt[it.expert];
    it.off = r.off[it.expert];
    kind = gu ? PW_KIND_GATE_UP : PW_KIND_DOWN;
    return it;
  };
  int pre_item = -1;
  if (static_cast<int>(blockIdx.x) < n_gu) {
    int kind0;
    const Item it0 = make_item(blockIdx.x, kind0);
    const BlockDesc d0 = *block_desc(p, it0.expert, kind0);
    if (d0.q >= 1 && d0.q <= PW_MAX_BITS && d0.K == p.H) {
      run_tile<PW_KIND_GATE_UP>(p, d0, it0, smem, r.perm, kTilePrologue);
      pre_item = blockIdx.x;
    }
  }
  // the previous kernel on the stream (possibly the previous forward, using the
  // same workspace) has finished and its writes are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) p.status[0] = s_int[3] ? PW_STATUS_NAN_LOGIT : 0u;
    for (int i = threadIdx.x; i < 1 + p.E + tiles_dn; i += blockDim.x) queue[i] = 0;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) st_release(p.sync, static_cast<int>(p.epoch));
    // the routing outputs the caller asked for
    const int P = p.T * p.k;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
      if (p.user_idx) p.user_idx[i] = r.idx[i];
      if (p.user_w) p.user_w[i] = r.w[i];
      if (p.user_perm) p.user_perm[i] = r.perm[i];
    }
    if (p.user_offsets)
      for (int e = threadIdx.x; e <= p.E; e += blockDim.x) p.user_offsets[e] = r.off[e];
    update_route_stats(p, r.perm, r.w, r.off);
  } else {
    if (threadIdx.x == 0) {
      const bool ok = wait_eq(p.sync, static_cast<int>(p.epoch));
      if (!ok) atomicOr(p.status, PW_STATUS_TIMEOUT);
      s_int[2] = ok;
    }
    __syncthreads();
    if (!s_int[2]) {
      cp_wait<0>();   // no copy of a pre-started tile outlives the CTA
      return;
    }
  }

  if (threadIdx.x == 0) s_int[0] = blockIdx.x;
  __syncthreads();
  for (int slot = 0;; slot ^= 1) {
    const int item = s_int[slot];
    if (item >= total) break;
    if (threadIdx.x == 0) s_int[slot ^ 1] = atomicAdd(queue, 1) + gridDim.x;   // claim the next one now
    int kind;
    const Item it = make_item(item, kind);
    const bool gu = kind == PW_KIND_GATE_UP;
    const BlockDesc d = *block_desc(p, it.expert, kind);
    const bool ok = d.q >= 1 && d.q <= PW_MAX_BITS && d.K == (gu ? p.H : p.I);
    if (!gu) {
      if (threadIdx.x == 0 && !wait_eq(&expert_done[it.expert], tiles_gu))
        atomicOr(p.status, PW_STATUS_TIMEOUT);
      __syncthreads();
    }
    if (ok) {
      if (gu) run_tile<PW_KIND_GATE_UP>(p, d, it, smem, r.perm, item == pre_item ? kTileResume : kTileWhole);
      else run_tile<PW_KIND_DOWN>(p, d, it, smem, r.perm);
    } else if (threadIdx.x == 0) {
      atomicOr(p.status, PW_STATUS_BAD_DESC);
    }
    // the h / y writers (threads below kTok * kRows) order their writes before the
    // counters below; the other threads wrote nothing other CTAs read
    if (threadIdx.x < kTok * kRows) __threadfence();
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
        combine_rows(p, r.w, r.inv, r0, min(r0 + kRows, p.H), 0, p.T, threadIdx.x, blockDim.x);
      }
    }
    __syncthreads();
  }
}

constexpr int kMaxDevices = 64;
int g_fused[kMaxDevices] = {};   // co-resident grid of the fused layer per device

}  // namespace

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
  // An ordinary launch of exactly the co-resident grid (every wait in the kernel
  // is on work that a running CTA has already claimed, or on CTA 0, which is
  // scheduled first), allowed to start while the previous kernel on the stream
  // finishes (programmatic stream serialisation; the kernel waits for it with
  // griddepcontrol.wait before it touches the workspace or the token rows).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g_fused[dev]);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_layer, p);
}

}  // namespace pw
