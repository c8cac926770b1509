// Prefill-sized expert GEMMs of the fused APL MoE layer on the 5th-generation
// tensor cores (sm_103a: TMA, mbarrier, tcgen05 MMA with the accumulator in TMEM).
//
// Source: PagedWeight technical summary, core components section 3 ("Fused
// Mixed-Precision Kernel": the kernel reads APL bit-planes and lookup tables
// directly, a different committed bitwidth per linear block).  With hundreds of
// tokens per expert the layer is a dense contraction, so the weights are
// dequantised once per tile into shared memory and multiplied on tensor cores.
//
// One CTA per SM, persistent over (expert, weight-row tile, group of up to 3
// token tiles) items, so each dequantised weight tile feeds up to 3 MMAs:
//  * the expert's token rows (gathered into expert order, fp16) arrive by TMA in
//    128 x 64 boxes with the 128-byte swizzle;
//  * bit-planes arrive by coalesced cp.async, two K steps (16 bytes per row and
//    plane) at a time, double buffered; each K step reads its q words per row
//    straight from the staged chunk;
//  * all 8 warps dequantise the 128 weight rows x 64 k of the same K step
//    straight into the K-major 128-byte-swizzled layout the MMA reads (SWAR bit
//    transpose of the plane words, byte-permute table addressing, fp16 table in
//    shared memory), then fence the async proxy;
//  * one thread issues tcgen05.mma kind::f16 (M = 128 tokens, N = 128 weight
//    rows, K = 16 per instruction, fp32 accumulate in TMEM) and commits to the
//    stage's mbarrier; the token tiles of step k+1 are fetched while step k
//    multiplies, so dequant, TMA and MMA overlap; only that thread waits on
//    mbarriers;
//  * the epilogue reads TMEM with tcgen05.ld: gate_up tiles (64 gate + 64 up
//    rows) write h = silu(gate) * up in fp16, down tiles write y in fp32.
// Every mbarrier wait is bounded and reports PW_STATUS_TIMEOUT.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "pw_route.cuh"

namespace pw {
namespace {

constexpr int kDqThreads = 256;                // dequantising warps 0..7
constexpr int kPThreads = kDqThreads + 32;     // + one TMA / MMA issue warp
constexpr int kBM = 128;                       // tokens per tile (MMA M)
constexpr int kBN = 128;                       // weight rows per tile (MMA N)
constexpr int kBK = 64;                        // K per stage: one 128-byte swizzle row of fp16
constexpr int kPStages = 2;
constexpr int kMT = 3;                         // token tiles sharing one dequantised weight tile
constexpr int kTileBytes = kBM * kBK * 2;      // 16 KB, A and B alike
constexpr int kPLutBytes = 256 * kBN * 2;      // fp16 [v][128 rows]
constexpr int kOffA = 0;                       // [stage][token tile] 16 KB boxes
constexpr int kOffB = kOffA + kPStages * kMT * kTileBytes;
constexpr int kOffLut = kOffB + kPStages * kTileBytes;
constexpr int kPlaneChunkBytes = PW_MAX_BITS * kBM * 16;   // 16 bytes (2 K steps) per row per plane
constexpr int kOffPl = kOffLut + kPLutBytes;               // [2 chunks][plane][row][4 words]
constexpr int kOffBar = kOffPl + 2 * kPlaneChunkBytes;
constexpr int kMiscBytes = 64 + 16 + 4 * (256 + 1) + 64;   // barriers, TMEM address, item prefix per expert
constexpr int kPSmemBytes = kOffBar + kMiscBytes + 1024;   // + slack to align the base to 1 KB
constexpr uint32_t kTmemCols = 512;           // kMT 128-column fp32 accumulators (power-of-two allocation)
constexpr long long kWaitLimit = 1ll << 22;

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Bounded wait for the phase of the given parity; false when the limit runs
// out or when another thread has raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
  for (long long i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (*abort) return false;
  }
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Barrier of the dequantising warps only (the issue warp keeps running).
__device__ __forceinline__ void named_sync_dq() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDqThreads) : "memory");
}

// ---------------------------------------------------------------- TMA / tcgen05

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFF) >> 4);          // start address      [0, 14)
  d |= static_cast<uint64_t>(1) << 16;                        // leading byte offset [16, 30)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride byte offset  [32, 46)
  d |= static_cast<uint64_t>(1) << 46;                        // version             [46, 48)
  d |= static_cast<uint64_t>(2) << 61;                        // 128-byte swizzle    [61, 64)
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D, M x N.
constexpr uint32_t kIdesc = (1u << 4)                             // D format: f32
                            | (0u << 7) | (0u << 10)              // A, B: f16
                            | (static_cast<uint32_t>(kBN >> 3) << 17)
                            | (static_cast<uint32_t>(kBM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void proxy_fence_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t prmt_p(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t bitsel_p(uint32_t a, uint32_t b, uint32_t m) {   // (a & ~m) | (b & m)
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xCA;" : "=r"(d) : "r"(m), "r"(b), "r"(a));
  return d;
}
__device__ __forceinline__ void swap_p(uint32_t& lo, uint32_t& hi, int s, uint32_t mask) {
  const uint32_t nlo = bitsel_p(lo, hi << s, mask << s);
  const uint32_t nhi = bitsel_p(hi, lo >> s, mask);
  lo = nlo;
  hi = nhi;
}
// Row r of o holds plane (q-1-r); afterwards byte bb of o[r] is the index of the
// element at bit 8bb + r of the page word.
__device__ __forceinline__ void transpose8(uint32_t (&o)[8]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) swap_p(o[r], o[r + 4], 4, 0x0F0F0F0Fu);
#pragma unroll
  for (int r = 0; r < 8; r += 4) {
    swap_p(o[r], o[r + 2], 2, 0x33333333u);
    swap_p(o[r + 1], o[r + 3], 2, 0x33333333u);
  }
#pragma unroll
  for (int r = 0; r < 8; r += 2) swap_p(o[r], o[r + 1], 1, 0x55555555u);
}

// Weight row of tile row i (-1 past the block).
template <int KIND>
__device__ __forceinline__ int wrow(const Fwd& p, int nt, int i) {
  if (KIND == PW_KIND_GATE_UP) {
    const int r = nt * (kBN / 2) + (i & 63);
    if (r >= p.I) return -1;
    return i < 64 ? r : p.I + r;
  }
  const int r = nt * kBN + i;
  return r < p.H ? r : -1;
}

template <int KIND>
__global__ void __launch_bounds__(kPThreads, 1)
k_prefill(const Fwd p, const __grid_constant__ CUtensorMap tmA) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1 KB-aligned base for the swizzled tiles, derived from the shared array
  // itself so the compiler keeps every access below in the shared window
  unsigned char* smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = saddr(smem);
  const uint32_t bar_full = sbase + kOffBar;          // [2] TMA of A arrived
  const uint32_t bar_mma = sbase + kOffBar + 16;      // [2] MMAs of the step done (B and A stage free)
  const uint32_t bar_b = sbase + kOffBar + 32;        // [2] B tile of the step dequantised
  int* s_misc = reinterpret_cast<int*>(smem + kOffBar + 64);   // [0] tmem addr, [1] abort, [4..] item starts
  __half* lut_s = reinterpret_cast<__half*>(smem + kOffLut);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E;
  const int K = (KIND == PW_KIND_GATE_UP) ? p.H : p.I;
  const int W = K >> 5;
  const int nksteps = K / kBK;
  const int ntiles = (KIND == PW_KIND_GATE_UP) ? p.I / (kBN / 2) : (p.H + kBN - 1) / kBN;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(s_misc)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_mma + 8 * s, 1);
      mbar_init(bar_b + 8 * s, kDqThreads);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_misc[1] = 0;
  }
  // items: per expert ceil(token tiles / kMT) groups x ntiles weight tiles
  int* s_start = s_misc + 4;   // [E+1] first item of each expert
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      s_start[e] = run;
      run += ((p.counts[e] + kBM * kMT - 1) / (kBM * kMT)) * ntiles;
    }
    s_start[E] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(s_misc[0]);
  const int total = s_start[E];
  const bool mma_warp = warp == kDqThreads / 32;

  // dequant role: tile row and which 32-k half of the K step
  const int row = tid & 127, half = (tid >> 7) & 1;
  // byte offset of the row's entry in a 256-byte table line: rows r and r + 64
  // share a 32-bit slot (r % 64), so the 32 rows a warp looks up at once sit in
  // 32 different banks whatever their indices
  const uint32_t rowoff = static_cast<uint32_t>(row & 63) * 4u + static_cast<uint32_t>(row >> 6) * 2u;
  const int lslot = static_cast<int>(rowoff >> 1);             // the same in fp16 entries
  uint32_t g = 0;                                              // K steps so far (stage ring), same in every warp

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int e = 0;
    while (s_start[e + 1] <= item) ++e;
    const int local = item - s_start[e];
    const int ngroups = (p.counts[e] + kBM * kMT - 1) / (kBM * kMT);
    const int nt = local / ngroups, mg = local % ngroups;
    const int row0 = p.offsets[e] + mg * kBM * kMT;            // first permuted pair of the group
    const int nvalid = min(kBM * kMT, p.counts[e] - mg * kBM * kMT);
    const int nm = (nvalid + kBM - 1) / kBM;                   // token tiles in this group
    const BlockDesc d = *block_desc(p, e, KIND);
    const int Q = d.q, V = 1 << Q;
    if (!PW_BOUNDS(p, e < E && row0 >= 0 && row0 + nvalid <= p.T * p.k && nt < ntiles, tid == 0)) continue;
    if (Q < 1 || Q > PW_MAX_BITS || d.K != K) {
      if (tid == 0) atomicOr(p.status, PW_STATUS_BAD_DESC);
      continue;
    }
    const uint32_t g0 = g;

    if (mma_warp) {
      // ---- TMA and MMA issue (one lane): A of step k goes to stage (g0+k)&1 once the
      // MMAs of step k-2 are done; the MMAs of step k wait for A and for B
      if (lane == 0 && !s_misc[1]) {
        auto wait_or_abort = [&](uint32_t bar, uint32_t parity) {
          if (mbar_wait(bar, parity, s_misc + 1)) return true;
          atomicOr(p.status, PW_STATUS_TIMEOUT);
          s_misc[1] = 1;
          return false;
        };
        auto load_a = [&](uint32_t gk, int k) {
          const uint32_t sa = gk & 1;
          mbar_expect_tx(bar_full + 8 * sa, nm * kTileBytes);
          for (int m = 0; m < nm; ++m)
            tma_load_2d(sbase + kOffA + (sa * kMT + m) * kTileBytes, &tmA, k * kBK, row0 + m * kBM,
                        bar_full + 8 * sa);
        };
        bool ok = true;
        // step 0's stage was last used by step g0-2: wait for its MMAs
        if (g0 >= 2) ok = wait_or_abort(bar_mma + 8 * (g0 & 1), ((g0 - 2) >> 1) & 1);
        if (ok) load_a(g0, 0);
        for (int ks = 0; ks < nksteps && ok; ++ks) {
          const uint32_t gk = g0 + ks, s = gk & 1;
          ok = wait_or_abort(bar_full + 8 * s, (gk >> 1) & 1) && wait_or_abort(bar_b + 8 * s, (gk >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t b0 = sbase + kOffB + s * kTileBytes;
          for (int m = 0; m < nm; ++m) {
            const uint32_t a0 = sbase + kOffA + (s * kMT + m) * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_f16(tmem + m * kBN, smem_desc(a0 + kk * 32), smem_desc(b0 + kk * 32), (ks | kk) != 0);
          }
          mma_commit(bar_mma + 8 * s);
          // step ks+1's tokens go to the stage of step ks-1 once its MMAs are done
          // (step ks's MMAs are queued behind them meanwhile)
          if (ks + 1 < nksteps) {
            if (gk >= 1) ok = wait_or_abort(bar_mma + 8 * (s ^ 1), ((gk - 1) >> 1) & 1);
            if (ok) load_a(gk + 1, ks + 1);
          }
        }
      }
      __syncwarp();
      g = g0 + nksteps;
      continue;
    }

    // ---- dequantisation (warps 0..7): LUT, plane chunks, one B tile per K step
    const int grow = wrow<KIND>(p, nt, row);
    // the previous item's dequant steps and epilogue are done by every dequant thread
    named_sync_dq();
    // the tile's table: LUT_q[row][v] fp16 -> lut_s[v][slot of row]
    // (rows of fewer than 8 entries, q < 3, are not 16-byte aligned: 2-byte loads)
    if (V < 8) {
      if (half == 0)
        for (int v = 0; v < V; ++v)
          reinterpret_cast<uint16_t*>(lut_s)[v * kBN + lslot] =
              grow >= 0 ? __ldg(d.lut + static_cast<size_t>(grow) * V + v) : static_cast<uint16_t>(0);
    }
    // four 16-byte loads in flight per thread before their values are stored
    for (int vc0 = half; V >= 8 && vc0 * 8 < V; vc0 += 8) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vc = vc0 + 2 * u;
        raw[u] = make_uint4(0, 0, 0, 0);
        if (grow >= 0 && vc * 8 < V)
          raw[u] = __ldg(reinterpret_cast<const uint4*>(d.lut + static_cast<size_t>(grow) * V + vc * 8));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vc = vc0 + 2 * u;
        if (vc * 8 >= V) break;
        const uint16_t* hv = reinterpret_cast<const uint16_t*>(&raw[u]);
#pragma unroll
        for (int j = 0; j < 8; ++j) reinterpret_cast<uint16_t*>(lut_s)[(vc * 8 + j) * kBN + lslot] = hv[j];
      }
    }
    // plane chunks: 16 bytes (4 words = K steps 2j, 2j+1) per row and plane;
    // thread (row, group) copies planes 4*group .. 4*group+3 of its row.  In
    // the page layout a row's word pairs are 64 words apart, so each chunk is
    // two 8-byte copies (32 consecutive rows' copies are contiguous)
    const int cgrp = half;
    const size_t prow = grow >= 0 ? (static_cast<size_t>(grow >> 5) * (W >> 1)) * 64 + (grow & 31) * 2 : 0;
    auto fetch_chunk = [&](int j) {
      if (grow >= 0 && 2 * j < nksteps) {
        unsigned char* dst = smem + kOffPl + (j & 1) * kPlaneChunkBytes + row * 16;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int pl = cgrp * 4 + u;
          const uint32_t* src = cgrp ? d.planes[4 + u] : d.planes[u];
          if (pl < Q) {
            const uint32_t* gsrc = src + prow + static_cast<size_t>(2 * j) * 64;
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(saddr(dst + pl * kBM * 16)),
                         "l"(gsrc));
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(saddr(dst + pl * kBM * 16 + 8)),
                         "l"(gsrc + 64));
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    fetch_chunk(0);
    fetch_chunk(1);
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    named_sync_dq();          // table and chunk 0 visible to every dequant thread

    const unsigned char* lutb = reinterpret_cast<const unsigned char*>(lut_s);
    for (int ks = 0; ks < nksteps; ++ks) {
      const uint32_t gk = g0 + ks, s = gk & 1;
      // B stage s was last read by the MMAs of step gk-2
      if (gk >= 2) {
        if (lane == 0 && !mbar_wait(bar_mma + 8 * s, ((gk - 2) >> 1) & 1, s_misc + 1)) {
          atomicOr(p.status, PW_STATUS_TIMEOUT);
          s_misc[1] = 1;
        }
        __syncwarp();
        tc_fence_after();
      }
      {
        // the row's plane words of this K step and half: word (ks & 1) * 2 + half of
        // the staged 16-byte chunk, plane q-1-r into o[r]
        const uint32_t* src = reinterpret_cast<const uint32_t*>(
            smem + kOffPl + ((ks >> 1) & 1) * kPlaneChunkBytes + row * 16) + (ks & 1) * 2 + half;
        uint32_t o[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) o[r] = (r < Q) ? src[(Q - 1 - r) * (kBM * 4)] : 0u;
        transpose8(o);
        unsigned char* tileB = smem + kOffB + s * kTileBytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          uint32_t hv[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const uint32_t a = prmt_p(o[r], rowoff, 0x5504u | (static_cast<uint32_t>(bb) << 4));
            hv[r] = *reinterpret_cast<const uint16_t*>(lutb + a);
          }
          // o[r] byte bb holds element 8bb + 2r (r < 4) or 8bb + 2(r-4) + 1 (r >= 4):
          // the page keeps a byte's even elements in its low half, odd in its high half
          uint4 pk;
          pk.x = hv[0] | (hv[4] << 16);
          pk.y = hv[1] | (hv[5] << 16);
          pk.z = hv[2] | (hv[6] << 16);
          pk.w = hv[3] | (hv[7] << 16);
          const int chunk = half * 4 + bb;
          *reinterpret_cast<uint4*>(tileB + ((chunk ^ (row & 7)) << 4)) = pk;
        }
      }
      proxy_fence_smem();   // generic-proxy writes of B visible to the tensor core
      mbar_arrive(bar_b + 8 * s);
      if (ks & 1) {
        // both K steps of chunk ks/2 are read by every thread: refill its buffer with
        // chunk ks/2 + 2 after chunk ks/2 + 1 has landed and is visible
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        named_sync_dq();
        fetch_chunk((ks >> 1) + 2);
      }
    }
    g = g0 + nksteps;

    // ---- epilogue: wait for the tile's last MMAs, then TMEM -> registers -> global
    {
      const uint32_t gl = g - 1;
      if (lane == 0 && !mbar_wait(bar_mma + 8 * (gl & 1), (gl >> 1) & 1, s_misc + 1)) {
        atomicOr(p.status, PW_STATUS_TIMEOUT);
        s_misc[1] = 1;
      }
      __syncwarp();
      tc_fence_after();
      // after an abort (a bounded wait gave up) every wait returns at once and the
      // accumulators are not read; the status word reports the failure
      if (!__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(s_misc + 1), 0)) {
        const int lg = warp & 3, ch = warp >> 2;
        for (int m = 0; m < nm; ++m) {
          const int tok = m * kBM + lg * 32 + lane;              // TMEM lane = token row of the tile
          const uint32_t lane_addr = tmem + m * kBN + (static_cast<uint32_t>(lg * 32) << 16);
          if (KIND == PW_KIND_GATE_UP) {
            float gv[32], uv[32];
            tmem_ld32(lane_addr + ch * 32, gv);
            tmem_ld32(lane_addr + 64 + ch * 32, uv);
            if (tok < nvalid) {
              __half* dst = p.hh + static_cast<size_t>(row0 + tok) * p.I + nt * 64 + ch * 32;
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                __half2 h2[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float a = gv[j + 2 * u], b = gv[j + 2 * u + 1];
                  const float ha = a / (1.f + expf(-a)) * uv[j + 2 * u];
                  const float hb = b / (1.f + expf(-b)) * uv[j + 2 * u + 1];
                  h2[u] = __floats2half2_rn(ha, hb);
                }
                *reinterpret_cast<uint4*>(dst + j) = *reinterpret_cast<const uint4*>(h2);
              }
            }
          } else {
            float yv[32];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              tmem_ld32(lane_addr + ch * 64 + c * 32, yv);
              if (tok < nvalid) {
                float* dst = p.y + static_cast<size_t>(row0 + tok) * p.H + nt * kBN + ch * 64 + c * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                  *reinterpret_cast<float4*>(dst + j) = make_float4(yv[j], yv[j + 1], yv[j + 2], yv[j + 3]);
              }
            }
          }
        }
      }
      // TMEM reads complete before this thread's next B arrival lets the MMA warp
      // overwrite the accumulators with the next tile's first MMAs
      tc_fence_before();
    }
  }

  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// X_perm[pos] = x[perm[pos] / k]: the expert-ordered token rows the GEMM reads by TMA.
__global__ void k_gather_x(Fwd p) {
  const int pos = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(p.perm[pos] / p.k) * p.H);
  uint4* dst = reinterpret_cast<uint4*>(p.xp + static_cast<size_t>(pos) * p.H);
  for (int i = threadIdx.x; i < p.H / 8; i += blockDim.x) dst[i] = src[i];
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
constexpr int kMaxDevicesP = 64;
int g_psms[kMaxDevicesP] = {};

cudaError_t make_map(CUtensorMap* m, const void* base, int rows, int cols) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {kBK, kBM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const Fwd& p, int kind, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesP) return cudaErrorInvalidDevice;
  if (g_psms[dev] == 0) {
    e = cudaFuncSetAttribute(k_prefill<PW_KIND_GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_prefill<PW_KIND_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
    int sms = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_psms[dev] = sms > 0 ? sms : 1;
  }
  const int P = p.T * p.k;
  CUtensorMap map;
  if (kind == PW_KIND_GATE_UP) {
    k_gather_x<<<P, 128, 0, s>>>(p);
    e = make_map(&map, p.xp, P, p.H);
    if (e != cudaSuccess) return e;
    k_prefill<PW_KIND_GATE_UP><<<g_psms[dev], kPThreads, kPSmemBytes, s>>>(p, map);
  } else {
    e = make_map(&map, p.hh, P, p.I);
    if (e != cudaSuccess) return e;
    k_prefill<PW_KIND_DOWN><<<g_psms[dev], kPThreads, kPSmemBytes, s>>>(p, map);
  }
  return cudaGetLastError();
}

}  // namespace pw
