// Decode-sized fused APL MoE layer (sm_103a): one persistent launch per layer.
//
// Source: PagedWeight technical summary, core components section 3 ("Fused
// Mixed-Precision Kernel": reads APL bit-planes and lookup tables directly,
// a different committed bitwidth per linear block within one fused operation).
//
// A decode batch gives each active expert a handful of tokens, so the layer
// streams every active block's q bit-planes and q-bit table from HBM once and
// keeps the tokens on chip.  What limits such a kernel is the instruction
// stream that turns plane bits into weights, so the design spends as few
// instructions per weight as it can:
//
//  * work items are 64-row tiles of one block (gate_up: 32 gate rows and the
//    32 matching up rows; down: 64 rows) for one pass of up to four of the
//    expert's tokens, laid out in a fixed order (largest gate_up cost first,
//    then all down tiles) and handed out by tickets in that order, so every
//    CTA knows its next items and loads their descriptors and tables ahead of
//    time; when the routed batch gives few down items (one token, long K),
//    each is split into K-ranges whose partial sums the combine adds in a
//    fixed order;
//  * lane l of every warp owns two rows of the tile (gate row l and up row l,
//    or rows l and 32 + l); the twelve warps split K;
//  * each warp streams its own plane words through a private cp.async ring of
//    four 2 KB half-stages (one coalesced 16-byte copy per lane and plane, the
//    pages being interleaved across 32-row groups; a unit of a q <= 4 block
//    takes one half-stage, a q >= 5 unit two) that
//    runs on into the warp's share of the next item, so the HBM stream does
//    not stop at item boundaries;
//  * the inner loop has two code paths, pair tables (q <= 4) and single
//    lookups (q >= 5), each for any q of its range (missing planes read as
//    zero plane slots), so that the hot code stays small.  The kernel is built
//    twice: with both paths for layers of hidden size >= 4096, and with the
//    single-lookup path alone (every q) for smaller ones, whose short items
//    do not repay the pair tables;
//  * q <= 4: pair tables.  The page keeps the even elements of every byte in
//    its low half and the odd ones in its high half, so a 4x4 bit transpose of
//    the q plane words nibble by nibble (four delta swaps per four words)
//    gives one byte per pair of neighbouring elements: the pair index
//    a | b << 4.  The row's pair table holds LUT[a] | LUT[b] << 16 at that
//    index, so one shared-memory lookup returns both fp16 weights of an MMA
//    register (rows rho and rho2 in the two halves of a 256-byte line);
//  * q >= 5: an 8x8 bit transpose (delta swaps) turns the plane words into one
//    index byte per element; one lookup per weight in a table whose 32-bit
//    slot (index, lane) holds both of the lane's rows' fp16 entries, so a
//    warp's 32 lookups hit 32 different banks whatever the indices, and one
//    byte permute packs two looked-up weights;
//  * the table window starts at a 64 KB-aligned shared address, so one byte
//    permute forms each lookup's full address (index in byte 1, lane offset in
//    byte 0, the window in bytes 2-3);
//  * the weights go straight from registers into the A operand of a
//    warp-level tensor-core MMA (m16n8k16, fp32 accumulate).  The MMA's 16
//    k-slots are split between the four lanes of a row group, and the token
//    operand is zero outside each lane's own column pair, so every lane
//    accumulates the dot products of its own two rows with two tokens (a
//    second MMA adds tokens 2 and 3);
//  * the K-warps' partial sums are added in a fixed order (bitwise
//    deterministic); gate_up items finish with h = silu(gate) * up (fp16),
//    down items with fp32 y rows; the CTA whose down item completes a 64-row
//    output tile combines it at its next item boundary.

#include <cuda_fp16.h>
#include <cstdint>

#include "pw_route.cuh"

namespace pw {
namespace {

constexpr int kThreads = 384;
constexpr int kWarps = kThreads / 32;
constexpr int kUnitWords = 2;      // plane words per row per ring stage
constexpr int kHalfStages = 4;     // ring of 2 KB half-stages per warp
constexpr int kTokPass = 4;        // tokens per pass over a tile (two MMA column sets)
constexpr int kGateUpTileRows = 32;   // gate rows per gate_up tile (plus as many up rows)
constexpr int kDownTileRows = 64;

// Shared memory: the table window, the warps' rings and one block of the rest
// ("misc": partial sums, the pair-table source, item descriptors, the layer's
// descriptors, routing results).  The window is 256 lines of 256 bytes at a
// 64 KB-aligned shared address; whatever precedes that address holds misc
// and as many rings as fit, the rest follows the window.
constexpr int kLine = 256;
constexpr int kTableBytes = 256 * kLine;
constexpr int kPlaneSlot = 512;                          // one plane of a unit: [row half][32 rows][2 words]
constexpr int kHalfStageBytes = 4 * kPlaneSlot;         // four plane slots
constexpr int kRingWarpBytes = kHalfStages * kHalfStageBytes;
constexpr int kSlots = 3;          // items in flight: current, next, the one after
constexpr int kRedOff = 0;                               // [warp][8][32 lanes] fp32 partial sums
constexpr int kScratchOff = kRedOff + kWarps * 8 * 32 * 4;   // [16 lines][32 lanes] single slots
constexpr int kDescOff = kScratchOff + 16 * 128;         // [kSlots] BlockDesc of the items in flight
constexpr int kCacheBlocks = 156;                        // the layer's descriptors when 2E fits
constexpr int kCacheOff = kDescOff + kSlots * 128;
constexpr int kRouteOff = kCacheOff + kCacheBlocks * 128;
constexpr int kCumOff = kRouteOff + route_smem_bytes();
constexpr int kItemOff = kCumOff + 2 * (kMaxE + 1) * 4;
constexpr int kMiscBytes = (kItemOff + 256 + 127) / 128 * 128;

// Placement for a window starting toff bytes into the dynamic shared memory.
struct Place {
  bool misc_first;   // misc before the window
  int nb;            // rings before the window
  int end;           // bytes used
};
__host__ __device__ constexpr Place place(int toff) {
  const bool mf = toff >= kMiscBytes;
  const int room = toff - (mf ? kMiscBytes : 0);
  const int nb = room / kRingWarpBytes < kWarps ? room / kRingWarpBytes : kWarps;
  return Place{mf, nb, toff + kTableBytes + (mf ? 0 : kMiscBytes) + (kWarps - nb) * kRingWarpBytes};
}
__host__ __device__ constexpr int smem_need() {
  int m = 0;
  for (int t = 0; t < 0x10000; t += 16) m = place(t).end > m ? place(t).end : m;
  return m;
}
constexpr int kSmemBytes = smem_need();
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

extern __shared__ __align__(128) unsigned char g_smem[];

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_wait_n(int n) {   // n = groups allowed to stay in flight
  if (n <= 0) cp_wait<0>();
  else if (n == 1) cp_wait<1>();
  else if (n == 2) cp_wait<2>();
  else cp_wait<3>();
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src) : "memory");
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
// (q-1-r) (zero for r >= q); afterwards byte bb of o[r] is the q-bit index
// (plane 0 most significant) of the element at bit 8*bb + r of the page word:
// element 8bb + 2r for r < 4, element 8bb + 2(r-4) + 1 for r >= 4.
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
// 4x4 bit transposes within every nibble.  Row r of the input holds plane
// (q-1-r) (zero for r >= q, q <= 4); afterwards nibble n of o[j] is the index
// of the element at bit 4n + j of the page word, so byte bb of o[j] is the
// pair index idx(8bb + 2j) | idx(8bb + 2j + 1) << 4.
__device__ __forceinline__ void planes_to_pairs(uint32_t (&o)[4]) {
  delta_swap(o[0], o[2], 2, 0x33333333u);
  delta_swap(o[1], o[3], 2, 0x33333333u);
  delta_swap(o[0], o[1], 1, 0x55555555u);
  delta_swap(o[2], o[3], 1, 0x55555555u);
}

// Table slot at shared address a.
__device__ __forceinline__ uint32_t lut_slot(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// Where the table, the rings and misc sit in this CTA's dynamic shared memory
// (computed once from the window address of g_smem).
struct Smem {
  unsigned char* table;   // 64 KB-aligned shared address
  unsigned char* misc;
  uint32_t table_hi;      // shared address of the table (bytes 2-3 only)
  uint32_t ring0, ring1;  // shared addresses: rings before / after the window
  int nb;                 // rings before the window
};
__device__ __forceinline__ Smem smem_layout() {
  Smem m;
  const uint32_t base = smem_addr(g_smem);
  const int toff = static_cast<int>((0x10000u - (base & 0xFFFFu)) & 0xFFFFu);
  const Place pl = place(toff);
  m.nb = pl.nb;
  m.table = g_smem + toff;
  m.table_hi = base + toff;
  m.misc = pl.misc_first ? g_smem : g_smem + toff + kTableBytes;
  m.ring0 = base + (pl.misc_first ? kMiscBytes : 0);
  m.ring1 = base + toff + kTableBytes + (pl.misc_first ? 0 : kMiscBytes);
  return m;
}
__device__ __forceinline__ uint32_t ring_of(const Smem& m, int warp) {
  return warp < m.nb ? m.ring0 + warp * kRingWarpBytes : m.ring1 + (warp - m.nb) * kRingWarpBytes;
}
__device__ __forceinline__ BlockDesc* desc_slot(const Smem& m, int sl) {
  return reinterpret_cast<BlockDesc*>(m.misc + kDescOff) + sl;
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld_nc16(const void* p) {   // read-only for the kernel's lifetime
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// ------------------------------------------------------------------ work items

struct ItemInfo {
  int valid, kind, expert, tile;
  int n;      // tokens of this pass (1..4)
  int off;    // permuted position of the pass's first token
  int need;   // down: gate_up items of the expert that must be done first
  int split;   // down: which of the nsplit K-ranges
  int nsplit;  // down: K-ranges of the forward's down items (1 for gate_up)
};

struct Plan {
  int nact, tiles_gu, tiles_dn, total_gu, total, down_per_tile;
  int ks;              // K-ranges per down item in this forward (<= p.ksplit)
  const int* cum_gu;   // [nact+1] first gate_up item of each cost rank
  const int* cum_dn;
};

// Item g of the layer's fixed order: gate_up items (experts by cost rank; per
// expert pass-major, then tile), then down items in the same expert order
// (per expert pass-major, then tile, then K-split).
__device__ ItemInfo item_of(int g, const Plan& pl, const RouteSmem& r, int ksplit) {
  ItemInfo it{};
  if (g < 0 || g >= pl.total) return it;
  const bool gu = g < pl.total_gu;
  const int* cum = gu ? pl.cum_gu : pl.cum_dn;
  const int gg = gu ? g : g - pl.total_gu;
  int lo = 0, hi = pl.nact - 1;   // last rank whose first item is <= gg
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= gg) lo = mid;
    else hi = mid - 1;
  }
  const int S = gu ? 1 : ksplit;
  const int tiles = (gu ? pl.tiles_gu : pl.tiles_dn) * S;
  const int rem = gg - cum[lo];
  const int e = r.lpt[1 + lo];
  const int pass = rem / tiles;
  const int cnt = r.cnt[e];
  it.valid = 1;
  it.kind = gu ? PW_KIND_GATE_UP : PW_KIND_DOWN;
  it.expert = e;
  it.tile = (rem % tiles) / S;
  it.split = (rem % tiles) % S;
  it.nsplit = S;
  it.n = min(kTokPass, cnt - pass * kTokPass);
  it.off = r.off[e] + pass * kTokPass;
  it.need = pl.tiles_gu * ((cnt + kTokPass - 1) / kTokPass);
  return it;
}

// Rows of lane l in a tile: rho (first half) and rho2 (second half).
__device__ __forceinline__ void lane_rows(const Fwd& p, const ItemInfo& it, int lane, int& rho, int& rho2) {
  if (it.kind == PW_KIND_GATE_UP) {
    rho = it.tile * kGateUpTileRows + lane;
    rho2 = p.I + rho;
  } else {
    rho = it.tile * kDownTileRows + lane;
    rho2 = rho + 32;
  }
}

// A descriptor is usable when its bitwidth and shape match the layer.
__device__ __forceinline__ bool desc_ok(const Fwd& p, const BlockDesc& d, int kind) {
  const bool gu = kind == PW_KIND_GATE_UP;
  return d.q >= 1 && d.q <= PW_MAX_BITS && d.K == (gu ? p.H : p.I) && d.R == (gu ? 2 * p.I : p.H);
}

// This warp's share of an item: plane words [w0, w1) of the item's K-range
// (K-split part `split` of `nsplit`), dealt word by word so that the twelve
// shares differ by at most one word, and the ring units (word pairs) that
// hold them, [u0, u1); a share that starts or ends inside a pair uses one of
// its two words.
__device__ __forceinline__ void warp_share(const BlockDesc& d, bool ok, int warp, int split, int nsplit, int& w0,
                                           int& w1, int& u0, int& u1) {
  const int W = ok ? (d.K >> 5) : 0;
  const int s0 = W * split / nsplit, n = W * (split + 1) / nsplit - s0;
  w0 = s0 + n * warp / kWarps;
  w1 = s0 + n * (warp + 1) / kWarps;
  u0 = w0 >> 1;
  u1 = w1 > w0 ? (w1 + 1) >> 1 : u0;
}

// ------------------------------------------------------------------ tables

// The next item's two table rows per lane, held in registers while the
// current item runs: thread (lane, wv) owns 8-entry chunks wv, wv + kWarps, ...
// (tables of fewer than 8 entries: warp 0 holds them whole in a[0] / b[0]).
constexpr int kLutChunks = (32 + kWarps - 1) / kWarps;   // 8-entry chunks per thread at q = 8
struct LutRegs {
  uint4 a[kLutChunks], b[kLutChunks];
};

__device__ __forceinline__ void lut_load(LutRegs& f, const BlockDesc& d, int rho, int rho2, int wv) {
  const int q = d.q, V = 1 << q;
  if (V < 8) {
    f.a[0] = f.b[0] = make_uint4(0u, 0u, 0u, 0u);
    if (wv == 0) {   // 2 or 4 entries per row
      const uint32_t* ra = reinterpret_cast<const uint32_t*>(d.lut + static_cast<size_t>(rho) * V);
      const uint32_t* rb = reinterpret_cast<const uint32_t*>(d.lut + static_cast<size_t>(rho2) * V);
      f.a[0].x = __ldg(ra);
      f.b[0].x = __ldg(rb);
      if (V == 4) {
        f.a[0].y = __ldg(ra + 1);
        f.b[0].y = __ldg(rb + 1);
      }
    }
    return;
  }
  const uint4* ra = reinterpret_cast<const uint4*>(d.lut + static_cast<size_t>(rho) * V);
  const uint4* rb = reinterpret_cast<const uint4*>(d.lut + static_cast<size_t>(rho2) * V);
#pragma unroll
  for (int j = 0; j < kLutChunks; ++j) {
    const int vc = wv + kWarps * j;
    if (vc * 8 < V) {
      f.a[j] = ld_nc16(ra + vc);
      f.b[j] = ld_nc16(rb + vc);
    }
  }
}

// Single-slot table: slot (v, lane) = (row rho entry v) | (row rho2 entry v) << 16
// at dst + v * stride + lane * 4.  Used as the table of q >= 5 items (stride: a
// window line) and as the source of the pair tables of q <= 4 items (stride
// 128, the scratch lines).
__device__ __forceinline__ void lut_store_single(unsigned char* dst, int stride, const LutRegs& f, int q,
                                                 int lane, int wv) {
  const int V = 1 << q;
  if (V < 8) {
    if (wv == 0) {
      const uint32_t wa[2] = {f.a[0].x, f.a[0].y};
      const uint32_t wb[2] = {f.b[0].x, f.b[0].y};
#pragma unroll
      for (int v = 0; v < 4; ++v)
        if (v < V)
          *reinterpret_cast<uint32_t*>(dst + v * stride + lane * 4) =
              prmt(wa[v >> 1], wb[v >> 1], (v & 1) ? 0x7632u : 0x5410u);
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < kLutChunks; ++j) {
    const int vc = wv + kWarps * j;
    if (vc * 8 < V) {
      const uint32_t aw[4] = {f.a[j].x, f.a[j].y, f.a[j].z, f.a[j].w};
      const uint32_t bw[4] = {f.b[j].x, f.b[j].y, f.b[j].z, f.b[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = vc * 8 + 2 * e;
        *reinterpret_cast<uint32_t*>(dst + v * stride + lane * 4) = prmt(aw[e], bw[e], 0x5410u);
        *reinterpret_cast<uint32_t*>(dst + (v + 1) * stride + lane * 4) = prmt(aw[e], bw[e], 0x7632u);
      }
    }
  }
}

// Pair tables of a q <= 4 item from its single slots in the scratch lines:
// line a | b << 4 of the window holds, for lane l, (rho entry a) | (rho entry
// b) << 16 at byte l * 4 and the same for rho2 at byte 128 + l * 4.  Each
// thread keeps its lane's 2^q single slots in registers; the work is cut into
// jobs (b, block of up to 8 a values), job j to warp j mod kWarps.
template <int Q>
__device__ __forceinline__ void pair_tables_q(unsigned char* table, const unsigned char* scratch, int lane,
                                              int wv) {
  constexpr int V = 1 << Q;
  constexpr int NB = V > 8 ? 2 : 1;   // blocks of a values
  constexpr int AB = V / NB;
  uint32_t sv[V];
#pragma unroll
  for (int v = 0; v < V; ++v) sv[v] = *reinterpret_cast<const uint32_t*>(scratch + v * 128 + lane * 4);
  for (int j = wv; j < V * NB; j += kWarps) {
    const int b = j % V;
    const uint32_t sb = *reinterpret_cast<const uint32_t*>(scratch + b * 128 + lane * 4);
    unsigned char* col = table + (b << 4) * kLine + lane * 4;
    if (j < V) {
#pragma unroll
      for (int a = 0; a < AB; ++a) {
        *reinterpret_cast<uint32_t*>(col + a * kLine) = prmt(sv[a], sb, 0x5410u);
        *reinterpret_cast<uint32_t*>(col + a * kLine + 128) = prmt(sv[a], sb, 0x7632u);
      }
    } else {
#pragma unroll
      for (int a = AB; a < V; ++a) {
        *reinterpret_cast<uint32_t*>(col + a * kLine) = prmt(sv[a], sb, 0x5410u);
        *reinterpret_cast<uint32_t*>(col + a * kLine + 128) = prmt(sv[a], sb, 0x7632u);
      }
    }
  }
}
__device__ __forceinline__ void pair_tables(unsigned char* table, const unsigned char* scratch, int q, int lane,
                                            int wv) {
  switch (q) {
    case 1: pair_tables_q<1>(table, scratch, lane, wv); break;
    case 2: pair_tables_q<2>(table, scratch, lane, wv); break;
    case 3: pair_tables_q<3>(table, scratch, lane, wv); break;
    default: pair_tables_q<4>(table, scratch, lane, wv); break;
  }
}

// ------------------------------------------------------------------ inner loop

// 16 bytes of a token row into x when pred is set (x keeps its value otherwise).
__device__ __forceinline__ void ld_x16(uint4& x, const void* ptr, bool pred) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " @p ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%5];\n}"
      : "+r"(x.x), "+r"(x.y), "+r"(x.z), "+r"(x.w)
      : "r"(static_cast<int>(pred)), "l"(ptr));
}

// The token operand of one plane word (32 k) for the two column sets, and the
// address of the next word's (refilled part by part as each part is used).
struct Tok {
  uint4 X0[4], X1[4];
  const uint4* x0;   // token rows of this lane (null: none)
  const uint4* x1;
  bool two;          // the pass has a third or fourth token (warp-uniform): second MMA column set
};

// One plane word of a q <= 4 block: o0 / o1 are rho's / rho2's pair indices
// (planes_to_pairs); lo0 / lo1 the lookup offsets of rho's / rho2's pair tables.
// MMA hh takes pairs j = 2hh (k-slots 2c, 2c+1) and 2hh + 1 (2c+8, 2c+9), i.e.
// elements 8bb + 4hh + {0, 1} and {2, 3}: the token operand's natural order.
__device__ __forceinline__ void word_mma_pairs(const uint32_t (&o0)[4], const uint32_t (&o1)[4], uint32_t lo0,
                                               uint32_t lo1, Tok& t, int gw, bool more, float (&acc)[2][2][4]) {
  const bool p0 = more && t.x0 != nullptr, p1 = more && t.x1 != nullptr;
#pragma unroll
  for (int bb = 0; bb < 4; ++bb) {
    const uint32_t sel = 0x7604u | (static_cast<uint32_t>(bb) << 4);
    uint32_t a[2][4];   // the byte lane's 8 lookups first, MMA hh = 0's four first
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      a[hh][0] = lut_slot(prmt(o0[2 * hh], lo0, sel));
      a[hh][1] = lut_slot(prmt(o1[2 * hh], lo1, sel));
      a[hh][2] = lut_slot(prmt(o0[2 * hh + 1], lo0, sel));
      a[hh][3] = lut_slot(prmt(o1[2 * hh + 1], lo1, sel));
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mma16816(acc[0][hh], a[hh], hh ? t.X0[bb].z : t.X0[bb].x, hh ? t.X0[bb].w : t.X0[bb].y);
      if (t.two) mma16816(acc[1][hh], a[hh], hh ? t.X1[bb].z : t.X1[bb].x, hh ? t.X1[bb].w : t.X1[bb].y);
    }
    ld_x16(t.X0[bb], t.x0 + (gw + 1) * 4 + bb, p0);
    if (t.two) ld_x16(t.X1[bb], t.x1 + (gw + 1) * 4 + bb, p1);
  }
}

// One plane word of a q >= 5 block: o0 / o1 are rho's / rho2's indices
// (planes_to_indices: o[r] byte bb is element 8bb + 2r, or 8bb + 2(r-4) + 1
// for r >= 4).  A lookup returns both rows' entries of one index; rho keeps
// the low halves, rho2 the high halves, two per MMA register.
__device__ __forceinline__ void word_mma_single(const uint32_t (&o0)[8], const uint32_t (&o1)[8], uint32_t lo0,
                                                Tok& t, int gw, bool more, float (&acc)[2][2][4]) {
  const bool p0 = more && t.x0 != nullptr, p1 = more && t.x1 != nullptr;
#pragma unroll
  for (int bb = 0; bb < 4; ++bb) {
    const uint32_t sel = 0x7604u | (static_cast<uint32_t>(bb) << 4);
    // the 16 lookups of the byte lane, those of MMA hh = 0 (rows 0, 4, 1, 5) first
    uint32_t s[8], u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = (i >> 1) + 4 * (i & 1);   // 0, 4, 1, 5, 2, 6, 3, 7
      s[r] = lut_slot(prmt(o0[r], lo0, sel));
      u[r] = lut_slot(prmt(o1[r], lo0, sel));
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // elements 8bb + 4hh + {0, 1}: rows 2hh and 4 + 2hh; {2, 3}: rows 2hh + 1 and 5 + 2hh
      uint32_t a[4];
      a[0] = prmt(s[2 * hh], s[4 + 2 * hh], 0x5410u);
      a[1] = prmt(u[2 * hh], u[4 + 2 * hh], 0x7632u);
      a[2] = prmt(s[2 * hh + 1], s[5 + 2 * hh], 0x5410u);
      a[3] = prmt(u[2 * hh + 1], u[5 + 2 * hh], 0x7632u);
      mma16816(acc[0][hh], a, hh ? t.X0[bb].z : t.X0[bb].x, hh ? t.X0[bb].w : t.X0[bb].y);
      if (t.two) mma16816(acc[1][hh], a, hh ? t.X1[bb].z : t.X1[bb].x, hh ? t.X1[bb].w : t.X1[bb].y);
    }
    ld_x16(t.X0[bb], t.x0 + (gw + 1) * 4 + bb, p0);
    if (t.two) ld_x16(t.X1[bb], t.x1 + (gw + 1) * 4 + bb, p1);
  }
}

// Where the warp's ring fetch stands: item (this CTA's local index), unit,
// end of the warp's units in that item, and what issuing a unit needs.  A unit
// is one word pair (64 k) of the tile's two 32-row groups; in the page layout
// each (plane, group, word pair) is 256 contiguous bytes, so lane l copies 16
// bytes: rows 2(l%16), 2(l%16)+1 of group l/16.
struct Fetch {
  int item, u, end, q;
  bool pair;
#ifdef PW_CHECK
  size_t words;      // plane words of the block (R * K / 32)
#endif         // the item's planes use the pair-table layout (four plane slots)
  size_t off;        // page word offset of this lane's 16 bytes at unit 0
  uint32_t desc;     // shared address of the item's descriptor
};

// A warp's ring: four 2 KB half-stages.  A unit of a q <= 4 item takes one
// half-stage (its planes in four plane slots), a unit of a q >= 5 item the two
// half-stages of one 4 KB half of the ring (eight slots; it starts at an even
// half-stage, leaving an odd one before it unused).  ih / ch count the half-stages issued /
// consumed (pads included), iu / cu the units; the unit being consumed starts
// at ch.
struct Ring {
  uint32_t base;
  int ih, ch, iu, cu;
};
// Pair tables for blocks of at most 4 bits, in the kernel built with them (kPairs).
template <bool kPairs>
__device__ __forceinline__ bool pair_mode(int q) { return kPairs && q <= 4; }
__device__ __forceinline__ int unit_halves(bool pair) { return pair ? 1 : 2; }

template <bool kPairs>
__device__ __forceinline__ void fetch_enter(Fetch& f, const Fwd& p, const Smem& sm, const ItemInfo* s_item,
                                            int item, int warp, int lane) {
  const int sl = item % kSlots;
  const ItemInfo& it = s_item[sl];
  const BlockDesc& d = *desc_slot(sm, sl);
  f.item = item;
  f.desc = smem_addr(&d);
  const bool ok = it.valid && desc_ok(p, d, it.kind);
  int w0, w1;
  warp_share(d, ok, warp, it.split, it.nsplit, w0, w1, f.u, f.end);
  const int h = lane >> 4;
  int grp;   // 32-row group of row half h
  if (it.kind == PW_KIND_GATE_UP) grp = h ? p.I / 32 + it.tile : it.tile;
  else grp = 2 * it.tile + h;
  f.q = d.q;
  f.pair = pair_mode<kPairs>(d.q);
#ifdef PW_CHECK
  f.words = static_cast<size_t>(d.R) * static_cast<size_t>(d.K) / 32;
#endif
  f.off = static_cast<size_t>(grp) * static_cast<size_t>(d.K >> 6) * 64 + (lane & 15) * 4;
}

// Issues units into the ring until it is full or the next unit belongs to an
// item that is not known yet (an item is known once its descriptor is in
// shared memory and it exists: items up to `known`).  The planes of a q-bit
// unit end at its last plane slot: plane p goes to slot s0 + p with s0 = 4 - q
// (one half-stage) or 8 - q (two), so that bit r of the index (plane q-1-r) is
// always slot 3 - r or 7 - r; the slots below s0 are zeroed.  The caller has
// synchronised the warp after the last read of the half-stages the issue may
// overwrite (everything before the unit being consumed).
template <bool kPairs>
__device__ __forceinline__ void fetch_fill(Fetch& f, const Fwd& p, const Smem& sm, const ItemInfo* s_item,
                                           int known, Ring& rg, int warp, int lane) {
  for (;;) {
    while (f.u == f.end) {   // the warp has no more units in this item
      if (f.item + 1 > known) return;
      fetch_enter<kPairs>(f, p, sm, s_item, f.item + 1, warp, lane);
    }
    const int sz = unit_halves(f.pair);
    const int pad = (sz == 2 && (rg.ih & 1)) ? 1 : 0;
    if (rg.ih + pad + sz > rg.ch + kHalfStages) return;   // full
    rg.ih += pad;
    const uint32_t dst = rg.base + (rg.ih & (kHalfStages - 1)) * kHalfStageBytes + (lane >> 4) * 256 +
                         (lane & 15) * 16;
    const size_t w = f.off + static_cast<size_t>(f.u) * 64;
    const int s0 = 4 * sz - f.q;   // first plane slot; the slots below it are zeroed
#pragma unroll
    for (int sl = 0; sl < PW_MAX_BITS; ++sl) {
      if (sl < s0) {
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst + sl * kPlaneSlot), "r"(0u) : "memory");
      } else if (sl < s0 + f.q) {
#ifdef PW_CHECK
        if (!PW_BOUNDS(p, w + 4 <= f.words, true)) {   // outside the page: zeros instead
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst + sl * kPlaneSlot), "r"(0u) : "memory");
          continue;
        }
#endif
        uint64_t base;
        asm volatile("ld.shared.u64 %0, [%1];" : "=l"(base) : "r"(f.desc + (sl - s0) * 8));
        const uint32_t* src = reinterpret_cast<const uint32_t*>(base) + w;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + sl * kPlaneSlot), "l"(src)
                     : "memory");
      }
    }
    cp_commit();
    rg.ih += sz;
    ++rg.iu;
    ++f.u;
  }
}

// The warp's units [u0, u1) of one item (its words [w0, w1)): ring stages in,
// transposes, lookups, MMAs.  Two code paths: pair tables (q <= 4, four plane slots) and single
// lookups (q >= 5, eight plane slots); missing planes read as zero slots.
template <bool kPairs, bool PAIR>
__device__ __forceinline__ void run_units(const Fwd& p, const Smem& sm, const ItemInfo* s_item, Fetch& f,
                                          int known, Ring& rg, int warp, int lane, uint32_t lo0, uint32_t lo1,
                                          int u0, int u1, int w0, int w1, Tok& t, float (&acc)[2][2][4]) {
  constexpr int NR = PAIR ? 4 : 8;   // index bits held (rows of the transposes)
  constexpr int SZ = PAIR ? 1 : 2;   // half-stages per unit
  for (int u = u0; u < u1; ++u) {
    cp_wait_n(rg.iu - rg.cu - 1);
    __syncwarp();   // every lane's copies of this unit visible; the previous unit is read
    if (SZ == 2 && (rg.ch & 1)) ++rg.ch;   // the issue's pad
    fetch_fill<kPairs>(f, p, sm, s_item, known, rg, warp, lane);
    const uint32_t st = rg.base + (rg.ch & (kHalfStages - 1)) * kHalfStageBytes + lane * 8;
    rg.ch += SZ;
    ++rg.cu;
#pragma unroll 1
    for (int wi = 0; wi < kUnitWords; ++wi) {
      const int gw = u * kUnitWords + wi;
      if (gw < w0 || gw >= w1) continue;   // the other word of a pair at the share's edge
      const bool more = gw + 1 < w1;
      uint32_t o0[NR], o1[NR];   // row r (bit r of the index) = slot NR-1-r
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        o0[r] = lds32(st + (NR - 1 - r) * kPlaneSlot + wi * 4);
        o1[r] = lds32(st + (NR - 1 - r) * kPlaneSlot + 256 + wi * 4);
      }
      if constexpr (PAIR) {
        planes_to_pairs(o0);
        planes_to_pairs(o1);
        word_mma_pairs(o0, o1, lo0, lo1, t, gw, more, acc);
      } else {
        planes_to_indices(o0);
        planes_to_indices(o1);
        word_mma_single(o0, o1, lo0, t, gw, more, acc);
      }
    }
  }
}

// 16-byte part of a block's descriptor: from the shared cache or global memory.
__device__ __forceinline__ uint4 desc_part(const Fwd& p, const Smem& sm, bool cached, int e, int kind, int part) {
  if (cached) return reinterpret_cast<const uint4*>(sm.misc + kCacheOff + (2 * e + kind) * 128)[part];
  return ld_nc16(reinterpret_cast<const uint4*>(block_desc(p, e, kind)) + part);
}

// ------------------------------------------------------------------ fused layer

constexpr int kSpinLimit = 1 << 22;   // ~0.3 s of polling before a wait gives up
constexpr int kSplitWaves = 3;        // down items wanted per CTA before K-splitting stops

__device__ __forceinline__ int ld_acquire(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* ptr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_add(int* ptr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}
// Bounded wait (one thread): true once *ptr >= want, false when the limit runs out.
__device__ bool wait_ge(const int* ptr, int want) {
  for (int i = 0; i < kSpinLimit; ++i) {
    if (ld_acquire(ptr) >= want) return true;
    __nanosleep(64);
  }
  return false;
}

// The first ticket of a claim under this forward's tag: the count the update
// returned, less the set-up bit (tickets taken while the forward was being set
// up follow the set-up CTA's tickets 0 and 1); -1 when the word holds another
// tag.
__device__ __forceinline__ int ticket_of(const Fwd& p, unsigned long long old) {
  if ((old & ~kCountMask) != p.tag) return -1;
  const unsigned long long c = old & kCountMask;
  return (c & kSetupBit) ? static_cast<int>(c & ~kSetupBit) + 2 : static_cast<int>(c);
}

// First claim of a CTA (one thread), right after the dependency wait; v is the
// ticket word as read at the kernel's start.  The first CTA to find the word
// under another tag sets the forward up (returns 1: tickets 0 and 1; the
// caller resets the counters, then clears the set-up bit); every other CTA
// takes two tickets at once (returns 0 with *first = its first ticket), or
// -1 if the word never settles.
__device__ int claim_first(const Fwd& p, unsigned long long v, int* first) {
  for (int i = 0; i < 64; ++i) {
    if ((v & ~kCountMask) == p.tag) {
      *first = ticket_of(p, add_relaxed_u64(p.sync, 2));
      return *first >= 0 ? 0 : -1;
    }
    const unsigned long long prev = cas_acq_rel_u64(p.sync, v, p.tag | kSetupBit);
    if (prev == v) return 1;
    v = prev;
  }
  return -1;
}

// Bounded wait (one thread) until the set-up CTA has reset the forward's
// counters and status (the set-up bit is clear): a CTA's first counter update,
// status bit or down-item wait comes after it.
__device__ bool wait_published(const Fwd& p) {
  for (int i = 0; i < kSpinLimit; ++i) {
    const unsigned long long v = ld_acquire_u64(p.sync);
    if ((v & ~kCountMask) == p.tag && !(v & kSetupBit)) return true;
    __nanosleep(64);
  }
  return false;
}

// A CTA's end of the forward (thread 0), in the build for captured CUDA
// graphs: it counts itself out, and the last CTA clears the ticket word, after
// every CTA's last ticket claim (each claim precedes its CTA's count).  The
// next forward on this workspace then sets up even when it carries the same
// tag, as the replays of one captured forward do.  (Eager calls take a new tag
// each and skip this: it costs about 1.5 % of a Mixtral-shaped layer.)
__device__ __noinline__ void leave_forward(unsigned long long* sync, unsigned long long tag, int n_counters,
                                           bool published) {
  for (int i = 0; !published && i < kSpinLimit; ++i) {   // as wait_published
    const unsigned long long v = ld_acquire_u64(sync);
    published = (v & ~kCountMask) == tag && !(v & kSetupBit);
    if (!published) __nanosleep(64);
  }
  if (!published) return;   // no set-up was seen: the counters are not this forward's
  int* exit_count = reinterpret_cast<int*>(sync + 1) + n_counters;
  __threadfence();
  if (atomicAdd(exit_count, 1) == static_cast<int>(gridDim.x) - 1) {
    __threadfence();
    st_release_u64(sync, 0ull);
  }
}

// Combine of one 64-row output tile once all its down items are done (the
// whole CTA): when the down items write parts (a workspace with room for a
// K-split), y = the ks parts added in split order (written to y for
// inspection), then out = residual + sum_j w * y.
__device__ void combine_tile(const Fwd& p, const RouteSmem& r, int tile, int ks, int tid) {
  const int r0 = tile * kDownTileRows, r1 = min(r0 + kDownTileRows, p.H);
  if (p.ksplit > 1) {
    const int P = p.T * p.k, n = r1 - r0;
    const size_t part = static_cast<size_t>(P) * p.H;
    for (int q = tid; q < P * n; q += kThreads) {
      const size_t at = static_cast<size_t>(q / n) * p.H + r0 + q % n;
      float v = 0.f;
      for (int sp = 0; sp < ks; ++sp) v += __ldcg(p.y_part + sp * part + at);
      p.y[at] = v;
    }
    __syncthreads();
  }
  combine_rows(p, r.w, r.inv, r0, r1, 0, p.T, tid, kThreads);
}

// One persistent launch (one CTA per SM, the co-resident grid) for the whole
// decode layer.  Every CTA routes the batch itself into shared memory (a few
// hundred logits, so no CTA waits for another's routing) and derives the
// layer's item order from it.  The items are handed out in that order by
// tickets: a CTA claims two at its start and one more at the start of each
// item, and works through its items in claim order.  Down items wait until
// their expert's gate_up items are done; all gate_up items precede all down
// items in the order, so every awaited item has been claimed by a CTA that is
// running and that reaches it without waiting on anything: the waits end
// whichever CTAs are resident.  The last down item of a 64-row output tile
// combines it.  Every wait is bounded and reports PW_STATUS_TIMEOUT instead of
// hanging.
template <bool kPairs, bool kGraph>
__global__ void __launch_bounds__(kThreads, 1) k_layer(Fwd p) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Smem sm = smem_layout();
  int* rs = reinterpret_cast<int*>(sm.misc + kRouteOff);
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
  int* cum_gu = reinterpret_cast<int*>(sm.misc + kCumOff);
  int* cum_dn = cum_gu + (kMaxE + 1);
  ItemInfo* s_item = reinterpret_cast<ItemInfo*>(sm.misc + kItemOff);
  unsigned char* scratch = sm.misc + kScratchOff;
  int* s_int = reinterpret_cast<int*>(s_item + kSlots);

  Plan pl;
  pl.tiles_gu = p.I / kGateUpTileRows;
  pl.tiles_dn = p.H / kDownTileRows;
  int* expert_done = reinterpret_cast<int*>(p.sync + 1);
  int* tile_done = expert_done + p.E;   // then the count of CTAs that finished this forward

  // The launch lets the next forward on the stream start on SMs this grid frees
  // (programmatic dependent launch): that forward routes its own batch while
  // this one finishes, and waits for it before touching the workspace.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the ticket word as it stands now (a hint for the claim; read again by its CAS)
  const unsigned long long tw = tid == 0 ? ld_relaxed_u64(p.sync) : 0ull;
  if (tid == 0) s_int[0] = 0;   // NaN logit seen
  // every block descriptor of the layer into shared memory (when they fit),
  // in flight while the batch is routed
  const bool cached = 2 * p.E <= kCacheBlocks;
  if (cached)
    for (int i = tid; i < 2 * p.E * 8; i += kThreads)
      cp_async16(sm.misc + kCacheOff + (i >> 3) * 128 + (i & 7) * 16,
                 reinterpret_cast<const uint4*>(p.desc + desc_index(p.layer, i >> 4, (i >> 3) & 1, p.E)) + (i & 7));
  cp_commit();
  __syncthreads();
  route_local(p, r, &s_int[0], kTokPass);   // reads only logits and descriptors
  pl.nact = r.lpt[0];
  if (warp == 0) {   // items per cost rank: tiles x passes; exclusive scan
    int run = 0;
    for (int a0 = 0; a0 <= pl.nact; a0 += 32) {
      const int a = a0 + lane;
      const int np = a < pl.nact ? (r.cnt[r.lpt[1 + a]] + kTokPass - 1) / kTokPass : 0;
      int incl = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (a <= pl.nact) {
        cum_gu[a] = (run + incl - np) * pl.tiles_gu;
        cum_dn[a] = run + incl - np;   // passes before rank a (scaled below)
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    // K-split of the down items: as many K-ranges (up to the workspace's
    // p.ksplit) as it takes for the down items to fill kSplitWaves waves of
    // the grid.  A few long down items (one token, two experts) leave most
    // CTAs idle at the end of the layer; more K-ranges than that only add item
    // boundaries and partial sums.  Measured on the Mixtral-8x7B-shaped layer:
    // batch 4 (384 unsplit down items) 352 us at 4 ranges, 344 at 1, 340 at 2;
    // batch 1 (128) 135 us at 4, 134 at 3.
    const int items_dn = run * pl.tiles_dn;
    const int want = kSplitWaves * static_cast<int>(gridDim.x);
    const int ks = items_dn > 0 ? max(1, min(p.ksplit, (want + items_dn - 1) / items_dn)) : 1;
    for (int a = lane; a <= pl.nact; a += 32) cum_dn[a] *= pl.tiles_dn * ks;
    if (lane == 0) s_int[4] = ks;
  }
  cp_wait<0>();   // the descriptor cache
  __syncthreads();
  pl.cum_gu = cum_gu;
  pl.cum_dn = cum_dn;
  pl.ks = s_int[4];
  pl.total_gu = cum_gu[pl.nact];
  pl.total = pl.total_gu + cum_dn[pl.nact];
  pl.down_per_tile = pl.tiles_dn > 0 ? cum_dn[pl.nact] / pl.tiles_dn : 0;

  // the previous kernel on the stream (possibly the previous forward, using the
  // same workspace) has finished and its writes are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) s_int[3] = claim_first(p, tw, &s_int[2]);
  __syncthreads();
  const int role = s_int[3];
  // published: this thread knows the forward's counters and status are reset
  // (tid 0 for counter updates and status bits, lane 0 of each warp for the
  // down-item waits)
  bool published = role == 1;
  if (role == 1) {
    // this CTA sets the forward up: counters to zero, the status word, then the
    // set-up bit cleared (tickets 0 and 1 are this CTA's)
    for (int i = tid; i < p.E + pl.tiles_dn + 1; i += kThreads) expert_done[i] = 0;   // and the exit count
    if (tid == 0) p.status[0] = s_int[0] ? PW_STATUS_NAN_LOGIT : 0u;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      add_release_u64(p.sync, 2ull - kSetupBit);
      s_int[2] = 0;
    }
    // the routing outputs the caller asked for, and the routing statistics
    const int P = p.T * p.k;
    for (int i = tid; i < P; i += kThreads) {
      if (p.user_idx) p.user_idx[i] = r.idx[i];
      if (p.user_w) p.user_w[i] = r.w[i];
      if (p.user_perm) p.user_perm[i] = r.perm[i];
    }
    if (p.user_offsets)
      for (int e = tid; e <= p.E; e += kThreads) p.user_offsets[e] = r.off[e];
    update_route_stats(p, r.perm, r.w, r.off);
  } else if (role < 0) {
    // the ticket word never settled (bounded): leave every item to the others
    if (tid == 0 && wait_published(p)) {
      atomicOr(p.status, PW_STATUS_TIMEOUT);
      if (kGraph) leave_forward(p.sync, p.tag, p.E + pl.tiles_dn, true);
    }
    return;
  }
  __syncthreads();
  // items of the first two tickets and their descriptors
  if (tid < 2) s_item[tid] = item_of(s_int[2] + tid, pl, r, pl.ks);
  __syncthreads();
  if (warp == 0 && lane < 16) {
    const int sl = lane >> 3, part = lane & 7;
    if (s_item[sl].valid)
      reinterpret_cast<uint4*>(desc_slot(sm, sl))[part] =
          desc_part(p, sm, cached, s_item[sl].expert, s_item[sl].kind, part);
  }
  __syncthreads();
  const uint32_t ring = ring_of(sm, warp);
  const uint32_t lo0 = sm.table_hi | (static_cast<uint32_t>(lane) * 4u);   // rho's lookups
  const uint32_t lo1 = lo0 + 128u;                                          // rho2's pair table
  Fetch f;
  Ring rg{ring, 0, 0, 0, 0};
  LutRegs lr;
  if (s_item[0].valid) {
    const BlockDesc& d0 = *desc_slot(sm, 0);
    int rho, rho2;
    lane_rows(p, s_item[0], lane, rho, rho2);
    const bool ok0 = desc_ok(p, d0, s_item[0].kind);
    if (ok0) lut_load(lr, d0, rho, rho2, warp);
    fetch_enter<kPairs>(f, p, sm, s_item, 0, warp, lane);
    fetch_fill<kPairs>(f, p, sm, s_item, s_item[1].valid ? 1 : 0, rg, warp, lane);
    if (ok0) {
      if (!pair_mode<kPairs>(d0.q)) {
        lut_store_single(sm.table, kLine, lr, d0.q, lane, warp);
      } else {
        lut_store_single(scratch, 128, lr, d0.q, lane, warp);
        __syncthreads();
        pair_tables(sm.table, scratch, d0.q, lane, warp);
      }
    }
  }
  __syncthreads();   // the first item's tables are complete

  // thread 0: the last down item's tile and the count its update returned,
  // looked at only at the next item boundary
  int pending_tile = -1, pending_old = -1;
  for (int i = 0; s_item[i % kSlots].valid; ++i) {
    const int sl = i % kSlots;
    const ItemInfo it = s_item[sl];
    const BlockDesc& d = *desc_slot(sm, sl);
    const bool gu = it.kind == PW_KIND_GATE_UP;
    const bool ok = desc_ok(p, d, it.kind) &&
                    PW_BOUNDS(p, it.expert >= 0 && it.expert < p.E && it.off >= 0 && it.off + it.n <= p.T * p.k &&
                                     it.tile >= 0 && it.tile < (gu ? pl.tiles_gu : pl.tiles_dn) &&
                                     it.split >= 0 && it.split < it.nsplit && it.nsplit <= (gu ? 1 : p.ksplit),
                              tid == 0);

    // item i+2's ticket: claimed now, looked at when this item ends
    const int sl1 = (i + 1) % kSlots, sl2 = (i + 2) % kSlots;
    const ItemInfo it1 = s_item[sl1];
    unsigned long long claim = 0;
    if (tid == 0 && it1.valid) claim = add_relaxed_u64(p.sync, 1);
    const int known = it1.valid ? i + 1 : i;   // the ring may run into item i+1
    // item i+1's tables, into registers until this item's lookups are done
    const BlockDesc& d1 = *desc_slot(sm, sl1);
    const bool ok1 = it1.valid && desc_ok(p, d1, it1.kind);
    if (ok1) {
      int rho, rho2;
      lane_rows(p, it1, lane, rho, rho2);
      lut_load(lr, d1, rho, rho2, warp);
    }

    int w0, w1, u0, u1;
    warp_share(d, ok, warp, it.split, it.nsplit, w0, w1, u0, u1);
    float acc[2][2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][hh][c] = 0.f;
    if (u0 < u1) {
      // this lane's token rows (lanes 9c + 4t carry token t of each column set)
      const int tl = (lane >> 2) - 2 * (lane & 3);
      Tok t;
      t.x0 = t.x1 = nullptr;
      t.two = it.n > 2;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = 2 * j + tl;
        if (tl >= 0 && tl <= 1 && tok < it.n) {
          const int pos = it.off + tok;
          const uint4* xr = reinterpret_cast<const uint4*>(gu ? p.x + static_cast<size_t>(r.perm[pos] / p.k) * p.H
                                                             : p.hh + static_cast<size_t>(pos) * p.I);
          if (j) t.x1 = xr;
          else t.x0 = xr;
        }
      }
      if (!gu) {   // h of this expert comes from its gate_up items
        if (lane == 0) {
          if (!published) published = wait_published(p);
          if (!published || !wait_ge(&expert_done[it.expert], it.need)) atomicOr(p.status, PW_STATUS_TIMEOUT);
        }
        __syncwarp();
      }
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        t.X0[k4] = make_uint4(0u, 0u, 0u, 0u);
        t.X1[k4] = make_uint4(0u, 0u, 0u, 0u);
        ld_x16(t.X0[k4], t.x0 + w0 * 4 + k4, t.x0 != nullptr);
        ld_x16(t.X1[k4], t.x1 + w0 * 4 + k4, t.x1 != nullptr);
      }
      if (pair_mode<kPairs>(d.q))
        run_units<kPairs, true>(p, sm, s_item, f, known, rg, warp, lane, lo0, lo1, u0, u1, w0, w1, t, acc);
      else
        run_units<kPairs, false>(p, sm, s_item, f, known, rg, warp, lane, lo0, lo1, u0, u1, w0, w1, t, acc);
    }
    // keep the ring running into the next item while this one finishes
    __syncwarp();
    fetch_fill<kPairs>(f, p, sm, s_item, known, rg, warp, lane);

    // ---- partial sums: red[warp][half * 4 + token][lane]
    float* red = reinterpret_cast<float*>(sm.misc + kRedOff);
    {
      float* rw = red + warp * 8 * 32;
      float v[8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {   // column set j: tokens 2j, 2j+1 of the rows rho / rho2
        v[2 * j] = acc[j][0][0] + acc[j][1][0];
        v[2 * j + 1] = acc[j][0][1] + acc[j][1][1];
        v[4 + 2 * j] = acc[j][0][2] + acc[j][1][2];
        v[4 + 2 * j + 1] = acc[j][0][3] + acc[j][1][3];
      }
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) rw[k8 * 32 + lane] = v[k8];
    }
    // a q <= 4 next item: its single slots into the scratch lines now (the
    // pair tables are built from them after the barrier)
    if (ok1 && pair_mode<kPairs>(d1.q)) lut_store_single(scratch, 128, lr, d1.q, lane, warp);
    // a down tile whose last item completed with the previous item: combine it now;
    // item i+2 from the ticket claimed at this item's start
    if (tid == 0) {
      s_int[1] = pending_old == pl.down_per_tile - 1 ? pending_tile : -1;
      s_item[sl2] = it1.valid ? item_of(ticket_of(p, claim), pl, r, pl.ks) : ItemInfo{};
    }
    __syncthreads();   // every lookup of this item is done; partials visible
    if (s_int[1] >= 0) combine_tile(p, r, s_int[1], pl.ks, tid);
    pending_tile = -1;
    pending_old = -1;

    if (ok1) {
      if (!pair_mode<kPairs>(d1.q)) lut_store_single(sm.table, kLine, lr, d1.q, lane, warp);
      else pair_tables(sm.table, scratch, d1.q, lane, warp);
    }
    if (warp == 0 && lane < 8 && s_item[sl2].valid)
      reinterpret_cast<uint4*>(desc_slot(sm, sl2))[lane] =
          desc_part(p, sm, cached, s_item[sl2].expert, s_item[sl2].kind, lane);
    auto red_at = [&](int w, int k8, int l) { return red[(w * 8 + k8) * 32 + l]; };
    if (gu) {
      if (tid < 32 * it.n) {
        const int l = tid & 31, t = tid >> 5;
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          g += red_at(w, t, l);
          u += red_at(w, 4 + t, l);
        }
        const float hv = g / (1.f + expf(-g)) * u;
        p.hh[static_cast<size_t>(it.off + t) * p.I + it.tile * kGateUpTileRows + l] = __float2half_rn(hv);
      }
    } else {
      if (tid < 64 * it.n) {
        const int l = tid & 31, hf = (tid >> 5) & 1, t = tid >> 6;
        float yv = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) yv += red_at(w, hf * 4 + t, l);
        p.y_part[(static_cast<size_t>(it.split) * p.T * p.k + it.off + t) * p.H + it.tile * kDownTileRows + hf * 32 +
                 l] = yv;
      }
    }
    // Outputs written; next item's tables and descriptor in place.  After the
    // barrier, thread 0's release-ordered counter update publishes every
    // thread's h / y writes (ordered before it by the barrier).  A gate_up
    // update is fire and forget; a down update returns the tile's count, which
    // thread 0 looks at only at the next item boundary (the atomic's round trip
    // overlaps the next item), where the CTA that completed the tile combines it.
    __syncthreads();
    if (tid == 0) {
      if (!published) published = wait_published(p);
      if (!ok || !published) atomicOr(p.status, published ? PW_STATUS_BAD_DESC : PW_STATUS_TIMEOUT);
      if (gu) {
        red_release_add(&expert_done[it.expert], 1);
      } else {
        pending_old = atom_acq_rel_add(&tile_done[it.tile], 1);
        pending_tile = it.tile;
      }
    }
  }
  if (tid == 0) s_int[1] = pending_old == pl.down_per_tile - 1 ? pending_tile : -1;
  __syncthreads();
  if (s_int[1] >= 0) combine_tile(p, r, s_int[1], pl.ks, tid);
  if (kGraph && tid == 0) leave_forward(p.sync, p.tag, p.E + pl.tiles_dn, published);
  cp_wait<0>();
}

constexpr int kMaxDevices = 64;
int g_fused[kMaxDevices] = {};   // co-resident grid of the fused layer per device

// Pair tables pay for their larger tables (64 KB rebuilt per q = 4 item) and
// the second inner loop only when items are long.  Measured on GB300: with
// them, Mixtral-8x7B-shaped decode layers (H = 4096) run 5 % faster, and
// Qwen1.5-MoE-shaped ones (H = 2048; gate_up items of 5 plane words per warp)
// 6 % slower, since the pair code also slows the q >= 5 loop.  So the kernel
// is built twice and the layer's hidden size picks one.
constexpr int kPairsMinH = 4096;

}  // namespace

cudaError_t launch_layer_fused(const Fwd& p, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (p.H % kDownTileRows != 0 || p.I % kGateUpTileRows != 0) return cudaErrorInvalidValue;
  if (g_fused[dev] == 0) {   // once per device: shared-memory opt-in and co-resident grid size
    const void* fns[4] = {reinterpret_cast<const void*>(k_layer<true, false>),
                          reinterpret_cast<const void*>(k_layer<false, false>),
                          reinterpret_cast<const void*>(k_layer<true, true>),
                          reinterpret_cast<const void*>(k_layer<false, true>)};
    int per_sm = 1 << 30, sms = 0;
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) {
      e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      int n = 0;
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fns[i], kThreads, kSmemBytes);
      per_sm = n < per_sm ? n : per_sm;
    }
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    g_fused[dev] = per_sm * sms;
  }
  // A call being captured into a CUDA graph gets the build that clears the
  // ticket word at its end (its replays repeat the capture's tag).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  const bool graph = cap != cudaStreamCaptureStatusNone;
  // An ordinary launch of the co-resident grid (items are handed out by
  // tickets, so the waits end even when only some CTAs are resident), allowed
  // to start while the previous kernel on the stream finishes (programmatic
  // stream serialisation; the kernel waits for it with griddepcontrol.wait
  // before it touches the workspace or the token rows).
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
  if (p.H >= kPairsMinH)
    return graph ? cudaLaunchKernelEx(&cfg, k_layer<true, true>, p) : cudaLaunchKernelEx(&cfg, k_layer<true, false>, p);
  return graph ? cudaLaunchKernelEx(&cfg, k_layer<false, true>, p) : cudaLaunchKernelEx(&cfg, k_layer<false, false>, p);
}

}  // namespace pw
