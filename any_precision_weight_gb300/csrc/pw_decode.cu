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
//    then all down tiles) and dealt round-robin to the CTAs, so every CTA knows
//    its next items and loads their descriptors and tables ahead of time;
//  * lane l of every warp owns two rows of the tile (gate row l and up row l,
//    or rows l and 32 + l); the twelve warps split K.  The two rows' q-bit
//    tables sit in shared memory as one 32-bit slot per (index, lane) holding
//    both rows' fp16 entries, so a warp's 32 lookups hit 32 different banks
//    whatever the indices;
//  * each warp streams its own plane words through a private two-stage
//    cp.async ring (one coalesced 16-byte copy per lane and plane, the pages
//    being interleaved across 32-row groups) that runs on into the warp's
//    share of the next item, so the HBM stream does not stop at item
//    boundaries;
//  * per 32-bit plane word, a lane turns q plane words into 32 indices with an
//    8x8 bit transpose (delta swaps), one byte permute per weight forms the
//    table address, and the looked-up fp16 weights go straight from registers
//    into the A operand of a warp-level tensor-core MMA (m16n8k16, fp32
//    accumulate).  The MMA's 16 k-slots are split between the four lanes of a
//    row group, and the token operand is zero outside each lane's own column
//    pair, so every lane accumulates the dot products of its own two rows with
//    two tokens (a second MMA adds tokens 2 and 3).  The MMA does the
//    multiply-adds that would otherwise cost two fp32 instructions per weight
//    and token;
//  * blocks of at most 3 bits use pair tables: the transposes' upper rows take
//    the plane words shifted by one element, so one lookup returns two
//    neighbouring weights already packed for the MMA;
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
constexpr int kStages = 2;         // ring stages per warp
constexpr int kTokPass = 4;        // tokens per pass over a tile (two MMA column sets)
constexpr int kGateUpTileRows = 32;   // gate rows per gate_up tile (plus as many up rows)
constexpr int kDownTileRows = 64;

// Shared memory.  Table line v (256 bytes) holds the 32 lanes' slots for index
// v in its first half; the second halves ("pieces", 128 bytes each) hold the
// split-K partial sums and the descriptors of the items in flight.  The table
// starts at a 64 KB-aligned shared address, so that one byte permute forms a
// lookup's complete address (index in byte 1, lane * 4 in byte 0, the table's
// 64 KB window in bytes 2-3).  The warps' rings fill the space before it and
// continue after it, followed by the routing results ("rest").
constexpr int kLine = 256;
constexpr int kTableBytes = 256 * kLine;
constexpr int kStageBytes = PW_MAX_BITS * 2 * 32 * 8;   // [plane][row half][lane] x 2 words
constexpr int kRingWarpBytes = kStages * kStageBytes;
constexpr int kSlots = 3;          // items in flight: current, next, the one after
constexpr int kRouteOff = 0;       // offsets within the rest area
constexpr int kCumOff = kRouteOff + route_smem_bytes();
constexpr int kItemOff = kCumOff + 2 * (kMaxE + 1) * 4;
constexpr int kRestBytes = kItemOff + 256;
// whatever the dynamic window's start, everything fits in: at most one ring's
// worth of bytes before the table is left unused
constexpr int kSmemBytes = (kWarps + 1) * kRingWarpBytes + kTableBytes + kRestBytes;
constexpr int kPieceRed = 0;       // warps x 8 (row half, token) x 32 lanes fp32
constexpr int kPieceDesc = kWarps * 8;   // one BlockDesc per item slot
constexpr int kPieceCache = kPieceDesc + kSlots;   // descriptors of every block of the layer
constexpr int kCacheBlocks = 256 - kPieceCache;    // (when 2 E fits)

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
  else cp_wait<2>();
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

// Table slot at shared address a.
__device__ __forceinline__ uint32_t lut_slot(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// Where the table, the rings and the rest area sit in this CTA's dynamic
// shared memory (computed once from the window address of g_smem).
struct Smem {
  unsigned char* table;   // 64 KB-aligned shared address
  unsigned char* rest;
  uint32_t table_hi;      // shared address of the table (bytes 2-3 only)
  int nb;                 // warps whose rings sit before the table
  uint32_t toff;
};
__device__ __forceinline__ Smem smem_layout() {
  Smem m;
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(g_smem));
  m.toff = (0x10000u - (base & 0xFFFFu)) & 0xFFFFu;
  m.nb = min(kWarps, static_cast<int>(m.toff / kRingWarpBytes));
  m.table = g_smem + m.toff;
  m.table_hi = base + m.toff;
  m.rest = m.table + kTableBytes + (kWarps - m.nb) * kRingWarpBytes;
  return m;
}
__device__ __forceinline__ uint32_t ring_of(const Smem& m, int warp) {
  const uint32_t off = warp < m.nb ? warp * kRingWarpBytes
                                   : m.toff + kTableBytes + (warp - m.nb) * kRingWarpBytes;
  return static_cast<uint32_t>(__cvta_generic_to_shared(g_smem)) + off;
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

// 128-byte piece n (second half of table line n).
__device__ __forceinline__ unsigned char* piece(unsigned char* table, int n) { return table + n * kLine + 128; }

// ------------------------------------------------------------------ work items

struct ItemInfo {
  int valid, kind, expert, tile;
  int n;      // tokens of this pass (1..4)
  int off;    // permuted position of the pass's first token
  int need;   // down: gate_up items of the expert that must be done first
  int pad;
};

struct Plan {
  int nact, tiles_gu, tiles_dn, total_gu, total, down_per_tile;
  const int* cum_gu;   // [nact+1] first gate_up item of each cost rank
  const int* cum_dn;
};

// Item g of the layer's fixed order: gate_up items (experts by cost rank; per
// expert pass-major, then tile), then down items in the same expert order.
__device__ ItemInfo item_of(int g, const Plan& pl, const RouteSmem& r) {
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
  const int tiles = gu ? pl.tiles_gu : pl.tiles_dn;
  const int rem = gg - cum[lo];
  const int e = r.lpt[1 + lo];
  const int pass = rem / tiles;
  const int cnt = r.cnt[e];
  it.valid = 1;
  it.kind = gu ? PW_KIND_GATE_UP : PW_KIND_DOWN;
  it.expert = e;
  it.tile = rem % tiles;
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

// This warp's plane-word units (2 words each) of an item: [u0, u1).
__device__ __forceinline__ void warp_units(const BlockDesc& d, bool ok, int warp, int& u0, int& u1) {
  const int U = ok ? (d.K >> 6) : 0;
  u0 = U * warp / kWarps;
  u1 = U * (warp + 1) / kWarps;
}

// ------------------------------------------------------------------ tables

// The next item's two table rows per lane, held in registers while the
// current item runs: thread (lane, wv) owns 8-entry chunks wv, wv + kWarps, ...
constexpr int kLutChunks = (32 + kWarps - 1) / kWarps;   // 8-entry chunks per thread at q = 8
struct LutRegs {
  uint4 a[kLutChunks], b[kLutChunks];
};

__device__ __forceinline__ void lut_load(LutRegs& f, const BlockDesc& d, int rho, int rho2, int wv) {
  const int q = d.q, V = 1 << q;
  if (q <= 3) {   // pair tables: every thread holds both rows' whole tables
    f.a[0] = f.b[0] = make_uint4(0u, 0u, 0u, 0u);
    if (V == 8) {
      f.a[0] = ld_nc16(reinterpret_cast<const uint4*>(d.lut + static_cast<size_t>(rho) * V));
      f.b[0] = ld_nc16(reinterpret_cast<const uint4*>(d.lut + static_cast<size_t>(rho2) * V));
    } else {   // 2 or 4 entries per row
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

// q >= 4: slot (v, lane) = (row rho entry v) | (row rho2 entry v) << 16 in line
// v.  q <= 3 (pair tables, indexed by a | b << 4 for two neighbouring weights'
// indices a, b < 8): line a | b << 4 holds (rho entry a) | (rho entry b) << 16,
// line (a | b << 4) + 128 the same for rho2; warp wv fills the lines of a = wv.
__device__ __forceinline__ void lut_store(unsigned char* table, const LutRegs& f, int q, int lane, int wv) {
  const int V = 1 << q;
  if (q <= 3) {
    const uint32_t wa[4] = {f.a[0].x, f.a[0].y, f.a[0].z, f.a[0].w};
    const uint32_t wb[4] = {f.b[0].x, f.b[0].y, f.b[0].z, f.b[0].w};
    const int a = wv;
    if (a < V) {
      // entry a of each row (a warp-uniform index: a funnel of selects)
      const uint32_t ta = (a & 4) ? ((a & 2) ? wa[3] : wa[2]) : ((a & 2) ? wa[1] : wa[0]);
      const uint32_t tb = (a & 4) ? ((a & 2) ? wb[3] : wb[2]) : ((a & 2) ? wb[1] : wb[0]);
      const uint32_t la = (a & 1) ? ta >> 16 : ta & 0xFFFFu;
      const uint32_t lb = (a & 1) ? tb >> 16 : tb & 0xFFFFu;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (b < V) {
          const uint32_t ha = (b & 1) ? (wa[b >> 1] & 0xFFFF0000u) : (wa[b >> 1] << 16);
          const uint32_t hb = (b & 1) ? (wb[b >> 1] & 0xFFFF0000u) : (wb[b >> 1] << 16);
          unsigned char* line = table + (a | (b << 4)) * kLine + lane * 4;
          *reinterpret_cast<uint32_t*>(line) = la | ha;
          *reinterpret_cast<uint32_t*>(line + 128 * kLine) = lb | hb;
        }
      }
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
        *reinterpret_cast<uint32_t*>(table + v * kLine + lane * 4) = prmt(aw[e], bw[e], 0x5410u);
        *reinterpret_cast<uint32_t*>(table + (v + 1) * kLine + lane * 4) = prmt(aw[e], bw[e], 0x7632u);
      }
    }
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

// One plane word (32 k) of the lane's two rows into the accumulators.
// o0 / o1: transposed indices of rho / rho2 (byte bb of o[r] = element 8bb + r);
// X0 / X1: token operand of the word for column sets 0 / 1, refilled with the
// next word's (x0n / x1n + 16 bytes per bb, when `more`) as each part is used.
__device__ __forceinline__ void word_mma(const uint32_t (&o0)[8], const uint32_t (&o1)[8], uint32_t laneoff,
                                         uint4 (&X0)[4], uint4 (&X1)[4], const uint4* x0n, const uint4* x1n,
                                         bool p0, bool p1, float (&acc)[2][2][4]) {
#pragma unroll
  for (int bb = 0; bb < 4; ++bb) {
    const uint32_t sel = 0x7604u | (static_cast<uint32_t>(bb) << 4);
    uint32_t s[8], t[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      s[r] = lut_slot(prmt(o0[r], laneoff, sel));
      t[r] = lut_slot(prmt(o1[r], laneoff, sel));
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // k-slots (2c, 2c+1) <- elements 8bb+4hh+{0,1}; (2c+8, 2c+9) <- +{2,3}
      uint32_t a[4];
      a[0] = prmt(s[4 * hh + 0], s[4 * hh + 1], 0x5410u);   // row rho
      a[1] = prmt(t[4 * hh + 0], t[4 * hh + 1], 0x7632u);   // row rho2
      a[2] = prmt(s[4 * hh + 2], s[4 * hh + 3], 0x5410u);
      a[3] = prmt(t[4 * hh + 2], t[4 * hh + 3], 0x7632u);
      mma16816(acc[0][hh], a, hh ? X0[bb].z : X0[bb].x, hh ? X0[bb].w : X0[bb].y);
      mma16816(acc[1][hh], a, hh ? X1[bb].z : X1[bb].x, hh ? X1[bb].w : X1[bb].y);
    }
    ld_x16(X0[bb], x0n + bb, p0);
    ld_x16(X1[bb], x1n + bb, p1);
  }
}

// The same for a q <= 3 block with pair tables: byte bb of o[r], r even, is
// the pair index of elements 8bb + r and 8bb + r + 1 (the transposes' upper
// rows are the plane words shifted by one element), so one lookup returns both
// fp16 weights of an A-register and no packing is needed; row rho2's indices
// carry bit 7 (its table sits 128 lines up).
__device__ __forceinline__ void word_mma_pair(const uint32_t (&o0)[8], const uint32_t (&o1)[8], uint32_t laneoff,
                                              uint4 (&X0)[4], uint4 (&X1)[4],
                                              const uint4* x0n, const uint4* x1n, bool p0, bool p1,
                                              float (&acc)[2][2][4]) {
#pragma unroll
  for (int bb = 0; bb < 4; ++bb) {
    const uint32_t sel = 0x7604u | (static_cast<uint32_t>(bb) << 4);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t a[4];
      a[0] = lut_slot(prmt(o0[4 * hh + 0], laneoff, sel));    // row rho, elements 8bb+4hh+{0,1}
      a[2] = lut_slot(prmt(o0[4 * hh + 2], laneoff, sel));    // row rho, elements +{2,3}
      a[1] = lut_slot(prmt(o1[4 * hh + 0], laneoff, sel));    // row rho2
      a[3] = lut_slot(prmt(o1[4 * hh + 2], laneoff, sel));
      mma16816(acc[0][hh], a, hh ? X0[bb].z : X0[bb].x, hh ? X0[bb].w : X0[bb].y);
      mma16816(acc[1][hh], a, hh ? X1[bb].z : X1[bb].x, hh ? X1[bb].w : X1[bb].y);
    }
    ld_x16(X0[bb], x0n + bb, p0);
    ld_x16(X1[bb], x1n + bb, p1);
  }
}

// Where the warp's ring fetch stands: item (this CTA's local index), unit,
// end of the warp's units in that item, and what issuing a unit needs.  A unit
// is one word pair (64 k) of the tile's two 32-row groups; in the page layout
// each (plane, group, word pair) is 256 contiguous bytes, so lane l copies 16
// bytes: rows 2(l%16), 2(l%16)+1 of group l/16.
struct Fetch {
  int item, u, end, q;
  size_t off;        // page word offset of this lane's 16 bytes at unit 0
  uint32_t desc;     // shared address of the item's descriptor
};

__device__ __forceinline__ void fetch_enter(Fetch& f, const Fwd& p, const Smem& sm, int item, int warp,
                                            int lane) {
  const int sl = item % kSlots;
  const ItemInfo& it = reinterpret_cast<const ItemInfo*>(sm.rest + kItemOff)[sl];
  const BlockDesc& d = *reinterpret_cast<const BlockDesc*>(piece(sm.table, kPieceDesc + sl));
  f.item = item;
  f.desc = smem_addr(&d);
  const bool ok = it.valid && desc_ok(p, d, it.kind);
  warp_units(d, ok, warp, f.u, f.end);
  const int h = lane >> 4;
  int grp;   // 32-row group of row half h
  if (it.kind == PW_KIND_GATE_UP) grp = h ? p.I / 32 + it.tile : it.tile;
  else grp = 2 * it.tile + h;
  f.q = d.q;
  f.off = static_cast<size_t>(grp) * static_cast<size_t>(d.K >> 6) * 64 + (lane & 15) * 4;
}

// Issues ring stages until kStages units are in flight or the next unit
// belongs to an item that is not known yet (an item is known once its
// descriptor is in shared memory and it exists: items up to `known`).
// `issued` counts units issued by this warp.  The caller has synchronised the
// warp after the last read of the stage that the next issue overwrites.
__device__ __forceinline__ void fetch_fill(Fetch& f, const Fwd& p, const Smem& sm, int known, int consumed,
                                           int& issued, int warp, int lane, uint32_t ring) {
  while (issued < consumed + kStages) {
    while (f.u == f.end) {   // the warp has no more units in this item
      if (f.item + 1 > known) return;
      fetch_enter(f, p, sm, f.item + 1, warp, lane);
    }
    // plane p of a q-plane item goes to stage slot 8 - q + p, so that plane
    // q-1-r is always slot 7-r; the slots below 8 - q are zeroed
    const uint32_t dst = ring + (issued % kStages) * kStageBytes + (lane >> 4) * 256 + (lane & 15) * 16;
    const size_t w = f.off + static_cast<size_t>(f.u) * 64;
    const int lo = PW_MAX_BITS - f.q;
#pragma unroll
    for (int sl = 0; sl < PW_MAX_BITS; ++sl) {
      if (sl >= lo) {
        uint64_t base;
        asm volatile("ld.shared.u64 %0, [%1];" : "=l"(base) : "r"(f.desc + (sl - lo) * 8));
        const uint32_t* src = reinterpret_cast<const uint32_t*>(base) + w;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst + sl * 512), "l"(src) : "memory");
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst + sl * 512), "r"(0u) : "memory");
      }
    }
    cp_commit();
    ++issued;
    ++f.u;
  }
}

// 16-byte part of a block's descriptor: from the shared cache or global memory.
__device__ __forceinline__ uint4 desc_part(const Fwd& p, const Smem& sm, bool cached, int e, int kind, int part) {
  if (cached) return reinterpret_cast<const uint4*>(piece(sm.table, kPieceCache + 2 * e + kind))[part];
  return ld_nc16(reinterpret_cast<const uint4*>(block_desc(p, e, kind)) + part);
}

// ------------------------------------------------------------------ fused layer

constexpr int kSpinLimit = 1 << 22;   // ~0.3 s of polling before a wait gives up

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

// The item a ticket-word update returned: its count under this forward's tag,
// or -1 when the word holds another tag or the set-up sentinel.
__device__ __forceinline__ int ticket_of(const Fwd& p, unsigned long long old) {
  if ((old & ~kCountMask) != p.tag) return -1;
  const unsigned long long c = old & kCountMask;
  return c == kSetupCount ? -1 : static_cast<int>(c);
}

// First claim of a CTA (one thread), right after the dependency wait: the
// first CTA to find the ticket word under another tag sets the forward up
// (returns 1; the caller resets the counters and then publishes the count);
// every other CTA waits (bounded) for the published tag and takes two tickets
// (returns 0 with *first = the first ticket, or -1 when the wait gave up).
__device__ int claim_first(const Fwd& p, int* first) {
  unsigned long long v = ld_acquire_u64(p.sync);
  if ((v & ~kCountMask) != p.tag && cas_acq_rel_u64(p.sync, v, p.tag | kSetupCount) == v) return 1;
  for (int i = 0; i < kSpinLimit; ++i) {
    v = ld_acquire_u64(p.sync);
    if ((v & ~kCountMask) == p.tag && (v & kCountMask) != kSetupCount) {
      *first = ticket_of(p, add_relaxed_u64(p.sync, 2));
      return *first >= 0 ? 0 : -1;
    }
    __nanosleep(64);
  }
  return -1;
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
__global__ void __launch_bounds__(kThreads, 1) k_layer(Fwd p) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Smem sm = smem_layout();
  int* rs = reinterpret_cast<int*>(sm.rest + kRouteOff);
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
  int* cum_gu = reinterpret_cast<int*>(sm.rest + kCumOff);
  int* cum_dn = cum_gu + (kMaxE + 1);
  ItemInfo* s_item = reinterpret_cast<ItemInfo*>(sm.rest + kItemOff);
  int* s_int = reinterpret_cast<int*>(s_item + kSlots);

  Plan pl;
  pl.tiles_gu = p.I / kGateUpTileRows;
  pl.tiles_dn = p.H / kDownTileRows;
  int* expert_done = reinterpret_cast<int*>(p.sync + 1);
  int* tile_done = expert_done + p.E;

  // The launch lets the next forward on the stream start on SMs this grid frees
  // (programmatic dependent launch): that forward routes its own batch while
  // this one finishes, and waits for it before touching the workspace.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) s_int[0] = 0;   // NaN logit seen
  // every block descriptor of the layer into shared memory (when they fit),
  // in flight while the batch is routed
  const bool cached = 2 * p.E <= kCacheBlocks;
  if (cached)
    for (int i = tid; i < 2 * p.E * 8; i += kThreads)
      cp_async16(piece(sm.table, kPieceCache + (i >> 3)) + (i & 7) * 16,
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
        cum_dn[a] = (run + incl - np) * pl.tiles_dn;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  cp_wait<0>();   // the descriptor cache
  __syncthreads();
  pl.cum_gu = cum_gu;
  pl.cum_dn = cum_dn;
  pl.total_gu = cum_gu[pl.nact];
  pl.total = pl.total_gu + cum_dn[pl.nact];
  pl.down_per_tile = pl.tiles_dn > 0 ? cum_dn[pl.nact] / pl.tiles_dn : 0;

  // the previous kernel on the stream (possibly the previous forward, using the
  // same workspace) has finished and its writes are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) s_int[3] = claim_first(p, &s_int[2]);
  __syncthreads();
  const int role = s_int[3];
  if (role == 1) {
    // this CTA sets the forward up: counters to zero, the status word, then the
    // ticket word's count (tickets 0 and 1 are this CTA's)
    for (int i = tid; i < p.E + pl.tiles_dn; i += kThreads) expert_done[i] = 0;
    if (tid == 0) p.status[0] = s_int[0] ? PW_STATUS_NAN_LOGIT : 0u;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release_u64(p.sync, p.tag | 2ull);
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
    // the set-up never published (bounded wait): leave every item to the others
    if (tid == 0) atomicOr(p.status, PW_STATUS_TIMEOUT);
    return;
  }
  __syncthreads();
  // items of the first two tickets and their descriptors
  if (tid < 2) s_item[tid] = item_of(s_int[2] + tid, pl, r);
  __syncthreads();
  if (warp == 0 && lane < 16) {
    const int sl = lane >> 3, part = lane & 7;
    if (s_item[sl].valid)
      reinterpret_cast<uint4*>(piece(sm.table, kPieceDesc + sl))[part] =
          desc_part(p, sm, cached, s_item[sl].expert, s_item[sl].kind, part);
  }
  __syncthreads();
  const uint32_t ring = ring_of(sm, warp);
  const uint32_t laneoff = sm.table_hi | (static_cast<uint32_t>(lane) * 4u);
  Fetch f;
  int issued = 0, consumed = 0;
  LutRegs lr;
  if (s_item[0].valid) {
    const BlockDesc& d0 = *reinterpret_cast<const BlockDesc*>(piece(sm.table, kPieceDesc));
    int rho, rho2;
    lane_rows(p, s_item[0], lane, rho, rho2);
    const bool ok0 = desc_ok(p, d0, s_item[0].kind);
    if (ok0) lut_load(lr, d0, rho, rho2, warp);
    fetch_enter(f, p, sm, 0, warp, lane);
    fetch_fill(f, p, sm, s_item[1].valid ? 1 : 0, consumed, issued, warp, lane, ring);
    if (ok0) lut_store(sm.table, lr, d0.q, lane, warp);
  }
  __syncthreads();   // the first item's tables are complete

  // thread 0: the last down item's tile and the count its update returned,
  // looked at only at the next item boundary
  int pending_tile = -1, pending_old = -1;
  for (int i = 0; s_item[i % kSlots].valid; ++i) {
    const int sl = i % kSlots;
    const ItemInfo it = s_item[sl];
    const BlockDesc& d = *reinterpret_cast<const BlockDesc*>(piece(sm.table, kPieceDesc + sl));
    const bool gu = it.kind == PW_KIND_GATE_UP;
    const bool ok = desc_ok(p, d, it.kind);
    if (!ok && tid == 0) atomicOr(p.status, PW_STATUS_BAD_DESC);

    // item i+2's ticket: claimed now, looked at when this item ends
    const int sl1 = (i + 1) % kSlots, sl2 = (i + 2) % kSlots;
    const ItemInfo it1 = s_item[sl1];
    unsigned long long claim = 0;
    if (tid == 0 && it1.valid) claim = add_relaxed_u64(p.sync, 1);
    const int known = it1.valid ? i + 1 : i;   // the ring may run into item i+1
    // item i+1's tables, into registers until this item's lookups are done
    const BlockDesc& d1 = *reinterpret_cast<const BlockDesc*>(piece(sm.table, kPieceDesc + sl1));
    const bool ok1 = it1.valid && desc_ok(p, d1, it1.kind);
    if (ok1) {
      int rho, rho2;
      lane_rows(p, it1, lane, rho, rho2);
      lut_load(lr, d1, rho, rho2, warp);
    }

    int u0, u1;
    warp_units(d, ok, warp, u0, u1);
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
      const uint4* xr[2] = {nullptr, nullptr};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = 2 * j + tl;
        if (tl >= 0 && tl <= 1 && tok < it.n) {
          const int pos = it.off + tok;
          xr[j] = reinterpret_cast<const uint4*>(gu ? p.x + static_cast<size_t>(r.perm[pos] / p.k) * p.H
                                                    : p.hh + static_cast<size_t>(pos) * p.I);
        }
      }
      if (!gu) {   // h of this expert comes from its gate_up items
        if (lane == 0 && !wait_ge(&expert_done[it.expert], it.need)) atomicOr(p.status, PW_STATUS_TIMEOUT);
        __syncwarp();
      }
      uint4 X0[4], X1[4];
      const int w0 = u0 * kUnitWords, w1 = u1 * kUnitWords;
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        X0[k4] = make_uint4(0u, 0u, 0u, 0u);
        X1[k4] = make_uint4(0u, 0u, 0u, 0u);
        ld_x16(X0[k4], xr[0] + w0 * 4 + k4, xr[0] != nullptr);
        ld_x16(X1[k4], xr[1] + w0 * 4 + k4, xr[1] != nullptr);
      }
      const bool pairq = d.q <= 3;
      for (int u = u0; u < u1; ++u) {
        cp_wait_n(issued - consumed - 1);
        __syncwarp();   // every lane's copies of this stage visible; the previous stage is read
        fetch_fill(f, p, sm, known, consumed, issued, warp, lane, ring);
        const uint32_t st = ring + (consumed % kStages) * kStageBytes + lane * 8;
        ++consumed;
        if (pairq) {   // q <= 3: the q plane words sit in slots 7..5
          uint2 pa[4], pb[4];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(pa[rr].x), "=r"(pa[rr].y) : "r"(st + (7 - rr) * 512));
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(pb[rr].x), "=r"(pb[rr].y) : "r"(st + (7 - rr) * 512 + 256));
          }
#pragma unroll
          for (int wi = 0; wi < kUnitWords; ++wi) {
            const int gw = u * kUnitWords + wi;
            uint32_t o0[8], o1[8];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              o0[rr] = wi ? pa[rr].y : pa[rr].x;
              o1[rr] = wi ? pb[rr].y : pb[rr].x;
              o0[rr + 4] = o0[rr] >> 1;
              o1[rr + 4] = o1[rr] >> 1;
            }
            planes_to_indices(o0);
            planes_to_indices(o1);
#pragma unroll
            for (int rr = 0; rr < 8; rr += 2) o1[rr] |= 0x80808080u;   // rho2's table: lines + 128
            const bool more = gw + 1 < w1;
            word_mma_pair(o0, o1, laneoff, X0, X1, xr[0] + (gw + 1) * 4, xr[1] + (gw + 1) * 4,
                          more && xr[0] != nullptr, more && xr[1] != nullptr, acc);
          }
          continue;
        }
        uint2 pv0[8], pv1[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(pv0[rr].x), "=r"(pv0[rr].y) : "r"(st + (7 - rr) * 512));
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(pv1[rr].x), "=r"(pv1[rr].y) : "r"(st + (7 - rr) * 512 + 256));
        }
#pragma unroll
        for (int wi = 0; wi < kUnitWords; ++wi) {
          const int gw = u * kUnitWords + wi;
          uint32_t o0[8], o1[8];
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            o0[rr] = wi ? pv0[rr].y : pv0[rr].x;
            o1[rr] = wi ? pv1[rr].y : pv1[rr].x;
          }
          planes_to_indices(o0);
          planes_to_indices(o1);
          const bool more = gw + 1 < w1;
          word_mma(o0, o1, laneoff, X0, X1, xr[0] + (gw + 1) * 4, xr[1] + (gw + 1) * 4,
                   more && xr[0] != nullptr, more && xr[1] != nullptr, acc);
        }
      }
    }
    // keep the ring running into the next item while this one finishes
    __syncwarp();
    fetch_fill(f, p, sm, known, consumed, issued, warp, lane, ring);

    // ---- partial sums: piece(warp * 8 + half * 4 + token)[lane]
    {
      float* red = reinterpret_cast<float*>(piece(sm.table, kPieceRed + warp * 8));
      float v[8];
#pragma unroll
      for (int j = 0; j < 2; ++j) {   // column set j: tokens 2j, 2j+1 of the rows rho / rho2
        v[2 * j] = acc[j][0][0] + acc[j][1][0];
        v[2 * j + 1] = acc[j][0][1] + acc[j][1][1];
        v[4 + 2 * j] = acc[j][0][2] + acc[j][1][2];
        v[4 + 2 * j + 1] = acc[j][0][3] + acc[j][1][3];
      }
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) red[k8 * (kLine / 4) + lane] = v[k8];
    }
    // a down tile whose last item completed with the previous item: combine it now;
    // item i+2 from the ticket claimed at this item's start
    if (tid == 0) {
      s_int[1] = pending_old == pl.down_per_tile - 1 ? pending_tile : -1;
      s_item[sl2] = it1.valid ? item_of(ticket_of(p, claim), pl, r) : ItemInfo{};
    }
    __syncthreads();   // every lookup of this item is done; partials visible
    if (s_int[1] >= 0) {
      const int r0 = s_int[1] * kDownTileRows;
      combine_rows(p, r.w, r.inv, r0, min(r0 + kDownTileRows, p.H), 0, p.T, tid, blockDim.x);
    }
    pending_tile = -1;
    pending_old = -1;

    if (ok1) lut_store(sm.table, lr, d1.q, lane, warp);
    if (warp == 0 && lane < 8 && s_item[sl2].valid)
      reinterpret_cast<uint4*>(piece(sm.table, kPieceDesc + sl2))[lane] =
          desc_part(p, sm, cached, s_item[sl2].expert, s_item[sl2].kind, lane);
    auto red_at = [&](int w, int k8, int l) {
      return reinterpret_cast<const float*>(piece(sm.table, kPieceRed + w * 8 + k8))[l];
    };
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
        p.y[static_cast<size_t>(it.off + t) * p.H + it.tile * kDownTileRows + hf * 32 + l] = yv;
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
  if (s_int[1] >= 0) {
    const int r0 = s_int[1] * kDownTileRows;
    combine_rows(p, r.w, r.inv, r0, min(r0 + kDownTileRows, p.H), 0, p.T, tid, blockDim.x);
  }
  cp_wait<0>();
}

constexpr int kMaxDevices = 64;
int g_fused[kMaxDevices] = {};   // co-resident grid of the fused layer per device

}  // namespace

cudaError_t launch_layer_fused(const Fwd& p, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (p.H % kDownTileRows != 0 || p.I % kGateUpTileRows != 0) return cudaErrorInvalidValue;
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
  return cudaLaunchKernelEx(&cfg, k_layer, p);
}

}  // namespace pw
