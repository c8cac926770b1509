// Device-side parameter block and helpers shared by the kernel files.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "pw_internal.h"

namespace pw {

// Everything one forward pass needs on the device, resolved by the host.
struct Fwd {
  const BlockDesc* desc;
  int layer, E, H, I, T, k, renorm;
  const __half* x;          // [T][H] fp16
  const float* logits;      // [T][E]
  const __half* residual;   // [T][H] or null
  __half* out;              // [T][H]
  int32_t* user_idx;
  float* user_w;
  int32_t* user_offsets;
  int32_t* user_perm;
  uint32_t* status;         // status word: low 32 bits of a tagged 64-bit word (see below)
  int32_t* idx;             // [T*k]
  float* w;                 // [T*k]
  int32_t* counts;          // [E]
  int32_t* offsets;         // [E+1]
  int32_t* perm;            // [T*k]
  int32_t* inv;             // [T*k]
  int32_t* active;          // [E+1] active experts: count, then ids (expert order)
  unsigned long long* sync; // fused path: [0] the ticket word; from byte 8, int32 counters:
                            // gate_up items done per expert [E], then down items done
                            // per 64-row tile of H
  unsigned long long tag;   // this forward's tag (bits 24..63): never 0, never repeated
  __half* hh;               // [T*k][I] h (fp16) in permuted order
  __half* xp;               // [T*k][H] token rows in permuted (expert) order, prefill GEMMs
  float* y;                 // [T*k][H]
  float* y_part;            // [ksplit][T*k][H] partial y of K-split down items (y when ksplit = 1)
  int ksplit;               // K-splits of a decode down item
  float* stats;             // [L][E] routing-mass moving average, or null
  float stats_alpha;        // its update weight
};

// The fused forward's ticket word.  A forward finds its workspace as the
// caller left it (fresh memory, an earlier forward's leftovers, anything), so
// nothing in it can be trusted until this forward has reset it.  The ticket
// word (64 bits) carries the forward's tag in bits 24..63 and a count in bits
// 0..23.  The first CTA to find the word under another tag swaps in the tag
// with the set-up bit (bit 23) as count and takes tickets 0 and 1; CTAs
// arriving meanwhile add their claims to the count at once (their tickets
// follow) but touch no counter or status word until the set-up CTA, having
// reset the forward's counters and status, clears the set-up bit.  The tag is
// a fixed byte 0xA5 above a 32-bit forward counter, so no index, count, small
// integer or float the workspace could hold (and no earlier forward's word)
// reads as the current tag.
constexpr unsigned long long kTagShift = 24;
constexpr unsigned long long kCountMask = (1ull << kTagShift) - 1;
constexpr unsigned long long kSetupBit = 1ull << 23;   // "being set up"

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* ptr) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* ptr, unsigned long long v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(ptr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long cas_acq_rel_u64(unsigned long long* ptr, unsigned long long cmp,
                                                              unsigned long long val) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;"
               : "=l"(old) : "l"(ptr), "l"(cmp), "l"(val) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* ptr) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void add_release_u64(unsigned long long* ptr, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(ptr), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long add_relaxed_u64(unsigned long long* ptr, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(ptr), "l"(v) : "memory");
  return old;
}

// Device-side bounds checks of the PW_CHECK build (libpw_check.so): a failed
// check sets PW_STATUS_BOUNDS and the caller skips the access; the kernels
// never trap.  In the normal build the checks compile away.
#ifdef PW_CHECK
__device__ __forceinline__ bool pw_in_bounds(const Fwd& p, bool ok, bool report) {
  if (!ok && report) atomicOr(p.status, PW_STATUS_BOUNDS);
  return ok;
}
#define PW_BOUNDS(p, cond, report) ::pw::pw_in_bounds((p), (cond), (report))
#else
#define PW_BOUNDS(p, cond, report) true
#endif

__device__ __forceinline__ const BlockDesc* block_desc(const Fwd& p, int e, int kind) {
  return p.desc + desc_index(p.layer, e, kind, p.E);
}

// The whole decode layer (routing, gate_up, down, combine) in one persistent
// launch; for batches of at most kFusedMaxT tokens.
constexpr int kFusedMaxT = 64;
cudaError_t launch_layer_fused(const Fwd& p, cudaStream_t s);
// Tensor-core GEMM of one block kind over all experts (prefill-sized batches);
// gate_up also gathers the token rows into expert order first.
cudaError_t launch_prefill(const Fwd& p, int kind, cudaStream_t s);

}  // namespace pw
