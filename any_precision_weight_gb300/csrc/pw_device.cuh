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
  uint32_t* status;         // status word; counters follow
  int32_t* idx;             // [T*k]
  float* w;                 // [T*k]
  int32_t* counts;          // [E]
  int32_t* offsets;         // [E+1]
  int32_t* perm;            // [T*k]
  int32_t* inv;             // [T*k]
  int32_t* active;          // [E+1] active experts: count, then ids (expert order)
  int32_t* act_lpt;         // [E+1] the same, most expensive gate_up block first
  int32_t* sync;            // fused path: [0] ready epoch, [1] work queue,
                            // [2, 2+E) gate_up tiles done per expert, then
                            // down items done per 32-row tile of H
  uint32_t epoch;           // nonzero, differs between consecutive fused forwards
  __half* hh;               // [T*k][I] h (fp16) in permuted order
  __half* xp;               // [T*k][H] token rows in permuted (expert) order, prefill GEMMs
  float* y;                 // [T*k][H]
  float* stats;             // [L][E] routing-mass moving average, or null
  float stats_alpha;        // its update weight
};

// Work-queue counters live right after the status word.
constexpr int kCtrGateUp = 1;
constexpr int kCtrDown = 2;

__device__ __forceinline__ const BlockDesc* block_desc(const Fwd& p, int e, int kind) {
  return p.desc + desc_index(p.layer, e, kind, p.E);
}

// The whole decode layer (routing, gate_up, down, combine) in one cooperative
// persistent launch; for batches of at most kFusedMaxT tokens.
constexpr int kFusedMaxT = 64;
cudaError_t launch_layer_fused(const Fwd& p, cudaStream_t s);
// Tensor-core GEMM of one block kind over all experts (prefill-sized batches);
// gate_up also gathers the token rows into expert order first.
cudaError_t launch_prefill(const Fwd& p, int kind, cudaStream_t s);

}  // namespace pw
