// Internal declarations shared by the host runtime (pw_runtime.cpp) and the
// kernels (pw_*.cu).  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pw.h"

#if defined(__CUDACC__)
#define PW_HD __host__ __device__
#else
#define PW_HD
#endif

namespace pw {

// Device-resident descriptor of one linear block: the page-table entry the
// kernels read (committed q_i and page addresses), 128 bytes, one per
// (layer, expert, kind).  Written only by stream-ordered commits.
struct alignas(128) BlockDesc {
  const uint32_t* planes[PW_MAX_BITS];  // plane pages; planes[p] valid for p < q
  const uint16_t* lut;                  // LUT_q, [R][2^q] fp16
  int32_t q;                            // committed bitwidth (0 = not registered)
  int32_t R, K;
  int32_t n_bits;
  int32_t b_min;
  int32_t pad[7];
};
static_assert(sizeof(BlockDesc) == 128, "descriptor size");

PW_HD inline size_t desc_index(int layer, int expert, int kind, int E) {
  return (static_cast<size_t>(layer) * E + expert) * 2 + kind;
}

// Workspace layout.  Every section starts on a 256-byte boundary.
struct Workspace {
  size_t status;     // uint32 status word (256 B section)
  size_t topk_idx;   // int32 [T*k]
  size_t topk_w;     // f32 [T*k]
  size_t counts;     // int32 [E]
  size_t offsets;    // int32 [E+1]
  size_t perm;       // int32 [T*k]
  size_t inv;        // int32 [T*k]
  size_t active;     // int32 [2][E+1]: active experts (count, ids); same, cost-sorted
  size_t sync;       // fused path: 64-bit ticket word, then int32 gate_up items done per
                     // expert, down items done per 64-row tile of H, CTAs finished
  size_t hh;         // fp16 [T*k][I] in perm order
  size_t xp;         // fp16 [T*k][H] token rows in perm order (prefill GEMMs)
  size_t y;          // f32 [T*k][H] in perm order
  size_t y_part;     // f32 [down_splits][T*k][H]: partial y of K-split down items (decode path)
  size_t x_in;       // fp16 [T][H]   (host-input staging)
  size_t logits_in;  // f32 [T][E]
  size_t resid_in;   // fp16 [T][H]
  size_t out_stage;  // fp16 [T][H]
  size_t total;
};

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// The decode path's batches (T <= 64 tokens, T*k <= 256 routed pairs).
PW_HD inline bool fused_batch(int T, int k) { return T <= 64 && T * k <= 256; }

// Largest K-split of a decode down item (64 rows x K = I) that the workspace
// makes room for: about I / H parts, so that a down item costs about as much
// as a gate_up item (64 rows x H), as long as every part keeps at least 24
// word pairs (2 per K-warp); 1 when I <= H.  The decode kernel uses fewer
// parts when the routed batch already gives enough down items.
PW_HD inline int down_splits(int H, int I) {
  int s = (I + H / 2) / H;
  const int cap = (I / 64) / 24;
  if (s > cap) s = cap;
  return s < 1 ? 1 : s;
}

inline Workspace workspace_layout(int T, int E, int k, int H, int I) {
  Workspace w{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
  const size_t P = static_cast<size_t>(T) * k;
  w.status = take(256);
  w.topk_idx = take(P * 4);
  w.topk_w = take(P * 4);
  w.counts = take(static_cast<size_t>(E) * 4);
  w.offsets = take(static_cast<size_t>(E + 1) * 4);
  w.perm = take(P * 4);
  w.inv = take(P * 4);
  w.active = take(static_cast<size_t>(E + 1) * 2 * 4);
  w.sync = take(8 + static_cast<size_t>(E + (H + 63) / 64 + 1) * 4);
  w.hh = take(P * I * 2);
  w.xp = take(P * H * 2);
  w.y = take(P * H * 4);
  const int S = fused_batch(T, k) ? down_splits(H, I) : 1;
  w.y_part = S > 1 ? take(static_cast<size_t>(S) * P * H * 4) : w.y;
  w.x_in = take(static_cast<size_t>(T) * H * 2);
  w.logits_in = take(static_cast<size_t>(T) * E * 4);
  w.resid_in = take(static_cast<size_t>(T) * H * 2);
  w.out_stage = take(static_cast<size_t>(T) * H * 2);
  w.total = o;
  return w;
}

// Arguments of one forward pass, resolved on the host.
struct ForwardArgs {
  const BlockDesc* desc;   // device descriptor array base
  int layer, E, H, I;
  const uint16_t* x;       // [T][H] fp16
  const float* logits;     // [T][E]
  int T, top_k, renorm;
  const uint16_t* residual;
  uint16_t* out;
  int32_t* user_idx;
  float* user_w;
  int32_t* user_offsets;
  int32_t* user_perm;
  unsigned char* ws;       // workspace base
  Workspace lay;
  cudaEvent_t prof[5];     // boundary events (pw_profile_attach), or all null
  float* stats;            // routing-mass statistics [L][E] (pw_stats_attach), or null
  float stats_alpha;
};

// Host helpers (pw_runtime.cpp): sets this thread's pw_last_error message and
// returns `code`; reads a table's expert count and sizes.
int set_error(int code, const char* msg);
int table_shape(const pw_table* t, int* E, int* H, int* I);

// Kernel launchers (pw_kernels.cu).  Return cudaSuccess or the launch error.
cudaError_t launch_commit(BlockDesc* dst, const BlockDesc& value, cudaStream_t s);

// Up to kCommitBatch descriptor writes carried by value in one launch.
constexpr int kCommitBatch = 192;
struct CommitBatch {
  int32_t n;
  uint32_t index[kCommitBatch];       // desc_index of each block
  uint32_t words[kCommitBatch][32];   // the 128-byte descriptors
};
static_assert(sizeof(CommitBatch) < 32000, "kernel parameter block limit");
cudaError_t launch_commit_batch(BlockDesc* table, const CommitBatch& b, cudaStream_t s);
cudaError_t launch_forward(const ForwardArgs& a, cudaStream_t s);

}  // namespace pw
