// Host runtime of the fused APL MoE layer: bit-plane packer and table builder,
// the weight page table with its stream-ordered commit and asynchronous reload
// protocol, and the forward entry points.
//
// Source of the behaviour: PagedWeight technical summary, core components
// section 1 ("Paged Weight Representation": per-block desired/committed
// bitwidth, page states GPU / CPU / in transfer) and section 3 ("Asynchronous
// Page Movement": offload to CPU memory, asynchronous reload, commits only at
// safe boundaries so inference is never interrupted).

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "pw_internal.h"

namespace {

thread_local std::string g_err;
thread_local cudaEvent_t g_prof[5] = {};   // one-shot, see pw_profile_attach

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PW_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- fp16 <-> fp64

double half_to_double(uint16_t h) {
  const int sign = h >> 15;
  const int ex = (h >> 10) & 31;
  const int man = h & 1023;
  double v;
  if (ex == 0) {
    v = std::ldexp(static_cast<double>(man), -24);
  } else if (ex == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(1024 + man), ex - 25);
  }
  return sign ? -v : v;
}

// Round to the nearest fp16, ties to even.
uint16_t double_to_half(double x) {
  if (std::isnan(x)) return 0x7E00;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (a >= 65520.0) return sign | 0x7C00;          // rounds to infinity
  if (a < std::ldexp(1.0, -14)) {                   // subnormal range, units of 2^-24
    const double m = std::nearbyint(std::ldexp(a, 24));   // default mode: half to even
    return sign | static_cast<uint16_t>(m);         // m == 1024 encodes 2^-14 exactly
  }
  int e2;
  const double f = std::frexp(a, &e2);              // a = f * 2^e2, f in [0.5, 1)
  int E = e2 - 1;                                   // a = s * 2^E, s in [1, 2)
  double mant = std::nearbyint((f * 2.0 - 1.0) * 1024.0);
  if (mant >= 1024.0) { mant = 0; E += 1; }
  if (E + 15 >= 31) return sign | 0x7C00;
  return sign | static_cast<uint16_t>(((E + 15) << 10) | static_cast<int>(mant));
}

// ---------------------------------------------------------------- table state

struct BlockState {
  bool registered = false;
  int n_bits = 0, b_min = 0, R = 0, K = 0;
  const uint32_t* host_planes = nullptr;
  const uint16_t* host_luts = nullptr;
  void* pages[PW_MAX_BITS] = {};
  void* d_luts = nullptr;
  int q = 0;                 // committed bitwidth (host mirror of the descriptor)
  int resident = 0;          // planes [0, resident) and tables b <= resident on device
  int pending = 0;           // target of the reload in flight (0: none)
  bool failed = false;       // the pending reload could not be enqueued or failed
  cudaEvent_t ev = nullptr;  // recorded after the reload's copies
};

}  // namespace

struct pw_table {
  int L = 0, E = 0, H = 0, I = 0;
  pw::BlockDesc* d_desc = nullptr;
  std::vector<BlockState> blocks;
  std::mutex mu;
  bool fail_next_reload = false;   // test hook, see pw_debug_fail_next_reload
};

namespace {

BlockState* block_of(pw_table* t, int layer, int expert, int kind) {
  if (!t || layer < 0 || layer >= t->L || expert < 0 || expert >= t->E || kind < 0 || kind > 1)
    return nullptr;
  return &t->blocks[pw::desc_index(layer, expert, kind, t->E)];
}

pw::BlockDesc make_desc(const BlockState& b, int q) {
  pw::BlockDesc d{};
  for (int p = 0; p < PW_MAX_BITS; ++p)
    d.planes[p] = (p < b.resident) ? static_cast<const uint32_t*>(b.pages[p]) : nullptr;
  d.lut = reinterpret_cast<const uint16_t*>(static_cast<const unsigned char*>(b.d_luts) +
                                            pw_lut_offset(b.R, b.b_min, q));
  d.q = q;
  d.R = b.R;
  d.K = b.K;
  d.n_bits = b.n_bits;
  d.b_min = b.b_min;
  return d;
}

int write_desc(pw_table* t, int layer, int expert, int kind, const BlockState& b, int q,
               cudaStream_t s) {
  const pw::BlockDesc d = make_desc(b, q);
  const cudaError_t e =
      pw::launch_commit(t->d_desc + pw::desc_index(layer, expert, kind, t->E), d, s);
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  return PW_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

namespace pw {

int set_error(int code, const char* msg) {
  g_err = msg;
  return code;
}

int table_shape(const pw_table* t, int* E, int* H, int* I) {
  if (!t) return PW_EINVAL;
  *E = t->E;
  *H = t->H;
  *I = t->I;
  return PW_OK;
}

}  // namespace pw

extern "C" {

const char* pw_last_error(void) { return g_err.c_str(); }

size_t pw_plane_bytes(int R, int K) {
  if (R <= 0 || K <= 0) return 0;
  return static_cast<size_t>(R) * K / 8;
}

size_t pw_lut_offset(int R, int b_min, int b) {
  size_t entries = 0;
  for (int c = b_min; c < b; ++c) entries += static_cast<size_t>(1) << c;
  return static_cast<size_t>(R) * entries * 2;
}

size_t pw_lut_bytes(int R, int b_min, int n_bits) {
  if (R <= 0 || b_min < 1 || n_bits > PW_MAX_BITS || b_min > n_bits) return 0;
  return pw_lut_offset(R, b_min, n_bits + 1);
}

int pw_pack(const uint8_t* idx, int R, int K, int n_bits, const uint16_t* parent_lut,
            int b_min, uint32_t* planes_out, uint16_t* luts_out) {
  if (!idx || !parent_lut || !planes_out || !luts_out) return fail(PW_EINVAL, "pw_pack: null pointer");
  if (R < 1 || K < 32 || K % 32)
    return fail(PW_EINVAL, "pw_pack: need R >= 1, K >= 32, K %% 32 == 0");
  if (n_bits < 1 || n_bits > PW_MAX_BITS || b_min < 1 || b_min > n_bits)
    return fail(PW_EINVAL, "pw_pack: need 1 <= b_min <= n_bits <= 8");
  const int W = K / 32;
  const size_t plane_words = static_cast<size_t>(R) * W;
  const int limit = 1 << n_bits;
  unsigned nthr = std::thread::hardware_concurrency();
  if (nthr == 0) nthr = 1;
  if (static_cast<size_t>(R) * K < (1u << 20)) nthr = 1;
  if (nthr > 64) nthr = 64;
  std::vector<int> bad_row(nthr, -1);
  auto work = [&](unsigned tid) {
    for (int r = static_cast<int>(tid); r < R; r += static_cast<int>(nthr)) {
      const uint8_t* row = idx + static_cast<size_t>(r) * K;
      for (int w = 0; w < W; ++w) {
        uint32_t words[PW_MAX_BITS] = {};
        for (int j = 0; j < 32; ++j) {
          const unsigned v = row[32 * w + j];
          if (static_cast<int>(v) >= limit) { bad_row[tid] = r; return; }
          for (int p = 0; p < n_bits; ++p) words[p] |= ((v >> (n_bits - 1 - p)) & 1u) << j;
        }
        for (int p = 0; p < n_bits; ++p)
          planes_out[p * plane_words + static_cast<size_t>(r) * W + w] = words[p];
      }
      // tables LUT_b for b = b_min..n_bits
      const uint16_t* par = parent_lut + static_cast<size_t>(r) * limit;
      for (int b = b_min; b <= n_bits; ++b) {
        uint16_t* dst = luts_out + pw_lut_offset(R, b_min, b) / 2 + static_cast<size_t>(r) * (1u << b);
        const int g = 1 << (n_bits - b);
        for (int j = 0; j < (1 << b); ++j) {
          if (g == 1) { dst[j] = par[j]; continue; }
          double s = 0.0;   // exact: a few hundred fp16 values fit in fp64's significand
          for (int i = 0; i < g; ++i) s += half_to_double(par[j * g + i]);
          dst[j] = double_to_half(s / g);
        }
      }
    }
  };
  if (nthr == 1) {
    work(0);
  } else {
    std::vector<std::thread> th;
    for (unsigned i = 0; i < nthr; ++i) th.emplace_back(work, i);
    for (auto& x : th) x.join();
  }
  for (int r : bad_row)
    if (r >= 0) return fail(PW_EINVAL, "pw_pack: row %d has an index >= 2^%d", r, n_bits);
  return PW_OK;
}

size_t pw_desc_bytes(int n_layers, int n_experts) {
  if (n_layers <= 0 || n_experts <= 0) return 0;
  return static_cast<size_t>(n_layers) * n_experts * 2 * sizeof(pw::BlockDesc);
}

int pw_table_create(pw_table** out, int n_layers, int n_experts, int H, int I, void* d_desc,
                    size_t desc_bytes, pw_stream_t s) {
  if (!out) return fail(PW_EINVAL, "pw_table_create: null out");
  *out = nullptr;
  if (n_layers < 1 || n_experts < 1 || n_experts > 256)
    return fail(PW_EINVAL, "pw_table_create: need n_layers >= 1, 1 <= n_experts <= 256");
  if (H < 128 || I < 128 || H % 128 || I % 128)
    return fail(PW_EINVAL, "pw_table_create: H and I must be positive multiples of 128");
  if (!d_desc || desc_bytes < pw_desc_bytes(n_layers, n_experts))
    return fail(PW_EINVAL, "pw_table_create: descriptor buffer smaller than pw_desc_bytes");
  if (reinterpret_cast<uintptr_t>(d_desc) % 128)
    return fail(PW_EINVAL, "pw_table_create: descriptor buffer must be 128-byte aligned");
  pw_table* t = new (std::nothrow) pw_table;
  if (!t) return fail(PW_ENOMEM, "pw_table_create: host allocation");
  t->L = n_layers;
  t->E = n_experts;
  t->H = H;
  t->I = I;
  t->d_desc = static_cast<pw::BlockDesc*>(d_desc);
  t->blocks.resize(static_cast<size_t>(n_layers) * n_experts * 2);
  const cudaError_t e = cudaMemsetAsync(d_desc, 0, pw_desc_bytes(n_layers, n_experts),
                                        reinterpret_cast<cudaStream_t>(s));
  if (e != cudaSuccess) {
    delete t;
    return cuda_fail(e, "pw_table_create: clearing descriptors");
  }
  *out = t;
  return PW_OK;
}

int pw_block_register(pw_table* t, int layer, int expert, int kind, int n_bits, int b_min,
                      const uint32_t* host_planes, const uint16_t* host_luts,
                      void* const* d_plane_pages, void* d_luts, int q_init, pw_stream_t s) {
  if (!t) return fail(PW_EINVAL, "pw_block_register: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b)
    return fail(PW_EINVAL, "pw_block_register: (layer %d, expert %d, kind %d) out of range", layer,
                expert, kind);
  if (n_bits < 1 || n_bits > PW_MAX_BITS || b_min < 1 || b_min > n_bits)
    return fail(PW_EINVAL, "pw_block_register: need 1 <= b_min <= n_bits <= 8");
  if (q_init < b_min || q_init > n_bits)
    return fail(PW_EINVAL, "pw_block_register: q_init %d outside [%d, %d]", q_init, b_min, n_bits);
  if (!host_planes || !host_luts || !d_plane_pages || !d_luts)
    return fail(PW_EINVAL, "pw_block_register: null pointer");
  if (b->pending) return fail(PW_EINVAL, "pw_block_register: a reload of this block is pending");
  const int R = kind == PW_KIND_GATE_UP ? 2 * t->I : t->H;
  const int K = kind == PW_KIND_GATE_UP ? t->H : t->I;
  for (int p = 0; p < n_bits; ++p) {
    if (p < q_init && !d_plane_pages[p])
      return fail(PW_EINVAL, "pw_block_register: plane page %d is null", p);
    if (d_plane_pages[p] && !aligned16(d_plane_pages[p]))
      return fail(PW_EINVAL, "pw_block_register: plane page %d not 16-byte aligned", p);
  }
  if (!aligned16(d_luts)) return fail(PW_EINVAL, "pw_block_register: tables not 16-byte aligned");
  BlockState nb;
  nb.registered = true;
  nb.n_bits = n_bits;
  nb.b_min = b_min;
  nb.R = R;
  nb.K = K;
  nb.host_planes = host_planes;
  nb.host_luts = host_luts;
  for (int p = 0; p < n_bits; ++p) nb.pages[p] = d_plane_pages[p];
  nb.d_luts = d_luts;
  nb.ev = b->ev;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  const size_t pb = pw_plane_bytes(R, K);
  for (int p = 0; p < q_init; ++p) {
    const cudaError_t e = cudaMemcpyAsync(nb.pages[p], host_planes + p * (pb / 4), pb,
                                          cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "pw_block_register: plane copy");
  }
  const cudaError_t e = cudaMemcpyAsync(d_luts, host_luts, pw_lut_offset(R, b_min, q_init + 1),
                                        cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "pw_block_register: table copy");
  nb.resident = q_init;
  nb.q = q_init;
  const int rc = write_desc(t, layer, expert, kind, nb, q_init, st);
  if (rc != PW_OK) return rc;
  *b = nb;
  return PW_OK;
}

int pw_reload_async(pw_table* t, int layer, int expert, int kind, int q_target, pw_stream_t copy) {
  if (!t) return fail(PW_EINVAL, "pw_reload_async: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_reload_async: block not registered");
  if (q_target < b->b_min || q_target > b->n_bits)
    return fail(PW_EINVAL, "pw_reload_async: q_target %d outside [%d, %d]", q_target, b->b_min,
                b->n_bits);
  if (b->pending && !b->failed)
    return fail(PW_EINVAL, "pw_reload_async: a reload of this block is pending");
  if (b->pending && b->failed) {     // retry after a failed reload: wait out its copies
    if (b->ev) cudaEventSynchronize(b->ev);
    b->pending = 0;
    b->failed = false;
  }
  if (q_target <= b->resident) return PW_OK;
  for (int p = b->resident; p < q_target; ++p)
    if (!b->pages[p]) return fail(PW_EINVAL, "pw_reload_async: no device page for plane %d", p);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(copy);
  if (!b->ev) {
    const cudaError_t e = cudaEventCreateWithFlags(&b->ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "pw_reload_async: event create");
  }
  b->failed = false;
  const size_t pb = pw_plane_bytes(b->R, b->K);
  cudaError_t e = cudaSuccess;
  if (t->fail_next_reload) {          // injected failure: nothing is enqueued
    t->fail_next_reload = false;
    e = cudaErrorInvalidValue;
  }
  for (int p = b->resident; p < q_target && e == cudaSuccess; ++p)
    e = cudaMemcpyAsync(b->pages[p], b->host_planes + p * (pb / 4), pb, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) {
    const size_t lo = pw_lut_offset(b->R, b->b_min, b->resident + 1);
    const size_t hi = pw_lut_offset(b->R, b->b_min, q_target + 1);
    e = cudaMemcpyAsync(static_cast<unsigned char*>(b->d_luts) + lo,
                        reinterpret_cast<const unsigned char*>(b->host_luts) + lo, hi - lo,
                        cudaMemcpyHostToDevice, st);
  }
  if (e == cudaSuccess) e = cudaEventRecord(b->ev, st);
  b->pending = q_target;
  if (e != cudaSuccess) {
    b->failed = true;
    return cuda_fail(e, "pw_reload_async: enqueue");
  }
  return PW_OK;
}

int pw_reload_query(pw_table* t, int layer, int expert, int kind) {
  if (!t) return fail(PW_EINVAL, "pw_reload_query: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_reload_query: block not registered");
  if (!b->pending) return 1;
  if (b->failed) return fail(PW_ERELOAD, "pw_reload_query: reload failed");
  const cudaError_t e = cudaEventQuery(b->ev);
  if (e == cudaSuccess) {
    b->resident = b->pending;   // copies done: visible to every later launch
    b->pending = 0;
    return 1;
  }
  if (e == cudaErrorNotReady) return 0;
  b->failed = true;
  return fail(PW_ERELOAD, "pw_reload_query: %s", cudaGetErrorString(e));
}

int pw_set_commit(pw_table* t, int layer, int expert, int kind, int q, pw_stream_t compute) {
  if (!t) return fail(PW_EINVAL, "pw_set_commit: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_set_commit: block not registered");
  if (q < b->b_min || q > b->n_bits)
    return fail(PW_EINVAL, "pw_set_commit: q %d outside [%d, %d]", q, b->b_min, b->n_bits);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(compute);
  if (q > b->resident) {
    if (!b->pending || b->pending < q)
      return fail(PW_ENOTRESIDENT, "pw_set_commit: q %d above the %d resident planes, no reload",
                  q, b->resident);
    if (b->failed) return fail(PW_ERELOAD, "pw_set_commit: the reload to %d failed", b->pending);
    const cudaError_t e = cudaStreamWaitEvent(st, b->ev, 0);
    if (e != cudaSuccess) return cuda_fail(e, "pw_set_commit: stream wait");
    // From here on the compute stream is ordered after the copies.
    b->resident = b->pending;
    b->pending = 0;
  }
  const int rc = write_desc(t, layer, expert, kind, *b, q, st);
  if (rc != PW_OK) return rc;
  b->q = q;
  return PW_OK;
}

int pw_block_state(pw_table* t, int layer, int expert, int kind, int* q, int* resident,
                   int* reload_target) {
  if (!t) return fail(PW_EINVAL, "pw_block_state: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b) return fail(PW_EINVAL, "pw_block_state: out of range");
  if (q) *q = b->registered ? b->q : 0;
  if (resident) *resident = b->registered ? b->resident : 0;
  if (reload_target) *reload_target = b->pending;
  return PW_OK;
}

int pw_debug_fail_next_reload(pw_table* t) {
  if (!t) return fail(PW_EINVAL, "pw_debug_fail_next_reload: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  t->fail_next_reload = true;
  return PW_OK;
}

int pw_table_destroy(pw_table* t) {
  if (!t) return PW_OK;
  for (auto& b : t->blocks)
    if (b.ev) {
      cudaEventSynchronize(b.ev);
      cudaEventDestroy(b.ev);
    }
  delete t;
  return PW_OK;
}

size_t pw_workspace_bytes(int T, int E, int top_k, int H, int I) {
  if (T < 0 || E < 1 || top_k < 1 || H < 1 || I < 1) return 0;
  return pw::workspace_layout(T, E, top_k, H, I).total;
}

static int forward_checks(pw_table* t, int layer, int T, int top_k, const void* ws,
                          size_t ws_bytes) {
  if (!t) return fail(PW_EINVAL, "pw_moe_forward: null table");
  if (layer < 0 || layer >= t->L)
    return fail(PW_EINVAL, "pw_moe_forward: layer %d out of range", layer);
  if (T < 0) return fail(PW_EINVAL, "pw_moe_forward: T < 0");
  if (top_k < 1 || top_k > t->E)
    return fail(PW_EINVAL, "pw_moe_forward: top_k %d outside [1, %d]", top_k, t->E);
  if (!ws || reinterpret_cast<uintptr_t>(ws) % 256)
    return fail(PW_EINVAL, "pw_moe_forward: workspace null or not 256-byte aligned");
  if (ws_bytes < pw::workspace_layout(T, t->E, top_k, t->H, t->I).total)
    return fail(PW_ENOMEM, "pw_moe_forward: workspace smaller than pw_workspace_bytes");
  for (int e = 0; e < t->E; ++e)
    for (int k = 0; k < 2; ++k)
      if (!t->blocks[pw::desc_index(layer, e, k, t->E)].registered)
        return fail(PW_EINVAL, "pw_moe_forward: block (%d, %d, %d) not registered", layer, e, k);
  return PW_OK;
}

int pw_moe_forward(pw_table* t, int layer, const void* x, const float* logits, int T, int top_k,
                   int renorm, const void* residual, void* out, int32_t* topk_idx, float* topk_w,
                   int32_t* offsets, int32_t* perm, void* workspace, size_t ws_bytes,
                   pw_stream_t compute) {
  const int rc = forward_checks(t, layer, T, top_k, workspace, ws_bytes);
  if (rc != PW_OK) return rc;
  if (T == 0) return PW_OK;
  if (!x || !logits || !out) return fail(PW_EINVAL, "pw_moe_forward: null x, logits or out");
  if (!aligned16(x) || !aligned16(out) || (residual && !aligned16(residual)))
    return fail(PW_EINVAL, "pw_moe_forward: x, residual and out must be 16-byte aligned");
  pw::ForwardArgs a{};
  a.desc = t->d_desc;
  a.layer = layer;
  a.E = t->E;
  a.H = t->H;
  a.I = t->I;
  a.x = static_cast<const uint16_t*>(x);
  a.logits = logits;
  a.T = T;
  a.top_k = top_k;
  a.renorm = renorm ? 1 : 0;
  a.residual = static_cast<const uint16_t*>(residual);
  a.out = static_cast<uint16_t*>(out);
  a.user_idx = topk_idx;
  a.user_w = topk_w;
  a.user_offsets = offsets;
  a.user_perm = perm;
  a.ws = static_cast<unsigned char*>(workspace);
  a.lay = pw::workspace_layout(T, t->E, top_k, t->H, t->I);
  for (int i = 0; i < 5; ++i) {
    a.prof[i] = g_prof[i];
    g_prof[i] = nullptr;
  }
  const cudaError_t e = pw::launch_forward(a, reinterpret_cast<cudaStream_t>(compute));
  if (e != cudaSuccess) return cuda_fail(e, "pw_moe_forward: launch");
  return PW_OK;
}

int pw_moe_forward_host(pw_table* t, int layer, const void* x_host, const float* logits_host,
                        int T, int top_k, int renorm, const void* residual_host, void* out_host,
                        void* workspace, size_t ws_bytes, pw_stream_t compute) {
  int rc = forward_checks(t, layer, T, top_k, workspace, ws_bytes);
  if (rc != PW_OK) return rc;
  if (T == 0) return PW_OK;
  if (!x_host || !logits_host || !out_host)
    return fail(PW_EINVAL, "pw_moe_forward_host: null x, logits or out");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(compute);
  const pw::Workspace lay = pw::workspace_layout(T, t->E, top_k, t->H, t->I);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const size_t xb = static_cast<size_t>(T) * t->H * 2;
  cudaError_t e = cudaMemcpyAsync(ws + lay.x_in, x_host, xb, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + lay.logits_in, logits_host, static_cast<size_t>(T) * t->E * 4,
                        cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && residual_host)
    e = cudaMemcpyAsync(ws + lay.resid_in, residual_host, xb, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "pw_moe_forward_host: input copy");
  rc = pw_moe_forward(t, layer, ws + lay.x_in, reinterpret_cast<const float*>(ws + lay.logits_in),
                      T, top_k, renorm, residual_host ? ws + lay.resid_in : nullptr,
                      ws + lay.out_stage, nullptr, nullptr, nullptr, nullptr, workspace, ws_bytes,
                      compute);
  if (rc != PW_OK) return rc;
  uint32_t status = 0;
  e = cudaMemcpyAsync(out_host, ws + lay.out_stage, xb, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&status, ws + lay.status, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "pw_moe_forward_host: output copy");
  if (status) return fail(PW_EDEVICE, "pw_moe_forward_host: device status 0x%x", status);
  return PW_OK;
}

int pw_profile_attach(void* const* events, int n_events) {
  for (int i = 0; i < 5; ++i)
    g_prof[i] = (events && n_events >= 5) ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  return PW_OK;
}

int pw_workspace_status(const void* workspace, pw_stream_t s, int* status) {
  if (!workspace || !status) return fail(PW_EINVAL, "pw_workspace_status: null pointer");
  uint32_t v = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
  cudaError_t e = cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "pw_workspace_status");
  *status = static_cast<int>(v);
  return PW_OK;
}

}  // extern "C"
