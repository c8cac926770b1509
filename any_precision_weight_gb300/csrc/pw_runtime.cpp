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
#include <algorithm>
#include <condition_variable>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <chrono>
#include <thread>
#include <vector>

#include <nvtx3/nvToolsExt.h>

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
  bool issued = false;       // the pending reload's copies and event are enqueued
  int commit_to = 0;         // submitted through the mover: commit this q on arrival
  cudaEvent_t ev = nullptr;  // recorded after the reload's copies
};

// One reload submitted to the mover.
struct MoveReq {
  int layer, expert, kind, q;
};

}  // namespace

struct pw_table {
  int L = 0, E = 0, H = 0, I = 0;
  pw::BlockDesc* d_desc = nullptr;
  std::vector<BlockState> blocks;
  std::mutex mu;
  std::condition_variable enqueued;   // signalled when a reload's enqueue phase ends
  bool fail_next_reload = false;   // test hook, see pw_debug_fail_next_reload
  float* stats = nullptr;          // routing-mass statistics [L][E] (pw_stats_attach)
  float stats_alpha = 0.f;

  // The reload mover (pw_mover_start): a host thread that takes submitted
  // reloads in order and enqueues them with a bound on the bytes in flight.
  // mover_mu guards the request queue and the mover's own fields; the table
  // lock mu guards block state and the arrival list.
  std::thread mover;
  std::mutex mover_mu;
  std::condition_variable mover_cv;
  std::deque<MoveReq> requests;
  bool mover_stop = false;
  int mover_busy = 0;                 // requests taken off the queue, not yet enqueued
  cudaStream_t mover_stream = nullptr;
  size_t mover_limit = 0;
  int mover_device = 0;
  int mover_error = PW_OK;            // first failure of the mover, reported by pw_commit_arrived
  std::string mover_error_msg;
  std::deque<size_t> arrivals;        // block indices enqueued by the mover, issue order (under mu)
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

// One block's reload.  The table lock is held only to check and claim the
// block and to publish the outcome, not while the copies are enqueued (an
// enqueue can block while the copy queue is full), so other host threads may
// query, commit and launch forward passes meanwhile.  A claimed block reads
// as in flight until its event is recorded.
int reload_one(pw_table* t, int layer, int expert, int kind, int q_target, cudaStream_t st) {
  BlockState c;               // what the enqueue phase needs, read under the lock
  bool inject = false;
  BlockState* b = nullptr;
  {
    std::lock_guard<std::mutex> lk(t->mu);
    b = block_of(t, layer, expert, kind);
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
    if (!b->ev) {
      const cudaError_t e = cudaEventCreateWithFlags(&b->ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(e, "pw_reload_async: event create");
    }
    inject = t->fail_next_reload;
    t->fail_next_reload = false;
    b->pending = q_target;
    b->failed = false;
    b->issued = false;
    c = *b;
  }
  const size_t pb = pw_plane_bytes(c.R, c.K);
  cudaError_t e = inject ? cudaErrorInvalidValue : cudaSuccess;   // injected: nothing enqueued
  // Planes are contiguous in the host store; consecutive device pages that are
  // also contiguous go in one copy.
  for (int p = c.resident; p < q_target && e == cudaSuccess;) {
    int p1 = p + 1;
    while (p1 < q_target && static_cast<unsigned char*>(c.pages[p1]) ==
                                static_cast<unsigned char*>(c.pages[p]) + (p1 - p) * pb)
      ++p1;
    e = cudaMemcpyAsync(c.pages[p], c.host_planes + p * (pb / 4), (p1 - p) * pb,
                        cudaMemcpyHostToDevice, st);
    p = p1;
  }
  if (e == cudaSuccess) {
    const size_t lo = pw_lut_offset(c.R, c.b_min, c.resident + 1);
    const size_t hi = pw_lut_offset(c.R, c.b_min, q_target + 1);
    e = cudaMemcpyAsync(static_cast<unsigned char*>(c.d_luts) + lo,
                        reinterpret_cast<const unsigned char*>(c.host_luts) + lo, hi - lo,
                        cudaMemcpyHostToDevice, st);
  }
  if (e == cudaSuccess) e = cudaEventRecord(c.ev, st);
  {
    std::lock_guard<std::mutex> lk(t->mu);
    if (e == cudaSuccess) b->issued = true;
    else b->failed = true;
  }
  t->enqueued.notify_all();
  if (e != cudaSuccess) return cuda_fail(e, "pw_reload_async: enqueue");
  return PW_OK;
}


// Bytes a reload of b to q would copy (planes above resident and their tables).
size_t reload_bytes(const BlockState& b, int q) {
  if (q <= b.resident) return 0;
  return static_cast<size_t>(q - b.resident) * pw_plane_bytes(b.R, b.K) +
         pw_lut_offset(b.R, b.b_min, q + 1) - pw_lut_offset(b.R, b.b_min, b.resident + 1);
}

// The mover thread: takes requests in order, keeps at most mover_limit bytes
// of copies in the copy queue (so that no enqueue blocks in the driver while
// other threads launch), and lists each enqueued block for pw_commit_arrived.
void mover_main(pw_table* t) {
  cudaSetDevice(t->mover_device);
  struct Flight {
    size_t bytes;
    cudaEvent_t ev;
  };
  std::deque<Flight> flight;
  std::vector<cudaEvent_t> spare;
  // a pool of completion events made before any request arrives, so that the
  // copies of a reload window are not interleaved with event creation
  for (int i = 0; i < 128; ++i) {
    cudaEvent_t ev = nullptr;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) break;
    spare.push_back(ev);
  }
  size_t inflight = 0;
  auto note_error = [t](int rc, const char* msg) {
    std::lock_guard<std::mutex> lk(t->mover_mu);
    if (t->mover_error == PW_OK) {
      t->mover_error = rc;
      t->mover_error_msg = msg;
    }
  };
  for (;;) {
    MoveReq r;
    {
      std::unique_lock<std::mutex> lk(t->mover_mu);
      t->mover_cv.wait(lk, [t] { return t->mover_stop || !t->requests.empty(); });
      if (t->mover_stop) break;
      r = t->requests.front();
      t->requests.pop_front();
      ++t->mover_busy;
    }
    size_t bytes = 0;
    size_t idx = 0;
    {
      std::lock_guard<std::mutex> lk(t->mu);
      BlockState* b = block_of(t, r.layer, r.expert, r.kind);
      if (b) {
        bytes = reload_bytes(*b, r.q);
        idx = pw::desc_index(r.layer, r.expert, r.kind, t->E);
      }
    }
    while (!flight.empty() && inflight + bytes > t->mover_limit) {
      const cudaError_t q = cudaEventQuery(flight.front().ev);
      if (q == cudaSuccess) {
        inflight -= flight.front().bytes;
        spare.push_back(flight.front().ev);
        flight.pop_front();
      } else if (q == cudaErrorNotReady) {
        std::this_thread::sleep_for(std::chrono::microseconds(20));
      } else {
        note_error(PW_ECUDA, cudaGetErrorString(q));
        break;
      }
    }
    const int rc = reload_one(t, r.layer, r.expert, r.kind, r.q, t->mover_stream);
    if (rc == PW_OK) {
      {
        std::lock_guard<std::mutex> lk(t->mu);
        t->blocks[idx].commit_to = r.q;
        t->arrivals.push_back(idx);
      }
      cudaEvent_t ev = nullptr;
      if (!spare.empty()) {
        ev = spare.back();
        spare.pop_back();
      } else if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
        ev = nullptr;
      }
      if (ev && cudaEventRecord(ev, t->mover_stream) == cudaSuccess) {
        flight.push_back({bytes, ev});
        inflight += bytes;
      } else if (ev) {
        spare.push_back(ev);
      }
    } else {
      note_error(rc, pw_last_error());
    }
    {
      std::lock_guard<std::mutex> lk(t->mover_mu);
      --t->mover_busy;
    }
    t->mover_cv.notify_all();
  }
  for (auto& f : flight) {
    cudaEventSynchronize(f.ev);
    cudaEventDestroy(f.ev);
  }
  for (auto ev : spare) cudaEventDestroy(ev);
}

void mover_stop(pw_table* t) {
  {
    std::lock_guard<std::mutex> lk(t->mover_mu);
    t->mover_stop = true;
  }
  t->mover_cv.notify_all();
  if (t->mover.joinable()) t->mover.join();
}

// Writes n descriptors (block index, committed q) on s, one launch per batch.
int commit_descs(pw_table* t, const std::vector<std::pair<size_t, int>>& list, cudaStream_t s) {
  static thread_local pw::CommitBatch batch;
  const size_t n = list.size();
  for (size_t i0 = 0; i0 < n; i0 += pw::kCommitBatch) {
    const int m = static_cast<int>(std::min<size_t>(pw::kCommitBatch, n - i0));
    batch.n = m;
    for (int j = 0; j < m; ++j) {
      const auto& it = list[i0 + j];
      const pw::BlockDesc d = make_desc(t->blocks[it.first], it.second);
      batch.index[j] = static_cast<uint32_t>(it.first);
      std::memcpy(batch.words[j], &d, sizeof d);
    }
    const cudaError_t e = pw::launch_commit_batch(t->d_desc, batch, s);
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    for (int j = 0; j < m; ++j) t->blocks[list[i0 + j].first].q = list[i0 + j].second;
  }
  return PW_OK;
}

// Checks that q may be committed for one block; no state changes.  lk holds
// t->mu; if another thread is still enqueueing the block's reload, waits for
// that to finish (the wait releases the lock).
int commit_check(pw_table* t, std::unique_lock<std::mutex>& lk, int layer, int expert, int kind,
                 int q, BlockState** out) {
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_set_commit: block not registered");
  if (q < b->b_min || q > b->n_bits)
    return fail(PW_EINVAL, "pw_set_commit: q %d outside [%d, %d]", q, b->b_min, b->n_bits);
  if (q > b->resident) {
    if (!b->pending || b->pending < q)
      return fail(PW_ENOTRESIDENT, "pw_set_commit: q %d above the %d resident planes, no reload",
                  q, b->resident);
    t->enqueued.wait(lk, [b] { return b->issued || b->failed || !b->pending; });
    if (q > b->resident) {
      if (b->failed) return fail(PW_ERELOAD, "pw_set_commit: the reload to %d failed", b->pending);
      if (!b->pending || b->pending < q)
        return fail(PW_ENOTRESIDENT, "pw_set_commit: q %d above the %d resident planes, no reload",
                    q, b->resident);
    }
  }
  *out = b;
  return PW_OK;
}

// Orders the compute stream after the block's reload when q needs its planes.
int commit_order(BlockState* b, int q, cudaStream_t st) {
  if (q <= b->resident) return PW_OK;
  const cudaError_t e = cudaStreamWaitEvent(st, b->ev, 0);
  if (e != cudaSuccess) return cuda_fail(e, "pw_set_commit: stream wait");
  // From here on the compute stream is ordered after the copies.
  b->resident = b->pending;
  b->pending = 0;
  return PW_OK;
}


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

// NVTX range around one C-ABI call (visible in Nsight timelines; a no-op when
// no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

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
  NvtxRange nvtx_range("pw_pack");
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
  // Bytes of an index that must be zero when n < 8, replicated over 8 indices.
  const uint64_t high = 0x0101010101010101ull * ((0xFFu << n_bits) & 0xFFu);
  auto work = [&](unsigned tid) {
    double sums[2 * 256];   // level b holds the 2^b sums of 2^(n-b) parents, at offset 2^b
    for (int r = static_cast<int>(tid); r < R; r += static_cast<int>(nthr)) {
      const uint8_t* row = idx + static_cast<size_t>(r) * K;
      uint64_t seen = 0;
      for (int w = 0; w < W; ++w) {
        // Four 8x8 bit transposes: byte i of y[g] holds bit i of indices 8g..8g+7,
        // index 8g+j at bit j, i.e. exactly byte g of the 32-bit word of bit i.
        uint64_t y[4];
        for (int g = 0; g < 4; ++g) {
          const uint8_t* b = row + 32 * w + 8 * g;
          uint64_t x = 0;
          for (int j = 0; j < 8; ++j) x |= static_cast<uint64_t>(b[j]) << (8 * j);
          seen |= x;
          uint64_t t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
          x ^= t ^ (t << 7);
          t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
          x ^= t ^ (t << 14);
          t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
          x ^= t ^ (t << 28);
          y[g] = x;
        }
        for (int p = 0; p < n_bits; ++p) {
          const int sh = 8 * (n_bits - 1 - p);   // plane p holds bit n-1-p
          const uint32_t word = static_cast<uint32_t>((y[0] >> sh) & 0xFF) |
                                static_cast<uint32_t>((y[1] >> sh) & 0xFF) << 8 |
                                static_cast<uint32_t>((y[2] >> sh) & 0xFF) << 16 |
                                static_cast<uint32_t>((y[3] >> sh) & 0xFF) << 24;
          planes_out[p * plane_words + static_cast<size_t>(r) * W + w] = word;
        }
      }
      if (seen & high) { bad_row[tid] = r; return; }
      // Tables LUT_b for b = b_min..n.  Entry j of LUT_b is the mean of parents
      // j*g .. j*g+g-1, g = 2^(n-b).  The sums are built level by level, each
      // the sum of two sums one level up; every fp16 value is an integer
      // multiple of 2^-24 below 2^16, so each partial sum is exact in fp64 and
      // equals the sum taken in any order.
      const uint16_t* par = parent_lut + static_cast<size_t>(r) * limit;
      for (int j = 0; j < limit; ++j) sums[limit + j] = half_to_double(par[j]);
      for (int b = n_bits - 1; b >= b_min; --b)
        for (int j = 0; j < (1 << b); ++j)
          sums[(1 << b) + j] = sums[(2 << b) + 2 * j] + sums[(2 << b) + 2 * j + 1];
      for (int b = b_min; b <= n_bits; ++b) {
        uint16_t* dst = luts_out + pw_lut_offset(R, b_min, b) / 2 + static_cast<size_t>(r) * (1u << b);
        const int g = 1 << (n_bits - b);
        if (g == 1) {
          for (int j = 0; j < limit; ++j) dst[j] = par[j];
          continue;
        }
        for (int j = 0; j < (1 << b); ++j) dst[j] = double_to_half(sums[(1 << b) + j] / g);
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

// Re-places the bits of a plane word for the device page: inside each byte the
// even elements (bits 0, 2, 4, 6) move to bits 0..3 and the odd ones (1, 3, 5,
// 7) to bits 4..7, each half in element order.  Two delta swaps: bits 1 <-> 2 of
// every nibble, then bit pairs 2-3 <-> 4-5 of every byte.
static inline uint32_t split_even_odd(uint32_t x) {
  uint32_t t = ((x >> 1) ^ x) & 0x22222222u;
  x ^= t ^ (t << 1);
  t = ((x >> 2) ^ x) & 0x0C0C0C0Cu;
  x ^= t ^ (t << 2);
  return x;
}

int pw_tile_planes(const uint32_t* planes, int n_bits, int R, int K, uint32_t* tiled_out) {
  NvtxRange nvtx_range("pw_tile_planes");
  if (!planes || !tiled_out) return fail(PW_EINVAL, "pw_tile_planes: null pointer");
  if (n_bits < 1 || n_bits > PW_MAX_BITS || R < 32 || R % 32 || K < 64 || K % 64)
    return fail(PW_EINVAL, "pw_tile_planes: need 1 <= n_bits <= 8, R %% 32 == 0, K %% 64 == 0");
  const size_t W = static_cast<size_t>(K) / 32, plane_words = static_cast<size_t>(R) * W;
  const uint32_t* lo = planes;
  const uint32_t* hi = planes + plane_words * n_bits;
  if (tiled_out < hi && lo < tiled_out + plane_words * n_bits)
    return fail(PW_EINVAL, "pw_tile_planes: input and output overlap");
  // word (p, r, w) -> p*R*W + ((r/32)*(W/2) + w/2)*64 + (r%32)*2 + w%2, bits
  // re-placed by split_even_odd; one task per (plane, group of 32 rows), spread
  // over CPU threads
  const int groups = R / 32, tasks = n_bits * groups;
  auto work = [&](int t0, int step) {
    for (int t = t0; t < tasks; t += step) {
      const int p = t / groups, g = t % groups;
      const uint32_t* src = planes + p * plane_words + static_cast<size_t>(g) * 32 * W;
      uint32_t* dst = tiled_out + p * plane_words + static_cast<size_t>(g) * 32 * W;
      for (int rr = 0; rr < 32; ++rr) {
        const uint32_t* row = src + static_cast<size_t>(rr) * W;
        uint32_t* d = dst + rr * 2;
        for (size_t w = 0; w < W; w += 2) {
          d[w * 32] = split_even_odd(row[w]);
          d[w * 32 + 1] = split_even_odd(row[w + 1]);
        }
      }
    }
  };
  unsigned nthr = std::thread::hardware_concurrency();
  if (nthr == 0) nthr = 1;
  if (plane_words * n_bits < (1u << 20)) nthr = 1;
  if (nthr > 32) nthr = 32;
  if (nthr == 1) {
    work(0, 1);
  } else {
    std::vector<std::thread> th;
    for (unsigned i = 0; i < nthr; ++i) th.emplace_back(work, static_cast<int>(i), static_cast<int>(nthr));
    for (auto& x : th) x.join();
  }
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
  NvtxRange nvtx_range("pw_block_register");
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
  if (!nb.ev) {
    // created here, not at the first reload: a reload window then issues only
    // copies (creating events inside it cost the first window most of its rate)
    const cudaError_t ee = cudaEventCreateWithFlags(&nb.ev, cudaEventDisableTiming);
    if (ee != cudaSuccess) return cuda_fail(ee, "pw_block_register: event create");
    b->ev = nb.ev;   // owned by the block from now on (destroyed with the table)
  }
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
  NvtxRange nvtx_range("pw_reload_async");
  if (!t) return fail(PW_EINVAL, "pw_reload_async: null table");
  return reload_one(t, layer, expert, kind, q_target, reinterpret_cast<cudaStream_t>(copy));
}

int pw_reload_many(pw_table* t, int n, const int* layer, const int* expert, const int* kind,
                   const int* q_target, pw_stream_t copy, int* n_done) {
  NvtxRange nvtx_range("pw_reload_many");
  if (n_done) *n_done = 0;
  if (!t) return fail(PW_EINVAL, "pw_reload_many: null table");
  if (n < 0 || (n > 0 && (!layer || !expert || !kind || !q_target)))
    return fail(PW_EINVAL, "pw_reload_many: bad count or null array");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(copy);
  for (int i = 0; i < n; ++i) {
    const int rc = reload_one(t, layer[i], expert[i], kind[i], q_target[i], st);
    if (rc != PW_OK) return rc;
    if (n_done) *n_done = i + 1;
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
  if (!b->issued) return 0;   // another thread is still enqueueing its copies
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
  NvtxRange nvtx_range("pw_set_commit");
  if (!t) return fail(PW_EINVAL, "pw_set_commit: null table");
  std::unique_lock<std::mutex> lk(t->mu);
  BlockState* b = nullptr;
  int rc = commit_check(t, lk, layer, expert, kind, q, &b);
  if (rc != PW_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(compute);
  rc = commit_order(b, q, st);
  if (rc != PW_OK) return rc;
  rc = write_desc(t, layer, expert, kind, *b, q, st);
  if (rc != PW_OK) return rc;
  b->q = q;
  return PW_OK;
}

int pw_set_commit_many(pw_table* t, int n, const int* layer, const int* expert, const int* kind,
                       const int* q, pw_stream_t compute) {
  NvtxRange nvtx_range("pw_set_commit_many");
  if (!t) return fail(PW_EINVAL, "pw_set_commit_many: null table");
  if (n < 0 || (n > 0 && (!layer || !expert || !kind || !q)))
    return fail(PW_EINVAL, "pw_set_commit_many: bad count or null array");
  std::unique_lock<std::mutex> lk(t->mu);
  std::vector<BlockState*> bs(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) {          // all or nothing: every entry is checked first
    const int rc = commit_check(t, lk, layer[i], expert[i], kind[i], q[i], &bs[i]);
    if (rc != PW_OK) return rc;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(compute);
  for (int i = 0; i < n; ++i) {
    const int rc = commit_order(bs[i], q[i], st);
    if (rc != PW_OK) return rc;
  }
  std::vector<std::pair<size_t, int>> list(static_cast<size_t>(n));
  for (int i = 0; i < n; ++i) list[i] = {pw::desc_index(layer[i], expert[i], kind[i], t->E), q[i]};
  const int rc = commit_descs(t, list, st);
  if (rc != PW_OK) return rc;
  return PW_OK;
}

int pw_mover_start(pw_table* t, pw_stream_t copy, size_t max_inflight_bytes) {
  if (!t) return fail(PW_EINVAL, "pw_mover_start: null table");
  if (max_inflight_bytes == 0) return fail(PW_EINVAL, "pw_mover_start: max_inflight_bytes is 0");
  std::lock_guard<std::mutex> lk(t->mover_mu);
  if (t->mover.joinable()) return fail(PW_EINVAL, "pw_mover_start: the mover is already running");
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "pw_mover_start: current device");
  t->mover_device = dev;
  t->mover_stream = reinterpret_cast<cudaStream_t>(copy);
  t->mover_limit = max_inflight_bytes;
  t->mover_stop = false;
  try {
    t->mover = std::thread(mover_main, t);
  } catch (...) {
    return fail(PW_ENOMEM, "pw_mover_start: could not start the thread");
  }
  return PW_OK;
}

int pw_mover_submit(pw_table* t, int n, const int* layer, const int* expert, const int* kind,
                    const int* q_target) {
  NvtxRange nvtx_range("pw_mover_submit");
  if (!t) return fail(PW_EINVAL, "pw_mover_submit: null table");
  if (n < 0 || (n > 0 && (!layer || !expert || !kind || !q_target)))
    return fail(PW_EINVAL, "pw_mover_submit: bad count or null array");
  {
    std::lock_guard<std::mutex> lk(t->mu);   // checked up front: all or nothing
    for (int i = 0; i < n; ++i) {
      const BlockState* b = block_of(t, layer[i], expert[i], kind[i]);
      if (!b || !b->registered)
        return fail(PW_EINVAL, "pw_mover_submit: entry %d: block not registered", i);
      if (q_target[i] < b->b_min || q_target[i] > b->n_bits)
        return fail(PW_EINVAL, "pw_mover_submit: entry %d: q %d outside [%d, %d]", i, q_target[i],
                    b->b_min, b->n_bits);
      for (int p = 0; p < q_target[i]; ++p)
        if (!b->pages[p])
          return fail(PW_EINVAL, "pw_mover_submit: entry %d: no device page for plane %d", i, p);
    }
  }
  {
    std::lock_guard<std::mutex> lk(t->mover_mu);
    if (!t->mover.joinable()) return fail(PW_EINVAL, "pw_mover_submit: the mover is not running");
    for (int i = 0; i < n; ++i) t->requests.push_back({layer[i], expert[i], kind[i], q_target[i]});
  }
  t->mover_cv.notify_all();
  return PW_OK;
}

int pw_plan_apply(pw_table* t, const int* desired, pw_stream_t compute, int* n_now, int* n_moved) {
  NvtxRange nvtx_range("pw_plan_apply");
  if (n_now) *n_now = 0;
  if (n_moved) *n_moved = 0;
  if (!t || !desired) return fail(PW_EINVAL, "pw_plan_apply: null table or plan");
  std::vector<std::pair<size_t, int>> now;
  std::vector<MoveReq> moves;
  {
    std::lock_guard<std::mutex> lk(t->mu);
    for (size_t i = 0; i < t->blocks.size(); ++i) {   // every entry checked before anything is done
      const int d = desired[i];
      if (d == 0) continue;
      const BlockState& b = t->blocks[i];
      if (!b.registered) return fail(PW_EINVAL, "pw_plan_apply: block %zu is not registered", i);
      if (d < b.b_min || d > b.n_bits)
        return fail(PW_EINVAL, "pw_plan_apply: block %zu: q %d outside [%d, %d]", i, d, b.b_min, b.n_bits);
      if (d == b.q) continue;
      if (d <= b.resident) {
        now.push_back({i, d});
        continue;
      }
      if (b.pending) return fail(PW_EINVAL, "pw_plan_apply: block %zu has a reload pending", i);
      for (int p = 0; p < d; ++p)
        if (!b.pages[p]) return fail(PW_EINVAL, "pw_plan_apply: block %zu has no page for plane %d", i, p);
      const int kind = static_cast<int>(i % 2), expert = static_cast<int>((i / 2) % t->E),
                layer = static_cast<int>(i / (2 * static_cast<size_t>(t->E)));
      moves.push_back({layer, expert, kind, d});
    }
    if (!moves.empty()) {
      std::lock_guard<std::mutex> mk(t->mover_mu);
      if (!t->mover.joinable())
        return fail(PW_EINVAL, "pw_plan_apply: %zu blocks need a reload and the mover is not running",
                    moves.size());
    }
    if (!now.empty()) {
      const int rc = commit_descs(t, now, reinterpret_cast<cudaStream_t>(compute));
      if (rc != PW_OK) return rc;
    }
  }
  if (!moves.empty()) {
    {
      std::lock_guard<std::mutex> mk(t->mover_mu);
      for (const MoveReq& r : moves) t->requests.push_back(r);
    }
    t->mover_cv.notify_all();
  }
  if (n_now) *n_now = static_cast<int>(now.size());
  if (n_moved) *n_moved = static_cast<int>(moves.size());
  return PW_OK;
}

int pw_commit_arrived(pw_table* t, pw_stream_t compute, int* n_committed, int* n_outstanding) {
  NvtxRange nvtx_range("pw_commit_arrived");
  if (n_committed) *n_committed = 0;
  if (n_outstanding) *n_outstanding = 0;
  if (!t) return fail(PW_EINVAL, "pw_commit_arrived: null table");
  int rc = PW_OK;
  std::vector<std::pair<size_t, int>> list;
  size_t left = 0;
  {
    std::lock_guard<std::mutex> lk(t->mu);
    while (!t->arrivals.empty()) {
      BlockState& b = t->blocks[t->arrivals.front()];
      if (b.pending) {
        if (b.failed) {
          rc = fail(PW_ERELOAD, "pw_commit_arrived: a reload failed; its block keeps q %d", b.q);
          b.commit_to = 0;
          t->arrivals.pop_front();
          continue;
        }
        if (!b.issued) break;
        const cudaError_t e = cudaEventQuery(b.ev);
        if (e == cudaErrorNotReady) break;   // copies on one stream land in issue order
        if (e != cudaSuccess) {
          rc = cuda_fail(e, "pw_commit_arrived: event query");
          break;
        }
        b.resident = b.pending;
        b.pending = 0;
      }
      if (b.commit_to && b.commit_to <= b.resident) list.push_back({t->arrivals.front(), b.commit_to});
      b.commit_to = 0;
      t->arrivals.pop_front();
    }
    if (!list.empty()) {
      const int c = commit_descs(t, list, reinterpret_cast<cudaStream_t>(compute));
      if (c != PW_OK) return c;
    }
    left = t->arrivals.size();
  }
  {
    std::lock_guard<std::mutex> lk(t->mover_mu);
    left += t->requests.size() + static_cast<size_t>(t->mover_busy);
    if (rc == PW_OK && t->mover_error != PW_OK) {
      rc = fail(t->mover_error, "pw_commit_arrived: mover: %s", t->mover_error_msg.c_str());
      t->mover_error = PW_OK;
      t->mover_error_msg.clear();
    }
  }
  if (n_committed) *n_committed = static_cast<int>(list.size());
  if (n_outstanding) *n_outstanding = static_cast<int>(left);
  return rc;
}

int pw_block_release(pw_table* t, int layer, int expert, int kind, int keep, void** released) {
  NvtxRange nvtx_range("pw_block_release");
  if (!t) return fail(PW_EINVAL, "pw_block_release: null table");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_block_release: block not registered");
  if (keep < b->q || keep > b->n_bits)
    return fail(PW_EINVAL, "pw_block_release: keep %d outside [committed q %d, %d]", keep, b->q, b->n_bits);
  if (b->pending) return fail(PW_EINVAL, "pw_block_release: a reload of this block is pending");
  for (int p = 0; p < PW_MAX_BITS; ++p) {
    void* page = nullptr;
    if (p >= keep && p < b->n_bits) {
      page = b->pages[p];
      b->pages[p] = nullptr;
    }
    if (released) released[p] = page;
  }
  if (b->resident > keep) b->resident = keep;
  return PW_OK;
}

int pw_block_attach_pages(pw_table* t, int layer, int expert, int kind, void* const* pages) {
  NvtxRange nvtx_range("pw_block_attach_pages");
  if (!t || !pages) return fail(PW_EINVAL, "pw_block_attach_pages: null table or pages");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_block_attach_pages: block not registered");
  if (b->pending) return fail(PW_EINVAL, "pw_block_attach_pages: a reload of this block is pending");
  for (int p = 0; p < b->n_bits; ++p) {   // all checked first
    if (!pages[p]) continue;
    if (p < b->resident && pages[p] != b->pages[p])
      return fail(PW_EINVAL, "pw_block_attach_pages: plane %d is resident on another page", p);
    if (!aligned16(pages[p])) return fail(PW_EINVAL, "pw_block_attach_pages: page %d not 16-byte aligned", p);
  }
  for (int p = b->resident; p < b->n_bits; ++p)
    if (pages[p]) b->pages[p] = pages[p];
  return PW_OK;
}

int pw_plane_states(pw_table* t, int layer, int expert, int kind, int* states) {
  if (!t || !states) return fail(PW_EINVAL, "pw_plane_states: null table or output");
  std::lock_guard<std::mutex> lk(t->mu);
  BlockState* b = block_of(t, layer, expert, kind);
  if (!b || !b->registered) return fail(PW_EINVAL, "pw_plane_states: block not registered");
  for (int p = 0; p < PW_MAX_BITS; ++p) {
    int st = PW_PLANE_HOST;
    if (p >= b->n_bits) st = PW_PLANE_HOST;
    else if (p < b->resident) st = PW_PLANE_DEVICE;
    else if (b->pending && !b->failed && p < b->pending) st = PW_PLANE_MOVING;
    else if (b->pages[p]) st = PW_PLANE_HOST_PAGED;
    states[p] = st;
  }
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
  mover_stop(t);
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

size_t pw_workspace_offset(int T, int E, int top_k, int H, int I, int section) {
  if (T < 0 || E < 1 || top_k < 1 || H < 1 || I < 1) return static_cast<size_t>(-1);
  const pw::Workspace w = pw::workspace_layout(T, E, top_k, H, I);
  if (section == PW_WS_H) return w.hh;
  if (section == PW_WS_Y) return w.y;
  return static_cast<size_t>(-1);
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
  NvtxRange nvtx_range("pw_moe_forward");
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
  {
    std::lock_guard<std::mutex> lk(t->mu);
    a.stats = t->stats;
    a.stats_alpha = t->stats_alpha;
  }
  const cudaError_t e = pw::launch_forward(a, reinterpret_cast<cudaStream_t>(compute));
  if (e != cudaSuccess) return cuda_fail(e, "pw_moe_forward: launch");
  return PW_OK;
}

int pw_moe_forward_host(pw_table* t, int layer, const void* x_host, const float* logits_host,
                        int T, int top_k, int renorm, const void* residual_host, void* out_host,
                        void* workspace, size_t ws_bytes, pw_stream_t compute) {
  NvtxRange nvtx_range("pw_moe_forward_host");
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

int pw_stats_attach(pw_table* t, float* d_stats, float alpha) {
  if (!t) return fail(PW_EINVAL, "pw_stats_attach: null table");
  if (d_stats && !(alpha > 0.f && alpha <= 1.f))
    return fail(PW_EINVAL, "pw_stats_attach: alpha must be in (0, 1]");
  if (d_stats && (reinterpret_cast<uintptr_t>(d_stats) & 3))
    return fail(PW_EINVAL, "pw_stats_attach: statistics buffer not 4-byte aligned");
  std::lock_guard<std::mutex> lk(t->mu);
  t->stats = d_stats;
  t->stats_alpha = d_stats ? alpha : 0.f;
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
