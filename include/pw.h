/*
 * pw.h -- C ABI of the fused mixed-precision APL MoE expert layer (GB300, sm_103a).
 *
 * Method: PagedWeight ("PagedWeight: Efficient MoE LLM Serving with Dynamic
 * Quality-Aware Weight Quantization").  Its technical summary's core components
 * name the pieces behind these calls:
 *   - section 1 "Paged Weight Representation": one unit per (layer, expert,
 *     gate_up|down) linear block; weights in APL's layered bit-plane format with
 *     associated lookup tables; a weight page table holding the desired (d_i) and
 *     committed (q_i) bitwidth of every block; pages resident on the GPU, on the
 *     CPU, or in transfer;
 *   - section 3 "Asynchronous Page Movement": pages reloaded asynchronously, a
 *     bitwidth commit applied only at a safe boundary so that inference never
 *     stops;
 *   - section 3 "Fused Mixed-Precision Kernel": one fused operation that reads
 *     bit-planes and tables directly, with a different bitwidth per block.
 *
 * Bit-plane layout (fixed by this library; the pages print none):
 *   parent index P[r][k] in [0, 2^n); plane p (p = 0 most significant) holds bit
 *   (n-1-p) of P; planes are stored plane-major per block, planes[p][r][K/32] as
 *   uint32, bit j of word w holding element k = 32w + j.  A b-bit weight uses the
 *   top b planes (index P >> (n-b)) and the row's own 2^b-entry fp16 table LUT_b.
 *   Each plane of a block is one page of R*K/8 bytes, so the planes below the
 *   committed bitwidth form a tail that can live on the CPU and be reloaded.
 *   Inside a device page the words are interleaved across groups of 32 rows
 *   and the bits of each word re-placed (pw_tile_planes), so that a warp's
 *   reads of 32 rows are contiguous.
 *
 * Block shapes: gate_up has R = 2I rows (rows [0, I) gate, [I, 2I) up) and
 * K = H columns; down has R = H rows and K = I columns.  H, I multiples of 128.
 *
 * Conventions for every call:
 *   - returns PW_OK (0) or a negative PW_E* status; nothing throws or exits;
 *     pw_last_error() gives a message for the last failure on this thread;
 *   - fp16 values are passed as uint16_t bit patterns or void*;
 *   - the library allocates no device memory: the caller owns every device
 *     buffer (plane pages, tables, descriptor array, workspace) and every stream;
 *     the library owns only the small host-side table object;
 *   - "device" pointers are CUDA device addresses on the current device; "host"
 *     pointers are CPU addresses (pinned where stated).
 */
#ifndef PW_H
#define PW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define PW_OK            0
#define PW_EINVAL       (-1)  /* bad argument, shape or state                     */
#define PW_ECUDA        (-2)  /* a CUDA runtime call or kernel launch failed      */
#define PW_ENOTRESIDENT (-3)  /* commit above the resident planes, no reload      */
#define PW_ERELOAD      (-4)  /* the reload this commit waits for has failed      */
#define PW_ETIMEOUT     (-5)  /* a bounded wait ran out                           */
#define PW_ENOMEM       (-6)  /* host allocation failed or workspace too small    */
#define PW_EDEVICE      (-7)  /* a kernel reported an error through the workspace */

/* Bits of the device status word (pw_workspace_status). */
#define PW_STATUS_NAN_LOGIT  1  /* a router logit was NaN (treated as -inf)     */
#define PW_STATUS_TIMEOUT    2  /* a bounded device-side wait gave up           */
#define PW_STATUS_BAD_DESC   4  /* an active block had no usable descriptor     */
#define PW_STATUS_BOUNDS     8  /* a device-side bounds check failed; the access
                                   was skipped (libpw_check.so, built with
                                   PW_CHECK, only)                             */

#define PW_KIND_GATE_UP 0
#define PW_KIND_DOWN    1
#define PW_MAX_BITS     8

typedef struct CUstream_st* pw_stream_t;   /* a cudaStream_t; NULL = default stream */
typedef struct pw_table pw_table;          /* opaque host-side page table           */

/* Message for the last failing call on this thread ("" if none). */
const char* pw_last_error(void);

/* ------------------------------------------------------------------ format (host) */

/* Bytes of one plane page of an R x K block: R*K/8. */
size_t pw_plane_bytes(int R, int K);

/* Bytes of the concatenated tables LUT_b, b = b_min..n_bits, each [R][2^b] fp16. */
size_t pw_lut_bytes(int R, int b_min, int n_bits);

/* Byte offset of LUT_b inside that concatenation (b_min <= b). */
size_t pw_lut_offset(int R, int b_min, int b);

/*
 * pw_pack -- bit-plane packer and table builder (host, CPU threads).
 * Source: "Paged Weight Representation" (layered bit-planes with associated
 * lookup tables).
 *   idx        host [R][K] uint8 parent indices, each < 2^n_bits
 *   parent_lut host [R][2^n_bits] fp16 table of the parent (n_bits-bit) weights
 *   planes_out host [n_bits][R][K/32] uint32, written in the layout above
 *   luts_out   host, pw_lut_bytes(R, b_min, n_bits) bytes: LUT_b for b = b_min..n_bits.
 *              LUT_n is the parent table; for b < n, LUT_b[r][j] is the mean of the
 *              2^(n-b) parent entries whose top b index bits equal j, computed in
 *              fp64 and rounded once to fp16 (nearest, ties to even).
 * Requirements: R >= 1, K >= 32, K % 32 == 0, 1 <= b_min <= n_bits <= 8.
 * Errors: PW_EINVAL for a bad shape, a null pointer or an index >= 2^n_bits
 * (nothing is guaranteed about the outputs then).
 */
int pw_pack(const uint8_t* idx, int R, int K, int n_bits, const uint16_t* parent_lut,
            int b_min, uint32_t* planes_out, uint16_t* luts_out);

/*
 * pw_tile_planes -- the device page layout of a block's planes (host, CPU).
 * Source: "Paged Weight Representation" (each plane one page); the order of
 * the words inside a page is this library's choice.
 * Reorders pw_pack's planes [n_bits][R][K/32] into the layout the kernels and
 * pw_block_register use: within each plane, rows are taken in groups of 32
 * and every pair of consecutive words along K is stored for the group's 32
 * rows side by side, [n_bits][R/32][K/64][32][2]; word w of row r of plane p
 * lands at p*R*(K/32) + ((r/32)*(K/64) + w/2)*64 + (r%32)*2 + w%2.  A warp
 * reading two words of 32 consecutive rows then reads 256 contiguous bytes.
 * Inside each word the bits are re-placed: of each byte's 8 elements, the even
 * ones (k%2 == 0) occupy bits 0..3 and the odd ones bits 4..7, in element
 * order (element j of the word at bit 8*(j/8) + (j%8)/2 + 4*(j%2)), so that
 * transposing 4 plane words nibble by nibble yields one byte per pair of
 * neighbouring elements.  Each plane is still one contiguous page of R*K/8
 * bytes, and a plane's bits never mix with another plane's.
 *   planes     host [n_bits][R][K/32] uint32 (pw_pack output), read only
 *   tiled_out  host, same size, must not overlap planes
 * Requirements: 1 <= n_bits <= 8, R % 32 == 0, K % 64 == 0.
 * Errors: PW_EINVAL (shape, null pointer, overlapping buffers).
 */
int pw_tile_planes(const uint32_t* planes, int n_bits, int R, int K, uint32_t* tiled_out);

/* ------------------------------------------------------------------ page table */

/* Bytes of the device descriptor array for n_layers x n_experts x 2 blocks. */
size_t pw_desc_bytes(int n_layers, int n_experts);

/*
 * pw_table_create -- the weight page table ("Paged Weight Representation":
 * per-block desired d_i and committed q_i).
 *   d_desc      device memory of at least pw_desc_bytes(n_layers, n_experts) bytes,
 *               128-byte aligned, owned by the caller, alive until pw_table_destroy.
 *               The kernels read each block's committed q_i and page addresses from
 *               it, so a commit needs no recompile and no host round trip.
 *   n_experts   1..256;  H, I: hidden and expert-intermediate sizes (multiples of 128).
 *   s           stream on which the descriptors are cleared (asynchronous).
 * Errors: PW_EINVAL (shapes, small or misaligned buffer), PW_ECUDA, PW_ENOMEM.
 */
int pw_table_create(pw_table** out, int n_layers, int n_experts, int H, int I,
                    void* d_desc, size_t desc_bytes, pw_stream_t s);

/*
 * pw_block_register -- attach one linear block (layer, expert, kind).
 *   host_planes  host planes in the page layout of pw_tile_planes (pw_pack output
 *                reordered by it), the backing store of every plane; pinned
 *                memory makes later reloads asynchronous.
 *                Must stay valid until pw_table_destroy.
 *   host_luts    host tables as written by pw_pack; same lifetime rule.
 *   d_plane_pages n_bits device pointers, page p holding plane p (R*K/8 bytes,
 *                16-byte aligned).  Pages for p >= q_init may be NULL if the block
 *                will never be reloaded that far.
 *   d_luts       device memory of pw_lut_bytes(R, b_min, n_bits) bytes (16-byte
 *                aligned) holding the tables in the pw_pack layout.
 *   q_init       committed bitwidth, b_min <= q_init <= n_bits.  Planes [0, q_init)
 *                and tables b <= q_init are copied host->device on s, then the
 *                descriptor is written on s; everything is ordered on s.
 * Errors: PW_EINVAL, PW_ECUDA.
 */
int pw_block_register(pw_table* t, int layer, int expert, int kind, int n_bits, int b_min,
                      const uint32_t* host_planes, const uint16_t* host_luts,
                      void* const* d_plane_pages, void* d_luts, int q_init, pw_stream_t s);

/*
 * pw_reload_async -- bring planes [resident, q_target) and tables
 * (resident, q_target] of one block from its host backing store to its device
 * pages ("Asynchronous Page Movement").  Enqueues host->device copies on the
 * copy stream and records an event after them; returns without waiting.  The
 * copies touch only planes and tables that no kernel reads at the committed
 * q <= resident, so they may overlap forward passes on another stream.
 * q_target <= resident is a no-op.  One reload per block may be pending at a time.
 * Errors: PW_EINVAL (q_target out of range, missing page, a reload already
 * pending), PW_ECUDA (a copy could not be enqueued: the block is marked failed
 * and a later commit above resident returns PW_ERELOAD).
 */
int pw_reload_async(pw_table* t, int layer, int expert, int kind, int q_target,
                    pw_stream_t copy);

/*
 * pw_reload_many -- pw_reload_async for n blocks in one call: block i is
 * (layer[i], expert[i], kind[i]) raised to q_target[i]; the four arrays are host
 * memory of n ints, read only during the call.  The table's lock is taken per
 * block, so another host thread may query and commit blocks while this call is
 * still enqueueing later ones.  Stops at the first block that fails, returning
 * its error code; *n_done (if not null) is the number of blocks enqueued
 * before it (n on success).  A runtime addition for planners that raise many
 * blocks at once; the pages describe per-block movement only.
 *
 * Threads: the table calls may be made from several host threads.  A reload
 * holds the table lock only while it checks and claims the block and when it
 * publishes the outcome, never while its copies are enqueued, so a planner
 * thread can run this while the decode thread launches forward passes,
 * queries and commits.  A block being enqueued reads as in flight
 * (pw_reload_query returns 0); a commit that needs it waits on the host until
 * its enqueue has finished.
 */
int pw_reload_many(pw_table* t, int n, const int* layer, const int* expert, const int* kind,
                   const int* q_target, pw_stream_t copy, int* n_done);

/*
 * pw_reload_query -- non-blocking completion check of a block's pending reload.
 * Returns 1 when the reload has completed (or none is pending), 0 while it is
 * in flight, PW_ERELOAD if it failed.
 */
int pw_reload_query(pw_table* t, int layer, int expert, int kind);

/*
 * pw_set_commit -- commit bitwidth q for one block at a stream-ordered safe
 * boundary ("bitwidth commits only at safe boundaries").  The descriptor write
 * is enqueued on the compute stream: forward passes enqueued on it before this
 * call read the old q, those after read q.  Raising q above the resident planes
 * requires a pending or completed reload to >= q: the compute stream then first
 * waits on the reload's event (no host wait).  Lowering q needs no copy.
 * Errors: PW_EINVAL (q outside [b_min, n_bits]), PW_ENOTRESIDENT (q above the
 * resident planes and no reload to q), PW_ERELOAD (that reload failed; q is
 * unchanged), PW_ECUDA.
 */
int pw_set_commit(pw_table* t, int layer, int expert, int kind, int q, pw_stream_t compute);

/*
 * pw_set_commit_many -- pw_set_commit for n blocks at one stream-ordered
 * boundary: block i is (layer[i], expert[i], kind[i]) committed at q[i]; host
 * arrays of n ints.  Every entry is checked before anything is enqueued, so on
 * PW_EINVAL / PW_ENOTRESIDENT / PW_ERELOAD no block changes.  The compute
 * stream waits on each raised block's reload event, then the descriptors are
 * written by one small kernel per 192 blocks instead of one per block.  If a
 * block appears twice, its last entry is the one that holds.  Errors as for
 * pw_set_commit.
 */
int pw_set_commit_many(pw_table* t, int n, const int* layer, const int* expert, const int* kind,
                       const int* q, pw_stream_t compute);

/*
 * The reload mover: a host thread owned by the table that carries out
 * submitted reloads in submission order on one copy stream, and a call the
 * decode loop makes at each step boundary to commit whatever has landed.
 * This is the asynchronous page movement of the pages ("Asynchronous Page
 * Movement": planes move while inference continues; a bitwidth is committed
 * only at a safe boundary) with the policy of when to enqueue moved into
 * native code: the decode thread makes one call per step instead of one per
 * block, and never blocks behind a full copy queue.
 *
 * pw_mover_start -- starts the mover on `copy` (a stream of the current
 * device).  It keeps at most max_inflight_bytes of reload copies enqueued and
 * not yet finished, so that its enqueues never block in the driver while other
 * threads launch.  Errors: PW_EINVAL (already running, zero limit), PW_ECUDA,
 * PW_ENOMEM (no thread).  pw_table_destroy stops it (requests not yet taken
 * are dropped; copies in flight are waited for).
 */
int pw_mover_start(pw_table* t, pw_stream_t copy, size_t max_inflight_bytes);

/*
 * pw_mover_submit -- queues reloads of n blocks (host arrays of n ints) to
 * q_target[i]; each block is committed at q_target[i] by the first
 * pw_commit_arrived after its copies have finished (a target at or below the
 * resident planes needs no copy and is committed at the next call).  All
 * entries are checked before any is queued.  Errors: PW_EINVAL (block not
 * registered, q outside [b_min, n_bits], a plane below q_target without a
 * device page, mover not running).  A failure later, in the mover, is
 * reported by the next pw_commit_arrived.
 */
int pw_mover_submit(pw_table* t, int n, const int* layer, const int* expert, const int* kind,
                    const int* q_target);

/*
 * pw_commit_arrived -- at a step boundary: commits, on the compute stream and
 * in one small launch per 192 blocks, every mover-submitted block whose copies
 * have finished (checked without waiting, in submission order, stopping at
 * the first that has not).  *n_committed = blocks committed by this call;
 * *n_outstanding = submitted blocks not yet committed (queued, being
 * enqueued, or in flight); either pointer may be null.  Errors: PW_ERELOAD
 * (a block's reload failed: it keeps its q; the others are still committed),
 * an error the mover met since the last call, PW_ECUDA.
 */
int pw_commit_arrived(pw_table* t, pw_stream_t compute, int* n_committed, int* n_outstanding);

/*
 * pw_stats_attach -- routing statistics as a by-product of the routing step
 * (the routing-mass input of the pages' runtime planner, "Quality-Aware Runtime
 * Planner": experts that receive more routing mass matter more).  d_stats is a
 * caller-owned device array of n_layers * n_experts floats, initialised by the
 * caller (zeros, or 1/E for a uniform prior).  Once attached, every forward
 * of layer l updates, on its stream and inside its routing kernel (no extra
 * launch), for every expert e:
 *   stats[l][e] <- (1 - alpha) * stats[l][e] + alpha * M_e,
 *   M_e = (1/T) * sum of the routing weights of the (token, slot) pairs routed to e,
 * summed in a fixed order (the same result on every run).  With renorm the
 * M_e of a batch sum to 1.  d_stats = null detaches.  Attach between forwards.
 * Errors: PW_EINVAL (null table, alpha outside (0, 1], misaligned buffer).
 */
int pw_stats_attach(pw_table* t, float* d_stats, float alpha);

/* ------------------------------------------------------------------ planner (host) */

/*
 * pw_plan_bits -- the quality-aware bitwidth planner ("Quality-Aware Runtime
 * Planner": offline Hessian-weighted sensitivity, online routing mass with
 * higher floors and damage multipliers for hot experts, a prompt residual
 * correcting the sensitivity; greedy lowest damage per byte saved until a
 * memory target is met).  Host only, no CUDA call.
 *
 * Per block i (host arrays of n_blocks): R[i] x K[i] weights, sens[i] the
 * offline sensitivity, resid[i] the prompt residual (resid may be null: 0),
 * mass[i] the routing mass of the block's expert.  The pages give no formulas;
 * this reading is used:
 *   s' = max(0, sens + resid), m = 1 + n_experts * mass,
 *   floor = hot_floor if mass >= hot_mass else b_min,
 *   damage of b -> b-1 bits = m * s' * R * K * (4^-(b-1) - 4^-b),
 *   bytes saved = R*K/8 + R * 2^b * 2 (one plane and the b-bit table).
 * Starting from n_bits everywhere, reductions are taken in increasing damage /
 * bytes saved (ties: lower block index) while the resident bytes exceed
 * target_bytes and some block is above its floor.  bits_out[i] receives the
 * planned bitwidth; *resident_out (if not null) the resident bytes of the plan
 * (above target_bytes when the floors stop it).
 * Errors: PW_EINVAL (null array, bad sizes, not 1 <= b_min <= hot_floor <= n_bits <= 8).
 */
int pw_plan_bits(int n_blocks, const int* R, const int* K, const double* sens, const double* resid,
                 const double* mass, int n_experts, double hot_mass, int hot_floor, int b_min,
                 int n_bits, double target_bytes, int* bits_out, int64_t* resident_out);

/*
 * pw_plan_apply -- carries out a plan on a table.  desired[] holds one
 * bitwidth per block in descriptor order ((layer * n_experts + expert) * 2 +
 * kind), 0 for "leave alone".  Blocks to lower, and blocks to raise whose
 * planes are already resident, are committed at once on the compute stream
 * (one batched commit); blocks to raise above their resident planes are
 * submitted to the mover (pw_mover_start must have been called) and commit
 * at a later pw_commit_arrived.  Every entry is checked before anything is
 * done.  *n_now / *n_moved (either may be null): blocks committed now / handed
 * to the mover.  Errors: PW_EINVAL (unregistered block with desired > 0, q out
 * of range, no page for a plane, mover not running while a reload is needed),
 * PW_ECUDA.
 */
int pw_plan_apply(pw_table* t, const int* desired, pw_stream_t compute, int* n_now, int* n_moved);

/* ------------------------------------------------------------------ offload */

/*
 * Page states of a plane ("Weight Page Table": pages are GPU-resident,
 * CPU-resident or in transfer).  The host backing store given to
 * pw_block_register holds every plane of the block for the table's lifetime
 * (weights never change), so a plane leaves the GPU by releasing its device
 * page; no device-to-host copy is needed.
 */
#define PW_PLANE_HOST 0        /* host copy only, no device page */
#define PW_PLANE_HOST_PAGED 1  /* host copy; a device page is attached but not filled */
#define PW_PLANE_MOVING 2      /* a reload into the device page is in flight */
#define PW_PLANE_DEVICE 3      /* resident on the device */

/*
 * pw_block_release -- offloads planes [keep, n_bits) of one block: they stop
 * being resident and their device pages are detached from the table and
 * returned in released[0..7] (null where no page was detached), for the
 * caller to free or reuse.  keep must be >= the committed q, so no forward
 * enqueued after this call reads them; forwards enqueued earlier at a higher
 * committed q may still be running, so reuse a released page only after the
 * compute stream has passed the commit that lowered q (for example after a
 * stream synchronisation or an event recorded after that commit).  Errors:
 * PW_EINVAL (keep outside [q, n_bits], a reload pending).
 */
int pw_block_release(pw_table* t, int layer, int expert, int kind, int keep, void** released);

/*
 * pw_block_attach_pages -- gives a block device pages for its non-resident
 * planes (pages[p] for p >= resident; null entries leave a plane as it is), so
 * that a later reload can fill them (page-pool reuse).  Each page holds
 * pw_plane_bytes(R, K) bytes, 16-byte aligned.  Errors: PW_EINVAL (a page for a
 * resident plane that differs from the current one, misaligned page, a reload
 * pending).
 */
int pw_block_attach_pages(pw_table* t, int layer, int expert, int kind, void* const* pages);

/* pw_plane_states -- the PW_PLANE_* state of planes 0..7 of one block (planes
 * at or above n_bits read PW_PLANE_HOST). */
int pw_plane_states(pw_table* t, int layer, int expert, int kind, int* states);

/* Host view of one block: committed q, resident planes, pending reload target (0 if none). */
int pw_block_state(pw_table* t, int layer, int expert, int kind, int* q, int* resident,
                   int* reload_target);

/*
 * pw_debug_fail_next_reload -- test hook for the failure path of the reload
 * protocol: the next pw_reload_async on this table behaves as if its first
 * host->device copy could not be enqueued (no copy is issued, the block is
 * marked failed, PW_ECUDA is returned).  Lets tests exercise PW_ERELOAD without
 * disturbing the GPU.
 */
int pw_debug_fail_next_reload(pw_table* t);

/* Destroys the host object (after synchronising its pending reload events). */
int pw_table_destroy(pw_table* t);

/* ------------------------------------------------------------------ forward */

/* Bytes of device workspace pw_moe_forward needs (and pw_moe_forward_host). */
size_t pw_workspace_bytes(int T, int E, int top_k, int H, int I);

/*
 * pw_workspace_offset -- where a forward leaves its intermediates inside a
 * workspace of pw_workspace_bytes(T, E, top_k, H, I) bytes, for inspection
 * after the forward (the next forward on the workspace overwrites them):
 *   PW_WS_H  h = silu(gate) * up, fp16 [T*top_k][I], row p = the pair at
 *            permuted position p (see `perm` of pw_moe_forward);
 *   PW_WS_Y  y = W_down . h, fp32 [T*top_k][H], same row order.
 * Returns the byte offset, or (size_t)-1 for a bad section or shape.
 */
#define PW_WS_H 0
#define PW_WS_Y 1
size_t pw_workspace_offset(int T, int E, int top_k, int H, int I, int section);

/*
 * pw_moe_forward -- one fused MoE expert layer ("Fused Mixed-Precision Kernel"):
 * top-k softmax routing, token->expert permutation (stable counting sort with
 * per-expert offsets), per-block-bitwidth dequantised gate_up GEMV/GEMM with
 * SiLU(gate)*up, down GEMV/GEMM, and the routing-weighted combine.
 *   x        device [T][H] fp16 tokens (16-byte aligned)
 *   logits   device [T][E] fp32 router logits (E = the table's n_experts)
 *   top_k    1 <= top_k <= E;  renorm: nonzero divides the top-k weights by their sum
 *   residual device [T][H] fp16 or NULL: added to the combined output
 *   out      device [T][H] fp16: residual + sum_j w[t][j] * y(t, j), rounded once
 *   topk_idx, topk_w  device [T][top_k] int32 / fp32 or NULL: experts in descending
 *            logit order (ties to the lower index) and their weights
 *   offsets  device [E+1] int32 or NULL: per-expert start of the permuted pairs
 *   perm     device [T*top_k] int32 or NULL: pair ids t*top_k+j in (expert, token) order
 *   workspace device, >= pw_workspace_bytes(T, E, top_k, H, I) bytes, 256-byte aligned;
 *            must not be shared by two calls in flight at once.
 * Every block (layer, e, kind) must be registered.  The call only enqueues work on
 * `compute` and never waits.  Arithmetic: fp16 in, fp32 accumulate, h kept in fp16,
 * y in fp32, out rounded to fp16.  A NaN logit is reported through the workspace
 * status word (see pw_workspace_status), not through the return value.
 * Decode-sized batches (T <= 64, T*top_k <= 256) run as one kernel launched with
 * programmatic dependent launch: it may start while the previous kernel on
 * `compute` is still running, and reads the logits and the block descriptors
 * before it waits for that kernel (it touches x, residual, out and the
 * workspace only after).  A kernel that lets its dependents start only when
 * it completes (every ordinary launch, and this library's commit kernels) is a
 * safe producer of the logits or descriptors; a kernel that releases its
 * dependents early must have written the logits before it does.  (The forward
 * itself releases its dependents at once; it writes neither.)
 * The workspace may hold anything when the call is made (fresh memory, an
 * earlier forward's leftovers): the forward itself resets what its CTAs share
 * before any of them uses it.  The decode kernel hands out its work items by
 * tickets in dependency order, so it finishes correctly even while another
 * kernel holds some of the SMs.
 * Each decode-sized call takes a new forward tag on the host, and the kernel
 * sets a forward up when the workspace's ticket word holds another tag.  A
 * call made while `compute` is being captured into a CUDA graph launches a
 * build of the kernel whose last CTA clears that word, so the graph may replay
 * the captured call (with the tag of its capture) any number of times in a row
 * on the same workspace.
 * PW_OK means only that the work was enqueued.  What happens on the device (a
 * NaN logit, a bounded device-side wait that ran out, an unusable block
 * descriptor) is reported only through the workspace status word: read it with
 * pw_workspace_status, or use pw_moe_forward_host, which returns PW_EDEVICE.
 * Errors: PW_EINVAL (shapes, unregistered block, misaligned pointer), PW_ENOMEM
 * (workspace too small), PW_ECUDA.
 */
int pw_moe_forward(pw_table* t, int layer, const void* x, const float* logits, int T,
                   int top_k, int renorm, const void* residual, void* out,
                   int32_t* topk_idx, float* topk_w, int32_t* offsets, int32_t* perm,
                   void* workspace, size_t ws_bytes, pw_stream_t compute);

/*
 * pw_moe_forward_host -- the same layer with HOST inputs and output: copies x,
 * logits (and residual) host->device into the workspace on `compute`, runs
 * pw_moe_forward, copies out device->host, and synchronises `compute` before
 * returning.  Host buffers should be pinned for full copy speed.
 * Errors: as pw_moe_forward, plus PW_EDEVICE when a kernel set a status bit.
 */
int pw_moe_forward_host(pw_table* t, int layer, const void* x_host, const float* logits_host,
                        int T, int top_k, int renorm, const void* residual_host,
                        void* out_host, void* workspace, size_t ws_bytes, pw_stream_t compute);

/*
 * pw_moe_forward_noalloc -- the same layer as pw_moe_forward for callers that
 * cannot allocate device memory (for example a runtime that reserves all of its
 * GPU memory at start-up and refuses later allocations, or a host that only
 * passes input and output buffers).  The paper has no counterpart: this is a
 * deployment convenience of this library.
 *   Scratch: a fixed 8 MiB device array inside the library, reserved on every
 *   GPU that loads it until the process exits; batches whose
 *   pw_workspace_bytes(T, E, top_k, H, I) exceeds 8 MiB are rejected with
 *   PW_ENOMEM and a message (use pw_moe_forward with your own workspace then).
 *   Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   The first call on a device (and the first after the device's context was
 *   reset) looks the array's address up on that device (this may load the
 *   library's kernels there); make that first call before capturing any stream.
 *   All calls share the one array and it keeps the previous call's contents;
 *   a call never trusts them (the forward resets what it shares between its
 *   CTAs itself).  Two calls whose GPU work overlaps in time race on it, so
 *   keep them on one stream or otherwise ordered.
 *   x, logits, residual, out, T, top_k, renorm, compute: as pw_moe_forward
 *   (no routing outputs).  Device-side conditions are reported through the
 *   array's status word: read it with pw_noalloc_status.
 * Errors: as pw_moe_forward, PW_ENOMEM when the batch does not fit, PW_ECUDA
 * when the address lookup fails.
 */
int pw_moe_forward_noalloc(pw_table* t, int layer, const void* x, const float* logits, int T,
                           int top_k, int renorm, const void* residual, void* out,
                           pw_stream_t compute);

/*
 * pw_workspace_status -- reads the device status word of a workspace after the
 * work already on stream s (synchronises s).  *status is 0 or an OR of the
 * PW_STATUS_* bits set by the last forward that used this workspace.
 */
int pw_workspace_status(const void* workspace, pw_stream_t s, int* status);

/*
 * pw_noalloc_status -- pw_workspace_status for the scratch array of
 * pw_moe_forward_noalloc on the current device: the PW_STATUS_* bits of the
 * last pw_moe_forward_noalloc whose work is on stream s or ordered before it
 * (synchronises s).  A noalloc call on another stream that overlaps in time
 * may already have replaced the word (the same race as the calls themselves).
 * Allocates nothing.  Errors: PW_EINVAL (null status), PW_ECUDA.
 */
int pw_noalloc_status(pw_stream_t s, int* status);

/*
 * pw_profile_attach -- measurement hook: the NEXT pw_moe_forward called on this
 * thread records the given CUDA events (cudaEvent_t handles created by the caller)
 * on its stream at its kernel boundaries, then forgets them:
 *   events[0] before the routing/permutation kernel, events[1] after it,
 *   events[2] after the gate_up kernel, events[3] after the down kernel,
 *   events[4] after the combine kernel.
 * n_events < 5 (or NULL) detaches.  The kernels themselves are unchanged.
 */
int pw_profile_attach(void* const* events, int n_events);

#ifdef __cplusplus
}
#endif
#endif /* PW_H */
