/*
 * ikbo.h -- C ABI of the GB300 (sm_103a) IKBO target-attention library.
 *
 * IKBO ("In-Kernel Broadcast Optimization: Co-Designing Kernels for RecSys
 * Inference", §1.1-§1.3 and §3.1 with Fig. 10): a request carries a few users
 * and many candidates.  Each candidate's query tokens attend to its own
 * user's history sequence (target attention, full/non-causal, §3), chosen
 * through a candidate-to-user map handed over by the inference runtime
 * (§1.3 item 3).  The kernels index the user's K/V through that map; no
 * per-candidate copy of a user tensor is ever materialised.
 *
 * Result, for every candidate c, head h and query token t
 * (u = cand_to_user[c], L_u = user_offsets[u+1] - user_offsets[u]):
 *
 *   s_j = scale * <q[c,h,t,:], k[user_offsets[u] + j, h, :]>      j < L_u
 *   out[c,h,t,:] = sum_j softmax(s)_j * v[user_offsets[u] + j, h, :]
 *
 * and an all-zero row when L_u == 0.
 *
 * Layouts (row-major, contiguous, bf16 = IEEE bfloat16):
 *   q, out        bf16 [n_cand, H, Lq, D]
 *   k_user, v_user bf16 [T, H, D], the users' sequences packed back to back
 *                 with no padding ("Optimizing Jagged Flash Attention with
 *                 TLX", introduction: jagged tensors plus an offsets tensor),
 *                 T = user_offsets[n_user]
 *   user_offsets  int32 [n_user + 1], user_offsets[0] = 0, non-decreasing
 *   cand_to_user  int32 [n_cand], values in [0, n_user); any order (sorted
 *                 input skips the internal grouping pass)
 *
 * Ownership: every pointer argument is owned by the caller and never freed
 * by the library.  Device-pointer entry points are asynchronous on `stream`
 * (a cudaStream_t; NULL = legacy default stream) and never synchronise the
 * host unless stated.  The library owns its scratch space (schedule, split
 * partials, tensor maps) and takes it, in stream order on `stream`, from a
 * stream-ordered memory pool of its own on the current device (made by the
 * first call that allocates; it keeps freed memory for later calls until
 * ikbo_shutdown).  The device's default pool is neither used nor changed.
 *
 * CUDA graphs: the device-pointer entry points (ikbo_attn_fwd and its
 * no-alloc, fused, multi-level and linear-compression variants) can be
 * captured on `stream`; their scratch allocations become graph memory
 * nodes and a programmatic dependent launch becomes a programmatic edge.
 * Make one call of each kind with the same device current before the
 * capture: the first call sets the kernels' attributes up.
 *
 * Errors: a negative status is returned at once, with nothing enqueued, for
 * anything the host can see (IKBO_ERR_NULL, _SHAPE, _ALIGN, _SCALE, _ALIAS,
 * _DEVICE).  Bad contents of the index tensors (a candidate mapped outside
 * [0, n_user), offsets that are not a jagged index) and bounded waits that
 * ran out can only be seen on the GPU: the kernels then skip all work (out
 * is left unchanged), never trap, and record the error in the error word of
 * the call's stream, which ikbo_get_device_error(stream) returns: each of
 * the first 63 streams of a device that make a call gets a word of its own
 * (later streams share one), so callers on different streams see only their
 * own errors.  A call captured in a CUDA graph records into the word of the
 * stream it was captured on.  A user's result depends on its
 * own rows of k/v only: rows of other users (which a key tile may reach)
 * never enter it, whatever their values, inf and NaN included.
 */
#ifndef IKBO_H
#define IKBO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* ikbo_stream_t;

enum ikbo_status {
  IKBO_OK = 0,
  IKBO_ERR_NULL = -1,    /* a required pointer is NULL */
  IKBO_ERR_SHAPE = -2,   /* D not 64/128, H < 1, Lq not in [1,128], n_cand < 0, n_user < 0 ... */
  IKBO_ERR_ALIGN = -3,   /* a tensor pointer is not 16-byte aligned */
  IKBO_ERR_SCALE = -4,   /* scale is not finite */
  IKBO_ERR_CUDA = -5,    /* a CUDA runtime/driver call failed (launch, pool allocation) */
  IKBO_ERR_INDEX = -6,   /* device: cand_to_user value outside [0, n_user) */
  IKBO_ERR_OFFSETS = -7, /* device: user_offsets[0] != 0 or decreasing */
  IKBO_ERR_TIMEOUT = -8, /* device: a bounded wait ran out */
  IKBO_ERR_ALIAS = -9,   /* out overlaps an input */
  IKBO_ERR_DEVICE = -10, /* current device is not a compute capability 10.3 GPU */
  IKBO_ERR_BUDGET = -11, /* broadcast path: mem_budget_bytes too small for one candidate */
  IKBO_ERR_SCRATCH = -12 /* ikbo_attn_fwd_noalloc: the call needs more than its fixed scratch */
};

/*
 * IKBO target attention, forward (the hot path).
 * "In-Kernel Broadcast Optimization: Co-Designing Kernels for RecSys
 * Inference", §3.1 (Fig. 10, right): candidates index their user's K/V at
 * run time instead of receiving a broadcast copy.
 *
 * Enqueues on `stream` one persistent tcgen05 attention kernel, which
 * validates the index tensors, groups candidates by user and plans its
 * work in its prologue (up to 20480 candidates and 1024 users; beyond, a
 * planning kernel runs first and the attention kernel reads its work list),
 * packs a user's candidates into 128-row query tiles, and streams that
 * user's K/V tiles through shared memory once per tile (once per two tiles
 * on the two-tile kernel, see ikbo_set_kernel).  When the (user, head)
 * units are few, the two CTAs of a cluster split a unit's keys and merge
 * their partial results through distributed shared memory.
 * All pointers are device pointers; q, k_user, v_user and out must be 16-byte
 * aligned; out must not overlap q, k_user or v_user.  n_cand == 0 is a no-op.
 */
int ikbo_attn_fwd(const void* q, const void* k_user, const void* v_user,
                  const int32_t* user_offsets, const int32_t* cand_to_user,
                  int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                  float scale, void* out, ikbo_stream_t stream);

/*
 * The explicit-broadcast comparison path the IKBO pages argue against
 * ("In-Kernel Broadcast Optimization", §1.4 item 1 and §3.1, Fig. 10 left):
 * K and V are first copied once per candidate into a [S_chunk, H, D] buffer
 * (S_chunk = sum of L_{u(c)} over a chunk of candidates), then the same
 * attention kernel runs with every candidate as its own "user".
 * Candidates are processed in chunks whose copies fit in mem_budget_bytes.
 * Same arguments and layouts as ikbo_attn_fwd.  This path reads
 * user_offsets and cand_to_user back to the host to size its chunks, so it
 * synchronises `stream` once per call.  Returns IKBO_ERR_BUDGET if one
 * candidate's copy does not fit the budget.
 */
int ikbo_broadcast_attn_fwd(const void* q, const void* k_user, const void* v_user,
                            const int32_t* user_offsets, const int32_t* cand_to_user,
                            int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                            float scale, void* out, size_t mem_budget_bytes,
                            ikbo_stream_t stream);

/*
 * ikbo_attn_fwd on HOST buffers (pinned memory recommended).  Copies the
 * inputs to device memory taken from the stream-ordered pool, runs the same
 * two kernels, copies out back and synchronises `stream` before returning.
 * The result is in `out` when the call returns IKBO_OK; device-side index
 * errors are returned directly (no separate ikbo_get_device_error needed).
 * user_offsets is read on the host (T = user_offsets[n_user]).
 */
int ikbo_attn_fwd_host(const void* q, const void* k_user, const void* v_user,
                       const int32_t* user_offsets, const int32_t* cand_to_user,
                       int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                       float scale, void* out, ikbo_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the error word of `stream`
 * on the current device (see "Errors" above): IKBO_OK, or IKBO_ERR_INDEX /
 * _OFFSETS / _TIMEOUT for the first kind of error that calls on `stream`
 * recorded since the word was last cleared.  Errors of calls on other
 * streams are not seen (except between streams past the first 63, which
 * share one word).
 */
int ikbo_get_device_error(ikbo_stream_t stream);

/* Static description of a status code. */
const char* ikbo_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int ikbo_version(void);

/*
 * Releases what the library holds on every device it has used.
 *   - Its events.
 *   - The pinned error-word copy of the host-buffer entry point.
 *   - Its own stream-ordered memory pool on each device, which keeps the
 *     scratch its calls freed: trimmed and destroyed here.
 *   - The streams' error words: cleared, and the streams forgotten.
 * It first waits for each such device's work to finish.  No other library
 * call may run meanwhile.  A later call sets the device up again.  The
 * no-alloc entry point's fixed array is part of the library image and is
 * not released.  Returns IKBO_OK, or IKBO_ERR_CUDA when a device call fails
 * (the release goes on for the other devices).
 */
int ikbo_shutdown(void);

/*
 * Kernel timing, for measurement.  When enabled, every ikbo_attn_fwd call
 * records CUDA events on its stream around its planning kernel and its
 * attention kernel; ikbo_get_timing() synchronises on the last call's events
 * and returns both durations in milliseconds.  After ikbo_broadcast_attn_fwd,
 * attn_ms is the whole GPU part of that path (copies, planning and attention
 * of every chunk) and plan_ms is 0.  Off by default.
 */
int ikbo_set_timing(int enable);
int ikbo_get_timing(float* plan_ms, float* attn_ms);

/*
 * Test hook.  flags = 1 makes the TMA producer of the attention kernel skip
 * arming the query-tile barrier, so the MMA and softmax warps wait until the
 * bound runs out: the kernel then records IKBO_ERR_TIMEOUT, skips all work
 * and exits normally (nothing traps, the context stays usable).
 * flags = 4, with a trace buffer set (ikbo_set_trace), also stamps the
 * prologue of every CTA into item slot 3 (not on the two-tile kernel with
 * Cluster Launch Control, whose grid has more CTAs than the buffer holds):
 * 0 entry, 1 barriers and tensor memory ready, 2 index tensors loaded,
 * 3 tensor maps set, 4 validated, 5 grouped, 6 units counted, 7 planned,
 * 8 cluster ready, 9 work done, 10 exit.  flags = 2 stamps the first item's tiles instead of items 1
 * and 2: softmax tiles 0-3 in slot 1 (points 4j .. 4j+3: scores seen,
 * row maximum done, maxima exchanged, P handed over) and MMA tiles 0-7 in
 * slot 2 (points 2j, 2j+1: S and PV issued).  The bits combine.
 * timeout_ns bounds every in-kernel wait (0 = the default of 2 s).
 * flags = 0 restores normal operation.
 */
int ikbo_set_debug(int flags, uint64_t timeout_ns);

/*
 * Test hook: the library's own stream-ordered pool on the current device
 * (see "Ownership" above).  Writes the bytes its allocations hold now and
 * the most they held at once since the last reset (0 and 0 before the first
 * allocating call); reset != 0 then restarts that high-water mark.  The
 * no-alloc entry point leaves both unchanged.  IKBO_ERR_CUDA when a CUDA
 * call fails.
 */
int ikbo_pool_usage(int reset, uint64_t* used_now, uint64_t* used_high);

/*
 * In-kernel timeline tracing, for profiling.  With a non-NULL device buffer
 * of at least (number of SMs) x 4 x 16 uint64 entries, later calls of the
 * tcgen05 kernel write %globaltimer stamps (ns) into it: entry
 * [(cta * 4 + item) * 16 + point] for the first 4 work items of every CTA,
 * at the points listed in csrc/ikbo_common.cuh (TracePoint), for CTAs with
 * an index below the number of SMs (the two-tile kernel with Cluster Launch
 * Control has more CTAs; the others are not traced).  Entries that are not
 * reached keep their old contents.  NULL switches tracing off (the default).
 * The caller owns the buffer.
 */
int ikbo_set_trace(uint64_t* device_buffer);

/*
 * Fused self + target attention ("In-Kernel Broadcast Optimization", §3.3):
 * in one launch, the target attention of ikbo_attn_fwd (q, out as there) and
 * the self-attention of every user's sequence over itself, with the same
 * keys and values and queries from the user side:
 *
 *   out_user[r, h, :] = sum_j softmax_j(scale * q_user[r, h, :] . k_user[o + j, h, :])
 *                       * v_user[o + j, h, :],   j = 0 .. L_u - 1,
 *
 * for every sequence row r of user u (o = user_offsets[u] <= r < user_offsets[u + 1]);
 * full attention, no causal mask.  Both kinds of query tile stream the same
 * user's K/V tiles.
 *
 *   q_user, out_user   bf16 [T, H, D], device memory, 16-byte aligned; out_user
 *                      shares no byte with any input or with out.
 *   T                  the number of sequence rows; user_offsets[n_user] must
 *                      equal it (checked on the device: IKBO_ERR_OFFSETS).
 *   other arguments    as ikbo_attn_fwd; n_cand may be 0 (self-attention
 *                      only; q, cand_to_user and out may then be NULL).
 *
 * Runs on the tcgen05 kernel that the automatic choice or ikbo_set_kernel
 * picks for the candidates (the one-tile kernel when the choice is the SIMT
 * kernel); on the two-tile kernel a self-attention item is two blocks of 128
 * sequence rows sharing the user's key tiles.  Planning is in-kernel:
 * n_cand <= 20480 and n_user <= 1024, else IKBO_ERR_SHAPE.  T < 0 or T >= 2^31: IKBO_ERR_SHAPE.  n_cand == 0 and T == 0:
 * no-op.  Errors and ownership otherwise as ikbo_attn_fwd.
 */
int ikbo_fused_attn_fwd(const void* q, const void* q_user, const void* k_user, const void* v_user,
                        const int32_t* user_offsets, const int32_t* cand_to_user, int64_t n_cand,
                        int64_t n_user, int64_t T, int32_t H, int32_t Lq, int32_t D, float scale,
                        void* out, void* out_user, ikbo_stream_t stream);

/*
 * IKBO linear compression ("In-Kernel Broadcast Optimization", §2): for every
 * candidate b of user u = cand_to_user[b], the compression of its K input
 * embeddings (its user's K_user, then its own K_cand, each of N values) by
 * W = [W_user | W_cand]:
 *
 *   out[b] = W_user @ X_user[u] + W_cand @ X_cand[b]         (M x N)
 *
 * The user term is computed once per user (accumulated in fp32, kept in bf16 in a library-owned
 * buffer) and added in the epilogue of the candidate product, so the user
 * block is never copied per candidate (§2.1-§2.3).  Two launches of one
 * tcgen05 kernel, the second a programmatic dependent of the first.
 *
 *   W_user  bf16 [M, K_user]        W_cand  bf16 [M, K_cand]
 *   X_user  bf16 [n_user, K_user, N]  X_cand  bf16 [n_cand, K_cand, N]
 *   out     bf16 [n_cand, M, N]; shares no byte with an input
 *   All device memory, 16-byte aligned (cand_to_user 4-byte aligned).
 *   K_user, K_cand: multiples of 8 (blocks zero-padded by the caller, which
 *   §2.2 shows to be exact); K_cand >= 8; K_user = 0 means no user block
 *   (then W_user, X_user, cand_to_user may be NULL).  N in {64, 128, 192, 256}.
 *   Accumulation in fp32; out rounded to bf16 (nearest even).
 * Errors: bad sizes IKBO_ERR_SHAPE, NULL IKBO_ERR_NULL, misaligned
 * IKBO_ERR_ALIGN, overlap IKBO_ERR_ALIAS; a cand_to_user value outside
 * [0, n_user) sets IKBO_ERR_INDEX in the device error word and that
 * candidate's rows are not written.  n_cand == 0: no-op.
 */
int ikbo_lce_fwd(const void* W_user, const void* W_cand, const void* X_user, const void* X_cand,
                 const int32_t* cand_to_user, int64_t n_cand, int64_t n_user, int32_t M,
                 int32_t K_user, int32_t K_cand, int32_t N, void* out, ikbo_stream_t stream);

/*
 * Linear compression over a user -> ads vendor -> ads item hierarchy ("In-Kernel
 * Broadcast Optimization", §5 with §2): an item's K input embeddings are its
 * user's block, its vendor's block and its own, so with v = item_to_vendor[i]
 * and u = vendor_to_user[v]
 *
 *   out[i] = W_user @ X_user[u] + W_vendor @ X_vendor[v] + W_item @ X_item[i]
 *
 * Each level's product is computed once per entry of that level: up to three
 * launches of the linear-compression kernel, each a programmatic dependent
 * of the one before, users (bf16 terms), then vendors (their product plus
 * their user's term, bf16), then items (their product plus their vendor's
 * term, to bf16).  No block is ever copied per vendor or per item.
 *
 *   W_user [M, K_user], W_vendor [M, K_vendor], W_item [M, K_item]    bf16
 *   X_user [n_user, K_user, N], X_vendor [n_vendor, K_vendor, N],
 *   X_item [n_item, K_item, N]                                         bf16
 *   item_to_vendor int32 [n_item], vendor_to_user int32 [n_vendor]; any order
 *   out bf16 [n_item, M, N]; shares no byte with an input
 *   All device memory, 16-byte aligned (the maps 4-byte aligned).
 *   K_user, K_vendor: multiples of 8, 0 = no such block (its W and X may then
 *   be NULL; with neither, the maps are not read and may be NULL; without a
 *   user block vendor_to_user is not read).  K_item: a multiple of 8, >= 8.
 *   N in {64, 128, 192, 256}.  Accumulation in fp32; out rounded to bf16.
 * Errors as ikbo_lce_fwd.  On the device: an item_to_vendor value outside
 * [0, n_vendor), or a vendor_to_user value outside [0, n_user) that an item
 * reaches, sets IKBO_ERR_INDEX and that item's rows are not written.
 * ikbo_get_timing, when enabled, reports the user level as its first value
 * and the vendor and item levels together as its second.  n_item == 0: no-op.
 */
int ikbo_ml_lce_fwd(const void* W_user, const void* W_vendor, const void* W_item,
                    const void* X_user, const void* X_vendor, const void* X_item,
                    const int32_t* item_to_vendor, const int32_t* vendor_to_user, int64_t n_item,
                    int64_t n_vendor, int64_t n_user, int32_t M, int32_t K_user, int32_t K_vendor,
                    int32_t K_item, int32_t N, void* out, ikbo_stream_t stream);

/*
 * Target attention over a user -> ads vendor -> ads item hierarchy ("In-Kernel
 * Broadcast Optimization", §5: a user sees several vendors, each vendor offers
 * several items; two nested broadcasts with independent, uneven ratios).  Every
 * item is a candidate: its Lq query tokens attend to the sequence of the user
 * its vendor belongs to,
 *
 *   u(i) = vendor_to_user[item_to_vendor[i]],
 *
 * and out is that of ikbo_attn_fwd with cand_to_user[i] = u(i).  The kernels
 * look the two maps up while they plan (in-kernel, or in the planning kernel
 * beyond the in-kernel limits); no per-item user map is passed in.
 *
 *   item_to_vendor  int32 [n_item], values in [0, n_vendor), any order
 *   vendor_to_user  int32 [n_vendor], values in [0, n_user), any order
 *   other arguments as ikbo_attn_fwd, with n_item in place of n_cand.
 * A value of either map out of range (only vendors that some item names are
 * read) sets IKBO_ERR_INDEX in the device error word and nothing is written.
 * n_item == 0: no-op.  n_vendor < 0 or >= 2^31: IKBO_ERR_SHAPE; n_vendor == 0
 * with items: IKBO_ERR_INDEX; vendor_to_user NULL: IKBO_ERR_NULL, not 4-byte
 * aligned: IKBO_ERR_ALIGN.  Kernel choice and other errors as ikbo_attn_fwd.
 */
int ikbo_ml_attn_fwd(const void* q, const void* k_user, const void* v_user,
                     const int32_t* user_offsets, const int32_t* item_to_vendor,
                     const int32_t* vendor_to_user, int64_t n_item, int64_t n_vendor,
                     int64_t n_user, int32_t H, int32_t Lq, int32_t D, float scale, void* out,
                     ikbo_stream_t stream);

/*
 * Selects the attention kernel for later calls on this thread.  Returns the
 * previous value.
 *   0  automatic (the default): 3 when the users have on average at least
 *      two query tiles each (n_cand >= 2 * c * n_user, c = floor(128 / Lq)),
 *      the batch makes at least 600 two-tile items
 *      (H * ceil(n_cand / (2 * c)) >= 600), or at least 200 for target
 *      attention alone with D = 128 and at most 256 users (the case that
 *      kernel 3 deals by Cluster Launch Control, each next item asked for
 *      late), and the inputs fit the in-kernel planning limits
 *      (n_cand <= 20480, n_user <= 1024); else 2;
 *   1  the SIMT kernel, kept as an independent GPU cross-check;
 *   2  the tcgen05/TMEM/TMA kernel with one query tile (up to 128 rows of one
 *      user's candidates) per work item, whose pair mode splits the keys of
 *      a unit over the two CTAs of a cluster when units are few;
 *   3  the tcgen05 kernel with two query tiles of the same user and head per
 *      work item, sharing each K/V tile between them (ping-pong of two
 *      softmax warpgroups); with at most 256 users its grid is one CTA per
 *      item (a bound on their number) and running CTAs take over the items
 *      of CTAs not yet started (Cluster Launch Control), longest first;
 *      inputs beyond the in-kernel planning limits run on kernel 2;
 *   4  the tcgen05 kernel with the key tiles of one query tile dealt to two
 *      softmax warpgroups in turn (even and odd tiles) and merged in the
 *      CTA, one unit per CTA when units are few; a unit far longer than the
 *      balanced share is cut into up to 8 key ranges on as many CTAs and
 *      merged by the first of them.  For batches of a few very long users
 *      (tens of thousands of keys); never chosen automatically, since the
 *      host cannot see the sequence lengths.  Inputs beyond the in-kernel
 *      planning limits run on kernel 2, and so do fused self + target calls.
 * Any other value selects 0.
 */
int ikbo_set_kernel(int which);

/*
 * The kernel (1 to 4 as above) that a call with these sizes would run with
 * this thread's current choice: ikbo_attn_fwd when self_rows < 0, else
 * ikbo_fused_attn_fwd over self_rows sequence rows (a fused call runs on
 * kernel 2 or 3).  Host arithmetic only: it touches no GPU.  Negative sizes,
 * H < 1, Lq outside [1, 128] or D other than 64 and 128 return
 * IKBO_ERR_SHAPE.
 */
int ikbo_selected_kernel(int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                         int64_t self_rows);

/*
 * Number of kernel launches that ikbo_attn_fwd (and ikbo_attn_fwd_host,
 * ikbo_attn_fwd_noalloc) makes for a batch of n_cand candidates over n_user
 * users with the current kernel choice of this thread: 0 for an empty batch,
 * 1 when the tcgen05 kernel plans in-kernel (n_cand <= 20480 and
 * n_user <= 1024), else 2 (a planning kernel, then the attention kernel).
 * Host arithmetic only: it touches no GPU.  Negative sizes return
 * IKBO_ERR_SHAPE.
 */
int ikbo_launches_per_call(int64_t n_cand, int64_t n_user);

/*
 * ikbo_attn_fwd without any memory allocation.  (The IKBO pages have no
 * counterpart to this entry point; it exists for deployment.)
 *
 * Some callers cannot let a library allocate GPU memory: a serving process
 * whose memory manager reserves the device memory up front and forbids any
 * later driver allocation, or a platform where stream-ordered memory pools
 * are unavailable.  ikbo_attn_fwd takes its scratch (work list, split
 * partials, tensor maps) from the stream-ordered pool on every call; this
 * variant takes it instead from one fixed array in device memory that is
 * part of the library (IKBO_NOALLOC_SCRATCH_BYTES = 40 MiB, held on every
 * GPU where the library is loaded until the process exits).  It allocates
 * no device memory and no pinned host memory (no cudaMalloc, cudaMallocAsync,
 * cudaMallocFromPoolAsync, cudaHostAlloc or cudaFree) and changes no memory
 * pool, on any call, the first included.
 *
 * Arguments, layouts, results and errors are those of ikbo_attn_fwd.  In
 * addition it returns IKBO_ERR_SCRATCH, with nothing enqueued, when the call
 * would need more scratch than the array holds (the need grows with n_cand,
 * n_user, H and D; every configuration in workloads.py, with every kernel
 * choice, needs under 30 MiB).
 *
 * The first call on a device sets the device up with that device current:
 * it queries the device's attributes, looks up the array's and the error
 * word's device addresses (cudaGetSymbolAddress) and sets the chosen
 * kernel's shared-memory attribute; make that first call before any stream
 * capture.  Every call on a device uses the same array.  What a call's
 * kernels read there is written earlier in the same call, except the flags
 * of units cut into key ranges, which carry a value unique to the call and
 * are reset after use; so a call never depends on what an earlier call left
 * there.  Two calls whose kernels overlap on the GPU (different streams, no
 * ordering between them) race on the array and give wrong results: order
 * them on one stream, or use ikbo_attn_fwd.
 */
#define IKBO_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)
int ikbo_attn_fwd_noalloc(const void* q, const void* k_user, const void* v_user,
                          const int32_t* user_offsets, const int32_t* cand_to_user,
                          int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                          float scale, void* out, ikbo_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IKBO_H */
