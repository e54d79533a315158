/*
 * spanla.h -- C ABI of libspanla, the packed linear-attention pass for GB300
 * (sm_103a).
 *
 * What a call computes ("Serving 0.88M TPS from Two RTXs and Mac Minis",
 * sections "The Workload", "Kernels" and "Long Requests"): unnormalised causal
 * linear attention, independently per head,
 *
 *     S_t = S_{t-1} + k_t v_t^T        o_t = S_t^T q_t      (inclusive diagonal)
 *
 * over a *packed pass*: one buffer of rows that holds many variable-length
 * views and many short branches.  Each view starts from S = 0.  Each branch
 * starts from the final state of its parent view (the state after the view's
 * last row) and runs over its own rows only; branches never see one another
 * (section "The Workload": branches attend to the view but not to each other).
 * The work follows the chunked form the "Kernels" section describes (each
 * chunk a few 64x64 matrix products; one scan of states covers every view of
 * the pass): a local state K^T V per piece of rows, the prefix of those states
 * over every view of the pass, and the output of every 128-row tile (masked
 * Q K^T V inside the tile plus Q S_prev).  For bf16 inputs the output work is
 * cut into one run of tiles per SM; a piece is the part of one view (per
 * head) inside one run, and the output kernel carries the state from tile to
 * tile on chip.  By default the whole bf16 pass is one cooperative launch
 * (the SMs sum the prefixes they need after a grid-wide counter); the
 * page's three launches (local states, one segmented scan, output) are the
 * alternative span_la_pass_variant selects.  For fp32 inputs the pieces are
 * 64-row chunks and every 128-row tile starts from its chunk's prefix.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  q, k, v and out are contiguous row-major [T][H][64] arrays in
 *   device memory (T = dims.total_rows, H = dims.num_heads), element type
 *   dims.dtype, base address 16-byte aligned.  States are contiguous fp32
 *   [n][H][64][64] arrays in device memory with S[i][j] at i*64 + j (i = key
 *   dimension, j = value dimension), 16-byte aligned.
 * Segments.  view_cu_seqlens (num_views + 1 entries) and branch_cu_seqlens
 *   (num_branches + 1 entries) are HOST int32 arrays of non-decreasing
 *   absolute row offsets into the same [T] buffer: segment s covers rows
 *   [cu[s], cu[s+1]).  Zero-length segments are allowed; a count of 0 is
 *   allowed (the array may then be NULL).  No two non-empty segments may
 *   overlap.  Rows in no segment are never read into a result and never
 *   written.  branch_parent (num_branches entries, HOST int32) names the
 *   parent of every branch.
 * Ownership.  The caller owns every buffer.  Host arrays are read only during
 *   the call.  The library allocates its workspace stream-ordered
 *   (cudaMallocAsync / cudaFreeAsync on `stream`) and frees it before the
 *   work completes on the stream.
 * Asynchrony.  A call only enqueues work on `stream` (a cudaStream_t on the
 *   current device; 0 = legacy default stream).  Outputs are valid once the
 *   stream has reached the call; inputs must stay unchanged until then.  The
 *   pass, branch and softmax calls do not synchronise the device: the
 *   per-device cache of launch plans (16 per device, keyed on the metadata,
 *   least recently used evicted) frees an evicted plan in stream order
 *   behind the calls that read it.  The cached plans, their events and the
 *   pinned staging buffers belong to the device's primary context and live
 *   until the process exits: do not call the library on a device after a
 *   cudaDeviceReset of that device.
 * Graphs.  The pass, branch and softmax calls may be recorded while `stream`
 *   is being captured into a CUDA graph: the recorded work replays on the
 *   buffers of the recorded call (their current contents), with its own
 *   workspace allocations in the graph.  The descriptor bytes of a recorded
 *   call are kept by the library for the life of the process.
 * Precision.  bf16 or fp32 inputs; the state and every accumulation are fp32.
 *   With fp32 inputs, fp32 operands (q, k, v, and the state and P tiles fed
 *   to the tensor cores) are split into two bf16 parts whose cross products
 *   are summed.  With bf16 inputs, P enters P v and the state enters q S
 *   rounded to bf16, like q, k and v themselves (the state itself stays
 *   fp32).  Outputs are rounded to the input type (round to nearest even).
 *   Results are deterministic run to run (no floating-point atomics).
 * Errors.  Metadata, shape, pointer and alignment problems are detected on the
 *   host before anything is enqueued; the call then returns an error code and
 *   writes nothing.  Device-side waits are bounded: a wait that runs out sets
 *   a device error word, the kernel returns without trapping, and
 *   span_la_check() reports SPAN_LA_ERR_TIMEOUT.  span_la_last_error_detail()
 *   describes the last failure on the calling thread.
 * Supported.  head_dim == 64, num_heads >= 1, total_rows < 2^31,
 *   dtype SPAN_LA_BF16 or SPAN_LA_F32, one GPU of compute capability 10.3.
 */
#ifndef SPANLA_H
#define SPANLA_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPAN_LA_BF16 = 0,
    SPAN_LA_F32 = 1
} span_la_dtype;

typedef enum {
    SPAN_LA_OK = 0,
    SPAN_LA_ERR_INVALID = 1,      /* bad metadata, pointer, alignment or size */
    SPAN_LA_ERR_UNSUPPORTED = 2,  /* head_dim != 64, unknown dtype, wrong GPU */
    SPAN_LA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
    SPAN_LA_ERR_NOMEM = 4,        /* workspace allocation failed */
    SPAN_LA_ERR_TIMEOUT = 5       /* a bounded device wait ran out */
} span_la_status;

typedef struct {
    int64_t total_rows;  /* T: rows of q, k, v and out */
    int32_t num_heads;   /* H */
    int32_t head_dim;    /* must be 64 */
    int32_t dtype;       /* span_la_dtype of q, k, v and out */
} span_la_dims;

/*
 * span_la_pass -- one packed pass over views and branches.
 *
 * Section "Kernels" (one scan per pass; shared branch passes with the small
 * kernels fused) and section "The Workload".  Computes o for every view row
 * and every branch row and writes each view's final state to view_state_out.
 * One cooperative launch for bf16 inputs by default (span_la_pass_variant).
 *
 *   q, k, v          device [T][H][64], dims.dtype
 *   view_cu_seqlens  host int32 [num_views + 1]
 *   branch_cu_seqlens host int32 [num_branches + 1]
 *   branch_parent    host int32 [num_branches], each in [0, num_views)
 *   out              device [T][H][64], dims.dtype; only segment rows written
 *   view_state_out   device fp32 [num_views][H][64][64]; required when
 *                    num_views > 0 (an empty view gets the zero state)
 *   stream           stream to enqueue on
 */
span_la_status span_la_pass(const void *q, const void *k, const void *v,
                            span_la_dims dims,
                            const int32_t *view_cu_seqlens, int32_t num_views,
                            const int32_t *branch_cu_seqlens, int32_t num_branches,
                            const int32_t *branch_parent,
                            void *out, float *view_state_out,
                            cudaStream_t stream);

/*
 * span_la_plan_prepare -- build and upload the launch plan of a later
 * span_la_pass, ahead of that call.
 *
 * Section "Batching in the Router": the router packs a pass from the
 * requests it has gathered, so the pass's metadata is known before its rows
 * reach the GPU.  Section "Kernels": a pass is launched from descriptors
 * built on the host from that metadata.  span_la_pass builds them on its first
 * call with new metadata (tens of microseconds of host time) and keeps them
 * in the per-device plan cache; this call does the same work earlier, for
 * example while the pass's q, k and v are still being copied in, so that the
 * pass itself finds the plan in the cache.  It computes nothing and touches
 * no q, k, v or output buffer.
 *
 *   dims             as the pass's dims (total_rows bounds the metadata;
 *                    num_heads and dtype select the plan)
 *   view_cu_seqlens, num_views, branch_cu_seqlens, num_branches,
 *   branch_parent    as for span_la_pass (host arrays, read during the call)
 *   stream           the descriptor upload is enqueued here (pinned staging,
 *                    stream ordered); a pass on another stream waits for it
 *                    through an event
 *   match            a span_la_pass on the same device with the same
 *                    metadata, num_heads, dtype and pass structure
 *                    (span_la_pass_variant) uses the prepared plan.  The
 *                    cache holds 16 plans per device, least recently used
 *                    evicted: a plan is lost if 16 others are used or
 *                    prepared after it and before its pass.  Preparing a
 *                    plan that is already cached only marks it as used
 *   errors           metadata problems as for span_la_pass, nothing
 *                    enqueued; SPAN_LA_ERR_UNSUPPORTED while `stream` is
 *                    being captured (captured passes do not use the cache);
 *                    SPAN_LA_ERR_NOMEM if the descriptor block cannot be
 *                    allocated (stream ordered, on `stream`)
 */
span_la_status span_la_plan_prepare(span_la_dims dims,
                                    const int32_t *view_cu_seqlens, int32_t num_views,
                                    const int32_t *branch_cu_seqlens, int32_t num_branches,
                                    const int32_t *branch_parent, cudaStream_t stream);

/*
 * span_la_branches_from_state -- branches only, each forking from a cached
 * view state.
 *
 * Section "Long Requests": branches only attend to their own view, so they can
 * be split into shards that each reuse the view's cached linear-attention
 * state instead of recomputing the view.  Equivalent to the branch rows of
 * span_la_pass when cached_state holds that pass's view_state_out.
 *
 *   cached_state     device fp32 [num_states][H][64][64]
 *   branch_parent    host int32 [num_branches], each in [0, num_states)
 *   out              device [T][H][64]; only branch rows written
 *   other arguments  as for span_la_pass
 */
span_la_status span_la_branches_from_state(const float *cached_state, int32_t num_states,
                                           const void *q, const void *k, const void *v,
                                           span_la_dims dims,
                                           const int32_t *branch_cu_seqlens,
                                           int32_t num_branches,
                                           const int32_t *branch_parent,
                                           void *out, cudaStream_t stream);

/*
 * span_la_pass_noalloc -- span_la_pass for callers that cannot allocate
 * device memory during a call.
 *
 * The pages have no counterpart of this entry point; it is a deployment aid.
 * span_la_pass takes its workspace from the stream-ordered allocator on every
 * call.  A caller that has handed the GPU's memory to its own pool, or that
 * runs where an allocation could block or fail at the wrong moment, can use
 * this variant instead: it computes the same pass with the same kernels, but
 * its workspace is one fixed 16 MiB array in device memory that belongs to the
 * library (every GPU on which it is used holds the array until the process
 * exits).  It calls no allocating routine.
 *
 *   arguments        as for span_la_pass; dims.dtype must be SPAN_LA_BF16
 *                    (fp32 inputs need per-call scratch: SPAN_LA_ERR_UNSUPPORTED)
 *   size limit       the descriptors (64 bytes per 128-row output tile of
 *                    one head) plus the workspace states (16 KiB fp32 each)
 *                    must fit in 16 MiB.  A piece is the part of one view-
 *                    head inside one SM's run of output tiles.  In the
 *                    one-launch structure (the default, span_la_pass_variant)
 *                    only a piece whose state another SM needs has a
 *                    workspace state, at most one per boundary between two
 *                    runs (fewer than the SM count), so the descriptors set
 *                    the limit: about 200,000 output tiles, i.e. some 25
 *                    million token-heads.  In the three-launch structure
 *                    every piece-head has one, about 1,000 in all: a pass
 *                    needs at most about (views + SMs) x heads of them (a
 *                    16-head pass of up to ~60 views fits on a 152-SM GPU).
 *                    A larger pass returns SPAN_LA_ERR_INVALID with the bytes
 *                    it needs, before anything is enqueued
 *   first call       the first call on a device looks up the array's device
 *                    address (cudaGetSymbolAddress with that device current)
 *                    and caches it; make that first call before any stream
 *                    capture, and do not use this entry point across a
 *                    cudaDeviceReset of that device (the cached address dies
 *                    with the context)
 *   memory           the array is reserved on every device whose context
 *                    loads the library's module that holds it: where it was
 *                    used, or on every device under eager module loading
 *                    (CUDA_MODULE_LOADING=EAGER); it stays until the process
 *                    exits
 *   sharing          every call uses the same array and leaves its contents
 *                    behind; calls whose work overlaps on the GPU (other
 *                    streams, other threads) race on it -- order them on one
 *                    stream
 *   errors           as for span_la_pass.  Device-side wait timeouts of this
 *                    path land in an error word of its own, which
 *                    span_la_check (on the same device) reads and clears
 *                    together with the library's main error word; the word
 *                    is not cleared by a call, so a timeout stays recorded
 *                    until span_la_check reports it
 */
span_la_status span_la_pass_noalloc(const void *q, const void *k, const void *v,
                                    span_la_dims dims,
                                    const int32_t *view_cu_seqlens, int32_t num_views,
                                    const int32_t *branch_cu_seqlens, int32_t num_branches,
                                    const int32_t *branch_parent,
                                    void *out, float *view_state_out,
                                    cudaStream_t stream);

/*
 * span_la_check -- synchronise `stream`, then report (and clear) the device
 * error words of the current device: the library's main word and, where
 * span_la_pass_noalloc has run on the device, that path's own word.  Returns
 * SPAN_LA_ERR_CUDA if the stream reports a CUDA error, SPAN_LA_ERR_TIMEOUT if
 * a kernel's bounded wait ran out, SPAN_LA_OK otherwise.  Allocates nothing.
 */
span_la_status span_la_check(cudaStream_t stream);

/* Static text for a status code. */
const char *span_la_status_string(span_la_status status);

/* Text describing the last failure of a call made on this host thread. */
const char *span_la_last_error_detail(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t span_la_version(void);

/*
 * span_la_selftest_wait_timeout -- failure-detection hook: enqueue one tiny
 * kernel whose bounded wait is on an mbarrier that nothing ever completes,
 * with a wait limit of `limit_us` microseconds (1 .. 1,000,000).  The kernel
 * gives up, sets the device error word and returns; span_la_check() then
 * reports SPAN_LA_ERR_TIMEOUT.  Used by the tests to show that a wait that
 * runs out neither traps nor hangs.
 */
span_la_status span_la_selftest_wait_timeout(int32_t limit_us, cudaStream_t stream);

/*
 * span_la_selftest_wait_timeout_noalloc -- the same failure-detection hook
 * for the error word of span_la_pass_noalloc: the probe kernel's wait runs
 * out after `limit_us` and sets that word; span_la_check() then reports
 * SPAN_LA_ERR_TIMEOUT.  Allocates nothing (the first use on a device looks
 * the word up, as span_la_pass_noalloc does).
 */
span_la_status span_la_selftest_wait_timeout_noalloc(int32_t limit_us, cudaStream_t stream);

/*
 * span_la_pass_variant -- how span_la_pass and span_la_pass_noalloc run a
 * bf16 pass (process-wide; calls made afterwards use it).  Both compute the
 * same result (up to the order of fp32 additions of states):
 *   SPAN_LA_PASS_ONE_LAUNCH (default): one cooperative launch.  Each CTA
 *     sums K^T V over its own pieces whose state another CTA needs, counts
 *     itself in a grid-wide counter, waits (bounded) for the others only
 *     where it needs their states and sums those itself; the CTA that holds a
 *     view's last tile computes the view's final state on chip, writes it to
 *     view_state_out and starts the view's branches in its run from it.  One
 *     scan per pass without a scan kernel ("Kernels": one scan per pass; the
 *     small kernels fused).
 *   SPAN_LA_PASS_THREE_LAUNCHES: span state -> segmented scan -> output, as
 *     the "Kernels" section lays the pass out.
 * fp32 passes and span_la_branches_from_state always take the launches of
 * their own path.  Unknown variant: SPAN_LA_ERR_INVALID.
 */
#define SPAN_LA_PASS_ONE_LAUNCH 0
#define SPAN_LA_PASS_THREE_LAUNCHES 1
span_la_status span_la_pass_variant(int32_t variant);

/*
 * span_la_fault_inject -- failure-detection hook on the host: with kind
 * SPAN_LA_FAULT_ALLOC, the library's next `count` device allocations
 * (workspace, descriptor blocks) fail as if the device were out of memory,
 * so the calls that make them return SPAN_LA_ERR_NOMEM before enqueueing any
 * kernel.  count = 0 clears it.  Process-wide; meant for tests.  Unknown kind
 * or count < 0: SPAN_LA_ERR_INVALID.
 */
#define SPAN_LA_FAULT_ALLOC 1
span_la_status span_la_fault_inject(int32_t kind, int32_t count);

/*
 * span_la_softmax_plan_stats -- host only, no CUDA call: the work units of
 * span_la_softmax_pass for this metadata, head count and number of CTAs
 * (normally the SM count), into stats[0..3]:
 *   stats[0] work items: (query tile of <= 128 rows, head) pairs
 *   stats[1] query rows those items cover (summed over heads)
 *   stats[2] key blocks the items process: each is one 128 x 128 x 64 Q K^T
 *            and one 128 x 64 x 128 P V product on the tensor cores
 *   stats[3] CTAs the launch uses
 * Returns SPAN_LA_ERR_INVALID on bad metadata, like the entry point.
 */
span_la_status span_la_softmax_plan_stats(const int32_t *view_cu_seqlens, int32_t num_views,
                                          const int32_t *branch_cu_seqlens, int32_t num_branches,
                                          const int32_t *branch_parent, int32_t num_heads,
                                          int32_t num_sms, int64_t *stats);

/*
 * span_la_plan_stats -- host only, no CUDA call: the work units a call with
 * this metadata, head count and dtype would launch on a GPU with `num_sms`
 * SMs (used to count the algorithmic bytes of each kernel), for the pass
 * variant in effect (span_la_pass_variant).  Every count is summed over the
 * heads.
 *   stats[0] state slots: 64-row chunk-heads (fp32) or piece-heads (bf16);
 *            in the one-launch pass, the pieces whose state another CTA reads
 *   stats[1] row-heads those slots cover (rows whose K and V are read to
 *            make them: by the state kernel, or in the one-launch pass's first
 *            phase)
 *   stats[2] runs of the segmented scan (0 in the one-launch pass)
 *   stats[3] final view states written (view-heads)
 *   stats[4] output tile-heads (<= 128 rows each)
 *   stats[5] row-heads those tiles cover
 *   stats[6] fp32 64x64 start-state reads of the output kernel (each state
 *            of a sum counted)
 *   stats[7] output pieces (fp32: tile-heads)
 *   stats[8] longest run of tiles of one output CTA (bf16; 1 for fp32)
 * from_state != 0 plans span_la_branches_from_state (views ignored).
 * Returns SPAN_LA_ERR_INVALID on bad metadata, like the entry points.
 */
span_la_status span_la_plan_stats(const int32_t *view_cu_seqlens, int32_t num_views,
                                  const int32_t *branch_cu_seqlens, int32_t num_branches,
                                  const int32_t *branch_parent, int32_t num_parents,
                                  int32_t from_state, int32_t num_heads, int32_t dtype,
                                  int32_t num_sms, int64_t *stats);

/*
 * Kernel profiling (tracing hook).  Kernels are numbered
 *   0 split_f32, 1 chunk_state, 3 tile_output (fp32 inputs),
 *   2 segmented_scan (both), 4 span_state, 5 span_output (bf16 inputs),
 *   6 softmax_attn (span_la_softmax_pass).
 * Launches of every kernel are always counted.  While profiling is enabled,
 * every launch is also bracketed by two CUDA events recorded on the call's
 * stream (one device only); span_la_profile_read() waits for the pending
 * events and adds their elapsed times up.  Enabling adds two event records per
 * launch and nothing else to the work on the stream.
 */
#define SPAN_LA_NUM_KERNELS 7

/* Turn event timing on (non-zero) or off. */
span_la_status span_la_profile_enable(int32_t enable);

/*
 * Per kernel id k < n (n <= SPAN_LA_NUM_KERNELS): ms_total[k] = summed event
 * time of its timed launches, timed[k] = launches timed, launches[k] = all
 * launches since the last reset.  Any of the three arrays may be NULL.
 * Synchronises on the pending events.
 */
span_la_status span_la_profile_read(double *ms_total, int64_t *timed, int64_t *launches,
                                    int32_t n);

/* Clear the counters and timings (waits for pending events first). */
span_la_status span_la_profile_reset(void);

/* Static name of kernel id k, or NULL. */
const char *span_la_kernel_name(int32_t k);

/*
 * span_la_softmax_pass -- one softmax-attention layer of the hybrid model over
 * the same packed rows ("Serving 0.88M TPS from Two RTXs and Mac Minis",
 * section "The Workload": a branch attends to its view and never to its
 * siblings; section "Long Requests": the softmax layers' K/V is the other
 * half of what a view contributes to its branches).  Per head h and row t:
 *
 *   o_t = sum_j softmax_j(scale * q_t . k_j) v_j,   lse_t = ln sum_j exp(scale * q_t . k_j),
 *
 * where a view row t sees the rows of its view up to and including t, and a
 * branch row t sees every row of its parent view plus the rows of its own
 * branch up to and including t.  Same metadata rules and layouts as
 * span_la_pass: q, k, v, out are device [T][H][64] bf16 (16-byte aligned);
 * accumulation is fp32 and the probabilities enter the P V product as bf16.
 *   scale    > 0, or 0 for 1/sqrt(64).  NaN, infinite or negative: INVALID.
 *   lse_out  device fp32 [T][H] (4-byte aligned) or NULL (not written).
 * Rows in no segment are not written.  dtype must be SPAN_LA_BF16, else
 * SPAN_LA_ERR_UNSUPPORTED.  One kernel launch on `stream`, asynchronous;
 * call span_la_check() to collect device-side wait timeouts.
 */
span_la_status span_la_softmax_pass(const void *q, const void *k, const void *v, span_la_dims dims,
                                    const int32_t *view_cu_seqlens, int32_t num_views,
                                    const int32_t *branch_cu_seqlens, int32_t num_branches,
                                    const int32_t *branch_parent, float scale, void *out,
                                    float *lse_out, cudaStream_t stream);

/*
 * span_la_softmax_branches_from_kv -- the softmax layer for branches only,
 * each attending to its parent view's K and V kept from an earlier pass (the
 * softmax half of the view cache: "Serving 0.88M TPS from Two RTXs and Mac
 * Minis", section "Long Requests") and to its own branch's rows up to itself.
 * Equals the branch rows of span_la_softmax_pass over the views and branches
 * together; the branches of one long request can be run as several calls
 * (shards) over the same view K/V.
 *   view_k, view_v   device bf16 [view_rows][H][64], 16-byte aligned; view p
 *                    is rows [view_cu_seqlens[p], view_cu_seqlens[p+1]) of them.
 *   q, k, v, out     device bf16 [T][H][64] (T = dims.total_rows) holding the
 *                    branch rows at branch_cu_seqlens; branch b's parent is
 *                    view branch_parent[b] of view_cu_seqlens.
 *   scale, lse_out   as span_la_softmax_pass.
 * Rows of out outside the branches are not written.
 */
span_la_status span_la_softmax_branches_from_kv(const void *view_k, const void *view_v, int64_t view_rows,
                                                const int32_t *view_cu_seqlens, int32_t num_views,
                                                const void *q, const void *k, const void *v,
                                                span_la_dims dims, const int32_t *branch_cu_seqlens,
                                                int32_t num_branches, const int32_t *branch_parent,
                                                float scale, void *out, float *lse_out,
                                                cudaStream_t stream);

/*
 * View-state cache ("Serving 0.88M TPS from Two RTXs and Mac Minis", section
 * "Long Requests": the shards of a long request reuse the view's cached state
 * instead of recomputing the view, 3.4x faster than without the cache).
 *
 * A cache holds up to `capacity` view final states of `num_heads` heads
 * (fp32 [H][64][64] each, 16 KiB per head) in device memory of the device
 * current at creation, under 64-bit keys the caller chooses (a request id, a
 * hash of the view's tokens).  When full, a put evicts the least recently
 * used entries; a lookup or a branch call that names a key counts as a use.
 * The cache orders its own device memory across streams with CUDA events: a
 * branch call waits for the put of each state it reads, and a put into a
 * slot waits for every earlier branch call that read the state it replaces,
 * on whatever streams they were enqueued.  The caller still orders the
 * states a put copies from (normally by putting on the stream of the pass
 * that wrote them).  A cache object may be used from several host threads
 * (calls are serialised by a lock); it is not tied to a stream, but puts and
 * branch calls must be made with its device current (else
 * SPAN_LA_ERR_INVALID).  Puts and
 * branch calls on a stream that is being captured into a CUDA graph return
 * SPAN_LA_ERR_UNSUPPORTED (the ordering events are per-call host state).
 */
typedef struct span_la_view_cache span_la_view_cache;

/* Create a cache (cudaMalloc of capacity * num_heads * 16 KiB).  capacity >= 1,
 * num_heads >= 1.  *cache receives the handle. */
span_la_status span_la_cache_create(int32_t num_heads, int32_t capacity, span_la_view_cache **cache);

/* Free the cache (synchronises the device first).  NULL is allowed. */
span_la_status span_la_cache_destroy(span_la_view_cache *cache);

/*
 * Insert or refresh n states: state i (device, fp32 [H][64][64] at
 * states + i * H * 4096) goes under keys[i] (host array of n distinct keys),
 * copied device-to-device on `stream`.  A key already present is overwritten
 * in place; new keys take free slots, then the least recently used slots of
 * keys not in this call.  1 <= n <= capacity.  A typical put follows a
 * span_la_pass on the same stream, with states = view_state_out.
 */
span_la_status span_la_cache_put(span_la_view_cache *cache, const uint64_t *keys, int32_t n,
                                 const float *states, cudaStream_t stream);

/* present[i] = 1 if keys[i] is cached (the entry counts as used), else 0.
 * keys and present are host arrays of n entries. */
span_la_status span_la_cache_contains(span_la_view_cache *cache, const uint64_t *keys, int32_t n,
                                      int32_t *present);

/*
 * Branches forking from cached view states: as span_la_branches_from_state,
 * with branch b starting from the state cached under parent_keys[b] (host
 * array of num_branches keys).  Every key must be present, else
 * SPAN_LA_ERR_INVALID and nothing is enqueued.  The branches of one long
 * request can be run as several calls (shards) over the same cached state.
 */
span_la_status span_la_cache_branches(span_la_view_cache *cache, const uint64_t *parent_keys,
                                      const void *q, const void *k, const void *v,
                                      span_la_dims dims, const int32_t *branch_cu_seqlens,
                                      int32_t num_branches, void *out, cudaStream_t stream);

/* stats[0..5] = entries, capacity, hits, misses, evictions, puts (counts of
 * keys; a hit or a miss is one key looked up by contains or by a branch call). */
span_la_status span_la_cache_stats(const span_la_view_cache *cache, int64_t *stats);

#ifdef __cplusplus
}
#endif

#endif /* SPANLA_H */
