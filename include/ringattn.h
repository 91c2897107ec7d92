/*
 * ringattn.h -- C ABI of libringattn: single-GPU ring-chunked attention
 * forward (and its backward pass) for NVIDIA GB300 (sm_103a).
 *
 * The method is the compute side of the "Ring Attention" fused kernel of the
 * mKernel overview page (chatgpz.de, German translation of the MarkTechPost
 * article), table "Die fünf verschmolzenen Kerne", row Ring Attention: the key
 * and value sequence is cut into blocks that rotate around a ring; the local
 * FlashAttention step consumes the block received before, folding it into a
 * running (max, sum, accumulator) triple, while the next block is being moved.
 * Here the P blocks ("chunks") all live in this GPU's memory: "moving the next
 * block" is the TMA staging of the next key/value tiles into shared memory
 * while the tensor cores consume the current ones.  Nothing crosses a GPU
 * boundary.
 *
 * Conventions shared by every call:
 *   - Every pointer to tensor data is a DEVICE pointer into memory the caller
 *     owns; the library never allocates, frees or retains caller memory.  The
 *     only library-owned device state is one status word per device (see
 *     ra_get_last_device_status), 4096 work-item counters per device for the
 *     forward kernel (32 KiB), the static scratch of ra_bwd_static, and the
 *     kernels' code.
 *   - ra_fwd and ra_fwd_block hand out their work items at run time through a
 *     counter in device memory that the launch leaves at zero when it ends.
 *     Eager launches take the device's 64 eager counters in turn: up to 64
 *     eager launches may be in flight on one device at once (on any streams).
 *     A launch recorded into a CUDA graph (its stream is capturing) keeps a
 *     counter of its own for every replay, one that no other launch of this
 *     process is ever given, so replays can run beside any eager launches and
 *     beside other graphs; one captured launch must not run concurrently with
 *     itself (replays of one graph in one stream are fine).  A process can
 *     record at most 4032 launches per device; later captures get
 *     RA_ERR_UNSUPPORTED.  ra_shutdown does not restart either sequence.
 *   - Every call enqueues work on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and returns without waiting; results are valid once the
 *     stream has reached the work.
 *   - Arguments are validated on the host before anything is launched; on any
 *     error nothing is launched and the outputs are untouched.
 *   - bf16 means IEEE-754 binary16-brain (1 sign, 8 exponent, 7 mantissa bits).
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ra_status {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, H % Hkv != 0, S % P != 0,
                             non-finite scale, n < 1 */
  RA_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle: D not 64/128,
                             S/P not a multiple of 128, pointer not 16-byte aligned,
                             negative scale, device is not sm_103, sizes past 2^31 rows
                             (ra_fwd, ra_fwd_block: past 2^30 128-row query tiles in
                             B*H*S/128) */
  RA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, attribute query,
                             tensor-map encode); ra_last_cuda_error() gives the code */
  RA_ERR_TIMEOUT = 4,     /* a bounded wait inside a kernel gave up (reported by
                             ra_get_last_device_status) */
  RA_ERR_BOUNDS = 5       /* bounds-checked builds only (ra_debug_build() == 1): a kernel
                             computed a global address outside its buffer and skipped the
                             access (reported by ra_get_last_device_status) */
} ra_status;

/*
 * ra_fwd -- ring-chunked attention forward.
 *
 * Computes, for batch b, query head h, query row s (all rows, all heads):
 *     g      = h / (H / Hkv)                        (grouped-query attention)
 *     x_t    = scale * <q[b,s,h,:], k[b,t,g,:]>      for allowed keys t
 *              (allowed: all t when causal == 0; t <= s when causal != 0)
 *     out[b,s,h,:] = sum_t softmax_t(x) * v[b,t,g,:]          (bf16, RNE)
 *     lse[b,h,s]   = ln sum_t exp(x_t)                        (fp32)
 * The keys are cut into P equal contiguous chunks of C = S/P rows.  A query
 * row in chunk i folds chunk i first (its own), then i-1, i-2, ... (the block
 * its ring predecessor would send), wrapping around for non-causal attention;
 * causal chunks j > i hold no allowed key and are skipped.  Each chunk is
 * folded with the online-softmax update (FlashAttention), so the result is
 * exact softmax attention up to floating-point rounding.
 *
 *   q    [B, S, H,   D] bf16, contiguous (row-major, D fastest)
 *   k, v [B, S, Hkv, D] bf16, contiguous
 *   out  [B, S, H,   D] bf16, contiguous, written
 *   lse  [B, H, S]      fp32, contiguous, written; may be NULL (not written)
 *   B, H, Hkv, S, D, P > 0;  H % Hkv == 0;  S % P == 0
 *   supported: D in {64, 128};  (S / P) % 128 == 0;  scale >= 0 and finite
 *   (scale == 0 is legal and gives uniform weights over the allowed keys)
 *   q, k, v, out 16-byte aligned; lse 4-byte aligned.
 *   out must not overlap q, k or v.
 *   Range: finite inputs.  The fp32 accumulators hold weights of up to 2^30
 *   per key tile relative to a running reference, so
 *   2^30 * (S / 128) * max|v| must stay below 2^128 (|v| < 2^80 up to 16 M
 *   keys); larger values can overflow to inf.
 * Returns RA_OK once the kernel is enqueued.  A kernel that had to give up a
 * bounded internal wait leaves out/lse partly written and records
 * RA_ERR_TIMEOUT for ra_get_last_device_status.
 */
ra_status ra_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                 int Hkv, int S, int D, int P, int causal, float scale, void* stream);

/*
 * ra_fwd_block -- one ring step: attention of a query block against one
 * key/value block at given global sequence positions, as a normalised
 * partial result.  This is what a ring rank computes on the block it has
 * just received (same page, table "Die fünf verschmolzenen Kerne", row Ring
 * Attention); ra_merge_partials then folds the partials of all blocks into the
 * exact result.
 *
 *   q    [B, Sq, H,   D] bf16: global query rows q_pos0 .. q_pos0+Sq-1
 *   k, v [B, Sk, Hkv, D] bf16: global key rows   k_pos0 .. k_pos0+Sk-1
 *   out  [B, Sq, H,   D] bf16, written: softmax over this block's allowed keys
 *        (causal: key position <= query position) applied to v
 *   lse  [B, H, Sq]      fp32, written: ln sum over those keys of exp(x_t);
 *        may be NULL
 *   A row with no allowed key in the block gets out = 0 and lse = -inf (it
 *   contributes nothing to a merge).
 *   supported: D in {64, 128}; Sq, Sk, q_pos0, k_pos0 multiples of 128;
 *   scale >= 0; q_pos0, k_pos0 >= 0 (RA_ERR_INVALID_ARG otherwise).
 * Same pointer, alignment, stream and error rules as ra_fwd.
 */
ra_status ra_fwd_block(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                       int H, int Hkv, int Sq, int Sk, int D, long long q_pos0, long long k_pos0,
                       int causal, float scale, void* stream);

/*
 * ra_merge_partials -- combine n normalised partial attention results that
 * were computed over disjoint key sets (for instance one per ring chunk) into
 * the result over their union: the online-softmax fold of the same page's
 * Ring Attention row, written in log-sum-exp form.
 *
 *   o_parts   [n, B, S, H, D]  bf16 (o_is_fp32 == 0) or fp32 (o_is_fp32 != 0);
 *             partial k holds O_k = (sum over its keys of e^{x_t} v_t) /
 *             (sum over its keys of e^{x_t}), as ra_fwd writes it
 *   lse_parts [n, B, H, S]     fp32; lse_k = ln(sum over its keys of e^{x_t});
 *             -inf marks a partial with no key, which contributes nothing (its
 *             o_parts entries are not read); every other lse_k must be finite
 *             (+inf or NaN make that row's out and lse NaN)
 *   out       [B, S, H, D]     bf16, written: sum_k e^{lse_k - lse} O_k
 *   lse       [B, H, S]        fp32, written: ln sum_k e^{lse_k}; may be NULL
 *   When every lse_k of a row is -inf the row gets out = 0 and lse = -inf.
 *   n >= 1; B, H, S, D > 0; D % 8 == 0; o_parts and out 16-byte aligned.
 */
ra_status ra_merge_partials(const void* o_parts, int o_is_fp32, const float* lse_parts, int n,
                            void* out, float* lse, int B, int H, int S, int D, void* stream);

/*
 * ra_bwd_workspace_bytes -- bytes of device workspace ra_bwd needs: two fp32
 * values per query row (8 * B * H * S).  Returns 0 if a size is not positive.
 */
unsigned long long ra_bwd_workspace_bytes(int B, int H, int S);

/*
 * ra_bwd -- gradients of ra_fwd's output with respect to q, k and v, for a
 * given gradient dout of the output (the loss sum(out * dout)).  The pages
 * describe no backward pass; this is the derivative of the definition in
 * ra_fwd's comment, with p_st = softmax_t(x) of query row s:
 *     dp_st   = <dout[b,s,h,:], v[b,t,g,:]>
 *     delta_s = <dout[b,s,h,:], out[b,s,h,:]>   (= sum_t p_st dp_st)
 *     ds_st   = p_st (dp_st - delta_s)
 *     dq[b,s,h,:] = scale * sum_t ds_st k[b,t,g,:]
 *     dk[b,t,g,:] = scale * sum over rows s and query heads h of group g of ds_st q[b,s,h,:]
 *     dv[b,t,g,:] =         sum over rows s and query heads h of group g of p_st dout[b,s,h,:]
 * p_st is recomputed from q, k and lse; the key tiles of each query tile are
 * visited in ra_fwd's ring order for P (only the rounding order depends on P).
 *
 *   q, out, dout [B, S, H, D] bf16, contiguous; out and lse as ra_fwd wrote
 *                them for the same q, k, v, P, causal and scale
 *   k, v         [B, S, Hkv, D] bf16, contiguous
 *   lse          [B, H, S] fp32 (natural log), 4-byte aligned
 *   dq           [B, S, H, D] bf16, written
 *   dk, dv       [B, S, Hkv, D] bf16, written
 *   workspace    device memory of workspace_bytes >= ra_bwd_workspace_bytes(B, H, S)
 *                bytes, owned by the caller, 16-byte aligned; overwritten (no
 *                initial contents needed); a workspace must not be shared by
 *                two ra_bwd calls that can run at the same time
 *   Same shape, support and stream rules as ra_fwd; every bf16 pointer 16-byte
 *   aligned; dq, dk, dv must not overlap each other or any input.
 * Enqueues three kernels on `stream` (per-row sums, dk/dv, dq).  Every output
 * element is written exactly once, so the result does not depend on timing.
 * Errors as ra_fwd; RA_ERR_INVALID_ARG also for a null lse or workspace and for
 * a workspace smaller than ra_bwd_workspace_bytes(B, H, S).
 */
ra_status ra_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, void* workspace,
                 unsigned long long workspace_bytes, int B, int H, int Hkv, int S, int D, int P,
                 int causal, float scale, void* stream);

/*
 * ra_bwd_static -- ra_bwd without a caller workspace, for callers that must
 * not allocate device memory per call.  (No counterpart on the pages: an
 * allocation-free form of this library's ra_bwd.)
 *
 * The per-row scratch (-lse*log2(e) and -delta, 8 bytes per query row) lives
 * in one fixed device array inside the library: 16 MiB, enough for
 * B*H*S <= 2^21 = 2,097,152 query rows.  Its address is looked up once per
 * device, when the library first sets that device up.  The call allocates
 * nothing (no cudaMalloc/cudaFree, no allocating library routine) and the
 * scratch needs no clearing: the first kernel writes every value the other
 * two read.
 *
 * Every call on a device shares that one array: two ra_bwd_static calls that
 * can run at the same time (on different streams, or from different host
 * threads) race on it and can return wrong gradients.  Issue them on one
 * stream, or use ra_bwd with a workspace per stream.
 *
 * Arguments, layouts, results and errors as ra_bwd without the workspace,
 * plus RA_ERR_UNSUPPORTED when B*H*S exceeds 2^21.
 */
ra_status ra_bwd_static(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                        int H, int Hkv, int S, int D, int P, int causal, float scale,
                        void* stream);

/*
 * ra_get_last_device_status -- synchronise `stream`, then read and clear this
 * device's sticky status word.  Returns RA_ERR_TIMEOUT if any kernel launched
 * since the previous query gave up a bounded wait (its outputs are then not
 * valid), RA_ERR_UNSUPPORTED if a kernel refused to run because the runtime
 * gave it a shared-memory base that is not 1024-byte aligned (the dk/dv kernel
 * of ra_bwd needs nearly all of a CTA's shared memory and cannot round the base
 * up; its outputs are then not written), RA_ERR_BOUNDS (bounds-checked builds
 * only) if a kernel skipped an access outside a buffer, RA_ERR_CUDA if the
 * synchronisation itself failed, else RA_OK.  With several bits set, the first
 * of timeout, bounds, layout in that order is reported.
 */
ra_status ra_get_last_device_status(void* stream);

/*
 * ra_measure_ceilings -- measure, on the current device, the two non-tensor
 * rates the forward's online softmax depends on (no counterpart on the pages;
 * a diagnostic of this library).  Per allowed (query, key) pair the softmax
 * computes one exp2 on the MUFU unit and a few fp32 operations, so these
 * rates bound the pairs per second beside the tensor-core roofline.
 * Runs microbenchmark kernels (one 1024-thread CTA per SM, about a
 * millisecond in all) on a stream of its own and waits for them; allocates
 * nothing (its timing records live in a 20 KiB library-owned device array).
 *   out[8] host doubles, written:
 *     [0] ex2 results per SM per clock      [1] ex2 results per second (whole GPU)
 *     [2] scalar fp32 FMA lanes / SM / clk  [3] scalar fp32 FMA lanes per second
 *     [4] packed f32x2 FMA lanes / SM / clk [5] packed f32x2 FMA lanes per second
 *     [6] mean SM clock during the runs (MHz) [7] SMs measured
 * Returns RA_ERR_INVALID_ARG for a NULL out, RA_ERR_UNSUPPORTED off sm_103,
 * RA_ERR_CUDA if a launch or copy fails.
 */
ra_status ra_measure_ceilings(double* out);

/* Human-readable name of a status code (static string, never NULL). */
const char* ra_status_string(ra_status s);

/* The cudaError_t value behind the most recent RA_ERR_CUDA on this thread. */
int ra_last_cuda_error(void);

/* Library version, (major << 16) | (minor << 8) | patch: 0.3.0 (0.3: the forward hands
   out its work items at run time through per-device counters). */
int ra_version(void);

/*
 * Test hook for the failure path: when `timeout_ns` > 0, subsequent ra_fwd
 * and ra_bwd launches on this process use that wait limit instead of the default (2 s);
 * when `skip_value_load` != 0 the producer deliberately never issues the
 * first value-tile copy (ra_fwd) or the first output-gradient tile copy of
 * the dk/dv kernel (ra_bwd, ra_bwd_static), so the consumer's bounded wait must
 * run out and the launch must report RA_ERR_TIMEOUT.  Pass (0, 0) to restore
 * normal launches.
 */
void ra_debug_set_fault(long long timeout_ns, int skip_value_load);

/*
 * Bounds-checked builds (no counterpart on the pages; a test facility).  The
 * library compiled with RA_DEBUG (libringattn_debug.so, built by
 * `python -m ring_chunked_attention_gb300.build --debug`) checks every global
 * address its kernels compute (output, lse, gradient and workspace rows, the
 * merge's partials; the tensor-map copies are bounded by the hardware) against
 * the buffer's size as the call's arguments give it.  An address outside it
 * sets a status bit and the access is skipped, with no trap: the next
 * ra_get_last_device_status returns RA_ERR_BOUNDS.  Other builds compile the
 * checks away.
 *   ra_debug_build: bit 0 set in a bounds-checked build, bit 1 in a traced
 *     build (below), 0 in the product build.
 *   ra_debug_set_bounds_trim: a test hook for bounds-checked builds; the last
 *     `elements` elements of every checked buffer count as outside it, so a
 *     test can see the checks fire without any access outside a buffer.  0
 *     (the default; negative values too) turns it off.  No effect in other
 *     builds.  Applies to launches made after the call.
 */
int ra_debug_build(void);
void ra_debug_set_bounds_trim(long long elements);

/*
 * Traced builds (a measurement facility, no counterpart on the pages).  The
 * library compiled with RA_TRACE (libringattn_trace.so, built by
 * `python -m ring_chunked_attention_gb300.build --trace`; the binding loads it
 * when the environment variable RA_TRACE is 1) counts clock cycles per role
 * in every CTA of the forward kernel: where its MMA warp, softmax warps and
 * producer thread wait or work.  Each CTA stores 32 counters when its roles
 * end (a launch first zeroes them all, so slots of CTAs it did not run read
 * 0); ra_trace_read synchronises the device and copies the counters of the
 * last forward launch's first n_ctas CTAs (at most 1024) into out
 * (n_ctas * 32 values, host memory).  The slot layout is given with
 * `python -m ring_chunked_attention_gb300.trace`, which runs a workload and
 * prints the per-step breakdown.  Returns RA_ERR_UNSUPPORTED in other builds,
 * RA_ERR_INVALID_ARG for a NULL out or n_ctas <= 0, RA_ERR_CUDA if the copy
 * fails.
 */
ra_status ra_trace_read(unsigned long long* out, int n_ctas);

/*
 * MMA issue order of ra_fwd and ra_fwd_block (no counterpart on the pages; an
 * implementation choice of this library).  The probabilities P_i of a query
 * tile are kept in tensor memory over the columns of the score tile S_i that
 * produced them, so the next S_i = Q_i K^T must not start before
 * O_i += P_i V has read them.  The PTX ISA orders two tcgen05.mma of one
 * thread directly only when they share the accumulator.  It also lists
 * tcgen05.mma -> tcgen05.shift and tcgen05.shift -> tcgen05.mma (same
 * cta_group) among the pairs that execute in issue order, and it orders
 * completion as seen through tcgen05.commit and an mbarrier wait.
 *   order 3 (default): per key/value step and query tile in turn, PV, a
 *     tcgen05.shift of 8 columns of S_i that hold consumed scores, the next
 *     S.  PV -> shift -> S execute in issue order, with no wait.
 *   order 0: the same with a wait for the PV's commit instead of the shift.
 *     Ordered by completion; the tensor pipe drains once per tile.
 *   order 1: per key/value step, both query tiles' PV products, then each
 *     tile's next S once the commit of its PV has arrived (no drain, but the
 *     two tiles' softmax work runs at the same time and competes; slower).
 *   order 2: per tile in turn, PV and the next S back to back with nothing
 *     between, relying on the tensor pipe executing MMAs with different
 *     accumulators in issue order, which no document states.  For measurement
 *     and tests only.
 * All four compute the same arithmetic; the test-suite checks that their
 * outputs are bit-identical.  Other values select order 3.  Launches with one
 * query tile per item (see ra_set_item_pairing) keep S and P in separate,
 * double-buffered columns, issue each S two steps ahead of its PV, and are
 * not affected by the order.  Applies to launches made after the call.
 */
void ra_set_mma_order(int order);

/*
 * How ra_fwd and ra_fwd_block group query tiles into work items (no
 * counterpart on the pages; an implementation choice of this library).  A
 * paired item is two 128-row query tiles that share one key/value stream (two
 * heads of a GQA group, or two consecutive tiles of one head); a single item
 * is one tile.  policy 0 (default): pair, unless that leaves fewer items than
 * the device has SMs, when single items shorten the heaviest item; 1: pair
 * whenever the shape allows; 2: never pair.  The grouping changes which SM
 * computes a tile, not its arithmetic: results are the same bits under every
 * policy.  The policy exists so that tests can reach every grouping at small
 * sizes.
 * Applies to launches made after the call.
 */
void ra_set_item_pairing(int policy);

/* Drop cached tensor maps and device queries and reset the debug and policy
 * settings.  The library's device arrays (status word, work-item counters,
 * the static scratch of ra_bwd_static) are file-scope device variables: they
 * stay allocated while the library is loaded, and ra_shutdown leaves them and
 * the counter sequences as they are, so launches still in flight are not
 * disturbed.  Each kernel's launch attributes are set once per device and
 * then reused, which also lets ra_fwd, ra_fwd_block and ra_bwd be recorded
 * into CUDA graphs; after a device reset (cudaDeviceReset), call ra_shutdown
 * so that they are set again. */
void ra_shutdown(void);

#ifdef __cplusplus
}
#endif
#endif /* RINGATTN_H */
