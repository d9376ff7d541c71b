/*
 * gdn.h -- C ABI of the GB300 GatedDeltaNet record / replay library (libgdn.so).
 *
 * The library runs the gated delta-rule recurrence step with innovation-tape
 * capture ("record"), the speculative-decode rollback that re-folds an
 * accepted tape prefix onto a state snapshot ("replay"), and the tiled GQA
 * head broadcast ("repeat"), as hand-written sm_103a CUDA kernels.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a pointer to caller-owned, densely packed,
 *   row-major DEVICE memory (any pointer the CUDA runtime can dereference
 *   from a kernel).  The library never allocates, frees, copies to the host
 *   or synchronises: it validates its arguments on the host, enqueues one
 *   kernel on `stream` (gdn_chunk_prefill: two) and returns.  Results are
 *   ready when the stream has reached that point.
 * - `stream` is a cudaStream_t (the typedef below is the same type);
 *   NULL means the legacy default stream.
 * - Kernels are enqueued as programmatic dependent launches: a kernel may
 *   be scheduled while the kernel before it on the stream is still running,
 *   but it reads and writes no global memory until that kernel has
 *   completed and its writes are visible, so the stream order of every
 *   memory access is that of ordinary launches (a kernel of the caller's
 *   between two calls is waited for as usual).
 * - Dimensions are int64_t and must be > 0 (a zero or negative dimension is
 *   GDN_ERR_INVALID_ARGUMENT, the rule the tiled-repeat page applies to its
 *   own shapes).
 * - Validation happens before any launch.  A non-GDN_OK status means nothing
 *   was enqueued, except GDN_ERR_CUDA, which reports a failed launch.
 *   gdn_last_error() returns a message for the last failure on the calling
 *   host thread.
 * - Floating-point tensors share one element type `dtype` (f32, bf16 or
 *   f16); the recurrent state is float32 (or `dtype` in the _tstate calls).
 *   The state and every step's scalars are float32 (see gdn_step_record for
 *   the bf16 tensor-core paths' split operands); values written in bf16/f16
 *   are rounded to nearest-even.
 *
 * Notation: B batch, T timesteps, Hk key heads, Hv value heads (Hv % Hk == 0,
 * G = Hv / Hk, key head of value head hv is hk = hv / G), Dk key dim, Dv
 * value dim.  The source page for record and replay is "metaltile-std 0.1.0
 * -- src/ffai/gated_delta_replay.rs" (module doc, kernels
 * gated_delta_step_record and state_replay); the source page for the repeat
 * is "mlx-native 0.6.5 -- ops/repeat_tiled.rs" (module doc "Mapping",
 * dispatch_repeat_tiled_f32).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 7

/* Same type as cudaStream_t. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARGUMENT = 1, /* bad shape, null pointer, overflow, overlap  */
    GDN_ERR_UNSUPPORTED = 2,      /* dtype or Dk outside the compiled set        */
    GDN_ERR_MISALIGNED = 3,       /* a pointer breaks its alignment requirement  */
    GDN_ERR_CUDA = 4              /* the CUDA runtime rejected the launch        */
} gdn_status;

typedef enum gdn_dtype {
    GDN_DTYPE_F32 = 0,
    GDN_DTYPE_BF16 = 1,
    GDN_DTYPE_F16 = 2
} gdn_dtype;

/* Which key head a value head reads (G = Hv / Hk). */
typedef enum gdn_gqa_mapping {
    GDN_GQA_BLOCK = 0, /* hk = hv / G: the record kernel's own rule             */
    GDN_GQA_TILED = 1  /* hk = hv % Hk: the head order of the tiled repeat
                          ("mlx-native repeat_tiled.rs", module doc "Mapping"),
                          read in place instead of materialised             */
} gdn_gqa_mapping;

/*
 * gdn_step_record -- T recurrence steps with delta-tape capture
 * (page: gated_delta_step_record; tape layout: module doc).
 *
 * For every state row s = state[b,hv,dv,:] (float32, Dk entries) and every
 * step t in 0..T-1 whose mask is on:
 *     s        <- g[b,t,hv] * s
 *     kv        = s . k[b,t,hk,:]
 *     delta     = (v[b,t,hv,dv] - kv) * beta[b,t,hv]
 *     delta_log[b,t,hv,dv] = delta
 *     s        <- s + k[b,t,hk,:] * delta
 *     y[b,t,hv,dv] = s . q[b,t,hk,:]
 * and state_out[b,hv,dv,:] = s after the last step.
 *
 * Arguments (shape, element type, alignment):
 *   q, k       [B,T,Hk,Dk]  dtype, 16-byte aligned
 *   v          [B,T,Hv,Dv]  dtype
 *   g, beta    [B,T,Hv]     dtype (g is a multiplicative decay, not a log)
 *   state_in   [B,Hv,Dv,Dk] float32, 16-byte aligned (the snapshot)
 *   mask       [B,T] uint32 or NULL.  NULL: every step is on.  A step with
 *              mask 0 is skipped: the state is unchanged and y, delta_log,
 *              k_log, g_log at (b,t) are NOT written (they keep whatever the
 *              caller put there).  Any nonzero value means on.
 *   y          [B,T,Hv,Dv]  dtype (output)
 *   state_out  [B,Hv,Dv,Dk] float32, 16-byte aligned (output).  May be the
 *              same pointer as state_in (in place); any other overlap with
 *              state_in is GDN_ERR_INVALID_ARGUMENT.
 *   delta_log  [B,T,Hv,Dv]  dtype (output, the innovation tape)
 *   k_log      [B,T,Hv,Dk]  dtype or NULL, 16-byte aligned (output): k
 *              expanded to value heads, k_log[b,t,hv,:] = k[b,t,hv/G,:],
 *              written where delta_log is
 *   g_log      [B,T,Hv]     dtype or NULL (output): copy of g, written where
 *              delta_log is
 *   Dk         32, 64, 128, 192 or 256 (else GDN_ERR_UNSUPPORTED); Dv any > 0
 * Outputs must not overlap inputs (other than the in-place state).
 *
 * Kernels and precision.  The call picks one of three kernels; all keep the
 * state in float32 and take every step's scalars (the decay products, the
 * reciprocals, the innovation) in float32:
 *   - FP32 steps (f32 / f16 inputs; bf16 calls the two below do not take):
 *     every product in float32, one rounding per state entry per step.
 *   - bf16, 7 <= T <= 16, Dk = 128, Dv a multiple of 128, v 16-byte aligned,
 *     state in float32: the tcgen05 kernel (one 16-step chunk per call,
 *     TMA-fed, accumulators in tensor memory).
 *   - other bf16 calls with T >= 12 and Dk of 64 or 128: mma.sync 16-step
 *     chunks.
 * The two tensor-core forms regroup a chunk's steps into products in which
 * the f32 state and the f32 per-row solve values enter as two bf16 terms
 * (hi + lo, 16 significant bits) against the exact bf16 k and q rows, with
 * f32 accumulation: each such product carries a relative error of about
 * 2^-17, well inside the 1e-3 that bf16 inputs are held to, but the results
 * are not bit-identical to the FP32-step kernel (and a bf16 tape is rounded
 * in either case).  The tcgen05 kernel solves each row's chunk in FP32.
 * Every kernel is deterministic run to run.
 */
gdn_status gdn_step_record(const void *q, const void *k, const void *v,
                           const void *g, const void *beta,
                           const float *state_in, const uint32_t *mask,
                           void *y, float *state_out, void *delta_log,
                           void *k_log, void *g_log,
                           int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                           int64_t Dk, int64_t Dv, gdn_dtype dtype,
                           gdn_stream_t stream);

/*
 * gdn_step_record_mapped -- gdn_step_record with a choice of GQA mapping.
 *
 * Identical to gdn_step_record (same arguments, layouts, errors) except that
 * the key head of value head hv is chosen by `mapping`:
 *   GDN_GQA_BLOCK  hk = hv / (Hv/Hk)  (gdn_step_record itself)
 *   GDN_GQA_TILED  hk = hv % Hk       (the result equals gqa_repeat_tiled of
 *                  q and k to Hv heads followed by gdn_step_record with
 *                  Hk = Hv, without the expanded copies)
 * k_log, when given, receives k[b,t,hk,:] under the same mapping.  An
 * unknown mapping value is GDN_ERR_INVALID_ARGUMENT.
 */
gdn_status gdn_step_record_mapped(const void *q, const void *k, const void *v,
                                  const void *g, const void *beta,
                                  const float *state_in, const uint32_t *mask,
                                  void *y, float *state_out, void *delta_log,
                                  void *k_log, void *g_log,
                                  int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                                  int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                                  gdn_dtype dtype, gdn_stream_t stream);

/*
 * gdn_step_record_tstate / gdn_state_replay_tstate -- record and replay with
 * the state stored in the input element type ("state in T", as the page's
 * kernels keep it) instead of float32.
 *
 * state_in / state_out are [B,Hv,Dv,Dk] in `dtype` (16-byte aligned).  The
 * state is widened exactly on load, every step runs in float32 as in
 * gdn_step_record, and the final state is rounded to nearest-even once on
 * store.  With dtype = GDN_DTYPE_F32 these are gdn_step_record_mapped and
 * gdn_state_replay (or _per_seq) exactly.  Everything else -- arguments,
 * layouts, mask rule, tape, errors -- is as documented for those calls;
 * gdn_state_replay_tstate takes the per-sequence counts of
 * gdn_state_replay_per_seq when accepted_per_seq is non-NULL (then
 * `accepted` is only checked to be >= 0), else the single count `accepted`.
 */
gdn_status gdn_step_record_tstate(const void *q, const void *k, const void *v,
                                  const void *g, const void *beta,
                                  const void *state_in, const uint32_t *mask,
                                  void *y, void *state_out, void *delta_log,
                                  void *k_log, void *g_log,
                                  int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                                  int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                                  gdn_dtype dtype, gdn_stream_t stream);

gdn_status gdn_state_replay_tstate(const void *delta_log, const void *k_log,
                                   const void *g_log, const void *state_in,
                                   const uint32_t *mask, void *state_out,
                                   int64_t B, int64_t T, int64_t Hv, int64_t Dk,
                                   int64_t Dv, int64_t accepted,
                                   const int32_t *accepted_per_seq,
                                   gdn_dtype dtype, gdn_stream_t stream);

/*
 * gdn_chunk_prefill -- the record recurrence for long calls, computed in
 * chunks of 16 steps on the tensor cores.
 *
 * Same mathematics, arguments, layouts, mask rule and errors as
 * gdn_step_record_mapped, with these differences:
 *   - delta_log, k_log and g_log are optional (NULL: not written); y and
 *     state_out are required.
 *   - The chunk form re-associates the sums of the step form (the pages give
 *     only the step form; the chunk form follows from it algebraically), so
 *     results agree with the step form to float32 rounding, not bit for bit:
 *     replaying its tape reproduces state_out to rounding, where a float32
 *     tape of gdn_step_record replays exactly.
 *   - It needs a caller-owned DEVICE workspace of at least
 *     gdn_chunk_prefill_workspace_size(B, T, Hv) bytes, 16-byte aligned
 *     (too small or NULL: GDN_ERR_INVALID_ARGUMENT).  Its contents on entry
 *     and exit are irrelevant to the caller; two calls in flight at once
 *     need two workspaces.
 * It enqueues two kernels on `stream` (the chunk-local matrices, then the
 * sequential scan over chunks).
 */
size_t gdn_chunk_prefill_workspace_size(int64_t B, int64_t T, int64_t Hv);

gdn_status gdn_chunk_prefill(const void *q, const void *k, const void *v,
                             const void *g, const void *beta,
                             const float *state_in, const uint32_t *mask,
                             void *y, float *state_out, void *delta_log,
                             void *k_log, void *g_log,
                             int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                             int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                             void *workspace, size_t workspace_bytes,
                             gdn_dtype dtype, gdn_stream_t stream);

/*
 * gdn_chunk_prefill_noalloc -- gdn_chunk_prefill without a caller workspace.
 *
 * The source pages have no counterpart to this entry point.  It is for
 * callers that cannot allocate device memory when they call: an inference
 * runtime that hands its whole HBM budget to its own pool allocator at start
 * and forbids allocations afterwards, a plugin or script host that receives
 * tensors but has no handle on the allocator that made them, or a serving
 * loop with a latency budget in which cudaMalloc (which may synchronise the
 * device) is not allowed.
 *
 * The workspace is a file-scope device array of 32 MiB inside the library (a
 * static __device__ object): every GPU on which the library's device code is
 * loaded holds those 32 MiB until the process exits, and no call allocates,
 * frees or synchronises anything.  Each call looks up the array's device
 * address for the current device (cudaGetSymbolAddress); the first call on a
 * device may also load the library's device code there, so make that first
 * call before any stream capture begins.  Problems whose workspace
 * (gdn_chunk_prefill_workspace_size) exceeds 32 MiB return
 * GDN_ERR_UNSUPPORTED before anything is launched.
 *
 * All calls on one device share the array, and each call leaves its contents
 * behind; a call writes every workspace entry it reads before reading it, so
 * nothing needs clearing between calls.  Calls whose kernels overlap in time
 * on one device race on the array and give wrong results: issue them on one
 * stream (or use gdn_chunk_prefill with a workspace per stream).  Results are
 * identical, bit for bit, to gdn_chunk_prefill with the same arguments; every
 * other argument, rule and error is as documented there.
 */
gdn_status gdn_chunk_prefill_noalloc(const void *q, const void *k, const void *v,
                                     const void *g, const void *beta,
                                     const float *state_in, const uint32_t *mask,
                                     void *y, float *state_out, void *delta_log,
                                     void *k_log, void *g_log,
                                     int64_t B, int64_t T, int64_t Hk, int64_t Hv,
                                     int64_t Dk, int64_t Dv, gdn_gqa_mapping mapping,
                                     gdn_dtype dtype, gdn_stream_t stream);

/*
 * gdn_state_replay -- rebuild the state after an accepted prefix of the tape
 * (page: state_replay; module doc: "re-folds the accepted prefix").
 *
 * For every state row and t in 0..T-1:
 *     do_step = (t < accepted) && (mask == NULL || mask[b,t] != 0)
 *     s <- do_step ? s * g_log[b,t,hv] + k_log[b,t,hv,:] * delta_log[b,t,hv,dv] : s
 * The select is a true select: tape slots of skipped steps are never read,
 * so they may hold anything (NaN, stale data).
 *
 *   delta_log  [B,T,Hv,Dv]  dtype
 *   k_log      [B,T,Hv,Dk]  dtype, 16-byte aligned (key rows expanded to value heads)
 *   g_log      [B,T,Hv]     dtype
 *   state_in   [B,Hv,Dv,Dk] float32, 16-byte aligned (the pre-record snapshot)
 *   mask       [B,T] uint32 or NULL (the mask record was given)
 *   state_out  [B,Hv,Dv,Dk] float32, 16-byte aligned; may equal state_in
 *   accepted   >= 0; values above T act as T; 0 copies state_in to state_out
 *
 * With a float32 tape written by gdn_step_record from the same snapshot and
 * mask, replay with accepted >= T reproduces record's state_out bit for bit,
 * and replay with accepted = a reproduces a record over the first a steps.
 *
 * Kernels: calls folding 2 to 16 steps with Dk = 128, a float32 state and
 * 16-byte aligned delta_log rows (base aligned, Dv * element size a multiple
 * of 16) run on a persistent kernel that streams 64-row state blocks and the
 * tape rows by TMA (one CTA per SM); the others on the FP32 kernel (one CTA
 * per 64-row block).  Both apply the same f32 operations in the same order,
 * so their results are bit-identical.  The persistent kernel's waits are
 * bounded as described at gdn_wait_status.  Past a fixed first share per
 * CTA, the persistent kernel hands its blocks out from a counter in library
 * memory, one of 256 slots taken round robin per launch and reset by the
 * launch itself; two launches that run at the same time must not share a
 * slot, so at most 255 other launches of this kernel may be in flight
 * alongside one (on any streams), and one captured graph that contains it
 * must not be instantiated twice and run concurrently.
 */
gdn_status gdn_state_replay(const void *delta_log, const void *k_log,
                            const void *g_log, const float *state_in,
                            const uint32_t *mask, float *state_out,
                            int64_t B, int64_t T, int64_t Hv, int64_t Dk,
                            int64_t Dv, int64_t accepted, gdn_dtype dtype,
                            gdn_stream_t stream);

/*
 * gdn_state_replay_per_seq -- gdn_state_replay with one accepted count per
 * sequence (speculative decoding accepts a different draft prefix in every
 * sequence of the batch; the page's kernel takes one count per dispatch).
 *
 *   accepted   [B] int32, DEVICE memory, 4-byte aligned, non-NULL.  Sequence
 *              b folds the steps t < accepted[b] whose mask is on; an entry
 *              < 0 acts as 0 (the sequence's state_out is its snapshot) and
 *              an entry > T acts as T.  Read by the kernel, so it may be
 *              produced by earlier work on the same stream.
 * Every other argument, layout and error is as for gdn_state_replay.  With
 * the same tape, sequence b's result equals gdn_state_replay with
 * accepted = accepted[b] (bit for bit).
 */
gdn_status gdn_state_replay_per_seq(const void *delta_log, const void *k_log,
                                    const void *g_log, const float *state_in,
                                    const uint32_t *mask, float *state_out,
                                    int64_t B, int64_t T, int64_t Hv, int64_t Dk,
                                    int64_t Dv, const int32_t *accepted,
                                    gdn_dtype dtype, gdn_stream_t stream);

/*
 * gdn_chunk_replay -- gdn_state_replay for long accepted prefixes, as one
 * tensor-core contraction.
 *
 * The replay fold is linear in the state and its updates do not read the
 * state, so it closes to
 *     s_out = Gam s_in + sum_t w_t delta_t k_t
 * over the folded steps t (t < accepted, mask on), with w_t the product of
 * g_log over the folded steps after t and Gam the product over all of them.
 * The library forms w and Gam, then runs the sum for every (b, hv) tile as a
 * (Dv x T) by (T x Dk) product on the tensor cores (tcgen05, tf32 operands
 * split into high and low parts, float32 accumulation).  Results agree with
 * gdn_state_replay to float32 rounding, not bit for bit; results are
 * run-to-run deterministic.
 *
 * Arguments, layouts and errors are those of gdn_state_replay, plus:
 *   accepted_per_seq  [B] int32 (device) or NULL: when given, sequence b folds
 *                     the steps t < accepted_per_seq[b] (entries < 0 act as 0,
 *                     > T as T) and `accepted` is only checked to be >= 0
 *   workspace         caller-owned device memory of at least
 *                     gdn_chunk_replay_workspace_size(B, T, Hv, Dk, Dv) bytes,
 *                     16-byte aligned; one workspace per call in flight
 * Only state_in, state_out and workspace need 16-byte alignment here.  It
 * enqueues two or three kernels on `stream` (the decay weights, the
 * contraction, and a fixed-order sum of partial results when the steps are
 * split over several CTAs per tile).
 */
size_t gdn_chunk_replay_workspace_size(int64_t B, int64_t T, int64_t Hv, int64_t Dk,
                                       int64_t Dv);

gdn_status gdn_chunk_replay(const void *delta_log, const void *k_log,
                            const void *g_log, const float *state_in,
                            const uint32_t *mask, float *state_out,
                            int64_t B, int64_t T, int64_t Hv, int64_t Dk,
                            int64_t Dv, int64_t accepted,
                            const int32_t *accepted_per_seq, void *workspace,
                            size_t workspace_bytes, gdn_dtype dtype,
                            gdn_stream_t stream);

/*
 * gqa_repeat_tiled -- tiled GQA broadcast (page: repeat_tiled.rs, "Mapping"):
 *     dst[t, hh, x] = src[t, hh % hg, x],  src [seq,hg,k] -> dst [seq,h,k]
 * A bit-exact copy.  Errors follow dispatch_repeat_tiled_f32: any dimension
 * <= 0, h % hg != 0, an element count or byte size that overflows, or
 * src_bytes / dst_bytes smaller than the shapes need ->
 * GDN_ERR_INVALID_ARGUMENT.  Any dtype of the enum is accepted; pointers
 * need only the element alignment (16-byte alignment with k * elemsize a
 * multiple of 16 takes the vector path).  src and dst must not overlap.
 */
gdn_status gqa_repeat_tiled(const void *src, void *dst,
                            int64_t seq, int64_t hg, int64_t h, int64_t k,
                            gdn_dtype dtype, size_t src_bytes, size_t dst_bytes,
                            gdn_stream_t stream);

/* Static name of a status code ("GDN_OK", ...); never NULL. */
const char *gdn_status_string(gdn_status status);

/* Message for the last non-OK status returned on the calling host thread
 * ("" if none).  Valid until the next call from the same thread. */
const char *gdn_last_error(void);

/* GDN_ABI_VERSION of the loaded library. */
int gdn_abi_version(void);

/*
 * gdn_wait_status -- whether a bounded wait of a pipelined (TMA / tcgen05) kernel ran out.
 *
 * The pipelined paths (the tcgen05 record kernel behind gdn_step_record and
 * gdn_step_record_mapped, the persistent replay behind gdn_state_replay and
 * gdn_state_replay_per_seq, and gdn_chunk_replay) run stages that wait on
 * each other through mbarriers.  Every such wait gives up after a
 * bound (about a second of GPU clock by default) instead of hanging; the
 * kernel then writes NaN to the state rows it could not finish, lets its
 * copies and products in flight land, and raises a device-side flag.  The
 * call that launched it still returned GDN_OK (it only enqueues work), so a
 * caller that wants to know reads the flag here: *expired is set to 1 if any
 * kernel raised it since the last call, else 0, and the flag is cleared.
 * The read is a synchronous device-to-host copy: call it after synchronising
 * the streams that ran the calls.  The pages have no counterpart.
 */
gdn_status gdn_wait_status(int *expired);

/*
 * Testing hooks (the pages have no counterpart).
 *
 * gdn_set_wait_bound -- the bound, in GPU clock cycles, on the pipeline
 * waits of the pipelined kernels launched after this call (0 restores the
 * default of 2e9 cycles).  A bound far below a kernel's normal waiting time
 * makes its waits run out, which exercises the expiry path above without any
 * fault: the drain after a failed wait always uses the default bound.
 * Process-wide; not meant for production calls.
 *
 * gdn_inject_wait_expiry -- while on (nonzero), every pipelined kernel
 * launched takes, before its pipeline starts, one wait on a barrier that
 * nothing completes, so that its bound runs out deterministically (pair it
 * with a short gdn_set_wait_bound: with the default bound each such kernel
 * waits about a second).  0 turns it off.
 *
 * gdn_force_launch_failures -- the next n calls that pass their argument
 * checks return GDN_ERR_CUDA (with a gdn_last_error message) before touching
 * the device, so a caller's handling of launch failures can be tested.
 * Process-wide; 0 cancels.
 */
gdn_status gdn_set_wait_bound(int64_t cycles);
gdn_status gdn_inject_wait_expiry(int on);
gdn_status gdn_force_launch_failures(int n);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
