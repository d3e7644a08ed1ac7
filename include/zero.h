/*
 * zero.h -- C ABI of the GB300 (sm_103a) ZeRO-DP partitioned mixed-precision
 * optimizer step.
 *
 * What the library computes (page titles and sections):
 *  - "01 - ZeRO memory math and Stage 1/2" (DeepSpeed ZeRO stages 1-2
 *    walkthrough), 4 (1)-(4): flatten a parameter group, pad it to a
 *    multiple of 2*world_size, split it into world_size contiguous shards
 *    (base = total // dp, remainder to the first ranks), and map tensors to
 *    shards;  6: the step -- overflow check (skip on inf/NaN), global gradient
 *    norm from per-shard partial sums, unscale and clip, Adam on the fp32
 *    shard, copy of the result to 16 bits in the rank's slot of the flat
 *    buffer, all-gather.
 *  - "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models"
 *    reading notes (papers.chlience.com), 3 (Adam is per coordinate, so the
 *    update of a shard needs only that shard's state), 4 (the averaged
 *    gradient shard g_bar^(k) = (1/N_d) sum_r g_r^(k), the reduce-scatter),
 *    7 and 9 (ZeRO-3: gather a layer's parameter shards before its forward
 *    and again before its backward; reduce its gradients onto the owner).
 *  - the ZeRO paper (Chinese translation, aiingo), 5.1-5.3 and Figure 1, and
 *    the CMU 11-868 lecture notes, slide 64: memory of model states per stage.
 *
 * One GPU holds every simulated rank: the N_d ranks' gradients are N_d
 * buffers in local HBM, the reduce-scatter is N_d coalesced reads fused into
 * the update, the scalar all-reduce of the norm is a fixed-order combine of
 * per-block partial sums on the device, and the all-gather destination is the
 * one flat 16-bit parameter buffer every simulated rank shares.
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA device (or managed) addresses on the current
 *    device; host pointers are plain CPU memory.  The caller owns every
 *    buffer; the library allocates no memory (zero_shard_step_noalloc's
 *    scratch is an array compiled into it; zero_shard_step_host creates two
 *    streams and a few events per device on its first call there) and carries
 *    no data from one call to the next (chained steps carry theirs in the
 *    caller's zero_chain).
 *  - Device work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and is asynchronous: results land in caller memory when
 *    the stream reaches them.  No entry point synchronises.
 *  - A negative return is an argument or launch error, reported before any
 *    work is enqueued when it is an argument error; zero_last_error() gives a
 *    message (per thread).  Conditions found on the device (overflow) are
 *    reported in zero_result, never by a trap.
 *  - 16-bit element offsets and counts are in elements, int64.
 *
 * Earlier descriptions of this interface used other names for some calls and
 * codes; each stands for the entry point given here:
 *  - zero_shard_stats (the reduce phase alone)   -> zero_shard_reduce
 *  - a `divisor` argument of the step            -> none: the averaging divisor
 *    is n_slices (N_d); the ZeRO-3 shard update, whose gradient is already
 *    averaged (divisor 1), is zero_shard_apply on the reduced shard
 *  - zero_workspace_bytes(n_shards, max_numel)  -> zero_workspace_bytes(void):
 *    the workspace has one fixed size, whatever the shards
 *  - ZERO_ENOMEM_WS                              -> ZERO_EWORKSPACE
 *  - an out-parameter "overflow flag + norm"     -> zero_result (overflow,
 *    applied, sumsq, grad_norm, clip_coef, grad_mult)
 *  - grad_slices / n_slices inside each shard    -> one grad_slices array per
 *    call (every shard of a step reads the same N_d slices) and a
 *    grad_offset per shard
 *  - zero3_reduce_bucket's separate device sumsq and overflow accumulators
 *                                                -> one zero_stats, an
 *    `accumulate` flag (0 starts it afresh) and the workspace for the
 *    per-block partial sums
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_MAX_SLICES 64   /* most gradient slices (ranks) one call reduces */
#define ZERO_MAX_SHARDS 64   /* most shards one call updates */

typedef enum {
    ZERO_OK = 0,
    ZERO_EINVAL = -1,      /* bad argument (null pointer, negative size, unknown dtype or mode) */
    ZERO_EALIGN = -2,      /* a pointer is not aligned to its element size */
    ZERO_EWORKSPACE = -3,  /* workspace missing or smaller than zero_workspace_bytes() */
    ZERO_ECUDA = -4,       /* a CUDA runtime call or launch failed */
    ZERO_ELIMIT = -5       /* more than ZERO_MAX_SLICES slices or ZERO_MAX_SHARDS shards; a call beyond
                              zero_shard_step_noalloc's scratch; (zero_result.status) a chained step outside
                              its scalar table */
} zero_status;

typedef enum { ZERO_F16 = 1, ZERO_BF16 = 2 } zero_dtype;

typedef enum {
    ZERO_PLAN_PADDED = 0,   /* pad to a multiple of 2*world_size, then split (the walkthrough's rule) */
    ZERO_PLAN_UNPADDED = 1  /* split the unpadded length; the remainder goes to the first ranks */
} zero_plan_mode;

/* ------------------------------------------------------------------------
 * Partition plan.  Host only.
 * Source: DeepSpeed ZeRO stages 1-2 walkthrough, 4 (1) flatten and align,
 * 4 (2) get_data_parallel_partitions (base = total // dp, remaining =
 * total % dp, remainder to the first ranks), 7 (start alignment).
 *
 * numels[n_tensors]          host, the group's tensors in declaration order
 * tensor_offsets[n_tensors]  host out, flat offset of each tensor
 * rank_offsets[world_size]   host out, first flat element of each rank's shard
 * rank_numels[world_size]    host out, shard sizes (sum = *padded_total)
 * padded_total, padding      host out, flat length after padding, and padding
 * Returns ZERO_OK or ZERO_EINVAL (n_tensors < 0, world_size < 1, negative
 * numel, unknown mode, null output).  Padding elements sit at the tail of the
 * last rank's shard; they are part of its shard.
 * ------------------------------------------------------------------------ */
int zero_plan(const int64_t* numels, int n_tensors, int world_size, int mode,
              int64_t* tensor_offsets, int64_t* rank_offsets, int64_t* rank_numels,
              int64_t* padded_total, int64_t* padding);

/* The tensors that overlap one rank's shard (params_in_partition and the
 * first offset of the walkthrough's 4 (4)): row k of out[4*k .. 4*k+3] is
 * (tensor index, first element inside the tensor, first element inside the
 * shard, length).  out must hold 4*n_tensors values.  Host only.  Returns the
 * number of rows (>= 0) or ZERO_EINVAL. */
int zero_plan_intersections(const int64_t* tensor_offsets, const int64_t* numels, int n_tensors,
                            int64_t rank_offset, int64_t rank_numel, int64_t* out);

/* ------------------------------------------------------------------------
 * Memory model of model states per device, in bytes.  Host only.
 * Source: ZeRO paper (Chinese translation), 5.1-5.3 and Figure 1; reading
 * notes 5.1-5.4; CMU 11-868 notes, slide 64.  K is the optimizer-state bytes
 * per parameter (12 for mixed-precision Adam):
 *   stage 0 (DP)        (4 + K) psi
 *   stage 1 (P_os)      4 psi + K psi / n_d
 *   stage 2 (P_os+g)    2 psi + (K + 2) psi / n_d
 *   stage 3 (P_os+g+p)  (4 + K) psi / n_d
 * Returns ZERO_OK or ZERO_EINVAL (stage outside 0..3, n_d < 1, psi or K < 0,
 * bytes_out null).
 * ------------------------------------------------------------------------ */
int zero_mem_model(double psi, double K, int n_d, int stage, double* bytes_out);

/* ------------------------------------------------------------------------
 * Plan-exact model states of one rank, with temporaries.  Host only.
 * Source: ZeRO paper (Chinese translation), 5.1-5.3 (which model states each
 * stage partitions), 3.2 and 6.2 (fused fp32 flat buffers: 6 GB for 1.5B
 * parameters, 12 GB for 3B).  zero_mem_model takes a rank's share as
 * psi / n_d; this takes the plan's own sizes, so padding and the remainder
 * ranks are counted:
 *   flat_numel   elements of a 16-bit flat buffer the stage keeps whole: the
 *                plan's padded total (zero_plan), or psi for stage 0
 *   shard_numel  this rank's shard (zero_plan's rank_numels[r]; for ZeRO-3 the
 *                sum of the rank's part of every unit)
 *   K            optimizer-state bytes per parameter (12 for mixed-precision Adam)
 *   state_sets   copies of the optimizer state held: 1 when updated in place,
 *                2 for the double-buffered state of the fused single pass
 *   fp32_temp_numel, b16_temp_numel  elements of fp32 and 16-bit temporaries
 *                (a fused flat buffer, a ZeRO-3 layer buffer, a bucket), or 0
 * bytes_out[5] = parameters, gradients, optimizer states, temporaries, total:
 *   parameters  2 flat_numel for stages 0-2, 2 shard_numel for stage 3
 *   gradients   2 flat_numel for stages 0-1, 2 shard_numel for stages 2-3
 *   states      K state_sets flat_numel for stage 0, K state_sets shard_numel otherwise
 *   temporaries 4 fp32_temp_numel + 2 b16_temp_numel
 * Returns ZERO_OK or ZERO_EINVAL (a negative size, stage outside 0..3,
 * state_sets < 1, K < 0, bytes_out null).
 * ------------------------------------------------------------------------ */
int zero_mem_model_plan(int64_t flat_numel, int64_t shard_numel, double K, int stage, int state_sets,
                        int64_t fp32_temp_numel, int64_t b16_temp_numel, double* bytes_out);

/* ------------------------------------------------------------------------
 * Communication volume per rank and step, in elements.  Host only.
 * Source: ZeRO paper (Chinese translation), 7.1 (a reduce-scatter or an
 * all-gather of Psi elements moves Psi; data parallelism's all-reduce is one
 * of each: 2 Psi), 7.2.1 (P_os+g: gradient reduce-scatter + parameter
 * all-gather, 2 Psi), 7.2.2 (P_os+g+p: parameter all-gathers for the forward
 * and the backward plus the gradient reduce-scatter, 3 Psi = 1.5x); reading
 * notes 5.5 (P_os with the optimised schedule: 2 Psi) and 4 (a ring moves
 * (N_d - 1)/N_d Psi per phase).
 * ring = 0 gives the pages' Psi-per-phase accounting, ring = 1 the ring's
 * exact figure.  Returns ZERO_OK or ZERO_EINVAL (stage outside 0..3, n_d < 1,
 * psi < 0, null output).
 * ------------------------------------------------------------------------ */
int zero_comm_volume(double psi, int n_d, int stage, int ring, double* elements_out);

/* Round-robin order of a group's tensors before flattening.  Host only.
 * Source: DeepSpeed ZeRO stages 1-2 walkthrough, 4.1 (round_robin_gradients):
 * tensor i goes to group i mod world_size and the groups are laid out one
 * after another, each in its original order, so that tensors adjacent in the
 * original (backward) order land in different ranks' shards.
 * order_out[k] = original index of the tensor placed k-th (n_tensors values);
 * feed the reordered sizes to zero_plan.  Returns ZERO_OK or ZERO_EINVAL. */
int zero_plan_round_robin(int n_tensors, int world_size, int64_t* order_out);

/* ------------------------------------------------------------------------
 * The step.
 * ------------------------------------------------------------------------ */

/* Hyper-parameters of one AdamW step (fp32, as the optimizer holds them).
 * step is t of THIS step, 1-based; the caller owns the counter and advances it
 * only when zero_result.applied is 1 (a skipped step does not count).
 * max_grad_norm <= 0 disables clipping. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay, max_grad_norm;
    int64_t step;
} zero_hyper;

/* One simulated rank's shard.
 * numel          elements in the shard (may be 0)
 * grad_offset    element offset of the shard inside every gradient slice
 *                (all-ranks view: the rank's flat offset into each rank's full
 *                gradient; rank-local view with staged slices: 0)
 * param_offset   element offset of the shard inside flat_param
 * *_in           device fp32 master weights, momentum and variance (numel each)
 * *_out          device fp32 outputs; equal to *_in for an in-place update, or a
 *                second state set (ping-pong) that lets the step run in one pass
 * grad_shard     device 16-bit reduced-gradient shard (numel), written by the
 *                two-pass path and read by zero_shard_apply; may be NULL for
 *                calls that take the single pass */
typedef struct {
    int64_t numel, grad_offset, param_offset;
    const float *master_in, *m_in, *v_in;
    float *master_out, *m_out, *v_out;
    void* grad_shard;
} zero_shard;

/* Running gradient statistics in device memory (the scalar all-reduce's
 * operands): sum of squares of the scaled reduced gradient and an overflow
 * flag (nonzero once an inf/NaN was reduced). */
typedef struct {
    double sumsq;
    int32_t overflow;
    int32_t reserved;
} zero_stats;

/* Outcome of a step, written to device (or mapped host) memory.
 * overflow   some reduced gradient element, or extra_overflow, was inf/NaN
 * applied    1 if the update was committed; 0 if the step was skipped --
 *            then the *_in state is the current state, and the parameters are
 *            as before the call (restored by the library where a speculative
 *            pass had written them)
 * path       which kernels ran the update: 1 = the fused single pass,
 *            2 = the apply pass (after the reduce pass), 3 = partial fused
 *            passes decided by zero_shard_step_commit
 * status     0, or ZERO_ELIMIT for a chained step whose t lies outside its
 *            scalar table (nothing is updated)
 * sumsq      sum of squares of the scaled reduced gradient plus extra_sumsq
 * grad_norm  sqrt(sumsq) / loss_scale
 * clip_coef  max_grad_norm / (grad_norm + 1e-6) when that is below 1, else 1
 * grad_mult  fp32(clip_coef / loss_scale), the multiplier applied to the
 *            reduced gradient before AdamW */
typedef struct {
    int32_t overflow, applied, path, status;
    double sumsq, grad_norm, clip_coef;
    float grad_mult, reserved;
} zero_result;

/* Bytes of device workspace the step calls need (zero_shard_step,
 * zero_shard_reduce, zero_shard_apply, zero3_reduce_bucket,
 * zero_shard_step_chained): per-block partial sums and flags, a completion
 * counter and the step's internal statistics.  The amount is fixed (it
 * depends on the most blocks a pass launches, not on the shard sizes), so the
 * call takes no size arguments.  The workspace must be zero-filled once before
 * its first use; every call leaves it ready for the next.  Calls that share a
 * workspace must not overlap on the device. */
size_t zero_workspace_bytes(void);

/* The whole partitioned step over n_shards shards that share one global
 * decision (all simulated ranks, or one rank's shard plus the other ranks'
 * statistics in extra_sumsq / extra_overflow).
 *
 * grad_slices[n_slices]  host array of device pointers: slice r is rank r's
 *                        16-bit gradient (grad_dtype); shard s reads elements
 *                        [grad_offset_s, grad_offset_s + numel_s) of each.
 *                        n_slices = N_d, the averaging divisor.
 * shards[n_shards]       host array
 * flat_param             device 16-bit (param_dtype) flat parameter buffer;
 *                        shard s writes [param_offset_s, + numel_s)
 * hyper                  host
 * loss_scale             S > 0; the reduced gradient is divided by it
 * extra_sumsq, extra_overflow   other ranks' share of the statistics
 * workspace              device, zero_workspace_bytes() bytes, see above
 * result                 device (or mapped host) zero_result
 *
 * Per element i of a shard, in this order: s = sum_r fp32(g_r[i]) in rank
 * order; a = round16(s / N_d); overflow if a is inf/NaN; sumsq += a^2;
 * after all shards: skip if any overflow; k = fp32(c / S) with the clip
 * coefficient c; g = a k; theta = theta * wdf; m = b1 m + (1-b1) g;
 * v = b2 v + (1-b2) g^2; theta = theta - ss * (m / (sqrt(v) * rb2 + eps));
 * flat_param[param_offset + i] = round16(theta), where wdf = fp32(1 - lr wd),
 * ss = fp32(lr / (1 - b1^t)) and rb2 = fp32(1 / sqrt(1 - b2^t)) are computed
 * in fp64 on the host.  Every fp32 operation is rounded on its own (no
 * contraction).
 *
 * Path: with clipping off and every shard's *_out distinct from its *_in, one
 * fused pass reads the slices and the *_in state once and writes the *_out
 * state and the parameters once; if the step is not applied a second, short
 * kernel restores the parameters from master_in (parameters always equal
 * round16(master)).  Otherwise two passes: reduce into grad_shard (required
 * then), then apply.  Both run 16-byte vectors where every slice address
 * (+ grad_offset), state pointer and grad_shard is 16-byte aligned, and
 * element by element otherwise; the state moves in 32-byte accesses where
 * every shard's six state pointers are 32-byte aligned (and, for the apply
 * pass, every grad_shard's vector loop starts on a 128-byte line).  The
 * choice changes no result.
 * Aliasing: apart from *_out == *_in (the in-place update), no output of a
 * call (a state array, a grad_shard, a shard's parameter range) may overlap
 * any input or any other output of the same call; the fused pass reads the
 * *_in state and the slices through the read-only cache while it writes.
 * Errors (all before any work is enqueued): ZERO_EINVAL, ZERO_EALIGN (16-bit
 * pointers must be 2-byte aligned, fp32 pointers 4-byte aligned),
 * ZERO_EWORKSPACE, ZERO_ELIMIT; ZERO_ECUDA if a launch fails. */
int zero_shard_step(const void* const* grad_slices, int n_slices, int grad_dtype,
                    const zero_shard* shards, int n_shards,
                    void* flat_param, int param_dtype,
                    const zero_hyper* hyper, float loss_scale,
                    double extra_sumsq, int extra_overflow,
                    void* workspace, size_t workspace_bytes,
                    zero_result* result, void* stream);

/* State initialisation, before the first step: for every shard, master_in[i]
 * = fp32(flat_param[param_offset + i]) (the exact widening of the 16-bit
 * value) and m_in[i] = v_in[i] = 0.
 * Source: DeepSpeed ZeRO stages 1-2 walkthrough, 4 (3): each rank keeps an
 * fp32 copy of its own partition of the 16-bit parameters (the master
 * weights); Adam's moments start at zero (reading notes, 3).
 * shards and flat_param as for zero_shard_step (all six state pointers set and
 * 4-byte aligned; only the *_in set is written; grad_offset and grad_shard
 * are not used); param_dtype is flat_param's.  Errors: ZERO_EINVAL,
 * ZERO_EALIGN, ZERO_ELIMIT (more than ZERO_MAX_SHARDS shards), ZERO_ECUDA. */
int zero_shard_init(const zero_shard* shards, int n_shards, const void* flat_param, int param_dtype,
                    void* stream);

/* First pass alone: reduce each shard's slices into its grad_shard
 * (a = round16(sum_r fp32(g_r) / n_slices), rank order) and add the shards'
 * sum of squares and overflow flag to *stats (device).  accumulate = 0 starts
 * *stats afresh; 1 adds to what is there (stream order makes successive calls
 * deterministic).  Arguments as for zero_shard_step. */
int zero_shard_reduce(const void* const* grad_slices, int n_slices, int grad_dtype,
                      const zero_shard* shards, int n_shards, int accumulate,
                      zero_stats* stats, void* workspace, size_t workspace_bytes, void* stream);

/* Second pass alone: read each shard's grad_shard and *stats (device), decide
 * skip and clip from stats->sumsq + extra_sumsq and stats->overflow |
 * extra_overflow, run AdamW from *_in to *_out and store the parameters, and
 * write *result.  For ZeRO-3 the parameters are the rank's own parameter
 * shard buffer (param_offset 0 there).  workspace as for zero_shard_step
 * (it must not be the one *stats lives in if that one is reused concurrently;
 * sharing the same workspace in stream order is fine). */
int zero_shard_apply(const zero_shard* shards, int n_shards, int grad_dtype,
                     void* flat_param, int param_dtype,
                     const zero_hyper* hyper, float loss_scale,
                     const zero_stats* stats, double extra_sumsq, int extra_overflow,
                     void* workspace, size_t workspace_bytes,
                     zero_result* result, void* stream);

/* ------------------------------------------------------------------------
 * ZeRO-3 per-layer steps.
 * Source: reading notes 7 and 9 (stage 3: all-gather a layer's parameter
 * shards before its forward and again before its backward; reduce-scatter its
 * gradients to the owner); ZeRO paper (Chinese translation) 7.2.2.
 * A unit (layer) of unit_numel elements is split into world_size equal parts
 * (unit_numel must divide by world_size); rank r keeps part r.
 * ------------------------------------------------------------------------ */

/* layer_out[r * P + j] = part_r[j] for j < P = unit_numel / world_size.
 * part_ptrs[world_size]: host array of device pointers, each P elements
 * (dtype); layer_out: device, unit_numel elements.  Bit-exact copy. */
int zero3_gather_layer(const void* const* part_ptrs, int world_size, int64_t unit_numel, int dtype,
                       void* layer_out, void* stream);

/* The owner-broadcast form of the same materialisation: each rank keeps one
 * contiguous segment of the flat parameter vector (the partition of
 * zero_plan), and a layer is rebuilt from the pieces of the owners' segments
 * it spans -- one or two pieces -- each broadcast by its owner.
 * Source: ZeRO paper (Chinese translation), 5.3 and 7.2.2 (the owner of a
 * partition broadcasts it before the forward of that part of the model, and
 * again before its backward); CMU 11-868 notes, slides 51-63.
 * layer_out = segment 0 | segment 1 | ...: segment_ptrs[n_segments] is a host
 * array of device pointers, segment_numels[n_segments] host element counts.
 * Bit-exact copy.  Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ELIMIT (more than
 * ZERO_MAX_SLICES segments), ZERO_ECUDA. */
int zero3_gather_segments(const void* const* segment_ptrs, const int64_t* segment_numels, int n_segments,
                          int dtype, void* layer_out, void* stream);

/* The same materialisation for a pipelined schedule: the gather of the next
 * unit runs on a side stream while the current unit computes.
 * Source: flycode100 ZeRO tutorial, section 4 (DeepSpeed prefetches the next
 * layer's parameters so that the all-gather overlaps with computation).
 * layer_out = segment 0 | segment 1 | ... exactly as zero3_gather_segments
 * (and, with world_size equal segments, as zero3_gather_layer).  The copy runs
 * on at most n_ctas CTAs (0 = one per SM), leaving the other SMs to whatever
 * else the GPU runs.  When every segment's source and its slot in layer_out
 * agree modulo 16 bytes, the bytes are moved by the TMA unit (bulk copies
 * through shared memory, one thread per CTA issuing them, about 100 GB/s per
 * CTA); otherwise the register-staged gather runs on at most n_ctas blocks.
 * status: device int32 the caller zero-fills; a CTA whose bounded wait for a
 * copy runs out sets bit 0 and stops, and layer_out is then incomplete.
 * Environment (read at each call; meant for tests): ZERO_GB300_SPIN_LIMIT=n
 * sets the tries per bounded wait (default 4194304); 0 makes every first
 * wait give up, which exercises the timeout path without hanging anything.
 * Errors (before any work): ZERO_EINVAL (NULL, negative sizes or n_ctas,
 * unknown dtype, status not 4-byte aligned), ZERO_EALIGN, ZERO_ELIMIT,
 * ZERO_ECUDA. */
int zero3_gather_bulk(const void* const* segment_ptrs, const int64_t* segment_numels, int n_segments, int dtype,
                      void* layer_out, int n_ctas, int32_t* status, void* stream);

/* The owner's share of the unit's gradient reduce-scatter:
 * grad_part[j] = round16(sum_r fp32(bucket_r[owner * P + j]) / world_size),
 * and the part's sum of squares / overflow added to *stats (accumulate as for
 * zero_shard_reduce).  bucket_ptrs[world_size]: host array of device pointers,
 * each a full unit (unit_numel elements).  grad_part: device, P elements. */
int zero3_reduce_bucket(const void* const* bucket_ptrs, int world_size, int owner, int64_t unit_numel,
                        int grad_dtype, void* grad_part, int accumulate, zero_stats* stats,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * The step without caller scratch.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory --
 * code that must not call cudaMalloc because it can synchronise the device
 * and stall other work, callers inside a program whose own allocator owns all
 * device memory, plugins that only receive device pointers through a C
 * interface, code that must not run out of memory in the middle of a step.
 *
 * It computes exactly what zero_shard_step computes, with the same arguments
 * except that there is no workspace, and grad_shard is not used: the step's
 * workspace and, on the two-pass path (clipping on, or some shard updated in
 * place), the shards' 16-bit reduced gradients live in one scratch array built
 * into the library -- WS (the zero_workspace_bytes() amount) plus 2097152
 * reduced-gradient elements, about 4 MB, held on every GPU that loads the
 * library until the process exits.  On the two-pass path the shards together
 * may need at most 2097152 elements (each shard's count rounded up to 128);
 * a larger call returns ZERO_ELIMIT and does nothing.  The fused single pass
 * has no such limit.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Every
 * call shares the array and clears its counter and statistics on `stream`
 * before its kernels run; calls whose work can overlap on the GPU (other
 * streams, other host threads) race on the array and must be serialised by
 * the caller.  No device memory is allocated or freed.
 * ------------------------------------------------------------------------ */
int zero_shard_step_noalloc(const void* const* grad_slices, int n_slices, int grad_dtype,
                            const zero_shard* shards, int n_shards,
                            void* flat_param, int param_dtype,
                            const zero_hyper* hyper, float loss_scale,
                            double extra_sumsq, int extra_overflow,
                            zero_result* result, void* stream);

/* ------------------------------------------------------------------------
 * Steps chained on the device.  zero_shard_step leaves the bookkeeping of a
 * step to the caller: it reads zero_result, swaps the state sets, advances
 * t or lowers S (DeepSpeed ZeRO stages 1-2 walkthrough, 6 step 1: on
 * overflow the optimizer is not called and the loss scale is lowered) -- one
 * device-to-host round trip per step.
 * Here that bookkeeping lives in device memory, so that any number of steps
 * can be enqueued (or captured in a CUDA graph and replayed) without the host
 * waiting on one.
 * ------------------------------------------------------------------------ */

/* Device-resident state of a chain of steps, owned by the caller.
 * cur         the current state set: 0 = every shard's *_in pointers, 1 = its
 *             *_out pointers; the step reads set cur and writes set 1 - cur
 * step        t of the next step (1-based)
 * loss_scale  S of the next step
 * applied, skipped, failed   steps applied, skipped on overflow, and ended
 *             with a nonzero status or an overflow at the loss-scale floor
 * min_loss_scale   floor of S: an overflow halves S only while S / 2 stays at
 *             or above it; <= 0 means 2^-126 (the smallest S whose
 *             reciprocal, the fused pass's multiplier, is finite in fp32)
 * After each step: applied -> step += 1 and cur ^= 1; overflow -> loss_scale
 * halves (no hysteresis, as zero_shard_step's callers do) and `skipped`
 * counts it, or, when halving would go below the floor, S stays and `failed`
 * counts it; a nonzero status (step outside the scalar table) changes nothing
 * but `failed`. */
typedef struct {
    int32_t cur, reserved;
    int64_t step;
    double loss_scale;
    int64_t applied, skipped, failed;
    double min_loss_scale;
} zero_chain;

/* The two step-dependent AdamW scalars for steps t0 .. t0 + n - 1, computed
 * on the host as zero_shard_step computes them (fp64, each rounded once to
 * fp32): table_out[2 i] = lr / (1 - beta1^t), table_out[2 i + 1] =
 * 1 / sqrt(1 - beta2^t) with t = t0 + i.  table_out: host, 2 n floats.  Copy
 * it to the device for zero_shard_step_chained.  hyper->step is ignored.
 * Returns ZERO_OK or ZERO_EINVAL (t0 < 1, n < 0, NULL pointers). */
int zero_adam_scalar_table(const zero_hyper* hyper, int64_t t0, int64_t n, float* table_out);

/* One step with its bookkeeping on the device: what zero_shard_step computes
 * for t = chain->step and S = chain->loss_scale, with the shards' two state
 * sets used by turns (chain->cur), then the chain updated as zero_chain
 * describes.  hyper->step is ignored.  Each shard's *_in and *_out must be
 * two distinct sets (no in-place update: the set read must survive a
 * skipped step).  Clipping (max_grad_norm > 0) takes the reduce and apply
 * passes and needs grad_shard; otherwise the fused pass.
 * scalar_table: device, 2 n_table floats from zero_adam_scalar_table for
 * steps table_t0 .. table_t0 + n_table - 1; a step outside it is not
 * applied and reports status ZERO_ELIMIT.  chain: device.  No host
 * synchronisation; the calls of a chain must run in stream order.
 * Errors as zero_shard_step, and ZERO_EINVAL for a NULL chain or table or a
 * shard updated in place. */
int zero_shard_step_chained(const void* const* grad_slices, int n_slices, int grad_dtype,
                            const zero_shard* shards, int n_shards,
                            void* flat_param, int param_dtype,
                            const zero_hyper* hyper, const float* scalar_table, int64_t table_t0,
                            int64_t n_table, zero_chain* chain,
                            double extra_sumsq, int extra_overflow,
                            void* workspace, size_t workspace_bytes,
                            zero_result* result, void* stream);

/* The apply pass with its bookkeeping on the device: what zero_shard_apply
 * computes for t = chain->step and S = chain->loss_scale, reading the state
 * set chain->cur of every shard and writing the other one, then the chain
 * updated as for zero_shard_step_chained.  The reduce pass before it needs
 * no step scalars, so a chained ZeRO-3 step is its gathers and bucket
 * reduces (zero3_gather_*, zero3_reduce_bucket) followed by this call, and a
 * chained clipped step is zero_shard_reduce followed by this call: neither
 * needs a host round trip between steps.  Unlike the fused pass, the apply
 * pass writes nothing on a skipped step, so a shard may update its state in
 * place (*_out == *_in; the chain's cur then changes nothing).
 * Arguments as zero_shard_apply, plus scalar_table, table_t0, n_table and
 * chain as for zero_shard_step_chained (hyper->step is ignored).  Errors as
 * zero_shard_apply, and ZERO_EINVAL for a NULL or misaligned chain or
 * table. */
int zero_shard_apply_chained(const zero_shard* shards, int n_shards, int grad_dtype,
                             void* flat_param, int param_dtype,
                             const zero_hyper* hyper, const float* scalar_table, int64_t table_t0,
                             int64_t n_table, zero_chain* chain,
                             const zero_stats* stats, double extra_sumsq, int extra_overflow,
                             void* workspace, size_t workspace_bytes,
                             zero_result* result, void* stream);

/* ------------------------------------------------------------------------
 * A step split into partial fused passes and a commit.
 * Source: reading notes 9 (ZeRO-3: after a unit's backward its gradients are
 * reduced onto the owner; the optimizer updates the owner's shard) and the
 * DeepSpeed ZeRO stages 1-2 walkthrough, 6 (skip the whole step on any
 * overflow).  Without clipping nothing of a shard's update depends on the
 * other shards but the skip decision, so each part of a shard can be reduced
 * and updated in one pass as soon as its gradients are ready -- for ZeRO-3,
 * right after each unit's bucket reduce-scatter -- speculatively, into the
 * second state set, with the decision taken once after the last part.  Per
 * element this moves 2 N_d + 26 bytes, where a reduce pass and an apply pass
 * move 2 N_d + 30.
 *
 * zero_shard_step_partial: what zero_shard_step's fused pass computes for
 * these shards (rank-order reduce of their slices, AdamW from *_in to *_out,
 * the parameters stored), with the shards' sum of squares and overflow flag
 * added to *stats (accumulate = 0 starts it afresh) instead of a decision.
 * Arguments as zero_shard_step, plus: max_grad_norm must be 0 (clipping
 * needs the global norm before any update), *_out distinct from *_in;
 * chain NULL takes t from hyper->step and S from loss_scale; otherwise t, S
 * and the state set in use come from the device chain and the scalar table
 * (as zero_shard_step_chained; loss_scale is ignored).  For a ZeRO-3 unit:
 * grad_slices are the world_size full-unit buckets, the shard is the owner's
 * part (grad_offset = owner * unit_numel / world_size) at its place in the
 * rank's parameter shard (flat_param, param_offset) and state.
 *
 * zero_shard_step_commit: the decision from *stats plus extra_sumsq /
 * extra_overflow, written to *result (path 3); on overflow the parameters of
 * every shard given (all the step's parts, or one shard spanning them) are
 * restored from the state set read, and the caller (or the chain) keeps
 * that set; a chain (may be NULL: then loss_scale is the step's S) is
 * updated as after zero_shard_step_chained, and a chained step whose t lies
 * outside [table_t0, table_t0 + n_table) is reported as ZERO_ELIMIT and not
 * applied.  The partial passes and the commit of one step must run in stream
 * order, on one workspace, with nothing between them that reads the *_out
 * state or relies on the parameters of a step that may be skipped.
 * Errors: ZERO_EINVAL (also for clipping or in-place state), ZERO_EALIGN,
 * ZERO_EWORKSPACE, ZERO_ELIMIT, ZERO_ECUDA, before any work is enqueued. */
int zero_shard_step_partial(const void* const* grad_slices, int n_slices, int grad_dtype,
                            const zero_shard* shards, int n_shards,
                            void* flat_param, int param_dtype,
                            const zero_hyper* hyper, float loss_scale,
                            const float* scalar_table, int64_t table_t0, int64_t n_table, zero_chain* chain,
                            int accumulate, zero_stats* stats,
                            void* workspace, size_t workspace_bytes, void* stream);

int zero_shard_step_commit(const zero_shard* shards, int n_shards, void* flat_param, int param_dtype,
                           float loss_scale, int64_t table_t0, int64_t n_table, zero_chain* chain,
                           const zero_stats* stats, double extra_sumsq, int extra_overflow,
                           zero_result* result, void* stream);

/* ------------------------------------------------------------------------
 * The step from host memory: gradients read from, parameters returned to,
 * page-locked host buffers.
 * Source: the DeepSpeed ZeRO stages 1-2 walkthrough, 6 (the step consumes
 * the ranks' gradients and ends with the updated 16-bit parameters, which
 * the all-gather hands back to the training loop).  The same step as
 * zero_shard_step, for a caller whose gradients arrive in host memory and
 * who wants the updated parameters there.
 *
 * The shards are cut into chunks of C elements.  Chunk j's piece of every
 * slice is copied up (on a stream of the library's) into slot j mod 4 of the
 * caller's device ring while the step's kernels run on `stream`: without
 * clipping and with two state sets, one partial fused pass per chunk (as
 * zero_shard_step_partial) and one commit (as zero_shard_step_commit: path
 * 3); otherwise one reduce pass per chunk into grad_shard, then the apply
 * pass (path 2).  After its partial pass each chunk's parameters are copied
 * down to host_param (on a third stream); a step the commit skips has its
 * parameters restored in flat_param and in host_param.  After the apply pass
 * the shards' parameters are copied down on `stream`.
 *
 * host_grad_slices[n_slices]  host array of pointers into page-locked host
 *                             memory (cudaHostAlloc or cudaHostRegister);
 *                             the layout of zero_shard_step's grad_slices
 * host_param                  page-locked host memory the device can
 *                             address, laid out as flat_param: shard s's
 *                             parameters land at [param_offset_s, + numel_s);
 *                             NULL = no copy down
 * staging, staging_bytes      device ring, 16-byte aligned:
 *                             C = staging_bytes / (4 * n_slices * 2) elements
 *                             rounded down to a multiple of 64; C >= 64
 * the rest                    as zero_shard_step (the caller keeps t, S and
 *                             the state set on the host: read *result)
 * Every copy and kernel of the call is ordered after the work enqueued on
 * `stream` before it, and `stream` waits for all of them (the copies down
 * included) before anything enqueued on it later; the host buffers must not
 * change until then.  Calls on one device share the library's two streams:
 * they are serialised on the host, and a ring must not be shared by calls
 * that are not ordered on the device.  Those streams and their events are
 * made by the first call on a device and kept until the process exits; they
 * do not survive cudaDeviceReset, so after a reset of a device this call must
 * not be made on it again in the same process.
 * Errors: ZERO_EINVAL (also for a host buffer that is not page-locked),
 * ZERO_EALIGN, ZERO_EWORKSPACE (also for a ring of fewer than 64 elements per
 * chunk), ZERO_ELIMIT, before any work is enqueued; ZERO_ECUDA. */
int zero_shard_step_host(const void* const* host_grad_slices, int n_slices, int grad_dtype,
                         const zero_shard* shards, int n_shards,
                         void* flat_param, int param_dtype, void* host_param,
                         const zero_hyper* hyper, float loss_scale,
                         double extra_sumsq, int extra_overflow,
                         void* staging, size_t staging_bytes,
                         void* workspace, size_t workspace_bytes,
                         zero_result* result, void* stream);

/* Message of the last error on this thread ("" if none). */
const char* zero_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_GB300_H */
