/*
 * ccl.h -- AllReduce, ReduceScatter and AllGather over p "rank" buffers that
 * all live in the memory of one GPU (NVIDIA GB300, sm_103a), or in pinned
 * host memory that GPU addresses directly.
 *
 * What is computed.  "Inside NCCL AllReduce", section "What all-reduce
 * promises": all-reduce combines one same-shaped buffer per rank element by
 * element (sum, prod, min, max or avg), and at the end all ranks hold the same
 * result; it equals a reduce-scatter (each rank ends owning the
 * finished reduction of one slice) followed by an all-gather (the finished
 * slices go to every rank).  Here the p ranks are p buffers one GPU
 * addresses; there are no peer GPUs and no messages.  Each element is reduced once, in fp32
 * for floating-point types (int32 for int32), in the exact rank order that
 * the schedule gives its chunk, and the finished value is written to every
 * destination in the same pass.
 *
 * Schedules (chunk c is elements [c*q + min(c, r), ...) with q = n / p,
 * r = n % p, i.e. p balanced chunks, larger ones first):
 *  - CCL_SCHED_RING: "Inside NCCL AllReduce", section "The ring, exactly as
 *    the kernel runs it" -- a chunk gathers one more rank's contribution per
 *    hop and completes at its owner.  Chunk c is accumulated in rank order
 *    (c+1) mod p, (c+2) mod p, ..., c (the three-GPU state table: chunk a
 *    starts as a1, adds a2, is completed by a0 on GPU 0).
 *  - CCL_SCHED_ALLPAIRS: "MSCCL, in depth", section "Writing an algorithm in
 *    MSCCLang" -- every rank sends slice r to owner r, which reduces it and
 *    broadcasts it; slice r is accumulated in rank order 0, 1, ..., p-1.
 *  - CCL_SCHED_CUSTOM: the per-chunk orders set by ccl_comm_set_schedule().
 *  - CCL_SCHED_AUTO: the alpha-beta cost model of "MSCCL, in depth" (sections
 *    "Why generic collectives leave time on the table" and "Worked example:
 *    all-pairs versus ring on 8 GPUs") picks ring or all-pairs; see
 *    ccl_select_schedule().
 *
 * Environment overrides, as NCCL's NCCL_ALGO and NCCL_PROTO: CCL_SCHEDULE=
 * ring|allpairs|auto, CCL_VARIANT=ldst|tma|tma_bulkred|auto and
 * CCL_SM_BUDGET=<k> apply only where the choice is left open -- schedule
 * CCL_SCHED_AUTO in the call, variant CCL_VARIANT_AUTO and SM budget 0 in the
 * communicator (ccl_set_launch); explicit values win.  CCL_VARIANT does not
 * apply to AllGather, which has one kernel.  An unset or empty variable
 * changes nothing; any other value outside these lists makes the call fail
 * with CCL_ERR_INVALID_ARG.
 *
 * Numerics.  fp16/bf16/fp32 inputs are widened exactly to fp32; partial
 * results stay fp32 for all p-1 steps; the result is rounded once to the
 * element type, round-to-nearest-even.  sum: fp32 add (no fused multiply-add);
 * prod: fp32 multiply; min/max: acc = (v < acc) ? v : acc (resp. >), so the
 * earlier operand in the schedule order wins ties; avg: each floating-point
 * contribution is multiplied by fl32(1/p) as it is read, and an int32 avg is
 * the wrapped int32 sum divided by p with truncation toward zero ("Inside
 * NCCL AllReduce", "What all-reduce promises").  int32 sum/prod wrap modulo
 * 2^32.  The ld/st and TMA copy variants and the one-phase executor keep this
 * order exactly (identical bits); the TMA bulk-reduce variant
 * (CCL_VARIANT_TMA_BULKRED) lets the memory system apply the adds and is held
 * to |err| <= 2 * p * eps(element type) * sum_k |x_k| per element instead (its
 * min/max pick the same value, but which of +0 and -0, or which NaN, is not
 * fixed); the stepwise-ring executor rounds each partial to the element type
 * at every hop (see ccl_variant_t).  A NaN that the ld/st or TMA variants'
 * min/max keep is the input's own bit pattern for fp16/bf16.
 *
 * Memory and ownership.  The caller allocates and owns every rank buffer
 * (device memory, e.g. from PyTorch).  A communicator copies the p input and
 * output pointers (host arrays are not retained) and allocates one small
 * device status block (256 bytes) that it frees in ccl_comm_destroy().  No
 * call allocates memory proportional to the message.  Rank buffers may also
 * be page-locked host memory the device can address with the same pointer
 * (cudaHostAlloc, or torch's pin_memory): the ld/st kernels then read and
 * write it directly over the host link, with no staging copy (tested for
 * AllReduce, ReduceScatter and AllGather with the ld/st variant).
 *
 * Asynchrony.  The collective calls check their arguments on the host,
 * enqueue kernels on `stream` (a cudaStream_t passed as void*, NULL = the
 * legacy default stream) and return without synchronising.  Errors detected
 * on the host are returned at once; a bounded device-side wait that gave up
 * is reported by ccl_comm_check().  Because they only enqueue, the
 * communicator collectives can be captured in a CUDA graph, provided each
 * variant and SM budget has run once on the device before capture (the first
 * launch sets kernel attributes).
 *
 * Alignment.  All pointers 16-byte aligned (and, for ReduceScatter /
 * AllGather, (n/p) * element size a multiple of 16) take the 128-bit vector
 * path; other layouts take a correct element-wise path (no error).
 *
 * Threads and streams.  A communicator must not be used from two host
 * threads at once.  Its collectives must also be ordered on the device: issue
 * them on one stream, or order the streams.  On large messages the TMA
 * variants and the SM-budget ld/st kernel hand out work from counters in the
 * communicator's status block, so two collectives of one communicator
 * running at the same time would share them.  Different
 * communicators are independent.  ccl_last_error() is per host thread.
 */
#ifndef CCL_H
#define CCL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CCL_API __attribute__((visibility("default")))
#else
#define CCL_API
#endif

#define CCL_MAX_RANKS 64
#define CCL_VERSION 10000 /* 1.0.0 */

typedef struct ccl_comm *ccl_comm_t;

typedef enum {
    CCL_OK = 0,
    CCL_ERR_INVALID_ARG = 1, /* bad pointer, size, alias, enum value, schedule table */
    CCL_ERR_UNSUPPORTED = 2, /* valid request the library does not serve (e.g. bulk-reduce of prod) */
    CCL_ERR_CUDA = 3,        /* a CUDA runtime call failed; ccl_last_error() names it */
    CCL_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (see ccl_comm_check) */
    CCL_ERR_NOMEM = 5,       /* host or device allocation failed */
    CCL_ERR_BOUNDS = 6       /* the checked build saw a kernel compute an access outside a rank
                                buffer and skipped it (see ccl_bounds_checked); never otherwise */
} ccl_status_t;

typedef enum { CCL_SUM = 0, CCL_PROD = 1, CCL_MIN = 2, CCL_MAX = 3, CCL_AVG = 4 } ccl_op_t;

typedef enum { CCL_F32 = 0, CCL_F16 = 1, CCL_BF16 = 2, CCL_I32 = 3 } ccl_dtype_t;

typedef enum {
    CCL_SCHED_AUTO = 0,
    CCL_SCHED_RING = 1,
    CCL_SCHED_ALLPAIRS = 2,
    CCL_SCHED_CUSTOM = 3
} ccl_schedule_t;

typedef enum {
    CCL_VARIANT_AUTO = 0,    /* the ld/st or the TMA kernel (the same bits), whichever the measured
                                launch table estimates faster for the call (see ccl_launch_estimate);
                                TMA only when the layout allows it */
    CCL_VARIANT_LDST = 1,    /* 128-bit register loads/stores, fixed order */
    CCL_VARIANT_TMA = 2,     /* cp.async.bulk into shared-memory stages, fixed order */
    CCL_VARIANT_TMA_BULKRED = 3, /* cp.reduce.async.bulk: order left to the memory system */
    /* Comparison executors (AllReduce only), for measuring the pages' other
     * algorithms on one GPU against the fused kernel: */
    CCL_VARIANT_RING_STEPWISE = 4, /* the ring hop by hop ("Inside NCCL AllReduce", "The ring, exactly as
                                      the kernel runs it"): 2(p-1) launches, each partial held in the element
                                      type in a rank buffer between hops (fp16/bf16 round at every hop; fp32
                                      and int32 give the fused bits); ring schedule only */
    CCL_VARIANT_ONE_PHASE = 5      /* one-phase all-pairs (MSCCL++ 1PA): every rank's output reduced
                                      independently from all p inputs (p^2 n s read); the fused bits;
                                      out of place only */
} ccl_variant_t;

/* ---------------------------------------------------------------------------
 * Communicator.
 * ------------------------------------------------------------------------- */

/* Create a communicator over p rank buffers.
 *  out        : receives the handle (host pointer, must not be NULL).
 *  p          : number of ranks, 1 <= p <= CCL_MAX_RANKS.
 *  rank_ptrs  : host array of p device pointers; rank_ptrs[r] is rank r's
 *               input buffer.  Copied; the array may be freed on return.
 *               Outputs default to the inputs (in place).
 * The current CUDA device at creation is the device every call runs on.
 * T-CCL, section "Programming Model": each rank passes its local buffer
 * and the communication group resolves the peers.
 * Errors: CCL_ERR_INVALID_ARG (NULL out/rank_ptrs, a NULL buffer, p out of
 * range), CCL_ERR_CUDA, CCL_ERR_NOMEM. */
CCL_API ccl_status_t ccl_comm_create(ccl_comm_t *out, int p, void *const *rank_ptrs);

/* Set the p output buffers (host array of device pointers, copied).  NULL
 * restores in-place operation (outputs = inputs).  T-CCL, section
 * "Programming Model": each rank passes its own buffer, and both in-place and
 * out-of-place operation are supported, as in NCCL.  In place means
 * out_ptrs[r] == rank_ptrs[r] for AllReduce and AllGather, and out_ptrs[r] ==
 * rank_ptrs[r] + r*n/p elements for ReduceScatter (NCCL's convention); any
 * other overlap is refused.  Aliasing is checked at each call, since only
 * then are sizes known.  Errors: CCL_ERR_INVALID_ARG (NULL comm, a NULL
 * output pointer). */
CCL_API ccl_status_t ccl_comm_set_outputs(ccl_comm_t comm, void *const *out_ptrs);

/* Set the per-chunk accumulation orders used by CCL_SCHED_CUSTOM.
 * order: host array of p*p bytes; order[c*p + k] is the k-th rank folded
 * into chunk c.  Rejected (CCL_ERR_INVALID_ARG) unless every row is a
 * permutation of 0..p-1 -- the validation of "MSCCL, in depth" (Check():
 * the program computes the declared collective). */
CCL_API ccl_status_t ccl_comm_set_schedule(ccl_comm_t comm, const uint8_t *order);

/* Launch shape.
 *  sm_budget : 0 = all SMs; k > 0 = at most k CTAs, so at most k SMs, the
 *              restricted-CTA-budget setting of T-CCL, section "Collective
 *              Operation Performance" (Fig. 4, Table IV).  Messages that need
 *              more than k CTAs of the regular kernel run one persistent,
 *              large CTA per SM.  Larger than the SM count = all SMs.  The
 *              comparison executors and ccl_allreduce_residual_rmsnorm always
 *              use every SM.
 *  variant   : a ccl_variant_t.  CCL_VARIANT_AUTO consults the launch table
 *              (ccl_launch_estimate).
 *  pipeline_chunk_bytes : 0 = the variant's default (measured per rank
 *              count and, for the TMA kernel, per SM budget).  For the TMA
 *              variants, the bytes per rank moved per pipeline stage
 *              (multiple of 16, 1 KiB .. 32 KiB; at most 16 KiB for the TMA
 *              kernel from 14 ranks, which brings the ranks through the
 *              stages eight at a time, or four above 8 KiB); a size whose
 *              stages do not fit in shared memory for the communicator's p
 *              is refused at the collective call (CCL_ERR_INVALID_ARG).  The
 *              ld/st kernels have no stages
 *              and ignore it.  Results of the fixed-order variants never
 *              depend on it.  This is the stage of the shared-memory pipeline
 *              (T-CCL, "Pipelined Copy and Reduction"), not the multi-MiB
 *              chunk of a ring pipeline between GPUs ("Inside NCCL
 *              AllReduce"): with every rank in one GPU's memory there is no
 *              hop to overlap with the next chunk, and such a chunk would only
 *              decide which CTA handles which part of the buffer when -- a
 *              choice the kernels make themselves (a device-wide work counter
 *              on large messages) and that cannot change any result.
 * Errors: CCL_ERR_INVALID_ARG for a negative budget, an unknown variant or a
 * chunk size outside the range. */
CCL_API ccl_status_t ccl_set_launch(ccl_comm_t comm, int sm_budget, int variant,
                            size_t pipeline_chunk_bytes);

/* Failure-detection hooks (tests).
 *  wait_limit_ns : bound on any single wait inside a kernel that waits (the
 *                  TMA variant's pipeline barriers); 0 restores the default
 *                  of 2 s.  On expiry the kernel records the wait in the
 *                  status block, stops, and ccl_comm_check() returns
 *                  CCL_ERR_TIMEOUT.
 *  stall_test    : 1 makes the TMA producer withhold its second tile, and the
 *                  fused RMSNorm's second CTA of a row withhold its partial
 *                  sum, so that a bounded wait runs out: the timeout path is
 *                  exercised without faulting or hanging the GPU.  2 (the
 *                  checked build only; nothing otherwise) makes the TMA
 *                  producer's bounds check of its second tile fail, so that
 *                  the CCL_ERR_BOUNDS path is exercised: the tile's copies
 *                  are not made.  0 = off.
 * Errors: CCL_ERR_INVALID_ARG for negative values or stall_test > 2. */
CCL_API ccl_status_t ccl_comm_set_debug(ccl_comm_t comm, long long wait_limit_ns, int stall_test);

/* Release the communicator and its device status block (no passage of the
 * pages: housekeeping).  Waits for nothing: the caller must not destroy a
 * communicator whose kernels are still in flight.  NULL is accepted.
 * Errors: CCL_ERR_CUDA if freeing the status block fails. */
CCL_API ccl_status_t ccl_comm_destroy(ccl_comm_t comm);

/* Synchronise the communicator's device and read its status block (no
 * passage of the pages: failure detection, housekeeping).
 * CCL_ERR_TIMEOUT if a bounded wait in a kernel gave up since the last
 * check, CCL_ERR_BOUNDS if (checked build) a kernel computed an access
 * outside a rank buffer and skipped it -- the block is then cleared --,
 * CCL_ERR_CUDA on a CUDA error, otherwise CCL_OK. */
CCL_API ccl_status_t ccl_comm_check(ccl_comm_t comm);

/* 1 if this library is the checked build (compiled with CCL_BOUNDS_CHECK:
 * every kernel tests the extent of each global access it computes against the
 * rank buffer it addresses, records the first violation in the status block
 * and skips the access), 0 for the default build (no passage of the pages:
 * housekeeping, a test aid; the measurements use the default build). */
CCL_API int ccl_bounds_checked(void);

/* ---------------------------------------------------------------------------
 * Collectives.  n is always the element count of one full rank buffer.
 * ------------------------------------------------------------------------- */

/* AllReduce ("Inside NCCL AllReduce", section "What all-reduce promises":
 * every rank ends with the same element-wise reduction of all p buffers; the
 * ring of "The ring, exactly as the kernel runs it" and the all-pairs program
 * of "MSCCL, in depth", "Writing an algorithm in MSCCLang", fix the order):
 * out[r][e] = reduction over ranks of in[k][e], for every r and
 * every e < n, each chunk in its schedule order.  In place (out[r] ==
 * in[r]) or out of place; any other overlap between an output and any
 * buffer is CCL_ERR_INVALID_ARG.  Any n >= 0 (n == 0 is a no-op).
 * Bytes moved: p*n*s read + p*n*s written. */
CCL_API ccl_status_t ccl_allreduce(ccl_comm_t comm, ccl_op_t op, ccl_dtype_t dtype, size_t n,
                           ccl_schedule_t schedule, void *stream);

/* ReduceScatter ("Inside NCCL AllReduce", "What all-reduce promises": each
 * rank ends owning the finished reduction of one slice; T-CCL, "Shard
 * Ownership": the owner of a shard produces its final value):
 * out[r][i] = element c_r + i of the reduction, 0 <= i < n/p,
 * where c_r = r*n/p: rank r receives its own chunk, written from offset 0.
 * Requires n % p == 0 (else CCL_ERR_INVALID_ARG, never a silent fallback).
 * In place in NCCL's sense (out[r] == in[r] + r*n/p elements) or disjoint.
 * Bytes moved: p*n*s read + n*s written. */
CCL_API ccl_status_t ccl_reduce_scatter(ccl_comm_t comm, ccl_op_t op, ccl_dtype_t dtype, size_t n,
                                ccl_schedule_t schedule, void *stream);

/* AllGather ("Inside NCCL AllReduce", "The ring, exactly as the kernel runs
 * it": in the all-gather half the finished chunks travel unchanged to every
 * rank; T-CCL, "Chunk and Window Decomposition": one load fanned out to every
 * destination): rank r contributes elements [r*n/p, (r+1)*n/p) of its input
 * buffer in[r] (n elements); every rank's output out[k] receives all n
 * elements, rank r's chunk at offset r*n/p.  Requires n % p == 0.  In place
 * (out[k] == in[k]: the owner's own chunk is not rewritten) or disjoint.
 * Bytes moved: n*s read + p*n*s written (in place: (p-1)*n*s written). */
CCL_API ccl_status_t ccl_all_gather(ccl_comm_t comm, ccl_dtype_t dtype, size_t n, void *stream);

/* AllReduce fused with the residual merge and RMSNorm, for a tensor-parallel
 * decode step ("Inside NCCL AllReduce", last section: the residual merge and
 * the RMSNorm after the all-reduce run inside the all-reduce kernel).  The
 * communicator's p input buffers are [rows, hidden] row-major (n = rows*hidden
 * elements each).  Per element:
 *   y   = the sum AllReduce of the p inputs, in the schedule's order (fp32,
 *         rounded to dtype) -- exactly ccl_allreduce's result;
 *   h   = round(y + residual_in)       -> residual_out (one buffer)
 *   out = round(h * (1/sqrt(mean_row(h^2) + eps)) * gamma[col]) -> every
 *         rank's output buffer.
 * dtype f32, f16 or bf16 (int32: CCL_ERR_UNSUPPORTED).  residual_in /
 * residual_out: device buffers of n elements; residual_out may equal
 * residual_in (in place) and must otherwise overlap nothing.  gamma: device
 * buffer of hidden elements.  Neither residual_in nor gamma may overlap an
 * output.  Rank buffers follow ccl_allreduce's aliasing rules.  The rounding
 * of y and h is exact; the row's mean square is summed in fp32 in a tree, so
 * out may differ from a fp64 evaluation by one unit in the last place of
 * dtype.  Bytes moved: (2p + 2) n s + hidden s.  When a row is spread over a
 * cluster of CTAs, their exchange of partial sums is a wait bounded by the
 * communicator's wait limit (ccl_comm_set_debug); one that gives up is
 * reported by ccl_comm_check() as CCL_ERR_TIMEOUT (that call's outputs are
 * then wrong; residual_out is complete). */
CCL_API ccl_status_t ccl_allreduce_residual_rmsnorm(ccl_comm_t comm, ccl_dtype_t dtype, size_t rows, size_t hidden,
                                                    const void *residual_in, void *residual_out, const void *gamma,
                                                    float eps, ccl_schedule_t schedule, void *stream);

/* AllReduce for callers that cannot allocate device memory.  The pages have
 * no counterpart: this entry point exists for code that may not call
 * cudaMalloc -- a plug-in inside an application that owns all device memory
 * and hands out only the buffers it manages (an inference server, a
 * framework's memory pool), a process whose memory budget is already
 * committed, or code that must not meet an out-of-memory failure once it is
 * running.  It needs no communicator and allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Computes exactly what ccl_allreduce computes (same chunks, same orders, same
 * bits) with the TMA variant's kernel and its static tile split (no tile
 * counter, so nothing but the status record is shared between calls):
 * out_ptrs[r][e] = reduction over k of
 * in_ptrs[k][e], e < n, for every r.  p in [1, 64]; in_ptrs / out_ptrs are host
 * arrays of p device pointers (in place: out_ptrs[r] == in_ptrs[r]; any other
 * overlap is CCL_ERR_INVALID_ARG); schedule is AUTO (cost model, no
 * environment override), RING or ALLPAIRS.  The buffers and every chunk
 * boundary must be 16-byte aligned, else CCL_ERR_UNSUPPORTED.
 *
 * Scratch: the kernel's only memory beyond the inputs and outputs is the
 * status record its bounded waits write (16 bytes).  It lives in a 256-byte
 * file-scope device array of this library (the stated maximum; a request
 * needing more is refused with CCL_ERR_INVALID_ARG), which every GPU that loads
 * the library holds until the process exits.  The first call on a device looks
 * up that array's device address; make that first call before any stream
 * capture.  All calls share the array and it keeps the last call's contents:
 * each call first waits for the work already queued on `stream` -- the
 * calling host thread blocks until that work is done -- and reads the record
 * the previous call left (returning CCL_ERR_TIMEOUT, without launching, if a
 * wait of that call gave up -- its outputs are then incomplete), then clears
 * it.  Calls that overlap on the GPU (other streams, other threads) race on
 * the record.
 * Errors: CCL_ERR_INVALID_ARG, CCL_ERR_UNSUPPORTED, CCL_ERR_TIMEOUT,
 * CCL_ERR_CUDA; messages through ccl_last_error(). */
CCL_API ccl_status_t ccl_allreduce_static(int p, void *const *in_ptrs, void *const *out_ptrs, ccl_op_t op,
                                          ccl_dtype_t dtype, size_t n, ccl_schedule_t schedule, void *stream);

/* Failure-detection hook of ccl_allreduce_static (tests); no passage of the
 * pages: housekeeping.  Sets, for every later call in this process, the bound
 * on any single wait of its kernel (0 restores the default of 2 s) and
 * whether its producer withholds the second tile (stall_test = 1), so that a
 * wait runs out on purpose and the next call reports CCL_ERR_TIMEOUT.
 * Nothing traps or faults.  Errors: CCL_ERR_INVALID_ARG for negative values
 * or stall_test > 1. */
CCL_API ccl_status_t ccl_allreduce_static_set_debug(long long wait_limit_ns, int stall_test);

/* ---------------------------------------------------------------------------
 * Host-side schedule builder and cost model (no GPU needed).
 * ------------------------------------------------------------------------- */

/* Build the per-chunk table of a schedule.
 *  bounds : host array of p+1 entries; chunk c is [bounds[c], bounds[c+1]).
 *  order  : host array of p*p bytes; order[c*p + k] = k-th rank folded into c.
 * schedule must be CCL_SCHED_RING or CCL_SCHED_ALLPAIRS.
 * The owner of chunk c (ReduceScatter destination) is rank c. */
CCL_API ccl_status_t ccl_schedule_build(int p, uint64_t n, ccl_schedule_t schedule,
                                uint64_t *bounds, uint8_t *order);

/* Validate a table: bounds partition [0, n) in order, every row of order is
 * a permutation of 0..p-1.  CCL_OK or CCL_ERR_INVALID_ARG. */
CCL_API ccl_status_t ccl_schedule_check(int p, uint64_t n, const uint64_t *bounds,
                                const uint8_t *order);

/* Alpha-beta model parameters ("MSCCL, in depth"): alpha_s per synchronised
 * step, link bandwidth in bytes/s, and the protocol efficiency each schedule
 * runs at (LL = 0.5, LL128 = 120/128 on the page). */
typedef struct {
    double alpha_s;
    double bw_bytes_per_s;
    double eff_ring;
    double eff_allpairs;
} ccl_cost_params_t;

/* Modelled time (seconds) of AllReduce of nbytes per rank over p ranks:
 * ring 2(p-1)*alpha + 2(p-1)/p * nbytes / (bw*eff_ring); all-pairs
 * 2*alpha + 2(p-1)/p * nbytes / (bw*eff_allpairs).  params NULL = the
 * page's worked-example values (2 us, 300 GB/s, 120/128, 0.5).
 * Returns a negative value for bad arguments. */
CCL_API double ccl_cost_estimate(int p, double nbytes, ccl_schedule_t schedule,
                         const ccl_cost_params_t *params);

/* The schedule AUTO resolves to: the lower modelled time (ties: ring). */
CCL_API ccl_schedule_t ccl_select_schedule(int p, double nbytes, const ccl_cost_params_t *params);

/* The measured launch table behind CCL_VARIANT_AUTO (T-CCL, section "Launch
 * Configuration Tuning": launch configurations profiled offline and ranked
 * per message size in a table the runtime consults).  The table, compiled
 * into the library, holds the per-call device time of an AllReduce (sum,
 * ring) with the ld/st and the TMA kernel at measured points: rank count,
 * element size, SM budget, bytes per rank (reducescatter_reduction_gb300/
 * calibrate.py measures it on the GPU it is for).  This call returns, in
 * *us, the table's estimate for p ranks of `dtype`, `sm_budget` (0 = every
 * SM; a budget at or above the table's SM count is every SM) and
 * `bytes_per_rank`, for variant CCL_VARIANT_LDST or CCL_VARIANT_TMA: the
 * nearest measured rank count and SM budget on a log scale (ties: the
 * larger), the element size itself, a power law between the two nearest
 * measured sizes, the smallest size's time below it, and the straight line
 * through the two largest sizes above it.  AUTO takes TMA exactly when its
 * estimate is below 0.98 times the ld/st one and the layout allows TMA
 * (16-byte aligned pointers and chunk boundaries).  No GPU is needed.
 * Errors: CCL_ERR_INVALID_ARG (NULL us, p outside [1, 64], unknown dtype,
 * negative budget, another variant), CCL_ERR_UNSUPPORTED (the table has no
 * point for this element size). */
CCL_API ccl_status_t ccl_launch_estimate(int p, ccl_dtype_t dtype, int sm_budget, size_t bytes_per_rank, int variant,
                                         double *us);

/* ---------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------- */

/* Message for the last non-OK status returned on this host thread (no
 * passage of the pages: housekeeping).  Never NULL; the string is owned by
 * the library and valid until the next call on this thread. */
CCL_API const char *ccl_last_error(void);

/* Description of the last kernel launch this communicator issued (kernel,
 * dtype, op, p, n, schedule, variant, grid, block, shared memory, SM budget,
 * counter=1 when CTAs or warps took work from a device-wide counter, and
 * inplace=1 when an output is an input, so that the kernels loaded without
 * ld.global.nc), so
 * that a caller can prove which path ran -- "MSCCL, in depth", section
 * "Deploying it": check that the custom algorithm actually ran instead of a
 * silent fallback.  Copies at most len-1 characters plus a terminating NUL
 * into buf; returns CCL_ERR_INVALID_ARG if comm or buf is NULL or len is 0. */
CCL_API ccl_status_t ccl_comm_last_launch(ccl_comm_t comm, char *buf, size_t len);

/* Number of kernels this communicator has launched since creation (no
 * passage of the pages: housekeeping; 0 for a NULL comm). */
CCL_API uint64_t ccl_comm_launch_count(ccl_comm_t comm);

/* CCL_VERSION of the loaded library (housekeeping). */
CCL_API int ccl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCL_H */
