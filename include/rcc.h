/*
 * rcc.h -- C ABI of librcc: tensor collectives over R logical ranks whose
 * buffers all live on one GPU, and the gradient-sync + fused AdamW step that
 * consumes them.
 *
 * Sources (page title, section):
 *   [ruCCL]   ruCCL README (ja): §2 "Tensor collective API" (register,
 *             all_reduce, broadcast, reduce, finish_collective,
 *             reset_collective), §3 "Registration and call contract",
 *             §4 "Errors and lifecycle", §5 "CUDA example" (4 logical ranks on
 *             GPU 0), §6 "Collective training" (all_reduce Mean of gradients,
 *             then optimizer.step).
 *   [RUDA-T]  RUDA docs "Training and saving state", section "Native PyTorch
 *             training on ruda:0": ruda_torch.AdamW(fused_step, max_grad_norm,
 *             hierarchical_stats), the 12-byte report read back before the
 *             update, skip on non-finite gradients, FP32 master weights and
 *             moments, one update kernel per parameter, fan-in-1024 statistics
 *             with at most two extra combine kernels and a reused reduction
 *             region of at most 49,200 bytes; ruda_torch.GradScaler.
 *   [Monarch] "Struct Communicator" (torch_sys_cuda::nccl): all_reduce,
 *             broadcast, reduce, all_gather_into_tensor, reduce_scatter_tensor,
 *             each issued on a stream, each returning a status.
 *
 * Conventions shared by every call:
 *   - Buffers are device memory on the session's GPU, owned by the caller.
 *     Per-rank arguments are arrays of R entries indexed by logical rank.
 *   - Calls validate everything on the host first (in the order of the
 *     status codes below) and launch nothing when they return an error.
 *   - Collectives are asynchronous on `stream`: they enqueue kernels and
 *     return without synchronising.  rcc_grad_sync_adamw synchronises once,
 *     to read its 12-byte report back.
 *   - Inputs are never written, except where a call documents an in-place
 *     form.  Outputs must not overlap each other or any input otherwise.
 *   - The current CUDA device must be the session's device.
 *   - Error text for the calling thread: rcc_last_error_message().
 *   - Kernels are launched with programmatic dependent launch: each waits
 *     for the kernel ahead of it on the stream to finish before touching
 *     memory, so ordering is that of a plain launch; only the launch latency
 *     overlaps.  Streams captured into a CUDA graph record these as
 *     programmatic edges.
 *
 * Environment (read once per process):
 *   RCC_WAIT_LIMIT_MS  limit of every host wait (default 120000).
 *   RCC_PDL=0          launch without programmatic dependent launch.
 *   RCC_VEC_BYTES=16   cap vector accesses at 16 bytes.
 *   RCC_CHAINS=n       parallel chains of per-tensor update launches
 *                      (1..32, default 16).
 *   RCC_AUTO_GRAPH=0   the default grad-sync flow never switches to graph
 *                      replay.
 *   RCC_NVTX=1         every call opens an NVTX range named after it (and the
 *                      grad-sync readback wait one of its own), for a profiler.
 */
#ifndef RCC_H
#define RCC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* rcc_stream_t;

#define RCC_MAX_RANKS 64

/* [ruCCL §4]: CollectiveError covers duplicate or missing registration, shape
 * mismatch, inconsistent reduction op or root, and an invalid broadcast
 * sender count; [Monarch] calls return a status or an error. */
typedef enum {
  RCC_OK = 0,
  RCC_ERR_DUPLICATE_REGISTRATION = 1, /* a live session already exists on that device */
  RCC_ERR_MISSING_REGISTRATION = 2,   /* dead handle, or a rank's required buffer is NULL */
  RCC_ERR_SHAPE_MISMATCH = 3,         /* per-rank counts differ; reduce_scatter count % R != 0 */
  RCC_ERR_INCONSISTENT_OP = 4,        /* per-rank ops differ, or an op is not an rcc_op */
  RCC_ERR_INCONSISTENT_ROOT = 5,      /* per-rank roots differ, or root outside [0, R) */
  RCC_ERR_BROADCAST_SENDERS = 6,      /* broadcast with a number of senders other than 1 */
  RCC_ERR_INVALID_ARGUMENT = 7,       /* anything else malformed (NULL array, bad dtype, overlap, ...) */
  RCC_ERR_TIMEOUT = 8,                /* a bounded wait for the GPU ran out */
  RCC_ERR_CUDA = 9                    /* a CUDA runtime call failed */
} rcc_status;

typedef enum { RCC_F32 = 0, RCC_BF16 = 1 } rcc_dtype;

/* Reduction operations.  [ruCCL §6] names Mean; sum, max and min complete the
 * set.  Arithmetic is fp32 for both dtypes (bf16 is widened exactly and the
 * result rounded once to nearest-even).  MEAN = fl32(sum / R).  MAX/MIN keep
 * the lowest rank's value among equals and return the quiet NaN 0x7FC00000
 * (bf16 0x7FC0) when any input is NaN. */
typedef enum { RCC_SUM = 0, RCC_MEAN = 1, RCC_MAX = 2, RCC_MIN = 3 } rcc_op;

/* Session flags.  RCC_DETERMINISTIC: sums fold ranks in the fixed order
 * 0, 1, ..., R-1 (acc = x0; acc = fl32(acc + x_r)), bit-identical to that
 * definition.  Without it sums use a pairwise tree over ranks (same traffic,
 * shorter dependency chain, results within the fp32 error bound).  MAX and
 * MIN are exact in both modes. */
#define RCC_DETERMINISTIC 0x1u
/* Session flag RCC_STEP_TIMING: rcc_grad_sync_adamw records CUDA events
 * between its phases, which rcc_last_step_times reads back.  A diagnostic: the
 * events sit between kernels that otherwise overlap their launches
 * (programmatic dependent launch), so a timed step can run a few microseconds
 * longer. */
#define RCC_STEP_TIMING 0x2u

/* Opaque session handle.  A finished or reset handle stays detectable: calls
 * on it return RCC_ERR_MISSING_REGISTRATION, never touch freed memory. */
typedef struct rcc_comm_s* rcc_comm;

/* ---- session lifecycle --------------------------------------------------- */

/* [ruCCL §2 register, §3: participants agree on the device count; §5: four
 * logical ranks on GPU 0].  Registers num_ranks (1..RCC_MAX_RANKS) logical
 * ranks on CUDA device `device` with element type `dtype`.  One live session
 * per device ("the local collective service", [ruCCL §2 reset_collective]);
 * a second registration on that device returns
 * RCC_ERR_DUPLICATE_REGISTRATION.  Makes no CUDA call: session scratch is
 * allocated on first use.  *out receives the handle. */
rcc_status rcc_register(int device, int num_ranks, rcc_dtype dtype,
                        unsigned flags, rcc_comm* out);

/* Replace the session flags (e.g. switch RCC_DETERMINISTIC) for later calls. */
rcc_status rcc_set_flags(rcc_comm comm, unsigned flags);

/* [ruCCL §2 finish_collective, §4 "normal termination"].  Waits for work
 * enqueued on `stream` (bounded: RCC_ERR_TIMEOUT after the limit), frees the
 * session's scratch and ends the session. */
rcc_status rcc_finish(rcc_comm comm, rcc_stream_t stream);

/* [ruCCL §2 reset_collective, §4: discards registration and in-flight
 * operation state; completes nothing, checkpoints nothing, recovers nothing].
 * Ends the session at once.  Kernels already enqueued run to completion on
 * the GPU (freeing the scratch waits for them); their results are not
 * reported.  A new rcc_register on the device succeeds afterwards. */
rcc_status rcc_reset(rcc_comm comm);

/* ---- collectives ---------------------------------------------------------
 * Every call: send/recv are arrays of R device pointers; counts, ops, roots
 * are arrays of R per-rank values that must agree ([ruCCL §3]: shape,
 * reduction op, root and other parameters must match).  A count of 0 is a
 * valid no-op.  Element type is the session's dtype. */

/* [ruCCL §2 all_reduce; §5 sum/mean with inputs unchanged; Monarch
 * all_reduce].  recv[r][i] = op(send[0][i], ..., send[R-1][i]) for every
 * rank r, i < counts[r].  Out of place; recv[r] == send[r] (in place) is also
 * accepted. */
rcc_status rcc_all_reduce(rcc_comm comm, const void* const* send,
                          void* const* recv, const size_t* counts,
                          const rcc_op* ops, rcc_stream_t stream);

/* [ruCCL §2 reduce: non-root participants receive nothing; Monarch reduce].
 * recv[root][i] = op_q send[q][i].  Only recv[root] is used (other entries
 * may be NULL and are never written).  recv[root] == send[root] (in place) is
 * accepted. */
rcc_status rcc_reduce(rcc_comm comm, const void* const* send,
                      void* const* recv, const size_t* counts,
                      const rcc_op* ops, const int* roots,
                      rcc_stream_t stream);

/* [ruCCL §2 broadcast: the sender passes Some(tensor), receivers None; §3:
 * each broadcast has exactly one sender; Monarch broadcast].  Exactly one
 * send[r] is non-NULL: that rank is the root.  recv[r][i] = send[root][i]
 * for every rank r whose recv[r] is non-NULL and not send[root] itself;
 * every non-root rank must supply recv[r]. */
rcc_status rcc_broadcast(rcc_comm comm, const void* const* send,
                         void* const* recv, const size_t* counts,
                         rcc_stream_t stream);

/* [Monarch reduce_scatter_tensor: reduce, then scatter].  in_counts[r] = N
 * elements per rank input, N % R == 0, shard n = N / R.
 * recv[r][j] = op_q send[q][r*n + j] for j < n (recv[r] holds n elements). */
rcc_status rcc_reduce_scatter(rcc_comm comm, const void* const* send,
                              void* const* recv, const size_t* in_counts,
                              const rcc_op* ops, rcc_stream_t stream);

/* [Monarch all_gather_into_tensor].  in_counts[r] = n elements per rank
 * input; recv[r] holds R*n elements: recv[r][q*n + j] = send[q][j]. */
rcc_status rcc_all_gather(rcc_comm comm, const void* const* send,
                          void* const* recv, const size_t* in_counts,
                          rcc_stream_t stream);

/* [Monarch all_to_all_single: split the input, scatter the split list to all
 * ranks, concatenate what each receives].  Equal splits: in_counts[r] = N
 * elements per rank, N % R == 0 (else RCC_ERR_SHAPE_MISMATCH), n = N / R;
 * recv[r] holds N elements and recv[r][q*n + j] = send[q][r*n + j].
 * No in-place form: outputs must not overlap any input. */
rcc_status rcc_all_to_all_single(rcc_comm comm, const void* const* send,
                                 void* const* recv, const size_t* in_counts,
                                 rcc_stream_t stream);

/* [Monarch all_gather: gather tensors from all ranks into a list of output
 * tensors].  in_counts[r] = n; recv has R*R entries, row-major by receiving
 * rank: recv[r*R + q] (n elements) receives send[q].  Rank r's own entry
 * recv[r*R + r] may be send[r] itself (nothing is copied for it).  One copy
 * pass per source rank. */
rcc_status rcc_all_gather_list(rcc_comm comm, const void* const* send,
                               void* const* recv, const size_t* in_counts,
                               rcc_stream_t stream);

/* ---- per-rank arrival ------------------------------------------------------
 * [ruCCL introduction and §1 (the in_process implementation: logical ranks
 * inside one process), §3: every
 * rank calls matching collectives in the same order with matching shape, op
 * and root; Monarch Communicator::new: one thread per rank].
 * Each logical rank -- typically its own host thread -- calls the *_rank form
 * with only its own buffers and its own stream.  The call returns once every
 * rank of the session has arrived: the last arrival checks that all ranks
 * called the same collective and agree (the group calls' checks and codes;
 * a different collective on some rank is RCC_ERR_INCONSISTENT_OP), makes the
 * kernel wait for the work each rank had queued on its stream, launches once,
 * and every rank's stream then waits for the kernel.  All ranks return the
 * same status.
 *   - A rank arriving twice for one collective: RCC_ERR_INVALID_ARGUMENT (to
 *     that call; the collective keeps waiting for the missing ranks).
 *   - Not every rank arriving within the wait limit (RCC_WAIT_LIMIT_MS,
 *     default 120 s): the waiting ranks get RCC_ERR_TIMEOUT and the
 *     collective is discarded.
 *   - rcc_reset or rcc_finish while ranks wait: they return
 *     RCC_ERR_MISSING_REGISTRATION ([ruCCL §4]: reset discards in-flight
 *     operation state).
 * Arguments mean what the group call's per-rank entries mean: for reduce only
 * the root's recv is used; for broadcast exactly one rank passes send. */
rcc_status rcc_all_reduce_rank(rcc_comm comm, int rank, const void* send, void* recv,
                               size_t count, rcc_op op, rcc_stream_t stream);
rcc_status rcc_reduce_rank(rcc_comm comm, int rank, const void* send, void* recv,
                           size_t count, rcc_op op, int root, rcc_stream_t stream);
rcc_status rcc_broadcast_rank(rcc_comm comm, int rank, const void* send, void* recv,
                              size_t count, rcc_stream_t stream);
rcc_status rcc_reduce_scatter_rank(rcc_comm comm, int rank, const void* send, void* recv,
                                   size_t in_count, rcc_op op, rcc_stream_t stream);
rcc_status rcc_all_gather_rank(rcc_comm comm, int rank, const void* send, void* recv,
                               size_t in_count, rcc_stream_t stream);

/* ---- gradient sync + fused AdamW ----------------------------------------- */

/* One parameter tensor as seen by every rank. */
typedef struct {
  size_t numel;                /* elements per rank (> 0) */
  const size_t* rank_numel;    /* optional [R]: each rank's own element count; all must
                                  equal numel ([ruCCL §6]: gradient shapes must match
                                  across ranks), else RCC_ERR_SHAPE_MISMATCH; NULL: skip */
  const float* const* grads;   /* [R] rank r's loss-scaled fp32 gradient; read only */
  float* const* params;        /* [replicas] fp32 master parameters, updated in place */
  float* const* exp_avg;       /* [replicas] fp32 first moments m, updated in place */
  float* const* exp_avg_sq;    /* [replicas] fp32 second moments v, updated in place */
  float* mean_grad;            /* optional [numel]: receives the unscaled mean gradient;
                                  NULL: not stored (the update re-reads the R grads) */
} rcc_param_set;

/* ruda_torch.AdamW options [RUDA-T] plus the published AdamW constants. */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
  double max_grad_norm;        /* > 0: clip when the global L2 norm exceeds it; <= 0: off */
  int32_t replicas;            /* optimizer-state copies: 1 or R (each rank its own) */
  int32_t hierarchical_stats;  /* 1: fan-in-1024 combines [RUDA-T] (none for <= 1024
                                  rows, at most two); 0: one flat final reduction */
  uint32_t elems_per_row;      /* elements summarised per statistics row; 0 = 8192;
                                  otherwise a multiple of 4 in [4, 2^24] */
  uint32_t flags;              /* 0 (the pages' flow) or RCC_ADAMW_* bits below */
} rcc_adamw_cfg;

/* rcc_adamw_cfg.flags.  By default the call reads the 12-byte report back,
 * decides on the host, then launches the updates ([RUDA-T]).  Once the same
 * tensors (32 or more) come three calls in a row, the default flow replays
 * those launches from a captured graph, as RCC_ADAMW_HOST_GRAPH does
 * (RCC_AUTO_GRAPH=0 keeps plain launches); the results are the same bits.
 * RCC_ADAMW_DEVICE_DECISION: one more kernel takes the same decision on the
 *   GPU from the report (identical arithmetic: IEEE double sqrt and division,
 *   one rounding to fp32), so the per-tensor updates are enqueued right behind
 *   the statistics; a skipped step launches updates that return at once.  The
 *   report is still read back before the call returns.  Like the default flow,
 *   it switches to replaying the per-tensor launches from a captured graph (as
 *   RCC_ADAMW_GRAPH) once the same tensors (32 or more) come three calls in a
 *   row (not with RCC_AUTO_GRAPH=0).
 * RCC_ADAMW_GRAPH: as DEVICE_DECISION, and the per-tensor update launches are
 *   captured once into a CUDA graph and replayed while the tensors' pointers
 *   and sizes stay the same (still one kernel node per parameter tensor).
 * RCC_ADAMW_MULTI_TENSOR: one update launch covers every tensor (one CTA per
 *   statistics row) instead of one launch per tensor -- a comparison point
 *   against the pages' one-kernel-per-parameter design; not with GRAPH.
 * RCC_ADAMW_HOST_GRAPH: the pages' order (report read back, decision on the
 *   host), then one 8-byte copy puts the decision in device memory and the
 *   captured per-tensor update graph of RCC_ADAMW_GRAPH is replayed instead of
 *   P separate launches; a skipped step launches nothing.  Takes no other
 *   flag. */
#define RCC_ADAMW_DEVICE_DECISION 0x1u
#define RCC_ADAMW_GRAPH 0x2u
#define RCC_ADAMW_MULTI_TENSOR 0x4u
#define RCC_ADAMW_HOST_GRAPH 0x8u

/* Optimizer step count and GradScaler state, owned by the caller, updated by
 * each call ([RUDA-T]: scale -> step -> update on the same GradScaler). */
typedef struct {
  int64_t step;                /* applied AdamW steps t (skipped steps do not count) */
  double scale;                /* loss scale S the gradients carry */
  double growth_factor;        /* S *= growth_factor after growth_interval finite steps */
  double backoff_factor;       /* S *= backoff_factor on a skipped step */
  int32_t growth_interval;
  int32_t growth_tracker;      /* consecutive finite steps since the last change */
} rcc_optim_state;

/* What one call did. */
typedef struct {
  double sum_sq;               /* sum of g^2 over finite unscaled mean gradients (fp64) */
  double grad_norm;            /* sqrt(sum_sq) */
  double scale_used;           /* the loss scale the gradients were divided by */
  uint32_t nonfinite;          /* non-finite unscaled mean gradient elements */
  int32_t skipped;             /* 1: whole step skipped (state untouched) */
  float clip_coef;             /* multiplier applied to g (1 when not clipped) */
  int32_t combine_launches;    /* extra hierarchical combine kernels launched (0..2) */
  uint64_t stats_rows;         /* rows written by the statistics kernel */
  uint64_t combine_region_bytes; /* bytes of the reused reduction region touched (<= 49,200) */
  uint64_t update_launches;    /* AdamW update kernels launched (num_params or 0) */
  uint32_t report_words[3];    /* the 12-byte report as read back: low and high 32-bit
                                  words of the fp64 sum of g^2, then the u32 count of
                                  non-finite g (saturated at 2^32 - 1) */
  int32_t combine_levels;      /* fan-in-1024 levels applied (0..2); one combine
                                  kernel each */
  int32_t updates_before_readback; /* 1: the update launches were enqueued before the
                                  readback (the device-decision flows); a skipped
                                  step's launches then return at once */
} rcc_step_report;

/* [ruCCL §6 + RUDA-T].  One data-parallel optimizer step over num_params
 * tensors:
 *   1. all_reduce Mean of the R loss-scaled gradients in rank order, then
 *      unscale: g = fl32(fl32(sum_q grads[q]) / R) * fl32(1 / S);
 *   2. read-only analysis: sum of g^2 (fp64) and a count of non-finite g,
 *      one 12-byte row per statistics block, fan-in-1024 combines (none for
 *      <= 1024 rows, at most two), a 12-byte report in device memory;
 *   3. the report is read back (the call's one synchronisation);
 *   4. any non-finite g (or norm) skips the whole step: parameters, moments
 *      and step count are untouched, S backs off;
 *   5. otherwise clip_coef = max_grad_norm / ||g|| when ||g|| > max_grad_norm,
 *      t = step + 1, and one AdamW update kernel per tensor updates every
 *      replica: p = p*(1 - lr*wd); m = b1*m + (1-b1)*g'; v = b2*v + (1-b2)*g'^2;
 *      p -= lr/(1-b1^t) * m / (sqrt(v)/sqrt(1-b2^t) + eps), g' = g*clip_coef;
 *      S grows after growth_interval finite steps.
 * Session dtype must be RCC_F32.  Gradients are never written (several ranks
 * or tensors may even share one gradient buffer).  The update kernels of
 * different tensors may run concurrently, so parameter, moment and
 * mean-gradient buffers must not overlap any other buffer of the call
 * (RCC_ERR_INVALID_ARGUMENT; checked whenever the set of buffers changes).
 * `state` is read and updated; `report` (may be NULL) receives what happened.
 * Returns RCC_ERR_TIMEOUT if the report did not arrive within the wait limit:
 * in the default and RCC_ADAMW_HOST_GRAPH flows nothing is then applied and
 * `state` is unchanged (the call may simply be repeated); in the
 * device-decision flows the queued updates still run, so the optimizer state
 * should be treated as unknown.  The next call on the session first waits
 * (bounded) for the abandoned call's queued work. */
rcc_status rcc_grad_sync_adamw(rcc_comm comm, const rcc_param_set* params,
                               int num_params, const rcc_adamw_cfg* cfg,
                               rcc_optim_state* state, rcc_step_report* report,
                               rcc_stream_t stream);

/* Phase times of the session's most recent rcc_grad_sync_adamw call, made
 * while the session had RCC_STEP_TIMING set, in milliseconds of GPU time
 * between CUDA events on the call's stream:
 *   out_ms[0] statistics kernel (mean, unscale, one row per block);
 *   out_ms[1] the fan-in-1024 combines and the 12-byte report;
 *   out_ms[2] from the report to the first update launch: in the default
 *             flow the readback, the host's decision and the launch issue;
 *             in the device-decision flows the decision kernel;
 *   out_ms[3] the update launches (0 launches on a skipped host-flow step).
 * Waits (bounded) for the call's work.  RCC_ERR_INVALID_ARGUMENT when the
 * session has no timed call. */
rcc_status rcc_last_step_times(rcc_comm comm, float out_ms[4]);

/* ---- gradient statistics without allocation ------------------------------- */

/* The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory at all -- code running while a stream is
 * being captured into a CUDA graph with allocation forbidden, processes whose
 * device memory belongs to another runtime or a fixed pool, or hosts that may
 * only pass buffers they already own.  rcc_grad_sync_adamw allocates session
 * scratch on first use; this call never does (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * It computes steps 1-2 of rcc_grad_sync_adamw for ONE parameter tensor:
 * g = fl32(fl32(sum_q grads[q]) / R) * fl32(1 / loss_scale), optionally
 * stored to mean_grad[numel] (device, may be NULL), and writes the 12-byte
 * report {low word, high word of the fp64 sum of g^2 over finite g, u32 count
 * of non-finite g} to `report` (device, 4-byte aligned).  Rows of 8192
 * elements and the fan-in-1024 combine are the same as rcc_grad_sync_adamw's
 * with its default elems_per_row, so the two give the same report.
 *
 * Limits and behaviour:
 *   - grads: host array of num_ranks (1..RCC_MAX_RANKS) device pointers;
 *     numel in [1, 134,217,728] (16,384 rows); anything larger returns
 *     RCC_ERR_INVALID_ARGUMENT.
 *   - The rows live in one file-scope device array of 196,800 bytes that every
 *     GPU which loads the library keeps until the process exits.  All calls
 *     share it: calls that overlap on the GPU (different streams, no ordering)
 *     race on it.  Every row is rewritten before it is read, so nothing needs
 *     clearing between calls.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: a cudaDeviceReset on
 *     that device invalidates it, so do not call this entry point after a
 *     device reset in the same process.
 *   - Asynchronous on `stream`; no session is needed. */
rcc_status rcc_grad_stats_noalloc(const float* const* grads, int num_ranks,
                                  size_t numel, double loss_scale,
                                  float* mean_grad, uint32_t* report,
                                  rcc_stream_t stream);

/* ---- diagnostics ---------------------------------------------------------- */

/* Message describing the calling thread's most recent error ("" if none). */
const char* rcc_last_error_message(void);

/* Fixed name of a status code. */
const char* rcc_status_string(rcc_status status);

/* Number of kernels this library has launched in the process so far. */
uint64_t rcc_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* RCC_H */
