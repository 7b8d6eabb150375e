/*
 * rcc_oracle.h -- CPU oracle for the librcc hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded CPU
 * restatement of what the collectives and the gradient-sync step compute.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA
 * library, and the library never calls it.
 *
 * Sources followed (page title, section):
 *   [ruCCL]    ruCCL README (ja): §2 "Tensor collective API", §3 "Registration
 *              and call contract", §4 "Errors and lifecycle", §5 "CUDA example",
 *              §6 "Collective training".
 *   [RUDA-T]   RUDA docs "Training and saving state": section "Native PyTorch
 *              training on ruda:0" (ruda_torch.AdamW fused step, GradScaler,
 *              12-byte report, hierarchical statistics).
 *   [Monarch]  "Struct Communicator" (torch_sys_cuda::nccl): all_reduce,
 *              reduce, broadcast, all_gather_into_tensor, reduce_scatter_tensor.
 *   AdamW itself is only named by the pages; its arithmetic follows the
 *   published decoupled-weight-decay Adam (Loshchilov & Hutter, "Decoupled
 *   Weight Decay Regularization", ICLR 2019, Algorithm 2) with Adam's bias
 *   correction (Kingma & Ba, 2015).
 *
 * Precision: the "rank order" functions reduce in fp32 exactly as the
 * deterministic mode is defined (acc = x_0; acc = fl32(acc + x_r) for
 * r = 1..R-1); the "f64" functions reduce in double as the accuracy reference.
 *
 * Parity status: every function here is pinned by tests that do not call it
 * twice (closed forms, exact integer sums, correctly rounded sums, hand-derived
 * rounding cases, library bf16 conversion, the byte layout of a packed
 * fp64 + u32 record).
 */
#ifndef RCC_ORACLE_H
#define RCC_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
#define ORC_F32 0
#define ORC_BF16 1
/* reduction operations */
#define ORC_SUM 0
#define ORC_MEAN 1
#define ORC_MAX 2
#define ORC_MIN 3

/* ---- element conversions ------------------------------------------------ */
float orc_bf16_to_f32(uint16_t b);
/* round-to-nearest-even fp32 -> bf16; NaN stays a quiet NaN */
uint16_t orc_f32_to_bf16_rne(float f);
/* round-to-nearest-even fp64 -> bf16 (one rounding, used for the fp64 reference) */
uint16_t orc_f64_to_bf16_rne(double d);
/* element-wise array forms of the two conversions above */
void orc_f32_to_bf16_rne_n(const float* x, size_t n, uint16_t* out);
void orc_f64_to_bf16_rne_n(const double* x, size_t n, uint16_t* out);

/* ---- per-element reductions over R rank buffers ------------------------- */
/* out[i] = op over x[0][i], ..., x[R-1][i]; fp32 rank-order fold. */
void orc_reduce_f32(int R, const float* const* x, size_t n, int op, float* out);
/* same in fp64 (sum/mean in double; max/min exact) */
void orc_reduce_f64(int R, const float* const* x, size_t n, int op, double* out);
/* bf16: widen exactly, fp32 rank-order fold, one RNE rounding to bf16 */
void orc_reduce_bf16(int R, const uint16_t* const* x, size_t n, int op, uint16_t* out);
/* bf16 inputs reduced in fp64 (accuracy reference before rounding) */
void orc_reduce_bf16_f64(int R, const uint16_t* const* x, size_t n, int op, double* out);
/* sum over ranks of |x_r[i]| in fp64 (the error-bound scale) */
void orc_abs_sum_f64(int R, const float* const* x, size_t n, double* out);

/* ---- collectives (dtype ORC_F32 or ORC_BF16; rank-order fp32 arithmetic) --
 * Return 0 on success, -1 on a bad argument.  Outputs may alias inputs only
 * where noted. */
/* recv[r][i] = op_q send[q][i] for every r (recv[r] == send[r] allowed) */
int orc_all_reduce(int R, int dtype, int op, const void* const* send,
                   void* const* recv, size_t n);
/* root_recv[i] = op_q send[q][i]; nothing else is written */
int orc_reduce(int R, int dtype, int op, const void* const* send,
               void* root_recv, size_t n);
/* recv[r][i] = root_send[i] for every r with recv[r] != NULL */
int orc_broadcast(int R, int dtype, const void* root_send, void* const* recv,
                  size_t n);
/* recv[r][j] = op_q send[q][r*n_shard + j], n_in = R*n_shard per rank */
int orc_reduce_scatter(int R, int dtype, int op, const void* const* send,
                       void* const* recv, size_t n_in);
/* recv[r][q*n_shard + j] = send[q][j] for every r, q */
int orc_all_gather(int R, int dtype, const void* const* send,
                   void* const* recv, size_t n_shard);

/* all_to_all_single with equal splits, n_in = R*n_shard per rank:
 * recv[r][q*n_shard + j] = send[q][r*n_shard + j] for every r, q */
int orc_all_to_all(int R, int dtype, const void* const* send, void* const* recv,
                   size_t n_in);

/* ---- gradient sync + AdamW ---------------------------------------------- */

/* Running statistics of the unscaled mean gradient. */
typedef struct {
  double sum;      /* compensated (Neumaier) running sum of g^2 */
  double comp;     /* its compensation term */
  uint64_t nonfinite;
  uint64_t count;
} orc_stats;

/* g[i] = fl32( fl32(sum_q grads[q][i] in rank order) / R ) * inv_scale, fp32 */
void orc_mean_unscale(int R, const float* const* grads, size_t n,
                      float inv_scale, float* g);
/* stats += { sum of g[i]^2 (fp64), count of non-finite g[i] } */
void orc_stats_accumulate(orc_stats* st, const float* g, size_t n);
double orc_stats_value(const orc_stats* st);

/* the host-side decision after the report is read back */
typedef struct {
  int skip;          /* 1: non-finite gradient or norm -> whole step skipped */
  double norm;       /* sqrt(sum g^2) */
  float clip_coef;   /* fl32(max_norm / norm) when norm > max_norm, else 1 */
} orc_decision;
void orc_decide(const orc_stats* st, double max_grad_norm, orc_decision* d);

/* per-step scalars: fp64 host arithmetic rounded once to fp32 */
typedef struct {
  float step_size;      /* lr / (1 - beta1^t) */
  float inv_bc2_sqrt;   /* 1 / sqrt(1 - beta2^t) */
  float decay;          /* 1 - lr * weight_decay */
  float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
} orc_adamw_scalars;
void orc_adamw_scalars_for(double lr, double beta1, double beta2, double eps,
                           double weight_decay, int64_t t,
                           orc_adamw_scalars* s);
/* one AdamW element update over n elements (fp32) */
void orc_adamw_update(const float* g, size_t n, float clip_coef,
                      const orc_adamw_scalars* s, float* p, float* m, float* v);

/* GradScaler state */
typedef struct {
  double scale;
  double growth_factor;
  double backoff_factor;
  int32_t growth_interval;
  int32_t growth_tracker;
} orc_scaler;
void orc_scaler_update(orc_scaler* sc, int found_inf);

/* One complete step over P parameter tensors (small and medium sizes):
 * grads[p*R + q] is rank q's loss-scaled gradient of tensor p; params,
 * exp_avg, exp_avg_sq[p] one fp32 copy per tensor; *step is the count of
 * applied steps (incremented unless skipped); scaler is updated.  The
 * statistics and decision are returned in *st and *d. */
void orc_grad_sync_adamw_step(int R, int P, const size_t* numel,
                              const float* const* grads, float* const* params,
                              float* const* exp_avg, float* const* exp_avg_sq,
                              double lr, double beta1, double beta2, double eps,
                              double weight_decay, double max_grad_norm,
                              int64_t* step, orc_scaler* scaler, orc_stats* st,
                              orc_decision* d);

/* the 12-byte report [RUDA-T: 12 bytes read back before the update; the page
 * fixes only the size]: {fp64 sum of squares, u32 non-finite count} as three
 * little-endian u32 words (low word of the sum, high word, count); a count
 * beyond 2^32 - 1 is stored as 2^32 - 1 */
void orc_report_pack(const orc_stats* st, uint32_t out[3]);

#ifdef __cplusplus
}
#endif
#endif /* RCC_ORACLE_H */
