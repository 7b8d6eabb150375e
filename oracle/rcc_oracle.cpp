/*
 * rcc_oracle.cpp -- CPU oracle for the librcc hot path (TEST INFRASTRUCTURE).
 *
 * Plain single-threaded loops, no SIMD intrinsics, no threads.  Built with
 * -O2 -ffp-contract=off so that every fp32 operation below is rounded once,
 * in the order written, on every host architecture.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load this library.
 * See rcc_oracle.h for the sources each function follows.
 */
#include "rcc_oracle.h"

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <vector>

namespace {

uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}
float bits_f32(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

/* The canonical quiet NaN every max/min result carries when any input is NaN. */
const uint32_t kCanonicalNaN = 0x7FC00000u;

/*
 * One element of the fp32 rank-order reduction.  [ruCCL §2 all_reduce /
 * reduce rows; Monarch all_reduce "reduce ... across all ranks"].  The
 * deterministic mode fixes the order: acc = x_0, then acc = fl32(acc + x_r)
 * for r = 1..R-1.  Mean is fl32(sum / R) with one IEEE division.  Max and min
 * keep the running value unless a later rank is strictly greater (smaller), so
 * equal values (including +0/-0) keep the lowest rank's bits; any NaN input
 * makes the result the canonical quiet NaN.
 */
float reduce_one_f32(int R, const float* xs, int op) {
  if (op == ORC_SUM || op == ORC_MEAN) {
    float acc = xs[0];
    for (int r = 1; r < R; ++r) acc = acc + xs[r];
    if (op == ORC_MEAN) acc = acc / (float)R;
    return acc;
  }
  float acc = xs[0];
  bool nan = std::isnan(xs[0]);
  for (int r = 1; r < R; ++r) {
    float x = xs[r];
    if (std::isnan(x)) {
      nan = true;
    } else if (op == ORC_MAX ? (x > acc) : (x < acc)) {
      acc = x;
    }
  }
  return nan ? bits_f32(kCanonicalNaN) : acc;
}

/* The same reduction carried out in double: the accuracy reference. */
double reduce_one_f64(int R, const double* xs, int op) {
  if (op == ORC_SUM || op == ORC_MEAN) {
    double acc = xs[0];
    for (int r = 1; r < R; ++r) acc = acc + xs[r];
    if (op == ORC_MEAN) acc = acc / (double)R;
    return acc;
  }
  double acc = xs[0];
  bool nan = std::isnan(xs[0]);
  for (int r = 1; r < R; ++r) {
    double x = xs[r];
    if (std::isnan(x)) {
      nan = true;
    } else if (op == ORC_MAX ? (x > acc) : (x < acc)) {
      acc = x;
    }
  }
  return nan ? (double)bits_f32(kCanonicalNaN) : acc;
}

bool valid_op(int op) { return op >= ORC_SUM && op <= ORC_MIN; }
bool valid_dtype(int dt) { return dt == ORC_F32 || dt == ORC_BF16; }
size_t elem_size(int dt) { return dt == ORC_F32 ? 4 : 2; }

/* reduce element i of R rank buffers (any dtype) into a buffer of the same dtype */
void reduce_elements(int R, int dtype, int op, const void* const* src,
                     size_t src_off, size_t n, void* dst) {
  std::vector<float> xs(R);
  for (size_t i = 0; i < n; ++i) {
    for (int r = 0; r < R; ++r) {
      if (dtype == ORC_F32)
        xs[r] = static_cast<const float*>(src[r])[src_off + i];
      else
        xs[r] = orc_bf16_to_f32(static_cast<const uint16_t*>(src[r])[src_off + i]);
    }
    float y = reduce_one_f32(R, xs.data(), op);
    if (dtype == ORC_F32)
      static_cast<float*>(dst)[i] = y;
    else
      static_cast<uint16_t*>(dst)[i] = orc_f32_to_bf16_rne(y);
  }
}

}  // namespace

extern "C" {

/* ---- element conversions ------------------------------------------------ */

float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/*
 * fp32 -> bf16 with round-to-nearest, ties to even: keep the top 16 bits of
 * the fp32 pattern, adding half of the dropped range (minus one when the kept
 * low bit is even) before truncating.  A NaN keeps its sign and high payload
 * and is forced quiet.
 */
uint16_t orc_f32_to_bf16_rne(float f) {
  uint32_t u = f32_bits(f);
  if (std::isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  uint32_t rounded = u + 0x7FFFu + lsb;
  return (uint16_t)(rounded >> 16);
}

/*
 * fp64 -> bf16 with a single round-to-nearest-even: scale by the bf16 spacing
 * of the value's binade (2^(e-8) for |d| in [2^(e-1), 2^e), 2^-133 below the
 * normal range), round the scaled value to an integer with nearbyint (the
 * default ties-to-even mode), scale back.  Results that reach 2^128 are Inf.
 */
uint16_t orc_f64_to_bf16_rne(double d) {
  if (std::isnan(d)) return 0x7FC0u;
  if (std::isinf(d) || d == 0.0) return orc_f32_to_bf16_rne((float)d);
  int e;
  std::frexp(d, &e); /* |d| in [2^(e-1), 2^e) */
  int q = e - 8;
  if (q < -133) q = -133;
  double r = std::nearbyint(std::ldexp(d, -q));
  double y = std::ldexp(r, q);
  if (std::fabs(y) >= std::ldexp(1.0, 128)) y = d > 0 ? INFINITY : -INFINITY;
  /* y has at most 8 significant bits, so it converts to fp32 exactly */
  return (uint16_t)(f32_bits((float)y) >> 16);
}

void orc_f32_to_bf16_rne_n(const float* x, size_t n, uint16_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16_rne(x[i]);
}

void orc_f64_to_bf16_rne_n(const double* x, size_t n, uint16_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16_rne(x[i]);
}

/* ---- per-element reductions --------------------------------------------- */

void orc_reduce_f32(int R, const float* const* x, size_t n, int op, float* out) {
  std::vector<float> xs(R);
  for (size_t i = 0; i < n; ++i) {
    for (int r = 0; r < R; ++r) xs[r] = x[r][i];
    out[i] = reduce_one_f32(R, xs.data(), op);
  }
}

void orc_reduce_f64(int R, const float* const* x, size_t n, int op, double* out) {
  std::vector<double> xs(R);
  for (size_t i = 0; i < n; ++i) {
    for (int r = 0; r < R; ++r) xs[r] = (double)x[r][i];
    out[i] = reduce_one_f64(R, xs.data(), op);
  }
}

void orc_reduce_bf16(int R, const uint16_t* const* x, size_t n, int op,
                     uint16_t* out) {
  const void* const* src = reinterpret_cast<const void* const*>(x);
  reduce_elements(R, ORC_BF16, op, src, 0, n, out);
}

void orc_reduce_bf16_f64(int R, const uint16_t* const* x, size_t n, int op,
                         double* out) {
  std::vector<double> xs(R);
  for (size_t i = 0; i < n; ++i) {
    for (int r = 0; r < R; ++r) xs[r] = (double)orc_bf16_to_f32(x[r][i]);
    out[i] = reduce_one_f64(R, xs.data(), op);
  }
}

void orc_abs_sum_f64(int R, const float* const* x, size_t n, double* out) {
  for (size_t i = 0; i < n; ++i) {
    double s = 0.0;
    for (int r = 0; r < R; ++r) s += std::fabs((double)x[r][i]);
    out[i] = s;
  }
}

/* ---- collectives --------------------------------------------------------- */

/*
 * all_reduce [ruCCL §2 "returns the reduced result to the participants";
 * §5 CUDA example: sum/mean of 257 FP32 elements over 4 logical ranks, inputs
 * unchanged; Monarch all_reduce].  The result is formed in a temporary first,
 * so an output that is its own rank's input (in place) reads unmodified data.
 */
int orc_all_reduce(int R, int dtype, int op, const void* const* send,
                   void* const* recv, size_t n) {
  if (R < 1 || !valid_dtype(dtype) || !valid_op(op)) return -1;
  if (n == 0) return 0;
  std::vector<unsigned char> tmp(n * elem_size(dtype));
  reduce_elements(R, dtype, op, send, 0, n, tmp.data());
  for (int r = 0; r < R; ++r) std::memcpy(recv[r], tmp.data(), tmp.size());
  return 0;
}

/* reduce to a root [ruCCL §2: non-root participants receive nothing;
 * Monarch reduce "writing the result out to tensor on the root rank"] */
int orc_reduce(int R, int dtype, int op, const void* const* send,
               void* root_recv, size_t n) {
  if (R < 1 || !valid_dtype(dtype) || !valid_op(op)) return -1;
  if (n == 0) return 0;
  std::vector<unsigned char> tmp(n * elem_size(dtype));
  reduce_elements(R, dtype, op, send, 0, n, tmp.data());
  std::memcpy(root_recv, tmp.data(), tmp.size());
  return 0;
}

/* broadcast [ruCCL §2: the sender passes Some(tensor), receivers None;
 * Monarch broadcast "data on the root rank to all the others"] */
int orc_broadcast(int R, int dtype, const void* root_send, void* const* recv,
                  size_t n) {
  if (R < 1 || !valid_dtype(dtype)) return -1;
  size_t bytes = n * elem_size(dtype);
  for (int r = 0; r < R; ++r)
    if (recv[r] != nullptr && recv[r] != root_send && bytes)
      std::memmove(recv[r], root_send, bytes);
  return 0;
}

/* reduce_scatter_tensor [Monarch: "Reduce, then scatters the result"]:
 * rank r receives the r-th of R equal shards of the reduced tensor. */
int orc_reduce_scatter(int R, int dtype, int op, const void* const* send,
                       void* const* recv, size_t n_in) {
  if (R < 1 || !valid_dtype(dtype) || !valid_op(op)) return -1;
  if (n_in % (size_t)R != 0) return -1;
  size_t shard = n_in / (size_t)R;
  for (int r = 0; r < R; ++r)
    reduce_elements(R, dtype, op, send, (size_t)r * shard, shard, recv[r]);
  return 0;
}

/* all_gather_into_tensor [Monarch: "Gather tensors from all ranks into a
 * single output tensor"]: rank q's input is placed at offset q*n_shard. */
int orc_all_gather(int R, int dtype, const void* const* send,
                   void* const* recv, size_t n_shard) {
  if (R < 1 || !valid_dtype(dtype)) return -1;
  size_t es = elem_size(dtype);
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q)
      std::memcpy(static_cast<unsigned char*>(recv[r]) + (size_t)q * n_shard * es,
                  send[q], n_shard * es);
  return 0;
}

/* all_to_all_single [Monarch: split the input, scatter the split list to
 * all ranks, concatenate what each receives]: equal splits, so rank q's
 * chunk r lands on rank r at position q. */
int orc_all_to_all(int R, int dtype, const void* const* send, void* const* recv,
                   size_t n_in) {
  if (R < 1 || !valid_dtype(dtype)) return -1;
  if (n_in % (size_t)R != 0) return -1;
  const size_t shard = n_in / (size_t)R, es = elem_size(dtype);
  for (int r = 0; r < R; ++r)
    for (int q = 0; q < R; ++q)
      std::memcpy(static_cast<unsigned char*>(recv[r]) + (size_t)q * shard * es,
                  static_cast<const unsigned char*>(send[q]) + (size_t)r * shard * es,
                  shard * es);
  return 0;
}

/* ---- gradient sync + AdamW ---------------------------------------------- */

/*
 * The gradient all-reduce with ReduceOperation::Mean [ruCCL §6], taken on the
 * loss-scaled gradients and then unscaled [RUDA-T native PyTorch section:
 * clipping happens "after unscale"]: mean in rank order, then one fp32
 * multiply by inv_scale = fl32(1/S).
 */
void orc_mean_unscale(int R, const float* const* grads, size_t n,
                      float inv_scale, float* g) {
  std::vector<float> xs(R);
  for (size_t i = 0; i < n; ++i) {
    for (int r = 0; r < R; ++r) xs[r] = grads[r][i];
    float mean = reduce_one_f32(R, xs.data(), ORC_MEAN);
    g[i] = mean * inv_scale;
  }
}

/*
 * Read-only gradient analysis [RUDA-T]: the squared L2 norm, summed in double
 * with Neumaier compensation (g^2 is exact in double), and the count of
 * non-finite elements.  Non-finite elements are counted, not summed: any of
 * them skips the step, so the sum is then unused.
 */
void orc_stats_accumulate(orc_stats* st, const float* g, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    st->count += 1;
    if (!std::isfinite(g[i])) {
      st->nonfinite += 1;
      continue;
    }
    double x = (double)g[i] * (double)g[i];
    double t = st->sum + x;
    if (std::fabs(st->sum) >= std::fabs(x))
      st->comp += (st->sum - t) + x;
    else
      st->comp += (x - t) + st->sum;
    st->sum = t;
  }
}

double orc_stats_value(const orc_stats* st) { return st->sum + st->comp; }

/*
 * The decision made on the host after the report is read back [RUDA-T]: a
 * non-finite gradient (or norm) skips the whole step; otherwise the global
 * L2 norm is clipped to max_grad_norm exactly when it exceeds it.
 */
void orc_decide(const orc_stats* st, double max_grad_norm, orc_decision* d) {
  double sumsq = orc_stats_value(st);
  d->norm = std::sqrt(sumsq);
  d->skip = (st->nonfinite > 0 || !std::isfinite(d->norm)) ? 1 : 0;
  d->clip_coef = 1.0f;
  if (!d->skip && max_grad_norm > 0.0 && d->norm > max_grad_norm)
    d->clip_coef = (float)(max_grad_norm / d->norm);
}

/* AdamW per-step scalars, fp64 on the host and rounded once to fp32
 * (bias corrections 1 - beta^t per Kingma & Ba; decoupled decay 1 - lr*wd). */
void orc_adamw_scalars_for(double lr, double beta1, double beta2, double eps,
                           double weight_decay, int64_t t,
                           orc_adamw_scalars* s) {
  double bc1 = 1.0 - std::pow(beta1, (double)t);
  double bc2 = 1.0 - std::pow(beta2, (double)t);
  s->step_size = (float)(lr / bc1);
  s->inv_bc2_sqrt = (float)(1.0 / std::sqrt(bc2));
  s->decay = (float)(1.0 - lr * weight_decay);
  s->beta1 = (float)beta1;
  s->one_minus_beta1 = (float)(1.0 - beta1);
  s->beta2 = (float)beta2;
  s->one_minus_beta2 = (float)(1.0 - beta2);
  s->eps = (float)eps;
}

/*
 * One AdamW update (Loshchilov & Hutter Algorithm 2 with the learning-rate-
 * scaled decay), fp32 master weights and moments [RUDA-T: "master parameters
 * and moments are FP32"], each operation rounded once:
 *   g' = g * coef                      clipped gradient
 *   p  = p * (1 - lr*wd)               decoupled weight decay
 *   m  = beta1*m + (1-beta1)*g'
 *   v  = beta2*v + (1-beta2)*(g'*g')
 *   p  = p - step_size * (m / (sqrt(v) * inv_bc2_sqrt + eps))
 */
void orc_adamw_update(const float* g, size_t n, float clip_coef,
                      const orc_adamw_scalars* s, float* p, float* m, float* v) {
  for (size_t i = 0; i < n; ++i) {
    float gp = g[i] * clip_coef;
    float pi = p[i] * s->decay;
    float mi = s->beta1 * m[i] + s->one_minus_beta1 * gp;
    float vi = s->beta2 * v[i] + s->one_minus_beta2 * (gp * gp);
    float denom = std::sqrt(vi) * s->inv_bc2_sqrt + s->eps;
    pi = pi - s->step_size * (mi / denom);
    p[i] = pi;
    m[i] = mi;
    v[i] = vi;
  }
}

/* GradScaler.update(): back off on an inf/NaN step, grow after
 * growth_interval consecutive finite steps [RUDA-T: scale -> step -> update
 * on the same GradScaler instance]. */
void orc_scaler_update(orc_scaler* sc, int found_inf) {
  if (found_inf) {
    sc->scale *= sc->backoff_factor;
    sc->growth_tracker = 0;
    return;
  }
  sc->growth_tracker += 1;
  if (sc->growth_tracker >= sc->growth_interval) {
    sc->scale *= sc->growth_factor;
    sc->growth_tracker = 0;
  }
}

/*
 * One full gradient-sync step in the pages' order [ruCCL §6; RUDA-T]:
 * all-reduce Mean + unscale -> read-only analysis -> report -> skip on
 * non-finite -> clip after unscale -> one AdamW update per parameter tensor
 * -> GradScaler update.
 */
void orc_grad_sync_adamw_step(int R, int P, const size_t* numel,
                              const float* const* grads, float* const* params,
                              float* const* exp_avg, float* const* exp_avg_sq,
                              double lr, double beta1, double beta2, double eps,
                              double weight_decay, double max_grad_norm,
                              int64_t* step, orc_scaler* scaler, orc_stats* st,
                              orc_decision* d) {
  float inv_scale = (float)(1.0 / scaler->scale);
  std::vector<std::vector<float>> g(P);
  *st = orc_stats{0.0, 0.0, 0, 0};
  for (int p = 0; p < P; ++p) {
    g[p].resize(numel[p]);
    orc_mean_unscale(R, grads + (size_t)p * R, numel[p], inv_scale, g[p].data());
    orc_stats_accumulate(st, g[p].data(), numel[p]);
  }
  orc_decide(st, max_grad_norm, d);
  if (d->skip) {
    orc_scaler_update(scaler, 1);
    return;
  }
  int64_t t = *step + 1;
  orc_adamw_scalars s;
  orc_adamw_scalars_for(lr, beta1, beta2, eps, weight_decay, t, &s);
  for (int p = 0; p < P; ++p)
    orc_adamw_update(g[p].data(), numel[p], d->clip_coef, &s, params[p],
                     exp_avg[p], exp_avg_sq[p]);
  *step = t;
  orc_scaler_update(scaler, 0);
}

void orc_report_pack(const orc_stats* st, uint32_t out[3]) {
  double s = orc_stats_value(st);
  uint64_t u;
  std::memcpy(&u, &s, 8);
  out[0] = (uint32_t)(u & 0xFFFFFFFFu);
  out[1] = (uint32_t)(u >> 32);
  out[2] = (uint32_t)(st->nonfinite > 0xFFFFFFFFull ? 0xFFFFFFFFu : st->nonfinite);
}

}  // extern "C"
