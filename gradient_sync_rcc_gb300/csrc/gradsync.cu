// gradsync.cu -- the gradient-sync + fused AdamW kernel chain.
//
// [ruCCL README §6 "Collective training"]: gradients are all-reduced with
// ReduceOperation::Mean, then handed to the optimizer step.
// [RUDA docs "Training and saving state", section "Native PyTorch training on
// ruda:0"]: ruda_torch.AdamW(fused_step, max_grad_norm, hierarchical_stats)
// does a read-only gradient analysis, global L2 clipping after unscale, and
// hierarchical statistics (fan-in 1024, at most two extra combine kernels, a
// reused reduction region of at most 49,200 bytes, none for <= 1024 rows);
// a 12-byte report is read back before the update; a non-finite gradient
// skips the whole step; master weights and moments are FP32; the update is one
// kernel per parameter, not one kernel for the whole model.
//
// Kernels (all launched with programmatic dependent launch, launch.cuh):
//   gs_stats_kernel   all_reduce Mean of the R scaled gradients + unscale,
//                     optional store of the mean gradient, and one 12-byte row
//                     {sum g^2 (fp64), non-finite count (u32)} per block
//   gs_combine_kernel one fan-in-1024 combine level: 1024 rows -> 1 row
//   gs_report_kernel  the last <= 1024 rows (or all rows, flat) -> report,
//                     also stored to the host's mapped readback slot
//   gs_decide_kernel  the host's skip / clip decision taken on the GPU (the
//                     device-decision flows)
//   gs_update_kernel  one launch per tensor: clip, decoupled decay, moments,
//                     bias-corrected step on every optimizer-state replica
//                     (32-byte accesses when every pointer allows)
//   gs_update_multi_kernel  the same update for every tensor in one launch
//                     (a comparison flow)
//
// Row layout: three u32 words {low, high word of the fp64 sum, count}.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "launch.cuh"
#include "rcc.h"
#include "rcc_internal.h"

namespace rcc {
namespace gs {

constexpr int kFanIn = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint4 ld_vec(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_vec(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// 32-byte global accesses (sm_100 and later): one request per warp for 1 KiB.
struct Words8 {
  uint32_t w[8];
};

// An L2 policy that marks lines evict-first, for data read or written once:
// the scaled gradients in the statistics pass, so that the mean gradient
// written beside them is what L2 keeps; the optimizer state and the mean
// gradient's second (last) read in the per-tensor update kernels.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ Words8 ld_vec8(const void* p, uint64_t l2_policy) {
  Words8 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
      : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
        "=r"(v.w[6]), "=r"(v.w[7])
      : "l"(p), "l"(l2_policy));
  return v;
}

// Write-back store: the mean gradient is read again by the update kernels
// right after, so it is left to stay in L2 as long as it can.
__device__ __forceinline__ void st_vec8(void* p, const Words8& v) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

// ---- per-thread sum of squares -------------------------------------------
// The squares are summed in a pair of fp32 words (value + running error) with
// error-free transformations: the product error fmaf(g, g, -g*g) is exact and
// TwoSum keeps the addition error, so a thread's partial is good to ~2^-44
// relative before it is widened to fp64 -- without spending GB300's scarce
// fp64 issue slots on every element.  Magnitudes outside [2^-40, 2^40] (where
// the error terms could underflow or the pair could overflow) go straight to
// an fp64 accumulator.  Non-finite values are counted and not summed.
struct SqAcc {
  float hi = 0.0f, lo = 0.0f;
  double wide = 0.0;
  uint32_t nonfinite = 0;
  __device__ __forceinline__ void add(float g) {
    const float a = fabsf(g);
    if (a <= 0x1p40f && a >= 0x1p-40f) {
      const float p = __fmul_rn(g, g);
      const float pe = __fmaf_rn(g, g, -p);
      const float t = __fadd_rn(hi, p);
      const float bp = __fsub_rn(t, hi);
      const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(t, bp)), __fsub_rn(p, bp));
      hi = t;
      lo = __fadd_rn(lo, __fadd_rn(err, pe));
    } else if (!(a <= 3.402823466e38f)) {  // Inf or NaN
      nonfinite += 1;
    } else if (a != 0.0f) {
      wide += (double)g * (double)g;
    }
  }
  __device__ __forceinline__ double value() const {
    return (double)hi + (double)lo + wide;
  }
};

// Block-wide sums of s (fp64) and c, written as one 12-byte row.  The count
// is summed in 64 bits and stored saturated at 2^32 - 1: a combine level adds
// up to 1024 rows of up to 2^24 elements each, and a wrapped count could read
// as zero and let a step with non-finite gradients through.
__device__ __forceinline__ void block_reduce_row(double s, uint64_t c, uint32_t* row) {
  __shared__ double ws[kWarps];
  __shared__ unsigned long long wc[kWarps];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s += __shfl_down_sync(0xFFFFFFFFu, s, off);
    c += __shfl_down_sync(0xFFFFFFFFu, (unsigned long long)c, off);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    ws[warp] = s;
    wc[warp] = c;
  }
  __syncthreads();
  if (warp == 0) {
    s = lane < kWarps ? ws[lane] : 0.0;
    c = lane < kWarps ? wc[lane] : 0ull;
#pragma unroll
    for (int off = kWarps / 2; off > 0; off >>= 1) {
      s += __shfl_down_sync(0xFFFFFFFFu, s, off);
      c += __shfl_down_sync(0xFFFFFFFFu, (unsigned long long)c, off);
    }
    if (lane == 0) {
      const unsigned long long u = (unsigned long long)__double_as_longlong(s);
      row[0] = (uint32_t)(u & 0xFFFFFFFFull);
      row[1] = (uint32_t)(u >> 32);
      row[2] = c > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)c;
    }
  }
}

// The 12 report words (written by this thread) to the host's mapped slot,
// then the call's sequence number once the words are visible system-wide: the
// host polls the sequence word and reads the report after it.
__device__ __forceinline__ void publish_report(const uint32_t* report, uint32_t* host_copy,
                                               uint32_t seq) {
  host_copy[0] = report[0];
  host_copy[1] = report[1];
  host_copy[2] = report[2];
  __threadfence_system();
  *reinterpret_cast<volatile uint32_t*>(host_copy + 3) = seq;
}

// The decision the host would take from the report: skip on any non-finite
// gradient or norm, otherwise clip when the norm exceeds max_grad_norm.  IEEE
// double sqrt and division, then one rounding to fp32: the same bits as the
// host's computation.
__device__ __forceinline__ void decide_from_report(const uint32_t* report, double max_norm,
                                                   GsDecision* out) {
  const double sum_sq =
      __longlong_as_double((long long)(((unsigned long long)report[1] << 32) | report[0]));
  const double norm = sqrt(sum_sq);
  const uint32_t skip = (report[2] > 0u || !isfinite(norm)) ? 1u : 0u;
  float coef = 1.0f;
  if (!skip && max_norm > 0.0 && norm > max_norm) coef = __double2float_rn(max_norm / norm);
  out->skip = skip;
  out->coef = coef;
}

// s / R rounded once.  For R a power of two the product s * (1/R) is the
// same correctly rounded quotient -- scaling by 2^-k rounds the same real
// number once, subnormal results included -- at a fraction of a division's
// instructions; other R divide.
__device__ __forceinline__ float div_by_ranks(float s, int R) {
  return (R & (R - 1)) == 0 ? __fmul_rn(s, __frcp_rn((float)R)) : __fdiv_rn(s, (float)R);
}

// mean of R scaled gradients in rank order, then unscale: both steps fp32 IEEE
__device__ __forceinline__ float mean_unscale(const float* x, int R, float inv_scale) {
  float s = x[0];
  for (int q = 1; q < R; ++q) s = __fadd_rn(s, x[q]);
  return __fmul_rn(div_by_ranks(s, R), inv_scale);
}

// Register budget: 3 CTAs per SM at eight ranks (8 x 32-byte vectors in
// flight per thread), 4 below that.
template <int RC>  // RC > 0: compile-time rank count; 0: runtime (a.R)
__global__ void __launch_bounds__(kThreads, RC >= 8 ? 3 : 4) gs_stats_kernel(const __grid_constant__ GsStatsArgs a) {
  pdl_wait_then_release();
  const uint64_t row = blockIdx.x;
  const int R = RC > 0 ? RC : a.R;
  // warp 0 finds the tensor owning this row (the last t with row_begin <=
  // row) and stages it and its R gradient pointers in shared memory, so the
  // descriptor loads happen once per CTA rather than once per warp
  __shared__ GsTensor s_t;
  __shared__ const float* s_g[kMaxRanks];
  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) {
      uint32_t lo = 0, hi = a.num_tensors - 1;
      while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (a.tensors[mid].row_begin <= row)
          lo = mid;
        else
          hi = mid - 1;
      }
      s_t = a.tensors[lo];
    }
    __syncwarp();
    for (int q = threadIdx.x; q < R; q += 32) s_g[q] = a.grads[s_t.grad_slot + q];
  }
  __syncthreads();
  const GsTensor t = s_t;
  // read from shared memory at each use (volatile): held in registers the R
  // pointers would push the eight-rank kernel past its register budget
  const float* const volatile* g = s_g;
  const uint64_t c0 = (row - t.row_begin) * (uint64_t)a.elems_per_row;
  uint64_t c1 = c0 + a.elems_per_row;
  if (c1 > t.numel) c1 = t.numel;

  SqAcc acc;
  uint64_t scalar_from = c0;
  if constexpr (RC > 0) {
    if (t.vec_ok & 4u) {
      // 32-byte vectors: the host sets bit 2 only when every gradient (and
      // the mean gradient) is 32-byte aligned and elems_per_row is a
      // multiple of 8, so c0 starts a vector
      const uint64_t v0 = c0 / 8, v1 = c1 / 8;
      scalar_from = v1 * 8;
      const uint64_t pol = l2_evict_first_policy();
      for (uint64_t v = v0 + threadIdx.x; v < v1; v += kThreads) {
        Words8 x[RC];
#pragma unroll
        for (int q = 0; q < RC; ++q) x[q] = ld_vec8(g[q] + v * 8, pol);
        Words8 m;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float col[RC];
#pragma unroll
          for (int q = 0; q < RC; ++q) col[q] = __uint_as_float(x[q].w[e]);
          const float me = mean_unscale(col, RC, a.inv_scale);
          acc.add(me);
          m.w[e] = __float_as_uint(me);
        }
        if (t.mean_grad) st_vec8(t.mean_grad + v * 8, m);
      }
    }
  }
  if (scalar_from == c0 && (t.vec_ok & 1u)) {
    // c0 is a multiple of 4 (elems_per_row is), so vectors start aligned;
    // two vectors per rank in flight, one at eight ranks (register budget)
    constexpr int kU4 = RC >= 8 ? 1 : 2;
    const uint64_t v0 = c0 / 4, v1 = c1 / 4;
    scalar_from = v1 * 4;
    for (uint64_t v = v0 + threadIdx.x; v < v1; v += kU4 * kThreads) {
      uint4 x[kU4][RC > 0 ? RC : 1];
      if constexpr (RC > 0) {
#pragma unroll
        for (int u = 0; u < kU4; ++u) {
          const uint64_t vi = v + (uint64_t)u * kThreads;
          if (vi < v1) {
#pragma unroll
            for (int q = 0; q < RC; ++q) x[u][q] = ld_vec(g[q] + vi * 4);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU4; ++u) {
        const uint64_t vi = v + (uint64_t)u * kThreads;
        if (vi >= v1) continue;
        float m[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (RC > 0) {
            float col[RC];
#pragma unroll
            for (int q = 0; q < RC; ++q)
              col[q] = __uint_as_float(e == 0 ? x[u][q].x : e == 1 ? x[u][q].y
                                        : e == 2 ? x[u][q].z : x[u][q].w);
            m[e] = mean_unscale(col, RC, a.inv_scale);
          } else {
            float s = g[0][vi * 4 + e];
            for (int q = 1; q < R; ++q) s = __fadd_rn(s, g[q][vi * 4 + e]);
            m[e] = __fmul_rn(div_by_ranks(s, R), a.inv_scale);
          }
          acc.add(m[e]);
        }
        if (t.mean_grad)
          st_vec(t.mean_grad + vi * 4, make_uint4(__float_as_uint(m[0]), __float_as_uint(m[1]),
                                                  __float_as_uint(m[2]), __float_as_uint(m[3])));
      }
    }
  }
  for (uint64_t i = scalar_from + threadIdx.x; i < c1; i += kThreads) {
    float s = g[0][i];
    for (int q = 1; q < R; ++q) s = __fadd_rn(s, g[q][i]);
    const float m = __fmul_rn(div_by_ranks(s, R), a.inv_scale);
    acc.add(m);
    if (t.mean_grad) t.mean_grad[i] = m;
  }
  block_reduce_row(acc.value(), acc.nonfinite, a.rows + row * 3);
}

__device__ __forceinline__ double row_sum(const uint32_t* r) {
  return __longlong_as_double((long long)(((unsigned long long)r[1] << 32) | r[0]));
}

// one combine level: block b reduces rows [b*1024, min((b+1)*1024, nrows))
__global__ void __launch_bounds__(kThreads)
    gs_combine_kernel(const uint32_t* __restrict__ in, uint64_t nrows, uint32_t* __restrict__ out) {
  pdl_wait_then_release();
  const uint64_t r0 = (uint64_t)blockIdx.x * kFanIn;
  double s = 0.0;
  uint64_t c = 0;
#pragma unroll
  for (int k = 0; k < kFanIn / kThreads; ++k) {
    const uint64_t r = r0 + threadIdx.x + (uint64_t)k * kThreads;
    if (r < nrows) {
      s += row_sum(in + r * 3);
      c += in[r * 3 + 2];
    }
  }
  block_reduce_row(s, c, out + (uint64_t)blockIdx.x * 3);
}

// the final reduction into the 12-byte report (one block, any row count);
// thread 0, which wrote the report, also stores it to the host's mapped slot
__global__ void __launch_bounds__(kThreads)
    gs_report_kernel(const uint32_t* __restrict__ in, uint64_t nrows, uint32_t* __restrict__ report,
                     uint32_t* __restrict__ host_copy, uint32_t seq) {
  pdl_wait_then_release();
  double s = 0.0;
  uint64_t c = 0;
  for (uint64_t r = threadIdx.x; r < nrows; r += kThreads) {
    s += row_sum(in + r * 3);
    c += in[r * 3 + 2];
  }
  block_reduce_row(s, c, report);
  if (host_copy && threadIdx.x == 0) publish_report(report, host_copy, seq);
}

// ---- AdamW update ---------------------------------------------------------
// Element arithmetic, each operation rounded once (no contraction):
//   g' = g*coef; p = p*decay; m = b1*m + (1-b1)*g'; v = b2*v + (1-b2)*(g'*g');
//   p = p - step_size * (m / (sqrt(v)*inv_bc2_sqrt + eps))
__device__ __forceinline__ void adamw_elem(float g, const AdamWScalars& s, float& p,
                                           float& m, float& v) {
  const float pd = __fmul_rn(p, s.decay);
  const float mi = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.one_minus_beta1, g));
  const float vi = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.one_minus_beta2, __fmul_rn(g, g)));
  const float denom = __fadd_rn(__fmul_rn(__fsqrt_rn(vi), s.inv_bc2_sqrt), s.eps);
  p = __fsub_rn(pd, __fmul_rn(s.step_size, __fdiv_rn(mi, denom)));
  m = mi;
  v = vi;
}

// ---- the update body shared by the per-tensor and multi-tensor kernels ----
// P: one tensor's state pointer table, params[0..rep), exp_avg[0..rep),
// exp_avg_sq[0..rep).  The gradient is the stored mean gradient, or it is
// recomputed from the R scaled gradients with the statistics kernel's
// arithmetic.

// The decision source: host values in the launch arguments, or (with a
// device decision) the skip flag, coefficient, scalars and inverse scale in
// device memory.  Fetched first, examined only after the first data loads are
// in flight.
struct StepView {
  GsDecision d;
  AdamWScalars sc;
  float inv_scale;
};

__device__ __forceinline__ StepView step_view(float clip, const AdamWScalars& s, float inv_scale,
                                            const GsDecision* decision,
                                            const AdamWScalars* dev_scalars) {
  StepView v;
  v.d.skip = 0u;
  v.d.coef = clip;
  v.sc = s;
  v.inv_scale = inv_scale;
  if (decision) {
    v.d = *decision;
    v.sc = *dev_scalars;
    v.inv_scale = v.sc.inv_scale;
  }
  return v;
}

// W consecutive floats: W = 4 (16-byte accesses) or W = 8 (32-byte accesses,
// used when every pointer of the tensor is 32-byte aligned).
template <int W>
struct FVec {
  float f[W];
};

// The update kernels' accesses carry the L2 policy `pol` when H is true (the
// per-tensor kernel: evict-first) and are plain 16-byte accesses when it is
// false (the multi-tensor launch, where the hinted form measured 7% slower on
// 1,024 tensors, 3.25 against 3.04 ms, whatever the policy).

// The mean gradient: read-only for the update kernel, read once.
template <int W, bool H>
__device__ __forceinline__ FVec<W> ld_grad(const float* p, uint64_t pol) {
  static_assert(H || W == 4, "plain accesses are 16-byte");
  FVec<W> v;
  if constexpr (!H) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.f[0]), "=f"(v.f[1]), "=f"(v.f[2]), "=f"(v.f[3])
                 : "l"(p));
  } else if constexpr (W == 4) {
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=f"(v.f[0]), "=f"(v.f[1]), "=f"(v.f[2]), "=f"(v.f[3])
                 : "l"(p), "l"(pol));
  } else {
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
        : "=f"(v.f[0]), "=f"(v.f[1]), "=f"(v.f[2]), "=f"(v.f[3]), "=f"(v.f[4]), "=f"(v.f[5]),
          "=f"(v.f[6]), "=f"(v.f[7])
        : "l"(p), "l"(pol));
  }
  return v;
}

// Scaled gradients and optimizer state: coherent loads (the state is written
// back by the same thread), no L1 allocation.
template <int W, bool H>
__device__ __forceinline__ FVec<W> ld_rw(const float* p, uint64_t pol) {
  static_assert(H || W == 4, "plain accesses are 16-byte");
  FVec<W> v;
  if constexpr (!H) {
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.f[0]), "=f"(v.f[1]), "=f"(v.f[2]), "=f"(v.f[3])
                 : "l"(p));
  } else if constexpr (W == 4) {
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=f"(v.f[0]), "=f"(v.f[1]), "=f"(v.f[2]), "=f"(v.f[3])
                 : "l"(p), "l"(pol));
  } else {
    asm volatile(
        "ld.global.L1::no_allocate.L2::cache_hint.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
        : "=f"(v.f[0]), "=f"(v.f[1]), "=f"(v.f[2]), "=f"(v.f[3]), "=f"(v.f[4]), "=f"(v.f[5]),
          "=f"(v.f[6]), "=f"(v.f[7])
        : "l"(p), "l"(pol));
  }
  return v;
}

// No "memory" clobber: the state loads and stores are all volatile asm, which
// stays in program order, and without the clobber the compiler may keep the
// tensor's pointers in registers instead of reloading them after every store.
template <int W, bool H>
__device__ __forceinline__ void st_rw(float* p, const FVec<W>& v, uint64_t pol) {
  static_assert(H || W == 4, "plain accesses are 16-byte");
  if constexpr (!H) {
    asm volatile("st.global.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.f[0]), "f"(v.f[1]),
                 "f"(v.f[2]), "f"(v.f[3]));
  } else if constexpr (W == 4) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(v.f[0]),
                 "f"(v.f[1]), "f"(v.f[2]), "f"(v.f[3]), "l"(pol));
  } else {
    asm volatile("st.global.L2::cache_hint.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8}, %9;" ::"l"(p),
                 "f"(v.f[0]), "f"(v.f[1]), "f"(v.f[2]), "f"(v.f[3]), "f"(v.f[4]), "f"(v.f[5]),
                 "f"(v.f[6]), "f"(v.f[7]), "l"(pol));
  }
}

// Elements [W*v, W*v + W) of one tensor.  Returns false (having written
// nothing) when the step is skipped.  The gradient and the first batch of
// state replicas are all loaded before any arithmetic; replicas beyond the
// batch (RB: 4 with 16-byte vectors; 1 with 32-byte ones, which keeps the
// kernel near 60 registers and 4 CTAs per SM) follow batch by batch.
// P(j): the tensor's state pointer j (params 0..rep), exp_avg rep..2rep,
// exp_avg_sq 2rep..3rep), from a table in device memory or from the launch
// arguments.
template <int REP, int W, bool H, typename StateAt>
__device__ __forceinline__ bool update_vec(StateAt P, int rep, const float* mean_grad,
                                           const float* const* grads, int R, uint64_t v,
                                           const StepView& sv, uint64_t pol) {
  constexpr int RBMAX = W == 8 ? 1 : 4;
  constexpr int RB = REP > 0 && REP < RBMAX ? REP : RBMAX;  // replicas per batch of loads
  const uint64_t off = v * W;
  FVec<W> g;
  if (mean_grad) {
    g = ld_grad<W, H>(mean_grad + off, pol);
  } else {
    g = ld_rw<W, H>(grads[0] + off, pol);
    for (int q = 1; q < R; ++q) {
      const FVec<W> y = ld_rw<W, H>(grads[q] + off, pol);
#pragma unroll
      for (int e = 0; e < W; ++e) g.f[e] = __fadd_rn(g.f[e], y.f[e]);
    }
  }
  FVec<W> p[RB], m[RB], w[RB];
#pragma unroll
  for (int k = 0; k < RB; ++k) {
    if (k < rep) {
      p[k] = ld_rw<W, H>(P(k) + off, pol);
      m[k] = ld_rw<W, H>(P(rep + k) + off, pol);
      w[k] = ld_rw<W, H>(P(2 * rep + k) + off, pol);
    }
  }
  if (sv.d.skip) return false;  // skipped step: state untouched
  if (!mean_grad) {
#pragma unroll
    for (int e = 0; e < W; ++e) g.f[e] = __fmul_rn(div_by_ranks(g.f[e], R), sv.inv_scale);
  }
#pragma unroll
  for (int e = 0; e < W; ++e) g.f[e] = __fmul_rn(g.f[e], sv.d.coef);
  for (int r0 = 0; r0 < rep; r0 += RB) {
    if (r0 > 0) {
#pragma unroll
      for (int k = 0; k < RB; ++k) {
        if (r0 + k < rep) {
          p[k] = ld_rw<W, H>(P(r0 + k) + off, pol);
          m[k] = ld_rw<W, H>(P(rep + r0 + k) + off, pol);
          w[k] = ld_rw<W, H>(P(2 * rep + r0 + k) + off, pol);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < RB; ++k) {
      if (r0 + k < rep) {
#pragma unroll
        for (int e = 0; e < W; ++e) adamw_elem(g.f[e], sv.sc, p[k].f[e], m[k].f[e], w[k].f[e]);
        st_rw<W, H>(P(r0 + k) + off, p[k], pol);
        st_rw<W, H>(P(rep + r0 + k) + off, m[k], pol);
        st_rw<W, H>(P(2 * rep + r0 + k) + off, w[k], pol);
      }
    }
  }
  return true;
}

// One element of one tensor (ragged tails and unaligned tensors); the caller
// has already checked the skip flag.
template <typename StateAt>
__device__ __forceinline__ void update_one(StateAt P, int rep, const float* mean_grad,
                                           const float* const* grads, int R, uint64_t i,
                                           const StepView& sv) {
  float g;
  if (mean_grad) {
    g = mean_grad[i];
  } else {
    float s = grads[0][i];
    for (int q = 1; q < R; ++q) s = __fadd_rn(s, grads[q][i]);
    g = __fmul_rn(div_by_ranks(s, R), sv.inv_scale);
  }
  g = __fmul_rn(g, sv.d.coef);
  for (int r = 0; r < rep; ++r) {
    float p = P(r)[i], m = P(rep + r)[i], w = P(2 * rep + r)[i];
    adamw_elem(g, sv.sc, p, m, w);
    P(r)[i] = p;
    P(rep + r)[i] = m;
    P(2 * rep + r)[i] = w;
  }
}

// One launch per tensor (the pages' design).  W: floats per vector (8 when
// the host found every pointer of the tensor 32-byte aligned, else 4; a.vec_ok
// 0 means scalars only).
template <int REP, int W>  // REP > 0: compile-time replica count; 0: runtime
__global__ void __launch_bounds__(kThreads) gs_update_kernel(const __grid_constant__ GsUpdateArgs a) {
  // The next kernel is released only once this CTA's vectors are done: these
  // kernels run on parallel chains, and CTAs released early would sit in SM
  // slots waiting while the other chains' kernels need them.
  pdl_wait();
  const int rep = REP > 0 ? REP : a.replicas;
  const StepView sv = step_view(a.clip_coef, a.s, a.inv_scale, a.decision, a.dev_scalars);
  const uint64_t nv = a.vec_ok ? a.numel / W : 0;
  const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
  const uint64_t nthreads = (uint64_t)gridDim.x * kThreads;
  const uint64_t pol = l2_evict_first_policy();
  auto body = [&](auto P) {
    for (uint64_t v = tid; v < nv; v += nthreads)
      if (!update_vec<REP, W, true>(P, rep, a.mean_grad, a.grads, a.R, v, sv, pol)) return;
    pdl_release();
    if (sv.d.skip) return;
    for (uint64_t i = nv * W + tid; i < a.numel; i += nthreads)
      update_one(P, rep, a.mean_grad, a.grads, a.R, i, sv);
  };
  // state pointers from the launch arguments (compile-time indices: constant
  // loads, no memory requests) when the host passed them by value
  if constexpr (REP > 0 && REP <= GsUpdateArgs::kInlineReplicas) {
    if (a.inl) {
      body([&](int j) { return a.inl_state[j]; });
      return;
    }
  }
  body([&](int j) { return a.state[j]; });
}

// One launch for every tensor: block b updates statistics row b (a chunk of
// elems_per_row elements of one tensor), the statistics kernel's partition.
template <int REP>
__global__ void __launch_bounds__(kThreads)
    gs_update_multi_kernel(const __grid_constant__ GsMultiUpdateArgs a) {
  pdl_wait_then_release();
  const int rep = REP > 0 ? REP : a.replicas;
  const StepView sv = step_view(a.clip_coef, a.s, a.inv_scale, a.decision, a.dev_scalars);
  const uint64_t row = blockIdx.x;
  uint32_t lo = 0, hi = a.num_tensors - 1;
  while (lo < hi) {
    const uint32_t mid = (lo + hi + 1) >> 1;
    if (a.tensors[mid].row_begin <= row)
      lo = mid;
    else
      hi = mid - 1;
  }
  const GsTensor t = a.tensors[lo];
  float* const* P = a.state + (size_t)lo * 3 * rep;
  const float* const* g = a.grads + t.grad_slot;
  const uint64_t c0 = (row - t.row_begin) * (uint64_t)a.elems_per_row;
  uint64_t c1 = c0 + a.elems_per_row;
  if (c1 > t.numel) c1 = t.numel;
  uint64_t scalar_from = c0;
  if (t.vec_ok & 2u) {
    const uint64_t v1 = c1 / 4;
    scalar_from = v1 * 4;
    auto at = [&](int j) { return P[j]; };
    for (uint64_t v = c0 / 4 + threadIdx.x; v < v1; v += kThreads)  // plain accesses: no policy
      if (!update_vec<REP, 4, false>(at, rep, t.mean_grad, g, a.R, v, sv, 0)) return;
  }
  if (sv.d.skip) return;
  for (uint64_t i = scalar_from + threadIdx.x; i < c1; i += kThreads)
    update_one([&](int j) { return P[j]; }, rep, t.mean_grad, g, a.R, i, sv);
}

// The decision kernel of the device-decision flows (decide_from_report above).
__global__ void gs_decide_kernel(const uint32_t* __restrict__ report, double max_norm,
                                 GsDecision* __restrict__ out) {
  pdl_wait_then_release();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  decide_from_report(report, max_norm, out);
}

int sm_count() {
  static int cached[256] = {};  // per device ordinal; benign race: same value
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 256) dev = 0;
  if (cached[dev] <= 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// Copies `words` 32-bit words from pinned host memory mapped into the
// device's address space, with SM loads instead of a copy engine: a small
// table then does not queue behind large host<->device copies that the caller
// has in flight on other streams.  The loads bypass the caches (ld.cv), since
// the host rewrites the staging memory between calls.
__global__ void __launch_bounds__(kThreads)
    gs_upload_kernel(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst, uint64_t words) {
  pdl_wait_then_release();
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < words;
       i += (uint64_t)gridDim.x * kThreads)
    dst[i] = __ldcv(src + i);
}

}  // namespace gs

cudaError_t launch_gs_stats(const GsStatsArgs& a, cudaStream_t stream) {
  if (a.total_rows == 0) return cudaSuccess;
  const dim3 grid((unsigned)a.total_rows), block(kThreads);
  switch (a.R) {
    case 1: return launch_kernel(gs::gs_stats_kernel<1>, grid, block, 0, stream, a);
    case 2: return launch_kernel(gs::gs_stats_kernel<2>, grid, block, 0, stream, a);
    case 4: return launch_kernel(gs::gs_stats_kernel<4>, grid, block, 0, stream, a);
    case 8: return launch_kernel(gs::gs_stats_kernel<8>, grid, block, 0, stream, a);
    default: return launch_kernel(gs::gs_stats_kernel<0>, grid, block, 0, stream, a);
  }
}

cudaError_t launch_gs_combine(const uint32_t* in, uint64_t nrows, uint32_t* out,
                              cudaStream_t stream) {
  const unsigned blocks = (unsigned)((nrows + gs::kFanIn - 1) / gs::kFanIn);
  return launch_kernel(gs::gs_combine_kernel, dim3(blocks), dim3(kThreads), 0, stream, in, nrows,
                       out);
}

cudaError_t launch_gs_report(const uint32_t* in, uint64_t nrows, uint32_t* report,
                             uint32_t* host_copy, uint32_t seq, cudaStream_t stream) {
  return launch_kernel(gs::gs_report_kernel, dim3(1), dim3(kThreads), 0, stream, in, nrows, report,
                       host_copy, seq);
}

cudaError_t launch_gs_update_multi(const GsMultiUpdateArgs& a, cudaStream_t stream) {
  if (a.total_rows == 0) return cudaSuccess;
  const dim3 grid((unsigned)a.total_rows), block(kThreads);
  switch (a.replicas) {
    case 1: return launch_kernel(gs::gs_update_multi_kernel<1>, grid, block, 0, stream, a);
    case 2: return launch_kernel(gs::gs_update_multi_kernel<2>, grid, block, 0, stream, a);
    case 4: return launch_kernel(gs::gs_update_multi_kernel<4>, grid, block, 0, stream, a);
    case 8: return launch_kernel(gs::gs_update_multi_kernel<8>, grid, block, 0, stream, a);
    default: return launch_kernel(gs::gs_update_multi_kernel<0>, grid, block, 0, stream, a);
  }
}

cudaError_t launch_host_upload(const void* src_mapped, void* dst, size_t bytes,
                               cudaStream_t stream) {
  const uint64_t words = bytes / 4;
  uint64_t blocks = (words + kThreads - 1) / kThreads;
  if (blocks > 64) blocks = 64;
  if (blocks < 1) blocks = 1;
  return launch_kernel(gs::gs_upload_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, stream,
                       static_cast<const uint32_t*>(src_mapped), static_cast<uint32_t*>(dst),
                       words);
}

cudaError_t launch_gs_decide(const uint32_t* report, double max_grad_norm, GsDecision* out,
                             cudaStream_t stream) {
  return launch_kernel(gs::gs_decide_kernel, dim3(1), dim3(32), 0, stream, report, max_grad_norm,
                       out);
}

template <int W>
cudaError_t launch_gs_update_w(const GsUpdateArgs& a, cudaStream_t stream) {
  const uint64_t units = a.vec_ok ? (a.numel + W - 1) / W : a.numel;
  uint64_t blocks = (units + kThreads - 1) / kThreads;
  // one vector per thread up to 64 CTAs per SM, grid-stride beyond
  const uint64_t cap = (uint64_t)gs::sm_count() * 64;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks), block(kThreads);
  switch (a.replicas) {
    case 1: return launch_kernel(gs::gs_update_kernel<1, W>, grid, block, 0, stream, a);
    case 2: return launch_kernel(gs::gs_update_kernel<2, W>, grid, block, 0, stream, a);
    case 4: return launch_kernel(gs::gs_update_kernel<4, W>, grid, block, 0, stream, a);
    case 8: return launch_kernel(gs::gs_update_kernel<8, W>, grid, block, 0, stream, a);
    default: return launch_kernel(gs::gs_update_kernel<0, W>, grid, block, 0, stream, a);
  }
}

cudaError_t launch_gs_update(const GsUpdateArgs& a, cudaStream_t stream) {
  return a.vec_ok == 32 ? launch_gs_update_w<8>(a, stream) : launch_gs_update_w<4>(a, stream);
}

// ---- statistics without allocation -----------------------------------------
// For callers that cannot allocate device memory at all: code running inside a
// CUDA-graph capture that forbids cudaMalloc, processes whose memory is owned
// by another runtime or pool, or integrations that may only pass their own
// buffers.  The statistics rows of one call live in this file-scope device
// array instead of session scratch.  Every GPU that loads the library holds it
// (196,800 bytes) until the process exits.  Host code may not use the array's
// name as a device address: rcc_grad_stats_noalloc looks the address up once
// per device with cudaGetSymbolAddress and passes it to the kernels.

namespace gs {

constexpr uint64_t kNoAllocMaxRows = 16384;
constexpr uint32_t kNoAllocElemsPerRow = 8192;
constexpr uint64_t kNoAllocMaxElems = kNoAllocMaxRows * kNoAllocElemsPerRow;
// statistics rows, then the <= 16 rows of the single combine level
static __device__ __align__(256) uint32_t g_noalloc_rows[(kNoAllocMaxRows + 16) * 3];

struct OneTensorArgs {
  const float* grads[kMaxRanks];  // R device pointers, passed by value
  float* mean_grad;
  uint32_t* rows;                 // device address of g_noalloc_rows
  uint64_t numel;
  int R;
  int vec_ok;
  float inv_scale;
};

// gs_stats_kernel for a single tensor whose R gradient pointers arrive in the
// launch arguments (no device pointer table, hence nothing to upload).
template <int RC>
__global__ void __launch_bounds__(kThreads)
    gs_stats_one_kernel(const __grid_constant__ OneTensorArgs a) {
  const uint64_t row = blockIdx.x;
  const int R = RC > 0 ? RC : a.R;
  const float* const* g = a.grads;
  const uint64_t c0 = row * (uint64_t)kNoAllocElemsPerRow;
  uint64_t c1 = c0 + kNoAllocElemsPerRow;
  if (c1 > a.numel) c1 = a.numel;

  SqAcc acc;
  uint64_t scalar_from = c0;
  if (a.vec_ok) {
    const uint64_t v0 = c0 / 4, v1 = c1 / 4;
    scalar_from = v1 * 4;
    for (uint64_t v = v0 + threadIdx.x; v < v1; v += 2 * kThreads) {
      uint4 x[2][RC > 0 ? RC : 1];
      if constexpr (RC > 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint64_t vi = v + (uint64_t)u * kThreads;
          if (vi < v1) {
#pragma unroll
            for (int q = 0; q < RC; ++q) x[u][q] = ld_vec(g[q] + vi * 4);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint64_t vi = v + (uint64_t)u * kThreads;
        if (vi >= v1) continue;
        float m[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (RC > 0) {
            float col[RC];
#pragma unroll
            for (int q = 0; q < RC; ++q)
              col[q] = __uint_as_float(e == 0 ? x[u][q].x : e == 1 ? x[u][q].y
                                        : e == 2 ? x[u][q].z : x[u][q].w);
            m[e] = mean_unscale(col, RC, a.inv_scale);
          } else {
            float s = g[0][vi * 4 + e];
            for (int q = 1; q < R; ++q) s = __fadd_rn(s, g[q][vi * 4 + e]);
            m[e] = __fmul_rn(__fdiv_rn(s, (float)R), a.inv_scale);
          }
          acc.add(m[e]);
        }
        if (a.mean_grad)
          st_vec(a.mean_grad + vi * 4, make_uint4(__float_as_uint(m[0]), __float_as_uint(m[1]),
                                                  __float_as_uint(m[2]), __float_as_uint(m[3])));
      }
    }
  }
  for (uint64_t i = scalar_from + threadIdx.x; i < c1; i += kThreads) {
    float s = g[0][i];
    for (int q = 1; q < R; ++q) s = __fadd_rn(s, g[q][i]);
    const float m = __fmul_rn(__fdiv_rn(s, (float)R), a.inv_scale);
    acc.add(m);
    if (a.mean_grad) a.mean_grad[i] = m;
  }
  block_reduce_row(acc.value(), acc.nonfinite, a.rows + row * 3);
}

}  // namespace gs

namespace {

std::mutex g_noalloc_mu;
// per device ordinal, set on first use and kept for the life of the process
// (a device reset would invalidate it; the header says not to call after one)
uint32_t* g_noalloc_dev_ptr[256] = {};

bool aligned16_ptr(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace rcc

extern "C" rcc_status rcc_grad_stats_noalloc(const float* const* grads, int num_ranks,
                                             size_t numel, double loss_scale,
                                             float* mean_grad, uint32_t* report,
                                             rcc_stream_t stream) {
  rcc::NvtxRange nvtx_range("rcc_grad_stats_noalloc");
  using namespace rcc;
  if (!grads || !report)
    return set_error(RCC_ERR_INVALID_ARGUMENT, "grads and report are required");
  if (num_ranks < 1 || num_ranks > kMaxRanks)
    return set_error(RCC_ERR_INVALID_ARGUMENT, "num_ranks outside [1, 64]");
  for (int r = 0; r < num_ranks; ++r)
    if (!grads[r]) return set_error(RCC_ERR_MISSING_REGISTRATION, "a rank supplies no gradient");
  if (numel == 0 || numel > gs::kNoAllocMaxElems)
    return set_error(RCC_ERR_INVALID_ARGUMENT,
                     "numel must be in [1, 134217728] (16384 rows of 8192 elements, the "
                     "size of the static statistics array)");
  if (!(std::isfinite(loss_scale) && loss_scale > 0.0))
    return set_error(RCC_ERR_INVALID_ARGUMENT, "loss_scale must be finite and > 0");
  if (reinterpret_cast<uintptr_t>(report) & 3u)
    return set_error(RCC_ERR_INVALID_ARGUMENT, "report must be 4-byte aligned");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(RCC_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= 256) return set_error(RCC_ERR_INVALID_ARGUMENT, "device ordinal >= 256");
  uint32_t* rows = nullptr;
  {
    // set-up, once per device, with that device current: the host-side name
    // of the array is not a device address, so fetch the real one
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_dev_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, gs::g_noalloc_rows);
      if (e != cudaSuccess) return set_error(RCC_ERR_CUDA, cudaGetErrorString(e));
      g_noalloc_dev_ptr[dev] = static_cast<uint32_t*>(p);
    }
    rows = g_noalloc_dev_ptr[dev];
  }
  gs::OneTensorArgs a{};
  bool vec = mean_grad == nullptr || aligned16_ptr(mean_grad);
  for (int r = 0; r < num_ranks; ++r) {
    a.grads[r] = grads[r];
    vec = vec && aligned16_ptr(grads[r]);
  }
  a.mean_grad = mean_grad;
  a.rows = rows;
  a.numel = numel;
  a.R = num_ranks;
  a.vec_ok = vec ? 1 : 0;
  a.inv_scale = (float)(1.0 / loss_scale);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const uint64_t nrows = (numel + gs::kNoAllocElemsPerRow - 1) / gs::kNoAllocElemsPerRow;
  const dim3 grid((unsigned)nrows);
  switch (num_ranks) {
    case 1: gs::gs_stats_one_kernel<1><<<grid, kThreads, 0, cs>>>(a); break;
    case 2: gs::gs_stats_one_kernel<2><<<grid, kThreads, 0, cs>>>(a); break;
    case 4: gs::gs_stats_one_kernel<4><<<grid, kThreads, 0, cs>>>(a); break;
    case 8: gs::gs_stats_one_kernel<8><<<grid, kThreads, 0, cs>>>(a); break;
    default: gs::gs_stats_one_kernel<0><<<grid, kThreads, 0, cs>>>(a); break;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return set_error(RCC_ERR_CUDA, cudaGetErrorString(e));
  uint64_t launched = 1;
  const uint32_t* src = rows;
  uint64_t n = nrows;
  if (n > (uint64_t)gs::kFanIn) {
    uint32_t* out = rows + gs::kNoAllocMaxRows * 3;
    if ((e = launch_gs_combine(src, n, out, cs)) != cudaSuccess)
      return set_error(RCC_ERR_CUDA, cudaGetErrorString(e));
    src = out;
    n = (n + gs::kFanIn - 1) / gs::kFanIn;
    ++launched;
  }
  if ((e = launch_gs_report(src, n, report, nullptr, 0u, cs)) != cudaSuccess)
    return set_error(RCC_ERR_CUDA, cudaGetErrorString(e));
  add_launches(launched + 1);
  return RCC_OK;
}
