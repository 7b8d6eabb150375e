// rcc_internal.h -- launch interface between the host layer (rcc_host.cpp)
// and the CUDA kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstddef>
#include <cstdint>
#include <cstdlib>

#include "rcc.h"

namespace rcc {

// RCC_NVTX=1 (read once per process): every C ABI call opens an NVTX range
// named after it, for a profiler's timeline.  Otherwise no NVTX call is made.
inline bool nvtx_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("RCC_NVTX");
    return v && v[0] == '1';
  }();
  return on;
}

struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name) : on(nvtx_enabled()) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kMaxRanks = 64;
constexpr int kThreads = 256;  // every collective / grad-sync kernel block

// Element-wise operation of a multi-pointer pass.
enum Red : int { kRedSum = 0, kRedMax = 1, kRedMin = 2, kRedCopy = 3 };

// One multi-pointer pass: for every segment s (blockIdx.y) and element i < n,
//   y = red(src_0[i], ..., src_{nsrc-1}[i])  (sources of segment s)
//   dst_d[i] = y for each destination d of segment s.
// Sources of segment s: src[s] alone when src_per_seg, else src[0..nsrc) each
// advanced by s * src_seg_stride elements.  Destinations likewise with
// dst_per_seg / dst_seg_stride.  This one shape covers all five collectives:
//   all_reduce      1 segment, R sources, R destinations
//   reduce          1 segment, R sources, 1 destination (the root's)
//   broadcast       1 segment, 1 source (root), R (or R-1) destinations
//   reduce_scatter  R segments, R sources at offset s*n, destination recv[s]
//   all_gather      R segments, source send[s], R destinations at offset s*n
//   all_to_all      R*R segments (a2a_ranks = R): segment q*R + r copies
//                   send[q] at offset r*n to recv[r] at offset q*n
struct MultiPtrArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  size_t n;
  size_t src_seg_stride;
  size_t dst_seg_stride;
  int nsrc;
  int ndst;
  int src_per_seg;
  int dst_per_seg;
  int a2a_ranks; // > 0: all-to-all addressing over this many ranks (see above)
  int mean_div;  // > 0: the sum is divided by this (IEEE division) before storing
  int vec_ok;    // alignment class in bytes (0, 16 or 32): every source and
                 // destination address, with segment offsets, is a multiple of
                 // it, so vectors of that many bytes may be used; with a
                 // `stage`, only the base addresses are
  int stage;     // kStageNone, or which side is aligned per segment (below)
};

// Segment offsets that are not vector-aligned while the base addresses are:
// kStageSources aligns the sources of each segment (reductions: vector loads,
// stores staged through shared memory); kStageDestinations aligns the
// destinations (copies: loads staged through shared memory, vector stores).
enum Stage : int { kStageNone = 0, kStageSources = 1, kStageDestinations = 2 };

// One launch of the pass for element type DT (0 fp32, 1 bf16) and reduction
// RED; FAST (sums over 4..8 sources) selects the pairwise tree.  Each
// combination the host names is instantiated in its own build object
// (collectives_part.cu).
namespace mp {
template <int DT, int RED, bool FAST>
cudaError_t launch_part(int nseg, const MultiPtrArgs& a, cudaStream_t stream);
}  // namespace mp

// ---- gradient sync -------------------------------------------------------

// Device-side description of one parameter tensor for the statistics kernel.
struct GsTensor {
  uint64_t numel;
  uint64_t row_begin;       // first statistics row of this tensor
  float* mean_grad;         // optional output of the unscaled mean gradient
  uint32_t grad_slot;       // index of this tensor's R grad pointers in the grad table
  uint32_t vec_ok;          // bit 0: all R grads (and mean_grad) 16-byte aligned;
                            // bit 1: so are all its state pointers (update vectors);
                            // bit 2: grads and mean_grad 32-byte aligned and rows
                            //        a multiple of 8 elements (32-byte statistics)
};

struct GsStatsArgs {
  const GsTensor* tensors;      // [num_tensors]
  const float* const* grads;    // [num_tensors * R] grad pointer table
  uint32_t* rows;               // [total_rows * 3]: {sum_sq lo, sum_sq hi, nonfinite}
  uint64_t total_rows;
  uint32_t num_tensors;
  uint32_t elems_per_row;
  int R;
  float inv_scale;
};

// Statistics pass: one 12-byte row per block.
cudaError_t launch_gs_stats(const GsStatsArgs& a, cudaStream_t stream);
// One fan-in-1024 combine level: ceil(nrows / 1024) output rows.
cudaError_t launch_gs_combine(const uint32_t* in, uint64_t nrows, uint32_t* out,
                              cudaStream_t stream);
// Copies `bytes` (a multiple of 4) from pinned host memory, given by its
// device alias, to device memory with a kernel (no copy engine).
cudaError_t launch_host_upload(const void* src_mapped, void* dst, size_t bytes,
                               cudaStream_t stream);
// Final reduction of nrows rows into the 12-byte report (one block); the
// same 12 bytes also go to `host_copy` (a mapped pinned slot) when non-null,
// followed by `seq` in host_copy[3] once they are visible to the host.
cudaError_t launch_gs_report(const uint32_t* in, uint64_t nrows, uint32_t* report,
                             uint32_t* host_copy, uint32_t seq, cudaStream_t stream);

struct AdamWScalars {
  float step_size;     // lr / (1 - beta1^t)
  float inv_bc2_sqrt;  // 1 / sqrt(1 - beta2^t)
  float decay;         // 1 - lr * wd
  float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
  float inv_scale;     // fl32(1 / S): used by the device-decision flow
};

// Written on the device by the decision kernel: the step is skipped, or every
// gradient is multiplied by coef.
struct GsDecision {
  uint32_t skip;
  float coef;
};

struct GsUpdateArgs {
  float* const* state;          // this tensor's state pointer table (device memory):
                                //   params[0..replicas), exp_avg[0..replicas), exp_avg_sq[0..replicas)
  const float* mean_grad;       // unscaled mean gradient, or NULL
  const float* const* grads;    // this tensor's R grads (device table), used when mean_grad is NULL
  uint64_t numel;
  int R;
  int replicas;
  int vec_ok;                   // alignment class of every pointer of the tensor, in
                                //   bytes: 32 (32-byte vectors), 16, or 0 (scalars)
  float inv_scale;
  float clip_coef;
  AdamWScalars s;
  const GsDecision* decision;       // device decision (skip, coef); NULL: use clip_coef and s
  const AdamWScalars* dev_scalars;  // device copy of the step scalars, used with decision
  // The state pointers by value when there are at most 4 copies: read from
  // the launch arguments instead of the table in device memory.  inl_state
  // has the table's layout.
  static constexpr int kInlineReplicas = 4;
  float* inl_state[3 * kInlineReplicas];
  int inl;                          // 1: use inl_state
};

cudaError_t launch_gs_update(const GsUpdateArgs& a, cudaStream_t stream);

// Every tensor's update in one launch (a comparison point for the one
// kernel per parameter the pages describe): block b updates statistics row b.
struct GsMultiUpdateArgs {
  const GsTensor* tensors;      // [num_tensors]
  const float* const* grads;    // grad pointer table
  float* const* state;          // state table: tensor p at p * 3 * replicas
  uint64_t total_rows;
  uint32_t num_tensors;
  uint32_t elems_per_row;
  int R;
  int replicas;
  float inv_scale;
  float clip_coef;
  AdamWScalars s;
  const GsDecision* decision;
  const AdamWScalars* dev_scalars;
};
cudaError_t launch_gs_update_multi(const GsMultiUpdateArgs& a, cudaStream_t stream);
// One thread turns the 12-byte report into the decision (same arithmetic as the host).
cudaError_t launch_gs_decide(const uint32_t* report, double max_grad_norm, GsDecision* out,
                             cudaStream_t stream);

// Host layer services for entry points defined outside rcc_host.cpp: record
// the calling thread's error text (returns st), count kernel launches.
rcc_status set_error(rcc_status st, const char* msg);
void add_launches(uint64_t n);

}  // namespace rcc
